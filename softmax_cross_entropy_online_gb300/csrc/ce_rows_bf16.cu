// Row-kernel instantiations for __nv_bfloat16 logits (one translation unit per type so
// the library's sources compile in parallel).
#include "ce_launch.cuh"

namespace ce {
CE_INSTANTIATE_ROWS(__nv_bfloat16)
}  // namespace ce
