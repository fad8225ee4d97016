// Row-kernel instantiations for float logits (one translation unit per type so
// the library's sources compile in parallel).
#include "ce_launch.cuh"

namespace ce {
CE_INSTANTIATE_ROWS(float)
}  // namespace ce
