// ce_launch.cuh -- launch helpers for the row kernels, instantiated once per
// element type in ce_rows_f32.cu / ce_rows_f16.cu / ce_rows_bf16.cu so the
// three translation units compile in parallel.
#pragma once

#include "ce_rows.cuh"
#include "ce_stream.cuh"

namespace ce {

// Raises a kernel's dynamic shared-memory limit to at least smem_bytes on the
// current device; remembered per (device, kernel), so repeated launches make
// no runtime call (defined in ce_api.cu).
cudaError_t ensure_max_smem(const void* fn, int smem_bytes);

// Programmatic dependent launch: a row kernel may be scheduled while the
// previous kernel on its stream finishes (its CTAs take SMs as that kernel's
// CTAs exit), and waits in griddep_wait() for that kernel's completion before
// it touches global memory.  Back-to-back calls overlap launch and scheduling
// with the previous call's tail (fp32 [32768, 4096] fwd+bwd: 167.7 -> 165.8 us).
// Writes the attribute into *a; returns the number of attributes written.
static inline int pdl_attr(cudaLaunchAttribute* a) {
  a->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a->val.programmaticStreamSerializationAllowed = 1;
  return 1;
}

// Instantiated shapes: NC consumer threads x CPT register-resident 16-byte
// chunks per thread.  Both hold 2048 chunks (32 KB) of a row slice per CTA.
//   NC = 256, CPT = 8: 9 warps, fewer threads with more elements each
//   NC = 512, CPT = 4: 17 warps, more threads with fewer elements each

template <typename T, int MODE, int NC, int CPT>
static const void* kptr() {
  return reinterpret_cast<const void*>(&ce_rows_kernel<T, MODE, NC, CPT>);
}

template <typename T, int NC, int CPT>
static const void* kptr_mode(int mode) {
  switch (mode) {
    case FWD: return kptr<T, FWD, NC, CPT>();
    case FWD_BWD: return kptr<T, FWD_BWD, NC, CPT>();
    case BWD: return kptr<T, BWD, NC, CPT>();
    case SOFTMAX: return kptr<T, SOFTMAX, NC, CPT>();
    default: return nullptr;
  }
}

// Kernel entry for (T, mode, variant); see kVariants.
template <typename T>
const void* rows_kernel_ptr(int mode, int variant) {
  switch (variant) {
    case 0: return kptr_mode<T, 256, 8>(mode);
    case 1: return kptr_mode<T, 512, 4>(mode);
    case 2: return kptr_mode<T, 128, 0>(mode);
    case 3: return kptr_mode<T, 256, 0>(mode);
    case 4: return kptr_mode<T, 512, 0>(mode);
    default: return nullptr;
  }
}

template <typename T>
cudaError_t rows_launch(int mode, int variant, const RowParams& p, int grid, int smem_bytes,
                        cudaStream_t stream) {
  const void* fn = rows_kernel_ptr<T>(mode, variant);
  const int NC = kVariants[variant].NC;
  if (fn == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = ensure_max_smem(fn, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(NC + 32), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (p.CL > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(p.CL);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  na += pdl_attr(attr + na);
  cfg.attrs = attr;
  cfg.numAttrs = na;
  void* args[] = {const_cast<RowParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// How many clusters (CTAs when CL == 1) of this kernel fit on the device at once.
template <typename T>
cudaError_t rows_max_active(int mode, int variant, int smem_bytes, int CL, int sm_count,
                            int* out) {
  const void* fn = rows_kernel_ptr<T>(mode, variant);
  const int NC = kVariants[variant].NC;
  if (fn == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = ensure_max_smem(fn, smem_bytes);
  if (e != cudaSuccess) return e;
  if (CL <= 1) {
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, NC + 32,
                                                      static_cast<size_t>(smem_bytes));
    *out = occ * sm_count;
    return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(CL), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(NC + 32), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(CL);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int ncl = 0;
  e = cudaOccupancyMaxActiveClusters(&ncl, fn, &cfg);
  *out = ncl;
  return e;
}

// ---- the warp-streaming kernel (ce_stream.cuh) ----
// kStreamKRes: register chunks a lane holds in the resident rows of the
// writing modes (0: stream the row twice)
constexpr int kStreamKRes = 16;

template <typename T>
const void* stream_kernel_ptr(int mode, bool resident) {
  switch (mode) {
    case FWD: return reinterpret_cast<const void*>(&ce_stream_kernel<T, FWD, 0>);
    case FWD_BWD:
      return resident ? reinterpret_cast<const void*>(&ce_stream_kernel<T, FWD_BWD, kStreamKRes>)
                      : reinterpret_cast<const void*>(&ce_stream_kernel<T, FWD_BWD, 0>);
    case BWD: return reinterpret_cast<const void*>(&ce_stream_kernel<T, BWD, 0>);
    case SOFTMAX:
      return resident ? reinterpret_cast<const void*>(&ce_stream_kernel<T, SOFTMAX, kStreamKRes>)
                      : reinterpret_cast<const void*>(&ce_stream_kernel<T, SOFTMAX, 0>);
    default: return nullptr;
  }
}

template <typename T>
cudaError_t stream_launch(int mode, bool resident, const StreamParams& p, int grid, int nwarps,
                          int smem_bytes, cudaStream_t stream) {
  const void* fn = stream_kernel_ptr<T>(mode, resident);
  if (fn == nullptr || nwarps < 1 || nwarps > kStreamMaxWarps) return cudaErrorInvalidValue;
  cudaError_t e = ensure_max_smem(fn, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(nwarps * 32), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = pdl_attr(attr);
  cfg.attrs = attr;
  void* args[] = {const_cast<StreamParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// CTAs of the streaming kernel that fit on one SM at once.
template <typename T>
cudaError_t stream_max_active(int mode, bool resident, int nwarps, int smem_bytes, int* per_sm) {
  const void* fn = stream_kernel_ptr<T>(mode, resident);
  if (fn == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = ensure_max_smem(fn, smem_bytes);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, fn, nwarps * 32,
                                                       static_cast<size_t>(smem_bytes));
}

#define CE_INSTANTIATE_ROWS(T)                                                                  \
  template const void* rows_kernel_ptr<T>(int, int);                                            \
  template cudaError_t rows_launch<T>(int, int, const RowParams&, int, int, cudaStream_t);      \
  template cudaError_t rows_max_active<T>(int, int, int, int, int, int*);                       \
  template const void* stream_kernel_ptr<T>(int, bool);                                         \
  template cudaError_t stream_launch<T>(int, bool, const StreamParams&, int, int, int,          \
                                        cudaStream_t);                                          \
  template cudaError_t stream_max_active<T>(int, bool, int, int, int*);

}  // namespace ce
