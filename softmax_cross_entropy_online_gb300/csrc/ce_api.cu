// ce_api.cu -- the C ABI (include/ce_gb300.h) of the cross-entropy rows:
// argument checks, the choice of kernel and launch shape for each (mode,
// dtype, V, M), the per-stream reduction scratch, the device error word, the
// launches, and the host helpers every entry point shares (ce_host.cuh).  Every
// computation happens in the kernels (ce_rows.cuh, ce_stream.cuh); this file
// only validates, plans and launches.  The tensor-core entry points (GEMM,
// fused linear + CE, attention) are in ce_api_tc.cu.
#include <array>
#include <atomic>
#include <cmath>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <thread>
#include <utility>

#include "../../include/ce_gb300.h"
#include "ce_host.cuh"
#include "ce_rows.cuh"
#include "ce_stream.cuh"

namespace ce {
template <typename T>
cudaError_t rows_launch(int mode, int variant, const RowParams& p, int grid, int smem_bytes,
                        cudaStream_t stream);
template <typename T>
cudaError_t rows_max_active(int mode, int variant, int smem_bytes, int CL, int sm_count,
                            int* out);
template <typename T>
cudaError_t stream_launch(int mode, bool resident, const StreamParams& p, int grid, int nwarps,
                          int smem_bytes, cudaStream_t stream);
template <typename T>
cudaError_t stream_max_active(int mode, bool resident, int nwarps, int smem_bytes, int* per_sm);
constexpr int kStreamKRes = 16;  // as in ce_launch.cuh
}  // namespace ce

namespace ce {
// Test hook: wait on a barrier that nothing completes; give up after limit_ns.
__global__ void ce_selftest_wait_kernel(unsigned int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    bool failed = false;
    mbar_wait<false>(smem_u32(&bar), 0u, err, failed, limit_ns);
    mbar_arrive(smem_u32(&bar));  // leave the barrier in a completed phase
  }
}

cudaError_t ensure_max_smem(const void* fn, int smem_bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> raised;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_pair(dev, fn);
  auto it = raised.find(key);
  if (it != raised.end() && it->second >= smem_bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess) raised[key] = smem_bytes;
  return e;
}

}  // namespace ce

// The device error word: bit 0 = a target outside [0, V), bit 1 = a bounded
// wait ran out.  One per device (each device's module has its own copy).
__device__ unsigned int g_ce_err_word;

namespace {

std::atomic<uint64_t> g_launches{0};

constexpr int kScratchPartials = 8192;   // > any persistent grid (152 SMs x 4 CTAs)

using ce_host::DeviceInfo;

std::mutex g_mu;
std::map<int, DeviceInfo> g_dev;
struct Scratch {
  double* partials = nullptr;
  unsigned int* ticket = nullptr;
};
std::map<std::pair<int, void*>, Scratch> g_scratch;

}  // namespace

namespace ce_host {

ce_status device_info(DeviceInfo& out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return CE_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ce_err_word) != cudaSuccess) return CE_ERR_CUDA;
    d.err = static_cast<unsigned int*>(p);
    it = g_dev.emplace(dev, d).first;
  }
  out = it->second;
  *dev_out = dev;
  return CE_OK;
}

void count_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace ce_host

namespace {

using ce_host::device_info;

// Reduction scratch for (device, stream): calls on one stream are ordered, so
// they can share it; different streams get their own.
ce_status scratch_for(int dev, void* stream, Scratch& out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(dev, stream);
  auto it = g_scratch.find(key);
  if (it == g_scratch.end()) {
    void* mem = nullptr;
    const size_t bytes = 256 + sizeof(double) * kScratchPartials;
    if (cudaMalloc(&mem, bytes) != cudaSuccess) return CE_ERR_CUDA;
    if (cudaMemset(mem, 0, 256) != cudaSuccess) return CE_ERR_CUDA;
    Scratch s;
    s.ticket = static_cast<unsigned int*>(mem);
    s.partials = reinterpret_cast<double*>(static_cast<char*>(mem) + 256);
    it = g_scratch.emplace(key, s).first;
  }
  out = it->second;
  return CE_OK;
}

int elem_size(ce_dtype d) {
  switch (d) {
    case CE_F32: return 4;
    case CE_F16: return 2;
    case CE_BF16: return 2;
    default: return 0;
  }
}

struct Plan {
  int variant = 0, R = 1, CL = 1, S = 0, stage_bytes = 0;
};

// Occupancy of a launch shape, looked up once per (device, kernel, shape):
// the runtime's occupancy query costs more host time than a small launch.
std::mutex g_occ_mu;
std::map<std::array<long long, 7>, int> g_occ;
template <typename F>
cudaError_t cached_occupancy(const std::array<long long, 7>& key, F query, int* out) {
  {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  const cudaError_t e = query(out);
  if (e == cudaSuccess) {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_occ[key] = *out;
  }
  return e;
}

constexpr int kMaxSliceBytes = 200 * 1024;  // one stage of one CTA, at most

// Upper bound of the 16-byte chunks one row (or R rows) can straddle.
long long chunks_for(long long bytes, bool aligned) {
  return aligned ? (bytes + 15) / 16 : (bytes + 15) / 16 + 1;
}

// Stage size of a launch shape, or 0 when the shape cannot hold the rows.
long long stage_bytes_for(int variant, int R, int CL, long long rb, bool aligned) {
  const int NC = ce::kVariants[variant].NC;
  const int CPT = ce::kVariants[variant].CPT;
  // a row group is a power of two of at least kMinGroupThreads threads: a
  // quarter warp, half a warp, or whole warps
  if (R < 1 || NC % R != 0) return 0;
  const int GT = NC / R;
  if (GT < ce::kMinGroupThreads || (GT & (GT - 1)) != 0) return 0;
  if (CL < 1 || CL > ce::kMaxCluster || (CL > 1 && R != 1)) return 0;
  const long long cpr = chunks_for(rb, aligned);
  if (CL == 1) {
    if (CPT > 0 && static_cast<long long>(NC / R) * CPT < cpr) return 0;
    return chunks_for(static_cast<long long>(R) * rb, aligned) * 16;
  }
  const long long per_cta = (cpr + CL - 1) / CL;
  if (CPT > 0 && per_cta > static_cast<long long>(NC) * CPT) return 0;
  return per_cta * 16;
}

// Default launch shapes of the unit kernel, from sweeps of every shape on
// GB300 (the forward and the longest rows default to the streaming kernel;
// these shapes serve them when the unit kernel is forced):
//  * rows up to 32 KB: R rows per unit of up to 64 KB.  The forward (read
//    only) uses 256 streaming consumer threads with one stage, three CTAs
//    per SM; the writing modes use 512 consumer threads with two stages, one
//    CTA per SM.
//  * rows of 32-54 KB, writing modes: two rows per unit, two stages.
//  * rows that fit one CTA twice over (up to ~108 KB): one row per unit and
//    no cluster, so no cross-CTA exchange: 512 threads with two stages for
//    the writing modes, 256 threads with one stage (two CTAs per SM) for the
//    forward.
//  * longer rows: split over a cluster into slices of at most 52 KB, 256
//    threads, two stages (two CTAs per SM); beyond 8 x 52 KB the slices grow
//    and each CTA keeps one stage.
// A small problem: rows of up to 32 KB and under one 64 KB unit per SM in all.
// There the launch and each unit's chain of latencies decide the time, not the
// bandwidth: the unit kernel's bandwidth shapes put one or two rows on each of
// the SMs' large CTAs.
bool small_problem(long long rb, bool aligned, long long M, int sm_count) {
  return chunks_for(rb, aligned) * 16 <= 32 * 1024 && M * rb <= sm_count * 64LL * 1024;
}

bool choose_plan(int mode, long long rb, bool aligned, long long M, int sm_count, Plan& pl) {
  const long long cpr = chunks_for(rb, aligned);
  if (small_problem(rb, aligned, M, sm_count)) {
    // 128-thread CTAs with one stage, R rows a unit with R the smallest power
    // of two that leaves at most one unit per SM.  Measured against the
    // bandwidth shapes: the fused fwd+bwd 3-15 % faster on eight shapes of
    // 0.5-4 MB (fp32 [256, 1024]: 7.4 against 8.7 us a call), the forward on
    // rows of up to 2 KB 11-13 % faster.  The forward on longer rows keeps the
    // streaming kernel, which this shape did not beat there.
    int R = 1;
    while ((M + R - 1) / R > sm_count && 128 / (2 * R) >= ce::kMinGroupThreads &&
           2 * R * rb <= 32 * 1024)
      R *= 2;
    for (; R >= 1; R /= 2) {
      const long long stage = stage_bytes_for(2, R, 1, rb, aligned);
      if (stage == 0) continue;
      pl = Plan{2, R, 1, 1, static_cast<int>(stage)};
      return true;
    }
  }
  if (cpr * 16 <= 32 * 1024) {
    // rows of up to 2 KB take the writing modes' shape in the forward too
    // (512 threads, 8-16 per row: 59% against 50% for fp32 V = 256)
    const bool fwd = mode == ce::FWD && rb > 2048;
    const int variant = fwd ? 3 : 4;
    const int NC = ce::kVariants[variant].NC;
    const long long budget = fwd ? 64 * 1024 : 128 * 1024;  // stage bytes per CTA
    int R = 1;
    // short rows share a warp: as few as kMinGroupThreads threads per row
    while (R * 2 <= NC / ce::kMinGroupThreads && static_cast<long long>(R) * 2 * rb <= 64 * 1024)
      R *= 2;
    const long long min_units = (fwd ? 3LL : 1LL) * sm_count;
    while (R > 1 && (M + R - 1) / R < min_units) R /= 2;
    for (; R >= 1; R /= 2) {
      const long long stage = stage_bytes_for(variant, R, 1, rb, aligned);
      if (stage == 0) continue;
      long long S = budget / stage;
      if (S > ce::kMaxStages) S = ce::kMaxStages;
      if (S < 1) S = 1;
      if (S * stage > 216 * 1024) continue;
      pl = Plan{variant, R, 1, static_cast<int>(S), static_cast<int>(stage)};
      return true;
    }
  }
  if (mode != ce::FWD && (M + 1) / 2 >= sm_count) {
    // rows of 32-54 KB in the writing modes: two rows per unit of up to 108 KB,
    // two stages (measured: 87-97% of the copy peak against 58-86% with one
    // row per unit, whose per-row merge is then amortised over too little)
    const long long stage = stage_bytes_for(4, 2, 1, rb, aligned);
    if (stage != 0 && 2 * stage <= 216 * 1024) {
      pl = Plan{4, 2, 1, 2, static_cast<int>(stage)};
      return true;
    }
  }
  {
    // the forward does best with two 256-thread CTAs per SM and one stage each
    const bool fwd = mode == ce::FWD;
    const int variant = fwd ? 3 : 4;
    const long long stage = stage_bytes_for(variant, 1, 1, rb, aligned);
    if (stage != 0 && 2 * stage <= 216 * 1024) {
      pl = Plan{variant, 1, 1, fwd ? 1 : 2, static_cast<int>(stage)};
      return true;
    }
  }
  for (int CL = 2; CL <= ce::kMaxCluster; ++CL) {
    const long long stage = stage_bytes_for(3, 1, CL, rb, aligned);
    if (stage == 0 || stage > 52 * 1024) continue;
    pl = Plan{3, 1, CL, 2, static_cast<int>(stage)};
    return true;
  }
  // very long rows: 8 CTAs with larger slices and one stage each, so that
  // several CTAs share an SM (measured: 513 KB rows run 1.6x faster than with
  // two stages and one CTA per SM)
  const long long stage = stage_bytes_for(3, 1, ce::kMaxCluster, rb, aligned);
  if (stage == 0 || stage > kMaxSliceBytes) return false;
  pl = Plan{3, 1, ce::kMaxCluster, 1, static_cast<int>(stage)};
  return true;
}

// Optional override for tuning sweeps: CE_PLAN="variant,R,CL,S" (variant
// indexes kVariants).  It is checked against the same limits as the automatic
// choice and ignored when it does not fit them.
void apply_env_plan(long long rb, bool aligned, Plan& pl) {
  const char* env = std::getenv("CE_PLAN");
  if (env == nullptr || *env == 0) return;
  int var = 0, R = 0, CL = 0, S = 0;
  if (std::sscanf(env, "%d,%d,%d,%d", &var, &R, &CL, &S) != 4) return;
  if (var < 0 || var >= ce::kNumVariants) return;
  const long long stage = stage_bytes_for(var, R, CL, rb, aligned);
  if (stage == 0 || S < 1 || S > ce::kMaxStages || stage * S > 220 * 1024) return;
  pl = Plan{var, R, CL, S, static_cast<int>(stage)};
}

// ---------------------------------------------------------------------------
// Launch shape of the warp-streaming kernel: nw warps per CTA (one CTA per
// SM), G warps per row, S ring slots of seg bytes per warp.
// ---------------------------------------------------------------------------
struct StreamPlan {
  int nw = 16, G = 1, S = 3, seg = 4096;
  bool res = false;  // resident rows (writing modes): one read of each row
};

// A resident plan holds every piece of a row in registers: 4 KB slots and at
// most 32 x kStreamKRes chunks a warp (the row's chunk count: exact for rows
// on the 16-byte grid, else an upper bound).
bool resident_fits(long long rb, bool aligned, int G, int seg) {
  const long long chunks = chunks_for(rb, aligned) + (aligned ? 0 : 1);
  return seg == 4096 && (chunks + G - 1) / G <= 32LL * ce::kStreamKRes;
}

// Launch shape of the streaming kernel, from sweeps on GB300 (16 warps per CTA
// with 4 KB slots beat every smaller CTA and other segment size measured):
//  * one pass (FWD, BWD): a warp per row while every warp gets at least six
//    rows; otherwise the fewest warps per row that give each group twelve,
//    keeping at least 8 KB of the row per warp.  Long pieces with enough rows
//    per group won (fp16 256 KB rows: 4 warps per row 97%, 16 warps 88%).
//  * two passes (FWD_BWD, SOFTMAX): 16 warps per row, so that the rows in
//    flight (one per CTA) stay in L2 until the second pass re-reads them.
bool choose_stream_plan(int mode, long long rb, int es, long long M, int sm_count,
                        StreamPlan& sp) {
  const int nw = ce::kStreamMaxWarps;
  const int seg = 4096;
  const bool two_pass = mode == ce::FWD_BWD || mode == ce::SOFTMAX;
  int G = 1;
  if (two_pass) {
    G = nw;
  } else if (mode == ce::FWD && es == 4) {
    // fp32 forward: pieces of 8 to 16 KB, one warp's two slots (measured on
    // rows of 8-64 KB: the best of G = 1..16 every time; 32 KB rows 95.7 ->
    // 87.4 us, 16 KB rows 90.4 -> 88.0 us against a warp per row)
    while (G < 8 && rb >= 16384LL * G) G *= 2;
  } else {
    const long long warps = static_cast<long long>(sm_count) * nw;
    if (M < 6 * warps) {
      while (G < nw && M * G < 12 * warps) G *= 2;
    }
    while (G > 1 && rb / G < 8192) G /= 2;
  }
  // rows shorter than a segment: one row per slot (the power of two that
  // holds every chunk a row can straddle), up to eight slots a warp
  int sg = seg;
  const long long row_span = (rb / 16 + 2) * 16;
  if (G == 1) {
    while (sg / 2 >= row_span && sg > 16) sg /= 2;
  }
  // ring depth per warp: two 4 KB slots for one pass, three for two passes
  // (measured: a third slot costs the one-pass modes up to 7%, and gains the
  // two-pass modes 2%); short rows take up to eight smaller slots
  const long long per_warp = two_pass ? 3 * 4096 : 2 * 4096;
  long long S = per_warp / sg;
  if (S < 2) S = 2;
  if (S > ce::kStreamMaxSlots) S = ce::kStreamMaxSlots;
  sp = StreamPlan{nw, G, static_cast<int>(S), sg};
  return true;
}

// Tuning overrides: CE_KERNEL=stream|unit forces a kernel; CE_SPLAN=
// "nw,G,S,seg[,res]" sets the streaming shape (seg a power of two of at least
// 16 bytes; res = 1 asks for resident rows in the writing modes), ignored
// unless it fits the kernel's limits.  Resident rows are never the default:
// measured, they tie with the unit kernel where pieces span two slots (fp32
// 4096: 90.3% against 90.1%) and lose where a row needs a whole CTA (bf16
// 50257: 54% against 78%, the CTA-wide merge stalls every warp's ring).
int env_kernel_choice() {
  const char* env = std::getenv("CE_KERNEL");
  if (env == nullptr) return 0;
  if (std::strcmp(env, "stream") == 0) return 1;
  if (std::strcmp(env, "unit") == 0) return 2;
  return 0;
}
void apply_env_stream_plan(int mode, long long rb, bool aligned, StreamPlan& sp) {
  const char* env = std::getenv("CE_SPLAN");
  if (env == nullptr || *env == 0) return;
  int nw = 0, G = 0, S = 0, seg = 0, res = 0;
  const int n = std::sscanf(env, "%d,%d,%d,%d,%d", &nw, &G, &S, &seg, &res);
  if (n != 4 && n != 5) return;
  if (nw < 1 || nw > ce::kStreamMaxWarps || G < 1 || (G & (G - 1)) != 0 || nw % G != 0) return;
  if (S < 1 || S > ce::kStreamMaxSlots || seg < 16 || (seg & (seg - 1)) != 0) return;
  if (static_cast<long long>(nw) * S * seg > 220 * 1024) return;
  const bool resident = res != 0 && (mode == ce::FWD_BWD || mode == ce::SOFTMAX);
  if (resident && !resident_fits(rb, aligned, G, seg)) return;
  sp = StreamPlan{nw, G, S, seg, resident};
}

// ---------------------------------------------------------------------------
// Reduction scratch for ce_fwd_bwd_inplace_noalloc.  It lives in the module's
// own device memory (a file-scope array), so that entry point never allocates:
// the first 256 bytes hold the ticket, then one fp64 partial sum per CTA.
// Every device that loads this library holds it until the process exits.
// ---------------------------------------------------------------------------
constexpr int kNoAllocPartials = 1024;
static __device__ __align__(256) unsigned char g_noalloc_scratch[256 + sizeof(double) * kNoAllocPartials];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_base[kMaxDevices] = {};

// The array's device address for the current device.  Host code only knows
// a host-side stand-in for the symbol, so the address is looked up once per
// device (with that device current) and kept.
ce_status noalloc_scratch(Scratch& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_base[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return CE_ERR_CUDA;
    g_noalloc_base[dev] = ptr;
  }
  char* base = static_cast<char*>(g_noalloc_base[dev]);
  out.ticket = reinterpret_cast<unsigned int*>(base);
  out.partials = reinterpret_cast<double*>(base + 256);
  return CE_OK;
}

}  // namespace

namespace ce_host {

// Suspend-time hint of the kernels' mbarrier waits (ns); CE_WAIT_HINT_NS
// overrides it for tuning sweeps.
unsigned int wait_hint_ns() {
  static const unsigned int hint = [] {
    const char* env = std::getenv("CE_WAIT_HINT_NS");
    long v = env ? std::strtol(env, nullptr, 10) : 0;
    return (v > 0 && v <= 1000000) ? static_cast<unsigned int>(v) : 20000u;
  }();
  return hint;
}

}  // namespace ce_host

namespace {

using ce_host::wait_hint_ns;

// Reduction scratch for a launch of `grid` CTAs: the module's static array
// (its ticket cleared on the stream first) or the per-stream buffer.
ce_status reduction_scratch(bool static_scratch, int dev, void* stream, int grid, Scratch& sc) {
  if (static_scratch) {
    if (grid > kNoAllocPartials) return CE_ERR_UNSUPPORTED;
    ce_status st = noalloc_scratch(sc);
    if (st != CE_OK) return st;
    if (cudaMemsetAsync(sc.ticket, 0, sizeof(unsigned int), static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return CE_ERR_CUDA;
    return CE_OK;
  }
  if (grid > kScratchPartials) return CE_ERR_UNSUPPORTED;
  return scratch_for(dev, stream, sc);
}

// The warp-streaming kernel; arguments already validated by launch_rows.
ce_status launch_stream(int mode, const void* logits, const int64_t* targets, const float* lse_in,
                        int64_t M, int64_t V, ce_dtype dtype, ce_reduction red, float* loss,
                        float* row_loss, float* lse_out, float grad_scale, void* stream,
                        const DeviceInfo& di, int dev, bool static_scratch, void* out_buf,
                        const StreamPlan& sp, __nv_bfloat16* g16 = nullptr,
                        long long g16_ld = 0) {
  const long long rb = static_cast<long long>(V) * elem_size(dtype);
  ce::StreamParams p;
  std::memset(&p, 0, sizeof(p));
  p.base = static_cast<char*>(const_cast<void*>(logits));
  p.targets = targets;
  p.lse_in = lse_in;
  p.row_loss = row_loss;
  p.lse_out = lse_out;
  p.loss = loss;
  p.err = di.err;
  p.M = M;
  p.V = V;
  p.row_bytes = rb;
  p.G = sp.G;
  int lg = 0;
  while ((1 << lg) < sp.G) ++lg;
  p.log_g = lg;
  p.S = sp.S;
  p.seg_bytes = sp.seg;
  {
    int sh = 0;
    while ((16 << sh) < sp.seg) ++sh;
    p.seg_shift = sh;
  }
  p.total_bytes = static_cast<long long>(M) * rb;
  p.wait_hint_ns = wait_hint_ns();
  p.out_delta = (out_buf == nullptr) ? 0
                                     : static_cast<long long>(reinterpret_cast<uintptr_t>(out_buf) -
                                                              reinterpret_cast<uintptr_t>(logits));
  p.grad_scale = grad_scale;
  p.mean = (red == CE_RED_MEAN) ? 1 : 0;
  p.g16 = g16;
  p.g16_ld = g16_ld;

  const int smem = sp.nw * sp.S * sp.seg;
  int per_sm = 0;
  cudaError_t e = cached_occupancy(
      {dev, sp.res ? 2 : 1, static_cast<long long>(dtype), mode, sp.nw, smem, 1},
      [&](int* out) {
        switch (dtype) {
          case CE_F32: return ce::stream_max_active<float>(mode, sp.res, sp.nw, smem, out);
          case CE_F16: return ce::stream_max_active<__half>(mode, sp.res, sp.nw, smem, out);
          default: return ce::stream_max_active<__nv_bfloat16>(mode, sp.res, sp.nw, smem, out);
        }
      },
      &per_sm);
  if (e != cudaSuccess || per_sm < 1) return CE_ERR_CUDA;
  const long long groups_per_cta = sp.nw / sp.G;
  long long grid = static_cast<long long>(per_sm) * di.sm_count;
  const long long need = (M + groups_per_cta - 1) / groups_per_cta;  // CTAs with a row
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;  // M == 0: one CTA writes the empty reduction

  if (loss != nullptr) {
    Scratch sc;
    const ce_status st = reduction_scratch(static_scratch, dev, stream, static_cast<int>(grid), sc);
    if (st != CE_OK) return st;
    p.partials = sc.partials;
    p.ticket = sc.ticket;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int g = static_cast<int>(grid);
  switch (dtype) {
    case CE_F32: e = ce::stream_launch<float>(mode, sp.res, p, g, sp.nw, smem, s); break;
    case CE_F16: e = ce::stream_launch<__half>(mode, sp.res, p, g, sp.nw, smem, s); break;
    default: e = ce::stream_launch<__nv_bfloat16>(mode, sp.res, p, g, sp.nw, smem, s); break;
  }
  if (e != cudaSuccess) return CE_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return CE_OK;
}

// Which row kernel runs a call (from sweeps on GB300): the streaming kernel
// for the forward on rows above 2 KB (1.1x to 2.3x the unit kernel) and for
// the writing modes once a row no longer fits one CTA's shared memory twice
// (where the unit kernel would split it over a cluster); the unit kernel for
// the writing modes on shorter rows, where its single read of each row
// (against the streaming kernel's read and L2 re-read) wins.
bool default_use_stream(int mode, long long rb, bool aligned) {
  // the forward: the unit kernel's sub-warp row groups for rows of up to 2 KB
  // (fp32 V = 256: 59% against the streaming kernel's 20%), streaming above
  if (mode == ce::FWD) return rb > 2048;
  const long long cpr = chunks_for(rb, aligned);
  return 2 * cpr * 16 > 216 * 1024;
}

// static_scratch: reduce through g_noalloc_scratch (its ticket is cleared on
// the stream before the launch) instead of the per-stream buffer.
// g16 (FWD_BWD on fp32 logits only): the gradient is written as bf16 rows of
// g16_ld elements into g16 instead of over the logits (streaming kernel).
ce_status launch_rows(int mode, const void* logits, const int64_t* targets, const float* lse_in,
                      int64_t M, int64_t V, ce_dtype dtype, ce_reduction red, float* loss,
                      float* row_loss, float* lse_out, float grad_scale, void* stream,
                      bool static_scratch = false, void* out_buf = nullptr,
                      __nv_bfloat16* g16 = nullptr, long long g16_ld = 0) {
  const int es = elem_size(dtype);
  if (es == 0) return CE_ERR_INVALID_ARG;
  if (red != CE_RED_MEAN && red != CE_RED_SUM && red != CE_RED_NONE) return CE_ERR_INVALID_ARG;
  if (M < 0 || V < 1) return CE_ERR_INVALID_ARG;
  if (M > 0 && (logits == nullptr || (targets == nullptr && mode != ce::SOFTMAX)))
    return CE_ERR_INVALID_ARG;
  if (mode == ce::BWD && M > 0 && lse_in == nullptr) return CE_ERR_INVALID_ARG;
  const uintptr_t lb = reinterpret_cast<uintptr_t>(logits);
  if (lb % es) return CE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(targets) % 8) return CE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(loss) % 4 || reinterpret_cast<uintptr_t>(row_loss) % 4 ||
      reinterpret_cast<uintptr_t>(lse_out) % 4 || reinterpret_cast<uintptr_t>(lse_in) % 4)
    return CE_ERR_INVALID_ARG;
  if (V > (INT64_MAX / 4) / es) return CE_ERR_INVALID_ARG;
  const long long rb = static_cast<long long>(V) * es;
  if (M > 0 && M > INT64_MAX / rb) return CE_ERR_INVALID_ARG;
  if (red == CE_RED_NONE) loss = nullptr;
  if (mode == ce::BWD) loss = nullptr;
  if (M == 0 && loss == nullptr) return CE_OK;

  DeviceInfo di;
  int dev = 0;
  ce_status st = device_info(di, &dev);
  if (st != CE_OK) return st;

  const bool aligned = (lb % 16 == 0) && (rb % 16 == 0);
  if (V > ce_max_vocab(dtype)) return CE_ERR_UNSUPPORTED;  // the same limit for both kernels
  if (g16 != nullptr) {
    if (mode != ce::FWD_BWD || dtype != CE_F32 || out_buf != nullptr || g16_ld < V ||
        (g16_ld % 4) || (reinterpret_cast<uintptr_t>(g16) % 16))
      return CE_ERR_INVALID_ARG;
    StreamPlan sp;
    if (!choose_stream_plan(mode, rb, es, M, di.sm_count, sp)) return CE_ERR_UNSUPPORTED;
    sp.res = false;
    return launch_stream(mode, logits, targets, lse_in, M, V, dtype, red, loss, row_loss, lse_out,
                         grad_scale, stream, di, dev, static_scratch, out_buf, sp, g16, g16_ld);
  }
  {
    const int forced = env_kernel_choice();
    const bool use_stream = forced == 1 || (forced == 0 && default_use_stream(mode, rb, aligned));
    StreamPlan sp;
    if (use_stream && choose_stream_plan(mode, rb, es, M, di.sm_count, sp)) {
      apply_env_stream_plan(mode, rb, aligned, sp);
      return launch_stream(mode, logits, targets, lse_in, M, V, dtype, red, loss, row_loss,
                           lse_out, grad_scale, stream, di, dev, static_scratch, out_buf, sp);
    }
  }
  Plan pl;
  if (!choose_plan(mode, rb, aligned, M, di.sm_count, pl)) return CE_ERR_UNSUPPORTED;
  apply_env_plan(rb, aligned, pl);

  ce::RowParams p;
  std::memset(&p, 0, sizeof(p));
  p.base = static_cast<char*>(const_cast<void*>(logits));
  p.targets = targets;
  p.lse_in = lse_in;
  p.row_loss = row_loss;
  p.lse_out = lse_out;
  p.loss = loss;
  p.err = di.err;
  p.M = M;
  p.V = V;
  p.row_bytes = rb;
  p.R = pl.R;
  p.CL = pl.CL;
  p.S = pl.S;
  p.stage_bytes = pl.stage_bytes;
  p.q_chunks = pl.stage_bytes / 16;
  p.wait_hint_ns = wait_hint_ns();
  {
    const int GT = ce::kVariants[pl.variant].NC / pl.R;  // a power of two
    int lg = 0;
    while ((1 << lg) < GT) ++lg;
    p.log_gt = lg;
  }
  p.n_units = (M + pl.R - 1) / pl.R;
  p.grad_scale = grad_scale;
  p.out_delta = (out_buf == nullptr) ? 0
                                     : static_cast<long long>(reinterpret_cast<uintptr_t>(out_buf) -
                                                              reinterpret_cast<uintptr_t>(logits));
  p.mean = (red == CE_RED_MEAN) ? 1 : 0;

  const int smem = pl.S * pl.stage_bytes;
  int max_active = 0;
  cudaError_t ce_err = cached_occupancy(
      {dev, 0, static_cast<long long>(dtype), mode, pl.variant, smem, pl.CL},
      [&](int* out) {
        switch (dtype) {
          case CE_F32: return ce::rows_max_active<float>(mode, pl.variant, smem, pl.CL, di.sm_count, out);
          case CE_F16: return ce::rows_max_active<__half>(mode, pl.variant, smem, pl.CL, di.sm_count, out);
          default: return ce::rows_max_active<__nv_bfloat16>(mode, pl.variant, smem, pl.CL, di.sm_count, out);
        }
      },
      &max_active);
  if (ce_err != cudaSuccess || max_active < 1) return CE_ERR_CUDA;
  long long nclusters = p.n_units < max_active ? p.n_units : max_active;
  if (nclusters < 1) nclusters = 1;  // M == 0: one cluster writes the empty reduction
  const int grid = static_cast<int>(nclusters * pl.CL);

  if (loss != nullptr) {
    Scratch sc;
    st = reduction_scratch(static_scratch, dev, stream, grid, sc);
    if (st != CE_OK) return st;
    p.partials = sc.partials;
    p.ticket = sc.ticket;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (dtype) {
    case CE_F32: ce_err = ce::rows_launch<float>(mode, pl.variant, p, grid, smem, s); break;
    case CE_F16: ce_err = ce::rows_launch<__half>(mode, pl.variant, p, grid, smem, s); break;
    default: ce_err = ce::rows_launch<__nv_bfloat16>(mode, pl.variant, p, grid, smem, s); break;
  }
  if (ce_err != cudaSuccess) return CE_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return CE_OK;
}

}  // namespace

extern "C" {

ce_status ce_forward(const void* logits, const int64_t* targets, int64_t M, int64_t V,
                     ce_dtype dtype, ce_reduction reduction, float* loss, float* row_loss,
                     float* lse, void* stream) {
  return launch_rows(ce::FWD, logits, targets, nullptr, M, V, dtype, reduction, loss, row_loss,
                     lse, 1.0f, stream);
}

ce_status ce_fwd_bwd_inplace(void* logits, const int64_t* targets, int64_t M, int64_t V,
                             ce_dtype dtype, ce_reduction reduction, float* loss,
                             float* row_loss, float* lse, void* stream) {
  const float scale = (reduction == CE_RED_MEAN && M > 0) ? 1.0f / static_cast<float>(M) : 1.0f;
  return launch_rows(ce::FWD_BWD, logits, targets, nullptr, M, V, dtype, reduction, loss,
                     row_loss, lse, scale, stream);
}

ce_status ce_fwd_bwd_inplace_noalloc(void* logits, const int64_t* targets, int64_t M, int64_t V,
                                     ce_dtype dtype, ce_reduction reduction, float* loss,
                                     float* row_loss, float* lse, void* stream) {
  const float scale = (reduction == CE_RED_MEAN && M > 0) ? 1.0f / static_cast<float>(M) : 1.0f;
  return launch_rows(ce::FWD_BWD, logits, targets, nullptr, M, V, dtype, reduction, loss,
                     row_loss, lse, scale, stream, /*static_scratch=*/true);
}

ce_status ce_softmax_forward(const void* logits, void* probs, int64_t M, int64_t V,
                             ce_dtype dtype, float* lse, void* stream) {
  const int es = elem_size(dtype);
  if (es == 0 || M < 0 || V < 1) return CE_ERR_INVALID_ARG;
  if (M > 0 && (logits == nullptr || probs == nullptr)) return CE_ERR_INVALID_ARG;
  if (M > 0 && probs != logits) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(logits), b = reinterpret_cast<uintptr_t>(probs);
    if (V > (INT64_MAX / 4) / es || M > (INT64_MAX / 4) / (V * es)) return CE_ERR_INVALID_ARG;
    const uintptr_t n = static_cast<uintptr_t>(M) * static_cast<uintptr_t>(V) * es;
    if (a < b + n && b < a + n) return CE_ERR_INVALID_ARG;  // partial overlap
    if ((a - b) % 16) return CE_ERR_UNSUPPORTED;  // both buffers on the same 16-byte phase
  }
  return launch_rows(ce::SOFTMAX, logits, nullptr, nullptr, M, V, dtype, CE_RED_NONE, nullptr,
                     nullptr, lse, 1.0f, stream, false, probs == logits ? nullptr : probs);
}

ce_status ce_backward_from_lse(void* logits, const int64_t* targets, const float* lse, int64_t M,
                               int64_t V, ce_dtype dtype, float scale, void* stream) {
  return launch_rows(ce::BWD, logits, targets, lse, M, V, dtype, CE_RED_NONE, nullptr, nullptr,
                     nullptr, scale, stream);
}

ce_status ce_check_errors(void* stream, int timeout_ms) {
  DeviceInfo di;
  int dev = 0;
  ce_status st = device_info(di, &dev);
  if (st != CE_OK) return st;
  static std::mutex mu;
  static std::map<int, unsigned int*> host_words;
  std::lock_guard<std::mutex> lk(mu);
  unsigned int*& hw = host_words[dev];
  if (hw == nullptr) {
    if (cudaHostAlloc(reinterpret_cast<void**>(&hw), sizeof(unsigned int), cudaHostAllocDefault) !=
        cudaSuccess)
      return CE_ERR_CUDA;
  }
  *hw = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(hw, di.err, sizeof(unsigned int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CE_ERR_CUDA;
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    cudaError_t q = cudaStreamQuery(s);
    if (q == cudaSuccess) break;
    if (q != cudaErrorNotReady) return CE_ERR_CUDA;
    if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms))
      return CE_ERR_TIMEOUT;
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  const unsigned int w = *hw;
  if (w != 0) {
    if (cudaMemsetAsync(di.err, 0, sizeof(unsigned int), s) != cudaSuccess) return CE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return CE_ERR_CUDA;
  }
  if (w & ce::ERR_WAIT_TIMEOUT) return CE_ERR_TIMEOUT;
  if (w & ce::ERR_TARGET_RANGE) return CE_ERR_TARGET_RANGE;
  return CE_OK;
}

const char* ce_status_string(ce_status status) {
  switch (status) {
    case CE_OK: return "CE_OK";
    case CE_ERR_INVALID_ARG: return "CE_ERR_INVALID_ARG";
    case CE_ERR_UNSUPPORTED: return "CE_ERR_UNSUPPORTED";
    case CE_ERR_TARGET_RANGE: return "CE_ERR_TARGET_RANGE";
    case CE_ERR_CUDA: return "CE_ERR_CUDA";
    case CE_ERR_TIMEOUT: return "CE_ERR_TIMEOUT";
    default: return "CE_ERR_UNKNOWN";
  }
}

int64_t ce_max_vocab(ce_dtype dtype) {
  const int es = elem_size(dtype);
  if (es == 0) return 0;
  // 8 CTAs x one stage of at most kMaxSliceBytes; a misaligned row straddles one more chunk
  const long long chunks = static_cast<long long>(ce::kMaxCluster) * (kMaxSliceBytes / 16);
  return (chunks - 2) * 16 / es;
}

uint64_t ce_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

ce_status ce_selftest_wait_timeout(void* stream, int timeout_us) {
  if (timeout_us < 1 || timeout_us > 1000000) return CE_ERR_INVALID_ARG;
  DeviceInfo di;
  int dev = 0;
  ce_status st = device_info(di, &dev);
  if (st != CE_OK) return st;
  ce::ce_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      di.err, static_cast<unsigned long long>(timeout_us) * 1000ull);
  if (cudaGetLastError() != cudaSuccess) return CE_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return CE_OK;
}

}  // extern "C"
