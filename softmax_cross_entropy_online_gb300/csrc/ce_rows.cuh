// ce_rows.cuh -- the row kernels of the softmax cross-entropy library (sm_103a).
//
// One kernel template covers the three row operations:
//   FWD      per-row lse and loss, deterministic mean        (ce_forward)
//   FWD_BWD  the same, then g = (softmax - onehot)*scale
//            written over the logits from the on-chip copy    (ce_fwd_bwd_inplace)
//   BWD      g from a stored lse, written over the logits      (ce_backward_from_lse)
//
// Definitions followed: the per-row "max, subtract, exp, sum, log" of the
// "POPCORNBENCH level-1 problem 95 transcript", its online (max, sum) pair
// and the associative merge of two pairs ("This is associative"); the row
// output log(sumexp) + max - x_target of the loss_kernel in "Cross Entropy
// Loss performance issue"; the fused in-place backward of "9 Triton kernels
// in 9 weeks" (week seven).  exp is evaluated as exp2(x * log2 e), the
// identity the flash-attention discussion on the Triton forum uses.
//
// Design (GB300-first, not a port of the pages' kernels):
//  * Persistent grid.  A "unit" is R consecutive rows (small V) or one row
//    split over a thread-block cluster of CL CTAs (large V).  Cluster c
//    processes units c, c + nclusters, ...; CTA `rank` of the cluster owns
//    the rank-th slice of every unit.
//  * Warp specialisation.  The last warp is the producer: it streams units
//    into an S-deep ring of shared-memory stages with 1-D TMA bulk copies
//    (cp.async.bulk, completion on an mbarrier), and writes gradients back
//    with bulk stores from the same stage.  The NC consumer threads compute.
//  * Rows need not be 16-byte aligned (odd V in 16-bit types).  A unit's
//    bytes [as, ae) are cut into 16-byte "chunks" aligned to absolute
//    addresses: chunk c covers [A0 - 16 + 16c, A0 + 16c) with A0 =
//    ceil16(as).  Interior chunks 1..nI move by TMA; the partial head chunk
//    (0) and tail chunk (nI + 1) are read and written element by element by
//    the consumer thread that owns them.  No byte outside the unit is ever
//    touched, so neighbouring units never race.
//  * Each consumer thread reads its chunks of the stage once for the row's
//    statistics: blocks of four chunks update an online pair (m_t, s_t), the
//    sum rescaled by exp(m_old - m_new) when a block raises the max, so every
//    element costs one exp2.  After the row's lse is known it reads them again
//    and writes g = exp(x - m_t) * exp(m_t - lse) * scale.  (The register-
//    resident shapes hold the row's chunks instead: max first, then the
//    sum.)  Thread pairs (m_t, s_t) merge by warp shuffles, then across the
//    row's warps through shared memory, then across the cluster through
//    distributed shared memory (each CTA stores its pair into every peer's
//    slot and arrives on the peer's mbarrier).
//  * Issue slots are the scarce resource once the stream runs at the copy
//    rate, so the streaming passes use the packed fp32 pair instructions
//    (fma/add/mul .f32x2: two rn operations, the same results, one issue)
//    and three-input maxima.
//  * Mean: each CTA sums its rows' losses in row order (fp64); the last CTA
//    to finish (integer ticket) adds the per-CTA partials in index order.
//    No floating-point atomics, bit-reproducible for a given grid.
//  * Every wait is bounded (mbarrier try_wait against %globaltimer).  On
//    timeout the thread records an error bit and carries on without
//    waiting again, so every launch ends and no barrier is left unmatched.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ce {

constexpr unsigned ERR_TARGET_RANGE = 1u;
constexpr unsigned ERR_WAIT_TIMEOUT = 2u;
constexpr unsigned long long WAIT_LIMIT_NS = 4000000000ull;  // 4 s per wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// SOFTMAX: p = exp(x - lse) (the fused softmax of "9 Triton kernels in 9
// weeks", week one), written over the logits or into a second buffer.
enum Mode : int { FWD = 0, FWD_BWD = 1, BWD = 2, SOFTMAX = 3 };

constexpr int kMaxStages = 16;
constexpr int kMaxCluster = 8;
// row groups of a CTA: a row takes GT = NC / R threads, at least 8 (a quarter
// warp: short rows put several rows in one warp)
constexpr int kMinGroupThreads = 8;
constexpr int kMaxRowGroups = 512 / kMinGroupThreads;

// The instantiated consumer shapes (NC consumer threads, CPT register-resident
// 16-byte chunks per thread; CPT == 0 re-reads shared memory instead).
struct Variant {
  int NC, CPT;
};
constexpr Variant kVariants[] = {{256, 8}, {512, 4}, {128, 0}, {256, 0}, {512, 0}};
constexpr int kNumVariants = 5;

struct RowParams {
  char* base;                 // logits (byte address)
  const int64_t* targets;     // [M]
  const float* lse_in;        // [M], BWD only
  float* row_loss;            // [M] or null
  float* lse_out;             // [M] or null
  float* loss;                // [1] or null
  double* partials;           // [gridDim.x] scratch when loss != null
  unsigned int* ticket;       // scratch counter when loss != null
  unsigned int* err;          // device error word
  long long M, V;
  long long row_bytes;        // V * sizeof(T)
  long long n_units;          // ceil(M / R)
  int R;                      // rows per unit (1 in cluster mode)
  int CL;                     // CTAs per cluster
  int S;                      // pipeline stages
  int stage_bytes;            // bytes of one stage (multiple of 16)
  int q_chunks;               // chunk window of one CTA per unit (stage_bytes / 16)
  int log_gt;                 // log2 of the consumer threads per row group
  unsigned int wait_hint_ns;  // suspend-time hint of the mbarrier waits
  long long out_delta;        // writes go to (address + out_delta); 0 = in place
  float grad_scale;           // FWD_BWD / BWD
  int mean;                   // 1: loss = sum / M, 0: loss = sum
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(tx)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   bar_cluster_addr)
               : "memory");
}
// try_wait with a suspend-time hint: a waiting thread sleeps (up to hint_ns)
// until the phase completes instead of spinning and taking issue slots from
// the warps that are computing.
template <bool kClusterScope>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  if (kClusterScope) {
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
  }
  return ok != 0;
}
// Bounded wait.  After this thread has once timed out (`failed`), later waits
// only poll once, so a launch that lost a barrier still ends promptly.
template <bool kClusterScope>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err,
                                          bool& failed, unsigned long long limit_ns,
                                          uint32_t hint_ns = 20000u) {
  if (mbar_try_wait<kClusterScope>(bar, parity, hint_ns)) return true;
  if (failed) return false;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait<kClusterScope>(bar, parity, hint_ns)) {
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, ERR_WAIT_TIMEOUT);
      failed = true;
      return false;
    }
  }
  return true;
}
// Non-blocking test of an mbarrier phase (parity): true once it has completed.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// The bounded wait for a phase that has usually completed already (CTA scope):
// a non-blocking test first, which returns sooner than the suspending wait does
// even on a completed phase.  Measured where it pays: the attention MMA issuer
// (-7 % at T = 4096) and the streaming kernel's ring slots (-1.7 % on fp16
// [8192, 131072] fwd+bwd); not in the unit kernel, whose stages are mostly
// still in flight when waited on.
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity, unsigned int* err,
                                               bool& failed, unsigned long long limit_ns,
                                               uint32_t hint_ns = 20000u) {
  if (mbar_test_wait(bar, parity)) return true;
  return mbar_wait<false>(bar, parity, err, failed, limit_ns, hint_ns);
}
// Programmatically dependent launch (see ce_launch.cuh): let the next kernel
// on the stream be scheduled as this grid's CTAs exit, and wait until the
// previous kernel has completed and its writes are visible.  Called by every
// thread before any access to global memory.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_smem),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(src_smem), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}
// named barrier `id` (1..15) over `nthreads` threads: one per row group, so
// the groups of a CTA do not wait for each other
__device__ __forceinline__ void group_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
// warp-wide max of a float in one instruction (NaN-ignoring, like fmaxf)
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max of three floats in one instruction (NaN-ignoring, like fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Packed fp32 pairs: one fma/add/mul.rn.f32x2 does the work of two rn scalar
// operations with the same results, in one issue slot.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// 2^(a log2e - h), 2^(b log2e - h): one packed FFMA and two EX2
__device__ __forceinline__ float2 ex2_pair(float a, float b, float h) {
  const float2 u = ffma2(make_float2(a, b), make_float2(kLog2e, kLog2e), make_float2(-h, -h));
  return make_float2(ex2(u.x), ex2(u.y));
}
// the same, times f (the gradient's row factor)
__device__ __forceinline__ void grad_pair(const float* x, float* g, float h, float f) {
  const float2 r = fmul2(ex2_pair(x[0], x[1], h), make_float2(f, f));
  g[0] = r.x;
  g[1] = r.y;
}
// e^u - 1 for the target's gradient, u = x_t - lse (<= 0 up to rounding).  Below
// u = -1/2 the difference ex2(u log2 e) - 1 loses nothing to cancellation (the
// result is at most -0.39).  Above it the Taylor series of e^u - 1 is summed
// through the u^8/8! term by Horner's rule: on |u| <= 1/2 the first omitted term
// is below 2^-26 of the result, so a target that holds nearly all the
// probability keeps its small gradient.  Branch-free; -inf gives -1, NaN stays
// NaN.
__device__ __forceinline__ float expm1_target(float u) {
  float p = fmaf(u, 1.f / 40320.f, 1.f / 5040.f);
  p = fmaf(u, p, 1.f / 720.f);
  p = fmaf(u, p, 1.f / 120.f);
  p = fmaf(u, p, 1.f / 24.f);
  p = fmaf(u, p, 1.f / 6.f);
  p = fmaf(u, p, 0.5f);
  p = fmaf(u, p, 1.f);
  const float series = u * p;
  const float diff = ex2(u * kLog2e) - 1.f;
  return u < -0.5f ? diff : series;
}

// Sum of a double over the warp by butterflies: every lane ends with the same
// bits (each step adds the same two operands on both lanes of a pair).
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// A running sum of row losses kept as an unevaluated pair hi + lo of floats:
// each step is Knuth's error-free TwoSum (the rounding error of hi + x goes
// into lo), so the pair carries about twice a float's precision and no
// double-precision instruction sits on a row's path.  A non-finite sum (an
// infinite or NaN row loss) is kept in hi with no error term.
struct PairSum {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float s = hi + x;
    const float bb = s - hi;
    const float e = (hi - (s - bb)) + (x - bb);
    lo += isfinite(s) ? e : 0.f;
    hi = s;
  }
  __device__ __forceinline__ double value() const {
    return static_cast<double>(hi) + static_cast<double>(lo);
  }
};

// Deterministic reduction of the loss over the grid, run by one whole warp of
// each CTA after the CTA's row-group sums sit in group_sums[0, n).  Lane j adds
// group sums j, j + 32, ... in order, a butterfly combines the lanes, and lane 0
// stores the CTA's partial and takes an integer ticket.  The CTA that takes the
// last ticket sums every partial the same way, with its loads all in flight at
// once (one L2 round trip, not one per CTA), writes the loss and re-arms the
// ticket.  Every addition's order is fixed by the launch shape, so the loss is
// bit-reproducible; no floating-point atomics are used.
__device__ __forceinline__ void loss_tail_warp(const double* group_sums, int n,
                                               double* partials, unsigned int* ticket,
                                               float* loss, long long M, int mean, int lane) {
  double part = 0.0;
  for (int j = lane; j < n; j += 32) part += group_sums[j];
  part = warp_sum_f64(part);
  unsigned int prev = 0;
  if (lane == 0) {
    partials[blockIdx.x] = part;
    __threadfence();
    prev = atomicAdd(ticket, 1u);
  }
  prev = __shfl_sync(0xffffffffu, prev, 0);
  if (prev != gridDim.x - 1) return;
  __threadfence();
  const int G = static_cast<int>(gridDim.x);
  double s = 0.0;
  int j = lane;
  for (; j + 32 * 7 < G; j += 32 * 8) {
    double v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __ldcg(partials + j + 32 * k);
#pragma unroll
    for (int k = 0; k < 8; ++k) s += v[k];
  }
  for (; j < G; j += 32) s += __ldcg(partials + j);
  s = warp_sum_f64(s);
  if (lane == 0) {
    *loss = static_cast<float>(mean ? s / static_cast<double>(M) : s);
    *ticket = 0u;  // ready for the next launch that uses this scratch
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// Element formats: 16 bytes = EPC elements; widen to fp32, narrow with RN.
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int EPC = 4;
  static constexpr int ES = 4;
  __device__ static __forceinline__ void unpack(uint4 q, float* v) {
    v[0] = __uint_as_float(q.x);
    v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z);
    v[3] = __uint_as_float(q.w);
  }
  __device__ static __forceinline__ uint4 pack(const float* g) {
    return make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                      __float_as_uint(g[3]));
  }
  __device__ static __forceinline__ float ld(const void* p) {
    return *static_cast<const volatile float*>(p);
  }
  __device__ static __forceinline__ float chunk_max(uint4 q) {
    return fmax3(__uint_as_float(q.x), __uint_as_float(q.y),
                 fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
  }
  // max of m and four chunks: a tree of three-input maxima
  __device__ static __forceinline__ float max4(uint4 a, uint4 b, uint4 c, uint4 d, float m) {
    const float m1 = fmax3(__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z));
    const float m2 = fmax3(__uint_as_float(a.w), __uint_as_float(b.x), __uint_as_float(b.y));
    const float m3 = fmax3(__uint_as_float(b.z), __uint_as_float(b.w), __uint_as_float(c.x));
    const float m4 = fmax3(__uint_as_float(c.y), __uint_as_float(c.z), __uint_as_float(c.w));
    const float m5 = fmax3(__uint_as_float(d.x), __uint_as_float(d.y), __uint_as_float(d.z));
    const float m6 = fmax3(__uint_as_float(d.w), m, m1);
    return fmax3(fmax3(m2, m3, m4), m5, m6);
  }
  __device__ static __forceinline__ void st(void* p, float g) { *static_cast<float*>(p) = g; }
};

template <>
struct Elem<__half> {
  static constexpr int EPC = 8;
  static constexpr int ES = 2;
  __device__ static __forceinline__ float2 w2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
  }
  __device__ static __forceinline__ uint32_t n2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ void unpack(uint4 q, float* v) {
    float2 a = w2(q.x), b = w2(q.y), c = w2(q.z), d = w2(q.w);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
  }
  __device__ static __forceinline__ uint4 pack(const float* g) {
    return make_uint4(n2(g[0], g[1]), n2(g[2], g[3]), n2(g[4], g[5]), n2(g[6], g[7]));
  }
  __device__ static __forceinline__ float ld(const void* p) {
    unsigned short u = *static_cast<const volatile unsigned short*>(p);
    return __half2float(__ushort_as_half(u));
  }
  // max of the 8 elements with packed half2 max (exact; NaN-ignoring like fmaxf)
  __device__ static __forceinline__ float chunk_max(uint4 q) {
    __half2 a = *reinterpret_cast<__half2*>(&q.x), b = *reinterpret_cast<__half2*>(&q.y);
    __half2 c = *reinterpret_cast<__half2*>(&q.z), d = *reinterpret_cast<__half2*>(&q.w);
    __half2 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(m), __high2float(m));
  }
  __device__ static __forceinline__ float max4(uint4 a, uint4 b, uint4 c, uint4 d, float m) {
    return fmaxf(m, fmaxf(fmaxf(chunk_max(a), chunk_max(b)), fmaxf(chunk_max(c), chunk_max(d))));
  }
  __device__ static __forceinline__ void st(void* p, float g) {
    *static_cast<unsigned short*>(p) = __half_as_ushort(__float2half_rn(g));
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int EPC = 8;
  static constexpr int ES = 2;
  __device__ static __forceinline__ uint32_t n2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ void unpack(uint4 q, float* v) {
    // bf16 is the upper half of an fp32: widening is a shift
    v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
    v[4] = __uint_as_float(q.z << 16); v[5] = __uint_as_float(q.z & 0xffff0000u);
    v[6] = __uint_as_float(q.w << 16); v[7] = __uint_as_float(q.w & 0xffff0000u);
  }
  __device__ static __forceinline__ uint4 pack(const float* g) {
    return make_uint4(n2(g[0], g[1]), n2(g[2], g[3]), n2(g[4], g[5]), n2(g[6], g[7]));
  }
  __device__ static __forceinline__ float ld(const void* p) {
    unsigned short u = *static_cast<const volatile unsigned short*>(p);
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
  // max of the 8 elements with packed bf16x2 max (exact; NaN-ignoring like fmaxf)
  __device__ static __forceinline__ float chunk_max(uint4 q) {
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&q.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&q.y);
    __nv_bfloat162 c = *reinterpret_cast<__nv_bfloat162*>(&q.z);
    __nv_bfloat162 d = *reinterpret_cast<__nv_bfloat162*>(&q.w);
    __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(m), __high2float(m));
  }
  __device__ static __forceinline__ float max4(uint4 a, uint4 b, uint4 c, uint4 d, float m) {
    return fmaxf(m, fmaxf(fmaxf(chunk_max(a), chunk_max(b)), fmaxf(chunk_max(c), chunk_max(d))));
  }
  __device__ static __forceinline__ void st(void* p, float g) {
    *static_cast<unsigned short*>(p) = __bfloat16_as_ushort(__float2bfloat16_rn(g));
  }
};

// ---------------------------------------------------------------------------
// Unit geometry (identical on producer and consumers)
// ---------------------------------------------------------------------------
struct UnitGeo {
  long long row0;   // first row of the unit
  int rows;         // rows in the unit
  long long as;     // absolute address of the unit's first byte
  int hb;           // bytes from `as` to the next 16-byte boundary A0 = as + hb
  int nI;           // interior chunks (1..nI)
  int w0, w1;       // this CTA's chunk window [w0, w1)
  bool head_ok;     // the partial head chunk 0 lies inside the tensor: load it by TMA
  bool tail_ok;     // the partial tail chunk nI + 1 lies inside the tensor: load it by TMA
};

__device__ __forceinline__ UnitGeo unit_geo(const RowParams& p, long long u, int rank) {
  UnitGeo g;
  g.row0 = u * p.R;  // the host guarantees CL * q_chunks covers every unit's chunks
  const long long rows = p.M - g.row0;
  g.rows = static_cast<int>(rows < p.R ? rows : p.R);
  const long long off = g.row0 * p.row_bytes;  // unit start, from the tensor base
  g.as = reinterpret_cast<long long>(p.base) + off;
  const int ub = g.rows * static_cast<int>(p.row_bytes);  // unit bytes (< 2^31)
  g.hb = static_cast<int>((-g.as) & 15);
  int c_first, c_last;
  if (ub > g.hb) {
    g.nI = (ub - g.hb) >> 4;
    c_last = ((ub - g.hb) & 15) ? g.nI + 1 : g.nI;
  } else {  // the whole unit sits before the first 16-byte boundary
    g.nI = 0;
    c_last = 0;
  }
  c_first = g.hb ? 0 : 1;
  const int Q = p.q_chunks;
  g.w0 = c_first + rank * Q;
  int w1 = g.w0 + Q;
  g.w1 = w1 < c_last + 1 ? w1 : c_last + 1;
  if (g.w1 < g.w0) g.w1 = g.w0;
  // A partial chunk also holds bytes of the neighbouring unit.  Reading those
  // (and ignoring them) is harmless as long as the 16 bytes lie inside the
  // tensor; writes to a partial chunk are always element by element.
  const long long total = p.M * p.row_bytes;
  g.head_ok = c_first == 0 && off + g.hb - 16 >= 0 && off + g.hb <= total;
  g.tail_ok = c_last == g.nI + 1 && off + g.hb + 16LL * (g.nI + 1) <= total;
  return g;
}

// chunk range [lo, hi) of this CTA's window written back by TMA: the interior
__device__ __forceinline__ void bulk_range(const UnitGeo& g, int& lo, int& hi) {
  lo = g.w0 > 1 ? g.w0 : 1;
  hi = g.w1 < g.nI + 1 ? g.w1 : g.nI + 1;
}
// chunk range read by TMA: the interior plus the partial head/tail chunks
// that lie inside the tensor
__device__ __forceinline__ void load_range(const UnitGeo& g, int& lo, int& hi) {
  const int l = g.head_ok ? 0 : 1;
  const int h = g.tail_ok ? g.nI + 2 : g.nI + 1;
  lo = g.w0 > l ? g.w0 : l;
  hi = g.w1 < h ? g.w1 : h;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// CPT > 0: each consumer thread keeps up to CPT full chunks of exp values in
// registers (one exp2 per element).  CPT == 0: the stage in shared memory is
// read once for the statistics and again for the backward (two exp2 per
// element, few registers, several CTAs per SM, and no register limit on the
// slice length).
template <int NC, int CPT>
struct MinBlocks {
  // streaming consumers: registers capped so that 5 (128 threads) or 3 (256
  // threads) CTAs fit on an SM; occupancy hides each CTA's per-unit latency
  static constexpr int value = CPT > 0 ? 1 : (NC <= 128 ? 5 : (NC <= 256 ? 3 : 1));
};

template <typename T, int MODE, int NC, int CPT>
__global__ void __launch_bounds__(NC + 32, (MinBlocks<NC, CPT>::value))
    ce_rows_kernel(const RowParams p) {
  griddep_wait();
  using E = Elem<T>;
  constexpr int EPC = E::EPC;
  constexpr int ES = E::ES;
  constexpr int NW = NC / 32;

  extern __shared__ __align__(128) unsigned char stage_mem[];
  __shared__ __align__(8) unsigned long long full_bar[kMaxStages];
  __shared__ __align__(8) unsigned long long done_bar[kMaxStages];
  __shared__ __align__(8) unsigned long long xbar[2];
  __shared__ __align__(16) float4 xslot[2][kMaxCluster];
  __shared__ float2 red[2][NW];
  __shared__ float xt_slot[2][NW];
  __shared__ double acc_slot[kMaxRowGroups];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int CL = p.CL;
  const int rank = static_cast<int>(blockIdx.x) % CL;
  const long long cid = blockIdx.x / CL;
  const long long ncl = gridDim.x / CL;
  const long long n_iter = (cid < p.n_units) ? (p.n_units - 1 - cid) / ncl + 1 : 0;
  const int S = p.S;
  const uint32_t stage0 = smem_u32(stage_mem);
  bool failed = false;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&done_bar[s]), NC);
    }
    mbar_init(smem_u32(&xbar[0]), CL);
    mbar_init(smem_u32(&xbar[1]), CL);
    fence_mbar_init_cluster();
  }
  __syncthreads();
  if (CL > 1) cluster_sync_all();  // peers' barriers exist before any remote arrive

  if (warp == NW) {
    // ======================= producer warp =======================
    // Loads run up to S - 1 units ahead of the consumers.  In the modes that
    // write, the gradient of unit j is stored as soon as the consumers release
    // its stage, and the stage is refilled once that store has been read out.
    if (lane == 0) {
      auto issue_load = [&](long long i, int s) {
        const UnitGeo g = unit_geo(p, cid + i * ncl, rank);
        int lo, hi;
        load_range(g, lo, hi);
        const uint32_t fb = smem_u32(&full_bar[s]);
        fence_proxy_async_smem();
        if (hi > lo) {
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>((hi - lo) * 16));
          bulk_load(stage0 + s * p.stage_bytes + (lo - g.w0) * 16,
                    reinterpret_cast<const void*>(g.as + g.hb - 16 + 16LL * lo),
                    static_cast<uint32_t>((hi - lo) * 16), fb);
        } else {
          mbar_arrive(fb);
        }
      };
      // Writing modes move a stage in kParts parts of fixed stage offsets: part
      // q of the refill is loaded as soon as part q of the previous unit's
      // store has been read out, so the store's tail and the load's head
      // overlap instead of following each other.
      constexpr int kParts = 4;
      auto part_of = [&](int a, int b, int q, int& pa, int& pb) {
        const int lo_q = (q * p.q_chunks) / kParts, hi_q = ((q + 1) * p.q_chunks) / kParts;
        pa = a > lo_q ? a : lo_q;
        pb = b < hi_q ? b : hi_q;
      };
      auto refill_in_parts = [&](long long i, int s) {
        const UnitGeo g = unit_geo(p, cid + i * ncl, rank);
        int lo, hi;
        load_range(g, lo, hi);
        const uint32_t fb = smem_u32(&full_bar[s]);
        if (hi > lo) {
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>((hi - lo) * 16));
        } else {
          mbar_arrive(fb);
        }
#pragma unroll
        for (int q = 0; q < kParts; ++q) {
          // parts 0..q of the store of this stage's previous unit are read out
          if (q == 0) bulk_wait_read<kParts - 1>();
          else if (q == 1) bulk_wait_read<kParts - 2>();
          else if (q == 2) bulk_wait_read<kParts - 3>();
          else bulk_wait_read<0>();
          int a, b;
          part_of(lo - g.w0, hi - g.w0, q, a, b);
          if (b > a) {
            fence_proxy_async_smem();
            bulk_load(stage0 + s * p.stage_bytes + a * 16,
                      reinterpret_cast<const void*>(g.as + g.hb - 16 + 16LL * (g.w0 + a)),
                      static_cast<uint32_t>((b - a) * 16), fb);
          }
        }
      };
      const long long pre = n_iter < S ? n_iter : S;
      for (long long i = 0; i < pre; ++i) issue_load(i, static_cast<int>(i));
      // A stage is refilled as soon as the store of its unit has been read out
      // of shared memory (lag 0): the loads then run S - 1 units ahead of the
      // consumers.  (The refill brings unit r + S, r = j - lag, which must not
      // be loaded yet, so any lag <= S - 1 is valid; a larger lag only shortens
      // the lookahead to S - 1 - lag units.)
      constexpr int lag = 0;  // the stage just stored is the one refilled
      int s = 0, sr = S - lag;  // stages of unit j and of unit j - lag (mod S)
      if (sr == S) sr = 0;
      uint32_t phase = 0;
      for (long long j = 0; j < n_iter; ++j) {
        mbar_wait<false>(smem_u32(&done_bar[s]), phase, p.err, failed, WAIT_LIMIT_NS, p.wait_hint_ns);
        if (MODE == FWD) {
          if (j + S < n_iter) issue_load(j + S, s);
        } else {
          const UnitGeo go = unit_geo(p, cid + j * ncl, rank);
          int lo, hi;
          bulk_range(go, lo, hi);
#pragma unroll
          for (int q = 0; q < kParts; ++q) {
            int a, b;
            part_of(lo - go.w0, hi - go.w0, q, a, b);
            if (b > a)
              bulk_store(reinterpret_cast<void*>(go.as + go.hb - 16 + 16LL * (go.w0 + a) + p.out_delta),
                         stage0 + s * p.stage_bytes + a * 16, (b - a) * 16);
            bulk_commit();  // one group per part (possibly empty) keeps the count exact
          }
          const long long r = j - lag;
          if (r >= 0 && r + S < n_iter) refill_in_parts(r + S, sr);
        }
        if (++s == S) { s = 0; phase ^= 1u; }
        if (++sr == S) sr = 0;
      }
      if (MODE != FWD) bulk_wait_all();
    }
  } else {
    // ======================= consumer warps =======================
    constexpr int LOG_ES = (ES == 4) ? 2 : 1;
    constexpr bool RESIDENT = CPT > 0;  // keep exp values in registers (else re-read smem)
    constexpr int KR = RESIDENT ? CPT : 1;
    const int R = p.R;
    const int GT = NC / R;     // threads per row group
    const int GW = GT / 32;    // warps per row group (0: several rows in a warp)
    const int grp = tid >> p.log_gt;  // row of the unit this thread works on
    const int gt = tid & (GT - 1);
    const int V = static_cast<int>(p.V);          // the host caps V * sizeof(T) far below 2^31
    const int rb = static_cast<int>(p.row_bytes);
    PairSum acc;  // this group's running loss sum (leader only)
    const bool leader = (gt == 0) && (rank == 0);

    int s = -1;
    uint32_t phase = 1;
    // the target (and, for BWD, the lse) of the next unit's row is fetched one
    // unit ahead, so its global-memory latency hides behind this unit's work
    long long t_next = -1;
    float lse_next = 0.f;
    {
      const long long row_first = cid * R + grp;
      if (MODE != SOFTMAX && n_iter > 0 && row_first < p.M) {
        t_next = __ldg(p.targets + row_first);
        if (MODE == BWD) lse_next = __ldg(p.lse_in + row_first);
      }
    }
    for (long long i = 0; i < n_iter; ++i) {
      if (++s == S) s = 0;
      if (s == 0) phase ^= 1u;
      const int b = static_cast<int>(i & 1);
      const UnitGeo g = unit_geo(p, cid + i * ncl, rank);
      const bool row_ok = grp < g.rows;
      const long long row = g.row0 + grp;
      const long long t = row_ok ? t_next : -1;
      const float lse_given = lse_next;
      if (i + 1 < n_iter) {
        const long long row_n = (cid + (i + 1) * ncl) * R + grp;
        if (MODE != SOFTMAX && row_n < p.M) {
          t_next = __ldg(p.targets + row_n);
          if (MODE == BWD) lse_next = __ldg(p.lse_in + row_n);
        }
      }
      const bool t_ok = row_ok && t >= 0 && t < V;

      // Offsets are taken from the start of chunk 0 (absolute as + hb - 16):
      // element e of this row lies at byte e*ES - d0 of that frame.
      const int d0 = g.hb - 16 - grp * rb;  // in (-16 - grp*rb, 0]
      int lo = (-d0) >> 4;                 // chunk holding the row's first byte
      int hi = ((rb - 1 - d0) >> 4) + 1;   // one past the chunk holding its last byte
      if (lo < g.w0) lo = g.w0;
      if (hi > g.w1) hi = g.w1;
      if (!row_ok) hi = lo;
      // "full" chunks: interior (moved by TMA) with all EPC slots inside the row;
      // the at most two edge chunks at either end, [lo, f0) and [f1, hi), are
      // handled element by element by threads gt = 0, 1.
      int f0 = (-d0 + 15) >> 4;
      if (f0 < 1) f0 = 1;
      int f1 = (rb - d0) >> 4;
      if (f1 > g.nI + 1) f1 = g.nI + 1;
      f0 = f0 < lo ? lo : (f0 > hi ? hi : f0);
      f1 = f1 < f0 ? f0 : (f1 > hi ? hi : f1);
      const int ce_front = (gt < f0 - lo) ? lo + gt : -1;  // this thread's edge chunks
      const int ce_back = (gt < hi - f1) ? f1 + gt : -1;
      const uint32_t sbase = stage0 + s * p.stage_bytes - g.w0 * 16;  // chunk c at sbase + 16c

      // target owner: the thread that processes the chunk holding x[row, t]
      const int tbo = t_ok ? static_cast<int>(t) * ES - d0 : 0;
      const int tc = t_ok ? (tbo >> 4) : -1;
      const bool t_smem = tc >= 1 && tc <= g.nI;  // written back through shared memory
      // chunk c's bytes are in the stage (interior, or a partial chunk loaded by TMA)
      auto in_stage = [&](int c) -> bool {
        return (c >= 1 && c <= g.nI) || (c == 0 && g.head_ok) || (c == g.nI + 1 && g.tail_ok);
      };
      bool owner = false;
      if (t_ok && tc >= lo && tc < hi) {
        owner = (tc < f0) ? (tc - lo == gt) : (tc >= f1 ? tc - f1 == gt : ((tc - f0) & (GT - 1)) == gt);
      }

      auto elem_ptr_global = [&](int e) -> char* {
        return reinterpret_cast<char*>(g.as + static_cast<long long>(grp) * rb +
                                       static_cast<long long>(e) * ES);
      };
      auto smem_ptr = [&](int byte_off) -> char* {
        return static_cast<char*>(__cvta_shared_to_generic(sbase + byte_off));
      };
      // values of an edge chunk, -inf outside the row: one 16-byte shared load
      // when the chunk is in the stage (the partial head/tail chunks normally
      // are), element loads from memory otherwise
      auto edge_load = [&](int c, float* v) {
        const int e0 = (d0 + 16 * c) >> LOG_ES;
        if (in_stage(c)) {
          E::unpack(lds128(sbase + 16 * c), v);
#pragma unroll
          for (int q = 0; q < EPC; ++q)
            if (!(e0 + q >= 0 && e0 + q < V)) v[q] = -INFINITY;
        } else {
#pragma unroll
          for (int q = 0; q < EPC; ++q) {
            const int e = e0 + q;
            v[q] = (e >= 0 && e < V) ? E::ld(elem_ptr_global(e)) : -INFINITY;
          }
        }
      };
      auto edge_store = [&](int c, const float* gv) {
        const int e0 = (d0 + 16 * c) >> LOG_ES;
        const bool in_smem = c >= 1 && c <= g.nI;
#pragma unroll
        for (int q = 0; q < EPC; ++q) {
          const int e = e0 + q;
          if (e >= 0 && e < V) {
            if (in_smem) E::st(smem_ptr(16 * c + q * ES), gv[q]);
            else E::st(elem_ptr_global(e) + p.out_delta, gv[q]);
          }
        }
      };

      mbar_wait<false>(smem_u32(&full_bar[s]), phase, p.err, failed, WAIT_LIMIT_NS, p.wait_hint_ns);

      float xt = 0.f;
      if (owner)
        xt = in_stage(tc) ? E::ld(smem_ptr(tbo)) : E::ld(elem_ptr_global(static_cast<int>(t)));

      if (MODE == BWD) {
        const float sc = p.grad_scale;
        // g = 2^(x log2e - lse log2e) * scale; the rounding of lse*log2e (lh)
        // is a common factor 2^(-ll) folded into the scale
        const float lh = lse_given * kLog2e;
        const float ll = fmaf(lse_given, kLog2e, -lh);
        const float scf = ex2(-ll) * sc;
        for (int c = f0 + gt; c < f1; c += GT) {
          float x[EPC], gv[EPC];
          E::unpack(lds128(sbase + 16 * c), x);
#pragma unroll
          for (int q = 0; q < EPC; q += 2) grad_pair(x + q, gv + q, lh, scf);
          sts128(sbase + 16 * c, E::pack(gv));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = h ? ce_back : ce_front;
          if (c >= 0) {
            float x[EPC], gv[EPC];
            edge_load(c, x);
#pragma unroll
            for (int q = 0; q < EPC; ++q) gv[q] = ex2((x[q] - lse_given) * kLog2e) * sc;
            edge_store(c, gv);
          }
        }
        if (owner) {
          // exp(x_t - lse) - 1 without cancellation when the target dominates
          const float gval = expm1_target(xt - lse_given) * sc;
          if (t_smem) E::st(smem_ptr(tbo), gval);
          else E::st(elem_ptr_global(static_cast<int>(t)), gval);
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&done_bar[s]));
        if (row_ok && !t_ok && gt == 0 && rank == 0) atomicOr(p.err, ERR_TARGET_RANGE);
        continue;
      }

      // ---- per-thread (max, sum) ----
      // e' = 2^(x log2e - mh) with mh = RN(m_t log2e) is a single FFMA + EX2.
      // Since x log2e - mh = (x - m_t) log2e + ml exactly up to the FFMA's own
      // rounding (ml = m_t log2e - mh, the same for every element of the
      // thread), e' = e * 2^ml: the common factor is divided out once per
      // thread, so logits sharing a large offset lose no accuracy.
      float v[KR][EPC];
      float mt = -INFINITY, mh = 0.f, ml = 0.f, st = 0.f;
      if (RESIDENT) {
#pragma unroll
        for (int k = 0; k < KR; ++k) {
          const int c = f0 + gt + k * GT;
          if (c < f1) {
            const uint4 q = lds128(sbase + 16 * c);
            mt = fmaxf(mt, E::chunk_max(q));
            E::unpack(q, v[k]);
          } else {
#pragma unroll
            for (int q = 0; q < EPC; ++q) v[k][q] = -INFINITY;
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = h ? ce_back : ce_front;
          if (c >= 0) {
            float x[EPC];
            edge_load(c, x);
#pragma unroll
            for (int q = 0; q < EPC; ++q) mt = fmaxf(mt, x[q]);
          }
        }
        const float mref = (mt == -INFINITY) ? 0.f : mt;
        mh = mref * kLog2e;
        ml = fmaf(mref, kLog2e, -mh);
#pragma unroll
        for (int k = 0; k < KR; ++k)
#pragma unroll
          for (int q = 0; q < EPC; ++q) {
            const float e = ex2(fmaf(v[k][q], kLog2e, -mh));
            v[k][q] = e;
            st += e;
          }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = h ? ce_back : ce_front;
          if (c >= 0) {
            float x[EPC];
            edge_load(c, x);
#pragma unroll
            for (int q = 0; q < EPC; ++q) st += ex2(fmaf(x[q], kLog2e, -mh));
          }
        }
      } else {
        // one pass over the stage: each block of four chunks updates an online
        // pair (m_t, s_t), the running sums rescaled by 2^(mh_old - mh_new)
        // (a factor 1 when the block does not raise the max: branch-free)
        float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);
        auto rescale_to = [&](float mn) {
          const float mhn = (mn == -INFINITY) ? 0.f : mn * kLog2e;
          const float r = (mt == -INFINITY) ? 0.f : ex2(mh - mhn);
          sa = fmul2(sa, make_float2(r, r));
          sb = fmul2(sb, make_float2(r, r));
          mt = mn;
          mh = mhn;
        };
        int c = f0 + gt;
        for (; c + 3 * GT < f1; c += 4 * GT) {
          const uint4 q0 = lds128(sbase + 16 * c), q1 = lds128(sbase + 16 * (c + GT));
          const uint4 q2 = lds128(sbase + 16 * (c + 2 * GT)), q3 = lds128(sbase + 16 * (c + 3 * GT));
          rescale_to(E::max4(q0, q1, q2, q3, mt));
          float x0[EPC], x1[EPC], x2[EPC], x3[EPC];
          E::unpack(q0, x0);
          E::unpack(q1, x1);
          E::unpack(q2, x2);
          E::unpack(q3, x3);
#pragma unroll
          for (int q = 0; q < EPC; q += 2) {
            sa = fadd2(sa, fadd2(ex2_pair(x0[q], x0[q + 1], mh), ex2_pair(x1[q], x1[q + 1], mh)));
            sb = fadd2(sb, fadd2(ex2_pair(x2[q], x2[q + 1], mh), ex2_pair(x3[q], x3[q + 1], mh)));
          }
        }
        for (; c < f1; c += GT) {
          const uint4 q0 = lds128(sbase + 16 * c);
          rescale_to(fmaxf(mt, E::chunk_max(q0)));
          float x[EPC];
          E::unpack(q0, x);
#pragma unroll
          for (int q = 0; q < EPC; q += 2) sa = fadd2(sa, ex2_pair(x[q], x[q + 1], mh));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ec = h ? ce_back : ce_front;
          if (ec >= 0) {
            float x[EPC];
            edge_load(ec, x);
            float em = mt;
#pragma unroll
            for (int q = 0; q < EPC; ++q) em = fmaxf(em, x[q]);
            rescale_to(em);
#pragma unroll
            for (int q = 0; q < EPC; q += 2) sa = fadd2(sa, ex2_pair(x[q], x[q + 1], mh));
          }
        }
        st = (sa.x + sa.y) + (sb.x + sb.y);
        const float mref = (mt == -INFINITY) ? 0.f : mt;
        ml = fmaf(mref, kLog2e, -mh);
      }
      if (MODE == FWD) {
        // every read of the stage is done: hand it back to the producer early
        mbar_arrive(smem_u32(&done_bar[s]));
      }

      // ---- merge (m, s): warp, then the row's warps ----
      // (st carries the factor 2^ml; it is removed in the same exp2 that
      // rescales the thread's sum to the warp max)
      const bool have_t = t_ok && tc >= g.w0 && tc < g.w1;  // this CTA holds x[row, t]
      float Mg, Sg, xrow = 0.f;
      if (GW == 0) {
        // GT lanes per row, groups aligned to GT lanes: butterflies over lane
        // distances below GT stay inside the row's group
        float mg = mt;
        for (int o = GT >> 1; o > 0; o >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
        float sg = (mt == -INFINITY) ? 0.f : st * ex2((mt - mg) * kLog2e - ml);
        for (int o = GT >> 1; o > 0; o >>= 1) sg += __shfl_xor_sync(0xffffffffu, sg, o);
        Mg = mg;
        Sg = sg;
        const unsigned gmask = ((GT == 32) ? 0xffffffffu : ((1u << GT) - 1u)) << (lane & ~(GT - 1));
        const unsigned own = __ballot_sync(0xffffffffu, owner) & gmask;
        const float xo = __shfl_sync(0xffffffffu, xt, own ? __ffs(own) - 1 : lane);
        if (have_t && own != 0u) xrow = xo;
      } else if (GW == 1) {
        const float mw = warp_max(mt);
        float sw = (mt == -INFINITY) ? 0.f : st * ex2((mt - mw) * kLog2e - ml);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sw += __shfl_down_sync(0xffffffffu, sw, o);
        // a row handled by one warp: the warp's pair is the row's pair, and the
        // target logit comes from the owner lane, with no shared memory or barrier
        Mg = mw;
        Sg = __shfl_sync(0xffffffffu, sw, 0);
        const unsigned own = __ballot_sync(0xffffffffu, owner);
        if (have_t && own != 0u) xrow = __shfl_sync(0xffffffffu, xt, __ffs(own) - 1);
      } else {
        const float mw = warp_max(mt);
        float sw = (mt == -INFINITY) ? 0.f : st * ex2((mt - mw) * kLog2e - ml);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sw += __shfl_down_sync(0xffffffffu, sw, o);
        if (lane == 0) red[b][warp] = make_float2(mw, sw);
        if (owner) xt_slot[b][grp] = xt;
        if (R == 1) consumer_sync(NC);
        else group_sync(1 + grp, GT);

        float2 r = (lane < GW) ? red[b][grp * GW + lane] : make_float2(-INFINITY, 0.f);
        Mg = warp_max(r.x);
        Sg = (r.x == -INFINITY) ? 0.f : r.y * ex2((r.x - Mg) * kLog2e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Sg += __shfl_down_sync(0xffffffffu, Sg, o);
        Sg = __shfl_sync(0xffffffffu, Sg, 0);
        xrow = have_t ? xt_slot[b][grp] : 0.f;
      }

      // ---- merge across the cluster through distributed shared memory ----
      if (CL > 1) {
        if (tid == 0) {
          const uint32_t my_slot = smem_u32(&xslot[b][rank]);
          const uint32_t my_bar = smem_u32(&xbar[b]);
          for (int k = 0; k < CL; ++k) {
            st_cluster_f4(map_to_rank(my_slot, k), Mg, Sg, xrow, have_t ? 1.f : 0.f);
            mbar_arrive_remote(map_to_rank(my_bar, k));
          }
        }
        mbar_wait<true>(smem_u32(&xbar[b]), static_cast<uint32_t>((i >> 1) & 1), p.err, failed,
                        WAIT_LIMIT_NS, p.wait_hint_ns);
        float4 xs = (lane < CL) ? xslot[b][lane] : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        const float Mc = warp_max(xs.x);
        float Sc = (xs.x == -INFINITY) ? 0.f : xs.y * ex2((xs.x - Mc) * kLog2e);
        float Xc = xs.w != 0.f ? xs.z : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          Sc += __shfl_down_sync(0xffffffffu, Sc, o);
          Xc += __shfl_down_sync(0xffffffffu, Xc, o);
        }
        Mg = Mc;
        Sg = __shfl_sync(0xffffffffu, Sc, 0);
        xrow = __shfl_sync(0xffffffffu, Xc, 0);
      }

      // ---- row outputs (one thread per row) ----
      if (leader && row_ok) {
        const float lnS = lg2(Sg) * kLn2;
        const float lse = Mg + lnS;
        // (m - x_t) + log S keeps the loss accurate when m and x_t are large
        const float rl = t_ok ? (Mg - xrow) + lnS : __int_as_float(0x7fc00000);
        if (p.row_loss) p.row_loss[row] = rl;
        if (p.lse_out) p.lse_out[row] = lse;
        acc.add(rl);
        if (!t_ok && MODE != SOFTMAX) atomicOr(p.err, ERR_TARGET_RANGE);
      }

      if (MODE == FWD_BWD || MODE == SOFTMAX) {
        // g = e' * 2^-ml * exp(m_t - lse) * scale, exp(m_t - lse) = 2^((m_t - M) log2e - log2 S)
        const float sc = p.grad_scale;
        const float f = ex2((mt - Mg) * kLog2e - lg2(Sg) - ml) * sc;
        if (RESIDENT) {
#pragma unroll
          for (int k = 0; k < KR; ++k) {
            const int c = f0 + gt + k * GT;
            if (c < f1) {
              float gv[EPC];
#pragma unroll
              for (int q = 0; q < EPC; ++q) gv[q] = v[k][q] * f;
              sts128(sbase + 16 * c, E::pack(gv));
            }
          }
        } else {
          int c = f0 + gt;
          for (; c + 3 * GT < f1; c += 4 * GT) {
            float x[4][EPC];
#pragma unroll
            for (int u = 0; u < 4; ++u) E::unpack(lds128(sbase + 16 * (c + u * GT)), x[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float gv[EPC];
#pragma unroll
              for (int q = 0; q < EPC; q += 2) grad_pair(x[u] + q, gv + q, mh, f);
              sts128(sbase + 16 * (c + u * GT), E::pack(gv));
            }
          }
          for (; c < f1; c += GT) {
            float x[EPC], gv[EPC];
            E::unpack(lds128(sbase + 16 * c), x);
#pragma unroll
            for (int q = 0; q < EPC; q += 2) grad_pair(x + q, gv + q, mh, f);
            sts128(sbase + 16 * c, E::pack(gv));
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = h ? ce_back : ce_front;
          if (c >= 0) {
            float x[EPC], gv[EPC];
            edge_load(c, x);
#pragma unroll
            for (int q = 0; q < EPC; ++q) gv[q] = ex2(fmaf(x[q], kLog2e, -mh)) * f;
            edge_store(c, gv);
          }
        }
        if (owner) {
          // exp(x_t - lse) - 1 without cancellation when the target dominates
          const float gval = expm1_target((xt - Mg) - lg2(Sg) * kLn2) * sc;
          if (t_smem) E::st(smem_ptr(tbo), gval);
          else E::st(elem_ptr_global(static_cast<int>(t)), gval);
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&done_bar[s]));
      }
    }

    // ---- deterministic reduction of the loss ----
    if (p.loss != nullptr) {
      if (gt == 0) acc_slot[grp] = acc.value();
      group_sync(15, NC);  // an id no row group uses
      if (warp == 0) loss_tail_warp(acc_slot, R, p.partials, p.ticket, p.loss, p.M, p.mean, lane);
    }
  }

  if (CL > 1) {
    __syncwarp();
    cluster_sync_all();  // no CTA leaves while a peer may still write into its shared memory
  }
}

}  // namespace ce
