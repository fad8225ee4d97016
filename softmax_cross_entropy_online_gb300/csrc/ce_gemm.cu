// ce_gemm.cu -- the dense contractions of the fused linear + cross-entropy
// ("9 Triton kernels in 9 weeks", week eight: the lm_head projection chunked
// into the loss), on the 5th-generation tensor cores of sm_103a:
//
//     D[M, N] (fp32)  =  A[M, K] . B[N, K]^T  (+ beta * D)
//
// with A and B bf16, each stored either K-major (K contiguous) or MN-major (M or
// N contiguous, i.e. the transpose): the fused path reads W, G and h in the
// layout they have, with no transpose pass.
//
// Design: a persistent kernel, one CTA per SM, warp-specialised.
//  * warp 0 (one thread) streams 128x64 tiles of A and 256x64 tiles of B into a
//    ring of shared-memory stages with TMA (cp.async.bulk.tensor, 128-byte
//    swizzle), completion counted on an mbarrier per stage;
//  * warp 1 allocates 512 TMEM columns (two 128x256 fp32 accumulators) and one
//    of its threads issues tcgen05.mma (M=128, N=256, K=16, bf16 -> fp32) from
//    the shared-memory descriptors; tcgen05.commit frees a stage when the MMAs
//    that read it are done and signals a full accumulator after the last k-tile;
//  * warps 2..5 are the epilogue: each reads its 32 TMEM lanes (tile rows) with
//    tcgen05.ld, 32 columns at a time, writes the 32 x 32 block into shared
//    memory (128-byte swizzle) and hands it to a TMA tensor store, or, to
//    accumulate (D += ...), a TMA tensor reduce-add done in L2; rows of D off the
//    16-byte grid are written by the warp instead, one row segment per access.
//    With two accumulators the epilogue of one tile overlaps the main loop of
//    the next.
// Every mbarrier wait is bounded (see ce_rows.cuh); TMEM is freed on every path.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "../../include/ce_gb300.h"
#include "ce_lce.cuh"
#include "ce_rows.cuh"
#include "ce_tc.cuh"

namespace ce {

constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;
constexpr int kGemmBK = 64;  // one 128-byte swizzle row of bf16
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192;
constexpr int kTileABytes = kGemmBM * kGemmBK * 2;  // 16 KB
constexpr int kTileBBytes = kGemmBN * kGemmBK * 2;  // 32 KB
constexpr int kStageBytes = kTileABytes + kTileBBytes;
constexpr int kEpiBytes = 32 * 32 * 4;  // one epilogue warp's 32 x 32 fp32 block
constexpr int kGemmSmem = kGemmStages * kStageBytes + 4 * kEpiBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;

struct GemmParams {
  int M, N, K;
  float* D;
  long long ldd;  // elements between rows of D
  float beta;     // 0: D = A B^T; 1: D += A B^T
  int use_tma;    // D written by TMA tensor stores / reduce-adds (rows 16-byte aligned)
  int tiles_m, tiles_n, k_tiles;
  int n_fast;     // tile order: 1 = N varies fastest (A the larger operand), 0 = M
  int a_mn, b_mn; // operand stored MN-major (M or N contiguous) instead of K-major
  int a_3d, b_3d; // MN-major operand loaded by one 3-D box per stage (M / N % 64 == 0)
  unsigned int* err;
  unsigned int wait_hint_ns;
  LceArgs lce;    // the fused linear + CE epilogue's work (LCE kernels only)
};

// instruction descriptor of kind::f16: D fp32, A and B bf16, N=256, M=128; bits
// 15 and 16 mark A and B as MN-major
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kGemmBN >> 3) << 17) |
                            ((kGemmBM >> 4) << 24);

// Tile order of the persistent grid: the CTAs running at the same time share
// the tiles of the smaller operand through L2 while the larger operand streams
// from HBM once (M fastest when B is the larger, N fastest when A is).
__device__ __forceinline__ void tile_coords(const GemmParams& p, int tile, int& tm, int& tn) {
  if (p.n_fast) {
    tn = tile % p.tiles_n;
    tm = tile / p.tiles_n;
  } else {
    tm = tile % p.tiles_m;
    tn = tile / p.tiles_m;
  }
}


// ---------------------------------------------------------------------------
// The fused linear + CE's gradient rows, formed by one warp per row from the
// stored fp32 logits and the row's per-tile (max, sum) pairs (ce_lce.cuh).
// ---------------------------------------------------------------------------

// Merge of two (max, sum of exp(x - max)) pairs: the larger max is kept and
// the other sum rescaled by exp(its max - the larger max); two empty pairs
// (-inf, 0) stay empty.
__device__ __forceinline__ void merge_pair(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  const float f1 = (m == -INFINITY) ? 0.f : ex2((m - mn) * kLog2e);
  const float f2 = (m2 == -INFINITY) ? 0.f : ex2((m2 - mn) * kLog2e);
  s = s * f1 + s2 * f2;
  m = mn;
}

// One warp's share of the gradient rows: a contiguous range of the chunk's
// 4-logit chunks (row-major over the rows), so every warp gets the same amount
// of work whatever the row count.  The warp walks it row by row: r the current
// row (done once r >= bg_rows), pos the next chunk in it (-1 until the row's
// pairs are merged), end_r / end_pos where the range stops, and the row's
// constants.
struct BgRow {
  int r, pos;           // the current row, and its next chunk (-1: pairs not merged yet)
  int start;            // where the warp's work in the next row to merge begins
  int end_r, end_pos;   // the range ends before chunk end_pos of row end_r
  long long t;          // the row's target
  float Lh, scf, gt;    // lse log2e = Lh + (correction in scf); scf = 2^-correction * scale; g_t
};

// Warp `gw` of `nwarps`: its range [gw * total / nwarps, (gw + 1) * total / nwarps)
// of the rows * ceil(V / 4) chunks.
__device__ __forceinline__ void bg_range(const LceArgs& a, BgRow& w, int gw, int nwarps) {
  const long long nch = (a.V + 3) >> 2;
  const long long total = static_cast<long long>(a.bg_rows) * nch;
  const long long g0 = total * gw / nwarps, g1 = total * (gw + 1) / nwarps;
  w.r = static_cast<int>(g0 / nch);
  w.start = static_cast<int>(g0 % nch);
  w.pos = -1;
  w.end_r = static_cast<int>(g1 / nch);
  w.end_pos = static_cast<int>(g1 % nch);
  if (g0 >= g1) w.r = w.end_r = a.bg_rows;  // an empty range
  w.t = -1;
  w.Lh = w.scf = w.gt = 0.f;
}

__device__ __forceinline__ bool bg_active(const LceArgs& a, const BgRow& w) {
  return w.r < w.end_r ||
         (w.r == w.end_r && w.r < a.bg_rows && w.end_pos > 0 && (w.pos < 0 || w.pos < w.end_pos));
}

// A row's constants from its per-tile pairs, the warp's lanes sharing the
// merge: the merged (m, s), ln s, lse log2e split into Lh + Lc (Lc a small
// correction taken once into the scale: scf = 2^-Lc * scale), and the target's
// gradient exp(x_t - lse) - 1 times the scale, without cancellation when the
// target dominates.
struct RowConsts {
  float m, lnS, Lh, scf, gt;
};
__device__ __forceinline__ RowConsts lce_row_consts(const float2* pp, int n_tiles, float xt,
                                                    float scale, int lane) {
  float m = -INFINITY, s = 0.f;
  for (int j = lane; j < n_tiles; j += 32) {
    const float2 q = __ldcg(pp + j);
    merge_pair(m, s, q.x, q.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge_pair(m, s, m2, s2);
  }
  const float mref = (m == -INFINITY) ? 0.f : m;
  const float mhr = mref * kLog2e;
  const float mlr = fmaf(mref, kLog2e, -mhr);
  const float l2s = lg2(s);
  const float Lh = mhr + l2s;
  const float bv = Lh - mhr;
  const float Lc = mlr + ((mhr - (Lh - bv)) + (l2s - bv));
  RowConsts c;
  c.m = m;
  c.lnS = l2s * kLn2;
  c.Lh = Lh;
  c.scf = ex2(-Lc) * scale;
  c.gt = expm1_target((xt - m) - c.lnS) * scale;
  return c;
}

// Merge row w.r's tile pairs into its log-sum-exp, write its row loss (the warp
// whose range holds the row's first chunk), and prepare the constants of its
// gradient; `start` is the chunk the warp's work in this row begins at.
__device__ __forceinline__ void bg_merge(const LceArgs& a, BgRow& w, int lane, int start) {
  const long long t = __ldg(a.bg_targets + w.r);
  const bool t_ok = t >= 0 && t < a.V;
  const float xt = t_ok ? __ldcg(a.bg_xt + w.r) : 0.f;
  const RowConsts c =
      lce_row_consts(a.bg_part + static_cast<long long>(w.r) * a.n_tiles, a.n_tiles, xt, a.scale, lane);
  w.t = t_ok ? t : -1;
  w.Lh = c.Lh;
  w.scf = c.scf;
  w.gt = c.gt;
  if (lane == 0 && start == 0) {
    a.bg_rl[w.r] = t_ok ? (c.m - xt) + c.lnS : __int_as_float(0x7fc00000);
    if (!t_ok) atomicOr(a.err, ERR_TARGET_RANGE);
  }
  w.pos = start;
}

// Up to NL x 32 consecutive 4-logit chunks of row w.r from w.pos on (not past
// the warp's range): g = exp(x - lse) * scale in bf16, the target's element
// overwritten by the lane that stored its chunk.  Moves w to the next row at
// the row's end.
template <int NL>
__device__ __forceinline__ void bg_chunks(const LceArgs& a, BgRow& w, int lane) {
  const int nrow = (a.V + 3) >> 2;
  const int nch = (w.r == w.end_r) ? w.end_pos : nrow;  // this row's last chunk + 1 for the warp
  const float* row = a.bg_logits + static_cast<long long>(w.r) * a.ldl;
  __nv_bfloat16* grow = a.bg_g16 + static_cast<long long>(w.r) * a.ldv;
  float4 x[NL];
#pragma unroll
  for (int k = 0; k < NL; ++k) {
    const int c = w.pos + lane + 32 * k;
    if (c < nch) x[k] = __ldcs(reinterpret_cast<const float4*>(row) + c);
  }
  const int tc = w.t >= 0 ? static_cast<int>(w.t >> 2) : -1;
#pragma unroll
  for (int k = 0; k < NL; ++k) {
    const int c = w.pos + lane + 32 * k;
    if (c < nch) {
      float g[4] = {ex2(fmaf(x[k].x, kLog2e, -w.Lh)) * w.scf, ex2(fmaf(x[k].y, kLog2e, -w.Lh)) * w.scf,
                    ex2(fmaf(x[k].z, kLog2e, -w.Lh)) * w.scf, ex2(fmaf(x[k].w, kLog2e, -w.Lh)) * w.scf};
      if (4 * c + 4 > a.V) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * c + e >= a.V) g[e] = 0.f;  // columns past V (never read as data)
      }
      const __nv_bfloat162 lo = __floats2bfloat162_rn(g[0], g[1]);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(g[2], g[3]);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&lo);
      u.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(grow + 4LL * c) = u;
      if (c == tc) grow[w.t] = __float2bfloat16_rn(w.gt);
    }
  }
  w.pos += 32 * NL;
  if (w.pos >= nch) {
    ++w.r;
    w.pos = -1;
  }
}

// One step of a warp's share: merge the next row's pairs, or form a slice.
template <int NL>
__device__ __forceinline__ void bg_step(const LceArgs& a, BgRow& w, int lane) {
  if (w.pos < 0) {
    bg_merge(a, w, lane, w.start);
    w.start = 0;  // every later row of the range starts at its first chunk
  } else {
    bg_chunks<NL>(a, w, lane);
  }
}

// A standalone pass over one chunk's rows (the last chunk of a call): a warp
// per row, rows r = warp, warp + nwarps, ...
__global__ void __launch_bounds__(256) lce_grad_rows_kernel(const LceArgs a) {
  const int lane = threadIdx.x & 31;
  const int nwarps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  BgRow w;
  bg_range(a, w, static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5), nwarps);
  while (bg_active(a, w)) bg_step<16>(a, w, lane);
}

// The lean schedule's merge pass: a warp per row of the chunk turns the row's
// pairs into its constants (a.rowc) and loss (a.rl); a target outside [0, V)
// gives a NaN loss, no one-hot term (-1 in the constants) and the error word.
__global__ void __launch_bounds__(256) lce_merge_rows_kernel(const LceArgs a) {
  const int lane = threadIdx.x & 31;
  const int nwarps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  for (int r = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5); r < a.rows;
       r += nwarps) {
    const long long t = __ldg(a.targets + r);
    const bool t_ok = t >= 0 && t < a.V;
    const float xt = t_ok ? __ldcg(a.xt + r) : 0.f;
    const RowConsts c =
        lce_row_consts(a.part + static_cast<long long>(r) * a.n_tiles, a.n_tiles, xt, a.scale, lane);
    if (lane == 0) {
      a.rowc[r] = make_float4(c.Lh, c.scf, c.gt, __int_as_float(t_ok ? static_cast<int>(t) : -1));
      a.rl[r] = t_ok ? (c.m - xt) + c.lnS : __int_as_float(0x7fc00000);
      if (!t_ok) atomicOr(a.err, ERR_TARGET_RANGE);
    }
  }
}

// A_MN / B_MN: the operands' layouts, fixed at compile time so that the
// K-major form runs exactly the code it would alone.  EPI (K-major operands
// only) extends the epilogue for the fused linear + CE:
//  * kLceStats: the logits GEMM, whose epilogue also reduces each row over each
//    tile to a (max, sum) pair and keeps the target logit; with p.lce.store it
//    stores the logits too and forms the previous chunk's gradient rows while
//    it waits for accumulators, without it stores nothing else;
//  * kLceGrad: the logits GEMM again, whose epilogue writes the bf16 gradient
//    exp(x - lse) * scale (the target's from the row's constants) instead of
//    the logits.
template <bool A_MN, bool B_MN, int EPI = 0>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tma_a,
                        const __grid_constant__ CUtensorMap tma_b,
                        const __grid_constant__ CUtensorMap tma_d, const GemmParams p) {
  constexpr bool LCE = EPI == kLceStats;
  constexpr bool GRAD = EPI == kLceGrad;
  extern __shared__ unsigned char gsm[];
  __shared__ __align__(8) unsigned long long full_bar[kGemmStages];
  __shared__ __align__(8) unsigned long long empty_bar[kGemmStages];
  __shared__ __align__(8) unsigned long long accf_bar[2];
  __shared__ __align__(8) unsigned long long acce_bar[2];
  __shared__ uint32_t tmem_slot;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = (smem_u32(gsm) + 1023u) & ~1023u;  // swizzle atoms need 1024 B
  bool failed = false;
  const unsigned int hint = p.wait_hint_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&accf_bar[a]), 1);
      mbar_init(smem_u32(&acce_bar[a]), 128);
    }
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int num_tiles = p.tiles_m * p.tiles_n;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int s = 0;
      uint32_t ph = 0;
      uint32_t filled = 0;  // stages that received at least one load
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        int tm, tn;
        tile_coords(p, tile, tm, tn);
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          mbar_wait<false>(smem_u32(&empty_bar[s]), ph ^ 1u, p.err, failed, WAIT_LIMIT_NS, hint);
          const uint32_t fb = smem_u32(&full_bar[s]);
          const uint32_t sa = sbase + s * kStageBytes;
          mbar_arrive_expect_tx(fb, kStageBytes);
          if (A_MN && p.a_3d) {
            tma_load_3d(sa, &tma_a, 0, kt * kGemmBK, tm * (kGemmBM / 64), fb);
          } else if (A_MN) {
            for (int j = 0; j < kGemmBM / 64; ++j)
              tma_load_2d(sa + j * 8192, &tma_a, tm * kGemmBM + 64 * j, kt * kGemmBK, fb);
          } else {
            tma_load_2d(sa, &tma_a, kt * kGemmBK, tm * kGemmBM, fb);
          }
          if (B_MN && p.b_3d) {
            tma_load_3d(sa + kTileABytes, &tma_b, 0, kt * kGemmBK, tn * (kGemmBN / 64), fb);
          } else if (B_MN) {
            for (int j = 0; j < kGemmBN / 64; ++j)
              tma_load_2d(sa + kTileABytes + j * 8192, &tma_b, tn * kGemmBN + 64 * j,
                          kt * kGemmBK, fb);
          } else {
            tma_load_2d(sa + kTileABytes, &tma_b, kt * kGemmBK, tn * kGemmBN, fb);
          }
          filled |= 1u << s;
          if (++s == kGemmStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // the CTA may not exit with a load in flight: wait (bounded) for the last
      // load of every stage (already complete unless a wait above timed out)
      for (int k = 0; k < kGemmStages; ++k) {
        if (!(filled & (1u << k))) continue;
        const uint32_t last_ph = (k < s) ? ph : (ph ^ 1u);
        mbar_wait<false>(smem_u32(&full_bar[k]), last_ph, p.err, failed, WAIT_LIMIT_NS, hint);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      int s = 0, a = 0;
      uint32_t ph = 0, aph = 0;
      constexpr uint32_t idesc = kIdesc | (A_MN ? (1u << 15) : 0u) | (B_MN ? (1u << 16) : 0u);
      // one MMA's K = 16 step: 32 bytes inside a K-major row, 2048 bytes (16
      // K-rows) in an MN-major tile; descriptors count 16-byte units
      constexpr uint64_t a_step = A_MN ? 128 : 2, b_step = B_MN ? 128 : 2;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        mbar_wait<false>(smem_u32(&acce_bar[a]), aph ^ 1u, p.err, failed, WAIT_LIMIT_NS, hint);
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(a * kGemmBN);
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          mbar_wait<false>(smem_u32(&full_bar[s]), ph, p.err, failed, WAIT_LIMIT_NS, hint);
          tc_fence_after();
          const uint32_t sa = sbase + s * kStageBytes;
          const uint64_t da = A_MN ? smem_desc_sw128_mn(sa) : smem_desc_sw128(sa);
          const uint64_t db =
              B_MN ? smem_desc_sw128_mn(sa + kTileABytes) : smem_desc_sw128(sa + kTileABytes);
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)
            umma_bf16(d_tmem, da + a_step * kk, db + b_step * kk, idesc, (kt | kk) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&empty_bar[s]));
          if (++s == kGemmStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        umma_commit(smem_u32(&accf_bar[a]));
        a ^= 1;
        if (a == 0) aph ^= 1u;
      }
    }
  } else {
    // ---------------- epilogue: warps 2..5 ----------------
    const int q = warp & 3;  // the TMEM lane quarter this warp may access
    // this warp's 32 x 32 fp32 block in shared memory, in the 128-byte swizzled
    // layout of the D tensor map: row r at 128 r, its 16-byte chunk c at chunk
    // c ^ (r & 7) (written by lane = row without more than 4-way conflicts,
    // read by lane = column without any)
    const uint32_t ebuf = sbase + kGemmStages * kStageBytes + q * kEpiBytes;
    int a = 0;
    uint32_t aph = 0;
    // LCE: this warp's background rows of the previous chunk
    BgRow bg;
    const bool bg_on = LCE && p.lce.bg_rows > 0;
    if (bg_on) bg_range(p.lce, bg, static_cast<int>(blockIdx.x) * 4 + q, static_cast<int>(gridDim.x) * 4);
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int tm, tn;
      tile_coords(p, tile, tm, tn);
      if (LCE) {
        // while the accumulator fills, form background gradient rows (a slice
        // takes a few microseconds; a tile's MMAs take about 25); once they run
        // out, wait as usual (bounded)
        while (!mbar_test_wait(smem_u32(&accf_bar[a]), aph)) {
          if (bg_on && bg_active(p.lce, bg)) {
            bg_step<16>(p.lce, bg, lane);
          } else {
            mbar_wait<false>(smem_u32(&accf_bar[a]), aph, p.err, failed, WAIT_LIMIT_NS, hint);
            break;
          }
        }
      } else {
        mbar_wait<false>(smem_u32(&accf_bar[a]), aph, p.err, failed, WAIT_LIMIT_NS, hint);
      }
      tc_fence_after();
      const int rbase = tm * kGemmBM + 32 * q;  // this warp's 32 rows of the tile
      if constexpr (GRAD) {
        // this thread's row (TMEM lane): g = 2^(x log2e - Lh) * scf, the
        // target's element from the row's constants; 64 columns (one
        // 128-byte swizzled row of bf16 per thread) per TMA store
        const int my_row = rbase + lane;
        float4 rc = make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
        if (my_row < p.lce.rows) rc = __ldg(p.lce.rowc + my_row);
        const int my_t = __float_as_int(rc.w);
#pragma unroll 1
        for (int cc = 0; cc < kGemmBN / 64; ++cc) {
          uint32_t r[64];
          const uint32_t ta = tmem + static_cast<uint32_t>(a * kGemmBN + cc * 64) +
                              (static_cast<uint32_t>(32 * q) << 16);
          tmem_ld32_nowait(ta, r);
          tmem_ld32_nowait(ta + 32, r + 32);
          tmem_wait_ld<64>(r);
          const int col0 = tn * kGemmBN + cc * 64;
          const int o = my_t - col0;  // the target's place in this block (none outside [0, 64))
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float g0 = ex2(fmaf(__uint_as_float(r[2 * j]), kLog2e, -rc.x)) * rc.y;
            float g1 = ex2(fmaf(__uint_as_float(r[2 * j + 1]), kLog2e, -rc.x)) * rc.y;
            if (o == 2 * j) g0 = rc.z;
            if (o == 2 * j + 1) g1 = rc.z;
            __nv_bfloat162 hv = __floats2bfloat162_rn(g0, g1);
            pk[j] = *reinterpret_cast<uint32_t*>(&hv);
          }
          // the previous block's store has read the buffer
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             ebuf + lane * 128 + 16 * (j ^ (lane & 7))),
                         "r"(pk[4 * j]), "r"(pk[4 * j + 1]), "r"(pk[4 * j + 2]), "r"(pk[4 * j + 3])
                         : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tma_d, ebuf, col0, rbase);
            bulk_commit();
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&acce_bar[a]));
        a ^= 1;
        if (a == 0) aph ^= 1u;
        continue;
      }
      // LCE: this thread's row (TMEM lane) and its running pair over the tile
      const int my_row = rbase + lane;
      long long my_t = -1;
      if (LCE && my_row < p.lce.rows) my_t = __ldg(p.lce.targets + my_row);
      float sm = -INFINITY, smh = 0.f, ss = 0.f, xtv = 0.f;
      bool hx = false;
#pragma unroll 1
      for (int cc = 0; cc < kGemmBN / 32; ++cc) {
        float v[32];
        tmem_ld32(tmem + static_cast<uint32_t>(a * kGemmBN + cc * 32) +
                      (static_cast<uint32_t>(32 * q) << 16),
                  v);
        const int col0 = tn * kGemmBN + cc * 32;
        if (LCE) {
          // the row's pair over these 32 columns (those past V excluded): the
          // max first, then one exp2 per value against the running reference
          const int nv = p.lce.V - col0;
          if (nv > 0) {
            float cm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (nv >= 32 || j < nv) cm = fmaxf(cm, v[j]);
            if (cm > sm) {
              const float nh = cm * kLog2e;
              ss = (sm == -INFINITY) ? 0.f : ss * ex2(smh - nh);
              sm = cm;
              smh = nh;
            }
            if (sm != -INFINITY) {
              float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (nv >= 32 || j < nv) a4[j & 3] += ex2(fmaf(v[j], kLog2e, -smh));
              ss += (a4[0] + a4[1]) + (a4[2] + a4[3]);
            }
            if (my_t >= col0 && my_t < col0 + 32) {
              const int o = static_cast<int>(my_t - col0);
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j == o) xtv = v[j];
              hx = true;
            }
          }
        }
        if (LCE && !p.lce.store) continue;  // the pairs only: nothing is stored
        if (p.use_tma) {
          // the previous block's store has read the buffer
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                           ebuf + lane * 128 + 16 * (j ^ (lane & 7))),
                       "f"(v[4 * j]), "f"(v[4 * j + 1]), "f"(v[4 * j + 2]), "f"(v[4 * j + 3])
                       : "memory");
        if (p.use_tma) {
          fence_proxy_async_smem();  // the block is visible to the TMA engine
          __syncwarp();
          if (lane == 0) {
            if (p.beta != 0.f) tma_reduce_add_2d(&tma_d, ebuf, col0, rbase);
            else tma_store_2d(&tma_d, ebuf, col0, rbase);
            bulk_commit();
          }
        } else {
          // rows of D off the 16-byte grid: lane = column, one row segment per access
          __syncwarp();
          const int col = col0 + lane;
          const bool col_ok = col < p.N;
          float* const dcol = p.D + col;
          const uint32_t rd = ebuf + 16 * (lane >> 2) + 4 * (lane & 3);
          float val[32];
#pragma unroll
          for (int r = 0; r < 32; ++r) {
            asm volatile("ld.shared.f32 %0, [%1];"
                         : "=f"(val[r])
                         : "r"((rd + r * 128) ^ (static_cast<uint32_t>(r & 7) << 4)));
          }
          if (p.beta != 0.f) {
            float old[32];
#pragma unroll
            for (int r = 0; r < 32; ++r)
              old[r] = (col_ok && rbase + r < p.M)
                           ? dcol[static_cast<long long>(rbase + r) * p.ldd]
                           : 0.f;
#pragma unroll
            for (int r = 0; r < 32; ++r) val[r] += old[r];
          }
#pragma unroll
          for (int r = 0; r < 32; ++r)
            if (col_ok && rbase + r < p.M) dcol[static_cast<long long>(rbase + r) * p.ldd] = val[r];
          __syncwarp();  // the block is read out before the next one is written
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&acce_bar[a]));
      if (LCE && my_row < p.lce.rows) {
        // the pair in natural units: ss counts 2^(x log2e - smh), smh rounded
        const float ml = (sm == -INFINITY) ? 0.f : fmaf(sm, kLog2e, -smh);
        p.lce.part[static_cast<long long>(my_row) * p.lce.n_tiles + tn] =
            make_float2(sm, (sm == -INFINITY) ? 0.f : ss * ex2(-ml));
        if (hx) p.lce.xt[my_row] = xtv;
      }
      a ^= 1;
      if (a == 0) aph ^= 1u;
    }
    // the rest of this warp's background rows
    if (bg_on) {
      while (bg_active(p.lce, bg)) bg_step<16>(p.lce, bg, lane);
    }
    // no CTA exits while a TMA store still reads its shared memory
    if (p.use_tma && lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// --- host side ---------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 tensor map over `rows` x `cols` (cols contiguous, row stride ld
// elements) with a box of box_rows x 64 and 128-byte swizzle: K-major tiles take
// box_rows = 128 / 256 rows of 64 K; MN-major tiles take 64 K-rows of 64
static bool make_map(CUtensorMap* map, const void* base, long long rows, long long cols,
                     long long ld, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor map of an MN-major operand whose MN extent is a multiple of
// 64: element (mn, k) at (mn % 64, k, mn / 64); one box of 64 x 64 x blocks
// lands the 64-wide blocks of a tile one after another (8 KB apart), the
// layout the MN-major descriptor expects, in a single copy
static bool make_map_mn3d(CUtensorMap* map, const void* base, long long k_rows, long long mn,
                          long long ld, int blocks) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(k_rows), static_cast<cuuint64_t>(mn / 64)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, 128};
  cuuint32_t box[3] = {64u, 64u, static_cast<cuuint32_t>(blocks)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 tensor map over D (rows x cols, row stride ld elements, a multiple
// of 4) with a box of 32 x 32 and 128-byte swizzle: the epilogue's blocks
static bool make_map_f32(CUtensorMap* map, void* base, long long rows, long long cols,
                         long long ld) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor map over the gradient rows G (rows x cols, row stride ld
// elements, a multiple of 8) with a box of 64 x 32 and 128-byte swizzle: the
// gradient epilogue's blocks (one 128-byte row of bf16 per thread)
static bool make_map_g16(CUtensorMap* map, void* base, long long rows, long long cols,
                         long long ld) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// D[M,N] = op(A) op(B)^T (+ beta D), bf16 inputs, fp32 D.  a_mn = false: A is
// [M, lda] with K contiguous; a_mn = true: A is stored [K, lda] with M contiguous
// (the transpose of a K-major A).  The same for B with N.  Requires lda, ldb
// multiples of 8 (16-byte row strides for TMA) and 16-byte aligned A and B;
// tiles reaching past M, N or K are zero-filled by TMA.
// lce (both operands K-major, beta = 0): the fused linear + CE's logits GEMM,
// with the epilogue work of ce_lce.cuh.  lce->mode kLceStats with lce->store
// needs D with rows on the 16-byte grid; without it, and in kLceGrad (which
// writes lce->g16, row stride lce->ldv, a multiple of 8), D is not used.
ce_status gemm_bf16(const void* A, long long lda, bool a_mn, const void* B, long long ldb,
                    bool b_mn, float* D, long long ldd, int M, int N, int K, float beta,
                    cudaStream_t stream, unsigned int* err, int sm_count,
                    unsigned int wait_hint_ns, const LceArgs* lce) {
  if (M <= 0 || N <= 0 || K <= 0) return CE_OK;
  if (lce != nullptr && (a_mn || b_mn || beta != 0.f)) return CE_ERR_UNSUPPORTED;
  const bool lce_d = lce == nullptr || (lce->mode == kLceStats && lce->store);  // D written
  if ((lda % 8) || (ldb % 8) || (lce_d && ldd < N)) return CE_ERR_UNSUPPORTED;
  if ((a_mn ? lda < M : lda < K) || (b_mn ? ldb < N : ldb < K)) return CE_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15))
    return CE_ERR_UNSUPPORTED;
  CUtensorMap ma, mb, md;
  // MN-major with an MN extent of whole 64-element blocks: one 3-D box per tile
  const bool a_3d = a_mn && (M % 64 == 0), b_3d = b_mn && (N % 64 == 0);
  const bool ok_a = a_3d ? make_map_mn3d(&ma, A, K, M, lda, kGemmBM / 64)
                         : (a_mn ? make_map(&ma, A, K, M, lda, 64) : make_map(&ma, A, M, K, lda, kGemmBM));
  const bool ok_b = b_3d ? make_map_mn3d(&mb, B, K, N, ldb, kGemmBN / 64)
                         : (b_mn ? make_map(&mb, B, K, N, ldb, 64) : make_map(&mb, B, N, K, ldb, kGemmBN));
  if (!ok_a || !ok_b) return CE_ERR_CUDA;
  // D by TMA when its rows sit on the 16-byte grid (the tensor map's stride rule)
  bool use_tma = lce_d && (ldd % 4 == 0) && ((reinterpret_cast<uintptr_t>(D) & 15) == 0);
  std::memset(&md, 0, sizeof(md));
  if (use_tma && !make_map_f32(&md, D, M, N, ldd)) return CE_ERR_CUDA;
  if (lce != nullptr && lce->mode == kLceGrad) {
    if (lce->g16 == nullptr || (lce->ldv % 8) || lce->ldv < N ||
        (reinterpret_cast<uintptr_t>(lce->g16) & 15))
      return CE_ERR_UNSUPPORTED;
    if (!make_map_g16(&md, lce->g16, M, N, lce->ldv)) return CE_ERR_CUDA;
    use_tma = true;  // the gradient blocks leave by TMA stores
  }
  GemmParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.D = D;
  p.ldd = ldd;
  p.beta = beta;
  p.use_tma = use_tma ? 1 : 0;
  p.tiles_m = (M + kGemmBM - 1) / kGemmBM;
  p.tiles_n = (N + kGemmBN - 1) / kGemmBN;
  p.k_tiles = (K + kGemmBK - 1) / kGemmBK;
  p.n_fast = M > N ? 1 : 0;  // A [M, K] the larger operand
  p.a_mn = a_mn ? 1 : 0;
  p.b_mn = b_mn ? 1 : 0;
  p.a_3d = a_3d ? 1 : 0;
  p.b_3d = b_3d ? 1 : 0;
  p.err = err;
  p.wait_hint_ns = wait_hint_ns;
  std::memset(&p.lce, 0, sizeof(p.lce));
  if (lce != nullptr) {
    if ((lce_d && !use_tma) || lce->n_tiles != p.tiles_n || lce->rows != M || lce->V != N ||
        (lce->mode != kLceStats && lce->mode != kLceGrad))
      return CE_ERR_UNSUPPORTED;
    p.lce = *lce;
  }
  auto kern = lce != nullptr ? (lce->mode == kLceGrad ? gemm_bf16_kernel<false, false, kLceGrad>
                                                      : gemm_bf16_kernel<false, false, kLceStats>)
              : a_mn ? (b_mn ? gemm_bf16_kernel<true, true> : gemm_bf16_kernel<true, false>)
                     : (b_mn ? gemm_bf16_kernel<false, true> : gemm_bf16_kernel<false, false>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem) !=
      cudaSuccess)
    return CE_ERR_CUDA;
  const int tiles = p.tiles_m * p.tiles_n;
  const int grid = tiles < sm_count ? tiles : sm_count;
  kern<<<grid, kGemmThreads, kGemmSmem, stream>>>(ma, mb, md, p);
  return cudaGetLastError() == cudaSuccess ? CE_OK : CE_ERR_CUDA;
}

}  // namespace ce

namespace ce {

// --- the mean of the row losses of the fused linear + cross-entropy ------------

// loss = (sum of rl[0..M)) / M: one CTA, each thread sums a fixed stride in
// fp64, then a fixed-order tree; deterministic, no atomics
__global__ void mean_rows_kernel(const float* __restrict__ rl, long long M, float* loss) {
  __shared__ double part[1024];
  double s = 0.0;
  for (long long i = threadIdx.x; i < M; i += blockDim.x) s += static_cast<double>(rl[i]);
  part[threadIdx.x] = s;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = static_cast<float>(part[0] / static_cast<double>(M));
}

ce_status launch_mean_rows(const float* rl, long long M, float* loss, cudaStream_t st) {
  mean_rows_kernel<<<1, 1024, 0, st>>>(rl, M, loss);
  return cudaGetLastError() == cudaSuccess ? CE_OK : CE_ERR_CUDA;
}

// The gradient rows of a.bg_rows rows (the last chunk of a fused linear + CE
// call), a warp per row, 8 warps a CTA.
ce_status launch_lce_merge_rows(const LceArgs& a, cudaStream_t st, int sm_count) {
  if (a.rows <= 0) return CE_OK;
  int grid = (a.rows + 7) / 8;
  if (grid > sm_count * 8) grid = sm_count * 8;
  lce_merge_rows_kernel<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? CE_OK : CE_ERR_CUDA;
}

ce_status launch_lce_grad_rows(const LceArgs& a, cudaStream_t st, int sm_count) {
  if (a.bg_rows <= 0) return CE_OK;
  int grid = (a.bg_rows + 7) / 8;
  if (grid > sm_count * 8) grid = sm_count * 8;
  lce_grad_rows_kernel<<<grid, 256, 0, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? CE_OK : CE_ERR_CUDA;
}

}  // namespace ce
