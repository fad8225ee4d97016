// ce_attention.cu -- the blockwise attention forward on the tcgen05 tensor
// cores of sm_103a: the workload of "How to optimize an existing Triton Kernel
// to make it faster?" (Triton discussion #8261), whose flash-attention-2
// listing keeps, per query row, a running max and a running normaliser over
// blocks of keys and rescales the output accumulator when the max grows --
// the same online (max, sum) pair as the cross-entropy rows.  For Q, K, V of
// shape [B * NH, T, D] (bf16), an optional additive mask [T, T] and/or the
// causal mask, and sm_scale:
//
//     O = softmax(Q K^T * sm_scale + mask) V        (fp32)
//     lse_i = log sum_j exp(S_ij)                    (fp32, optional)
//
// Design (persistent, one CTA per SM, 320 threads; a work item is 128 query
// rows of one head; neighbouring CTAs work on the same head so its K and V
// are read from L2; under the causal mask query tiles are paired so every
// work unit costs the same):
//  * warp 0 (one thread) loads each item's Q tile (two buffers: the next
//    item's Q arrives while this one computes) and streams K tiles of 128
//    keys into a three-stage ring and V tiles into a two-stage ring with TMA
//    (128-byte swizzle; K K-major for S = Q K^T, V MN-major for O = P V, so
//    neither is transposed); K runs one tile ahead of V within an item (an
//    item's last V is loaded with it), each K stage refilled once its score
//    MMA has read it;
//  * warp 1 allocates all 512 TMEM columns -- two 128 x 128 fp32 score
//    buffers, the D-column output accumulator, two bf16 weight buffers P --
//    and one thread issues the MMAs: scores run two tiles ahead, S_{j+2} =
//    Q K_{j+2}^T issued as soon as the softmax holds S_j in registers and
//    before O += P_j V_j (A operand P read from TMEM), so the tensor cores
//    always have the next scores queued while the softmax warps work;
//  * warps 2..9 give each query row two threads (TMEM lane = row; two warps
//    per lane quarter), each with 64 of a tile's 128 keys: they load those
//    scores into registers (freeing the score buffer), swap partial maxima
//    through shared memory for the tile max (one named barrier per swap: each
//    thread writes the slot it read at the previous swap), move the row's reference max only
//    when the tile max exceeds it by more than 2^8 (then each rescales its half
//    of the row of O in TMEM after the previous P V has run), write
//    P = 2^(s c - ref) as bf16 into TMEM and add it to their share of the
//    normaliser l.  At the end of the item the two shares are summed and each
//    thread stages its half of O / l (fp32, or rounded to bf16) in shared
//    memory (one block per warp at a time) for TMA tensor stores; lse is
//    written by the first.  For D = 128 the staging blocks are the item's own
//    Q buffer (its score MMAs have all run by then), which the producer
//    reloads only after each warp's stores have read it.
//  * exp is exp2 of the score in log2 units: s * sm_scale * log2(e).  The
//    softmax warps issue the most instructions per tile, so the exponent
//    arguments and the normaliser's partial sums use paired fp32 instructions
//    (fma / add .f32x2, rounded as the scalar ones) and the tile max a
//    three-input max: the same results from fewer instructions.
// Every mbarrier wait is bounded; TMEM is freed on every path.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "../../include/ce_gb300.h"
#include "ce_rows.cuh"
#include "ce_tc.cuh"

namespace ce {

constexpr int kAttBQ = 128;  // query rows of a work item
constexpr int kAttBK = 128;  // keys of a tile
constexpr int kAttSoftmaxWarps = 8;  // two per TMEM lane quarter, 64 keys of a tile each
constexpr int kAttSoftmax = 32 * kAttSoftmaxWarps;
constexpr int kAttThreads = 64 + kAttSoftmax;
// TMEM columns: scores S0 [0, 128) and S1 [128, 256), the output accumulator
// O [256, 256 + D), the bf16 weights P0 [384, 448) and P1 [448, 512) (two to
// a 32-bit column)
constexpr uint32_t kAttTmemCols = 512;
constexpr uint32_t kAttTmemO = 256;
constexpr uint32_t kAttTmemP = 384;

struct AttnParams {
  const float* mask;   // [T, T] additive, or null
  float* lse;          // [BH, T], or null
  int T, BH;
  int causal;          // 1: keys after the query are masked (and their tiles skipped)
  float scale_log2;    // sm_scale * log2(e)
  float inv_scale;     // 1 / sm_scale: a mask entry in units of the unscaled score
  int q_tiles;         // ceil(T / 128)
  int n_pairs;         // ceil(q_tiles / 2)
  int n_units;         // work units: BH * n_pairs (causal) or BH * q_tiles
  unsigned int* err;
  unsigned int wait_hint_ns;
};

constexpr int kAttKStages = 3;  // K ring depth: scores run two tiles ahead
template <int D>
struct AttnSmem {
  static constexpr int kQ = kAttBQ * D * 2;  // Q: D / 64 K-major blocks of 128 rows x 128 B
  static constexpr int kK = kAttBK * D * 2;  // K: the same layout
  static constexpr int kV = kAttBK * D * 2;  // V: D / 64 MN-major blocks of 128 keys x 128 B
  // output staging: 32 rows x 128 B a warp, in the item's own Q buffer when it
  // is large enough (its score MMAs have all run by then), else a region of its own
  static constexpr int kStageNeed = kAttSoftmaxWarps * 4096;
  static constexpr bool kStageInQ = kQ >= kStageNeed;
  static constexpr int kStage = kStageInQ ? 0 : kStageNeed;
  static constexpr int kTotal = 2 * kQ + kAttKStages * kK + 2 * kV + kStage + 1024;  // + slack
};

// The reference max of a row moves only when a tile's max exceeds it by more
// than this (log2 units): until then the weights 2^(y - ref) stay below 2^8,
// exact enough in fp32 and bf16, and the accumulator is not rescaled.
constexpr float kRescaleLog2 = 8.f;

// OUT16: the output is rounded to bf16 (else fp32)
template <int D, bool OUT16>
__global__ void __launch_bounds__(kAttThreads, 1)
    attention_fwd_kernel(const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_o, const AttnParams p) {
  griddep_wait();  // the previous kernel on the stream has completed (dependent launch)
  using L = AttnSmem<D>;
  extern __shared__ unsigned char att_smem[];
  __shared__ __align__(8) unsigned long long q_full[2], q_empty[2], o_free;
  __shared__ __align__(8) unsigned long long k_full[kAttKStages], k_empty[kAttKStages];
  __shared__ __align__(8) unsigned long long v_full[2], v_empty[2];
  __shared__ __align__(8) unsigned long long s_full[2], s_free[2];
  __shared__ __align__(8) unsigned long long p_full[2], pv_done[2];
  __shared__ uint32_t tmem_slot;
  __shared__ float red[2][kAttBQ];  // [key half][row]: a row's two partial maxima or normalisers

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t base = (smem_u32(att_smem) + 1023u) & ~1023u;  // swizzle atoms need 1024 B
  const uint32_t sq0 = base;                      // two Q buffers (items alternate)
  const uint32_t sk0 = sq0 + 2 * L::kQ;           // three K stages
  const uint32_t sv0 = sk0 + kAttKStages * L::kK; // two V stages
  const uint32_t so0 = sv0 + 2 * L::kV;           // output staging (when not in Q)
  bool failed = false;
  const unsigned int hint = p.wait_hint_ns;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&o_free), kAttSoftmax);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&q_full[s]), 1);
      // the score MMAs' commit and, when the output is staged in the Q buffer,
      // each softmax warp once its stores have read it
      mbar_init(smem_u32(&q_empty[s]), 1 + (L::kStageInQ ? kAttSoftmaxWarps : 0));
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&s_free[s]), kAttSoftmax);
      mbar_init(smem_u32(&p_full[s]), kAttSoftmax);
      mbar_init(smem_u32(&pv_done[s]), 1);
    }
    for (int s = 0; s < kAttKStages; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    fence_mbar_init_cluster();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_slot)),
                 "r"(kAttTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  // Work units, handed out round-robin to the persistent CTAs.  Neighbouring
  // units belong to the same head, so the CTAs running together share that
  // head's K and V through L2.  Without the causal mask a unit is one
  // (head, query tile) item.  With it, unit u of a head pairs query tile
  // q_tiles - 1 - u (u + 1 key tiles from the end) with query tile u, so
  // every unit costs q_tiles + 1 key tiles and the grid ends evenly.
  auto items_in = [&](int u) {
    if (!p.causal) return 1;
    const int pr = u % p.n_pairs;
    return (p.q_tiles - 1 - pr != pr) ? 2 : 1;
  };
  auto item_of = [&](int u, int sub, int& bh, int& qt) {
    if (!p.causal) {
      bh = u / p.q_tiles;
      qt = u % p.q_tiles;
      return;
    }
    bh = u / p.n_pairs;
    const int pr = u % p.n_pairs;
    qt = sub == 0 ? p.q_tiles - 1 - pr : pr;
  };
  auto tiles_of = [&](int qt) {
    const int kv_end = p.causal ? min(p.T, (qt + 1) * kAttBQ) : p.T;
    return (kv_end + kAttBK - 1) / kAttBK;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      // K tile g is issued before V tile g - 1: S = Q K^T runs ahead of O += P V,
      // so each K stage is refilled as soon as its score MMA has read it
      long long g = 0;  // key tiles loaded, over all items
      int it = 0;
      int v_bh = -1, v_j = 0;  // the V tile still to load (tile g - 1)
      auto load_v = [&](long long t, int bh, int j) {
        const int st = static_cast<int>(t & 1);
        if (t >= 2)
          mbar_wait<false>(smem_u32(&v_empty[st]), static_cast<uint32_t>(((t >> 1) - 1) & 1),
                           p.err, failed, WAIT_LIMIT_NS, hint);
        const uint32_t fb = smem_u32(&v_full[st]);
        mbar_arrive_expect_tx(fb, L::kV);
        for (int db = 0; db < D / 64; ++db)
          for (int kh = 0; kh < 2; ++kh)
            tma_load_3d(sv0 + st * L::kV + db * 16384 + kh * 8192, &map_v, 64 * db,
                        j * kAttBK + 64 * kh, bh, fb);
      };
      for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
        for (int sub = 0; sub < items_in(u); ++sub, ++it) {
          int bh, qt;
          item_of(u, sub, bh, qt);
          const int n = tiles_of(qt);
          // Q buffer it % 2: the score MMAs of item it - 2 have read it (and the
          // stores of that item's output, staged there, have read it)
          const int qb = it & 1;
          if (it >= 2)
            mbar_wait<false>(smem_u32(&q_empty[qb]), static_cast<uint32_t>(((it >> 1) - 1) & 1),
                             p.err, failed, WAIT_LIMIT_NS, hint);
          mbar_arrive_expect_tx(smem_u32(&q_full[qb]), L::kQ);
          for (int kb = 0; kb < D / 64; ++kb)
            tma_load_3d(sq0 + qb * L::kQ + kb * 16384, &map_q, 64 * kb, qt * kAttBQ, bh,
                        smem_u32(&q_full[qb]));
          for (int j = 0; j < n; ++j, ++g) {
            const int st = static_cast<int>(g % kAttKStages);
            if (g >= kAttKStages)
              mbar_wait<false>(smem_u32(&k_empty[st]),
                               static_cast<uint32_t>((g / kAttKStages - 1) & 1), p.err, failed,
                               WAIT_LIMIT_NS, hint);
            const uint32_t fb = smem_u32(&k_full[st]);
            mbar_arrive_expect_tx(fb, L::kK);
            for (int kb = 0; kb < D / 64; ++kb)
              tma_load_3d(sk0 + st * L::kK + kb * 16384, &map_k, 64 * kb, j * kAttBK, bh, fb);
            if (v_bh >= 0) load_v(g - 1, v_bh, v_j);
            v_bh = bh;
            v_j = j;
          }
          // the item's last V now, not after the next item's Q: that Q buffer
          // may still hold an output being stored, and a one-tile item's P V
          // would wait for this V behind it
          load_v(g - 1, bh, n - 1);
          v_bh = -1;
        }
      }
      // drain: no copy into this CTA's shared memory is in flight when it exits
      // (the MMA thread has waited on these phases already unless a wait failed)
      bool drain_failed = false;
      for (int t = it - 2 < 0 ? 0 : it - 2; t < it; ++t)
        mbar_wait<false>(smem_u32(&q_full[t & 1]), static_cast<uint32_t>((t >> 1) & 1), p.err,
                         drain_failed, WAIT_LIMIT_NS, hint);
      for (long long t = g - kAttKStages < 0 ? 0 : g - kAttKStages; t < g; ++t)
        mbar_wait<false>(smem_u32(&k_full[t % kAttKStages]),
                         static_cast<uint32_t>((t / kAttKStages) & 1), p.err, drain_failed,
                         WAIT_LIMIT_NS, hint);
      for (long long t = g - 2 < 0 ? 0 : g - 2; t < g; ++t)
        mbar_wait<false>(smem_u32(&v_full[t & 1]), static_cast<uint32_t>((t >> 1) & 1), p.err,
                         drain_failed, WAIT_LIMIT_NS, hint);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      // S = Q K^T: M = 128 queries, N = 128 keys, both operands K-major (K = D)
      constexpr uint32_t idesc_s = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) |
                                   ((128u >> 4) << 24);
      // O += P V: M = 128 queries, N = D, A = P in TMEM (K = keys), B = V MN-major
      constexpr uint32_t idesc_o = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                                   ((static_cast<uint32_t>(D) >> 3) << 17) | ((128u >> 4) << 24);
      long long g = 0;   // score tiles issued, over all items
      long long gp = 0;  // P V tiles issued, over all items
      int it = 0;
      uint32_t sq = sq0;  // this item's Q buffer
      // shared-memory descriptors built once: a buffer's descriptor advances by
      // (bytes >> 4) in its start-address field (the buffers sit below 256 KB
      // on 16-byte boundaries, so the field never carries)
      const uint64_t dk = smem_desc_sw128(sk0);
      const uint64_t dv = smem_desc_sw128_mn(sv0, 16384);
      // S_gs into score buffer gs % 2 from K stage gs % 3, once the softmax holds
      // the buffer's previous scores (tile gs - 2) in registers
      auto issue_s = [&](long long gs) {
        const int st = static_cast<int>(gs & 1);
        const int ks = static_cast<int>(gs % kAttKStages);
        mbar_wait_fast(smem_u32(&k_full[ks]), static_cast<uint32_t>((gs / kAttKStages) & 1),
                         p.err, failed, WAIT_LIMIT_NS, hint);
        if (gs >= 2)
          mbar_wait_fast(smem_u32(&s_free[st]), static_cast<uint32_t>(((gs >> 1) - 1) & 1),
                           p.err, failed, WAIT_LIMIT_NS, hint);
        tc_fence_after();
        const uint64_t da = smem_desc_sw128(sq);
        const uint64_t db = dk + static_cast<uint64_t>(ks * (L::kK >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          umma_bf16(tmem + st * 128, da + off, db + off, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&s_full[st]));
        umma_commit(smem_u32(&k_empty[ks]));
      };
      for (int u = blockIdx.x; u < p.n_units; u += gridDim.x)
      for (int sub = 0; sub < items_in(u); ++sub, ++it) {
        int bh, qt;
        item_of(u, sub, bh, qt);
        const int n = tiles_of(qt);
        const int qb = it & 1;
        sq = sq0 + qb * L::kQ;
        mbar_wait_fast(smem_u32(&q_full[qb]), static_cast<uint32_t>((it >> 1) & 1), p.err,
                         failed, WAIT_LIMIT_NS, hint);
        tc_fence_after();
        // scores run two tiles ahead of P V: S_{j+2} is issued as soon as the
        // softmax has read S_j, before P V of tile j
        issue_s(g++);
        if (n > 1) issue_s(g++);
        if (n <= 2) umma_commit(smem_u32(&q_empty[qb]));  // every MMA reading Q is issued
        for (int j = 0; j < n; ++j) {
          if (j + 2 < n) {
            issue_s(g++);
            if (j + 3 == n) umma_commit(smem_u32(&q_empty[qb]));
          }
          // the previous item's output has been read out of TMEM
          if (j == 0 && it > 0)
            mbar_wait_fast(smem_u32(&o_free), static_cast<uint32_t>((it - 1) & 1), p.err, failed,
                             WAIT_LIMIT_NS, hint);
          const int pb = static_cast<int>(gp & 1);  // P buffer and V stage of this tile
          mbar_wait_fast(smem_u32(&p_full[pb]), static_cast<uint32_t>((gp >> 1) & 1), p.err,
                           failed, WAIT_LIMIT_NS, hint);
          mbar_wait_fast(smem_u32(&v_full[pb]), static_cast<uint32_t>((gp >> 1) & 1), p.err,
                           failed, WAIT_LIMIT_NS, hint);
          tc_fence_after();
          const uint64_t dbv = dv + static_cast<uint64_t>(pb * (L::kV >> 4));
          const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < kAttBK / 16; ++kk) {
            // P: 16 keys = 8 columns; V: 64-wide D blocks of 128 keys x 128 B
            // 16 KB apart, 16 keys = 2 KB
            umma_bf16_ts(tmem + kAttTmemO, tmem + kAttTmemP + 64 * pb + 8 * kk,
                         dbv + static_cast<uint64_t>(kk * (2048 >> 4)), idesc_o,
                         kk > 0 ? 1u : acc0);
          }
          umma_commit(smem_u32(&pv_done[pb]));
          umma_commit(smem_u32(&v_empty[pb]));
          ++gp;
        }
      }
      // drain: every MMA has finished before TMEM is released
      bool drain_failed = false;
      if (gp > 0)
        mbar_wait_fast(smem_u32(&pv_done[(gp - 1) & 1]), static_cast<uint32_t>(((gp - 1) >> 1) & 1),
                         p.err, drain_failed, WAIT_LIMIT_NS, hint);
    }
  } else {
    // ------- softmax warps 2..9: one query row and 64 keys of a tile per thread -------
    const int q = warp & 3;           // the TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;    // which 64 keys of each tile (and half of O's columns)
    const int r = 32 * q + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t eoff = (warp - 2) * 4096;  // this warp's output staging block
    const float c = p.scale_log2;                   // > 0: the max of s * c is c * max(s)
    constexpr int kOC = D / 64;                     // output chunks of 32 columns per thread
    // wait until P V of global tile t has finished
    auto wait_pv = [&](long long t) {
      mbar_wait<false>(smem_u32(&pv_done[t & 1]), static_cast<uint32_t>((t >> 1) & 1), p.err,
                       failed, WAIT_LIMIT_NS, hint);
    };
    // the two threads of a row swap a value through red[][r] with one meeting
    // (a named barrier per lane quarter) after the writes.  Each thread writes
    // the slot it read at the previous swap, whose value the partner wrote for
    // it alone, so no write can overtake the partner's pending read: that read
    // is of the other slot
    int par = 0;
    auto swap = [&](float v) {
      red[h ^ par][r] = v;
      group_sync(1 + q, 64);
      const float w = red[h ^ par ^ 1][r];
      par ^= 1;
      return w;
    };
    long long g = 0;  // score tiles consumed, over all items
    int it = 0;
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x)
    for (int sub = 0; sub < items_in(u); ++sub, ++it) {
      int bh, qt;
      item_of(u, sub, bh, qt);
      const int n = tiles_of(qt);
      const int row = qt * kAttBQ + r;
      const bool row_ok = row < p.T;
      const float* mrow = (p.mask != nullptr && row_ok) ? p.mask + static_cast<long long>(row) * p.T
                                                        : nullptr;
      float m_ref = -INFINITY;  // reference max of O and l (log2 units), the same in both threads
      float l = 0.f;            // this thread's share of the normaliser, relative to m_ref
      const uint32_t ebuf = (L::kStageInQ ? sq0 + (it & 1) * L::kQ : so0) + eoff;
      for (int j = 0; j < n; ++j, ++g) {
        const int st = static_cast<int>(g & 1);
        mbar_wait<false>(smem_u32(&s_full[st]), static_cast<uint32_t>((g >> 1) & 1), p.err,
                         failed, WAIT_LIMIT_NS, hint);
        tc_fence_after();
        uint32_t sr[64];
        const uint32_t ts = tmem + st * 128 + 64 * h + lane_off;
        tmem_ld32_nowait(ts, sr);
        tmem_ld32_nowait(ts + 32, sr + 32);
        tmem_wait_ld<64>(sr);
        // the scores are in registers: the buffer may take the next tile's scores
        tc_fence_before();
        mbar_arrive(smem_u32(&s_free[st]));
        if (L::kStageInQ && j == 0 && it > 0) {
          // the previous item's output stores have read its Q buffer: release it
          if (lane == 0) {
            bulk_wait_read<0>();
            mbar_arrive(smem_u32(&q_empty[(it - 1) & 1]));
          }
          __syncwarp();
        }
        float* x = reinterpret_cast<float*>(sr);
        const int kv0 = j * kAttBK + 64 * h;  // this thread's first key
        // one decision for the whole CTA: does any key of this tile need a mask?
        const bool masked = p.mask != nullptr || j * kAttBK + kAttBK > p.T ||
                            (p.causal && j * kAttBK + kAttBK - 1 > qt * kAttBQ);
        float mx[8];
        if (!masked) {
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = x[i];
#pragma unroll
          for (int i = 8; i < 64; i += 16)  // two more scores per partial max and instruction
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mx[k] = (i + 8 < 64) ? fmax3(mx[k], x[i + k], x[i + 8 + k]) : fmaxf(mx[k], x[i + k]);
        } else {
          // keys kv0 + i with i > lim are hidden (past T, or after the query).
          // Two loops, with and without the additive mask: a test of the mask
          // pointer inside the unrolled loop made every causal diagonal tile
          // about twice as slow as a clear one.
          const int lim = (p.causal ? min(row, p.T - 1) : p.T - 1) - kv0;
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
          if (mrow != nullptr) {
            // the additive mask joins the unscaled score as mask / sm_scale, so
            // both paths share one exponent, and a zero entry changes no bit
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              const float y = fmaf(__ldg(mrow + min(kv0 + i, p.T - 1)), p.inv_scale, x[i]);
              x[i] = (i > lim) ? -INFINITY : y;
              mx[i & 7] = fmaxf(mx[i & 7], x[i]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              x[i] = (i > lim) ? -INFINITY : x[i];
              mx[i & 7] = fmaxf(mx[i & 7], x[i]);
            }
          }
        }
        const float pm = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                               fmaxf(mx[6], mx[7]));
        const float mt = c * fmaxf(pm, swap(pm));  // the row's tile max (log2 units)
        if (j == 0) {
          m_ref = mt;  // this tile's P V overwrites O
        } else if (__any_sync(0xffffffffu, mt > m_ref + kRescaleLog2)) {
          // move the reference: O and l are rescaled by alpha = 2^(old - new),
          // after the previous P V has finished and before this tile's is issued
          // (the partner warp takes the same decision: it sees the same maxima)
          const float m_new = fmaxf(m_ref, mt);
          const float alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
          wait_pv(g - 1);
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < kOC; ++cc) {
            const uint32_t to = tmem + kAttTmemO + 32 * (kOC * h + cc) + lane_off;
            float o[32];
            tmem_ld32(to, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(to, o);
          }
          l *= alpha;
          m_ref = m_new;
        }
        const float ref = (m_ref == -INFINITY) ? 0.f : m_ref;
        float2 sm2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sm2[i] = make_float2(0.f, 0.f);
        const float2 c2 = make_float2(c, c), nr2 = make_float2(-ref, -ref);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 y = ffma2(make_float2(x[i], x[i + 1]), c2, nr2);
          x[i] = ex2(y.x);
          x[i + 1] = ex2(y.y);
          sm2[(i & 7) >> 1] = fadd2(sm2[(i & 7) >> 1], make_float2(x[i], x[i + 1]));
        }
        l += ((sm2[0].x + sm2[0].y) + (sm2[1].x + sm2[1].y)) +
             ((sm2[2].x + sm2[2].y) + (sm2[3].x + sm2[3].y));
        // P, rounded to bf16, two keys to a column (the lower key in the low
        // half), into TMEM buffer g % 2 -- free once P V of tile g - 2 has run
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
          pk[i] = *reinterpret_cast<uint32_t*>(&hv);
        }
        if (g >= 2) wait_pv(g - 2);
        tc_fence_after();
        tmem_st32_nowait(tmem + kAttTmemP + 64 * st + 32 * h + lane_off, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&p_full[st]));
      }
      // ---- the item's output: O / l through shared memory and TMA stores ----
      const float lt = l + swap(l);
      wait_pv(g - 1);
      tc_fence_after();
      if (h == 0 && p.lse != nullptr && row_ok) {
        const float mref = (m_ref == -INFINITY) ? 0.f : m_ref;
        p.lse[static_cast<long long>(bh) * p.T + row] = (mref + lg2(lt)) * 0.6931471805599453f;
      }
      const float inv_l = 1.f / lt;
      if constexpr (OUT16) {
        // this thread's half of the row, rounded to bf16: D bytes, one staging
        // row (128-byte rows with the 128-byte swizzle for D = 128, plain
        // 64-byte rows for D = 64) and one TMA store per warp
        uint32_t pk[D / 4];
#pragma unroll
        for (int cc = 0; cc < kOC; ++cc) {
          float o[32];
          tmem_ld32(tmem + kAttTmemO + 32 * (kOC * h + cc) + lane_off, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 hv = __floats2bfloat162_rn(o[2 * i] * inv_l, o[2 * i + 1] * inv_l);
            pk[16 * cc + i] = *reinterpret_cast<uint32_t*>(&hv);
          }
        }
        // the staging block: the store issued before has read it
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          const uint32_t a = (D == 128) ? ebuf + lane * 128 + 16 * (jj ^ (lane & 7))
                                        : ebuf + lane * 64 + 16 * jj;
          sts128(a, make_uint4(pk[4 * jj], pk[4 * jj + 1], pk[4 * jj + 2], pk[4 * jj + 3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && qt * kAttBQ + 32 * q < p.T) {  // blocks wholly past T are not stored
          tma_store_3d(&map_o, ebuf, (D / 2) * h, qt * kAttBQ + 32 * q, bh);
          bulk_commit();
        }
      } else {
#pragma unroll 1
        for (int cc = 0; cc < kOC; ++cc) {
          const int col = 32 * (kOC * h + cc);
          float o[32];
          tmem_ld32(tmem + kAttTmemO + col + lane_off, o);
          // the staging block: the store issued before has read it
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(
                             ebuf + lane * 128 + 16 * (jj ^ (lane & 7))),
                         "f"(o[4 * jj] * inv_l), "f"(o[4 * jj + 1] * inv_l),
                         "f"(o[4 * jj + 2] * inv_l), "f"(o[4 * jj + 3] * inv_l)
                         : "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && qt * kAttBQ + 32 * q < p.T) {  // blocks wholly past T are not stored
            tma_store_3d(&map_o, ebuf, col, qt * kAttBQ + 32 * q, bh);
            bulk_commit();
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&o_free));
    }
    // no CTA exits while a TMA store still reads its shared memory
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kAttTmemCols)
                 : "memory");
  }
}

// --- host side ---------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 att_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 3-D map over [BH, T, D] (D contiguous) with a box of box_d x box_t x 1
static bool att_map(CUtensorMap* map, CUtensorMapDataType type, int esize, const void* base,
                    int BH, int T, int D, int box_d, int box_t,
                    CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = att_encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * esize,
                           static_cast<cuuint64_t>(T) * D * esize};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_d), static_cast<cuuint32_t>(box_t), 1u};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, type, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool OUT16>
static ce_status attention_launch(const void* Q, const void* K, const void* V, const float* mask,
                                  int causal, int BH, int T, float sm_scale, void* O, float* lse,
                                  cudaStream_t stream, unsigned int* err, int sm_count,
                                  unsigned int wait_hint_ns) {
  CUtensorMap mq, mk, mv, mo;
  if (!att_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, Q, BH, T, D, 64, kAttBQ) ||
      !att_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, BH, T, D, 64, kAttBK) ||
      !att_map(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, V, BH, T, D, 64, 64) ||
      !(OUT16 ? att_map(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, O, BH, T, D, D / 2, 32,
                        D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE)
              : att_map(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, O, BH, T, D, 32, 32)))
    return CE_ERR_CUDA;
  AttnParams p;
  p.mask = mask;
  p.lse = lse;
  p.T = T;
  p.BH = BH;
  p.causal = causal;
  p.scale_log2 = sm_scale * kLog2e;
  p.inv_scale = 1.f / sm_scale;
  p.q_tiles = (T + kAttBQ - 1) / kAttBQ;
  p.n_pairs = (p.q_tiles + 1) / 2;
  p.n_units = BH * (causal ? p.n_pairs : p.q_tiles);
  p.err = err;
  p.wait_hint_ns = wait_hint_ns;
  if (BH == 0 || T == 0) return CE_OK;
  // 512 TMEM columns per CTA: the shared-memory request keeps one CTA per SM,
  // so no CTA ever waits in tcgen05.alloc for a neighbour to finish
  const int smem = AttnSmem<D>::kTotal > (128 << 10) ? AttnSmem<D>::kTotal : (128 << 10);
  if (cudaFuncSetAttribute(attention_fwd_kernel<D, OUT16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return CE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attention_fwd_kernel<D, OUT16>, kAttThreads,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    return CE_ERR_CUDA;
  if (per_sm != 1) return CE_ERR_UNSUPPORTED;
  long long grid = sm_count;
  if (grid > p.n_units) grid = p.n_units;
  // launched as programmatically dependent, like the row kernels: the next
  // call's CTAs take SMs as this call's exit, and wait before touching memory
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kAttThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attention_fwd_kernel<D, OUT16>, mq, mk, mv, mo, p) == cudaSuccess
             ? CE_OK
             : CE_ERR_CUDA;
}

ce_status attention_forward(const void* Q, const void* K, const void* V, const float* mask,
                            int causal, int BH, int T, int D, float sm_scale, void* O,
                            bool out_bf16, float* lse, cudaStream_t stream, unsigned int* err,
                            int sm_count, unsigned int wait_hint_ns) {
  if (D == 64)
    return out_bf16 ? attention_launch<64, true>(Q, K, V, mask, causal, BH, T, sm_scale, O, lse,
                                                 stream, err, sm_count, wait_hint_ns)
                    : attention_launch<64, false>(Q, K, V, mask, causal, BH, T, sm_scale, O, lse,
                                                  stream, err, sm_count, wait_hint_ns);
  if (D == 128)
    return out_bf16 ? attention_launch<128, true>(Q, K, V, mask, causal, BH, T, sm_scale, O, lse,
                                                  stream, err, sm_count, wait_hint_ns)
                    : attention_launch<128, false>(Q, K, V, mask, causal, BH, T, sm_scale, O,
                                                   lse, stream, err, sm_count, wait_hint_ns);
  return CE_ERR_UNSUPPORTED;
}

}  // namespace ce
