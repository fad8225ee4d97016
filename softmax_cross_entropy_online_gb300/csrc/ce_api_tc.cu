// ce_api_tc.cu -- the C ABI (include/ce_gb300.h) of the tensor-core paths:
// the tcgen05 GEMM, the fused linear + cross-entropy ("9 Triton kernels in 9
// weeks", week eight) and its two schedules, and the blockwise attention
// forward.  Argument checks, workspace layout and launches only; the kernels
// are in ce_gemm.cu and ce_attention.cu.
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/ce_gb300.h"
#include "ce_host.cuh"
#include "ce_lce.cuh"

namespace ce {
ce_status gemm_bf16(const void* A, long long lda, bool a_mn, const void* B, long long ldb,
                    bool b_mn, float* D, long long ldd, int M, int N, int K, float beta,
                    cudaStream_t stream, unsigned int* err, int sm_count,
                    unsigned int wait_hint_ns, const LceArgs* lce = nullptr);
ce_status launch_mean_rows(const float* rl, long long M, float* loss, cudaStream_t st);
ce_status launch_lce_grad_rows(const LceArgs& a, cudaStream_t st, int sm_count);
ce_status launch_lce_merge_rows(const LceArgs& a, cudaStream_t st, int sm_count);
ce_status attention_forward(const void* Q, const void* K, const void* V, const float* mask,
                            int causal, int BH, int T, int D, float sm_scale, void* O,
                            bool out_bf16, float* lse, cudaStream_t stream, unsigned int* err,
                            int sm_count, unsigned int wait_hint_ns);
}  // namespace ce

namespace {

using ce_host::DeviceInfo;
using ce_host::device_info;
using ce_host::wait_hint_ns;

// Workspace of the fused linear + cross-entropy for row chunks of `mc` rows.
//
// Fused schedule (a workspace of linear_ce_workspace_size_fused bytes): two
// fp32 logits buffers [mc, ldl] (ldl = V rounded up to a multiple of 4), two
// per-tile pair buffers [mc, n_tiles] and two target-logit buffers [mc], the
// bf16 gradient rows G [M, ldv] of every row (ldv = V rounded up to a multiple
// of 8) and the row losses [M].  The logits GEMM of chunk k writes buffer
// k % 2 and its epilogue reduces each row over each tile to a (max, sum) pair;
// its epilogue warps form chunk k - 1's gradient rows from buffer (k - 1) % 2
// meanwhile; a standalone pass forms the last chunk's.  dH and dW are then
// each one GEMM over all rows.
//
// Lean schedule (the default, and any workspace short of the fused one): no
// logits are stored.  Per chunk, one pair buffer [mc, n_tiles], one target-
// logit buffer [mc], the row constants [mc] and the chunk's bf16 G [mc, ldv],
// plus the row losses [M]: the logits GEMM keeps only the pairs, a merge pass
// turns them into the row constants and losses, a second logits GEMM writes G
// from its accumulators, and dH and dW are contracted before the next chunk
// (dW accumulated over the chunks).
//
// The GEMMs read W, G and h in their stored layouts (MN-major operands where K
// is not contiguous), so nothing is transposed.
struct LinearWs {
  size_t logits[2], part[2], xt[2], rowc, g16, rl, total;
};
size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
LinearWs linear_ws_layout(long long M, long long V, long long mc, bool fused) {
  const long long ldv = (V + 7) / 8 * 8;
  const long long ldl = (V + 3) / 4 * 4;
  const long long nt = (V + ce::kLceTileCols - 1) / ce::kLceTileCols;
  LinearWs w;
  std::memset(&w, 0, sizeof(w));
  size_t off = 0;
  const int nbuf = fused ? 2 : 1;
  if (fused) {
    for (int b = 0; b < 2; ++b) {
      w.logits[b] = off;
      off += round256(static_cast<size_t>(mc) * ldl * 4);
    }
  }
  for (int b = 0; b < nbuf; ++b) {
    w.part[b] = off;
    off += round256(static_cast<size_t>(mc) * nt * 8);
    w.xt[b] = off;
    off += round256(static_cast<size_t>(mc) * 4);
  }
  if (!fused) {
    w.rowc = off;
    off += round256(static_cast<size_t>(mc) * 16);
  }
  w.g16 = off;
  off += round256(static_cast<size_t>(fused ? M : mc) * ldv * 2);
  w.rl = off;
  off += round256(static_cast<size_t>(M) * 4);
  w.total = off;
  return w;
}
constexpr long long kLinearDefaultChunk = 2048;   // the fused schedule's row chunk
constexpr long long kLinearLeanMaxChunk = 2560;   // the lean schedule's largest row chunk

// The lean schedule's row chunk: among the multiples of 128 up to the largest
// that fits the workspace (and kLinearLeanMaxChunk), or all of M, the one whose
// per-chunk dH GEMMs (ceil(rows / 128) x ceil(H / 256) tiles each) take the
// fewest waves over the SMs, then the fewest chunks; 0 if none fits.
long long lean_chunk(long long M, long long H, long long V, int sms, size_t ws) {
  const long long tn = (H + 255) / 256;
  long long best = 0, best_waves = 0, best_chunks = 0;
  auto consider = [&](long long mc) {
    if (linear_ws_layout(M, V, mc, false).total > ws) return;
    long long waves = 0, chunks = 0;
    for (long long m0 = 0; m0 < M; m0 += mc, ++chunks) {
      const long long rows = (M - m0) < mc ? (M - m0) : mc;
      waves += ((rows + 127) / 128 * tn + sms - 1) / sms;
    }
    if (best == 0 || waves < best_waves || (waves == best_waves && chunks < best_chunks)) {
      best = mc;
      best_waves = waves;
      best_chunks = chunks;
    }
  };
  if (M <= kLinearLeanMaxChunk) consider(M);
  for (long long mc = 128; mc <= kLinearLeanMaxChunk && mc < M; mc += 128) consider(mc);
  return best;
}

}  // namespace

extern "C" {

ce_status ce_gemm_bf16(const void* A, int64_t lda, int a_mn, const void* B, int64_t ldb,
                       int b_mn, float* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                       float beta, void* stream) {
  if (M < 0 || N < 0 || K < 0 || (M > 0 && N > 0 && (A == nullptr || B == nullptr || D == nullptr)))
    return CE_ERR_INVALID_ARG;
  if ((a_mn != 0 && a_mn != 1) || (b_mn != 0 && b_mn != 1)) return CE_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return CE_ERR_UNSUPPORTED;
  if (beta != 0.f && beta != 1.f) return CE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(D) % 4) return CE_ERR_INVALID_ARG;
  DeviceInfo di;
  int dev = 0;
  ce_status st = device_info(di, &dev);
  if (st != CE_OK) return st;
  st = ce::gemm_bf16(A, lda, a_mn != 0, B, ldb, b_mn != 0, D, ldd, static_cast<int>(M),
                     static_cast<int>(N), static_cast<int>(K), beta,
                     static_cast<cudaStream_t>(stream), di.err, di.sm_count, wait_hint_ns());
  if (st == CE_OK) ce_host::count_launches(1);
  return st;
}

ce_status ce_attention_forward(const void* q, const void* k, const void* v, const float* mask,
                               int causal, int64_t B, int64_t NH, int64_t T, int64_t D,
                               float sm_scale, void* out, ce_dtype out_dtype, float* lse,
                               void* stream) {
  if (B < 0 || NH < 0 || T < 0 || (causal != 0 && causal != 1) || !std::isfinite(sm_scale) ||
      !(sm_scale > 0.f) || !std::isfinite(1.f / sm_scale))
    return CE_ERR_INVALID_ARG;
  if (out_dtype != CE_F32 && out_dtype != CE_F16 && out_dtype != CE_BF16) return CE_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return CE_ERR_UNSUPPORTED;
  if (out_dtype == CE_F16) return CE_ERR_UNSUPPORTED;
  int64_t BH = 0;
  if (__builtin_mul_overflow(B, NH, &BH)) return CE_ERR_UNSUPPORTED;
  if (BH == 0 || T == 0) return CE_OK;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return CE_ERR_INVALID_ARG;
  if (T > INT32_MAX || BH > INT32_MAX) return CE_ERR_UNSUPPORTED;
  // the kernel counts (head, 128-row query tile) items in 32-bit integers
  if (BH * ((T + 127) / 128) > INT32_MAX) return CE_ERR_UNSUPPORTED;
  auto mis = [](const void* ptr, uintptr_t a) { return reinterpret_cast<uintptr_t>(ptr) % a != 0; };
  if (mis(q, 16) || mis(k, 16) || mis(v, 16) || mis(out, 16) || (mask && mis(mask, 4)) ||
      (lse && mis(lse, 4)))
    return CE_ERR_INVALID_ARG;
  DeviceInfo di;
  int dev = 0;
  ce_status st = device_info(di, &dev);
  if (st != CE_OK) return st;
  st = ce::attention_forward(q, k, v, mask, causal, static_cast<int>(BH), static_cast<int>(T),
                             static_cast<int>(D), sm_scale, out, out_dtype == CE_BF16, lse,
                             static_cast<cudaStream_t>(stream), di.err, di.sm_count,
                             wait_hint_ns());
  if (st == CE_OK) ce_host::count_launches(1);
  return st;
}

ce_status ce_gemm_bf16_tn(const void* A, int64_t lda, const void* B, int64_t ldb, float* D,
                          int64_t ldd, int64_t M, int64_t N, int64_t K, float beta,
                          void* stream) {
  return ce_gemm_bf16(A, lda, 0, B, ldb, 0, D, ldd, M, N, K, beta, stream);
}

size_t linear_ce_workspace_size(int64_t M, int64_t H, int64_t V) {
  if (M < 0 || H < 1 || V < 1) return 0;
  const long long Mr = M > 0 ? M : 1;
  const long long mc = Mr < kLinearLeanMaxChunk ? Mr : kLinearLeanMaxChunk;
  return linear_ws_layout(Mr, V, mc, false).total;
}

size_t linear_ce_workspace_size_fused(int64_t M, int64_t H, int64_t V) {
  if (M < 0 || H < 1 || V < 1) return 0;
  const long long Mr = M > 0 ? M : 1;
  const long long mc = Mr < kLinearDefaultChunk ? Mr : kLinearDefaultChunk;
  return linear_ws_layout(Mr, V, mc, true).total;
}

ce_status linear_ce_fwd_bwd(const void* h, const void* W, const int64_t* targets, int64_t M,
                            int64_t H, int64_t V, float* loss, float* dH, float* dW,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 1 || H < 1 || V < 1) return CE_ERR_INVALID_ARG;
  if (!h || !W || !targets || !loss || !dH || !dW || !workspace) return CE_ERR_INVALID_ARG;
  if ((H % 8) || (reinterpret_cast<uintptr_t>(h) % 16) || (reinterpret_cast<uintptr_t>(W) % 16))
    return CE_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(workspace) % 256) || (reinterpret_cast<uintptr_t>(dH) % 16) ||
      (reinterpret_cast<uintptr_t>(dW) % 16) || (reinterpret_cast<uintptr_t>(targets) % 8) ||
      (reinterpret_cast<uintptr_t>(loss) % 4))
    return CE_ERR_INVALID_ARG;
  if (M > INT32_MAX || H > INT32_MAX || V > INT32_MAX) return CE_ERR_UNSUPPORTED;
  DeviceInfo di;
  int dev = 0;
  ce_status st = device_info(di, &dev);
  if (st != CE_OK) return st;
  // the schedule and row chunk: the largest chunk (a multiple of 128, or all of
  // M) whose workspace fits the fused schedule, else the lean schedule's chunk
  long long mc = M < kLinearDefaultChunk ? M : kLinearDefaultChunk;
  bool fused = true;
  while (linear_ws_layout(M, V, mc, true).total > workspace_bytes && mc > 128)
    mc = (mc / 2 + 127) / 128 * 128;
  if (linear_ws_layout(M, V, mc, true).total > workspace_bytes) {
    fused = false;
    mc = lean_chunk(M, H, V, di.sm_count, workspace_bytes);
    if (mc == 0) return CE_ERR_INVALID_ARG;
  }
  const LinearWs L = linear_ws_layout(M, V, mc, fused);
  const int nt = static_cast<int>((V + ce::kLceTileCols - 1) / ce::kLceTileCols);
  char* ws = static_cast<char*>(workspace);
  auto* g16 = reinterpret_cast<__nv_bfloat16*>(ws + L.g16);
  auto* rl = reinterpret_cast<float*>(ws + L.rl);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long ldv = (V + 7) / 8 * 8;
  const long long ldl = (V + 3) / 4 * 4;
  const unsigned hint = wait_hint_ns();
  const int sms = di.sm_count;
  const auto* Wb = static_cast<const __nv_bfloat16*>(W);
  const auto* hb = static_cast<const __nv_bfloat16*>(h);
  uint64_t launches = 0;
  const float scale = 1.0f / static_cast<float>(M);
  if (fused) {
    ce::LceArgs prev;  // the chunk whose gradient rows are still to be formed
    std::memset(&prev, 0, sizeof(prev));
    int k = 0;
    for (long long m0 = 0; m0 < M; m0 += mc, ++k) {
      const long long rows = (M - m0) < mc ? (M - m0) : mc;
      const int b = k & 1;
      auto* logits = reinterpret_cast<float*>(ws + L.logits[b]);
      ce::LceArgs a;
      std::memset(&a, 0, sizeof(a));
      a.part = reinterpret_cast<float2*>(ws + L.part[b]);
      a.xt = reinterpret_cast<float*>(ws + L.xt[b]);
      a.targets = targets + m0;
      a.rows = static_cast<int>(rows);
      a.V = static_cast<int>(V);
      a.n_tiles = nt;
      a.mode = ce::kLceStats;
      a.store = 1;
      a.ldl = ldl;
      a.ldv = ldv;
      a.scale = scale;
      a.err = di.err;
      // the previous chunk's gradient rows, formed by this GEMM's epilogue warps
      a.bg_logits = prev.bg_logits;
      a.bg_part = prev.bg_part;
      a.bg_xt = prev.bg_xt;
      a.bg_targets = prev.bg_targets;
      a.bg_g16 = prev.bg_g16;
      a.bg_rl = prev.bg_rl;
      a.bg_rows = prev.bg_rows;
      // logits[rows, V] = h_c W^T: both operands K-major (K = H)
      if ((st = ce::gemm_bf16(hb + m0 * H, H, false, Wb, H, false, logits, ldl,
                              static_cast<int>(rows), static_cast<int>(V), static_cast<int>(H),
                              0.f, s, di.err, sms, hint, &a)) != CE_OK)
        return st;
      ++launches;
      prev = a;
      prev.bg_logits = logits;
      prev.bg_part = a.part;
      prev.bg_xt = a.xt;
      prev.bg_targets = targets + m0;
      prev.bg_g16 = g16 + m0 * ldv;
      prev.bg_rl = rl + m0;
      prev.bg_rows = static_cast<int>(rows);
    }
    // the last chunk's gradient rows
    if ((st = ce::launch_lce_grad_rows(prev, s, sms)) != CE_OK) return st;
    ++launches;
    // dH = G W over every row at once (K = V), dW = G^T h written once (K = M)
    if ((st = ce::gemm_bf16(g16, ldv, false, Wb, H, true, dH, H, static_cast<int>(M),
                            static_cast<int>(H), static_cast<int>(V), 0.f, s, di.err, sms,
                            hint)) != CE_OK)
      return st;
    if ((st = ce::gemm_bf16(g16, ldv, true, hb, H, true, dW, H, static_cast<int>(V),
                            static_cast<int>(H), static_cast<int>(M), 0.f, s, di.err, sms,
                            hint)) != CE_OK)
      return st;
    launches += 2;
  } else {
    for (long long m0 = 0; m0 < M; m0 += mc) {
      const long long rows = (M - m0) < mc ? (M - m0) : mc;
      const auto* hc = hb + m0 * H;
      ce::LceArgs a;
      std::memset(&a, 0, sizeof(a));
      a.part = reinterpret_cast<float2*>(ws + L.part[0]);
      a.xt = reinterpret_cast<float*>(ws + L.xt[0]);
      a.targets = targets + m0;
      a.rows = static_cast<int>(rows);
      a.V = static_cast<int>(V);
      a.n_tiles = nt;
      a.mode = ce::kLceStats;
      a.store = 0;
      a.rowc = reinterpret_cast<float4*>(ws + L.rowc);
      a.rl = rl + m0;
      a.g16 = g16;
      a.ldv = ldv;
      a.scale = scale;
      a.err = di.err;
      // the logits' per-tile pairs and target logits (logits = h_c W^T, K = H), no logits
      if ((st = ce::gemm_bf16(hc, H, false, Wb, H, false, nullptr, 0, static_cast<int>(rows),
                              static_cast<int>(V), static_cast<int>(H), 0.f, s, di.err, sms, hint,
                              &a)) != CE_OK)
        return st;
      // each row's log-sum-exp constants and loss
      if ((st = ce::launch_lce_merge_rows(a, s, sms)) != CE_OK) return st;
      // the logits again, their epilogue writing G [rows, ldv] in bf16
      a.mode = ce::kLceGrad;
      if ((st = ce::gemm_bf16(hc, H, false, Wb, H, false, nullptr, 0, static_cast<int>(rows),
                              static_cast<int>(V), static_cast<int>(H), 0.f, s, di.err, sms, hint,
                              &a)) != CE_OK)
        return st;
      // dH[rows] = G W: A = G K-major (K = V), B = W read MN-major ([V, H], H contiguous)
      if ((st = ce::gemm_bf16(g16, ldv, false, Wb, H, true, dH + m0 * H, H,
                              static_cast<int>(rows), static_cast<int>(H), static_cast<int>(V),
                              0.f, s, di.err, sms, hint)) != CE_OK)
        return st;
      // dW (+)= G^T h_c: A = G read MN-major ([rows, V], V contiguous), B = h_c read
      // MN-major ([rows, H], H contiguous), K = rows
      if ((st = ce::gemm_bf16(g16, ldv, true, hc, H, true, dW, H, static_cast<int>(V),
                              static_cast<int>(H), static_cast<int>(rows), m0 == 0 ? 0.f : 1.f,
                              s, di.err, sms, hint)) != CE_OK)
        return st;
      launches += 5;
    }
  }
  if ((st = ce::launch_mean_rows(rl, M, loss, s)) != CE_OK) return st;
  ++launches;
  ce_host::count_launches(launches);
  return CE_OK;
}

}  // extern "C"
