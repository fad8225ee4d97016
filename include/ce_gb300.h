/*
 * ce_gb300.h -- C ABI of the GB300 (sm_103a) softmax cross-entropy library.
 *
 * What is computed.  For logits x [M, V] (row-major, contiguous, row i at
 * byte offset i*V*sizeof(dtype)) and integer targets t [M]:
 *
 *     m_i      = max_j x_ij
 *     lse_i    = m_i + log sum_j exp(x_ij - m_i)
 *     row_i    = lse_i - x_{i,t_i}
 *     loss     = (1/M) sum_i row_i      (mean)   or   sum_i row_i   (sum)
 *     g_ij     = (exp(x_ij - lse_i) - [j == t_i]) * scale
 *
 * with scale = 1/M for the mean and 1 for sum/none.  Sources: the per-row
 * definition "max, subtract, exp, sum, log" with mean reduction in the
 * "POPCORNBENCH level-1 problem 95 transcript" (cross-entropy CUDA kernel);
 * the loss_kernel output formula (log(sumexp) + max - target logit) in
 * "Cross Entropy Loss performance issue" (Triton issue #5509); the fused
 * forward+backward that writes the gradient over the logits buffer in
 * "9 Triton kernels in 9 weeks", week seven.
 *
 * Conventions shared by every entry point:
 *  - Every buffer pointer (logits, targets, loss, row_loss, lse, and the
 *    operands and outputs of the GEMM, linear+CE and attention calls) is a
 *    DEVICE pointer on the current CUDA device.  The caller owns all of them;
 *    the library never frees or keeps them.  The library does not look up
 *    where a pointer lives: a host pointer, or one into another device's
 *    memory, is the caller's error and faults the kernel (the Python binding
 *    refuses such tensors before calling).  `stream` is a cudaStream_t
 *    (NULL = legacy default stream); every call is asynchronous and
 *    stream-ordered.
 *  - logits must be aligned to the element size, targets to 8 bytes and
 *    the float outputs to 4 bytes.  Rows need not be 16-byte aligned.
 *  - Arithmetic is fp32 (16-bit inputs widen exactly); loss, row_loss and
 *    lse are fp32; gradients are rounded to the logits' dtype
 *    (round-to-nearest-even, subnormals kept).
 *  - The mean is deterministic: no floating-point atomics are used; for a
 *    given device and shape the same inputs give bit-identical outputs.
 *  - Errors detectable on the host return before anything is launched.  A
 *    target outside [0, V) does not stop the call: that row's loss is NaN,
 *    its gradient is softmax*scale (no one-hot term), and a device error
 *    word is set; ce_check_errors reports it.  Nothing traps.
 *  - The reducing calls (a mean or sum loss) use a small library-owned device
 *    buffer, one per (device, stream) pair: 256 + 8 * 8192 bytes (about
 *    64 KB), created by cudaMalloc on the first reducing call on that stream
 *    and kept until the process exits (the library never frees it).  A caller
 *    that reduces on many short-lived streams therefore holds 64 KB per
 *    stream it has used; reduce on a few long-lived streams, or use
 *    ce_fwd_bwd_inplace_noalloc.  Make the first reducing call on a stream
 *    outside CUDA graph capture.
 *  - Per device, the library looks up and keeps device addresses (its error
 *    word, its static scratch) and launch shapes on first use.  After
 *    cudaDeviceReset, or any other teardown of the device's primary context,
 *    those kept addresses are stale: do not call the library again in that
 *    process after a reset.
 */
#ifndef CE_GB300_H
#define CE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CE_OK = 0,
  CE_ERR_INVALID_ARG = 1,  /* bad size, null or misaligned pointer, bad enum */
  CE_ERR_UNSUPPORTED = 2,  /* V beyond ce_max_vocab(dtype), or a layout a kernel cannot take */
  CE_ERR_TARGET_RANGE = 3, /* (ce_check_errors) a target was outside [0, V) */
  CE_ERR_CUDA = 4,         /* a CUDA runtime call or a launch failed */
  CE_ERR_TIMEOUT = 5       /* (ce_check_errors) a bounded wait ran out */
} ce_status;

typedef enum { CE_F32 = 0, CE_F16 = 1, CE_BF16 = 2 } ce_dtype;

typedef enum { CE_RED_MEAN = 0, CE_RED_SUM = 1, CE_RED_NONE = 2 } ce_reduction;

/*
 * ce_forward -- loss forward: one streaming pass over the logits with an
 * online (max, sum-of-exp) per row, the target-logit gather, and the
 * reduction.  The online recurrence and its pairwise merge are the ones
 * the transcript derives ("online softmax algorithm", "This is
 * associative").
 *
 *   logits    [M, V] of `dtype`, read only.
 *   targets   [M] int64 class indices.
 *   M >= 0, V >= 1.
 *   reduction CE_RED_MEAN / CE_RED_SUM write *loss; CE_RED_NONE ignores it.
 *   loss      [1] fp32 or NULL (then no reduction is computed).
 *   row_loss  [M] fp32 or NULL.   lse [M] fp32 or NULL.
 *   M == 0: mean writes NaN, sum writes 0.
 */
ce_status ce_forward(const void* logits, const int64_t* targets, int64_t M, int64_t V,
                     ce_dtype dtype, ce_reduction reduction, float* loss, float* row_loss,
                     float* lse, void* stream);

/*
 * ce_fwd_bwd_inplace -- fused forward + backward ("9 Triton kernels in 9
 * weeks", week seven): computes everything ce_forward does and overwrites
 * the logits with g = (softmax - onehot) * scale, scale = 1/M (mean) or 1
 * (sum, none).  Each logit is read from HBM once and written once.
 *
 *   logits    [M, V] of `dtype`, read and overwritten with the gradient.
 *   Other arguments as in ce_forward.  row_loss and lse must not alias
 *   the logits.
 */
ce_status ce_fwd_bwd_inplace(void* logits, const int64_t* targets, int64_t M, int64_t V,
                             ce_dtype dtype, ce_reduction reduction, float* loss,
                             float* row_loss, float* lse, void* stream);

/*
 * ce_softmax_forward -- fused softmax, p = exp(x - lse) per row, in one read
 * and one write of HBM ("9 Triton kernels in 9 weeks", week one: the three
 * passes of a softmax fused into one).  Same row machinery as ce_forward.
 *
 *   logits [M, V] of `dtype`, read.  probs [M, V] of `dtype`: either the
 *   logits pointer itself (in place) or a buffer that does not overlap it and
 *   whose address differs from the logits' by a multiple of 16 bytes (else
 *   CE_ERR_UNSUPPORTED).  lse [M] fp32 or NULL.  No targets.
 */
ce_status ce_softmax_forward(const void* logits, void* probs, int64_t M, int64_t V,
                             ce_dtype dtype, float* lse, void* stream);

/*
 * ce_fwd_bwd_inplace_noalloc -- ce_fwd_bwd_inplace for callers that must not
 * allocate device memory.  (The source pages have no counterpart; this is a
 * deployment variant of the fused kernel.)
 *
 * Who needs it: a caller whose allocator owns the whole device memory budget
 * and forbids stray allocations, or one that cannot afford the implicit
 * device synchronisation a cudaMalloc/cudaFree may cause in a timed loop.
 * ce_fwd_bwd_inplace creates a small reduction buffer with cudaMalloc on the
 * first reducing call on each stream; this entry point never calls
 * cudaMalloc, cudaFree or any other allocating routine.
 *
 * Same arguments, results and errors as ce_fwd_bwd_inplace.  The reduction
 * scratch is a fixed array inside the library's device code (one fp64
 * partial sum per CTA, at most 1024 CTAs, about 8 KB), held by every device
 * that loads the library until the process exits.  A launch that would need
 * more than 1024 CTAs returns CE_ERR_UNSUPPORTED (no GB300 launch shape does).
 *
 *  - Set-up: the first call on each device (with that device current) looks
 *    up the array's device address once; make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array.  Each call clears its
 *    counter on `stream` before the launch, so a call never depends on the
 *    previous call's leftovers, but calls whose executions overlap on the GPU
 *    (different streams, no ordering between them) race and can produce a
 *    wrong loss.  Order them on one stream or with events.
 */
ce_status ce_fwd_bwd_inplace_noalloc(void* logits, const int64_t* targets, int64_t M, int64_t V,
                                     ce_dtype dtype, ce_reduction reduction, float* loss,
                                     float* row_loss, float* lse, void* stream);

/*
 * ce_backward_from_lse -- gradient only, from a stored per-row lse:
 * g = (exp(x - lse_i) - onehot) * scale written over the logits.  This is
 * the backward half of the fused kernel of "9 Triton kernels in 9 weeks",
 * week seven (the gradient of the mean loss, softmax minus the one-hot
 * target over M, written into the logits buffer), run from an lse saved by
 * the forward of "POPCORNBENCH level-1 problem 95 transcript"'s definition
 * (log_sum_exp per row).  Use it when the forward ran earlier (ce_forward
 * with lse != NULL); `scale` is the upstream gradient of each row loss (1/M
 * for a mean).  Each logit is read once and written once.
 *
 *   logits [M, V] read and overwritten; targets [M] int64; lse [M] fp32.
 */
ce_status ce_backward_from_lse(void* logits, const int64_t* targets, const float* lse,
                               int64_t M, int64_t V, ce_dtype dtype, float scale,
                               void* stream);

/*
 * linear_ce_fwd_bwd -- fused linear + cross-entropy ("9 Triton kernels in 9
 * weeks", week eight: the lm_head projection chunked into the loss to cut its
 * activation memory).  For hidden states h [M, H] and the lm_head weight
 * W [V, H], with logits = h W^T:
 *
 *     loss = mean_i CE(logits_i, t_i)
 *     dH   = G W          [M, H]      G = (softmax(logits) - onehot) / M
 *     dW   = G^T h        [V, H]
 *
 * Rows are processed in chunks; the schedule follows the workspace.
 *  * Lean schedule (linear_ce_workspace_size bytes, the default): the logits
 *    are never stored.  Per chunk, a tcgen05 logits GEMM reduces each row
 *    over each 256-column tile of its accumulator to a (max, sum of exp) pair
 *    and keeps the target logit; a pass merges each row's pairs into its
 *    log-sum-exp and loss; a second logits GEMM recomputes the tiles and its
 *    epilogue writes the chunk's bf16 G straight from the accumulator; then
 *    dH rows = G W and dW (+)= G^T h.  Four GEMMs' work, about 0.66 GB of
 *    workspace for M = 8192, V = 128256 (the unfused fp32 logits and their
 *    gradient would take 8.4 GB).
 *  * Fused schedule (linear_ce_workspace_size_fused bytes or more): each
 *    2048-row chunk's fp32 logits go to one of two chunk buffers (the [M, V]
 *    logits never exist at once) while the epilogue forms the same pairs; the
 *    next chunk's GEMM epilogue warps turn them into the previous chunk's bf16
 *    G rows and row losses from the stored logits; G is kept whole and dH and
 *    dW are each one GEMM over all rows.  Three GEMMs' work, about 4.2 GB.
 *    A workspace between the two takes the fused schedule with a smaller
 *    chunk while it fits (down to 128 rows), else the lean one.
 * The GEMMs read W, G and h in their stored layouts, with fp32 accumulation.
 *
 *   h        [M, H] bf16, row-major; W [V, H] bf16, row-major (device).
 *            H must be a multiple of 8; h and W 16-byte aligned.
 *   targets  [M] int64.   loss [1] fp32.   dH [M, H] fp32.   dW [V, H] fp32.
 *   workspace  device memory (256-byte aligned, owned by the caller) of
 *            workspace_bytes: at least the lean schedule's need for 128-row
 *            chunks (about 128 * (2 V + 8 V / 256 + 20) + 4 M bytes), else
 *            CE_ERR_INVALID_ARG.
 *   A target outside [0, V) gives that row a NaN loss (so the mean is NaN),
 *   drops its one-hot term and sets the device error word (ce_check_errors).
 *   G is rounded to bf16 before the two gradient GEMMs; logits, the loss
 *   and every accumulation are fp32.
 */
ce_status linear_ce_fwd_bwd(const void* h, const void* W, const int64_t* targets, int64_t M,
                            int64_t H, int64_t V, float* loss, float* dH, float* dW,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes of linear_ce_fwd_bwd's lean schedule at its largest row
 * chunk (2560, or M, rows): the chunk's bf16 G [rows, V rounded up to a
 * multiple of 8], its per-tile pairs, target logits and row constants, and the
 * fp32 row losses [M]; about 0.66 GB for M = 8192, V = 128256 (0 on bad
 * sizes). */
size_t linear_ce_workspace_size(int64_t M, int64_t H, int64_t V);

/* Workspace bytes of linear_ce_fwd_bwd's fused schedule at its row chunk of
 * 2048 (or M) rows: two fp32 logits chunks [2048, V rounded up to a multiple
 * of 4], their per-tile pairs and target logits, bf16 G [M, V rounded up to a
 * multiple of 8] and the fp32 row losses; about 4.2 GB for M = 8192,
 * V = 128256 (0 on bad sizes). */
size_t linear_ce_workspace_size_fused(int64_t M, int64_t H, int64_t V);

/*
 * ce_gemm_bf16 -- the tensor-core contraction under linear_ce_fwd_bwd, exposed
 * on its own: D[M, N] = sum_k A(m, k) B(n, k) (beta = 0) or D += ... (beta = 1)
 * in fp32, A and B bf16.  a_mn = 0: A is [M, lda] with K contiguous,
 * A(m, k) = A[m * lda + k]; a_mn = 1: A is stored transposed, [K, lda] with M
 * contiguous, A(m, k) = A[k * lda + m].  The same for B with N (b_mn).  Row
 * strides lda, ldb in elements, multiples of 8; A and B 16-byte aligned; D
 * fp32 with row stride ldd >= N.  A persistent tcgen05 kernel: TMA into shared
 * memory, MMAs into TMEM accumulators, an epilogue through shared memory and
 * TMA tensor stores (or tensor reduce-adds for beta = 1).  Errors: null
 * pointers, a_mn / b_mn outside {0, 1}, beta outside {0, 1} ->
 * CE_ERR_INVALID_ARG; bad strides or alignment -> CE_ERR_UNSUPPORTED.
 */
ce_status ce_gemm_bf16(const void* A, int64_t lda, int a_mn, const void* B, int64_t ldb,
                       int b_mn, float* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                       float beta, void* stream);

/*
 * ce_gemm_bf16_tn -- ce_gemm_bf16 with both operands K-major:
 * D[M, N] = A[M, K] B[N, K]^T (beta = 0) or D += A B^T (beta = 1).
 */
ce_status ce_gemm_bf16_tn(const void* A, int64_t lda, const void* B, int64_t ldb, float* D,
                          int64_t ldd, int64_t M, int64_t N, int64_t K, float beta,
                          void* stream);

/*
 * ce_attention_forward -- blockwise (flash-attention-2 style) attention
 * forward on the tensor cores: the workload of "How to optimize an existing
 * Triton Kernel to make it faster?" (Triton discussion #8261), whose forward
 * keeps a running row max and a running normaliser over blocks of keys, the
 * same online (max, sum) pair as the cross-entropy rows.  Per head:
 *
 *     S   = Q K^T * sm_scale + mask        (+ the causal mask if causal != 0)
 *     out = softmax_rows(S) V
 *     lse = log sum_j exp(S_ij)            (per query row)
 *
 *   q, k, v  [B, NH, T, D] bf16, contiguous, 16-byte aligned (device).
 *            D is 64 or 128.
 *   mask     [T, T] fp32 additive mask (row = query), or NULL.  -inf hides
 *            a key.  Combined with causal it is added before the causal mask.
 *   causal   1: key j is hidden from query i when j > i (and the key blocks
 *            wholly above the diagonal are skipped); 0: no causal mask.
 *   sm_scale the score scale (the page uses 1/sqrt(D)); positive, with a finite
 *            reciprocal (a mask entry enters as mask / sm_scale on the unscaled
 *            score, so finite entries must stay below 2^127 sm_scale in size).
 *   out      [B, NH, T, D] of out_dtype, 16-byte aligned (device, caller-owned).
 *   out_dtype CE_F32, or CE_BF16 (the page's output is allocated like q).
 *   lse      [B, NH, T] fp32 (device) or NULL.
 * Arithmetic: bf16 products with fp32 accumulation for Q K^T; the softmax in
 * fp32 (exponentials in base 2 of the score times log2(e)); P is rounded to
 * bf16 for P V, accumulated in fp32; out = O / l in fp32, rounded to nearest
 * even for CE_BF16.  A row whose every key is hidden gives NaN outputs and
 * lse = -inf (the definition's 0/0).
 * Errors: null pointers, B, NH or T < 0, causal outside {0, 1}, sm_scale not
 * positive with a finite reciprocal, out_dtype not a ce_dtype, misaligned
 * pointers -> CE_ERR_INVALID_ARG; D not 64 or 128, out_dtype CE_F16, or T,
 * B*NH or B*NH*ceil(T/128) above 2^31-1 -> CE_ERR_UNSUPPORTED.
 */
ce_status ce_attention_forward(const void* q, const void* k, const void* v, const float* mask,
                               int causal, int64_t B, int64_t NH, int64_t T, int64_t D,
                               float sm_scale, void* out, ce_dtype out_dtype, float* lse,
                               void* stream);

/*
 * ce_check_errors -- wait (at most timeout_ms) for `stream` to drain, then
 * read and clear the current device's error word.  Returns CE_OK,
 * CE_ERR_TARGET_RANGE (some target was outside [0, V)), CE_ERR_TIMEOUT (the
 * stream did not drain in time, or a kernel's bounded wait ran out), or
 * CE_ERR_CUDA.
 */
ce_status ce_check_errors(void* stream, int timeout_ms);

/* Human-readable name of a status. Never NULL. */
const char* ce_status_string(ce_status status);

/* Largest V the row kernels accept for `dtype` (0 for a bad dtype). */
int64_t ce_max_vocab(ce_dtype dtype);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t ce_launch_count(void);

/*
 * ce_selftest_wait_timeout -- test hook for the bounded-wait machinery:
 * launches one tiny kernel that waits on a barrier nothing will complete,
 * gives up after timeout_us microseconds and sets the device error word,
 * so that a following ce_check_errors returns CE_ERR_TIMEOUT.  It never
 * hangs the GPU.  1 <= timeout_us <= 1000000.
 */
ce_status ce_selftest_wait_timeout(void* stream, int timeout_us);

#ifdef __cplusplus
}
#endif

#endif /* CE_GB300_H */
