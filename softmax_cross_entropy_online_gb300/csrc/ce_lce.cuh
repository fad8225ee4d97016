// ce_lce.cuh -- the work the fused linear + cross-entropy does around its logits
// GEMM ("9 Triton kernels in 9 weeks", week eight: the lm_head projection
// chunked into the loss).  Shared by the GEMM (ce_gemm.cu), whose epilogue
// produces it, and the host schedule (ce_api.cu), which lays it out.
//
//  * Per chunk of rows, the logits GEMM's epilogue reduces each row over each
//    256-column tile of its accumulator to a pair (max, sum of exp(x - max)),
//    the online pair of the "POPCORNBENCH level-1 problem 95 transcript", and
//    keeps the row's target logit.
//  * Fused schedule: the epilogue also stores the chunk's fp32 logits.  While
//    the tensor cores run the next chunk, the same epilogue warps merge a
//    row's pairs ("This is associative") into its log-sum-exp and form the
//    row's bf16 gradient (softmax - onehot) * scale from the stored logits in
//    one pass, with the row loss: the work is spread over the idle time of the
//    epilogue warps (a tile's MMAs take about ten times its epilogue).  A
//    standalone kernel does the last chunk.
//  * Lean schedule: no logits are stored.  A warp per row merges the pairs
//    into the row's constants (its log-sum-exp, the target's gradient) and
//    loss; a second logits GEMM then recomputes each tile and its epilogue
//    writes the bf16 gradient straight from the accumulator.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ce {

constexpr int kLceTileCols = 256;  // the logits GEMM's tile width (its BN)
constexpr int kLceStats = 1;  // epilogue: the pairs and target logits (and the logits if store)
constexpr int kLceGrad = 2;   // epilogue: bf16 G = (softmax - onehot) * scale from the row constants

struct LceArgs {
  // this launch's chunk, written by the logits GEMM's epilogue
  float2* part;            // [rows][n_tiles]: (max, sum of exp(x - max)) per row and tile
  float* xt;               // [rows]: the row's target logit (written by the tile holding it)
  const int64_t* targets;  // [rows]: this chunk's targets
  int rows;                // rows of this chunk (the GEMM's M)
  int V;                   // columns of the logits (the GEMM's N)
  int n_tiles;             // ceil(V / 256)
  int mode;                // kLceStats or kLceGrad
  int store;               // kLceStats: also store the fp32 logits (the fused schedule)
  // lean schedule: a row's constants {lse log2e (high part), 2^-(its low part)
  // * scale, the target's gradient, the target or -1 as int bits}, written by
  // the merge pass with the row losses, read by the gradient pass
  float4* rowc;            // [rows]
  float* rl;               // [rows]: the row losses (merge pass)
  __nv_bfloat16* g16;      // [rows][ldv]: the gradient pass's output
  // the chunk whose gradient rows are formed (the previous one in the GEMM's
  // epilogue, the last one in the standalone kernel); bg_rows = 0: none
  const float* bg_logits;   // [bg_rows][ldl] fp32 logits
  const float2* bg_part;    // [bg_rows][n_tiles]
  const float* bg_xt;       // [bg_rows]
  const int64_t* bg_targets;  // [bg_rows]
  __nv_bfloat16* bg_g16;    // [bg_rows][ldv]: the bf16 gradient rows
  float* bg_rl;             // [bg_rows]: the row losses
  int bg_rows;
  long long ldl;            // row stride of the logits in elements (a multiple of 4)
  long long ldv;            // row stride of G in elements (a multiple of 8)
  float scale;              // the gradient scale (1 / M of the whole batch)
  unsigned int* err;        // the device error word
};

}  // namespace ce
