// Mixture-of-experts feed-forward of the target (see moe.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"
#include "layers.h"
#include "partials.cuh"

namespace df {

struct MoeBufs {
  int32_t* topk_id;     // [R][k] chosen experts, by probability (lower id first among equals)
  float* topk_w;        // [R][k] their renormalised weights
  int32_t* counts;      // [E] tokens routed to each expert
  int32_t* offsets;     // [E] first row of each expert in the expert-ordered buffers
  int32_t* pos_of;      // [R][k] expert-ordered row of (token, choice)
  int32_t* pair_token;  // [R k] token of each expert-ordered row
  df_bf16* xp;          // [R k][d] normed rows in expert order
  df_bf16* act;         // [R k][Fe] SwiGLU activations
  float* out;           // [R k][d] expert outputs
  int4* chunks;         // grouped GEMM work list: {expert, first row, rows, 0}
  int32_t* n_chunks;    // its length
};

// Bytes of each MoeBufs array for R rows, in the order above (each 256-byte aligned by the
// caller's carver); returns their sum.
constexpr int kMoeBufCount = 11;
size_t moe_buf_elems(int R, int k, int E, int d, int Fe, size_t* sizes /* [kMoeBufCount] */);

// router logits (partial tiles of x . W_router^T) -> topk_id, topk_w; NaN logits -> DF_ERR_NAN
int launch_moe_route(const PartialView& pv, int R, int E, int k, MoeBufs& m, int* status, cudaStream_t st);
// topk_id -> counts, offsets, pos_of, pair_token, the grouped GEMM's chunk list; then
// xp = x[pair_token]
int launch_moe_dispatch(const df_bf16* x, int R, int d, int E, int k, int Fe, MoeBufs& m, int* status,
                        cudaStream_t st);
// grouped expert products: act = SwiGLU(xp . W_gate_up[e]^T), out = act . W_down[e]^T
int launch_moe_experts(const df_bf16* w_gate_up, const df_bf16* w_down, int R, int d, int E, int k, int Fe,
                       MoeBufs& m, int* status, cudaStream_t st);
// h += sum_j w_j out[pos_of[t][j]];  then RMSNorm like res_norm (a.pv unused); P = R k rows of out
int launch_moe_combine(const MoeBufs& m, int k, int P, const ResNormArgs& a, int* status, cudaStream_t st);

}  // namespace df
