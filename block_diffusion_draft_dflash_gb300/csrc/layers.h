// Launch arguments of the row-wise layer kernels (see layers.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"
#include "partials.cuh"

namespace df {

struct RmsNormArgs {
  const float* in;        // fp32 residual rows, row stride d
  const df_bf16* gain;    // [d]
  df_bf16* out;           // bf16 rows, row stride ld_out
  int ld_out;
  int rows, d;
  float eps;
  // output row o reads input row (o / group_out) * group_in + in_off + o % group_out
  int group_out, group_in, in_off;
  float* zero;            // optional buffer to clear (next GEMM's accumulator)
  long long zero_count;
  df_bf16* capture;       // optional: bf16 copy of the input rows (row stride ld_capture)
  int ld_capture;
};

// Consumer of a projection whose output is added to the residual stream (or, with
// h == null, taken as is), followed by RMSNorm:  h[t] += y[t];  out[o] = RMSNorm(h[t]) * gain.
struct ResNormArgs {
  PartialView pv;         // partial tiles of y (d features)
  float* h;               // residual rows [tokens][d], updated in place; null: no residual
  int d;
  const df_bf16* gain;
  float eps;
  df_bf16* out;           // bf16 rows, row stride ld_out
  int ld_out;
  int rows;               // output rows
  int group_out, group_in, in_off;  // out row o <- token (o / group_out) * group_in + in_off + o % group_out
  df_bf16* capture;       // optional bf16 copy of the new residual row, by token (row stride ld_capture)
  int ld_capture;
};

// Consumer of the gate/up projection: act[t][f] = silu(y[t][f]) * y[t][F + f] (bf16).
struct SwigluArgs {
  PartialView pv;
  int rows, F;
  df_bf16* act;
};

struct QkRopeArgs {
  const float* qkv;       // [rows][ld_qkv] fp32: q heads, k heads, v heads (hd 128); or
  PartialView pv;         //   pv.part != null: read the projection's partial tiles (tile = head)
  int ld_qkv;
  int b, TA, TB;          // rows: b*TA "query" rows, then b*TB context rows
  const int32_t* base;    // [b] first slot (cache length before the step)
  const int32_t* nnew;    // [b] context rows per sequence (TB rows) and offset of TA rows; may be null
  const int32_t* depth;   // [b][TA] position offsets of TA rows; null = row index
  int Hq, Hkv;
  const df_bf16* q_norm;
  const df_bf16* k_norm;
  float eps, theta;
  df_bf16* q_out;         // [b*TA][Hq][128]
  df_bf16* k_plane;       // [b][Hkv][cap][128]
  df_bf16* v_plane;       // [b][Hkv][128][cap]
  int cap;
  int* status;
  const float2* rope;     // [rows][64] (cos, sin) of pair i at the row's position (launch_rope_table)
  double inv_freq[64];    // theta^(-2i/128), filled by launch_rope_table
};

int launch_embed(const df_bf16* E, int d, int V, const int32_t* tok, const int32_t* bonus, int L, int mask_id,
                 float* h, int rows, int* status, cudaStream_t st);
int launch_rmsnorm(const RmsNormArgs& a, cudaStream_t st);
// Rotary table of every row of a forward (the positions are the same in every layer).
int launch_rope_table(const QkRopeArgs& a, float2* table, cudaStream_t st);
int launch_qk_rope(const QkRopeArgs& a, cudaStream_t st);
int launch_res_norm(const ResNormArgs& a, cudaStream_t st);
int launch_swiglu_partial(const SwigluArgs& a, cudaStream_t st);
// In-place log-softmax of rows whose (max, sum exp) partials came from the LM-head GEMM.
int launch_logsoftmax_from_stats(float* x, int rows, int V, const float* stats, int n_stats, float* lse,
                                 cudaStream_t st);
int launch_argmax_finalize(const unsigned long long* amax, int rows, int32_t* out, cudaStream_t st);
// Draw keys (draw_key() in common.cuh) of `rows` token rows, for the LM head's temperature
// draw.  Row t draws the token at absolute position pos_t of sequence s_t: given per row
// (row_seq, row_pos) when row_seq is non-NULL; otherwise the rows are b sequences of T tree
// (or chain) nodes, s_t = t / T, pos_t = cache_len[s_t] + (depth ? depth[t] : t % T) + 1.
int launch_draw_keys(int rows, uint64_t seed, const int32_t* row_seq, const int32_t* row_pos, int T,
                     const int32_t* cache_len, const int32_t* depth, uint32_t* keys, cudaStream_t st);

}  // namespace df
