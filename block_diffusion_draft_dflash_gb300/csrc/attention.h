// Launch arguments of the tensor-core attention kernel (see attention.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"

namespace df {

constexpr int kAttnMaxSplits = 64;

// Rows: for sequence s, query node i (0 <= i < T), head h: q[s][i][h][128].
// Keys of sequence s: slots [0, dense_len[s] + dense_add) all visible, then a tail of
// tail_len slots of which row i sees slot j iff bit j of anc[s][i] is set.
struct AttnArgs {
  int b, T, Hq, Hkv, cap;
  const df_bf16* q;        // [b][T][Hq][128]
  const df_bf16* k_plane;  // [b][Hkv][cap][128]
  const df_bf16* v_plane;  // [b][Hkv][128][cap]
  const int32_t* dense_len;
  int dense_add;
  int tail_len;
  const uint32_t* anc;     // [b][T][ceil(tail_len/32)], or null: then the tail is causal
                           //   (row i sees tail slots 0 .. i) if `causal`, else not visible
  int causal;
  float scale;
  int nsplit;
  df_bf16* out;            // [b][T][Hq][128]
  float* o_part;           // [nsplit][b*T*Hq][128]  (nsplit > 1)
  float* ml_part;          // [nsplit][b*T*Hq][2]
  int* status;
};

struct AttnParams {
  int b, T, Hq, Hkv, cap;
  const int32_t* dense_len;
  int dense_add, tail_len;
  const uint32_t* anc;
  int W;
  int causal;
  float scale;
  int n_qtiles, nsplit;
  df_bf16* out;
  float* o_part;
  float* ml_part;
  int* status;
};

int launch_attention(const AttnArgs& a, cudaStream_t st);
int attn_num_splits(int b, int Hkv, int n_qtiles, int max_keys);
size_t attn_partial_bytes(int b, int T, int Hq, int nsplit);

}  // namespace df
