// Greedy acceptance and KV-cache compaction.
//
// Method: summary of "Accelerating Speculative Decoding with Block Diffusion Draft
// Trees" (bluediary8.tistory.com/1288), section "방법론 자세히 보기": the verifier follows
// the target's outputs down the tree, accepts the longest matching path and compacts the
// KV cache so that rejected branches disappear.
//
// accept_walk_kernel: one warp per sequence.  At each step the 32 lanes scan the tree
//   for the child of the current node whose token equals the target's choice there
//   (children of one node carry distinct tokens, so at most one matches).
// compact_kernel: one CTA per (layer, sequence, kv head) moves the accepted nodes' K rows
//   (and the matching V columns, V being stored transposed) from slot N + idx_j to slot
//   N + j.  A later destination can be an earlier source (idx_j' == j), so every CTA
//   loads all its sources into registers before it stores anything.
// gather_feat_kernel: copies the feature rows of the root and the accepted path into the
//   drafter's pending-context buffer.
#include "common.cuh"
#include "checked.cuh"
#include "trace.h"

namespace df {

constexpr int kMaxPath = 32;

struct AcceptScratch {   // per sequence, in the workspace
  int32_t n_old;         // cache length before this step
  int32_t a;             // accepted nodes (excluding the root)
  int32_t path[kMaxPath];
};

__global__ void __launch_bounds__(32) accept_walk_kernel(int n_tree, int max_new, const int32_t* __restrict__ choice,
                                                         const int32_t* __restrict__ tok,
                                                         const int32_t* __restrict__ parent, int32_t* cache_len,
                                                         int cap, int32_t* n_new, int32_t* acc_tok, int32_t* n_acc,
                                                         int32_t* new_bonus, int32_t* src_slot,
                                                         AcceptScratch* scratch, int* status) {
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.x, lane = threadIdx.x;
  const int32_t* ch = choice + (size_t)s * n_tree;
  const int32_t* tk = tok + (size_t)s * n_tree;
  const int32_t* pa = parent + (size_t)s * n_tree;
  __shared__ int32_t path[kMaxPath];
  int cur = 0, a = 0;
  while (a < kMaxPath) {
    const int want = ch[cur];
    int found = 0x7fffffff;
    for (int c = 1 + lane; c < n_tree; c += 32)
      if (pa[c] == cur && tk[c] == want) found = min(found, c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
    if (found == 0x7fffffff) break;
    if (lane == 0) path[a] = found;
    cur = found;
    ++a;
  }
  __syncwarp();
  const int32_t N = cache_len[s];
  if (a + 1 > max_new) {
    if (lane == 0) set_status(status, DF_ERR_CAPACITY, s);
    a = max_new - 1;
  }
  const int bonus = ch[cur];
  for (int j = lane; j < max_new; j += 32) {
    const int32_t t = j < a ? tk[path[j]] : (j == a ? bonus : -1);
    acc_tok[(size_t)s * max_new + j] = t;
    src_slot[(size_t)s * max_new + j] = j < a ? N + path[j] : -1;
  }
  for (int j = lane; j < a; j += 32) scratch[s].path[j] = path[j];
  if (lane == 0) {
    scratch[s].n_old = N;
    scratch[s].a = a;
    n_acc[s] = a;
    n_new[s] = a + 1;
    new_bonus[s] = bonus;
    cache_len[s] = min(N + 1 + a, cap);
  }
}

// grid: (n_layers * b * Hkv, 2): y = 0 moves K rows, y = 1 moves V columns.
__global__ void __launch_bounds__(256) compact_kernel(df_bf16* k_cache, df_bf16* v_cache, int b, int Hkv, int cap,
                                                      const AcceptScratch* __restrict__ scratch, int* status) {
  pdl_wait();
  pdl_trigger();
  constexpr int HD = 128;
  const int lhs = blockIdx.x;                 // ((layer * b) + s) * Hkv + h
  const int s = (lhs / Hkv) % b;
  const int a = scratch[s].a;
  if (a == 0) return;
  const int N = scratch[s].n_old;
  const size_t plane = (size_t)lhs * cap * HD;  // one (layer, s, head) plane, cap*HD elements
  const int tid = threadIdx.x;
  if (blockIdx.y == 0) {
    // K: rows of 128 bf16 = 16 x 16-byte chunks; a <= 31 rows -> <= 496 chunks.
    uint4* base = reinterpret_cast<uint4*>(k_cache + plane);
    uint4 buf[2];
    int dst[2];
    const int total = a * 16;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int c = tid + r * 256;
      dst[r] = -1;
      if (c < total) {
        const int j = c >> 4, w = c & 15;
        const int src_slot = N + scratch[s].path[j];
        if (DF_IN_BOUNDS(src_slot >= 0 && src_slot < cap && N + 1 + j < cap, status, 40)) {
          buf[r] = base[(size_t)src_slot * 16 + w];
          dst[r] = (N + 1 + j) * 16 + w;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (dst[r] >= 0) base[dst[r]] = buf[r];
  } else {
    // V^T: [hd][cap]; move column N + idx_j to column N + 1 + j for all 128 rows.
    df_bf16* base = v_cache + plane;
    const int total = a * HD;  // <= 31 * 128 = 3968 elements
    df_bf16 buf[16];
    int dst[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int c = tid + r * 256;
      dst[r] = -1;
      if (c < total) {
        const int row = c / a, j = c % a;
        const int src_slot = N + scratch[s].path[j];
        if (DF_IN_BOUNDS(src_slot >= 0 && src_slot < cap && N + 1 + j < cap, status, 41)) {
          buf[r] = base[(size_t)row * cap + src_slot];
          dst[r] = row * cap + N + 1 + j;
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 16; ++r)
      if (dst[r] >= 0) base[dst[r]] = buf[r];
  }
}

// grid: (b, max_new); copies feature row (root or path node) j of sequence s.
__global__ void __launch_bounds__(256) gather_feat_kernel(const df_bf16* __restrict__ tree_feat, int n_tree,
                                                          int feat_dim, df_bf16* __restrict__ new_feat, int max_new,
                                                          const AcceptScratch* __restrict__ scratch, int* status) {
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.x, j = blockIdx.y;
  if (j > scratch[s].a) return;
  const int node = j == 0 ? 0 : scratch[s].path[j - 1];
  if (!DF_IN_BOUNDS(node >= 0 && node < n_tree, status, 42)) return;
  const uint4* src = reinterpret_cast<const uint4*>(tree_feat + ((size_t)s * n_tree + node) * feat_dim);
  uint4* dst = reinterpret_cast<uint4*>(new_feat + ((size_t)s * max_new + j) * feat_dim);
  for (int i = threadIdx.x; i < feat_dim / 8; i += blockDim.x) dst[i] = src[i];
}

size_t accept_scratch_bytes(int b) { return (size_t)b * sizeof(AcceptScratch); }

int launch_accept(int b, int n_tree, const int32_t* choice, const int32_t* tok, const int32_t* parent,
                  df_bf16* k_cache, df_bf16* v_cache, int n_layers, int Hkv, int cap, int32_t* cache_len,
                  const df_bf16* tree_feat, int feat_dim, df_bf16* new_feat, int max_new, int32_t* n_new,
                  int32_t* acc_tok, int32_t* n_acc, int32_t* new_bonus, int32_t* src_slot, void* scratch,
                  int* status, cudaStream_t st) {
  DF_TRACE("accept_compact", st);
  AcceptScratch* sc = reinterpret_cast<AcceptScratch*>(scratch);
  launch_k(accept_walk_kernel, dim3(b), dim3(32), 0, st, n_tree, max_new, choice, tok, parent, cache_len, cap, n_new, acc_tok, n_acc,
                                       new_bonus, src_slot, sc, status);
  if (k_cache && v_cache && n_layers > 0)
    launch_k(compact_kernel, dim3(dim3(n_layers * b * Hkv, 2)), dim3(256), 0, st, k_cache, v_cache, b, Hkv, cap, sc,
             status);
  if (tree_feat && new_feat)
    launch_k(gather_feat_kernel, dim3(dim3(b, max_new)), dim3(256), 0, st, tree_feat, n_tree, feat_dim, new_feat, max_new, sc,
             status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace df
