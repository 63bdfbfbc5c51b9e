// Host-side description of one weight-streaming GEMM launch (see gemm.cu).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace df {

enum GemmMode { kGemmAtomicAdd = 0, kGemmStore = 1, kGemmArgmax = 2, kGemmPartial = 3 };

struct PartialView;

struct GemmDesc {
  const void* X;   // [M][K] bf16, row stride ldx elements
  const void* W;   // [N][K] bf16, row stride ldw elements
  int M, N, K;
  long long ldx, ldw;
  int mode;
  float* out;      // kGemmAtomicAdd: out[t*ldo + n] += ...;  kGemmStore: out[t*ldo + n] = ...
  int ldo;
  unsigned long long* amax;  // kGemmArgmax: per-token packed (value key << 32 | ~index), max-reduced
  const uint32_t* draw_key;  // kGemmArgmax, optional: per-token draw keys (draw_key()); the argmax is
                             // then taken over value * inv_temp + Gumbel noise (a temperature draw)
  float inv_temp;
  float* stats;    // kGemmStore, optional: [M][4 * ceil(N/128)] float2 (max, sum exp(x - max)) partials
  int* status;
  float* part;     // kGemmPartial: slot buffer (size from gemm_partial_bytes)
  PartialView* view;  // kGemmPartial: filled with what consumers need to read the slots
  int min_k_per_cta;  // kGemmPartial, optional: launch few enough CTAs that each takes at least
                      // this many k-steps (fewer pieces per tile for a tiny weight; 0 = no limit)
};

int launch_gemm(const GemmDesc& g, cudaStream_t st);
// Bytes of partial-tile slots a kGemmPartial launch of this shape writes.
size_t gemm_partial_bytes(int M, int N, int K, int min_k_per_cta = 0);
int make_tmap_2d(struct CUtensorMap_st* out, const void* ptr, long long rows, long long cols, long long ld, int box_rows);

}  // namespace df
