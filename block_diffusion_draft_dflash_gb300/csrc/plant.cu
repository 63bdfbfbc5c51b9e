// Acceptance planting for synthetic models (benchmark and test harness; the pages have no
// counterpart).  Random-init drafters almost never agree with random-init targets, so a
// known fraction of agreement is planted into the drafter's log-probs: for sequence s and
// draft position d (1..D), with probability `rate`, row d becomes the log-softmax of its
// logits with `bias` added at the reference token r = ref[s][pos[s]][d - 1] (the token the
// harness expects the target to choose at depth d when the block starts at position
// pos[s]):
//   lp'_i = lp_i - c  (i != r),   lp'_r = lp_r + bias - c,   c = log(1 + p_r (e^bias - 1)),
// where p_r = exp(lp_r).  The choice is a counter-based hash of (seed, s, pos[s], d), so a
// captured graph replays a different draw at every step (pos grows) with no host input.
// With miss_bias > 0, a row not chosen is a near miss instead of a random guess: `bias` goes
// to a decoy token (a second hash of the draw picks it, never r) and `miss_bias` to r, so
// the two lead the row, r usually second (about e^(miss_bias - bias) of the decoy's mass): a
// tree holds both branches, a single chain only the first.  miss_bias = 0 leaves such rows
// as they are.
#include "common.cuh"
#include "nvtx.h"
#include "trace.h"

namespace df {

DF_DEV uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

// grid: b * D rows; block 512.  One block per row: the correction c is taken from the row
// before any of it is rewritten.
__global__ void __launch_bounds__(512) plant_logprobs_kernel(float* __restrict__ lp, int D, int V,
                                                             const int32_t* __restrict__ ref, int n_pos,
                                                             const int32_t* __restrict__ pos, float rate, float bias,
                                                             float miss_bias, unsigned long long seed) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, s = row / D, d = row % D + 1;
  const int p0 = pos[s];
  if (p0 < 0 || p0 >= n_pos) return;
  const uint64_t h = splitmix64(seed ^ splitmix64(((uint64_t)s << 40) ^ ((uint64_t)(uint32_t)p0 << 8) ^ (uint64_t)d));
  const double u = (double)(h >> 11) * (1.0 / 9007199254740992.0);  // uniform [0, 1)
  const bool hit = u < (double)rate;
  if (!hit && !(miss_bias > 0.f)) return;
  const int r = ref[((size_t)s * n_pos + p0) * D + d - 1];
  if (r < 0 || r >= V) return;  // no reference for this block
  const float add_r = hit ? bias : miss_bias;
  const int decoy = hit || V < 2 ? -1 : (int)(((uint64_t)r + 1 + splitmix64(h) % (uint64_t)(V - 1)) % (uint64_t)V);
  float* x = lp + (size_t)row * V;
  __shared__ float c_sh;
  if (threadIdx.x == 0) {
    // log of the biased row's normaliser: 1 + p_r (e^add_r - 1) [+ p_decoy (e^bias - 1)]
    double zm1 = exp((double)x[r]) * expm1((double)add_r);
    if (decoy >= 0) zm1 += exp((double)x[decoy]) * expm1((double)bias);
    c_sh = (float)log1p(zm1);
  }
  __syncthreads();
  const float c = c_sh;
  for (int i = threadIdx.x; i < V; i += blockDim.x)
    x[i] = (i == r ? x[i] + add_r : i == decoy ? x[i] + bias : x[i]) - c;
}

}  // namespace df

extern "C" int dflash_plant_logprobs(float* logprobs, int b, int D, int V, const int32_t* ref, int n_pos,
                                     const int32_t* pos, float rate, float bias, float miss_bias,
                                     unsigned long long seed, df_stream stream) {
  DF_NVTX("dflash_plant_logprobs");
  if (b < 0 || D < 1 || V < 1 || n_pos < 0) return DF_ERR_ARG;
  if (b == 0 || n_pos == 0) return DF_OK;
  if (!logprobs || !ref || !pos) return DF_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  DF_TRACE("plant", st);
  df::launch_k(df::plant_logprobs_kernel, dim3(b * D), dim3(512), 0, st, logprobs, D, V, ref, n_pos, pos, rate,
               bias, miss_bias, seed);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
