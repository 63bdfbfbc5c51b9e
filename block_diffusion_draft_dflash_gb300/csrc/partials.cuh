// Reading the partial tiles a stream-K GEMM leaves behind (see gemm.cu, kGemmPartial).
//
// The GEMM splits its (tile, k-step) iteration space evenly over its CTAs.  Inside its
// range a CTA meets consecutive tiles; for each one (a "segment") it stores its fp32
// accumulator, [BN tokens][128 features], to a slot of its own.  It also records, for
// every tile, the slots that hold its pieces in CTA order (tile_slot[tile][0 .. cnt-1]),
// so that a reader sums exactly those, always in the same order: the result is
// deterministic and needs no atomics.
#pragma once
#include "common.cuh"

namespace df {

struct PartialView {
  const float* part;        // [slots][BN][128]
  const int* tile_cnt;      // [tiles]
  const int* tile_slot;     // [tiles][maxc]
  int maxc, BN, n_ttiles;
};

// Output (token t, rows r..r+3 of weight tile w) as a float4 (r a multiple of 4).
DF_DEV float4 partial_sum4(const PartialView& v, int w, int t, int r) {
  int tt = 0, j = t;
  if (v.n_ttiles > 1) { tt = t / v.BN; j = t - tt * v.BN; }
  const int tile = w * v.n_ttiles + tt;
  const int n = v.tile_cnt[tile];
  const int* sl = v.tile_slot + (size_t)tile * v.maxc;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* base = v.part + (size_t)j * 128 + r;
  const size_t slot_stride = (size_t)v.BN * 128;
#pragma unroll 4
  for (int i = 0; i < n; ++i) {
    const float4 x = __ldcg(reinterpret_cast<const float4*>(base + (size_t)sl[i] * slot_stride));
    acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
  }
  return acc;
}

// The four values (lane, lane+32, lane+64, lane+96) of token t in weight tile w.
DF_DEV void partial_sum_strided4(const PartialView& v, int w, int t, int lane, float* out) {
  int tt = 0, j = t;
  if (v.n_ttiles > 1) { tt = t / v.BN; j = t - tt * v.BN; }
  const int tile = w * v.n_ttiles + tt;
  const int n = v.tile_cnt[tile];
  const int* sl = v.tile_slot + (size_t)tile * v.maxc;
  out[0] = out[1] = out[2] = out[3] = 0.f;
  const float* base = v.part + (size_t)j * 128 + lane;
  const size_t slot_stride = (size_t)v.BN * 128;
#pragma unroll 4
  for (int i = 0; i < n; ++i) {
    const float* p = base + (size_t)sl[i] * slot_stride;
    out[0] += __ldcg(p); out[1] += __ldcg(p + 32); out[2] += __ldcg(p + 64); out[3] += __ldcg(p + 96);
  }
}

}  // namespace df
