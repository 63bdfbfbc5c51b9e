// Reading the partial tiles a stream-K GEMM leaves behind (see gemm.cu, kGemmPartial).
//
// The GEMM splits its (tile, k-step) iteration space evenly over its CTAs.  Inside its
// range a CTA meets consecutive tiles; for each one (a "segment") it stores its fp32
// accumulator, [BN tokens][128 features], to a slot of its own.  It also records, for
// every tile, the slots that hold its pieces in CTA order (after the count in meta[tile]),
// so that a reader sums exactly those, always in the same order: the result is
// deterministic and needs no atomics.
#pragma once
#include "common.cuh"

namespace df {

struct PartialView {
  const float* part;  // [slots][BN][128]
  const int* meta;    // [tiles][meta_stride]: piece count, then the pieces' slots in CTA order
  int meta_stride;    // a multiple of 4 (so a tile's list starts 16-byte aligned)
  int BN, n_ttiles;
};

DF_DEV void add4(float4& a, const float4& b) { a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w; }

// Sums f(slot) over a tile's pieces in their recorded order.  The count and the first three
// slots arrive in one 16-byte load, so the data loads of up to three pieces issue after a
// single dependent round trip.
template <class T, class F>
DF_DEV T sum_pieces(const PartialView& v, int tile, F f) {
  const int4* m = reinterpret_cast<const int4*>(v.meta + (size_t)tile * v.meta_stride);
  const int4 h = __ldcg(m);
  T acc = f(h.y);
  if (h.x > 1) acc += f(h.z);
  if (h.x > 2) acc += f(h.w);
  for (int i = 3; i < h.x; i += 4) {
    const int4 q = __ldcg(m + (i + 1) / 4);
    acc += f(q.x);
    if (i + 1 < h.x) acc += f(q.y);
    if (i + 2 < h.x) acc += f(q.z);
    if (i + 3 < h.x) acc += f(q.w);
  }
  return acc;
}

struct Sum4 {
  float4 v;
  DF_DEV Sum4(float4 x) : v(x) {}
  DF_DEV Sum4& operator+=(const Sum4& o) { add4(v, o.v); return *this; }
};
struct Strided4 {
  float a, b, c, d;
  DF_DEV Strided4& operator+=(const Strided4& o) { a += o.a; b += o.b; c += o.c; d += o.d; return *this; }
};

DF_DEV void tile_of(const PartialView& v, int w, int t, int& tile, int& j) {
  int tt = 0;
  j = t;
  if (v.n_ttiles > 1) { tt = t / v.BN; j = t - tt * v.BN; }
  tile = w * v.n_ttiles + tt;
}

// Output (token t, rows r..r+3 of weight tile w) as a float4 (r a multiple of 4).
DF_DEV float4 partial_sum4(const PartialView& v, int w, int t, int r) {
  int tile, j;
  tile_of(v, w, t, tile, j);
  const float* base = v.part + (size_t)j * 128 + r;
  const size_t stride = (size_t)v.BN * 128;
  return sum_pieces<Sum4>(v, tile, [&](int s) {
    return Sum4(__ldcg(reinterpret_cast<const float4*>(base + (size_t)s * stride)));
  }).v;
}

// The four values (lane, lane+32, lane+64, lane+96) of token t in weight tile w.
DF_DEV void partial_sum_strided4(const PartialView& v, int w, int t, int lane, float* out) {
  int tile, j;
  tile_of(v, w, t, tile, j);
  const float* base = v.part + (size_t)j * 128 + lane;
  const size_t stride = (size_t)v.BN * 128;
  const Strided4 r = sum_pieces<Strided4>(v, tile, [&](int s) {
    const float* p = base + (size_t)s * stride;
    return Strided4{__ldcg(p), __ldcg(p + 32), __ldcg(p + 64), __ldcg(p + 96)};
  });
  out[0] = r.a; out[1] = r.b; out[2] = r.c; out[3] = r.d;
}

}  // namespace df
