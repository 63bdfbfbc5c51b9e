// Row-wise kernels around the GEMMs of a decoder layer (all memory-bound, SIMT):
//   embed_rows_kernel      residual stream <- token embedding rows (fp32)
//   rmsnorm_kernel         bf16 GEMM input <- RMSNorm(fp32 residual) * gain; can also
//                          zero the next GEMM's fp32 accumulator and capture the residual
//                          rows as bf16 feature rows (the drafter's context features)
//   rope_table_kernel      (cos, sin) of every row's rotary angles, once per forward
//   qk_norm_rope_kernel    per-head RMSNorm of q and k, rotary embedding, q to its buffer,
//                          k and v into their cache slots (v transposed)
//   res_norm_kernel        partial tiles of a projection + residual, then RMSNorm
//   swiglu_partial_kernel  bf16 act <- silu(gate) * up from the gate/up partial tiles
//   lse_from_stats_kernel  log-sum-exp of each LM-head row from the GEMM's softmax partials
//   sub_lse_kernel         x - lse, in place (the drafter's log-probs)
//   argmax_finalize_kernel token id from the packed argmax keys
//   draw_keys_kernel       per-row keys of the LM head's temperature draw
// Readings: Qwen3-style pre-norm layer (see the oracle); RMSNorm eps and rotary base
// come from the model config.
#include "common.cuh"
#include "layers.h"
#include "trace.h"

namespace df {

// grid: rows; block 256.  tok_mode 0: tok[r]; 1: drafter block row (bonus / mask).
__global__ void __launch_bounds__(256) embed_rows_kernel(const df_bf16* __restrict__ E, int d, int V,
                                                         const int32_t* __restrict__ tok, const int32_t* __restrict__ bonus,
                                                         int L, int mask_id, float* __restrict__ h, int* status) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  int t;
  if (bonus) {
    const int s = r / L, i = r % L;
    t = i == 0 ? bonus[s] : mask_id;
  } else {
    t = tok[r];
  }
  if (t < 0 || t >= V) {
    if (threadIdx.x == 0) set_status(status, DF_ERR_ARG, r);
    t = 0;
  }
  const uint2* src = reinterpret_cast<const uint2*>(E + (size_t)t * d);  // 4 bf16
  float4* dst = reinterpret_cast<float4*>(h + (size_t)r * d);
  for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
    const uint2 u = src[i];
    dst[i] = make_float4(bf16_to_f(u.x & 0xFFFF), bf16_to_f(u.x >> 16), bf16_to_f(u.y & 0xFFFF), bf16_to_f(u.y >> 16));
  }
}

// grid: out rows (+ extra blocks that only zero); block 256.  d multiple of 4.
__global__ void __launch_bounds__(256) rmsnorm_kernel(RmsNormArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8];
  const int o = blockIdx.x;
  // zeroing of the next accumulator, spread over all blocks
  if (a.zero && a.zero_count) {
    const long long per = (a.zero_count + gridDim.x - 1) / gridDim.x;
    const long long z0 = per * o, z1 = min(z0 + per, a.zero_count);
    for (long long i = z0 + threadIdx.x; i < z1; i += blockDim.x) a.zero[i] = 0.f;
  }
  if (o >= a.rows) return;
  const int in_row = (o / a.group_out) * a.group_in + a.in_off + (o % a.group_out);
  const float4* x = reinterpret_cast<const float4*>(a.in + (size_t)in_row * a.d);
  const int n4 = a.d / 4;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = x[i];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
  const float inv = rsqrtf(tot / a.d + a.eps);
  const uint2* g = reinterpret_cast<const uint2*>(a.gain);
  uint2* y = reinterpret_cast<uint2*>(a.out + (size_t)o * a.ld_out);
  uint2* cap = a.capture ? reinterpret_cast<uint2*>(a.capture + (size_t)in_row * a.ld_capture) : nullptr;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = x[i];
    const uint2 gw = g[i];
    const float g0 = bf16_to_f(gw.x & 0xFFFF), g1 = bf16_to_f(gw.x >> 16), g2 = bf16_to_f(gw.y & 0xFFFF),
                g3 = bf16_to_f(gw.y >> 16);
    uint2 r;
    r.x = (uint32_t)f_to_bf16(v.x * inv * g0) | ((uint32_t)f_to_bf16(v.y * inv * g1) << 16);
    r.y = (uint32_t)f_to_bf16(v.z * inv * g2) | ((uint32_t)f_to_bf16(v.w * inv * g3) << 16);
    y[i] = r;
    if (cap) {
      uint2 c;
      c.x = (uint32_t)f_to_bf16(v.x) | ((uint32_t)f_to_bf16(v.y) << 16);
      c.y = (uint32_t)f_to_bf16(v.z) | ((uint32_t)f_to_bf16(v.w) << 16);
      cap[i] = c;
    }
  }
}

// Row r of a q/k/v projection: its sequence, cache slot and rotary position.  Rows
// 0 .. b*TA-1 are query rows (slot after the sequence's new context rows, position offset by
// depth); the b*TB context rows follow.  Returns false for a context row beyond its
// sequence's count (nothing to write).
DF_DEV bool qk_row(const QkRopeArgs& a, int r, int& s, int& slot, int& pos, bool& write_q) {
  const int nA = a.b * a.TA;
  if (r < nA) {
    s = r / a.TA;
    const int i = r % a.TA;
    const int base = a.base[s] + (a.nnew ? a.nnew[s] : 0);
    slot = base + i;
    pos = base + (a.depth ? a.depth[r] : i);
    write_q = true;
    return true;
  }
  const int rr = r - nA;
  s = rr / a.TB;
  const int j = rr % a.TB;
  slot = pos = a.base[s] + j;
  write_q = false;
  return j < a.nnew[s];
}

// grid: rows; block 64: (cos, sin) of pos * theta^(-2i/128) for pair i = threadIdx.x.
// The angle is reduced mod 2 pi in fp64 so that large positions keep full fp32 accuracy
// in sincosf.
__global__ void __launch_bounds__(64) rope_table_kernel(QkRopeArgs a, float2* __restrict__ table) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, i = threadIdx.x;
  int s, slot, pos;
  bool write_q;
  if (!qk_row(a, r, s, slot, pos, write_q)) return;
  const double twopi = 6.283185307179586476925286766559, inv_twopi = 0.15915494309189533576888376337251;
  double ang = (double)pos * a.inv_freq[i];
  ang -= twopi * rint(ang * inv_twopi);
  float sn, cs;
  sincosf((float)ang, &sn, &cs);
  table[(size_t)r * 64 + i] = make_float2(cs, sn);
}

// grid: (rows, ceil((Hq + 2 Hkv) / (8 KH))); block 256: warp w handles heads
// blockIdx.y * 8 KH + w + 8 i, i < KH.
// Lane l owns elements l, l+32, l+64, l+96 of a 128-wide head, so both rotary pairs
// (i, i+64) of the lane stay in the lane.
constexpr int kQkHeads = 3;
template <int KH>  // heads per warp
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(QkRopeArgs a) {
  pdl_wait();
  pdl_trigger();
  constexpr int HD = 128;
  const int r = blockIdx.x;
  int s, slot, pos;
  bool write_q;
  if (!qk_row(a, r, s, slot, pos, write_q)) return;
  if (slot >= a.cap) {
    if (threadIdx.x == 0) set_status(a.status, DF_ERR_CAPACITY, r);
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const float* row = a.qkv ? a.qkv + (size_t)r * a.ld_qkv : nullptr;
  const float2 cs0 = a.rope[(size_t)r * 64 + lane], cs1 = a.rope[(size_t)r * 64 + lane + 32];
  const float c0 = cs0.x, s0 = cs0.y, c1 = cs1.x, s1 = cs1.y;
  const int nh = a.Hq + 2 * a.Hkv;
  // this warp's heads: h0 + i * nw, i < KH; every head's loads are issued before any is used
  const int h0 = blockIdx.y * nw * KH + warp;
  float v[KH][4];
#pragma unroll
  for (int i = 0; i < KH; ++i) {
    const int h = h0 + i * nw;
    v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.f;
    if (h >= nh || (!write_q && h < a.Hq)) continue;
    if (a.pv.part) {
      partial_sum_strided4(a.pv, h, r, lane, v[i]);
    } else {
      const float* x = row + h * HD;
      v[i][0] = x[lane]; v[i][1] = x[lane + 32]; v[i][2] = x[lane + 64]; v[i][3] = x[lane + 96];
    }
  }
#pragma unroll
  for (int i = 0; i < KH; ++i) {
    const int h = h0 + i * nw;
    if (h >= nh || (!write_q && h < a.Hq)) continue;
    float v0 = v[i][0], v1 = v[i][1], v2 = v[i][2], v3 = v[i][3];
    if (h < a.Hq + a.Hkv) {
      const df_bf16* gain = h < a.Hq ? a.q_norm : a.k_norm;
      const float ms = warp_sum(v0 * v0 + v1 * v1 + v2 * v2 + v3 * v3) / HD;
      const float inv = rsqrtf(ms + a.eps);
      v0 *= inv * bf16_to_f(gain[lane]);
      v1 *= inv * bf16_to_f(gain[lane + 32]);
      v2 *= inv * bf16_to_f(gain[lane + 64]);
      v3 *= inv * bf16_to_f(gain[lane + 96]);
      // rotate-half: (x_i, x_{i+64}) -> (x_i c - x_{i+64} s, x_{i+64} c + x_i s)
      const float r0 = v0 * c0 - v2 * s0, r2 = v2 * c0 + v0 * s0;
      const float r1 = v1 * c1 - v3 * s1, r3 = v3 * c1 + v1 * s1;
      v0 = r0; v1 = r1; v2 = r2; v3 = r3;
    }
    if (h < a.Hq) {
      df_bf16* q = a.q_out + ((size_t)r * a.Hq + h) * HD;
      q[lane] = f_to_bf16(v0); q[lane + 32] = f_to_bf16(v1); q[lane + 64] = f_to_bf16(v2); q[lane + 96] = f_to_bf16(v3);
    } else if (h < a.Hq + a.Hkv) {
      const int kh = h - a.Hq;
      df_bf16* k = a.k_plane + (((size_t)s * a.Hkv + kh) * a.cap + slot) * HD;
      k[lane] = f_to_bf16(v0); k[lane + 32] = f_to_bf16(v1); k[lane + 64] = f_to_bf16(v2); k[lane + 96] = f_to_bf16(v3);
    } else {
      const int vh = h - a.Hq - a.Hkv;
      df_bf16* vt = a.v_plane + ((size_t)s * a.Hkv + vh) * HD * (size_t)a.cap + slot;
      vt[(size_t)lane * a.cap] = f_to_bf16(v0);
      vt[(size_t)(lane + 32) * a.cap] = f_to_bf16(v1);
      vt[(size_t)(lane + 64) * a.cap] = f_to_bf16(v2);
      vt[(size_t)(lane + 96) * a.cap] = f_to_bf16(v3);
    }
  }
}

// grid: output rows; block min(d/4, 1024) threads (one float4 of the row each, two
// passes for d > 4096).  d a multiple of 128 and at most 8192.
__global__ void __launch_bounds__(1024) res_norm_kernel(ResNormArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  const int o = blockIdx.x;
  const int t = (o / a.group_out) * a.group_in + a.in_off + (o % a.group_out);
  float4 v[2];
  const int per = blockDim.x * 4;
  float ss = 0.f;
  float* hrow = a.h ? a.h + (size_t)t * a.d : nullptr;
  // every load first (the residual rows and both partial sums), the residual stores after:
  // a store between them would keep the second element's loads behind the first's
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int n = i * per + threadIdx.x * 4;
    v[i] = n < a.d ? partial_sum4(a.pv, n >> 7, t, n & 127) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float4 hv[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  if (hrow) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int n = i * per + threadIdx.x * 4;
      if (n < a.d) hv[i] = *reinterpret_cast<const float4*>(hrow + n);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int n = i * per + threadIdx.x * 4;
    if (n >= a.d) continue;
    float4& y = v[i];
    if (hrow) {
      y.x += hv[i].x; y.y += hv[i].y; y.z += hv[i].z; y.w += hv[i].w;
      *reinterpret_cast<float4*>(hrow + n) = y;
    }
    ss += y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
  }
  ss = warp_sum(ss);
  const int nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < nw; ++w) tot += red[w];
  const float inv = rsqrtf(tot / a.d + a.eps);
  const uint2* g = reinterpret_cast<const uint2*>(a.gain);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int n = i * per + threadIdx.x * 4;
    if (n >= a.d) continue;
    const float4 y = v[i];
    const uint2 gw = g[n / 4];
    uint2 r;
    r.x = (uint32_t)f_to_bf16(y.x * inv * bf16_to_f(gw.x & 0xFFFF)) |
          ((uint32_t)f_to_bf16(y.y * inv * bf16_to_f(gw.x >> 16)) << 16);
    r.y = (uint32_t)f_to_bf16(y.z * inv * bf16_to_f(gw.y & 0xFFFF)) |
          ((uint32_t)f_to_bf16(y.w * inv * bf16_to_f(gw.y >> 16)) << 16);
    *reinterpret_cast<uint2*>(a.out + (size_t)o * a.ld_out + n) = r;
    if (a.capture) {
      uint2 c;
      c.x = (uint32_t)f_to_bf16(y.x) | ((uint32_t)f_to_bf16(y.y) << 16);
      c.y = (uint32_t)f_to_bf16(y.z) | ((uint32_t)f_to_bf16(y.w) << 16);
      *reinterpret_cast<uint2*>(a.capture + (size_t)t * a.ld_capture + n) = c;
    }
  }
}

// grid: (rows, ceil(F / 1024)) (rows in x: y is limited to 65535); block 256; 4 features
// per thread.
__global__ void __launch_bounds__(256) swiglu_partial_kernel(SwigluArgs a) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int f = (blockIdx.y * 256 + threadIdx.x) * 4;
  if (f >= a.F) return;
  const float4 g = partial_sum4(a.pv, f >> 7, t, f & 127);
  const int fu = a.F + f;
  const float4 u = partial_sum4(a.pv, fu >> 7, t, fu & 127);
  auto sl = [](float x) { return x / (1.f + __expf(-x)); };
  uint2 o;
  o.x = (uint32_t)f_to_bf16(sl(g.x) * u.x) | ((uint32_t)f_to_bf16(sl(g.y) * u.y) << 16);
  o.y = (uint32_t)f_to_bf16(sl(g.z) * u.z) | ((uint32_t)f_to_bf16(sl(g.w) * u.w) << 16);
  *reinterpret_cast<uint2*>(a.act + (size_t)t * a.F + f) = o;
}

// lse[r] from the GEMM epilogue's (max, sum exp) partials of row r.
__global__ void __launch_bounds__(1024) lse_from_stats_kernel(const float2* __restrict__ stats, int n_stats,
                                                              float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sm[32], ss[32];
  const float2* st = stats + (size_t)blockIdx.x * n_stats;
  float m = -INFINITY, s = 0.f;
  for (int i = threadIdx.x; i < n_stats; i += blockDim.x) {
    const float2 v = st[i];
    if (v.x == -INFINITY) continue;
    if (v.x > m) { s = s * __expf(m - v.x) + v.y; m = v.x; }
    else s += v.y * __expf(v.x - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float mm = fmaxf(m, m2);
    s = (m == -INFINITY ? 0.f : s * __expf(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * __expf(m2 - mm));
    m = mm;
  }
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) { sm[w] = m; ss[w] = s; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) M = fmaxf(M, sm[i]);
    float S = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) S += sm[i] == -INFINITY ? 0.f : ss[i] * __expf(sm[i] - M);
    lse[blockIdx.x] = M + logf(S);
  }
}

// x[r][i] -= lse[r] over a grid of (row, chunk) blocks (rows in x).
__global__ void __launch_bounds__(256) sub_lse_kernel(float* __restrict__ x, int V, const float* __restrict__ lse) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const float l = lse[r];
  float* row = x + (size_t)r * V;
  if ((V & 3) == 0) {
    // float4s, four per thread loaded before any is written back (an in-place update would
    // otherwise keep each load behind the previous store)
    constexpr int U = 4;
    const int V4 = V >> 2, chunk4 = (V4 + gridDim.y - 1) / gridDim.y;
    const int q0 = blockIdx.y * chunk4, q1 = min(V4, q0 + chunk4);
    float4* row4 = reinterpret_cast<float4*>(row);
    for (int q = q0 + threadIdx.x; q < q1; q += blockDim.x * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (q + u * (int)blockDim.x < q1) v[u] = row4[q + u * blockDim.x];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (q + u * (int)blockDim.x >= q1) continue;
        v[u].x -= l; v[u].y -= l; v[u].z -= l; v[u].w -= l;
        row4[q + u * blockDim.x] = v[u];
      }
    }
    return;
  }
  const int chunk = (V + gridDim.y - 1) / gridDim.y;
  const int i0 = blockIdx.y * chunk, i1 = min(V, i0 + chunk);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) row[i] -= l;
}

__global__ void argmax_finalize_kernel(const unsigned long long* __restrict__ amax, int rows, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r < rows) out[r] = (int32_t)(~(uint32_t)(amax[r] & 0xFFFFFFFFull));
}

__global__ void draw_keys_kernel(int rows, uint64_t seed, const int32_t* __restrict__ row_seq,
                                 const int32_t* __restrict__ row_pos, int T, const int32_t* __restrict__ cache_len,
                                 const int32_t* __restrict__ depth, uint32_t* __restrict__ keys) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= rows) return;
  int s, n;
  if (row_seq) {
    s = row_seq[t];
    n = row_pos[t];
  } else {
    s = t / T;
    n = cache_len[s] + (depth ? depth[t] : t - s * T) + 1;
  }
  keys[t] = draw_key(seed, s, n);
}

// ----------------------------------------------------------------------------- launchers
int launch_embed(const df_bf16* E, int d, int V, const int32_t* tok, const int32_t* bonus, int L, int mask_id,
                 float* h, int rows, int* status, cudaStream_t st) {
  DF_TRACE("embed", st);
  launch_k(embed_rows_kernel, dim3(rows), dim3(256), 0, st, E, d, V, tok, bonus, L, mask_id, h, status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
int launch_rmsnorm(const RmsNormArgs& a, cudaStream_t st) {
  int grid = a.rows;
  if (a.zero && a.zero_count && grid < 296) grid = 296;
  DF_TRACE("rmsnorm", st);
  launch_k(rmsnorm_kernel, dim3(grid), dim3(256), 0, st, a);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
int launch_rope_table(const QkRopeArgs& a_in, float2* table, cudaStream_t st) {
  const int rows = a_in.b * (a_in.TA + a_in.TB);
  if (rows == 0) return DF_OK;
  QkRopeArgs a = a_in;
  for (int i = 0; i < 64; ++i) a.inv_freq[i] = pow((double)a.theta, -2.0 * i / 128.0);
  DF_TRACE("rope_table", st);
  launch_k(rope_table_kernel, dim3(rows), dim3(64), 0, st, a, table);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
int launch_qk_rope(const QkRopeArgs& a, cudaStream_t st) {
  const int rows = a.b * (a.TA + a.TB);
  if (rows == 0) return DF_OK;
  if (!a.rope) return DF_ERR_ARG;
  DF_TRACE("qk_norm_rope", st);
  // kQkHeads heads per warp: one row's 48 heads in 2 blocks of 8 warps, so the whole grid is
  // resident beside the q/k/v GEMM
  launch_k(qk_norm_rope_kernel<kQkHeads>, dim3(dim3(rows, (a.Hq + 2 * a.Hkv + 8 * kQkHeads - 1) / (8 * kQkHeads))),
           dim3(256), 0, st, a);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
int launch_res_norm(const ResNormArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return DF_OK;
  if (a.d % 128 || a.d > 8192) return DF_ERR_SHAPE;
  DF_TRACE("residual_norm", st);
  // two float4 per thread when the row is long enough: 512-thread blocks leave room for two
  // of them beside a GEMM CTA, so every row's block is resident before the GEMM ends
  int threads = a.d >= 2048 ? a.d / 8 : a.d / 4;
  if (threads > 1024) threads = 1024;
  threads = (threads + 31) / 32 * 32;
  launch_k(res_norm_kernel, dim3(a.rows), dim3(threads), 0, st, a);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
int launch_swiglu_partial(const SwigluArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return DF_OK;
  DF_TRACE("swiglu", st);
  launch_k(swiglu_partial_kernel, dim3(dim3(a.rows, (a.F + 1023) / 1024)), dim3(256), 0, st, a);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
int launch_logsoftmax_from_stats(float* x, int rows, int V, const float* stats, int n_stats, float* lse,
                                 cudaStream_t st) {
  DF_TRACE("logsoftmax", st);
  launch_k(lse_from_stats_kernel, dim3(rows), dim3(1024), 0, st, reinterpret_cast<const float2*>(stats), n_stats, lse);
  launch_k(sub_lse_kernel, dim3(dim3(rows, 32)), dim3(256), 0, st, x, V, lse);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
int launch_draw_keys(int rows, uint64_t seed, const int32_t* row_seq, const int32_t* row_pos, int T,
                     const int32_t* cache_len, const int32_t* depth, uint32_t* keys, cudaStream_t st) {
  DF_TRACE("draw_keys", st);
  launch_k(draw_keys_kernel, dim3((rows + 255) / 256), dim3(256), 0, st, rows, seed, row_seq, row_pos, T, cache_len,
           depth, keys);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
int launch_argmax_finalize(const unsigned long long* amax, int rows, int32_t* out, cudaStream_t st) {
  DF_TRACE("argmax_finalize", st);
  launch_k(argmax_finalize_kernel, dim3((rows + 255) / 256), dim3(256), 0, st, amax, rows, out);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace df
