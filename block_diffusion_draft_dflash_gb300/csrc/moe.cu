// Mixture-of-experts feed-forward of the target, for the mixture-of-experts target the
// pages evaluate (Qwen3-Coder-30B-A3B: [DFlash] SGLang results, summary of "Accelerating
// Speculative Decoding with Block Diffusion Draft Trees", section "실험 결과").  Reading of
// its feed-forward (Qwen3-MoE): a router softmax over the experts, the top-k experts per
// token with weights renormalised to sum 1, each expert a SwiGLU feed-forward.
//
//   moe_route_kernel    one warp per token: sums the router logits' partial tiles, fp32
//                       softmax, k rounds of a warp maximum (lower expert id first among
//                       equal probabilities), renormalised weights
//   moe_permute_kernel  one CTA: stable counting sort of the (token, choice) pairs by
//                       expert (ties by token, then choice), expert offsets and counts
//   moe_gather_kernel   normed rows copied into expert order
//   moe_gemm_kernel     grouped GEMM on tcgen05 over the stacked expert weights: the rows
//                       of each expert in chunks of at most 256 (the chunk list is built by
//                       the dispatch on the device), one work item per (chunk, 128 output
//                       features), persistent CTAs taking items round robin; a k-step loads
//                       the item's 128 x 64 weight tile once and the chunk's rows in 64-row
//                       boxes, and one MMA of N = the chunk's rows (rounded up to 16) uses
//                       them, so an expert's weights are streamed once per chunk however
//                       many rows it holds; gate/up items load 64 gate rows and the matching
//                       64 up rows, and the epilogue writes silu(g) * u
//   moe_combine_kernel  h += sum_j w_j expert_out_j, then RMSNorm (as res_norm)
// No host synchronisation: the routing stays on the device, so a step is graph-capturable.
#include "common.cuh"
#include "checked.cuh"
#include "gemm.h"
#include "moe.h"
#include "runtime.h"
#include "trace.h"

namespace df {

constexpr int kMoeThreads = 192;
constexpr int kMoeBK = 64;
constexpr int kMoeChunk = 256;  // rows of one expert per work item at most (MMA N <= 256)
constexpr uint32_t kMoeWBytes = 128 * kMoeBK * 2;  // 128 weight rows x 64
constexpr uint32_t kMoeXBox = 64 * kMoeBK * 2;     // 64 token rows x 64
// The k-steps' operands sit in a ring of bytes: a k-step takes its weight tile plus as many
// 64-row boxes as its chunk needs (24 to 48 KB), so small chunks keep more k-steps in flight.
constexpr uint32_t kMoeRing = 192 * 1024;
constexpr int kMoeSlots = 8;    // k-steps in flight at most (kMoeRing / the smallest k-step)
constexpr int kMoeXPitch = 33;  // gate/up exchange buffer: [64 features][32 tokens], padded
enum { kMoeGateUp = 0, kMoeDown = 1 };

// ------------------------------------------------------------------------------ routing
// grid: ceil(R / 8); block 256: one warp per token.  E a multiple of 32, at most 256.
__global__ void __launch_bounds__(256) moe_route_kernel(PartialView pv, int R, int E, int k,
                                                        int32_t* __restrict__ topk_id, float* __restrict__ topk_w,
                                                        int* status) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= R) return;
  constexpr int kMaxPer = 8;  // E / 32 <= 8
  const int per = E / 32;
  float lg[kMaxPer];
#pragma unroll
  for (int w = 0; w < kMaxPer / 4; ++w)
    if (4 * w < per) partial_sum_strided4(pv, w, t, lane, lg + 4 * w);  // experts 128 w + lane + 32 i
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i)
    if (i < per) m = fmaxf(m, lg[i]);
  m = warp_max(m);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i)
    if (i < per) { lg[i] = __expf(lg[i] - m); s += lg[i]; }
  s = warp_sum(s);
  const float inv = 1.f / s;
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) lg[i] = i < per ? lg[i] * inv : -1.f;  // probabilities; -1 = taken / absent
  float wsum = 0.f;
  for (int j = 0; j < k; ++j) {
    // this lane's best (probability desc, expert id asc), then the warp's
    unsigned long long best = 0ull;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
      const int e = (i / 4) * 128 + (i % 4) * 32 + lane;
      const unsigned long long key =
          lg[i] >= 0.f ? (((unsigned long long)float_key(lg[i]) << 32) | (uint32_t)(~(uint32_t)e)) : 0ull;
      if (key > best) { best = key; bi = i; }
    }
    const uint32_t top_hi = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32));
    const uint32_t top_lo = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32) == top_hi ? (uint32_t)best : 0u);
    // no candidate left only when the logits were NaN: route to expert j with weight 0
    const bool none = top_hi == 0u;
    const int e = none ? j : (int)(~top_lo);
    const float pe = none ? 0.f : key_float(top_hi);
    if (none && lane == 0) set_status(status, DF_ERR_NAN, 30);
    if (best == (((unsigned long long)top_hi << 32) | top_lo)) lg[bi] = -1.f;  // the owner drops it
    if (lane == 0) {
      topk_id[(size_t)t * k + j] = e;
      topk_w[(size_t)t * k + j] = pe;
    }
    wsum += pe;
  }
  __syncwarp();
  if (lane < k) topk_w[(size_t)t * k + lane] = wsum > 0.f ? topk_w[(size_t)t * k + lane] / wsum : 0.f;
}

// One CTA of 1024 threads: a stable counting sort of the pairs p = t k + j by expert.
// Warp w takes the contiguous pairs [w c, (w + 1) c), c = ceil(P / 32): it counts them per
// expert (lanes with equal experts found by a match), every expert's rows are then laid out
// warp after warp, and each warp walks its pairs again to place them in order.  Also the
// grouped GEMM's work list: each expert's rows split evenly into chunks of at most m rows,
// m in {256, 192, 128, 64} chosen to minimise the busiest CTA's bytes per k-step summed
// over its items (ceil(items / ctas) x (the weight tile + the widest chunk's row boxes),
// items = chunks x n_wt feature tiles): few experts holding many rows get smaller chunks,
// so that the items spread over all CTAs.
constexpr int kPermWarps = 32;
__constant__ int kChunkCand[4] = {256, 192, 128, 64};
__global__ void __launch_bounds__(kPermWarps * 32) moe_permute_kernel(int P, int E, int k,
                                                                     const int32_t* __restrict__ topk_id,
                                                                     int32_t* __restrict__ counts,
                                                                     int32_t* __restrict__ offsets,
                                                                     int32_t* __restrict__ pos_of,
                                                                     int32_t* __restrict__ pair_token,
                                                                     int4* __restrict__ chunks,
                                                                     int32_t* __restrict__ n_chunks, int n_wt,
                                                                     int ctas) {
  pdl_wait();
  pdl_trigger();
  __shared__ int cnt[kPermWarps][256];  // per warp and expert: a count, then the warp's first row
  __shared__ int tot[256], first[256], nch[256], ch0[256];  // per expert
  __shared__ int cand_chunks[4], cand_boxes[4];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < kPermWarps * 256; i += blockDim.x) (&cnt[0][0])[i] = 0;
  if (threadIdx.x < 4) { cand_chunks[threadIdx.x] = 0; cand_boxes[threadIdx.x] = 0; }
  __syncthreads();
  const int per_warp = (P + kPermWarps - 1) / kPermWarps;
  const int p_lo = min(P, warp * per_warp), p_hi = min(P, p_lo + per_warp);
  for (int p0 = p_lo; p0 < p_hi; p0 += 32) {
    const int p = p0 + lane;
    int id = p < p_hi ? topk_id[p] : -1;
    if (id >= E) id = -1;  // cannot come from the router; kept out of the tables
    const unsigned peers = __match_any_sync(0xffffffffu, id);
    if (id >= 0 && lane == __ffs(peers) - 1) cnt[warp][id] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int acc = 0;
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = cnt[w][e];
      cnt[w][e] = acc;
      acc += c;
    }
    tot[e] = acc;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int n = (acc + kChunkCand[c] - 1) / kChunkCand[c];
      if (n) {
        atomicAdd(&cand_chunks[c], n);
        atomicMax(&cand_boxes[c], ((acc + n - 1) / n + 63) / 64);
      }
    }
  }
  __syncthreads();
  int m = kChunkCand[0];
  long long best = -1;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const long long cost = ((long long)cand_chunks[c] * n_wt + ctas - 1) / ctas * (2 + cand_boxes[c]);
    if (best < 0 || cost < best) { best = cost; m = kChunkCand[c]; }
  }
  for (int e = threadIdx.x; e < E; e += blockDim.x) nch[e] = (tot[e] + m - 1) / m;
  __syncthreads();
  if (warp == 0) {  // exclusive scans of the rows and the chunks, 32 experts at a time (E % 32 == 0)
    int run = 0, run_c = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int v = tot[e0 + lane], vc = nch[e0 + lane];
      int x = v, xc = vc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o), yc = __shfl_up_sync(0xffffffffu, xc, o);
        if (lane >= o) { x += y; xc += yc; }
      }
      counts[e0 + lane] = v;
      offsets[e0 + lane] = run + x - v;
      first[e0 + lane] = run + x - v;
      ch0[e0 + lane] = run_c + xc - vc;
      run += __shfl_sync(0xffffffffu, x, 31);
      run_c += __shfl_sync(0xffffffffu, xc, 31);
    }
    if (lane == 0) *n_chunks = run_c;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = tot[e], n = nch[e];
    int row = first[e];
    for (int i = 0; i < n; ++i) {
      const int rows = c / n + (i < c % n ? 1 : 0);
      chunks[ch0[e] + i] = make_int4(e, row, rows, 0);
      row += rows;
    }
  }
  for (int p0 = p_lo; p0 < p_hi; p0 += 32) {
    const int p = p0 + lane;
    int id = p < p_hi ? topk_id[p] : -1;
    if (id >= E) id = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, id);
    const int before = id >= 0 ? cnt[warp][id] : 0;
    __syncwarp();
    if (id >= 0) {
      const int pos = first[id] + before + __popc(peers & ((1u << lane) - 1u));
      pos_of[p] = pos;
      pair_token[pos] = p / k;
      if (lane == __ffs(peers) - 1) cnt[warp][id] = before + __popc(peers);
    }
    __syncwarp();
  }
}

// grid: P; block 128: row pos of xp <- row pair_token[pos] of x (d / 8 uint4 per row)
__global__ void __launch_bounds__(128) moe_gather_kernel(const df_bf16* __restrict__ x, int d, int R,
                                                         const int32_t* __restrict__ pair_token,
                                                         df_bf16* __restrict__ xp, int* status) {
  pdl_wait();
  pdl_trigger();
  const int pos = blockIdx.x;
  const int t = pair_token[pos];
  if (!DF_IN_BOUNDS(t >= 0 && t < R, status, 50)) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d);
  uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)pos * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = src[i];
}

// ------------------------------------------------------------------------- grouped GEMM
struct MoeGemmParams {
  int n_wt, k_iters;        // items: n_chunks x n_wt (feature tiles innermost)
  const int4* chunks;       // {expert, first expert-ordered row, rows, 0}
  const int32_t* n_chunks;
  int Fe, d;
  df_bf16* act;             // gate/up: [P][Fe]
  float* out;               // down: [P][d]
  int* status;
};

template <int MODE>
__global__ void __launch_bounds__(kMoeThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const MoeGemmParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int S = kMoeSlots;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kMoeRing);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = bars + 2 * S + 2;
  uint64_t* mma_drain = bars + 2 * S + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  uint32_t* slot_off = reinterpret_cast<uint32_t*>(bars + 2 * S + 6);  // [S] ring offset of each k-step
  float* xbuf = reinterpret_cast<float*>(bars + 2 * S + 6 + S / 2);   // gate/up epilogue: up values

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&tfull[i], 1); mbar_init(&tempty[i], 128); }
    mbar_init(mma_drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, 2 * kMoeChunk); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the chunk list and the expert-ordered rows come from the previous kernels
  pdl_trigger();
  const int n_items = *p.n_chunks * p.n_wt;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp keeps the ring's books in lockstep (waits end in warp votes), one
    // elected lane issuing the copies.
    const bool leader = elect_one();
    const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
    uint32_t head = 0, used = 0;  // next free byte of the ring; bytes held by k-steps in flight
    uint32_t held[S];             // bytes each slot holds (a wrapped k-step also holds the skipped tail)
    long long issued = 0, released = 0;
    bool ok = true;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int4 ch = p.chunks[it / p.n_wt];
      const int wt = it % p.n_wt, nbox = (ch.z + 63) >> 6;
      const uint32_t need = kMoeWBytes + nbox * kMoeXBox;
      for (int k = 0; k < p.k_iters; ++k) {
        uint32_t start = head, take = need;
        if (head + need > kMoeRing) { start = 0; take = kMoeRing - head + need; }
        // the oldest k-steps give their bytes back until this one fits and a slot is free
        while (used + take > kMoeRing || issued - released == S) {
          const int so = (int)(released % S);
          if (!__all_sync(0xffffffffu, mbar_wait(&empty[so], (uint32_t)((released / S) & 1), p.status, 21))) { ok = false; break; }
          used -= held[so];
          ++released;
        }
        if (!ok) break;
        const int sl = (int)(issued % S);
        held[sl] = take;
        used += take;
        head = start + need;
        if (leader) {
          slot_off[sl] = start;
          unsigned char* sb = smem + start;
          mbar_arrive_expect_tx(&full[sl], need);
          if (MODE == kMoeGateUp) {
            const int g0 = ch.x * 2 * p.Fe + wt * 64;  // 64 gate rows, then the matching 64 up rows
            tma_load_2d(sb, &tmW, &full[sl], k * kMoeBK, g0, pol_w);
            tma_load_2d(sb + kMoeWBytes / 2, &tmW, &full[sl], k * kMoeBK, g0 + p.Fe, pol_w);
          } else {
            tma_load_2d(sb, &tmW, &full[sl], k * kMoeBK, ch.x * p.d + wt * 128, pol_w);
          }
          for (int j = 0; j < nbox; ++j)
            tma_load_2d(sb + kMoeWBytes + j * kMoeXBox, &tmX, &full[sl], k * kMoeBK, ch.y + 64 * j, pol_x);
        }
        __syncwarp();
        ++issued;
      }
    }
    // every load issued has landed before the CTA may exit (bounded waits)
    if (leader)
      for (long long g = issued - S > released ? issued - S : released; g < issued; ++g)
        mbar_wait(&full[g % S], (uint32_t)((g / S) & 1), nullptr, 0);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp walks the k-steps in lockstep (every wait ends in a warp vote), so the
    // operand descriptors are warp-uniform values; one elected lane issues the MMAs and
    // their commits.
    const bool leader = elect_one();
    long long g = 0;  // k-steps consumed
    int si = 0;
    bool ok = true, issued_any = false;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int4 ch = p.chunks[it / p.n_wt];
      const uint32_t idesc = idesc_bf16_f32(128, (ch.z + 15) & ~15);
      const int acc = si & 1, use = si >> 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], (use & 1) ^ 1, p.status, 22))) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * kMoeChunk;
      for (int k = 0; k < p.k_iters; ++k, ++g) {
        const int sl = (int)(g % S);
        if (!__all_sync(0xffffffffu, mbar_wait(&full[sl], (uint32_t)((g / S) & 1), p.status, 23))) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + slot_off[sl]);
        const uint64_t adesc = sdesc_kmajor_sw128(sa), bdesc = sdesc_kmajor_sw128(sa + kMoeWBytes);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kMoeBK / 16; ++kk)
            mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, (k > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[sl]);
        }
        __syncwarp();
        issued_any = true;
      }
      if (!ok) break;
      if (leader) mma_commit(&tfull[acc]);
      __syncwarp();
      ++si;
    }
    if (issued_any && !ok) {
      // giving up: the MMAs already issued must finish before TMEM is freed
      if (leader) mma_commit(mma_drain);
      __syncwarp();
      mbar_wait(mma_drain, 0, nullptr, 0);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3;      // TMEM lane quarter: weight rows 32 q .. 32 q + 31
    const int r = q * 32 + lane;
    int si = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      const int4 ch = p.chunks[it / p.n_wt];
      const int wt = it % p.n_wt;
      const int acc = si & 1, use = si >> 1;
      // the four epilogue warps leave together (they meet at named barriers below)
      const bool ok = mbar_wait(&tfull[acc], use & 1, p.status, 24);
      uint32_t all_ok;
      asm volatile("{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.and.pred b, 1, 128, a;\n"
                   " selp.u32 %0, 1, 0, b;\n}" : "=r"(all_ok) : "r"((uint32_t)ok) : "memory");
      if (!all_ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * kMoeChunk;
      for (int c0 = 0; c0 < ch.z; c0 += 32) {  // 32 token columns at a time
        float v[32];
        tmem_ld16(taddr + c0, v);
        tmem_ld16(taddr + c0 + 16, v + 16);
        tmem_ld_wait();
        const int nc = min(32, ch.z - c0);
        const size_t row0 = (size_t)ch.y + c0;
        if (MODE == kMoeGateUp) {
          // weight rows 0..63: gate of features 64 wt + r; rows 64..127: the matching up
          asm volatile("bar.sync 1, 128;" ::: "memory");  // the previous columns' readers are done
          if (r >= 64)
#pragma unroll
            for (int c = 0; c < 32; ++c) xbuf[(r - 64) * kMoeXPitch + c] = v[c];
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (r < 64) {
            df_bf16* dst = p.act + row0 * p.Fe + wt * 64 + r;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              if (c < nc) {
                const float g = v[c], u = xbuf[r * kMoeXPitch + c];
                dst[(size_t)c * p.Fe] = f_to_bf16(g / (1.f + __expf(-g)) * u);
              }
            }
          }
        } else {
          float* dst = p.out + row0 * p.d + wt * 128 + r;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c < nc) dst[(size_t)c * p.d] = v[c];
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);  // all of this accumulator's columns are read
      ++si;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, 2 * kMoeChunk);
  }
}

// ----------------------------------------------------------------------------- combine
// grid: output rows; block d / 8 threads (two float4 each), d a multiple of 256, <= 8192.
// The row's k (weight, expert-ordered row) pairs are staged in shared memory first, so the
// expert outputs' loads of several choices are in flight together.
__global__ void __launch_bounds__(1024) moe_combine_kernel(ResNormArgs a, const float* __restrict__ out,
                                                           const float* __restrict__ topk_w,
                                                           const int32_t* __restrict__ pos_of, int k, int P,
                                                           int* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  __shared__ float w_sh[32];
  __shared__ int pos_sh[32];
  const int o = blockIdx.x;
  const int t = (o / a.group_out) * a.group_in + a.in_off + (o % a.group_out);
  if (threadIdx.x < k) {
    const int pos = pos_of[(size_t)t * k + threadIdx.x];
    const bool ok = DF_IN_BOUNDS(pos >= 0 && pos < P, status, 51);
    w_sh[threadIdx.x] = ok ? topk_w[(size_t)t * k + threadIdx.x] : 0.f;
    pos_sh[threadIdx.x] = ok ? pos : 0;
  }
  __syncthreads();
  const int per = blockDim.x * 4;
  const int n_[2] = {(int)threadIdx.x * 4, per + (int)threadIdx.x * 4};
  float4 v[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
#pragma unroll 4
  for (int j = 0; j < k; ++j) {  // choices in order: a fixed summation order
    const float w = w_sh[j];
    const float* row = out + (size_t)pos_sh[j] * a.d;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if (n_[i] >= a.d) continue;
      const float4 e = __ldcg(reinterpret_cast<const float4*>(row + n_[i]));
      v[i].x += w * e.x; v[i].y += w * e.y; v[i].z += w * e.z; v[i].w += w * e.w;
    }
  }
  float ss = 0.f;
  float* hrow = a.h + (size_t)t * a.d;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (n_[i] >= a.d) continue;
    const float4 hv = *reinterpret_cast<const float4*>(hrow + n_[i]);
    float4& y = v[i];
    y.x += hv.x; y.y += hv.y; y.z += hv.z; y.w += hv.w;
    *reinterpret_cast<float4*>(hrow + n_[i]) = y;
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

// ----------------------------------------------------------------------------- host
// chunks of at least 64 rows (the smallest chunk size the dispatch chooses): sum over the
// experts of ceil(c_e / 64) <= E + R k / 64
int moe_max_chunks(int R, int k, int E) { return E + R * k / 64 + 1; }

size_t moe_buf_elems(int R, int k, int E, int d, int Fe, size_t* sz) {
  const size_t P = (size_t)R * k;
  sz[0] = P * 4;            // topk_id
  sz[1] = P * 4;            // topk_w
  sz[2] = (size_t)E * 4;    // counts
  sz[3] = (size_t)E * 4;    // offsets
  sz[4] = P * 4;            // pos_of
  sz[5] = P * 4;            // pair_token
  sz[6] = P * d * 2;        // xp
  sz[7] = P * Fe * 2;       // act
  sz[8] = P * d * 4;        // out
  sz[9] = (size_t)moe_max_chunks(R, k, E) * 16;  // chunks
  sz[10] = 16;              // n_chunks
  size_t t = 0;
  for (int i = 0; i < kMoeBufCount; ++i) t += sz[i];
  return t;
}

int launch_moe_route(const PartialView& pv, int R, int E, int k, MoeBufs& m, int* status, cudaStream_t st) {
  if (E % 32 || E > 256 || k < 1 || k > 32 || k > E) return DF_ERR_SHAPE;
  DF_TRACE("moe_route", st);
  launch_k(moe_route_kernel, dim3((R + 7) / 8), dim3(256), 0, st, pv, R, E, k, m.topk_id, m.topk_w, status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_moe_dispatch(const df_bf16* x, int R, int d, int E, int k, int Fe, MoeBufs& m, int* status,
                        cudaStream_t st) {
  DF_TRACE("moe_dispatch", st);
  const int P = R * k;
  launch_k(moe_permute_kernel, dim3(1), dim3(kPermWarps * 32), 0, st, P, E, k, m.topk_id, m.counts, m.offsets,
           m.pos_of, m.pair_token, m.chunks, m.n_chunks, Fe / 64, num_sms());
  launch_k(moe_gather_kernel, dim3(P), dim3(128), 0, st, x, d, R, m.pair_token, m.xp, status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_moe_experts(const df_bf16* w_gate_up, const df_bf16* w_down, int R, int d, int E, int k, int Fe,
                       MoeBufs& m, int* status, cudaStream_t st) {
  if (Fe % 64 || d % 128) return DF_ERR_SHAPE;
  const int P = R * k;
  const size_t smem = 1024 + kMoeRing + (2 * kMoeSlots + 6 + kMoeSlots / 2) * 8 + 64 * kMoeXPitch * 4;
  if (ensure_dynamic_smem(moe_gemm_kernel<kMoeGateUp>, smem) != cudaSuccess ||
      ensure_dynamic_smem(moe_gemm_kernel<kMoeDown>, smem) != cudaSuccess)
    return DF_ERR_CUDA;
  CUtensorMap tw1, tx1, tw2, tx2;
  // gate/up: stacked [E * 2 Fe][d] weights in 64-row boxes; token rows xp [P][d] in 64-row boxes
  if (make_tmap_2d(&tw1, w_gate_up, (long long)E * 2 * Fe, d, d, 64) || make_tmap_2d(&tx1, m.xp, P, d, d, 64))
    return DF_ERR_CUDA;
  // down: stacked [E * d][Fe] weights in 128-row boxes; token rows act [P][Fe]
  if (make_tmap_2d(&tw2, w_down, (long long)E * d, Fe, Fe, 128) || make_tmap_2d(&tx2, m.act, P, Fe, Fe, 64))
    return DF_ERR_CUDA;
  MoeGemmParams p{};
  p.chunks = m.chunks;
  p.n_chunks = m.n_chunks;
  p.Fe = Fe;
  p.d = d;
  p.act = m.act;
  p.out = m.out;
  p.status = status;
  const int grid = num_sms();
  {
    DF_TRACE("moe_gemm_gate_up", st);
    p.n_wt = Fe / 64;
    p.k_iters = d / kMoeBK;
    launch_k(moe_gemm_kernel<kMoeGateUp>, dim3(grid), dim3(kMoeThreads), smem, st, tw1, tx1, p);
  }
  {
    DF_TRACE("moe_gemm_down", st);
    p.n_wt = d / 128;
    p.k_iters = Fe / kMoeBK;
    launch_k(moe_gemm_kernel<kMoeDown>, dim3(grid), dim3(kMoeThreads), smem, st, tw2, tx2, p);
  }
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

int launch_moe_combine(const MoeBufs& m, int k, int P, const ResNormArgs& a, int* status, cudaStream_t st) {
  if (a.rows <= 0) return DF_OK;
  if (a.d % 256 || a.d > 8192 || !a.h) return DF_ERR_SHAPE;
  DF_TRACE("moe_combine", st);
  launch_k(moe_combine_kernel, dim3(a.rows), dim3(a.d / 8), 0, st, a, m.out, m.topk_w, m.pos_of, k, P, status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace df
