// Weight-streaming GEMM on 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
//   out[t][n] (+)= sum_k X[t][k] * W[n][k]        X: [M tokens][K] bf16, W: [N][K] bf16
//
// The token count is small in every projection of the speculative step (16 to a few
// hundred rows per sequence) while the weights are large, so the kernel is organised
// around streaming W exactly once from HBM:
//   * swap-AB: the MMA's 128-row A operand is a 128-row slice of W and the token tile is
//     the MMA's N dimension (16..256, a multiple of 16), so a 16-token drafter GEMM still
//     runs full-width tensor instructions;
//   * persistent CTAs (one per SM) split the (tile, k-block) iteration space evenly
//     ("stream-K"), so the grid stays full however few 128-row weight tiles there are;
//   * warp roles: warp 0 issues TMA loads into a multi-stage shared-memory ring (a stage
//     = one 128 x 64 weight tile + the token rows' 64-wide k-slice), warp 1 owns the TMEM
//     allocation and one lane issues tcgen05.mma, warps 2-5 drain the TMEM accumulators
//     (double-buffered when two fit in 512 columns) and write the epilogue;
//   * epilogues: partial slots (each CTA stores every tile piece it computed to a slot of
//     its own and lists it for the tile; the next kernel sums a tile's pieces in a fixed
//     order, so results are deterministic with no atomics; see partials.cuh), fp32
//     reduction-add or store (whole tiles), or fused argmax over the output features
//     (whole tiles; the target LM head writes no logits).
// Every mbarrier wait is bounded (common.cuh); a timeout is recorded in the status word.
#include <stdio.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "common.cuh"
#include "gemm.h"
#include "partials.cuh"
#include "runtime.h"
#include "trace.h"

namespace df {

constexpr int kGemmThreads = 192;
constexpr int kBM = 128;  // weight rows per tile (MMA M)
constexpr int kBK = 64;   // k per stage (one 128-byte swizzle row)
constexpr int kArgChunks = 16;  // argmax epilogue: running maxima of up to 16 x 32 token columns
constexpr int kMaxGrid = 192;   // CTAs a launch may use (iteration ranges passed as parameters)
#ifndef DF_GEMM_DRAIN_DELTA
#define DF_GEMM_DRAIN_DELTA -1
#endif
constexpr int kDrainDelta = DF_GEMM_DRAIN_DELTA;  // drain cost in k-steps (-1: BN / 64 when not double-buffered)

struct GemmParams {
  int M, N, K;
  int n_ttiles, BN, k_iters;
  int sub0, sub1;   // token tile = two MMA widths (sub1 = 0 when BN <= 256)
  int nbuf;         // TMEM accumulator buffers (2 when 2*BN fits in 512 columns)
  int w_keep;       // 1: weights are re-read by later token tiles (keep them in L2)
  long long total_iters;
  int whole_tiles;  // 1: each CTA owns whole tiles (store / argmax epilogues)
  float* out;
  int ldo;
  unsigned long long* amax;  // argmax keys [M]
  const uint32_t* draw_key;  // argmax: per-token draw keys, or NULL (greedy)
  float inv_temp;
  float* part;               // kGemmPartial: [G * max_seg][BN][128] fp32 slots
  int* meta;                 // kGemmPartial: [tiles][meta_stride] piece count, then slots in CTA order
  int meta_stride;
  int max_seg;
  float2* stats;             // kGemmStore: optional per (token, weight tile, warp) (max, sum exp(x - max))
  int n_stats;               // = 4 * number of weight tiles
  int* status;
  int stages;
  int starts[kMaxGrid + 1];  // CTA c owns iterations [starts[c], starts[c + 1])
};

struct Segment {
  long long tile;
  int k0, k1;
};

// Iteration range of CTA c (chosen on the host, see gemm_partition) and its decomposition
// into per-tile segments.
DF_DEV void cta_range(const GemmParams& p, long long& it0, long long& it1) {
  it0 = p.starts[blockIdx.x];
  it1 = p.starts[blockIdx.x + 1];
}
// The CTA whose range holds iteration `it` (the ranges are contiguous and ascending).
DF_DEV int cta_of(const GemmParams& p, long long it) {
  int lo = 0, hi = (int)gridDim.x - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.starts[mid] <= it) lo = mid; else hi = mid - 1;
  }
  return lo;
}
DF_DEV bool next_segment(const GemmParams& p, long long& it, long long it1, Segment& s) {
  if (it >= it1) return false;
  s.tile = it / p.k_iters;
  s.k0 = (int)(it - s.tile * p.k_iters);
  const long long tile_end = (s.tile + 1) * p.k_iters;
  const long long e = tile_end < it1 ? tile_end : it1;
  s.k1 = s.k0 + (int)(e - it);
  it = e;
  return true;
}

// Argmax epilogue.  Keys are (order-preserving float bits << 32) | ~row, so the maximum
// key is the largest value and, among equal values, the lowest row (token id).
//
// argmax_tile: for every token column of the tile, the maximum key over this warp's 32
// rows, folded into the warp's running maxima (shared memory, run[chunk * 32 + lane]).
// 32 columns at a time: a transposing butterfly (offsets 16, 8, 4, 2, 1) halves the
// columns each lane holds while taking maxima, so lane L ends with column L after 31
// exchanges instead of 5 per column.
// DRAW: the keys are of value * inv_temp + draw_noise(key of the column's token, row), the
// product and the sum rounded separately (no fused multiply-add), so that a temperature
// draw is the argmax the same way; dk = the tile's per-column draw keys, nk columns valid.
template <bool DRAW>
DF_DEV void argmax_tile(uint32_t taddr, int BN, int n, bool n_ok, unsigned long long* run, int lane,
                        const uint32_t* dk = nullptr, int nk = 0, float inv_temp = 1.f) {
  for (int c0 = 0; c0 < BN; c0 += 32) {
    float v[32];
    tmem_ld16(taddr + c0, v);
    const bool two = c0 + 16 < BN;  // BN is a multiple of 16; never read past the tile
    if (two) tmem_ld16(taddr + c0 + 16, v + 16);
    tmem_ld_wait();
    if constexpr (DRAW) {
      const uint32_t mine = c0 + lane < nk ? dk[c0 + lane] : 0u;  // lane j: column c0 + j's key
#pragma unroll
      for (int j = 0; j < 32; ++j)
        v[j] = __fadd_rn(__fmul_rn(v[j], inv_temp), draw_noise(__shfl_sync(0xffffffffu, mine, j), n));
    }
    unsigned long long k[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
      k[j] = (n_ok && (j < 16 || two)) ? (((unsigned long long)float_key(v[j]) << 32) | (uint32_t)(~(uint32_t)n)) : 0ull;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const bool hi = (lane & off) != 0;  // keep the upper half of the current columns
#pragma unroll
      for (int i = 0; i < off; ++i) {
        const unsigned long long keep = hi ? k[i + off] : k[i];
        const unsigned long long send = hi ? k[i] : k[i + off];
        const unsigned long long got = __shfl_xor_sync(0xffffffffu, send, off);
        k[i] = keep > got ? keep : got;
      }
    }
    unsigned long long& r = run[(c0 >> 5) * 32 + lane];
    if (k[0] > r) r = k[0];
  }
}

// Publishes the running maxima of token tile tt (one atomic per column) and clears them.
template <class P>
DF_DEV void argmax_flush(const P& p, unsigned long long* run, int tt, int lane) {
  for (int c = 0; c * 32 < p.BN; ++c) {
    const int col = c * 32 + lane, t = tt * p.BN + col;
    unsigned long long& r = run[c * 32 + lane];
    if (col < p.BN && t < p.M && r) atomicMax(p.amax + t, r);
    r = 0ull;
  }
}

// MODE is the epilogue (GemmMode): one instantiation per epilogue keeps each kernel's code
// small and free of per-element mode branches.
template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmX1, const GemmParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = p.BN, S = p.stages;
  const uint32_t w_bytes = kBM * kBK * 2, x_bytes = (uint32_t)BN * kBK * 2;
  const uint32_t stage_bytes = w_bytes + x_bytes;  // multiple of 1024 (BN multiple of 16... see host)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * stage_bytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = bars + 2 * S + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
  uint64_t* mma_drain = bars + 2 * S + 5;  // completion of every MMA issued, when the issuer gives up
  // argmax epilogue: per warp, per 32-column chunk, per lane (= column) running maximum key
  unsigned long long* run_max = reinterpret_cast<unsigned long long*>(bars + 2 * S + 6);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int acc_cols = p.nbuf * BN;
  const uint32_t tmem_cols = acc_cols <= 32 ? 32 : acc_cols <= 64 ? 64 : acc_cols <= 128 ? 128 : acc_cols <= 256 ? 256 : 512;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&tfull[i], 1); mbar_init(&tempty[i], 128); }
    mbar_init(mma_drain, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    if (p.sub1) tma_prefetch_desc(&tmX1);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, tmem_cols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  long long it0, it1;
  cta_range(p, it0, it1);
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    // The whole warp walks the k-steps in lockstep (waits end in warp votes), one elected
    // lane issuing the copies; the (weight tile, token tile, k) coordinates advance
    // incrementally from the range's first k-step.
    const bool leader = elect_one();
    const uint64_t pol_w = p.w_keep ? policy_evict_last() : policy_evict_first(), pol_x = policy_evict_last();
    const long long n = it1 - it0;
    struct Pos {
      int wt, tt, k;
    };
    Pos pos0;
    {
      const long long tile = it0 / p.k_iters;
      pos0.k = (int)(it0 - tile * p.k_iters);
      pos0.wt = (int)(tile / p.n_ttiles);
      pos0.tt = (int)(tile % p.n_ttiles);
    }
    auto advance = [&](Pos& q) {
      if (++q.k == p.k_iters) {
        q.k = 0;
        if (++q.tt == p.n_ttiles) { q.tt = 0; ++q.wt; }
      }
    };
    auto load_x = [&](int st, const Pos& q) {
      unsigned char* xb = smem + (size_t)st * stage_bytes + w_bytes;
      tma_load_2d(xb, &tmX, &full[st], q.k * kBK, q.tt * BN, pol_x);
      if (p.sub1) tma_load_2d(xb + p.sub0 * 128, &tmX1, &full[st], q.k * kBK, q.tt * BN + p.sub0, pol_x);
    };
    // Weights are constant: the first ring's worth of weight tiles is requested before the
    // previous kernel has finished.  Each stage's transaction count covers both halves, so
    // it completes only once its token rows (loaded after the wait) have arrived too.
    const int npre = (int)(n < S ? n : S);
    Pos q = pos0;
    for (int i = 0; i < npre; ++i, advance(q)) {
      if (leader) {
        mbar_arrive_expect_tx(&full[i], stage_bytes);
        tma_load_2d(smem + (size_t)i * stage_bytes, &tmW, &full[i], q.k * kBK, q.wt * kBM, pol_w);
      }
    }
    pdl_wait();  // token rows are the previous kernel's output
    q = pos0;
    for (int i = 0; i < npre; ++i, advance(q))
      if (leader) load_x(i, q);
    int stage = npre % S;
    uint32_t phase = npre == S ? 1u : 0u;
    long long issued = npre;
    for (long long i = npre; i < n; ++i, advance(q)) {
      if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], phase ^ 1, p.status, 1))) break;
      if (leader) {
        mbar_arrive_expect_tx(&full[stage], stage_bytes);
        tma_load_2d(smem + (size_t)stage * stage_bytes, &tmW, &full[stage], q.k * kBK, q.wt * kBM, pol_w);
        load_x(stage, q);
      }
      __syncwarp();
      ++issued;
      if (++stage == S) { stage = 0; phase ^= 1; }
    }
    if (leader) {
      // Drain: every load issued must have landed before the CTA may exit, also when the MMA
      // issuer gave up before consuming it (bounded waits; already complete in normal runs).
      const long long m = issued < S ? issued : S;
      int st = stage;
      uint32_t ph = phase;
      for (long long i = 0; i < m; ++i) {
        if (--st < 0) { st = S - 1; ph ^= 1; }
        mbar_wait(&full[st], ph, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp walks the stages in lockstep (every wait ends in a warp vote), so the
    // operand descriptors are warp-uniform values; one elected lane issues the MMAs and
    // their commits.
    const uint32_t idesc0 = idesc_bf16_f32(kBM, p.sub0);
    const uint32_t idesc1 = idesc_bf16_f32(kBM, p.sub1 ? p.sub1 : 16);
    const bool leader = elect_one();
    int stage = 0;
    uint32_t phase = 0;
    long long it = it0;
    Segment sg;
    int si = 0;
    // failure-path test hook: with the header's hold word set, issue no MMA and give up (the
    // producer then finds no stage released, times out and drains its loads)
    bool ok = __all_sync(0xffffffffu, !leader || wait_hold_clear(p.status, 5)), issued_any = false;
    while (ok && next_segment(p, it, it1, sg)) {
      const int acc = si % p.nbuf, use = si / p.nbuf;
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], (use & 1) ^ 1, p.status, 2))) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int k = sg.k0; k < sg.k1; ++k) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, p.status, 3))) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + (size_t)stage * stage_bytes);
        const uint64_t adesc = sdesc_kmajor_sw128(sa);
        const uint64_t bdesc = sdesc_kmajor_sw128(sa + w_bytes);
        const uint64_t bdesc1 = sdesc_kmajor_sw128(sa + w_bytes + p.sub0 * 128);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t accum = (k > sg.k0 || kk > 0) ? 1u : 0u;
            mma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc0, accum);
            if (p.sub1) mma_bf16(d_tmem + p.sub0, adesc + 2 * kk, bdesc1 + 2 * kk, idesc1, accum);
          }
          mma_commit(&empty[stage]);
        }
        __syncwarp();
        issued_any = true;
        if (++stage == S) { stage = 0; phase ^= 1; }
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
    // Partial slots and outputs may still be read by the previous kernel: wait for it.
    pdl_wait();
    pdl_trigger();
    if (MODE == kGemmPartial && threadIdx.x == 64 && it1 > it0) {
      // Register this CTA's segments in the per-tile slot lists.  The CTA's place among a
      // tile's contributors is its distance from the CTA that owns the tile's first k-step.
      const long long k = p.k_iters;
      const long long t_first = it0 / k, t_last = (it1 - 1) / k;
      for (long long t = t_first; t <= t_last; ++t) {
        int pos = 0;
        if (t * k < it0) pos = (int)blockIdx.x - cta_of(p, t * k);  // CTA holding iteration t*k is first
        p.meta[t * p.meta_stride + 1 + pos] = (int)(blockIdx.x * p.max_seg + (t - t_first));
        if ((t + 1) * k <= it1) p.meta[t * p.meta_stride] = pos + 1;  // this CTA holds the tile's last k-step
      }
    }
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    unsigned long long* run = run_max + (size_t)(warp - 2) * kArgChunks * 32;
    int run_tt = 0;
    if constexpr (MODE == kGemmArgmax) {
      for (int i = lane; i < kArgChunks * 32; i += 32) run[i] = 0ull;
      __syncwarp();
    }
    long long it = it0;
    Segment sg;
    int si = 0;
    while (next_segment(p, it, it1, sg)) {
      const int acc = si % p.nbuf, use = si / p.nbuf;
      // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], use & 1, p.status, 4))) break;
      tc_fence_after();
      const int wt = (int)(sg.tile / p.n_ttiles), tt = (int)(sg.tile % p.n_ttiles);
      const int n = wt * kBM + q * 32 + lane;
      const bool n_ok = n < p.N;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if constexpr (MODE == kGemmArgmax) {
        if (tt != run_tt) {  // a new token tile: publish the finished one's maxima
          argmax_flush(p, run, run_tt, lane);
          run_tt = tt;
        }
        if (p.draw_key)
          argmax_tile<true>(taddr, BN, n, n_ok, run, lane, p.draw_key + (size_t)tt * BN, p.M - tt * BN, p.inv_temp);
        else
          argmax_tile<false>(taddr, BN, n, n_ok, run, lane);
      } else if constexpr (MODE == kGemmPartial) {
        // this segment's accumulator -> its slot, [token][feature row], plain stores; 64
        // columns per TMEM round trip, then 16 at a time for the rest
        float* dst = p.part + ((size_t)blockIdx.x * p.max_seg + si) * BN * 128 + q * 32 + lane;
        int c0 = 0;
        for (; c0 + 64 <= BN; c0 += 64) {
          float v[64];
#pragma unroll
          for (int c = 0; c < 64; c += 16) tmem_ld16(taddr + c0 + c, v + c);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 64; ++j) dst[(size_t)(c0 + j) * 128] = v[j];
        }
        for (; c0 < BN; c0 += 16) {
          float v[16];
          tmem_ld16(taddr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) dst[(size_t)(c0 + j) * 128] = v[j];
        }
      } else
      for (int c0 = 0; c0 < BN; c0 += 16) {
        float v[16];
        tmem_ld16(taddr + c0, v);
        tmem_ld_wait();
        const int t0 = tt * BN + c0;
        if constexpr (MODE == kGemmAtomicAdd) {
          if (n_ok)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (t0 + j < p.M) atomicAdd(p.out + (size_t)(t0 + j) * p.ldo + n, v[j]);
        } else if constexpr (MODE == kGemmStore) {
          if (n_ok)
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (t0 + j < p.M) p.out[(size_t)(t0 + j) * p.ldo + n] = v[j];
          if (p.stats) {
            // softmax statistics of this warp's 32 output rows, per token column
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float x = n_ok ? v[j] : -INFINITY;
              const float m = warp_max(x);
              const float e = (m == -INFINITY) ? 0.f : warp_sum(__expf(x - m));
              if (lane == j && t0 + j < p.M)
                p.stats[(size_t)(t0 + j) * p.n_stats + wt * 4 + q] = make_float2(m, e);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      ++si;
    }
    if constexpr (MODE == kGemmArgmax) argmax_flush(p, run, run_tt, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// ----------------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Encodes (and caches) a 2D bf16 tensor map: `rows` x `cols` (cols contiguous, row
// stride `ld` elements), box = box_rows x 64 columns, 128-byte swizzle.
int make_tmap_2d(CUtensorMap* out, const void* ptr, long long rows, long long cols, long long ld, int box_rows) {
  struct Key {
    const void* p; long long r, c, ld; int b;
    bool operator==(const Key& o) const { return p == o.p && r == o.r && c == o.c && ld == o.ld && b == o.b; }
  };
  struct H {
    size_t operator()(const Key& k) const {
      return std::hash<const void*>()(k.p) ^ (std::hash<long long>()(k.r * 1315423911ll + k.c * 2654435761ll + k.ld) << 1) ^ k.b;
    }
  };
  static std::mutex mu;
  static std::unordered_map<Key, CUtensorMap, H> cache;
  const Key key{ptr, rows, cols, ld, box_rows};
  {
    std::lock_guard<std::mutex> g(mu);
    auto itc = cache.find(key);
    if (itc != cache.end()) { *out = itc->second; return DF_OK; }
  }
  EncodeTiledFn enc = get_encode();
  if (!enc) return DF_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return DF_ERR_CUDA;
  {
    std::lock_guard<std::mutex> g(mu);
    if (cache.size() > 4096) cache.clear();
    cache.emplace(key, m);
  }
  *out = m;
  return DF_OK;
}

// Token tile.  Up to 512 tokens form one tile (two MMAs of N <= 256 per k-step, one
// TMEM buffer), so every weight k-chunk is streamed once; beyond that, equal tiles of at
// most 256 (double-buffered TMEM) with the weights kept in L2 for the later tiles.
int gemm_token_tile(int M) {
  if (M <= 512) return (M + 15) / 16 * 16;
  const int nt = (M + 255) / 256;
  int bn = (M + nt - 1) / nt;
  return (bn + 15) / 16 * 16;
}

// Split of a launch's iteration space over its CTAs.
//
// Whole-tile epilogues: tiles spread evenly.  Partial-tile epilogue (stream-K): contiguous
// iteration ranges of equal *cost*, where a range that crosses a tile boundary is charged
// `delta` extra iterations per crossing when the accumulator is not double-buffered (its MMA
// waits for the previous tile's drain; delta = the drain time in k-steps, about BN / 64).
// The smallest feasible maximum cost is found by bisection with a greedy fill; CTAs left
// without work are not launched.
struct Partition {
  int G;                      // CTAs launched
  int starts[kMaxGrid + 1];
  int max_seg, maxc;          // most segments of one CTA, most pieces of one tile
};

static void make_partition(long long total, long long k_iters, int G, bool whole_tiles, int delta, Partition& P) {
  P.G = 0;
  if (whole_tiles) {
    const long long tiles = total / k_iters;
    for (int c = 0; c <= G; ++c) P.starts[c] = (int)((tiles * c / G) * k_iters);
    P.G = G;
  } else {
    // furthest end of a range that starts at s and may cost C
    auto reach = [&](long long s, long long C) {
      long long end = s, budget = C;
      while (end < total) {
        const long long lim = std::min((end / k_iters + 1) * k_iters, total);
        if (end + budget <= lim) return end + budget;
        budget -= lim - end;
        end = lim;
        if (end >= total) break;
        budget -= delta;  // going on past a tile boundary costs a drain
        if (budget <= 0) break;
      }
      return end;
    };
    auto ranges = [&](long long C) {  // greedy fill: ranges needed at cost C (G + 1 = too many)
      int n = 0;
      for (long long s = 0; s < total;) {
        const long long e = reach(s, C);
        if (e <= s || ++n > G) return G + 1;
        s = e;
      }
      return n;
    };
    long long lo = (total + G - 1) / G, hi = lo;
    while (ranges(hi) > G) hi *= 2;
    while (lo < hi) {
      const long long mid = (lo + hi) / 2;
      if (ranges(mid) <= G) hi = mid; else lo = mid + 1;
    }
    long long s = 0;
    P.starts[0] = 0;
    while (s < total) {
      s = reach(s, lo);
      P.starts[++P.G] = (int)s;
    }
  }
  P.max_seg = 1;
  P.maxc = 1;
  std::vector<int> pieces(total / k_iters, 0);
  for (int c = 0; c < P.G; ++c) {
    if (P.starts[c + 1] <= P.starts[c]) continue;
    const long long t0 = P.starts[c] / k_iters, t1 = (P.starts[c + 1] - 1) / k_iters;
    P.max_seg = std::max(P.max_seg, (int)(t1 - t0 + 1));
    for (long long t = t0; t <= t1; ++t) P.maxc = std::max(P.maxc, ++pieces[t]);
  }
}

// The partition of a launch of this shape (cached: it depends on the shape and the SM count only).
static const Partition& gemm_partition(int M, int N, int K, bool whole_tiles, int min_k_per_cta = 0) {
  const int BN = gemm_token_tile(M);
  const long long n_tt = (M + BN - 1) / BN, k_iters = K / kBK;
  const long long tiles = (long long)((N + kBM - 1) / kBM) * n_tt;
  const long long total = tiles * k_iters;
  long long G = std::min<long long>(num_sms(), kMaxGrid);
  G = std::min(G, whole_tiles ? tiles : total);
  if (!whole_tiles && min_k_per_cta > 1) G = std::max(1LL, std::min(G, total / min_k_per_cta));
  const int nbuf = 2 * BN <= 512 ? 2 : 1;
  const int delta = kDrainDelta >= 0 ? kDrainDelta : (nbuf == 2 ? 0 : (BN + 63) / 64);
  static std::mutex mu;
  static std::map<std::tuple<long long, long long, long long, bool, int>, Partition> cache;
  std::lock_guard<std::mutex> g(mu);
  auto key = std::make_tuple(total, k_iters, G, whole_tiles, delta);
  auto it = cache.find(key);
  if (it == cache.end()) {
    Partition P;
    make_partition(total, k_iters, (int)G, whole_tiles, delta, P);
    it = cache.emplace(key, P).first;
  }
  return it->second;
}

// Layout of a partial buffer: slots [grid * max_seg][BN][128] fp32, then per tile its piece
// count and slot list, meta[tiles][meta_stride] (meta_stride >= maxc + 1, a multiple of 4).
struct PartialLayout {
  size_t slots_bytes, total_bytes;
  long long tiles;
  int max_seg, maxc, meta_stride;
};
static PartialLayout partial_layout(int M, int N, int K, const Partition& P) {
  PartialLayout L;
  const int BN = gemm_token_tile(M);
  L.tiles = (long long)((N + kBM - 1) / kBM) * ((M + BN - 1) / BN);
  L.max_seg = P.max_seg;
  L.maxc = P.maxc;
  L.slots_bytes = (size_t)P.G * L.max_seg * BN * 128 * 4;
  L.meta_stride = (L.maxc + 1 + 3) / 4 * 4;
  L.total_bytes = L.slots_bytes + (size_t)L.tiles * 4 * L.meta_stride + 64;
  return L;
}

size_t gemm_partial_bytes(int M, int N, int K, int min_k_per_cta) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  return partial_layout(M, N, K, gemm_partition(M, N, K, false, min_k_per_cta)).total_bytes;
}

int launch_gemm(const GemmDesc& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0) return DF_OK;
  if (g.K % kBK != 0 || g.K <= 0) return DF_ERR_SHAPE;
  const int BN = gemm_token_tile(g.M);
  const int sub0 = BN < 256 ? BN : 256, sub1 = BN - sub0;
  CUtensorMap tw, tx, tx1;
  int rc = make_tmap_2d(&tw, g.W, g.N, g.K, g.ldw, kBM);
  if (rc) return rc;
  rc = make_tmap_2d(&tx, g.X, g.M, g.K, g.ldx, sub0);
  if (rc) return rc;
  tx1 = tx;
  if (sub1) {
    rc = make_tmap_2d(&tx1, g.X, g.M, g.K, g.ldx, sub1);
    if (rc) return rc;
  }
  GemmParams p{};
  p.sub0 = sub0;
  p.sub1 = sub1;
  p.nbuf = 2 * BN <= 512 ? 2 : 1;
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.n_ttiles = (g.M + BN - 1) / BN;
  p.w_keep = p.n_ttiles > 1;
  p.BN = BN;
  p.k_iters = g.K / kBK;
  const long long tiles = (long long)((g.N + kBM - 1) / kBM) * p.n_ttiles;
  p.total_iters = tiles * p.k_iters;
  p.whole_tiles = g.mode == kGemmStore || g.mode == kGemmArgmax;
  p.out = g.out;
  p.ldo = g.ldo;
  p.amax = g.amax;
  p.draw_key = g.draw_key;
  p.inv_temp = g.inv_temp;
  p.stats = reinterpret_cast<float2*>(g.stats);
  p.n_stats = 4 * ((g.N + kBM - 1) / kBM);
  p.status = g.status;
  const uint32_t stage_bytes = kBM * kBK * 2 + BN * kBK * 2;
  int stages = (int)((200 * 1024) / stage_bytes);
  if (stages > 8) stages = 8;
  if (stages < 2) stages = 2;
  p.stages = stages;
  const size_t smem = 1024 + (size_t)stages * stage_bytes + (2 * stages + 6) * 8 +
                      (g.mode == kGemmArgmax ? 4 * kArgChunks * 32 * 8 : 0);
  cudaError_t attr_err = cudaSuccess;
  switch (g.mode) {
    case kGemmPartial: attr_err = ensure_dynamic_smem(gemm_bf16_tc_kernel<kGemmPartial>, smem); break;
    case kGemmAtomicAdd: attr_err = ensure_dynamic_smem(gemm_bf16_tc_kernel<kGemmAtomicAdd>, smem); break;
    case kGemmStore: attr_err = ensure_dynamic_smem(gemm_bf16_tc_kernel<kGemmStore>, smem); break;
    case kGemmArgmax: attr_err = ensure_dynamic_smem(gemm_bf16_tc_kernel<kGemmArgmax>, smem); break;
    default: return DF_ERR_ARG;
  }
  if (attr_err != cudaSuccess) return DF_ERR_CUDA;
  const Partition& P = gemm_partition(g.M, g.N, g.K, p.whole_tiles, g.mode == kGemmPartial ? g.min_k_per_cta : 0);
  const long long grid = P.G;
  for (int c = 0; c <= P.G; ++c) p.starts[c] = P.starts[c];
  if (g.mode == kGemmPartial) {
    if (!g.part || !g.view) return DF_ERR_ARG;
    const PartialLayout L = partial_layout(g.M, g.N, g.K, P);
    unsigned char* base = reinterpret_cast<unsigned char*>(g.part);
    p.part = g.part;
    p.max_seg = L.max_seg;
    p.meta = reinterpret_cast<int*>(base + L.slots_bytes);
    p.meta_stride = L.meta_stride;
    PartialView& v = *g.view;
    v.part = g.part;
    v.meta = p.meta;
    v.meta_stride = L.meta_stride;
    v.BN = BN;
    v.n_ttiles = p.n_ttiles;
  }
  // trace tag: the kernel class, then the launch shape (M x N x K)
  char tag[48] = {0};
  if (trace_on())
    snprintf(tag, sizeof tag, "%s %dx%dx%d", g.mode == kGemmArgmax ? "gemm_lmhead_argmax"
                                             : g.mode == kGemmStore ? "gemm_lmhead_logits" : "gemm",
             g.M, g.N, g.K);
  DF_TRACE(tag, st);
  const dim3 gd((unsigned)grid), bd(kGemmThreads);
  switch (g.mode) {
    case kGemmPartial: launch_k(gemm_bf16_tc_kernel<kGemmPartial>, gd, bd, smem, st, tw, tx, tx1, p); break;
    case kGemmAtomicAdd: launch_k(gemm_bf16_tc_kernel<kGemmAtomicAdd>, gd, bd, smem, st, tw, tx, tx1, p); break;
    case kGemmStore: launch_k(gemm_bf16_tc_kernel<kGemmStore>, gd, bd, smem, st, tw, tx, tx1, p); break;
    case kGemmArgmax: launch_k(gemm_bf16_tc_kernel<kGemmArgmax>, gd, bd, smem, st, tw, tx, tx1, p); break;
    default: return DF_ERR_ARG;
  }
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace df
