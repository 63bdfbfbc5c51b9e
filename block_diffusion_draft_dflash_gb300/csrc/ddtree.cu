// DDTree construction on the GPU: per-position top-K, then best-first max-heap selection
// of the B most probable prefixes, then the ancestor bitsets of the flattened tree.
//
// Method: summary of "Accelerating Speculative Decoding with Block Diffusion Draft
// Trees" (bluediary8.tistory.com/1288), section "방법론 자세히 보기": the best B-node
// tree is the set of B prefixes with the highest prefix probability under the factorized
// per-position distribution, found by a best-first max-heap in O(B log B).
//
// Top-K, per (sequence, position) row of V log-probs, on order-preserving 32-bit keys:
//   * with scratch in the workspace (ddtree_build), three passes over 8192-key chunks
//     spread over the whole GPU: a histogram of the top 12 key bits, a collect pass that
//     keeps every key above the K-th key's bin and the candidates inside it, and a final
//     per-row select + bitonic sort by (log-prob desc, token id asc);
//   * otherwise, or when a row's candidates overflow, topk_rows_kernel: one CTA per row,
//     radix select (12 + 12 + 8 bit digits, MSB first, warp-aggregated shared-memory
//     histograms) for the K-th largest key T, a gather of every key > T and the lowest-id
//     keys == T, and the same sort.
// Kernel 2 (ddtree_heap_kernel, or ddtree_tourney_kernel from 256 nodes on): one CTA per
//   sequence.  One warp runs the best-first selection: each candidate is a single 64-bit key
//   whose integer order is the tree's total order (score desc, depth asc, parent index asc,
//   rank asc); the live candidates are held in the warp's registers (every pop a warp-wide
//   maximum over them) or, for larger budgets, one per node in a three-level tournament in
//   shared memory (every pop two slot updates and their group maxima).  The CTA then writes
//   the node arrays and the ancestor bitsets (one warp per row; each lane owns a 32-bit word).
#include "common.cuh"
#include "runtime.h"
#include "trace.h"

namespace df {

constexpr int kTopkThreads = 1024;
constexpr int kTourneyMinB = 256;  // budgets from which the selection runs as a tournament
constexpr int kMaxK = 2048;

DF_DEV void hist_add(uint32_t* hist, uint32_t digit, bool active) {
  // Lanes with the same digit add once through their leader.
  const uint32_t lanes = __ballot_sync(0xffffffffu, active);
  if (!active) return;
  const uint32_t peers = __match_any_sync(lanes, digit);
  const int lane = threadIdx.x & 31;
  if ((__ffs(peers) - 1) == lane) atomicAdd(&hist[digit], __popc(peers));
}

// Inclusive block scan of one value per thread (1024 threads).
DF_DEV uint32_t block_scan_incl(uint32_t v, uint32_t* warp_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_tmp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    warp_tmp[lane] = w;
  }
  __syncthreads();
  const uint32_t off = warp ? warp_tmp[warp - 1] : 0u;
  __syncthreads();
  return v + off;
}

// Whole-row radix top-K by one CTA of 1024 threads (also the fallback of the chunked
// path when the threshold bin holds too many candidates, e.g. rows of equal values).
// Block-wide bitonic sort, descending; n a power of two.  One thread per compared pair:
// pair p joins element lo (p with a 0 inserted at the stride's bit) and lo + stride.
DF_DEV void bitonic_desc(unsigned long long* a, int n) {
  const int half = n >> 1;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int p = threadIdx.x; p < half; p += blockDim.x) {
        const int lo = ((p & ~(stride - 1)) << 1) | (p & (stride - 1));
        const int hi = lo + stride;
        const unsigned long long x = a[lo], y = a[hi];
        const bool desc = (lo & size) == 0;
        if (desc ? (x < y) : (x > y)) { a[lo] = y; a[hi] = x; }
      }
      __syncthreads();
    }
  }
}

template <bool kVec4>
DF_DEV void topk_row_full(const float* __restrict__ lp, size_t row, int V, int K, int32_t* __restrict__ out_id,
                          float* __restrict__ out_val, int* status) {
  __shared__ uint32_t hist[4096];
  __shared__ uint32_t warp_tmp[32];
  __shared__ unsigned long long sel[kMaxK];
  __shared__ uint32_t sh_bin, sh_above, sh_ngt, sh_eq_base, sh_nan;
  const int tid = threadIdx.x;
  const float* x = lp + row * (size_t)V;
  if (tid == 0) { sh_nan = 0; sh_ngt = 0; sh_eq_base = 0; }

  uint32_t prefix = 0;
  int krem = K;
  const int shifts[3] = {20, 8, 0};
  const int widths[3] = {12, 12, 8};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass], width = widths[pass], nb = 1 << width;
    for (int i = tid; i < nb; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t mask = nb - 1;
    const int hi_shift = shift + width;  // bits above this digit must equal `prefix`
    auto visit = [&](float f, bool valid) {
      const uint32_t k = float_key(f);
      bool take = valid;
      if (pass == 0) {
        if (valid && isnan(f)) { sh_nan = 1; take = false; }
      } else {
        take = take && ((k >> hi_shift) == prefix);
      }
      hist_add(hist, (k >> shift) & mask, take);
    };
    if (kVec4) {
      const float4* x4 = reinterpret_cast<const float4*>(x);
      const int n4 = V >> 2;
      for (int base = 0; base < n4; base += kTopkThreads) {
        const int i = base + tid;
        float4 f = (i < n4) ? __ldg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        const bool ok = i < n4;
        visit(f.x, ok); visit(f.y, ok); visit(f.z, ok); visit(f.w, ok);
      }
    } else {
      for (int base = 0; base < V; base += kTopkThreads) {
        const int i = base + tid;
        visit(i < V ? __ldg(x + i) : 0.f, i < V);
      }
    }
    __syncthreads();
    if (sh_nan) {
      if (tid == 0) set_status(status, DF_ERR_NAN, (int)row);
      return;
    }
    // Bins in descending key order: position p <-> bin nb-1-p.  Thread t owns positions
    // [t*per, (t+1)*per) where per = nb / 1024 (or one position for t < nb if nb < 1024).
    const int per = nb >= kTopkThreads ? nb / kTopkThreads : 1;
    const bool owns = nb >= kTopkThreads || tid < nb;
    uint32_t local = 0;
    if (owns)
      for (int j = 0; j < per; ++j) local += hist[nb - 1 - (tid * per + j)];
    const uint32_t incl = block_scan_incl(local, warp_tmp);
    const uint32_t excl = incl - local;
    if (owns && excl < (uint32_t)krem && (uint32_t)krem <= incl) {
      uint32_t acc = excl;
      for (int j = 0; j < per; ++j) {
        const int bin = nb - 1 - (tid * per + j);
        const uint32_t c = hist[bin];
        if (acc + c >= (uint32_t)krem) { sh_bin = bin; sh_above = acc; break; }
        acc += c;
      }
    }
    __syncthreads();
    prefix = (prefix << width) | sh_bin;
    krem -= (int)sh_above;
    __syncthreads();
  }
  // prefix == T (the K-th largest key); krem = how many keys equal to T are taken.
  const uint32_t T = prefix;
  const uint32_t n_eq_total = hist[T & 0xFF];
  const int n_gt = K - krem;
  const bool need_lowest = n_eq_total > (uint32_t)krem;  // ties straddle the cut
  // Gather keys > T (any order), and keys == T when all of them are taken.
  auto put = [&](float f, int i, bool valid) {
    if (!valid) return;
    const uint32_t k = float_key(f);
    if (k > T || (k == T && !need_lowest)) {
      const uint32_t pos = atomicAdd(&sh_ngt, 1u);
      if (pos < (uint32_t)kMaxK) sel[pos] = ((unsigned long long)k << 32) | (uint32_t)(~(uint32_t)i);
    }
  };
  if (kVec4) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int n4 = V >> 2;
    for (int i = tid; i < n4; i += kTopkThreads) {
      const float4 f = __ldg(x4 + i);
      put(f.x, 4 * i, true); put(f.y, 4 * i + 1, true); put(f.z, 4 * i + 2, true); put(f.w, 4 * i + 3, true);
    }
  } else {
    for (int i = tid; i < V; i += kTopkThreads) put(__ldg(x + i), i, true);
  }
  __syncthreads();
  if (need_lowest) {
    // Take the krem lowest indices with key == T, scanning in index order.
    for (int base = 0; base < V; base += kTopkThreads) {
      const int i = base + tid;
      const bool eq = i < V && float_key(__ldg(x + i)) == T;
      const uint32_t incl = block_scan_incl(eq ? 1u : 0u, warp_tmp);
      const uint32_t rank = sh_eq_base + incl - (eq ? 1u : 0u);
      if (eq && rank < (uint32_t)krem)
        sel[n_gt + rank] = ((unsigned long long)T << 32) | (uint32_t)(~(uint32_t)i);
      __syncthreads();
      if (tid == kTopkThreads - 1) sh_eq_base += incl;
      __syncthreads();
      if (sh_eq_base >= (uint32_t)krem) break;
    }
  }
  // Bitonic sort (descending) of K entries padded to a power of two with zeros.
  int n = 1;
  while (n < K) n <<= 1;
  for (int i = K + tid; i < n; i += kTopkThreads) sel[i] = 0ull;
  __syncthreads();
  bitonic_desc(sel, n);
  for (int r = tid; r < K; r += kTopkThreads) {
    const unsigned long long c = sel[r];
    out_id[row * K + r] = (int32_t)(~(uint32_t)(c & 0xFFFFFFFFull));
    out_val[row * K + r] = key_float((uint32_t)(c >> 32));
  }
}

template <bool kVec4>
__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(const float* __restrict__ lp, int V, int K,
                                                                 int32_t* __restrict__ out_id,
                                                                 float* __restrict__ out_val, int* status) {
  pdl_wait();
  pdl_trigger();
  topk_row_full<kVec4>(lp, blockIdx.x, V, K, out_id, out_val, status);
}

// ----------------------------------------------------------------------------- sampled top-K
// One read of the log-probs per row when scratch is available:
//   topk_sample:  a 1/16 sample of the row (every 16th line of 32 floats) and histograms of
//                 its top 12 key bits, then of the next 12 bits inside the chosen bin, give
//                 a threshold key t at or below the K-th largest key with high probability
//                 (where the sample's count from the top reaches K/16 plus a 4-sigma margin);
//   topk_collect: every key >= t is appended to the row's candidate list (gathered per
//                 block in shared memory, one global reservation per block), NaN reported;
//   topk_final:   if K <= candidates <= capacity, a bitonic sort by (key desc, id asc) of
//                 the candidates gives the top K exactly (every key above the K-th largest
//                 is at least t).  Otherwise the row is redone by the whole-row select.
constexpr int kChunk = 8192;          // keys per collect block
constexpr int kChunkThreads = 512;
constexpr int kSampleLines = 16;      // one line of 32 keys in 16 is sampled
constexpr int kCapCand = 8192;        // candidates kept per row
constexpr int kSampleU = 8;           // sampled lines a warp loads before counting them
constexpr int kLocCand = 2048;        // candidates one collect block holds (more: the row falls back)

struct TopkRow {     // per row, in the workspace
  uint32_t thr, count, pad0, pad1;
};

__global__ void __launch_bounds__(256) topk_sample_kernel(const float* __restrict__ lp, int V, int K,
                                                          TopkRow* __restrict__ sc) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t hist[4096];
  __shared__ uint32_t warp_tmp[8];
  __shared__ uint32_t sh_bin, sh_found;
  const size_t row = blockIdx.x;
  const float* x = lp + row * (size_t)V;
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) { sh_bin = 0; sh_found = 0; }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int n_lines = V / 32;
  int n_sample = 0;
  // the sampled lines' loads are issued kSampleU at a time (independent DRAM round trips)
  for (int l0 = warp * kSampleLines; l0 < n_lines; l0 += nw * kSampleLines * kSampleU) {
    float f[kSampleU];
#pragma unroll
    for (int u = 0; u < kSampleU; ++u) {
      const int l = l0 + u * nw * kSampleLines;
      f[u] = l < n_lines ? __ldg(x + (size_t)l * 32 + lane) : __int_as_float(0x7fc00000);  // NaN: skipped
    }
#pragma unroll
    for (int u = 0; u < kSampleU; ++u)
      if (!isnan(f[u])) atomicAdd(&hist[float_key(f[u]) >> 20], 1u);
  }
  n_sample = ((n_lines + kSampleLines - 1) / kSampleLines) * 32;
  __syncthreads();
  // the sample rank to reach: K / 16 plus a margin of 4 standard deviations
  const float kr = (float)K / kSampleLines;
  const uint32_t r = (uint32_t)ceilf(kr + 4.f * sqrtf(kr) + 4.f);
  // bins in descending order, 16 per thread; inclusive scan of the per-thread sums
  uint32_t local = 0;
  for (int j = 0; j < 16; ++j) local += hist[4095 - (threadIdx.x * 16 + j)];
  uint32_t v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tmp[warp] = v;
  __syncthreads();
  uint32_t off = 0;
  for (int w = 0; w < warp; ++w) off += warp_tmp[w];
  const uint32_t incl = v + off, excl = incl - local;
  if (excl < r && r <= incl) {
    uint32_t acc = excl;
    for (int j = 0; j < 16; ++j) {
      const int bin = 4095 - (threadIdx.x * 16 + j);
      acc += hist[bin];
      if (acc >= r) { sh_bin = bin; sh_found = 1; break; }
    }
  }
  __syncthreads();
  // second level: the next 12 key bits of the sampled keys inside that bin, counted from the
  // top; the rank still to reach inside the bin is r minus the sample count above it
  const uint32_t hi_bin = sh_bin;
  const bool found = sh_found != 0;
  uint32_t above = 0;
  if (found) {
    // count of sampled keys in bins above hi_bin (warp-strided sum, then block sum)
    uint32_t a = 0;
    for (int b2 = (int)hi_bin + 1 + threadIdx.x; b2 < 4096; b2 += blockDim.x) a += hist[b2];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    __syncthreads();
    if (lane == 0) warp_tmp[warp] = a;
    __syncthreads();
    for (int w = 0; w < nw; ++w) above += warp_tmp[w];
    __syncthreads();
    for (int i = threadIdx.x; i < 4096; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int l0 = warp * kSampleLines; l0 < n_lines; l0 += nw * kSampleLines * kSampleU) {
      float f[kSampleU];
#pragma unroll
      for (int u = 0; u < kSampleU; ++u) {
        const int l = l0 + u * nw * kSampleLines;
        f[u] = l < n_lines ? __ldg(x + (size_t)l * 32 + lane) : __int_as_float(0x7fc00000);
      }
#pragma unroll
      for (int u = 0; u < kSampleU; ++u) {
        const uint32_t k = float_key(f[u]);
        if (!isnan(f[u]) && (k >> 20) == hi_bin) atomicAdd(&hist[(k >> 8) & 0xFFF], 1u);
      }
    }
    __syncthreads();
    const uint32_t r2 = r - above;  // >= 1: the bin holds the r-th sampled key
    if (threadIdx.x == 0) sh_bin = hi_bin << 12;  // (the whole bin, should the search below miss)
    __syncthreads();
    local = 0;
    for (int j = 0; j < 16; ++j) local += hist[4095 - (threadIdx.x * 16 + j)];
    v = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t nn = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += nn;
    }
    __syncthreads();
    if (lane == 31) warp_tmp[warp] = v;
    __syncthreads();
    uint32_t off2 = 0;
    for (int w = 0; w < warp; ++w) off2 += warp_tmp[w];
    const uint32_t incl2 = v + off2, excl2 = incl2 - local;
    if (excl2 < r2 && r2 <= incl2) {
      uint32_t acc = excl2;
      for (int j = 0; j < 16; ++j) {
        const int bin = 4095 - (threadIdx.x * 16 + j);
        acc += hist[bin];
        if (acc >= r2) { sh_bin = (hi_bin << 12) | (uint32_t)bin; break; }
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    // too small a sample for the rank: take every key (the count check then decides)
    sc[row].thr = (found && (uint32_t)n_sample >= r) ? (sh_bin << 8) : 0u;
    sc[row].count = 0;
  }
}

template <bool kVec4>
__global__ void __launch_bounds__(kChunkThreads) topk_collect_kernel(const float* __restrict__ lp, int V,
                                                                     TopkRow* __restrict__ sc,
                                                                     unsigned long long* __restrict__ cand,
                                                                     int* status) {
  pdl_wait();
  pdl_trigger();
  // candidates of this chunk gather in shared memory first; one global reservation per block
  __shared__ unsigned long long loc[kLocCand];
  __shared__ uint32_t n_loc, base;
  const size_t row = blockIdx.y;
  const float* x = lp + row * (size_t)V;
  if (threadIdx.x == 0) n_loc = 0;
  __syncthreads();
  const uint32_t t = sc[row].thr;
  const int lane = threadIdx.x & 31;
  const int i0 = blockIdx.x * kChunk, i1 = min(V, i0 + kChunk);
  bool nan = false;
  auto put = [&](float f, int i, bool valid) {
    nan |= valid && isnan(f);
    const uint32_t k = float_key(f);
    const bool take = valid && k >= t;
    const uint32_t m = __ballot_sync(0xffffffffu, take);
    if (!m) return;
    uint32_t b0 = 0;
    if (lane == __ffs(m) - 1) b0 = atomicAdd(&n_loc, (uint32_t)__popc(m));
    b0 = __shfl_sync(0xffffffffu, b0, __ffs(m) - 1);
    const uint32_t pos = b0 + __popc(m & ((1u << lane) - 1u));
    if (take && pos < (uint32_t)kLocCand) loc[pos] = ((unsigned long long)k << 32) | (uint32_t)(~(uint32_t)i);
  };
  if (kVec4) {
    // every load of the chunk is issued before any is used: one DRAM round trip per block
    constexpr int kPer = kChunk / 4 / kChunkThreads;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float4 f[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int q = i0 / 4 + u * kChunkThreads + threadIdx.x;
      f[u] = q * 4 < i1 ? __ldg(x4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int q = i0 / 4 + u * kChunkThreads + threadIdx.x;
      const bool ok = q * 4 < i1;
      put(f[u].x, 4 * q, ok); put(f[u].y, 4 * q + 1, ok); put(f[u].z, 4 * q + 2, ok); put(f[u].w, 4 * q + 3, ok);
    }
  } else {
    for (int b = i0; b < i1; b += blockDim.x) {
      const int i = b + threadIdx.x;
      const bool ok = i < i1;
      put(ok ? __ldg(x + i) : 0.f, i, ok);
    }
  }
  if (__any_sync(0xffffffffu, nan) && lane == 0) set_status(status, DF_ERR_NAN, (int)row);
  __syncthreads();
  const uint32_t n = n_loc;
  // a block holding more than kLocCand candidates pushes the row's count past the capacity,
  // so the row is redone by the whole-row select
  if (threadIdx.x == 0) base = atomicAdd(&sc[row].count, n > (uint32_t)kLocCand ? (uint32_t)kCapCand + 1 : n);
  __syncthreads();
  if (n <= (uint32_t)kLocCand)
    for (uint32_t j = threadIdx.x; j < n; j += blockDim.x)
      if (base + j < (uint32_t)kCapCand) cand[row * kCapCand + base + j] = loc[j];
}


template <bool kVec4>
__global__ void __launch_bounds__(kTopkThreads) topk_final_kernel(const float* __restrict__ lp, int V, int K,
                                                                  const TopkRow* __restrict__ sc,
                                                                  const unsigned long long* __restrict__ cand,
                                                                  int32_t* __restrict__ out_id,
                                                                  float* __restrict__ out_val, int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ unsigned long long keys[];  // [kCapCand]
  const size_t row = blockIdx.x;
  if (status && *(volatile int*)status == DF_ERR_NAN) return;
  const uint32_t n_c = sc[row].count;
  if (n_c < (uint32_t)K || n_c > (uint32_t)kCapCand) {  // the threshold missed: whole-row select
    topk_row_full<kVec4>(lp, row, V, K, out_id, out_val, status);
    return;
  }
  int n = 1;
  while (n < (int)n_c) n <<= 1;
  for (int i = threadIdx.x; i < n; i += blockDim.x) keys[i] = i < (int)n_c ? cand[row * kCapCand + i] : 0ull;
  __syncthreads();
  bitonic_desc(keys, n);
  for (int r = threadIdx.x; r < K; r += blockDim.x) {
    const unsigned long long c = keys[r];
    out_id[row * K + r] = (int32_t)(~(uint32_t)(c & 0xFFFFFFFFull));
    out_val[row * K + r] = key_float((uint32_t)(c >> 32));
  }
}

size_t topk_chunked_scratch_bytes(int rows) {
  return (size_t)rows * (sizeof(TopkRow) + (size_t)kCapCand * 8) + 1024;
}

// ----------------------------------------------------------------------------- heap
// 64-bit heap key, larger = earlier in the tree's total order:
//   [63:32] float_key(score)  [31:27] 31-depth  [26:16] 2047-parent  [15:5] 2047-rank
DF_DEV unsigned long long heap_key(float s, int depth, int parent, int rank) {
  return ((unsigned long long)float_key(s) << 32) | ((uint32_t)(31 - depth) << 27) |
         ((uint32_t)(2047 - parent) << 16) | ((uint32_t)(2047 - rank) << 5);
}

// The selected nodes (shared memory) -> the tree's arrays and ancestor bitsets (whole CTA).
DF_DEV void write_tree(int s, int n, int D, int K, const int32_t* __restrict__ topk_id,
                       const int32_t* __restrict__ root_tok, const int32_t* n_par, const int32_t* n_dep,
                       const int32_t* n_rank, const float* n_score, int32_t* __restrict__ tok,
                       int32_t* __restrict__ parent, int32_t* __restrict__ depth, float* __restrict__ score,
                       uint32_t* __restrict__ anc) {
  const int tid = threadIdx.x, W = (n + 31) / 32;
  const size_t o = (size_t)s * n;
  const int32_t* gid = topk_id + (size_t)s * D * K;
  for (int i = tid; i < n; i += blockDim.x) {
    tok[o + i] = i == 0 ? (root_tok ? root_tok[s] : -1) : gid[(n_dep[i] - 1) * K + n_rank[i]];
    parent[o + i] = n_par[i];
    depth[o + i] = n_dep[i];
    score[o + i] = n_score[i];
  }
  // Ancestor bitsets: one warp per row, lane w owns words w, w+32, ...
  const int lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  uint32_t* arow = anc + (size_t)s * n * W;
  for (int i = warp; i < n; i += nwarps) {
    for (int w0 = 0; w0 < W; w0 += 32) {
      const int w = w0 + lane;
      uint32_t bits = 0;
      for (int j = i; j >= 0; j = n_par[j])
        if ((j >> 5) == w) bits |= 1u << (j & 31);
      if (w < W) arow[(size_t)i * W + w] = bits;
    }
  }
}

// One CTA per sequence; warp 0 runs the best-first selection.  The live candidates (at most
// B + 1) sit in the warp's registers, NREG per lane, densely packed: candidate c lives in
// lane c % 32, register c / 32.  Each pop takes the lane maxima, a warp maximum (two redux steps)
// and a ballot for the owner; the last candidate fills the hole; the successors (first
// child, next sibling) are appended.  Keys are unique, so the maximum is unique.
template <int NREG>
__global__ void __launch_bounds__(256) ddtree_heap_kernel(const int32_t* __restrict__ topk_id,
                                                          const float* __restrict__ topk_val, int D, int K, int B,
                                                          const int32_t* __restrict__ root_tok,
                                                          int32_t* __restrict__ tok, int32_t* __restrict__ parent,
                                                          int32_t* __restrict__ depth, float* __restrict__ score,
                                                          uint32_t* __restrict__ anc, const int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  const int s = blockIdx.x, tid = threadIdx.x;
  const int n = B + 1;
  float* val = reinterpret_cast<float*>(smem);                                       // [D][K]
  int32_t* n_par = reinterpret_cast<int32_t*>(val + ((D * K + 1) & ~1));             // [n]
  int32_t* n_dep = n_par + n;                                                        // [n]
  int32_t* n_rank = n_dep + n;                                                       // [n]
  float* n_score = reinterpret_cast<float*>(n_rank + n);                             // [n]

  if (status && *(volatile const int*)status == DF_ERR_NAN) return;  // NaN found by top-K
  const float* gval = topk_val + (size_t)s * D * K;
  for (int i = tid; i < D * K; i += blockDim.x) val[i] = gval[i];
  __syncthreads();

  if (tid < 32) {
    const int lane = tid;
    unsigned long long cand[NREG];
#pragma unroll
    for (int i = 0; i < NREG; ++i) cand[i] = 0ull;  // 0 = empty (no key is 0)
    int cnt = 0;
    auto append = [&](unsigned long long key) {  // warp-uniform
      const int li = cnt & 31, ri = cnt >> 5;
#pragma unroll
      for (int i = 0; i < NREG; ++i)
        if (i == ri && lane == li) cand[i] = key;
      ++cnt;
    };
    // every lane writes the node arrays (same value), so every lane reads its own writes
    n_par[0] = -1; n_dep[0] = 0; n_rank[0] = -1; n_score[0] = 0.f;
    if (B > 0) append(heap_key(0.f + val[0], 1, 0, 0));
    for (int idx = 1; idx <= B; ++idx) {
      // lane maximum as a tree (depth log2 NREG, not a chain through every register)
      unsigned long long t[NREG];
#pragma unroll
      for (int i = 0; i < NREG; ++i) t[i] = cand[i];
#pragma unroll
      for (int st = 1; st < NREG; st <<= 1)
#pragma unroll
        for (int i = 0; i + st < NREG; i += 2 * st) t[i] = t[i] > t[i + st] ? t[i] : t[i + st];
      const unsigned long long best = t[0];
      // warp maximum of the 64-bit lane maxima: the high words with one redux, then the low
      // words among the lanes that hold the top high word
      const uint32_t top_hi = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32));
      const bool at_hi = (uint32_t)(best >> 32) == top_hi;
      const uint32_t top_lo = __reduce_max_sync(0xffffffffu, at_hi ? (uint32_t)best : 0u);
      const unsigned long long top = ((unsigned long long)top_hi << 32) | top_lo;
      // the last candidate moves into the popped one's place (keys are unique, so exactly one
      // register of one lane equals `top`); then the last place is cleared
      const int last = cnt - 1, ll = last & 31, lr = last >> 5;
      unsigned long long lv = 0ull;
#pragma unroll
      for (int i = 0; i < NREG; ++i) lv |= (i == lr) ? cand[i] : 0ull;
      lv = __shfl_sync(0xffffffffu, lv, ll);
#pragma unroll
      for (int i = 0; i < NREG; ++i) cand[i] = cand[i] == top ? lv : cand[i];
#pragma unroll
      for (int i = 0; i < NREG; ++i)
        if (lane == ll && i == lr) cand[i] = 0ull;
      --cnt;
      const uint32_t lo = (uint32_t)top;
      const int dep = 31 - (int)(lo >> 27);
      const int par = 2047 - (int)((lo >> 16) & 0x7FF);
      const int r = 2047 - (int)((lo >> 5) & 0x7FF);
      const float sc = key_float((uint32_t)(top >> 32));
      n_par[idx] = par; n_dep[idx] = dep; n_rank[idx] = r; n_score[idx] = sc;
      if (dep < D) append(heap_key(sc + val[dep * K], dep + 1, idx, 0));
      if (r + 1 < K) append(heap_key(n_score[par] + val[(dep - 1) * K + r + 1], dep, par, r + 1));
    }
  }
  __syncthreads();
  write_tree(s, n, D, K, topk_id, root_tok, n_par, n_dep, n_rank, n_score, tok, parent, depth, score, anc);
}

// Warp-wide maximum of a 64-bit key: the high words with one redux, then the low words among
// the lanes that hold the top high word.
DF_DEV unsigned long long warp_max_key(unsigned long long v) {
  const uint32_t hi = __reduce_max_sync(0xffffffffu, (uint32_t)(v >> 32));
  const uint32_t lo = __reduce_max_sync(0xffffffffu, (uint32_t)(v >> 32) == hi ? (uint32_t)v : 0u);
  return ((unsigned long long)hi << 32) | lo;
}

// The same best-first selection with the candidates in a three-level tournament in shared
// memory instead of registers.  Every node holds at most one live candidate, its best child
// not yet selected: selecting a child c of p replaces p's candidate by c's next sibling and
// gives c its first child.  So the candidates sit in slots indexed by node (leaf[p]), and a
// selection changes two slots; a change recomputes the maximum of the slot's group of 32
// (one warp maximum), of that group's group of 32, and of the few top groups.  The keys,
// hence the order of selection, are those of ddtree_heap_kernel.
__global__ void __launch_bounds__(256) ddtree_tourney_kernel(const int32_t* __restrict__ topk_id,
                                                             const float* __restrict__ topk_val, int D, int K, int B,
                                                             const int32_t* __restrict__ root_tok,
                                                             int32_t* __restrict__ tok, int32_t* __restrict__ parent,
                                                             int32_t* __restrict__ depth, float* __restrict__ score,
                                                             uint32_t* __restrict__ anc, const int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char smem[];
  const int s = blockIdx.x, tid = threadIdx.x;
  const int n = B + 1;
  const int n0 = (n + 31) & ~31, n1 = ((n0 >> 5) + 31) & ~31, n2 = n1 >> 5;  // level sizes (n2 <= 32)
  unsigned long long* leaf = reinterpret_cast<unsigned long long*>(smem);  // [n0] candidate of each node
  unsigned long long* lv1 = leaf + n0;                                     // [n1] maxima of 32 leaves
  unsigned long long* lv2 = lv1 + n1;                                      // [n2] maxima of 32 lv1 entries
  float* val = reinterpret_cast<float*>(lv2 + ((n2 + 1) & ~1));            // [D][K]
  int32_t* n_par = reinterpret_cast<int32_t*>(val + ((D * K + 1) & ~1));   // [n]
  int32_t* n_dep = n_par + n;
  int32_t* n_rank = n_dep + n;
  float* n_score = reinterpret_cast<float*>(n_rank + n);

  if (status && *(volatile const int*)status == DF_ERR_NAN) return;  // NaN found by top-K
  const float* gval = topk_val + (size_t)s * D * K;
  for (int i = tid; i < D * K; i += blockDim.x) val[i] = gval[i];
  for (int i = tid; i < n0 + n1 + n2; i += blockDim.x) leaf[i] = 0ull;  // 0 = no candidate
  __syncthreads();

  if (tid < 32) {
    const int lane = tid;
    n_par[0] = -1; n_dep[0] = 0; n_rank[0] = -1; n_score[0] = 0.f;
    // up to 2048 nodes the (at most 64) lv1 maxima are read directly for the top (two levels)
    const bool two_level = n1 <= 64;
    // a slot changed: its group maxima up to the top
    auto fix = [&](int x) {
      const int g1 = x >> 5, g2 = g1 >> 5;
      __syncwarp();
      const unsigned long long m1 = warp_max_key(leaf[(g1 << 5) + lane]);
      if (lane == 0) lv1[g1] = m1;
      __syncwarp();
      if (two_level) return;
      const unsigned long long m2 = warp_max_key(lv1[(g2 << 5) + lane]);
      if (lane == 0) lv2[g2] = m2;
      __syncwarp();
    };
    if (B > 0) {
      if (lane == 0) leaf[0] = heap_key(0.f + val[0], 1, 0, 0);
      fix(0);
    }
    for (int idx = 1; idx <= B; ++idx) {
      unsigned long long t0;
      if (two_level) {
        const unsigned long long a = lv1[lane], c = lane + 32 < n1 ? lv1[lane + 32] : 0ull;
        t0 = a > c ? a : c;
      } else {
        t0 = lane < n2 ? lv2[lane] : 0ull;
      }
      const unsigned long long top = warp_max_key(t0);
      const uint32_t lo = (uint32_t)top;
      const int dep = 31 - (int)(lo >> 27);
      const int par = 2047 - (int)((lo >> 16) & 0x7FF);
      const int r = 2047 - (int)((lo >> 5) & 0x7FF);
      const float sc = key_float((uint32_t)(top >> 32));
      // every lane writes the node arrays (same value), so every lane reads its own writes
      n_par[idx] = par; n_dep[idx] = dep; n_rank[idx] = r; n_score[idx] = sc;
      const unsigned long long sib = r + 1 < K ? heap_key(n_score[par] + val[(dep - 1) * K + r + 1], dep, par, r + 1) : 0ull;
      const unsigned long long kid = dep < D ? heap_key(sc + val[dep * K], dep + 1, idx, 0) : 0ull;
      __syncwarp();
      if (lane == 0) { leaf[par] = sib; leaf[idx] = kid; }
      fix(par);
      if ((idx >> 5) != (par >> 5)) fix(idx);
    }
  }
  __syncthreads();
  write_tree(s, n, D, K, topk_id, root_tok, n_par, n_dep, n_rank, n_score, tok, parent, depth, score, anc);
}

size_t ddtree_tourney_smem(int D, int K, int B) {
  const int n = B + 1;
  const int n0 = (n + 31) & ~31, n1 = ((n0 >> 5) + 31) & ~31, n2 = n1 >> 5;
  return (size_t)(n0 + n1 + ((n2 + 1) & ~1)) * 8 + (size_t)((D * K + 1) & ~1) * 4 + (size_t)n * 16;
}

}  // namespace df

// ----------------------------------------------------------------------------- host
namespace df {
size_t ddtree_heap_smem(int D, int K, int B) {
  const int n = B + 1;
  return (size_t)((D * K + 1) & ~1) * 4 + (size_t)n * 16;
}

__global__ void zero_u32_kernel(uint32_t* p, size_t n) {
  pdl_wait();
  pdl_trigger();
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) p[i] = 0;
}

int launch_ddtree(const float* lp, int b, int D, int V, int B, const int32_t* root_tok, int32_t* tok,
                  int32_t* parent, int32_t* depth, float* score, uint32_t* anc, int32_t* topk_id,
                  float* topk_val, int* status, cudaStream_t st, void* chunk_scratch) {
  const int K = B < V ? B : V;
  if (B > 0) {
    const int rows = b * D;
    if (chunk_scratch && V >= 4 * kChunk) {
      // sampled threshold, one collecting read, exact select (whole-row select per row as fallback)
      unsigned char* base = static_cast<unsigned char*>(chunk_scratch);
      TopkRow* sc = reinterpret_cast<TopkRow*>(base);
      unsigned long long* cand = reinterpret_cast<unsigned long long*>(
          (reinterpret_cast<uintptr_t>(sc + rows) + 255) & ~uintptr_t(255));
      {
        DF_TRACE("topk_sample", st);
        launch_k(topk_sample_kernel, dim3(rows), dim3(256), 0, st, lp, V, K, sc);
      }
      const dim3 grid((V + kChunk - 1) / kChunk, rows);
      const size_t smem = (size_t)kCapCand * 8;
      if (ensure_dynamic_smem(topk_final_kernel<true>, smem) != cudaSuccess ||
          ensure_dynamic_smem(topk_final_kernel<false>, smem) != cudaSuccess)
        return DF_ERR_CUDA;
      {
        DF_TRACE("topk_collect", st);
        if ((V & 3) == 0) launch_k(topk_collect_kernel<true>, grid, dim3(kChunkThreads), 0, st, lp, V, sc, cand, status);
        else launch_k(topk_collect_kernel<false>, grid, dim3(kChunkThreads), 0, st, lp, V, sc, cand, status);
      }
      DF_TRACE("topk_select", st);
      if ((V & 3) == 0)
        launch_k(topk_final_kernel<true>, dim3(rows), dim3(kTopkThreads), smem, st, lp, V, K, sc, cand, topk_id,
                 topk_val, status);
      else
        launch_k(topk_final_kernel<false>, dim3(rows), dim3(kTopkThreads), smem, st, lp, V, K, sc, cand, topk_id,
                 topk_val, status);
    } else if ((V & 3) == 0) {
      DF_TRACE("topk", st);
      launch_k(topk_rows_kernel<true>, dim3(rows), dim3(kTopkThreads), 0, st, lp, V, K, topk_id, topk_val, status);
    } else {
      DF_TRACE("topk", st);
      launch_k(topk_rows_kernel<false>, dim3(rows), dim3(kTopkThreads), 0, st, lp, V, K, topk_id, topk_val, status);
    }
  }
  const size_t smem = ddtree_heap_smem(D, K > 0 ? K : 1, B);
  // registers per lane for the live candidates (at most B + 1)
  const int nreg = (B + 1 + 31) / 32;
  auto launch = [&](auto kern) -> int {
    if (ensure_dynamic_smem(kern, smem) != cudaSuccess) return DF_ERR_CUDA;
    DF_TRACE("ddtree_heap", st);
    launch_k(kern, dim3(b), dim3(256), smem, st, topk_id, topk_val, D, K > 0 ? K : 1, B, root_tok, tok, parent, depth,
             score, anc, status);
    return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
  };
  // the tournament in shared memory from 256 nodes on (its cost grows with log B, the
  // registers' with B: equal at 256, 2.8x faster at 1024), when it fits beside the log-probs
  const size_t smem_t = ddtree_tourney_smem(D, K > 0 ? K : 1, B);
  if (B >= kTourneyMinB && smem_t <= 227 * 1024) {
    if (ensure_dynamic_smem(ddtree_tourney_kernel, smem_t) != cudaSuccess) return DF_ERR_CUDA;
    DF_TRACE("ddtree_heap", st);
    launch_k(ddtree_tourney_kernel, dim3(b), dim3(256), smem_t, st, topk_id, topk_val, D, K > 0 ? K : 1, B, root_tok,
             tok, parent, depth, score, anc, status);
    return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
  }
  if (nreg <= 1) return launch(ddtree_heap_kernel<1>);
  if (nreg <= 2) return launch(ddtree_heap_kernel<2>);
  if (nreg <= 4) return launch(ddtree_heap_kernel<4>);
  if (nreg <= 9) return launch(ddtree_heap_kernel<9>);
  if (nreg <= 17) return launch(ddtree_heap_kernel<17>);
  if (nreg <= 33) return launch(ddtree_heap_kernel<33>);
  if (nreg <= 65) return launch(ddtree_heap_kernel<65>);
  return DF_ERR_SHAPE;
}

// ----------------------------------------------------------------------------- chain
// Vanilla DFlash draft (summary of "Accelerating Speculative Decoding with Block Diffusion
// Draft Trees", section "실험 결과", compares it with DDTree at the same block size): the
// drafter's most likely token at every position, verified as one causal chain.
//
// chain_argmax_kernel: grid (ceil(V / kChunk), rows), one block per 8192-entry chunk of a
//   row; the block's maximum key ((order-preserving log-prob bits << 32) | ~token id, so
//   the largest value wins and, among equal values, the lowest id) is folded into the
//   row's key with one 64-bit atomic maximum.
// chain_finalize_kernel: one warp per sequence: node i (1..D) carries position i's token,
//   parent i - 1, depth i, score = fp32 sum of log-probs root first; ancestor row i has
//   bits 0..i set.
__global__ void __launch_bounds__(kChunkThreads) chain_argmax_kernel(const float* __restrict__ lp, int V,
                                                                     unsigned long long* __restrict__ keys,
                                                                     int* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned long long red[kChunkThreads / 32];
  const size_t row = blockIdx.y;
  const float* x = lp + row * (size_t)V;
  const int i0 = blockIdx.x * kChunk, i1 = min(V, i0 + kChunk);
  unsigned long long best = 0ull;
  bool nan = false;
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const float f = __ldg(x + i);
    nan |= isnan(f);
    const unsigned long long k = ((unsigned long long)float_key(f) << 32) | (uint32_t)(~(uint32_t)i);
    best = k > best ? k : best;
  }
  if (__any_sync(0xffffffffu, nan) && (threadIdx.x & 31) == 0) set_status(status, DF_ERR_NAN, (int)row);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
    best = y > best ? y : best;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) best = red[w] > best ? red[w] : best;
    atomicMax(keys + row, best);
  }
}

__global__ void __launch_bounds__(32) chain_finalize_kernel(const unsigned long long* __restrict__ keys, int D,
                                                            const int32_t* __restrict__ root_tok,
                                                            int32_t* __restrict__ tok, int32_t* __restrict__ parent,
                                                            int32_t* __restrict__ depth, float* __restrict__ score,
                                                            uint32_t* __restrict__ anc, const int* status) {
  pdl_wait();
  pdl_trigger();
  if (status && *(volatile const int*)status == DF_ERR_NAN) return;
  const int s = blockIdx.x, lane = threadIdx.x;
  const int n = D + 1, W = (n + 31) / 32;
  const size_t o = (size_t)s * n;
  if (lane == 0) {
    float sc = 0.f;
    tok[o] = root_tok ? root_tok[s] : -1;
    parent[o] = -1;
    depth[o] = 0;
    score[o] = 0.f;
    for (int i = 1; i <= D; ++i) {
      const unsigned long long k = keys[(size_t)s * D + i - 1];
      sc = sc + key_float((uint32_t)(k >> 32));
      tok[o + i] = (int32_t)(~(uint32_t)(k & 0xFFFFFFFFull));
      parent[o + i] = i - 1;
      depth[o + i] = i;
      score[o + i] = sc;
    }
  }
  for (int e = lane; e < n * W; e += 32) {
    const int i = e / W, w = e % W;
    const int nb = i + 1 - 32 * w;  // bits 0..i set
    anc[o * W + e] = nb >= 32 ? 0xFFFFFFFFu : (nb <= 0 ? 0u : ((1u << nb) - 1u));
  }
}

int launch_chain(const float* lp, int b, int D, int V, const int32_t* root_tok, int32_t* tok, int32_t* parent,
                 int32_t* depth, float* score, uint32_t* anc, unsigned long long* keys, int* status, cudaStream_t st) {
  DF_TRACE("chain", st);
  const int rows = b * D;
  launch_k(zero_u32_kernel, dim3((unsigned)((2 * rows + 255) / 256)), dim3(256), 0, st,
           reinterpret_cast<uint32_t*>(keys), (size_t)2 * rows);
  launch_k(chain_argmax_kernel, dim3((V + kChunk - 1) / kChunk, rows), dim3(kChunkThreads), 0, st, lp, V, keys,
           status);
  launch_k(chain_finalize_kernel, dim3(b), dim3(32), 0, st, keys, D, root_tok, tok, parent, depth, score, anc,
           status);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}
}  // namespace df
