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
// Kernel 2 (ddtree_heap_kernel): one CTA per sequence.  One warp runs the best-first
//   selection: each candidate is a single 64-bit key whose integer order is the tree's
//   total order (score desc, depth asc, parent index asc, rank asc), the live candidates
//   are held in the warp's registers and every pop is a warp-wide maximum.  The CTA then
//   writes the node arrays and the ancestor bitsets (one warp per row; each lane owns a
//   32-bit word).
#include "common.cuh"
#include "runtime.h"
#include "trace.h"

namespace df {

constexpr int kTopkThreads = 1024;
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
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n; i += kTopkThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long a = sel[i], b = sel[j];
          const bool desc = (i & size) == 0;
          if (desc ? (a < b) : (a > b)) { sel[i] = b; sel[j] = a; }
        }
      }
      __syncthreads();
    }
  }
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

// ----------------------------------------------------------------------------- chunked top-K
// Pass A: per (chunk, row) CTA, histogram of the top 12 key bits into hist[row][4096].
// Pass B: per (chunk, row) CTA, threshold bin t from hist (the bin holding the K-th
//         largest key); keys in bins above t go to hi[row] (all of them are selected),
//         keys in bin t to eq[row] (candidates), with per-row counters.
// Pass C: per row, the K - |hi| best candidates of eq by (key desc, id asc) join hi and
//         the K winners are sorted.  If eq overflowed, the row is redone by topk_row_full.
constexpr int kChunk = 8192;
constexpr int kCapEq = 4096;
constexpr int kChunkThreads = 512;

struct TopkScratch {     // per row
  uint32_t cnt_hi, cnt_eq, thr_bin, above;
};

__global__ void __launch_bounds__(kChunkThreads) topk_hist_kernel(const float* __restrict__ lp, int V,
                                                                  uint32_t* __restrict__ ghist, int* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t hist[4096];
  __shared__ uint32_t sh_nan;
  const size_t row = blockIdx.y;
  const float* x = lp + row * (size_t)V;
  for (int i = threadIdx.x; i < 4096; i += blockDim.x) hist[i] = 0;
  if (threadIdx.x == 0) sh_nan = 0;
  __syncthreads();
  const int i0 = blockIdx.x * kChunk, i1 = min(V, i0 + kChunk);
  for (int base = i0; base < i1; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const bool ok = i < i1;
    const float f = ok ? __ldg(x + i) : 0.f;
    const bool nan = ok && isnan(f);
    if (nan) sh_nan = 1;
    hist_add(hist, float_key(f) >> 20, ok && !nan);
  }
  __syncthreads();
  if (sh_nan && threadIdx.x == 0) set_status(status, DF_ERR_NAN, (int)row);
  uint32_t* g = ghist + row * 4096;
  for (int i = threadIdx.x; i < 4096; i += blockDim.x)
    if (hist[i]) atomicAdd(g + i, hist[i]);
}

__global__ void __launch_bounds__(kChunkThreads) topk_collect_kernel(const float* __restrict__ lp, int V, int K,
                                                                     const uint32_t* __restrict__ ghist,
                                                                     TopkScratch* __restrict__ sc,
                                                                     unsigned long long* __restrict__ hi,
                                                                     unsigned long long* __restrict__ eq) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t warp_tmp[32];
  __shared__ uint32_t sh_bin, sh_above;
  const size_t row = blockIdx.y;
  const uint32_t* h = ghist + row * 4096;
  // descending bins, 8 per thread (512 threads x 8 = 4096)
  uint32_t local = 0;
  for (int j = 0; j < 8; ++j) local += h[4095 - (threadIdx.x * 8 + j)];
  // inclusive scan over 512 threads
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t v = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < (kChunkThreads >> 5) ? warp_tmp[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < (kChunkThreads >> 5)) warp_tmp[lane] = w;
  }
  __syncthreads();
  const uint32_t incl = v + (warp ? warp_tmp[warp - 1] : 0u);
  const uint32_t excl = incl - local;
  if (excl < (uint32_t)K && (uint32_t)K <= incl) {
    uint32_t acc = excl;
    for (int j = 0; j < 8; ++j) {
      const int bin = 4095 - (threadIdx.x * 8 + j);
      if (acc + h[bin] >= (uint32_t)K) { sh_bin = bin; sh_above = acc; break; }
      acc += h[bin];
    }
  }
  __syncthreads();
  const uint32_t tb = sh_bin;
  if (blockIdx.x == 0 && threadIdx.x == 0) { sc[row].thr_bin = tb; sc[row].above = sh_above; }
  const float* x = lp + row * (size_t)V;
  const int i0 = blockIdx.x * kChunk, i1 = min(V, i0 + kChunk);
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const uint32_t k = float_key(__ldg(x + i));
    const uint32_t d = k >> 20;
    if (d < tb) continue;
    const unsigned long long c = ((unsigned long long)k << 32) | (uint32_t)(~(uint32_t)i);
    if (d > tb) {
      const uint32_t pos = atomicAdd(&sc[row].cnt_hi, 1u);
      if (pos < (uint32_t)kMaxK) hi[row * kMaxK + pos] = c;
    } else {
      const uint32_t pos = atomicAdd(&sc[row].cnt_eq, 1u);
      if (pos < (uint32_t)kCapEq) eq[row * kCapEq + pos] = c;
    }
  }
}

DF_DEV void bitonic_desc(unsigned long long* a, int n) {  // n power of two, block-wide
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long x = a[i], y = a[j];
          const bool desc = (i & size) == 0;
          if (desc ? (x < y) : (x > y)) { a[i] = y; a[j] = x; }
        }
      }
      __syncthreads();
    }
  }
}

template <bool kVec4>
__global__ void __launch_bounds__(kTopkThreads) topk_final_kernel(const float* __restrict__ lp, int V, int K,
                                                                  const TopkScratch* __restrict__ sc,
                                                                  const unsigned long long* __restrict__ hi,
                                                                  const unsigned long long* __restrict__ eq,
                                                                  int32_t* __restrict__ out_id,
                                                                  float* __restrict__ out_val, int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ unsigned long long cand[];  // [kCapEq] then [kMaxK]
  const size_t row = blockIdx.x;
  if (status && *(volatile int*)status == DF_ERR_NAN) return;
  const uint32_t n_eq = sc[row].cnt_eq, n_hi = sc[row].above;
  if (n_eq > (uint32_t)kCapEq) {  // threshold bin too crowded: whole-row path
    topk_row_full<kVec4>(lp, row, V, K, out_id, out_val, status);
    return;
  }
  unsigned long long* e = cand;
  unsigned long long* w = cand + kCapEq;
  int n = 1;
  while (n < (int)n_eq) n <<= 1;
  for (int i = threadIdx.x; i < n; i += blockDim.x) e[i] = i < (int)n_eq ? eq[row * kCapEq + i] : 0ull;
  int nk = 1;
  while (nk < K) nk <<= 1;
  for (int i = threadIdx.x; i < nk; i += blockDim.x) w[i] = i < (int)n_hi ? hi[row * kMaxK + i] : 0ull;
  __syncthreads();
  bitonic_desc(e, n);
  const int need = K - (int)n_hi;
  for (int i = threadIdx.x; i < need; i += blockDim.x) w[n_hi + i] = e[i];
  __syncthreads();
  bitonic_desc(w, nk);
  for (int r = threadIdx.x; r < K; r += blockDim.x) {
    const unsigned long long c = w[r];
    out_id[row * K + r] = (int32_t)(~(uint32_t)(c & 0xFFFFFFFFull));
    out_val[row * K + r] = key_float((uint32_t)(c >> 32));
  }
}

size_t topk_chunked_scratch_bytes(int rows) {
  return (size_t)rows * (4096 * 4 + sizeof(TopkScratch) + kMaxK * 8 + kCapEq * 8) + 1024;
}

// ----------------------------------------------------------------------------- heap
// 64-bit heap key, larger = earlier in the tree's total order:
//   [63:32] float_key(score)  [31:27] 31-depth  [26:16] 2047-parent  [15:5] 2047-rank
DF_DEV unsigned long long heap_key(float s, int depth, int parent, int rank) {
  return ((unsigned long long)float_key(s) << 32) | ((uint32_t)(31 - depth) << 27) |
         ((uint32_t)(2047 - parent) << 16) | ((uint32_t)(2047 - rank) << 5);
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
  const int W = (n + 31) / 32;
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
      unsigned long long best = cand[0];
      int bi = 0;
#pragma unroll
      for (int i = 1; i < NREG; ++i)
        if (cand[i] > best) { best = cand[i]; bi = i; }
      // warp maximum of the 64-bit lane maxima: the high words with one redux, then the low
      // words among the lanes that hold the top high word
      const uint32_t top_hi = __reduce_max_sync(0xffffffffu, (uint32_t)(best >> 32));
      const bool at_hi = (uint32_t)(best >> 32) == top_hi;
      const uint32_t top_lo = __reduce_max_sync(0xffffffffu, at_hi ? (uint32_t)best : 0u);
      const unsigned long long top = ((unsigned long long)top_hi << 32) | top_lo;
      const int owner = __ffs(__ballot_sync(0xffffffffu, best == top)) - 1;
      const int hole = __shfl_sync(0xffffffffu, bi, owner);
      // the last candidate moves into the hole (or the hole is the last one)
      const int last = cnt - 1, ll = last & 31, lr = last >> 5;
      unsigned long long lv = 0ull;
#pragma unroll
      for (int i = 0; i < NREG; ++i)
        if (i == lr) lv = cand[i];
      lv = __shfl_sync(0xffffffffu, lv, ll);
#pragma unroll
      for (int i = 0; i < NREG; ++i)
        if (lane == owner && i == hole) cand[i] = lv;
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
    DF_TRACE("topk", st);
    const int rows = b * D;
    if (chunk_scratch) {
      // chunked path: histogram, collect, final select (falls back per row when needed)
      unsigned char* base = static_cast<unsigned char*>(chunk_scratch);
      uint32_t* ghist = reinterpret_cast<uint32_t*>(base);
      TopkScratch* sc = reinterpret_cast<TopkScratch*>(ghist + (size_t)rows * 4096);
      unsigned long long* hi = reinterpret_cast<unsigned long long*>(
          (reinterpret_cast<uintptr_t>(sc + rows) + 255) & ~uintptr_t(255));
      unsigned long long* eq = hi + (size_t)rows * kMaxK;
      const size_t nzero = (size_t)rows * 4096 + (size_t)rows * (sizeof(TopkScratch) / 4);
      launch_k(zero_u32_kernel, dim3((unsigned)((nzero + 1023) / 1024 < 1024 ? (nzero + 1023) / 1024 : 1024)), dim3(1024), 0, st, 
          ghist, nzero);
      const dim3 grid((V + kChunk - 1) / kChunk, rows);
      launch_k(topk_hist_kernel, dim3(grid), dim3(kChunkThreads), 0, st, lp, V, ghist, status);
      launch_k(topk_collect_kernel, dim3(grid), dim3(kChunkThreads), 0, st, lp, V, K, ghist, sc, hi, eq);
      const size_t smem = (size_t)(kCapEq + kMaxK) * 8;
      if (ensure_dynamic_smem(topk_final_kernel<true>, smem) != cudaSuccess ||
          ensure_dynamic_smem(topk_final_kernel<false>, smem) != cudaSuccess)
        return DF_ERR_CUDA;
      if ((V & 3) == 0)
        launch_k(topk_final_kernel<true>, dim3(rows), dim3(kTopkThreads), smem, st, lp, V, K, sc, hi, eq, topk_id, topk_val, status);
      else
        launch_k(topk_final_kernel<false>, dim3(rows), dim3(kTopkThreads), smem, st, lp, V, K, sc, hi, eq, topk_id, topk_val, status);
    } else if ((V & 3) == 0) {
      launch_k(topk_rows_kernel<true>, dim3(rows), dim3(kTopkThreads), 0, st, lp, V, K, topk_id, topk_val, status);
    } else {
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
