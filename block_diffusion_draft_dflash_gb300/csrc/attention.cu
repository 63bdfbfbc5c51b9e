// Attention of a block of query rows over a sequence's KV cache, on tcgen05 tensor cores.
//
// Serves both attention calls of the speculative step:
//   * tree verification (summary of "Accelerating Speculative Decoding with Block
//     Diffusion Draft Trees", section "방법론 자세히 보기"): every flattened tree row
//     sees the whole cache [0, N) and, among the tree's own slots N .. N+T-1, only its
//     ancestors and itself (bit j of its ancestor row);
//   * the drafter ("DFlash: Block Diffusion for Flash Speculative Decoding 논문 정리",
//     sections "DFlash의 핵심 아이디어" and "학습 방식도 추론 시나리오에 맞춰 바꿨다"):
//     every block row sees every injected context slot and every block row, no mask.
// Both are "dense prefix [0, dense_len) + optional ancestor-masked tail".
//
// Tile: 128 query rows = (128 / G) consecutive tree nodes x the G query heads that share
// one kv head (GQA), so one K/V tile feeds all 128 rows.  Per 128-key block:
//   S = Q K^T   (tcgen05.mma, M=128 N=128 K=128, accumulator in TMEM, triple-buffered)
//   softmax     (one TMEM lane = one query row, exp2 domain, running max / sum; the
//                ancestor mask is applied as 32-bit words per key group)
//   O += P V    (P written bf16 into TMEM over its own S, the MMA reading A from TMEM;
//                V stored transposed in the cache so that its tile is K-major)
// Warp roles: warps 0 .. 4 kCG - 1 softmax/epilogue (kCG warps per 32-row group, one per
// 128/kCG-column group, exchanging row maxima through shared memory), then a Q/K TMA
// producer warp, the TMEM owner + MMA issuer warp and a V TMA producer warp.  The MMA warp
// (in lockstep, one elected lane issuing) issues whichever product has its operands (S of a
// later block, or PV of the oldest block whose P is written), S first, so neither a late K
// nor a late V tile holds up the other product.
// The key range of a sequence is split over CTAs (split-KV) when the grid would
// otherwise not fill the GPU; partial (O, max, sum) are merged by attn_combine_kernel.
#include "attention.h"
#include "common.cuh"
#include "runtime.h"
#include "trace.h"

namespace df {

constexpr int kCG = 2;                       // column groups per query row (one warp each)
constexpr int kCols = 128 / kCG;             // S columns (keys) and O columns (head dims) per thread
constexpr int kSoftThreads = 128 * kCG;      // softmax / epilogue threads
constexpr int kTmaWarp = 4 * kCG, kMmaWarp = 4 * kCG + 1, kVWarp = 4 * kCG + 2;
constexpr int kAttnThreads = kSoftThreads + 96;  // + Q/K TMA warp, MMA warp, V TMA warp
constexpr int kKB = 128;     // keys per block
constexpr int kSBufs = 3;                    // S/P buffers in TMEM (128 columns each)
constexpr uint32_t kOCol = kSBufs * 128;     // O accumulator columns [384, 512)
constexpr int kKStages = 2;  // K tiles are free again once S = Q K^T has run
constexpr int kVStages = 3;  // V tiles are free again once O += P V has run (the longer wait)
constexpr uint32_t kTileBytes = 128 * 128 * 2;  // one 128x128 bf16 tile = 2 swizzled slabs

DF_DEV int floordiv32(int t) { return t >= 0 ? (t >> 5) : -((-t + 31) >> 5); }

// 32 ancestor bits for tail indices t0 .. t0+31 (bit c <-> t0 + c); out of range -> 0.
DF_DEV uint32_t anc_bits32(const uint32_t* row, int W, int t0) {
  const int w = floordiv32(t0);
  const int sh = t0 - 32 * w;
  const uint32_t lo = (w >= 0 && w < W) ? row[w] : 0u;
  const uint32_t hi = (w + 1 >= 0 && w + 1 < W) ? row[w + 1] : 0u;
  return sh ? ((lo >> sh) | (hi << (32 - sh))) : lo;
}

// Causal tail bits for tail indices t0 .. t0+31: set where 0 <= t <= node (a chain whose
// node i sees tail slots 0 .. i).
DF_DEV uint32_t causal_bits32(int t0, int node) {
  const int lo = t0 < 0 ? -t0 : 0;           // first bit with t >= 0
  const int hi = node - t0 + 1;              // bits below hi have t <= node
  if (hi <= lo || lo >= 32) return 0u;
  const uint32_t below_hi = hi >= 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u);
  const uint32_t from_lo = lo == 0 ? 0xFFFFFFFFu : ~((1u << lo) - 1u);
  return below_hi & from_lo;
}

// Dense bits for keys j0 .. j0+31: set where j < dense_len.
DF_DEV uint32_t dense_bits32(int j0, int dense_len) {
  const int n = dense_len - j0;
  return n >= 32 ? 0xFFFFFFFFu : (n <= 0 ? 0u : ((1u << n) - 1u));
}

// Named-barrier AND over the softmax threads (barrier 1): every thread gets the same
// answer, so the group leaves its loop together.
DF_DEV bool group_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r) : "r"((uint32_t)v), "r"(kSoftThreads) : "memory");
  return r != 0;
}
DF_DEV void group_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kSoftThreads) : "memory"); }

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* q_smem = smem;                                  // 32 KB
  unsigned char* k_smem = smem + kTileBytes;                     // kKStages x 32 KB
  unsigned char* v_smem = k_smem + kKStages * kTileBytes;        // kVStages x 32 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(v_smem + kVStages * kTileBytes);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kKStages;
  uint64_t* v_full = k_empty + kKStages;
  uint64_t* v_empty = v_full + kVStages;
  uint64_t* s_full = v_empty + kVStages;
  // One P barrier and one PV barrier per S buffer: each is reused only every third block,
  // which no waiter can fall a whole phase behind (a parity wait cannot tell phases two
  // apart).  Softmax of block j runs only after S_j, and S_j follows PV_{j-2} on the tensor
  // core, so at most PV_{j-1} is still pending when block j's softmax looks at O.
  uint64_t* p_full = s_full + kSBufs;
  uint64_t* o_done = p_full + kSBufs;
  uint64_t* mma_drain = o_done + kSBufs;  // completion of every MMA issued, when the issuer gives up
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  __shared__ float red_max[2][kCG][128];  // [block parity][column group][row]
  __shared__ float red_sum[kCG][128];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kKStages; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1); }
    for (int i = 0; i < kVStages; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1); }
    for (int i = 0; i < kSBufs; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < kSBufs; ++i) { mbar_init(&p_full[i], kSoftThreads); mbar_init(&o_done[i], 1); }
    mbar_init(mma_drain, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // everything below reads what earlier kernels wrote (q, the caches, the lengths)
  pdl_wait();
  pdl_trigger();
  // work unit -> (sequence, kv head, query tile, split)
  int u = blockIdx.x;
  const int split = u % p.nsplit; u /= p.nsplit;
  const int qt = u % p.n_qtiles; u /= p.n_qtiles;
  const int kvh = u % p.Hkv;
  const int s = u / p.Hkv;
  const int G = p.Hq / p.Hkv, NPT = 128 / G;
  const int dense_len = p.dense_len[s] + p.dense_add;
  // a causal chain: no row of this tile sees a tail slot past the tile's last node, so the
  // key blocks beyond it are not visited at all
  const int last_node = min(p.T, (qt + 1) * NPT) - 1;
  const int Lk = dense_len + (p.causal ? min(p.tail_len, last_node + 1) : p.tail_len);
  const int nb = (Lk + kKB - 1) / kKB;
  const int kb0 = (int)((long long)nb * split / p.nsplit), kb1 = (int)((long long)nb * (split + 1) / p.nsplit);
  const int nblk = kb1 - kb0;
  // TMEM: S/P of block j at cols 128 (j % 3) .. +127, O at 384-511.  P
  // (bf16 pairs) overwrites its own S in place: column group g at cols [g kCols, g kCols + kCols/2).
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp || warp == kVWarp) {
    // ------------------------------------------------------------ TMA producers
    // One warp loads Q and the K tiles, another the V tiles: a wait for a free K slot never
    // holds up a V load, or the other way round.
    if (lane == 0 && nblk > 0) {
      const uint64_t pol_q = policy_evict_first(), pol_kv = policy_evict_last();
      const int plane = s * p.Hkv + kvh;
      const bool is_k = warp == kTmaWarp;
      if (is_k) {
        mbar_arrive_expect_tx(q_full, kTileBytes);
        const int qz = s * p.T + qt * NPT;
        tma_load_3d(q_smem, &tmQ, q_full, 0, kvh * G, qz, pol_q);
        tma_load_3d(q_smem + kTileBytes / 2, &tmQ, q_full, 64, kvh * G, qz, pol_q);
      }
      const int NS = is_k ? kKStages : kVStages;
      uint64_t* fullb = is_k ? k_full : v_full;
      uint64_t* emptyb = is_k ? k_empty : v_empty;
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % NS;
        if (!mbar_wait(&emptyb[st], ((j / NS) & 1) ^ 1, p.status, is_k ? 11 : 15)) break;
        const int key0 = (kb0 + j) * kKB;
        mbar_arrive_expect_tx(&fullb[st], kTileBytes);
        if (is_k) {
          unsigned char* kb = k_smem + st * kTileBytes;
          tma_load_2d(kb, &tmK, &fullb[st], 0, plane * p.cap + key0, pol_kv);
          tma_load_2d(kb + kTileBytes / 2, &tmK, &fullb[st], 64, plane * p.cap + key0, pol_kv);
        } else {
          unsigned char* vb = v_smem + st * kTileBytes;
          tma_load_2d(vb, &tmV, &fullb[st], key0, plane * 128, pol_kv);
          tma_load_2d(vb + kTileBytes / 2, &tmV, &fullb[st], key0 + 64, plane * 128, pol_kv);
        }
        ++issued;
      }
      // every load issued must have landed before the CTA may exit, also when the MMA issuer
      // gave up before consuming it (bounded waits; already complete in normal runs)
      if (is_k) mbar_wait(q_full, 0, nullptr, 0);
      for (int j = issued - NS > 0 ? issued - NS : 0; j < issued; ++j)
        mbar_wait(&fullb[j % NS], (j / NS) & 1, nullptr, 0);
    }
  } else if (warp == kMmaWarp) {
    if (nblk > 0) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the issue loop in lockstep (every decision is a warp vote), so
      // the operand descriptors are warp-uniform values; one elected lane issues the MMAs
      // and their commits.
      const uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t qa = smem_u32(q_smem);
      const bool leader = elect_one();
      bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, p.status, 12));
      tc_fence_after();
      // operands already present: issue only
      auto issue_pv = [&](int j) {
        tc_fence_after();
        const uint32_t vb = smem_u32(v_smem + (j % kVStages) * kTileBytes);
        const uint32_t pt = tmem + (j % kSBufs) * 128;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {  // keys 16kk..16kk+15: P of column group 16kk / kCols
            constexpr int kPer = kCols / 16;  // 16-key steps per column group
            const uint32_t boff = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
            mma_bf16_ts(tmem + kOCol, pt + (kk / kPer) * kCols + (kk % kPer) * 8, sdesc_kmajor_sw128(vb + boff), idesc,
                        (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&o_done[j % kSBufs]);
          mma_commit(&v_empty[j % kVStages]);
        }
        __syncwarp();
      };
      auto issue_s = [&](int j) {
        tc_fence_after();
        const int st = j % kKStages;
        const uint32_t kb = smem_u32(k_smem + st * kTileBytes);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
            mma_bf16(tmem + (j % kSBufs) * 128, sdesc_kmajor_sw128(qa + off), sdesc_kmajor_sw128(kb + off), idesc,
                     kk > 0 ? 1u : 0u);
          }
          mma_commit(&s_full[j % kSBufs]);
          mma_commit(&k_empty[st]);
        }
        __syncwarp();
      };
      // Whichever product has its operands goes next, S first (its scores gate the next
      // softmax block), so a late K tile never holds up a ready PV or the other way round.
      // S_k reuses the buffer of block k - 3, so it waits until PV_{k-3} has been issued:
      // the tensor core runs one CTA's MMAs in issue order, so a buffer is rewritten only
      // after its P was read, and S_k complete implies every PV up to k - 3 complete.
      // A barrier phase seen complete by any lane is complete, so each test is an any-vote.
      int s_next = 0, pv_next = 0, idle = 0;
      uint64_t t_idle = 0;  // time of the first idle check since the last issue (0: none yet)
      const uint64_t limit = wait_limit(p.status);
      while (ok && pv_next < nblk) {
        if (s_next < nblk && s_next - pv_next < kSBufs &&
            __any_sync(0xffffffffu, mbar_test_wait(&k_full[s_next % kKStages], (s_next / kKStages) & 1))) {
          issue_s(s_next++);
        } else if (pv_next < s_next &&
                   __any_sync(0xffffffffu, mbar_test_wait(&p_full[pv_next % kSBufs], (pv_next / kSBufs) & 1) &&
                                               mbar_test_wait(&v_full[pv_next % kVStages], (pv_next / kVStages) & 1))) {
          issue_pv(pv_next++);
        } else {
          if ((++idle & 1023) == 0) {  // bounded: give up after the wait limit without progress
            const uint64_t now = __shfl_sync(0xffffffffu, globaltimer(), 0);
            if (t_idle == 0) t_idle = now;
            else if (now - t_idle > limit) {
              if (leader) set_status(p.status, DF_ERR_TIMEOUT, 13);
              ok = false;
            }
            if (__any_sync(0xffffffffu, p.status && *(volatile int*)p.status == DF_ERR_TIMEOUT)) ok = false;
          }
          continue;
        }
        idle = 0;
        t_idle = 0;
      }
      if (!ok && (s_next > 0 || pv_next > 0)) {
        // giving up: the MMAs already issued must finish before TMEM is freed
        if (leader) mma_commit(mma_drain);
        __syncwarp();
        mbar_wait(mma_drain, 0, nullptr, 0);
      }
    }
  } else {
    // ------------------------------------------------ softmax / epilogue (warps 0 .. 4 kCG - 1)
    // Warp w owns TMEM lanes 32*(w%4)..+31 (one query row per thread) and column group
    // g = w/4: S columns [g kCols, (g+1) kCols) (keys) and the same O columns (head dims).
    const int grp = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // query row == TMEM lane
    const int node = qt * NPT + r / G, head = kvh * G + r % G;
    const bool row_ok = node < p.T;
    const bool warp_live = __any_sync(0xffffffffu, row_ok);
    const uint32_t* anc_row = (p.anc && row_ok) ? p.anc + ((size_t)s * p.T + node) * p.W : nullptr;
    const float scale2 = p.scale * 1.4426950408889634f;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float m_run = -INFINITY, l_part = 0.f;
    bool ok = true;
    // Lazy rescaling: the running max m_run (raw-score units) only moves when a block raises
    // the row max by more than 8 in log2 units; P = 2^(scale2 (s - m_run)) then stays below
    // 2^8, and O and the running sum are rescaled only on those rare moves.
    constexpr float kRescale = 8.f;
    for (int j = 0; j < nblk; ++j) {
      // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
      const bool w1 = __all_sync(0xffffffffu, mbar_wait(&s_full[j % kSBufs], (j / kSBufs) & 1, p.status, 16));
      float sv[kCols];
      float mpart = -INFINITY;
      const uint32_t sp = tmem + lane_base + (j % kSBufs) * 128 + grp * kCols;  // this group's S (then P)
      if (w1) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kCols; c += 16) tmem_ld16(sp + c, sv + c);
        tmem_ld_wait();
        // Raw scores; the softmax scale is folded into the exponent below.  Only blocks
        // that reach past the dense prefix need the admission mask.
        const int key0 = (kb0 + j) * kKB + grp * kCols;
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if ((kb0 + j + 1) * kKB > dense_len) {
          uint32_t adm[kCols / 32];
#pragma unroll
          for (int g = 0; g < kCols / 32; ++g) {
            const int j0 = key0 + 32 * g;
            uint32_t bits = row_ok ? dense_bits32(j0, dense_len) : 0u;
            if (anc_row) bits |= anc_bits32(anc_row, p.W, j0 - dense_len);
            else if (p.causal && row_ok) bits |= causal_bits32(j0 - dense_len, node);
            adm[g] = bits;
          }
#pragma unroll
          for (int c = 0; c < kCols; ++c) {
            if (!((adm[c >> 5] >> (c & 31)) & 1u)) sv[c] = -INFINITY;
            m4[c & 3] = fmaxf(m4[c & 3], sv[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < kCols; ++c) m4[c & 3] = fmaxf(m4[c & 3], sv[c]);
        }
        mpart = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      } else {
#pragma unroll
        for (int c = 0; c < kCols; ++c) sv[c] = -INFINITY;
      }
      red_max[j & 1][grp][r] = mpart;
      if (!group_and(w1 && ok)) { ok = false; break; }  // uniform across the softmax threads
      float mx = red_max[j & 1][0][r];  // raw-score units
#pragma unroll
      for (int g = 1; g < kCG; ++g) mx = fmaxf(mx, red_max[j & 1][g][r]);
      float alpha = 1.f;
      if ((mx - m_run) * scale2 > kRescale) {  // also taken on the first admitted key (m_run = -inf)
        alpha = ex2_approx((m_run - mx) * scale2);  // 0 when m_run = -inf
        m_run = mx;
      }
      uint32_t packed[kCols / 2];
      if (warp_live && m_run != -INFINITY) {
        const float mb = -m_run * scale2;
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < kCols; c += 4) {  // three additions per four probabilities
          const float p0 = ex2_approx(fmaf(sv[c], scale2, mb)), p1 = ex2_approx(fmaf(sv[c + 1], scale2, mb));
          const float p2 = ex2_approx(fmaf(sv[c + 2], scale2, mb)), p3 = ex2_approx(fmaf(sv[c + 3], scale2, mb));
          s4[(c >> 2) & 3] += (p0 + p1) + (p2 + p3);
          packed[c >> 1] = pack_bf16x2(p0, p1);
          packed[(c >> 1) + 1] = pack_bf16x2(p2, p3);
        }
        l_part = l_part * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
      } else {
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) packed[c] = 0u;
      }
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O must hold PV of every earlier block before it is rescaled
        ok = mbar_wait(&o_done[(j - 1) % kSBufs], ((j - 1) / kSBufs) & 1, p.status, 17) && ok;
        tc_fence_after();
        const uint32_t oaddr = tmem + lane_base + kOCol + grp * kCols;
#pragma unroll
        for (int c = 0; c < kCols; c += 16) {
          float o[16];
          tmem_ld16(oaddr + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= alpha;
          tmem_st16(oaddr + c, o);
        }
      }
      // P over this group's (already loaded) S columns
      static_assert(kCols == 32 || kCols == 64, "column groups of 32 or 64");
      if constexpr (kCols == 64) {
        tmem_st32(sp, packed);
      } else {
        float pf[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pf[i] = __uint_as_float(packed[i]);
        tmem_st16(sp, pf);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[j % kSBufs]);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok && nblk > 0) ok = mbar_wait(&o_done[(nblk - 1) % kSBufs], ((nblk - 1) / kSBufs) & 1, p.status, 18);
    tc_fence_after();
    red_sum[grp][r] = l_part;
    group_sync();
    float l_run = red_sum[0][r];
#pragma unroll
    for (int g = 1; g < kCG; ++g) l_run += red_sum[g][r];
    const size_t grow = ((size_t)s * p.T + node) * p.Hq + head;  // global query row
    const uint32_t oaddr = tmem + lane_base + kOCol + grp * kCols;
    if (p.nsplit == 1) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(p.out + grow * 128 + grp * kCols);
#pragma unroll
      for (int c = 0; c < kCols; c += 16) {
        float o[16];
        if (nblk > 0) { tmem_ld16(oaddr + c, o); tmem_ld_wait(); }
        else {
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = 0.f;
        }
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = (uint32_t)f_to_bf16(o[2 * i] * inv) | ((uint32_t)f_to_bf16(o[2 * i + 1] * inv) << 16);
        if (row_ok) {
          dst[c / 8] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[c / 8 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    } else {
      const size_t nrows = (size_t)p.b * p.T * p.Hq;
      float* op = p.o_part + ((size_t)split * nrows + grow) * 128 + grp * kCols;
#pragma unroll
      for (int c = 0; c < kCols; c += 16) {
        float o[16];
        if (nblk > 0) { tmem_ld16(oaddr + c, o); tmem_ld_wait(); }
        else {
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = 0.f;
        }
        if (row_ok)
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(op + c + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
      }
      if (row_ok && grp == 0) {
        p.ml_part[((size_t)split * nrows + grow) * 2] = m_run * scale2;  // log2 units for the combine
        p.ml_part[((size_t)split * nrows + grow) * 2 + 1] = l_run;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) {
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
}

// One warp per query row: out = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j.
constexpr int kCombineFast = 4;  // splits merged from one round of loads
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ ml_part, int nsplit,
                                                           long long nrows, df_bf16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (nsplit <= kCombineFast) {
    // every split's (max, sum) and O slice in one round of (predicated) loads
    float m[kCombineFast], l[kCombineFast];
    float4 o[kCombineFast];
#pragma unroll
    for (int j = 0; j < kCombineFast; ++j) {
      const bool on = j < nsplit;
      const size_t at = (size_t)j * nrows + row;
      m[j] = on ? ml_part[at * 2] : -INFINITY;
      l[j] = on ? ml_part[at * 2 + 1] : 0.f;
      o[j] = on ? reinterpret_cast<const float4*>(o_part + at * 128)[lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float M = m[0];
#pragma unroll
    for (int j = 1; j < kCombineFast; ++j) M = fmaxf(M, m[j]);
#pragma unroll
    for (int j = 0; j < kCombineFast; ++j) {
      const float w = m[j] == -INFINITY ? 0.f : exp2f(m[j] - M);
      L += w * l[j];
      acc.x += w * o[j].x; acc.y += w * o[j].y; acc.z += w * o[j].z; acc.w += w * o[j].w;
    }
  } else {
    float M = -INFINITY;
    for (int j = 0; j < nsplit; ++j) M = fmaxf(M, ml_part[((size_t)j * nrows + row) * 2]);
    for (int j = 0; j < nsplit; ++j) {
      const float m = ml_part[((size_t)j * nrows + row) * 2];
      if (m == -INFINITY) continue;
      const float w = exp2f(m - M);
      L += w * ml_part[((size_t)j * nrows + row) * 2 + 1];
      const float4 o = reinterpret_cast<const float4*>(o_part + ((size_t)j * nrows + row) * 128)[lane];
      acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint2 r;
  r.x = (uint32_t)f_to_bf16(acc.x * inv) | ((uint32_t)f_to_bf16(acc.y * inv) << 16);
  r.y = (uint32_t)f_to_bf16(acc.z * inv) | ((uint32_t)f_to_bf16(acc.w * inv) << 16);
  reinterpret_cast<uint2*>(out + row * 128)[lane] = r;
}

// ----------------------------------------------------------------------------- host
static int make_tmap(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                     const cuuint32_t* box) {
  typedef CUresult (*Fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*, const cuuint64_t*,
                         const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                         CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Fn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return DF_ERR_CUDA;
    fn = reinterpret_cast<Fn>(f);
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DF_OK : DF_ERR_CUDA;
}

int attn_num_splits(int b, int Hkv, int n_qtiles, int max_keys) {
  const int units = b * Hkv * n_qtiles;
  const int nsm = num_sms();
  const int nb = (max_keys + kKB - 1) / kKB;
  // fill one wave: as many splits as whole copies of the unit set fit on the SMs
  int ns = units >= nsm ? 1 : nsm / units;
  if (ns > nb) ns = nb;
  if (ns > kAttnMaxSplits) ns = kAttnMaxSplits;
  if (ns < 1) ns = 1;
  return ns;
}

int launch_attention(const AttnArgs& a, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  const int NPT = 128 / G;
  const int n_qtiles = (a.T + NPT - 1) / NPT;
  CUtensorMap tq, tk, tv;
  {
    cuuint64_t dims[3] = {128, (cuuint64_t)a.Hq, (cuuint64_t)a.b * a.T};
    cuuint64_t str[2] = {(cuuint64_t)128 * 2, (cuuint64_t)a.Hq * 128 * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)NPT};
    if (make_tmap(&tq, a.q, 3, dims, str, box)) return DF_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {128, (cuuint64_t)a.b * a.Hkv * a.cap};
    cuuint64_t str[1] = {(cuuint64_t)128 * 2};
    cuuint32_t box[2] = {64, 128};
    if (make_tmap(&tk, a.k_plane, 2, dims, str, box)) return DF_ERR_CUDA;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.cap, (cuuint64_t)a.b * a.Hkv * 128};
    cuuint64_t str[1] = {(cuuint64_t)a.cap * 2};
    cuuint32_t box[2] = {64, 128};
    if (make_tmap(&tv, a.v_plane, 2, dims, str, box)) return DF_ERR_CUDA;
  }
  AttnParams p{};
  p.b = a.b; p.T = a.T; p.Hq = a.Hq; p.Hkv = a.Hkv; p.cap = a.cap;
  p.dense_len = a.dense_len; p.dense_add = a.dense_add; p.tail_len = a.tail_len;
  p.anc = a.anc; p.W = a.anc ? (a.tail_len + 31) / 32 : 0;
  p.causal = a.anc ? 0 : a.causal;
  p.scale = a.scale;
  p.n_qtiles = n_qtiles;
  p.nsplit = a.nsplit;
  p.out = a.out; p.o_part = a.o_part; p.ml_part = a.ml_part;
  p.status = a.status;
  const size_t smem = 1024 + kTileBytes * (1 + kKStages + kVStages) + 256;
  if (ensure_dynamic_smem(attn_tc_kernel, smem) != cudaSuccess) return DF_ERR_CUDA;
  const int grid = a.b * a.Hkv * n_qtiles * a.nsplit;
  {
    DF_TRACE(a.anc ? "attention_tree" : a.causal ? "attention_causal" : "attention_draft", st);
    launch_k(attn_tc_kernel, dim3(grid), dim3(kAttnThreads), smem, st, tq, tk, tv, p);
  }
  if (cudaGetLastError() != cudaSuccess) return DF_ERR_CUDA;
  if (a.nsplit > 1) {
    DF_TRACE("attention_combine", st);
    const long long nrows = (long long)a.b * a.T * a.Hq;
    launch_k(attn_combine_kernel, dim3((unsigned)((nrows + 7) / 8)), dim3(256), 0, st, a.o_part, a.ml_part, a.nsplit, nrows, a.out);
    if (cudaGetLastError() != cudaSuccess) return DF_ERR_CUDA;
  }
  return DF_OK;
}

size_t attn_partial_bytes(int b, int T, int Hq, int nsplit) {
  const size_t rows = (size_t)b * T * Hq;
  return nsplit > 1 ? rows * nsplit * (128 * 4 + 8) : 0;
}

}  // namespace df
