// Shared device helpers for the sm_103a kernels: status word, bounded mbarrier waits,
// TMA (cp.async.bulk.tensor) loads, tcgen05 (TMEM allocation, MMA, commit, loads),
// and small numeric utilities.  Every wait is bounded by wall-clock time; on expiry the
// waiter records DF_ERR_TIMEOUT in the workspace status word and returns false, so no
// kernel here can spin forever.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/dflash.h"

#define DF_DEV __device__ __forceinline__
#define DF_HD __host__ __device__ __forceinline__

namespace df {

// --------------------------------------------------------------------------- status
struct WsHeader {        // first 256 bytes of every workspace
  int status;            // first device-side error code (0 = none)
  int detail;            // kernel-specific detail for that error
  unsigned long long wait_limit_ns;  // limit of every bounded wait (0 = kWaitLimitNs)
  int hold;              // test hook: nonzero makes each GEMM wait (bounded) for it to read 0
  int pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header size");
static_assert(offsetof(WsHeader, wait_limit_ns) == 8 && offsetof(WsHeader, hold) == 16, "header layout");

DF_DEV void set_status(int* status, int code, int detail = 0) {
  if (status && atomicCAS(status, 0, code) == 0) status[1] = detail;
}

DF_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// The wait limit of a workspace: its header's setting, else kWaitLimitNs.  Waits given no
// status word (the drains of a kernel that is giving up) always use kWaitLimitNs.
DF_DEV uint64_t wait_limit(const int* status) {
  if (!status) return kWaitLimitNs;
  const uint64_t l = *reinterpret_cast<const volatile unsigned long long*>(status + 2);
  return l ? l : kWaitLimitNs;
}

// --------------------------------------------------------------------------- smem / mbarrier
DF_DEV uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

DF_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
DF_DEV void fence_barrier_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
DF_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

DF_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar)) : "memory");
}
DF_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
DF_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Non-blocking probe of the same phase (try_wait may suspend the thread for a while).
DF_DEV bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of `bar` to complete.  Returns false (and records a
// timeout) if it does not complete within the workspace's wait limit (wait_limit).
DF_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, int* status, int where) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer(), limit = wait_limit(status);
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit) {
      set_status(status, DF_ERR_TIMEOUT, where);
      return false;
    }
    if (status && *(volatile int*)status == DF_ERR_TIMEOUT) return false;  // another role gave up
  }
}

// Test hook of the failure path: while the workspace header's `hold` word is nonzero the
// caller waits, bounded by the workspace's wait limit; returns false (and records
// DF_ERR_TIMEOUT) if the word is still set at the limit.  Nothing in the library sets the
// word, so a kernel that finds it set always times out, having issued no work.
DF_DEV bool wait_hold_clear(int* status, int where) {
  if (!status) return true;
  const volatile int* hold = status + 4;
  if (*hold == 0) return true;
  const uint64_t t0 = globaltimer(), limit = wait_limit(status);
  while (*hold != 0) {
    if (globaltimer() - t0 > limit) {
      set_status(status, DF_ERR_TIMEOUT, where);
      return false;
    }
    __nanosleep(1000);
  }
  return true;
}

// --------------------------------------------------------------------------- TMA
DF_DEV void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
DF_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
DF_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
DF_DEV void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
DF_DEV void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
        "l"(policy)
      : "memory");
}

// --------------------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor, K-major operand, 128-byte swizzle: rows of 64 bf16
// (128 B), 8-row swizzle atoms of 1024 B stacked at stride 1024 B.  Start addresses
// advance by 32 B per K=16 step inside the atom.
DF_DEV uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);        // start address
  d |= (uint64_t)(16 >> 4) << 16;                 // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;               // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                         // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                         // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                  // D format: f32
         | (1u << 7)                // A format: bf16
         | (1u << 10)               // B format: bf16
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

DF_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
DF_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
DF_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// One lane of a converged warp (the lowest active one), chosen with a warp-uniform
// predicate: MMAs issued under it keep their operand descriptors in warp-uniform values.
DF_DEV bool elect_one() {
  uint32_t r;
  asm volatile("{\n .reg .b32 x;\n .reg .pred p;\n elect.sync x|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(r));
  return r != 0;
}

DF_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DF_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, one instruction (K = 16 for bf16).
DF_DEV void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once all previously issued MMAs of this thread have completed.
DF_DEV void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns per thread.
DF_DEV void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
DF_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
DF_DEV void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
      : "memory");
}
// 32 lanes x 32 bits, 32 consecutive columns per thread.
DF_DEV void tmem_st32(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M x 16, bf16 pairs per 32-bit column) read from
// tensor memory.
DF_DEV void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
DF_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// --------------------------------------------------------------------------- dependent launch
// Every kernel of the library is launched with programmatic stream serialization: it may
// start while its predecessor in the stream is still running.  pdl_wait() blocks until the
// predecessor has completed and its memory is visible.  Each kernel calls pdl_trigger()
// only after its own pdl_wait(), so a successor can launch only once this kernel's
// predecessor is complete: code before pdl_wait() overlaps the immediate predecessor at
// most, and must not touch memory that the predecessor reads or writes.
DF_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DF_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// --------------------------------------------------------------------------- numerics
// Order-preserving map of fp32 onto uint32 (larger float -> larger key; -0 < +0).
DF_DEV uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
DF_DEV float key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

DF_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
DF_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 2^x with the hardware approximation (flush-to-zero), one MUFU operation.
DF_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Two floats -> packed bf16x2 (low = a), round to nearest even, one instruction.
DF_DEV uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

DF_DEV float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
DF_DEV uint16_t f_to_bf16(float f) {  // round to nearest even
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// --------------------------------------------------------------------------- drawing tokens
// Temperature-T draws of the target's token are Gumbel-max: argmax_v (logit_v / T + g_v),
// g_v = -log(-log u_v), with u_v from a counter-based generator keyed to (seed, sequence,
// position of the drawn token, v): the 32-bit finalizer of MurmurHash3 (A. Appleby, public
// domain) applied in a fixed chain.  Keying to the absolute position makes speculative
// decoding reproduce plain sampling under the same seed.
DF_HD uint32_t fmix32(uint32_t h) {
  h ^= h >> 16;
  h *= 0x85EBCA6Bu;
  h ^= h >> 13;
  h *= 0xC2B2AE35u;
  h ^= h >> 16;
  return h;
}
// Key of the draw for sequence s at absolute position n.
DF_HD uint32_t draw_key(uint64_t seed, int s, int n) {
  uint32_t a = fmix32((uint32_t)seed ^ (0x9E3779B9u * (uint32_t)(s + 1)));
  a = fmix32(a ^ (uint32_t)(seed >> 32));
  return fmix32(a + 0xC2B2AE35u * (uint32_t)n);
}
// g_v of token v for the draw keyed by k; u = (23 random bits + 1/2) / 2^23, exact in fp32
// and inside [2^-24, 1 - 2^-24].  The inner logarithm is the accurate one: for u near 1,
// -log u is tiny and an approximate logarithm's absolute error would dominate it.
DF_DEV float draw_noise(uint32_t k, int v) {
  const uint32_t h = fmix32(k ^ ((uint32_t)v * 0x27D4EB2Fu));
  const float u = ((float)(h >> 9) + 0.5f) * (1.f / 8388608.f);
  return -__logf(-logf(u));
}

}  // namespace df
