// ddtree_build_static: the DDTree builder for callers that cannot hand the library a
// workspace.  Its scratch (the per-position top-K lists and a status word) is a fixed
// array in device memory that belongs to the library, so the call itself allocates
// nothing.  See include/dflash.h for the contract.
#include <mutex>

#include "common.cuh"
#include "nvtx.h"

namespace df {
int launch_ddtree(const float* lp, int b, int D, int V, int B, const int32_t* root_tok, int32_t* tok,
                  int32_t* parent, int32_t* depth, float* score, uint32_t* anc, int32_t* topk_id, float* topk_val,
                  int* status, cudaStream_t st, void* chunk_scratch);
size_t ddtree_heap_smem(int D, int K, int B);
}  // namespace df

namespace {

// Largest b * D * min(B, V) the fixed scratch holds (one int32 id + one fp32 value each).
constexpr long long kStaticTopkEntries = 1ll << 18;
constexpr size_t kHeaderBytes = 256;

// Loaded with the library on every device that uses it and kept until the process exits.
static __device__ __align__(256) unsigned char g_ddtree_scratch[kHeaderBytes + kStaticTopkEntries * 8];

// Device address of g_ddtree_scratch, looked up once per device (host code cannot use the
// symbol itself as a device pointer).
void* scratch_address(int* rc) {
  static std::mutex mu;
  static void* addr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    *rc = DF_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ddtree_scratch) != cudaSuccess || !p) {
      *rc = DF_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *rc = DF_OK;
  return addr[dev];
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int ddtree_build_static(const float* logprobs, int b, int D, int V, int B, const int32_t* root_tok,
                                   int32_t* tok, int32_t* parent, int32_t* depth, float* score, uint32_t* anc,
                                   df_stream stream) {
  DF_NVTX("ddtree_build_static");
  if (b < 0 || D < 1 || D > 31 || V < 2 || B < 0 || B > 2048) return DF_ERR_ARG;
  {
    double total = 0, p = 1;
    for (int k = 1; k <= D && total < 1e9; ++k) { p *= V; total += p; }
    if ((double)B > total) return DF_ERR_ARG;
  }
  if (b == 0) return DF_OK;
  if (!logprobs || !tok || !parent || !depth || !score || !anc) return DF_ERR_ARG;
  if (!al16(logprobs) || !al16(tok) || !al16(parent) || !al16(depth) || !al16(score) || !al16(anc)) return DF_ERR_ALIGN;
  const int K = B < V ? (B > 0 ? B : 1) : V;
  if ((long long)b * D * K > kStaticTopkEntries) return DF_ERR_WORKSPACE;  // beyond the fixed scratch
  if (df::ddtree_heap_smem(D, K, B) > 227 * 1024) return DF_ERR_SHAPE;
  int rc = DF_OK;
  unsigned char* base = static_cast<unsigned char*>(scratch_address(&rc));
  if (rc != DF_OK) return rc;
  cudaStream_t st = (cudaStream_t)stream;
  // The status word must read zero before the kernels run (a NaN left by an earlier call
  // would otherwise make the heap kernel skip its work).
  if (cudaMemsetAsync(base, 0, kHeaderBytes, st) != cudaSuccess) return DF_ERR_CUDA;
  int32_t* topk_id = reinterpret_cast<int32_t*>(base + kHeaderBytes);
  float* topk_val = reinterpret_cast<float*>(base + kHeaderBytes + (size_t)kStaticTopkEntries * 4);
  // the whole-row top-K path needs no scratch beyond the top-K lists
  return df::launch_ddtree(logprobs, b, D, V, B, root_tok, tok, parent, depth, score, anc, topk_id, topk_val,
                           reinterpret_cast<int*>(base), st, nullptr);
}
