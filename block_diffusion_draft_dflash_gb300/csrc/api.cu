// C ABI entry points (include/dflash.h): argument checks, workspace carving and the
// launch sequences of the composite calls.  No device memory is allocated here.
#include <stdio.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "attention.h"
#include "common.cuh"
#include "gemm.h"
#include "layers.h"
#include "moe.h"
#include "nvtx.h"

namespace df {
int launch_ddtree(const float* lp, int b, int D, int V, int B, const int32_t* root_tok, int32_t* tok,
                  int32_t* parent, int32_t* depth, float* score, uint32_t* anc, int32_t* topk_id, float* topk_val,
                  int* status, cudaStream_t st, void* chunk_scratch);
size_t ddtree_heap_smem(int D, int K, int B);
int launch_chain(const float* lp, int b, int D, int V, const int32_t* root_tok, int32_t* tok, int32_t* parent,
                 int32_t* depth, float* score, uint32_t* anc, unsigned long long* keys, int* status, cudaStream_t st);
size_t topk_chunked_scratch_bytes(int rows);
size_t accept_scratch_bytes(int b);
int launch_accept(int b, int n_tree, const int32_t* choice, const int32_t* tok, const int32_t* parent,
                  df_bf16* k_cache, df_bf16* v_cache, int n_layers, int Hkv, int cap, int32_t* cache_len,
                  const df_bf16* tree_feat, int feat_dim, df_bf16* new_feat, int max_new, int32_t* n_new,
                  int32_t* acc_tok, int32_t* n_acc, int32_t* new_bonus, int32_t* src_slot, void* scratch,
                  int* status, cudaStream_t st);

namespace {

constexpr size_t kAlign = 256;
inline size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Bump allocator over a caller-provided workspace (or a size counter when base is null).
struct Carver {
  unsigned char* base;
  size_t off = kAlign;  // the first 256 bytes hold the status header
  explicit Carver(void* b) : base(static_cast<unsigned char*>(b)) {}
  template <class T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = up(off + count * sizeof(T));
    return p;
  }
};

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
inline int* status_of(void* ws) { return reinterpret_cast<int*>(ws); }

#define DF_TRY(x)            \
  do {                       \
    int _rc = (x);           \
    if (_rc != DF_OK) return _rc; \
  } while (0)

// Router GEMM (E <= 256 weight rows): each CTA takes at least this many k-steps.
constexpr int kRouterMinK = 4;

bool cfg_ok(const df_model_cfg* c) {
  if (!c || c->n_experts < 0) return false;
  const bool moe = c->n_experts > 0;
  if (moe && (c->n_experts % 32 || c->n_experts > 256 || c->top_k < 1 || c->top_k > 32 || c->top_k > c->n_experts ||
              c->d_expert <= 0 || c->d_expert % 64 || c->d_model % 256))
    return false;
  return c->n_layers > 0 && c->d_model > 0 && c->d_model % 64 == 0 && c->head_dim == 128 && c->n_kv_heads > 0 &&
         c->n_q_heads % c->n_kv_heads == 0 && (128 % (c->n_q_heads / c->n_kv_heads)) == 0 &&
         (c->n_q_heads / c->n_kv_heads) <= 8 && (moe || (c->d_ff > 0 && c->d_ff % 64 == 0)) && c->vocab >= 2 &&
         c->n_feat_layers >= 0 && c->n_feat_layers <= 8;
}

struct LayerBufs {
  float* h;         // [R][d] residual stream
  df_bf16* x;       // [Rx][d] normed GEMM input (query rows, then context rows)
  df_bf16* q;       // [R][Hq*hd]
  df_bf16* attn;    // [R][Hq*hd]
  df_bf16* act;     // [R][F]
  float* part;      // GEMM partial-tile slots, reused by every projection
  float* o_part;    // attention split-KV partials
  float* ml_part;
  float2* rope;     // [Rx][64] rotary (cos, sin) of every q/k/v row, filled once per forward
  MoeBufs moe;      // mixture-of-experts layers only
};

int nsplit_for(int b, int T, int Hq, int Hkv, int max_keys) {
  const int G = Hq / Hkv, NPT = 128 / G;
  return attn_num_splits(b, Hkv, (T + NPT - 1) / NPT, max_keys);
}

// Largest partial-slot buffer any projection of a layer needs.
size_t layer_partial_bytes(const df_model_cfg* c, int R, int Rx) {
  const int d = c->d_model, F = c->d_ff, qd = c->n_q_heads * 128, nqkv = (c->n_q_heads + 2 * c->n_kv_heads) * 128;
  size_t m = gemm_partial_bytes(Rx, nqkv, d);
  m = std::max(m, gemm_partial_bytes(R, d, qd));
  if (c->n_experts > 0) {
    m = std::max(m, gemm_partial_bytes(R, c->n_experts, d, kRouterMinK));  // router logits
  } else {
    m = std::max(m, gemm_partial_bytes(R, 2 * F, d));
    m = std::max(m, gemm_partial_bytes(R, d, F));
  }
  return m;
}

// One pre-norm decoder layer over R query rows; x already holds RMSNorm(h) * attn_norm
// for them (and the context rows R .. Rx-1, which only enter the q/k/v projection).
// Each projection writes partial tiles that the next kernel reduces and consumes:
//   q/k/v -> q/k norm + rotation + cache;  o -> residual + RMSNorm;
//   gate/up -> SwiGLU;  down -> residual + the next RMSNorm (+ feature capture).
struct LayerRun {
  const df_model_cfg* cfg;
  const df_layer_weights* w;
  int layer;           // index in the model
  int b, T;            // R = b*T query rows
  int Rx;              // rows of the q/k/v projection (R plus context rows)
  QkRopeArgs qk;       // filled except the layer-specific fields
  AttnArgs at;         // filled except q/k/v/out
  ResNormArgs out;     // down consumer: gain, destination rows and mapping, capture
  int* status;
};

int run_layer(const LayerRun& L, LayerBufs& B, cudaStream_t st) {
  const df_model_cfg& c = *L.cfg;
  const int d = c.d_model, hd = 128, Hq = c.n_q_heads, Hkv = c.n_kv_heads, F = c.d_ff;
  const int nqkv = (Hq + 2 * Hkv) * hd;
  const int R = L.b * L.T;
  PartialView pv{};
  GemmDesc g{};
  g.X = B.x; g.W = L.w->w_qkv; g.M = L.Rx; g.N = nqkv; g.K = d; g.ldx = d; g.ldw = d;
  g.mode = kGemmPartial; g.part = B.part; g.view = &pv; g.status = L.status;
  DF_TRY(launch_gemm(g, st));
  QkRopeArgs qk = L.qk;
  qk.qkv = nullptr; qk.pv = pv; qk.ld_qkv = nqkv; qk.q_norm = L.w->q_norm; qk.k_norm = L.w->k_norm; qk.q_out = B.q;
  qk.rope = B.rope;
  DF_TRY(launch_qk_rope(qk, st));
  AttnArgs at = L.at;
  at.q = B.q; at.k_plane = qk.k_plane; at.v_plane = qk.v_plane; at.out = B.attn;
  at.o_part = B.o_part; at.ml_part = B.ml_part;
  DF_TRY(launch_attention(at, st));
  g = GemmDesc{};
  g.X = B.attn; g.W = L.w->w_o; g.M = R; g.N = d; g.K = Hq * hd; g.ldx = Hq * hd; g.ldw = Hq * hd;
  g.mode = kGemmPartial; g.part = B.part; g.view = &pv; g.status = L.status;
  DF_TRY(launch_gemm(g, st));
  ResNormArgs rn{};
  rn.pv = pv; rn.h = B.h; rn.d = d; rn.gain = L.w->mlp_norm; rn.eps = c.rms_eps; rn.out = B.x; rn.ld_out = d;
  rn.rows = R; rn.group_out = 1; rn.group_in = 1; rn.in_off = 0;
  DF_TRY(launch_res_norm(rn, st));
  if (c.n_experts > 0) {
    // mixture of experts: router logits -> top-k routing -> expert order -> grouped expert
    // products (SwiGLU fused into the gate/up one) -> weighted combine + residual + next norm
    g = GemmDesc{};
    g.X = B.x; g.W = L.w->w_router; g.M = R; g.N = c.n_experts; g.K = d; g.ldx = d; g.ldw = d;
    g.mode = kGemmPartial; g.part = B.part; g.view = &pv; g.status = L.status;
    g.min_k_per_cta = kRouterMinK;  // a weight of E <= 256 rows: a few pieces per tile, not one per CTA
    DF_TRY(launch_gemm(g, st));
    MoeBufs m = B.moe;
    m.counts += (size_t)L.layer * c.n_experts;  // each layer's expert counts are kept
    DF_TRY(launch_moe_route(pv, R, c.n_experts, c.top_k, m, L.status, st));
    DF_TRY(launch_moe_dispatch(B.x, R, d, c.n_experts, c.top_k, c.d_expert, m, L.status, st));
    DF_TRY(launch_moe_experts(L.w->w_experts_gate_up, L.w->w_experts_down, R, d, c.n_experts, c.top_k, c.d_expert,
                              m, L.status, st));
    rn = L.out;
    rn.h = B.h; rn.d = d; rn.eps = c.rms_eps;
    return launch_moe_combine(m, c.top_k, R * c.top_k, rn, L.status, st);
  }
  g = GemmDesc{};
  g.X = B.x; g.W = L.w->w_gate_up; g.M = R; g.N = 2 * F; g.K = d; g.ldx = d; g.ldw = d;
  g.mode = kGemmPartial; g.part = B.part; g.view = &pv; g.status = L.status;
  DF_TRY(launch_gemm(g, st));
  SwigluArgs sw{};
  sw.pv = pv; sw.rows = R; sw.F = F; sw.act = B.act;
  DF_TRY(launch_swiglu_partial(sw, st));
  g = GemmDesc{};
  g.X = B.act; g.W = L.w->w_down; g.M = R; g.N = d; g.K = F; g.ldx = F; g.ldw = F;
  g.mode = kGemmPartial; g.part = B.part; g.view = &pv; g.status = L.status;
  DF_TRY(launch_gemm(g, st));
  rn = L.out;
  rn.pv = pv; rn.h = B.h; rn.d = d; rn.eps = c.rms_eps;
  DF_TRY(launch_res_norm(rn, st));
  return DF_OK;
}

// ---------------------------------------------------------------------------- layouts
struct TargetWs {
  LayerBufs B;
  unsigned long long* amax;
  uint32_t* draw_key;  // per-row keys of the LM head's temperature draw
};
size_t target_ws(const df_model_cfg* c, int b, int n_tree, void* base, TargetWs* out) {
  const int d = c->d_model, Hq = c->n_q_heads, Hkv = c->n_kv_heads, F = c->d_ff;
  const size_t R = (size_t)b * n_tree;
  Carver cv(base);
  TargetWs w{};
  w.B.h = cv.take<float>(R * d);
  w.B.x = cv.take<df_bf16>(R * d);
  w.B.q = cv.take<df_bf16>(R * Hq * 128);
  w.B.attn = cv.take<df_bf16>(R * Hq * 128);
  w.B.act = cv.take<df_bf16>(R * (c->n_experts > 0 ? 1 : F));
  w.B.part = cv.take<float>(layer_partial_bytes(c, (int)R, (int)R) / 4 + 1);
  w.amax = cv.take<unsigned long long>(R);
  w.draw_key = cv.take<uint32_t>(R);
  if (c->n_experts > 0) {
    size_t sz[kMoeBufCount];
    moe_buf_elems((int)R, c->top_k, c->n_experts, d, c->d_expert, sz);
    sz[2] *= c->n_layers;  // expert counts of every layer
    MoeBufs& m = w.B.moe;
    m.topk_id = cv.take<int32_t>(sz[0] / 4);
    m.topk_w = cv.take<float>(sz[1] / 4);
    m.counts = cv.take<int32_t>(sz[2] / 4);
    m.offsets = cv.take<int32_t>(sz[3] / 4);
    m.pos_of = cv.take<int32_t>(sz[4] / 4);
    m.pair_token = cv.take<int32_t>(sz[5] / 4);
    m.xp = cv.take<df_bf16>(sz[6] / 2);
    m.act = cv.take<df_bf16>(sz[7] / 2);
    m.out = cv.take<float>(sz[8] / 4);
    m.chunks = cv.take<int4>(sz[9] / 16);
    m.n_chunks = cv.take<int32_t>(sz[10] / 4);
  }
  w.B.rope = cv.take<float2>(R * 64);
  // split-KV partials sized for the largest split this call could choose (cache up to 2^20 keys)
  const int ns = nsplit_for(b, n_tree, Hq, Hkv, 1 << 20);
  const size_t pb = attn_partial_bytes(b, n_tree, Hq, ns);
  w.B.o_part = cv.take<float>(pb / 4);
  w.B.ml_part = w.B.o_part ? w.B.o_part + (size_t)ns * R * Hq * 128 : nullptr;
  if (out) *out = w;
  return cv.off;
}

struct DraftWs {
  LayerBufs B;
  df_bf16* xl;        // [b*(L-1)][d]
  int32_t* len_new;   // [b]
  float* stats;       // [b*(L-1)][4*ceil(V/128)][2] LM-head softmax partials
  float* lse;         // [b*(L-1)]
};
size_t draft_ws(const df_model_cfg* c, int b, int max_new, void* base, DraftWs* out) {
  const int d = c->d_model, Hq = c->n_q_heads, Hkv = c->n_kv_heads, F = c->d_ff, L = c->block_size;
  const size_t R = (size_t)b * L, Rc = (size_t)b * max_new;
  Carver cv(base);
  DraftWs w{};
  w.B.h = cv.take<float>(R * d);
  w.B.x = cv.take<df_bf16>((R + Rc) * d);
  w.B.q = cv.take<df_bf16>(R * Hq * 128);
  w.B.attn = cv.take<df_bf16>(R * Hq * 128);
  w.B.act = cv.take<df_bf16>(R * F);
  size_t pbytes = layer_partial_bytes(c, (int)R, (int)(R + Rc));
  if (Rc) pbytes = std::max(pbytes, gemm_partial_bytes((int)Rc, d, c->n_feat_layers * d));
  w.B.part = cv.take<float>(pbytes / 4 + 1);
  w.xl = cv.take<df_bf16>((size_t)b * (L - 1) * d);
  w.len_new = cv.take<int32_t>(b);
  w.stats = cv.take<float>((size_t)b * (L - 1) * 4 * ((c->vocab + 127) / 128) * 2);
  w.lse = cv.take<float>((size_t)b * (L - 1));
  w.B.rope = cv.take<float2>((R + Rc) * 64);
  const int ns = nsplit_for(b, L, Hq, Hkv, 1 << 20);
  const size_t pb = attn_partial_bytes(b, L, Hq, ns);
  w.B.o_part = cv.take<float>(pb / 4);
  w.B.ml_part = w.B.o_part ? w.B.o_part + (size_t)ns * R * Hq * 128 : nullptr;
  if (out) *out = w;
  return cv.off;
}

__global__ void len_new_kernel(const int32_t* len, const int32_t* add, int32_t* out, int b) {
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < b) out[s] = len[s] + add[s];
}
__global__ void copy_len_kernel(const int32_t* src, int32_t* dst, int b) {
  pdl_wait();
  pdl_trigger();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < b) dst[s] = src[s];
}
}  // namespace
}  // namespace df

using namespace df;

extern "C" {

const char* dflash_status_string(int s) {
  switch (s) {
    case DF_OK: return "ok";
    case DF_ERR_ARG: return "invalid argument";
    case DF_ERR_SHAPE: return "unsupported shape";
    case DF_ERR_ALIGN: return "pointer not 16-byte aligned";
    case DF_ERR_CAPACITY: return "cache capacity exceeded";
    case DF_ERR_CUDA: return "CUDA runtime error";
    case DF_ERR_NAN: return "NaN log-probability";
    case DF_ERR_TIMEOUT: return "device-side wait timed out";
    case DF_ERR_NOT_IMPLEMENTED: return "not implemented";
    case DF_ERR_WORKSPACE: return "workspace missing or too small";
    case DF_ERR_DEVICE: return "device is not compute capability 10.3";
    case DF_ERR_BOUNDS: return "device-side index check failed (checked build)";
    default: return "unknown status";
  }
}

int dflash_check_device(void) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DF_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return (major == 10 && minor == 3) ? DF_OK : DF_ERR_DEVICE;
}

int dflash_workspace_status(void* ws, df_stream stream) {
  if (!ws) return DF_ERR_WORKSPACE;
  int h[2] = {0, 0};
  if (cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess) return DF_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DF_ERR_CUDA;
  if (h[0] != 0) {
    int z[2] = {0, 0};
    if (cudaMemcpy(ws, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return DF_ERR_CUDA;
  }
  return h[0];
}

// ------------------------------------------------------------------------------- ddtree
size_t ddtree_build_workspace_size(int b, int D, int V, int B) {
  const int K = B < V ? (B > 0 ? B : 1) : V;
  Carver cv(nullptr);
  cv.take<int32_t>((size_t)b * D * K);
  cv.take<float>((size_t)b * D * K);
  cv.take<unsigned char>(topk_chunked_scratch_bytes(b * D));
  return cv.off;
}

int ddtree_build(const float* logprobs, int b, int D, int V, int B, const int32_t* root_tok, int32_t* tok,
                 int32_t* parent, int32_t* depth, float* score, uint32_t* anc, void* ws, size_t ws_bytes,
                 df_stream stream) {
  DF_NVTX("ddtree_build");
  if (b < 0 || D < 1 || D > 31 || V < 2 || B < 0 || B > 2048) return DF_ERR_ARG;
  // B must not exceed the number of prefixes sum_{k<=D} V^k
  {
    double total = 0, p = 1;
    for (int k = 1; k <= D && total < 1e9; ++k) { p *= V; total += p; }
    if ((double)B > total) return DF_ERR_ARG;
  }
  if (b == 0) return DF_OK;
  if (!logprobs || !tok || !parent || !depth || !score || !anc) return DF_ERR_ARG;
  if (!al16(logprobs) || !al16(tok) || !al16(parent) || !al16(depth) || !al16(score) || !al16(anc)) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < ddtree_build_workspace_size(b, D, V, B)) return DF_ERR_WORKSPACE;
  const int K = B < V ? (B > 0 ? B : 1) : V;
  if (ddtree_heap_smem(D, K, B) > 227 * 1024) return DF_ERR_SHAPE;
  Carver cv(ws);
  int32_t* tid = cv.take<int32_t>((size_t)b * D * K);
  float* tval = cv.take<float>((size_t)b * D * K);
  void* chunk = cv.take<unsigned char>(topk_chunked_scratch_bytes(b * D));
  return launch_ddtree(logprobs, b, D, V, B, root_tok, tok, parent, depth, score, anc, tid, tval, status_of(ws),
                       (cudaStream_t)stream, chunk);
}

// -------------------------------------------------------------------------- chain
size_t dflash_chain_build_workspace_size(int b, int D) {
  Carver cv(nullptr);
  cv.take<unsigned long long>((size_t)(b > 0 ? b : 1) * (D > 0 ? D : 1));
  return cv.off;
}

int dflash_chain_build(const float* logprobs, int b, int D, int V, const int32_t* root_tok, int32_t* tok,
                       int32_t* parent, int32_t* depth, float* score, uint32_t* anc, void* ws, size_t ws_bytes,
                       df_stream stream) {
  DF_NVTX("dflash_chain_build");
  if (b < 0 || D < 1 || D > 31 || V < 1) return DF_ERR_ARG;
  if (b == 0) return DF_OK;
  if (!logprobs || !tok || !parent || !depth || !score || !anc) return DF_ERR_ARG;
  if (!al16(logprobs) || !al16(tok) || !al16(parent) || !al16(depth) || !al16(score) || !al16(anc)) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < dflash_chain_build_workspace_size(b, D)) return DF_ERR_WORKSPACE;
  Carver cv(ws);
  unsigned long long* keys = cv.take<unsigned long long>((size_t)b * D);
  return launch_chain(logprobs, b, D, V, root_tok, tok, parent, depth, score, anc, keys, status_of(ws),
                      (cudaStream_t)stream);
}

// ------------------------------------------------------------------------- attention
size_t tree_verify_attention_workspace_size(int b, int n_tree, int Hq, int Hkv, int hd, int cap) {
  (void)hd;
  if (Hkv <= 0 || Hq % Hkv) return kAlign;
  const int ns = nsplit_for(b, n_tree, Hq, Hkv, cap);
  Carver cv(nullptr);
  cv.take<unsigned char>(attn_partial_bytes(b, n_tree, Hq, ns));
  return cv.off;
}

int tree_verify_attention(int b, int n_tree, int Hq, int Hkv, int hd, const df_bf16* q, const df_bf16* k_cache,
                          const df_bf16* v_cache, int cap, const int32_t* cache_len, const uint32_t* anc, float scale,
                          df_bf16* out, void* ws, size_t ws_bytes, df_stream stream) {
  DF_NVTX("tree_verify_attention");
  if (b < 0 || n_tree < 1 || Hkv <= 0 || Hq % Hkv || cap <= 0) return DF_ERR_ARG;
  const int G = Hq / Hkv;
  if (hd != 128 || G > 8 || (128 % G) || cap % 8) return DF_ERR_SHAPE;
  if (b == 0) return DF_OK;
  if (!q || !k_cache || !v_cache || !cache_len || !anc || !out) return DF_ERR_ARG;
  if (!al16(q) || !al16(k_cache) || !al16(v_cache) || !al16(anc) || !al16(out)) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < tree_verify_attention_workspace_size(b, n_tree, Hq, Hkv, hd, cap)) return DF_ERR_WORKSPACE;
  Carver cv(ws);
  const int ns = nsplit_for(b, n_tree, Hq, Hkv, cap);
  float* part = cv.take<float>(attn_partial_bytes(b, n_tree, Hq, ns) / 4);
  AttnArgs a{};
  a.b = b; a.T = n_tree; a.Hq = Hq; a.Hkv = Hkv; a.cap = cap;
  a.q = q; a.k_plane = k_cache; a.v_plane = v_cache;
  a.dense_len = cache_len; a.dense_add = 0; a.tail_len = n_tree; a.anc = anc;
  a.scale = scale; a.nsplit = ns; a.out = out;
  a.o_part = part; a.ml_part = part ? part + (size_t)ns * b * n_tree * Hq * 128 : nullptr;
  a.status = status_of(ws);
  return launch_attention(a, (cudaStream_t)stream);
}

// --------------------------------------------------------------------- accept/compact
size_t accept_and_compact_workspace_size(int b, int n_tree) {
  (void)n_tree;
  Carver cv(nullptr);
  cv.take<unsigned char>(accept_scratch_bytes(b));
  return cv.off;
}

int accept_and_compact(int b, int n_tree, const int32_t* choice, const int32_t* tok, const int32_t* parent,
                       df_bf16* k_cache, df_bf16* v_cache, int n_layers, int Hkv, int hd, int cap,
                       int32_t* cache_len, const df_bf16* tree_feat, int feat_dim, df_bf16* new_feat, int max_new,
                       int32_t* n_new, int32_t* acc_tok, int32_t* n_acc, int32_t* new_bonus, int32_t* src_slot,
                       void* ws, size_t ws_bytes, df_stream stream) {
  DF_NVTX("accept_and_compact");
  if (b < 0 || n_tree < 1 || max_new < 1 || n_layers < 0 || cap <= 0) return DF_ERR_ARG;
  if (n_layers > 0 && (hd != 128 || Hkv <= 0)) return DF_ERR_SHAPE;
  if (b == 0) return DF_OK;
  if (!choice || !tok || !parent || !cache_len || !n_new || !acc_tok || !n_acc || !new_bonus || !src_slot)
    return DF_ERR_ARG;
  if ((tree_feat == nullptr) != (new_feat == nullptr)) return DF_ERR_ARG;
  if (tree_feat && (feat_dim <= 0 || feat_dim % 8 || !al16(tree_feat) || !al16(new_feat))) return DF_ERR_ALIGN;
  if (n_layers > 0 && (!k_cache || !v_cache)) return DF_ERR_ARG;
  if (k_cache && (!al16(k_cache) || !al16(v_cache))) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < accept_and_compact_workspace_size(b, n_tree)) return DF_ERR_WORKSPACE;
  Carver cv(ws);
  void* scratch = cv.take<unsigned char>(accept_scratch_bytes(b));
  return launch_accept(b, n_tree, choice, tok, parent, k_cache, v_cache, n_layers, Hkv, cap, cache_len, tree_feat,
                       feat_dim, new_feat, max_new, n_new, acc_tok, n_acc, new_bonus, src_slot, scratch,
                       status_of(ws), (cudaStream_t)stream);
}

// ------------------------------------------------------------------ target tree forward
size_t dflash_target_tree_forward_workspace_size(const df_model_cfg* tcfg, int b, int n_tree) {
  if (!cfg_ok(tcfg) || b < 0 || n_tree < 1) return kAlign;
  return target_ws(tcfg, b, n_tree, nullptr, nullptr);
}

// Every layer carries the weights its feed-forward kind needs, 16-byte aligned (TMA).
int layers_ok(const df_model_cfg* c, const df_model_weights* w) {
  for (int i = 0; i < c->n_layers; ++i) {
    const df_layer_weights& L = w->layers[i];
    const void* need[] = {L.attn_norm, L.w_qkv, L.q_norm, L.k_norm, L.w_o, L.mlp_norm,
                          c->n_experts > 0 ? (const void*)L.w_router : (const void*)L.w_gate_up,
                          c->n_experts > 0 ? (const void*)L.w_experts_gate_up : (const void*)L.w_down,
                          c->n_experts > 0 ? (const void*)L.w_experts_down : (const void*)L.w_down};
    for (const void* q : need) {
      if (!q) return DF_ERR_ARG;
      if (!al16(q)) return DF_ERR_ALIGN;
    }
  }
  return DF_OK;
}

int dflash_target_expert_counts(const df_model_cfg* c, int b, int n_tree, const void* ws, size_t ws_bytes,
                                int32_t* counts, df_stream stream) {
  if (!cfg_ok(c) || c->n_experts == 0) return DF_ERR_SHAPE;
  if (b <= 0 || n_tree < 1 || !ws || !counts) return DF_ERR_ARG;
  if (ws_bytes < dflash_target_tree_forward_workspace_size(c, b, n_tree)) return DF_ERR_WORKSPACE;
  TargetWs W;
  target_ws(c, b, n_tree, const_cast<void*>(ws), &W);
  const size_t bytes = (size_t)c->n_layers * c->n_experts * sizeof(int32_t);
  return cudaMemcpyAsync(counts, W.B.moe.counts, bytes, cudaMemcpyDeviceToDevice, (cudaStream_t)stream) == cudaSuccess
             ? DF_OK
             : DF_ERR_CUDA;
}

// The target's forward over the flattened tree; the choice per node is the argmax
// (temperature 0) or a temperature draw keyed to (seed, sequence, position).
static int target_forward_run(const df_model_cfg* c, const df_model_weights* w, int b, int n_tree, const int32_t* tok,
                              const int32_t* depth, const uint32_t* anc, df_bf16* k_cache, df_bf16* v_cache, int cap,
                              const int32_t* cache_len, int32_t* choice, df_bf16* tree_feat, void* ws,
                              size_t ws_bytes, float temperature, uint64_t seed, cudaStream_t st) {
  if (!cfg_ok(c)) return DF_ERR_SHAPE;
  if (!w || !w->layers || !w->embed || !w->final_norm || b < 0 || n_tree < 1 || cap <= 0) return DF_ERR_ARG;
  DF_TRY(layers_ok(c, w));
  if (cap % 8) return DF_ERR_SHAPE;
  if (b == 0) return DF_OK;
  if (!tok || !k_cache || !v_cache || !cache_len || !choice) return DF_ERR_ARG;
  if ((depth == nullptr) != (anc == nullptr)) return DF_ERR_ARG;  // both NULL: a causal chain
  if (!al16(k_cache) || !al16(v_cache) || (anc && !al16(anc)) || (tree_feat && !al16(tree_feat))) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < dflash_target_tree_forward_workspace_size(c, b, n_tree)) return DF_ERR_WORKSPACE;
  TargetWs W;
  target_ws(c, b, n_tree, ws, &W);
  int* status = status_of(ws);
  const int d = c->d_model, R = b * n_tree, nf = c->n_feat_layers, Hkv = c->n_kv_heads;
  const size_t plane = (size_t)b * Hkv * cap * 128;
  DF_TRY(launch_embed(w->embed, d, c->vocab, tok, nullptr, 1, 0, W.B.h, R, status, st));
  auto feat_slot = [&](int done_layers) -> int {
    for (int f = 0; f < nf; ++f)
      if (c->feat_layers[f] == done_layers) return f;
    return -1;
  };
  {
    RmsNormArgs rn{};
    rn.in = W.B.h; rn.gain = w->layers[0].attn_norm; rn.out = W.B.x; rn.ld_out = d; rn.rows = R; rn.d = d;
    rn.eps = c->rms_eps; rn.group_out = 1; rn.group_in = 1;
    rn.zero = reinterpret_cast<float*>(W.amax); rn.zero_count = 2LL * R;  // LM-head argmax keys start at 0
    DF_TRY(launch_rmsnorm(rn, st));
  }
  for (int li = 0; li < c->n_layers; ++li) {
    LayerRun L{};
    L.cfg = c; L.w = &w->layers[li]; L.layer = li; L.b = b; L.T = n_tree; L.Rx = R; L.status = status;
    QkRopeArgs& qk = L.qk;
    qk.b = b; qk.TA = n_tree; qk.TB = 0; qk.base = cache_len; qk.nnew = nullptr; qk.depth = depth;
    qk.Hq = c->n_q_heads; qk.Hkv = Hkv; qk.eps = c->rms_eps; qk.theta = c->rope_theta;
    qk.k_plane = k_cache + (size_t)li * plane; qk.v_plane = v_cache + (size_t)li * plane; qk.cap = cap;
    qk.status = status;
    if (li == 0) DF_TRY(launch_rope_table(qk, W.B.rope, st));
    AttnArgs& at = L.at;
    at.b = b; at.T = n_tree; at.Hq = c->n_q_heads; at.Hkv = Hkv; at.cap = cap;
    at.dense_len = cache_len; at.dense_add = 0; at.tail_len = n_tree; at.anc = anc; at.causal = anc == nullptr;
    at.scale = 1.0f / sqrtf(128.f);
    at.nsplit = nsplit_for(b, n_tree, c->n_q_heads, Hkv, cap);
    at.status = status;
    ResNormArgs& o = L.out;  // after the down projection: next layer's input norm (or the final norm)
    o.gain = li + 1 < c->n_layers ? w->layers[li + 1].attn_norm : w->final_norm;
    o.out = W.B.x; o.ld_out = d; o.rows = R; o.group_out = 1; o.group_in = 1; o.in_off = 0;
    const int f = tree_feat ? feat_slot(li + 1) : -1;
    o.capture = f >= 0 ? tree_feat + (size_t)f * d : nullptr;
    o.ld_capture = nf * d;
    DF_TRY(run_layer(L, W.B, st));
  }
  GemmDesc g{};
  g.X = W.B.x; g.W = w->embed; g.M = R; g.N = c->vocab; g.K = d; g.ldx = d; g.ldw = d;
  g.mode = kGemmArgmax; g.amax = W.amax; g.status = status;
  if (temperature > 0.f) {
    DF_TRY(launch_draw_keys(R, seed, nullptr, nullptr, n_tree, cache_len, depth, W.draw_key, st));
    g.draw_key = W.draw_key;
    g.inv_temp = (float)(1.0 / (double)temperature);
  }
  DF_TRY(launch_gemm(g, st));
  return launch_argmax_finalize(W.amax, R, choice, st);
}

int dflash_target_tree_forward(const df_model_cfg* c, const df_model_weights* w, int b, int n_tree, const int32_t* tok,
                               const int32_t* depth, const uint32_t* anc, df_bf16* k_cache, df_bf16* v_cache, int cap,
                               const int32_t* cache_len, int32_t* choice, df_bf16* tree_feat, void* ws,
                               size_t ws_bytes, df_stream stream) {
  DF_NVTX("dflash_target_tree_forward");
  return target_forward_run(c, w, b, n_tree, tok, depth, anc, k_cache, v_cache, cap, cache_len, choice, tree_feat, ws,
                            ws_bytes, 0.f, 0, (cudaStream_t)stream);
}

int dflash_target_tree_forward_sampled(const df_model_cfg* c, const df_model_weights* w, int b, int n_tree,
                                       const int32_t* tok, const int32_t* depth, const uint32_t* anc,
                                       df_bf16* k_cache, df_bf16* v_cache, int cap, const int32_t* cache_len,
                                       float temperature, uint64_t seed, int32_t* choice, df_bf16* tree_feat,
                                       void* ws, size_t ws_bytes, df_stream stream) {
  DF_NVTX("dflash_target_tree_forward_sampled");
  if (!(temperature > 0.f) || !std::isfinite(temperature)) return DF_ERR_ARG;
  return target_forward_run(c, w, b, n_tree, tok, depth, anc, k_cache, v_cache, cap, cache_len, choice, tree_feat, ws,
                            ws_bytes, temperature, seed, (cudaStream_t)stream);
}

// ------------------------------------------------------------------------ draft block
size_t dflash_draft_block_workspace_size(const df_model_cfg* dcfg, int b, int max_new) {
  if (!cfg_ok(dcfg) || b < 0 || max_new < 0 || dcfg->block_size < 2 || dcfg->n_experts != 0) return kAlign;
  return draft_ws(dcfg, b, max_new, nullptr, nullptr);
}

int dflash_draft_block(const df_model_cfg* c, const df_model_weights* w, int b, const df_bf16* new_feat, int max_new,
                       const int32_t* n_new, df_bf16* ctx_k, df_bf16* ctx_v, int32_t* ctx_len, int cap,
                       const int32_t* bonus, float* logprobs, void* ws, size_t ws_bytes, df_stream stream) {
  DF_NVTX("dflash_draft_block");
  if (!cfg_ok(c) || c->block_size < 2 || c->n_feat_layers < 1 || c->n_experts != 0) return DF_ERR_SHAPE;
  if (!w || !w->layers || !w->embed || !w->final_norm || !w->fc || !w->fc_norm) return DF_ERR_ARG;
  if (b < 0 || max_new < 0 || cap <= 0) return DF_ERR_ARG;
  DF_TRY(layers_ok(c, w));
  if (cap % 8) return DF_ERR_SHAPE;
  if (b == 0) return DF_OK;
  if ((max_new > 0 && (!new_feat || !n_new)) || !ctx_k || !ctx_v || !ctx_len || !bonus || !logprobs) return DF_ERR_ARG;
  if ((new_feat && !al16(new_feat)) || !al16(ctx_k) || !al16(ctx_v) || !al16(logprobs)) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < dflash_draft_block_workspace_size(c, b, max_new)) return DF_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  DraftWs W;
  draft_ws(c, b, max_new, ws, &W);
  int* status = status_of(ws);
  const int d = c->d_model, L = c->block_size, Hkv = c->n_kv_heads, nf = c->n_feat_layers;
  const int R = b * L, Rc = b * max_new;
  const size_t plane = (size_t)b * Hkv * cap * 128;
  if (max_new > 0) {
    launch_k(len_new_kernel, dim3((b + 255) / 256), dim3(256), 0, st, ctx_len, n_new, W.len_new, b);
    // context fusion: c = RMSNorm(fc . f) into the context rows of x
    PartialView pv{};
    GemmDesc g{};
    g.X = new_feat; g.W = w->fc; g.M = Rc; g.N = d; g.K = nf * d; g.ldx = (long long)nf * d; g.ldw = (long long)nf * d;
    g.mode = kGemmPartial; g.part = W.B.part; g.view = &pv; g.status = status;
    DF_TRY(launch_gemm(g, st));
    ResNormArgs rn{};
    rn.pv = pv; rn.h = nullptr; rn.d = d; rn.gain = w->fc_norm; rn.eps = c->rms_eps; rn.out = W.B.x + (size_t)R * d;
    rn.ld_out = d; rn.rows = Rc; rn.group_out = 1; rn.group_in = 1; rn.in_off = 0;
    DF_TRY(launch_res_norm(rn, st));
  } else {
    launch_k(copy_len_kernel, dim3((b + 255) / 256), dim3(256), 0, st, ctx_len, W.len_new, b);
  }
  DF_TRY(launch_embed(w->embed, d, c->vocab, nullptr, bonus, L, c->mask_id, W.B.h, R, status, st));
  {
    RmsNormArgs rn{};
    rn.in = W.B.h; rn.gain = w->layers[0].attn_norm; rn.out = W.B.x; rn.ld_out = d; rn.rows = R; rn.d = d;
    rn.eps = c->rms_eps; rn.group_out = 1; rn.group_in = 1;
    DF_TRY(launch_rmsnorm(rn, st));
  }
  for (int li = 0; li < c->n_layers; ++li) {
    LayerRun Lr{};
    Lr.cfg = c; Lr.w = &w->layers[li]; Lr.b = b; Lr.T = L; Lr.Rx = R + Rc; Lr.status = status;
    QkRopeArgs& qk = Lr.qk;
    qk.b = b; qk.TA = L; qk.TB = max_new; qk.base = ctx_len; qk.nnew = max_new > 0 ? n_new : nullptr;
    qk.depth = nullptr;
    qk.Hq = c->n_q_heads; qk.Hkv = Hkv; qk.eps = c->rms_eps; qk.theta = c->rope_theta;
    qk.k_plane = ctx_k + (size_t)li * plane; qk.v_plane = ctx_v + (size_t)li * plane; qk.cap = cap;
    qk.status = status;
    if (li == 0) DF_TRY(launch_rope_table(qk, W.B.rope, st));
    AttnArgs& at = Lr.at;
    at.b = b; at.T = L; at.Hq = c->n_q_heads; at.Hkv = Hkv; at.cap = cap;
    at.dense_len = W.len_new; at.dense_add = L; at.tail_len = 0; at.anc = nullptr;
    at.scale = 1.0f / sqrtf(128.f);
    at.nsplit = nsplit_for(b, L, c->n_q_heads, Hkv, cap);
    at.status = status;
    ResNormArgs& o = Lr.out;
    if (li + 1 < c->n_layers) {
      o.gain = w->layers[li + 1].attn_norm; o.out = W.B.x; o.rows = R; o.group_out = 1; o.group_in = 1; o.in_off = 0;
    } else {  // final norm of rows 1..L-1 of every block, straight into the LM-head input
      o.gain = w->final_norm; o.out = W.xl; o.rows = b * (L - 1); o.group_out = L - 1; o.group_in = L; o.in_off = 1;
    }
    o.ld_out = d;
    DF_TRY(run_layer(Lr, W.B, st));
  }
  GemmDesc g{};
  g.X = W.xl; g.W = w->embed; g.M = b * (L - 1); g.N = c->vocab; g.K = d; g.ldx = d; g.ldw = d;
  g.mode = kGemmStore; g.out = logprobs; g.ldo = c->vocab; g.status = status; g.stats = W.stats;
  DF_TRY(launch_gemm(g, st));
  DF_TRY(launch_logsoftmax_from_stats(logprobs, b * (L - 1), c->vocab, W.stats, 4 * ((c->vocab + 127) / 128), W.lse,
                                      st));
  launch_k(copy_len_kernel, dim3((b + 255) / 256), dim3(256), 0, st, W.len_new, ctx_len, b);
  return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // extern "C"

extern "C" {
size_t dflash_linear_workspace_size(void) { return 256; }

size_t dflash_linear_argmax_workspace_size(int M) {
  Carver cv(nullptr);
  cv.take<unsigned long long>(M > 0 ? (size_t)M : 1);
  return cv.off;
}

int dflash_linear_argmax(const df_bf16* X, const df_bf16* W, int M, int N, int K, int32_t* out, void* ws,
                         size_t ws_bytes, df_stream stream) {
  DF_NVTX("dflash_linear_argmax");
  if (M < 0 || N <= 0 || K <= 0) return DF_ERR_ARG;
  if (K % 64) return DF_ERR_SHAPE;
  if (M == 0) return DF_OK;
  if (!X || !W || !out) return DF_ERR_ARG;
  if (!al16(X) || !al16(W)) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < dflash_linear_argmax_workspace_size(M)) return DF_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  Carver cv(ws);
  unsigned long long* keys = cv.take<unsigned long long>((size_t)M);
  if (cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * M, st) != cudaSuccess) return DF_ERR_CUDA;
  GemmDesc g{};
  g.X = X; g.W = W; g.M = M; g.N = N; g.K = K; g.ldx = K; g.ldw = K;
  g.mode = kGemmArgmax; g.amax = keys; g.status = status_of(ws);
  DF_TRY(launch_gemm(g, st));
  return launch_argmax_finalize(keys, M, out, st);
}

size_t dflash_linear_sample_workspace_size(int M) {
  Carver cv(nullptr);
  cv.take<unsigned long long>(M > 0 ? (size_t)M : 1);
  cv.take<uint32_t>(M > 0 ? (size_t)M : 1);
  return cv.off;
}

int dflash_linear_sample(const df_bf16* X, const df_bf16* W, int M, int N, int K, float temperature, uint64_t seed,
                         const int32_t* row_seq, const int32_t* row_pos, int32_t* out, void* ws, size_t ws_bytes,
                         df_stream stream) {
  DF_NVTX("dflash_linear_sample");
  if (M < 0 || N <= 0 || K <= 0 || !(temperature > 0.f) || !std::isfinite(temperature)) return DF_ERR_ARG;
  if (K % 64) return DF_ERR_SHAPE;
  if (M == 0) return DF_OK;
  if (!X || !W || !out || !row_seq || !row_pos) return DF_ERR_ARG;
  if (!al16(X) || !al16(W)) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < dflash_linear_sample_workspace_size(M)) return DF_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  Carver cv(ws);
  unsigned long long* keys = cv.take<unsigned long long>((size_t)M);
  uint32_t* dkeys = cv.take<uint32_t>((size_t)M);
  if (cudaMemsetAsync(keys, 0, sizeof(unsigned long long) * M, st) != cudaSuccess) return DF_ERR_CUDA;
  DF_TRY(launch_draw_keys(M, seed, row_seq, row_pos, 0, nullptr, nullptr, dkeys, st));
  GemmDesc g{};
  g.X = X; g.W = W; g.M = M; g.N = N; g.K = K; g.ldx = K; g.ldw = K;
  g.mode = kGemmArgmax; g.amax = keys; g.status = status_of(ws);
  g.draw_key = dkeys; g.inv_temp = (float)(1.0 / (double)temperature);
  DF_TRY(launch_gemm(g, st));
  return launch_argmax_finalize(keys, M, out, st);
}

size_t dflash_linear_logsoftmax_workspace_size(int M, int N) {
  Carver cv(nullptr);
  const size_t rows = M > 0 ? (size_t)M : 1, tiles = N > 0 ? (size_t)(N + 127) / 128 : 1;
  cv.take<float>(rows * 4 * tiles * 2);  // per (row, weight tile, warp) (max, sum exp) pairs
  cv.take<float>(rows);                  // log-sum-exp per row
  return cv.off;
}

int dflash_linear_logsoftmax(const df_bf16* X, const df_bf16* W, int M, int N, int K, float* out, void* ws,
                             size_t ws_bytes, df_stream stream) {
  DF_NVTX("dflash_linear_logsoftmax");
  if (M < 0 || N <= 0 || K <= 0) return DF_ERR_ARG;
  if (K % 64) return DF_ERR_SHAPE;
  if (M == 0) return DF_OK;
  if (!X || !W || !out) return DF_ERR_ARG;
  if (!al16(X) || !al16(W) || !al16(out)) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < dflash_linear_logsoftmax_workspace_size(M, N)) return DF_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  Carver cv(ws);
  const int n_stats = 4 * ((N + 127) / 128);
  float* stats = cv.take<float>((size_t)M * n_stats * 2);
  float* lse = cv.take<float>((size_t)M);
  // exactly the drafter's LM-head sequence: logits + softmax partials, then x - lse
  GemmDesc g{};
  g.X = X; g.W = W; g.M = M; g.N = N; g.K = K; g.ldx = K; g.ldw = K;
  g.mode = kGemmStore; g.out = out; g.ldo = N; g.status = status_of(ws); g.stats = stats;
  DF_TRY(launch_gemm(g, st));
  return launch_logsoftmax_from_stats(out, M, N, stats, n_stats, lse, st);
}

int dflash_workspace_configure(void* ws, unsigned long long wait_limit_ns, int hold, df_stream stream) {
  if (!ws) return DF_ERR_WORKSPACE;
  struct {
    unsigned long long limit;
    int hold;
  } h{wait_limit_ns, hold};
  unsigned char* base = static_cast<unsigned char*>(ws);
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(base + offsetof(WsHeader, wait_limit_ns), &h.limit, sizeof(h.limit), cudaMemcpyHostToDevice,
                      st) != cudaSuccess ||
      cudaMemcpyAsync(base + offsetof(WsHeader, hold), &h.hold, sizeof(h.hold), cudaMemcpyHostToDevice, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return DF_ERR_CUDA;
  return DF_OK;
}

int dflash_linear(const df_bf16* X, const df_bf16* W, int M, int N, int K, float* out, int accumulate, void* ws,
                  size_t ws_bytes, df_stream stream) {
  DF_NVTX("dflash_linear");
  if (M < 0 || N < 0 || K <= 0) return DF_ERR_ARG;
  if (K % 64) return DF_ERR_SHAPE;
  if (M == 0 || N == 0) return DF_OK;
  if (!X || !W || !out) return DF_ERR_ARG;
  if (!al16(X) || !al16(W) || !al16(out)) return DF_ERR_ALIGN;
  if (!ws || ws_bytes < dflash_linear_workspace_size()) return DF_ERR_WORKSPACE;
  GemmDesc g{};
  g.X = X; g.W = W; g.M = M; g.N = N; g.K = K; g.ldx = K; g.ldw = K;
  g.mode = accumulate ? kGemmAtomicAdd : kGemmStore;
  g.out = out; g.ldo = N; g.status = status_of(ws);
  return launch_gemm(g, (cudaStream_t)stream);
}
}
