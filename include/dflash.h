/*
 * dflash.h -- C ABI of the GB300 (sm_103a) speculative-step library.
 *
 * One speculative step of a block-diffusion drafter (DFlash) with draft trees (DDTree):
 *   dflash_draft_block         drafter forward: context fusion + KV injection, one
 *                              bidirectional pass over the block, per-position log-probs
 *   ddtree_build               top-K per position + best-first max-heap tree of B nodes
 *   dflash_target_tree_forward target forward over the flattened tree (its attention
 *                              layers call tree_verify_attention), greedy choice per node
 *                              (_sampled: the target's temperature draw per node)
 *   tree_verify_attention      ancestor-only attention of tree rows over the KV cache
 *   accept_and_compact         greedy longest-path walk and KV-cache compaction
 *
 * Sources (page title, section):
 *   [DFlash]  "DFlash: Block Diffusion for Flash Speculative Decoding 논문 정리"
 *             (honbul.tistory.com/178)
 *   [DDTree]  summary of "Accelerating Speculative Decoding with Block Diffusion Draft
 *             Trees" (bluediary8.tistory.com/1288)
 *
 * Conventions (every call):
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the library never
 *     allocates device memory and never frees what it is given.  Scratch space is the
 *     caller's `ws` buffer of at least the size the matching *_workspace_size() returns
 *     (256-byte aligned).  A workspace may be reused by later calls on the same stream.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and performs no host synchronisation, so a sequence of calls can be
 *     captured into a CUDA graph once the first call has run outside capture.
 *   - Tensors are dense and row-major in the order their shape is written.  bf16 tensors
 *     are passed as uint16_t bit patterns (df_bf16).  Every pointer must be 16-byte
 *     aligned (DF_ERR_ALIGN otherwise).
 *   - Host-detectable errors are returned at once and nothing is launched.  Errors the
 *     GPU finds (NaN log-probs, an exhausted wait, a full cache) are recorded in the
 *     workspace's status word; dflash_workspace_status() returns and clears it.  Every
 *     device-side wait is bounded (2 s unless dflash_workspace_configure sets otherwise).
 *   - Host-side state (kernel attributes, SM counts, tensor maps) is kept per device, so
 *     one process may use the library on several GPUs in turn.
 *   - The cache layout is [layer][batch][kv_head][slot][head_dim] for K and
 *     [layer][batch][kv_head][head_dim][slot] for V (V is stored transposed so that
 *     every tensor-core operand is K-major).  Slot s of a sequence holds the token at
 *     position s.
 *   - Head dimension is 128 and d_model, d_ff are multiples of 64.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t df_bf16;                 /* bf16 bit pattern                        */
typedef struct CUstream_st* df_stream;    /* same type as cudaStream_t               */

enum {
  DF_OK = 0,
  DF_ERR_ARG = -1,             /* bad scalar argument or null pointer                */
  DF_ERR_SHAPE = -2,           /* unsupported shape (head_dim != 128, ...)           */
  DF_ERR_ALIGN = -3,           /* a pointer is not 16-byte aligned                   */
  DF_ERR_CAPACITY = -4,        /* cache capacity too small for the requested writes  */
  DF_ERR_CUDA = -5,            /* a CUDA runtime call failed                         */
  DF_ERR_NAN = -6,             /* NaN log-probability seen on the device             */
  DF_ERR_TIMEOUT = -7,         /* a bounded device-side wait ran out                 */
  DF_ERR_NOT_IMPLEMENTED = -8,
  DF_ERR_WORKSPACE = -9,       /* workspace missing or smaller than required         */
  DF_ERR_DEVICE = -10,         /* current device is not compute capability 10.3      */
  DF_ERR_BOUNDS = -11          /* a device-side index check failed (DFLASH_CHECKED builds
                                  only; the access was skipped, detail = the check's id)   */
};

/* Shape of one decoder-only transformer (Qwen3 family layout). */
typedef struct {
  int32_t n_layers, d_model, n_q_heads, n_kv_heads, head_dim, d_ff, vocab;
  int32_t n_feat_layers;       /* target: number of layers whose outputs form the   */
  int32_t feat_layers[8];      /*   drafter's context row (1-indexed, ascending);    */
                               /* drafter: n_feat_layers = how many such rows it fuses */
  int32_t block_size;          /* drafter: L (row 0 bonus, rows 1..L-1 mask)         */
  int32_t mask_id;             /* drafter: mask token id                             */
  float rms_eps, rope_theta;
  int32_t n_experts;           /* target: 0 = dense feed-forward; else a mixture of   */
  int32_t top_k;               /*   n_experts SwiGLU experts of width d_expert, top_k  */
  int32_t d_expert;            /*   per token (n_experts a multiple of 32, <= 256;     */
                               /*   d_expert a multiple of 64; d_model of 256)         */
} df_model_cfg;

/* One decoder layer's weights (all bf16, row-major [out][in]). */
typedef struct {
  const df_bf16* attn_norm;    /* [d]                                                */
  const df_bf16* w_qkv;        /* [(Hq + 2 Hkv) * hd][d]: q heads, then k, then v    */
  const df_bf16* q_norm;       /* [hd]                                               */
  const df_bf16* k_norm;       /* [hd]                                               */
  const df_bf16* w_o;          /* [d][Hq * hd]                                       */
  const df_bf16* mlp_norm;     /* [d]                                                */
  const df_bf16* w_gate_up;    /* [2 F][d]: gate rows 0..F-1, up rows F..2F-1        */
  const df_bf16* w_down;       /* [d][F]                                             */
  /* mixture-of-experts layers (n_experts > 0; w_gate_up and w_down unused):          */
  const df_bf16* w_router;     /* [E][d]                                             */
  const df_bf16* w_experts_gate_up;  /* [E][2 Fe][d]: per expert gate rows, then up  */
  const df_bf16* w_experts_down;     /* [E][d][Fe]                                   */
} df_layer_weights;

typedef struct {
  const df_layer_weights* layers;  /* HOST array of n_layers entries                */
  const df_bf16* final_norm;       /* [d]                                           */
  const df_bf16* embed;            /* [V][d] token embedding = tied LM head (shared) */
  const df_bf16* fc;               /* drafter only: [d][n_feat * d]                 */
  const df_bf16* fc_norm;          /* drafter only: [d]                             */
} df_model_weights;

/* ------------------------------------------------------------------------------------
 * dflash_draft_block -- one drafter forward (DFlash).
 *
 * [DFlash] "DFlash의 핵심 아이디어" (1, 2): hidden states from several target layers are
 * fused into a compressed context signal that every drafter layer attends to as memory;
 * (3): the drafter fills all masked positions of a short block in one forward pass.
 * [DFlash] "학습 방식도 추론 시나리오에 맞춰 바꿨다": positions of one block see each
 * other; embedding and LM head are the target's.  [DDTree] "핵심 아이디어": the input
 * is the masked block after the bonus token, the output one distribution per position.
 *
 * Steps: for each sequence s, the n_new[s] rows of new_feat (concatenated residual
 * outputs of the target's feature layers at positions ctx_len[s] + j) become
 * c = RMSNorm(fc . f); every drafter layer projects c with its own W_k / W_v (k-norm,
 * rotation at the position) and appends it to its context cache; ctx_len[s] += n_new[s].
 * Then the block [bonus[s], mask x (L-1)] at positions ctx_len[s] .. ctx_len[s]+L-1
 * runs through the layers, each row attending to every context slot and every block
 * row (no mask).  Rows 1..L-1 give log-probs (fp32 log-softmax of the logits).
 *
 *   dcfg, dw      drafter shape / weights (dw->embed is the shared embedding); a dense
 *                 feed-forward (n_experts = 0)
 *   new_feat      [b][max_new][n_feat * d] bf16; rows >= n_new[s] are ignored
 *   n_new         [b] int32, 0 <= n_new <= max_new
 *   ctx_k         [n_layers][b][Hkv][cap][hd] bf16, in/out
 *   ctx_v         [n_layers][b][Hkv][hd][cap] bf16, in/out
 *   ctx_len       [b] int32, in/out; needs ctx_len + n_new + L <= cap (slots past the
 *                 context are scratch for the block's own keys)
 *   bonus         [b] int32 block row-0 token
 *   logprobs      [b][L-1][V] fp32 out
 * ------------------------------------------------------------------------------------ */
size_t dflash_draft_block_workspace_size(const df_model_cfg* dcfg, int b, int max_new);
int dflash_draft_block(const df_model_cfg* dcfg, const df_model_weights* dw, int b,
                       const df_bf16* new_feat, int max_new, const int32_t* n_new,
                       df_bf16* ctx_k, df_bf16* ctx_v, int32_t* ctx_len, int cap,
                       const int32_t* bonus, float* logprobs,
                       void* ws, size_t ws_bytes, df_stream stream);

/* ------------------------------------------------------------------------------------
 * ddtree_build -- optimal draft tree under a node budget (DDTree).
 *
 * [DDTree] "방법론 자세히 보기": expected acceptance length equals the sum of the tree
 * nodes' prefix probabilities, so the best tree of B nodes is the B most probable
 * prefixes of the factorized per-position distribution, found by a best-first max-heap
 * in O(B log B).
 *
 * Order: prefix score (fp32 sum of its log-probs, root first) descending, then depth
 * ascending, then the parent's place in this order, then the token's rank at its depth
 * (per-position lists sorted by log-prob descending, token id ascending).
 *
 *   logprobs  [b][D][V] fp32 (position d+1 at row d); NaN -> DF_ERR_NAN (device)
 *   root_tok  [b] int32 or NULL: written to tok[s][0] (else -1)
 *   tok, parent, depth  [b][B+1] int32; index 0 = root (parent -1, depth 0); nodes
 *             1..B in pop order, so parents precede children
 *   score     [b][B+1] fp32 log prefix probability (root 0)
 *   anc       [b][B+1][ceil((B+1)/32)] uint32; bit j of row i set iff node j is node i
 *             or one of its ancestors (bit 0 = root always set)
 * Limits: 1 <= D <= 31, 0 <= B <= 2048, B <= sum_{k<=D} V^k, V >= 2.
 * ------------------------------------------------------------------------------------ */
size_t ddtree_build_workspace_size(int b, int D, int V, int B);
int ddtree_build(const float* logprobs, int b, int D, int V, int B, const int32_t* root_tok,
                 int32_t* tok, int32_t* parent, int32_t* depth, float* score, uint32_t* anc,
                 void* ws, size_t ws_bytes, df_stream stream);

/* ------------------------------------------------------------------------------------
 * ddtree_build_static -- ddtree_build for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this call: it exists for integration only.  Some
 * callers cannot call cudaMalloc or hand over a workspace, e.g. a host framework that
 * owns every device allocation and exposes none to plug-ins, a serving loop that may not
 * allocate while a CUDA graph is being captured, or a runtime whose memory pool is fixed
 * at start-up.  This variant takes the same inputs and outputs as ddtree_build (same
 * layouts, limits and results) but keeps its scratch -- the per-position top-K lists and
 * a status word -- in a fixed array inside the library's device image (about 2 MiB,
 * present on every GPU that loads the library until the process exits).  It calls no
 * cudaMalloc, cudaFree or allocating library routine.
 *   - Size limit: b * D * min(B, V) <= 262144; larger calls return DF_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current); make that first call before any stream capture.
 *   - Every call shares the one array, so calls that may overlap on the GPU (other
 *     streams, other host threads) race: serialise them.  Each call clears the status
 *     word first; the top-K lists are fully rewritten before they are read.
 *   - Device-side errors cannot be handed back (there is no workspace to read): when a
 *     log-probability is NaN the outputs of that call are left unwritten.
 *   - The looked-up address is kept for the life of the process: the library must not be
 *     used on a device after its primary context has been reset (cudaDeviceReset).
 * ------------------------------------------------------------------------------------ */
int ddtree_build_static(const float* logprobs, int b, int D, int V, int B, const int32_t* root_tok,
                        int32_t* tok, int32_t* parent, int32_t* depth, float* score, uint32_t* anc,
                        df_stream stream);

/* ------------------------------------------------------------------------------------
 * dflash_chain_build -- the vanilla DFlash draft: one chain of the per-position argmax.
 *
 * [DDTree] "실험 결과": DDTree is compared with plain DFlash at the same block size, which
 * verifies the drafter's block as it is: the most likely token at every position, one
 * causal chain.  [DFlash] "DFlash의 핵심 아이디어" (3): the block is drafted in one pass
 * and checked by the target in one pass.
 *
 * Same inputs and output layout as ddtree_build with B = D: node i (1..D) is position i's
 * most likely token (lowest id among exactly equal log-probs), parent i - 1, depth i,
 * score = fp32 sum of the log-probs of positions 1..i added root first; ancestor row i has
 * bits 0..i set (a causal mask).  NaN log-probs -> DF_ERR_NAN (device), outputs unwritten.
 *   logprobs  [b][D][V] fp32;  root_tok [b] or NULL (tok[s][0] = -1)
 *   tok, parent, depth [b][D+1] int32;  score [b][D+1] fp32;  anc [b][D+1][ceil((D+1)/32)]
 * Limits: 1 <= D <= 31, V >= 1.
 * ------------------------------------------------------------------------------------ */
size_t dflash_chain_build_workspace_size(int b, int D);
int dflash_chain_build(const float* logprobs, int b, int D, int V, const int32_t* root_tok,
                       int32_t* tok, int32_t* parent, int32_t* depth, float* score, uint32_t* anc,
                       void* ws, size_t ws_bytes, df_stream stream);

/* ------------------------------------------------------------------------------------
 * tree_verify_attention -- ancestor-only attention of flattened tree rows (DDTree).
 *
 * [DDTree] "방법론 자세히 보기": the flattened tree goes through the target in one pass;
 * an ancestor-only mask lets each token see only the tokens on its own root path.
 *
 * Row (s, i, h) attends cache slots [0, N) (N = cache_len[s]) and tree slots N + j for
 * every j with bit j of anc[s][i] set, softmax(scale q.k) weighted V, fp32 inside.
 * The tree's own K/V must already be in slots N .. N + n_tree - 1.
 *
 *   q         [b][n_tree][Hq][hd] bf16 (rotated)
 *   k_cache   [b][Hkv][cap][hd] bf16 (one layer),  v_cache [b][Hkv][hd][cap] bf16
 *   cache_len [b] int32, N + n_tree <= cap
 *   anc       [b][n_tree][ceil(n_tree/32)] uint32
 *   out       [b][n_tree][Hq][hd] bf16
 * Limits: hd = 128; Hq a multiple of Hkv with Hq/Hkv in {1,2,4,8}; n_tree >= 1;
 *         cap a multiple of 8.  Cache slots that no row may see must still hold finite
 *         values (zero-initialise caches): masked keys get weight 0, and 0 * NaN = NaN.
 * ------------------------------------------------------------------------------------ */
size_t tree_verify_attention_workspace_size(int b, int n_tree, int Hq, int Hkv, int hd, int cap);
int tree_verify_attention(int b, int n_tree, int Hq, int Hkv, int hd,
                          const df_bf16* q, const df_bf16* k_cache, const df_bf16* v_cache,
                          int cap, const int32_t* cache_len, const uint32_t* anc, float scale,
                          df_bf16* out, void* ws, size_t ws_bytes, df_stream stream);

/* ------------------------------------------------------------------------------------
 * dflash_target_tree_forward -- the target's single forward over a flattened tree.
 *
 * [DDTree] "핵심 아이디어" / "방법론 자세히 보기": the tree is verified in one target
 * forward pass under the ancestor-only mask.
 *
 * The target's feed-forward may be a mixture of experts (tcfg->n_experts > 0: [DFlash]
 * and [DDTree] "실험 결과" evaluate Qwen3-Coder-30B-A3B; read as the Qwen3-MoE layer: a
 * router softmax over the experts, the top_k experts per token, weights renormalised to
 * sum 1, SwiGLU experts).  Routing stays on the device (no host synchronisation).
 *
 * Node i of sequence s (token tok[s][i]) is rotated at position cache_len[s] + depth[s][i];
 * its K/V go to slot cache_len[s] + i of every layer; attention is tree_verify_attention.
 * Outputs the greedy choice (argmax, lowest id on ties) after every node and the residual
 * outputs of the feature layers.  With n_tree = 1 this is one plain decode step; with a
 * chain it is a prompt pass ([DFlash] "DFlash의 핵심 아이디어" (1, 2): the prompt's
 * feature rows become the drafter's first context).
 *
 *   tok, depth [b][n_tree] int32;  anc [b][n_tree][ceil(n_tree/32)] uint32
 *             depth and anc both NULL: the rows are a chain (a causal prompt pass): row i
 *             is rotated at cache_len + i and sees tree slots 0 .. i
 *   k_cache   [n_layers][b][Hkv][cap][hd],  v_cache [n_layers][b][Hkv][hd][cap]  bf16
 *   cache_len [b] int32 (not modified); needs cache_len + n_tree <= cap
 *   choice    [b][n_tree] int32 out
 *   tree_feat [b][n_tree][n_feat * d] bf16 out (may be NULL)
 * ------------------------------------------------------------------------------------ */
size_t dflash_target_tree_forward_workspace_size(const df_model_cfg* tcfg, int b, int n_tree);
int dflash_target_tree_forward(const df_model_cfg* tcfg, const df_model_weights* tw, int b,
                               int n_tree, const int32_t* tok, const int32_t* depth,
                               const uint32_t* anc, df_bf16* k_cache, df_bf16* v_cache, int cap,
                               const int32_t* cache_len, int32_t* choice, df_bf16* tree_feat,
                               void* ws, size_t ws_bytes, df_stream stream);

/* dflash_target_tree_forward_sampled -- as dflash_target_tree_forward, with the choice
 * after every node drawn from the target's distribution at temperature T instead of its
 * argmax.
 *
 * [DFlash] and [DDTree] "실험 결과" evaluate temperature 1.0 but state no acceptance rule.
 * Reading: the verifier follows the target's own outputs ([DDTree] "방법론 자세히 보기"),
 * so at temperature T the output after node i is a token the target draws, and
 * accept_and_compact walks the tree along the drawn tokens unchanged; every emitted token
 * is then the target's own draw (lossless).  The draw is Gumbel-max, argmax over v of
 * fp32(logit_v * (1/T)) + g_v, g_v = -log(-log u_v), u_v = (23 bits of a counter-based hash +
 * 1/2) / 2^23 keyed to (seed, sequence s, position N_s + depth_i + 1 of the drawn token, v)
 * (MurmurHash3's 32-bit finalizer in a fixed chain, also exposed through
 * dflash_linear_sample).  Keyed to the absolute position, speculative decoding emits the
 * tokens plain sampling emits under the same seed.
 *   temperature > 0 and finite (DF_ERR_ARG otherwise); seed: any 64-bit value.  Every other
 *   argument and the workspace are those of dflash_target_tree_forward.
 * ------------------------------------------------------------------------------------ */
int dflash_target_tree_forward_sampled(const df_model_cfg* tcfg, const df_model_weights* tw,
                                       int b, int n_tree, const int32_t* tok,
                                       const int32_t* depth, const uint32_t* anc,
                                       df_bf16* k_cache, df_bf16* v_cache, int cap,
                                       const int32_t* cache_len, float temperature, uint64_t seed,
                                       int32_t* choice, df_bf16* tree_feat, void* ws,
                                       size_t ws_bytes, df_stream stream);

/* dflash_target_expert_counts -- routing statistics of the last mixture-of-experts
 * dflash_target_tree_forward run on this workspace (same tcfg, b, n_tree): per layer, the
 * rows routed to each expert (each row goes to top_k distinct experts, so a layer's counts
 * sum to b * n_tree * top_k).  Stream-ordered device-to-device copy.
 *   counts [n_layers][n_experts] int32 out (device)
 * Errors: DF_ERR_SHAPE for a dense target, DF_ERR_WORKSPACE for a smaller workspace.  */
int dflash_target_expert_counts(const df_model_cfg* tcfg, int b, int n_tree, const void* ws,
                                size_t ws_bytes, int32_t* counts, df_stream stream);

/* ------------------------------------------------------------------------------------
 * accept_and_compact -- greedy acceptance and KV-cache compaction (DDTree).
 *
 * [DDTree] "방법론 자세히 보기": the verifier follows the target's outputs down the tree,
 * accepts the longest matching path and compacts the KV cache, dropping rejected
 * branches.
 *
 * Walk: cur = root; while some child c of cur has tok[c] == choice[cur], move to c.
 * The a accepted nodes (depth 1..a) are moved to slots N+1..N+a of every layer (K and V);
 * cache_len[s] becomes N + 1 + a.  Their feature rows, after the root's, go to new_feat.
 *
 *   choice, tok, parent  [b][n_tree] int32
 *   k_cache, v_cache     all layers, layouts as in the conventions; in/out
 *   cache_len            [b] int32 in/out
 *   tree_feat            [b][n_tree][feat_dim] bf16 (may be NULL with new_feat NULL)
 *   new_feat             [b][max_new][feat_dim] bf16 out: rows 0..a (root, path);
 *                        max_new >= deepest path + 1
 *   n_new                [b] int32 out = a + 1
 *   acc_tok              [b][max_new] int32 out: accepted tokens then the new bonus
 *   n_acc                [b] int32 out = a
 *   new_bonus            [b] int32 out: choice at the last accepted node
 *   src_slot             [b][max_new] int32 out: source slot of slot N+1+j (j < a), -1 after
 * ------------------------------------------------------------------------------------ */
size_t accept_and_compact_workspace_size(int b, int n_tree);
int accept_and_compact(int b, int n_tree, const int32_t* choice, const int32_t* tok,
                       const int32_t* parent, df_bf16* k_cache, df_bf16* v_cache,
                       int n_layers, int Hkv, int hd, int cap, int32_t* cache_len,
                       const df_bf16* tree_feat, int feat_dim, df_bf16* new_feat, int max_new,
                       int32_t* n_new, int32_t* acc_tok, int32_t* n_acc, int32_t* new_bonus,
                       int32_t* src_slot, void* ws, size_t ws_bytes, df_stream stream);

/* ------------------------------------------------------------------------------------
 * dflash_linear -- building block: out (+)= X . W^T on the tensor cores.
 *
 * Every projection of the step (q/k/v, o, gate/up, down, context fusion, LM head) is
 * this product of a few token rows with a large weight matrix; exposed for custom
 * composites and tests.
 *   X [M][K] bf16, W [N][K] bf16, K a multiple of 64, out [M][N] fp32.
 *   accumulate = 1: out += X W^T (out must be initialised); 0: out = X W^T.
 * ------------------------------------------------------------------------------------ */
size_t dflash_linear_workspace_size(void);
int dflash_linear(const df_bf16* X, const df_bf16* W, int M, int N, int K, float* out, int accumulate,
                  void* ws, size_t ws_bytes, df_stream stream);

/* dflash_linear_argmax -- out[t] = argmax_n (X W^T)[t][n], lowest n among equal maxima: the
 * target's LM head of dflash_target_tree_forward (the logits are never written).
 *   X [M][K] bf16, W [N][K] bf16, K a multiple of 64, out [M] int32.
 *   Workspace: dflash_linear_argmax_workspace_size(M) bytes (per-row keys + status). */
size_t dflash_linear_argmax_workspace_size(int M);
int dflash_linear_argmax(const df_bf16* X, const df_bf16* W, int M, int N, int K, int32_t* out,
                         void* ws, size_t ws_bytes, df_stream stream);

/* dflash_linear_sample -- out[t] = the token row t draws at temperature T from
 * softmax((X W^T)[t] / T): the LM head of dflash_target_tree_forward_sampled, with each row's
 * draw keyed to (seed, row_seq[t], row_pos[t]) instead of to the tree (see that call).
 *   X [M][K] bf16, W [N][K] bf16, K a multiple of 64; row_seq, row_pos [M] int32 (device);
 *   temperature > 0 and finite (DF_ERR_ARG otherwise); out [M] int32.
 *   Workspace: dflash_linear_sample_workspace_size(M) bytes. */
size_t dflash_linear_sample_workspace_size(int M);
int dflash_linear_sample(const df_bf16* X, const df_bf16* W, int M, int N, int K, float temperature,
                         uint64_t seed, const int32_t* row_seq, const int32_t* row_pos, int32_t* out,
                         void* ws, size_t ws_bytes, df_stream stream);

/* dflash_linear_logsoftmax -- out[t][n] = log-softmax over n of (X W^T)[t]: the drafter's LM
 * head of dflash_draft_block, exactly its sequence of kernels (logits stored with per-tile
 * softmax partials, then the log-sum-exp of each row subtracted).
 * [DDTree] "핵심 아이디어": the drafter gives one distribution per block position, and the
 * tree builder reads those distributions as log-probabilities.
 *   X [M][K] bf16, W [N][K] bf16, K a multiple of 64, out [M][N] fp32.
 *   Workspace: dflash_linear_logsoftmax_workspace_size(M, N) bytes. */
size_t dflash_linear_logsoftmax_workspace_size(int M, int N);
int dflash_linear_logsoftmax(const df_bf16* X, const df_bf16* W, int M, int N, int K, float* out,
                             void* ws, size_t ws_bytes, df_stream stream);

/* ------------------------------------------------------------------------------------
 * dflash_plant_logprobs -- acceptance planting for synthetic models (benchmark and test
 * harness; the pages have no counterpart).
 *
 * Random-init drafters almost never agree with random-init targets.  For sequence s and
 * draft position d (1..D), with probability `rate`, row d of the log-probs becomes the
 * log-softmax of its logits with `bias` added at the reference token r = ref[s][pos[s]][d-1]:
 * lp'_i = lp_i - c (i != r), lp'_r = lp_r + bias - c, c = log(1 + exp(lp_r)(e^bias - 1)).
 * The draw is a counter-based hash (splitmix64) of (seed, s, pos[s], d): no host input per
 * step, so the call can sit in a captured graph.  With miss_bias > 0 a row not drawn is a
 * near miss: `bias` goes to a decoy token d != r (picked by a second splitmix64 of the draw:
 * d = (r + 1 + splitmix64(h) mod (V - 1)) mod V) and `miss_bias` to r, both renormalised as
 * above: the decoy and r lead the row, r usually second (a drafter whose miss still holds
 * the target's token); miss_bias = 0 leaves such rows as they are.  Rows with no reference (pos[s] outside [0, n_pos) or a negative
 * entry) are left as they are.
 *   logprobs [b][D][V] fp32 in/out
 *   ref      [b][n_pos][D] int32: the tokens expected at depths 1..D of a block whose row 0
 *            (the bonus token) is at position p
 *   pos      [b] int32: position of the block's row 0 (the target's cache length)
 * ------------------------------------------------------------------------------------ */
int dflash_plant_logprobs(float* logprobs, int b, int D, int V, const int32_t* ref, int n_pos,
                          const int32_t* pos, float rate, float bias, float miss_bias,
                          unsigned long long seed, df_stream stream);

/* ------------------------------------------------------------------------------------
 * Status and device queries.
 * ------------------------------------------------------------------------------------ */
/* Launch tracing, off by default.  While on, every kernel launch of the library (outside
 * stream capture) is bracketed by a pair of CUDA events on its stream.
 * dflash_trace_read synchronises on those events, writes up to max_entries per-tag totals
 * (names: max_entries x 64 chars, NUL-terminated; total_ms; count), clears the record and
 * returns the number of tags written.  A tag is the kernel class, optionally followed by a
 * space and the launch's shape (GEMMs: "M x N x K"). */
int dflash_trace_enable(int on);
int dflash_trace_read(int max_entries, char* names, double* total_ms, int* count);
/* Reads and clears the device status word of a workspace (synchronises `stream`).
 * Returns DF_OK or the first device-side error recorded since the last read. */
int dflash_workspace_status(void* ws, df_stream stream);
/* Failure-path settings of a workspace (synchronises `stream`), kept until changed:
 *   wait_limit_ns  limit of every bounded device-side wait of calls using this workspace
 *                  (0 = the default, 2 s); a wait that runs out records DF_ERR_TIMEOUT and
 *                  its kernel returns without touching TMEM or shared memory still in use
 *   hold           test hook: nonzero makes every projection GEMM of such a call wait for
 *                  the word to read 0 before it issues any tensor-core work.  Nothing clears
 *                  it, so the wait runs out and the call reports DF_ERR_TIMEOUT; set 0 to go on.
 * Zero-initialised workspaces start with both at 0. */
int dflash_workspace_configure(void* ws, unsigned long long wait_limit_ns, int hold, df_stream stream);
/* Static text for a status code. */
const char* dflash_status_string(int status);
/* DF_OK if the current CUDA device is compute capability 10.3 (GB300). */
int dflash_check_device(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
