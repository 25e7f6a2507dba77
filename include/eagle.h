/*
 * eagle.h -- C ABI of libeagle: one EAGLE / EAGLE-2 draft-and-verify round on
 * a single GB300 GPU (sm_103a).
 *
 * Sources (the three pages this library restates; cited by title + section):
 *   [A] "EAGLE 推测解码为什么比 Medusa 快？（含 EAGLE-2 动态草稿树）" (zzszmyf.github.io)
 *   [B] "eagle-feature-level-speculative-decoding" (charlestar.github.io)
 *   [C] "EAGLE 完全拆解：特征级草稿模型如何把投机解码推到 3 倍以上" (pinghaoyang.com.cn)
 *
 * The round is a transaction ([B] "KV Cache 必须按事务提交"):
 *   draft (eagle_draft_step, per tree layer) -> tree (eagle_tree_expand_rerank)
 *   -> verify attention (eagle_tree_verify_attn) -> accept (eagle_accept)
 *   -> commit the accepted path (eagle_commit).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer in a struct or argument is a DEVICE pointer unless it is
 *    marked "host".  Buffers are owned by the caller; no call allocates,
 *    frees or retains device memory.  Scratch space comes from the caller's
 *    workspace, sized by eagle_create.
 *  - bf16 values are passed as uint16_t bit patterns.  Matrices are row-major
 *    [out][ld] (PyTorch Linear layout) with row pitch ld >= in, ld % 8 == 0.
 *  - Device pointers must be 16-byte aligned, else EAGLE_ERR_ALIGN.
 *  - Every call is asynchronous on the given stream and does not synchronise
 *    the host (except eagle_read_device_status).  Shape, capacity and tree
 *    checks run on the host before any launch and return a status; errors
 *    only the device can see (non-finite logits, an exhausted distribution,
 *    a wait that timed out) set the status word in the workspace, read with
 *    eagle_read_device_status.  Nothing aborts, traps or asserts.
 *  - One context per stream at a time: calls that share a workspace must not
 *    overlap on the device.
 *
 * Round state layout (our layout; the pages fix the rules, not the storage)
 * -------------------------------------------------------------------------
 *  - B requests.  Request b's round starts from f_last[b] (the verified
 *    feature of position L_b - 1) and t_next[b], the already-committed token
 *    at position L_b ([A] §6.1 / §7.1: the first draft token comes from
 *    q == p and is accepted with probability 1).  t_next is the tree root.
 *  - Expanded nodes (nodes the draft head runs on) occupy slots
 *    e = 0 .. E-1 per request; e = 0 is the root.  Each has K drawn
 *    children (e, r), r = draw rank.  Layer l of the plan runs the draft head
 *    on slots [layer_e0[l], layer_e0[l] + layer_rows[l]) of every request.
 *  - The verified tree has S = 1 + m slots per request: slot 0 = root, slots
 *    1..m sorted by (depth, selection rank).  anc[s] bit j (word j / 64) is set iff slot j
 *    is an ancestor of s or j == s ([B] "Tree Attention": M_uv = 0 iff v is
 *    an ancestor of u or v = u).  A node at depth delta sits at position
 *    L_b + delta.
 */
#ifndef EAGLE_H
#define EAGLE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EAGLE_OK = 0,
  EAGLE_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, bad plan */
  EAGLE_ERR_SHAPE = 2,         /* dims unsupported or inconsistent */
  EAGLE_ERR_ALIGN = 3,         /* a pointer or pitch breaks the 16-byte rule */
  EAGLE_ERR_CAPACITY = 4,      /* beyond the limits given to eagle_create */
  EAGLE_ERR_INVALID_TREE = 5,  /* template malformed / selection not connected */
  EAGLE_ERR_NUMERIC = 6,       /* non-finite logits or a zero-mass distribution */
  EAGLE_ERR_TIMEOUT = 7,       /* a device-side wait gave up (kernel returned early) */
  EAGLE_ERR_UNSUPPORTED = 8,   /* no device, wrong architecture */
  EAGLE_ERR_CUDA = 9           /* a CUDA runtime call failed */
} eagle_status;

#define EAGLE_MAX_NODES 256    /* tree slots and expanded slots per request */
/* Ancestor masks over n slots take EAGLE_MASK_WORDS(n) 64-bit words per
 * slot: bit j of a mask is bit j % 64 of word j / 64.  Up to 64 slots that is
 * one word, so trees of up to 63 retained nodes keep one u64 per slot. */
#define EAGLE_MASK_WORDS(n) (((n) + 63) / 64)
#define EAGLE_MAX_CHILDREN 16  /* drawn children per expanded node */
#define EAGLE_MAX_LAYERS 128   /* target layers one commit can append */
#define EAGLE_MAX_VOCAB 32768  /* keeps every exact sampling product below 2^128 */

typedef struct eagle_ctx eagle_ctx;

/* Model shape of the draft head's decoder layer ([A] §4.1, [B] "草稿头到底包含什么"):
 * FC 2d -> d with bias, then a LLaMA pre-norm layer (RMSNorm, RoPE
 * rotate-half, GQA attention, SwiGLU MLP) and the shared LM head. */
typedef struct {
  int d;            /* hidden size; multiple of 64 */
  int n_q_heads;    /* Hq; Hq * head_dim multiple of 64 */
  int n_kv_heads;   /* Hkv; Hq % Hkv == 0; Hkv * head_dim multiple of 64 */
  int head_dim;     /* dh in {16, 32, 64, 128} */
  int d_ff;         /* F (any value >= 8) */
  int vocab;        /* V <= EAGLE_MAX_VOCAB */
  float rms_eps;    /* RMSNorm epsilon (1e-5) */
  float rope_theta; /* RoPE base (10000) */
} eagle_dims;

/* Capacities fixed at creation; calls beyond them return EAGLE_ERR_CAPACITY. */
typedef struct {
  int max_batch;      /* requests per call, <= 65535 */
  int max_rows;       /* draft rows per step (batch x rows per request), <= 256 */
  int max_expanded;   /* expanded slots per request, <= EAGLE_MAX_NODES */
  int max_children;   /* children per expanded node, <= EAGLE_MAX_CHILDREN */
  int max_tree;       /* tree slots per request incl. root, <= EAGLE_MAX_NODES */
  int max_prefix;     /* longest prefix KV (draft or target) in rows */
} eagle_limits;

/* Tree plan (host struct, built by eagle_plan_eagle2 / eagle_plan_static).
 * kind 0: EAGLE-2 dynamic tree ([A] §10.3): layer 0 = root; layer l >= 1
 * expands the top_k nodes of layer l by value (value = product of draft
 * confidences along the path); FINAL keeps the top_m of all drawn nodes by
 * (value desc, depth asc, creation order asc).
 * kind 1: static template ([B] "从一条草稿变成一棵候选树"): nodes listed by depth,
 * node i is child number node_rank[i] of node_parent[i] (-1 = root). */
typedef struct {
  int kind;
  int top_k;                            /* children drawn per expanded node */
  int depth;                            /* layers below the root */
  int top_m;                            /* retained nodes (excl. root) */
  int n_expanded;                       /* expanded slots the plan uses */
  int n_layers;                         /* draft layers (= depth for kind 0) */
  int layer_e0[EAGLE_MAX_NODES];        /* first expanded slot of draft layer l */
  int layer_rows[EAGLE_MAX_NODES];      /* expanded slots of draft layer l */
  int n_nodes;                          /* kind 1: template nodes */
  int16_t node_parent[EAGLE_MAX_NODES]; /* kind 1: template index of the parent, -1 root */
  int16_t node_rank[EAGLE_MAX_NODES];   /* kind 1: child number under the parent */
  int16_t node_depth[EAGLE_MAX_NODES];  /* filled by eagle_plan_static */
  int16_t node_exp[EAGLE_MAX_NODES];    /* filled: expanded slot of the node or -1 */
} eagle_plan;

/* Draft head weights.  bf16 matrices [out][ld]; fp32 vectors. */
typedef struct {
  const uint16_t* w_fc;  int ld_fc;     /* [d][ld], in = 2d: columns 0..d-1 feature, d..2d-1 embedding */
  const float* b_fc;                    /* [d] */
  const float* g1;                      /* [d] RMSNorm gain before attention */
  const uint16_t* wq;    int ld_q;      /* [Hq*dh][ld], in = d */
  const uint16_t* wk;    int ld_k;      /* [Hkv*dh][ld] */
  const uint16_t* wv;    int ld_v;      /* [Hkv*dh][ld] */
  const uint16_t* wo;    int ld_o;      /* [d][ld], in = Hq*dh */
  const float* g2;                      /* [d] RMSNorm gain before the MLP */
  const uint16_t* w_gate; int ld_gate;  /* [F][ld], in = d */
  const uint16_t* w_up;   int ld_up;    /* [F][ld] */
  const uint16_t* w_down; int ld_down;  /* [d][ld], in = F */
  const uint16_t* embed;  int ld_embed; /* [V][ld] frozen target embedding, in = d */
  const uint16_t* w_lm;   int ld_lm;    /* [V][ld] frozen target LM head, in = d */
} eagle_draft_weights;

/* Block-table (paged) addressing of a KV cache ([C] "工程落地时真正要看什么":
 * the authoritative KV of accepted tokens lives in blocks that the serving
 * system's cache manager allocates; [B] "KV Cache 必须按事务提交": the commit
 * may land through block-table remapping, the logical state being the same).
 * With block_table == NULL the cache is contiguous, [B][cap][Hkv][dh].
 * Otherwise its k and v are block pools [n_blocks][block_size][Hkv][dh] and
 * position p < cap of request b is row p % block_size of block
 * block_table[b * (cap / block_size) + p / block_size]; a table entry < 0 (or
 * >= n_blocks) marks a block that is not allocated.  block_size is a power of
 * two that divides cap (EAGLE_ERR_INVALID_ARG otherwise).  The caller owns
 * the table and the blocks: the library reads the table and never changes it.
 * Rows of an unallocated block inside a request's length read as zeros and set
 * EAGLE_ERR_INVALID_ARG in the status word; a commit whose rows would land in
 * an unallocated block is refused (EAGLE_ERR_CAPACITY, see eagle_commit). */
typedef struct {
  const int32_t* block_table;  /* [B][cap / block_size] block ids (device), NULL: contiguous */
  int block_size;              /* rows per block */
  int n_blocks;                /* blocks in each pool */
} eagle_paging;

/* A KV cache of one attention layer: [B][cap][Hkv][dh] bf16, or block pools
 * addressed through `paging` (all zero: contiguous). */
typedef struct {
  uint16_t* k;
  uint16_t* v;
  int cap;                 /* rows per request */
  const int32_t* len;      /* [B] valid rows per request (device) */
  eagle_paging paging;     /* target caches only: the draft cache stays contiguous */
} eagle_kv;

/* Per-round request inputs. */
typedef struct {
  const int32_t* t_next;   /* [B] committed token at the root position */
  const float* f_last;     /* [B][d] verified feature of position L_b - 1 */
  const int32_t* pos0;     /* [B] root position L_b */
} eagle_requests;

/* Sampling controls ([A] §6.2).  temperature[b] <= 0 selects greedy for
 * request b (children = top-k logits; acceptance = target argmax walk).
 * Uniforms: Philox4x32-10 (Salmon et al., SC'11), key = (seed, 0x000EA61E),
 * counter = (draw index, node slot, purpose << 16 | request, round_id),
 * word 0; purpose 0 = child draw, 1 = accept test, 2 = final draw. */
typedef struct {
  const float* temperature;  /* [B] (device) */
  uint32_t seed;
  uint32_t round_id;
} eagle_sampling;

/* Expanded-node pool ([A] §10.3: the EAGLE-2 candidate set), [B][E] arrays
 * with E = max_expanded; anc is [B][E][EAGLE_MASK_WORDS(E)]. */
typedef struct {
  int32_t* token;       /* -1 marks an inactive slot */
  int32_t* parent;      /* expanded slot of the parent, -1 for the root */
  int32_t* rank;        /* draw rank under the parent */
  int32_t* depth;
  double*  value;       /* product of draft confidences root..node (root = 1) */
  uint64_t* anc;        /* bit j: expanded slot j is an ancestor or the node itself */
  int32_t* child_exp;   /* [B][E][K] expanded slot made from child (e, r), or -1 */
} eagle_pool;

/* Drawn children of each expanded node, in draw order: [B][E][K]. */
typedef struct {
  int32_t* token;       /* -1 when the draft distribution ran out of mass */
  float* prob;          /* q_e(token), the draft confidence */
} eagle_children;

/* Per-expanded-node outputs of the draft head. */
typedef struct {
  float* f_hat;         /* [B][E][d]  predicted feature f^ ([A] §4.1) */
  float* logits;        /* [B][E][V]  z = LM_Head(f^) */
  float* probs;         /* [B][E][V]  q = softmax(z / T) (T = 1 for greedy requests) */
  float* k_tree;        /* [B][E][Hkv][dh] fp32: the draft layer's K of each expanded row (post-RoPE) */
  float* v_tree;        /* [B][E][Hkv][dh] fp32 */
} eagle_draft_out;

/* Flattened verification tree, [B][S] arrays with S = tree stride; anc is
 * [B][S][EAGLE_MASK_WORDS(S)]. */
typedef struct {
  int32_t* token;
  int32_t* parent;      /* tree slot of the parent, -1 for slot 0 */
  int32_t* depth;
  int32_t* pos;         /* L_b + depth */
  int32_t* exp;         /* expanded slot of the node, or -1 if never expanded */
  uint64_t* anc;        /* ancestor-or-self bitmask over tree slots */
  int32_t* child_slot;  /* [B][E][K] tree slot of drawn child (e, r), -1 if pruned */
  int32_t* size;        /* [B] 1 + retained nodes */
  int stride;           /* S: slots allocated per request (>= 1 + top_m) */
} eagle_tree;

/* Acceptance result ([B] "Greedy 验证" / "随机采样验证"). */
typedef struct {
  int32_t* accept_len;  /* [B] accepted tree nodes below the root */
  int32_t* path;        /* [B][path_cap] tree slots, path[0] = 0 (root) */
  int32_t* final_token; /* [B] correction / bonus / residual token = next round's t_next */
  int32_t* last_slot;   /* [B] tree slot of the last accepted node (its true feature
                           becomes the next round's f_last) */
  int path_cap;         /* >= plan depth + 1 */
} eagle_accept_out;

typedef enum { EAGLE_PHASE_ROOT = 0, EAGLE_PHASE_FRONTIER = 1, EAGLE_PHASE_FINAL = 2 } eagle_phase;

/* ---- lifecycle ------------------------------------------------------------ */

/* Validates dims/limits against this library and the current device
 * (sm_103 required), returns a host-only context and the workspace size the
 * caller must allocate (device, 256-byte aligned).  Allocates no device memory.
 * Shape checks run before the device check, so they can be exercised
 * without a GPU. */
eagle_status eagle_create(eagle_ctx** out, const eagle_dims* dims, const eagle_limits* limits,
                          size_t* workspace_bytes);
eagle_status eagle_destroy(eagle_ctx* ctx);

/* Zeroes the workspace (counters and padding must start at zero).  Call once
 * after allocating it, and after any call that returned an error mid-flight. */
eagle_status eagle_workspace_init(eagle_ctx* ctx, void* workspace, cudaStream_t stream);

/* Reads and clears the device status word (synchronises `stream`). */
eagle_status eagle_read_device_status(eagle_ctx* ctx, void* workspace, cudaStream_t stream,
                                      int* status_out);

const char* eagle_status_string(eagle_status s);

/* Checks the device-side failure path of the kernels' waits.  Every wait of
 * the library's kernels on a barrier (a tile landing, a tensor-core result,
 * another warp's hand-off) is bounded: after 2 s it gives up, sets
 * EAGLE_ERR_TIMEOUT in the status word and returns, so a lost arrival ends
 * the launch with an error instead of a hang and the context stays usable.
 * One wait is on other CTAs of the same launch: when every tile of a
 * contraction is split and the whole grid fits the GPU at once, a split
 * tile's contributors wait for one another before sharing its epilogue; a
 * kernel of another stream that kept enough SMs busy for 2 s while the
 * grid started would end that launch with EAGLE_ERR_TIMEOUT.
 * This launches one CTA whose only wait, that same bounded wait, is on a
 * barrier nothing arrives at: about 2 s later the status word holds
 * EAGLE_ERR_TIMEOUT (read and clear it with eagle_read_device_status).
 * Asynchronous on `stream`; returns EAGLE_OK once launched (EAGLE_ERR_CUDA on
 * a launch failure, EAGLE_ERR_INVALID_ARG / EAGLE_ERR_ALIGN for the context
 * or workspace). */
eagle_status eagle_wait_selftest(eagle_ctx* ctx, void* workspace, cudaStream_t stream);

/* ---- plans (host only) ---------------------------------------------------- */

/* EAGLE-2 plan: layers 0..depth-1 run on 1, top_k, ..., top_k rows per request;
 * n_expanded = 1 + top_k * (depth - 1); FINAL keeps top_m of the
 * n_expanded * top_k drawn nodes. */
eagle_status eagle_plan_eagle2(eagle_plan* out, int top_k, int depth, int top_m);

/* Static plan from a template given as (parent, rank) per node, listed by
 * depth; every node's parent must precede it.  top_k = 1 + max rank. */
eagle_status eagle_plan_static(eagle_plan* out, int n_nodes, const int16_t* node_parent,
                               const int16_t* node_rank);

/* ---- the round ------------------------------------------------------------ */

/* eagle_draft_step -- run the draft head on draft layer `layer` of the plan
 * ([A] §4.1, §6.1; [B] "Advanced Token", "草稿头到底包含什么"; [C] "draft head 的结构和目标函数").
 * For every request b and expanded slot e of the layer (row token t =
 * pool.token[b][e], parent feature f = f_last[b] if e == 0 else
 * out.f_hat[b][pool.parent[b][e]], position pos0[b] + pool.depth[b][e]):
 *   h  = W_fc [f ; E[t]] + b_fc
 *   q,k,v = RoPE(W_{q,k,v} RMSNorm(h; g1))      k, v -> out.k_tree/v_tree[b][e]
 *   o  = softmax(q k^T / sqrt(dh)) v over draft_kv rows 0..len[b]-1 and the
 *        draft K/V of the expanded slots whose bit is set in pool.anc[b][e]
 *   h2 = h + W_o o;  f^ = h2 + W_down(SiLU(W_gate b) * W_up b), b = RMSNorm(h2; g2)
 *   z  = W_lm f^;  q = softmax(z / T)
 *   children: greedy -> the plan's top_k largest z (ties to the lower id);
 *             sampling -> top_k draws without replacement from q, each
 *             t = (u32 * S) >> 32 on weights floor(q * 2^40) (exact integers).
 * Rows whose token is -1 produce children -1.  Reads the pool written by
 * eagle_tree_expand_rerank; writes out[b][e] and children[b][e] for the
 * layer's slots only.  Row count = batch * layer_rows[layer] <= max_rows. */
eagle_status eagle_draft_step(eagle_ctx* ctx, const eagle_plan* plan, int layer, int batch,
                              const eagle_draft_weights* w, const eagle_requests* req,
                              const eagle_kv* draft_kv, const eagle_pool* pool,
                              const eagle_draft_out* out, const eagle_children* children,
                              const eagle_sampling* s, void* workspace, cudaStream_t stream);

/* eagle_tree_expand_rerank -- tree construction ([A] §10.3; [C] "EAGLE-2：固定树变成上下文感知动态树").
 *   ROOT     (layer ignored): slot 0 of every request = t_next, value 1.
 *   FRONTIER (layer l >= 1): the expanded slots of draft layer l from the
 *            children of layer l-1 -- EAGLE-2: top_k by (value desc, parent
 *            slot asc, draw rank asc), value = value(parent) * q (fp64);
 *            static: the template's nodes at depth l that have children.
 *   FINAL    : the verification tree -- EAGLE-2: top_m drawn nodes by
 *            (value desc, depth asc, parent slot asc, rank asc), connected
 *            because value never grows along a path and ties go shallower;
 *            static: every template node.  Flattens, fills parent/depth/pos/
 *            exp/anc/child_slot/size.  A selection that is not connected sets
 *            EAGLE_ERR_INVALID_TREE in the device status word. */
eagle_status eagle_tree_expand_rerank(eagle_ctx* ctx, const eagle_plan* plan, int phase, int layer,
                                      int batch, const eagle_requests* req,
                                      const eagle_children* children, const eagle_pool* pool,
                                      const eagle_tree* tree, void* workspace, cudaStream_t stream);

/* eagle_tree_verify_attn -- tree-masked attention of one target layer
 * ([B] "Tree Attention 如何一次验证多条路径"; [A] §12 item 5):
 *   out[b][s][h] = softmax(scale * q[b][s][h] . K^T) V over prefix rows
 *   0..prefix.len[b]-1 and tree slots j < tree.size[b] with bit j of
 *   tree.anc[b][s]; kv head = h / (Hq / Hkv).  A length beyond the cache
 *   (prefix.len[b] > prefix.cap) is read as prefix.cap rows and sets
 *   EAGLE_ERR_CAPACITY in the status word.  The prefix may be paged
 *   (prefix.paging): its rows are then read through the block table.
 * q: [B][S][Hq][dh] bf16; k_tree, v_tree: [B][S][Hkv][dh] bf16; out: [B][S][Hq][dh] fp32,
 * S = tree.stride.  Slots s >= tree.size[b] are not written. */
eagle_status eagle_tree_verify_attn(eagle_ctx* ctx, int batch, const uint16_t* q,
                                    const uint16_t* k_tree, const uint16_t* v_tree,
                                    const eagle_kv* prefix, const eagle_tree* tree, float scale,
                                    float* out, void* workspace, cudaStream_t stream);

/* eagle_tree_verify_attn_noalloc -- eagle_tree_verify_attn without a
 * workspace argument.  None of the three pages has a counterpart: this is a
 * deployment convenience around the same kernel, not part of the method.
 *
 * Who needs it: callers that cannot hand the library device memory -- a
 * plain C host that links only libeagle and owns no device allocator, or a
 * serving loop whose device memory is fully reserved at start-up and may not
 * allocate per call.  The call allocates nothing: no cudaMalloc / cudaFree
 * and no allocating library.  The split partials and the per-(request,
 * kv head) arrival counters live in a fixed 32 MiB static device array
 * inside libeagle, one per device.
 *
 * Limit: batch * n_kv_heads <= 16384 and
 *   batch * tree.stride * n_q_heads * (splits + 1) * (head_dim + 4) * 4 bytes
 *   <= 32 MiB - 64 KiB,
 * splits being the prefix split count the library picks (<= 31 and
 * <= 2 * SMs / (batch * n_kv_heads) - 1, at most one per 64 rows of
 * prefix.cap).  Example: batch 1, 32 query heads of 128, stride 27, 8
 * splits: 4.1 MB.
 * Beyond the limit the call returns EAGLE_ERR_CAPACITY and launches nothing;
 * use eagle_tree_verify_attn with a workspace instead.
 *
 * Zero state: the counters must be zero when a call starts.  The first call
 * on a device looks up the array's address, zeroes the counters on `stream`
 * and waits for `stream`; make that first call before any stream capture
 * begins.  Every call leaves the counters at zero again.  The partials need
 * no initial value.
 *
 * Races: every call on one device shares the one array.  Two calls whose
 * kernels may overlap in time (different streams with no ordering between
 * them, or several host threads) corrupt each other's partials and counters;
 * order them, e.g. on one stream.
 *
 * Arguments, layouts, results and the other errors: as eagle_tree_verify_attn. */
eagle_status eagle_tree_verify_attn_noalloc(eagle_ctx* ctx, int batch, const uint16_t* q,
                                            const uint16_t* k_tree, const uint16_t* v_tree,
                                            const eagle_kv* prefix, const eagle_tree* tree, float scale,
                                            float* out, cudaStream_t stream);

/* eagle_accept -- acceptance on the verified tree ([A] §6.2; [B] "Greedy 验证",
 * "随机采样验证"; [C] "为什么普通草稿模型不够理想").
 * target_logits [B][S][V] fp32 (the target's logits at every tree slot).
 * Writes target_argmax [B][S] (ties to the lower id) and, for sampling
 * requests, target_probs [B][S][V] = softmax(logits / T), then walks the tree:
 *  greedy   : descend while a retained child carries the target argmax; the
 *             final token is the argmax at the last node (correction or bonus).
 *  sampling : at node u test its drawn children in draw order; candidate i
 *             (drawn from q with candidates 0..i-1 removed, Q_i) is accepted
 *             iff u32 * Q_i[x] * sum(P) < P[x] * sum(Q_i) * 2^32 (integer
 *             weights floor(. * 2^40), i.e. r < p/q); accepted and retained ->
 *             descend with P = target weights of the child; accepted but
 *             pruned -> final token; rejected -> P = max(0, P sum(Q_i) - Q_i sum(P))
 *             shifted right until max < 2^40.  No candidate left -> final
 *             token = one draw from P.
 * q_probs = eagle_draft_out.probs. */
eagle_status eagle_accept(eagle_ctx* ctx, const eagle_plan* plan, int batch, const eagle_tree* tree,
                          const eagle_children* children, const float* target_logits,
                          const float* q_probs, const eagle_sampling* s, float* target_probs,
                          int32_t* target_argmax, const eagle_accept_out* out,
                          void* workspace, cudaStream_t stream);

/* The walk of eagle_accept alone, on given target probabilities (fp32
 * [B][S][V]) and argmax ([B][S]); for callers that compute p themselves. */
eagle_status eagle_accept_from_probs(eagle_ctx* ctx, const eagle_plan* plan, int batch,
                                     const eagle_tree* tree, const eagle_children* children,
                                     const float* target_probs, const int32_t* target_argmax,
                                     const float* q_probs, const eagle_sampling* s,
                                     const eagle_accept_out* out, void* workspace,
                                     cudaStream_t stream);

/* Commit outputs. */
typedef struct {
  float* f_commit;      /* [B][path_cap][d] true features of path slots 0..a */
  int32_t* tok_commit;  /* [B][path_cap + 1] tokens of path slots 0..a, then the final token */
  float* f_last;        /* [B][d] next round's f_last = true feature of the last accepted slot */
  int32_t* t_next;      /* [B] next round's root token = final token */
  int32_t* prefix_len;  /* [B] L_b + 1 + a */
  int32_t* draft_len;   /* [B] draft_kv.len[b] + 1 (the root's draft row is appended) */
} eagle_commit_out;

/* eagle_commit -- the commit transaction ([B] "KV Cache 必须按事务提交"; [A] §6.2
 * closing remark and §12 item 3): for every layer l < n_layers, copy the
 * tree K/V rows of path slots 0..a of request b to target cache rows
 * L_b..L_b+a (L_b = target_kv_len[b]); gather the true features f_true[b][path];
 * append the root's draft K/V (its row used the verified f_last; rounded to the
 * cache's bf16) to the draft cache at row draft_kv.len[b]; rejected branches
 * are simply not copied.
 * k_tree_layers / v_tree_layers / k_cache_layers / v_cache_layers are HOST
 * arrays of n_layers device pointers ([B][S][Hkv][dh] and [B][kv_cap][Hkv][dh]).
 * target_paging (host pointer, NULL: contiguous caches) pages every target
 * layer's cache through one block table: k_cache_layers[l] / v_cache_layers[l]
 * are then layer l's block pools and row L_b + i lands in the block that the
 * table maps position L_b + i to (eagle_paging).
 * f_true: [B][S][d] fp32.  Output buffers must not alias inputs.
 * Capacity (checked on the device, where the lengths live): a request whose
 * target cache cannot take its 1 + a rows (L_b + 1 + a > kv_cap), or whose
 * draft cache is full (draft_kv.len[b] >= draft_kv.cap), is not committed:
 * no cache row of it is written, prefix_len / draft_len keep the old
 * lengths, its other outputs are unspecified, and EAGLE_ERR_CAPACITY is set
 * in the workspace's status word.  With target_paging, a request any of whose
 * 1 + a rows maps to an unallocated block is refused the same way. */
eagle_status eagle_commit(eagle_ctx* ctx, int batch, const eagle_accept_out* acc,
                          const eagle_tree* tree, const float* f_true, int n_layers,
                          const uint16_t* const* k_tree_layers, const uint16_t* const* v_tree_layers,
                          uint16_t* const* k_cache_layers, uint16_t* const* v_cache_layers,
                          int kv_cap, const int32_t* target_kv_len, const eagle_paging* target_paging,
                          const eagle_draft_out* draft, const eagle_kv* draft_kv,
                          const eagle_commit_out* out, void* workspace, cudaStream_t stream);

/* eagle_draft_refresh -- the draft layer's K/V of the accepted path's
 * positions, computed from the target's true features, appended to the
 * draft cache: after a round the drafter continues from the committed path,
 * not from its own drafted features ([B] "KV Cache 必须按事务提交"; [A] §6.2
 * closing remark; [C] "工程落地时真正要看什么").  With the round's root at
 * position L_b = pos0[b] and a = acc.accept_len[b] accepted nodes, for
 * i = 1 .. a (at most acc.path_cap - 1):
 *   x = [cm.f_commit[b][i-1] ; E[cm.tok_commit[b][i]]]   (true feature of
 *       position L_b + i - 1, token at position L_b + i)
 *   k, v = RoPE(W_{k,v} RMSNorm(W_fc x + b_fc; g1)) at position L_b + i
 * go (bf16) to draft_kv rows draft_kv.len[b] + i - 1, and
 * len_out[b] = draft_kv.len[b] + a.  The root's own row (position L_b) was
 * appended by eagle_commit, so pass draft_kv.len = that call's
 * cm.draft_len; the next round's root row (the final token at L_b + a + 1)
 * comes from its own first draft step.  Run once over a prompt (f_commit =
 * the prompt's features, tok_commit = its tokens, accept_len = rows) it
 * fills the draft cache for a new request.
 * Layouts: cm.f_commit [B][acc.path_cap][d] fp32, cm.tok_commit
 * [B][acc.path_cap + 1]; batch * (acc.path_cap - 1) <= max_rows
 * (EAGLE_ERR_CAPACITY).  A request whose cache cannot take its a rows
 * writes none and keeps its length (EAGLE_ERR_CAPACITY in the status word).
 * len_out must not alias draft_kv.len (EAGLE_ERR_INVALID_ARG).  Streams the
 * FC and the K / V projection weights once. */
eagle_status eagle_draft_refresh(eagle_ctx* ctx, int batch, const eagle_draft_weights* w,
                                 const eagle_accept_out* acc, const eagle_commit_out* cm, const int32_t* pos0,
                                 const eagle_kv* draft_kv, int32_t* len_out, void* workspace,
                                 cudaStream_t stream);

/* eagle_fuse_features -- the EAGLE-3 input ([C] "EAGLE-3：放弃 feature
 * prediction，改成多层特征融合与 training-time test"): the target's low-, middle-
 * and high-layer features of a position, each of dimension d, concatenated
 * and compressed back to d,
 *   g[j] = W_fuse [l_j ; m_j ; h_j] (+ b_fuse),
 * for n_rows rows.  g then takes the place of the feature f everywhere the
 * round reads a target feature: the round's f_last, and the true features
 * of the tree slots (f_true) that eagle_commit gathers and
 * eagle_draft_refresh reads; drafted rows still carry the draft's own
 * outputs, as in EAGLE-1 and EAGLE-2.
 * w_fuse [d][ld_fuse] bf16 (ld_fuse >= 3d, % 8 == 0), columns 0..d-1 take
 * l, d..2d-1 m, 2d..3d-1 h; b_fuse [d] fp32 or NULL (no bias); lmh
 * [n_rows][3d] fp32; g_out [n_rows][d] fp32; n_rows <= max_rows
 * (EAGLE_ERR_CAPACITY).  Streams W_fuse once. */
eagle_status eagle_fuse_features(eagle_ctx* ctx, const uint16_t* w_fuse, int ld_fuse, const float* b_fuse,
                                 int n_rows, const float* lmh, float* g_out, void* workspace,
                                 cudaStream_t stream);

/* ---- measurement --------------------------------------------------------- */

/* Kernel timing hook: while enabled, the library records a CUDA event before
 * and after every launch of kernel class `kernel_id` on the launching stream,
 * up to `capacity` pairs.  Events are created here (host-side objects, not
 * device memory). */
typedef enum {
  EAGLE_K_ALL = -1, EAGLE_K_GEMM_FC = 0, EAGLE_K_GEMM_QKV = 1, EAGLE_K_GEMM_O = 2,
  EAGLE_K_GEMM_GATEUP = 3, EAGLE_K_GEMM_DOWN = 4, EAGLE_K_GEMM_LM = 5, EAGLE_K_DRAFT_ATTN = 6,
  EAGLE_K_SELECT = 7, EAGLE_K_TREE = 8, EAGLE_K_VERIFY_ATTN = 9, EAGLE_K_ACCEPT = 10,
  EAGLE_K_COMMIT = 11, EAGLE_K_PREP = 12, EAGLE_K_REFRESH = 13, EAGLE_K_FUSE = 14
} eagle_kernel_id;
eagle_status eagle_trace_enable(eagle_ctx* ctx, int kernel_id, int capacity);
/* Synchronises the recorded events; writes up to `cap` durations in ms, the
 * kernel class of each (ids_out may be NULL) and the count. */
eagle_status eagle_trace_read(eagle_ctx* ctx, float* ms_out, int* ids_out, int cap, int* n_out);
eagle_status eagle_trace_disable(eagle_ctx* ctx);

/* Launch timestamps, for measuring kernels inside an untraced round (a CUDA
 * graph replay keeps the programmatic overlap between kernels, which event
 * pairs around each launch would break).  While enabled, the i-th launch
 * issued through this context (counted from enable; launches captured into a
 * graph keep their slot on every replay) has thread 0 of each CTA record
 * %globaltimer nanoseconds into stamps[3i] (atomic min, when the CTA
 * starts), stamps[3i+1] (atomic min, when it has passed its wait for the
 * preceding kernels' results) and stamps[3i+2] (atomic max, when the thread
 * leaves the kernel).  `stamps` is a caller-owned device buffer of
 * 3 * capacity uint64_t that the caller sets to (UINT64_MAX, UINT64_MAX, 0)
 * triples before each run it measures; launches beyond `capacity` are not
 * recorded.  Costs one atomic per CTA and stamp. */
eagle_status eagle_stamps_enable(eagle_ctx* ctx, uint64_t* stamps, int capacity);
/* Stops assigning stamp slots; writes the kernel class (eagle_kernel_id) of
 * each stamped launch, in order, to ids_out (up to cap) and their count. */
eagle_status eagle_stamps_disable(eagle_ctx* ctx, int* ids_out, int cap, int* n_out);

/* Kernels this context has launched so far (host-side count). */
long long eagle_launch_count(const eagle_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_H */
