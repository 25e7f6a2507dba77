// The C ABI of libeagle: argument validation, workspace layout, plans and
// the sequencing of each call's kernels on the caller's stream.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <set>
#include <tuple>

#include "internal.h"

using namespace eagle;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define EAGLE_REQUIRE(cond, code) \
  do {                            \
    if (!(cond)) return (code);   \
  } while (0)
#define EAGLE_PTR(p)                                      \
  do {                                                    \
    if (!(p)) return EAGLE_ERR_INVALID_ARG;               \
    if (!aligned16(p)) return EAGLE_ERR_ALIGN;            \
  } while (0)
#define EAGLE_CUDA(expr)                                  \
  do {                                                    \
    if ((expr) != cudaSuccess) return EAGLE_ERR_CUDA;     \
  } while (0)

eagle_status check_dims(const eagle_dims* d) {
  EAGLE_REQUIRE(d, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(d->d > 0 && d->d % 64 == 0, EAGLE_ERR_SHAPE);
  EAGLE_REQUIRE(d->head_dim == 16 || d->head_dim == 32 || d->head_dim == 64 || d->head_dim == 128,
                EAGLE_ERR_SHAPE);
  EAGLE_REQUIRE(d->n_q_heads > 0 && d->n_kv_heads > 0 && d->n_q_heads % d->n_kv_heads == 0, EAGLE_ERR_SHAPE);
  EAGLE_REQUIRE((d->n_q_heads * d->head_dim) % 64 == 0 && (d->n_kv_heads * d->head_dim) % 64 == 0,
                EAGLE_ERR_SHAPE);
  EAGLE_REQUIRE(d->d_ff >= 8, EAGLE_ERR_SHAPE);
  EAGLE_REQUIRE(d->vocab >= 2 && d->vocab <= EAGLE_MAX_VOCAB, EAGLE_ERR_SHAPE);
  EAGLE_REQUIRE(d->rms_eps >= 0.f && std::isfinite(d->rms_eps), EAGLE_ERR_SHAPE);
  EAGLE_REQUIRE(d->rope_theta > 1.f && std::isfinite(d->rope_theta), EAGLE_ERR_SHAPE);
  return EAGLE_OK;
}

eagle_status check_limits(const eagle_limits* l) {
  EAGLE_REQUIRE(l, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(l->max_batch >= 1 && l->max_batch <= 65535, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(l->max_rows >= 1 && l->max_rows <= 256, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(l->max_expanded >= 1 && l->max_expanded <= EAGLE_MAX_NODES, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(l->max_children >= 1 && l->max_children <= EAGLE_MAX_CHILDREN, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(l->max_tree >= 1 && l->max_tree <= EAGLE_MAX_NODES, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(l->max_prefix >= 1, EAGLE_ERR_CAPACITY);
  return EAGLE_OK;
}

eagle_status check_plan(const eagle_ctx* c, const eagle_plan* p) {
  EAGLE_REQUIRE(p, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(p->kind == 0 || p->kind == 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(p->top_k >= 1 && p->top_k <= c->lim.max_children, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(p->n_expanded >= 1 && p->n_expanded <= c->lim.max_expanded, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(p->n_layers >= 1 && p->n_layers <= EAGLE_MAX_NODES, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(p->top_m >= 1 && p->top_m + 1 <= c->lim.max_tree, EAGLE_ERR_CAPACITY);
  return EAGLE_OK;
}

int splits_bound(const eagle_ctx* c, int pairs) { return attn_splits_bound(c, pairs, c->lim.max_prefix); }

void layout(eagle_ctx* c) {
  const eagle_dims& D = c->dims;
  const eagle_limits& L = c->lim;
  Workspace& W = c->ws;
  W.npmax = padded_rows(L.max_rows);
  auto r64 = [](int x) { return (x + 63) / 64 * 64; };
  W.kp_fc = r64(2 * D.d);
  W.kp_qkv = W.kp_gu = W.kp_lm = r64(D.d);
  W.kp_o = r64(D.n_q_heads * D.head_dim);
  W.kp_down = r64(D.d_ff);
  W.kp_fuse = r64(3 * D.d);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + std::max<size_t>(bytes, 1), 256);
    return o;
  };
  const size_t np2 = 2 * static_cast<size_t>(W.npmax);
  W.status = take(256);
  W.b_fc = take(np2 * W.kp_fc * 2);
  W.b_qkv = take(np2 * W.kp_qkv * 2);
  W.b_o = take(np2 * W.kp_o * 2);
  W.b_gu = take(np2 * W.kp_gu * 2);
  W.b_down = take(np2 * W.kp_down * 2);
  W.b_lm = take(np2 * W.kp_lm * 2);
  W.b_fuse = take(np2 * W.kp_fuse * 2);
  W.h = take(static_cast<size_t>(L.max_rows) * D.d * 4);
  W.h2 = take(static_cast<size_t>(L.max_rows) * D.d * 4);
  W.qrow = take(static_cast<size_t>(L.max_rows) * D.n_q_heads * D.head_dim * 4);
  const int tiles_d = ceil_div(D.d, 128);
  W.ss_fc = take(static_cast<size_t>(L.max_rows) * tiles_d * 4);
  W.ss_o = take(static_cast<size_t>(L.max_rows) * tiles_d * 4);
  W.max_mtiles = std::max({tiles_d, ceil_div((D.n_q_heads + 2 * D.n_kv_heads) * D.head_dim, 128),
                           ceil_div(D.d_ff, 64), ceil_div(D.vocab, 128)});
  // split-tile partial slots t + cta: t < max_mtiles, cta < grid <= 2 * SMs
  W.gemm_part = take(static_cast<size_t>(W.max_mtiles + 2 * c->sm_count) * L.max_rows * 128 * 4);
  W.gemm_cnt = take(static_cast<size_t>(N_EPI) * W.max_mtiles * 4);
  // partial records of the widest attention launch: b requests use
  // splits_bound(b * Hkv) + 1 records per query row; past the batch where
  // the splits reach 1 the count grows as 2b, so the largest batch covers
  // every batch beyond the scanned ones
  size_t records = 0;
  const int scan = std::min(L.max_batch, 4096);
  for (int i = 0; i <= scan; ++i) {
    const int b = i < scan ? i + 1 : L.max_batch;
    const size_t s1 = static_cast<size_t>(splits_bound(c, b * D.n_kv_heads) + 1);
    records = std::max(records, static_cast<size_t>(L.max_rows) * D.n_q_heads * s1);
    records = std::max(records, static_cast<size_t>(b) * L.max_tree * D.n_q_heads * s1);
  }
  W.attn_part = take(records * (D.head_dim + 4) * 4);
  W.attn_cnt = take(static_cast<size_t>(2) * L.max_batch * D.n_kv_heads * 4);
  W.total = off;
}

eagle_status check_weights(const eagle_ctx* c, const eagle_draft_weights* w) {
  EAGLE_REQUIRE(w, EAGLE_ERR_INVALID_ARG);
  const eagle_dims& D = c->dims;
  const int qd = D.n_q_heads * D.head_dim;
  const struct { const void* p; int ld; int in; } mats[] = {
      {w->w_fc, w->ld_fc, 2 * D.d}, {w->wq, w->ld_q, D.d},        {w->wk, w->ld_k, D.d},
      {w->wv, w->ld_v, D.d},        {w->wo, w->ld_o, qd},         {w->w_gate, w->ld_gate, D.d},
      {w->w_up, w->ld_up, D.d},     {w->w_down, w->ld_down, D.d_ff}, {w->embed, w->ld_embed, D.d},
      {w->w_lm, w->ld_lm, D.d}};
  for (const auto& m : mats) {
    EAGLE_PTR(m.p);
    EAGLE_REQUIRE(m.ld >= m.in, EAGLE_ERR_SHAPE);
    EAGLE_REQUIRE(m.ld % 8 == 0, EAGLE_ERR_ALIGN);
  }
  EAGLE_PTR(w->b_fc);
  EAGLE_PTR(w->g1);
  EAGLE_PTR(w->g2);
  return EAGLE_OK;
}

eagle_status check_pool(const eagle_pool* p) {
  EAGLE_REQUIRE(p, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(p->token); EAGLE_PTR(p->parent); EAGLE_PTR(p->rank); EAGLE_PTR(p->depth);
  EAGLE_PTR(p->value); EAGLE_PTR(p->anc); EAGLE_PTR(p->child_exp);
  return EAGLE_OK;
}

eagle_status check_tree(const eagle_ctx* c, const eagle_tree* t) {
  EAGLE_REQUIRE(t, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(t->token); EAGLE_PTR(t->parent); EAGLE_PTR(t->depth); EAGLE_PTR(t->pos);
  EAGLE_PTR(t->exp); EAGLE_PTR(t->anc); EAGLE_PTR(t->child_slot); EAGLE_PTR(t->size);
  EAGLE_REQUIRE(t->stride >= 1 && t->stride <= c->lim.max_tree, EAGLE_ERR_CAPACITY);
  return EAGLE_OK;
}

eagle_status check_children(const eagle_children* ch) {
  EAGLE_REQUIRE(ch, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(ch->token);
  EAGLE_PTR(ch->prob);
  return EAGLE_OK;
}

// A block table (if any) over a cache of cap rows per request: block_size a
// power of two dividing cap, at least one block in the pools.
eagle_status check_paging(const eagle_paging* pg, int cap) {
  if (pg == nullptr || pg->block_table == nullptr) return EAGLE_OK;
  EAGLE_PTR(pg->block_table);
  const int bs = pg->block_size;
  EAGLE_REQUIRE(bs >= 1 && (bs & (bs - 1)) == 0 && cap % bs == 0, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(pg->n_blocks >= 1, EAGLE_ERR_INVALID_ARG);
  return EAGLE_OK;
}

// paged: the cache may be addressed through a block table (target caches);
// the draft cache is always contiguous
eagle_status check_kv(const eagle_ctx* c, const eagle_kv* kv, bool paged = false) {
  EAGLE_REQUIRE(kv, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(kv->k); EAGLE_PTR(kv->v); EAGLE_PTR(kv->len);
  EAGLE_REQUIRE(kv->cap >= 1, EAGLE_ERR_SHAPE);
  // the workspace's attention records are sized for caches up to max_prefix
  EAGLE_REQUIRE(kv->cap <= c->lim.max_prefix, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(paged || kv->paging.block_table == nullptr, EAGLE_ERR_INVALID_ARG);
  return check_paging(&kv->paging, kv->cap);
}

eagle_status check_ws(const void* ws) {
  EAGLE_REQUIRE(ws, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, EAGLE_ERR_ALIGN);
  return EAGLE_OK;
}

}  // namespace

namespace eagle {

namespace {
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CtxQuery {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
  CtxQuery() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(fn);
  }
};

std::mutex once_mu;
std::set<std::tuple<unsigned long long, const void*, int>> once_done;
}  // namespace

bool current_context_id(unsigned long long* id) {
  static const CtxQuery q;
  if (!q.get_current || !q.get_id) return false;
  CUcontext c = nullptr;
  if (q.get_current(&c) != CUDA_SUCCESS) return false;
  if (c == nullptr) {
    // no current context yet: select the device, which makes its primary
    // context current (the runtime initialises it there)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return false;
    if (q.get_current(&c) != CUDA_SUCCESS || c == nullptr) return false;
  }
  return q.get_id(c, id) == CUDA_SUCCESS;
}

cudaError_t cluster_nonportable_once(const void* kernel) {
  unsigned long long id = 0;
  if (!current_context_id(&id)) return cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  const auto key = std::make_tuple(id, kernel, -1);
  std::lock_guard<std::mutex> lock(once_mu);
  if (once_done.count(key)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) once_done.insert(key);
  return e;
}

cudaError_t smem_limit_once(const void* kernel, int bytes) {
  unsigned long long id = 0;
  if (!current_context_id(&id)) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  const auto key = std::make_tuple(id, kernel, bytes);
  std::lock_guard<std::mutex> lock(once_mu);
  if (once_done.count(key)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) once_done.insert(key);
  return e;
}

void trace_before(eagle_ctx* ctx, int kernel_id, cudaStream_t s) {
  TraceState& t = ctx->trace;
  if (t.kernel_id == -2 || (t.kernel_id != -1 && t.kernel_id != kernel_id) || t.n >= t.capacity) return;
  // external records: inside a stream capture they become timing nodes of the graph
  cudaEventRecordWithFlags(t.events[2 * t.n], s, cudaEventRecordExternal);
}
void trace_after(eagle_ctx* ctx, int kernel_id, cudaStream_t s) {
  TraceState& t = ctx->trace;
  if (t.kernel_id == -2 || (t.kernel_id != -1 && t.kernel_id != kernel_id) || t.n >= t.capacity) return;
  cudaEventRecordWithFlags(t.events[2 * t.n + 1], s, cudaEventRecordExternal);
  t.ids[t.n] = kernel_id;
  ++t.n;
}

}  // namespace eagle

extern "C" {

const char* eagle_status_string(eagle_status s) {
  switch (s) {
    case EAGLE_OK: return "ok";
    case EAGLE_ERR_INVALID_ARG: return "invalid argument";
    case EAGLE_ERR_SHAPE: return "unsupported or inconsistent shape";
    case EAGLE_ERR_ALIGN: return "pointer or pitch not 16-byte aligned";
    case EAGLE_ERR_CAPACITY: return "beyond the context's capacity";
    case EAGLE_ERR_INVALID_TREE: return "invalid tree";
    case EAGLE_ERR_NUMERIC: return "non-finite values or zero-mass distribution";
    case EAGLE_ERR_TIMEOUT: return "device-side wait timed out";
    case EAGLE_ERR_UNSUPPORTED: return "unsupported device";
    case EAGLE_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

eagle_status eagle_create(eagle_ctx** out, const eagle_dims* dims, const eagle_limits* limits,
                          size_t* workspace_bytes) {
  EAGLE_REQUIRE(out && workspace_bytes, EAGLE_ERR_INVALID_ARG);
  *out = nullptr;
  eagle_status st = check_dims(dims);
  if (st != EAGLE_OK) return st;
  st = check_limits(limits);
  if (st != EAGLE_OK) return st;
  int dev = 0, n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) {
    cudaGetLastError();
    return EAGLE_ERR_UNSUPPORTED;
  }
  EAGLE_CUDA(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  EAGLE_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (!(prop.major == 10 && prop.minor == 3)) return EAGLE_ERR_UNSUPPORTED;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return EAGLE_ERR_UNSUPPORTED;
  eagle_ctx* c = new eagle_ctx();
  c->dims = *dims;
  c->lim = *limits;
  c->device = dev;
  c->sm_count = prop.multiProcessorCount;
  c->encode = reinterpret_cast<EncodeTiledFn>(fn);
  layout(c);
  *workspace_bytes = c->ws.total;
  *out = c;
  return EAGLE_OK;
}

eagle_status eagle_destroy(eagle_ctx* ctx) {
  if (!ctx) return EAGLE_ERR_INVALID_ARG;
  for (cudaEvent_t e : ctx->trace.events) cudaEventDestroy(e);
  delete ctx;
  return EAGLE_OK;
}

eagle_status eagle_workspace_init(eagle_ctx* ctx, void* workspace, cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  eagle_status st = check_ws(workspace);
  if (st != EAGLE_OK) return st;
  EAGLE_CUDA(cudaMemsetAsync(workspace, 0, ctx->ws.total, stream));
  return EAGLE_OK;
}

eagle_status eagle_read_device_status(eagle_ctx* ctx, void* workspace, cudaStream_t stream, int* status_out) {
  EAGLE_REQUIRE(ctx && status_out, EAGLE_ERR_INVALID_ARG);
  eagle_status st = check_ws(workspace);
  if (st != EAGLE_OK) return st;
  int v = 0;
  EAGLE_CUDA(cudaMemcpyAsync(&v, ws_ptr<int>(workspace, ctx->ws.status), sizeof(int), cudaMemcpyDeviceToHost,
                             stream));
  EAGLE_CUDA(cudaStreamSynchronize(stream));
  EAGLE_CUDA(cudaMemsetAsync(ws_ptr<int>(workspace, ctx->ws.status), 0, sizeof(int), stream));
  EAGLE_CUDA(cudaStreamSynchronize(stream));
  *status_out = v;
  return EAGLE_OK;
}

eagle_status eagle_plan_eagle2(eagle_plan* out, int top_k, int depth, int top_m) {
  EAGLE_REQUIRE(out, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(top_k >= 1 && top_k <= EAGLE_MAX_CHILDREN, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(depth >= 1, EAGLE_ERR_INVALID_ARG);
  const int n_exp = 1 + top_k * (depth - 1);
  EAGLE_REQUIRE(n_exp <= EAGLE_MAX_NODES, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(top_m >= 1 && top_m + 1 <= EAGLE_MAX_NODES && top_m <= n_exp * top_k, EAGLE_ERR_CAPACITY);
  std::memset(out, 0, sizeof(*out));
  out->kind = 0;
  out->top_k = top_k;
  out->depth = depth;
  out->top_m = top_m;
  out->n_expanded = n_exp;
  out->n_layers = depth;
  out->layer_e0[0] = 0;
  out->layer_rows[0] = 1;
  for (int l = 1; l < depth; ++l) {
    out->layer_e0[l] = 1 + (l - 1) * top_k;
    out->layer_rows[l] = top_k;
  }
  return EAGLE_OK;
}

eagle_status eagle_plan_static(eagle_plan* out, int n_nodes, const int16_t* node_parent,
                               const int16_t* node_rank) {
  EAGLE_REQUIRE(out && node_parent && node_rank, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(n_nodes >= 1 && n_nodes + 1 <= EAGLE_MAX_NODES, EAGLE_ERR_CAPACITY);
  eagle_plan p;
  std::memset(&p, 0, sizeof(p));
  p.kind = 1;
  p.n_nodes = n_nodes;
  int kmax = 0, dmax = 0;
  bool has_child[EAGLE_MAX_NODES] = {false};
  for (int i = 0; i < n_nodes; ++i) {
    const int par = node_parent[i], r = node_rank[i];
    EAGLE_REQUIRE(par >= -1 && par < i, EAGLE_ERR_INVALID_TREE);
    EAGLE_REQUIRE(r >= 0 && r < EAGLE_MAX_CHILDREN, EAGLE_ERR_INVALID_TREE);
    for (int j = 0; j < i; ++j)
      EAGLE_REQUIRE(!(node_parent[j] == par && node_rank[j] == r), EAGLE_ERR_INVALID_TREE);
    p.node_parent[i] = static_cast<int16_t>(par);
    p.node_rank[i] = static_cast<int16_t>(r);
    const int dep = par < 0 ? 1 : p.node_depth[par] + 1;
    EAGLE_REQUIRE(i == 0 || dep >= p.node_depth[i - 1], EAGLE_ERR_INVALID_TREE);   // listed by depth
    p.node_depth[i] = static_cast<int16_t>(dep);
    if (par >= 0) has_child[par] = true;
    kmax = std::max(kmax, r + 1);
    dmax = std::max(dmax, dep);
  }
  int e = 1;
  for (int i = 0; i < n_nodes; ++i) p.node_exp[i] = has_child[i] ? static_cast<int16_t>(e++) : -1;
  EAGLE_REQUIRE(e <= EAGLE_MAX_NODES, EAGLE_ERR_CAPACITY);
  p.top_k = kmax;
  p.depth = dmax;
  p.top_m = n_nodes;
  p.n_expanded = e;
  p.n_layers = dmax;
  p.layer_e0[0] = 0;
  p.layer_rows[0] = 1;
  int next = 1;
  for (int l = 1; l < dmax; ++l) {
    int rows = 0;
    for (int i = 0; i < n_nodes; ++i)
      if (has_child[i] && p.node_depth[i] == l) ++rows;
    p.layer_e0[l] = next;
    p.layer_rows[l] = rows;
    next += rows;
  }
  *out = p;
  return EAGLE_OK;
}

eagle_status eagle_draft_step(eagle_ctx* ctx, const eagle_plan* plan, int layer, int batch,
                              const eagle_draft_weights* w, const eagle_requests* req, const eagle_kv* draft_kv,
                              const eagle_pool* pool, const eagle_draft_out* out, const eagle_children* children,
                              const eagle_sampling* s, void* workspace, cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  eagle_status st = check_plan(ctx, plan);
  if (st != EAGLE_OK) return st;
  EAGLE_REQUIRE(layer >= 0 && layer < plan->n_layers, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(batch >= 1 && batch <= ctx->lim.max_batch, EAGLE_ERR_CAPACITY);
  const int rpr = plan->layer_rows[layer];
  EAGLE_REQUIRE(rpr >= 1, EAGLE_ERR_INVALID_ARG);
  const int n = batch * rpr;
  EAGLE_REQUIRE(n <= ctx->lim.max_rows, EAGLE_ERR_CAPACITY);
  if ((st = check_weights(ctx, w)) != EAGLE_OK) return st;
  EAGLE_REQUIRE(req, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(req->f_last); EAGLE_PTR(req->pos0);
  if ((st = check_kv(ctx, draft_kv)) != EAGLE_OK) return st;
  if ((st = check_pool(pool)) != EAGLE_OK) return st;
  EAGLE_REQUIRE(out, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(out->f_hat); EAGLE_PTR(out->logits); EAGLE_PTR(out->probs); EAGLE_PTR(out->k_tree);
  EAGLE_PTR(out->v_tree);
  if ((st = check_children(children)) != EAGLE_OK) return st;
  EAGLE_REQUIRE(s, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(s->temperature);
  if ((st = check_ws(workspace)) != EAGLE_OK) return st;

  DraftLaunch L{};
  L.plan = plan;
  L.layer = layer;
  L.batch = batch;
  L.e0 = plan->layer_e0[layer];
  L.rpr = rpr;
  L.n = n;
  L.NP = padded_rows(n);
  L.k = plan->top_k;
  L.w = w;
  L.req = req;
  L.draft_kv = draft_kv;
  L.pool = pool;
  L.out = out;
  L.children = children;
  L.s = s;
  L.ws = workspace;
  EAGLE_CUDA(launch_prep_fc(ctx, L, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_FC, L, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_QKV, L, stream));
  EAGLE_CUDA(launch_draft_attn(ctx, L, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_O, L, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_GATEUP, L, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_DOWN, L, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_LM, L, stream));
  EAGLE_CUDA(launch_select(ctx, L, stream));
  return EAGLE_OK;
}

eagle_status eagle_draft_refresh(eagle_ctx* ctx, int batch, const eagle_draft_weights* w, const eagle_accept_out* acc,
                                 const eagle_commit_out* cm, const int32_t* pos0, const eagle_kv* draft_kv,
                                 int32_t* len_out, void* workspace, cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(batch >= 1 && batch <= ctx->lim.max_batch, EAGLE_ERR_CAPACITY);
  eagle_status st = check_weights(ctx, w);
  if (st != EAGLE_OK) return st;
  EAGLE_REQUIRE(acc && cm, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(acc->accept_len);
  EAGLE_REQUIRE(acc->path_cap >= 2, EAGLE_ERR_SHAPE);
  EAGLE_PTR(cm->f_commit); EAGLE_PTR(cm->tok_commit);
  EAGLE_PTR(pos0);
  if ((st = check_kv(ctx, draft_kv)) != EAGLE_OK) return st;
  EAGLE_PTR(len_out);
  EAGLE_REQUIRE(len_out != draft_kv->len, EAGLE_ERR_INVALID_ARG);
  if ((st = check_ws(workspace)) != EAGLE_OK) return st;
  const int R = acc->path_cap - 1;
  EAGLE_REQUIRE(static_cast<long long>(batch) * R <= ctx->lim.max_rows, EAGLE_ERR_CAPACITY);
  eagle_requests req{};
  req.pos0 = pos0;
  DraftLaunch L{};
  L.batch = batch;
  L.rpr = R;
  L.e0 = 0;
  L.n = batch * R;
  L.NP = padded_rows(L.n);
  L.k = 1;
  L.w = w;
  L.req = &req;
  L.ws = workspace;
  L.refresh_kv = draft_kv;
  L.refresh_n = acc->accept_len;
  EAGLE_CUDA(launch_prep_refresh(ctx, L, cm->f_commit, cm->tok_commit, acc->path_cap, len_out, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_FC, L, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_KV, L, stream));
  return EAGLE_OK;
}

eagle_status eagle_fuse_features(eagle_ctx* ctx, const uint16_t* w_fuse, int ld_fuse, const float* b_fuse, int n_rows,
                                 const float* lmh, float* g_out, void* workspace, cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(w_fuse);
  EAGLE_REQUIRE(ld_fuse >= 3 * ctx->dims.d, EAGLE_ERR_SHAPE);
  EAGLE_REQUIRE(ld_fuse % 8 == 0, EAGLE_ERR_ALIGN);
  if (b_fuse) EAGLE_PTR(b_fuse);
  EAGLE_REQUIRE(n_rows >= 1 && n_rows <= ctx->lim.max_rows, EAGLE_ERR_CAPACITY);
  EAGLE_PTR(lmh); EAGLE_PTR(g_out);
  eagle_status st = check_ws(workspace);
  if (st != EAGLE_OK) return st;
  DraftLaunch L{};
  L.batch = 1;
  L.rpr = n_rows;
  L.n = n_rows;
  L.NP = padded_rows(n_rows);
  L.k = 1;
  L.ws = workspace;
  L.w_fuse = w_fuse;
  L.ld_fuse = ld_fuse;
  L.b_fuse = b_fuse;
  L.g_out = g_out;
  EAGLE_CUDA(launch_prep_fuse(ctx, L, lmh, stream));
  EAGLE_CUDA(launch_gemm(ctx, EPI_FUSE, L, stream));
  return EAGLE_OK;
}

eagle_status eagle_tree_expand_rerank(eagle_ctx* ctx, const eagle_plan* plan, int phase, int layer, int batch,
                                      const eagle_requests* req, const eagle_children* children,
                                      const eagle_pool* pool, const eagle_tree* tree, void* workspace,
                                      cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  eagle_status st = check_plan(ctx, plan);
  if (st != EAGLE_OK) return st;
  EAGLE_REQUIRE(batch >= 1 && batch <= ctx->lim.max_batch, EAGLE_ERR_CAPACITY);
  if ((st = check_pool(pool)) != EAGLE_OK) return st;
  if ((st = check_ws(workspace)) != EAGLE_OK) return st;
  EAGLE_REQUIRE(req, EAGLE_ERR_INVALID_ARG);
  if (phase == EAGLE_PHASE_ROOT) {
    EAGLE_PTR(req->t_next);
  } else if (phase == EAGLE_PHASE_FRONTIER) {
    EAGLE_REQUIRE(layer >= 1 && layer < plan->n_layers, EAGLE_ERR_INVALID_ARG);
    if ((st = check_children(children)) != EAGLE_OK) return st;
  } else if (phase == EAGLE_PHASE_FINAL) {
    if ((st = check_children(children)) != EAGLE_OK) return st;
    if ((st = check_tree(ctx, tree)) != EAGLE_OK) return st;
    EAGLE_PTR(req->pos0);
    EAGLE_REQUIRE(tree->stride >= 1 + plan->top_m, EAGLE_ERR_CAPACITY);
  } else {
    return EAGLE_ERR_INVALID_ARG;
  }
  EAGLE_CUDA(launch_tree(ctx, plan, phase, layer, batch, req, children, pool,
                         phase == EAGLE_PHASE_FINAL ? tree : nullptr, ws_ptr<int>(workspace, ctx->ws.status),
                         stream));
  return EAGLE_OK;
}

eagle_status eagle_tree_verify_attn(eagle_ctx* ctx, int batch, const uint16_t* q, const uint16_t* k_tree,
                                    const uint16_t* v_tree, const eagle_kv* prefix, const eagle_tree* tree,
                                    float scale, float* out, void* workspace, cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(batch >= 1 && batch <= ctx->lim.max_batch, EAGLE_ERR_CAPACITY);
  EAGLE_PTR(q); EAGLE_PTR(k_tree); EAGLE_PTR(v_tree); EAGLE_PTR(out);
  eagle_status st = check_kv(ctx, prefix, true);
  if (st != EAGLE_OK) return st;
  if ((st = check_tree(ctx, tree)) != EAGLE_OK) return st;
  if ((st = check_ws(workspace)) != EAGLE_OK) return st;
  EAGLE_REQUIRE(std::isfinite(scale) && scale > 0.f, EAGLE_ERR_INVALID_ARG);
  EAGLE_CUDA(launch_verify_attn(ctx, batch, q, k_tree, v_tree, prefix, tree, scale, out, workspace, stream));
  return EAGLE_OK;
}

eagle_status eagle_tree_verify_attn_noalloc(eagle_ctx* ctx, int batch, const uint16_t* q, const uint16_t* k_tree,
                                            const uint16_t* v_tree, const eagle_kv* prefix, const eagle_tree* tree,
                                            float scale, float* out, cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(batch >= 1 && batch <= ctx->lim.max_batch, EAGLE_ERR_CAPACITY);
  EAGLE_PTR(q); EAGLE_PTR(k_tree); EAGLE_PTR(v_tree); EAGLE_PTR(out);
  eagle_status st = check_kv(ctx, prefix, true);
  if (st != EAGLE_OK) return st;
  if ((st = check_tree(ctx, tree)) != EAGLE_OK) return st;
  EAGLE_REQUIRE(std::isfinite(scale) && scale > 0.f, EAGLE_ERR_INVALID_ARG);
  return launch_verify_attn_noalloc(ctx, batch, q, k_tree, v_tree, prefix, tree, scale, out, stream);
}

static eagle_status check_accept(eagle_ctx* ctx, const eagle_plan* plan, int batch, const eagle_tree* tree,
                                 const eagle_children* children, const float* q_probs, const eagle_sampling* s,
                                 const eagle_accept_out* out, void* workspace) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  eagle_status st = check_plan(ctx, plan);
  if (st != EAGLE_OK) return st;
  EAGLE_REQUIRE(batch >= 1 && batch <= ctx->lim.max_batch, EAGLE_ERR_CAPACITY);
  if ((st = check_tree(ctx, tree)) != EAGLE_OK) return st;
  if ((st = check_children(children)) != EAGLE_OK) return st;
  EAGLE_PTR(q_probs);
  EAGLE_REQUIRE(s, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(s->temperature);
  EAGLE_REQUIRE(out, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(out->accept_len); EAGLE_PTR(out->path); EAGLE_PTR(out->final_token); EAGLE_PTR(out->last_slot);
  EAGLE_REQUIRE(out->path_cap >= plan->depth + 1, EAGLE_ERR_CAPACITY);
  return check_ws(workspace);
}

eagle_status eagle_accept(eagle_ctx* ctx, const eagle_plan* plan, int batch, const eagle_tree* tree,
                          const eagle_children* children, const float* target_logits, const float* q_probs,
                          const eagle_sampling* s, float* target_probs, int32_t* target_argmax,
                          const eagle_accept_out* out, void* workspace, cudaStream_t stream) {
  eagle_status st = check_accept(ctx, plan, batch, tree, children, q_probs, s, out, workspace);
  if (st != EAGLE_OK) return st;
  EAGLE_PTR(target_logits); EAGLE_PTR(target_probs); EAGLE_PTR(target_argmax);
  EAGLE_CUDA(launch_target_softmax(ctx, batch, tree, target_logits, s->temperature, target_probs, target_argmax,
                                   workspace, stream));
  EAGLE_CUDA(launch_accept_walk(ctx, plan, batch, tree, children, target_probs, target_argmax, q_probs, s, out,
                                workspace, stream));
  return EAGLE_OK;
}

eagle_status eagle_accept_from_probs(eagle_ctx* ctx, const eagle_plan* plan, int batch, const eagle_tree* tree,
                                     const eagle_children* children, const float* target_probs,
                                     const int32_t* target_argmax, const float* q_probs, const eagle_sampling* s,
                                     const eagle_accept_out* out, void* workspace, cudaStream_t stream) {
  eagle_status st = check_accept(ctx, plan, batch, tree, children, q_probs, s, out, workspace);
  if (st != EAGLE_OK) return st;
  EAGLE_PTR(target_probs); EAGLE_PTR(target_argmax);
  EAGLE_CUDA(launch_accept_walk(ctx, plan, batch, tree, children, target_probs, target_argmax, q_probs, s, out,
                                workspace, stream));
  return EAGLE_OK;
}

eagle_status eagle_commit(eagle_ctx* ctx, int batch, const eagle_accept_out* acc, const eagle_tree* tree,
                          const float* f_true, int n_layers, const uint16_t* const* k_tree_layers,
                          const uint16_t* const* v_tree_layers, uint16_t* const* k_cache_layers,
                          uint16_t* const* v_cache_layers, int kv_cap, const int32_t* target_kv_len,
                          const eagle_paging* target_paging, const eagle_draft_out* draft,
                          const eagle_kv* draft_kv, const eagle_commit_out* out, void* workspace,
                          cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  EAGLE_REQUIRE(batch >= 1 && batch <= ctx->lim.max_batch, EAGLE_ERR_CAPACITY);
  EAGLE_REQUIRE(acc, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(acc->accept_len); EAGLE_PTR(acc->path); EAGLE_PTR(acc->final_token); EAGLE_PTR(acc->last_slot);
  EAGLE_REQUIRE(acc->path_cap >= 1, EAGLE_ERR_CAPACITY);
  eagle_status st = check_tree(ctx, tree);
  if (st != EAGLE_OK) return st;
  EAGLE_PTR(f_true);
  EAGLE_REQUIRE(n_layers >= 0 && n_layers <= EAGLE_MAX_LAYERS, EAGLE_ERR_CAPACITY);
  if (n_layers > 0) {
    EAGLE_REQUIRE(k_tree_layers && v_tree_layers && k_cache_layers && v_cache_layers, EAGLE_ERR_INVALID_ARG);
    for (int l = 0; l < n_layers; ++l) {
      EAGLE_PTR(k_tree_layers[l]); EAGLE_PTR(v_tree_layers[l]);
      EAGLE_PTR(k_cache_layers[l]); EAGLE_PTR(v_cache_layers[l]);
    }
  }
  EAGLE_REQUIRE(kv_cap >= 1, EAGLE_ERR_SHAPE);
  EAGLE_PTR(target_kv_len);
  if ((st = check_paging(target_paging, kv_cap)) != EAGLE_OK) return st;
  EAGLE_REQUIRE(out, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(out->f_commit); EAGLE_PTR(out->tok_commit); EAGLE_PTR(out->f_last); EAGLE_PTR(out->t_next);
  EAGLE_PTR(out->prefix_len);
  if (draft || draft_kv) {
    EAGLE_REQUIRE(draft && draft_kv, EAGLE_ERR_INVALID_ARG);
    EAGLE_PTR(draft->k_tree); EAGLE_PTR(draft->v_tree);
    if ((st = check_kv(ctx, draft_kv)) != EAGLE_OK) return st;
    EAGLE_PTR(out->draft_len);
  }
  if ((st = check_ws(workspace)) != EAGLE_OK) return st;
  CommitLaunch C{};
  C.batch = batch;
  C.n_layers = n_layers;
  C.kv_cap = kv_cap;
  C.paged = paged_of(target_paging, kv_cap);
  C.acc = acc;
  C.tree = tree;
  C.f_true = f_true;
  C.kt = k_tree_layers;
  C.vt = v_tree_layers;
  C.kc = k_cache_layers;
  C.vc = v_cache_layers;
  C.kv_len = target_kv_len;
  C.draft = draft;
  C.draft_kv = draft_kv;
  C.out = out;
  C.status = ws_ptr<int>(workspace, ctx->ws.status);
  EAGLE_CUDA(launch_commit(ctx, C, stream));
  return EAGLE_OK;
}

eagle_status eagle_trace_enable(eagle_ctx* ctx, int kernel_id, int capacity) {
  EAGLE_REQUIRE(ctx && capacity >= 1 && kernel_id >= -1 && kernel_id <= EAGLE_K_FUSE, EAGLE_ERR_INVALID_ARG);
  TraceState& t = ctx->trace;
  while (static_cast<int>(t.events.size()) < 2 * capacity) {
    cudaEvent_t e;
    EAGLE_CUDA(cudaEventCreate(&e));
    t.events.push_back(e);
  }
  t.ids.assign(capacity, -1);
  t.capacity = capacity;
  t.kernel_id = kernel_id;
  t.n = 0;
  return EAGLE_OK;
}

eagle_status eagle_trace_read(eagle_ctx* ctx, float* ms_out, int* ids_out, int cap, int* n_out) {
  EAGLE_REQUIRE(ctx && n_out && (ms_out || cap == 0), EAGLE_ERR_INVALID_ARG);
  TraceState& t = ctx->trace;
  const int n = std::min(t.n, cap);
  for (int i = 0; i < n; ++i) {
    EAGLE_CUDA(cudaEventSynchronize(t.events[2 * i + 1]));
    float ms = 0.f;
    EAGLE_CUDA(cudaEventElapsedTime(&ms, t.events[2 * i], t.events[2 * i + 1]));
    ms_out[i] = ms;
    if (ids_out) ids_out[i] = t.ids[i];
  }
  *n_out = n;
  return EAGLE_OK;
}

eagle_status eagle_trace_disable(eagle_ctx* ctx) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  ctx->trace.kernel_id = -2;
  ctx->trace.n = 0;
  return EAGLE_OK;
}

eagle_status eagle_stamps_enable(eagle_ctx* ctx, uint64_t* stamps, int capacity) {
  EAGLE_REQUIRE(ctx && capacity >= 1, EAGLE_ERR_INVALID_ARG);
  EAGLE_PTR(stamps);
  ctx->stamps = stamps;
  ctx->stamp_cap = capacity;
  ctx->stamp_ids.clear();
  return EAGLE_OK;
}

eagle_status eagle_stamps_disable(eagle_ctx* ctx, int* ids_out, int cap, int* n_out) {
  EAGLE_REQUIRE(ctx && n_out && (ids_out || cap == 0), EAGLE_ERR_INVALID_ARG);
  const int n = static_cast<int>(ctx->stamp_ids.size());
  for (int i = 0; i < n && i < cap; ++i) ids_out[i] = ctx->stamp_ids[i];
  *n_out = n;
  ctx->stamps = nullptr;
  ctx->stamp_cap = 0;
  ctx->stamp_ids.clear();
  return EAGLE_OK;
}

eagle_status eagle_wait_selftest(eagle_ctx* ctx, void* workspace, cudaStream_t stream) {
  EAGLE_REQUIRE(ctx, EAGLE_ERR_INVALID_ARG);
  eagle_status st = check_ws(workspace);
  if (st != EAGLE_OK) return st;
  EAGLE_CUDA(eagle::launch_wait_selftest(ctx, workspace, stream));
  return EAGLE_OK;
}

long long eagle_launch_count(const eagle_ctx* ctx) { return ctx ? ctx->launches : -1; }

}  // extern "C"
