// Tree construction on the device, one CTA per request ([A] §10.3; [C]
// "EAGLE-2：固定树变成上下文感知动态树").
//  ROOT     : slot 0 = t_next with value 1; every other expanded slot inactive.
//  FRONTIER : EAGLE-2 -- candidates are the k drawn children of the previous
//             layer's expanded nodes, value = value(parent) * q (fp64); keep
//             the top_k by (value desc, parent slot asc, draw rank asc) as the
//             new layer.  Static -- the template's nodes of this depth that
//             have children.
//  FINAL    : EAGLE-2 -- keep the top_m drawn nodes of the whole pool by
//             (value desc, depth asc, parent slot asc, rank asc); value never
//             grows along a path and ties go to the shallower node, so the
//             kept set is a connected tree.  Static -- every template node.
//             Then flatten: slots 1..m by (depth asc, selection rank asc),
//             parent slots, positions, ancestor bitmasks.
// Ancestor masks take EAGLE_MASK_WORDS(n) words per slot (n = expanded
// slots for the pool, tree slots for the tree): bit j is bit j % 64 of word
// j / 64.  A tree slot's mask is built by its own thread walking the parent
// chain to the root, every word in registers.
// A frontier layer's ranks come from counting (one warp per candidate, its
// lanes comparing the candidate's key with every other valid key in turn
// and summing the counts); the final selection's from a bitonic sort of the
// whole pool's candidates by the same total order (a few hundred keys: the
// counting's n^2 comparisons took ~30 us on one SM).  Both are exact and
// independent of thread order.  Node values
// are non-negative fp64 products, whose bit patterns order like the values
// as unsigned integers: the counting loops compare those (GB300 runs fp64
// comparisons at a small fraction of the integer rate).
#include "internal.h"
#include "common.cuh"

namespace eagle {
namespace {

constexpr int TREE_THREADS = 1024;
constexpr int TREE_WARPS = TREE_THREADS / 32;
constexpr int MAX_WORDS = EAGLE_MASK_WORDS(EAGLE_MAX_NODES);

struct TreeParams {
  eagle_plan plan;
  int phase, layer;
  int E, K, S;
  int WE, WS;                     // mask words per pool slot, per tree slot
  const int32_t* t_next;
  const int32_t* pos0;
  const int32_t* ctok;
  const float* cprob;
  int32_t* p_token;
  int32_t* p_parent;
  int32_t* p_rank;
  int32_t* p_depth;
  double* p_value;
  uint64_t* p_anc;
  int32_t* p_child_exp;
  int32_t* t_token;
  int32_t* t_parent;
  int32_t* t_depth;
  int32_t* t_pos;
  int32_t* t_exp;
  uint64_t* t_anc;
  int32_t* t_child_slot;
  int32_t* t_size;
  int* status;
  uint64_t* stamp;
};

// key order: true if entry a ranks before entry b (value keys: the bits of
// non-negative doubles, larger first; then depth, then creation order)
__device__ __forceinline__ bool before(uint64_t va, int da, int ca, uint64_t vb, int db, int cb) {
  if (va != vb) return va > vb;
  if (da != db) return da < db;
  return ca < cb;
}

__device__ __forceinline__ uint64_t value_key(double v) {
  return static_cast<uint64_t>(__double_as_longlong(v));
}

// Mask word w of the pool slot e of request b (pb = b * E).
__device__ __forceinline__ uint64_t& pool_anc(const TreeParams& p, size_t pb, int e, int w) {
  return p.p_anc[(pb + e) * p.WE + w];
}

__host__ __device__ inline int pow2_at_least(int n) {
  int v = 1;
  while (v < n) v <<= 1;
  return v;
}

// Dynamic shared memory of the kernel: the E * K drawn candidates of a
// request, their sort order (padded to a power of two) and the parent slot
// of every tree slot.
size_t tree_smem_bytes(int E, int K, int S) {
  const size_t n = static_cast<size_t>(E) * K;
  return n * (sizeof(double) + sizeof(uint64_t) + 3 * sizeof(int)) +
         static_cast<size_t>(pow2_at_least(static_cast<int>(n))) * sizeof(int) + static_cast<size_t>(S) * sizeof(int);
}

// Candidate a goes before candidate b in the final order: valid ones first
// by the selection order, then invalid and padding entries by index.
__device__ __forceinline__ bool cand_before(int a, int b, const uint64_t* key, const int* dep, int n) {
  const bool va = a < n && dep[a] >= 0, vb = b < n && dep[b] >= 0;
  if (va != vb) return va;
  if (!va) return a < b;
  return before(key[a], dep[a], a, key[b], dep[b], b);
}

// Block-wide bitonic sort of order[0, n2) (n2 a power of two) by cand_before.
__device__ void sort_candidates(int* order, int n2, const uint64_t* key, const int* dep, int n) {
  for (int k2 = 2; k2 <= n2; k2 <<= 1)
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += TREE_THREADS) {
        const int l = i ^ j;
        if (l > i) {
          const int a = order[i], b = order[l];
          const bool swap = (i & k2) == 0 ? cand_before(b, a, key, dep, n) : cand_before(a, b, key, dep, n);
          if (swap) {
            order[i] = b;
            order[l] = a;
          }
        }
      }
      __syncthreads();
    }
}

__global__ void __launch_bounds__(TREE_THREADS) tree_kernel(const TreeParams p) {
  const LaunchStamp ls(p.stamp);
  pdl_wait();      // predecessor outputs visible from here on
  ls.waited();
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem_tree[];
  const int n_pool = p.E * p.K;
  double* s_val = reinterpret_cast<double*>(smem_tree);
  uint64_t* s_key = reinterpret_cast<uint64_t*>(s_val + n_pool);
  int* s_dep = reinterpret_cast<int*>(s_key + n_pool);
  int* s_rank = s_dep + n_pool;
  int* s_slot = s_rank + n_pool;
  int* s_order = s_slot + n_pool;
  int* s_parent_slot = s_order + pow2_at_least(n_pool);
  __shared__ int s_count;

  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int E = p.E, K = p.K, S = p.S;
  const eagle_plan& pl = p.plan;
  const size_t pb = static_cast<size_t>(b) * E;

  if (p.phase == EAGLE_PHASE_ROOT) {
    for (int i = tid; i < E * K; i += TREE_THREADS) p.p_child_exp[pb * K + i] = -1;
    for (int e = tid; e < E; e += TREE_THREADS) {
      const bool root = e == 0;
      p.p_token[pb + e] = root ? p.t_next[b] : -1;
      p.p_parent[pb + e] = -1;
      p.p_rank[pb + e] = 0;
      p.p_depth[pb + e] = 0;
      p.p_value[pb + e] = root ? 1.0 : -1.0;
      for (int w = 0; w < p.WE; ++w) pool_anc(p, pb, e, w) = root && w == 0 ? 1ull : 0ull;
    }
    return;
  }

  if (p.phase == EAGLE_PHASE_FRONTIER) {
    const int l = p.layer;
    if (pl.kind == 1) {
      for (int i = tid; i < pl.n_nodes; i += TREE_THREADS) {
        if (pl.node_depth[i] != l || pl.node_exp[i] < 0) continue;
        const int par_e = pl.node_parent[i] < 0 ? 0 : pl.node_exp[pl.node_parent[i]];
        const int r = pl.node_rank[i];
        const int e_new = pl.node_exp[i];
        const int tok = p.ctok[(pb + par_e) * K + r];
        const bool ok = p.p_token[pb + par_e] >= 0 && tok >= 0;
        p.p_token[pb + e_new] = ok ? tok : -1;
        p.p_parent[pb + e_new] = par_e;
        p.p_rank[pb + e_new] = r;
        p.p_depth[pb + e_new] = l;
        p.p_value[pb + e_new] =
            ok ? p.p_value[pb + par_e] * static_cast<double>(p.cprob[(pb + par_e) * K + r]) : -1.0;
        for (int w = 0; w < p.WE; ++w)
          pool_anc(p, pb, e_new, w) =
              ok ? (pool_anc(p, pb, par_e, w) | (w == (e_new >> 6) ? 1ull << (e_new & 63) : 0ull)) : 0ull;
        if (ok) p.p_child_exp[(pb + par_e) * K + r] = e_new;
      }
      return;
    }
    const int e_prev = pl.layer_e0[l - 1], n_prev = pl.layer_rows[l - 1];
    const int e_new0 = pl.layer_e0[l], n_new = pl.layer_rows[l];
    const int k = pl.top_k;
    const int n_c = n_prev * k;
    if (tid == 0) s_count = 0;
    __syncthreads();
    for (int c = tid; c < n_c; c += TREE_THREADS) {
      const int e = e_prev + c / k, r = c % k;
      const int tok = p.ctok[(pb + e) * K + r];
      const bool valid = p.p_token[pb + e] >= 0 && tok >= 0;
      s_val[c] = valid ? p.p_value[pb + e] * static_cast<double>(p.cprob[(pb + e) * K + r]) : -1.0;
      s_key[c] = valid ? value_key(s_val[c]) : 0ull;
      s_dep[c] = valid ? 1 : 0;
      if (valid) atomicAdd(&s_count, 1);
    }
    __syncthreads();
    const int lane = tid & 31;
    for (int c = tid >> 5; c < n_c; c += TREE_WARPS) {
      if (!s_dep[c]) continue;                 // the same for the whole warp
      const uint64_t kc = s_key[c];
      int cnt = 0;
      for (int o = lane; o < n_c; o += 32)
        if (s_dep[o] && before(s_key[o], 0, o, kc, 0, c)) ++cnt;
      const int rank = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(cnt)));
      if (rank >= n_new) continue;
      const int e = e_prev + c / k, r = c % k;
      const int e_new = e_new0 + rank;
      if (lane == 0) {
        p.p_token[pb + e_new] = p.ctok[(pb + e) * K + r];
        p.p_parent[pb + e_new] = e;
        p.p_rank[pb + e_new] = r;
        p.p_depth[pb + e_new] = p.p_depth[pb + e] + 1;
        p.p_value[pb + e_new] = s_val[c];
        p.p_child_exp[(pb + e) * K + r] = e_new;
      }
      for (int w = lane; w < p.WE; w += 32)
        pool_anc(p, pb, e_new, w) = pool_anc(p, pb, e, w) | (w == (e_new >> 6) ? 1ull << (e_new & 63) : 0ull);
    }
    for (int i = tid; i < n_new; i += TREE_THREADS) {
      if (i < s_count) continue;
      const int e_new = e_new0 + i;
      p.p_token[pb + e_new] = -1;
      p.p_parent[pb + e_new] = -1;
      p.p_rank[pb + e_new] = 0;
      p.p_depth[pb + e_new] = l;
      p.p_value[pb + e_new] = -1.0;
      for (int w = 0; w < p.WE; ++w) pool_anc(p, pb, e_new, w) = 0ull;
    }
    return;
  }

  // ---------------- FINAL ----------------
  const size_t tb = static_cast<size_t>(b) * S;
  for (int i = tid; i < E * K; i += TREE_THREADS) p.t_child_slot[pb * K + i] = -1;
  int n_sel = 0;
  if (pl.kind == 1) {
    n_sel = pl.n_nodes;
    __syncthreads();
    for (int i = tid; i < pl.n_nodes; i += TREE_THREADS) {
      const int par_e = pl.node_parent[i] < 0 ? 0 : pl.node_exp[pl.node_parent[i]];
      const int r = pl.node_rank[i];
      const int s = i + 1;
      const int tok = p.ctok[(pb + par_e) * K + r];
      const bool ok = p.p_token[pb + par_e] >= 0 && tok >= 0;
      p.t_token[tb + s] = ok ? tok : -1;
      const int ps = pl.node_parent[i] < 0 ? 0 : pl.node_parent[i] + 1;
      p.t_parent[tb + s] = ps;
      s_parent_slot[s] = ps;
      p.t_depth[tb + s] = pl.node_depth[i];
      p.t_pos[tb + s] = p.pos0[b] + pl.node_depth[i];
      p.t_exp[tb + s] = pl.node_exp[i];
      p.t_child_slot[(pb + par_e) * K + r] = s;
    }
  } else {
    const int k = pl.top_k, m = pl.top_m;
    const int n_c = pl.n_expanded * k;
    if (tid == 0) s_count = 0;
    __syncthreads();
    for (int c = tid; c < n_c; c += TREE_THREADS) {
      const int e = c / k, r = c % k;
      const int tok = p.ctok[(pb + e) * K + r];
      const bool valid = p.p_token[pb + e] >= 0 && tok >= 0;
      s_val[c] = valid ? p.p_value[pb + e] * static_cast<double>(p.cprob[(pb + e) * K + r]) : -1.0;
      s_key[c] = valid ? value_key(s_val[c]) : 0ull;
      s_dep[c] = valid ? p.p_depth[pb + e] + 1 : -1;
      s_slot[c] = -1;
      if (valid) atomicAdd(&s_count, 1);
    }
    __syncthreads();
    // every candidate's rank (its position in the sorted order; the
    // s_count valid ones come first)
    const int n2 = pow2_at_least(n_c);
    for (int i = tid; i < n2; i += TREE_THREADS) s_order[i] = i;
    __syncthreads();
    sort_candidates(s_order, n2, s_key, s_dep, n_c);
    for (int i = tid; i < n_c; i += TREE_THREADS) {
      const int c = s_order[i];
      s_rank[c] = s_dep[c] >= 0 ? i : INT32_MAX;
    }
    n_sel = min(m, s_count);
    // slots of the kept ones, s_order[0, n_sel): by (depth, rank)
    for (int i = tid; i < n_sel; i += TREE_THREADS) {
      const int c = s_order[i], dc = s_dep[c];
      int pos = 0;
      for (int j = 0; j < n_sel; ++j) {
        const int dj = s_dep[s_order[j]];
        if (dj < dc || (dj == dc && j < i)) ++pos;
      }
      s_slot[c] = 1 + pos;
    }
    __syncthreads();
    for (int c = tid; c < n_c; c += TREE_THREADS) {
      const int s = s_slot[c];
      if (s < 0) continue;
      const int e = c / k, r = c % k;
      int ps = 0;
      if (e != 0) {
        const int pc = p.p_parent[pb + e] * k + p.p_rank[pb + e];
        ps = (pc >= 0 && pc < n_c) ? s_slot[pc] : -1;
        if (ps < 0) {
          set_status(p.status, EAGLE_ERR_INVALID_TREE);
          ps = 0;
        }
      }
      p.t_token[tb + s] = p.ctok[(pb + e) * K + r];
      p.t_parent[tb + s] = ps;
      s_parent_slot[s] = ps;
      p.t_depth[tb + s] = s_dep[c];
      p.t_pos[tb + s] = p.pos0[b] + s_dep[c];
      p.t_exp[tb + s] = p.p_child_exp[(pb + e) * K + r];
      p.t_child_slot[(pb + e) * K + r] = s;
    }
  }
  if (tid == 0) s_parent_slot[0] = -1;
  __syncthreads();
  const int size = 1 + n_sel;
  if (tid == 0) {
    p.t_size[b] = size;
    p.t_token[tb] = p.p_token[pb];
    p.t_parent[tb] = -1;
    p.t_depth[tb] = 0;
    p.t_pos[tb] = p.pos0[b];
    p.t_exp[tb] = 0;
  }
  // ancestor-or-self masks: slot s walks its parent chain (parents precede
  // their children, so the walk ends at the root within s steps)
  for (int s = tid; s < S; s += TREE_THREADS) {
    uint64_t m[MAX_WORDS];
#pragma unroll
    for (int w = 0; w < MAX_WORDS; ++w) m[w] = 0ull;
    if (s < size) {
      int u = s;
      for (int steps = 0; u >= 0 && steps <= s; ++steps) {
#pragma unroll
        for (int w = 0; w < MAX_WORDS; ++w)
          if (w == (u >> 6)) m[w] |= 1ull << (u & 63);
        const int pu = u == 0 ? -1 : s_parent_slot[u];
        if (u != 0 && !(pu >= 0 && pu < u)) {
          set_status(p.status, EAGLE_ERR_INVALID_TREE);
          break;
        }
        u = pu;
      }
    } else {
      p.t_token[tb + s] = -1;
      p.t_parent[tb + s] = -1;
      p.t_depth[tb + s] = 0;
      p.t_pos[tb + s] = 0;
      p.t_exp[tb + s] = -1;
    }
#pragma unroll
    for (int w = 0; w < MAX_WORDS; ++w)
      if (w < p.WS) p.t_anc[(tb + s) * p.WS + w] = m[w];
  }
}

}  // namespace

cudaError_t launch_tree(eagle_ctx* ctx, const eagle_plan* plan, int phase, int layer, int batch,
                        const eagle_requests* req, const eagle_children* ch, const eagle_pool* pool,
                        const eagle_tree* tree, int* status, cudaStream_t st) {
  TreeParams p{};
  p.plan = *plan;
  p.phase = phase;
  p.layer = layer;
  p.E = ctx->lim.max_expanded;
  p.K = ctx->lim.max_children;
  p.WE = EAGLE_MASK_WORDS(p.E);
  p.t_next = req ? req->t_next : nullptr;
  p.pos0 = req ? req->pos0 : nullptr;
  p.ctok = ch ? ch->token : nullptr;
  p.cprob = ch ? ch->prob : nullptr;
  p.p_token = pool->token;
  p.p_parent = pool->parent;
  p.p_rank = pool->rank;
  p.p_depth = pool->depth;
  p.p_value = pool->value;
  p.p_anc = pool->anc;
  p.p_child_exp = pool->child_exp;
  if (tree) {
    p.S = tree->stride;
    p.WS = EAGLE_MASK_WORDS(p.S);
    p.t_token = tree->token;
    p.t_parent = tree->parent;
    p.t_depth = tree->depth;
    p.t_pos = tree->pos;
    p.t_exp = tree->exp;
    p.t_anc = tree->anc;
    p.t_child_slot = tree->child_slot;
    p.t_size = tree->size;
  }
  p.status = status;
  p.stamp = stamp_slot(ctx, EAGLE_K_TREE);
  const size_t smem = tree_smem_bytes(p.E, p.K, tree ? p.S : 1);
  {
    // the attribute is set once per context, to what the largest limits need
    const size_t most = tree_smem_bytes(EAGLE_MAX_NODES, EAGLE_MAX_CHILDREN, EAGLE_MAX_NODES);
    const cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(tree_kernel), static_cast<int>(most));
    if (e != cudaSuccess) return e;
  }
  trace_before(ctx, EAGLE_K_TREE, st);
  const cudaError_t e = launch_pdl(tree_kernel, dim3(batch), dim3(TREE_THREADS), smem, st, p);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_TREE, st);
  return e;
}

}  // namespace eagle
