// Acceptance on the verified tree ([A] §6.2; [B] "Greedy 验证", "随机采样验证";
// [C] "为什么普通草稿模型不够理想").
//  target_softmax: per (request, tree slot): argmax of the target logits
//    (ties to the lower id) and, for sampling requests, p = softmax(z / T).
//  accept_walk: one CTA per request walks from the root.
//    greedy   -- descend while a retained child carries the target argmax;
//                the argmax at the last node is the correction/bonus token.
//    sampling -- recursive multi-candidate rejection sampling in exact
//                integers: weights P = floor(p * 2^40) of the current node's
//                target distribution; candidate i (the i-th drawn child, drawn
//                from q without the earlier ones, Q_i) is accepted iff
//                u32 * Q_i[x] * sum(P) < P[x] * sum(Q_i) * 2^32 (r < p/q);
//                on rejection P <- max(0, P sum(Q_i) - Q_i sum(P)) >> shift
//                (the residual norm(max(0, p - q)), rescaled below 2^40).
//                Accepted and retained -> descend; accepted but pruned ->
//                final token; no candidate left -> final = one draw from P.
#include "internal.h"
#include "common.cuh"

namespace eagle {
namespace {

constexpr int SM_THREADS = 1024;

__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(SM_THREADS)
    target_softmax_kernel(const float* __restrict__ logits, const float* __restrict__ temperature,
                          const int32_t* __restrict__ tree_size, int S, int V, float* __restrict__ probs,
                          int32_t* __restrict__ argmax, int* status, uint64_t* stamp) {
  const LaunchStamp lstamp(stamp);
  pdl_wait();      // predecessor outputs visible from here on
  lstamp.waited();
  pdl_trigger();
  __shared__ float red_f[32];
  __shared__ int red_i[32];
  const int s = blockIdx.x, b = blockIdx.y;
  if (s >= tree_size[b]) return;
  const size_t row = static_cast<size_t>(b) * S + s;
  const float* z = logits + row * V;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  float bv = -INFINITY;
  int bi = INT32_MAX;
  bool bad = false;
  for (int v = tid; v < V; v += SM_THREADS) {
    const float x = z[v];
    if (!isfinite(x)) bad = true;
    if (ranks_before(x, v, bv, bi)) { bv = x; bi = v; }
  }
  if (bad) set_status(status, EAGLE_ERR_NUMERIC);
  warp_argmax(bv, bi);
  if (lane == 0) { red_f[wid] = bv; red_i[wid] = bi; }
  __syncthreads();
  if (wid == 0) {
    const int nw = SM_THREADS / 32;
    bv = lane < nw ? red_f[lane] : -INFINITY;
    bi = lane < nw ? red_i[lane] : INT32_MAX;
    warp_argmax(bv, bi);
    if (lane == 0) { red_f[0] = bv; red_i[0] = bi; }
  }
  __syncthreads();
  const float m = red_f[0];
  if (tid == 0) argmax[row] = red_i[0] == INT32_MAX ? -1 : red_i[0];   // -1: no finite logit
  const float T = temperature[b];
  if (!(T > 0.f)) return;
  const float inv_t = 1.0f / T;
  __syncthreads();
  float ls = 0.f;
  for (int v = tid; v < V; v += SM_THREADS) ls += expf((z[v] - m) * inv_t);
  const float tot = block_sum(ls, red_f);
  const float inv = 1.0f / tot;
  float* pr = probs + row * V;
  for (int v = tid; v < V; v += SM_THREADS) pr[v] = expf((z[v] - m) * inv_t) * inv;
}

typedef unsigned __int128 u128;

__device__ __forceinline__ int bitlen128(u128 x) {
  const uint64_t hi = static_cast<uint64_t>(x >> 64), lo = static_cast<uint64_t>(x);
  if (hi) return 128 - __clzll(static_cast<long long>(hi));
  if (lo) return 64 - __clzll(static_cast<long long>(lo));
  return 0;
}

struct WalkParams {
  int K, k, E, S, V, path_cap;
  const int32_t* t_token;
  const int32_t* t_parent;
  const int32_t* t_exp;
  const int32_t* t_child_slot;
  const int32_t* t_size;
  const int32_t* ctok;
  const float* probs;      // [B][S][V]
  const int32_t* argmax;   // [B][S]
  const float* q;          // [B][E][V]
  const float* temperature;
  uint32_t seed, round_id;
  uint64_t* scratch;       // [B][V] current weights P
  int32_t* accept_len;
  int32_t* path;
  int32_t* final_token;
  int32_t* last_slot;
  int* status;
  uint64_t* stamp;
};

__global__ void __launch_bounds__(SM_THREADS) accept_walk_kernel(const WalkParams p) {
  const LaunchStamp ls(p.stamp);
  pdl_wait();      // predecessor outputs visible from here on
  ls.waited();
  pdl_trigger();
  __shared__ uint64_t red_u[32];
  __shared__ int red_i[32];
  __shared__ uint64_t tprefix[SM_THREADS];
  __shared__ int s_taken[EAGLE_MAX_CHILDREN];
  __shared__ uint64_t s_px;
  __shared__ int s_flag, s_u, s_final;
  const int b = blockIdx.x, tid = threadIdx.x;
  const size_t tb = static_cast<size_t>(b) * p.S;
  const float T = p.temperature[b];
  int32_t* path = p.path + static_cast<size_t>(b) * p.path_cap;

  if (!(T > 0.f)) {  // greedy walk, over the tree staged in shared memory
    __shared__ int s_par[EAGLE_MAX_NODES], s_tok[EAGLE_MAX_NODES], s_am[EAGLE_MAX_NODES];
    const int size = min(p.t_size[b], min(p.S, EAGLE_MAX_NODES));
    for (int c = tid; c < size; c += blockDim.x) {
      s_par[c] = p.t_parent[tb + c];
      s_tok[c] = p.t_token[tb + c];
      s_am[c] = p.argmax[tb + c];
    }
    __syncthreads();
    if (tid == 0) {
      int u = 0, a = 0;
      path[0] = 0;
      int g = s_am[0];
      while (true) {
        int nxt = -1;
        for (int c = 1; c < size; ++c)
          if (s_par[c] == u && s_tok[c] == g) { nxt = c; break; }
        if (nxt < 0 || a + 1 >= p.path_cap) break;
        u = nxt;
        path[++a] = u;
        g = s_am[u];
      }
      p.accept_len[b] = a;
      p.final_token[b] = g;
      p.last_slot[b] = u;
    }
    return;
  }

  const int per = (p.V + SM_THREADS - 1) / SM_THREADS;
  const int v0 = tid * per, v1 = min(p.V, v0 + per);
  uint64_t* P = p.scratch + static_cast<size_t>(b) * p.V;
  int u = 0, a = 0;
  if (tid == 0) path[0] = 0;
  int final_tok = -1;
  while (true) {
    // P = target weights of node u
    const float* pu = p.probs + (tb + u) * p.V;
    uint64_t ls = 0;
    for (int v = v0; v < v1; ++v) {
      const uint64_t w = quantize_prob(pu[v]);
      P[v] = w;
      ls += w;
    }
    uint64_t SP = block_sum_u64(ls, red_u);
    int e = p.t_exp[tb + u];
    if (e >= p.E) {                   // not an expanded slot of this layout
      if (tid == 0) set_status(p.status, EAGLE_ERR_INVALID_TREE);
      e = -1;
    }
    bool descended = false;
    if (e >= 0) {
      const float* qe = p.q + (static_cast<size_t>(b) * p.E + e) * p.V;
      uint64_t lq = 0;
      for (int v = v0; v < v1; ++v) lq += quantize_prob(qe[v]);
      const uint64_t SQ = block_sum_u64(lq, red_u);
      uint64_t taken_w = 0;
      int n_taken = 0;
      for (int i = 0; i < p.k; ++i) {
        const int x = p.ctok[(static_cast<size_t>(b) * p.E + e) * p.K + i];
        if (x < 0) break;
        if (x >= p.V) {                 // not a token: the node's candidates end here
          if (tid == 0) set_status(p.status, EAGLE_ERR_INVALID_ARG);
          break;
        }
        const uint64_t SQi = SQ - taken_w;
        __syncthreads();
        if (x >= v0 && x < v1) s_px = P[x];
        __syncthreads();
        if (tid == 0) {
          const uint64_t Qx = quantize_prob(qe[x]);
          const uint32_t r = round_uniform(p.seed, i, u, PURPOSE_ACCEPT, b, p.round_id);
          const u128 lhs = static_cast<u128>(r) * Qx * SP;
          const u128 rhs = (static_cast<u128>(s_px) * SQi) << 32;
          s_flag = lhs < rhs ? 1 : 0;
          if (s_flag) s_u = p.t_child_slot[(static_cast<size_t>(b) * p.E + e) * p.K + i];
        }
        __syncthreads();
        if (s_flag) {
          int slot = s_u;
          if (slot >= p.S) {            // outside the tree: treated as pruned
            if (tid == 0) set_status(p.status, EAGLE_ERR_INVALID_TREE);
            slot = -1;
          }
          if (slot >= 0 && a + 1 < p.path_cap) {
            u = slot;
            ++a;
            if (tid == 0) path[a] = u;
            descended = true;
          } else {
            // accepted but pruned: x is the final token (a full path cannot
            // occur: path_cap >= depth + 1 is checked on the host)
            if (slot >= 0) set_status(p.status, EAGLE_ERR_CAPACITY);
            final_tok = x;
          }
          break;
        }
        // rejection: residual max(0, P sum(Q_i) - Q_i sum(P)), rescaled below 2^40
        int lbits = 0;
        for (int v = v0; v < v1; ++v) {
          bool tk = false;
          for (int t = 0; t < n_taken; ++t) tk |= s_taken[t] == v;
          const uint64_t qv = tk ? 0ull : quantize_prob(qe[v]);
          const u128 A = static_cast<u128>(P[v]) * SQi, Bq = static_cast<u128>(qv) * SP;
          const u128 rr = A > Bq ? A - Bq : static_cast<u128>(0);
          lbits = max(lbits, bitlen128(rr));
        }
        const int bits = block_max_i(lbits, red_i);
        const int shift = bits > QBITS ? bits - QBITS : 0;
        uint64_t ls2 = 0;
        for (int v = v0; v < v1; ++v) {
          bool tk = false;
          for (int t = 0; t < n_taken; ++t) tk |= s_taken[t] == v;
          const uint64_t qv = tk ? 0ull : quantize_prob(qe[v]);
          const u128 A = static_cast<u128>(P[v]) * SQi, Bq = static_cast<u128>(qv) * SP;
          const u128 rr = A > Bq ? A - Bq : static_cast<u128>(0);
          const uint64_t w = static_cast<uint64_t>(rr >> shift);
          P[v] = w;
          ls2 += w;
        }
        SP = block_sum_u64(ls2, red_u);
        __syncthreads();
        if (tid == 0) s_taken[n_taken] = x;
        taken_w += quantize_prob(qe[x]);
        ++n_taken;
        __syncthreads();
      }
    }
    if (descended) continue;          // reload P for the accepted child
    if (final_tok < 0) {
      // one draw from P: thread slices, inclusive scan, search
      uint64_t ls3 = 0;
      for (int v = v0; v < v1; ++v) ls3 += P[v];
      __syncthreads();
      tprefix[tid] = ls3;
      __syncthreads();
      for (int off = 1; off < SM_THREADS; off <<= 1) {
        const uint64_t add = tid >= off ? tprefix[tid - off] : 0ull;
        __syncthreads();
        tprefix[tid] += add;
        __syncthreads();
      }
      if (tid == 0) {
        const uint64_t tot = tprefix[SM_THREADS - 1];
        int pick = -1;
        if (tot > 0) {
          const uint32_t r = round_uniform(p.seed, 0, u, PURPOSE_FINAL, b, p.round_id);
          const uint64_t t = scale_uniform(r, tot);
          int lo = 0, hi = SM_THREADS - 1;
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (tprefix[mid] > t) hi = mid; else lo = mid + 1;
          }
          uint64_t run = lo > 0 ? tprefix[lo - 1] : 0ull;
          const int s0 = lo * per, s1 = min(p.V, s0 + per);
          for (int v = s0; v < s1; ++v) {
            run += P[v];
            if (run > t) { pick = v; break; }
          }
        }
        if (pick < 0) set_status(p.status, EAGLE_ERR_NUMERIC);
        s_final = pick;
      }
      __syncthreads();
      final_tok = s_final;
    }
    break;
  }
  if (tid == 0) {
    p.accept_len[b] = a;
    p.final_token[b] = final_tok;
    p.last_slot[b] = u;
  }
}

}  // namespace

cudaError_t launch_target_softmax(eagle_ctx* ctx, int batch, const eagle_tree* tree, const float* logits,
                                  const float* temperature, float* probs, int32_t* argmax, void* ws,
                                  cudaStream_t st) {
  dim3 grid(tree->stride, batch);
  uint64_t* stamp = stamp_slot(ctx, EAGLE_K_ACCEPT);
  trace_before(ctx, EAGLE_K_ACCEPT, st);
  const cudaError_t e = launch_pdl(target_softmax_kernel, grid, dim3(SM_THREADS), 0, st, logits, temperature,
                                   tree->size, tree->stride, ctx->dims.vocab, probs, argmax,
                                   ws_ptr<int>(ws, ctx->ws.status), stamp);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_ACCEPT, st);
  return e;
}

cudaError_t launch_accept_walk(eagle_ctx* ctx, const eagle_plan* plan, int batch, const eagle_tree* tree,
                               const eagle_children* ch, const float* probs, const int32_t* argmax,
                               const float* q_probs, const eagle_sampling* s, const eagle_accept_out* out,
                               void* ws, cudaStream_t st) {
  WalkParams p{};
  p.K = ctx->lim.max_children;
  p.k = plan->top_k;
  p.E = ctx->lim.max_expanded;
  p.S = tree->stride;
  p.V = ctx->dims.vocab;
  p.path_cap = out->path_cap;
  p.t_token = tree->token;
  p.t_parent = tree->parent;
  p.t_exp = tree->exp;
  p.t_child_slot = tree->child_slot;
  p.t_size = tree->size;
  p.ctok = ch->token;
  p.probs = probs;
  p.argmax = argmax;
  p.q = q_probs;
  p.temperature = s->temperature;
  p.seed = s->seed;
  p.round_id = s->round_id;
  p.scratch = ws_ptr<uint64_t>(ws, ctx->ws.accept_scratch);
  p.accept_len = out->accept_len;
  p.path = out->path;
  p.final_token = out->final_token;
  p.last_slot = out->last_slot;
  p.status = ws_ptr<int>(ws, ctx->ws.status);
  p.stamp = stamp_slot(ctx, EAGLE_K_ACCEPT);
  trace_before(ctx, EAGLE_K_ACCEPT, st);
  const cudaError_t e = launch_pdl(accept_walk_kernel, dim3(batch), dim3(SM_THREADS), 0, st, p);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_ACCEPT, st);
  return e;
}

}  // namespace eagle
