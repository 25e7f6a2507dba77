// Acceptance on the verified tree ([A] §6.2; [B] "Greedy 验证", "随机采样验证";
// [C] "为什么普通草稿模型不够理想").
//  target_softmax: per (request, tree slot): argmax of the target logits
//    (ties to the lower id) and, for sampling requests, p = softmax(z / T).
//  accept_walk: one cluster per request walks from the root.
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
#include "sm100.cuh"

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
  int32_t* accept_len;
  int32_t* path;
  int32_t* final_token;
  int32_t* last_slot;
  int* status;
  uint64_t* stamp;
};

// The walk: one cluster of WALK_CL CTAs per request.  The sampling walk
// spreads the vocabulary over the cluster, WALK_PER consecutive entries per
// thread (the weights P of the current node and the taken-candidate marks
// stay in registers); sums and maxima are CTA reductions whose per-CTA
// values every CTA pushes to every other through distributed shared memory
// before a cluster barrier, so every CTA holds the same totals and takes the
// same decisions.  A candidate's weight P[x] is read from the CTA that owns
// x.  A value published by the n-th barrier sits in slot n % 2, rewritten
// only two barriers later, after every CTA has read it.  The greedy walk is
// rank 0's alone.
constexpr int WALK_CL = 8;
constexpr int WALK_THREADS = 512;
constexpr int WALK_PER = 8;
static_assert(WALK_CL * WALK_THREADS * WALK_PER >= EAGLE_MAX_VOCAB, "one cluster covers the largest vocabulary");

__global__ void __cluster_dims__(WALK_CL, 1, 1) __launch_bounds__(WALK_THREADS)
    accept_walk_kernel(const WalkParams p) {
  const LaunchStamp ls(p.stamp);
  pdl_wait();      // predecessor outputs visible from here on
  ls.waited();
  pdl_trigger();
  __shared__ uint64_t red_u[32];
  __shared__ int red_i[32];
  __shared__ uint64_t x_a[2][WALK_CL], x_b[2][WALK_CL];   // per-CTA values, by barrier parity
  __shared__ uint64_t x_px[2];                            // P at the next candidate (its owner CTA)
  __shared__ int x_pick[2];                               // the final draw (rank 0)
  const int b = blockIdx.x / WALK_CL;
  const uint32_t rank = sm100::cluster_rank();
  const int tid = threadIdx.x;
  const size_t tb = static_cast<size_t>(b) * p.S;
  const float T = p.temperature[b];
  int32_t* path = p.path + static_cast<size_t>(b) * p.path_cap;

  if (!(T > 0.f)) {  // greedy walk, over the tree staged in shared memory
    if (rank != 0) return;
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

  sm100::cluster_sync();                     // every CTA of the cluster has started
  int ph = 0;                                // cluster barriers passed since
  const bool lead = rank == 0 && tid == 0;
  const int V = p.V;
  const int v0 = (static_cast<int>(rank) * WALK_THREADS + tid) * WALK_PER;
  auto owner = [](int v) { return static_cast<uint32_t>(v / (WALK_THREADS * WALK_PER)); };
  // this CTA's value v (held by every thread) into slot ph % 2 of every CTA
  auto publish = [&](uint64_t (*xs)[WALK_CL], uint64_t v) {
    if (tid < WALK_CL) sm100::dsmem_st_u64(sm100::dsmem_addr(&xs[ph & 1][rank], tid), v);
  };
  auto barrier = [&]() {
    sm100::cluster_sync();
    ++ph;
  };
  auto total = [&](uint64_t (*xs)[WALK_CL]) {  // the published values' sum, in rank order
    uint64_t t = 0;
    for (int c = 0; c < WALK_CL; ++c) t += xs[(ph - 1) & 1][c];
    return t;
  };
  const int32_t* ctok_b = p.ctok + static_cast<size_t>(b) * p.E * p.K;

  int u = 0, a = 0, final_tok = -1;
  if (lead) path[0] = 0;
  uint64_t P[WALK_PER];
  while (true) {
    // P = target weights of node u; Q = draft weights of its expanded slot
    const float* pu = p.probs + (tb + u) * V;
    uint64_t lp = 0;
#pragma unroll
    for (int j = 0; j < WALK_PER; ++j) {
      P[j] = v0 + j < V ? quantize_prob(pu[v0 + j]) : 0ull;
      lp += P[j];
    }
    int e = p.t_exp[tb + u];
    if (e >= p.E) {                   // not an expanded slot of this layout
      if (lead) set_status(p.status, EAGLE_ERR_INVALID_TREE);
      e = -1;
    }
    const float* qe = e >= 0 ? p.q + (static_cast<size_t>(b) * p.E + e) * V : nullptr;
    uint64_t lq = 0;
    if (qe) {
#pragma unroll
      for (int j = 0; j < WALK_PER; ++j) lq += v0 + j < V ? quantize_prob(qe[v0 + j]) : 0ull;
    }
    const uint64_t cp = block_sum_u64(lp, red_u);
    const uint64_t cq = block_sum_u64(lq, red_u);
    publish(x_a, cp);
    publish(x_b, cq);
    if (e >= 0 && p.k > 0) {          // P at the first candidate, from its owner
      const int x0 = ctok_b[e * p.K];
      if (x0 >= v0 && x0 < v0 + WALK_PER && x0 < V) x_px[ph & 1] = P[x0 - v0];
    }
    barrier();
    uint64_t SP = total(x_a);
    const uint64_t SQ = total(x_b);
    bool descended = false;
    if (e >= 0) {
      uint64_t taken_w = 0;
      uint32_t tmask = 0;             // this thread's entries drawn as earlier candidates
      for (int i = 0; i < p.k; ++i) {
        const int x = ctok_b[e * p.K + i];
        if (x < 0) break;
        if (x >= V) {                 // not a token: the node's candidates end here
          if (lead) set_status(p.status, EAGLE_ERR_INVALID_ARG);
          break;
        }
        const uint64_t SQi = SQ - taken_w;
        const uint64_t px = sm100::dsmem_ld_u64(sm100::dsmem_addr(&x_px[(ph - 1) & 1], owner(x)));
        const uint64_t Qx = quantize_prob(qe[x]);
        const uint32_t r = round_uniform(p.seed, i, u, PURPOSE_ACCEPT, b, p.round_id);
        const u128 lhs = static_cast<u128>(r) * Qx * SP;
        const u128 rhs = (static_cast<u128>(px) * SQi) << 32;
        if (lhs < rhs) {
          int slot = p.t_child_slot[(static_cast<size_t>(b) * p.E + e) * p.K + i];
          if (slot >= p.S) {          // outside the tree: treated as pruned
            if (lead) set_status(p.status, EAGLE_ERR_INVALID_TREE);
            slot = -1;
          }
          if (slot >= 0 && a + 1 < p.path_cap) {
            u = slot;
            ++a;
            if (lead) path[a] = u;
            descended = true;
          } else {
            // accepted but pruned: x is the final token (a full path cannot
            // occur: path_cap >= depth + 1 is checked on the host)
            if (slot >= 0 && lead) set_status(p.status, EAGLE_ERR_CAPACITY);
            final_tok = x;
          }
          break;
        }
        // rejection: residual max(0, P sum(Q_i) - Q_i sum(P)), rescaled below 2^40
        int lbits = 0;
#pragma unroll
        for (int j = 0; j < WALK_PER; ++j) {
          if (v0 + j >= V) continue;
          const uint64_t qv = ((tmask >> j) & 1u) ? 0ull : quantize_prob(qe[v0 + j]);
          const u128 A = static_cast<u128>(P[j]) * SQi, Bq = static_cast<u128>(qv) * SP;
          lbits = max(lbits, bitlen128(A > Bq ? A - Bq : static_cast<u128>(0)));
        }
        publish(x_a, static_cast<uint64_t>(block_max_i(lbits, red_i)));
        barrier();
        int bits = 0;
        for (int c = 0; c < WALK_CL; ++c) bits = max(bits, static_cast<int>(x_a[(ph - 1) & 1][c]));
        const int shift = bits > QBITS ? bits - QBITS : 0;
        uint64_t l2 = 0;
#pragma unroll
        for (int j = 0; j < WALK_PER; ++j) {
          if (v0 + j >= V) continue;
          const uint64_t qv = ((tmask >> j) & 1u) ? 0ull : quantize_prob(qe[v0 + j]);
          const u128 A = static_cast<u128>(P[j]) * SQi, Bq = static_cast<u128>(qv) * SP;
          P[j] = static_cast<uint64_t>((A > Bq ? A - Bq : static_cast<u128>(0)) >> shift);
          l2 += P[j];
        }
        publish(x_b, block_sum_u64(l2, red_u));
        if (i + 1 < p.k) {            // the next candidate's new weight, from its owner
          const int xn = ctok_b[e * p.K + i + 1];
          if (xn >= v0 && xn < v0 + WALK_PER && xn < V) x_px[ph & 1] = P[xn - v0];
        }
        barrier();
        SP = total(x_b);
        if (x >= v0 && x < v0 + WALK_PER) tmask |= 1u << (x - v0);
        taken_w += Qx;
      }
    }
    if (descended) continue;          // reload P for the accepted child
    if (final_tok < 0) {
      // one draw from P: the entry whose inclusive prefix first exceeds
      // t = floor(u32 * sum / 2^32), scanning entries in vocabulary order
      uint64_t l3 = 0;
#pragma unroll
      for (int j = 0; j < WALK_PER; ++j) l3 += P[j];
      const int lane = tid & 31, wid = tid >> 5;
      uint64_t incl = l3;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      __syncthreads();
      if (lane == 31) red_u[wid] = incl;
      __syncthreads();
      uint64_t before = incl - l3, cta = 0;
      for (int w = 0; w < WALK_THREADS / 32; ++w) {
        if (w < wid) before += red_u[w];
        cta += red_u[w];
      }
      publish(x_a, cta);
      barrier();
      uint64_t tot = 0;
      for (int c = 0; c < WALK_CL; ++c) {
        const uint64_t tc = x_a[(ph - 1) & 1][c];
        if (c < static_cast<int>(rank)) before += tc;
        tot += tc;
      }
      if (tot > 0) {
        const uint32_t r = round_uniform(p.seed, 0, u, PURPOSE_FINAL, b, p.round_id);
        const uint64_t t = scale_uniform(r, tot);
        if (l3 > 0 && before <= t && t - before < l3) {
          uint64_t run = before;
          int pick = -1;
#pragma unroll
          for (int j = 0; j < WALK_PER; ++j) {
            run += P[j];
            if (pick < 0 && run > t) pick = v0 + j;
          }
          sm100::dsmem_st_s32(sm100::dsmem_addr(&x_pick[ph & 1], 0), pick);
        }
        barrier();
        final_tok = rank == 0 ? x_pick[(ph - 1) & 1] : 0;
        if (final_tok < 0 && lead) set_status(p.status, EAGLE_ERR_NUMERIC);
      } else {
        if (lead) set_status(p.status, EAGLE_ERR_NUMERIC);
        final_tok = -1;
      }
    }
    break;
  }
  if (lead) {
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
  p.accept_len = out->accept_len;
  p.path = out->path;
  p.final_token = out->final_token;
  p.last_slot = out->last_slot;
  p.status = ws_ptr<int>(ws, ctx->ws.status);
  p.stamp = stamp_slot(ctx, EAGLE_K_ACCEPT);
  trace_before(ctx, EAGLE_K_ACCEPT, st);
  const cudaError_t e = launch_pdl(accept_walk_kernel, dim3(batch * WALK_CL), dim3(WALK_THREADS), 0, st, p);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_ACCEPT, st);
  return e;
}

}  // namespace eagle
