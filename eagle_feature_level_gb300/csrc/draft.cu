// Draft-step kernels around the contractions:
//  * prep_fc: gathers each row's FC input x = [f ; E[t]] ([A] §4.1: the
//    feature of the parent position and the embedding of the shifted token)
//    into the FC's bf16 hi/lo operand;
//  * select: q = softmax(z / T) of each row's LM-head logits, then the row's
//    children -- greedy: the k largest logits, ties to the lower token id;
//    sampling: k draws without replacement from q on exact integer weights
//    floor(q * 2^40) with the round's Philox stream ([A] §6.1: t ~ q).
#include "internal.h"
#include "sm100.cuh"

namespace eagle {
namespace {

// One thread per 8 consecutive columns of x = [f ; E[t]] (d is a multiple of
// 64, so a group never straddles the two halves); grid (rows, column groups).
__global__ void prep_fc_kernel(const float* __restrict__ f_last, const float* __restrict__ f_hat,
                               const int32_t* __restrict__ token, const int32_t* __restrict__ parent,
                               const uint16_t* __restrict__ embed, int ld_embed, int d, int E, int rpr, int e0,
                               int NP, int kp, uint16_t* __restrict__ bfc) {
  const int j = blockIdx.x;
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (c0 >= 2 * d) return;
  const int b = j / rpr, e = e0 + j % rpr;
  const int tok = token[static_cast<size_t>(b) * E + e];
  float x[8];
  if (tok < 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = 0.f;
  } else if (c0 < d) {
    const float* feat = e == 0 ? f_last + static_cast<size_t>(b) * d
                               : f_hat + (static_cast<size_t>(b) * E + parent[static_cast<size_t>(b) * E + e]) * d;
    const float4 a = *reinterpret_cast<const float4*>(feat + c0);
    const float4 c = *reinterpret_cast<const float4*>(feat + c0 + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
  } else {
    const uint4 r = *reinterpret_cast<const uint4*>(embed + static_cast<size_t>(tok) * ld_embed + (c0 - d));
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  uint16_t h[8], l[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) split_bf16(x[i], h[i], l[i]);
  uint4 hv, lv;
  hv.x = h[0] | (uint32_t(h[1]) << 16); hv.y = h[2] | (uint32_t(h[3]) << 16);
  hv.z = h[4] | (uint32_t(h[5]) << 16); hv.w = h[6] | (uint32_t(h[7]) << 16);
  lv.x = l[0] | (uint32_t(l[1]) << 16); lv.y = l[2] | (uint32_t(l[3]) << 16);
  lv.z = l[4] | (uint32_t(l[5]) << 16); lv.w = l[6] | (uint32_t(l[7]) << 16);
  *reinterpret_cast<uint4*>(bfc + static_cast<size_t>(j) * kp + c0) = hv;
  *reinterpret_cast<uint4*>(bfc + static_cast<size_t>(NP + j) * kp + c0) = lv;
}

constexpr int SEL_THREADS = 512;

// (value desc, id asc) total order: true if a ranks before b.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Shared-memory slot of vocabulary entry v: one pad word per 32 entries, so
// both strided (v = tid + i * 1024) and per-thread contiguous chunks of 32
// entries hit 32 distinct banks.
__device__ __forceinline__ int pad32(int v) { return v + (v >> 5); }

struct SelParams {
  const float* logits;     // [B][E][V]
  float* probs;            // [B][E][V]
  int32_t* child_tok;      // [B][E][K]
  float* child_prob;
  const int32_t* token;    // pool.token [B][E]
  const float* temperature;
  int V, E, K, k, rpr, e0;
  uint32_t seed, round_id;
  int* status;
};

// One CTA per draft row.  Logits are read once (coalesced) into shared
// memory; max, exp, sum and q all work there; q is written back coalesced.
__global__ void __launch_bounds__(SEL_THREADS) select_kernel(const SelParams p) {
  extern __shared__ float qs[];                  // [pad32(V)]
  __shared__ float red_f[32];
  __shared__ int red_i[32];
  __shared__ uint64_t tprefix[SEL_THREADS];      // inclusive prefix of per-thread weight sums
  __shared__ int s_taken[EAGLE_MAX_CHILDREN];
  __shared__ uint64_t s_wtaken[EAGLE_MAX_CHILDREN];

  const int j = blockIdx.x;
  const int b = j / p.rpr, e = p.e0 + j % p.rpr;
  const size_t node = static_cast<size_t>(b) * p.E + e;
  const float* z = p.logits + node * p.V;
  float* q = p.probs + node * p.V;
  int32_t* ct = p.child_tok + node * p.K;
  float* cp = p.child_prob + node * p.K;
  const int tid = threadIdx.x;
  if (p.token[node] < 0) {
    if (tid < p.K) { ct[tid] = -1; cp[tid] = 0.f; }
    return;
  }
  const float T = p.temperature[b];
  const bool greedy = !(T > 0.f);
  const float inv_t = greedy ? 1.0f : 1.0f / T;
  const int V = p.V;

  // pass 1: stage logits, row max, per-thread top-k (greedy).  Loads are
  // issued in batches of 8 ahead of the insertion; the top-k list lives in
  // registers (fully unrolled bubble insertion, no dynamic indexing).
  float tv[EAGLE_MAX_CHILDREN];
  int ti[EAGLE_MAX_CHILDREN];
#pragma unroll
  for (int s = 0; s < EAGLE_MAX_CHILDREN; ++s) { tv[s] = -INFINITY; ti[s] = INT32_MAX; }
  float lmax = -INFINITY;
  bool bad = false;
  for (int base = tid; base < V; base += 8 * SEL_THREADS) {
    float xs[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = base + u * SEL_THREADS;
      xs[u] = v < V ? __ldg(z + v) : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int v = base + u * SEL_THREADS;
      if (v >= V) break;
      const float x = xs[u];
      qs[pad32(v)] = x;
      if (!isfinite(x)) bad = true;
      lmax = fmaxf(lmax, x);
      if (greedy && ranks_before(x, v, tv[EAGLE_MAX_CHILDREN - 1], ti[EAGLE_MAX_CHILDREN - 1])) {
        float cv = x;
        int ci = v;
#pragma unroll
        for (int s = 0; s < EAGLE_MAX_CHILDREN; ++s) {
          if (ranks_before(cv, ci, tv[s], ti[s])) {
            const float tf = tv[s]; tv[s] = cv; cv = tf;
            const int tn = ti[s]; ti[s] = ci; ci = tn;
          }
        }
      }
    }
  }
  if (bad) set_status(p.status, EAGLE_ERR_NUMERIC);
  const float m = block_max(lmax, red_f);
  // pass 2: exponentials and their sum (fixed-order reduction)
  float lsum = 0.f;
  for (int v = tid; v < V; v += SEL_THREADS) {
    const float ex = expf((qs[pad32(v)] - m) * inv_t);
    qs[pad32(v)] = ex;
    lsum += ex;
  }
  const float invS = 1.0f / block_sum(lsum, red_f);
  // pass 3: q, in shared memory and to the output row
  for (int v = tid; v < V; v += SEL_THREADS) {
    const float qv = qs[pad32(v)] * invS;
    qs[pad32(v)] = qv;
    q[v] = qv;
  }
  __syncthreads();

  if (greedy) {
    // k rounds of a block-wide argmax over each thread's next candidate
    int ptr = 0;
    const int lane = tid & 31, wid = tid >> 5;
    for (int r = 0; r < p.k; ++r) {
      float bv = -INFINITY;
      int bi = INT32_MAX;
#pragma unroll
      for (int s = 0; s < EAGLE_MAX_CHILDREN; ++s)
        if (s == ptr) { bv = tv[s]; bi = ti[s]; }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      __syncthreads();
      if (lane == 0) { red_f[wid] = bv; red_i[wid] = bi; }
      __syncthreads();
      if (wid == 0) {
        bv = red_f[lane];
        bi = red_i[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) red_i[0] = bi;
      }
      __syncthreads();
      const int win = red_i[0];
      if (bi != INT32_MAX && win == bi && ptr < EAGLE_MAX_CHILDREN) {
        // this thread's candidate won (ids are unique across threads)
        bool mine = false;
#pragma unroll
        for (int s = 0; s < EAGLE_MAX_CHILDREN; ++s)
          if (s == ptr) mine = ti[s] == win;
        if (mine) ++ptr;
      }
      if (tid == 0) {
        const bool ok = win != INT32_MAX && win < V;
        ct[r] = ok ? win : -1;
        cp[r] = ok ? qs[pad32(win)] : 0.f;
      }
    }
    if (tid == 0)
      for (int r = p.k; r < p.K; ++r) { ct[r] = -1; cp[r] = 0.f; }
    return;
  }

  // sampling: exact integer weights over contiguous per-thread chunks, a
  // block-wide inclusive scan of the chunk sums, then k sequential draws
  const int per = (V + SEL_THREADS - 1) / SEL_THREADS;
  const int v0 = tid * per, v1 = min(V, v0 + per);
  uint64_t wsum = 0;
  for (int v = v0; v < v1; ++v) wsum += quantize_prob(qs[pad32(v)]);
  tprefix[tid] = wsum;
  __syncthreads();
  for (int off = 1; off < SEL_THREADS; off <<= 1) {
    const uint64_t add = tid >= off ? tprefix[tid - off] : 0ull;
    __syncthreads();
    tprefix[tid] += add;
    __syncthreads();
  }
  if (tid == 0) {
    uint64_t remaining = tprefix[SEL_THREADS - 1];
    int n_taken = 0;
    for (int r = 0; r < p.k; ++r) {
      if (remaining == 0) { ct[r] = -1; cp[r] = 0.f; continue; }
      const uint32_t u = round_uniform(p.seed, r, e, PURPOSE_DRAW, b, p.round_id);
      const uint64_t t = scale_uniform(u, remaining);
      // inclusive prefix at the end of chunk tt, minus the weights already drawn
      auto adj_prefix = [&](int tt) {
        uint64_t v = tprefix[tt];
        const int end = min(V, (tt + 1) * per);
        for (int x = 0; x < n_taken; ++x)
          if (s_taken[x] < end) v -= s_wtaken[x];
        return v;
      };
      int lo = 0, hi = SEL_THREADS - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (adj_prefix(mid) > t) hi = mid; else lo = mid + 1;
      }
      uint64_t run = lo > 0 ? adj_prefix(lo - 1) : 0ull;
      int pick = -1;
      const int s0 = lo * per, s1 = min(V, s0 + per);
      for (int v = s0; v < s1; ++v) {
        bool taken = false;
        for (int x = 0; x < n_taken; ++x) taken |= s_taken[x] == v;
        if (taken) continue;
        run += quantize_prob(qs[pad32(v)]);
        if (run > t) { pick = v; break; }
      }
      if (pick < 0) {      // cannot happen with consistent prefix sums
        set_status(p.status, EAGLE_ERR_NUMERIC);
        ct[r] = -1; cp[r] = 0.f;
        continue;
      }
      const uint64_t wp = quantize_prob(qs[pad32(pick)]);
      s_taken[n_taken] = pick;
      s_wtaken[n_taken] = wp;
      ++n_taken;
      remaining -= wp;
      ct[r] = pick;
      cp[r] = qs[pad32(pick)];
    }
    for (int r = p.k; r < p.K; ++r) { ct[r] = -1; cp[r] = 0.f; }
  }
}

}  // namespace

cudaError_t launch_prep_fc(eagle_ctx* ctx, const DraftLaunch& L, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  trace_before(ctx, EAGLE_K_PREP, st);
  const dim3 grid(L.n, ceil_div(2 * D.d / 8, 128));
  prep_fc_kernel<<<grid, 128, 0, st>>>(L.req->f_last, L.out->f_hat, L.pool->token, L.pool->parent, L.w->embed,
                                     L.w->ld_embed, D.d, ctx->lim.max_expanded, L.rpr, L.e0, L.NP,
                                     ctx->ws.kp_fc, ws_ptr<uint16_t>(L.ws, ctx->ws.b_fc));
  ctx->launches++;
  trace_after(ctx, EAGLE_K_PREP, st);
  return cudaGetLastError();
}

cudaError_t launch_select(eagle_ctx* ctx, const DraftLaunch& L, cudaStream_t st) {
  SelParams p{};
  p.logits = L.out->logits;
  p.probs = L.out->probs;
  p.child_tok = L.children->token;
  p.child_prob = L.children->prob;
  p.token = L.pool->token;
  p.temperature = L.s->temperature;
  p.V = ctx->dims.vocab;
  p.E = ctx->lim.max_expanded;
  p.K = ctx->lim.max_children;
  p.k = L.k;
  p.rpr = L.rpr;
  p.e0 = L.e0;
  p.seed = L.s->seed;
  p.round_id = L.s->round_id;
  p.status = ws_ptr<int>(L.ws, ctx->ws.status);
  const size_t smem = static_cast<size_t>(p.V + (p.V >> 5) + 1) * sizeof(float);
  static size_t attr = 0;
  if (smem > attr) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr = smem;
  }
  trace_before(ctx, EAGLE_K_SELECT, st);
  select_kernel<<<L.n, SEL_THREADS, smem, st>>>(p);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_SELECT, st);
  return cudaGetLastError();
}

}  // namespace eagle
