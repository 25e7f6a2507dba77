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

__global__ void prep_fc_kernel(const float* __restrict__ f_last, const float* __restrict__ f_hat,
                               const int32_t* __restrict__ token, const int32_t* __restrict__ parent,
                               const uint16_t* __restrict__ embed, int ld_embed, int d, int E, int rpr, int e0,
                               int NP, int kp, uint16_t* __restrict__ bfc) {
  const int j = blockIdx.x;
  const int b = j / rpr, e = e0 + j % rpr;
  const int tok = token[static_cast<size_t>(b) * E + e];
  const float* feat = nullptr;
  if (tok >= 0) {
    if (e == 0) feat = f_last + static_cast<size_t>(b) * d;
    else feat = f_hat + (static_cast<size_t>(b) * E + parent[static_cast<size_t>(b) * E + e]) * d;
  }
  uint16_t* hi = bfc + static_cast<size_t>(j) * kp;
  uint16_t* lo = bfc + static_cast<size_t>(NP + j) * kp;
  for (int c = threadIdx.x; c < 2 * d; c += blockDim.x) {
    float x = 0.f;
    if (tok >= 0) x = c < d ? feat[c] : bf16_to_f32(embed[static_cast<size_t>(tok) * ld_embed + (c - d)]);
    uint16_t h16, l16;
    split_bf16(x, h16, l16);
    hi[c] = h16;
    lo[c] = l16;
  }
}

constexpr int SEL_THREADS = 1024;
constexpr int SEL_PER_THREAD = 32;     // V <= 32768

// (value desc, id asc) total order: true if a ranks before b.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

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

__global__ void __launch_bounds__(SEL_THREADS) select_kernel(const SelParams p) {
  __shared__ float red_f[32];
  __shared__ int red_i[32];
  __shared__ uint64_t tprefix[SEL_THREADS];   // inclusive prefix of per-thread weight sums
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
  const int per = (p.V + SEL_THREADS - 1) / SEL_THREADS;
  const int v0 = tid * per, v1 = min(p.V, v0 + per);

  float zl[SEL_PER_THREAD];
  float lmax = -INFINITY;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < SEL_PER_THREAD; ++i) {
    const int v = v0 + i;
    const bool in = i < per && v < v1;
    zl[i] = in ? z[v] : -INFINITY;
    if (in && !isfinite(zl[i])) bad = true;
    lmax = fmaxf(lmax, zl[i]);
  }
  if (bad) set_status(p.status, EAGLE_ERR_NUMERIC);
  const float m = block_max(lmax, red_f);
  float lsum = 0.f;
  float el[SEL_PER_THREAD];
#pragma unroll
  for (int i = 0; i < SEL_PER_THREAD; ++i) {
    el[i] = (i < per && v0 + i < v1) ? expf((zl[i] - m) * inv_t) : 0.f;
    lsum += el[i];
  }
  const float S = block_sum(lsum, red_f);
  const float invS = 1.0f / S;
#pragma unroll
  for (int i = 0; i < SEL_PER_THREAD; ++i) {
    if (i < per && v0 + i < v1) {
      el[i] *= invS;
      q[v0 + i] = el[i];
    }
  }

  if (greedy) {
    // per-thread top-k of its slice, then k rounds of a block-wide argmax
    float tv[EAGLE_MAX_CHILDREN];
    int ti[EAGLE_MAX_CHILDREN];
    int cnt = 0;
    for (int i = 0; i < per && v0 + i < v1; ++i) {
      const float v = zl[i];
      const int id = v0 + i;
      if (cnt == p.k && !ranks_before(v, id, tv[cnt - 1], ti[cnt - 1])) continue;
      int pos = cnt < p.k ? cnt : p.k - 1;
      while (pos > 0 && ranks_before(v, id, tv[pos - 1], ti[pos - 1])) {
        tv[pos] = tv[pos - 1];
        ti[pos] = ti[pos - 1];
        --pos;
      }
      tv[pos] = v;
      ti[pos] = id;
      if (cnt < p.k) ++cnt;
    }
    int ptr = 0;
    const int lane = tid & 31, wid = tid >> 5;
    for (int r = 0; r < p.k; ++r) {
      float bv = ptr < cnt ? tv[ptr] : -INFINITY;
      int bi = ptr < cnt ? ti[ptr] : INT32_MAX;
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
      if (ptr < cnt && ti[ptr] == win) ++ptr;
      if (tid == 0) {
        const bool ok = win != INT32_MAX && win < p.V;
        ct[r] = ok ? win : -1;
        cp[r] = ok ? q[win] : 0.f;
      }
    }
    if (tid == 0)
      for (int r = p.k; r < p.K; ++r) { ct[r] = -1; cp[r] = 0.f; }
    return;
  }

  // sampling: exact integer weights, per-thread sums, block-wide inclusive scan
  uint64_t wsum = 0;
#pragma unroll
  for (int i = 0; i < SEL_PER_THREAD; ++i)
    if (i < per && v0 + i < v1) wsum += quantize_prob(el[i]);
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
      // adjusted inclusive prefix at the end of thread slice tt
      auto adj_prefix = [&](int tt) {
        uint64_t v = tprefix[tt];
        const int end = min(p.V, (tt + 1) * per);
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
      const int s0 = lo * per, s1 = min(p.V, s0 + per);
      for (int v = s0; v < s1; ++v) {
        bool taken = false;
        for (int x = 0; x < n_taken; ++x) taken |= s_taken[x] == v;
        if (taken) continue;
        run += quantize_prob(q[v]);
        if (run > t) { pick = v; break; }
      }
      if (pick < 0) {      // cannot happen with consistent prefix sums
        set_status(p.status, EAGLE_ERR_NUMERIC);
        ct[r] = -1; cp[r] = 0.f;
        continue;
      }
      const uint64_t wp = quantize_prob(q[pick]);
      s_taken[n_taken] = pick;
      s_wtaken[n_taken] = wp;
      ++n_taken;
      remaining -= wp;
      ct[r] = pick;
      cp[r] = q[pick];
    }
    for (int r = p.k; r < p.K; ++r) { ct[r] = -1; cp[r] = 0.f; }
  }
}

}  // namespace

cudaError_t launch_prep_fc(eagle_ctx* ctx, const DraftLaunch& L, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  trace_before(ctx, EAGLE_K_PREP, st);
  prep_fc_kernel<<<L.n, 256, 0, st>>>(L.req->f_last, L.out->f_hat, L.pool->token, L.pool->parent, L.w->embed,
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
  trace_before(ctx, EAGLE_K_SELECT, st);
  select_kernel<<<L.n, SEL_THREADS, 0, st>>>(p);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_SELECT, st);
  return cudaGetLastError();
}

}  // namespace eagle
