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
                               int NP, int kp, uint16_t* __restrict__ bfc, uint64_t* stamp) {
  const LaunchStamp ls(stamp);
  // The FC contraction after this kernel may be scheduled now (its CTAs
  // start streaming weights); triggering before the wait in the kernels
  // ahead of this one would bring it in while the LM head still streams.
  pdl_trigger();
  pdl_wait();      // predecessor outputs visible from here on
  ls.waited();
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

// EAGLE-3 feature fusion input ([C] "EAGLE-3：放弃 feature prediction，改成多层
// 特征融合与 training-time test": g = FC([l; m; h])): row j of [l ; m ; h]
// (fp32 [n][3d]) into the fusion contraction's bf16 hi/lo operand.
__global__ void prep_fuse_kernel(const float* __restrict__ lmh, int d3, int NP, int kp, uint16_t* __restrict__ bop,
                                 uint64_t* stamp) {
  const LaunchStamp ls(stamp);
  pdl_trigger();
  pdl_wait();
  ls.waited();
  const int j = blockIdx.x;
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (c0 >= d3) return;
  const float* row = lmh + static_cast<size_t>(j) * d3 + c0;
  const float4 a = *reinterpret_cast<const float4*>(row);
  const float4 c = *reinterpret_cast<const float4*>(row + 4);
  const float x[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
  uint16_t h[8], l[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) split_bf16(x[u], h[u], l[u]);
  uint4 hv, lv;
  hv.x = h[0] | (uint32_t(h[1]) << 16); hv.y = h[2] | (uint32_t(h[3]) << 16);
  hv.z = h[4] | (uint32_t(h[5]) << 16); hv.w = h[6] | (uint32_t(h[7]) << 16);
  lv.x = l[0] | (uint32_t(l[1]) << 16); lv.y = l[2] | (uint32_t(l[3]) << 16);
  lv.z = l[4] | (uint32_t(l[5]) << 16); lv.w = l[6] | (uint32_t(l[7]) << 16);
  *reinterpret_cast<uint4*>(bop + static_cast<size_t>(j) * kp + c0) = hv;
  *reinterpret_cast<uint4*>(bop + static_cast<size_t>(NP + j) * kp + c0) = lv;
}

// Draft-cache refresh rows ([B] "KV Cache 必须按事务提交": the drafter
// continues from the committed path; [A] §6.2 closing remark): row
// j = b * R + i - 1 (i = 1 .. R) is x = [f_commit[b][i-1] ; E[tok_commit[b][i]]]
// -- the true feature of accepted position i - 1 and the token at position
// i -- when i <= accept_len[b], else zero.  Same operand layout as
// prep_fc_kernel.  The first thread of each request also writes its new
// cache length (len + a when the cache takes all a rows, else len, with
// EAGLE_ERR_CAPACITY).
__global__ void prep_refresh_kernel(const float* __restrict__ f_commit, const int32_t* __restrict__ tok_commit,
                                    const int32_t* __restrict__ n_act, const int32_t* __restrict__ kv_len, int kv_cap,
                                    int32_t* __restrict__ len_out, int path_cap, int R,
                                    const uint16_t* __restrict__ embed, int ld_embed, int d, int V, int NP, int kp,
                                    uint16_t* __restrict__ bfc, int* status, uint64_t* stamp) {
  const LaunchStamp ls(stamp);
  pdl_trigger();
  pdl_wait();      // the acceptance and commit outputs are visible from here on
  ls.waited();
  const int j = blockIdx.x;
  const int b = j / R, i = j % R + 1;
  const int a = min(max(n_act[b], 0), R);
  if (i == 1 && blockIdx.y == 0 && threadIdx.x == 0) {
    const int len = kv_len[b];
    const bool room = len >= 0 && len + a <= kv_cap;
    len_out[b] = room ? len + a : len;
    if (!room) set_status(status, EAGLE_ERR_CAPACITY);
  }
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * 8;
  if (c0 >= 2 * d) return;
  int tok = i <= a ? tok_commit[static_cast<size_t>(b) * (path_cap + 1) + i] : -1;
  if (tok >= V) {
    if (c0 == 0) set_status(status, EAGLE_ERR_INVALID_ARG);
    tok = -1;
  }
  float x[8];
  if (tok < 0) {
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = 0.f;
  } else if (c0 < d) {
    const float* feat = f_commit + (static_cast<size_t>(b) * path_cap + (i - 1)) * d;
    const float4 f0 = *reinterpret_cast<const float4*>(feat + c0);
    const float4 f1 = *reinterpret_cast<const float4*>(feat + c0 + 4);
    x[0] = f0.x; x[1] = f0.y; x[2] = f0.z; x[3] = f0.w; x[4] = f1.x; x[5] = f1.y; x[6] = f1.z; x[7] = f1.w;
  } else {
    const uint4 r = *reinterpret_cast<const uint4*>(embed + static_cast<size_t>(tok) * ld_embed + (c0 - d));
    const uint32_t wv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      x[2 * u] = __uint_as_float(wv[u] << 16);
      x[2 * u + 1] = __uint_as_float(wv[u] & 0xffff0000u);
    }
  }
  uint16_t h[8], l[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) split_bf16(x[u], h[u], l[u]);
  uint4 hv, lv;
  hv.x = h[0] | (uint32_t(h[1]) << 16); hv.y = h[2] | (uint32_t(h[3]) << 16);
  hv.z = h[4] | (uint32_t(h[5]) << 16); hv.w = h[6] | (uint32_t(h[7]) << 16);
  lv.x = l[0] | (uint32_t(l[1]) << 16); lv.y = l[2] | (uint32_t(l[3]) << 16);
  lv.z = l[4] | (uint32_t(l[5]) << 16); lv.w = l[6] | (uint32_t(l[7]) << 16);
  *reinterpret_cast<uint4*>(bfc + static_cast<size_t>(j) * kp + c0) = hv;
  *reinterpret_cast<uint4*>(bfc + static_cast<size_t>(NP + j) * kp + c0) = lv;
}

// select: a cluster of SEL_CL CTAs per row, each CTA one contiguous
// SEL_THREADS * SEL_PER slice of the vocabulary, SEL_PER consecutive logits
// per thread held in registers.  Row max, sum, top-k candidates and sampling
// draws are exchanged through distributed shared memory; every CTA reduces
// the exchanged partials in rank order, so all see the same max and sum.
constexpr int SEL_CL = 8;
constexpr int SEL_THREADS = 256;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_PER = 16;
constexpr int SEL_SLICE = SEL_THREADS * SEL_PER;
static_assert(SEL_CL * SEL_SLICE >= EAGLE_MAX_VOCAB, "one cluster covers the largest vocabulary");
static_assert(SEL_CL * EAGLE_MAX_CHILDREN <= 128 && SEL_WARPS * EAGLE_MAX_CHILDREN <= 128,
              "candidate lists fit four per lane");
static_assert(SEL_WARPS == SEL_CL, "rank 0 merges the lists of CTA w in its warp w");
// 32-bit words of the select kernel's shared buffer: the greedy lists or the
// sampling per-thread totals, whichever is larger
constexpr int SEL_GREEDY_WORDS = (2 * SEL_CL * SEL_WARPS + 3 * SEL_CL + 3 * SEL_WARPS) * EAGLE_MAX_CHILDREN;
constexpr int SEL_SAMPLE_WORDS = 2 * SEL_CL * SEL_THREADS;
constexpr int SEL_UNION_WORDS = SEL_GREEDY_WORDS > SEL_SAMPLE_WORDS ? SEL_GREEDY_WORDS : SEL_SAMPLE_WORDS;

// (value desc, id asc) total order: true if a ranks before b.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// One warp: the k best of n <= 128 candidates (z, id, q), in order, to out.
// Lane l holds candidates l, l + 32, l + 64, l + 96.
__device__ __forceinline__ void warp_merge_topk(const float* cz, const int* ci, const float* cq, int n, int k,
                                                float* oz, int* oi, float* oq) {
  const int lane = threadIdx.x & 31;
  float z[4];
  int id[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = lane + 32 * u;
    z[u] = c < n ? cz[c] : -INFINITY;
    id[u] = c < n ? ci[c] : INT32_MAX;
  }
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = INT32_MAX, bs = -1;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (ranks_before(z[u], id[u], bv, bi)) { bv = z[u]; bi = id[u]; bs = u; }
    float wv = bv;
    int wi = bi;
    warp_argmax(wv, wi);
    if (bs >= 0 && wi == bi && bi != INT32_MAX) {   // this lane holds the winner
      const int c = lane + 32 * bs;
      if (oz) oz[r] = z[bs];
      oi[r] = bi;
      oq[r] = cq[c];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (u == bs) { z[u] = -INFINITY; id[u] = INT32_MAX; }
    }
    if (wi == INT32_MAX && lane == 0) {               // fewer than k candidates
      if (oz) oz[r] = -INFINITY;
      oi[r] = INT32_MAX;
      oq[r] = 0.f;
    }
  }
  __syncwarp();
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
  uint64_t* stamp;
};

__global__ void __cluster_dims__(SEL_CL, 1, 1) __launch_bounds__(SEL_THREADS) select_kernel(const SelParams p) {
  const LaunchStamp ls(p.stamp);
  // Phase 0 of the cluster barrier: every CTA arrives as it starts and waits
  // just before its first access to another CTA's shared memory, which is
  // then known to have started.
  sm100::cluster_arrive_relaxed();
  pdl_wait();      // predecessor outputs visible from here on
  ls.waited();
  pdl_trigger();
  __shared__ float s_red[SEL_WARPS];
  __shared__ float s_cmax[SEL_CL], s_csum[SEL_CL];         // per-rank partials (pushed)
  __shared__ uint64_t s_ctot[SEL_CL];
  __shared__ uint64_t s_wt[SEL_WARPS];                       // sampling: integer weight totals per warp
  // sampling, rank 0: every CTA's per-warp weight totals (pushed), and the
  // draws so far (token, weight)
  __shared__ uint64_t s_gwt[SEL_CL * SEL_WARPS];
  __shared__ int s_dtok[EAGLE_MAX_CHILDREN];
  __shared__ uint64_t s_dw[EAGLE_MAX_CHILDREN];
  // One buffer serves either path (a cluster's row is greedy or sampled in
  // every CTA), which keeps the kernel's shared memory small enough for its
  // CTAs to be resident beside the LM-head contraction they follow, so that
  // they start before it ends.  Greedy, rank 0: every warp's list of every
  // CTA (pushed), each CTA's merged list, the final list.  Sampling, rank 0:
  // every CTA's per-thread weight totals (pushed).
  __shared__ __align__(16) uint32_t s_un[SEL_UNION_WORDS];
  float* s_gz = reinterpret_cast<float*>(s_un);
  int* s_gi = reinterpret_cast<int*>(s_gz + SEL_CL * SEL_WARPS * EAGLE_MAX_CHILDREN);
  float* s_cz = reinterpret_cast<float*>(s_gi + SEL_CL * SEL_WARPS * EAGLE_MAX_CHILDREN);
  float* s_cq = s_cz + SEL_CL * EAGLE_MAX_CHILDREN;
  int* s_ci = reinterpret_cast<int*>(s_cq + SEL_CL * EAGLE_MAX_CHILDREN);
  float* s_wz = reinterpret_cast<float*>(s_ci + SEL_CL * EAGLE_MAX_CHILDREN);
  float* s_wq = s_wz + SEL_WARPS * EAGLE_MAX_CHILDREN;
  int* s_wi = reinterpret_cast<int*>(s_wq + SEL_WARPS * EAGLE_MAX_CHILDREN);
  uint64_t* s_gtt = reinterpret_cast<uint64_t*>(s_un);

  const int row = blockIdx.x / SEL_CL;
  const uint32_t rank = sm100::cluster_rank();
  const int b = row / p.rpr, e = p.e0 + row % p.rpr;
  const size_t node = static_cast<size_t>(b) * p.E + e;
  int32_t* ct = p.child_tok + node * p.K;
  float* cp = p.child_prob + node * p.K;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (p.token[node] < 0) {                   // uniform over the cluster: no barrier is waited on
    if (rank == 0 && tid < p.K) { ct[tid] = -1; cp[tid] = 0.f; }
    return;
  }
  const float T = p.temperature[b];
  const bool greedy = !(T > 0.f);
  const float inv_t = greedy ? 1.0f : 1.0f / T;
  const int V = p.V, k = p.k;
  const int v0 = static_cast<int>(rank) * SEL_SLICE + tid * SEL_PER;
  const float* zrow = p.logits + node * V;
  float* qrow = p.probs + node * V;
  const bool vec = (V & 3) == 0 && v0 + SEL_PER <= V;

  // logits, finiteness, slice max
  float x[SEL_PER];
  if (vec) {
#pragma unroll
    for (int u = 0; u < SEL_PER / 4; ++u) {
      const float4 f = __ldg(reinterpret_cast<const float4*>(zrow + v0) + u);
      x[4 * u] = f.x; x[4 * u + 1] = f.y; x[4 * u + 2] = f.z; x[4 * u + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < SEL_PER; ++u) x[u] = v0 + u < V ? __ldg(zrow + v0 + u) : -INFINITY;
  }
  float lmax = -INFINITY;
  bool bad = false;
#pragma unroll
  for (int u = 0; u < SEL_PER; ++u) {
    if (v0 + u < V) {
      bad |= !isfinite(x[u]);
      lmax = fmaxf(lmax, x[u]);
    }
  }
  if (bad) set_status(p.status, EAGLE_ERR_NUMERIC);
  lmax = warp_max_redux(lmax);
  if (lane == 0) s_red[wid] = lmax;
  __syncthreads();
  sm100::cluster_wait();                     // phase 0: every CTA of the cluster has started
  if (tid < SEL_CL) {                        // push this CTA's max to every rank
    float m = s_red[0];
    for (int w = 1; w < SEL_WARPS; ++w) m = fmaxf(m, s_red[w]);
    sm100::dsmem_st_f32(sm100::dsmem_addr(&s_cmax[rank], tid), m);
  }
  sm100::cluster_arrive();                   // phase 1: the maxima
  if (greedy) {
    // each warp's k best (logit desc, id asc) go straight into rank 0's
    // table while the maxima travel (no softmax statistic is needed to rank
    // them; the probabilities come later)
    uint32_t taken = 0;
    float bv = -INFINITY;
    int bi = INT32_MAX, bs = -1;
#pragma unroll
    for (int u = 0; u < SEL_PER; ++u)
      if (v0 + u < V && ranks_before(x[u], v0 + u, bv, bi)) { bv = x[u]; bi = v0 + u; bs = u; }
    const int gbase = (static_cast<int>(rank) * SEL_WARPS + wid) * k;
    for (int r = 0; r < k; ++r) {
      float wv = bv;
      int wi = bi;
      warp_argmax(wv, wi);
      if (bs >= 0 && wi == bi && bi != INT32_MAX) {
        sm100::dsmem_st_f32(sm100::dsmem_addr(&s_gz[gbase + r], 0), bv);
        sm100::dsmem_st_s32(sm100::dsmem_addr(&s_gi[gbase + r], 0), bi);
        taken |= 1u << bs;
        bv = -INFINITY; bi = INT32_MAX; bs = -1;
#pragma unroll
        for (int u = 0; u < SEL_PER; ++u)
          if (!((taken >> u) & 1u) && v0 + u < V && ranks_before(x[u], v0 + u, bv, bi)) {
            bv = x[u]; bi = v0 + u; bs = u;
          }
      }
      if (wi == INT32_MAX && lane == 0) {
        sm100::dsmem_st_f32(sm100::dsmem_addr(&s_gz[gbase + r], 0), -INFINITY);
        sm100::dsmem_st_s32(sm100::dsmem_addr(&s_gi[gbase + r], 0), INT32_MAX);
      }
    }
  }
  sm100::cluster_wait();
  float m = s_cmax[0];
  for (int c = 1; c < SEL_CL; ++c) m = fmaxf(m, s_cmax[c]);

  // exponentials, slice sum in a fixed order, cluster sum in rank order
  float ex[SEL_PER];
  float lsum = 0.f;
#pragma unroll
  for (int u = 0; u < SEL_PER; ++u) {
    ex[u] = v0 + u < V ? expf((x[u] - m) * inv_t) : 0.f;
    lsum += ex[u];
  }
  lsum = warp_sum(lsum);
  __syncthreads();                           // s_red reuse
  if (lane == 0) s_red[wid] = lsum;
  __syncthreads();
  if (tid < SEL_CL) {
    float sum = 0.f;
    for (int w = 0; w < SEL_WARPS; ++w) sum += s_red[w];
    sm100::dsmem_st_f32(sm100::dsmem_addr(&s_csum[rank], tid), sum);
  }
  sm100::cluster_sync();
  float S = 0.f;
  for (int c = 0; c < SEL_CL; ++c) S += s_csum[c];
  const float invS = 1.0f / S;
  float q[SEL_PER];
#pragma unroll
  for (int u = 0; u < SEL_PER; ++u) q[u] = ex[u] * invS;
  if (vec) {
#pragma unroll
    for (int u = 0; u < SEL_PER / 4; ++u)
      reinterpret_cast<float4*>(qrow + v0)[u] = make_float4(q[4 * u], q[4 * u + 1], q[4 * u + 2], q[4 * u + 3]);
  } else {
#pragma unroll
    for (int u = 0; u < SEL_PER; ++u)
      if (v0 + u < V) qrow[v0 + u] = q[u];
  }

  if (greedy) {
    // rank 0 merges the cluster's lists (complete since the second barrier):
    // warp w the lists of CTA w, then warp 0 the CTAs' lists; a child's
    // probability is its q entry, recomputed by the same expression
    if (rank != 0) return;
    warp_merge_topk(s_gz + wid * SEL_WARPS * k, s_gi + wid * SEL_WARPS * k, s_gz + wid * SEL_WARPS * k,
                    SEL_WARPS * k, k, s_cz + wid * k, s_ci + wid * k, s_cq + wid * k);
    __syncthreads();
    if (wid != 0) return;
    warp_merge_topk(s_cz, s_ci, s_cq, SEL_CL * k, k, s_wz, s_wi, s_wq);
    if (lane < p.K) {
      const bool ok = lane < k && s_wi[lane] != INT32_MAX && s_wi[lane] < V;
      ct[lane] = ok ? s_wi[lane] : -1;
      cp[lane] = ok ? expf((s_wz[lane] - m) * inv_t) * invS : 0.f;
    }
    return;
  }

  // sampling: exact integer weights floor(q 2^40).  Every CTA pushes its
  // per-thread and per-warp weight totals into rank 0's shared memory; one
  // warp of rank 0 then makes the k draws without replacement, each by
  // descending from the CTAs' totals to a warp's and a thread's (local
  // reads) and to that thread's entries (their weights again from q, which
  // every CTA wrote before the barrier), the weights already drawn taken out
  // at every level: the token is the first one, in vocabulary order, at
  // which the running sum of the remaining weights exceeds
  // t = floor(u32 * remaining / 2^32).  After the barrier no CTA touches
  // another's shared memory, so the CTAs other than rank 0 leave at once
  // (with many rows, later clusters take their SMs: 13B batch 8, 270 ->
  // 199 us of selection per round).
  uint64_t wsum = 0;
#pragma unroll
  for (int u = 0; u < SEL_PER; ++u) wsum += v0 + u < V ? quantize_prob(q[u]) : 0ull;
  sm100::dsmem_st_u64(sm100::dsmem_addr(&s_gtt[rank * SEL_THREADS + tid], 0), wsum);
  const uint64_t wtot = warp_sum_u64(wsum);
  if (lane == 0) {
    s_wt[wid] = wtot;
    sm100::dsmem_st_u64(sm100::dsmem_addr(&s_gwt[rank * SEL_WARPS + wid], 0), wtot);
  }
  __syncthreads();
  if (tid < SEL_CL) {                        // this CTA's total, to every rank
    uint64_t cta_total = 0;
    for (int w = 0; w < SEL_WARPS; ++w) cta_total += s_wt[w];
    sm100::dsmem_st_u64(sm100::dsmem_addr(&s_ctot[rank], tid), cta_total);
  }
  sm100::cluster_sync();                     // every CTA's weights and totals are in place
  if (rank == 0 && wid == 0) {
    uint64_t total = 0;
    for (int c = 0; c < SEL_CL; ++c) total += s_ctot[c];
    int pk_tok = -1;                         // lane r: the r-th drawn token, its weight and q
    float pk_q = 0.f;
    uint64_t picked = 0;
    int n_drawn = 0;
    bool lost = false;
    // the first lane whose inclusive running sum of adj exceeds t (-1: none);
    // t becomes the offset inside that lane's range
    auto descend = [&](uint64_t adj, uint64_t& t) {
      uint64_t incl = adj;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const unsigned m = __ballot_sync(0xffffffffu, incl > t);
      if (m == 0u) return -1;
      const int f = __ffs(m) - 1;
      t -= __shfl_sync(0xffffffffu, incl - adj, f);
      return f;
    };
    // adj minus the weights of the earlier draws that fall in [lo_v, hi_v)
    // (each lane reads the draws from shared memory: no chain of shuffles)
    auto minus_drawn = [&](uint64_t adj, int lo_v, int hi_v, int r) {
      for (int s2 = 0; s2 < r; ++s2) {
        const int tk = s_dtok[s2];
        if (tk >= lo_v && tk < hi_v) adj -= s_dw[s2];
      }
      return adj;
    };
    for (int r = 0; r < k; ++r) {
      const uint64_t remaining = total - picked;
      if (remaining == 0) break;             // the distribution ran out of mass
      const uint32_t u32 = round_uniform(p.seed, r, e, PURPOSE_DRAW, b, p.round_id);
      uint64_t t = scale_uniform(u32, remaining);
      // CTA, warp, thread, entry
      uint64_t adj = lane < SEL_CL ? s_ctot[lane] : 0ull;
      adj = minus_drawn(adj, lane * SEL_SLICE, (lane + 1) * SEL_SLICE, r);
      const int c = descend(lane < SEL_CL ? adj : 0ull, t);
      if (c < 0) { lost = true; break; }
      const int cb = c * SEL_SLICE;
      adj = lane < SEL_WARPS ? s_gwt[c * SEL_WARPS + lane] : 0ull;
      adj = minus_drawn(adj, cb + lane * 32 * SEL_PER, cb + (lane + 1) * 32 * SEL_PER, r);
      const int w = descend(lane < SEL_WARPS ? adj : 0ull, t);
      if (w < 0) { lost = true; break; }
      const int th = w * 32 + lane;
      adj = s_gtt[c * SEL_THREADS + th];
      adj = minus_drawn(adj, cb + th * SEL_PER, cb + (th + 1) * SEL_PER, r);
      const int j = descend(adj, t);
      if (j < 0) { lost = true; break; }
      const int tb = cb + (w * 32 + j) * SEL_PER;
      const uint64_t wraw = lane < SEL_PER && tb + lane < V ? quantize_prob(qrow[tb + lane]) : 0ull;
      adj = minus_drawn(wraw, tb + lane, tb + lane + 1, r);
      const int u = descend(lane < SEL_PER ? adj : 0ull, t);
      if (u < 0) { lost = true; break; }
      const int tok = tb + u;
      const uint64_t wt = __shfl_sync(0xffffffffu, wraw, u);
      if (lane == r) {
        pk_tok = tok;
        pk_q = qrow[tok];                    // written by its CTA before the barrier
        s_dtok[r] = tok;
        s_dw[r] = wt;
      }
      __syncwarp();                          // the next draw's lanes read this one
      picked += wt;
      ++n_drawn;
    }
    if (lane < p.K) {
      const bool ok = lane < k && lane < n_drawn;
      ct[lane] = ok ? pk_tok : -1;
      cp[lane] = ok ? pk_q : 0.f;
    }
    if (lost && lane == 0) set_status(p.status, EAGLE_ERR_NUMERIC);
  }
}

}  // namespace

cudaError_t launch_prep_fc(eagle_ctx* ctx, const DraftLaunch& L, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  trace_before(ctx, EAGLE_K_PREP, st);
  const dim3 grid(L.n, ceil_div(2 * D.d / 8, 128));
  uint64_t* stamp = stamp_slot(ctx, EAGLE_K_PREP);
  const cudaError_t e =
      launch_pdl(prep_fc_kernel, grid, dim3(128), 0, st, L.req->f_last, L.out->f_hat, L.pool->token, L.pool->parent,
                 L.w->embed, L.w->ld_embed, D.d, ctx->lim.max_expanded, L.rpr, L.e0, L.NP, ctx->ws.kp_fc,
                 ws_ptr<uint16_t>(L.ws, ctx->ws.b_fc), stamp);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_PREP, st);
  return e;
}

cudaError_t launch_prep_fuse(eagle_ctx* ctx, const DraftLaunch& L, const float* lmh, cudaStream_t st) {
  const int d3 = 3 * ctx->dims.d;
  const dim3 grid(L.n, ceil_div(d3 / 8, 128));
  uint64_t* stamp = stamp_slot(ctx, EAGLE_K_FUSE);
  trace_before(ctx, EAGLE_K_FUSE, st);
  const cudaError_t e = launch_pdl(prep_fuse_kernel, grid, dim3(128), 0, st, lmh, d3, L.NP, ctx->ws.kp_fuse,
                                   ws_ptr<uint16_t>(L.ws, ctx->ws.b_fuse), stamp);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_FUSE, st);
  return e;
}

cudaError_t launch_prep_refresh(eagle_ctx* ctx, const DraftLaunch& L, const float* f_commit,
                                const int32_t* tok_commit, int path_cap, int32_t* len_out, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  const dim3 grid(L.n, ceil_div(2 * D.d / 8, 128));
  uint64_t* stamp = stamp_slot(ctx, EAGLE_K_REFRESH);
  trace_before(ctx, EAGLE_K_REFRESH, st);
  const cudaError_t e =
      launch_pdl(prep_refresh_kernel, grid, dim3(128), 0, st, f_commit, tok_commit, L.refresh_n, L.refresh_kv->len,
                 L.refresh_kv->cap, len_out, path_cap, L.rpr, L.w->embed, L.w->ld_embed, D.d, D.vocab, L.NP,
                 ctx->ws.kp_fc, ws_ptr<uint16_t>(L.ws, ctx->ws.b_fc), ws_ptr<int>(L.ws, ctx->ws.status), stamp);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_REFRESH, st);
  return e;
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
  p.stamp = stamp_slot(ctx, EAGLE_K_SELECT);
  trace_before(ctx, EAGLE_K_SELECT, st);
  const cudaError_t e = launch_pdl(select_kernel, dim3(L.n * SEL_CL), dim3(SEL_THREADS), 0, st, p);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_SELECT, st);
  return e;
}

}  // namespace eagle
