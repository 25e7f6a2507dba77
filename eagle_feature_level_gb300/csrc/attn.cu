// Tree-masked attention, shared by the draft layer and the target's
// verification layer ([B] "Tree Attention 如何一次验证多条路径": node u sees the
// committed prefix plus the tree nodes that are its ancestors or itself).
//
// Split-KV layout: one CTA per (prefix split or tree part, request, kv head).
// Every query row of the request that maps to this kv head (tree nodes x GQA
// group) consumes the same shared-memory K/V tile, so prefix KV bytes are
// read from HBM once per call however many tree nodes there are.  Each CTA
// writes (max, sum, unnormalised output) partials; the last CTA of a
// (request, kv head) merges them in split order.  The ancestor mask of each
// query row lives in a register (one 64-bit word) and is tested per tree key.
#include "internal.h"
#include "sm100.cuh"

namespace eagle {
namespace {

constexpr int TILE = 64;          // KV rows per shared-memory tile
constexpr int THREADS = 256;
constexpr int MAX_DH = 128;

struct AttnParams {
  int mode;                       // 0 draft, 1 verify
  int B, Hq, Hkv, dh, G;
  int n_splits, chunk;            // prefix splits and rows per split
  int rows_cap;                   // query nodes per request (draft: rows per request; verify: tree stride)
  const float* q_f32;             // draft: [n][Hq*dh] fp32
  const uint16_t* q_bf16;         // verify: [B][S][Hq][dh] bf16
  const uint16_t* kp;             // prefix KV [B][cap][Hkv][dh] bf16
  const uint16_t* vp;
  int kv_cap;
  const int32_t* kv_len;
  const float* kt_f32;            // draft: tree K/V [B][E][Hkv][dh] fp32
  const float* vt_f32;
  const uint16_t* kt_bf16;        // verify: tree K/V [B][S][Hkv][dh] bf16
  const uint16_t* vt_bf16;
  int tree_cap;                   // E or S
  const uint64_t* anc;            // draft: pool.anc [B][E]; verify: tree.anc [B][S]
  const int32_t* tree_size;       // verify: [B]
  int e0;                         // draft: first expanded slot of this layer
  float scale;
  float* out_f32;                 // verify: [B][S][Hq][dh]
  uint16_t* b_o;                  // draft: next GEMM operand (hi/lo), [2NP][bo_ld]
  int NP, bo_ld;
  float* part;
  int* counters;
};

__device__ __forceinline__ int n_nodes(const AttnParams& p, int b) {
  return p.mode == 0 ? p.rows_cap : min(p.tree_size[b], p.rows_cap);
}

__device__ __forceinline__ size_t q_index(const AttnParams& p, int b, int node, int hq) {
  return ((static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq) * p.dh;
}

__device__ __forceinline__ uint64_t row_mask(const AttnParams& p, int b, int node) {
  if (p.mode == 0) return p.anc[static_cast<size_t>(b) * p.tree_cap + p.e0 + node];
  return p.anc[static_cast<size_t>(b) * p.tree_cap + node];
}

// fp32 K/V tiles in dynamic shared memory: [TILE][dh + 4] each; the 4-word
// row pad keeps lane-per-row float4 reads conflict-free.  Each thread issues
// all of its loads for the tile (K and V, up to 4 pieces each) before
// converting and storing, so the tile costs one memory latency, not one per
// piece.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* dst) {
  float4 a, b;
  a.x = __uint_as_float(w.x << 16); a.y = __uint_as_float(w.x & 0xffff0000u);
  a.z = __uint_as_float(w.y << 16); a.w = __uint_as_float(w.y & 0xffff0000u);
  b.x = __uint_as_float(w.z << 16); b.y = __uint_as_float(w.z & 0xffff0000u);
  b.z = __uint_as_float(w.w << 16); b.w = __uint_as_float(w.w & 0xffff0000u);
  *reinterpret_cast<float4*>(dst) = a;
  *reinterpret_cast<float4*>(dst + 4) = b;
}

__device__ __forceinline__ void stage_kv(float* sk, float* sv, int ld, const uint16_t* kb, const uint16_t* vb,
                                         const float* kf, const float* vf, size_t row0, size_t row_stride, int nt,
                                         int dh) {
  if (kf) {
    const int pieces = dh / 4, total = nt * pieces;
    for (int base = threadIdx.x; base < total; base += 2 * THREADS) {
      float4 kk[2], vv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = base + u * THREADS;
        if (idx < total) {
          const int r = idx / pieces, c = idx % pieces;
          kk[u] = __ldg(reinterpret_cast<const float4*>(kf + row0 + r * row_stride) + c);
          vv[u] = __ldg(reinterpret_cast<const float4*>(vf + row0 + r * row_stride) + c);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = base + u * THREADS;
        if (idx < total) {
          const int r = idx / pieces, c = idx % pieces;
          *reinterpret_cast<float4*>(sk + r * ld + c * 4) = kk[u];
          *reinterpret_cast<float4*>(sv + r * ld + c * 4) = vv[u];
        }
      }
    }
  } else {
    const int pieces = dh / 8, total = nt * pieces;
    for (int base = threadIdx.x; base < total; base += 2 * THREADS) {
      uint4 kk[2], vv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = base + u * THREADS;
        if (idx < total) {
          const int r = idx / pieces, c = idx % pieces;
          kk[u] = __ldg(reinterpret_cast<const uint4*>(kb + row0 + r * row_stride) + c);
          vv[u] = __ldg(reinterpret_cast<const uint4*>(vb + row0 + r * row_stride) + c);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int idx = base + u * THREADS;
        if (idx < total) {
          const int r = idx / pieces, c = idx % pieces;
          bf16x8_to_f32(kk[u], sk + r * ld + c * 8);
          bf16x8_to_f32(vv[u], sv + r * ld + c * 8);
        }
      }
    }
  }
}

__global__ void __launch_bounds__(THREADS, 2) tree_attn_kernel(const AttnParams p) {
  extern __shared__ __align__(16) float smem_kv[];
  __shared__ __align__(16) float sq[8][MAX_DH];
  __shared__ int s_last;

  const int split = blockIdx.x;              // split == n_splits: the tree part
  const int pair = blockIdx.y;
  const int b = pair / p.Hkv, h = pair % p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dh = p.dh;
  const int ld = dh + 4;
  float* sk = smem_kv;
  float* sv = smem_kv + TILE * ld;
  const int nodes = n_nodes(p, b);
  const int R = nodes * p.G;
  const bool is_tree = split == p.n_splits;
  int lo = 0, hi = 0;
  if (!is_tree) {
    const int L = p.kv_len[b];
    lo = split * p.chunk;
    hi = min(L, lo + p.chunk);
  } else {
    hi = p.mode == 0 ? p.tree_cap : min(p.tree_size[b], p.tree_cap);
  }
  const int rec = dh + 2;
  const size_t row_stride = static_cast<size_t>(p.Hkv) * dh;

  // Each warp owns query rows r = r0 + warp + 8 i (i < 8); running state in registers.
  for (int r0 = 0; r0 < R; r0 += 64) {
    float m_run[8], l_run[8], acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      m_run[i] = -INFINITY;
      l_run[i] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
    }
    for (int t0 = lo; t0 < hi; t0 += TILE) {
      const int nt = min(TILE, hi - t0);
      __syncthreads();
      if (!is_tree) {
        const size_t row0 = ((static_cast<size_t>(b) * p.kv_cap + t0) * p.Hkv + h) * dh;
        stage_kv(sk, sv, ld, p.kp, p.vp, nullptr, nullptr, row0, row_stride, nt, dh);
      } else {
        const size_t row0 = ((static_cast<size_t>(b) * p.tree_cap + t0) * p.Hkv + h) * dh;
        stage_kv(sk, sv, ld, p.kt_bf16, p.vt_bf16, p.kt_f32, p.vt_f32, row0, row_stride, nt, dh);
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = r0 + warp + 8 * i;
        if (r >= R) break;
        const int node = r / p.G, hq = h * p.G + r % p.G;
        const size_t qo = q_index(p, b, node, hq);
        for (int d = lane; d < dh; d += 32)
          sq[warp][d] = p.mode == 0 ? p.q_f32[qo + d] : bf16_to_f32(p.q_bf16[qo + d]);
        __syncwarp();
        const uint64_t mask = is_tree ? row_mask(p, b, node) : ~0ull;
        float sc[2];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int j = lane + 32 * half;
          float s = -INFINITY;
          const bool vis = j < nt && (!is_tree || ((mask >> (t0 + j)) & 1ull));
          if (vis) {
            const float* kr = sk + j * ld;
            float dot = 0.f;
            for (int d0 = 0; d0 < dh; d0 += 4) {
              const float4 kv = *reinterpret_cast<const float4*>(kr + d0);
              const float4 qv = *reinterpret_cast<const float4*>(&sq[warp][d0]);
              dot = fmaf(qv.x, kv.x, dot);
              dot = fmaf(qv.y, kv.y, dot);
              dot = fmaf(qv.z, kv.z, dot);
              dot = fmaf(qv.w, kv.w, dot);
            }
            s = dot * p.scale;
          }
          sc[half] = s;
        }
        const float tmax = warp_max(fmaxf(sc[0], sc[1]));
        __syncwarp();
        if (tmax == -INFINITY) continue;
        const float m_new = fmaxf(m_run[i], tmax);
        const float corr = __expf(m_run[i] - m_new);
        const float p0 = sc[0] == -INFINITY ? 0.f : __expf(sc[0] - m_new);
        const float p1 = sc[1] == -INFINITY ? 0.f : __expf(sc[1] - m_new);
        l_run[i] = l_run[i] * corr + warp_sum(p0 + p1);
        m_run[i] = m_new;
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] *= corr;
        for (int j = 0; j < nt; ++j) {
          const float pj = __shfl_sync(0xffffffffu, j < 32 ? p0 : p1, j & 31);
          if (pj == 0.f) continue;
          const float* vr = sv + j * ld;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int d = lane + 32 * c;
            if (d < dh) acc[i][c] = fmaf(pj, vr[d], acc[i][c]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + warp + 8 * i;
      if (r >= R) break;
      const int node = r / p.G, hq = h * p.G + r % p.G;
      const size_t qi = (static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq;
      float* dst = p.part + (qi * (p.n_splits + 1) + split) * rec;
      if (lane == 0) {
        dst[0] = m_run[i];
        dst[1] = l_run[i];
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        if (d < dh) dst[2 + d] = acc[i][c];
      }
    }
  }

  // the last CTA of this (request, kv head) merges the splits in order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&p.counters[pair], 1);
    s_last = prev == p.n_splits;
    if (s_last) p.counters[pair] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int r = warp; r < R; r += 8) {
    const int node = r / p.G, hq = h * p.G + r % p.G;
    const size_t qi = (static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq;
    const float* src = p.part + qi * (p.n_splits + 1) * rec;
    // lane s holds split s (n_splits + 1 <= 32): all partial headers load at once
    const int ns = p.n_splits + 1;
    const float ms = lane < ns ? __ldcg(src + lane * rec) : -INFINITY;
    const float ls = lane < ns ? __ldcg(src + lane * rec + 1) : 0.f;
    const float M = warp_max(ms);
    const float wgt = ms == -INFINITY ? 0.f : __expf(ms - M);
    const float Lsum = warp_sum(wgt * ls);
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < ns; s0 += 8) {
      float vals[8][4];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = s0 + u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int d = lane + 32 * c;
          vals[u][c] = (s < ns && d < dh) ? __ldcg(src + s * rec + 2 + d) : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float ws = __shfl_sync(0xffffffffu, wgt, (s0 + u) & 31);
#pragma unroll
        for (int c = 0; c < 4; ++c) o[c] = fmaf(ws, vals[u][c], o[c]);
      }
    }
    const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int d = lane + 32 * c;
      if (d >= dh) continue;
      const float v = o[c] * inv;
      if (p.mode == 1) {
        p.out_f32[((static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq) * dh + d] = v;
      } else {
        const int j = b * p.rows_cap + node;
        const int col = hq * dh + d;
        uint16_t hi16, lo16;
        split_bf16(v, hi16, lo16);
        p.b_o[static_cast<size_t>(j) * p.bo_ld + col] = hi16;
        p.b_o[static_cast<size_t>(p.NP + j) * p.bo_ld + col] = lo16;
      }
    }
  }
}

}  // namespace

int attn_splits(const eagle_ctx* ctx, int pairs, int cap) {
  int want = ceil_div(2 * ctx->sm_count, pairs < 1 ? 1 : pairs);
  const int by_len = ceil_div(cap < 1 ? 1 : cap, TILE);
  if (want > by_len) want = by_len;
  if (want < 1) want = 1;
  if (want > 31) want = 31;        // n_splits + 1 records fit one warp in the merge
  return want;
}

static cudaError_t run_attn(eagle_ctx* ctx, AttnParams& p, int kernel_id, cudaStream_t st) {
  p.n_splits = attn_splits(ctx, p.B * p.Hkv, p.kv_cap);
  p.chunk = ceil_div(ceil_div(p.kv_cap, p.n_splits), TILE) * TILE;
  dim3 grid(p.n_splits + 1, p.B * p.Hkv);
  const size_t smem = static_cast<size_t>(2) * TILE * (p.dh + 4) * sizeof(float);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(tree_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(2 * TILE * (MAX_DH + 4) * sizeof(float)));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  trace_before(ctx, kernel_id, st);
  tree_attn_kernel<<<grid, THREADS, smem, st>>>(p);
  ctx->launches++;
  trace_after(ctx, kernel_id, st);
  return cudaGetLastError();
}

cudaError_t launch_draft_attn(eagle_ctx* ctx, const DraftLaunch& L, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  const Workspace& W = ctx->ws;
  AttnParams p{};
  p.mode = 0;
  p.B = L.batch;
  p.Hq = D.n_q_heads;
  p.Hkv = D.n_kv_heads;
  p.dh = D.head_dim;
  p.G = D.n_q_heads / D.n_kv_heads;
  p.rows_cap = L.rpr;
  p.q_f32 = ws_ptr<float>(L.ws, W.qrow);
  p.kp = L.draft_kv->k;
  p.vp = L.draft_kv->v;
  p.kv_cap = L.draft_kv->cap;
  p.kv_len = L.draft_kv->len;
  p.kt_f32 = L.out->k_tree;
  p.vt_f32 = L.out->v_tree;
  p.tree_cap = ctx->lim.max_expanded;
  p.anc = L.pool->anc;
  p.e0 = L.e0;
  p.scale = 1.0f / sqrtf(static_cast<float>(D.head_dim));
  p.b_o = ws_ptr<uint16_t>(L.ws, W.b_o);
  p.NP = L.NP;
  p.bo_ld = W.kp_o;
  p.part = ws_ptr<float>(L.ws, W.attn_part);
  p.counters = ws_ptr<int>(L.ws, W.attn_cnt);
  return run_attn(ctx, p, EAGLE_K_DRAFT_ATTN, st);
}

cudaError_t launch_verify_attn(eagle_ctx* ctx, int batch, const uint16_t* q, const uint16_t* kt,
                               const uint16_t* vt, const eagle_kv* prefix, const eagle_tree* tree,
                               float scale, float* out, void* ws, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  const Workspace& W = ctx->ws;
  AttnParams p{};
  p.mode = 1;
  p.B = batch;
  p.Hq = D.n_q_heads;
  p.Hkv = D.n_kv_heads;
  p.dh = D.head_dim;
  p.G = D.n_q_heads / D.n_kv_heads;
  p.rows_cap = tree->stride;
  p.q_bf16 = q;
  p.kp = prefix->k;
  p.vp = prefix->v;
  p.kv_cap = prefix->cap;
  p.kv_len = prefix->len;
  p.kt_bf16 = kt;
  p.vt_bf16 = vt;
  p.tree_cap = tree->stride;
  p.anc = tree->anc;
  p.tree_size = tree->size;
  p.scale = scale;
  p.out_f32 = out;
  p.part = ws_ptr<float>(ws, W.attn_part);
  p.counters = ws_ptr<int>(ws, W.attn_cnt) + ctx->lim.max_batch * D.n_kv_heads;
  return run_attn(ctx, p, EAGLE_K_VERIFY_ATTN, st);
}

}  // namespace eagle
