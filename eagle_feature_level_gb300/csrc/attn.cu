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
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "sm100.cuh"

namespace eagle {
namespace {

constexpr int TILE = 64;          // KV rows per shared-memory tile
constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int MAX_DH = 128;
constexpr int RW = 8;             // query rows a warp owns in one pass
constexpr int ROWS_PASS = WARPS * RW;
constexpr int PF = TILE * (MAX_DH / 8) / THREADS;   // 16-byte prefix pieces per thread per K (or V) tile

struct AttnParams {
  int mode;                       // 0 draft, 1 verify
  int B, Hq, Hkv, dh, G;
  int n_splits, chunk;            // prefix splits and rows per split (a multiple of TILE)
  int rows_cap;                   // query nodes per request (draft: rows per request; verify: tree stride)
  int rows_pass;                  // query rows staged per pass: min(ROWS_PASS, rows_cap * G)
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

__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* dst) {
  float4 a, b;
  a.x = __uint_as_float(w.x << 16); a.y = __uint_as_float(w.x & 0xffff0000u);
  a.z = __uint_as_float(w.y << 16); a.w = __uint_as_float(w.y & 0xffff0000u);
  b.x = __uint_as_float(w.z << 16); b.y = __uint_as_float(w.z & 0xffff0000u);
  b.z = __uint_as_float(w.w << 16); b.w = __uint_as_float(w.w & 0xffff0000u);
  *reinterpret_cast<float4*>(dst) = a;
  *reinterpret_cast<float4*>(dst + 4) = b;
}

// A bf16 prefix tile in flight: piece i of this thread is row (tid + i*THREADS)
// / (dh/8), 8 columns.  Loads are issued for the next tile before the current
// one is consumed; rows past the tile's end stay zero.
struct PrefixTile {
  uint4 k[PF], v[PF];
};

// 16-byte read-only load whose L2 line is replaced first (the prefix KV is
// read once per launch).
__device__ __forceinline__ uint4 ld_stream16(const void* ptr, uint64_t policy) {
  uint4 r;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr), "l"(policy));
  return r;
}

__device__ __forceinline__ void prefix_load(PrefixTile& t, const uint16_t* kb, const uint16_t* vb, size_t row0,
                                            size_t row_stride, int nt, int dh) {
  const uint64_t policy = sm100::l2_policy_evict_first();
  const int pieces = dh >> 3;
#pragma unroll
  for (int i = 0; i < PF; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    const int r = idx / pieces, c = idx - r * pieces;
    if (r < nt) {
      t.k[i] = ld_stream16(reinterpret_cast<const uint4*>(kb + row0 + r * row_stride) + c, policy);
      t.v[i] = ld_stream16(reinterpret_cast<const uint4*>(vb + row0 + r * row_stride) + c, policy);
    } else {
      t.k[i] = make_uint4(0u, 0u, 0u, 0u);
      t.v[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

__device__ __forceinline__ void prefix_store(const PrefixTile& t, float* sk, float* sv, int ld, int dh) {
  const int pieces = dh >> 3;
#pragma unroll
  for (int i = 0; i < PF; ++i) {
    const int idx = threadIdx.x + i * THREADS;
    const int r = idx / pieces, c = idx - r * pieces;
    if (r < TILE) {
      bf16x8_to_f32(t.k[i], sk + r * ld + c * 8);
      bf16x8_to_f32(t.v[i], sv + r * ld + c * 8);
    }
  }
}

// The tree part (at most one tile): fp32 (draft) or bf16 (verify) rows, zero past nt.
__device__ __forceinline__ void tree_stage(const AttnParams& p, float* sk, float* sv, int ld, size_t row0,
                                           size_t row_stride, int nt) {
  const int dh = p.dh;
  if (p.mode == 0) {
    const int pieces = dh >> 2;
    for (int idx = threadIdx.x; idx < TILE * pieces; idx += THREADS) {
      const int r = idx / pieces, c = idx - r * pieces;
      float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
      if (r < nt) {
        kk = __ldg(reinterpret_cast<const float4*>(p.kt_f32 + row0 + r * row_stride) + c);
        vv = __ldg(reinterpret_cast<const float4*>(p.vt_f32 + row0 + r * row_stride) + c);
      }
      *reinterpret_cast<float4*>(sk + r * ld + c * 4) = kk;
      *reinterpret_cast<float4*>(sv + r * ld + c * 4) = vv;
    }
  } else {
    const int pieces = dh >> 3;
    for (int idx = threadIdx.x; idx < TILE * pieces; idx += THREADS) {
      const int r = idx / pieces, c = idx - r * pieces;
      uint4 kk = make_uint4(0u, 0u, 0u, 0u), vv = kk;
      if (r < nt) {
        kk = __ldg(reinterpret_cast<const uint4*>(p.kt_bf16 + row0 + r * row_stride) + c);
        vv = __ldg(reinterpret_cast<const uint4*>(p.vt_bf16 + row0 + r * row_stride) + c);
      }
      bf16x8_to_f32(kk, sk + r * ld + c * 8);
      bf16x8_to_f32(vv, sv + r * ld + c * 8);
    }
  }
}

// Per-CTA constants of one attention launch, shared by the pass bodies.
struct PassCtx {
  int b, h, warp, lane, dh, ld, lo, hi, rec, split, dcol;
  bool is_tree, has_cols;
  size_t row_stride;
  float *sk, *sv, *sq, *sp;
  uint64_t* s_mask;
};

// One pass over this CTA's keys for query rows r0 .. r0 + rp - 1; warp w owns
// rows w + 8 i, i < nr <= NR.  The kernel is instantiated for NR = 1, 2, 4, 8
// (chosen from the launch's rows per pass) so that a warp issues work only
// for row slots that can exist: with one query row per warp the unrolled
// code of eight would cost eight times the issue slots.
template <int NR>
__device__ __forceinline__ void attn_pass(const AttnParams& p, const PassCtx& x, int r0, int rp) {
  const int b = x.b, h = x.h, warp = x.warp, lane = x.lane, dh = x.dh, ld = x.ld, lo = x.lo, hi = x.hi;
  const int rec = x.rec, split = x.split, dcol = x.dcol;
  const bool is_tree = x.is_tree, has_cols = x.has_cols;
  const size_t row_stride = x.row_stride;
  float *sk = x.sk, *sv = x.sv, *sq = x.sq, *sp = x.sp;
  uint64_t* s_mask = x.s_mask;
  const int nr = rp > warp ? (rp - warp + WARPS - 1) / WARPS : 0;   // <= NR
  // The prefix KV is not written by the kernels of this draft step: its
  // first tile is requested before waiting on the predecessor.
  PrefixTile pre;
  if (!is_tree && lo < hi)
    prefix_load(pre, p.kp, p.vp, ((static_cast<size_t>(b) * p.kv_cap + lo) * p.Hkv + h) * dh, row_stride,
                min(TILE, hi - lo), dh);
  if (r0 == 0) pdl_wait();                 // q rows, tree K/V and masks come from the predecessors
  __syncthreads();                         // previous pass done with sq
  for (int idx = threadIdx.x; idx < rp * (dh >> 2); idx += THREADS) {
    const int rr = idx / (dh >> 2), c = idx - rr * (dh >> 2);
    const int r = r0 + rr, node = r / p.G, hq = h * p.G + r % p.G;
    const size_t qo = q_index(p, b, node, hq) + 4 * c;
    float4 v;
    if (p.mode == 0) {
      v = *reinterpret_cast<const float4*>(p.q_f32 + qo);
    } else {
      const uint2 w = *reinterpret_cast<const uint2*>(p.q_bf16 + qo);
      v.x = __uint_as_float(w.x << 16); v.y = __uint_as_float(w.x & 0xffff0000u);
      v.z = __uint_as_float(w.y << 16); v.w = __uint_as_float(w.y & 0xffff0000u);
    }
    *reinterpret_cast<float4*>(sq + rr * dh + 4 * c) = v;
  }
  if (is_tree && lane < RW && lane < nr)
    s_mask[warp * RW + lane] = row_mask(p, b, (r0 + warp + WARPS * lane) / p.G);
  float m_run[NR], l_run[NR], acc[NR][4];
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
  }

  for (int t0 = lo; t0 < hi; t0 += TILE) {
    const int nt = min(TILE, hi - t0);
    __syncthreads();                       // all warps done with the previous tile
    if (!is_tree) {
      prefix_store(pre, sk, sv, ld, dh);
      if (t0 + TILE < hi)                  // next tile's loads fly while this one is consumed
        prefix_load(pre, p.kp, p.vp, ((static_cast<size_t>(b) * p.kv_cap + t0 + TILE) * p.Hkv + h) * dh,
                    row_stride, min(TILE, hi - t0 - TILE), dh);
    } else {
      tree_stage(p, sk, sv, ld, ((static_cast<size_t>(b) * p.tree_cap + t0) * p.Hkv + h) * dh, row_stride, nt);
    }
    __syncthreads();
    if (nr == 0) continue;

    // scores of keys lane and lane + 32 for each owned row
    float s0[NR], s1[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) { s0[i] = 0.f; s1[i] = 0.f; }
    const float* k0 = sk + lane * ld;
    const float* k1 = sk + (lane + 32) * ld;
    for (int d = 0; d < dh; d += 4) {
      const float4 a = *reinterpret_cast<const float4*>(k0 + d);
      const float4 c = *reinterpret_cast<const float4*>(k1 + d);
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        if (i < nr) {
          const float4 q = *reinterpret_cast<const float4*>(sq + (warp + WARPS * i) * dh + d);
          // plain FMA chains: the 2 x NR independent (row, key) sums give the ILP
          s0[i] = fmaf(q.w, a.w, fmaf(q.z, a.z, fmaf(q.y, a.y, fmaf(q.x, a.x, s0[i]))));
          s1[i] = fmaf(q.w, c.w, fmaf(q.z, c.z, fmaf(q.y, c.y, fmaf(q.x, c.x, s1[i]))));
        }
      }
    }
    // online softmax per row; probabilities to this warp's shared rows
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      if (i < nr) {
        // tree keys: one tile (t0 == 0), bit j of the row's ancestor mask
        const uint64_t mask = is_tree ? s_mask[warp * RW + i] : ~0ull;
        const bool v0 = lane < nt && ((mask >> lane) & 1ull);
        const bool v1 = lane + 32 < nt && ((mask >> (lane + 32)) & 1ull);
        const float a = v0 ? s0[i] * p.scale : -INFINITY;
        const float c = v1 ? s1[i] * p.scale : -INFINITY;
        const float m_new = fmaxf(m_run[i], warp_max(fmaxf(a, c)));
        float p0 = 0.f, p1 = 0.f, corr = 1.f;
        if (m_new != -INFINITY) {
          p0 = __expf(a - m_new);
          p1 = __expf(c - m_new);
          corr = __expf(m_run[i] - m_new);
        }
        l_run[i] = l_run[i] * corr + warp_sum(p0 + p1);
        m_run[i] = m_new;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) acc[i][c4] *= corr;
        sp[i * TILE + lane] = p0;
        sp[i * TILE + lane + 32] = p1;
      }
    }
    __syncwarp();
    // acc += P V over the tile, 4 keys per step (V rows past nt are zero)
    if (has_cols) {
      for (int j = 0; j < nt; j += 4) {
        float4 vv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) vv[u] = *reinterpret_cast<const float4*>(sv + (j + u) * ld + dcol);
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          if (i < nr) {
            const float4 pj = *reinterpret_cast<const float4*>(sp + i * TILE + j);
            acc[i][0] = fmaf(pj.x, vv[0].x, fmaf(pj.y, vv[1].x, fmaf(pj.z, vv[2].x, fmaf(pj.w, vv[3].x, acc[i][0]))));
            acc[i][1] = fmaf(pj.x, vv[0].y, fmaf(pj.y, vv[1].y, fmaf(pj.z, vv[2].y, fmaf(pj.w, vv[3].y, acc[i][1]))));
            acc[i][2] = fmaf(pj.x, vv[0].z, fmaf(pj.y, vv[1].z, fmaf(pj.z, vv[2].z, fmaf(pj.w, vv[3].z, acc[i][2]))));
            acc[i][3] = fmaf(pj.x, vv[0].w, fmaf(pj.y, vv[1].w, fmaf(pj.z, vv[2].w, fmaf(pj.w, vv[3].w, acc[i][3]))));
          }
        }
      }
    }
    __syncwarp();
  }
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    if (i < nr) {
      const int r = r0 + warp + WARPS * i;
      const int node = r / p.G, hq = h * p.G + r % p.G;
      const size_t qi = (static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq;
      float* dst = p.part + (qi * (p.n_splits + 1) + split) * rec;
      if (lane == 0) {
        dst[0] = m_run[i];
        dst[1] = l_run[i];
      }
      if (has_cols) {
#pragma unroll
        for (int c = 0; c < 4; ++c) dst[2 + dcol + c] = acc[i][c];
      }
    }
  }
}

// Dynamic shared memory: K tile, V tile ([TILE][dh+4] fp32 each; the 4-word
// pad makes lane-per-row float4 reads conflict-free), the pass's query rows
// [rows_pass][dh] and each warp's probabilities [WARPS][RW][TILE].
//
// Warp w owns query rows w + 8 i of the pass: it scores them against the tile
// (lane = keys lane and lane + 32), runs the online softmax and accumulates
// P V for them (lane = 4 output columns), so after the tile is staged no
// further block-wide barrier is needed.
template <int NR>
__global__ void __launch_bounds__(THREADS, 2) tree_attn_kernel(const AttnParams p) {
  pdl_trigger();
  if (p.mode == 1) pdl_wait();               // verification reads the tree's size first
  extern __shared__ __align__(16) float smem_attn[];
  __shared__ int s_last;
  __shared__ uint64_t s_mask[ROWS_PASS];     // ancestor masks of the tree part's rows

  const int split = blockIdx.x;              // split == n_splits: the tree part
  const int pair = blockIdx.y;
  const int b = pair / p.Hkv, h = pair % p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dh = p.dh;
  const int ld = dh + 4;
  float* sk = smem_attn;
  float* sv = sk + TILE * ld;
  float* sq = sv + TILE * ld;
  float* sp = sq + p.rows_pass * dh + (warp * RW) * TILE;
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
  const int dcol = 4 * lane;                 // this lane's output columns
  const bool has_cols = dcol < dh;

  const PassCtx x{b, h, warp, lane, dh, ld, lo, hi, rec, split, dcol, is_tree, has_cols, row_stride,
                  sk, sv, sq, sp, s_mask};
  for (int r0 = 0; r0 < R; r0 += p.rows_pass) {
    attn_pass<NR>(p, x, r0, min(p.rows_pass, R - r0));
  }

  pdl_wait();                                 // (no-op once waited; a pass-less CTA waits here)
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
  const int tiles = ceil_div(cap < 1 ? 1 : cap, TILE);
  // one wave at two CTAs per SM, the tree part's CTA included
  int want = 2 * ctx->sm_count / (pairs < 1 ? 1 : pairs) - 1;
  if (want > tiles) want = tiles;
  if (want > 31) want = 31;        // n_splits + 1 records fit one warp in the merge
  if (want < 1) want = 1;
  const int per = ceil_div(tiles, want);
  return ceil_div(tiles, per);     // every split non-empty at full length
}

template <int NR>
static cudaError_t launch_attn_nr(const AttnParams& p, dim3 grid, size_t smem, cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    const size_t most = (static_cast<size_t>(2) * TILE * (MAX_DH + 4) + static_cast<size_t>(ROWS_PASS) * MAX_DH +
                         static_cast<size_t>(WARPS) * RW * TILE) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(tree_attn_kernel<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(most));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(tree_attn_kernel<NR>, grid, dim3(THREADS), smem, st, p);
}

static cudaError_t run_attn(eagle_ctx* ctx, AttnParams& p, int kernel_id, cudaStream_t st) {
  p.n_splits = attn_splits(ctx, p.B * p.Hkv, p.kv_cap);
  p.chunk = ceil_div(ceil_div(p.kv_cap, TILE), p.n_splits) * TILE;
  p.rows_pass = std::min(ROWS_PASS, p.rows_cap * p.G);
  dim3 grid(p.n_splits + 1, p.B * p.Hkv);
  const size_t smem = (static_cast<size_t>(2) * TILE * (p.dh + 4) + static_cast<size_t>(p.rows_pass) * p.dh +
                       static_cast<size_t>(WARPS) * RW * TILE) * sizeof(float);
  const int per_warp = ceil_div(p.rows_pass, WARPS);
  trace_before(ctx, kernel_id, st);
  cudaError_t e;
  if (per_warp <= 1) e = launch_attn_nr<1>(p, grid, smem, st);
  else if (per_warp <= 2) e = launch_attn_nr<2>(p, grid, smem, st);
  else if (per_warp <= 4) e = launch_attn_nr<4>(p, grid, smem, st);
  else e = launch_attn_nr<RW>(p, grid, smem, st);
  ctx->launches++;
  trace_after(ctx, kernel_id, st);
  return e;
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

// ---- verify attention from a fixed device scratch (no workspace) ----------
//
// For callers that cannot hand the library device memory (a C host that
// links only libeagle and owns no allocator, a serving loop whose memory is
// fully reserved at start-up): the split partials and the arrival counters
// of eagle_tree_verify_attn_noalloc live in this file-scope array, one per
// device, instead of the caller's workspace.  Layout: [0, 64 KiB) int
// counters, one per (request, kv head), which must be zero when a call
// starts; then the fp32 partial records, which need no initial value.
constexpr size_t kScratchBytes = static_cast<size_t>(32) << 20;
constexpr size_t kScratchCounterBytes = static_cast<size_t>(64) << 10;
constexpr int kScratchMaxPairs = static_cast<int>(kScratchCounterBytes / sizeof(int));
constexpr int kScratchMaxDevices = 64;

static __device__ __align__(256) unsigned char verify_scratch[kScratchBytes];

namespace {
std::mutex scratch_mu;
void* scratch_base[kScratchMaxDevices] = {};
}  // namespace

size_t verify_scratch_need(const eagle_ctx* ctx, int batch, const eagle_kv* prefix, const eagle_tree* tree) {
  const eagle_dims& D = ctx->dims;
  const int splits = attn_splits(ctx, batch * D.n_kv_heads, prefix->cap);
  const size_t records = static_cast<size_t>(batch) * tree->stride * D.n_q_heads * (splits + 1);
  return records * (D.head_dim + 2) * sizeof(float);
}

eagle_status launch_verify_attn_noalloc(eagle_ctx* ctx, int batch, const uint16_t* q, const uint16_t* kt,
                                        const uint16_t* vt, const eagle_kv* prefix, const eagle_tree* tree,
                                        float scale, float* out, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  if (batch * D.n_kv_heads > kScratchMaxPairs ||
      verify_scratch_need(ctx, batch, prefix, tree) > kScratchBytes - kScratchCounterBytes)
    return EAGLE_ERR_CAPACITY;                 // nothing launched
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kScratchMaxDevices) return EAGLE_ERR_CUDA;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(scratch_mu);
    base = scratch_base[dev];
    if (base == nullptr) {
      // first call on this device: the array's address, then zeroed counters
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, verify_scratch) != cudaSuccess) return EAGLE_ERR_CUDA;
      if (cudaMemsetAsync(ptr, 0, kScratchCounterBytes, st) != cudaSuccess) return EAGLE_ERR_CUDA;
      if (cudaStreamSynchronize(st) != cudaSuccess) return EAGLE_ERR_CUDA;
      scratch_base[dev] = base = ptr;
    }
  }
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
  // the last CTA of each (request, kv head) puts its counter back to zero
  p.counters = static_cast<int*>(base);
  p.part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kScratchCounterBytes);
  return run_attn(ctx, p, EAGLE_K_VERIFY_ATTN, st) == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // namespace eagle
