// Tree-masked attention, shared by the draft layer and the target's
// verification layer ([B] "Tree Attention 如何一次验证多条路径": node u sees the
// committed prefix plus the tree nodes that are its ancestors or itself).
//
// Split-KV layout: one CTA per (prefix split or tree part, request, kv head).
// Every query row of the request that maps to this kv head (tree nodes x
// GQA group) consumes the same shared-memory K/V tile, so prefix KV bytes
// are read from HBM once per call however many tree nodes there are.  Each
// CTA writes (max, sum, unnormalised output) partials; the last CTA of a
// (request, kv head) merges them in split order.  The ancestor mask of each
// query row is one 64-bit word, tested per tree key.
//
// Two kernels share this layout.  The draft layer's (a few fp32 query rows
// per request and layer) runs on the CUDA cores, one wave at four CTAs per
// SM.  The verification layer's (every tree node at once, bf16 queries)
// runs its products on the tensor cores (warp-level bf16 MMA tiles, fp32
// accumulation), one wave at two CTAs per SM.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "sm100.cuh"

namespace eagle {
namespace {

constexpr int TILE = 64;          // prefix / verify-tree keys per shared-memory tile (bf16)
constexpr int TILE_F32 = 32;      // draft-tree keys per tile (fp32, or bf16 hi + lo: same bytes)
constexpr int THREADS = 128;
constexpr int WARPS = THREADS / 32;
constexpr int MAX_DH = 128;
constexpr int RW = 8;             // CUDA-core kernel: query rows a warp owns in one pass, at most
constexpr int ROWS_PASS = WARPS * RW;   // query rows per pass (tensor-core kernel: two 16-row tiles)
constexpr int MASKW = EAGLE_MASK_WORDS(EAGLE_MAX_NODES);   // ancestor-mask words a row can have
constexpr int KLD = MAX_DH + 8;   // bf16 row pitch in shared memory (elements): ldmatrix rows hit distinct banks
constexpr int MLD = MAX_DH + 4;   // fp32 row pitch of a warp's softmax state in the intra-CTA merge

// Shared-memory bytes of one K+V tile buffer: 64 bf16 rows of K then of V,
// 32 fp32 rows of each, or 32 bf16 rows each of K hi, K lo, V hi, V lo.
constexpr size_t TILE_BYTES = static_cast<size_t>(2) * TILE * KLD * 2;
static_assert(static_cast<size_t>(2) * TILE_F32 * (MAX_DH + 4) * 4 <= TILE_BYTES, "fp32 half tile fits a buffer");
// Tensor-core kernel with nw warps: query rows per pass (32 with four warps,
// 16 per warp with eight), their bf16 hi and lo copies, and the nw / 2 warp
// states of 16 rows that reuse that space in the intra-CTA merge.
__host__ __device__ constexpr int mma_rows(int nw) { return nw == 4 ? 32 : 16 * nw; }
__host__ __device__ constexpr size_t q_bytes(int nw) { return static_cast<size_t>(2) * mma_rows(nw) * KLD * 2; }
__host__ __device__ constexpr size_t mrg_bytes(int nw) { return static_cast<size_t>(nw / 2) * 16 * MLD * 4; }
static_assert(mrg_bytes(4) <= q_bytes(4) && mrg_bytes(8) <= q_bytes(8), "the merge states reuse the query rows' space");
constexpr size_t Q_BYTES = q_bytes(4);

struct AttnParams {
  int mode;                       // 0 draft, 1 verify
  int B, Hq, Hkv, dh, G;
  int n_splits, chunk;            // prefix splits and rows per split (a multiple of TILE)
  int n_buf;                      // tile buffers per CTA (2: the next prefix tile streams in)
  int rows_cap;                   // query nodes per request (draft: rows per request; verify: tree stride)
  int rows_pass;                  // CUDA-core kernel: query rows staged per pass, min(ROWS_PASS, rows_cap * G)
  const float* q_f32;             // draft: [n][Hq*dh] fp32
  const uint16_t* q_bf16;         // verify: [B][S][Hq][dh] bf16
  const uint16_t* kp;             // prefix KV [B][cap][Hkv][dh] bf16, or block pools (paged)
  const uint16_t* vp;
  int kv_cap;
  PagedKv paged;                  // verify: the prefix through a block table (table null: contiguous)
  const int32_t* kv_len;
  const float* kt_f32;            // draft: tree K/V [B][E][Hkv][dh] fp32
  const float* vt_f32;
  const uint16_t* kt_bf16;        // verify: tree K/V [B][S][Hkv][dh] bf16
  const uint16_t* vt_bf16;
  int tree_cap;                   // E or S
  const uint64_t* anc;            // draft: pool.anc [B][E][W]; verify: tree.anc [B][S][W]
  int mask_words;                 // W = EAGLE_MASK_WORDS(tree_cap)
  const int32_t* tree_size;       // verify: [B]
  int e0;                         // draft: first expanded slot of this layer
  float scale;
  float* out_f32;                 // verify: [B][S][Hq][dh]
  uint16_t* b_o;                  // draft: next GEMM operand (hi/lo), [2NP][bo_ld]
  int NP, bo_ld;
  float* part;                    // partial records [query row][split][dh + 4]
  int* counters;
  int cluster;                    // tensor-core kernel: the splits of a (request, kv head) form a cluster
                                  // and merge through distributed shared memory (part, counters unused)
  int recs_off;                   // with cluster: byte offset of the CTA's records [rows][dh + 4] in shared memory
  int tma;                        // tcgen05 kernel: whole prefix tiles by TMA through the launch's tensor maps
  int box_rows;                   // keys per TMA box: 64, or the block size of a paged prefix
  int stages;                     // tcgen05 kernel: K/V ring stages
  int* status;                    // device status word (null: not reported)
  uint64_t* stamp;                // launch timestamps (null: off)
};

// Prefix rows of request b that exist: a length beyond the cache is read as
// the whole cache and reported once per (request, kv head) pair.
__device__ __forceinline__ int prefix_rows(const AttnParams& p, int b, bool report) {
  const int L = p.kv_len[b];
  if (L > p.kv_cap) {
    if (report) set_status(p.status, EAGLE_ERR_CAPACITY);
    return p.kv_cap;
  }
  return L;
}

__device__ __forceinline__ int n_nodes(const AttnParams& p, int b) {
  return p.mode == 0 ? p.rows_cap : min(p.tree_size[b], p.rows_cap);
}

__device__ __forceinline__ size_t q_index(const AttnParams& p, int b, int node, int hq) {
  return ((static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq) * p.dh;
}

// Word w of a query row's ancestor mask (tree keys j with bit j % 64 of
// word j / 64 set are visible to the row).
__device__ __forceinline__ uint64_t row_mask(const AttnParams& p, int b, int node, int w) {
  const size_t slot = static_cast<size_t>(b) * p.tree_cap + (p.mode == 0 ? p.e0 + node : node);
  return p.anc[slot * p.mask_words + w];
}

// A query row's mask words into shared memory (MASKW per row, unused ones zero).
__device__ __forceinline__ void load_row_mask(const AttnParams& p, uint64_t* dst, int b, int node) {
#pragma unroll
  for (int w = 0; w < MASKW; ++w) dst[w] = w < p.mask_words ? row_mask(p, b, node, w) : 0ull;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(sm100::smem_u32(dst)), "l"(src),
               "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async16_cg(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// Waits until at most n (0..3, larger taken as 3) copy groups are pending.
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  if (n <= 0) cp_async_wait<0>();
  else if (n == 1) cp_async_wait<1>();
  else if (n == 2) cp_async_wait<2>();
  else cp_async_wait<3>();
}

// Copies one bf16 tile (keys t0 .. t0 + nt - 1 of kv head h) into buf as K
// rows [TILE][KLD] then V rows; rows past nt are zeroed.  Issued by all
// threads as 16-byte asynchronous copies (one commit group per tile).
__device__ __forceinline__ void stage_bf16(uint16_t* buf, const uint16_t* kb, const uint16_t* vb, size_t row0,
                                           size_t row_stride, int nt, int dh, uint64_t policy) {
  uint16_t* sk = buf;
  uint16_t* sv = buf + TILE * KLD;
  const int pieces = dh >> 3;
  for (int idx = threadIdx.x; idx < TILE * pieces; idx += blockDim.x) {
    const int r = idx / pieces, c = idx - r * pieces;
    if (r < nt) {
      cp_async16(sk + r * KLD + 8 * c, kb + row0 + r * row_stride + 8 * c, policy);
      cp_async16(sv + r * KLD + 8 * c, vb + row0 + r * row_stride + 8 * c, policy);
    } else {
      *reinterpret_cast<uint4*>(sk + r * KLD + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sv + r * KLD + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  cp_async_commit();
}

// Prefix keys t0 .. t0 + nt - 1 of request b, kv head h, staged like
// stage_bf16 but read through the block table; rows of an unallocated block
// are zero and reported.
__device__ __forceinline__ void stage_bf16_paged(uint16_t* buf, const AttnParams& p, int b, int h, int t0, int nt,
                                                 uint64_t policy) {
  uint16_t* sk = buf;
  uint16_t* sv = buf + TILE * KLD;
  const int dh = p.dh, pieces = dh >> 3;
  for (int idx = threadIdx.x; idx < TILE * pieces; idx += blockDim.x) {
    const int r = idx / pieces, c = idx - r * pieces;
    bool loaded = false;
    if (r < nt) {
      const long long row = paged_row(p.paged, b, t0 + r);
      if (row >= 0) {
        const size_t off = (static_cast<size_t>(row) * p.Hkv + h) * dh + 8 * c;
        cp_async16(sk + r * KLD + 8 * c, p.kp + off, policy);
        cp_async16(sv + r * KLD + 8 * c, p.vp + off, policy);
        loaded = true;
      } else if (c == 0) {
        set_status(p.status, EAGLE_ERR_INVALID_ARG);
      }
    }
    if (!loaded) {
      *reinterpret_cast<uint4*>(sk + r * KLD + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sv + r * KLD + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  cp_async_commit();
}

// Final output of one query row from the merged split states: o / L, as
// fp32 (verification) or as the next GEMM's hi / lo bf16 operand (draft).
__device__ __forceinline__ void write_merged_row(const AttnParams& p, int b, int node, int hq, const float (&o)[4],
                                                 float Lsum, int lane) {
  const int dh = p.dh;
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

// The splits of one (request, kv head) as one thread-block cluster: each
// CTA has left its records [row][dh + 4] (max, sum, 2 unused, output) in its
// own shared memory at `recs`; CTA `rank` merges the rows r = rank (mod
// splits + 1), warp by warp, reading every split's record of the row from
// that split's CTA.  The arithmetic and its order are those of the merge
// through global memory (the splits' weights in a warp, then the outputs
// summed split by split).  Every thread of every CTA of the cluster calls it.
__device__ __noinline__ void cluster_merge(const AttnParams& p, const float* recs, int R, int b, int h, int warp,
                                           int lane) {
  const int dh = p.dh, rec = dh + 4;
  __syncthreads();
  sm100::cluster_sync();                     // every CTA's records are complete
  const int ns = p.n_splits + 1;
  const int rank = static_cast<int>(sm100::cluster_rank());
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  for (int r = rank + ns * warp; r < R; r += ns * nwarps) {
    const int node = r / p.G, hq = h * p.G + r % p.G;
    const float* mine = recs + static_cast<size_t>(r) * rec;
    const float ms = lane < ns ? sm100::dsmem_ld_f32(sm100::dsmem_addr(mine, lane)) : -INFINITY;
    const float ls = lane < ns ? sm100::dsmem_ld_f32(sm100::dsmem_addr(mine + 1, lane)) : 0.f;
    const float M = warp_max(ms);
    const float wgt = ms == -INFINITY ? 0.f : __expf(ms - M);
    const float Lsum = warp_sum(wgt * ls);
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int sp = 0; sp < ns; ++sp) {
      const float ws = __shfl_sync(0xffffffffu, wgt, sp);
      const uint32_t rs = sm100::dsmem_addr(mine + 4, sp);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        if (d < dh) o[c] = fmaf(ws, sm100::dsmem_ld_f32(rs + 4u * static_cast<uint32_t>(d)), o[c]);
      }
    }
    write_merged_row(p, b, node, hq, o, Lsum, lane);
  }
  sm100::cluster_sync();                     // no CTA leaves while a peer still reads its records
}

// ---- draft layer: CUDA cores -------------------------------------------------

// Copies draft-tree keys k0 .. k0 + nt - 1 (fp32, at most TILE_F32) into buf
// as K rows [TILE_F32][dh + 4] then V rows; rows past nt are zeroed.
__device__ __forceinline__ void stage_f32(float* buf, const float* kf, const float* vf, size_t row0,
                                          size_t row_stride, int nt, int dh) {
  const int ld = dh + 4;
  float* sk = buf;
  float* sv = buf + TILE_F32 * ld;
  const int pieces = dh >> 2;
  const uint64_t policy = sm100::l2_policy_evict_first();
  for (int idx = threadIdx.x; idx < TILE_F32 * pieces; idx += blockDim.x) {
    const int r = idx / pieces, c = idx - r * pieces;
    if (r < nt) {
      cp_async16(sk + r * ld + 4 * c, kf + row0 + r * row_stride + 4 * c, policy);
      cp_async16(sv + r * ld + 4 * c, vf + row0 + r * row_stride + 4 * c, policy);
    } else {
      *reinterpret_cast<float4*>(sk + r * ld + 4 * c) = make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(sv + r * ld + 4 * c) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  cp_async_commit();
}

__device__ __forceinline__ float4 bf16x4(uint2 w) {
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u), __uint_as_float(w.y << 16),
                     __uint_as_float(w.y & 0xffff0000u));
}

// Running softmax state of the rows a warp owns in a pass.
template <int NR>
struct RowState {
  float m[NR], l[NR], acc[NR][4];
};

// One staged tile against the warp's rows: scores of the lane's keys (lane
// and lane + 32 for a bf16 tile, lane for an fp32 half tile), the online
// softmax, and acc += P V (lane = 4 output columns).  `tmask` holds bit j of
// tile key j for the tree part (all ones for prefix tiles).
template <int NR, bool F32>
__device__ __forceinline__ void tile_compute(const AttnParams& p, RowState<NR>& st, const void* buf, const float* sq,
                                             float* sp, const uint64_t* s_mask, int warp, int lane, int nr, int nt,
                                             int key_base, bool is_tree) {
  const int dh = p.dh;
  constexpr int KEYS = F32 ? TILE_F32 : TILE;
  float s0[NR], s1[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) { s0[i] = 0.f; s1[i] = 0.f; }
  if (F32) {
    const int ld = dh + 4;
    const float* k0 = static_cast<const float*>(buf) + lane * ld;
    for (int d = 0; d < dh; d += 4) {
      const float4 a = *reinterpret_cast<const float4*>(k0 + d);
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        if (i < nr) {
          const float4 q = *reinterpret_cast<const float4*>(sq + (warp + WARPS * i) * dh + d);
          s0[i] = fmaf(q.w, a.w, fmaf(q.z, a.z, fmaf(q.y, a.y, fmaf(q.x, a.x, s0[i]))));
        }
      }
    }
  } else {
    const uint16_t* k0 = static_cast<const uint16_t*>(buf) + lane * KLD;
    const uint16_t* k1 = k0 + 32 * KLD;
    for (int d = 0; d < dh; d += 8) {
      const uint4 wa = *reinterpret_cast<const uint4*>(k0 + d);
      const uint4 wc = *reinterpret_cast<const uint4*>(k1 + d);
      const float4 a0 = bf16x4(make_uint2(wa.x, wa.y)), a1 = bf16x4(make_uint2(wa.z, wa.w));
      const float4 c0 = bf16x4(make_uint2(wc.x, wc.y)), c1 = bf16x4(make_uint2(wc.z, wc.w));
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        if (i < nr) {
          const float* qr = sq + (warp + WARPS * i) * dh + d;
          const float4 q0 = *reinterpret_cast<const float4*>(qr);
          const float4 q1 = *reinterpret_cast<const float4*>(qr + 4);
          float x = fmaf(q0.w, a0.w, fmaf(q0.z, a0.z, fmaf(q0.y, a0.y, fmaf(q0.x, a0.x, s0[i]))));
          s0[i] = fmaf(q1.w, a1.w, fmaf(q1.z, a1.z, fmaf(q1.y, a1.y, fmaf(q1.x, a1.x, x))));
          float y = fmaf(q0.w, c0.w, fmaf(q0.z, c0.z, fmaf(q0.y, c0.y, fmaf(q0.x, c0.x, s1[i]))));
          s1[i] = fmaf(q1.w, c1.w, fmaf(q1.z, c1.z, fmaf(q1.y, c1.y, fmaf(q1.x, c1.x, y))));
        }
      }
    }
  }
  // online softmax per row; probabilities to this warp's shared rows
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    if (i < nr) {
      // tree keys: bit key_base + j of the row's ancestor mask; a tile (64
      // bf16 or 32 fp32 keys, starting at a multiple of its size) lies in
      // one mask word
      const uint64_t mask = is_tree ? s_mask[(warp * RW + i) * MASKW + (key_base >> 6)] : ~0ull;
      const int kb = key_base & 63;
      const int j0 = lane, j1 = lane + 32;
      const bool v0 = j0 < nt && ((mask >> (kb + j0)) & 1ull);
      const bool v1 = !F32 && j1 < nt && ((mask >> (kb + (j1 & 63))) & 1ull);
      const float a = v0 ? s0[i] * p.scale : -INFINITY;
      const float c = v1 ? s1[i] * p.scale : -INFINITY;
      const float m_new = fmaxf(st.m[i], warp_max_redux(fmaxf(a, c)));
      float p0 = 0.f, p1 = 0.f, corr = 1.f;
      if (m_new != -INFINITY) {
        p0 = __expf(a - m_new);
        p1 = __expf(c - m_new);
        corr = __expf(st.m[i] - m_new);
      }
      st.l[i] = st.l[i] * corr + warp_sum(p0 + p1);
      st.m[i] = m_new;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) st.acc[i][c4] *= corr;
      sp[i * TILE + lane] = p0;
      if (!F32) sp[i * TILE + lane + 32] = p1;
    }
  }
  __syncwarp();
  // acc += P V over the tile, 4 keys per step (rows past nt are zero)
  const int dcol = 4 * lane;
  if (dcol < dh) {
    for (int j = 0; j < nt; j += 4) {
      float4 vv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (F32) {
          vv[u] = *reinterpret_cast<const float4*>(static_cast<const float*>(buf) + (KEYS + j + u) * (dh + 4) + dcol);
        } else {
          vv[u] = bf16x4(*reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(buf) + (KEYS + j + u) * KLD +
                                                         dcol));
        }
      }
#pragma unroll
      for (int i = 0; i < NR; ++i) {
        if (i < nr) {
          const float4 pj = *reinterpret_cast<const float4*>(sp + i * TILE + j);
          st.acc[i][0] = fmaf(pj.x, vv[0].x, fmaf(pj.y, vv[1].x, fmaf(pj.z, vv[2].x, fmaf(pj.w, vv[3].x, st.acc[i][0]))));
          st.acc[i][1] = fmaf(pj.x, vv[0].y, fmaf(pj.y, vv[1].y, fmaf(pj.z, vv[2].y, fmaf(pj.w, vv[3].y, st.acc[i][1]))));
          st.acc[i][2] = fmaf(pj.x, vv[0].z, fmaf(pj.y, vv[1].z, fmaf(pj.z, vv[2].z, fmaf(pj.w, vv[3].z, st.acc[i][2]))));
          st.acc[i][3] = fmaf(pj.x, vv[0].w, fmaf(pj.y, vv[1].w, fmaf(pj.z, vv[2].w, fmaf(pj.w, vv[3].w, st.acc[i][3]))));
        }
      }
    }
  }
  __syncwarp();
}

// Dynamic shared memory: n_buf tile buffers (TILE_BYTES each), the pass's
// query rows [rows_pass][dh] fp32, and each warp's probabilities
// [WARPS][RW][TILE].
//
// One CTA per (prefix split or tree part, request, kv head).  Warp w owns
// query rows w + 4 i of a pass: it scores them against the staged tile,
// runs the online softmax and accumulates P V for them, so a staged tile
// needs no further block-wide barrier.  Prefix tiles are bf16 copied by
// cp.async (the next one streams in while the current one is consumed when a
// split holds several); the draft's fp32 tree part is consumed as two
// 32-key halves of the same buffer.  The kernel is instantiated for NR = 1,
// 2, 4, 8 rows per warp so that a warp issues work only for row slots that
// can exist.
template <int NR>
__global__ void __launch_bounds__(THREADS, 4) tree_attn_kernel(const AttnParams p) {
  const LaunchStamp ls(p.stamp);
  pdl_trigger();
  if (p.mode == 1) {
    pdl_wait();                              // verification reads the tree's size first
    ls.waited();
  }
  extern __shared__ __align__(16) uint8_t smem_attn[];
  __shared__ int s_last;
  __shared__ uint64_t s_mask[ROWS_PASS * MASKW];   // ancestor masks of the tree part's rows

  const int split = blockIdx.x;              // split == n_splits: the tree part
  const int pair = blockIdx.y;
  const int b = pair / p.Hkv, h = pair % p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dh = p.dh;
  uint8_t* bufs = smem_attn;
  float* sq = reinterpret_cast<float*>(smem_attn + p.n_buf * TILE_BYTES);
  float* sp = sq + p.rows_pass * dh + (warp * RW) * TILE;
  const int nodes = n_nodes(p, b);
  const int R = nodes * p.G;
  const bool is_tree = split == p.n_splits;
  const bool tree_f32 = is_tree && p.mode == 0;
  int lo = 0, hi = 0;
  if (!is_tree) {
    const int L = prefix_rows(p, b, split == 0 && threadIdx.x == 0);
    lo = split * p.chunk;
    hi = min(L, lo + p.chunk);
  } else {
    hi = p.mode == 0 ? p.tree_cap : min(p.tree_size[b], p.tree_cap);
  }
  const int rec = dh + 4;                    // partial record: max, sum, 2 unused, output[dh]
  const size_t row_stride = static_cast<size_t>(p.Hkv) * dh;
  const uint64_t policy = sm100::l2_policy_evict_first();
  const int step = tree_f32 ? TILE_F32 : TILE;
  const int n_tiles = hi > lo ? (hi - lo + step - 1) / step : 0;
  // A split whose keys fit one buffer stages them once for every pass.
  const bool resident = n_tiles <= 1;

  auto stage = [&](int tile, int which) {
    uint8_t* buf = bufs + which * TILE_BYTES;
    const int t0 = lo + tile * step, nt = min(step, hi - t0);
    if (tree_f32)
      stage_f32(reinterpret_cast<float*>(buf), p.kt_f32, p.vt_f32,
                ((static_cast<size_t>(b) * p.tree_cap + t0) * p.Hkv + h) * dh, row_stride, nt, dh);
    else if (is_tree)
      stage_bf16(reinterpret_cast<uint16_t*>(buf), p.kt_bf16, p.vt_bf16,
                 ((static_cast<size_t>(b) * p.tree_cap + t0) * p.Hkv + h) * dh, row_stride, nt, dh, policy);
    else if (p.paged.table)
      stage_bf16_paged(reinterpret_cast<uint16_t*>(buf), p, b, h, t0, nt, policy);
    else
      stage_bf16(reinterpret_cast<uint16_t*>(buf), p.kp, p.vp,
                 ((static_cast<size_t>(b) * p.kv_cap + t0) * p.Hkv + h) * dh, row_stride, nt, dh, policy);
  };
  // The prefix KV is not written by the kernels of this draft step: its
  // first tile is requested before waiting on the predecessor.
  if (!is_tree && n_tiles > 0) stage(0, 0);
  pdl_wait();                                // q rows, tree K/V and masks come from the predecessors
  ls.waited();
  if (is_tree && n_tiles > 0) stage(0, 0);

  for (int r0 = 0; r0 < R; r0 += p.rows_pass) {
    const int rp = min(p.rows_pass, R - r0);
    const int nr = rp > warp ? (rp - warp + WARPS - 1) / WARPS : 0;   // <= NR
    if (r0 > 0) __syncthreads();             // the previous pass is done with sq (and the buffers)
    for (int idx = threadIdx.x; idx < rp * (dh >> 2); idx += THREADS) {
      const int rr = idx / (dh >> 2), c = idx - rr * (dh >> 2);
      const int r = r0 + rr, node = r / p.G, hq = h * p.G + r % p.G;
      const size_t qo = q_index(p, b, node, hq) + 4 * c;
      float4 v;
      if (p.mode == 0) {
        v = *reinterpret_cast<const float4*>(p.q_f32 + qo);
      } else {
        const uint2 w = *reinterpret_cast<const uint2*>(p.q_bf16 + qo);
        v = bf16x4(w);
      }
      *reinterpret_cast<float4*>(sq + rr * dh + 4 * c) = v;
    }
    if (is_tree && lane < RW && lane < nr)
      load_row_mask(p, s_mask + (warp * RW + lane) * MASKW, b, (r0 + warp + WARPS * lane) / p.G);
    RowState<NR> st;
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      st.m[i] = -INFINITY;
      st.l[i] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) st.acc[i][c] = 0.f;
    }
    for (int tile = 0; tile < n_tiles; ++tile) {
      const int which = p.n_buf > 1 ? (tile & 1) : 0;
      if (!resident) {
        // staged earlier: tile 0 of the first pass (prologue), or by the
        // previous iteration's prefetch when two buffers alternate
        const bool staged = (r0 == 0 && tile == 0) || (p.n_buf > 1 && tile > 0);
        if (!staged) {
          __syncthreads();                   // every warp is done with this buffer
          stage(tile, which);
        }
        if (p.n_buf > 1 && tile + 1 < n_tiles) {
          __syncthreads();                   // the other buffer's previous tile is consumed
          stage(tile + 1, which ^ 1);
          cp_async_wait<1>();                // this tile's copies have landed
        } else {
          cp_async_wait<0>();
        }
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      if (nr > 0) {
        const int t0 = lo + tile * step;
        const int nt = min(step, hi - t0);
        const uint8_t* buf = bufs + which * TILE_BYTES;
        if (tree_f32)
          tile_compute<NR, true>(p, st, buf, sq, sp, s_mask, warp, lane, nr, nt, t0, true);
        else
          tile_compute<NR, false>(p, st, buf, sq, sp, s_mask, warp, lane, nr, nt, is_tree ? t0 : 0, is_tree);
      }
    }
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      if (i < nr) {
        const int r = r0 + warp + WARPS * i;
        const int node = r / p.G, hq = h * p.G + r % p.G;
        const size_t qi = (static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq;
        float* dst = p.cluster ? reinterpret_cast<float*>(smem_attn + p.recs_off) + static_cast<size_t>(r) * rec
                               : p.part + (qi * (p.n_splits + 1) + split) * rec;
        if (lane == 0) {
          dst[0] = st.m[i];
          dst[1] = st.l[i];
        }
        const int dcol = 4 * lane;
        if (dcol < dh)
          *reinterpret_cast<float4*>(dst + 4 + dcol) = make_float4(st.acc[i][0], st.acc[i][1], st.acc[i][2], st.acc[i][3]);
      }
    }
  }
  cp_async_wait<0>();                        // nothing may land after the CTA has left

  if (p.cluster) {
    cluster_merge(p, reinterpret_cast<const float*>(smem_attn + p.recs_off), R, b, h, warp, lane);
    return;
  }

  // the last CTA of this (request, kv head) merges the splits in order
  __syncthreads();                           // every thread's partial records come first
  if (threadIdx.x == 0) {
    const int prev = arrive_acq_rel(&p.counters[pair]);
    s_last = prev == p.n_splits;
    if (s_last) p.counters[pair] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  for (int r = warp; r < R; r += WARPS) {
    const int node = r / p.G, hq = h * p.G + r % p.G;
    const size_t qi = (static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq;
    const float* src = p.part + qi * (p.n_splits + 1) * rec;
    // lane s holds split s (n_splits + 1 <= 32): all partial headers, and
    // the outputs of the first 16 splits, are requested at once
    const int ns = p.n_splits + 1;
    const float ms = lane < ns ? __ldcg(src + lane * rec) : -INFINITY;
    const float ls = lane < ns ? __ldcg(src + lane * rec + 1) : 0.f;
    float first[16][4];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int d = lane + 32 * c;
        first[u][c] = (u < ns && d < dh) ? __ldcg(src + u * rec + 4 + d) : 0.f;
      }
    }
    const float M = warp_max(ms);
    const float wgt = ms == -INFINITY ? 0.f : __expf(ms - M);
    const float Lsum = warp_sum(wgt * ls);
    float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float ws = __shfl_sync(0xffffffffu, wgt, u);
#pragma unroll
      for (int c = 0; c < 4; ++c) o[c] = fmaf(ws, first[u][c], o[c]);
    }
    for (int s0 = 16; s0 < ns; s0 += 8) {
      float vals[8][4];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int s = s0 + u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int d = lane + 32 * c;
          vals[u][c] = (s < ns && d < dh) ? __ldcg(src + s * rec + 4 + d) : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float ws = __shfl_sync(0xffffffffu, wgt, (s0 + u) & 31);
#pragma unroll
        for (int c = 0; c < 4; ++c) o[c] = fmaf(ws, vals[u][c], o[c]);
      }
    }
    write_merged_row(p, b, node, hq, o, Lsum, lane);
  }
}

// ---- verification layer: tensor cores ----------------------------------------

// ---- warp-level bf16 tensor-core tiles (m16n8k16, fp32 accumulate) ---------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const uint16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(sm100::smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const uint16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(sm100::smem_u32(p)));
}
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (x, y) -> bf16x2 hi = RN(x, y) and lo = RN of the remainders; x in the low half
__device__ __forceinline__ void split_pair(float x, float y, uint32_t& hi, uint32_t& lo) {
  uint16_t xh, xl, yh, yl;
  split_bf16(x, xh, xl);
  split_bf16(y, yh, yl);
  hi = static_cast<uint32_t>(xh) | (static_cast<uint32_t>(yh) << 16);
  lo = static_cast<uint32_t>(xl) | (static_cast<uint32_t>(yl) << 16);
}

// Draft-tree keys k0 .. k0 + nt - 1 (fp32, at most TILE_F32) into buf as bf16
// hi / lo pairs: K hi [TILE_F32][KLD], K lo, then V hi at row TILE (the same
// place as a bf16 tile's V), V lo; rows past nt are zeroed.
__device__ __forceinline__ void stage_f32_split(uint16_t* buf, const float* kf, const float* vf, size_t row0,
                                                size_t row_stride, int nt, int dh) {
  const int pieces = dh >> 2;
  for (int idx = threadIdx.x; idx < TILE_F32 * pieces; idx += blockDim.x) {
    const int r = idx / pieces, c = idx - r * pieces;
    float4 k = make_float4(0.f, 0.f, 0.f, 0.f), v = k;
    if (r < nt) {
      k = __ldcg(reinterpret_cast<const float4*>(kf + row0 + r * row_stride + 4 * c));
      v = __ldcg(reinterpret_cast<const float4*>(vf + row0 + r * row_stride + 4 * c));
    }
    uint32_t h0, l0, h1, l1;
    const int o = r * KLD + 4 * c;
    split_pair(k.x, k.y, h0, l0);
    split_pair(k.z, k.w, h1, l1);
    *reinterpret_cast<uint2*>(buf + o) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(buf + TILE_F32 * KLD + o) = make_uint2(l0, l1);
    split_pair(v.x, v.y, h0, l0);
    split_pair(v.z, v.w, h1, l1);
    *reinterpret_cast<uint2*>(buf + TILE * KLD + o) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(buf + (TILE + TILE_F32) * KLD + o) = make_uint2(l0, l1);
  }
  cp_async_commit();                         // an empty group: one group per staged tile, as the others
}

// Online-softmax state of one warp: rows g and g + 8 of its 16-row tile
// (g = lane / 4), output columns 8 j + 2 (lane % 4) + {0, 1} of each 8-wide
// column tile j (the m16n8 accumulator layout).
struct WarpState {
  float m[2], l[2];
  float o[MAX_DH / 8][4];
};

// One warp, one staged tile: rows [16 mt, 16 mt + 16) of the pass against
// tile keys [k_lo, k_lo + 8 NKT).  S = Q K^T on the tensor cores (Q as bf16
// hi + lo when it is fp32; K hi + lo for the draft's fp32 tree keys), scale,
// mask (keys past nt; tree keys outside the row's ancestor set), online
// softmax in registers, then O += P V with P split into bf16 hi + lo taken
// straight from the score accumulators.
template <int NKT>
__device__ __forceinline__ void tile_mma(const AttnParams& p, WarpState& st, const uint16_t* buf, bool kv_lo,
                                         const uint16_t* qhi, const uint16_t* qlo, int mt, int k_lo, int nt,
                                         int key_base, bool is_tree, uint64_t mask_a, uint64_t mask_b, int lane) {
  const int dh = p.dh;
  const int tq = lane & 3;
  const uint16_t* sk = buf;
  const uint16_t* skl = buf + TILE_F32 * KLD;
  const uint16_t* sv = buf + TILE * KLD;
  const uint16_t* svl = buf + (TILE + TILE_F32) * KLD;
  float s[NKT][4];
#pragma unroll
  for (int j = 0; j < NKT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
  const int qrow = 16 * mt + (lane & 15), qcol = (lane >> 4) * 8;
  const int krow = k_lo + (lane & 7) + ((lane >> 4) << 3), kcol = ((lane >> 3) & 1) * 8;
  for (int kk = 0; kk < dh; kk += 16) {
    uint32_t a[4], al[4];
    ldsm_x4(a, qhi + qrow * KLD + kk + qcol);
    if (qlo != nullptr) ldsm_x4(al, qlo + qrow * KLD + kk + qcol);
#pragma unroll
    for (int j = 0; j < NKT; j += 2) {
      uint32_t bk[4];
      ldsm_x4(bk, sk + (krow + 8 * j) * KLD + kk + kcol);
      mma_bf16_16816(s[j], a, bk[0], bk[1]);
      mma_bf16_16816(s[j + 1], a, bk[2], bk[3]);
      if (qlo != nullptr) {
        mma_bf16_16816(s[j], al, bk[0], bk[1]);
        mma_bf16_16816(s[j + 1], al, bk[2], bk[3]);
      }
      if (kv_lo) {
        ldsm_x4(bk, skl + (krow + 8 * j) * KLD + kk + kcol);
        mma_bf16_16816(s[j], a, bk[0], bk[1]);
        mma_bf16_16816(s[j + 1], a, bk[2], bk[3]);
      }
    }
  }
  // scale and mask; the rows' maxima over this warp's keys (a quad shares a row)
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < NKT; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = k_lo + 8 * j + 2 * tq + (e & 1);
      const uint64_t mk = e < 2 ? mask_a : mask_b;
      const bool ok = key < nt && (!is_tree || ((mk >> (key_base + key)) & 1ull));
      s[j][e] = ok ? s[j][e] * p.scale : -INFINITY;
      mx[e >> 1] = fmaxf(mx[e >> 1], s[j][e]);
    }
  }
  float corr[2], sum[2] = {0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    const float m_new = fmaxf(st.m[r], mx[r]);
    corr[r] = m_new == -INFINITY ? 1.f : __expf(st.m[r] - m_new);
    mx[r] = m_new;
  }
#pragma unroll
  for (int j = 0; j < NKT; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float m_new = mx[e >> 1];
      const float pe = m_new == -INFINITY ? 0.f : __expf(s[j][e] - m_new);
      s[j][e] = pe;
      sum[e >> 1] += pe;
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 1);
    sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], 2);
    st.l[r] = st.l[r] * corr[r] + sum[r];
    st.m[r] = mx[r];
  }
#pragma unroll
  for (int j = 0; j < MAX_DH / 8; ++j) {
    st.o[j][0] *= corr[0];
    st.o[j][1] *= corr[0];
    st.o[j][2] *= corr[1];
    st.o[j][3] *= corr[1];
  }
  // O += P V, 16 keys per step: the score accumulators of column tiles 2q
  // and 2q + 1 are the A fragment of keys [16 q, 16 q + 16)
  const int vrow = k_lo + (lane & 7) + ((lane >> 3) & 1) * 8, vcol = (lane >> 4) * 8;
#pragma unroll
  for (int q = 0; q < NKT / 2; ++q) {
    uint32_t ah[4], alo[4];
    split_pair(s[2 * q][0], s[2 * q][1], ah[0], alo[0]);
    split_pair(s[2 * q][2], s[2 * q][3], ah[1], alo[1]);
    split_pair(s[2 * q + 1][0], s[2 * q + 1][1], ah[2], alo[2]);
    split_pair(s[2 * q + 1][2], s[2 * q + 1][3], ah[3], alo[3]);
#pragma unroll
    for (int j = 0; j < MAX_DH / 8; j += 2) {
      if (8 * j < dh) {
        uint32_t bv[4];
        ldsm_x4_t(bv, sv + (vrow + 16 * q) * KLD + 8 * j + vcol);
        mma_bf16_16816(st.o[j], ah, bv[0], bv[1]);
        mma_bf16_16816(st.o[j + 1], ah, bv[2], bv[3]);
        mma_bf16_16816(st.o[j], alo, bv[0], bv[1]);
        mma_bf16_16816(st.o[j + 1], alo, bv[2], bv[3]);
        if (kv_lo) {
          ldsm_x4_t(bv, svl + (vrow + 16 * q) * KLD + 8 * j + vcol);
          mma_bf16_16816(st.o[j], ah, bv[0], bv[1]);
          mma_bf16_16816(st.o[j + 1], ah, bv[2], bv[3]);
        }
      }
    }
  }
}

// st <- merge(st, the state stored at slot): the usual rescale to the
// larger maximum.
__device__ __forceinline__ void merge_state(WarpState& st, const float* slot, int dh, int lane) {
  const int g = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const float* row = slot + (g + 8 * r) * MLD;
    const float mb = row[MAX_DH], lb = row[MAX_DH + 1];
    const float m = fmaxf(st.m[r], mb);
    const float wa = m == -INFINITY ? 0.f : __expf(st.m[r] - m);
    const float wb = m == -INFINITY ? 0.f : __expf(mb - m);
    st.l[r] = st.l[r] * wa + lb * wb;
    st.m[r] = m;
#pragma unroll
    for (int j = 0; j < MAX_DH / 8; ++j) {
      if (8 * j < dh) {
        const float2 ob = *reinterpret_cast<const float2*>(row + 8 * j + 2 * tq);
        st.o[j][2 * r] = st.o[j][2 * r] * wa + ob.x * wb;
        st.o[j][2 * r + 1] = st.o[j][2 * r + 1] * wa + ob.y * wb;
      }
    }
  }
}

__device__ __forceinline__ void store_state(const WarpState& st, float* slot, int dh, int lane) {
  const int g = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float* row = slot + (g + 8 * r) * MLD;
    if (tq == 0) {
      row[MAX_DH] = st.m[r];
      row[MAX_DH + 1] = st.l[r];
    }
#pragma unroll
    for (int j = 0; j < MAX_DH / 8; ++j)
      if (8 * j < dh) *reinterpret_cast<float2*>(row + 8 * j + 2 * tq) = make_float2(st.o[j][2 * r], st.o[j][2 * r + 1]);
  }
}

// Dynamic shared memory: n_buf tile buffers (TILE_BYTES each) and the
// pass's query rows as bf16 hi [16 NW][KLD] and lo, whose space holds the
// warp states of the intra-CTA merge once the pass's tiles are done; at the
// end, the merging CTA reuses all of it to stage partial records.
//
// One CTA of NW warps per (prefix split or tree part, request, kv head):
// four warps at two CTAs per SM, or eight at one when a kv head has more
// than 32 query rows (fewer passes, each re-reading the split's tiles).  A
// pass covers up to 16 NW query rows (tree nodes x GQA group) as MT tiles of
// 16 (a power of two); the NW / MT warps of a row tile split every staged
// key tile between them,
// each keeping its own online softmax, and are merged (in a fixed order) at
// the end of the pass.  Prefix tiles are bf16 copied by cp.async (the next
// one streams in while the current one is consumed when a split holds
// several); the draft's fp32 tree keys are split into bf16 hi + lo as they
// are staged, 32 keys per tile.
template <int NW>
__global__ void __launch_bounds__(32 * NW, NW == 4 ? 2 : 1) tree_attn_mma_kernel(const AttnParams p) {
  constexpr int kThreads = 32 * NW;
  constexpr int kRows = mma_rows(NW);        // query rows per pass
  const LaunchStamp ls(p.stamp);
  pdl_trigger();
  extern __shared__ __align__(16) uint8_t smem_attn[];
  __shared__ int s_last;
  __shared__ uint64_t s_mask[kRows * MASKW];   // ancestor masks of the pass's rows (tree part)

  const int split = blockIdx.x;              // split == n_splits: the tree part
  const int pair = blockIdx.y;
  const int b = pair / p.Hkv, h = pair % p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dh = p.dh;
  uint8_t* bufs = smem_attn;
  uint16_t* qhi = reinterpret_cast<uint16_t*>(smem_attn + p.n_buf * TILE_BYTES);
  uint16_t* qlo = qhi + kRows * KLD;
  float* mrg = reinterpret_cast<float*>(qhi);   // after a pass's last tile, the query rows are dead
  const bool is_tree = split == p.n_splits;
  const bool tree_f32 = is_tree && p.mode == 0;
  // The prefix and its length are this round's inputs, written by no kernel
  // of the round: a prefix split's range and tiles are known (and its tiles
  // requested) before the dependency wait.  The tree part's size, the query
  // rows and the tree K/V come from the predecessors.
  int lo = 0, hi = 0;
  if (!is_tree) {
    const int L = prefix_rows(p, b, split == 0 && threadIdx.x == 0);
    lo = split * p.chunk;
    hi = min(L, lo + p.chunk);
  }
  const int rec = dh + 4;                    // partial record: max, sum, 2 unused, output[dh]
  const size_t row_stride = static_cast<size_t>(p.Hkv) * dh;
  const uint64_t policy = sm100::l2_policy_evict_first();
  const int step = tree_f32 ? TILE_F32 : TILE;

  auto stage = [&](int tile, int which) {
    uint16_t* buf = reinterpret_cast<uint16_t*>(bufs + which * TILE_BYTES);
    const int t0 = lo + tile * step, nt = min(step, hi - t0);
    if (tree_f32)
      stage_f32_split(buf, p.kt_f32, p.vt_f32, ((static_cast<size_t>(b) * p.tree_cap + t0) * p.Hkv + h) * dh,
                      row_stride, nt, dh);
    else if (is_tree)
      stage_bf16(buf, p.kt_bf16, p.vt_bf16, ((static_cast<size_t>(b) * p.tree_cap + t0) * p.Hkv + h) * dh,
                 row_stride, nt, dh, policy);
    else if (p.paged.table)
      stage_bf16_paged(buf, p, b, h, t0, nt, policy);
    else
      stage_bf16(buf, p.kp, p.vp, ((static_cast<size_t>(b) * p.kv_cap + t0) * p.Hkv + h) * dh, row_stride, nt, dh,
                 policy);
  };
  // tiles [0, staged) of the current pass have been requested; a split
  // whose tiles all fit the buffers stages them once for every pass
  int n_tiles = hi > lo ? (hi - lo + step - 1) / step : 0;
  int staged = 0;
  if (!is_tree) {
    for (; staged < n_tiles && staged < p.n_buf; ++staged) stage(staged, staged);
  }
  pdl_wait();                                // q rows, tree K/V, masks and the tree's size
  ls.waited();
  const int nodes = n_nodes(p, b);
  const int R = nodes * p.G;
  if (is_tree) {
    hi = p.mode == 0 ? p.tree_cap : min(p.tree_size[b], p.tree_cap);
    n_tiles = hi > lo ? (hi - lo + step - 1) / step : 0;
    for (; staged < n_tiles && staged < p.n_buf; ++staged) stage(staged, staged);
  }
  const bool resident = n_tiles <= p.n_buf;

  for (int r0 = 0; r0 < R; r0 += kRows) {
    const int rp = min(kRows, R - r0);
    int MT = 1;                              // 16-row tiles of the pass (a power of two)
    while (16 * MT < rp && MT < kRows / 16) MT <<= 1;
    const int KS = NW / MT;                  // warps sharing a row tile
    const int mt = warp % MT, ks = warp / MT;
    if (r0 > 0) {
      __syncthreads();                       // the previous pass is done with the query rows and buffers
      if (!resident) staged = 0;
    }
    // query rows of the pass as bf16 hi (+ lo for fp32 queries); rows past rp are zero
    for (int idx = threadIdx.x; idx < 16 * MT * (dh >> 2); idx += kThreads) {
      const int rr = idx / (dh >> 2), c = idx - rr * (dh >> 2);
      uint2 wh = make_uint2(0u, 0u), wl = make_uint2(0u, 0u);
      if (rr < rp) {
        const int r = r0 + rr, node = r / p.G, hq = h * p.G + r % p.G;
        const size_t qo = q_index(p, b, node, hq) + 4 * c;
        if (p.mode == 0) {
          const float4 v = *reinterpret_cast<const float4*>(p.q_f32 + qo);
          split_pair(v.x, v.y, wh.x, wl.x);
          split_pair(v.z, v.w, wh.y, wl.y);
        } else {
          wh = *reinterpret_cast<const uint2*>(p.q_bf16 + qo);
        }
      }
      *reinterpret_cast<uint2*>(qhi + rr * KLD + 4 * c) = wh;
      if (p.mode == 0) *reinterpret_cast<uint2*>(qlo + rr * KLD + 4 * c) = wl;
    }
    if (is_tree && threadIdx.x < kRows) {
      if (threadIdx.x < rp) {
        load_row_mask(p, s_mask + threadIdx.x * MASKW, b, (r0 + threadIdx.x) / p.G);
      } else {
#pragma unroll
        for (int w = 0; w < MASKW; ++w) s_mask[threadIdx.x * MASKW + w] = 0ull;
      }
    }
    WarpState st;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
#pragma unroll
    for (int j = 0; j < MAX_DH / 8; ++j) st.o[j][0] = st.o[j][1] = st.o[j][2] = st.o[j][3] = 0.f;
    for (int tile = 0; tile < n_tiles; ++tile) {
      // a ring of n_buf buffers: tile t in buffer t % n_buf, up to n_buf
      // tiles requested ahead; the buffer refilled here held the tile that
      // the previous iteration consumed
      const int which = tile % p.n_buf;
      if (staged < n_tiles && staged < tile + p.n_buf) {
        __syncthreads();                     // every warp is done with the buffers being refilled
        for (; staged < n_tiles && staged < tile + p.n_buf; ++staged) stage(staged, staged % p.n_buf);
      }
      cp_async_wait_upto(staged - tile - 1);   // this tile's copies have landed (later ones may fly)
      __syncthreads();
      const int t0 = lo + tile * step;
      const int nt = min(step, hi - t0);
      const int kpw = max(16, step / KS);    // keys per warp: 16, 32 or 64
      const int k_lo = ks * kpw;
      if (k_lo < nt) {
        const uint16_t* buf = reinterpret_cast<const uint16_t*>(bufs + which * TILE_BYTES);
        // a tree tile lies in one mask word (it starts at a multiple of its size)
        const int mw = is_tree ? (t0 >> 6) : 0;
        const uint64_t ma = is_tree ? s_mask[(16 * mt + (lane >> 2)) * MASKW + mw] : ~0ull;
        const uint64_t mb = is_tree ? s_mask[(16 * mt + (lane >> 2) + 8) * MASKW + mw] : ~0ull;
        const uint16_t* ql = p.mode == 0 ? qlo : nullptr;
        const int kb = is_tree ? (t0 & 63) : 0;
        if (kpw == 16) {
          tile_mma<2>(p, st, buf, tree_f32, qhi, ql, mt, k_lo, nt, kb, is_tree, ma, mb, lane);
        } else if (kpw == 32) {
          tile_mma<4>(p, st, buf, tree_f32, qhi, ql, mt, k_lo, nt, kb, is_tree, ma, mb, lane);
        } else {
          // 64 keys per warp: one warp per row tile, which only the
          // eight-warp kernel's 128-row passes produce
          if constexpr (kRows / 16 == NW)
            tile_mma<8>(p, st, buf, tree_f32, qhi, ql, mt, k_lo, nt, kb, is_tree, ma, mb, lane);
        }
      }
    }
    // merge the KS warps of each row tile pairwise, in a fixed order
    for (int d = 1; d < KS; d <<= 1) {
      __syncthreads();
      const int slot = mt + MT * (ks / (2 * d));          // < NW / 2
      if (ks % (2 * d) == d) store_state(st, mrg + slot * 16 * MLD, dh, lane);
      __syncthreads();
      if (ks % (2 * d) == 0) merge_state(st, mrg + slot * 16 * MLD, dh, lane);
    }
    if (ks == 0) {
      const int g = lane >> 2, tq = lane & 3;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int rr = 16 * mt + g + 8 * r;
        if (rr >= rp) continue;
        const int row = r0 + rr, node = row / p.G, hq = h * p.G + row % p.G;
        const size_t qi = (static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq;
        float* dst = p.cluster ? reinterpret_cast<float*>(smem_attn + p.recs_off) + static_cast<size_t>(row) * rec
                               : p.part + (qi * (p.n_splits + 1) + split) * rec;
        if (tq == 0) {
          dst[0] = st.m[r];
          dst[1] = st.l[r];
        }
#pragma unroll
        for (int j = 0; j < MAX_DH / 8; ++j)
          if (8 * j < dh)
            *reinterpret_cast<float2*>(dst + 4 + 8 * j + 2 * tq) = make_float2(st.o[j][2 * r], st.o[j][2 * r + 1]);
      }
    }
  }
  cp_async_wait<0>();                        // nothing may land after the CTA has left

  if (p.cluster) {
    cluster_merge(p, reinterpret_cast<const float*>(smem_attn + p.recs_off), R, b, h, warp, lane);
    return;
  }

  // the last CTA of this (request, kv head) merges the splits in order
  __syncthreads();                           // every thread's partial records come first
  if (threadIdx.x == 0) {
    const int prev = arrive_acq_rel(&p.counters[pair]);
    s_last = prev == p.n_splits;
    if (s_last) p.counters[pair] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  // Every record of a batch of rows is copied into shared memory at once
  // (16-byte asynchronous copies: a row's ns records are contiguous), then a
  // warp per row merges from shared memory: lane s < ns holds split s's
  // header, lane c sums columns c + 32 i.
  const int ns = p.n_splits + 1;
  float* stg = reinterpret_cast<float*>(smem_attn);
  const int row_floats = ns * rec;
  const size_t smem_floats = (p.n_buf * TILE_BYTES + q_bytes(NW)) / sizeof(float);
  const int batch = max(1, static_cast<int>(smem_floats / row_floats));
  for (int rb = 0; rb < R; rb += batch) {
    const int nb = min(batch, R - rb);
    __syncthreads();                         // the previous batch is merged
    for (int i = 0; i < nb; ++i) {
      const int r = rb + i, node = r / p.G, hq = h * p.G + r % p.G;
      const size_t qi = (static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq;
      const float* src = p.part + qi * ns * rec;
      for (int k = 4 * threadIdx.x; k < row_floats; k += 4 * kThreads) cp_async16_cg(stg + i * row_floats + k, src + k);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    for (int i = warp; i < nb; i += NW) {
      const int r = rb + i, node = r / p.G, hq = h * p.G + r % p.G;
      const float* srow = stg + i * row_floats;
      const float ms = lane < ns ? srow[lane * rec] : -INFINITY;
      const float ls = lane < ns ? srow[lane * rec + 1] : 0.f;
      const float M = warp_max(ms);
      const float wgt = ms == -INFINITY ? 0.f : __expf(ms - M);
      const float Lsum = warp_sum(wgt * ls);
      float o[4] = {0.f, 0.f, 0.f, 0.f};
      for (int s = 0; s < ns; ++s) {
        const float ws = __shfl_sync(0xffffffffu, wgt, s);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int d = lane + 32 * c;
          if (d < dh) o[c] = fmaf(ws, srow[s * rec + 4 + d], o[c]);
        }
      }
      write_merged_row(p, b, node, hq, o, Lsum, lane);
    }
  }
  cp_async_wait<0>();
}


// ---- tcgen05 attention with warp roles (dh 128) -------------------------------
//
// One CTA of 640 threads per (prefix split, block of 128 query rows, request
// and kv head); the last split also takes the tree part, its online softmax
// continuing over the tree keys.  Roles:
//   warps 0-1   loaders, warp 0 of every tile's K and warp 1 of its V, each
//               with its own ring barriers: K is released when S has been
//               computed, V when P V has, so the K stream runs a whole ring
//               ahead of S (one ring for both measured load-latency bound).
//               A whole prefix tile comes by TMA (boxes of 64 dims x 64 keys,
//               or x one block of a paged prefix); a partial tile, a tile
//               with an unallocated block and the verification tree's tiles
//               by 16-byte asynchronous copies with the missing rows zeroed;
//               the draft tree's fp32 keys and values as bf16 hi + lo pairs,
//               32 keys a tile.
//   warps 2-3   MMA issuers, one thread each (warp 2 for the even tiles,
//               warp 3 for the odd ones -- one issuer measured starved of
//               issue slots by the busy softmax warps): S = Q K^T into the
//               group's S buffer in tensor memory, O += P V with P read from
//               tensor memory.
//   warps 4-19  softmax, four warpgroups: thread = query row = its tensor-
//               memory lane (warp % 4 selects the 32-lane quarter), and
//               warpgroup g takes quarter g of each tile's keys: its partial
//               row maximum, exchanged with the other three through shared
//               memory (one barrier of the softmax warps a tile); P = 2^(s c
//               - m) (c = scale log2 e) of its keys as bf16 hi + lo into
//               tensor memory; its share of the row sum; quarter g of O's
//               columns when O is rescaled and at the end.
// Warps whose 32 rows all lie past a block's rows (a few-row draft layer)
// only keep the barrier protocol.
// The four warpgroups (rather than two taking all of a row's keys each) hide
// the latency of the per-tile chain -- tensor-memory load, maximum,
// exponentials, hi / lo split, tensor-memory store -- measured as the limit.
// P is relative to a per-row reference maximum m (log2 units), raised -- O
// and the sums rescaled in place -- only when a tile's maximum passes it by
// more than WS_RESCALE (natural units): P stays below e^WS_RESCALE and O / l
// does not depend on when m was raised.  Pipelining: K / V stages in a ring
// (kv_full / kv_empty barriers); S double-buffered, so S(t + 1) is ready
// while the softmax of tile t runs, and S(t + 2) is issued as soon as that
// softmax has loaded S(t) (s_free), before P(t) V(t); P double-buffered; O
// accumulating in tensor memory over all tiles.  Draft rows (fp32 queries) enter S as hi + lo: S = Qhi K +
// Qlo K; the draft tree's keys as hi + lo too: S = Qhi Khi + Qlo Khi + Qhi
// Klo and O += Phi Vhi + Plo Vhi + Phi Vlo.
// Shared-memory operands use the 128-byte swizzle (1024-byte atoms of 8 rows
// x 128 bytes, 16-byte chunk j of row r at chunk j ^ (r % 8)): Q as two
// k-blocks [128 rows][64 dims] (draft: hi, then lo); a ring stage as K [64
// keys][64 dims] x 2 halves, then V alike -- what TMA writes for boxes of 64
// dims x 64 keys -- K being the K-major B operand of Q K^T and V the MN-major
// B operand of P V; a draft-tree stage as K hi, K lo, V hi, V lo of 32 keys.
constexpr int WS_LOAD_WARPS = 2;
constexpr int WS_MMA_WARP = 2;                      // and 3
constexpr int WS_SOFT_WARP0 = 4;
constexpr int WS_SOFT_WGS = 4;                      // softmax warpgroups
constexpr int WS_GROUP_WGS = 2;                     // ... in two groups of two, a group for every other tile
constexpr int WS_GROUP_THREADS = 128 * WS_GROUP_WGS;
constexpr int WS_THREADS = 32 * (WS_SOFT_WARP0 + 4 * WS_SOFT_WGS);
constexpr int WS_SOFT_THREADS = 128 * WS_SOFT_WGS;
constexpr int WS_ROWS = 128;
constexpr int WS_KEYS = 64;                         // keys per prefix / verification-tree tile
constexpr int WS_FKEYS = 32;                        // keys per draft-tree tile
constexpr int WS_DH = 128;
constexpr uint32_t WS_STAGE = 32768;                // one ring stage: K then V
constexpr uint32_t WS_HALF = 8192;                  // 64 keys x 64 dims of bf16
constexpr uint32_t WS_FHALF = 4096;                 // 32 keys x 64 dims of bf16
constexpr uint32_t WS_QHALF = 16384;                // 128 rows x 64 dims of bf16
constexpr uint32_t WS_BUDGET = 196608;              // Q + ring stages
constexpr int WS_MAX_STAGES = 5;
constexpr size_t WS_SMEM = WS_BUDGET + 1024;        // + room to align the base to 1024 bytes
constexpr float WS_RESCALE = 8.0f;
constexpr float WS_LOG2E = 1.4426950408889634f;
constexpr int WS_MAX_RECS = 16;                     // prefix splits of a (request, kv head) at most
constexpr uint32_t WS_TM_S = 0;                     // S of group 0 / 1: columns 0 / 64
constexpr uint32_t WS_TM_O = 128;                   // O of group 0 / 1: columns 128-255 / 384-511
constexpr uint32_t WS_TM_O_STEP = 256;
constexpr uint32_t WS_TM_P = 256;                   // P of group 0 / 1: 256 / 320 (hi, then lo 32 columns on)
constexpr uint32_t WS_TM_COLS = 512;
constexpr int WS_BAR_SOFT = 1;                      // named barriers: all softmax warps, then one per group
constexpr int WS_BAR_GROUP = 2;

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a swizzled
// block of 128-byte rows.
__device__ __forceinline__ uint32_t ws_sw(int row, int chunk) {
  return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}
// 32 lanes x 32 consecutive 32-bit columns (thread i: lane quarter * 32 + i).
__device__ __forceinline__ void ws_tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void ws_tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 lanes x 4 consecutive 32-bit columns, stored.
__device__ __forceinline__ void ws_tmem_st4(uint32_t taddr, const uint32_t (&w)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3])
               : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns, stored.
__device__ __forceinline__ void ws_tmem_st8(uint32_t taddr, const uint32_t (&w)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns, stored.
__device__ __forceinline__ void ws_tmem_st16(uint32_t taddr, const uint32_t (&w)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
               : "memory");
}
// Shared-memory descriptors as two 32-bit words.  The high word (8-row group
// stride 1024 bytes, version 1, 128-byte swizzle) is the same for every
// operand here; the low word is (address >> 4) | (leading byte offset >> 4)
// << 16, so an operand that many bytes on is the low word plus (bytes >> 4)
// (the address field never carries: operands end below 256 KB).
constexpr uint32_t WS_DESC_HI = (1024u >> 4) | (1u << 14) | (2u << 29);
__device__ __forceinline__ uint32_t ws_desc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr >> 4) & 0x3FFFu) | ((lbo >> 4) << 16);
}
// The two MMA forms from 32-bit descriptor words; `acc` false only for the
// first MMA of an accumulation.
__device__ __forceinline__ void ws_mma_ss32(uint32_t d_tmem, uint32_t alo, uint32_t blo, uint32_t hi, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 a, b;\n setp.ne.b32 p, %5, 0;\n mov.b64 a, {%1, %3};\n mov.b64 b, {%2, %3};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(alo), "r"(blo), "r"(hi), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void ws_mma_ts32(uint32_t d_tmem, uint32_t a_tmem, uint32_t blo, uint32_t hi, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 b;\n setp.ne.b32 p, %5, 0;\n mov.b64 b, {%2, %3};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(blo), "r"(hi), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ float ws_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (x, y) -> bf16x2 hi = RN(x, y) and lo = RN of the remainders, x in the low
// half (the same values as split_pair, two conversions per pair).
__device__ __forceinline__ void ws_split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Tile t of a CTA: prefix tiles of the split first, then (last split) the
// tree's.  k0 = its first key (prefix position or tree slot), nk = its keys.
struct WsTiles {
  int lo, hi, n_pre, tree_keys, n;
  bool draft;
  __device__ __forceinline__ void at(int t, bool& tree, bool& f32, int& k0, int& nk) const {
    tree = t >= n_pre;
    f32 = draft && tree;
    if (tree) {
      const int kt = draft ? WS_FKEYS : WS_KEYS;
      k0 = (t - n_pre) * kt;
      nk = min(kt, tree_keys - k0);
    } else {
      k0 = lo + t * WS_KEYS;
      nk = min(WS_KEYS, hi - k0);
    }
  }
};

// Whether prefix tile [k0, k0 + 64) may come by TMA: the launch has tensor
// maps, the tile is whole, and every block of a paged prefix it spans exists.
__device__ __forceinline__ bool ws_tma_ok(const AttnParams& p, int b, int k0, int nk) {
  if (!p.tma || nk != WS_KEYS) return false;
  if (!p.paged.table) return true;
  for (int r = 0; r < WS_KEYS; r += p.box_rows) {
    const int blk = p.paged.table[static_cast<size_t>(b) * p.paged.per_req + ((k0 + r) >> p.paged.shift)];
    if (blk < 0 || blk >= p.paged.n_blocks) return false;
  }
  return true;
}
// Requests half `m` (0: K, 1: V) of prefix tile [k0, k0 + 64) of kv head h
// into its place in stage `st` (one thread).
__device__ __forceinline__ void ws_tma_half(const AttnParams& p, const CUtensorMap* map, uint8_t* st, uint64_t* bar,
                                            int m, int b, int h, int k0) {
  sm100::mbar_arrive_expect_tx(bar, WS_STAGE / 2);
  for (int r = 0; r < WS_KEYS; r += p.box_rows) {
    const int row = p.paged.table ? static_cast<int>(paged_row(p.paged, b, k0 + r)) : b * p.kv_cap + k0 + r;
#pragma unroll
    for (int half = 0; half < 2; ++half)
      sm100::tma_load_3d(st + m * 2 * WS_HALF + half * WS_HALF + r * 128, map, 64 * half, h, row, bar);
  }
}
// Half m (0: K, 1: V) of a bf16 tile by 16-byte asynchronous copies (one
// warp): prefix keys (through the block table when paged; a row of an
// unallocated block is zero and reported) or verification-tree keys; rows
// past nk are zero.  Returns once the copies have landed.
__device__ __forceinline__ void ws_copy_half(const AttnParams& p, uint8_t* st, int m, int b, int h, bool tree, int k0,
                                             int nk, int lane) {
  const uint16_t* src_base = m == 0 ? (tree ? p.kt_bf16 : p.kp) : (tree ? p.vt_bf16 : p.vp);
  uint8_t* dst = st + m * 2 * WS_HALF;
  for (int idx = lane; idx < WS_KEYS * 16; idx += 32) {
    const int key = idx >> 4, c = idx & 15;
    const uint32_t off = (c >> 3) * WS_HALF + ws_sw(key, c & 7);
    long long row = -1;
    if (key < nk) {
      if (tree) {
        row = static_cast<long long>(b) * p.tree_cap + k0 + key;
      } else if (p.paged.table) {
        row = paged_row(p.paged, b, k0 + key);
        if (row < 0 && c == 0 && m == 0) set_status(p.status, EAGLE_ERR_INVALID_ARG);
      } else {
        row = static_cast<long long>(b) * p.kv_cap + k0 + key;
      }
    }
    if (row >= 0)
      cp_async16_cg(dst + off, src_base + (static_cast<size_t>(row) * p.Hkv + h) * WS_DH + 8 * c);
    else
      *reinterpret_cast<uint4*>(dst + off) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_async_commit();
  cp_async_wait<0>();
}
// Half m (0: K, 1: V) of a draft-tree tile (one warp): fp32 rows k0 .. k0 +
// nk - 1 (nk <= 32) as bf16 hi then lo, each two 4 KB dim halves of 32 rows.
__device__ __forceinline__ void ws_split_half(const AttnParams& p, uint8_t* st, int m, int b, int h, int k0, int nk,
                                              int lane) {
  constexpr int PER = WS_FKEYS * 16 / 32;    // 8-dim chunks per lane
  constexpr int BATCH = 4;
  static_assert(PER % BATCH == 0, "whole batches");
  const float* src_base = m == 0 ? p.kt_f32 : p.vt_f32;
  uint8_t* dst = st + m * 2 * WS_HALF;
  for (int i0 = 0; i0 < PER; i0 += BATCH) {
    float4 x[BATCH][2];
#pragma unroll
    for (int i = 0; i < BATCH; ++i) {
      const int idx = lane + 32 * (i0 + i);
      const int key = idx >> 4, c = idx & 15;
      x[i][0] = x[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (key < nk) {
        const size_t src = ((static_cast<size_t>(b) * p.tree_cap + k0 + key) * p.Hkv + h) * WS_DH + 8 * c;
        x[i][0] = __ldcg(reinterpret_cast<const float4*>(src_base + src));
        x[i][1] = __ldcg(reinterpret_cast<const float4*>(src_base + src + 4));
      }
    }
#pragma unroll
    for (int i = 0; i < BATCH; ++i) {
      const int idx = lane + 32 * (i0 + i);
      const int key = idx >> 4, c = idx & 15;
      const uint32_t off = (c >> 3) * WS_FHALF + ws_sw(key, c & 7);
      const float4 a = x[i][0], z = x[i][1];
      uint4 hi, lo;
      ws_split2(a.x, a.y, hi.x, lo.x);
      ws_split2(a.z, a.w, hi.y, lo.y);
      ws_split2(z.x, z.y, hi.z, lo.z);
      ws_split2(z.z, z.w, hi.w, lo.w);
      *reinterpret_cast<uint4*>(dst + off) = hi;
      *reinterpret_cast<uint4*>(dst + WS_HALF + off) = lo;
    }
  }
}

// Waits (every lane of the warp) for the phase of `bar` with the given
// parity; the result is the same in every lane.
__device__ __forceinline__ bool ws_warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = sm100::mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// The softmax of one tile t (KT keys) of group G = t % 2 for this thread's
// row and its warpgroup's half w of the keys: see the kernel's description.
// `full`: every key visible (a whole prefix tile); otherwise key j is
// visible when j < nk and bit j of mk is set.  The row maximum is the larger
// of the group's two warpgroups' partial maxima, exchanged through s_pmax
// [group][2][2][128] with one barrier of the group's warps; every thread of
// the group calls this once per tile of the group, `work` false after an
// abort (the barrier is still passed, nothing else done) and `rows` false
// for a warp none of whose rows the block has (barrier and arrivals only).
// Returns false when a wait gave up.
template <int KT>
__device__ __forceinline__ bool ws_softmax_tile(bool work, bool rows, uint32_t tmem, uint32_t lane_base, int t, int w,
                                                int row, bool full, uint64_t mk, int nk, float c, float& m_ref,
                                                float& l_part, uint64_t* o_done, uint64_t* s_free, float* s_pmax,
                                                volatile int* abort) {
  constexpr int KPT = KT / WS_GROUP_WGS;     // this thread's keys: 32 of 64 or 16 of 32
  const int G = t & 1, u = t >> 1;           // the group and its own tile count
  const int j0 = KPT * w;
  float sv[KPT];
  // With c > 0 the maximum is taken over the raw scores and the scale enters
  // with the exponent (one FFMA per key); otherwise the scores are scaled
  // first.  Invisible keys are -inf.
  const bool pos = c > 0.f;
  const float ec = pos ? c : 1.f;
  float pm = -INFINITY;
  if (work && !rows) {
    // a warp whose 32 rows all lie past the block's: it only keeps the
    // barrier protocol (its P stays unwritten: those O rows are never read)
    __syncwarp();
    if ((threadIdx.x & 31) == 0) sm100::mbar_arrive(&s_free[G]);
  }
  if (work && rows) {
    if constexpr (KPT == 32) {
      ws_tmem_ld32(tmem + WS_TM_S + 64u * G + lane_base + j0, sv);
    } else {
      ws_tmem_ld16(tmem + WS_TM_S + 64u * G + lane_base + j0, sv);
    }
    sm100::tmem_wait_ld();
    // this warp is done with S buffer G: S(t + 2) may be issued into it
    sm100::tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) sm100::mbar_arrive(&s_free[G]);
    if (!pos) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) sv[j] *= c;
    }
    if (!full) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) sv[j] = (j0 + j < nk && ((mk >> (j0 + j)) & 1ull)) ? sv[j] : -INFINITY;
    }
    float mx[4];                             // four independent chains
#pragma unroll
    for (int i = 0; i < 4; ++i) mx[i] = sv[i];
#pragma unroll
    for (int j = 4; j < KPT; ++j) mx[j & 3] = fmaxf(mx[j & 3], sv[j]);
    pm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
  }
  float* pmx = s_pmax + ((G * 2 + (u & 1)) * WS_GROUP_WGS) * WS_ROWS;
  pmx[w * WS_ROWS + row] = pm;
  if (G) sm100::named_barrier(WS_BAR_GROUP + 1, WS_GROUP_THREADS);
  else sm100::named_barrier(WS_BAR_GROUP, WS_GROUP_THREADS);
  if (!work || !rows) return true;
  const float mt = fmaxf(pmx[row], pmx[WS_ROWS + row]) * ec;   // the tile's maximum, log2 units
  const bool raise = mt > m_ref + WS_RESCALE * WS_LOG2E || (m_ref == -INFINITY && mt != -INFINITY);
  const bool rescale = raise && m_ref != -INFINITY;
  // P V of the group's previous tile t - 2 is done with O_G and with P buffer G
  if (t >= 2 && !ws_warp_wait(&o_done[G], static_cast<uint32_t>((u - 1) & 1), abort)) return false;
  if (__any_sync(0xffffffffu, rescale)) {
    // O_G of the warp's rows times 2^(m_old - m_new) (a finite reference
    // comes from an earlier tile of the group); this warpgroup's half of the columns
    sm100::tc_fence_after();
    const float f = rescale ? ws_exp2(m_ref - mt) : 1.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float v16[16];
      const uint32_t ta = tmem + WS_TM_O + WS_TM_O_STEP * G + lane_base + 64 * w + 16 * q;
      ws_tmem_ld16(ta, v16);
      sm100::tmem_wait_ld();
      uint32_t x[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) x[j] = __float_as_uint(v16[j] * f);
      ws_tmem_st16(ta, x);
    }
    sm100::tmem_wait_st();
    if (rescale) l_part *= f;
  }
  if (raise) m_ref = mt;
  const float nm = m_ref == -INFINITY ? 0.f : -m_ref;   // (with m = -inf every key is -inf: P = 0)
  float part[2] = {0.f, 0.f};
  // keys j0 .. j0 + KPT - 1 are P columns j0 / 2 .. (two bf16 a column), hi then lo 32 columns on
  const uint32_t pcol = tmem + WS_TM_P + 64u * G + lane_base + j0 / 2;
  uint32_t hw[KPT / 2], lw[KPT / 2];
#pragma unroll
  for (int i = 0; i < KPT / 2; ++i) {
    const float e0 = ws_exp2(fmaf(sv[2 * i], ec, nm)), e1 = ws_exp2(fmaf(sv[2 * i + 1], ec, nm));
    part[0] += e0;
    part[1] += e1;
    ws_split2(e0, e1, hw[i], lw[i]);
  }
  l_part += part[0] + part[1];
  if constexpr (KPT == 32) {
    ws_tmem_st16(pcol, hw);
    ws_tmem_st16(pcol + 32, lw);
  } else {
    ws_tmem_st8(pcol, hw);
    ws_tmem_st8(pcol + 32, lw);
  }
  sm100::tmem_wait_st();
  return true;
}

__global__ void __launch_bounds__(WS_THREADS, 1)
    tree_attn_ws_kernel(const AttnParams p, const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap) {
  const LaunchStamp ls(p.stamp);
  extern __shared__ uint8_t smem_ws_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_ws_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  // per stage and half (0: K, 1: V): loaded / released by its MMAs
  __shared__ uint64_t s_full[2][WS_MAX_STAGES], s_empty[2][WS_MAX_STAGES];
  __shared__ uint64_t s_s_full[2], s_s_free[2], s_p_full[2], s_o_done[2], s_mma_done[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_never, s_pre, s_last;
  __shared__ uint64_t s_mask[WS_ROWS * MASKW];
  __shared__ float s_m[2][WS_ROWS], s_l[2][WS_GROUP_WGS][WS_ROWS];
  __shared__ float s_pmax[2 * 2 * WS_GROUP_WGS * WS_ROWS];

  const int split = blockIdx.x, rb = blockIdx.y, pair = blockIdx.z;
  const int b = pair / p.Hkv, h = pair % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool draft = p.mode == 0;
  const int NST = p.stages;
  const uint32_t q_bytes = draft ? 4 * WS_QHALF : 2 * WS_QHALF;
  uint8_t* ring = sm + q_bytes;
  volatile int* abort_flag = &s_abort;
  volatile int* never = &s_never;

  WsTiles T;
  T.draft = draft;
  {
    const int L = prefix_rows(p, b, split == 0 && rb == 0 && tid == 0);
    T.lo = split * p.chunk;
    T.hi = min(L, T.lo + p.chunk);
  }
  T.n_pre = T.hi > T.lo ? (T.hi - T.lo + WS_KEYS - 1) / WS_KEYS : 0;
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      for (int m = 0; m < 2; ++m) {
        sm100::mbar_init(&s_full[m][s], 1);
        sm100::mbar_init(&s_empty[m][s], 1);
      }
    }
    for (int i = 0; i < 2; ++i) {
      sm100::mbar_init(&s_s_full[i], 1);
      sm100::mbar_init(&s_s_free[i], 4 * WS_GROUP_WGS);   // one arrival per warp of group i
      sm100::mbar_init(&s_p_full[i], 4 * WS_GROUP_WGS);
      sm100::mbar_init(&s_o_done[i], 1);
    }
    sm100::mbar_init(&s_mma_done[0], 1);
    sm100::mbar_init(&s_mma_done[1], 1);
    s_abort = 0;
    s_never = 0;
    sm100::fence_barrier_init();
    // The prefix is this round's input, written by no kernel of the round:
    // the split's first whole tiles are requested before the dependency wait.
    int pre = 0;
    for (; pre < min(NST, T.n_pre); ++pre) {
      const int k0 = T.lo + pre * WS_KEYS;
      if (!ws_tma_ok(p, b, k0, min(WS_KEYS, T.hi - k0))) break;
      ws_tma_half(p, &kmap, ring + pre * WS_STAGE, &s_full[0][pre], 0, b, h, k0);
      ws_tma_half(p, &vmap, ring + pre * WS_STAGE, &s_full[1][pre], 1, b, h, k0);
    }
    s_pre = pre;
  }
  pdl_wait();                                // q rows, tree K/V, masks and the tree's size
  ls.waited();
  const int R = n_nodes(p, b) * p.G;
  const int r0 = rb * WS_ROWS;
  const int rows_here = max(0, min(WS_ROWS, R - r0));
  const bool last_split = split == p.n_splits - 1;
  T.tree_keys = !last_split ? 0
                            : (draft ? min(p.e0 + p.rows_cap, p.tree_cap) : min(p.tree_size[b], p.tree_cap));
  const int n_tree = (T.tree_keys + (draft ? WS_FKEYS : WS_KEYS) - 1) / (draft ? WS_FKEYS : WS_KEYS);
  T.n = rows_here > 0 ? T.n_pre + n_tree : 0;
  const int n_tiles = T.n;

  // Tensor memory only after the wait (every kernel this one waits for has
  // finished), and dependents start only once every CTA holds its columns.
  if (warp == WS_MMA_WARP) {
    sm100::tmem_alloc(&s_tmem, WS_TM_COLS);
    sm100::tmem_relinquish();
  }
  if (warp >= WS_SOFT_WARP0 && n_tiles > 0) {
    // the block's query rows (rows past the block's: zero), then the masks
    const int st = tid - 32 * WS_SOFT_WARP0;
    for (int idx = st; idx < WS_ROWS * 16; idx += WS_SOFT_THREADS) {
      const int rr = idx >> 4, c = idx & 15;
      const uint32_t off = (c >> 3) * WS_QHALF + ws_sw(rr, c & 7);
      uint4 vh = make_uint4(0u, 0u, 0u, 0u), vl = vh;
      if (rr < rows_here) {
        const int r = r0 + rr, node = r / p.G, hq = h * p.G + r % p.G;
        const size_t qo = q_index(p, b, node, hq) + 8 * c;
        if (draft) {
          const float4 a = *reinterpret_cast<const float4*>(p.q_f32 + qo);
          const float4 z = *reinterpret_cast<const float4*>(p.q_f32 + qo + 4);
          ws_split2(a.x, a.y, vh.x, vl.x);
          ws_split2(a.z, a.w, vh.y, vl.y);
          ws_split2(z.x, z.y, vh.z, vl.z);
          ws_split2(z.z, z.w, vh.w, vl.w);
        } else {
          vh = *reinterpret_cast<const uint4*>(p.q_bf16 + qo);
        }
      }
      *reinterpret_cast<uint4*>(sm + off) = vh;
      if (draft) *reinterpret_cast<uint4*>(sm + 2 * WS_QHALF + off) = vl;
    }
    if (n_tree > 0 && st < WS_ROWS) {
      if (st < rows_here) {
        load_row_mask(p, s_mask + st * MASKW, b, (r0 + st) / p.G);
      } else {
#pragma unroll
        for (int w = 0; w < MASKW; ++w) s_mask[st * MASKW + w] = 0ull;
      }
    }
    sm100::fence_proxy_async_smem();         // generic-proxy stores -> tensor-core reads
  }
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  pdl_trigger();
  const uint32_t tmem = s_tmem;
  const uint32_t sbase = sm100::smem_u32(sm);
  const uint32_t rbase = sbase + q_bytes;

  constexpr int OC = WS_DH / WS_SOFT_WGS;     // output columns per softmax thread
  float o[OC];
#pragma unroll
  for (int j = 0; j < OC; ++j) o[j] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  const int sw = warp - WS_SOFT_WARP0;       // softmax warp
  const int grp = sw >> 3, w = (sw >> 2) & 1, quarter = warp & 3;
  const int c0 = OC * (2 * w + grp);          // this thread's output columns
  const int row = quarter * 32 + lane;

  if (warp < WS_LOAD_WARPS) {
    // ---- loaders: warp 0 the K halves, warp 1 the V halves, each a ring ahead ----
    const int m = warp;
    const CUtensorMap* map = m == 0 ? &kmap : &vmap;
    int t = s_pre;
    for (; t < n_tiles; ++t) {
      const int s = t % NST;
      bool ok = true;
      if (lane == 0 && t >= NST)
        ok = sm100::mbar_wait(&s_empty[m][s], static_cast<uint32_t>((t / NST - 1) & 1), abort_flag);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
        if (lane == 0) {
          set_status(p.status, EAGLE_ERR_TIMEOUT);
          s_abort = 1;
        }
        break;
      }
      bool tree, f32;
      int k0, nk;
      T.at(t, tree, f32, k0, nk);
      if (!tree && ws_tma_ok(p, b, k0, nk)) {          // the same decision in every lane
        if (lane == 0) ws_tma_half(p, map, ring + s * WS_STAGE, &s_full[m][s], m, b, h, k0);
      } else {
        if (f32) ws_split_half(p, ring + s * WS_STAGE, m, b, h, k0, nk, lane);
        else ws_copy_half(p, ring + s * WS_STAGE, m, b, h, tree, k0, nk, lane);
        sm100::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(&s_full[m][s]);
      }
    }
    // no TMA copy may still be landing when the CTA leaves
    const int issued = max(t, s_pre);
    if (lane == 0)
      for (int u = max(0, issued - NST); u < issued; ++u)
        sm100::mbar_wait(&s_full[m][u % NST], static_cast<uint32_t>((u / NST) & 1), never);
  } else if (warp == WS_MMA_WARP || warp == WS_MMA_WARP + 1) {
    // ---- MMA issuers: lane 0 of warp 2 for the even tiles (softmax group 0),
    // of warp 3 for the odd ones (group 1) ----
    const int G = warp - WS_MMA_WARP;
    if (lane == 0 && n_tiles > G) {
      const uint32_t id_s64 = sm100::idesc_bf16_f32(WS_ROWS, WS_KEYS);
      const uint32_t id_s32 = sm100::idesc_bf16_f32(WS_ROWS, WS_FKEYS);
      const uint32_t id_pv = sm100::idesc_bf16_f32(WS_ROWS, WS_DH) | (1u << 16);   // B (V) MN-major
      // S(t) = Q K(t)^T and O += P(t) V(t), each issued as one run of MMAs
      // (alternating the two measured 2.4x slower).  The issuing loop is kept
      // lean -- descriptors formed once per tile, every MMA's offset a
      // constant -- since a dependent MMA chain issues at the rate this
      // thread reaches it.
      const uint32_t hi = WS_DESC_HI;
      const uint32_t qlo = ws_desc_lo(sbase, 16);                 // Q hi, k-block 0
      // stage base of tile t's K and V; stage and phase tracked incrementally
      auto issue_s = [&](int t, int st) {
        sm100::tc_fence_after();
        const uint32_t stg = rbase + static_cast<uint32_t>(st) * WS_STAGE;
        const uint32_t d = tmem + WS_TM_S + 64u * static_cast<uint32_t>(t & 1);
        const uint32_t klo = ws_desc_lo(stg, 16);
        if (!(draft && t >= T.n_pre)) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)                 // Q hi against K
            ws_mma_ss32(d, qlo + (((kk >> 2) * WS_QHALF + (kk & 3) * 32) >> 4),
                        klo + (((kk >> 2) * WS_HALF + (kk & 3) * 32) >> 4), hi, id_s64, kk > 0 ? 1u : 0u);
          if (draft) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)               // Q lo against K
              ws_mma_ss32(d, qlo + ((2 * WS_QHALF + (kk >> 2) * WS_QHALF + (kk & 3) * 32) >> 4),
                          klo + (((kk >> 2) * WS_HALF + (kk & 3) * 32) >> 4), hi, id_s64, 1u);
          }
        } else {
#pragma unroll
          for (int pr = 0; pr < 3; ++pr)                 // Qhi Khi, Qlo Khi, Qhi Klo
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              ws_mma_ss32(d, qlo + (((pr == 1 ? 2 * WS_QHALF : 0u) + (kk >> 2) * WS_QHALF + (kk & 3) * 32) >> 4),
                          klo + (((pr == 2 ? WS_HALF : 0u) + (kk >> 2) * WS_FHALF + (kk & 3) * 32) >> 4), hi, id_s32,
                          (pr | kk) != 0 ? 1u : 0u);
        }
        sm100::mma_commit(&s_s_full[t & 1]);
        sm100::mma_commit(&s_empty[0][st]);
      };
      auto issue_pv = [&](int t, int st) {
        const uint32_t stg = rbase + static_cast<uint32_t>(st) * WS_STAGE;
        const uint32_t pt = tmem + WS_TM_P + 64u * static_cast<uint32_t>(t & 1);
        const uint32_t od = tmem + WS_TM_O + WS_TM_O_STEP * static_cast<uint32_t>(t & 1);
        const uint32_t first = t >= 2 ? 1u : 0u;            // the first tile of each group starts its O
        if (!(draft && t >= T.n_pre)) {
          const uint32_t vlo = ws_desc_lo(stg + 2 * WS_HALF, WS_HALF);
#pragma unroll
          for (int i = 0; i < 8; ++i)                    // P hi, then P lo, against V
            ws_mma_ts32(od, pt + 32u * (i >> 2) + 8u * (i & 3), vlo + (((i & 3) * 2048) >> 4), hi, id_pv,
                        i > 0 ? 1u : first);
        } else {
          const uint32_t vlo = ws_desc_lo(stg + 2 * WS_HALF, WS_FHALF);
#pragma unroll
          for (int i = 0; i < 6; ++i) {                  // Phi Vhi, Plo Vhi, Phi Vlo
            const int pr = i >> 1, kk = i & 1;
            ws_mma_ts32(od, pt + (pr == 1 ? 32u : 0u) + 8u * kk,
                        vlo + (((pr == 2 ? WS_HALF : 0u) + kk * 2048) >> 4), hi, id_pv, i > 0 ? 1u : first);
          }
        }
        sm100::mma_commit(&s_o_done[t & 1]);
        sm100::mma_commit(&s_empty[1][st]);
      };
      // stage and fill phase of tile t
      auto stage_of = [&](int t) { return t % NST; };
      auto phase_of = [&](int t) { return static_cast<uint32_t>((t / NST) & 1); };
      bool ok = sm100::mbar_wait(&s_full[0][stage_of(G)], phase_of(G), abort_flag);
      if (ok) issue_s(G, stage_of(G));
      for (int t = G; ok && t < n_tiles; t += 2) {
        // S(t + 2) into this group's S buffer as soon as the group's softmax
        // of tile t has read S(t) from it (it then runs while that softmax
        // does), then O += P(t) V(t) once P(t) is written
        if (t + 2 < n_tiles) {
          const int st = stage_of(t + 2);
          ok = sm100::mbar_wait(&s_s_free[G], static_cast<uint32_t>((t >> 1) & 1), abort_flag) &&
               sm100::mbar_wait(&s_full[0][st], phase_of(t + 2), abort_flag);
          if (!ok) break;
          issue_s(t + 2, st);
        }
        const int sv = stage_of(t);
        ok = sm100::mbar_wait(&s_p_full[G], static_cast<uint32_t>((t >> 1) & 1), abort_flag) &&
             sm100::mbar_wait(&s_full[1][sv], phase_of(t), abort_flag);
        if (!ok) break;
        sm100::tc_fence_after();
        issue_pv(t, sv);
      }
      if (!ok) {
        set_status(p.status, EAGLE_ERR_TIMEOUT);
        s_abort = 1;
      }
      // every MMA issued here has completed before the tensor memory goes
      sm100::mma_commit(&s_mma_done[G]);
      sm100::mbar_wait(&s_mma_done[G], 0u, never);
    }
  } else if (warp >= WS_SOFT_WARP0) {
    // ---- softmax: group grp takes the tiles t = grp (mod 2) ----
    // Every warp of the group passes each of the group's tile barriers once,
    // also after an abort or with no rows of the block (in a warp that has
    // some, rows past the block's have zero queries: finite, never written out).
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const bool warp_rows = quarter * 32 < rows_here;   // (the rest of a few-row block is padding)
    const float c = p.scale * WS_LOG2E;
    float m_ref = -INFINITY, l_part = 0.f;
    bool ok = true;
    for (int t = grp; t < n_tiles; t += 2) {
      bool work = ok && !*abort_flag;
      if (work) {
        work = ws_warp_wait(&s_s_full[grp], static_cast<uint32_t>((t >> 1) & 1), abort_flag);
        ok = work;
        sm100::tc_fence_after();
      }
      bool tree, f32;
      int k0, nk;
      T.at(t, tree, f32, k0, nk);
      const bool full = !tree && nk == WS_KEYS;
      const uint64_t mk = tree ? (s_mask[row * MASKW + (k0 >> 6)] >> (k0 & 63)) : ~0ull;
      const bool done = f32 ? ws_softmax_tile<WS_FKEYS>(work, warp_rows, tmem, lane_base, t, w, row, full, mk, nk, c,
                                                        m_ref, l_part, s_o_done, s_s_free, s_pmax, abort_flag)
                            : ws_softmax_tile<WS_KEYS>(work, warp_rows, tmem, lane_base, t, w, row, full, mk, nk, c,
                                                       m_ref, l_part, s_o_done, s_s_free, s_pmax, abort_flag);
      if (work && !done) ok = false;
      sm100::tc_fence_before();
      __syncwarp();
      if (work && ok && lane == 0) sm100::mbar_arrive(&s_p_full[grp]);
    }
    // the group's last P V
    if (ok && n_tiles > grp) {
      const int tl = grp + 2 * ((n_tiles - 1 - grp) / 2);
      ok = ws_warp_wait(&s_o_done[grp], static_cast<uint32_t>((tl >> 1) & 1), abort_flag);
    }
    if (!ok) {
      if (lane == 0) set_status(p.status, EAGLE_ERR_TIMEOUT);
      s_abort = 1;
    }
    // the two groups' states of the row: m (alike in a group's warpgroups), l in parts
    if (w == 0) s_m[grp][row] = m_ref;
    s_l[grp][w][row] = l_part;
    sm100::named_barrier(WS_BAR_SOFT, WS_SOFT_THREADS);
    const float m0 = s_m[0][row], m1 = s_m[1][row];
    const float M = fmaxf(m0, m1);
    const float a0 = m0 == -INFINITY ? 0.f : ws_exp2(m0 - M), a1 = m1 == -INFINITY ? 0.f : ws_exp2(m1 - M);
    m_run = M;
    l_run = a0 * (s_l[0][0][row] + s_l[0][1][row]) + a1 * (s_l[1][0][row] + s_l[1][1][row]);
    // output columns c0 .. c0 + OC - 1: a0 O_0 + a1 O_1 (an O with weight 0 is not read: it may never have been written)
    if (ok && !*abort_flag && warp_rows) {
      sm100::tc_fence_after();
#pragma unroll
      for (int gi = 0; gi < 2; ++gi) {
        const float a = gi ? a1 : a0;
        if (__any_sync(0xffffffffu, a != 0.f)) {
          float v[OC];
          ws_tmem_ld32(tmem + WS_TM_O + WS_TM_O_STEP * gi + lane_base + c0, v);
          sm100::tmem_wait_ld();
          if (a != 0.f) {
#pragma unroll
            for (int j = 0; j < OC; ++j) o[j] = fmaf(a, v[j], o[j]);
          }
        }
      }
    }
  }
  sm100::tc_fence_before();
  __syncthreads();
  if (warp == WS_MMA_WARP) {
    sm100::tc_fence_after();
    sm100::tmem_dealloc(tmem, WS_TM_COLS);
  }
  if (s_abort) return;

  // this thread's output columns c0 .. c0 + OC - 1 of its row
  // (a row with no key in this split keeps max -inf, sum 0, output 0)
  const bool has_row = warp >= WS_SOFT_WARP0 && row < rows_here;
  const int r = r0 + row;
  const int node = r / p.G, hq = h * p.G + r % p.G;
  const size_t qi = (static_cast<size_t>(b) * p.rows_cap + node) * p.Hq + hq;
  if (p.n_splits == 1) {
    if (!has_row) return;
    const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
    if (!draft) {
      float* dst = p.out_f32 + qi * WS_DH + c0;
#pragma unroll
      for (int q = 0; q < OC / 4; ++q)
        *reinterpret_cast<float4*>(dst + 4 * q) =
            make_float4(o[4 * q] * inv, o[4 * q + 1] * inv, o[4 * q + 2] * inv, o[4 * q + 3] * inv);
    } else {
      const size_t j = static_cast<size_t>(b) * p.rows_cap + node;
      uint16_t* dh = p.b_o + j * p.bo_ld + hq * WS_DH + c0;
      uint16_t* dl = p.b_o + (static_cast<size_t>(p.NP) + j) * p.bo_ld + hq * WS_DH + c0;
#pragma unroll
      for (int q = 0; q < OC / 8; ++q) {
        uint4 hi, lo;
        ws_split2(o[8 * q] * inv, o[8 * q + 1] * inv, hi.x, lo.x);
        ws_split2(o[8 * q + 2] * inv, o[8 * q + 3] * inv, hi.y, lo.y);
        ws_split2(o[8 * q + 4] * inv, o[8 * q + 5] * inv, hi.z, lo.z);
        ws_split2(o[8 * q + 6] * inv, o[8 * q + 7] * inv, hi.w, lo.w);
        *reinterpret_cast<uint4*>(dh + 8 * q) = hi;
        *reinterpret_cast<uint4*>(dl + 8 * q) = lo;
      }
    }
    return;
  }
  // several splits: records [query row][split][dh + 4] (max in log2 units,
  // sum, 2 unused, output), then the last CTA of the (request, kv head)
  // merges every row in split order
  const int rec = WS_DH + 4;
  const int ns = p.n_splits;
  if (has_row) {
    float* dst = p.part + (qi * ns + split) * rec;
    if (c0 == 0) {
      dst[0] = m_run;
      dst[1] = l_run;
    }
#pragma unroll
    for (int q = 0; q < OC / 4; ++q)
      *reinterpret_cast<float4*>(dst + 4 + c0 + 4 * q) = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  }
  __syncthreads();                           // every thread's records come first
  if (tid == 0) {
    const int prev = arrive_acq_rel(&p.counters[pair]);
    s_last = prev == ns * static_cast<int>(gridDim.y) - 1;
    if (s_last) p.counters[pair] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  for (int rr = warp; rr < R; rr += WS_THREADS / 32) {
    const int nd = rr / p.G, hh = h * p.G + rr % p.G;
    const float* src = p.part + ((static_cast<size_t>(b) * p.rows_cap + nd) * p.Hq + hh) * ns * rec;
    const float ms = lane < ns ? __ldcg(src + lane * rec) : -INFINITY;
    const float lsv = lane < ns ? __ldcg(src + lane * rec + 1) : 0.f;
    float vals[WS_MAX_RECS][4];
#pragma unroll
    for (int u = 0; u < WS_MAX_RECS; ++u)
#pragma unroll
      for (int q = 0; q < 4; ++q) vals[u][q] = u < ns ? __ldcg(src + u * rec + 4 + lane + 32 * q) : 0.f;
    const float M = warp_max(ms);
    const float wgt = ms == -INFINITY ? 0.f : ws_exp2(ms - M);
    const float Lsum = warp_sum(wgt * lsv);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < WS_MAX_RECS; ++u) {
      const float ws = __shfl_sync(0xffffffffu, wgt, u);
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[q] = fmaf(ws, vals[u][q], acc[q]);
    }
    write_merged_row(p, b, nd, hh, acc, Lsum, lane);
  }
}

}  // namespace

int attn_splits(const eagle_ctx* ctx, int pairs, int cap, int per_sm) {
  const int tiles = ceil_div(cap < 1 ? 1 : cap, TILE);
  // one wave at per_sm CTAs per SM, the tree part's CTA included
  int want = attn_splits_bound(ctx, pairs, cap, per_sm);
  if (want > tiles) want = tiles;
  const int per = ceil_div(tiles, want);
  return ceil_div(tiles, per);     // every split non-empty at full length
}

// CTAs per SM each kernel is sized for (its split count makes one wave).
constexpr int kDraftPerSm = 4;
constexpr int kVerifyPerSm = 2;
// Dynamic shared memory of the tensor-core kernel: four warps at two CTAs
// per SM, eight warps at one.
constexpr size_t kMmaSmemMost = static_cast<size_t>(112) << 10;
constexpr size_t kMma8SmemMost = static_cast<size_t>(216) << 10;
// Dynamic shared memory the CUDA-core kernel may use: two tile buffers, a
// full pass of query rows and score rows, and the records of up to 16 rows.
constexpr size_t kCoreSmemMost = 2 * TILE_BYTES + (static_cast<size_t>(ROWS_PASS) * MAX_DH +
                                                   static_cast<size_t>(WARPS) * RW * TILE) * sizeof(float) +
                                 static_cast<size_t>(16) * (MAX_DH + 4) * sizeof(float);
// CTAs of one cluster at most (above 8 the size is not portable).
constexpr int kClusterMost = 16;
// Shared memory of an SM, and what each resident CTA costs beyond its
// dynamic shared memory (static arrays and the reserved kilobyte).
constexpr size_t kSmemPerSm = static_cast<size_t>(228) << 10;
constexpr size_t kSmemPerCta = static_cast<size_t>(3) << 10;

template <int NR>
static cudaError_t launch_attn_nr(const AttnParams& p, dim3 grid, size_t smem, cudaStream_t st) {
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(tree_attn_kernel<NR>), static_cast<int>(kCoreSmemMost));
  if (e == cudaSuccess && p.cluster) e = cluster_nonportable_once(reinterpret_cast<const void*>(tree_attn_kernel<NR>));
  if (e != cudaSuccess) return e;
  return p.cluster ? launch_pdl_cluster(tree_attn_kernel<NR>, grid, dim3(THREADS), smem, st, p.n_splits + 1, p)
                   : launch_pdl(tree_attn_kernel<NR>, grid, dim3(THREADS), smem, st, p);
}

template <int NW>
static cudaError_t launch_mma(const AttnParams& p, dim3 grid, size_t smem, cudaStream_t st, size_t most) {
  const void* k = reinterpret_cast<const void*>(tree_attn_mma_kernel<NW>);
  cudaError_t e = smem_limit_once(k, static_cast<int>(most));
  if (e == cudaSuccess && p.cluster) e = cluster_nonportable_once(k);
  if (e != cudaSuccess) return e;
  return p.cluster ? launch_pdl_cluster(tree_attn_mma_kernel<NW>, grid, dim3(32 * NW), smem, st, p.n_splits + 1, p)
                   : launch_pdl(tree_attn_mma_kernel<NW>, grid, dim3(32 * NW), smem, st, p);
}

// Query rows per (request, kv head) from which the draft layer's attention
// runs on the tensor cores too.  Measured: 10 rows (EAGLE-2, k = 10) take
// 25 us per launch there against 46 on the CUDA cores at the 7B shape (13B:
// 217 against 368); 1 to 4 rows (the static tree) are faster on the CUDA
// cores (10 against 15 us), most of a 16-row tile being padding.
constexpr int kDraftMmaRows = 8;

// Query rows per (request, kv head) from which the attention (dh 128) runs
// on the tcgen05 kernel.  Measured at the 7B shape: the static tree's 26
// verification rows 20 -> 16 us per round against warp-level MMA; the draft
// layer's 1-4 rows 48 -> 72 us (slower: a 128-row block of padding).
constexpr int kDraftTcRows = 8;
constexpr int kVerifyTcRows = 16;

// A bf16 KV array [rows][Hkv][dh 128] as a 3-D tensor map {dh, kv head, row}
// with boxes of 64 dims x 1 head x box_rows rows in the 128-byte swizzle.
static bool encode_kv_map(eagle_ctx* ctx, CUtensorMap* map, const void* ptr, int Hkv, long long rows, int box_rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(WS_DH), static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(WS_DH) * 2, static_cast<cuuint64_t>(Hkv) * WS_DH * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  return ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tcgen05 kernel (dh 128): as many prefix splits (at most WS_MAX_RECS,
// and never more records per row than the workspace and the no-allocation
// scratch hold) as one wave of CTAs, one per SM, needs.  Whole prefix tiles
// come by TMA when the caches allow it (16-byte aligned, a paged block of at
// least 8 rows, rows addressable with 32-bit coordinates); otherwise every
// tile is copied by the loader warps.
static cudaError_t run_attn_ws(eagle_ctx* ctx, AttnParams& p, int kernel_id, cudaStream_t st) {
  const int rows = p.rows_cap * p.G;
  const int row_blocks = ceil_div(rows, WS_ROWS);
  const int pairs = p.B * p.Hkv;
  const int tiles = ceil_div(p.kv_cap, TILE);
  int want = ctx->sm_count / (pairs * row_blocks);     // whole waves only
  want = std::min(want, std::min(WS_MAX_RECS, tiles));
  want = std::min(want, attn_splits(ctx, pairs, p.kv_cap, kVerifyPerSm) + 1);
  want = std::max(want, 1);
  const int per = ceil_div(tiles, want);
  p.n_splits = ceil_div(tiles, per);         // every split non-empty at full length
  p.chunk = per * TILE;
  p.stages = static_cast<int>((WS_BUDGET - (p.mode == 0 ? 4u : 2u) * WS_QHALF) / WS_STAGE);
  const bool paged = p.paged.table != nullptr;
  const int bs = paged ? (1 << p.paged.shift) : WS_KEYS;
  const long long rows_total =
      paged ? (static_cast<long long>(p.paged.n_blocks) << p.paged.shift) : static_cast<long long>(p.B) * p.kv_cap;
  auto aligned16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  p.box_rows = std::min(WS_KEYS, bs);
  p.tma = bs >= 8 && rows_total < (1ll << 31) && aligned16(p.kp) && aligned16(p.vp);
  CUtensorMap km, vm;
  std::memset(&km, 0, sizeof(km));
  std::memset(&vm, 0, sizeof(vm));
  if (p.tma && !(encode_kv_map(ctx, &km, p.kp, p.Hkv, rows_total, p.box_rows) &&
                 encode_kv_map(ctx, &vm, p.vp, p.Hkv, rows_total, p.box_rows)))
    p.tma = 0;
  dim3 grid(p.n_splits, row_blocks, pairs);
  p.stamp = stamp_slot(ctx, kernel_id);
  trace_before(ctx, kernel_id, st);
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(tree_attn_ws_kernel), static_cast<int>(WS_SMEM));
  if (e == cudaSuccess) e = launch_pdl(tree_attn_ws_kernel, grid, dim3(WS_THREADS), WS_SMEM, st, p, km, vm);
  ctx->launches++;
  trace_after(ctx, kernel_id, st);
  return e;
}

static cudaError_t run_attn(eagle_ctx* ctx, AttnParams& p, int kernel_id, cudaStream_t st) {
  if (p.dh % 16 != 0 || p.dh > MAX_DH) return cudaErrorInvalidValue;
  if (p.dh == WS_DH && ((p.mode == 1 && p.rows_cap * p.G >= kVerifyTcRows) ||
                        (p.mode == 0 && p.rows_cap * p.G >= kDraftTcRows)))
    return run_attn_ws(ctx, p, kernel_id, st);
  const bool mma = p.mode == 1 || p.rows_cap * p.G >= kDraftMmaRows;
  const int tiles = ceil_div(p.kv_cap, TILE);
  const int rows = p.rows_cap * p.G;
  p.rows_pass = std::min(ROWS_PASS, rows);
  // tensor cores: eight warps per CTA (one CTA per SM, 128-row passes) when
  // a kv head has more query rows than four four-warp passes take.
  // Measured at the 70B shape: 488 verification rows 4.7 -> 4.0 ms; 80
  // draft rows 4.5 -> 5.1 ms (slower: a CTA per SM); 61 rows about even.
  const int nw = mma && rows > 4 * ROWS_PASS ? 8 : 4;
  const int per_sm_most = mma ? (nw == 8 ? 1 : kVerifyPerSm) : kDraftPerSm;
  p.n_splits = attn_splits(ctx, p.B * p.Hkv, p.kv_cap, per_sm_most);
  // Tile buffers of a split of tps key tiles (two: the next tile streams in
  // while the current one is consumed; a deeper ring measured no faster at
  // the 70B shape), and the dynamic shared memory of such a launch.
  auto nbuf_for = [&](int tps) { return std::min(tps, 2); };
  auto smem_for = [&](int tps) {
    const size_t bufs = static_cast<size_t>(nbuf_for(tps)) * TILE_BYTES;
    return mma ? bufs + q_bytes(nw)
               : bufs + (static_cast<size_t>(p.rows_pass) * p.dh + static_cast<size_t>(WARPS) * RW * TILE) *
                            sizeof(float);
  };
  // Waves of a launch of `splits` prefix splits whose CTAs take `smem`
  // bytes of dynamic shared memory each.
  const int pairs = p.B * p.Hkv;
  auto waves = [&](int splits, size_t smem) {
    int per_sm = static_cast<int>(kSmemPerSm / (smem + kSmemPerCta));
    per_sm = std::max(1, std::min(per_sm, per_sm_most));
    return ceil_div((splits + 1) * pairs, per_sm * ctx->sm_count);
  };
  // The splits of a (request, kv head) merge inside one cluster when they
  // fit one (at most kClusterMost CTAs, the tree part's included), every
  // row's record fits beside the tiles and the launch is one wave;
  // otherwise the last CTA to finish merges them through global memory.
  // Measured: fewer, longer splits to fit a cluster are slower (the tiles
  // of a split load one after another), and so are clusters over several
  // waves (whole clusters wait for room in one GPC: 13B draft attention
  // 1.8 -> 3.8 ms).
  if (p.n_splits + 1 <= kClusterMost) {
    const size_t recs = static_cast<size_t>(rows) * (p.dh + 4) * sizeof(float);
    const size_t base = smem_for(ceil_div(tiles, p.n_splits));
    const size_t most = mma ? (nw == 8 ? kMma8SmemMost : kMmaSmemMost) : kCoreSmemMost;
    if (base + recs <= most && waves(p.n_splits, base + recs) == 1) {
      p.cluster = 1;
      p.recs_off = static_cast<int>(base);
    }
  }
  const int tiles_per_split = ceil_div(tiles, p.n_splits);
  p.chunk = tiles_per_split * TILE;
  p.n_buf = nbuf_for(tiles_per_split);
  const size_t smem = smem_for(tiles_per_split) +
                      (p.cluster ? static_cast<size_t>(rows) * (p.dh + 4) * sizeof(float) : 0);
  const int ns = p.n_splits + 1;
  dim3 grid(ns, p.B * p.Hkv);
  p.stamp = stamp_slot(ctx, kernel_id);
  trace_before(ctx, kernel_id, st);
  cudaError_t e;
  if (mma) {
    e = nw == 8 ? launch_mma<8>(p, grid, smem, st, kMma8SmemMost) : launch_mma<4>(p, grid, smem, st, kMmaSmemMost);
  } else {
    const int per_warp = ceil_div(p.rows_pass, WARPS);
    if (per_warp <= 1) e = launch_attn_nr<1>(p, grid, smem, st);
    else if (per_warp <= 2) e = launch_attn_nr<2>(p, grid, smem, st);
    else if (per_warp <= 4) e = launch_attn_nr<4>(p, grid, smem, st);
    else e = launch_attn_nr<RW>(p, grid, smem, st);
  }
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
  p.mask_words = EAGLE_MASK_WORDS(p.tree_cap);
  p.e0 = L.e0;
  p.scale = 1.0f / sqrtf(static_cast<float>(D.head_dim));
  p.b_o = ws_ptr<uint16_t>(L.ws, W.b_o);
  p.NP = L.NP;
  p.bo_ld = W.kp_o;
  p.part = ws_ptr<float>(L.ws, W.attn_part);
  p.counters = ws_ptr<int>(L.ws, W.attn_cnt);
  p.status = ws_ptr<int>(L.ws, W.status);
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
  p.paged = paged_of(&prefix->paging, prefix->cap);
  p.kv_len = prefix->len;
  p.kt_bf16 = kt;
  p.vt_bf16 = vt;
  p.tree_cap = tree->stride;
  p.anc = tree->anc;
  p.mask_words = EAGLE_MASK_WORDS(p.tree_cap);
  p.tree_size = tree->size;
  p.scale = scale;
  p.out_f32 = out;
  p.part = ws_ptr<float>(ws, W.attn_part);
  p.counters = ws_ptr<int>(ws, W.attn_cnt) + ctx->lim.max_batch * D.n_kv_heads;
  p.status = ws_ptr<int>(ws, W.status);
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

static __device__ __align__(256) unsigned char verify_scratch[kScratchBytes];

namespace {
// The array's address in each CUDA context that has used it, keyed by the
// context's id: a context re-created after cudaDeviceReset has a new id, so
// its array is looked up and its counters zeroed again.
std::mutex scratch_mu;
std::vector<std::pair<unsigned long long, void*>> scratch_base;
}  // namespace

size_t verify_scratch_need(const eagle_ctx* ctx, int batch, const eagle_kv* prefix, const eagle_tree* tree) {
  const eagle_dims& D = ctx->dims;
  const int splits = attn_splits(ctx, batch * D.n_kv_heads, prefix->cap, kVerifyPerSm);
  const size_t records = static_cast<size_t>(batch) * tree->stride * D.n_q_heads * (splits + 1);
  return records * (D.head_dim + 4) * sizeof(float);
}

eagle_status launch_verify_attn_noalloc(eagle_ctx* ctx, int batch, const uint16_t* q, const uint16_t* kt,
                                        const uint16_t* vt, const eagle_kv* prefix, const eagle_tree* tree,
                                        float scale, float* out, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  if (batch * D.n_kv_heads > kScratchMaxPairs ||
      verify_scratch_need(ctx, batch, prefix, tree) > kScratchBytes - kScratchCounterBytes)
    return EAGLE_ERR_CAPACITY;                 // nothing launched
  unsigned long long cid = 0;
  if (!current_context_id(&cid)) return EAGLE_ERR_CUDA;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(scratch_mu);
    for (const auto& kv : scratch_base)
      if (kv.first == cid) base = kv.second;
    if (base == nullptr) {
      // first call in this context: the set-up below would synchronise the
      // stream, which a capture does not allow -- refuse before touching it
      cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return EAGLE_ERR_CUDA;
      if (cap != cudaStreamCaptureStatusNone) return EAGLE_ERR_INVALID_ARG;
      // the array's address, then zeroed counters
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, verify_scratch) != cudaSuccess) return EAGLE_ERR_CUDA;
      if (cudaMemsetAsync(ptr, 0, kScratchCounterBytes, st) != cudaSuccess) return EAGLE_ERR_CUDA;
      if (cudaStreamSynchronize(st) != cudaSuccess) return EAGLE_ERR_CUDA;
      scratch_base.emplace_back(cid, ptr);
      base = ptr;
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
  p.paged = paged_of(&prefix->paging, prefix->cap);
  p.kv_len = prefix->len;
  p.kt_bf16 = kt;
  p.vt_bf16 = vt;
  p.tree_cap = tree->stride;
  p.anc = tree->anc;
  p.mask_words = EAGLE_MASK_WORDS(p.tree_cap);
  p.tree_size = tree->size;
  p.scale = scale;
  p.out_f32 = out;
  // the last CTA of each (request, kv head) puts its counter back to zero
  p.counters = static_cast<int*>(base);
  p.part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kScratchCounterBytes);
  return run_attn(ctx, p, EAGLE_K_VERIFY_ATTN, st) == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // namespace eagle
