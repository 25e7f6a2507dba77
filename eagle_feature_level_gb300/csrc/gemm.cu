// Weight-streaming GEMM for the draft head's contractions (FC, QKV, O,
// gate/up, down, LM head), Y[n][out] = X[n][K] . W[out][K]^T with n = draft
// rows (1..256) and W streamed from HBM exactly once per launch.
//
// Blackwell design:
//  * a pipeline stage holds 128 weight rows x kps k-blocks of 64 (kps = 2
//    unless the activation tile is large): each 64-row half is one TMA box of
//    a 4-D tensor map {64 k, 8 rows, k-block, 8-row group}, so every request
//    fetches kps x 128 contiguous bytes per weight row (HBM streams markedly
//    faster at 256 B per row than at 128 B); shared memory receives
//    [group][k-block][8 rows][128 B] with the 128-byte swizzle, which the MMA
//    reads with an 8-row group stride of kps x 1024 B.  The 4-D map covers
//    only whole k-blocks and whole 8-row groups, so it never reads past a row
//    pitch or the last row; a half that reaches a matrix's row tail or K tail
//    is fetched as 8 x kps boxes {64 k, 8 rows} of a 2-D map over the used
//    [rows][K] extent, whose out-of-range elements fill with zeros;
//  * the activation tile arrives the same way (one 4-D box); stages cycle
//    through a multi-stage shared-memory ring guarded by mbarriers;
//  * one thread issues tcgen05.mma (M = 128 weight rows, N = activation rows,
//    "swap-AB"), accumulating in tensor memory; a commit per stage releases the
//    ring slot;
//  * activations enter as two bf16 halves (x = hi + lo), stacked along N, so
//    the fp32 activation keeps ~16 mantissa bits while the weights stay bf16;
//  * work is split stream-K style: the (tile, k-block) units are divided
//    evenly over the CTAs, so every SM streams the same number of bytes.
//    Contractions with fewer 128-row tiles than SMs run two CTAs per SM with
//    half-size rings (every tile split); the others run one CTA per SM, the
//    stream-K share of the leftover tiles first, then whole tiles of their
//    own with the epilogue straight from tensor memory.  For a split tile
//    each CTA writes its fp32 partial and arrives on the tile's counter; the
//    last to arrive sums the partials in CTA order (deterministic);
//  * the epilogue of that last CTA fuses the layer's elementwise work: bias,
//    residual adds, RMSNorm scaling (sum of squares carried as per-tile
//    partials), RoPE, SiLU-gating, the bf16 hi/lo split of the next
//    contraction's input, and the scatter into per-node outputs.
// Warp roles: warp 0 = TMA producer, warp 1 = MMA issuer and tensor-memory
// owner, warps 2-5 = epilogue (one tensor-memory lane quarter each).
#include "internal.h"
#include "sm100.cuh"

namespace eagle {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;                     // elements per k-block (one 128-byte swizzle row)
constexpr int KBLK_BYTES = BK * 2;
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
// Activation rows per epilogue chunk: 16, or 32 when a launch has more than
// 16 rows (each chunk's row inputs and split partials cost a round trip to
// L2, which the finalizing CTA waits for; the smaller chunk keeps the shared
// memory of few-row launches as it was).
constexpr int XCH_MAX = 32;

struct GemmParams {
  int epi;
  int n, NP, kb, m_tiles;
  long long total_units;
  int mblk[3];
  int n_mats;
  int two_mma;
  int tmem_cols, acc_stride, n_acc, stages;
  int kps;                  // k-blocks per stage
  int xr;                   // activation rows per epilogue chunk (16 or XCH_MAX)
  int coop;                 // every CTA resident at once: split tiles finalized by all their contributors
  uint32_t a_stage_bytes, b_stage_bytes;
  int full_rows[3];         // rows of each matrix in whole 8-row groups
  int full_kb;              // whole 64-wide k-blocks of K
  int sk_tiles;             // tiles [0, sk_tiles) split stream-K over all CTAs (processed first)
  int dp_waves;             // then tiles sk_tiles + c + i * grid, i < dp_waves, owned by CTA c alone
  int sk_whole;             // fewer stream-K units than CTAs: tile c < sk_tiles whole to CTA c
  int rpr, e0, E;
  int d, F, V, Hq, Hkv, dh;
  float eps;
  double ln_theta;
  const float* bias;
  const float* gain;
  const float* ss_in;
  int ss_in_tiles;
  float* ss_out;
  const float* resid;
  float* out_f32;
  uint16_t* bnext;
  int kp_next;
  float* qrow;
  float* k_tree;
  float* v_tree;
  const int32_t* pos0;
  const int32_t* depth;
  float* part;
  int* counters;
  int* status;
  uint64_t* stamp;
  // EPI_KV (draft-cache refresh): bf16 cache [B][kv_cap_rows][Hkv][dh]
  uint16_t* kc;
  uint16_t* vc;
  int kv_cap_rows;
  const int32_t* kv_len;
  const int32_t* n_act;
};

struct Smem {
  uint8_t* a;       // stages x a_stage_bytes
  uint8_t* b;       // stages x b_stage_bytes
  uint64_t* full;
  uint64_t* empty;
  uint64_t* tfull;  // [2]
  uint64_t* tempty; // [2]
  uint32_t* tmem_holder;
  int* flags;       // [0] abort, [1] last-arriver, [2] wait ok
  float* xch;       // [xr][128]
  float* red;       // [4][32]
  float* rs;        // [32]
  int* rowi;        // [2 * XCH_MAX]
  float* stg2;      // [xr][sw], 16-byte aligned: the tile's row inputs from earlier kernels (last)
};

// sw: floats per staged row input (BM residual columns, or a row's norm
// partials at a stride of ss_in_tiles + 1), so s.stg2 holds xr * sw floats.
__host__ __device__ inline size_t smem_bytes_for(int stages, uint32_t a_stage, uint32_t b_stage, int xr, int sw) {
  size_t s = 1024;                                  // alignment slack
  s += static_cast<size_t>(stages) * (a_stage + b_stage);
  s += (2 * stages + 4) * 8 + 64;
  s += static_cast<size_t>(xr) * BM * 4 + 4 * 32 * 4 + 32 * 4 + 2 * XCH_MAX * 4 + static_cast<size_t>(xr) * sw * 4;
  return s;
}

__device__ inline Smem carve(uint8_t* raw, const GemmParams& p) {
  uintptr_t base = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023);
  uint8_t* ptr = reinterpret_cast<uint8_t*>(base);
  Smem s;
  s.a = ptr;
  ptr += static_cast<size_t>(p.stages) * p.a_stage_bytes;
  s.b = ptr;
  ptr += static_cast<size_t>(p.stages) * p.b_stage_bytes;
  s.full = reinterpret_cast<uint64_t*>(ptr);
  s.empty = s.full + p.stages;
  s.tfull = s.empty + p.stages;
  s.tempty = s.tfull + 2;
  s.tmem_holder = reinterpret_cast<uint32_t*>(s.tempty + 2);
  s.flags = reinterpret_cast<int*>(s.tmem_holder + 4);
  s.xch = reinterpret_cast<float*>(s.flags + 12);
  s.red = s.xch + p.xr * BM;
  s.rs = s.red + 4 * 32;
  s.rowi = reinterpret_cast<int*>(s.rs + 32);
  s.stg2 = reinterpret_cast<float*>(s.rowi + 2 * XCH_MAX);
  return s;
}

// CTA that owns k-block unit u under the even split of T units over G CTAs
// (CTA c owns [floor(c T / G), floor((c+1) T / G))).
__device__ __forceinline__ int cta_of_unit(long long u, long long T, int G) {
  return static_cast<int>(((u + 1) * G - 1) / T);
}

// The CTA's work: first its even share [sk_begin, sk_end) of the stream-K
// units (tiles [0, sk_tiles), kb units each), then dp_waves whole tiles of
// its own.  Virtual unit v in [0, n_units) names the v-th unit it processes.
struct CtaWork {
  long long sk_begin, sk_end;
  int cta, grid;
  __device__ long long n_units(const GemmParams& p) const {
    return (sk_end - sk_begin) + static_cast<long long>(p.dp_waves) * p.kb;
  }
  __device__ long long unit(const GemmParams& p, long long v) const {
    const long long n_sk = sk_end - sk_begin;
    if (v < n_sk) return sk_begin + v;
    const long long w = (v - n_sk) / p.kb, k = (v - n_sk) % p.kb;
    return (static_cast<long long>(p.sk_tiles) + cta + w * grid) * p.kb + k;
  }
  // segment seg: tile t, virtual units [v0, v1); false past the last one
  __device__ bool segment(const GemmParams& p, int seg, int& t, long long& v0, long long& v1) const {
    const long long n_sk = sk_end - sk_begin;
    const int n_sk_seg = n_sk > 0 ? static_cast<int>((sk_end - 1) / p.kb - sk_begin / p.kb + 1) : 0;
    if (seg < n_sk_seg) {
      t = static_cast<int>(sk_begin / p.kb) + seg;
      const long long u0 = max(sk_begin, static_cast<long long>(t) * p.kb);
      const long long u1 = min(sk_end, static_cast<long long>(t + 1) * p.kb);
      v0 = u0 - sk_begin;
      v1 = u1 - sk_begin;
      return true;
    }
    const int w = seg - n_sk_seg;
    if (w >= p.dp_waves) return false;
    t = p.sk_tiles + cta + w * grid;
    v0 = n_sk + static_cast<long long>(w) * p.kb;
    v1 = v0 + p.kb;
    return true;
  }
};

__device__ __forceinline__ CtaWork cta_work(const GemmParams& p) {
  CtaWork wk;
  wk.cta = blockIdx.x;
  wk.grid = gridDim.x;
  const long long U = static_cast<long long>(p.sk_tiles) * p.kb;
  if (p.sk_whole) {
    // an even split would leave CTAs without units, and a tile's
    // contributors would no longer be every CTA between its first and last
    wk.sk_begin = wk.cta < p.sk_tiles ? static_cast<long long>(wk.cta) * p.kb : U;
    wk.sk_end = wk.cta < p.sk_tiles ? static_cast<long long>(wk.cta + 1) * p.kb : U;
    return wk;
  }
  wk.sk_begin = static_cast<long long>(wk.cta) * U / wk.grid;
  wk.sk_end = static_cast<long long>(wk.cta + 1) * U / wk.grid;
  return wk;
}

__device__ __forceinline__ void locate_box(const GemmParams& p, int t, int half, int& map, int& row) {
  if (p.epi == EPI_GATEUP) {          // box 0: gate rows, box 1: up rows of the same 64 columns
    map = half;
    row = t * 64;
    return;
  }
  const int blk = 2 * t + half;
  int prev = 0;
  for (int i = 0; i < p.n_mats; ++i) {
    if (blk < p.mblk[i] || i == p.n_mats - 1) {
      map = i;
      row = (blk - prev) * 64;
      return;
    }
    prev = p.mblk[i];
  }
  map = 0;
  row = 0;
}

__device__ __forceinline__ void put_split(uint16_t* buf, int NP, int kp, int j, int col, float x) {
  uint16_t hi, lo;
  split_bf16(x, hi, lo);
  buf[static_cast<size_t>(j) * kp + col] = hi;
  buf[static_cast<size_t>(NP + j) * kp + col] = lo;
}

// RoPE angle pos * f reduced to about [-pi, pi] in fp32: f = f_hi + f_lo,
// the product's rounding error recovered with an FMA, then Cody-Waite
// reduction by 2 pi = C1 + C2 + C3 (Cody & Waite, "Software Manual for the
// Elementary Functions", 1980), C1 carrying 8 significant bits so k * C1 is
// exact for the |k| < 2^16 that positions below 2^18 can produce.
__device__ __forceinline__ float rope_angle(int pos, float f_hi, float f_lo) {
  constexpr float C1 = 6.28125f;
  constexpr float C2 = 1.9353071795864769253e-3f;
  constexpr float C3 = static_cast<float>(1.9353071795864769253e-3 - static_cast<double>(C2));
  const float P = static_cast<float>(pos);            // exact: pos < 2^24
  const float a = P * f_hi;
  const float a_lo = fmaf(P, f_lo, fmaf(P, f_hi, -a));
  const float k = rintf(a * 0.15915494309189535f);
  float r = a - k * C1;                                // exact
  r = fmaf(-k, C2, r);
  r = fmaf(-k, C3, r);
  return r + a_lo;
}

// 16-byte global -> shared copies that bypass L1 (the sources are rewritten
// by other CTAs and kernels), issued without waiting.
__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The 128 epilogue threads copy n contiguous floats (n % 4 == 0, both ends
// 16-byte aligned) into shared memory.
__device__ __forceinline__ void stage_block(float* dst, const float* src, int n, int et) {
  for (int i = 4 * et; i < n; i += 4 * EPI_THREADS) cp_async16(dst + i, src + i);
}

// Per-column constants of the fused epilogue for tile row m of tile t.
struct EpiCol {
  int gi, qd, kd, head, di, partner;
  bool rope, is_v, rot_first, d_col;
  float f_hi, f_lo, col_bias, col_gain;
};

__device__ __noinline__ EpiCol epi_column(const GemmParams& p, int t, int m) {
  EpiCol c;
  c.gi = t * BM + m;
  c.qd = p.epi == EPI_KV ? 0 : p.Hq * p.dh;   // the refresh projects K and V only
  c.kd = p.Hkv * p.dh;
  const int half = p.dh >> 1;
  c.rope = false; c.is_v = false; c.rot_first = false;
  c.head = 0; c.di = 0; c.partner = m;
  c.f_hi = 0.f; c.f_lo = 0.f;          // inverse frequency as an unevaluated float pair
  if ((p.epi == EPI_QKV || p.epi == EPI_KV) && c.gi < c.qd + 2 * c.kd) {
    c.is_v = c.gi >= c.qd + c.kd;
    const int base = c.gi < c.qd ? 0 : (c.gi < c.qd + c.kd ? c.qd : c.qd + c.kd);
    c.head = (c.gi - base) / p.dh;
    c.di = (c.gi - base) % p.dh;
    c.rot_first = c.di < half;
    c.partner = c.rot_first ? m + half : m - half;
    c.rope = !c.is_v;
    const double inv_freq = exp(-(2.0 * (c.rot_first ? c.di : c.di - half) / p.dh) * p.ln_theta);
    c.f_hi = static_cast<float>(inv_freq);
    c.f_lo = static_cast<float>(inv_freq - static_cast<double>(c.f_hi));
  }
  c.d_col = c.gi < p.d;
  c.col_bias = 0.f; c.col_gain = 0.f;
  if (p.epi == EPI_FC && c.d_col) { c.col_bias = p.bias[c.gi]; c.col_gain = p.gain[c.gi]; }
  if (p.epi == EPI_FUSE && c.d_col && p.bias != nullptr) c.col_bias = p.bias[c.gi];
  if (p.epi == EPI_O && c.d_col) c.col_gain = p.gain[c.gi];
  return c;
}

// Issue the asynchronous copies of rows jc .. jc + nj - 1's inputs from
// earlier kernels into s.stg2 (residual rows for O / down, RMSNorm partial
// sums for QKV / gate-up) and, for QKV, the rows' RoPE positions into
// s.rowi.  Completion: cp_async_wait_all + an epilogue barrier.
__device__ __noinline__ void stage_row_inputs(const GemmParams& p, const Smem& s, int t, int jc, int nj, int m) {
  const int et = m;
  const int tiles = p.ss_in_tiles;
  if (p.epi == EPI_O || p.epi == EPI_DOWN) {                      // residual rows, this tile's columns
    const int ncol = min(BM, p.d - t * BM);                         // a multiple of 64
    for (int i = et; i < nj * (BM / 4); i += EPI_THREADS) {
      const int r = i / (BM / 4), q = 4 * (i % (BM / 4));
      if (q < ncol) cp_async16(s.stg2 + r * BM + q, p.resid + static_cast<size_t>(jc + r) * p.d + t * BM + q);
    }
  } else if (p.epi == EPI_QKV || p.epi == EPI_GATEUP || p.epi == EPI_KV) {   // norm partials of rows jc..jc+nj-1
    // row r at stg2 + r * (tiles + 1): with a stride one longer than the
    // row, the threads summing one row each no longer share a bank
    const float* ss = p.ss_in + static_cast<size_t>(jc) * tiles;
    const int n = nj * tiles;
#pragma unroll 4
    for (int i = et; i < n; i += EPI_THREADS) {
      const int r = i / tiles;
      s.stg2[i + r] = __ldcg(ss + i);
    }
    if (p.epi == EPI_QKV && m < nj) {
      const int j = jc + m, b = j / p.rpr, e = p.e0 + j % p.rpr;
      s.rowi[m] = p.pos0[b] + p.depth[static_cast<size_t>(b) * p.E + e];
    }
    if (p.epi == EPI_KV && m < nj) {
      // refresh row (b, i): position pos0[b] + i, cache row len[b] + i - 1;
      // all of a request's rows or none (the cache must take them all)
      const int j = jc + m, b = j / p.rpr, i = j % p.rpr + 1;
      const int len = p.kv_len[b], a = min(max(p.n_act[b], 0), p.rpr);
      const bool room = len >= 0 && len + a <= p.kv_cap_rows;
      s.rowi[m] = p.pos0[b] + i;
      s.rowi[XCH_MAX + m] = (i <= a && room) ? len + i - 1 : -1;
    }
  }
}

// Steps 2-3 of a tile's epilogue for rows jc .. jc + nj - 1, whose summed
// accumulators are in s.xch: wait for the rows' inputs written by earlier
// kernels (the caller has issued their copies into s.stg2), then the
// contraction's elementwise work.  Ends with the epilogue warps
// synchronised.
__device__ __noinline__ void epilogue_chunk(const GemmParams& p, const Smem& s, const EpiCol& col, int t, int jc,
                                            int nj, int m) {
  // the shared rows' pointers in registers: the loops' global stores could
  // otherwise alias the Smem fields, forcing a re-read per row
  float* const xch = s.xch;
  const float* const stg2 = s.stg2;
  const float* const rs = s.rs;
  const int* const rowi = s.rowi;
  float* const red = s.red;
  const int gi = col.gi, qd = col.qd, kd = col.kd, head = col.head, di = col.di, partner = col.partner;
  const bool rope = col.rope, is_v = col.is_v, rot_first = col.rot_first, d_col = col.d_col;
  const float f_hi = col.f_hi, f_lo = col.f_lo, col_bias = col.col_bias, col_gain = col.col_gain;
  // 2. row inputs written by earlier kernels (staged in s.stg2)
  const int tiles = p.ss_in_tiles;
  cp_async_wait_all();
  sm100::named_barrier(1, EPI_THREADS);
  if ((p.epi == EPI_O || p.epi == EPI_DOWN) && d_col) {
#pragma unroll 1
    for (int jj = 0; jj < nj; ++jj) xch[jj * BM + m] += stg2[jj * BM + m];
  }
  if ((p.epi == EPI_QKV || p.epi == EPI_GATEUP || p.epi == EPI_KV) && m < nj) {   // RMSNorm scale of input row jc + m
    const float* ss = stg2 + m * (tiles + 1);
    float acc4[4] = {0.f, 0.f, 0.f, 0.f};
    int i = 0;
#pragma unroll 1
    for (; i + 4 <= tiles; i += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) acc4[u] += ss[i + u];
    }
#pragma unroll 1
    for (; i < tiles; ++i) acc4[0] += ss[i];
    const float tot = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
    s.rs[m] = 1.0f / sqrtf(tot / static_cast<float>(p.d) + p.eps);
  }
  sm100::named_barrier(1, EPI_THREADS);
  // 3. the contraction's elementwise epilogue, one activation row at a time
  if (p.epi == EPI_FC || p.epi == EPI_O) {
    float* const out = p.out_f32;
    uint16_t* const bn = p.bnext;
    const int NP = p.NP, kpn = p.kp_next, d = p.d;
#pragma unroll 1
    for (int jj = 0; jj < nj; ++jj) {
      const int j = jc + jj;
      float v = 0.f;
      if (d_col) {
        v = xch[jj * BM + m] + col_bias;
        out[static_cast<size_t>(j) * d + gi] = v;
        put_split(bn, NP, kpn, j, gi, v * col_gain);
      }
      xch[jj * BM + m] = v;
    }
    sm100::named_barrier(1, EPI_THREADS);
    // sum of squares of the tile's columns of each row (next RMSNorm): warp
    // w sums columns 32w .. 32w + 31 of row r = lane (the rotated start keeps
    // the lanes on distinct banks), then thread r adds the four warp sums
    {
      const int w = m >> 5, r = m & 31;
      if (r < nj) {
        float sq = 0.f;
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
          const float x = xch[r * BM + 32 * w + ((k + r) & 31)];
          sq = fmaf(x, x, sq);
        }
        red[w * 32 + r] = sq;
      }
      sm100::named_barrier(1, EPI_THREADS);
      if (m < nj)
        p.ss_out[static_cast<size_t>(jc + m) * p.m_tiles + t] =
            (red[m] + red[32 + m]) + (red[64 + m] + red[96 + m]);
    }
  } else if (p.epi == EPI_QKV) {
    if (gi < qd + 2 * kd) {
      float* const qrow = p.qrow;
      float* const dst = is_v ? p.v_tree : p.k_tree;
      const int rpr = p.rpr, e0 = p.e0, E = p.E, Hkv = p.Hkv, dh = p.dh;
#pragma unroll 1
      for (int jj = 0; jj < nj; ++jj) {
        const int j = jc + jj;
        const int b = j / rpr, e = e0 + j % rpr;
        const float sc = rs[jj];
        float v = xch[jj * BM + m] * sc;
        if (rope) {
          float sn, cs;
          sincosf(rope_angle(rowi[jj], f_hi, f_lo), &sn, &cs);
          const float other = xch[jj * BM + partner] * sc;
          v = rot_first ? v * cs - other * sn : v * cs + other * sn;
        }
        if (gi < qd)
          qrow[static_cast<size_t>(j) * qd + gi] = v;
        else
          dst[((static_cast<size_t>(b) * E + e) * Hkv + head) * dh + di] = v;
      }
    }
  } else if (p.epi == EPI_KV) {
    if (gi < 2 * kd) {
      uint16_t* const dst = is_v ? p.vc : p.kc;
      const int rpr = p.rpr, Hkv = p.Hkv, dh = p.dh, cap = p.kv_cap_rows;
#pragma unroll 1
      for (int jj = 0; jj < nj; ++jj) {
        const int row = rowi[XCH_MAX + jj];
        if (row < 0) continue;                 // inactive row, or the cache cannot take the request's rows
        const int b = (jc + jj) / rpr;
        const float sc = rs[jj];
        float v = xch[jj * BM + m] * sc;
        if (rope) {
          float sn, cs;
          sincosf(rope_angle(rowi[jj], f_hi, f_lo), &sn, &cs);
          const float other = xch[jj * BM + partner] * sc;
          v = rot_first ? v * cs - other * sn : v * cs + other * sn;
        }
        dst[((static_cast<size_t>(b) * cap + row) * Hkv + head) * dh + di] = f32_to_bf16(v);
      }
    }
  } else if (p.epi == EPI_FUSE) {
    if (d_col) {
      float* const out = p.out_f32;
      const int d = p.d;
#pragma unroll 1
      for (int jj = 0; jj < nj; ++jj) out[static_cast<size_t>(jc + jj) * d + gi] = xch[jj * BM + m] + col_bias;
    }
  } else if (p.epi == EPI_GATEUP) {
    const int c = t * 64 + m;
    if (m < 64 && c < p.F) {
      uint16_t* const bn = p.bnext;
      const int NP = p.NP, kpn = p.kp_next;
#pragma unroll 1
      for (int jj = 0; jj < nj; ++jj) {
        const float sc = rs[jj];
        const float g = xch[jj * BM + m] * sc, u = xch[jj * BM + m + 64] * sc;
        put_split(bn, NP, kpn, jc + jj, c, g / (1.0f + expf(-g)) * u);
      }
    }
  } else if (p.epi == EPI_DOWN) {
    if (d_col) {
      float* const out = p.out_f32;
      uint16_t* const bn = p.bnext;
      const int NP = p.NP, kpn = p.kp_next, d = p.d, rpr = p.rpr, e0 = p.e0, E = p.E;
#pragma unroll 1
      for (int jj = 0; jj < nj; ++jj) {
        const int j = jc + jj;
        const int b = j / rpr, e = e0 + j % rpr;
        const float v = xch[jj * BM + m];
        out[(static_cast<size_t>(b) * E + e) * d + gi] = v;
        put_split(bn, NP, kpn, j, gi, v);
      }
    }
  } else {  // EPI_LM
    if (gi < p.V) {
      float* const out = p.out_f32;
      const int rpr = p.rpr, e0 = p.e0, E = p.E, V = p.V;
#pragma unroll 1
      for (int jj = 0; jj < nj; ++jj) {
        const int j = jc + jj;
        const int b = j / rpr, e = e0 + j % rpr;
        out[(static_cast<size_t>(b) * E + e) * V + gi] = xch[jj * BM + m];
      }
    }
  }
  sm100::named_barrier(1, EPI_THREADS);
}

// Final epilogue of tile t: sum the partials of CTAs [c_first, c_last] and
// apply the contraction's fused elementwise work.  `m` is the tile row this
// thread owns (its tensor-memory lane).  It runs once per tile, cold, at the
// end of the stream, so its chain of memory latencies is on the kernel's
// critical path.  `area` (cap floats, 16-byte aligned) is the idle pipeline
// ring when this is the CTA's last tile, else null: when every contributor's
// partial fits in it beside their sum, the partials of all rows arrive in
// one batch of asynchronous copies issued from compact loops (many in
// flight, one wait); otherwise each chunk of xr rows is loaded straight from
// L2, 16 rows x four CTAs' loads in flight at a time (staging one
// contributor's 160 rows at a time through the ring took ~7 us a batch).  Either
// way every element is summed in CTA order (deterministic, and the same
// order on both routes).
__device__ __noinline__ void finalize_tile(const GemmParams& p, const Smem& s, const EpiCol& col, int t,
                                           int c_first, int c_last, int m, float* area, int cap) {
  const int et = m;                    // epilogue thread index == tile row
  const int C = c_last - c_first + 1;
  const int blk = p.n * BM;            // one CTA's partial of the tile: n rows
  const float* part = p.part + static_cast<size_t>(t + c_first) * blk;
  float* const xch = s.xch;            // in registers (see epilogue_chunk)
  if (area != nullptr && cap - blk >= C * blk) {   // every contributor's partial in one batch
    float* acc = area;
    float* stage = area + blk;
    const int cb = min(C, (cap - blk) / blk);
    sm100::fence_proxy_async_smem();   // the ring's last reads were the tensor cores'
#pragma unroll 1
    for (int c0 = 0; c0 < C; c0 += cb) {
      const int cn = min(cb, C - c0);
      stage_block(stage, part + static_cast<size_t>(c0) * blk, cn * blk, et);
      cp_async_wait_all();
      sm100::named_barrier(1, EPI_THREADS);
#pragma unroll 1
      for (int i = 4 * et; i < blk; i += 4 * EPI_THREADS) {
        float4 a = c0 == 0 ? *reinterpret_cast<const float4*>(stage + i) : *reinterpret_cast<const float4*>(acc + i);
#pragma unroll 4
        for (int c = c0 == 0 ? 1 : 0; c < cn; ++c) {
          const float4 x = *reinterpret_cast<const float4*>(stage + static_cast<size_t>(c) * blk + i);
          a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
        }
        *reinterpret_cast<float4*>(acc + i) = a;
      }
      sm100::named_barrier(1, EPI_THREADS);
    }
    for (int jc = 0; jc < p.n; jc += p.xr) {
      const int nj = min(p.xr, p.n - jc);
      if (jc > 0) stage_row_inputs(p, s, t, jc, nj, m);   // chunk 0's row inputs were staged early
#pragma unroll 1
      for (int jj = 0; jj < nj; ++jj) xch[jj * BM + m] = acc[(jc + jj) * BM + m];
      sm100::named_barrier(1, EPI_THREADS);
      epilogue_chunk(p, s, col, t, jc, nj, m);
    }
    return;
  }
  for (int jc = 0; jc < p.n; jc += p.xr) {
    const int nj = min(p.xr, p.n - jc);
    // 0. the chunk's row inputs, by asynchronous copies that land while the
    //    partials below are read (chunk 0's were staged early)
    if (jc > 0) stage_row_inputs(p, s, t, jc, nj, m);
    // 1. partials of the contributing CTAs (each one contiguous block of nj
    //    rows), read straight from L2 16 rows x four CTAs at a time (64
    //    independent loads in flight per thread, where staging them CTA by
    //    CTA cost one round trip and a barrier each) and summed in CTA order
#pragma unroll 1
    for (int h = 0; h < nj; h += 16) {
      const int nh = min(16, nj - h);
      const float* src = part + static_cast<size_t>(jc + h) * BM + m;
      float a[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) a[jj] = jj < nh ? __ldcg(src + jj * BM) : 0.f;
#pragma unroll 4
      for (int c = 1; c < C; ++c) {
        const float* sc = src + static_cast<size_t>(c) * blk;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          if (jj < nh) a[jj] += __ldcg(sc + jj * BM);
      }
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        if (jj < nh) xch[(h + jj) * BM + m] = a[jj];
    }
    sm100::named_barrier(1, EPI_THREADS);
    epilogue_chunk(p, s, col, t, jc, nj, m);
  }
}

// Cooperative final epilogue of split tile t (p.coop): every one of its C
// contributors, once all C partials are written, sums them (in CTA order, as
// finalize_tile does) for its own share [r0, r1) of the activation rows and
// runs the fused elementwise work on those rows, so the tile's epilogue is
// spread over its C CTAs instead of waiting on one.  Rows below xr were
// staged at the segment's start.
__device__ __noinline__ void finalize_rows(const GemmParams& p, const Smem& s, const EpiCol& col, int t,
                                           int c_first, int C, int m, int r0, int r1) {
  const int blk = p.n * BM;
  const float* part = p.part + static_cast<size_t>(t + c_first) * blk;
  float* const xch = s.xch;
  for (int jc = r0; jc < r1; jc += p.xr) {
    const int nj = min(p.xr, r1 - jc);
    if (jc > 0) stage_row_inputs(p, s, t, jc, nj, m);
#pragma unroll 1
    for (int h = 0; h < nj; h += 16) {
      const int nh = min(16, nj - h);
      const float* src = part + static_cast<size_t>(jc + h) * BM + m;
      float a[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) a[jj] = jj < nh ? __ldcg(src + jj * BM) : 0.f;
#pragma unroll 4
      for (int c = 1; c < C; ++c) {
        const float* sc = src + static_cast<size_t>(c) * blk;
#pragma unroll
        for (int jj = 0; jj < 16; ++jj)
          if (jj < nh) a[jj] += __ldcg(sc + jj * BM);
      }
#pragma unroll
      for (int jj = 0; jj < 16; ++jj)
        if (jj < nh) xch[(h + jj) * BM + m] = a[jj];
    }
    sm100::named_barrier(1, EPI_THREADS);
    epilogue_chunk(p, s, col, t, jc, nj, m);
  }
}

// Tensor maps of one launch: the (up to three) weight matrices as 4-D
// grouped maps, their 2-D tail maps, and the activation operand.
struct GemmMaps {
  const CUtensorMap *a0, *a1, *a2, *t0, *t1, *t2, *b;
};

// Weight rows of unit u into ring slot st (two 64-row halves).
__device__ __forceinline__ void issue_a(const GemmParams& p, const Smem& s, const GemmMaps& mp, long long u, int st,
                                        uint64_t policy) {
  const uint32_t group_bytes = static_cast<uint32_t>(p.kps) * 1024u;
  const int t = static_cast<int>(u / p.kb), kz = static_cast<int>(u % p.kb) * p.kps;
  uint8_t* a_dst = s.a + static_cast<size_t>(st) * p.a_stage_bytes;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    int map, row;
    locate_box(p, t, h, map, row);
    uint8_t* dst = a_dst + h * 8 * group_bytes;
    if (row + 64 <= p.full_rows[map] && kz + p.kps <= p.full_kb) {
      const CUtensorMap* m4 = map == 0 ? mp.a0 : (map == 1 ? mp.a1 : mp.a2);
      sm100::tma_load_4d_hint(dst, m4, 0, 0, kz, row >> 3, &s.full[st], policy);
    } else {                                     // row or K tail: 8-row x 64-k boxes, zero past the end
      const CUtensorMap* m2 = map == 0 ? mp.t0 : (map == 1 ? mp.t1 : mp.t2);
#pragma unroll 1
      for (int g = 0; g < 8; ++g)
        for (int c = 0; c < p.kps; ++c)
          sm100::tma_load_2d_hint(dst + g * group_bytes + c * 1024, m2, (kz + c) * BK, row + 8 * g, &s.full[st],
                                  policy);
    }
  }
}

// Activation rows (the previous kernel's output) of unit u into slot st.
__device__ __forceinline__ void issue_b(const GemmParams& p, const Smem& s, const GemmMaps& mp, long long u, int st) {
  const int kz = static_cast<int>(u % p.kb) * p.kps;
  sm100::tma_load_4d(s.b + static_cast<size_t>(st) * p.b_stage_bytes, mp.b, 0, 0, kz, 0, &s.full[st]);
}

__device__ __forceinline__ long long first_ring(const GemmParams& p, const CtaWork& wk) {
  return min(static_cast<long long>(p.stages), wk.n_units(p));
}

// TMA producer (warp 0; lane 0 issues) over the CTA's units in order.  The
// first ring's weights do not depend on the previous kernel: they stream
// while it drains.  Their activation boxes are issued by warp 2
// (gemm_produce_first_b) as soon as the previous kernel has completed, so a
// CTA that starts late is not held up behind its own weight requests.
__device__ __forceinline__ void gemm_produce(const GemmParams& p, const Smem& s, const GemmMaps& mp, int lane,
                                             const CtaWork& wk, volatile int* abort_flag, const LaunchStamp& ls) {
  const long long nv = wk.n_units(p);
  const long long n_pre = first_ring(p, wk);
  if (lane == 0)
    for (long long i = 0; i < n_pre; ++i)
      sm100::mbar_arrive_expect_tx(&s.full[i], p.a_stage_bytes + p.b_stage_bytes);
  __syncwarp();
  sm100::named_barrier_arrive(2, 64);          // the first ring's expected bytes are set
  if (lane != 0) return;
  const uint64_t policy = sm100::l2_policy_evict_first();   // weights are read once per launch
  for (long long i = 0; i < n_pre; ++i) issue_a(p, s, mp, wk.unit(p, i), static_cast<int>(i), policy);
  pdl_wait();
  ls.waited();
  long long issued = n_pre;
  int stage = static_cast<int>(n_pre % p.stages);
  uint32_t phase = n_pre == p.stages ? 1u : 0u;
  for (long long v = n_pre; v < nv; ++v) {
    const long long u = wk.unit(p, v);
    if (!sm100::mbar_wait(&s.empty[stage], phase ^ 1u, abort_flag)) {
      *abort_flag = 1;
      set_status(p.status, EAGLE_ERR_TIMEOUT);
      break;
    }
    sm100::mbar_arrive_expect_tx(&s.full[stage], p.a_stage_bytes + p.b_stage_bytes);
    issue_a(p, s, mp, u, stage, policy);
    issue_b(p, s, mp, u, stage);
    ++issued;
    if (++stage == p.stages) { stage = 0; phase ^= 1u; }
  }
  if (*abort_flag) {
    // let copies already in flight land before the CTA exits
    const long long pending = issued < p.stages ? issued : p.stages;
    for (long long i = 0; i < pending; ++i) {
      stage = stage == 0 ? p.stages - 1 : stage - 1;
      if (stage == p.stages - 1) phase ^= 1u;
      const uint64_t t0 = globaltimer_ns();
      while (!sm100::mbar_try_wait(&s.full[stage], phase) && globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
      }
    }
  }
}

// Warp 2, before its epilogue work: the activation boxes of the first ring.
__device__ __forceinline__ void gemm_produce_first_b(const GemmParams& p, const Smem& s, const GemmMaps& mp, int lane,
                                                     const CtaWork& wk) {
  sm100::named_barrier(2, 64);                 // warp 0 has set the expected bytes
  if (lane == 0) {
    pdl_wait();
    const long long n_pre = first_ring(p, wk);
    for (long long i = 0; i < n_pre; ++i) issue_b(p, s, mp, wk.unit(p, i), static_cast<int>(i));
  }
  __syncwarp();
}

// One MMA from 32-bit shared-memory descriptor words: lo = (address >> 4) |
// (leading byte offset >> 4) << 16, hi = the stride / version / swizzle word
// shared by both operands (an operand that many bytes on is lo + bytes >> 4:
// the 14-bit address field never carries, shared memory ending below 256 KB).
__device__ __forceinline__ void mma_lo_hi(uint32_t d_tmem, uint32_t alo, uint32_t blo, uint32_t hi, uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 a, b;\n setp.ne.b32 p, %5, 0;\n mov.b64 a, {%1, %3};\n mov.b64 b, {%2, %3};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(alo), "r"(blo), "r"(hi), "r"(idesc), "r"(acc));
}

// MMA issuer (warp 1, lane 0): one accumulator per tile segment of the
// CTA's work, double-buffered in tensor memory when two fit.  The issuing
// loop is kept lean -- descriptor words advanced by adds, every MMA's offset
// within a stage a constant, the stage shape (KPS2: two k-blocks per stage;
// TWO: the hi and lo halves as separate MMAs) a template parameter with no
// branch between MMAs -- since the MMAs issue only as fast as this thread
// reaches them (a runtime test of either flag between the MMAs doubled the
// issue time per MMA).
template <bool KPS2, bool TWO>
__device__ __forceinline__ void gemm_mma_loop(const GemmParams& p, const Smem& s, uint32_t tmem_base,
                                              const CtaWork& wk, volatile int* abort_flag) {
  const uint32_t n_total = 2u * p.NP;
  const uint32_t idesc = TWO ? sm100::idesc_bf16_f32(BM, p.NP) : sm100::idesc_bf16_f32(BM, n_total);
  const uint32_t sbo = static_cast<uint32_t>(p.kps) * 1024u;
  const uint32_t hi = ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
  const uint32_t a_lo0 = ((sm100::smem_u32(s.a) >> 4) & 0x3FFFu) | (1u << 16);   // stage 0; leading byte offset 16
  const uint32_t b_lo0 = ((sm100::smem_u32(s.b) >> 4) & 0x3FFFu) | (1u << 16);
  const uint32_t a_step = p.a_stage_bytes >> 4, b_step = p.b_stage_bytes >> 4;
  const uint32_t b2 = (static_cast<uint32_t>(p.NP >> 3) * sbo) >> 4;          // second activation half
  uint32_t a_lo = a_lo0, b_lo = b_lo0;                                           // the current stage's words
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  int t;
  long long v0, v1;
  for (int seg = 0; ok && wk.segment(p, seg, t, v0, v1); ++seg) {
    const int buf = seg % p.n_acc;
    const uint32_t aph = static_cast<uint32_t>(seg / p.n_acc) & 1u;
    if (!sm100::mbar_wait(&s.tempty[buf], aph ^ 1u, abort_flag)) {
      *abort_flag = 1;
      set_status(p.status, EAGLE_ERR_TIMEOUT);
      break;
    }
    sm100::tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * p.acc_stride);
    for (long long v = v0; v < v1; ++v) {
      if (!sm100::mbar_wait(&s.full[stage], phase, abort_flag)) {
        *abort_flag = 1;
        set_status(p.status, EAGLE_ERR_TIMEOUT);
        ok = false;
        break;
      }
      sm100::tc_fence_after();
      const uint32_t first = v != v0 ? 1u : 0u;        // only the segment's first MMA starts the sum
      // k-block c, step kk: offset c * 1024 + kk * 32 bytes in both operands
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (c == 1 && !KPS2) break;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((c * 1024 + kk * 32) >> 4);
          const uint32_t acc = (c > 0 || kk > 0) ? 1u : first;
          mma_lo_hi(d_tmem, a_lo + off, b_lo + off, hi, idesc, acc);
          if (TWO) mma_lo_hi(d_tmem + p.NP, a_lo + off, b_lo + b2 + off, hi, idesc, acc);
        }
      }
      sm100::mma_commit(&s.empty[stage]);
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
        a_lo = a_lo0;
        b_lo = b_lo0;
      } else {
        a_lo += a_step;
        b_lo += b_step;
      }
    }
    if (!ok) break;
    sm100::mma_commit(&s.tfull[buf]);
  }
}

__device__ __forceinline__ void gemm_mma(const GemmParams& p, const Smem& s, int lane, uint32_t tmem_base,
                                         const CtaWork& wk, volatile int* abort_flag) {
  if (lane != 0) return;
  if (p.kps == 2) {
    if (p.two_mma) gemm_mma_loop<true, true>(p, s, tmem_base, wk, abort_flag);
    else gemm_mma_loop<true, false>(p, s, tmem_base, wk, abort_flag);
  } else {
    if (p.two_mma) gemm_mma_loop<false, true>(p, s, tmem_base, wk, abort_flag);
    else gemm_mma_loop<false, false>(p, s, tmem_base, wk, abort_flag);
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 2)
    gemm_stream_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
                       const __grid_constant__ CUtensorMap mA2, const __grid_constant__ CUtensorMap mT0,
                       const __grid_constant__ CUtensorMap mT1, const __grid_constant__ CUtensorMap mT2,
                       const __grid_constant__ CUtensorMap mB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const Smem s = carve(smem_raw, p);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const CtaWork wk = cta_work(p);
  const long long U_sk = static_cast<long long>(p.sk_tiles) * p.kb;
  volatile int* abort_flag = s.flags;
  const GemmMaps maps{&mA0, &mA1, &mA2, &mT0, &mT1, &mT2, &mB};
  const LaunchStamp ls(p.stamp);
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      sm100::mbar_init(&s.full[i], 1);
      sm100::mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      sm100::mbar_init(&s.tfull[i], 1);
      sm100::mbar_init(&s.tempty[i], 4);
    }
    s.flags[0] = 0;
    s.flags[1] = 0;
    s.flags[2] = 0;
    sm100::fence_barrier_init();
    sm100::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    sm100::tma_prefetch_desc(&mA0);
    if (p.n_mats > 1) sm100::tma_prefetch_desc(&mA1);
    if (p.n_mats > 2) sm100::tma_prefetch_desc(&mA2);
    sm100::tma_prefetch_desc(&mB);
  }
  if (warp == 1) {
    sm100::tmem_alloc(s.tmem_holder, p.tmem_cols);
    sm100::tmem_relinquish();
  }
  sm100::tc_fence_before();
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem_base = *s.tmem_holder;

  if (warp == 0) {
    gemm_produce(p, s, maps, lane, wk, abort_flag, ls);
    __syncwarp();
  } else if (warp == 1) {
    gemm_mma(p, s, lane, tmem_base, wk, abort_flag);
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    if (warp == 2) gemm_produce_first_b(p, s, maps, lane, wk);
    pdl_wait();                                 // residuals, norms, positions of earlier kernels
    const int et = threadIdx.x - 64;            // 0..127
    const int quarter = warp & 3;               // tensor-memory lanes this warp may read
    const int m = quarter * 32 + lane;          // tile row held by this thread
    int t;
    long long v0, v1;
    for (int seg = 0; wk.segment(p, seg, t, v0, v1); ++seg) {
      const int buf = seg % p.n_acc;
      const uint32_t aph = static_cast<uint32_t>(seg / p.n_acc) & 1u;
      // While the tile streams: its epilogue constants and the first row
      // chunk's inputs from earlier kernels.
      const EpiCol col = epi_column(p, t, m);
      cp_async_wait_all();                      // the previous segment's copies into s.stg2 have landed
      sm100::named_barrier(1, EPI_THREADS);
      stage_row_inputs(p, s, t, 0, min(p.xr, p.n), m);
      if (et == 0) s.flags[2] = sm100::mbar_wait(&s.tfull[buf], aph, abort_flag) ? 1 : 0;
      sm100::named_barrier(1, EPI_THREADS);
      if (!s.flags[2]) {
        if (et == 0) {
          *abort_flag = 1;
          set_status(p.status, EAGLE_ERR_TIMEOUT);
        }
        cp_async_wait_all();
        break;
      }
      sm100::tc_fence_after();
      const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(buf * p.acc_stride);
      int c_first = cta, c_last = cta;
      if (t < p.sk_tiles && !p.sk_whole) {
        c_first = cta_of_unit(static_cast<long long>(t) * p.kb, U_sk, G);
        c_last = cta_of_unit(static_cast<long long>(t) * p.kb + p.kb - 1, U_sk, G);
      }
      if (c_first == c_last && p.n_acc == 1 && t >= p.sk_tiles && t + G < p.m_tiles) {
        // the whole tile is this CTA's and its only accumulator is wanted by
        // the CTA's next tile: the summed accumulator goes to this CTA's own
        // slot in global memory at once, freeing tensor memory for the next
        // tile's MMAs while the epilogue runs from the slot
        const int slot = p.sk_tiles + G + cta;
        for (int c0 = 0; c0 < p.NP; c0 += 8) {
          float hi[8], lo[8];
          sm100::tmem_ld8(lane_addr + c0, hi);
          sm100::tmem_ld8(lane_addr + p.NP + c0, lo);
          sm100::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int j = c0 + i;
            if (j < p.n) p.part[(static_cast<size_t>(slot) * p.n + j) * BM + m] = hi[i] + lo[i];
          }
        }
        sm100::tc_fence_before();
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(&s.tempty[buf]);
        // each thread reads back only what it wrote (its tile row m)
        finalize_rows(p, s, col, t, slot - t, 1, m, 0, p.n);
        sm100::named_barrier(1, EPI_THREADS);
        continue;
      }
      if (c_first == c_last) {
        // the whole tile is this CTA's: epilogue straight from tensor memory
        for (int jc = 0; jc < p.n; jc += p.xr) {
          const int nj = min(p.xr, p.n - jc);
          // this chunk's row inputs stream in while its accumulators are read
          // (chunk 0's were staged before the accumulators were ready)
          if (jc > 0) stage_row_inputs(p, s, t, jc, nj, m);
          for (int c0 = 0; c0 < nj; c0 += 8) {
            float hi[8], lo[8];
            sm100::tmem_ld8(lane_addr + jc + c0, hi);
            sm100::tmem_ld8(lane_addr + p.NP + jc + c0, lo);
            sm100::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (c0 + i < nj) s.xch[(c0 + i) * BM + m] = hi[i] + lo[i];
          }
          sm100::named_barrier(1, EPI_THREADS);
          epilogue_chunk(p, s, col, t, jc, nj, m);
        }
        sm100::tc_fence_before();
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(&s.tempty[buf]);
        continue;
      }
      const int slot = t + cta;
      for (int c0 = 0; c0 < p.NP; c0 += 8) {
        float hi[8], lo[8];
        sm100::tmem_ld8(lane_addr + c0, hi);
        sm100::tmem_ld8(lane_addr + p.NP + c0, lo);
        sm100::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int j = c0 + i;
          if (j < p.n) p.part[(static_cast<size_t>(slot) * p.n + j) * BM + m] = hi[i] + lo[i];
        }
      }
      sm100::tc_fence_before();
      __syncwarp();
      if (lane == 0) sm100::mbar_arrive(&s.tempty[buf]);
      sm100::named_barrier(1, EPI_THREADS);     // every epilogue thread's partial stores come first
      if (p.coop) {
        // The contributors for which tile t is their last segment wait for
        // every partial, then finalize a share of its activation rows each;
        // the one whose work continues past the tile (the last contributor,
        // unless it stops inside it) only arrives.  The counter counts C
        // arrivals, then the W waiters' departures; the last one resets it.
        const int C = c_last - c_first + 1;
        const long long end_last = static_cast<long long>(c_last + 1) * U_sk / G;   // c_last's share ends here
        const int lastw = end_last <= static_cast<long long>(t + 1) * p.kb ? c_last : c_last - 1;
        const int W = lastw - c_first + 1;
        if (cta > lastw) {
          if (et == 0) arrive_acq_rel(&p.counters[t]);
          continue;
        }
        if (et == 0) {
          arrive_acq_rel(&p.counters[t]);
          const uint64_t w0 = globaltimer_ns();
          int ok = 1;
          while (ld_acquire(&p.counters[t]) < C) {
            if (*abort_flag || globaltimer_ns() - w0 > WAIT_LIMIT_NS) {
              ok = 0;
              break;
            }
            __nanosleep(64);
          }
          s.flags[1] = ok;
        }
        sm100::named_barrier(1, EPI_THREADS);
        if (!s.flags[1]) {
          if (et == 0) {
            *abort_flag = 1;
            set_status(p.status, EAGLE_ERR_TIMEOUT);
          }
          cp_async_wait_all();
          break;
        }
        const int ci = cta - c_first;
        const int r0 = static_cast<int>(static_cast<long long>(ci) * p.n / W);
        const int r1 = static_cast<int>(static_cast<long long>(ci + 1) * p.n / W);
        if (r0 < r1) finalize_rows(p, s, col, t, c_first, C, m, r0, r1);
        sm100::named_barrier(1, EPI_THREADS);
        if (et == 0 && arrive_acq_rel(&p.counters[t]) == C + W - 1) p.counters[t] = 0;
        continue;
      }
      if (et == 0) {
        const int prev = arrive_acq_rel(&p.counters[t]);
        const int last = prev == c_last - c_first;
        if (last) p.counters[t] = 0;
        s.flags[1] = last;
      }
      sm100::named_barrier(1, EPI_THREADS);
      if (s.flags[1]) {
        // on the CTA's last tile the pipeline ring is idle: all of its loads
        // were consumed by MMAs that have completed
        int t2;
        long long w0, w1;
        const bool last_seg = !wk.segment(p, seg + 1, t2, w0, w1);
        float* area = last_seg ? reinterpret_cast<float*>(s.a) : nullptr;
        const int cap = static_cast<int>(static_cast<size_t>(p.stages) * (p.a_stage_bytes + p.b_stage_bytes) / 4);
        finalize_tile(p, s, col, t, c_first, c_last, m, area, cap);
      }
      sm100::named_barrier(1, EPI_THREADS);
    }
    cp_async_wait_all();                        // no copy may land after the CTA has left
  }
  __syncthreads();
  if (warp == 1) {
    sm100::tc_fence_after();
    sm100::tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// [rows][ld] bf16 matrix seen as {64 k, 8 rows, k-block, 8-row group} over
// its whole k-blocks and whole 8-row groups only (every element the map can
// address lies inside the used [rows][K] extent); box = kps k-blocks x
// box_groups groups.
bool encode_grouped(eagle_ctx* ctx, CUtensorMap* map, const void* ptr, int K, int rows, int ld_elems, int kps,
                    int box_groups) {
  const int groups = rows / 8 > 0 ? rows / 8 : 1;   // a dimension under one unit is never addressed
  const int kblocks = K / BK > 0 ? K / BK : 1;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(BK), 8, static_cast<cuuint64_t>(kblocks),
                        static_cast<cuuint64_t>(groups)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(ld_elems) * 2, KBLK_BYTES,
                           static_cast<cuuint64_t>(ld_elems) * 16};
  cuuint32_t box[4] = {BK, 8, static_cast<cuuint32_t>(kps), static_cast<cuuint32_t>(box_groups)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The used [rows][K] extent as a 2-D map; box = 64 k x 8 rows (elements
// past K or past the last row read as zero).
bool encode_tail(eagle_ctx* ctx, CUtensorMap* map, const void* ptr, int K, int rows, int ld_elems) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_elems) * 2};
  cuuint32_t box[2] = {BK, 8};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = ctx->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(eagle_ctx* ctx, int epi, const DraftLaunch& L, cudaStream_t st) {
  const eagle_dims& D = ctx->dims;
  const Workspace& W = ctx->ws;
  const eagle_draft_weights* w = L.w;
  const int qd = D.n_q_heads * D.head_dim, kd = D.n_kv_heads * D.head_dim;
  GemmParams p{};
  p.epi = epi;
  p.n = L.n;
  p.NP = L.NP;
  p.rpr = L.rpr;
  p.e0 = L.e0;
  p.E = ctx->lim.max_expanded;
  p.d = D.d;
  p.F = D.d_ff;
  p.V = D.vocab;
  p.Hq = D.n_q_heads;
  p.Hkv = D.n_kv_heads;
  p.dh = D.head_dim;
  p.eps = D.rms_eps;
  p.ln_theta = log(static_cast<double>(D.rope_theta));
  p.status = ws_ptr<int>(L.ws, W.status);
  p.part = ws_ptr<float>(L.ws, W.gemm_part);
  p.counters = ws_ptr<int>(L.ws, W.gemm_cnt) + epi * W.max_mtiles;
  const int tiles_d = ceil_div(D.d, BM);

  const uint16_t* mats[3] = {nullptr, nullptr, nullptr};
  int rows[3] = {0, 0, 0}, lds[3] = {0, 0, 0};
  int K = 0, kp_in = 0;
  size_t b_in = 0;
  int n_out = 0;
  switch (epi) {
    case EPI_FC:
      mats[0] = w->w_fc; rows[0] = D.d; lds[0] = w->ld_fc; K = 2 * D.d;
      b_in = W.b_fc; kp_in = W.kp_fc; n_out = D.d;
      p.bias = w->b_fc; p.gain = w->g1;
      p.out_f32 = ws_ptr<float>(L.ws, W.h);
      p.bnext = ws_ptr<uint16_t>(L.ws, W.b_qkv); p.kp_next = W.kp_qkv;
      p.ss_out = ws_ptr<float>(L.ws, W.ss_fc);
      break;
    case EPI_QKV:
      mats[0] = w->wq; rows[0] = qd; lds[0] = w->ld_q;
      mats[1] = w->wk; rows[1] = kd; lds[1] = w->ld_k;
      mats[2] = w->wv; rows[2] = kd; lds[2] = w->ld_v;
      K = D.d; b_in = W.b_qkv; kp_in = W.kp_qkv; n_out = qd + 2 * kd;
      p.ss_in = ws_ptr<float>(L.ws, W.ss_fc); p.ss_in_tiles = tiles_d;
      p.qrow = ws_ptr<float>(L.ws, W.qrow);
      p.k_tree = L.out->k_tree; p.v_tree = L.out->v_tree;
      p.pos0 = L.req->pos0; p.depth = L.pool->depth;
      break;
    case EPI_O:
      mats[0] = w->wo; rows[0] = D.d; lds[0] = w->ld_o; K = qd;
      b_in = W.b_o; kp_in = W.kp_o; n_out = D.d;
      p.gain = w->g2;
      p.resid = ws_ptr<float>(L.ws, W.h);
      p.out_f32 = ws_ptr<float>(L.ws, W.h2);
      p.bnext = ws_ptr<uint16_t>(L.ws, W.b_gu); p.kp_next = W.kp_gu;
      p.ss_out = ws_ptr<float>(L.ws, W.ss_o);
      break;
    case EPI_GATEUP:
      mats[0] = w->w_gate; rows[0] = D.d_ff; lds[0] = w->ld_gate;
      mats[1] = w->w_up; rows[1] = D.d_ff; lds[1] = w->ld_up;
      K = D.d; b_in = W.b_gu; kp_in = W.kp_gu; n_out = 2 * D.d_ff;
      p.ss_in = ws_ptr<float>(L.ws, W.ss_o); p.ss_in_tiles = tiles_d;
      p.bnext = ws_ptr<uint16_t>(L.ws, W.b_down); p.kp_next = W.kp_down;
      break;
    case EPI_DOWN:
      mats[0] = w->w_down; rows[0] = D.d; lds[0] = w->ld_down; K = D.d_ff;
      b_in = W.b_down; kp_in = W.kp_down; n_out = D.d;
      p.resid = ws_ptr<float>(L.ws, W.h2);
      p.out_f32 = L.out->f_hat;
      p.bnext = ws_ptr<uint16_t>(L.ws, W.b_lm); p.kp_next = W.kp_lm;
      break;
    case EPI_KV:
      mats[0] = w->wk; rows[0] = kd; lds[0] = w->ld_k;
      mats[1] = w->wv; rows[1] = kd; lds[1] = w->ld_v;
      K = D.d; b_in = W.b_qkv; kp_in = W.kp_qkv; n_out = 2 * kd;
      p.ss_in = ws_ptr<float>(L.ws, W.ss_fc); p.ss_in_tiles = tiles_d;
      p.pos0 = L.req->pos0;
      p.kc = L.refresh_kv->k; p.vc = L.refresh_kv->v;
      p.kv_cap_rows = L.refresh_kv->cap; p.kv_len = L.refresh_kv->len;
      p.n_act = L.refresh_n;
      break;
    case EPI_FUSE:
      mats[0] = L.w_fuse; rows[0] = D.d; lds[0] = L.ld_fuse; K = 3 * D.d;
      b_in = W.b_fuse; kp_in = W.kp_fuse; n_out = D.d;
      p.bias = L.b_fuse;
      p.out_f32 = L.g_out;
      break;
    default:  // EPI_LM
      mats[0] = w->w_lm; rows[0] = D.vocab; lds[0] = w->ld_lm; K = D.d;
      b_in = W.b_lm; kp_in = W.kp_lm; n_out = D.vocab;
      p.out_f32 = L.out->logits;
      break;
  }
  p.n_mats = epi == EPI_QKV ? 3 : (epi == EPI_GATEUP || epi == EPI_KV ? 2 : 1);
  int cum = 0;
  for (int i = 0; i < p.n_mats; ++i) {
    cum += ceil_div(rows[i], 64);
    p.mblk[i] = cum;
  }
  p.m_tiles = epi == EPI_GATEUP ? ceil_div(D.d_ff, 64) : ceil_div(n_out, BM);
  p.two_mma = 2 * p.NP > 256 ? 1 : 0;
  for (int i = 0; i < 3; ++i) p.full_rows[i] = i < p.n_mats ? rows[i] / 8 * 8 : 0;
  p.full_kb = K / BK;
  p.xr = p.n > 16 ? XCH_MAX : 16;
  const int sw = p.ss_in_tiles + 1 > BM ? p.ss_in_tiles + 1 : BM;
  const int acc_cols = 2 * p.NP;
  p.acc_stride = acc_cols < 32 ? 32 : (acc_cols + 31) / 32 * 32;
  p.n_acc = 2 * p.acc_stride <= 512 ? 2 : 1;
  const int need = p.n_acc * p.acc_stride;
  int cols = 32;
  while (cols < need) cols <<= 1;
  p.tmem_cols = cols;
  // Contractions with fewer tiles than SMs (every tile split) run two CTAs
  // per SM with half-size rings when two fit (shared memory and tensor
  // memory): a CTA of the next kernel can then start on an SM as soon as one
  // of the two leaves, instead of waiting for the SM's last finalizing CTA.
  // The others keep one CTA per SM (whole tiles of their own at the end).
  const size_t half_cap = static_cast<size_t>(113) * 1024;
  const int per_sm = p.m_tiles < ctx->sm_count && cols <= 256 &&
                     smem_bytes_for(2, BM * KBLK_BYTES, 2 * p.NP * KBLK_BYTES, p.xr, sw) <= half_cap ? 2 : 1;
  const size_t smem_cap = per_sm == 2 ? half_cap : 232448;
  const int min_ring = per_sm == 2 ? 2 : 3;
  // two k-blocks per stage while that still leaves a ring of min_ring stages
  p.kps = smem_bytes_for(min_ring, BM * KBLK_BYTES * 2, 2 * p.NP * KBLK_BYTES * 2, p.xr, sw) <= smem_cap ? 2 : 1;
  p.a_stage_bytes = static_cast<uint32_t>(BM * KBLK_BYTES * p.kps);
  p.b_stage_bytes = static_cast<uint32_t>(2 * p.NP * KBLK_BYTES * p.kps);
  p.kb = ceil_div(K, BK * p.kps);
  p.total_units = static_cast<long long>(p.m_tiles) * p.kb;

  int stages = 8;
  while (stages > 2 && smem_bytes_for(stages, p.a_stage_bytes, p.b_stage_bytes, p.xr, sw) > smem_cap) --stages;
  p.stages = stages;
  size_t smem = smem_bytes_for(stages, p.a_stage_bytes, p.b_stage_bytes, p.xr, sw);
  if (smem > smem_cap) return cudaErrorInvalidConfiguration;
  if (per_sm == 1 && smem < 120 * 1024) smem = 120 * 1024;    // keeps one CTA per SM

  CUtensorMap maps[3], tails[3], mb;
  for (int i = 0; i < 3; ++i) {
    const int src = i < p.n_mats ? i : 0;
    if (!encode_grouped(ctx, &maps[i], mats[src], K, rows[src], lds[src], p.kps, 8)) return cudaErrorInvalidValue;
    if (!encode_tail(ctx, &tails[i], mats[src], K, rows[src], lds[src])) return cudaErrorInvalidValue;
  }
  if (!encode_grouped(ctx, &mb, ws_ptr<uint16_t>(L.ws, b_in), kp_in, 2 * p.NP, kp_in, p.kps, 2 * p.NP / 8))
    return cudaErrorInvalidValue;

  {
    const cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(gemm_stream_kernel), 232448);
    if (e != cudaSuccess) return e;
  }
  int grid = per_sm * ctx->sm_count;
  if (p.total_units < grid) grid = static_cast<int>(p.total_units);
  // whole waves of tiles go data-parallel at the end of every CTA's work;
  // the remaining tiles are split stream-K and processed first
  p.dp_waves = p.m_tiles / grid;
  p.sk_tiles = p.m_tiles - p.dp_waves * grid;
  p.sk_whole = p.sk_tiles > 0 && static_cast<long long>(p.sk_tiles) * p.kb < grid ? 1 : 0;
  // the split tiles' contributors wait for one another only when every tile
  // is split (no data-parallel tiles follow a CTA's split ones) and the whole
  // grid is resident at once; else the last arriver finalizes alone
  {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemm_stream_kernel, NUM_THREADS, smem) != cudaSuccess)
      occ = 0;
    p.coop = p.dp_waves == 0 && occ >= per_sm && grid <= occ * ctx->sm_count ? 1 : 0;
  }
  // partial slots t + cta of split tiles, and sk_tiles + grid + cta of the
  // own tiles' accumulators (one accumulator, more than one own tile), stay
  // inside the workspace's array
  if (p.sk_tiles > 0 && p.sk_tiles - 1 + grid - 1 >= W.max_mtiles + 2 * ctx->sm_count)
    return cudaErrorInvalidConfiguration;
  if (p.n_acc == 1 && p.dp_waves > 1 && p.sk_tiles + 2 * grid - 1 >= W.max_mtiles + 2 * ctx->sm_count)
    return cudaErrorInvalidConfiguration;
  const int kid = epi == EPI_KV ? static_cast<int>(EAGLE_K_REFRESH)
                                 : (epi == EPI_FUSE ? static_cast<int>(EAGLE_K_FUSE) : epi);
  p.stamp = stamp_slot(ctx, kid);
  trace_before(ctx, kid, st);
  const cudaError_t e = launch_pdl(gemm_stream_kernel, dim3(grid), dim3(NUM_THREADS), smem, st, maps[0], maps[1],
                                   maps[2], tails[0], tails[1], tails[2], mb, p);
  ctx->launches++;
  trace_after(ctx, kid, st);
  return e;
}

}  // namespace eagle
