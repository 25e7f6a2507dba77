// The commit transaction ([B] "KV Cache 必须按事务提交"; [A] §6.2 closing remark,
// §12 item 3): the root and the accepted path become authoritative, rejected
// branches are dropped by not copying them.  One CTA per (request, path
// position): it copies that slot's K/V row of every target layer into the
// cache at position L_b + i and gathers its true feature.  One more CTA per
// request, running beside them, writes the next round's state and appends
// the root's draft K/V row.
#include "internal.h"
#include "common.cuh"
#include "sm100.cuh"

namespace eagle {
namespace {

struct CommitParams {
  int n_layers, kv_cap, S, E, d, row_elems, path_cap, draft_cap;
  PagedKv paged;                  // target caches through a block table (table null: contiguous)
  const uint16_t* kt[EAGLE_MAX_LAYERS];
  const uint16_t* vt[EAGLE_MAX_LAYERS];
  uint16_t* kc[EAGLE_MAX_LAYERS];
  uint16_t* vc[EAGLE_MAX_LAYERS];
  const int32_t* accept_len;
  const int32_t* path;
  const int32_t* final_token;
  const int32_t* last_slot;
  const int32_t* t_token;
  const float* f_true;
  const int32_t* kv_len;
  const float* dk_tree;
  const float* dv_tree;
  uint16_t* dk;
  uint16_t* dv;
  const int32_t* draft_len;
  float* f_commit;
  int32_t* tok_commit;
  float* f_last;
  int32_t* t_next;
  int32_t* prefix_len_out;
  int32_t* draft_len_out;
  int* status;
  uint64_t* stamp;
};

// rows are whole multiples of 8 bf16 (16 bytes)
__device__ __forceinline__ void copy_row(uint16_t* dst, const uint16_t* src, int elems) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int i = threadIdx.x; i < elems / 8; i += blockDim.x) d4[i] = s4[i];
}

__global__ void commit_kernel(const CommitParams p) {
  const LaunchStamp ls(p.stamp);
  pdl_wait();      // predecessor outputs visible from here on
  ls.waited();
  pdl_trigger();
  const int b = blockIdx.x, i = blockIdx.y;
  const int a = p.accept_len[b];
  const int L = p.kv_len[b];
  // a request whose cache cannot take the path commits nothing (checked
  // alike by every CTA of the request; the state CTA reports it): the rows
  // L .. L + a must exist and, in a paged cache, lie in allocated blocks
  bool room = L >= 0 && static_cast<long long>(L) + 1 + a <= p.kv_cap;
  if (room && p.paged.table)
    for (int pos = L; room && pos <= L + a; pos = ((pos >> p.paged.shift) + 1) << p.paged.shift)
      room = paged_row(p.paged, b, pos) >= 0;
  const bool draft_room = p.dk == nullptr || (p.draft_len[b] >= 0 && p.draft_len[b] < p.draft_cap);
  if (i == p.path_cap) {
    if (!room || !draft_room) {
      if (threadIdx.x == 0) {
        p.prefix_len_out[b] = L;
        if (p.dk) p.draft_len_out[b] = p.draft_len[b];
        set_status(p.status, EAGLE_ERR_CAPACITY);
      }
      return;
    }
    // next round's state: the last accepted slot's true feature, the bonus
    // token, the new prefix length; the root's draft K/V row (fp32 -> bf16,
    // four elements per load) appended to the draft cache
    const int last = p.last_slot[b];
    const float4* fl = reinterpret_cast<const float4*>(p.f_true + (static_cast<size_t>(b) * p.S + last) * p.d);
    float4* fo = reinterpret_cast<float4*>(p.f_last + static_cast<size_t>(b) * p.d);
    for (int c = threadIdx.x; c < p.d / 4; c += blockDim.x) fo[c] = fl[c];
    if (threadIdx.x == 0) {
      p.t_next[b] = p.final_token[b];
      p.prefix_len_out[b] = L + 1 + a;
    }
    if (p.dk) {
      const int Ld = p.draft_len[b];
      const size_t src = (static_cast<size_t>(b) * p.E + 0) * p.row_elems;
      const size_t dst = (static_cast<size_t>(b) * p.draft_cap + Ld) * p.row_elems;
      const float4* ks = reinterpret_cast<const float4*>(p.dk_tree + src);
      const float4* vs = reinterpret_cast<const float4*>(p.dv_tree + src);
      uint2* kd = reinterpret_cast<uint2*>(p.dk + dst);
      uint2* vd = reinterpret_cast<uint2*>(p.dv + dst);
      for (int c = threadIdx.x; c < p.row_elems / 4; c += blockDim.x) {
        const float4 k = ks[c], v = vs[c];
        kd[c] = make_uint2(f32_to_bf16(k.x) | (static_cast<uint32_t>(f32_to_bf16(k.y)) << 16),
                           f32_to_bf16(k.z) | (static_cast<uint32_t>(f32_to_bf16(k.w)) << 16));
        vd[c] = make_uint2(f32_to_bf16(v.x) | (static_cast<uint32_t>(f32_to_bf16(v.y)) << 16),
                           f32_to_bf16(v.z) | (static_cast<uint32_t>(f32_to_bf16(v.w)) << 16));
      }
      if (threadIdx.x == 0) p.draft_len_out[b] = Ld + 1;
    }
    return;
  }
  if (i > a || !room || !draft_room) return;
  const int slot = p.path[static_cast<size_t>(b) * p.path_cap + i];
  const size_t row = p.paged.table ? static_cast<size_t>(paged_row(p.paged, b, L + i))
                                    : static_cast<size_t>(b) * p.kv_cap + L + i;
  for (int l = 0; l < p.n_layers; ++l) {
    const size_t src = (static_cast<size_t>(b) * p.S + slot) * p.row_elems;
    const size_t dst = row * p.row_elems;
    copy_row(p.kc[l] + dst, p.kt[l] + src, p.row_elems);
    copy_row(p.vc[l] + dst, p.vt[l] + src, p.row_elems);
  }
  const float4* f = reinterpret_cast<const float4*>(p.f_true + (static_cast<size_t>(b) * p.S + slot) * p.d);
  float4* fc = reinterpret_cast<float4*>(p.f_commit + (static_cast<size_t>(b) * p.path_cap + i) * p.d);
  for (int c = threadIdx.x; c < p.d / 4; c += blockDim.x) fc[c] = f[c];
  if (threadIdx.x == 0) {
    int32_t* tc = p.tok_commit + static_cast<size_t>(b) * (p.path_cap + 1);
    tc[i] = p.t_token[static_cast<size_t>(b) * p.S + slot];
    if (i == a) tc[a + 1] = p.final_token[b];
  }
}

}  // namespace

cudaError_t launch_commit(eagle_ctx* ctx, const CommitLaunch& C, cudaStream_t st) {
  CommitParams p{};
  p.n_layers = C.n_layers;
  p.kv_cap = C.kv_cap;
  p.paged = C.paged;
  p.S = C.tree->stride;
  p.E = ctx->lim.max_expanded;
  p.d = ctx->dims.d;
  p.row_elems = ctx->dims.n_kv_heads * ctx->dims.head_dim;
  p.path_cap = C.acc->path_cap;
  for (int l = 0; l < C.n_layers; ++l) {
    p.kt[l] = C.kt[l];
    p.vt[l] = C.vt[l];
    p.kc[l] = C.kc[l];
    p.vc[l] = C.vc[l];
  }
  p.accept_len = C.acc->accept_len;
  p.path = C.acc->path;
  p.final_token = C.acc->final_token;
  p.last_slot = C.acc->last_slot;
  p.t_token = C.tree->token;
  p.f_true = C.f_true;
  p.kv_len = C.kv_len;
  if (C.draft && C.draft_kv) {
    p.dk_tree = C.draft->k_tree;
    p.dv_tree = C.draft->v_tree;
    p.dk = C.draft_kv->k;
    p.dv = C.draft_kv->v;
    p.draft_cap = C.draft_kv->cap;
    p.draft_len = C.draft_kv->len;
  }
  p.f_commit = C.out->f_commit;
  p.tok_commit = C.out->tok_commit;
  p.f_last = C.out->f_last;
  p.t_next = C.out->t_next;
  p.prefix_len_out = C.out->prefix_len;
  p.draft_len_out = C.out->draft_len;
  p.status = C.status;
  p.stamp = stamp_slot(ctx, EAGLE_K_COMMIT);
  dim3 grid(C.batch, C.acc->path_cap + 1);
  trace_before(ctx, EAGLE_K_COMMIT, st);
  const cudaError_t e = launch_pdl(commit_kernel, grid, dim3(512), 0, st, p);
  ctx->launches++;
  trace_after(ctx, EAGLE_K_COMMIT, st);
  return e;
}

// ---- the bounded wait, checked ------------------------------------------------
//
// One CTA whose only wait is the library's bounded barrier wait on a barrier
// nothing arrives at: it gives up after the device wait limit and reports
// EAGLE_ERR_TIMEOUT in the status word, as every kernel's barrier wait does,
// and returns (nothing is in flight when it leaves).
namespace {
__global__ void wait_selftest_kernel(int* status) {
  __shared__ uint64_t s_bar;
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    s_abort = 0;
    sm100::mbar_init(&s_bar, 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !sm100::mbar_wait(&s_bar, 0u, &s_abort)) set_status(status, EAGLE_ERR_TIMEOUT);
}
}  // namespace

cudaError_t launch_wait_selftest(eagle_ctx* ctx, void* ws, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(ws_ptr<int>(ws, ctx->ws.status));
  ctx->launches++;
  return cudaGetLastError();
}

}  // namespace eagle
