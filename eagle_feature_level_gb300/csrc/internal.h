// Host-side internals of libeagle: the context, the workspace layout and the
// launchers each kernel file provides.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>
#include <vector>

#include "../../include/eagle.h"

namespace eagle {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// GEMM epilogue kinds (one per contraction of the draft step, and the K/V
// projection of the draft-cache refresh).
enum Epi : int { EPI_FC = 0, EPI_QKV = 1, EPI_O = 2, EPI_GATEUP = 3, EPI_DOWN = 4, EPI_LM = 5, EPI_KV = 6,
                 EPI_FUSE = 7 };
constexpr int N_EPI = 8;

// Activation rows are padded to NP; the GEMM's B operand holds the bf16 "hi"
// parts in rows [0, NP) and the "lo" parts in rows [NP, 2NP).  NP is a
// multiple of 8 (one MMA of N = 2NP <= 256) or of 16 beyond 128 rows (two
// MMAs of N = NP).
inline int padded_rows(int n) {
  if (n <= 8) return 8;
  if (n <= 128) return (n + 7) / 8 * 8;
  return (n + 15) / 16 * 16;
}

struct Workspace {
  size_t status;                 // int status word
  size_t b_fc, b_qkv, b_o, b_gu, b_down, b_lm, b_fuse;   // bf16 [2*NPmax][Kpad]
  int kp_fc, kp_qkv, kp_o, kp_gu, kp_down, kp_lm, kp_fuse;
  size_t h, h2;                  // fp32 [max_rows][d]
  size_t qrow;                   // fp32 [max_rows][Hq*dh]
  size_t ss_fc, ss_o;            // fp32 [max_rows][tiles of d]
  size_t gemm_part;              // fp32 [(max_mtiles + 2 * SMs) * max_rows * 128]
  size_t gemm_cnt;               // int [N_EPI][max_mtiles]
  size_t attn_part;              // fp32 partial (m, l, acc[dh]) records
  size_t attn_cnt;               // int [2][max_batch * Hkv]
  size_t total;
  int max_mtiles;
  int npmax;
};

struct TraceState {
  int kernel_id = -2;            // -2: disabled
  int capacity = 0;
  std::vector<cudaEvent_t> events;   // pairs
  std::vector<int> ids;              // kernel class of each pair
  int n = 0;
};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace eagle

struct eagle_ctx {
  eagle_dims dims;
  eagle_limits lim;
  int device = 0;
  int sm_count = 0;
  eagle::Workspace ws;
  eagle::TraceState trace;
  long long launches = 0;
  eagle::EncodeTiledFn encode = nullptr;
  // launch timestamps (eagle_stamps_enable): caller-owned device pairs
  uint64_t* stamps = nullptr;
  int stamp_cap = 0;
  std::vector<int> stamp_ids;        // kernel class of each stamped launch
};

namespace eagle {

// Every kernel of the library is launched with programmatic stream
// serialization: the next kernel in the stream may be scheduled while this
// one drains, and waits in-kernel (griddepcontrol.wait) before touching what
// its predecessor wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                      int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The calling thread's current CUDA context as a process-unique id (the
// driver never reuses one, so a context re-created after cudaDeviceReset gets
// a new id).  Makes the device's primary context current if none is.  False
// if the id cannot be determined.
bool current_context_id(unsigned long long* id);

// cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
// bytes), done once per (current context, kernel, bytes): function
// attributes belong to a context, so every device and every re-created
// context gets its own.
cudaError_t smem_limit_once(const void* kernel, int bytes);
// cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
// 1) (clusters of up to 16 CTAs), once per (current context, kernel).
cudaError_t cluster_nonportable_once(const void* kernel);

// The timestamp pair of the next launch (of kernel class `kernel_id`) while
// stamps are enabled, else null.
inline uint64_t* stamp_slot(eagle_ctx* ctx, int kernel_id) {
  if (!ctx->stamps || static_cast<int>(ctx->stamp_ids.size()) >= ctx->stamp_cap) return nullptr;
  uint64_t* s = ctx->stamps + 3 * ctx->stamp_ids.size();
  ctx->stamp_ids.push_back(kernel_id);
  return s;
}

// Launch bookkeeping: optional CUDA-event trace around kernels of one class.
void trace_before(eagle_ctx* ctx, int kernel_id, cudaStream_t s);
void trace_after(eagle_ctx* ctx, int kernel_id, cudaStream_t s);

template <typename T>
inline T* ws_ptr(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

struct DraftLaunch {
  const eagle_plan* plan;
  int layer, batch, e0, rpr, n, NP, k;
  const eagle_draft_weights* w;
  const eagle_requests* req;
  const eagle_kv* draft_kv;
  const eagle_pool* pool;
  const eagle_draft_out* out;
  const eagle_children* children;
  const eagle_sampling* s;
  void* ws;
  // draft-cache refresh (EPI_KV): rows j = b * rpr + i - 1 for i = 1 .. rpr
  const eagle_kv* refresh_kv;     // cache; row of (b, i) = len[b] + i - 1
  const int32_t* refresh_n;       // [B] active rows of request b
  // feature fusion (EPI_FUSE): g[j] = W_fuse [l; m; h]_j (+ b_fuse)
  const uint16_t* w_fuse;
  int ld_fuse;
  const float* b_fuse;
  float* g_out;
};

cudaError_t launch_prep_fc(eagle_ctx* ctx, const DraftLaunch& L, cudaStream_t st);
cudaError_t launch_gemm(eagle_ctx* ctx, int epi, const DraftLaunch& L, cudaStream_t st);
cudaError_t launch_draft_attn(eagle_ctx* ctx, const DraftLaunch& L, cudaStream_t st);
cudaError_t launch_select(eagle_ctx* ctx, const DraftLaunch& L, cudaStream_t st);
// Gathers the refresh rows [f_commit[b][i-1] ; E[tok_commit[b][i]]] into the
// FC operand and writes len_out = len + active rows.
// Gathers rows of [l ; m ; h] (fp32 [n][3d]) into the fusion operand.
cudaError_t launch_prep_fuse(eagle_ctx* ctx, const DraftLaunch& L, const float* lmh, cudaStream_t st);
cudaError_t launch_prep_refresh(eagle_ctx* ctx, const DraftLaunch& L, const float* f_commit,
                                const int32_t* tok_commit, int path_cap, int32_t* len_out, cudaStream_t st);

cudaError_t launch_tree(eagle_ctx* ctx, const eagle_plan* plan, int phase, int layer, int batch,
                        const eagle_requests* req, const eagle_children* ch, const eagle_pool* pool,
                        const eagle_tree* tree, int* status, cudaStream_t st);

cudaError_t launch_verify_attn(eagle_ctx* ctx, int batch, const uint16_t* q, const uint16_t* kt,
                               const uint16_t* vt, const eagle_kv* prefix, const eagle_tree* tree,
                               float scale, float* out, void* ws, cudaStream_t st);
// eagle_tree_verify_attn_noalloc: the same kernel with its partials and
// counters in a fixed static device array; EAGLE_ERR_CAPACITY when the call
// does not fit it (nothing launched).
eagle_status launch_verify_attn_noalloc(eagle_ctx* ctx, int batch, const uint16_t* q, const uint16_t* kt,
                                        const uint16_t* vt, const eagle_kv* prefix, const eagle_tree* tree,
                                        float scale, float* out, cudaStream_t st);

cudaError_t launch_target_softmax(eagle_ctx* ctx, int batch, const eagle_tree* tree, const float* logits,
                                  const float* temperature, float* probs, int32_t* argmax, void* ws,
                                  cudaStream_t st);
cudaError_t launch_accept_walk(eagle_ctx* ctx, const eagle_plan* plan, int batch, const eagle_tree* tree,
                               const eagle_children* ch, const float* probs, const int32_t* argmax,
                               const float* q_probs, const eagle_sampling* s, const eagle_accept_out* out,
                               void* ws, cudaStream_t st);

// Block-table addressing of a paged KV cache: position pos of request b is
// row pos % 2^shift of block table[b * per_req + pos / 2^shift] of the pool
// (eagle_paging); table == nullptr: contiguous [B][cap] rows.
struct PagedKv {
  const int32_t* table;
  int shift;              // log2(block_size)
  int per_req;            // table entries per request (cap / block_size)
  int n_blocks;
};

inline PagedKv paged_of(const eagle_paging* pg, int cap) {
  PagedKv k{};
  if (pg == nullptr || pg->block_table == nullptr) return k;
  k.table = pg->block_table;
  while ((1 << k.shift) < pg->block_size) ++k.shift;
  k.per_req = cap / pg->block_size;
  k.n_blocks = pg->n_blocks;
  return k;
}

struct CommitLaunch {
  int batch, n_layers, kv_cap;
  PagedKv paged;          // target caches
  const eagle_accept_out* acc;
  const eagle_tree* tree;
  const float* f_true;
  const uint16_t* const* kt;
  const uint16_t* const* vt;
  uint16_t* const* kc;
  uint16_t* const* vc;
  const int32_t* kv_len;
  const eagle_draft_out* draft;
  const eagle_kv* draft_kv;
  const eagle_commit_out* out;
  int* status;
};
cudaError_t launch_commit(eagle_ctx* ctx, const CommitLaunch& C, cudaStream_t st);
cudaError_t launch_wait_selftest(eagle_ctx* ctx, void* ws, cudaStream_t st);

// Prefix splits of the split-KV attention for `pairs` (request, kv head)
// pairs over a cache of `cap` rows, for a kernel run at per_sm CTAs per SM.
int attn_splits(const eagle_ctx* ctx, int pairs, int cap, int per_sm);
// Most prefix splits an attention launch over `pairs` (request, kv head)
// pairs and a cache of `cap` rows uses: enough for one wave at per_sm CTAs
// per SM (four, the most any attention kernel runs at, by default) with the
// tree part's CTA, and at least enough that no split holds more than 8 key
// tiles of 64 (long or ragged prefixes: many short CTAs, not a few long
// ones); at most 31, so that a warp holds every split's record in the merge.
inline int attn_splits_bound(const eagle_ctx* ctx, int pairs, int cap, int per_sm = 4) {
  int s = per_sm * ctx->sm_count / (pairs < 1 ? 1 : pairs) - 1;
  const int tiles = ((cap < 1 ? 1 : cap) + 63) / 64;
  if (s < (tiles + 7) / 8) s = (tiles + 7) / 8;
  if (s > 31) s = 31;
  return s < 1 ? 1 : s;
}

}  // namespace eagle
