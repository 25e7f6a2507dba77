// Device helpers shared by the libeagle kernels: bf16 bit handling, the
// hi/lo bf16 split of fp32 activations, Philox4x32-10, block reductions and
// the device status word.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/eagle.h"

namespace eagle {

// ---- bf16 as raw bits ------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Round-to-nearest-even fp32 -> bf16 bits.
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi): two bf16 operands whose
// sum carries ~16 mantissa bits, so bf16 tensor-core products of fp32
// activations keep fp32-level accuracy.
__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  hi = f32_to_bf16(x);
  lo = f32_to_bf16(x - bf16_to_f32(hi));
}

// ---- programmatic dependent launch -------------------------------------------
// Kernels are launched so that the next kernel in the stream may start while
// this one drains.  pdl_wait: block until every preceding grid has completed
// and its memory is visible (each thread that reads a predecessor's output or
// writes global memory passes it first); pdl_trigger: let the next grid be
// scheduled (it still waits for this grid to complete before its reads).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---- Philox4x32-10 (Salmon et al., SC'11) -----------------------------------
// Four 32-bit counter words, two key words, ten rounds; words 0 and 2 are
// multiplied by the two round constants, the key is bumped by the Weyl
// constants between rounds.
struct Philox4 { uint32_t x, y, z, w; };

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return {c0, c1, c2, c3};
}

enum : uint32_t { PURPOSE_DRAW = 0, PURPOSE_ACCEPT = 1, PURPOSE_FINAL = 2, KEY_TAG = 0x000EA61Eu };

// The round's uniform stream: key (seed, tag), counter
// (draw index, node slot, purpose << 16 | request, round), word 0.
__device__ __forceinline__ uint32_t round_uniform(uint32_t seed, uint32_t draw_index, uint32_t slot,
                                                  uint32_t purpose, uint32_t request, uint32_t round_id) {
  return philox4x32_10(draw_index, slot, (purpose << 16) | request, round_id, seed, KEY_TAG).x;
}

// t = floor(u32 * S / 2^32) for S < 2^63.
__device__ __forceinline__ uint64_t scale_uniform(uint32_t u, uint64_t S) {
  const uint64_t lo = static_cast<uint64_t>(u) * (S & 0xffffffffull);
  const uint64_t hi = static_cast<uint64_t>(u) * (S >> 32);
  return hi + (lo >> 32);
}

constexpr int QBITS = 40;

// W = floor(p * 2^40) for p in [0, 2^24), exactly, in integer arithmetic
// (no fp64 pipe, which GB300 runs at a small fraction of its integer rate):
// a finite positive fp32 p is m * 2^(E - 150) with the significand m (hidden
// bit included; E the biased exponent, E = 1 for subnormals), so
// p * 2^40 = m * 2^(E - 110), a shift of m.  Zero, negative, infinite and
// NaN inputs carry no mass (0).
__device__ __forceinline__ uint64_t quantize_prob(float p) {
  const uint32_t u = __float_as_uint(p);
  const uint32_t E = (u >> 23) & 0xffu;
  if ((u >> 31) != 0u || E == 0xffu || E > 150u) return 0ull;
  const uint64_t m = E != 0u ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
  const int sh = static_cast<int>(E != 0u ? E : 1u) - 110;
  return sh >= 0 ? (m << sh) : (sh > -32 ? (m >> -sh) : 0ull);
}

// ---- reductions -----------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide reductions over blockDim.x threads (multiple of 32, <= 1024),
// with a fixed combination order (deterministic).  `scratch` holds >= 32
// entries; every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) scratch[wid] = v;
  __syncthreads();
  float r = lane < nw ? scratch[lane] : 0.f;
  r = warp_sum(r);
  return r;
}
__device__ __forceinline__ float block_max(float v, float* scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) scratch[wid] = v;
  __syncthreads();
  float r = lane < nw ? scratch[lane] : -INFINITY;
  return warp_max(r);
}
__device__ __forceinline__ uint64_t block_sum_u64(uint64_t v, uint64_t* scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum_u64(v);
  __syncthreads();
  if (lane == 0) scratch[wid] = v;
  __syncthreads();
  uint64_t r = lane < nw ? scratch[lane] : 0ull;
  return warp_sum_u64(r);
}
__device__ __forceinline__ int block_max_i(int v, int* scratch) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max_i(v);
  __syncthreads();
  if (lane == 0) scratch[wid] = v;
  __syncthreads();
  int r = lane < nw ? scratch[lane] : INT32_MIN;
  return warp_max_i(r);
}

// Order-preserving unsigned image of a non-NaN float (-0 taken as +0, so
// equal values tie exactly as they do under ranks_before), and its inverse.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The warp's largest non-NaN value on every lane, in one reduction (-0 and
// +0 compare equal; the result is then +0).
__device__ __forceinline__ float warp_max_redux(float v) {
  return key_value(__reduce_max_sync(0xffffffffu, order_key(v)));
}

// The warp's best (v, i) -- larger v first, then smaller i -- on every lane: two warp-wide
// integer reductions (largest key, then smallest id among the lanes that
// hold it).  Ids are non-negative; INT32_MAX marks an empty lane.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
  const uint32_t key = order_key(v);
  const uint32_t best = __reduce_max_sync(0xffffffffu, key);
  const uint32_t id = __reduce_min_sync(0xffffffffu, key == best ? static_cast<uint32_t>(i) : 0xffffffffu);
  v = key_value(best);
  i = static_cast<int>(id);
}

// ---- last-arriver counters ------------------------------------------------
// One thread's arrival on a per-tile (or per-pair) counter, issued after a
// CTA barrier that follows the CTA's partial-result stores.  Release is
// cumulative over the barrier, so the CTA that observes the final count sees
// those stores; acquire makes the earlier arrivals' stores visible here (the
// rest of the CTA reads them after the next barrier).  Takes the place of a
// full fence on every thread before and after a relaxed atomic.
__device__ __forceinline__ int arrive_acq_rel(int* counter) {
  int prev;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(counter) : "memory");
  return prev;
}

// A counter's value with acquire semantics at GPU scope: once it shows every
// arrival, the stores the arrivals released are visible to this thread (and,
// after a CTA barrier, to the rest of its CTA).
__device__ __forceinline__ int ld_acquire(const int* counter) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
  return v;
}

// ---- device status word -----------------------------------------------------
// First int of the workspace.  The first error wins; later ones are dropped.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Block-table addressing of a paged KV cache (PagedKv): the pool row of
// position pos of request b, or -1 when that block is not allocated.
__device__ __forceinline__ long long paged_row(const PagedKv& pg, int b, int pos) {
  const int blk = pg.table[static_cast<size_t>(b) * pg.per_req + (pos >> pg.shift)];
  if (blk < 0 || blk >= pg.n_blocks) return -1;
  return (static_cast<long long>(blk) << pg.shift) + (pos & ((1 << pg.shift) - 1));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- launch timestamps (measurement) ---------------------------------------
// With a non-null slot, thread 0 of every CTA records %globaltimer three
// times: when it starts (atomic min into slot[0]), when it has passed the
// dependency wait (atomic min into slot[1]: the earliest moment a CTA of this
// launch could use its predecessors' outputs) and when it leaves the kernel
// (atomic max into slot[2]).  A null slot costs one test.
struct LaunchStamp {
  unsigned long long* slot;
  __device__ explicit LaunchStamp(uint64_t* s)
      : slot(threadIdx.x == 0 ? reinterpret_cast<unsigned long long*>(s) : nullptr) {
    if (slot) atomicMin(slot, static_cast<unsigned long long>(globaltimer_ns()));
  }
  __device__ void waited() const {
    if (slot) atomicMin(slot + 1, static_cast<unsigned long long>(globaltimer_ns()));
  }
  __device__ ~LaunchStamp() {
    if (slot) atomicMax(slot + 2, static_cast<unsigned long long>(globaltimer_ns()));
  }
};

// A device-side wait gives up after this long and reports EAGLE_ERR_TIMEOUT.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

}  // namespace eagle
