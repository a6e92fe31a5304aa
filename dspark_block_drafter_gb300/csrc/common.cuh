// Shared device helpers of the DSpark kernels: element loads, the (value, id) order
// used by every argmax / top-k, and the sticky device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dspark {

// Bits of the device error word (first word of the workspace control block).
enum : uint32_t {
  kErrBadToken = 1u,   // an anchor / previous token outside [0, V)
  kErrTimeout = 2u,    // a bounded wait gave up
  kErrPrepared = 4u,   // the prepared head buffer was made for other weights or sizes
};

// Words of the workspace control block after the error word: counters of the latest
// pass (the block is zeroed at the start of every pass), read by dspark_pass_stats.
enum : int {
  kCtrlOnTheFly = 1,   // (slot, block) pairs the pruned walk evaluated without a table
  kCtrlEveryRow = 2,   //   of those, over every head row (the candidate list overflowed)
  kCtrlDenseOver = 3,  // (slot, block) top-k lists of the dense chain that overflowed and
                       //   were recomputed over every head row
  kCtrlGemmTiles = 4,  // tiles claimed by the lm_head GEMM's dynamic schedule
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Candidate order: larger value first, and among equal values the lower id first.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  // bitwise, not short-circuit: no branch, so warps do not diverge on it
  return (va > vb) | ((va == vb) & (ia < ib));
}

// 64-bit key whose unsigned order is the candidate order above: the float is mapped
// to an order-preserving unsigned integer in the high half and the id is inverted in
// the low half, so a larger key means a larger value or, for equal values, a lower id.
__device__ __forceinline__ unsigned long long order_key(float v, int id) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ int key_id(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}
__device__ __forceinline__ float key_value(unsigned long long k) {
  uint32_t u = (uint32_t)(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  return __uint_as_float(u);
}

// 32-bit key whose signed order is the order of the floats (for integer max reductions)
__device__ __forceinline__ int order_key32(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7FFFFFFF;
}
__device__ __forceinline__ float order_key32_value(int k) {
  return __int_as_float(k >= 0 ? k : k ^ 0x7FFFFFFF);
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel still runs; it must wait for that
// kernel's completion (and memory) before touching its results.  The previous kernel
// lets it start early by signalling.  Both are no-ops without such a launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_signal() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// Warp-wide best (value, id) under the candidate order.
__device__ __forceinline__ void warp_best(float& v, int& id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    int oi = __shfl_xor_sync(0xFFFFFFFFu, id, o);
    if (better(ov, oi, v, id)) { v = ov; id = oi; }
  }
}

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

}  // namespace dspark
