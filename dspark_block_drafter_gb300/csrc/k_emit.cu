// The emittable-row set of a reduced draft vocabulary given in the bias form: a full-V
// head whose lm_bias marks the rows the draft cannot emit (a bias at or below -1e8).
// llama.cpp PR #26275 ("dspark: support speculators-format checkpoints") gives the
// reduced vocabulary both as such an expanded head and as a compact head with a d2t
// map; dspark_prepare_head turns the first into the second on the device, so that every
// proposal works on the emittable rows only:
//   1. the rows with bias > -1e8, in increasing order (count per chunk, then each chunk
//      scanned at its offset), padded to a multiple of 8 with copies of the last one;
//   2. their lm_head rows, markov_w2 columns and biases, gathered into the prepared
//      buffer (padding rows: zero weights and a bias of -1e30, so they never win).
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kChunk = 4096;          // bias entries per CTA of the scan
constexpr int kScanThreads = 1024;    // four entries per thread

__device__ __forceinline__ bool emittable(float bias) { return bias > kEmitMaskLevel; }

__global__ void __launch_bounds__(256)
emit_count(const float* __restrict__ bias, int V, int* __restrict__ count) {
  int n = 0;
  for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x)
    n += emittable(bias[v]) ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
  if ((threadIdx.x & 31) == 0 && n) atomicAdd(count, n);
}

__global__ void __launch_bounds__(256)
emit_chunk_counts(const float* __restrict__ bias, int V, int* __restrict__ chunk_count) {
  __shared__ int s;
  if (threadIdx.x == 0) s = 0;
  __syncthreads();
  const int v0 = blockIdx.x * kChunk;
  int n = 0;
  for (int v = v0 + threadIdx.x; v < min(V, v0 + kChunk); v += blockDim.x)
    n += emittable(bias[v]) ? 1 : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, o);
  if ((threadIdx.x & 31) == 0 && n) atomicAdd(&s, n);
  __syncthreads();
  if (threadIdx.x == 0) chunk_count[blockIdx.x] = s;
}

// Chunk c writes its emittable rows, in order, from the sum of the earlier chunks' counts.
__global__ void __launch_bounds__(kScanThreads)
emit_list(const float* __restrict__ bias, int V, const int* __restrict__ chunk_count,
          int32_t* __restrict__ list) {
  __shared__ int s_warp[kScanThreads / 32];
  __shared__ int s_base;
  const int c = blockIdx.x, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  if (tid == 0) {
    int b = 0;
    for (int q = 0; q < c; ++q) b += chunk_count[q];
    s_base = b;
  }
  // this thread's four consecutive entries
  const int v0 = c * kChunk + 4 * tid;
  bool f[4];
  int n = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    f[t] = v0 + t < V && emittable(bias[v0 + t]);
    n += f[t] ? 1 : 0;
  }
  // exclusive scan of n over the CTA: within the warp, then over the warps
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kScanThreads / 32 ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kScanThreads / 32) s_warp[lane] = w;          // inclusive over the warps
  }
  __syncthreads();
  int pos = s_base + (warp > 0 ? s_warp[warp - 1] : 0) + incl - n;
#pragma unroll
  for (int t = 0; t < 4; ++t)
    if (f[t]) list[pos++] = v0 + t;
}

// Padding entries n_emit .. n_pad - 1: copies of the last emittable row.
__global__ void emit_pad(int32_t* list, int n_emit, int n_pad) {
  const int j = n_emit + threadIdx.x;
  if (j < n_pad) list[j] = list[n_emit - 1];
}

// rows_c[j][:] = rows[list[j]][:] (16-byte chunks), zero for padding rows
__global__ void __launch_bounds__(256)
emit_gather_rows(const uint4* __restrict__ rows, const int32_t* __restrict__ list, int n_emit,
                 int n_pad, int chunks_per_row, uint4* __restrict__ rows_c) {
  const size_t total = (size_t)n_pad * chunks_per_row;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(e / chunks_per_row), q = (int)(e % chunks_per_row);
    rows_c[e] = j < n_emit ? rows[(size_t)list[j] * chunks_per_row + q] : make_uint4(0, 0, 0, 0);
  }
}

// w2_c[k][j] = w2[k][list[j]], zero for padding columns
__global__ void __launch_bounds__(256)
emit_gather_cols(const __nv_bfloat16* __restrict__ w2, const int32_t* __restrict__ list,
                 int n_emit, int n_pad, int V, int r, __nv_bfloat16* __restrict__ w2_c) {
  const size_t total = (size_t)r * n_pad;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (size_t)gridDim.x * blockDim.x) {
    const int k = (int)(e / n_pad), j = (int)(e % n_pad);
    w2_c[e] = j < n_emit ? w2[(size_t)k * V + list[j]] : __float2bfloat16(0.f);
  }
}

// bias_c[j] = bias[list[j]], -1e30 for padding rows
__global__ void __launch_bounds__(256)
emit_gather_bias(const float* __restrict__ bias, const int32_t* __restrict__ list, int n_emit,
                 int n_pad, float* __restrict__ bias_c) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j < n_pad) bias_c[j] = j < n_emit ? bias[list[j]] : -1e30f;
}

__global__ void emit_header(CompactHeader* dst, const CompactHeader h) { *dst = h; }

}  // namespace

CompactLayout plan_compact(int V, int H, int r, int n_pad) {
  CompactLayout l{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  l.header = take(sizeof(CompactHeader));
  l.list = take(sizeof(int32_t) * (size_t)n_pad);
  l.chunk_count = take(sizeof(int) * (size_t)((V + kChunk - 1) / kChunk + 1));
  l.lm_head = take(sizeof(__nv_bfloat16) * (size_t)n_pad * H);
  l.w2 = take(sizeof(__nv_bfloat16) * (size_t)r * n_pad);
  l.bias = take(sizeof(float) * (size_t)n_pad);
  l.prepared = off;
  l.total = off + plan_prepared(n_pad, r).total;
  return l;
}

cudaError_t launch_emit_count(const float* bias, int V, int* count, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(count, 0, sizeof(int), stream);
  if (e != cudaSuccess) return e;
  const int grid = std::min(1024, (V + 255) / 256);
  emit_count<<<grid, 256, 0, stream>>>(bias, V, count);
  return cudaGetLastError();
}

cudaError_t launch_prepare_compact(const void* lm_head, const float* bias, const void* w1,
                                   const void* w2, int V, int H, int r, int n_emit, int n_pad,
                                   void* prepared, cudaStream_t stream) {
  const CompactLayout l = plan_compact(V, H, r, n_pad);
  char* base = (char*)prepared;
  int32_t* list = (int32_t*)(base + l.list);
  int* cc = (int*)(base + l.chunk_count);
  const int chunks = (V + kChunk - 1) / kChunk;
  emit_chunk_counts<<<chunks, 256, 0, stream>>>(bias, V, cc);
  emit_list<<<chunks, kScanThreads, 0, stream>>>(bias, V, cc, list);
  if (n_pad > n_emit) emit_pad<<<1, 32, 0, stream>>>(list, n_emit, n_pad);
  const int cpr = H / 8;                                  // 16-byte chunks of a bf16 row
  const size_t rows_total = (size_t)n_pad * cpr;
  emit_gather_rows<<<(unsigned)std::min<size_t>(4096, (rows_total + 255) / 256), 256, 0,
                     stream>>>((const uint4*)lm_head, list, n_emit, n_pad, cpr,
                               (uint4*)(base + l.lm_head));
  const size_t cols_total = (size_t)r * n_pad;
  emit_gather_cols<<<(unsigned)std::min<size_t>(4096, (cols_total + 255) / 256), 256, 0,
                     stream>>>((const __nv_bfloat16*)w2, list, n_emit, n_pad, V, r,
                               (__nv_bfloat16*)(base + l.w2));
  emit_gather_bias<<<(n_pad + 255) / 256, 256, 0, stream>>>(bias, list, n_emit, n_pad,
                                                            (float*)(base + l.bias));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // the pruned chain's preparation of the compact head
  e = launch_prepare_head(w1, base + l.w2, V, r, n_pad, base + l.prepared, stream);
  if (e != cudaSuccess) return e;
  CompactHeader h{};
  h.magic = kCompactMagic;
  h.V = V;
  h.H = H;
  h.r = r;
  h.n_emit = n_emit;
  h.n_pad = n_pad;
  h.lm_head = (unsigned long long)(uintptr_t)lm_head;
  h.lm_bias = (unsigned long long)(uintptr_t)bias;
  h.w1 = (unsigned long long)(uintptr_t)w1;
  h.w2 = (unsigned long long)(uintptr_t)w2;
  emit_header<<<1, 1, 0, stream>>>((CompactHeader*)(base + l.header), h);
  return cudaGetLastError();
}

}  // namespace dspark
