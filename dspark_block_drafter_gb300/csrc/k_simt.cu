// CUDA-core (FMA) kernels of the proposal: base logits of the fp32 operand type, and
// the Markov-corrected greedy chain one slot at a time.  Every sum is accumulated in
// fp32.
#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kTileM = 64, kTileV = 64, kTileK = 16;

// z[i][v][b] = sum_h hidden[b, ifp + i, h] * lm_head[v, h] + lm_bias[v]
// (llama.cpp commit 6fed9f6, the proposal formula's logits(i)); prediction row
// m = i * B + b.
template <typename T>
__global__ void __launch_bounds__(256)
base_logits_simt(const T* __restrict__ hidden, const T* __restrict__ W,
                 const float* __restrict__ bias, float* __restrict__ z, int B, int L_in,
                 int N, int ifp, int H, int Vh, size_t Vhp, size_t ldb) {
  __shared__ float As[kTileK][kTileM + 4];
  __shared__ float Ws[kTileK][kTileV + 4];
  const int M = B * N;
  const int m0 = blockIdx.y * kTileM, v0 = blockIdx.x * kTileV;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += kTileK) {
    for (int e = threadIdx.x; e < kTileM * kTileK; e += 256) {
      int mm = e / kTileK, kk = e % kTileK;
      int m = m0 + mm, k = k0 + kk;
      float a = 0.f;
      if (m < M && k < H) {
        int i = m / B, b = m % B;
        a = to_f32(hidden[((size_t)b * L_in + ifp + i) * H + k]);
      }
      As[kk][mm] = a;
      int v = v0 + mm;
      float w = 0.f;
      if (v < Vh && k < H) w = to_f32(W[(size_t)v * H + k]);
      Ws[kk][mm] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTileK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q] = As[kk][ty * 4 + q];
        w[q] = Ws[kk][tx * 4 + q];
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(a[p], w[q], acc[p][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    int m = m0 + ty * 4 + p;
    if (m >= M) continue;
    const int i = m / B, b = m % B;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int v = v0 + tx * 4 + q;
      if (v < Vh) z[((size_t)i * Vhp + v) * ldb + b] = acc[p][q] + (bias ? bias[v] : 0.f);
    }
  }
}

// One chain step, part 1: zc[b][v] = z[i][b][v] + sum_k markov_w1[prev_b, k] *
// markov_w2[k, v] for every head row v (the proposal formula's logits'(i)).
template <typename T>
__global__ void __launch_bounds__(256)
markov_step_simt(const float* __restrict__ z_i, const T* __restrict__ w1,
                 const T* __restrict__ w2, const int32_t* __restrict__ prev,
                 float* __restrict__ zc, float* __restrict__ logits, int slot, int B,
                 int N, int Vh, size_t ldb, size_t ldz, int r, int V, uint32_t* err) {
  extern __shared__ float u[];  // [r]
  const int b = blockIdx.y;
  int p = prev[b];
  if (p < 0 || p >= V) {
    if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(err, kErrBadToken);
    p = 0;
  }
  for (int k = threadIdx.x; k < r; k += blockDim.x) u[k] = to_f32(w1[(size_t)p * r + k]);
  __syncthreads();
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= Vh) return;
  float acc = 0.f;
  for (int k = 0; k < r; ++k) acc = fmaf(u[k], to_f32(w2[(size_t)k * Vh + v]), acc);
  float x = z_i[(size_t)v * ldb + b] + acc;
  zc[(size_t)b * ldz + v] = x;
  if (logits) logits[((size_t)b * N + slot) * Vh + v] = x;
}

// Block-wide best candidate of a row strictly after (pv, pid) in the candidate order.
__device__ void block_best_after(const float* __restrict__ row, int n, size_t stride, float pv,
                                 int pid, bool first, float& out_v, int& out_id) {
  __shared__ float sv[32];
  __shared__ int si[32];
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  for (int v = threadIdx.x; v < n; v += blockDim.x) {
    float x = row[(size_t)v * stride];
    if (!first && !better(pv, pid, x, v)) continue;  // not strictly after the previous pick
    if (better(x, v, bv, bi)) { bv = x; bi = v; }
  }
  warp_best(bv, bi);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) { sv[w] = bv; si[w] = bi; }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x / 32;
    bv = l < nw ? sv[l] : -INFINITY;
    bi = l < nw ? si[l] : 0x7FFFFFFF;
    warp_best(bv, bi);
    if (l == 0) { sv[0] = bv; si[0] = bi; }
  }
  __syncthreads();
  out_v = sv[0];
  out_id = si[0] == 0x7FFFFFFF ? 0 : si[0];  // only when every value is NaN
  __syncthreads();
}

// One chain step, part 2: the slot's argmax (the next prev) and its top-k.
// Ids are head rows, mapped to token ids through d2t when the head is compact (d2t is
// increasing, so the row order and the token order agree).
__global__ void __launch_bounds__(1024)
select_step_simt(const float* __restrict__ zc, const float* __restrict__ z_i,
                 const int32_t* __restrict__ d2t, int topk_markov, int k,
                 int32_t* __restrict__ draft, int32_t* __restrict__ topk_ids,
                 float* __restrict__ topk_vals, int32_t* __restrict__ prev, int slot,
                 int N, int Vh, size_t ldb, size_t ldz) {
  const int b = blockIdx.x;
  const float* row_c = zc + (size_t)b * ldz;
  float bv;
  int bi;
  block_best_after(row_c, Vh, 1, 0.f, 0, true, bv, bi);
  const int tok = d2t ? d2t[bi] : bi;
  if (threadIdx.x == 0) {
    draft[(size_t)b * N + slot] = tok;
    prev[b] = tok;
  }
  if (!topk_ids && !topk_vals) return;
  // ranked row: the corrected logits (contiguous) or the base logits (stride ldb)
  const float* row_r = topk_markov ? row_c : z_i + b;
  const size_t stride = topk_markov ? 1 : ldb;
  float pv = 0.f;
  int pid = 0;
  for (int j = 0; j < k; ++j) {
    block_best_after(row_r, Vh, stride, pv, pid, j == 0, bv, bi);
    if (threadIdx.x == 0) {
      size_t o = ((size_t)b * N + slot) * k + j;
      if (topk_ids) topk_ids[o] = d2t ? d2t[bi] : bi;
      if (topk_vals) topk_vals[o] = bv;
    }
    pv = bv;
    pid = bi;
  }
}

template <typename T>
cudaError_t base_logits_t(const ProposePlan& p) {
  dim3 grid((p.Vh + kTileV - 1) / kTileV, (p.B * p.N + kTileM - 1) / kTileM);
  base_logits_simt<T><<<grid, 256, 0, p.stream>>>(
      (const T*)p.hidden, (const T*)p.lm_head, p.lm_bias, p.z, p.B, p.L_in, p.N, p.ifp,
      p.H, p.Vh, p.Vhp, p.ldb);
  return cudaGetLastError();
}

template <typename T>
cudaError_t chain_t(const ProposePlan& p) {
  for (int i = 0; i < p.N; ++i) {
    const int32_t* prev = i == 0 ? p.anchors : p.prev;
    const float* z_i = p.z + (size_t)i * p.Vhp * p.ldb;
    dim3 g1((p.Vh + 255) / 256, p.B);
    markov_step_simt<T><<<g1, 256, p.r * sizeof(float), p.stream>>>(
        z_i, (const T*)p.w1, (const T*)p.w2, prev, p.zc, p.logits, i, p.B, p.N, p.Vh,
        p.ldb, p.ldz, p.r, p.V, p.ctrl);
    select_step_simt<<<p.B, 1024, 0, p.stream>>>(p.zc, z_i, p.d2t, p.topk_markov, p.k,
                                                  p.draft, p.topk_ids, p.topk_vals,
                                                  p.prev, i, p.N, p.Vh, p.ldb, p.ldz);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_base_logits_simt(const ProposePlan& p) {
  return base_logits_t<float>(p);   // the bf16 operand type runs on the tensor cores
}

cudaError_t launch_chain_simt(const ProposePlan& p) {
  return p.dtype == 0 ? chain_t<float>(p) : chain_t<__nv_bfloat16>(p);
}

}  // namespace dspark
