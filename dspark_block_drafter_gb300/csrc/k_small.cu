// Small kernels of the path: the zeroing of a pass's control block, the confidence head
// with the truncation length, the greedy verify/accept step, and the self-test of the
// bounded device-side wait.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dspark {

namespace {

// The control block of a pass (error word, counters, barrier words, winner keys, bound
// maxima) back to zero.  It lets the kernel after it be scheduled at once: that kernel,
// launched as a dependent, waits for this one to finish before it reads or writes any of
// these words.
__global__ void __launch_bounds__(256) zero_block(uint4* __restrict__ p, size_t n16) {
  pdl_signal();
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n16;
       e += (size_t)gridDim.x * blockDim.x)
    p[e] = make_uint4(0u, 0u, 0u, 0u);
}

// conf[b, i] = sigmoid(h[b, ifp + i] . w_conf + b_conf) and n_draft[b] = the first slot
// with conf < conf_min, else N (llama.cpp commit 6fed9f6, "spec: add confidence-based
// draft pruning for DSpark": a block ends at its first slot whose confidence falls under
// the threshold, and a threshold of 0 turns this off).  One CTA per block; warps take
// slots round-robin.
template <typename T>
__global__ void __launch_bounds__(512)
conf_truncate(const T* __restrict__ hidden, const T* __restrict__ w_conf, float b_conf,
              int L_in, int N, int ifp, int H, float conf_min, float* __restrict__ conf,
              int32_t* __restrict__ n_draft) {
  extern __shared__ float sconf[];  // [N]
  const int b = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
  if (w_conf) {
    for (int i = warp; i < N; i += nw) {
      const T* h = hidden + ((size_t)b * L_in + ifp + i) * H;
      float acc = 0.f;
      constexpr int kVec = 16 / sizeof(T);            // elements per 16-byte load
      const bool vec = (H % kVec == 0) && ((uintptr_t)h % 16 == 0) && ((uintptr_t)w_conf % 16 == 0);
      int c0 = 0;
      if (vec) {
        const uint4* h4 = reinterpret_cast<const uint4*>(h);
        const uint4* w4 = reinterpret_cast<const uint4*>(w_conf);
        const int n4 = H / kVec;
#pragma unroll 4
        for (int q = lane; q < n4; q += 32) {
          const uint4 hv = h4[q], wv = w4[q];
          const T* he = reinterpret_cast<const T*>(&hv);
          const T* we = reinterpret_cast<const T*>(&wv);
#pragma unroll
          for (int e = 0; e < kVec; ++e) acc = fmaf(to_f32(he[e]), to_f32(we[e]), acc);
        }
        c0 = H;
      }
      for (int c = c0 + lane; c < H; c += 32) acc = fmaf(to_f32(h[c]), to_f32(w_conf[c]), acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      if (lane == 0) {
        float c = 1.f / (1.f + expf(-(acc + b_conf)));
        sconf[i] = c;
        conf[(size_t)b * N + i] = c;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int n = N;
    if (w_conf && conf_min > 0.f) {
      for (int i = 0; i < N; ++i)
        if (sconf[i] < conf_min) { n = i; break; }
    }
    n_draft[b] = n;
  }
}

// Greedy verify/accept, which DSpark takes over from DFlash as it is (llama.cpp commit
// 6fed9f6, the verify paragraph of the squash log; greedy decoding stays lossless).  One
// warp per block: a ballot over the slot comparisons finds the first mismatch.
__global__ void __launch_bounds__(256)
verify_kernel(int B, int N, const int32_t* __restrict__ draft,
              const int32_t* __restrict__ n_draft, const int32_t* __restrict__ target,
              int32_t* __restrict__ accepted, int32_t* __restrict__ bonus,
              int32_t* __restrict__ emitted) {
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  pdl_wait();                                        // the draft of the proposal
  if (b >= B) return;
  const int nd = min(max(n_draft[b], 0), N);
  const int32_t* d = draft + (size_t)b * N;
  const int32_t* t = target + (size_t)b * (N + 1);
  int a = nd;
  for (int j0 = 0; j0 < nd; j0 += 32) {
    const int j = j0 + lane;
    const bool mismatch = j < nd && d[j] != t[j];
    const unsigned m = __ballot_sync(0xFFFFFFFFu, mismatch);
    if (m) { a = j0 + __ffs(m) - 1; break; }
  }
  const int bo = t[a];
  if (lane == 0) {
    accepted[b] = a;
    bonus[b] = bo;
  }
  if (emitted)
    for (int j = lane; j <= N; j += 32)
      emitted[(size_t)b * (N + 1) + j] = j < a ? d[j] : (j == a ? bo : -1);
}

// Verify of the top-k candidate lattice (the DDTree consumer; lucebox PR #626, description:
// the tree's candidates are the per-slot top-k with the Markov bias; onnxruntime-genai
// PR #2490, the DFlash 2 / DSpark builder commits: the runtime walks the drafter's
// candidate lattice greedily).  Every candidate of slot i is a child of every candidate
// of slot i - 1, so the greedy target, whose argmax after an accepted prefix is its own
// token target[b, i], goes one level deeper exactly when that token is among slot i's
// candidates.  One warp per block: lane i scans the k candidates of depth i, a ballot
// finds the first depth without the target's token.
__global__ void __launch_bounds__(256)
tree_verify_kernel(int B, int N, int k, const int32_t* __restrict__ topk_ids,
                   const int32_t* __restrict__ n_draft, const int32_t* __restrict__ target,
                   int32_t* __restrict__ accepted, int32_t* __restrict__ bonus,
                   int32_t* __restrict__ emitted, int32_t* __restrict__ path) {
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  pdl_wait();                                        // the lattice of the proposal
  if (b >= B) return;
  const int nd = min(max(n_draft[b], 0), N);
  const int32_t* t = target + (size_t)b * (N + 1);
  // rank of the target's token among depth j's candidates, or -1
  auto rank_at = [&](int j) {
    const int32_t* c = topk_ids + ((size_t)b * N + j) * k;
    const int32_t want = t[j];
    for (int q = 0; q < k; ++q)
      if (c[q] == want) return q;
    return -1;
  };
  int a = nd;
  for (int j0 = 0; j0 < nd; j0 += 32) {
    const int j = j0 + lane;
    const bool miss = j < nd && rank_at(j) < 0;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, miss);
    if (m) { a = j0 + __ffs(m) - 1; break; }
  }
  const int bo = t[a];
  if (lane == 0) {
    accepted[b] = a;
    bonus[b] = bo;
  }
  // the accepted tokens are the target's own, then the bonus token
  if (emitted)
    for (int j = lane; j <= N; j += 32)
      emitted[(size_t)b * (N + 1) + j] = j <= a ? t[j] : -1;
  if (path)
    for (int j = lane; j < N; j += 32)
      path[(size_t)b * N + j] = j < a ? rank_at(j) : -1;
}

// Self-test of the bounded wait that every pipeline of the library relies on: one thread
// waits on a fresh mbarrier that nothing ever arrives on, through the same ptx::mbar_wait
// the GEMM and the chain pipelines use.  When the clock budget runs out (or, with
// pre_abort, at once through the abort flag) the wait gives up and the kernel raises the
// timeout bit of the error word, exactly as a pipeline that lost a copy would.
__global__ void __launch_bounds__(32)
wait_selftest(uint32_t* __restrict__ err, long long budget, int pre_abort) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    abort_flag = pre_abort;
    ptx::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, budget, &abort_flag))
    flag_error(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t* err, long long budget, int pre_abort,
                                 cudaStream_t stream) {
  wait_selftest<<<1, 32, 0, stream>>>(err, budget, pre_abort);
  return cudaGetLastError();
}

cudaError_t launch_zero_block(void* p, size_t bytes, cudaStream_t stream) {
  if (bytes % 16 != 0 || ((uintptr_t)p & 15) != 0) return cudaErrorInvalidValue;
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<size_t>(256, (n16 + 255) / 256);
  zero_block<<<grid, 256, 0, stream>>>((uint4*)p, n16);
  return cudaGetLastError();
}

cudaError_t launch_conf(const ProposePlan& p) {
  float* conf = p.conf ? p.conf : p.conf_ws;
  size_t smem = sizeof(float) * (size_t)p.N;
  const int threads = 32 * std::min(16, std::max(1, p.N));   // one warp per slot
  if (p.dtype == 0)
    conf_truncate<float><<<p.B, threads, smem, p.stream>>>(
        (const float*)p.conf_hidden, (const float*)p.w_conf, p.b_conf, p.L_in, p.N, p.ifp, p.H,
        p.conf_min, conf, p.n_draft);
  else
    conf_truncate<__nv_bfloat16><<<p.B, threads, smem, p.stream>>>(
        (const __nv_bfloat16*)p.conf_hidden, (const __nv_bfloat16*)p.w_conf, p.b_conf, p.L_in,
        p.N, p.ifp, p.H, p.conf_min, conf, p.n_draft);
  return cudaGetLastError();
}

cudaError_t launch_verify(int B, int N, const int32_t* draft, const int32_t* n_draft,
                          const int32_t* target, int32_t* accepted, int32_t* bonus,
                          int32_t* emitted, cudaStream_t stream) {
  const int warps_per_cta = 8;
  return launch_dependent(verify_kernel, dim3((B + warps_per_cta - 1) / warps_per_cta),
                          dim3(32 * warps_per_cta), 0, stream, B, N, draft, n_draft, target,
                          accepted, bonus, emitted);
}

cudaError_t launch_tree_verify(int B, int N, int k, const int32_t* topk_ids,
                               const int32_t* n_draft, const int32_t* target,
                               int32_t* accepted, int32_t* bonus, int32_t* emitted,
                               int32_t* path, cudaStream_t stream) {
  const int warps_per_cta = 8;
  return launch_dependent(tree_verify_kernel, dim3((B + warps_per_cta - 1) / warps_per_cta),
                          dim3(32 * warps_per_cta), 0, stream, B, N, k, topk_ids, n_draft,
                          target, accepted, bonus, emitted, path);
}

}  // namespace dspark
