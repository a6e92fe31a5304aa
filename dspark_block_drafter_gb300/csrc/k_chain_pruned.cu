// Exact-bound candidate pruning of the Markov chain: one CTA per block, no grid-wide
// synchronisation, the Markov term evaluated only where it can change the result.
//
// For slot i of block b with previous token p, u = markov_w1[p] and the corrected logit
// of head row v is  z'[v] = z[v] + u . w2[:, v]  (llama.cpp commit 6fed9f6, the proposal
// formula).  By Cauchy-Schwarz |u . w2[:, v]| <= |u| |w2[:, v]|, so with U = |u|,
// cn[v] = |w2[:, v]| and, per 128-row tile T, zmax[T] = max z and cmax[T] = max cn:
//   * each tile holds a row with z' >= lb[T] = zmax[T] - U cmax[T]  (its z-maximum);
//   * theta = the k-th largest lb[T] is therefore <= the k-th largest z';
//   * a row can reach the top k only if ub[v] = z[v] + U cn[v] >= theta, and a tile only
//     if zmax[T] + U cmax[T] >= theta.
// The kernel evaluates z' exactly (fp32) for the rows that pass and selects the argmax
// (the next previous token) and the top-k among them.  Both bounds carry a small margin
// for fp32 rounding, so the selection equals that of evaluating every row.  Any number
// of candidates is handled (the buffer is flushed and reduced to its best k as it
// fills), so the pruning only changes the cost, never the result.
//
// One-time preparation (dspark_prepare_head) stores markov_w2 transposed ([V_head][r],
// so a row's Markov weights are 512 contiguous bytes at r = 256), the column norms cn
// and their per-tile maxima.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxKeep = 33;                 // survivors of a reduction: top_k <= 32, + argmax
// candidate buffer entries: one round of appends (kWarps tiles of kTile rows) on top of
// the survivors of a reduction
constexpr int kCand = kWarps * kTile + 64;
static_assert(kCand >= kWarps * kTile + kMaxKeep, "candidate buffer too small");
constexpr float kRelMargin = 1.0f / 1024;    // fp32 rounding margins of the bounds
constexpr float kAbsMargin = 1e-4f;

// ------------------------------------------------------------------ preparation
// w2t[v][k] = w2[k][v] through 32 x 32 shared-memory tiles.
__global__ void __launch_bounds__(256)
prepare_transpose(const __nv_bfloat16* __restrict__ w2, int r, int Vh, size_t Vhp,
                  __nv_bfloat16* __restrict__ w2t) {
  __shared__ unsigned short tile[32][34];
  const int v0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;     // 32 x 8
  for (int y = ty; y < 32; y += 8) {
    const int k = k0 + y, v = v0 + tx;
    tile[y][tx] = (k < r && v < Vh) ? __bfloat16_as_ushort(w2[(size_t)k * Vh + v]) : 0;
  }
  __syncthreads();
  for (int y = ty; y < 32; y += 8) {
    const int v = v0 + y, k = k0 + tx;
    if (v < (int)Vhp && k < r) w2t[(size_t)v * r + k] = __ushort_as_bfloat16(tile[tx][y]);
  }
}

// cnorm[v] = |w2[:, v]| (fp32 sum of squares of the bf16 values), one warp per row of
// w2t; cnmax[T] = the maximum over the tile (rows past V_head have norm 0).
__global__ void __launch_bounds__(kTile)
prepare_norms(const __nv_bfloat16* __restrict__ w2t, int r, size_t Vhp,
              float* __restrict__ cnorm, float* __restrict__ cnmax) {
  __shared__ float s_max[kTile / 32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float tile_max = 0.f;
  for (int v = blockIdx.x * kTile + warp; v < (int)((blockIdx.x + 1) * kTile); v += kTile / 32) {
    float s = 0.f;
    for (int k = lane; k < r; k += 32) {
      const float w = __bfloat162float(w2t[(size_t)v * r + k]);
      s = fmaf(w, w, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float n = sqrtf(s);
    if (lane == 0) cnorm[v] = n;
    tile_max = fmaxf(tile_max, n);
  }
  if (lane == 0) s_max[warp] = tile_max;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.f;
    for (int w = 0; w < kTile / 32; ++w) m = fmaxf(m, s_max[w]);
    cnmax[blockIdx.x] = m;
  }
}

// ------------------------------------------------------------------ the chain
struct PrunedArgs {
  const float* z;          // [N][Vhp][ldb]
  const float* zmax;       // [N][B][T]
  size_t Vhp, ldb;
  const __nv_bfloat16* w1;   // [V][r]
  const __nv_bfloat16* w2t;  // [Vhp][r]
  const float* cnorm;      // [Vhp]
  const float* cnmax;      // [T]
  const int32_t* anchors;
  const int32_t* d2t;
  int32_t* draft;          // [B][N]
  int32_t* topk_ids;       // [B][N][k] or NULL
  float* topk_vals;
  uint32_t* err;
  int B, N, V, Vh, r, T, k, zrank, want_topk;
};

struct Cand {
  float x;     // corrected logit (NaN until evaluated)
  float z;     // base logit
  int v;       // head row
};

// Block-wide best (value, id) under the candidate order among buffer entries strictly
// after (pv, pid) (or all, when first); the value is x or z.  Every thread returns it.
__device__ void block_pick(const Cand* buf, int n, bool by_z, bool first, float pv, int pid,
                           float& out_v, int& out_id, float* s_v, int* s_i) {
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  for (int j = threadIdx.x; j < n; j += kThreads) {
    const float x = by_z ? buf[j].z : buf[j].x;
    const int id = buf[j].v;
    if (!first && !better(pv, pid, x, id)) continue;
    if (better(x, id, bv, bi)) {
      bv = x;
      bi = id;
    }
  }
  warp_best(bv, bi);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  __syncthreads();
  if (l == 0) {
    s_v[w] = bv;
    s_i[w] = bi;
  }
  __syncthreads();
  bv = l < kWarps ? s_v[l] : -INFINITY;
  bi = l < kWarps ? s_i[l] : 0x7FFFFFFF;
  warp_best(bv, bi);
  out_v = bv;
  out_id = bi;
}

// Block-wide k-th best of vals[0..n) (ids = indices) under the candidate order;
// -inf when n < k.
__device__ float block_kth(const float* vals, int n, int k, float* s_v, int* s_i) {
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  float pv = 0.f, res = -INFINITY;
  int pid = 0;
  for (int q = 0; q < k; ++q) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int t = threadIdx.x; t < n; t += kThreads)
      if ((q == 0 || better(pv, pid, vals[t], t)) && better(vals[t], t, bv, bi)) {
        bv = vals[t];
        bi = t;
      }
    warp_best(bv, bi);
    __syncthreads();
    if (l == 0) {
      s_v[w] = bv;
      s_i[w] = bi;
    }
    __syncthreads();
    bv = l < kWarps ? s_v[l] : -INFINITY;
    bi = l < kWarps ? s_i[l] : 0x7FFFFFFF;
    warp_best(bv, bi);
    pv = bv;
    pid = bi;
    res = bv;
  }
  return n < k ? -INFINITY : res;
}

// Corrected logits of every buffer entry not evaluated yet (x is NaN): one warp per
// entry, u from shared memory, the row of markov_w2 transposed from global memory.
__device__ void evaluate(Cand* buf, int n, const float* s_u, const __nv_bfloat16* w2t, int r) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int e = warp; e < n; e += kWarps) {
    if (buf[e].x == buf[e].x) continue;
    const __nv_bfloat16* w = w2t + (size_t)buf[e].v * r;
    float s = 0.f;
    for (int q = lane * 8; q < r; q += 32 * 8) {
      if ((r & 7) == 0) {
        const uint4 raw = *reinterpret_cast<const uint4*>(w + q);
        const __nv_bfloat16* e8 = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
        for (int c = 0; c < 8; ++c) s = fmaf(s_u[q + c], __bfloat162float(e8[c]), s);
      } else {
        for (int c = 0; c < 8 && q + c < r; ++c) s = fmaf(s_u[q + c], __bfloat162float(w[q + c]), s);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if (lane == 0) buf[e].x = buf[e].z + s;
  }
}

// Evaluate the buffer and shrink it to the entries that can still matter: the best kk by
// the ranked value and the best by corrected logit.  Called by the whole block.
__device__ void reduce_buffer(Cand* buf, int* s_n, int kk, bool by_z, const float* s_u,
                              const __nv_bfloat16* w2t, int r, float* s_v, int* s_i,
                              int* s_keep, Cand* s_stage) {
  const int n = *s_n;
  evaluate(buf, n, s_u, w2t, r);
  __syncthreads();
  // pick the survivors' head rows first, then gather them to the front
  int nk = 0;
  float pv = 0.f;
  int pid = 0;
  for (int q = 0; q < kk && q < n; ++q) {
    float bv;
    int bi;
    block_pick(buf, n, by_z, q == 0, pv, pid, bv, bi, s_v, s_i);
    if (threadIdx.x == 0) s_keep[nk] = bi;
    ++nk;
    pv = bv;
    pid = bi;
  }
  float av;
  int ai;
  block_pick(buf, n, false, true, 0.f, 0, av, ai, s_v, s_i);
  __syncthreads();
  bool have = false;
  for (int q = 0; q < nk; ++q) have |= s_keep[q] == ai;
  if (!have) {
    if (threadIdx.x == 0) s_keep[nk] = ai;
    ++nk;
  }
  __syncthreads();
  // copy the survivors out to a staging area, then back to the front of the buffer
  for (int j = threadIdx.x; j < n; j += kThreads)
    for (int q = 0; q < nk; ++q)
      if (buf[j].v == s_keep[q]) s_stage[q] = buf[j];
  __syncthreads();
  if (threadIdx.x < nk) buf[threadIdx.x] = s_stage[threadIdx.x];
  if (threadIdx.x == 0) *s_n = nk;
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
chain_pruned(const PrunedArgs a) {
  extern __shared__ float smem[];
  float* s_u = smem;                                   // [r]
  float* s_cnmax = s_u + ((a.r + 3) & ~3);             // [T]
  float* s_lb = s_cnmax + ((a.T + 3) & ~3);            // [T]
  Cand* buf = (Cand*)(s_lb + ((a.T + 3) & ~3));        // [kCand]
  __shared__ float s_red_v[kWarps];
  __shared__ int s_red_i[kWarps];
  __shared__ int s_n, s_prev, s_ntiles;
  __shared__ int s_tiles[kThreads];
  __shared__ int s_keep[kMaxKeep];
  __shared__ Cand s_stage[kMaxKeep];
  __shared__ float s_U;

  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  for (int t = tid; t < a.T; t += kThreads) s_cnmax[t] = a.cnmax[t];
  if (tid == 0) s_prev = a.anchors[b];
  const int kk = a.want_topk ? a.k : 1;                // ranks kept
  __syncthreads();

  for (int step = 0; step < a.N; ++step) {
    // -------- u = markov_w1[prev] and its norm (rounded up by a small margin)
    int p = s_prev;
    if (p < 0 || p >= a.V) {
      if (tid == 0) flag_error(a.err, kErrBadToken);
      p = 0;
    }
    float ss = 0.f;
    for (int q = tid; q < a.r; q += kThreads) {
      const float u = __bfloat162float(a.w1[(size_t)p * a.r + q]);
      s_u[q] = u;
      ss = fmaf(u, u, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (lane == 0) s_red_v[warp] = ss;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int w = 0; w < kWarps; ++w) t += s_red_v[w];
      s_U = sqrtf(t) * (1.f + kRelMargin);
      s_n = 0;
    }
    __syncthreads();
    const float U = s_U;
    const float* zm = a.zmax + ((size_t)step * a.B + b) * a.T;
    // -------- thresholds
    for (int t = tid; t < a.T; t += kThreads)
      s_lb[t] = zm[t] - U * s_cnmax[t] * (1.f + kRelMargin) - kAbsMargin;
    __syncthreads();
    // corrected logits: the k-th best lower bound (only the argmax when ranking z)
    const float theta_x = block_kth(s_lb, a.T, a.zrank ? 1 : kk, s_red_v, s_red_i);
    float theta_z = INFINITY;
    if (a.zrank) {
      __syncthreads();
      for (int t = tid; t < a.T; t += kThreads) s_lb[t] = zm[t];
      __syncthreads();
      theta_z = block_kth(s_lb, a.T, kk, s_red_v, s_red_i) - kAbsMargin;
    }
    // -------- candidates
    const float* z_i = a.z + (size_t)step * a.Vhp * a.ldb + b;
    for (int t0 = 0; t0 < a.T; t0 += kThreads) {
      __syncthreads();
      if (tid == 0) s_ntiles = 0;
      __syncthreads();
      {
        const int t = t0 + tid;
        if (t < a.T) {
          const bool cx = zm[t] + U * s_cnmax[t] * (1.f + kRelMargin) + kAbsMargin >= theta_x;
          const bool cz = zm[t] >= theta_z;
          if (cx || cz) s_tiles[atomicAdd(&s_ntiles, 1)] = t;
        }
      }
      __syncthreads();
      const int nt = s_ntiles;
      for (int j0 = 0; j0 < nt; j0 += kWarps) {
        if (s_n + kWarps * kTile > kCand)
          reduce_buffer(buf, &s_n, kk, a.zrank != 0, s_u, a.w2t, a.r, s_red_v, s_red_i, s_keep,
                        s_stage);
        const int j = j0 + warp;
        if (j < nt) {
          const int t = s_tiles[j];
#pragma unroll
          for (int q = 0; q < kTile / 32; ++q) {
            const int v = t * kTile + q * 32 + lane;
            bool take = false;
            float zv = -INFINITY;
            if (v < a.Vh) {
              zv = z_i[(size_t)v * a.ldb];
              const float ub = zv + U * a.cnorm[v] * (1.f + kRelMargin) + kAbsMargin;
              take = ub >= theta_x || zv >= theta_z;
            }
            const unsigned m = __ballot_sync(0xFFFFFFFFu, take);
            int base = 0;
            if (lane == 0 && m) base = atomicAdd(&s_n, __popc(m));
            base = __shfl_sync(0xFFFFFFFFu, base, 0);
            if (take) {
              const int slot = base + __popc(m & ((1u << lane) - 1));
              buf[slot].z = zv;
              buf[slot].v = v;
              buf[slot].x = NAN;            // evaluated later
            }
          }
        }
        __syncthreads();
      }
    }
    // -------- evaluation and selection
    const int n = s_n;
    evaluate(buf, n, s_u, a.w2t, a.r);
    __syncthreads();
    float av;
    int ai;
    block_pick(buf, n, false, true, 0.f, 0, av, ai, s_red_v, s_red_i);
    if (ai < 0 || ai >= a.Vh) ai = 0;       // only if every candidate value was NaN
    const int tok = a.d2t ? a.d2t[ai] : ai;
    if (tid == 0) {
      a.draft[(size_t)b * a.N + step] = tok;
      s_prev = tok;
    }
    if (a.want_topk) {
      float pv = 0.f;
      int pid = 0;
      for (int q = 0; q < a.k; ++q) {
        float bv;
        int bi;
        block_pick(buf, n, a.zrank != 0, q == 0, pv, pid, bv, bi, s_red_v, s_red_i);
        if (tid == 0) {
          const size_t o = ((size_t)b * a.N + step) * a.k + q;
          const int row = (bi >= 0 && bi < a.Vh) ? bi : 0;   // fewer candidates than k:
                                                              // impossible for k <= V_head
          if (a.topk_ids) a.topk_ids[o] = a.d2t ? a.d2t[row] : row;
          if (a.topk_vals) a.topk_vals[o] = bv;
        }
        pv = bv;
        pid = bi;
      }
    }
    __syncthreads();
  }
}

}  // namespace

PreparedLayout plan_prepared(int Vh, int r) {
  PreparedLayout l{};
  l.Vhp = align_up((size_t)Vh, kTile);
  l.tiles = l.Vhp / kTile;
  size_t off = 0;
  l.w2t = off;
  off = align_up(off + l.Vhp * r * sizeof(__nv_bfloat16), 256);
  l.cnorm = off;
  off = align_up(off + l.Vhp * sizeof(float), 256);
  l.cnmax = off;
  off = align_up(off + l.tiles * sizeof(float), 256);
  l.total = off;
  return l;
}

cudaError_t launch_prepare_head(const void* w2, int r, int Vh, void* prepared,
                                cudaStream_t stream) {
  const PreparedLayout l = plan_prepared(Vh, r);
  char* base = (char*)prepared;
  __nv_bfloat16* w2t = (__nv_bfloat16*)(base + l.w2t);
  dim3 g1((unsigned)(l.Vhp / 32), (unsigned)((r + 31) / 32));
  prepare_transpose<<<g1, 256, 0, stream>>>((const __nv_bfloat16*)w2, r, Vh, l.Vhp, w2t);
  prepare_norms<<<(unsigned)l.tiles, kTile, 0, stream>>>(w2t, r, l.Vhp,
                                                         (float*)(base + l.cnorm),
                                                         (float*)(base + l.cnmax));
  return cudaGetLastError();
}

cudaError_t launch_chain_pruned(const ProposePlan& p) {
  PrunedArgs a{};
  a.z = p.z;
  a.zmax = p.zmax;
  a.Vhp = p.Vhp;
  a.ldb = p.ldb;
  a.w1 = (const __nv_bfloat16*)p.w1;
  a.w2t = p.w2t;
  a.cnorm = p.cnorm;
  a.cnmax = p.cnmax;
  a.anchors = p.anchors;
  a.d2t = p.d2t;
  a.draft = p.draft;
  a.topk_ids = p.topk_ids;
  a.topk_vals = p.topk_vals;
  a.err = p.ctrl;
  a.B = p.B;
  a.N = p.N;
  a.V = p.V;
  a.Vh = p.Vh;
  a.r = p.r;
  a.T = (int)(p.Vhp / kTile);
  a.k = p.k;
  a.want_topk = (p.topk_ids || p.topk_vals) ? 1 : 0;
  a.zrank = (a.want_topk && !p.topk_markov) ? 1 : 0;
  const size_t smem = sizeof(float) * (((a.r + 3) & ~3) + 2 * ((a.T + 3) & ~3)) +
                      sizeof(Cand) * kCand;
  cudaError_t e = cudaFuncSetAttribute(chain_pruned, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  chain_pruned<<<p.B, kThreads, smem, p.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dspark
