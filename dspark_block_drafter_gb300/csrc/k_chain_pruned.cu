// Exact-bound candidate pruning of the Markov chain.
//
// For slot i of block b with previous token p, u = markov_w1[p] and the corrected logit
// of head row v is  z'[v] = z[v] + u . w2[:, v]  (llama.cpp commit 6fed9f6, the proposal
// formula).  By Cauchy-Schwarz |u . w2[:, v]| <= |u| |w2[:, v]| <= Umax cn[v], where
// Umax = max_p |markov_w1[p]| and cn[v] = |w2[:, v]|.  With, per 128-row tile T,
// zmax[T] = max z (emitted by the lm_head GEMM) and cmax[T] = max cn:
//   * each tile holds a row with z' >= lb[T] = zmax[T] - Umax cmax[T] (its z-maximum);
//   * theta = the k-th largest lb[T] is therefore <= the k-th largest z';
//   * a row can reach the top k only if ub[v] = z[v] + Umax cn[v] >= theta, and a tile
//     only if zmax[T] + Umax cmax[T] >= theta.
// None of this depends on the previous token, so the candidate rows of every (slot,
// block) are found by one fully parallel kernel; the sequential chain then evaluates z'
// exactly (fp32) for the candidates only (their markov_w2 rows prefetched one slot
// ahead) and selects the argmax (the next previous token) and the top-k.  The bounds
// carry a small margin for fp32 rounding, so the selection equals that of evaluating
// every row.  A (slot, block) with more candidates than the list holds is evaluated
// over every row instead, so the pruning only changes the cost, never the result.
//
// One-time preparation (dspark_prepare_head) stores markov_w2 transposed ([V_head][r],
// a row's Markov weights contiguous), the column norms cn, their per-tile maxima and
// Umax.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kTile = 128;
constexpr int kThreads = 256;
constexpr int kCap = 512;                    // candidate list entries per (slot, block)
constexpr int kRowsMax = 64;                 // candidates whose rows are staged per slot
constexpr size_t kRowsBytes = 128 * 1024;     // shared memory for both staging buffers
constexpr int kCandThreads = 512;            // threads of the candidate pass
constexpr int kCandWarps = kCandThreads / 32;
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

// Umax: the largest Euclidean norm of a markov_w1 row (one warp per row; positive
// floats compare like their bit patterns, so an unsigned atomicMax keeps the maximum).
__global__ void __launch_bounds__(256)
prepare_w1max(const __nv_bfloat16* __restrict__ w1, int V, int r, unsigned* __restrict__ out) {
  const int lane = threadIdx.x % 32;
  const int row0 = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int rows = gridDim.x * blockDim.x / 32;
  float best = 0.f;
  for (int p = row0; p < V; p += rows) {
    float s = 0.f;
    for (int k = lane; k < r; k += 32) {
      const float w = __bfloat162float(w1[(size_t)p * r + k]);
      s = fmaf(w, w, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    best = fmaxf(best, sqrtf(s));
  }
  if (lane == 0) atomicMax(out, __float_as_uint(best));
}

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

// Warp-wide best (value, id) among vals/ids[0..n) strictly after (pv, pid) (all when
// first).  Called by all 32 lanes of one warp; every lane returns the result.
__device__ __forceinline__ void warp_pick(const float* vals, const int* ids, int n, bool first,
                                          float pv, int pid, float& out_v, int& out_id) {
  const int lane = threadIdx.x % 32;
  float bv = -INFINITY;
  int bi = 0x7FFFFFFF;
  for (int j = lane; j < n; j += 32) {
    const float x = vals[j];
    const int id = ids ? ids[j] : j;
    if (!first && !better(pv, pid, x, id)) continue;
    if (better(x, id, bv, bi)) {
      bv = x;
      bi = id;
    }
  }
  warp_best(bv, bi);
  out_v = bv;
  out_id = bi;
}

// Block-wide k-th best of vals[0..n) (ids = indices), with two block barriers: every
// warp selects the best k of its stride, then warp 0 selects from those.  -inf when
// n < k.  Uses scratch[] (>= kWarps * k floats and ints).
__device__ float block_kth_fast(const float* vals, int n, int k, float* sc_v, int* sc_i,
                                float* s_out) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nw = blockDim.x / 32;
  // warp w covers indices [w * chunk, (w + 1) * chunk)
  const int chunk = (n + nw - 1) / nw;
  const int lo = min(n, warp * chunk), hi = min(n, lo + chunk);
  float pv = 0.f;
  int pid = 0;
  for (int q = 0; q < k; ++q) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
    for (int t = lo + lane; t < hi; t += 32)
      if ((q == 0 || better(pv, pid, vals[t], t)) && better(vals[t], t, bv, bi)) {
        bv = vals[t];
        bi = t;
      }
    warp_best(bv, bi);
    if (lane == 0) {
      sc_v[warp * k + q] = bv;
      sc_i[warp * k + q] = bi;
    }
    pv = bv;
    pid = bi;
  }
  __syncthreads();
  if (warp == 0) {
    float rv = -INFINITY;
    pv = 0.f;
    pid = 0;
    for (int q = 0; q < k; ++q) {
      float bv;
      int bi;
      warp_pick(sc_v, sc_i, nw * k, q == 0, pv, pid, bv, bi);
      pv = bv;
      pid = bi;
      rv = bv;
    }
    if (lane == 0) *s_out = n < k ? -INFINITY : rv;
  }
  __syncthreads();
  return *s_out;
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


// ------------------------------------------------------------------ candidates
struct CandArgs {
  const float* z;          // [N][Vhp][ldb]
  const float* zmax;       // [N][B][T]
  size_t Vhp, ldb;
  const float* cnorm;      // [Vhp]
  const float* cnmax;      // [T]
  const unsigned* w1max;   // Umax as float bits
  int32_t* cand_v;         // [N][B][kCap]
  float* cand_z;           // [N][B][kCap]
  int32_t* cand_n;         // [N][B] (zeroed; may exceed kCap: the list overflowed)
  int B, N, Vh, T, kk, zrank;
};

// One CTA per (slot, block): thresholds, candidate tiles, candidate rows.
__global__ void __launch_bounds__(kCandThreads)
pruned_candidates(const CandArgs a) {
  extern __shared__ float smem[];
  float* s_lb = smem;                                   // [T]
  int* s_tiles = (int*)(s_lb + ((a.T + 3) & ~3));       // [T]
  __shared__ float s_sc_v[kCandWarps * 32];
  __shared__ int s_sc_i[kCandWarps * 32];
  __shared__ float s_theta;
  __shared__ int s_ntiles;
  const int b = blockIdx.x, i = blockIdx.y;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float* zm = a.zmax + ((size_t)i * a.B + b) * a.T;
  const float umax = __uint_as_float(*a.w1max) * (1.f + kRelMargin);
  for (int t = tid; t < a.T; t += kCandThreads)
    s_lb[t] = zm[t] - umax * a.cnmax[t] * (1.f + kRelMargin) - kAbsMargin;
  if (tid == 0) s_ntiles = 0;
  __syncthreads();
  const float theta_x =
      block_kth_fast(s_lb, a.T, a.zrank ? 1 : a.kk, s_sc_v, s_sc_i, &s_theta);
  float theta_z = INFINITY;
  if (a.zrank) {
    for (int t = tid; t < a.T; t += kCandThreads) s_lb[t] = zm[t];
    __syncthreads();
    theta_z = block_kth_fast(s_lb, a.T, a.kk, s_sc_v, s_sc_i, &s_theta) - kAbsMargin;
  }
  for (int t = tid; t < a.T; t += kCandThreads) {
    const bool cx = zm[t] + umax * a.cnmax[t] * (1.f + kRelMargin) + kAbsMargin >= theta_x;
    if (cx || zm[t] >= theta_z) s_tiles[atomicAdd(&s_ntiles, 1)] = t;
  }
  __syncthreads();
  const int nt = s_ntiles;
  const float* z_i = a.z + (size_t)i * a.Vhp * a.ldb + b;
  int32_t* cv = a.cand_v + ((size_t)i * a.B + b) * kCap;
  float* cz = a.cand_z + ((size_t)i * a.B + b) * kCap;
  int32_t* cn = a.cand_n + (size_t)i * a.B + b;
  for (int j = warp; j < nt; j += kCandWarps) {
    const int t = s_tiles[j];
#pragma unroll
    for (int q = 0; q < kTile / 32; ++q) {
      const int v = t * kTile + q * 32 + lane;
      bool take = false;
      float zv = -INFINITY;
      if (v < a.Vh) {
        zv = z_i[(size_t)v * a.ldb];
        const float ub = zv + umax * a.cnorm[v] * (1.f + kRelMargin) + kAbsMargin;
        take = ub >= theta_x || zv >= theta_z;
      }
      const unsigned m = __ballot_sync(0xFFFFFFFFu, take);
      int base = 0;
      if (lane == 0 && m) base = atomicAdd(cn, __popc(m));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (take) {
        const int slot = base + __popc(m & ((1u << lane) - 1));
        if (slot < kCap) {
          cv[slot] = v;
          cz[slot] = zv;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ the chain
struct PrunedArgs {
  const float* z;            // [N][Vhp][ldb] (only read on list overflow)
  size_t Vhp, ldb;
  const __nv_bfloat16* w1;   // [V][r]
  const __nv_bfloat16* w2t;  // [Vhp][r]
  const int32_t* cand_v;
  const float* cand_z;
  const int32_t* cand_n;
  const int32_t* anchors;
  const int32_t* d2t;
  int32_t* draft;            // [B][N]
  int32_t* topk_ids;         // [B][N][k] or NULL
  float* topk_vals;
  uint32_t* err;
  int B, N, V, Vh, r, k, kk, zrank, want_topk;
  int rows_cap;              // candidates whose rows are staged per slot
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_prev() {    // all but the latest group
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// Stage the markov_w2 rows and the markov_w1 rows (the candidate as a previous token)
// of the first `cap` candidates of a list into shared memory.
__device__ void stage_rows(const int32_t* s_v, int n, int cap, const __nv_bfloat16* w2t,
                           const __nv_bfloat16* w1, const int32_t* d2t, int r,
                           __nv_bfloat16* rows2, __nv_bfloat16* rows1) {
  const int chunks_per_row = r / 8;                      // r % 8 == 0 on this path
  const int total = min(n, cap) * chunks_per_row;
  for (int c = threadIdx.x; c < total; c += kThreads) {
    const int j = c / chunks_per_row, q = c % chunks_per_row;
    const int v = s_v[j];
    const int tok = d2t ? d2t[v] : v;
    cp_async16(rows2 + (size_t)j * r + q * 8, w2t + (size_t)v * r + q * 8);
    cp_async16(rows1 + (size_t)j * r + q * 8, w1 + (size_t)tok * r + q * 8);
  }
}

// z' = z + u . w2[:, v] for list entries [0, n): eight lanes per entry.  Lane `sub`
// takes the 8-element chunks sub, sub + 8, ... of the row, so that the eight lanes of an
// entry read consecutive 16-byte chunks of the row and of u (no bank conflicts); rows
// [0, cap) come from shared memory, later ones from global memory.
__device__ void evaluate_list(Cand* buf, int n, int cap, const float* s_u,
                              const __nv_bfloat16* rows, const __nv_bfloat16* w2t, int r) {
  const int sub = threadIdx.x % 8;
  const int chunks = r / 8;                              // r % 8 == 0 on this path
  for (int e0 = 0; e0 < n; e0 += kThreads / 8) {
    const int e = e0 + threadIdx.x / 8;
    float s0 = 0.f, s1 = 0.f;
    if (e < n) {
      const __nv_bfloat16* w = e < cap ? rows + (size_t)e * r : w2t + (size_t)buf[e].v * r;
      for (int c = sub; c < chunks; c += 8) {
        const uint4 raw = *reinterpret_cast<const uint4*>(w + c * 8);
        const float4 u0 = *reinterpret_cast<const float4*>(s_u + c * 8);
        const float4 u1 = *reinterpret_cast<const float4*>(s_u + c * 8 + 4);
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
        const float2 w01 = __bfloat1622float2(p2[0]), w23 = __bfloat1622float2(p2[1]);
        const float2 w45 = __bfloat1622float2(p2[2]), w67 = __bfloat1622float2(p2[3]);
        s0 = fmaf(u0.x, w01.x, s0);
        s1 = fmaf(u0.y, w01.y, s1);
        s0 = fmaf(u0.z, w23.x, s0);
        s1 = fmaf(u0.w, w23.y, s1);
        s0 = fmaf(u1.x, w45.x, s0);
        s1 = fmaf(u1.y, w45.y, s1);
        s0 = fmaf(u1.z, w67.x, s0);
        s1 = fmaf(u1.w, w67.y, s1);
      }
    }
    float s = s0 + s1;
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 4);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
    s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
    if (e < n && sub == 0) buf[e].x = buf[e].z + s;
  }
}

// One CTA per block walks its N slots.  The candidate lists, the markov_w2 rows and the
// markov_w1 rows of slot i + 1 are staged while slot i is evaluated, so that a slot's
// critical path touches shared memory only.
__global__ void __launch_bounds__(kThreads)
chain_pruned(const PrunedArgs a) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const size_t rows_elems = (size_t)a.rows_cap * a.r;
  __nv_bfloat16* s_rows2 = (__nv_bfloat16*)dsm;                  // [2][rows_cap][r]
  __nv_bfloat16* s_rows1 = s_rows2 + 2 * rows_elems;              // [2][rows_cap][r]
  float* s_u = (float*)(s_rows1 + 2 * rows_elems);                // [r]
  int32_t* s_lv = (int32_t*)(s_u + ((a.r + 3) & ~3));             // [2][kCap]
  float* s_lz = (float*)(s_lv + 2 * kCap);                        // [2][kCap]
  Cand* buf = (Cand*)(s_lz + 2 * kCap);                           // [kCand]
  __shared__ float s_red_v[kWarps];
  __shared__ int s_red_i[kWarps];
  __shared__ int s_n[2], s_nfull, s_prev, s_sel;
  __shared__ int s_keep[kMaxKeep];
  __shared__ Cand s_stage[kMaxKeep];

  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  auto list_base = [&](int i) { return ((size_t)i * a.B + b) * kCap; };
  auto load_list = [&](int i, int slot) {
    const int n = a.cand_n[(size_t)i * a.B + b];
    const int m = min(n, kCap);
    for (int j = tid; j < m; j += kThreads) {
      s_lv[slot * kCap + j] = a.cand_v[list_base(i) + j];
      s_lz[slot * kCap + j] = a.cand_z[list_base(i) + j];
    }
    if (tid == 0) s_n[slot] = n;
  };
  // slot 0: u from the anchor, list and rows of slot 0, list of slot 1
  {
    int p = a.anchors[b];
    if (p < 0 || p >= a.V) {
      if (tid == 0) flag_error(a.err, kErrBadToken);
      p = 0;
    }
    for (int q = tid; q < a.r; q += kThreads) s_u[q] = __bfloat162float(a.w1[(size_t)p * a.r + q]);
    load_list(0, 0);
    if (a.N > 1) load_list(1, 1);
    __syncthreads();
    if (s_n[0] <= kCap)
      stage_rows(s_lv, s_n[0], a.rows_cap, a.w2t, a.w1, a.d2t, a.r, s_rows2, s_rows1);
    cp_async_commit();
  }

  for (int step = 0; step < a.N; ++step) {
    const int cur = step & 1, nxt = cur ^ 1;
    // -------- stage the next slot's rows (its list is in), fetch the list after it
    if (step + 1 < a.N && s_n[nxt] <= kCap)
      stage_rows(s_lv + nxt * kCap, s_n[nxt], a.rows_cap, a.w2t, a.w1, a.d2t, a.r,
                 s_rows2 + nxt * rows_elems, s_rows1 + nxt * rows_elems);
    cp_async_commit();
    // the list two slots ahead: plain loads issued now (the whole kCap slots, so that no
    // instruction waits on the count), stored to shared memory after this slot
    int nv2 = 0, v2[kCap / kThreads];
    float z2[kCap / kThreads];
    if (step + 2 < a.N) {
      nv2 = a.cand_n[(size_t)(step + 2) * a.B + b];
#pragma unroll
      for (int q = 0; q < kCap / kThreads; ++q) {
        const int j = tid + q * kThreads;
        v2[q] = a.cand_v[list_base(step + 2) + j];
        z2[q] = a.cand_z[list_base(step + 2) + j];
      }
    }
    cp_async_wait_prev();                      // this slot's rows
    __syncthreads();
    const int n = s_n[cur];
    float av;
    int ai;
    int nsel;
    if (n <= kCap) {
      // -------- exact z' of the candidates
      for (int j = tid; j < n; j += kThreads) {
        buf[j].v = s_lv[cur * kCap + j];
        buf[j].z = s_lz[cur * kCap + j];
      }
      __syncthreads();
      evaluate_list(buf, n, a.rows_cap, s_u, s_rows2 + cur * rows_elems, a.w2t, a.r);
      __syncthreads();
      nsel = n;
    } else {
      // -------- the list overflowed: every row, streamed through the buffer
      if (tid == 0) s_nfull = 0;
      __syncthreads();
      const float* z_i = a.z + (size_t)step * a.Vhp * a.ldb + b;
      for (int v0 = 0; v0 < a.Vh; v0 += kCand - kMaxKeep) {
        const int cnt = min(kCand - kMaxKeep, a.Vh - v0);
        const int base = s_nfull;
        __syncthreads();
        for (int j = tid; j < cnt; j += kThreads) {
          buf[base + j].v = v0 + j;
          buf[base + j].z = z_i[(size_t)(v0 + j) * a.ldb];
          buf[base + j].x = NAN;
        }
        __syncthreads();
        if (tid == 0) s_nfull = base + cnt;
        __syncthreads();
        reduce_buffer(buf, &s_nfull, a.kk, a.zrank != 0, s_u, a.w2t, a.r, s_red_v, s_red_i,
                      s_keep, s_stage);
      }
      nsel = s_nfull;
    }
    // -------- selection: each entry counts the entries that beat it (its rank)
    if (nsel <= kThreads) {
      if (tid == 0) s_sel = -1;
      __syncthreads();
      if (tid < nsel) {
        const float x = buf[tid].x, zz = buf[tid].z;
        const int v = buf[tid].v;
        const float rk = a.zrank ? zz : x;
        int rank_x = 0, rank_r = 0;
        for (int j = 0; j < nsel; ++j) {
          const float xj = buf[j].x;
          const float rj = a.zrank ? buf[j].z : xj;
          const int vj = buf[j].v;
          rank_x += better(xj, vj, x, v);
          rank_r += better(rj, vj, rk, v);
        }
        if (rank_x == 0) {                     // the argmax: the next previous token
          const int tok = a.d2t ? a.d2t[v] : v;
          a.draft[(size_t)b * a.N + step] = tok;
          s_prev = tok;
          s_sel = tid;
        }
        if (a.want_topk && rank_r < a.k) {
          const size_t o = ((size_t)b * a.N + step) * a.k + rank_r;
          if (a.topk_ids) a.topk_ids[o] = a.d2t ? a.d2t[v] : v;
          if (a.topk_vals) a.topk_vals[o] = rk;
        }
      }
      __syncthreads();
    } else {
      block_pick(buf, nsel, false, true, 0.f, 0, av, ai, s_red_v, s_red_i);
      if (ai < 0 || ai >= a.Vh) ai = 0;      // only if every candidate value was NaN
      const int tok = a.d2t ? a.d2t[ai] : ai;
      if (tid == 0) {
        a.draft[(size_t)b * a.N + step] = tok;
        s_prev = tok;
        s_sel = -1;
      }
      if (a.want_topk) {
        float pv = 0.f;
        int pid = 0;
        for (int q = 0; q < a.k; ++q) {
          float bv;
          int bi;
          block_pick(buf, nsel, a.zrank != 0, q == 0, pv, pid, bv, bi, s_red_v, s_red_i);
          if (tid == 0) {
            const size_t o = ((size_t)b * a.N + step) * a.k + q;
            const int row = (bi >= 0 && bi < a.Vh) ? bi : 0;   // fewer candidates than k:
                                                                // impossible, k <= V_head
            if (a.topk_ids) a.topk_ids[o] = a.d2t ? a.d2t[row] : row;
            if (a.topk_vals) a.topk_vals[o] = bv;
          }
          pv = bv;
          pid = bi;
        }
      }
      __syncthreads();
    }
    // -------- the next slot's u: staged with this slot's candidates when possible
    {
      const int sel = s_sel;
      int p = s_prev;
      if (p < 0 || p >= a.V) {
        if (tid == 0) flag_error(a.err, kErrBadToken);
        p = 0;
      }
      if (sel >= 0 && sel < a.rows_cap && n <= kCap) {
        const __nv_bfloat16* src = s_rows1 + cur * rows_elems + (size_t)sel * a.r;
        for (int q = tid; q < a.r; q += kThreads) s_u[q] = __bfloat162float(src[q]);
      } else {
        for (int q = tid; q < a.r; q += kThreads)
          s_u[q] = __bfloat162float(a.w1[(size_t)p * a.r + q]);
      }
      // the list two slots ahead lands where this slot's list was
      if (step + 2 < a.N) {
        const int m = min(nv2, kCap);
#pragma unroll
        for (int q = 0; q < kCap / kThreads; ++q) {
          const int j = tid + q * kThreads;
          if (j < m) {
            s_lv[cur * kCap + j] = v2[q];
            s_lz[cur * kCap + j] = z2[q];
          }
        }
        if (tid == 0) s_n[cur] = nv2;
      }
      __syncthreads();
    }
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
  l.w1max = off;
  off = align_up(off + sizeof(unsigned), 256);
  l.total = off;
  return l;
}

size_t pruned_list_bytes(int B, int N) {
  return (size_t)N * B * kCap * (sizeof(int32_t) + sizeof(float));
}

cudaError_t launch_prepare_head(const void* w1, const void* w2, int V, int r, int Vh,
                                void* prepared, cudaStream_t stream) {
  const PreparedLayout l = plan_prepared(Vh, r);
  char* base = (char*)prepared;
  __nv_bfloat16* w2t = (__nv_bfloat16*)(base + l.w2t);
  dim3 g1((unsigned)(l.Vhp / 32), (unsigned)((r + 31) / 32));
  prepare_transpose<<<g1, 256, 0, stream>>>((const __nv_bfloat16*)w2, r, Vh, l.Vhp, w2t);
  prepare_norms<<<(unsigned)l.tiles, kTile, 0, stream>>>(w2t, r, l.Vhp,
                                                         (float*)(base + l.cnorm),
                                                         (float*)(base + l.cnmax));
  cudaError_t e = cudaMemsetAsync(base + l.w1max, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  const int rows_per_cta = 8;
  const int grid = std::min(4096, (V + rows_per_cta - 1) / rows_per_cta);
  prepare_w1max<<<grid, 256, 0, stream>>>((const __nv_bfloat16*)w1, V, r,
                                          (unsigned*)(base + l.w1max));
  return cudaGetLastError();
}

cudaError_t launch_chain_pruned(const ProposePlan& p) {
  const int T = (int)(p.Vhp / kTile);
  const bool want_topk = p.topk_ids || p.topk_vals;
  const int kk = want_topk ? p.k : 1;
  const int zrank = (want_topk && !p.topk_markov) ? 1 : 0;
  {
    CandArgs c{};
    c.z = p.z;
    c.zmax = p.zmax;
    c.Vhp = p.Vhp;
    c.ldb = p.ldb;
    c.cnorm = p.cnorm;
    c.cnmax = p.cnmax;
    c.w1max = p.w1max;
    c.cand_v = p.cand_v;
    c.cand_z = p.cand_z;
    c.cand_n = p.cand_n;
    c.B = p.B;
    c.N = p.N;
    c.Vh = p.Vh;
    c.T = T;
    c.kk = kk;
    c.zrank = zrank;
    const size_t smem = sizeof(float) * 2 * ((T + 3) & ~3);
    cudaError_t e = cudaFuncSetAttribute(pruned_candidates,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    pruned_candidates<<<dim3(p.B, p.N), kCandThreads, smem, p.stream>>>(c);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  PrunedArgs a{};
  a.z = p.z;
  a.Vhp = p.Vhp;
  a.ldb = p.ldb;
  a.w1 = (const __nv_bfloat16*)p.w1;
  a.w2t = p.w2t;
  a.cand_v = p.cand_v;
  a.cand_z = p.cand_z;
  a.cand_n = p.cand_n;
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
  a.k = p.k;
  a.kk = kk;
  a.zrank = zrank;
  a.want_topk = want_topk ? 1 : 0;
  a.rows_cap = (int)std::min<size_t>(kRowsMax, kRowsBytes / (4 * sizeof(__nv_bfloat16) * a.r));
  const size_t smem = sizeof(__nv_bfloat16) * 4 * (size_t)a.rows_cap * a.r +
                      sizeof(float) * ((a.r + 3) & ~3) +
                      (sizeof(int32_t) + sizeof(float)) * 2 * kCap + sizeof(Cand) * kCand;
  cudaError_t e = cudaFuncSetAttribute(chain_pruned, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  chain_pruned<<<p.B, kThreads, smem, p.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace dspark
