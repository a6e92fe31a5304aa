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
// None of this depends on the previous token.  So one fully parallel kernel, one CTA per
// (slot i, block b), finds the candidate rows C(i) of the slot (theta of rank k) and the
// rows A(i - 1) that can be the previous slot's argmax (theta of rank 1); the previous
// token of slot i is the head row chosen in slot i - 1, which lies in A(i - 1) (slot 0:
// the anchor).  It then evaluates z' exactly (fp32) for every pair of a possible previous
// row and a candidate: a small table.  The sequential walk over a block's slots, run by
// the last of the block's CTAs to finish its table, is left with table lookups per slot;
// the top-k of the rows taken is copied from the tables.  The bounds carry a margin for
// fp32 rounding, so every selection equals that of evaluating every row.  Where a list
// or a table would not fit (loose bounds), the walk evaluates that slot on the fly, over
// every row if need be, so the pruning only changes the cost, never the result.
//
// The lm_head GEMM applies the same bounds to leave out tiles of z that cannot reach a
// slot's top k (zwritten says which); such a tile counts here as one whose upper bound
// is -inf.
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
constexpr int kThreads = 256;                // threads of the kernels
constexpr int kWarps = kThreads / 32;
static_assert((kWarps & (kWarps - 1)) == 0 && kWarps <= 32, "warp count: a power of two");
constexpr int kCap = 512;                    // candidate list entries per (slot, block)
constexpr int kCapA = 16;                    // possible previous rows tabulated per slot
constexpr int kTabC = 128;                   // candidates tabulated per slot
constexpr int kRowsChunk = 32;               // markov_w2 rows staged at a time
constexpr int kMaxKeep = 33;                 // survivors of a reduction: top_k <= 32, + argmax
// candidate buffer entries: one round of appends (kWarps tiles of kTile rows) on top of
// the survivors of a reduction
constexpr int kCand = kWarps * kTile + 64;
static_assert(kCand >= kWarps * kTile + kMaxKeep, "candidate buffer too small");
constexpr float kRelMargin = kPrunedRelMargin;    // fp32 rounding margins of the bounds
constexpr float kAbsMargin = kPrunedAbsMargin;

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

// The header goes in last, so that a buffer whose preparation did not finish reads as
// unprepared.
__global__ void prepare_header(PreparedHeader* dst, const PreparedHeader h) { *dst = h; }

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



// ------------------------------------------------------------------ tables
// Bitonic sort of the warp's 32 (value, id) pairs into the candidate order: afterwards
// lane q holds the q-th best.
__device__ __forceinline__ void warp_sort(float& v, int& id) {
  const int lane = threadIdx.x % 32;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, stride);
      const int oid = __shfl_xor_sync(0xFFFFFFFFu, id, stride);
      // blocks of `size` lanes alternate between best-first and worst-first; the lower
      // lane of a pair keeps the better entry in a best-first block
      const bool best_first = ((lane & size) == 0) | (size == 32);
      const bool lower = (lane & stride) == 0;
      const bool ob = better(ov, oid, v, id), mb = better(v, id, ov, oid);
      const bool take = (best_first == lower) ? ob : mb;
      v = take ? ov : v;
      id = take ? oid : id;
    }
  }
}

// A lower bound on the k-th largest of the values the block's threads hold (k <= 32):
// the k-th largest of the per-thread values, which the caller made the maxima of
// disjoint subsets.  Since those maxima are a subset of the underlying values, their
// k-th largest never exceeds the true one; it equals it unless two of the top k share a
// thread.  Every warp sorts its 32, then warp 0 merges the warps' best k.
__device__ float block_kth_of_maxima(float val, int k, float* s_top, float* s_out) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (k == 1) {
    // the largest: a plain block maximum
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) val = fmaxf(val, __shfl_xor_sync(0xFFFFFFFFu, val, o));
    if (lane == 0) s_top[warp] = val;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = s_top[0];
      for (int w = 1; w < kWarps; ++w) m = fmaxf(m, s_top[w]);
      *s_out = m;
    }
    __syncthreads();
    return *s_out;
  }
  int id = lane;
  warp_sort(val, id);
  if (lane < k) s_top[warp * 32 + lane] = val;
  __syncthreads();
  if (warp == 0) {
    // k rounds over the heads of the warps' sorted lists (lanes 0 .. kWarps-1)
    int h = 0;
    float last = -INFINITY;
    for (int q = 0; q < k; ++q) {
      float c = (lane < kWarps && h < k) ? s_top[lane * 32 + h] : -INFINITY;
      int ci = lane;
#pragma unroll
      for (int o = kWarps / 2; o > 0; o >>= 1) {
        const float oc = __shfl_xor_sync(0xFFFFFFFFu, c, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, ci, o);
        const bool t = better(oc, oi, c, ci);
        c = t ? oc : c;
        ci = t ? oi : ci;
      }
      c = __shfl_sync(0xFFFFFFFFu, c, 0);            // lanes >= kWarps ran their own
      ci = __shfl_sync(0xFFFFFFFFu, ci, 0);          // groups; lane 0's group is the one
      h += (lane == ci);
      last = c;
    }
    if (lane == 0) *s_out = last;
  }
  __syncthreads();
  return *s_out;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

struct TableArgs {
  const float* z;            // octet layout (z_octet_index)
  const float* zmax;         // [N][B][T]
  const uint8_t* zw;         // [N][B][T]: 0 where the GEMM left the tile's z out, or NULL
  size_t Vhp, ldb;
  const float* cnorm;        // [Vhp]
  const float* cnmax;        // [T]
  const unsigned* w1max;     // Umax as float bits
  const __nv_bfloat16* w1;   // [V][r]
  const __nv_bfloat16* w2t;  // [Vhp][r]
  const int32_t* anchors;
  const int32_t* d2t;
  const __nv_bfloat16* hidden;   // [B][L_in][H], read for the confidence head
  const __nv_bfloat16* w_conf;   // [H] or NULL
  float b_conf;
  float* conf;               // [B][N]
  int32_t* cand_v;           // [N][B][kCap]
  float* cand_z;             // [N][B][kCap]
  int32_t* cand_n;           // [N][B] (above kCap: the list overflowed)
  int32_t* prev_v;           // [N][B][kCapA]
  int32_t* prev_n;           // [N][B] (above kCapA: too many to tabulate)
  int32_t* amax;             // [N][B][kCapA]: head row of the argmax given each prev row
  int32_t* tk_id;            // [N][B][kCapA][k]: top-k tokens given each prev row
  float* tk_val;             // [N][B][kCapA][k]
  uint32_t* err;
  int* walk_done;            // [B], zero at the start of the pass: table CTAs done per block
  const int32_t* nd_in;      // [B] cuts computed before the chain (adaptive block length:
                             // slots from the cut on are skipped), or NULL
  const PreparedHeader* prep;    // the prepared buffer's header
  PreparedHeader prep_want;      // what it must say for this head
  int B, N, V, Vh, T, r, k, kk, zrank, want_topk, L_in, ifp, H;
};

// One list of candidate tiles of a (slot, block) row of z: rows whose upper bound
// reaches theta_x or whose base logit reaches theta_z go to s_v (and s_z, when given):
// at most cap are kept, *s_cnt counts them all.
struct RowScan {
  size_t slot;
  const int* tiles;
  int ntiles;
  float theta_x, theta_z;
  int32_t* s_v;
  float* s_z;
  int cap;
  int* s_cnt;
};

// Both lists of a (slot, block) in one pass: one warp per tile, four rows a lane, and
// each warp loads four tiles (of either list) before it looks at them, so the rows of
// both lists cost one round of memory latency.  zrow(v) = z + z_octet_index(slot, v, b).
__device__ void scan_rows(const float* z, size_t b, size_t Vhp, size_t ldb, const float* cnorm,
                          float umax, int Vh, const RowScan& l0, const RowScan& l1) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  constexpr int kTilesPerRound = 4;
  const int ntiles = l0.ntiles + l1.ntiles;
  for (int j0 = warp; j0 < ntiles; j0 += kTilesPerRound * kWarps) {
    float4 z4[kTilesPerRound], c4[kTilesPerRound];
    int v0[kTilesPerRound];
#pragma unroll
    for (int h = 0; h < kTilesPerRound; ++h) {
      const int j = j0 + h * kWarps;
      v0[h] = -1;
      if (j < ntiles) {
        const RowScan& l = j < l0.ntiles ? l0 : l1;
        v0[h] = l.tiles[j < l0.ntiles ? j : j - l0.ntiles] * kTile + lane * 4;
        z4[h] = *reinterpret_cast<const float4*>(z + z_octet_index(l.slot, v0[h], b, Vhp, ldb));
        c4[h] = *reinterpret_cast<const float4*>(cnorm + v0[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < kTilesPerRound; ++h) {
      const int j = j0 + h * kWarps;
      if (j >= ntiles) break;                        // warp-uniform
      const RowScan& l = j < l0.ntiles ? l0 : l1;
      const float zq[4] = {z4[h].x, z4[h].y, z4[h].z, z4[h].w};
      const float cq[4] = {c4[h].x, c4[h].y, c4[h].z, c4[h].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int v = v0[h] + q;
        const bool take =
            (v < Vh) & ((zq[q] + umax * cq[q] * (1.f + kRelMargin) + kAbsMargin >= l.theta_x) |
                        (zq[q] >= l.theta_z));
        const unsigned m = __ballot_sync(0xFFFFFFFFu, take);
        if (m == 0) continue;
        int base = 0;
        if (lane == 0) base = atomicAdd(l.s_cnt, __popc(m));
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        if (take) {
          const int slot = base + __popc(m & ((1u << lane) - 1));
          if (slot < l.cap) {
            l.s_v[slot] = v;
            if (l.s_z) l.s_z[slot] = zq[q];
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ the walk
struct SelectArgs {
  const float* z;            // octet layout (read only to evaluate every row)
  const int32_t* nd_in;      // [B] cuts computed before the chain (adaptive block length:
                             // slots from the cut on are not drafted), or NULL
  const uint8_t* zw;         // [N][B][T]: 0 where the GEMM left the tile's z out, or NULL
  int T;
  size_t Vhp, ldb;
  const __nv_bfloat16* w1;   // [V][r]
  const __nv_bfloat16* w2t;  // [Vhp][r]
  const int32_t* cand_v;
  const float* cand_z;
  const int32_t* cand_n;
  const int32_t* prev_v;
  const int32_t* prev_n;
  const int32_t* amax;
  const int32_t* tk_id;
  const float* tk_val;
  const int32_t* anchors;
  const int32_t* d2t;
  const float* conf;         // [B][N], or NULL without a confidence head
  float conf_min;
  int32_t* n_draft;          // [B]
  int32_t* draft;            // [B][N]
  int32_t* topk_ids;         // [B][N][k] or NULL
  float* topk_vals;
  uint32_t* err;             // the control words: [0] error word, [1] slots evaluated on the
                             // fly (no table), [2] of those, over every head row
  int B, N, V, Vh, r, k, kk, zrank, want_topk;
};

constexpr int kMaxSlots = 256;               // prediction slots of the bf16 path

// z' = z + u . w2[:, v] for buffer entries [0, n), rows read from global memory: eight
// lanes per entry, lane `sub` taking the 8-element chunks sub, sub + 8, ... of the row.
__device__ void evaluate_list(Cand* buf, int n, const float* s_u, const __nv_bfloat16* w2t,
                              int r) {
  const int sub = threadIdx.x % 8;
  const int chunks = r / 8;                              // r % 8 == 0 on this path
  for (int e0 = 0; e0 < n; e0 += kThreads / 8) {
    const int e = e0 + threadIdx.x / 8;
    float s0 = 0.f, s1 = 0.f;
    if (e < n) {
      const __nv_bfloat16* w = w2t + (size_t)buf[e].v * r;
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

// Shared memory of the walk of one block, carved from the CTA's dynamic shared memory.
// (All of it overlays the tables' shared memory, which the walk no longer needs, so that
// the kernel's static shared memory stays small: four CTAs must fit an SM.)
__host__ __device__ inline size_t walk_smem_bytes(int r, int N) {
  return sizeof(float) * ((r + 3) & ~3) + sizeof(Cand) * (kCand + kMaxKeep) +
         sizeof(int) * 4 * (size_t)N + sizeof(int32_t) * 2 * (size_t)N * kCapA +
         sizeof(float) * (size_t)N + sizeof(float) * kWarps + sizeof(int) * kWarps +
         sizeof(int) * (3 + kMaxKeep) + 8 + sizeof(int2) * (size_t)N * kCapA;
}

// The walk of block b over its N slots, by the whole CTA (the last of the block's table
// CTAs to finish).  A tabulated slot is a lookup: the previous row's index in A(i - 1),
// then the argmax stored for it; warp 0 walks those alone.  A slot without a table (a
// list that overflowed, too many previous rows, a previous row not found) is evaluated
// on the fly by the whole CTA, over every row if need be.
__device__ void walk_block(const SelectArgs& a, int b, uint8_t* dsm) {
  float* s_u = (float*)dsm;                                    // [r]
  Cand* buf = (Cand*)(s_u + ((a.r + 3) & ~3));                 // [kCand]
  Cand* s_stage = buf + kCand;                                 // [kMaxKeep]
  int* s_nc = (int*)(s_stage + kMaxKeep);                      // [N] each
  int* s_na = s_nc + a.N;
  int* s_pi = s_na + a.N;
  int* s_row = s_pi + a.N;
  int32_t (*s_av)[kCapA] = reinterpret_cast<int32_t (*)[kCapA]>(s_row + a.N);   // [N][kCapA]
  int32_t (*s_am)[kCapA] = s_av + a.N;
  float* s_conf = reinterpret_cast<float*>(s_am + a.N);        // [N]
  float* s_red_v = s_conf + a.N;                               // [kWarps]
  int* s_red_i = reinterpret_cast<int*>(s_red_v + kWarps);     // [kWarps]
  int* s_keep = s_red_i + kWarps;                              // [kMaxKeep]
  int& s_nfull = s_keep[kMaxKeep];
  int& s_prev = s_keep[kMaxKeep + 1];
  int& s_stop = s_keep[kMaxKeep + 2];
  int2 (*s_step)[kCapA] = reinterpret_cast<int2 (*)[kCapA]>(
      ((uintptr_t)(s_keep + kMaxKeep + 3) + 7) & ~(uintptr_t)7);                  // [N][kCapA]
  const int tid = threadIdx.x;
  // slots to draft: all, or (adaptive block length) those before the precomputed cut
  const int cut = a.nd_in ? min(max(a.nd_in[b], 0), a.N) : a.N;

  // ---- counts, the previous rows and argmax rows of every slot, and the confidences,
  //      in one round of copies (entries past a slot's count, or of a slot without a
  //      table, are copied but never read)
  for (int i = tid; i < cut; i += kThreads) {
    cp_async4(&s_nc[i], a.cand_n + (size_t)i * a.B + b);
    cp_async4(&s_na[i], a.prev_n + (size_t)i * a.B + b);
  }
  if (a.conf && !a.nd_in)
    for (int i = tid; i < a.N; i += kThreads) cp_async4(&s_conf[i], a.conf + (size_t)b * a.N + i);
  for (int e = tid; e < cut * kCapA; e += kThreads) {
    const int i = e / kCapA, p = e % kCapA;
    const size_t o = ((size_t)i * a.B + b) * kCapA + p;
    cp_async4(&s_av[i][p], a.prev_v + o);
    cp_async4(&s_am[i][p], a.amax + o);
  }
  cp_async_wait_all();
  __syncthreads();
  auto tabulated = [&](int i) {
    return s_nc[i] >= 1 && s_nc[i] <= kTabC && s_na[i] >= 1 && s_na[i] <= kCapA;
  };

  // ---- the steps of the walk, all at once: for a tabulated slot i and a possible
  //      previous row p of it (index into A(i - 1)), step[i][p] = {the row the table
  //      chose for p, the index in A(i) of that row (its first listing there)}; the row
  //      is -1 where the walk stops at slot i (it is not valid), the index -1 where it
  //      stops after slot i (slot i + 1 has no table or does not list the row)
  for (int e = tid; e < cut * kCapA; e += kThreads) {
    const int i = e / kCapA, p = e % kCapA;
    int2 st = make_int2(-1, -1);
    if (tabulated(i) && p < s_na[i]) {
      const int row = s_am[i][p];
      if (row >= 0 && row < a.Vh) {
        st.x = row;
        if (i + 1 < cut && tabulated(i + 1))
          for (int q = 0; q < s_na[i + 1]; ++q)
            if (s_av[i + 1][q] == row) {
              st.y = q;
              break;
            }
      }
    }
    s_step[i][p] = st;
  }
  __syncthreads();
  // ---- thread 0 follows the steps through the tabulated slots as far as they go (slot
  //      0's only previous row is the anchor): one shared-memory load per slot
  if (tid == 0) {
    int prev = -1, step = 0, pi = 0;
    for (; step < cut && pi >= 0; ++step) {
      const int2 st = s_step[step][pi];
      if (st.x < 0) break;
      s_pi[step] = pi;
      s_row[step] = st.x;                            // drafted after the walk
      prev = st.x;
      pi = st.y;
    }
    s_stop = step;
    s_prev = prev;
  }
  __syncthreads();
  for (int step = s_stop; step < cut; ++step) {
    // -------- a tabulated slot whose previous row is listed: a lookup
    if (tid == 0) {
      int pi = -1;
      if (tabulated(step)) {
        if (step == 0) {
          pi = 0;
        } else {
          for (int p = 0; p < s_na[step]; ++p)
            if (s_av[step][p] == s_prev) {
              pi = p;
              break;
            }
        }
        if (pi >= 0) {
          const int row = s_am[step][pi];
          if (row >= 0 && row < a.Vh) {
            s_prev = row;
            s_row[step] = row;
          } else {
            pi = -1;
          }
        }
      }
      s_pi[step] = pi;
    }
    __syncthreads();
    if (s_pi[step] >= 0) continue;
    // -------- on the fly: u of the previous token, z' of the list (or of every row)
    if (tid == 0) atomicAdd(a.err + kCtrlOnTheFly, 1u);
    {
      int p;
      if (step == 0) {
        p = a.anchors[b];
      } else {
        const int pv = s_prev;
        p = (pv >= 0 && pv < a.Vh) ? (a.d2t ? a.d2t[pv] : pv) : -1;
      }
      if (p < 0 || p >= a.V) {
        if (tid == 0) flag_error(a.err, kErrBadToken);
        p = 0;
      }
      for (int q = tid; q < a.r; q += kThreads)
        s_u[q] = __bfloat162float(a.w1[(size_t)p * a.r + q]);
    }
    const int n = s_nc[step];
    const size_t ib = (size_t)step * a.B + b;
    int nsel;
    __syncthreads();
    if (n >= 1 && n <= kCap) {
      for (int j = tid; j < n; j += kThreads) {
        buf[j].v = a.cand_v[ib * kCap + j];
        buf[j].z = a.cand_z[ib * kCap + j];
        buf[j].x = NAN;
      }
      __syncthreads();
      evaluate_list(buf, n, s_u, a.w2t, a.r);
      __syncthreads();
      nsel = n;
    } else {
      // the list overflowed: every row, streamed through the buffer
      if (tid == 0) {
        s_nfull = 0;
        atomicAdd(a.err + kCtrlEveryRow, 1u);
      }
      __syncthreads();
      for (int v0 = 0; v0 < a.Vh; v0 += kCand - kMaxKeep) {
        const int cnt = min(kCand - kMaxKeep, a.Vh - v0);
        const int base = s_nfull;
        __syncthreads();
        for (int j = tid; j < cnt; j += kThreads) {
          const int v = v0 + j;
          // rows of a tile the GEMM left out cannot reach this slot's top k
          const bool in = !a.zw || a.zw[((size_t)step * a.B + b) * a.T + v / kTile];
          buf[base + j].v = v;
          buf[base + j].z = in ? a.z[z_octet_index(step, v, b, a.Vhp, a.ldb)] : -INFINITY;
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
    // -------- selection over the evaluated entries: argmax, then the top-k
    float av;
    int ai;
    block_pick(buf, nsel, false, true, 0.f, 0, av, ai, s_red_v, s_red_i);
    if (ai < 0 || ai >= a.Vh) ai = 0;                  // only if every value was NaN
    if (tid == 0) {
      s_row[step] = ai;
      s_prev = ai;
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
          const int row = (bi >= 0 && bi < a.Vh) ? bi : 0;
          if (a.topk_ids) a.topk_ids[o] = a.d2t ? a.d2t[row] : row;
          if (a.topk_vals) a.topk_vals[o] = bv;
        }
        pv = bv;
        pid = bi;
      }
    }
    __syncthreads();
  }

  // ---- the draft (every slot's chosen head row as a token) and the top-k of the
  //      looked-up slots (the entries stored for the chosen previous row): all loads
  //      first, then the stores
  for (int e = tid; e < a.N * a.k; e += kThreads) {
    int tok = -1;                                    // past the cut: not drafted
    if (e < a.N && e < cut) {
      const int row = s_row[e];
      tok = a.d2t ? a.d2t[row] : row;
    }
    const int i = e / a.k, q = e % a.k;
    bool put = false;
    int id = -1;
    float val = NAN;
    if (a.want_topk) {
      if (i >= cut) {
        put = true;                                  // past the cut: not drafted
      } else if (s_pi[i] >= 0) {                     // (else written by the on-the-fly step)
        const size_t src = (((size_t)i * a.B + b) * kCapA + s_pi[i]) * a.k + q;
        if (a.topk_ids) id = a.tk_id[src];
        if (a.topk_vals) val = a.tk_val[src];
        put = true;
      }
    }
    if (e < a.N) a.draft[(size_t)b * a.N + e] = tok;
    if (put) {
      const size_t dst = ((size_t)b * a.N + i) * a.k + q;
      if (a.topk_ids) a.topk_ids[dst] = id;
      if (a.topk_vals) a.topk_vals[dst] = val;
    }
  }
  // ---- truncation at the first slot whose confidence is below conf_min (llama.cpp
  //      commit 6fed9f6, "spec: add confidence-based draft pruning for DSpark")
  //      (already computed, before the GEMM, with the adaptive block length)
  if (tid == 0 && !a.nd_in) {
    int nd = a.N;
    if (a.conf && a.conf_min > 0.f)
      for (int i = 0; i < a.N; ++i)
        if (s_conf[i] < a.conf_min) {
          nd = i;
          break;
        }
    a.n_draft[b] = nd;
  }
}

// One CTA per (block, slot i): candidate rows C(i) (bound of rank kk), the rows A(i - 1)
// that can be the argmax of slot i - 1 (bound of rank 1; slot 0: the anchor), z' exactly
// for every pair in A(i - 1) x C(i), and from it, for each possible previous row, the
// argmax and the top-k of slot i.  Also the slot's confidence.
// Four CTAs per SM (at most 64 registers a thread), so that the B x N CTAs of the
// Qwen3-8B-shaped batch (512) run in one wave on 152 SMs.
__device__ __forceinline__ void table_work(const TableArgs& a, uint8_t* dsm, int b, int i) {
  const int T4 = (a.T + 3) & ~3;
  float* s_ub = (float*)dsm;                                   // [T4] upper bounds, slot i
  float* s_up = s_ub + T4;                                     // [T4] upper bounds, slot i-1
  int* s_tc = (int*)(s_up + T4);                               // [T4] tiles of C(i)
  int* s_ta = s_tc + T4;                                       // [T4] tiles of A(i-1)
  int32_t* s_cv = (int32_t*)(s_ta + T4);                       // [kCap]
  float* s_cz = (float*)(s_cv + kCap);                         // [kCap]
  float* s_x = s_cz + kCap;                                    // [kCapA][kTabC]
  __nv_bfloat16* s_w1 = (__nv_bfloat16*)(s_x + kCapA * kTabC); // [kCapA][r]
  __nv_bfloat16* s_w2 = s_w1 + (size_t)kCapA * a.r;            // [kRowsChunk][r]
  __shared__ float s_top[kWarps * 32];
  __shared__ float s_theta, s_red[kWarps], s_cpart[kWarps];
  __shared__ int s_ntc, s_nta, s_nc, s_na;
  __shared__ int32_t s_av[kCapA];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const float umax = __uint_as_float(*a.w1max) * (1.f + kRelMargin);
  const float* zm = a.zmax + ((size_t)i * a.B + b) * a.T;
  const float* zp = i > 0 ? a.zmax + ((size_t)(i - 1) * a.B + b) * a.T : nullptr;
  // Tiles the GEMM left out of z had an upper bound below a lower bound of their slot's
  // threshold, so they hold no candidate: their upper bounds are set to -inf here.
  const uint8_t* wi = a.zw ? a.zw + ((size_t)i * a.B + b) * a.T : nullptr;
  const uint8_t* wp = (a.zw && zp) ? a.zw + ((size_t)(i - 1) * a.B + b) * a.T : nullptr;

  if (tid == 0) {
    s_ntc = 0;
    s_nta = 0;
    s_nc = 0;
    s_na = 0;
  }
  // ---- bounds of slot i and slot i - 1, and the confidence, all warps sharing both;
  //      each thread keeps the maxima of the lower bounds / tile maxima it saw
  float mp = -INFINITY;                              // slot i-1's lower bounds
  float mlb = -INFINITY, mzm = -INFINITY;            // slot i's lower bounds, tile maxima
  {
    // loads of up to kBoundsUnroll tiles per thread are issued before any is used
    constexpr int kBoundsUnroll = 8;
    const int stride = kThreads;
    for (int t0 = tid; t0 < a.T; t0 += kBoundsUnroll * stride) {
      float c[kBoundsUnroll], z0[kBoundsUnroll], z1[kBoundsUnroll];
      unsigned w0 = 0, w1 = 0;                       // bit u: tile t0 + u * stride stored
#pragma unroll
      for (int u = 0; u < kBoundsUnroll; ++u) {
        const int t = t0 + u * stride;
        const bool in = t < a.T;
        c[u] = in ? a.cnmax[t] : 0.f;
        z0[u] = in ? zm[t] : -INFINITY;
        z1[u] = (in && zp) ? zp[t] : -INFINITY;
        w0 |= (unsigned)(!(in && wi) || wi[t] != 0) << u;
        w1 |= (unsigned)(!(in && wp) || wp[t] != 0) << u;
      }
#pragma unroll
      for (int u = 0; u < kBoundsUnroll; ++u) {
        const int t = t0 + u * stride;
        if (t >= a.T) break;
        const float d = umax * c[u] * (1.f + kRelMargin) + kAbsMargin;
        mlb = fmaxf(mlb, z0[u] - d);
        mzm = fmaxf(mzm, z0[u]);
        s_ub[t] = (w0 >> u) & 1 ? z0[u] + d : -INFINITY;
        if (zp) {
          s_up[t] = (w1 >> u) & 1 ? z1[u] + d : -INFINITY;
          mp = fmaxf(mp, z1[u] - d);
        }
      }
    }
  }
  if (a.w_conf) {
    // sigmoid(h . w_conf + b_conf) (llama.cpp commit 6fed9f6, "spec: add confidence-based
    // draft pruning for DSpark"): each thread a few 16-byte chunks of the dot product,
    // summed over the warp here and over the warps after the barrier
    const __nv_bfloat16* h = a.hidden + ((size_t)b * a.L_in + a.ifp + i) * a.H;
    float acc = 0.f;
    if ((a.H % 8) == 0 && ((uintptr_t)h % 16) == 0 && ((uintptr_t)a.w_conf % 16) == 0) {
      const uint4* h4 = reinterpret_cast<const uint4*>(h);
      const uint4* w4 = reinterpret_cast<const uint4*>(a.w_conf);
      const int n4 = a.H / 8;
#pragma unroll 2
      for (int q = tid; q < n4; q += kThreads) {
        const uint4 hv = h4[q], wv = w4[q];
        const __nv_bfloat16* he = reinterpret_cast<const __nv_bfloat16*>(&hv);
        const __nv_bfloat16* we = reinterpret_cast<const __nv_bfloat16*>(&wv);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(to_f32(he[e]), to_f32(we[e]), acc);
      }
    } else {
      for (int c = tid; c < a.H; c += kThreads) acc = fmaf(to_f32(h[c]), to_f32(a.w_conf[c]), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) s_cpart[warp] = acc;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mp = fmaxf(mp, __shfl_xor_sync(0xFFFFFFFFu, mp, o));
  if (lane == 0) s_red[warp] = mp;
  __syncthreads();
  if (a.w_conf && tid == 0) {
    float acc = 0.f;
    for (int w = 0; w < kWarps; ++w) acc += s_cpart[w];
    a.conf[(size_t)b * a.N + i] = 1.f / (1.f + expf(-(acc + a.b_conf)));
  }
  // ---- thresholds: rank kk of slot i's lower bounds (rank 1 when the top-k ranks base
  //      logits, which then take rank kk of the tile maxima); rank 1 of slot i-1's
  const float theta_x = block_kth_of_maxima(mlb, a.zrank ? 1 : a.kk, s_top, &s_theta);
  float theta_z = INFINITY;
  if (a.zrank) theta_z = block_kth_of_maxima(mzm, a.kk, s_top, &s_theta) - kAbsMargin;
  float theta1 = s_red[0];
  for (int w = 1; w < kWarps; ++w) theta1 = fmaxf(theta1, s_red[w]);
  // ---- candidate tiles of both lists
  for (int t = tid; t < a.T; t += kThreads) {
    if (s_ub[t] >= theta_x || (a.zrank && zm[t] >= theta_z)) s_tc[atomicAdd(&s_ntc, 1)] = t;
    if (zp && s_up[t] >= theta1) s_ta[atomicAdd(&s_nta, 1)] = t;
  }
  __syncthreads();
  // ---- their rows
  {
    const RowScan lc{(size_t)i, s_tc, s_ntc, theta_x, theta_z, s_cv, s_cz, kCap, &s_nc};
    const RowScan lp{zp ? (size_t)(i - 1) : 0, s_ta, zp ? s_nta : 0, theta1, INFINITY,
                     s_av, nullptr, kCapA, &s_na};
    scan_rows(a.z, b, a.Vhp, a.ldb, a.cnorm, umax, a.Vh, lc, lp);
  }
  if (!zp && tid == 0) {
    int p = a.anchors[b];
    if (p < 0 || p >= a.V) {
      flag_error(a.err, kErrBadToken);
      p = 0;
    }
    s_av[0] = p;                                     // slot 0: the anchor (a token)
    s_na = 1;
  }
  __syncthreads();
  // ---- the lists
  const int nc = s_nc, na = s_na;
  const size_t ib = (size_t)i * a.B + b;
  for (int j = tid; j < min(nc, kCap); j += kThreads) {
    a.cand_v[ib * kCap + j] = s_cv[j];
    a.cand_z[ib * kCap + j] = s_cz[j];
  }
  for (int j = tid; j < min(na, kCapA); j += kThreads) a.prev_v[ib * kCapA + j] = s_av[j];
  if (tid == 0) {
    a.cand_n[ib] = nc;
    a.prev_n[ib] = na;
  }
  // (a slot without a table is evaluated on the fly by the walk)
  if (nc >= 1 && nc <= kTabC && na >= 1 && na <= kCapA) {
    // ---- z' = z + markov_w1[p] . w2[:, v] for every p in A(i - 1), v in C(i): eight lanes
    //      per pair, the same summation order as the on-the-fly evaluation
    const int chunks = a.r / 8;                        // r % 8 == 0 on this path
    for (int c = tid; c < na * chunks; c += kThreads) {
      const int p = c / chunks, q = c % chunks;
      int tok = (i == 0 || !a.d2t) ? s_av[p] : a.d2t[s_av[p]];
      if (tok < 0 || tok >= a.V) {
        flag_error(a.err, kErrBadToken);
        tok = 0;
      }
      cp_async16(s_w1 + (size_t)p * a.r + q * 8, a.w1 + (size_t)tok * a.r + q * 8);
    }
    for (int c0 = 0; c0 < nc; c0 += kRowsChunk) {
      const int cnt = min(kRowsChunk, nc - c0);
      for (int c = tid; c < cnt * chunks; c += kThreads) {
        const int e = c / chunks, q = c % chunks;
        cp_async16(s_w2 + (size_t)e * a.r + q * 8, a.w2t + (size_t)s_cv[c0 + e] * a.r + q * 8);
      }
      cp_async_wait_all();
      __syncthreads();
      const int pairs = na * cnt, sub = tid % 8;
      for (int q0 = 0; q0 < pairs; q0 += kThreads / 8) {
        const int pr = q0 + tid / 8;
        float s0 = 0.f, s1 = 0.f;
        if (pr < pairs) {
          const __nv_bfloat16* u = s_w1 + (size_t)(pr / cnt) * a.r;
          const __nv_bfloat16* w = s_w2 + (size_t)(pr % cnt) * a.r;
          for (int ch = sub; ch < chunks; ch += 8) {
            const uint4 ru = *reinterpret_cast<const uint4*>(u + ch * 8);
            const uint4 rw = *reinterpret_cast<const uint4*>(w + ch * 8);
            const __nv_bfloat162* pu = reinterpret_cast<const __nv_bfloat162*>(&ru);
            const __nv_bfloat162* pw = reinterpret_cast<const __nv_bfloat162*>(&rw);
  #pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float2 fu = __bfloat1622float2(pu[h]), fw = __bfloat1622float2(pw[h]);
              s0 = fmaf(fu.x, fw.x, s0);
              s1 = fmaf(fu.y, fw.y, s1);
            }
          }
        }
        float s = s0 + s1;
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 4);
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 2);
        s += __shfl_xor_sync(0xFFFFFFFFu, s, 1);
        if (pr < pairs && sub == 0) {
          const int e = pr % cnt;
          s_x[(pr / cnt) * kTabC + c0 + e] = s_cz[c0 + e] + s;
        }
      }
      __syncthreads();
    }
    // ---- for each possible previous row: the argmax (the next previous row) and the top-k
    for (int p = warp; p < na; p += kWarps) {
      const float* x = s_x + p * kTabC;
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
      for (int c = lane; c < nc; c += 32)
        if (better(x[c], s_cv[c], bv, bi)) {
          bv = x[c];
          bi = s_cv[c];
        }
      warp_best(bv, bi);
      if (lane == 0) a.amax[ib * kCapA + p] = (bi >= 0 && bi < a.Vh) ? bi : -1;
      if (!a.want_topk) continue;
      const float* rk = a.zrank ? s_cz : x;
      if (a.k == 1 && !a.zrank) {
        // the top 1 of the corrected logits is the argmax just found (same order)
        if (lane == 0) {
          const size_t o = ib * kCapA + p;
          const int row = (bi >= 0 && bi < a.Vh) ? bi : 0;
          a.tk_id[o] = a.d2t ? a.d2t[row] : row;
          a.tk_val[o] = bv;
        }
        continue;
      }
      if (nc <= 32 && a.k > 1) {
        // one entry per lane: sort the warp, lane q holds the q-th
        float v = lane < nc ? rk[lane] : -INFINITY;
        int id = lane < nc ? s_cv[lane] : 0x7FFFFFFF;
        warp_sort(v, id);
        if (lane < a.k) {
          const size_t o = (ib * kCapA + p) * a.k + lane;
          const int row = (id >= 0 && id < a.Vh) ? id : 0;
          a.tk_id[o] = a.d2t ? a.d2t[row] : row;
          a.tk_val[o] = v;
        }
        continue;
      }
      float pv = 0.f;
      int pid = 0;
      for (int q = 0; q < a.k; ++q) {
        bv = -INFINITY;
        bi = 0x7FFFFFFF;
        for (int c = lane; c < nc; c += 32) {
          const float val = rk[c];
          const int id = s_cv[c];
          if (q > 0 && !better(pv, pid, val, id)) continue;
          if (better(val, id, bv, bi)) {
            bv = val;
            bi = id;
          }
        }
        warp_best(bv, bi);
        if (lane == 0) {
          const size_t o = (ib * kCapA + p) * a.k + q;
          const int row = (bi >= 0 && bi < a.Vh) ? bi : 0;
          a.tk_id[o] = a.d2t ? a.d2t[row] : row;
          a.tk_val[o] = bv;
        }
        pv = bv;
        pid = bi;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 4)
pruned_table(const TableArgs a, const SelectArgs sel) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const int b = blockIdx.x, i = blockIdx.y;
  const int tid = threadIdx.x;
  pdl_signal();
  pdl_wait();                                        // z and zmax of the lm_head GEMM
  // a prepared buffer made for other weights or sizes: nothing in it is read, nothing
  // is drafted, and the error word says why
  if (!prepared_matches(a.prep, a.prep_want)) {
    if (tid == 0 && b == 0 && i == 0) flag_error(a.err, kErrPrepared);
    return;
  }
  // with the adaptive block length, a slot from the block's cut on is not drafted
  if (!a.nd_in || i < a.nd_in[b]) table_work(a, dsm, b, i);
  // ---- the last of the block's N CTAs to get here walks the block (the others' lists
  //      and tables are in global memory by then)
  __shared__ int s_last;
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(a.walk_done + b, 1) == a.N - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  walk_block(sel, b, dsm);
}

}  // namespace

PreparedLayout plan_prepared(int Vh, int r) {
  PreparedLayout l{};
  l.Vhp = align_up((size_t)Vh, kTile);
  l.tiles = l.Vhp / kTile;
  size_t off = 0;
  l.header = off;
  off = align_up(off + sizeof(PreparedHeader), 256);
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

PrunedLists plan_pruned_lists(int B, int N, int k) {
  PrunedLists l{};
  const size_t nb = (size_t)N * B;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  l.cand_v = take(sizeof(int32_t) * nb * kCap);
  l.cand_z = take(sizeof(float) * nb * kCap);
  l.cand_n = take(sizeof(int32_t) * nb);
  l.prev_v = take(sizeof(int32_t) * nb * kCapA);
  l.prev_n = take(sizeof(int32_t) * nb);
  l.amax = take(sizeof(int32_t) * nb * kCapA);
  l.tk_id = take(sizeof(int32_t) * nb * kCapA * k);
  l.tk_val = take(sizeof(float) * nb * kCapA * k);
  l.total = off;
  return l;
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
  PreparedHeader h{};
  h.magic = kPreparedMagic;
  h.V = V;
  h.Vh = Vh;
  h.r = r;
  h.w1 = (unsigned long long)(uintptr_t)w1;
  h.w2 = (unsigned long long)(uintptr_t)w2;
  prepare_header<<<1, 1, 0, stream>>>((PreparedHeader*)(base + l.header), h);
  return cudaGetLastError();
}

cudaError_t launch_chain_pruned(const ProposePlan& p) {
  const int T = (int)(p.Vhp / kTile);
  const bool want_topk = p.topk_ids || p.topk_vals;
  const int kk = want_topk ? p.k : 1;
  const int zrank = (want_topk && !p.topk_markov) ? 1 : 0;
  if (!p.z_octet || p.N > kMaxSlots || p.r % 8 != 0 || !p.walk_done || !p.prep)
    return cudaErrorInvalidValue;
  TableArgs t{};
  t.z = p.z;
  t.zmax = p.zmax;
  t.zw = p.zwritten;
  t.Vhp = p.Vhp;
  t.ldb = p.ldb;
  t.cnorm = p.cnorm;
  t.cnmax = p.cnmax;
  t.w1max = p.w1max;
  t.w1 = (const __nv_bfloat16*)p.w1;
  t.w2t = p.w2t;
  t.anchors = p.anchors;
  t.d2t = p.d2t;
  t.hidden = (const __nv_bfloat16*)p.conf_hidden;
  // (with the adaptive block length the confidences are already computed)
  t.w_conf = p.skip_truncated ? nullptr : (const __nv_bfloat16*)p.w_conf;
  t.b_conf = p.b_conf;
  t.conf = p.conf ? p.conf : p.conf_ws;
  t.cand_v = p.cand_v;
  t.cand_z = p.cand_z;
  t.cand_n = p.cand_n;
  t.prev_v = p.prev_v;
  t.prev_n = p.prev_n;
  t.amax = p.amax;
  t.tk_id = p.tk_id;
  t.tk_val = p.tk_val;
  t.err = p.ctrl;
  t.walk_done = p.walk_done;
  t.nd_in = p.skip_truncated ? p.n_draft : nullptr;
  t.prep = p.prep;
  t.prep_want = p.prep_want;
  t.B = p.B;
  t.N = p.N;
  t.V = p.V;
  t.Vh = p.Vh;
  t.T = T;
  t.r = p.r;
  t.k = p.k;
  t.kk = kk;
  t.zrank = zrank;
  t.want_topk = want_topk ? 1 : 0;
  t.L_in = p.L_in;
  t.ifp = p.ifp;
  t.H = p.H;
  SelectArgs s{};
  s.z = p.z;
  s.zw = p.zwritten;
  s.T = T;
  s.Vhp = p.Vhp;
  s.ldb = p.ldb;
  s.w1 = (const __nv_bfloat16*)p.w1;
  s.w2t = p.w2t;
  s.cand_v = p.cand_v;
  s.cand_z = p.cand_z;
  s.cand_n = p.cand_n;
  s.prev_v = p.prev_v;
  s.prev_n = p.prev_n;
  s.amax = p.amax;
  s.tk_id = p.tk_id;
  s.tk_val = p.tk_val;
  s.anchors = p.anchors;
  s.d2t = p.d2t;
  s.conf = p.w_conf ? (p.conf ? p.conf : p.conf_ws) : nullptr;
  s.conf_min = p.conf_min;
  s.n_draft = p.n_draft;
  s.draft = p.draft;
  s.topk_ids = p.topk_ids;
  s.topk_vals = p.topk_vals;
  s.err = p.ctrl;
  s.B = p.B;
  s.N = p.N;
  s.V = p.V;
  s.Vh = p.Vh;
  s.r = p.r;
  s.k = p.k;
  s.kk = kk;
  s.zrank = zrank;
  s.want_topk = want_topk ? 1 : 0;
  s.nd_in = p.skip_truncated ? p.n_draft : nullptr;
  // the tables' shared memory, or the walk's when it needs more
  const size_t T4 = (size_t)((T + 3) & ~3);
  const size_t table_smem = sizeof(float) * 4 * T4 + (sizeof(int32_t) + sizeof(float)) * kCap +
                            sizeof(float) * kCapA * kTabC +
                            sizeof(__nv_bfloat16) * (size_t)(kCapA + kRowsChunk) * p.r;
  const size_t smem = std::max(table_smem, walk_smem_bytes(p.r, p.N));
  const cudaError_t e = raise_smem_limit(reinterpret_cast<const void*>(pruned_table), smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(pruned_table, dim3(p.B, p.N), dim3(kThreads), smem, p.stream, t, s);
}

}  // namespace dspark
