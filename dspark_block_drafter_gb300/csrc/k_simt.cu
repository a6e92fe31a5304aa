// CUDA-core (FMA) kernels of the proposal for the fp32 operand type: the base logits,
// and the Markov-corrected greedy chain over all slots in one cooperative launch.  Every
// sum is accumulated in fp32.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kTileM = 64, kTileV = 64, kTileK = 16;
constexpr int kGemmStages = 4;          // K-tiles in flight (cp.async ring)

__device__ __forceinline__ void cp_async4_zfill(float* dst, const float* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// z[i][v][b] = sum_h hidden[b, ifp + i, h] * lm_head[v, h] + lm_bias[v]
// (llama.cpp commit 6fed9f6, the proposal formula's logits(i)); prediction row
// m = i * B + b.  64 x 64 output tiles; the K-tiles stream through a ring of
// kGemmStages shared-memory stages filled by cp.async, so several are in flight at once
// (small problems are bound by the latency of these loads, not by their bytes).
__global__ void __launch_bounds__(256)
base_logits_simt(const float* __restrict__ hidden, const float* __restrict__ W,
                 const float* __restrict__ bias, float* __restrict__ z, int B, int L_in,
                 int N, int ifp, int H, int Vh, size_t Vhp, size_t ldb) {
  __shared__ float As[kGemmStages][kTileK][kTileM + 4];
  __shared__ float Ws[kGemmStages][kTileK][kTileV + 4];
  const int M = B * N;
  const int m0 = blockIdx.y * kTileM, v0 = blockIdx.x * kTileV;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int nk = (H + kTileK - 1) / kTileK;
  auto issue = [&](int kt) {
    if (kt < nk) {
      const int k0 = kt * kTileK, st = kt % kGemmStages;
      for (int e = threadIdx.x; e < kTileM * kTileK; e += 256) {
        const int mm = e / kTileK, kk = e % kTileK;
        const int m = m0 + mm, k = k0 + kk, v = v0 + mm;
        const bool va = m < M && k < H, vw = v < Vh && k < H;
        const int i = va ? m / B : 0, b = va ? m % B : 0;
        cp_async4_zfill(&As[st][kk][mm],
                        va ? &hidden[((size_t)b * L_in + ifp + i) * H + k] : hidden, va);
        cp_async4_zfill(&Ws[st][kk][mm], vw ? &W[(size_t)v * H + k] : W, vw);
      }
    }
    cp_async_commit();                                // (an empty group past the end)
  };
  float acc[4][4] = {};
#pragma unroll
  for (int s = 0; s < kGemmStages - 1; ++s) issue(s);
  for (int kt = 0; kt < nk; ++kt) {
    issue(kt + kGemmStages - 1);
    cp_async_wait<kGemmStages - 1>();                  // K-tile kt has landed
    __syncthreads();
    const int st = kt % kGemmStages;
#pragma unroll
    for (int kk = 0; kk < kTileK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q] = As[st][kk][ty * 4 + q];
        w[q] = Ws[st][kk][tx * 4 + q];
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(a[p], w[q], acc[p][q]);
    }
    __syncthreads();                                  // before the stage is refilled
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

// The Markov-corrected greedy chain over all slots in one cooperative launch (the
// proposal formula's logits'(i) = logits(i) + markov_w2^T markov_w1[prev(i)], prev(i) the
// argmax of slot i - 1).  CTA c owns the contiguous head rows [v0, v1); per slot and
// block it evaluates its rows (thread = row), posts its best (value, row) with a 64-bit
// atomicMax, and lists its k best ranked rows; a grid barrier then makes the slot's
// winners the next slot's previous tokens.  After the last slot the CTAs' warps merge
// the lists into each (slot, block)'s top k.
// Sums in fp32 in the order k = 0 .. r - 1, as the oracle's dot product lists them.
constexpr int kSimtThreads = 256;
constexpr int kSkinnyRows = kSimtFusedRows;   // prediction rows of the few-row GEMM forms
constexpr long long kSimtWaitBudget = 2000000000ll;   // ~1 s of SM clocks

struct SimtArgs {
  const float* z;               // base logits [N][Vhp][ldb]
  const float* w1;              // [V][r]
  const float* w2;              // [r][Vh]
  const int32_t* anchors;
  const int32_t* d2t;
  int32_t* draft;               // [B][N]
  int32_t* topk_ids;            // [B][N][k] written from the winners (k = 1 over
  float* topk_vals;             //   corrected logits), or NULL
  int32_t* topk_out_ids;        // [B][N][k] written by the merge of the lists, or NULL
  float* topk_out_vals;
  float* logits;                // [B][N][Vh] or NULL
  float* zc;                    // this slot's corrected logits [B][ldz]
  float* cand_val;              // [N][B][G][k] each CTA's k best ranked rows
  int32_t* cand_id;
  unsigned long long* keys;     // [N][B] winners
  unsigned* bar;
  uint32_t* err;
  size_t Vhp, ldb, ldz;
  int B, N, V, Vh, r, k, topk_markov, lists;
  int chunk;                    // blocks evaluated together (their markov_w1 rows in smem)
  // small problems: the base logits (each thread its own head row, the hidden rows
  // staged in shared memory) and the confidence head inside this kernel
  int fused;
  const float* hidden;          // [B][L_in][H]
  const float* lm_head;         // [Vh][H]
  const float* lm_bias;         // [Vh] or NULL
  const float* conf_hidden;     // [B][L_in][H]
  const float* w_conf;          // [H] or NULL
  float b_conf, conf_min;
  float* conf;                  // [B][N]
  int32_t* n_draft;             // [B]
  float* zk;                    // fused, with top-k: every slot's ranked values [N][B][ldz]
  int L_in, ifp, H;
};

__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

constexpr int kSimtMaxChunk = 8;                      // blocks evaluated together, at most
constexpr int kSimtRegRank = 32;                      // ranks whose column stays in registers
constexpr int kSimtWarps = kSimtThreads / 32;
constexpr int kSimtMaxK = 32;

// The best (value, row) over the CTA of each of the chunk's cb blocks, from every
// thread's candidates bv[j], bi[j]: warp reductions, then a pass over the warps' results
// in shared memory.  Every thread gets the results back in bv, bi.
template <int CH>
__device__ __forceinline__ void cta_best_chunk(float (&bv)[CH], int (&bi)[CH], int cb,
                                               float (*sv)[kSimtWarps], int (*si)[kSimtWarps]) {
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
#pragma unroll
  for (int j = 0; j < CH; ++j) {
    if (j >= cb) break;                               // (uniform)
    warp_best(bv[j], bi[j]);
    if (l == 0) {
      sv[j][w] = bv[j];
      si[j][w] = bi[j];
    }
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < CH; ++j) {
    if (j >= cb) break;
    float v = sv[j][0];
    int id = si[j][0];
#pragma unroll
    for (int q = 1; q < kSimtWarps; ++q)
      if (better(sv[j][q], si[j][q], v, id)) {
        v = sv[j][q];
        id = si[j][q];
      }
    bv[j] = v;
    bi[j] = id;
  }
  __syncthreads();                                    // (before sv, si are reused)
}

// The top k of (slot i, block b) from the G CTAs' lists: k rounds of a warp-wide best,
// each strictly after the previous pick.  Called by one whole warp.
__device__ void merge_lists(const SimtArgs& a, int i, int b, int G) {
  const int lane = threadIdx.x % 32;
  const size_t base = ((size_t)i * a.B + b) * G * a.k;
  const int n = G * a.k;
  // up to 8 entries per lane are read once and kept in registers; the rest are re-read
  constexpr int kKeep = 8;
  float cv[kKeep];
  int ci[kKeep];
#pragma unroll
  for (int t = 0; t < kKeep; ++t) {
    const int e = lane + 32 * t;
    cv[t] = e < n ? __ldcg(&a.cand_val[base + e]) : -INFINITY;
    ci[t] = e < n ? __ldcg(&a.cand_id[base + e]) : 0x7FFFFFFF;
  }
  float pv = 0.f;
  int pid = 0;
  for (int q = 0; q < a.k; ++q) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int t = 0; t < kKeep; ++t) {
      const float x = cv[t];
      const int id = ci[t];
      if (id != 0x7FFFFFFF && (q == 0 || better(pv, pid, x, id)) && better(x, id, bv, bi)) {
        bv = x;
        bi = id;
      }
    }
    for (int e = lane + 32 * kKeep; e < n; e += 32) {
      const float x = __ldcg(&a.cand_val[base + e]);
      const int id = __ldcg(&a.cand_id[base + e]);
      if (id == 0x7FFFFFFF) continue;                 // a CTA with fewer than k rows
      if ((q == 0 || better(pv, pid, x, id)) && better(x, id, bv, bi)) {
        bv = x;
        bi = id;
      }
    }
    warp_best(bv, bi);
    if (lane == 0) {
      const size_t o = ((size_t)b * a.N + i) * a.k + q;
      const int row = bi == 0x7FFFFFFF ? 0 : bi;
      if (a.topk_out_ids) a.topk_out_ids[o] = a.d2t ? a.d2t[row] : row;
      if (a.topk_out_vals) a.topk_out_vals[o] = bv;
    }
    pv = bv;
    pid = bi;
  }
}

// CH: blocks evaluated together (a.chunk <= CH of them per chunk); WR: the rank is at
// most kSimtRegRank, and each thread keeps its first row's markov_w2 column in registers
// (the same every slot).  The code of one instantiation is sized to what it runs: a
// kernel this latency-bound stalls on instruction fetch when it is larger.
template <int CH, bool WR>
__global__ void __launch_bounds__(kSimtThreads)
chain_simt(const SimtArgs a) {
  extern __shared__ float s_u[];                      // [chunk][r]: markov_w1 of the prev;
                                                      // fused: then [M][H] hidden rows and
                                                      // [M][threads] base logits
  __shared__ float sv[CH][kSimtWarps];
  __shared__ int si[CH][kSimtWarps];
  __shared__ float s_lv[CH][kSimtWarps][kSimtMaxK];   // each warp's k best of each block
  __shared__ int s_li[CH][kSimtWarps][kSimtMaxK];
  __shared__ float s_rk[CH][kSimtThreads];            // each thread's first row's ranked value
  __shared__ int s_prev[CH];
  __shared__ int s_abort;
  const int G = gridDim.x, c = blockIdx.x, tid = threadIdx.x;
  const int warp = tid / 32, lane = tid % 32;
  const int v0 = (int)((long long)c * a.Vh / G), v1 = (int)((long long)(c + 1) * a.Vh / G);
  // this thread's first row: its values stay in registers (the rest are re-read)
  const int vr = v0 + tid;
  float wreg[WR ? kSimtRegRank : 1];
  if (WR) {
#pragma unroll
    for (int q = 0; q < (WR ? kSimtRegRank : 1); ++q)
      wreg[q] = (vr < v1 && q < a.r) ? a.w2[(size_t)q * a.Vh + vr] : 0.f;
  }
  if (tid == 0) s_abort = 0;
  const int M = a.B * a.N;
  float* s_h = s_u + (((size_t)a.chunk * a.r + 3) & ~(size_t)3);   // (16-byte aligned)
  float* s_zf = s_h + (size_t)M * a.H;
  if (a.fused) {
    // this CTA's lm_head rows into L2 first (they are read below, a few rows at a time)
    {
      const char* slab = reinterpret_cast<const char*>(a.lm_head + (size_t)v0 * a.H);
      const size_t bytes = sizeof(float) * (size_t)(v1 - v0) * a.H;
      for (size_t o = (size_t)tid * 128; o < bytes; o += (size_t)kSimtThreads * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(slab + o));
    }
    // the base logits of this thread's row for every prediction row m = i * B + b
    // (the proposal formula's logits(i)): hidden rows staged in shared memory, the
    // lm_head row streamed in 16-byte chunks
    for (int e = tid; e < M * a.H; e += kSimtThreads) {
      const int m = e / a.H, kk = e % a.H;
      s_h[e] = a.hidden[((size_t)(m % a.B) * a.L_in + a.ifp + m / a.B) * a.H + kk];
    }
    __syncthreads();
    // warp w takes an eighth of the CTA's rows, kRowsAtOnce at a time: the lanes read
    // those lm_head rows in 16-byte chunks (coalesced, all requested before any is used),
    // each keeps a partial sum per (row, prediction row), and a butterfly over the lane
    // bits 4..1 leaves lanes 2m and 2m + 1 with prediction row m's sum (lane bit 0 adds
    // the last pair)
    {
      constexpr int kRowsAtOnce = 4;
      const bool vec = (a.H % 4) == 0 && ((uintptr_t)a.lm_head % 16) == 0;
      const int per_w = (v1 - v0 + kSimtWarps - 1) / kSimtWarps;
      const int wbeg = v0 + warp * per_w, wend = min(v1, wbeg + per_w);
      for (int g = wbeg; g < wend; g += kRowsAtOnce) {
        float part[kRowsAtOnce][kSkinnyRows];
#pragma unroll
        for (int rr = 0; rr < kRowsAtOnce; ++rr)
#pragma unroll
          for (int m = 0; m < kSkinnyRows; ++m) part[rr][m] = 0.f;
        if (vec) {
          for (int k0 = 0; k0 < a.H; k0 += 256) {           // two chunks per lane and row
            float4 w4[kRowsAtOnce][2];
#pragma unroll
            for (int rr = 0; rr < kRowsAtOnce; ++rr)
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const int kk = k0 + 128 * t + 4 * lane;
                w4[rr][t] = (g + rr < wend && kk < a.H)
                                ? *reinterpret_cast<const float4*>(a.lm_head + (size_t)(g + rr) * a.H + kk)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int kk = k0 + 128 * t + 4 * lane;
              if (kk >= a.H) break;
#pragma unroll
              for (int m = 0; m < kSkinnyRows; ++m) {
                if (m >= M) break;
                const float4 h = *reinterpret_cast<const float4*>(s_h + (size_t)m * a.H + kk);
#pragma unroll
                for (int rr = 0; rr < kRowsAtOnce; ++rr)
                  part[rr][m] = fmaf(h.w, w4[rr][t].w, fmaf(h.z, w4[rr][t].z,
                                     fmaf(h.y, w4[rr][t].y, fmaf(h.x, w4[rr][t].x, part[rr][m]))));
              }
            }
          }
        } else {
          for (int kk = lane; kk < a.H; kk += 32) {
            float w[kRowsAtOnce];
#pragma unroll
            for (int rr = 0; rr < kRowsAtOnce; ++rr)
              w[rr] = g + rr < wend ? a.lm_head[(size_t)(g + rr) * a.H + kk] : 0.f;
#pragma unroll
            for (int m = 0; m < kSkinnyRows; ++m) {
              if (m >= M) break;
              const float h = s_h[(size_t)m * a.H + kk];
#pragma unroll
              for (int rr = 0; rr < kRowsAtOnce; ++rr) part[rr][m] = fmaf(h, w[rr], part[rr][m]);
            }
          }
        }
#pragma unroll
        for (int rr = 0; rr < kRowsAtOnce; ++rr) {
          // butterfly: at bit o the lane keeps the half of its sums selected by that bit
#pragma unroll
          for (int o = kSkinnyRows; o > 1; o >>= 1) {
            const int half = o / 2;
            const bool upper = (lane & half * 2) != 0;    // lane bits 4, 3, 2, 1
#pragma unroll
            for (int q = 0; q < half; ++q) {
              const float send = upper ? part[rr][q] : part[rr][q + half];
              const float keep = upper ? part[rr][q + half] : part[rr][q];
              part[rr][q] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, half * 2);
            }
          }
          part[rr][0] += __shfl_xor_sync(0xFFFFFFFFu, part[rr][0], 1);
          const int m = lane >> 1, v = g + rr;
          if ((lane & 1) == 0 && m < M && v < wend)
            s_zf[(size_t)m * kSimtThreads + (v - v0)] =
                part[rr][0] + (a.lm_bias ? a.lm_bias[v] : 0.f);
        }
      }
    }
    __syncthreads();
    // the confidence head: one (block, slot) dot product per warp of the grid
    if (a.w_conf) {
      for (int e = c * kSimtWarps + warp; e < M; e += G * kSimtWarps) {
        const int i = e / a.B, b = e % a.B;
        const float* h = a.conf_hidden + ((size_t)b * a.L_in + a.ifp + i) * a.H;
        float acc = 0.f;
        for (int kk = lane; kk < a.H; kk += 32) acc = fmaf(h[kk], a.w_conf[kk], acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
        if (lane == 0) a.conf[(size_t)b * a.N + i] = 1.f / (1.f + expf(-(acc + a.b_conf)));
      }
    }
  }
  for (int i = 0; i < a.N; ++i) {
    const float* z_i = a.z + (size_t)i * a.Vhp * a.ldb;
    for (int b0 = 0; b0 < a.B; b0 += a.chunk) {
      const int cb = min(a.chunk, a.B - b0);
      if (tid < cb) {
        const int b = b0 + tid;
        int p;
        if (i == 0) {
          p = a.anchors[b];
        } else {
          const int row = key_id(__ldcg(&a.keys[(size_t)(i - 1) * a.B + b]));
          p = (row >= 0 && row < a.Vh) ? (a.d2t ? a.d2t[row] : row) : -1;
        }
        if (p < 0 || p >= a.V) {
          if (c == 0) flag_error(a.err, kErrBadToken);
          p = 0;
        }
        s_prev[tid] = p;
      }
      __syncthreads();
      for (int e = tid; e < cb * a.r; e += kSimtThreads)
        s_u[e] = a.w1[(size_t)s_prev[e / a.r] * a.r + e % a.r];
      __syncthreads();
      float bv[CH];
      int bi[CH];
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        bv[j] = -INFINITY;
        bi[j] = 0x7FFFFFFF;
        s_rk[j][tid] = -INFINITY;
      }
      for (int v = vr; v < v1; v += kSimtThreads) {
        float acc[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) acc[j] = 0.f;
        if (WR && v == vr) {
#pragma unroll
          for (int q = 0; q < (WR ? kSimtRegRank : 1); ++q) {
            if (q >= a.r) break;
#pragma unroll
            for (int j = 0; j < CH; ++j)
              if (j < cb) acc[j] = fmaf(s_u[j * a.r + q], wreg[q], acc[j]);
          }
        } else {
          // eight loads issued together, then their products (in the order q = 0 .. r-1)
          for (int q0 = 0; q0 < a.r; q0 += 8) {
            float w[8];
#pragma unroll
            for (int t = 0; t < 8; ++t)
              w[t] = q0 + t < a.r ? a.w2[(size_t)(q0 + t) * a.Vh + v] : 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              if (q0 + t >= a.r) break;
#pragma unroll
              for (int j = 0; j < CH; ++j)
                if (j < cb) acc[j] = fmaf(s_u[j * a.r + q0 + t], w[t], acc[j]);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          if (j >= cb) break;
          const int b = b0 + j;
          const float zb = a.fused ? s_zf[(size_t)(i * a.B + b) * kSimtThreads + tid]
                                   : z_i[(size_t)v * a.ldb + b];
          const float x = zb + acc[j];
          if (a.lists) {
            if (a.fused)
              a.zk[((size_t)i * a.B + b) * a.ldz + v] = a.topk_markov ? x : zb;
            else
              a.zc[(size_t)b * a.ldz + v] = x;
          }
          if (a.logits) a.logits[((size_t)b * a.N + i) * a.Vh + v] = x;
          if (v == vr) s_rk[j][tid] = a.topk_markov ? x : zb;
          if (better(x, v, bv[j], bi[j])) {
            bv[j] = x;
            bi[j] = v;
          }
        }
      }
      cta_best_chunk<CH>(bv, bi, cb, sv, si);
      if (tid < cb) {
        const int b = b0 + tid;
        float v = 0.f;
        int id = 0x7FFFFFFF;
#pragma unroll
        for (int j = 0; j < CH; ++j)
          if (j == tid) {
            v = bv[j];
            id = bi[j];
          }
        if (id != 0x7FFFFFFF) {
          atomicMax(&a.keys[(size_t)i * a.B + b], order_key(v + 0.0f, id));
          // the markov_w1 row of this CTA's best: the next slot reads one of the G such
          // rows of the block, so each is brought into L2 while the grid meets
          if (i + 1 < a.N) {
            const int p = a.d2t ? a.d2t[id] : id;
            if (p >= 0 && p < a.V)
              for (int o = 0; o < a.r; o += 32)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(a.w1 + (size_t)p * a.r + o));
          }
        }
      }
      if (a.lists && !a.fused) {
        // each warp's k best ranked rows of each block (each strictly after the previous
        // pick; the ranked value: corrected, or base logits), without block-wide syncs
#pragma unroll 1
        for (int j = 0; j < cb; ++j) {
          const int b = b0 + j;
          float pv = 0.f;
          int pid = 0;
          for (int q = 0; q < a.k; ++q) {
            float qv = -INFINITY;
            int qi = 0x7FFFFFFF;
            for (int v = vr; v < v1; v += kSimtThreads) {
              const float x = v == vr ? s_rk[j][tid]
                                      : (a.topk_markov ? a.zc[(size_t)b * a.ldz + v]
                                                       : z_i[(size_t)v * a.ldb + b]);
              if ((q == 0 || better(pv, pid, x, v)) && better(x, v, qv, qi)) {
                qv = x;
                qi = v;
              }
            }
            warp_best(qv, qi);
            if (lane == 0) {
              s_lv[j][warp][q] = qv;
              s_li[j][warp][q] = qi;
            }
            pv = qv;
            pid = qi;
          }
        }
        __syncthreads();
        // warp j merges the warps' lists of block j into the CTA's k best
        if (warp < cb) {
          const int j = warp;
          const int n = kSimtWarps * a.k;
          float pv = 0.f;
          int pid = 0;
          const size_t o = (((size_t)i * a.B + b0 + j) * G + c) * a.k;
          for (int q = 0; q < a.k; ++q) {
            float qv = -INFINITY;
            int qi = 0x7FFFFFFF;
            for (int e = lane; e < n; e += 32) {
              const float x = s_lv[j][e / a.k][e % a.k];
              const int id = s_li[j][e / a.k][e % a.k];
              if (id != 0x7FFFFFFF && (q == 0 || better(pv, pid, x, id)) &&
                  better(x, id, qv, qi)) {
                qv = x;
                qi = id;
              }
            }
            warp_best(qv, qi);
            if (lane == 0) {
              a.cand_val[o + q] = qv;
              a.cand_id[o + q] = qi;
            }
            pv = qv;
            pid = qi;
          }
        }
        __syncthreads();                              // (before the lists are reused)
      }
    }
    // the next slot's base logits of this CTA's rows into L2 while the grid meets
    if (i + 1 < a.N && !a.fused)
      for (int v = vr; v < v1; v += kSimtThreads)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a.z + ((size_t)(i + 1) * a.Vhp + v) * a.ldb));
    // every CTA has posted slot i's winners: the grid barrier (release / acquire)
    __syncthreads();
    if (tid == 0) {
      red_release_add_u32(a.bar, 1u);
      const unsigned target = (unsigned)(i + 1) * (unsigned)G;
      const long long t0 = clock64();
      while (ld_acquire_u32(a.bar) < target) {
        if (clock64() - t0 > kSimtWaitBudget) {
          flag_error(a.err, kErrTimeout);
          s_abort = 1;
          break;
        }
        __nanosleep(32);
      }
    }
    __syncthreads();
    if (s_abort) return;
  }
  // the top k of every (slot, block) from the CTAs' lists (all complete after the last
  // barrier): warp w of CTA c merges pairs c * kSimtWarps + w, c * kSimtWarps + w + G *
  // kSimtWarps, ...
  if (a.lists && !a.fused) {
    for (int e = c * kSimtWarps + warp; e < a.N * a.B; e += G * kSimtWarps)
      merge_lists(a, e / a.B, e % a.B, G);
  }
  // fused: the top k of each (slot, block) over all its rows, one CTA per pair (k rounds
  // of a CTA-wide best, each strictly after the previous pick)
  if (a.lists && a.fused) {
    for (int e = c; e < a.N * a.B; e += G) {
      const int i = e / a.B, b = e % a.B;
      const float* row = a.zk + (size_t)e * a.ldz;
      // the first 16 of each thread's rows read once into registers, the rest re-read
      constexpr int kKeep = 16;
      float cv[kKeep];
#pragma unroll
      for (int t = 0; t < kKeep; ++t) {
        const int v = tid + kSimtThreads * t;
        cv[t] = v < a.Vh ? __ldcg(row + v) : -INFINITY;
      }
      float pv = 0.f;
      int pid = 0;
      for (int q = 0; q < a.k; ++q) {
        float qv[1] = {-INFINITY};
        int qi[1] = {0x7FFFFFFF};
#pragma unroll
        for (int t = 0; t < kKeep; ++t) {
          const int v = tid + kSimtThreads * t;
          const float x = cv[t];
          if (v < a.Vh && (q == 0 || better(pv, pid, x, v)) && better(x, v, qv[0], qi[0])) {
            qv[0] = x;
            qi[0] = v;
          }
        }
        for (int v = tid + kSimtThreads * kKeep; v < a.Vh; v += kSimtThreads) {
          const float x = __ldcg(row + v);
          if ((q == 0 || better(pv, pid, x, v)) && better(x, v, qv[0], qi[0])) {
            qv[0] = x;
            qi[0] = v;
          }
        }
        cta_best_chunk<1>(qv, qi, 1, sv, si);
        if (tid == 0) {
          const size_t o = ((size_t)b * a.N + i) * a.k + q;
          const int r0 = qi[0] == 0x7FFFFFFF ? 0 : qi[0];
          if (a.topk_out_ids) a.topk_out_ids[o] = a.d2t ? a.d2t[r0] : r0;
          if (a.topk_out_vals) a.topk_out_vals[o] = qv[0];
        }
        pv = qv[0];
        pid = qi[0];
      }
    }
  }
  // fused: the truncation of each block at its first slot with confidence below
  // conf_min (none when conf_min <= 0 or without a confidence head)
  if (a.fused && c == 0) {
    for (int b = tid; b < a.B; b += kSimtThreads) {
      int n = a.N;
      if (a.w_conf && a.conf_min > 0.f)
        for (int i = 0; i < a.N; ++i)
          if (__ldcg(&a.conf[(size_t)b * a.N + i]) < a.conf_min) {
            n = i;
            break;
          }
      a.n_draft[b] = n;
    }
  }
  // the draft (and, for k = 1 over corrected logits, the top-1) from the winners
  if (c == 0) {
    for (int e = tid; e < a.N * a.B; e += kSimtThreads) {
      const int i = e / a.B, b = e % a.B;
      const unsigned long long key = __ldcg(&a.keys[(size_t)i * a.B + b]);
      int row = key_id(key);
      row = (row >= 0 && row < a.Vh) ? row : 0;
      const int tok = a.d2t ? a.d2t[row] : row;
      a.draft[(size_t)b * a.N + i] = tok;
      if (a.topk_ids) a.topk_ids[(size_t)b * a.N + i] = tok;
      if (a.topk_vals) a.topk_vals[(size_t)b * a.N + i] = key_value(key);
    }
  }
}

// The same base logits for few prediction rows (M <= kSkinnyRows, their hidden states
// within 48 KB): the hidden rows are staged in shared memory, and each warp takes whole
// lm_head rows, one 16-byte chunk per lane at a time, reducing its M partial sums over
// the warp.  (Bound by the latency of reading lm_head once.)

__global__ void __launch_bounds__(256)
base_logits_skinny(const float* __restrict__ hidden, const float* __restrict__ W,
                   const float* __restrict__ bias, float* __restrict__ z, int B, int L_in,
                   int N, int ifp, int H, int Vh, size_t Vhp, size_t ldb) {
  extern __shared__ float s_h[];                      // [M][H]
  const int M = B * N;
  for (int e = threadIdx.x; e < M * H; e += 256) {
    const int m = e / H, k = e % H;
    const int i = m / B, b = m % B;
    s_h[e] = hidden[((size_t)b * L_in + ifp + i) * H + k];
  }
  __syncthreads();
  const int lane = threadIdx.x % 32;
  const int warps = gridDim.x * 8, gw = blockIdx.x * 8 + threadIdx.x / 32;
  const bool vec = (H % 4) == 0 && ((uintptr_t)W % 16) == 0;   // 16-byte row chunks
  for (int v = gw; v < Vh; v += warps) {
    float acc[kSkinnyRows];
#pragma unroll
    for (int m = 0; m < kSkinnyRows; ++m) acc[m] = 0.f;
    const float* wr = W + (size_t)v * H;
    if (vec) {
      for (int k = lane * 4; k < H; k += 128) {
        const float4 w = *reinterpret_cast<const float4*>(wr + k);
#pragma unroll
        for (int m = 0; m < kSkinnyRows; ++m) {
          if (m >= M) break;
          const float4 h = *reinterpret_cast<const float4*>(s_h + (size_t)m * H + k);
          acc[m] = fmaf(h.x, w.x, fmaf(h.y, w.y, fmaf(h.z, w.z, fmaf(h.w, w.w, acc[m]))));
        }
      }
    } else {
      for (int k = lane; k < H; k += 32) {
        const float w = wr[k];
#pragma unroll
        for (int m = 0; m < kSkinnyRows; ++m) {
          if (m >= M) break;
          acc[m] = fmaf(s_h[(size_t)m * H + k], w, acc[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < kSkinnyRows; ++m) {
      if (m >= M) break;
      float x = acc[m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
      if (lane == 0) {
        const int i = m / B, b = m % B;
        z[((size_t)i * Vhp + v) * ldb + b] = x + (bias ? bias[v] : 0.f);
      }
    }
  }
}

cudaError_t base_logits(const ProposePlan& p) {
  const int M = p.B * p.N;
  if (M <= kSkinnyRows && (size_t)M * p.H * sizeof(float) <= 48 * 1024) {
    int sms = 0;
    cudaError_t e = device_sms(&sms);
    if (e != cudaSuccess) return e;
    const int warps_needed = p.Vh;                      // one lm_head row per warp at most
    const int grid = std::max(1, std::min(4 * sms, (warps_needed + 7) / 8));
    base_logits_skinny<<<grid, 256, sizeof(float) * (size_t)M * p.H, p.stream>>>(
        (const float*)p.hidden, (const float*)p.lm_head, p.lm_bias, p.z, p.B, p.L_in, p.N,
        p.ifp, p.H, p.Vh, p.Vhp, p.ldb);
    return cudaGetLastError();
  }
  dim3 grid((p.Vh + kTileV - 1) / kTileV, (p.B * p.N + kTileM - 1) / kTileM);
  base_logits_simt<<<grid, 256, 0, p.stream>>>(
      (const float*)p.hidden, (const float*)p.lm_head, p.lm_bias, p.z, p.B, p.L_in, p.N,
      p.ifp, p.H, p.Vh, p.Vhp, p.ldb);
  return cudaGetLastError();
}

const void* simt_kernel(int ch, bool wr) {
  switch (ch * 2 + (wr ? 1 : 0)) {
    case 2: return reinterpret_cast<const void*>(chain_simt<1, false>);
    case 3: return reinterpret_cast<const void*>(chain_simt<1, true>);
    case 4: return reinterpret_cast<const void*>(chain_simt<2, false>);
    case 5: return reinterpret_cast<const void*>(chain_simt<2, true>);
    case 8: return reinterpret_cast<const void*>(chain_simt<4, false>);
    case 9: return reinterpret_cast<const void*>(chain_simt<4, true>);
    case 16: return reinterpret_cast<const void*>(chain_simt<8, false>);
    default: return reinterpret_cast<const void*>(chain_simt<8, true>);
  }
}

// Launch shape of the fp32 chain: blocks per chunk, the instantiation, and whether the
// base logits and the confidence head run inside it (small problems: at most
// kSkinnyRows prediction rows whose hidden states fit 32 KB, one head row per thread,
// no adaptive block length).
struct SimtShape {
  int chunk, ch, G;
  bool wr, fused;
  size_t smem;
  const void* kern;
};

cudaError_t simt_shape(int B, int N, int H, int Vh, int r, bool skip_truncated, SimtShape* sh) {
  const int cap = std::max(1, (48 * 1024 / 4) / std::max(r, 1));
  sh->chunk = std::max(1, std::min({kSimtMaxChunk, B, cap}));
  sh->ch = sh->chunk <= 1 ? 1 : sh->chunk <= 2 ? 2 : sh->chunk <= 4 ? 4 : 8;
  sh->wr = r <= kSimtRegRank;
  sh->kern = simt_kernel(sh->ch, sh->wr);
  const size_t M = (size_t)B * N;
  const size_t base = sizeof(float) * (size_t)r * sh->chunk;
  const size_t fused_smem = base + 16 + sizeof(float) * (M * H + M * kSimtThreads);
  int sms = 0, per_sm = 0;
  cudaError_t e = device_sms(&sms);
  if (e != cudaSuccess) return e;
  sh->fused = false;
  if (!skip_truncated && M <= kSkinnyRows && M * H * sizeof(float) <= 32 * 1024 &&
      (long long)Vh <= (long long)simt_chain_ctas_max(Vh) * kSimtThreads) {
    e = raise_smem_limit(sh->kern, fused_smem);
    if (e == cudaSuccess) e = blocks_per_sm(sh->kern, kSimtThreads, fused_smem, &per_sm);
    if (e != cudaSuccess) return e;
    // (about 32 head rows per CTA: the base logits then use every SM)
    const int G = std::max(1, std::min({(Vh + 31) / 32, sms * per_sm, kChainMaxCtas}));
    if (per_sm >= 1 && (long long)Vh <= (long long)G * kSimtThreads) {
      sh->fused = true;
      sh->smem = fused_smem;
      sh->G = G;
      return cudaSuccess;
    }
  }
  sh->smem = base;
  // (the dynamic part may need the opt-in: the kernel's static lists take up to 17 KB)
  e = raise_smem_limit(sh->kern, sh->smem);
  if (e == cudaSuccess) e = blocks_per_sm(sh->kern, kSimtThreads, sh->smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  sh->G = std::max(1, std::min(simt_chain_ctas_max(Vh), sms * per_sm));
  return cudaSuccess;
}

cudaError_t chain_fused(const ProposePlan& p) {
  SimtShape sh;
  cudaError_t e = simt_shape(p.B, p.N, p.H, p.Vh, p.r, p.skip_truncated, &sh);
  if (e != cudaSuccess) return e;
  const int G = sh.G;
  const bool want_topk = p.topk_ids || p.topk_vals;
  const bool lists = want_topk && (p.k > 1 || !p.topk_markov);
  SimtArgs a{};
  a.z = p.z;
  a.w1 = (const float*)p.w1;
  a.w2 = (const float*)p.w2;
  a.anchors = p.anchors;
  a.d2t = p.d2t;
  a.draft = p.draft;
  a.topk_ids = lists ? nullptr : p.topk_ids;
  a.topk_vals = lists ? nullptr : p.topk_vals;
  a.topk_out_ids = lists ? p.topk_ids : nullptr;
  a.topk_out_vals = lists ? p.topk_vals : nullptr;
  a.logits = p.logits;
  a.zc = p.zc;
  a.cand_val = p.cand_val;
  a.cand_id = p.cand_id;
  a.keys = p.keys;
  a.bar = p.bar;
  a.err = p.ctrl;
  a.Vhp = p.Vhp;
  a.ldb = p.ldb;
  a.ldz = p.ldz;
  a.B = p.B;
  a.N = p.N;
  a.V = p.V;
  a.Vh = p.Vh;
  a.r = p.r;
  a.k = p.k;
  a.topk_markov = p.topk_markov;
  a.lists = lists ? 1 : 0;
  a.chunk = sh.chunk;
  a.fused = sh.fused ? 1 : 0;
  a.hidden = (const float*)p.hidden;
  a.lm_head = (const float*)p.lm_head;
  a.lm_bias = p.lm_bias;
  a.conf_hidden = (const float*)p.conf_hidden;
  a.w_conf = (const float*)p.w_conf;
  a.b_conf = p.b_conf;
  a.conf_min = p.conf_min;
  a.conf = p.conf ? p.conf : p.conf_ws;
  a.n_draft = p.n_draft;
  a.zk = p.zk;
  a.L_in = p.L_in;
  a.ifp = p.ifp;
  a.H = p.H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kSimtThreads);
  cfg.dynamicSmemBytes = sh.smem;
  cfg.stream = p.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&a};
  return cudaLaunchKernelExC(&cfg, sh.kern, args);
}

}  // namespace

cudaError_t launch_base_logits_simt(const ProposePlan& p) {
  return base_logits(p);            // (the bf16 operand type runs on the tensor cores)
}

cudaError_t launch_chain_simt(const ProposePlan& p) { return chain_fused(p); }

bool simt_fused(int B, int N, int H, int Vh, int r, bool skip_truncated) {
  SimtShape sh;
  if (simt_shape(B, N, H, Vh, r, skip_truncated, &sh) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return sh.fused;
}

// CTAs of the fp32 chain at most: one per 256 head rows, within the list capacity
int simt_chain_ctas_max(int Vh) { return std::min(kChainMaxCtas, (Vh + 255) / 256); }

}  // namespace dspark
