// The Markov-corrected greedy chain on the 5th-generation tensor cores, one persistent
// cooperative kernel for all N slots of a group of up to 32 blocks.
//
// llama.cpp commit 6fed9f6 ("spec: add DSpark speculative decoding", the proposal
// formula):
//   logits'(i) = logits(i) + markov_w2^T . markov_w1[prev(i)]
//   prev(0) = anchor,  prev(i > 0) = argmax logits'(i - 1)
// sequential over the slots, vectorised over the blocks.
//
// Each CTA owns a fixed, contiguous range of 128-row vocabulary tiles.  Per slot:
//   1. the epilogue warps gather u[b] = markov_w1[prev_b] (bf16, K-major, 128-byte
//      swizzled) into shared memory: the MMA's B operand, N = blocks padded to 16;
//   2. the producer warp streams markov_w2 tiles [r x 128] by TMA (MN-major A operand;
//      the tiles are the same every slot, so the producer runs ahead across slots);
//   3. the MMA warp issues m[v, b] = sum_k w2[k, v] * u[b, k] (tcgen05, M = 128 head
//      rows) into a ring of TMEM accumulators;
//   4. the epilogue adds the base logits z[i][b][v], transposes 32 x 32 panels through
//      shared memory so that lane b owns block b, and keeps per-lane running argmax
//      (always over the corrected logits) and top-k (over corrected or base logits);
//   5. the CTA's best candidate per block goes to a 64-bit order key with atomicMax,
//      its top-k list to a partial buffer; a bounded grid barrier ends the slot and
//      every CTA reads the winners as the next slot's previous tokens.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dspark {

namespace {

constexpr int kTileV = 128;
constexpr int kKB = 64;                                 // K rows per stage
constexpr uint32_t kHalf = 64 * kKB * 2;                // one 64-column half: 8 KB
constexpr uint32_t kStage = 2 * kHalf;                  // 16 KB
constexpr int kEpiWarps = 8;                            // two groups of four
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kProducerWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1;
constexpr int kThreads = 32 * (kEpiWarps + 2);
constexpr int kPanel = 32 * 33;                         // one padded 32 x 32 transpose panel
constexpr long long kWaitBudget = 2000000000ll;         // ~1 s of SM clocks

struct ChainArgs {
  const float* z;       // base logits [N][Vhp][ldb]
  size_t Vhp, ldb;
  const __nv_bfloat16* w1;
  const int32_t* anchors;
  const int32_t* d2t;
  int32_t* draft;
  float* logits;
  float* part_val;
  int32_t* part_id;
  unsigned long long* keys;
  unsigned int* bar;
  uint32_t* err;
  int B, b0, Bg, N, V, Vh, r, k, want_topk;
  int n_mma, kb_count, tiles, stages, n_acc;
  uint32_t acc_stride, tmem_cols;
  uint32_t u_kb_bytes;      // n_mma * 128
  uint32_t scratch_bytes;
};

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

// All epilogue threads agree on whether to stop: one thread samples the abort flag
// between two named barriers and everyone reads that sample.
__device__ __forceinline__ bool epi_agree_abort(volatile int* abort_flag,
                                                volatile int* decision, int tid) {
  epi_sync();
  if (tid == 0) *decision = *abort_flag;
  epi_sync();
  return *decision != 0;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive floats from a 16-byte aligned row holding `avail` valid entries; the
// rest read as -inf.
__device__ __forceinline__ void load_z32(const float* row, bool ok, long long avail,
                                         float (&zv)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (ok && 4 * q < avail) f = __ldcs(reinterpret_cast<const float4*>(row) + q);
    zv[4 * q] = f.x;
    zv[4 * q + 1] = f.y;
    zv[4 * q + 2] = f.z;
    zv[4 * q + 3] = f.w;
  }
}

// Insert (v, id) into a sorted list of KT entries (best first); the last one drops out.
template <int KT>
__device__ __forceinline__ void list_insert(float (&lv)[KT], int (&li)[KT], float v, int id) {
#pragma unroll
  for (int q = 0; q < KT; ++q) {
    if (better(v, id, lv[q], li[q])) {
      const float tv = lv[q];
      const int ti = li[q];
      lv[q] = v;
      li[q] = id;
      v = tv;
      id = ti;
    }
  }
}

// KT: size of the per-lane candidate lists (>= top_k; 1 when no list is kept).
// NCH: 32-block chunks per group of blocks.  ZRANK: top-k ranks the base logits.
template <int KT, int NCH, bool ZRANK>
__global__ void __launch_bounds__(kThreads, 1)
chain_tc(const __grid_constant__ CUtensorMap tm_w2, const ChainArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* s_w2 = smem;
  uint8_t* s_u = s_w2 + (size_t)a.stages * kStage;
  float* s_scr = (float*)(s_u + (size_t)a.kb_count * a.u_kb_bytes);
  uint8_t* tail = (uint8_t*)s_scr + a.scratch_bytes;
  uint64_t* full = (uint64_t*)tail;
  uint64_t* empty = full + a.stages;
  uint64_t* acc_full = empty + a.stages;
  uint64_t* acc_empty = acc_full + a.n_acc;
  uint64_t* u_ready = acc_empty + a.n_acc;
  uint64_t* drain = u_ready + 1;
  int32_t* s_prev = (int32_t*)(drain + 1);               // [64]
  uint32_t* tmem_slot = (uint32_t*)(s_prev + 64);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  volatile int* s_decision = abort_flag + 1;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int q = 0; q < a.n_acc; ++q) {
      ptx::mbar_init(&acc_full[q], 1);
      ptx::mbar_init(&acc_empty[q], 128);       // the four warps of one group
    }
    ptx::mbar_init(u_ready, 1);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) ptx::tma_prefetch_desc(&tm_w2);
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, a.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int t_begin = (int)((long long)blockIdx.x * a.tiles / G);
  const int t_end = (int)((long long)(blockIdx.x + 1) * a.tiles / G);
  const int nt = t_end - t_begin;

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(a.err, kErrTimeout);
  };

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int step = 0; ok && step < a.N; ++step)
        for (int t = t_begin; ok && t < t_end; ++t)
          for (int kb = 0; kb < a.kb_count; ++kb, ++it) {
            const uint32_t s = it % a.stages, ph = (it / a.stages) & 1;
            if (!ptx::mbar_wait(&empty[s], ph ^ 1, kWaitBudget, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* dst = s_w2 + (size_t)s * kStage;
            ptx::mbar_arrive_expect_tx(&full[s], kStage);
            ptx::tma_load_2d(dst, &tm_w2, &full[s], t * kTileV, kb * kKB);
            ptx::tma_load_2d(dst + kHalf, &tm_w2, &full[s], t * kTileV + 64, kb * kKB);
          }
      if (!ok) {
        give_up();
        const uint32_t first = it > (uint32_t)a.stages ? it - a.stages : 0;
        for (uint32_t j = first; j < it; ++j)
          ptx::mbar_wait(&full[j % a.stages], (j / a.stages) & 1, kWaitBudget, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16_f32(kTileV, a.n_mma, /*A MN-major*/ 1, 0);
      uint32_t it = 0;
      bool ok = true;
      for (int step = 0; ok && step < a.N; ++step) {
        if (!ptx::mbar_wait(u_ready, step & 1, kWaitBudget, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t u0 = ptx::smem_u32(s_u);
        for (int lt = 0; ok && lt < nt; ++lt) {
          const uint32_t gl = (uint32_t)(step * nt + lt);
          const uint32_t acc = gl % a.n_acc, aph = (gl / a.n_acc) & 1;
          if (!ptx::mbar_wait(&acc_empty[acc], aph ^ 1, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d = tmem + acc * a.acc_stride;
          for (int kb = 0; kb < a.kb_count; ++kb, ++it) {
            const uint32_t s = it % a.stages, ph = (it / a.stages) & 1;
            if (!ptx::mbar_wait(&full[s], ph, kWaitBudget, abort_flag)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t w0 = ptx::smem_u32(s_w2 + (size_t)s * kStage);
            const uint32_t b0 = u0 + kb * a.u_kb_bytes;
#pragma unroll
            for (int kk = 0; kk < kKB / 16; ++kk)
              ptx::mma_f16(d, ptx::desc_mnmajor_sw128(w0 + kk * 2048, kHalf, 1024),
                           ptx::desc_kmajor_sw128(b0 + kk * 32), idesc, (kb | kk) != 0);
            ptx::mma_commit(&empty[s]);
          }
          if (ok) ptx::mma_commit(&acc_full[acc]);
        }
      }
      if (!ok) give_up();
      ptx::mma_commit(drain);
      ptx::mbar_wait(drain, 0, kWaitBudget, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int tid = threadIdx.x;                    // 0..255
    const int quad = warp % 4, grp = warp / 4;      // TMEM lane quadrant, tile parity
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float* scr_x = s_scr + warp * (ZRANK ? 2 : 1) * kPanel;
    float* scr_z = scr_x + kPanel;
    bool ok = true;
    for (int step = 0; ok && step < a.N; ++step) {
      // -------- 1. previous tokens of this slot
      if (tid < a.Bg) {
        int p;
        if (step == 0) {
          p = a.anchors[a.b0 + tid];
        } else {
          const unsigned long long key = __ldcg(&a.keys[(size_t)(step - 1) * a.B + a.b0 + tid]);
          const int row = key_id(key);
          p = a.d2t ? a.d2t[row] : row;
          if (blockIdx.x == 0) a.draft[(size_t)(a.b0 + tid) * a.N + step - 1] = p;
        }
        if (p < 0 || p >= a.V) {
          flag_error(a.err, kErrBadToken);
          p = 0;
        }
        s_prev[tid] = p;
      }
      epi_sync();
      // -------- 2. u = markov_w1[prev] into the swizzled K-major B operand
      {
        const int per_row = a.kb_count * 8;
        const int chunks = a.n_mma * per_row;
        for (int base = 0; base < chunks; base += 4 * kEpiThreads) {
          uint4 val[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int idx = base + q * kEpiThreads + tid;
            val[q] = make_uint4(0, 0, 0, 0);
            const int n = idx / per_row, rem = idx % per_row;
            if (idx < chunks && n < a.Bg) {
              const int k0 = (rem / 8) * kKB + (rem % 8) * 8;
              const __nv_bfloat16* src = a.w1 + (size_t)s_prev[n] * a.r + k0;
              if ((a.r & 7) == 0 && k0 + 8 <= a.r) {
                val[q] = __ldg(reinterpret_cast<const uint4*>(src));
              } else {                                 // ragged rank: element-wise
                uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  if (k0 + c < a.r)
                    w[c / 2] |= (uint32_t)__bfloat16_as_ushort(src[c]) << (16 * (c % 2));
                val[q] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int idx = base + q * kEpiThreads + tid;
            if (idx < chunks) {
              const int n = idx / per_row, rem = idx % per_row;
              const int kb = rem / 8, j = rem % 8;
              *reinterpret_cast<uint4*>(s_u + (size_t)kb * a.u_kb_bytes + n * 128 +
                                        ((j ^ (n & 7)) << 4)) = val[q];
            }
          }
        }
      }
      fence_proxy_async();
      epi_sync();
      if (tid == 0) ptx::mbar_arrive(u_ready);

      // -------- 3. tiles of this group: base logits + Markov term, running argmax/top-k
      float amax_v[NCH], thr_v[NCH];
      int amax_i[NCH], thr_i[NCH];
      float lv[NCH][KT];
      int li[NCH][KT];
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        amax_v[c] = thr_v[c] = -INFINITY;
        amax_i[c] = thr_i[c] = 0x7FFFFFFF;
#pragma unroll
        for (int q = 0; q < KT; ++q) {
          lv[c][q] = -INFINITY;
          li[c][q] = 0x7FFFFFFF;
        }
      }
      const float* z_i = a.z + (size_t)step * a.Vhp * a.ldb;
      for (int lt = grp; lt < nt; lt += 2) {
        const int t = t_begin + lt;
        const int v = t * kTileV + quad * 32 + lane;
        const bool v_ok = v < a.Vh;
        const int id0 = t * kTileV + quad * 32;          // id of candidate j is id0 + j
        // base logits of this head row for the chunk's 32 blocks: contiguous, 16-byte loads
        const float* zrow = z_i + (size_t)v * a.ldb + a.b0;
        float zv[32];
        load_z32(zrow, v_ok, a.ldb - a.b0, zv);
        const uint32_t gl = (uint32_t)(step * nt + lt);
        const uint32_t acc = gl % a.n_acc, aph = (gl / a.n_acc) & 1;
        ok = __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&acc_full[acc], aph, kWaitBudget, abort_flag));
        if (!ok) break;
        ptx::tc_fence_after();
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(tmem + lane_base + acc * a.acc_stride + c * 32, r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = zv[j] + __uint_as_float(r[j]);
            scr_x[j * 33 + lane] = x;
            if (ZRANK) scr_z[j * 33 + lane] = zv[j];
            if (a.logits && v_ok && c * 32 + j < a.Bg)
              a.logits[((size_t)(a.b0 + c * 32 + j) * a.N + step) * a.Vh + v] = x;
          }
          if (c + 1 < NCH)                                 // next chunk's base logits
            load_z32(zrow + (c + 1) * 32, v_ok, (long long)a.ldb - a.b0 - (c + 1) * 32, zv);
          __syncwarp();
#pragma unroll 4
          for (int j = 0; j < 32; ++j) {
            const int id = id0 + j;
            if (id < a.Vh) {                               // uniform over the warp
              const float x = scr_x[lane * 33 + j];
              if (better(x, id, amax_v[c], amax_i[c])) {
                amax_v[c] = x;
                amax_i[c] = id;
              }
              if (KT > 1 || ZRANK) {
                const float rk = ZRANK ? scr_z[lane * 33 + j] : x;
                if (better(rk, id, thr_v[c], thr_i[c])) {  // beats the list's last entry
                  list_insert<KT>(lv[c], li[c], rk, id);
                  thr_v[c] = lv[c][KT - 1];
                  thr_i[c] = li[c][KT - 1];
                }
              }
            }
          }
          __syncwarp();
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&acc_empty[acc]);
      }
      // a warp that gave up raises the flag; the others then stop waiting, and all take
      // the same decision here (the named barriers below need every epilogue thread)
      if (!ok) give_up();
      if (epi_agree_abort(abort_flag, s_decision, tid)) {
        ok = false;
        break;
      }
      // -------- 4. merge the eight warps, publish the CTA's candidates
      constexpr int KL = (KT > 1 || ZRANK) ? KT : 1;   // entries per lane list in smem
      constexpr int BS = NCH * 32;                     // block stride of the merge arrays
      float* m_av = s_scr;                             // [8][BS]
      int* m_ai = (int*)(m_av + kEpiWarps * BS);       // [8][BS]
      float* m_lv = (float*)(m_ai + kEpiWarps * BS);   // [8][BS][KL]
      int* m_li = (int*)(m_lv + kEpiWarps * BS * KL);  // [8][BS][KL]
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        const int b = c * 32 + lane;
        m_av[warp * BS + b] = amax_v[c];
        m_ai[warp * BS + b] = amax_i[c];
        if (KT > 1 || ZRANK) {
#pragma unroll
          for (int q = 0; q < KL; ++q) {
            m_lv[(warp * BS + b) * KL + q] = lv[c][q];
            m_li[(warp * BS + b) * KL + q] = li[c][q];
          }
        }
      }
      epi_sync();
      if (tid < a.Bg) {                                // argmax of each block
        const int b = tid;
        float bv = m_av[b];
        int bi = m_ai[b];
#pragma unroll
        for (int w = 1; w < kEpiWarps; ++w)
          if (better(m_av[w * BS + b], m_ai[w * BS + b], bv, bi)) {
            bv = m_av[w * BS + b];
            bi = m_ai[w * BS + b];
          }
        if (bi != 0x7FFFFFFF) atomicMax(&a.keys[(size_t)step * a.B + a.b0 + b], order_key(bv, bi));
      }
      if (a.want_topk) {
        // one warp per block: k rounds of a warp-wide best among the 8 lists' entries
        // strictly after the previous pick
        for (int b = warp; b < a.Bg; b += kEpiWarps) {
          const size_t o = (((size_t)step * a.B + a.b0 + b) * G + blockIdx.x) * a.k;
          float pv = 0.f;
          int pid = 0;
          for (int q = 0; q < a.k; ++q) {
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF;
            for (int e = lane; e < kEpiWarps * KL; e += 32) {
              const int w = e / KL, s2 = e % KL;
              const float x = (KT > 1 || ZRANK) ? m_lv[(w * BS + b) * KL + s2] : m_av[w * BS + b];
              const int xi = (KT > 1 || ZRANK) ? m_li[(w * BS + b) * KL + s2] : m_ai[w * BS + b];
              if ((q == 0 || better(pv, pid, x, xi)) && better(x, xi, bv, bi)) {
                bv = x;
                bi = xi;
              }
            }
            warp_best(bv, bi);
            if (lane == 0) {
              a.part_val[o + q] = bv;
              a.part_id[o + q] = bi;
            }
            pv = bv;
            pid = bi;
          }
        }
      }
      // -------- 5. grid barrier: every CTA has published this slot
      __threadfence();
      epi_sync();
      if (tid == 0) {
        atomicAdd(a.bar, 1u);
        const unsigned target = (unsigned)(step + 1) * (unsigned)G;
        const long long t0 = clock64();
        while (ld_acquire(a.bar) < target) {
          if (clock64() - t0 > kWaitBudget) {
            give_up();
            break;
          }
        }
      }
      if (epi_agree_abort(abort_flag, s_decision, tid)) {
        ok = false;
        break;
      }
    }
    if (ok && blockIdx.x == 0 && tid < a.Bg) {
      const unsigned long long key = __ldcg(&a.keys[(size_t)(a.N - 1) * a.B + a.b0 + tid]);
      const int row = key_id(key);
      a.draft[(size_t)(a.b0 + tid) * a.N + a.N - 1] = a.d2t ? a.d2t[row] : row;
    }
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, a.tmem_cols);
  }
}

// Merge of the per-CTA top-k lists of every (slot, block) into the sorted output.
template <int KMAX>
__global__ void __launch_bounds__(256)
topk_merge(const float* __restrict__ part_val, const int32_t* __restrict__ part_id, int G,
           int k, int B, int N, const int32_t* __restrict__ d2t, int32_t* __restrict__ ids,
           float* __restrict__ vals) {
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (w >= B * N) return;
  const int i = w / B, b = w % B;
  const size_t base = ((size_t)i * B + b) * G * k;
  float lv[KMAX];
  int li[KMAX];
#pragma unroll
  for (int q = 0; q < KMAX; ++q) {
    lv[q] = -INFINITY;
    li[q] = 0x7FFFFFFF;
  }
  for (int c = lane; c < G * k; c += 32) {
    const float x = part_val[base + c];
    const int xi = part_id[base + c];
    if (better(x, xi, lv[KMAX - 1], li[KMAX - 1])) list_insert<KMAX>(lv, li, x, xi);
  }
  // k rounds of a warp-wide pick of the best list head
  for (int q = 0; q < k; ++q) {
    float bv = lv[0];
    int bi = li[0];
    warp_best(bv, bi);
    if (li[0] == bi && lv[0] == bv) {      // the winning lane pops its head
#pragma unroll
      for (int s = 0; s + 1 < KMAX; ++s) {
        lv[s] = lv[s + 1];
        li[s] = li[s + 1];
      }
      lv[KMAX - 1] = -INFINITY;
      li[KMAX - 1] = 0x7FFFFFFF;
    }
    if (lane == 0) {
      const size_t o = ((size_t)b * N + i) * k + q;
      const int row = bi == 0x7FFFFFFF ? 0 : bi;
      if (ids) ids[o] = d2t ? d2t[row] : row;
      if (vals) vals[o] = bv;
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

template <int KT, int NCH, bool ZRANK>
cudaError_t launch_chain_inst(const CUtensorMap& tm, const ChainArgs& a, int grid, size_t smem,
                              cudaStream_t stream) {
  auto kern = chain_tc<KT, NCH, ZRANK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm, a);
}

}  // namespace

cudaError_t launch_chain_tc(const ProposePlan& p) {
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = (p.Vh + kTileV - 1) / kTileV;
  const int grid = std::max(1, std::min({sms, tiles, kChainMaxCtas}));
  const bool want_topk = p.topk_ids || p.topk_vals;
  const bool zrank = want_topk && !p.topk_markov;
  // per-lane list size: none when only the argmax is needed (or when the argmax is the
  // whole top-1), else the smallest of 8 / 32 that holds top_k
  const int kt = (!want_topk || (p.k == 1 && p.topk_markov)) ? 1 : (p.k <= 8 ? 8 : 32);
  const int group = 32;                        // blocks per launch: one per lane

  CUtensorMap tm;
  {
    cuuint64_t dims[2] = {(cuuint64_t)p.Vh, (cuuint64_t)p.r};
    cuuint64_t strides[1] = {(cuuint64_t)p.Vh * 2};
    cuuint32_t box[2] = {64, kKB};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)p.w2, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  for (int b0 = 0; b0 < p.B; b0 += group) {
    ChainArgs a{};
    a.z = p.z;
    a.Vhp = p.Vhp;
    a.ldb = p.ldb;
    a.w1 = (const __nv_bfloat16*)p.w1;
    a.anchors = p.anchors;
    a.d2t = p.d2t;
    a.draft = p.draft;
    a.logits = p.logits;
    a.part_val = p.part_val;
    a.part_id = p.part_id;
    a.keys = p.keys;
    a.bar = p.bar + b0 / 32;
    a.err = p.ctrl;
    a.B = p.B;
    a.b0 = b0;
    a.Bg = std::min(group, p.B - b0);
    a.N = p.N;
    a.V = p.V;
    a.Vh = p.Vh;
    a.r = p.r;
    a.k = p.k;
    a.want_topk = want_topk ? 1 : 0;
    a.n_mma = (a.Bg + 15) / 16 * 16;
    a.kb_count = (p.r + kKB - 1) / kKB;
    a.tiles = tiles;
    a.acc_stride = (uint32_t)((a.n_mma + 31) / 32 * 32);
    a.n_acc = 4;
    uint32_t cols = 32;
    while (cols < a.n_acc * a.acc_stride) cols <<= 1;
    a.tmem_cols = cols;
    a.u_kb_bytes = (uint32_t)a.n_mma * 128;
    const int kl = (kt > 1 || zrank) ? kt : 1;
    const size_t transpose = (size_t)kEpiWarps * (zrank ? 2 : 1) * kPanel * sizeof(float);
    const size_t bs = a.Bg <= 32 ? 32 : 64;
    const size_t merge = (size_t)kEpiWarps * bs * 8 + (size_t)kEpiWarps * bs * kl * 8;
    a.scratch_bytes = (uint32_t)align_up(std::max(transpose, merge), 1024);
    const size_t fixed = 1024 + (size_t)a.kb_count * a.u_kb_bytes + a.scratch_bytes + 1024;
    const size_t budget = 225 * 1024;
    if (fixed + 2 * kStage > budget) return cudaErrorInvalidConfiguration;
    a.stages = (int)std::min<size_t>(12, (budget - fixed) / kStage);
    const size_t smem = fixed + (size_t)a.stages * kStage;
    cudaError_t e;
    if (kt == 1)
      e = zrank ? launch_chain_inst<1, 1, true>(tm, a, grid, smem, p.stream)
                : launch_chain_inst<1, 1, false>(tm, a, grid, smem, p.stream);
    else if (kt == 8)
      e = zrank ? launch_chain_inst<8, 1, true>(tm, a, grid, smem, p.stream)
                : launch_chain_inst<8, 1, false>(tm, a, grid, smem, p.stream);
    else
      e = zrank ? launch_chain_inst<32, 1, true>(tm, a, grid, smem, p.stream)
                : launch_chain_inst<32, 1, false>(tm, a, grid, smem, p.stream);
    if (e != cudaSuccess) return e;
  }
  const int kmax = p.k <= 1 ? 1 : (p.k <= 8 ? 8 : 32);
  if (want_topk) {
    const int warps = p.B * p.N;
    const int threads = 256;
    const int blocks = (warps * 32 + threads - 1) / threads;
    if (kmax == 1)
      topk_merge<1><<<blocks, threads, 0, p.stream>>>(p.part_val, p.part_id, grid, p.k, p.B,
                                                      p.N, p.d2t, p.topk_ids, p.topk_vals);
    else if (kmax == 8)
      topk_merge<8><<<blocks, threads, 0, p.stream>>>(p.part_val, p.part_id, grid, p.k, p.B,
                                                      p.N, p.d2t, p.topk_ids, p.topk_vals);
    else
      topk_merge<32><<<blocks, threads, 0, p.stream>>>(p.part_val, p.part_id, grid, p.k, p.B,
                                                       p.N, p.d2t, p.topk_ids, p.topk_vals);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace dspark
