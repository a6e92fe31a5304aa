// The Markov-corrected greedy chain evaluated over every head row (the dense form), one
// persistent cooperative kernel for all N slots of a group of up to 32 blocks.
//
// llama.cpp commit 6fed9f6 ("spec: add DSpark speculative decoding", the proposal
// formula):
//   logits'(i) = logits(i) + markov_w2^T . markov_w1[prev(i)]
//   prev(0) = anchor,  prev(i > 0) = argmax logits'(i - 1)
// sequential over the slots, vectorised over the blocks.
//
// Each CTA owns a fixed, contiguous range of 128-row vocabulary tiles, and TMEM holds the
// Markov terms of all of them for one slot (tiles x blocks fp32 columns, two slots' worth
// when that fits).  Per slot:
//   1. the epilogue warps gather u[b] = markov_w1[prev_b] into shared memory: the MMA's
//      B operand (K-major, 128-byte swizzled; N = blocks padded to 16 or 32);
//   2. two producer warps stream markov_w2 in [K-rows x 128 columns] stages by TMA
//      (MN-major A operand; the same tiles every slot, so they run ahead across slots),
//      and a third streams the slot's base logits z, [128 rows x 32 blocks] per tile,
//      with an evict-first L2 policy (z is read once; markov_w2 stays in L2);
//   3. the MMA thread issues m[v, b] = sum_k w2[k, v] u[b, k] for every tile (tcgen05,
//      M = 128 head rows) into the slot's TMEM columns;
//   4. pass 1 (the critical path): every epilogue warp takes every tile, thread = one
//      head row of its TMEM lane quadrant x half of the blocks; z' = z + m goes back into
//      TMEM, and each thread keeps a running best per block (value and tile).  After the
//      last tile a shuffle network gives each lane one block's best of the warp, shared
//      memory the CTA's, a 64-bit atomicMax the grid's; each block's thread then arrives
//      on the grid barrier with a release and pulls the markov_w1 row of its CTA's best
//      into L2 (the next slot gathers one of those rows);
//   5. once the barrier completes, the epilogue gathers the next slot's u (so its MMAs
//      start) and then, while they run, finds this slot's top-k candidates: every CTA
//      also posted its best value of each block into one of 2k bucket maxima (the CTA
//      index picks the bucket), so each bucket maximum is a distinct element and the
//      k-th largest of them is a lower bound of the block's k-th largest value.  Rows at
//      or above it, read back from TMEM, are appended to a short global list per (slot,
//      block) -- about k of them over the whole grid.  After the kernel, topk_final
//      sorts each list; a list that overflowed (massive ties) is recomputed exactly over
//      every head row instead.
// Every wait is bounded (about a second of clocks): on expiry the kernel raises the
// timeout bit of the error word and winds down.
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
constexpr uint32_t kZStage = kTileV * 32 * 4;           // base logits of a tile: 16 KB
constexpr int kEpiWarps = 8;                            // 4 TMEM quadrants x 2 block halves
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kMmaWarp = 8, kZWarp = 9, kW2Warp = 10;   // two markov_w2 producers: 10, 11
constexpr int kThreads = 32 * 12;
constexpr int kZStages = 3;
constexpr long long kWaitBudget = 2000000000ll;         // ~1 s of SM clocks

struct DenseArgs {
  const __nv_bfloat16* w1;
  const int32_t* anchors;
  const int32_t* d2t;
  int32_t* draft;
  int32_t* topk_ids;      // written here only for k = 1 over corrected logits (the argmax)
  float* topk_vals;
  float* logits;
  float* cand_val;        // [N][B][G][kDenseLocal] rows at or above the top-k bound
  int32_t* cand_id;
  int32_t* cand_cnt;      // [N][B][G] how many this CTA found
  uint32_t* bucket;       // [N][B][kDenseBuckets] maxima of the CTAs' best values
  unsigned long long* keys;
  unsigned int* bar;
  uint32_t* err;
  size_t Vhp;
  int B, b0, Bg, N, V, Vh, r, k;
  int n_mma, kstages, kb_count, tiles, tmax, dbuf, stages, nb;   // nb: buckets in use
  int ks;                 // markov_w2 K-rows per stage: 256 (two 32 KB boxes) or 128
  uint32_t box, stage;    // bytes of one 64-column box and of a stage (two boxes)
  uint32_t u_kb_bytes, tmem_cols;
};

// Named barrier of the epilogue warps.  The non-.aligned form: a warp may reach it
// diverged (one thread polls the grid barrier while the others wait here).
__device__ __forceinline__ void epi_sync() {
  asm volatile("barrier.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
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

// -0 and +0 are equal values (the lower id decides between them), but not equal keys:
// keys are taken of x + 0, which is +0 for both.
__device__ __forceinline__ float canon(float x) { return __fadd_rn(x, 0.0f); }

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// NK MMAs of K = 16 over one markov_w2 stage: A advances 16 K-rows (2048 bytes) per MMA,
// B 32 bytes inside its 64-K swizzle block and bstep (16-byte units) between blocks.  The
// descriptors' 14-bit address fields stay below 2^14 (shared memory < 256 KB), so the
// sums carry into nothing.
template <int NK>
__device__ __forceinline__ void mma_run(uint32_t d, uint64_t ad, uint64_t bd, uint32_t bstep,
                                        uint32_t idesc, bool accumulate_first) {
#pragma unroll
  for (int kk = 0; kk < NK; ++kk)
    ptx::mma_f16(d, ad + (uint64_t)(kk * 128), bd + (uint64_t)((kk / 4) * bstep + (kk % 4) * 2),
                 idesc, (kk > 0 || accumulate_first) ? 1u : 0u);
}

template <bool ZRANK, bool TOPK>
__global__ void __launch_bounds__(kThreads, 1)
chain_dense(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_z,
            const DenseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* s_w2 = smem;
  uint8_t* s_z = s_w2 + (size_t)a.stages * a.stage;
  uint8_t* s_u = s_z + (size_t)kZStages * kZStage;
  float* s_bv = (float*)(s_u + (size_t)a.kb_count * a.u_kb_bytes);   // [8][32]
  int* s_bi = (int*)(s_bv + kEpiWarps * 32);                           // [8][32]
  float* s_zb = (float*)(s_bi + kEpiWarps * 32);                       // [8][32]
  float* s_thv = s_zb + kEpiWarps * 32;                                // [32]
  int32_t* s_prev = (int32_t*)(s_thv + 32);                            // [32]
  int* s_cnt = s_prev + 32;                                            // [32]
  uint64_t* full = (uint64_t*)(((uintptr_t)(s_cnt + 32) + 7) & ~(uintptr_t)7);
  uint64_t* empty = full + a.stages;
  uint64_t* zfull = empty + a.stages;
  uint64_t* zempty = zfull + kZStages;
  uint64_t* acc_full = zempty + kZStages;                              // [2][tmax]
  uint64_t* tmem_free = acc_full + 2 * a.tmax;                         // [2]
  uint64_t* u_ready = tmem_free + 2;
  uint64_t* drain = u_ready + 1;
  uint32_t* tmem_slot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  volatile int* s_decision = abort_flag + 1;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int G = gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kZStages; ++s) {
      ptx::mbar_init(&zfull[s], 1);
      ptx::mbar_init(&zempty[s], kEpiWarps);      // every epilogue warp reads every tile
    }
    for (int q = 0; q < 2 * a.tmax; ++q) ptx::mbar_init(&acc_full[q], 1);
    ptx::mbar_init(&tmem_free[0], 1);
    ptx::mbar_init(&tmem_free[1], 1);
    ptx::mbar_init(u_ready, 1);
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kZWarp && lane == 0) ptx::tma_prefetch_desc(&tm_z);
  if (warp == kW2Warp && lane == 0) ptx::tma_prefetch_desc(&tm_w2);
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
  // TMEM columns of slot s's tile lt: buffer (s & 1) when two slots fit, else buffer 0
  auto col_of = [&](int s, int lt) -> uint32_t {
    return (uint32_t)(((a.dbuf ? (s & 1) : 0) * a.tmax + lt) * a.n_mma);
  };

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(a.err, kErrTimeout);
  };

  if (warp == kW2Warp || warp == kW2Warp + 1) {
    // ---------------------------------------------------------- markov_w2 producers
    // Producer j loads the stages of even (j = 0) or odd (j = 1) iteration numbers.
    // A stage is 2 x (ks / 128) boxes of 128 K-rows x 64 columns (16 KB), one per lane:
    // several issuing threads keep more boxes in flight than one.
    {
      const uint32_t j = (uint32_t)(warp - kW2Warp);
      const uint32_t per_slot = (uint32_t)(nt * a.kstages);
      const uint32_t total = per_slot * (uint32_t)a.N;
      const int nbox = 2 * (a.ks / 128);
      uint32_t it = j, issued_last = 0;
      bool ok = true, any = false;
      for (; ok && it < total; it += 2) {
        const uint32_t s = it % a.stages, ph = (it / a.stages) & 1;
        // (every lane waits: a warp whose lanes sit diverged in a wait slows the warp
        // collectives of the whole SM)
        const bool w_ok =
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait_sleep(&empty[s], ph ^ 1, kWaitBudget, abort_flag));
        if (w_ok && lane == 0) ptx::mbar_arrive_expect_tx(&full[s], a.stage);
        __syncwarp();
        if (!w_ok) {
          ok = false;
          break;
        }
        const uint32_t w = it % per_slot;
        const int t = t_begin + (int)(w / a.kstages), kst = (int)(w % a.kstages);
        if (lane < nbox) {
          const int half = lane & 1, kq = lane >> 1;        // column half, 128-row block
          uint8_t* dst = s_w2 + (size_t)s * a.stage + half * a.box + kq * 16384;
          ptx::tma_load_2d(dst, &tm_w2, &full[s], t * kTileV + half * 64, kst * a.ks + kq * 128);
        }
        issued_last = it;
        any = true;
      }
      if (!ok && lane == 0) {
        give_up();
        // the copies of this producer still in flight (among the last `stages` issued)
        // land before the CTA winds down
        if (any) {
          const uint32_t lo =
              issued_last + 1 > (uint32_t)a.stages ? issued_last + 1 - a.stages : 0;
          for (uint32_t i2 = lo; i2 <= issued_last; ++i2)
            if ((i2 & 1) == j)
              ptx::mbar_wait_sleep(&full[i2 % a.stages], (i2 / a.stages) & 1, kWaitBudget, nullptr);
        }
      }
    }
  } else if (warp == kZWarp) {
    // ---------------------------------------------------------- base-logit producer
    // (all lanes run the loop in step; lane 0 issues)
    {
      const uint32_t total = (uint32_t)(nt * a.N);
      const uint64_t z_policy = ptx::l2_policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (; ok && it < total; ++it) {
        const uint32_t s = it % kZStages, ph = (it / kZStages) & 1;
        if (!__all_sync(0xFFFFFFFFu,
                        ptx::mbar_wait_sleep(&zempty[s], ph ^ 1, kWaitBudget, abort_flag))) {
          ok = false;
          break;
        }
        const int slot = (int)(it / nt), t = t_begin + (int)(it % nt);
        if (lane == 0) {
          // (each tile of z is read once: its lines go first, so that markov_w2, read
          // again every slot, keeps its place in L2)
          ptx::mbar_arrive_expect_tx(&zfull[s], kZStage);
          ptx::tma_load_2d_hint(s_z + (size_t)s * kZStage, &tm_z, &zfull[s], a.b0,
                                (int)((size_t)slot * a.Vhp) + t * kTileV, z_policy);
        }
        __syncwarp();
      }
      if (!ok && lane == 0) {
        give_up();
        const uint32_t first = it > (uint32_t)kZStages ? it - kZStages : 0;
        for (uint32_t q = first; q < it; ++q)
          ptx::mbar_wait_sleep(&zfull[q % kZStages], (q / kZStages) & 1, kWaitBudget, nullptr);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    // (all lanes run the loop in step and wait together; lane 0 issues)
    {
      const uint32_t idesc = ptx::idesc_bf16_f32(kTileV, a.n_mma, /*A MN-major*/ 1, 0);
      const uint32_t u0 = ptx::smem_u32(s_u);
      const uint32_t bstep = a.u_kb_bytes >> 4;          // u's 64-K blocks, in 16-byte units
      uint32_t s_it = 0, ph_it = 0;                      // ring position of the next stage
      bool ok = true;
      for (int step = 0; ok && step < a.N; ++step) {
        if (!__all_sync(0xFFFFFFFFu,
                        ptx::mbar_wait_sleep(u_ready, step & 1, kWaitBudget, abort_flag))) {
          ok = false;
          break;
        }
        const int buf = a.dbuf ? (step & 1) : 0;
        const int use = a.dbuf ? (step >> 1) : step;
        if (use > 0 && !__all_sync(0xFFFFFFFFu, ptx::mbar_wait_sleep(&tmem_free[buf], (use - 1) & 1,
                                                                      kWaitBudget, abort_flag))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (int lt = 0; ok && lt < nt; ++lt) {
          const uint32_t d = tmem + col_of(step, lt);
          for (int kst = 0; kst < a.kstages; ++kst) {
            if (!__all_sync(0xFFFFFFFFu,
                            ptx::mbar_wait_sleep(&full[s_it], ph_it, kWaitBudget, abort_flag))) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            if (lane == 0) {
              // the stage's MMAs as one straight run from two base descriptors (the tensor
              // pipe queues only a little ahead of this thread, so per-MMA work idles it)
              const uint64_t ad = ptx::desc_mnmajor_sw128(
                  ptx::smem_u32(s_w2 + (size_t)s_it * a.stage), a.box, 1024);
              const uint64_t bd =
                  ptx::desc_kmajor_sw128(u0 + (uint32_t)(kst * (a.ks / 64)) * a.u_kb_bytes);
              if (a.ks == 256)
                mma_run<16>(d, ad, bd, bstep, idesc, kst != 0);
              else
                mma_run<8>(d, ad, bd, bstep, idesc, kst != 0);
              ptx::mma_commit(&empty[s_it]);
            }
            __syncwarp();
            if (++s_it == (uint32_t)a.stages) {
              s_it = 0;
              ph_it ^= 1u;
            }
          }
          if (ok && lane == 0) ptx::mma_commit(&acc_full[(a.dbuf ? (step & 1) : 0) * a.tmax + lt]);
          __syncwarp();
        }
      }
      if (!ok && lane == 0) give_up();
      if (lane == 0) {
        ptx::mma_commit(drain);
        ptx::mbar_wait_sleep(drain, 0, kWaitBudget, nullptr);
      }
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int tid = threadIdx.x;                    // 0..255
    const int quad = warp % 4;                      // TMEM lane quadrant
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int row = quad * 32 + lane;               // row of the tile this thread owns
    // the blocks (TMEM columns) of this warp: one half of the MMA's N, 16 or 8 of them
    const int ncw = a.n_mma / 2, c0w = (warp / 4) * ncw;

    // u = markov_w1[prev] for the group's blocks into the swizzled K-major B operand
    // (zero past r and past the group's blocks); prev from s_prev
    auto gather_u = [&]() {
      const int per_row = a.kb_count * 8;             // 16-byte chunks of one row of u
      const int chunks = a.n_mma * per_row;
      for (int base = 0; base < chunks; base += 4 * kEpiThreads) {
        uint4 val[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int idx = base + q * kEpiThreads + tid;
          val[q] = make_uint4(0, 0, 0, 0);
          const int n = idx / per_row, rem = idx % per_row;
          if (idx < chunks && n < a.Bg) {
            const int k0 = (rem / 8) * 64 + (rem % 8) * 8;
            const __nv_bfloat16* src = a.w1 + (size_t)s_prev[n] * a.r + k0;
            if ((a.r & 7) == 0 && k0 + 8 <= a.r) {
              val[q] = __ldg(reinterpret_cast<const uint4*>(src));
            } else if (k0 < a.r) {                     // ragged rank: element-wise
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
      fence_proxy_async();                            // (the MMA reads u through the
      epi_sync();                                     //  async proxy)
      if (tid == 0) ptx::mbar_arrive(u_ready);
    };
    // the previous tokens of slot `step`: the anchors, or the winners of slot step - 1
    // (which block 0 also writes out as that slot's draft)
    auto load_prev = [&](int step) {
      if (tid < a.Bg) {
        int p;
        if (step == 0) {
          p = a.anchors[a.b0 + tid];
        } else {
          const unsigned long long key = __ldcg(&a.keys[(size_t)(step - 1) * a.B + a.b0 + tid]);
          const int hrow = key_id(key);
          p = a.d2t ? a.d2t[hrow] : hrow;
          if (blockIdx.x == 0) {
            const size_t o = (size_t)(a.b0 + tid) * a.N + step - 1;
            a.draft[o] = p;
            if (a.topk_ids) a.topk_ids[o] = p;
            if (a.topk_vals) a.topk_vals[o] = key_value(key);
          }
        }
        if (p < 0 || p >= a.V) {
          flag_error(a.err, kErrBadToken);
          p = 0;
        }
        s_prev[tid] = p;
      }
      epi_sync();
    };

    // Bound of each block's top k for slot `step`: the k-th largest of its nb bucket
    // maxima (an empty bucket reads as -inf).  One warp per block, lane j ranks bucket j
    // (ties by index); a warp's four blocks load their buckets together.
    constexpr int kPer = 32 / kEpiWarps;
    auto load_bound = [&](int step, uint32_t (&kb)[kPer]) {
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int c = warp + q * kEpiWarps;
        const size_t sb = (size_t)step * a.B + a.b0 + c;
        kb[q] = (c < a.Bg && lane < a.nb) ? __ldcg(&a.bucket[sb * kDenseBuckets + lane]) : 0u;
      }
    };
    auto rank_bound = [&](const uint32_t (&kb)[kPer]) {
      // (the warp's blocks ranked together and nb even: 2 x kPer independent shuffles
      // in flight per step)
      int rank[kPer];
#pragma unroll
      for (int q = 0; q < kPer; ++q) rank[q] = 0;
      for (int h = 0; h < a.nb; h += 2) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
#pragma unroll
          for (int q = 0; q < kPer; ++q) {
            const uint32_t y = __shfl_sync(0xFFFFFFFFu, kb[q], h + e);
            rank[q] += (y > kb[q]) | ((y == kb[q]) & (h + e < lane));
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const int c = warp + q * kEpiWarps;
        if (c < a.Bg && lane < a.nb && rank[q] == a.k - 1)
          s_thv[c] = kb[q] == 0u ? -INFINITY : order_key32_value((int)(kb[q] ^ 0x80000000u));
      }
    };
    // The rows of tile lt of slot `step` at or above their block's bound (in s_thv) go
    // to this CTA's list of the block: a few over the whole grid.
    auto scan_tile = [&](int step, int lt) {
      const int v = (t_begin + lt) * kTileV + row;
      const uint32_t taddr = tmem + lane_base + col_of(step, lt);
      for (int c0 = c0w; c0 < c0w + ncw && c0 < a.Bg; c0 += 8) {
        uint32_t r[8];
        __syncwarp();                                     // (after the divergent appends)
        ptx::tmem_ld_32x32b_x8(taddr + c0, r);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float x = __uint_as_float(r[j]);
          if (v < a.Vh && c0 + j < a.Bg && x >= s_thv[c0 + j]) {
            // a place in this CTA's list (shared-memory counter), then plain stores:
            // nothing waits on the memory system while markov_w2 streams
            const int e = atomicAdd(&s_cnt[c0 + j], 1);
            if (e < kDenseLocal) {
              const size_t o =
                  (((size_t)step * a.B + a.b0 + c0 + j) * G + blockIdx.x) * kDenseLocal + e;
              a.cand_val[o] = x;
              a.cand_id[o] = v;
            }
          }
        }
      }
      __syncwarp();
    };
    // After a slot's scan: this CTA's count of each block's candidates (more than
    // kDenseLocal: its list overflowed), and the counters restart.  (After an epi_sync.)
    auto publish_counts = [&](int step) {
      if (tid < a.Bg) {
        a.cand_cnt[((size_t)step * a.B + a.b0 + tid) * G + blockIdx.x] = s_cnt[tid];
        s_cnt[tid] = 0;
      }
    };
    // With two TMEM buffers, slot s's scan runs inside slot s + 1's first pass, tile by
    // tile, before each tile's wait for its MMA; with one it runs after the barrier.
    const bool fuse = TOPK && a.dbuf;

    bool ok = true;
    if (tid < 32) s_cnt[tid] = 0;
    load_prev(0);
    gather_u();
    for (int step = 0; ok && step < a.N; ++step) {
      const int buf = a.dbuf ? (step & 1) : 0;
      const int use = a.dbuf ? (step >> 1) : step;
      // -------- 3. pass 1: z' = z + m (back into TMEM for the top-k pass).  Every warp
      //            takes every tile: its TMEM lane quadrant (32 rows) and its half of the
      //            blocks, so a tile's work is spread over all eight warps.  Each thread
      //            keeps, per block, the best of its own rows over the slot's tiles (the
      //            value and the tile); the warp's 32 rows are reduced once, after the
      //            last tile, so a tile costs no cross-lane work.  (Compared as floats:
      //            -0 and +0 are equal, as they are as values; the value published is
      //            canonical.)
      float bx[16];                                       // best z' of block c0w + j, or -inf
      uint32_t btile[4];                                  // its tile: byte j % 4 of word j / 4
#pragma unroll
      for (int j = 0; j < 16; ++j) bx[j] = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q) btile[q] = 0u;
      if (ZRANK) {
        if (lane < ncw) s_zb[quad * 32 + c0w + lane] = -INFINITY;
        __syncwarp();
      }
      const bool wide = ncw == 16;                        // (else 8 blocks per warp)
      const int nblk = min(ncw, a.Bg - c0w);              // this warp's blocks in the group
      const uint32_t blk_mask = nblk > 0 ? (nblk >= 32 ? ~0u : (1u << nblk) - 1u) : 0u;
      for (int lt = 0; lt < nt; ++lt) {
        const int v = (t_begin + lt) * kTileV + row;
        const bool v_ok = v < a.Vh;
        const bool scan_prev = fuse && step > 0;
        uint32_t rp[16];                                  // the previous slot's z' (fused scan)
        if (scan_prev) {
          const uint32_t pa = tmem + lane_base + col_of(step - 1, lt) + c0w;
          __syncwarp();
          if (wide)
            ptx::tmem_ld_32x32b_x16(pa, rp);
          else
            ptx::tmem_ld_32x32b_x8(pa, *reinterpret_cast<uint32_t(*)[8]>(&rp[0]));
        }
        const uint32_t zit = (uint32_t)(step * nt + lt);
        const uint32_t zs = zit % kZStages, zph = (zit / kZStages) & 1;
        bool w_ok = ptx::mbar_wait_sleep(&zfull[zs], zph, kWaitBudget, abort_flag);
        w_ok = w_ok && ptx::mbar_wait_sleep(&acc_full[buf * a.tmax + lt], use & 1, kWaitBudget,
                                            abort_flag);
        ok = __all_sync(0xFFFFFFFFu, w_ok);
        if (!ok) {
          ptx::tmem_ld_wait();
          break;
        }
        ptx::tc_fence_after();
        const uint32_t taddr = tmem + lane_base + col_of(step, lt) + c0w;
        uint32_t r[16];                                   // this slot's Markov terms
        if (wide)
          ptx::tmem_ld_32x32b_x16(taddr, r);
        else
          ptx::tmem_ld_32x32b_x8(taddr, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
        const uint8_t* zrow = s_z + (size_t)zs * kZStage + (size_t)row * 128;
        float zv[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {                     // 16-byte chunk c0w / 4 + q of the
          if (q >= 2 && !wide) break;                     // row, swizzled
          const int ch = c0w / 4 + q;
          const float4 f = *reinterpret_cast<const float4*>(zrow + ((ch ^ (row & 7)) << 4));
          zv[4 * q] = f.x;
          zv[4 * q + 1] = f.y;
          zv[4 * q + 2] = f.z;
          zv[4 * q + 3] = f.w;
        }
        ptx::tmem_ld_wait();
        // the previous slot's candidates of this tile: rows at or above their block's
        // bound.  The bounds are read first and the hits found without a branch, so that
        // nothing serialises the loop; hits themselves are rare.
        if (scan_prev) {
          uint32_t hit = 0;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q >= 2 && !wide) break;
            const float4 t4 = *reinterpret_cast<const float4*>(s_thv + c0w + 4 * q);
            hit |= (__uint_as_float(rp[4 * q]) >= t4.x ? 1u : 0u) << (4 * q);
            hit |= (__uint_as_float(rp[4 * q + 1]) >= t4.y ? 1u : 0u) << (4 * q + 1);
            hit |= (__uint_as_float(rp[4 * q + 2]) >= t4.z ? 1u : 0u) << (4 * q + 2);
            hit |= (__uint_as_float(rp[4 * q + 3]) >= t4.w ? 1u : 0u) << (4 * q + 3);
          }
          hit &= v_ok ? blk_mask : 0u;
          while (hit) {
            const int j = __ffs(hit) - 1;
            hit &= hit - 1;
            uint32_t xb = rp[0];
#pragma unroll
            for (int q = 1; q < 16; ++q) xb = j == q ? rp[q] : xb;
            const int c = c0w + j;
            const int e = atomicAdd(&s_cnt[c], 1);
            if (e < kDenseLocal) {
              const size_t o =
                  (((size_t)(step - 1) * a.B + a.b0 + c) * G + blockIdx.x) * kDenseLocal + e;
              a.cand_val[o] = __uint_as_float(xb);
              a.cand_id[o] = v;
            }
          }
        }
        __syncwarp();
        if (a.logits && v_ok) {                           // (tests only)
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (j < ncw && c0w + j < a.Bg)
              a.logits[((size_t)(a.b0 + c0w + j) * a.N + step) * a.Vh + v] =
                  zv[j] + __uint_as_float(r[j]);
        }
        // z' = z + m (or -inf past the head), back into r for the top-k scan, and the
        // thread's running best of each block (strict: on equal values the earlier tile,
        // the lower row, stays)
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j >= 8 && !wide) break;
          const float x = v_ok ? zv[j] + __uint_as_float(r[j]) : -INFINITY;
          if (x > bx[j]) {
            bx[j] = x;
            btile[j / 4] = (btile[j / 4] & ~(0xFFu << (8 * (j % 4)))) |
                           ((uint32_t)lt << (8 * (j % 4)));
          }
          r[j] = __float_as_uint(ZRANK ? (v_ok ? zv[j] : -INFINITY) : x);
        }
        if (ZRANK) {                                      // the largest base logit of each
          float mzv = -INFINITY;                          // block over the warp's rows
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j >= 8 && !wide) break;
            const int mz = __reduce_max_sync(0xFFFFFFFFu, order_key32(v_ok ? zv[j] : -INFINITY));
            if (lane == j) mzv = order_key32_value(mz);
          }
          if (lane < ncw)
            s_zb[quad * 32 + c0w + lane] = fmaxf(s_zb[quad * 32 + c0w + lane], mzv);
        }
        __syncwarp();
        if (TOPK) {
          if (wide)
            ptx::tmem_st_32x32b_x16(taddr, r);
          else
            ptx::tmem_st_32x32b_x8(taddr, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
          ptx::tmem_st_wait();
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&zempty[zs]);
      }
      // the warp's best of each of its blocks over its 32 rows: a transposing butterfly
      // on (value, row) pairs over lane bits 3..0, halving the blocks a lane holds at each
      // step, then one plain step over bit 4; lanes j and j + 16 end with block c0w + j
      // (on equal values the lower row wins)
      if (ok) {
        float key[16];
        int rw[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = (int)((btile[j / 4] >> (8 * (j % 4))) & 0xFFu);
          key[j] = bx[j];
          rw[j] = bx[j] == -INFINITY ? 0x7FFFFFFF : (t_begin + t) * kTileV + row;
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int i = 0; i < o; ++i) {
            const float send_k = upper ? key[i] : key[i + o];
            const int send_r = upper ? rw[i] : rw[i + o];
            const float keep_k = upper ? key[i + o] : key[i];
            const int keep_r = upper ? rw[i + o] : rw[i];
            const float got_k = __shfl_xor_sync(0xFFFFFFFFu, send_k, o);
            const int got_r = __shfl_xor_sync(0xFFFFFFFFu, send_r, o);
            const bool take = got_k > keep_k || (got_k == keep_k && got_r < keep_r);
            key[i] = take ? got_k : keep_k;
            rw[i] = take ? got_r : keep_r;
          }
        }
        {
          const float got_k = __shfl_xor_sync(0xFFFFFFFFu, key[0], 16);
          const int got_r = __shfl_xor_sync(0xFFFFFFFFu, rw[0], 16);
          if (got_k > key[0] || (got_k == key[0] && got_r < rw[0])) {
            key[0] = got_k;
            rw[0] = got_r;
          }
        }
        if (lane < ncw) {
          s_bv[quad * 32 + c0w + lane] = canon(key[0]);
          s_bi[quad * 32 + c0w + lane] = rw[0];
        }
      }
      // a warp that gave up raises the flag; the others then stop waiting, and all take
      // the same decision here (the named barriers below need every epilogue thread)
      if (!ok) give_up();
      if (epi_agree_abort(abort_flag, s_decision, tid)) {
        ok = false;
        break;
      }
      // -------- 4. argmax: the warps' bests (in shared memory), then the grid
      ptx::tc_fence_before();
      epi_sync();
      // (fused: every warp has scanned the previous slot's TMEM columns; they are free)
      if (fuse && step > 0) {
        if (tid == 0) ptx::mbar_arrive(&tmem_free[(step - 1) & 1]);
        publish_counts(step - 1);
      }
      if (tid < a.Bg) {
        float bv = s_bv[tid];
        int bi = s_bi[tid];
        float bz = ZRANK ? s_zb[tid] : 0.f;
#pragma unroll
        for (int q = 1; q < 4; ++q) {                     // the four lane quadrants
          if (better(s_bv[q * 32 + tid], s_bi[q * 32 + tid], bv, bi)) {
            bv = s_bv[q * 32 + tid];
            bi = s_bi[q * 32 + tid];
          }
          if (ZRANK) bz = fmaxf(bz, s_zb[q * 32 + tid]);
        }
        const size_t sb = (size_t)step * a.B + a.b0 + tid;
        if (bi != 0x7FFFFFFF) atomicMax(&a.keys[sb], order_key(canon(bv), bi));
        // this CTA's best ranked value of the block: a distinct element per CTA, so the
        // bucket maxima are distinct elements too
        if (TOPK)
          atomicMax(&a.bucket[sb * kDenseBuckets + blockIdx.x % a.nb],
                    (uint32_t)order_key32(canon(ZRANK ? bz : bv)) ^ 0x80000000u);
        // arrive on the grid barrier; the release orders this thread's atomics first
        red_release_add(a.bar, 1u);
        // the markov_w1 row of this CTA's best: the next slot gathers one of the G such
        // rows of the block, so each is brought into L2 while the grid meets
        if (bi != 0x7FFFFFFF && step + 1 < a.N) {
          const int p = a.d2t ? __ldg(a.d2t + bi) : bi;
          if (p >= 0 && p < a.V) {
            const char* src = reinterpret_cast<const char*>(a.w1 + (size_t)p * a.r);
            for (int o = 0; o < a.r * 2; o += 128) ptx::prefetch_l2(src + o);
          }
        }
      }
      // -------- 5. the grid barrier: every CTA has published this slot's winners.
      //            (Warp 0 polls with all its lanes, in step.)
      if (warp == 0) {
        const unsigned target = (unsigned)(step + 1) * (unsigned)G * (unsigned)a.Bg;
        const long long t0 = clock64();
        while (__all_sync(0xFFFFFFFFu, ld_acquire(a.bar) < target)) {
          if (__any_sync(0xFFFFFFFFu, clock64() - t0 > kWaitBudget)) {
            if (lane == 0) give_up();
            break;
          }
          __nanosleep(32);
        }
      }
      if (epi_agree_abort(abort_flag, s_decision, tid)) {
        ok = false;
        break;
      }
      // -------- 6. the next slot's previous tokens and u: its MMAs start.  (This slot's
      //            bucket maxima are loaded first, while the memory system is quiet.)
      uint32_t kb[kPer];
      if (TOPK) load_bound(step, kb);
      load_prev(step + 1);
      if (step + 1 < a.N) gather_u();
      // -------- 7. this slot's top-k scan: fused into the next slot's first pass, or
      //            here when TMEM holds one slot
      if (TOPK) {
        rank_bound(kb);
        epi_sync();
        if (!fuse || step + 1 == a.N) {
          for (int lt = 0; lt < nt; ++lt) scan_tile(step, lt);
          epi_sync();
          publish_counts(step);
        }
      }
      if (!fuse) {
        // this slot's TMEM columns are free for the MMA of a later slot
        __syncwarp();
        ptx::tc_fence_before();
        epi_sync();
        if (tid == 0) ptx::mbar_arrive(&tmem_free[buf]);
      }
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

// The top-k of every (slot, block), one CTA each, from the dense chain's candidate list:
// every row at or above a lower bound of the k-th largest ranked value, so the list holds
// the top k.  Sorted by (value descending, id ascending); a list that overflowed is
// replaced by an exact evaluation of every head row of that slot and block.
struct FinalArgs {
  const float* cand_val;            // [N][B][G][kDenseLocal]
  const int32_t* cand_id;
  const int32_t* cand_cnt;          // [N][B][G]
  const unsigned long long* keys;   // [N][B] winners (previous tokens of the recompute)
  const int32_t* anchors;
  const int32_t* d2t;
  const float* z;                   // base logits [N][Vhp][ldb]
  const __nv_bfloat16* w1;
  const __nv_bfloat16* w2;          // [r][Vh]
  int32_t* ids;
  float* vals;
  uint32_t* err;
  size_t Vhp, ldb;
  int B, N, V, Vh, r, k, zrank, G;
};

constexpr int kFinalThreads = 256;

__global__ void __launch_bounds__(kFinalThreads)
topk_final(const FinalArgs a) {
  const int i = blockIdx.x / a.B, b = blockIdx.x % a.B;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const size_t sb = (size_t)i * a.B + b;
  __shared__ float s_v[kDenseCap];
  __shared__ int s_i[kDenseCap];
  __shared__ float s_wv[kFinalThreads / 32];
  __shared__ int s_wi[kFinalThreads / 32];
  __shared__ float s_u[512];
  __shared__ int s_n, s_over;
  auto out = [&](int q, float v, int id) {
    const size_t o = ((size_t)b * a.N + i) * a.k + q;
    const int hrow = (id >= 0 && id < a.Vh) ? id : 0;
    if (a.ids) a.ids[o] = a.d2t ? a.d2t[hrow] : hrow;
    if (a.vals) a.vals[o] = v;
  };
  if (tid == 0) {
    s_n = 0;
    s_over = 0;
  }
  __syncthreads();
  // the CTAs' lists of this slot and block, gathered into one (thread t: CTA t)
  for (int t = tid; t < a.G; t += kFinalThreads) {
    const int n = a.cand_cnt[sb * a.G + t];
    if (n > kDenseLocal) s_over = 1;
    for (int e = 0; e < min(n, kDenseLocal); ++e) {
      const int pos = atomicAdd(&s_n, 1);
      if (pos < kDenseCap) {
        s_v[pos] = a.cand_val[(sb * a.G + t) * kDenseLocal + e];
        s_i[pos] = a.cand_id[(sb * a.G + t) * kDenseLocal + e];
      } else {
        s_over = 1;
      }
    }
  }
  __syncthreads();
  if (!s_over) {
    if (warp != 0) return;
    const int n = s_n;
    // k rounds of a warp-wide best strictly after the previous pick
    float pv = 0.f;
    int pid = 0;
    for (int q = 0; q < a.k; ++q) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
      for (int e = lane; e < n; e += 32)
        if ((q == 0 || better(pv, pid, s_v[e], s_i[e])) && better(s_v[e], s_i[e], bv, bi)) {
          bv = s_v[e];
          bi = s_i[e];
        }
      warp_best(bv, bi);
      if (lane == 0) out(q, bv, bi);
      pv = bv;
      pid = bi;
    }
    return;
  }
  // overflow: every head row of this slot and block, exactly as the chain evaluates it
  if (tid == 0) atomicAdd(a.err + kCtrlDenseOver, 1u);
  int prev;
  if (i == 0) {
    prev = a.anchors[b];
  } else {
    const int hrow = key_id(a.keys[(size_t)(i - 1) * a.B + b]);
    prev = a.d2t ? a.d2t[hrow] : hrow;
  }
  if (prev < 0 || prev >= a.V) {
    if (tid == 0) flag_error(a.err, kErrBadToken);
    prev = 0;
  }
  for (int k = tid; k < a.r; k += kFinalThreads)
    s_u[k] = __bfloat162float(a.w1[(size_t)prev * a.r + k]);
  __syncthreads();
  // each thread's best k (sorted) over its rows, then k rounds of a CTA-wide best
  constexpr int KM = 32;
  float lv[KM];
  int li[KM];
  for (int q = 0; q < KM; ++q) {
    lv[q] = -INFINITY;
    li[q] = 0x7FFFFFFF;
  }
  for (int v = tid; v < a.Vh; v += kFinalThreads) {
    const float z = a.z[((size_t)i * a.Vhp + v) * a.ldb + b];
    float m = 0.f;
    for (int k = 0; k < a.r; ++k)
      m = fmaf(s_u[k], __bfloat162float(a.w2[(size_t)k * a.Vh + v]), m);
    float x = a.zrank ? z : z + m;
    int xi = v;
    for (int q = 0; q < a.k; ++q)
      if (better(x, xi, lv[q], li[q])) {
        const float tv = lv[q];
        const int ti = li[q];
        lv[q] = x;
        li[q] = xi;
        x = tv;
        xi = ti;
      }
  }
  int head = 0;
  for (int q = 0; q < a.k; ++q) {
    float bv = head < a.k ? lv[head] : -INFINITY;
    int bi = head < a.k ? li[head] : 0x7FFFFFFF;
    warp_best(bv, bi);
    if (lane == 0) {
      s_wv[warp] = bv;
      s_wi[warp] = bi;
    }
    __syncthreads();
    if (warp == 0) {
      float cv = lane < kFinalThreads / 32 ? s_wv[lane] : -INFINITY;
      int ci = lane < kFinalThreads / 32 ? s_wi[lane] : 0x7FFFFFFF;
      warp_best(cv, ci);
      if (lane == 0) {
        out(q, cv, ci);
        s_wi[0] = ci;
      }
    }
    __syncthreads();
    if (head < a.k && li[head] == s_wi[0]) ++head;   // the winner's thread moves on
    __syncthreads();
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

template <bool ZRANK, bool TOPK>
cudaError_t launch_dense_inst(const CUtensorMap& tw, const CUtensorMap& tz, const DenseArgs& a,
                              int grid, size_t smem, cudaStream_t stream) {
  auto kern = chain_dense<ZRANK, TOPK>;
  int per_sm = 0;
  cudaError_t e = blocks_per_sm(reinterpret_cast<const void*>(kern), kThreads, smem, &per_sm);
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
  return cudaLaunchKernelEx(&cfg, kern, tw, tz, a);
}

}  // namespace

// Blocks per launch of the dense chain for this vocabulary: 32, or 16 when the Markov
// terms of 32 blocks over a CTA's tiles would not fit TMEM; 0 when neither fits.
int dense_chain_group(int Vh, int sms) {
  const int tiles = (Vh + kTileV - 1) / kTileV;
  const int grid = std::max(1, std::min({sms, tiles, kChainMaxCtas}));
  const int tmax = (tiles + grid - 1) / grid;
  if (tmax * 32 <= 512) return 32;
  if (tmax * 16 <= 512) return 16;
  return 0;
}

cudaError_t launch_chain_dense(const ProposePlan& p) {
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  int sms = 0;
  const cudaError_t es = device_sms(&sms);
  if (es != cudaSuccess) return es;
  const int tiles = (p.Vh + kTileV - 1) / kTileV;
  const int grid = std::max(1, std::min({sms, tiles, kChainMaxCtas}));
  const int tmax = (tiles + grid - 1) / grid;
  const int group = dense_chain_group(p.Vh, sms);
  if (group == 0) return cudaErrorNotSupported;
  const bool want_topk = p.topk_ids || p.topk_vals;
  const bool zrank = want_topk && !p.topk_markov;
  // with k = 1 over the corrected logits the top-1 is the argmax: written with the draft
  const bool topk_pass = want_topk && (p.k > 1 || zrank);

  // markov_w2 stages of 256 K-rows (a whole 128-row tile of a rank-256 head: 64 KB), or
  // 128 when the rank is at most 128.  Each stage costs one mbarrier round trip between
  // the TMA and the MMA whatever its size, so the stages are as large as the rank allows.
  const int ks = p.r <= 128 ? 128 : 256;
  CUtensorMap tw, tz;
  {
    cuuint64_t dims[2] = {(cuuint64_t)p.Vh, (cuuint64_t)p.r};
    cuuint64_t strides[1] = {(cuuint64_t)p.Vh * 2};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)p.w2, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // base logits z[N][Vhp][ldb] as a 2-D array of N * Vhp rows of ldb floats; a box is
    // one tile's 128 rows x 32 blocks (columns past ldb read as zero and are unused)
    cuuint64_t dims[2] = {(cuuint64_t)p.ldb, (cuuint64_t)p.N * p.Vhp};
    cuuint64_t strides[1] = {(cuuint64_t)p.ldb * 4};
    cuuint32_t box[2] = {32, kTileV};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tz, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void*)p.z, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  for (int b0 = 0; b0 < p.B; b0 += group) {
    DenseArgs a{};
    a.w1 = (const __nv_bfloat16*)p.w1;
    a.anchors = p.anchors;
    a.d2t = p.d2t;
    a.draft = p.draft;
    a.topk_ids = (want_topk && !topk_pass) ? p.topk_ids : nullptr;
    a.topk_vals = (want_topk && !topk_pass) ? p.topk_vals : nullptr;
    a.logits = p.logits;
    a.cand_val = p.cand_val;
    a.cand_id = p.cand_id;
    a.cand_cnt = p.cand_cnt;
    a.bucket = p.bucket;
    a.keys = p.keys;
    a.bar = p.bar + b0 / 16;
    a.err = p.ctrl;
    a.Vhp = p.Vhp;
    a.B = p.B;
    a.b0 = b0;
    a.Bg = std::min(group, p.B - b0);
    a.N = p.N;
    a.V = p.V;
    a.Vh = p.Vh;
    a.r = p.r;
    a.k = p.k;
    a.n_mma = a.Bg <= 16 ? 16 : 32;
    a.ks = ks;
    a.box = 64u * ks * 2;
    a.stage = 2 * a.box;
    a.kstages = (p.r + ks - 1) / ks;
    a.kb_count = a.kstages * (ks / 64);
    a.tiles = tiles;
    a.tmax = tmax;
    a.dbuf = 2 * tmax * a.n_mma <= 512 ? 1 : 0;
    uint32_t cols = 32;
    while (cols < (uint32_t)((a.dbuf ? 2 : 1) * tmax * a.n_mma)) cols <<= 1;
    a.tmem_cols = cols;
    a.u_kb_bytes = (uint32_t)a.n_mma * 128;
    a.nb = std::min(kDenseBuckets, std::max(2, 2 * p.k));
    // s_bv, s_bi, s_zb, s_thv, s_prev, s_cnt; then the barriers and four words
    const size_t misc = (size_t)3 * kEpiWarps * 32 * 4 + 3 * 32 * 4 + 8 +
                        8 * ((size_t)2 * 4 + 2 * kZStages + 2 * tmax + 4) + 16;
    const size_t fixed = 1024 + (size_t)kZStages * kZStage +
                         (size_t)a.kb_count * a.u_kb_bytes + misc;
    const size_t budget = 225 * 1024;
    if (fixed + 2 * a.stage > budget) return cudaErrorInvalidConfiguration;
    a.stages = (int)std::min<size_t>(4, (budget - fixed) / a.stage);
    const size_t smem = fixed + (size_t)a.stages * a.stage;
    cudaError_t e;
    if (topk_pass)
      e = zrank ? launch_dense_inst<true, true>(tw, tz, a, grid, smem, p.stream)
                : launch_dense_inst<false, true>(tw, tz, a, grid, smem, p.stream);
    else
      e = launch_dense_inst<false, false>(tw, tz, a, grid, smem, p.stream);
    if (e != cudaSuccess) return e;
  }
  if (topk_pass) {
    FinalArgs f{};
    f.cand_val = p.cand_val;
    f.cand_id = p.cand_id;
    f.cand_cnt = p.cand_cnt;
    f.keys = p.keys;
    f.anchors = p.anchors;
    f.d2t = p.d2t;
    f.z = p.z;
    f.w1 = (const __nv_bfloat16*)p.w1;
    f.w2 = (const __nv_bfloat16*)p.w2;
    f.ids = p.topk_ids;
    f.vals = p.topk_vals;
    f.err = p.ctrl;
    f.Vhp = p.Vhp;
    f.ldb = p.ldb;
    f.B = p.B;
    f.N = p.N;
    f.V = p.V;
    f.Vh = p.Vh;
    f.r = p.r;
    f.k = p.k;
    f.zrank = zrank ? 1 : 0;
    f.G = grid;
    if (p.r > 512) return cudaErrorInvalidValue;
    topk_final<<<p.B * p.N, kFinalThreads, 0, p.stream>>>(f);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace dspark
