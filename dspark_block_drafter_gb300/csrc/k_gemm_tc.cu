// Base logits on the 5th-generation tensor cores (bf16 in, fp32 accumulate in TMEM).
//
//   z[i][v][b] = sum_h hidden[b, ifp + i, h] * lm_head[v, h] + lm_bias[v]
//
// (llama.cpp commit 6fed9f6, "spec: add DSpark speculative decoding": logits(i) of the
// proposal formula.)  A tile is 128 (or, for a CTA pair, 256) head rows by an N-tile of
// Ni slots x BB blocks (blocks fastest, up to 256 prediction rows).  By default the GEMM
// runs "swap-AB": the MMA's M dimension is the head rows and its N dimension the
// prediction rows, so a small batch still fills the instruction.  The pruned chain's
// octet layout of z keeps 8 head rows of one (slot, block) in one 32-byte sector; the
// dense chain's layout keeps the blocks of one (slot, head row) contiguous.
//
// Persistent and warp-specialised, one CTA per SM:
//   warp 4      TMA producer: lm_head tile [128 x 64] and hidden tile [Ni, BB, 64] per
//               K-block (two K-blocks per copy when H allows) into a ring of
//               shared-memory stages (128-byte swizzle)
//   warp 5      MMA issuer: tcgen05.mma (K = 16) per K-block into a TMEM accumulator;
//               tcgen05.commit frees the stage, and the accumulator when the tile ends
//   warps 0-3   epilogue: tcgen05.ld of their 32 TMEM lanes, + bias, fp32 stores of z,
//               per-tile maxima for the pruned chain
// Two TMEM accumulators alternate so that the epilogue of one tile overlaps the MMAs of
// the next.  Tiles are ordered vocabulary-major: CTAs that run side by side share the
// same lm_head tile through L2, so lm_head streams from HBM once.  Single CTAs claim
// their tiles from a counter as they go (a CTA that streams faster takes more of them);
// pairs take every units-th tile.
//
// When a tile's slots split evenly in two, CTAs run in pairs (a cluster of two on one
// TPC) on 256-row tiles with M = 256 MMAs (cta_group::2): each CTA stages its own 128
// lm_head rows and half of the hidden rows, so a pair moves two thirds of the bytes
// through shared memory and L2 that two single CTAs would.  The leader (rank 0) posts
// the byte count of both halves on its own barrier, both CTAs' copies count against it,
// the leader issues the MMAs, and the commits arrive in both CTAs.  A pair whose N-tile
// is exactly 256 prediction rows runs the other way round (PM = 1, see logits_gemm_tc):
// one prediction row per epilogue thread, and tiles of z that cannot reach a slot's top
// k are not stored.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dspark {

namespace {

constexpr int kBlockV = 128;      // MMA M: head rows per tile
constexpr int kBlockK = 64;       // one 128-byte swizzle row of bf16
constexpr uint32_t kStageA = kBlockV * kBlockK * 2;   // 16 KB
constexpr int kThreads = 192;
constexpr int kMaxLiveTiles = 64;     // N-tiles the adaptive block length can leave out
constexpr int kTileRing = 4;          // claimed tile indices in flight (dynamic schedule)
constexpr int kBarBytes = 512;        // shared memory of the barriers and the tile ring
#ifndef DSPARK_GEMM_BUCKET_X
#define DSPARK_GEMM_BUCKET_X 2
#endif
// Per (slot, block) row, the GEMM keeps zbound_k x kBucketX maxima of tile lower bounds
// (when zbound_k <= 8), of which the zbound_k-th largest bounds the threshold.
constexpr int kBucketX = DSPARK_GEMM_BUCKET_X;
constexpr long long kWaitBudget = 2000000000ll;       // ~1 s of SM clocks
#ifndef DSPARK_GEMM_MAX_KPB
#define DSPARK_GEMM_MAX_KPB 2
#endif
constexpr int kMaxKpb = DSPARK_GEMM_MAX_KPB;          // K-blocks per stage, at most

struct GemmArgs {
  float* z;
  size_t Vhp, ldb;
  float* zmax;     // [N][B][zm_tiles] per-tile maxima of z, or NULL
  // Tiles of z that cannot matter (PM = 1 only; zbound_k = 0 stores every tile): see the
  // PM = 1 epilogue.
  uint32_t* zbound;        // [N][NB][B] maxima of tile lower bounds (order keys), NB =
                           // zbound_k x kBucketX for zbound_k <= 8, else zbound_k
  uint8_t* zwritten;       // [N][B][zm_tiles]
  const float* cnmax;      // [zm_tiles] largest markov_w2 column norm of each tile
  const unsigned* w1max;   // largest markov_w1 row norm (float bits)
  const PreparedHeader* prep;  // header of the prepared buffer cnmax and w1max lie in
  PreparedHeader prep_want;    // what it must say (otherwise every tile is stored)
  int zbound_k;
  // Dynamic schedule (CG = 1): after its first tile (unit), a CTA claims tile units + the
  // old value of *tile_ctr, which starts at 0 for the launch; NULL: tile unit + j units.
  unsigned* tile_ctr;
  const int32_t* n_draft;  // [B] cuts computed before the GEMM (adaptive block length), or
                           // NULL: every row is drafted
  int octet;       // z layout: [N][Vhp / 8][ldb][8] (1) or [N][Vhp][ldb] (0)
  const float* bias;
  uint32_t* err;
  int B, N, ifp, Vh;
  int BB, Ni;      // blocks and slots per N-tile
  int n_bt;        // N-tiles along the blocks (the slot index is tile / n_bt)
  int bn_mma;      // MMA N (rows of the B operand per stage), multiple of 16
  int acc_stride;  // TMEM columns between the two accumulators (multiple of 32)
  int kpb;         // 64-wide K-blocks per stage, each loaded operand one copy per stage
  int n_tiles, v_tiles, num_kb, stages;
  int zm_tiles;    // 128-row tiles of the vocabulary (zmax row length)
  uint32_t tmem_cols;
};

// Valid prediction rows of N-tile nt: slots and blocks it covers.
__device__ __forceinline__ void ntile_extent(const GemmArgs& g, int nt, int& i0, int& ni,
                                             int& bb0, int& nb) {
  const int it = nt / g.n_bt, bt = nt % g.n_bt;
  i0 = it * g.Ni;
  ni = min(g.Ni, g.N - i0);
  bb0 = bt * g.BB;
  nb = min(g.BB, g.B - bb0);
}

// CG = 1: one CTA per 128-row tile (cta_group::1).  CG = 2: a cluster of two CTAs
// shares a 256-row tile with M = 256 pair MMAs (cta_group::2): each CTA stages its
// 128 lm_head rows and half of the prediction rows, the leader (rank 0) issues the MMAs,
// and each CTA's TMEM receives its own 128 rows of the result.
//
// PM = 1 (pairs whose N-tile holds exactly 256 prediction rows): the same staged tiles
// enter the MMA the other way round, the prediction rows as M and the pair's 256 lm_head
// rows as N, so that a TMEM lane holds one prediction row across 256 head rows.  The
// epilogue then takes each 128-row tile maximum within one thread and stores each z
// octet (8 head rows of one prediction row, 32 contiguous bytes) with one instruction:
// far fewer instructions than the PM = 0 epilogue, which matters because the MMA thread
// shares the SM's issue and memory pipes with it.
template <int CG, int PM>
__global__ void __launch_bounds__(kThreads, 1)
logits_gemm_tc(const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ CUtensorMap tm_h, const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t b_rows = (uint32_t)g.bn_mma / CG;            // B rows staged by this CTA
  const uint32_t b_sub = b_rows * kBlockK * 2;                 // one K-block of them
  const uint32_t b_stage = b_sub * g.kpb;
  const uint32_t a_stage = kStageA * g.kpb;
  uint8_t* sA = smem;
  uint8_t* sB = sA + (size_t)g.stages * a_stage;
  uint64_t* full = (uint64_t*)(sB + (size_t)g.stages * b_stage);
  uint64_t* empty = full + g.stages;
  uint64_t* acc_full = empty + g.stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* tile_bar = drain + 1;                         // epilogue warps, per tile:
  uint64_t* tile_bar2 = tile_bar + 1;                     // maxima in / maxima out
  uint32_t* tmem_slot = (uint32_t*)(tile_bar2 + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  // the dynamic schedule's mailbox: tile indices posted by the producer, in order
  uint64_t* ring_full = tile_bar2 + 2;                    // an index is posted
  uint64_t* ring_free = ring_full + kTileRing;            // every reader has taken it
  volatile int* s_ring = (volatile int*)(ring_free + kTileRing);
  // column maxima of the tile over the four epilogue warps, as order-preserving keys
  int* s_cmax = (int*)((uint8_t*)smem + g.stages * (a_stage + b_stage) + kBarBytes);   // [256]
  int* s_live = s_cmax + 256;          // [1 + kMaxLiveTiles]: count, then the live N-tiles

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = CG == 2 ? ptx::cluster_ctarank() : 0;
  const bool leader = rank == 0;
  const int unit = CG == 2 ? (int)(blockIdx.x / 2) : (int)blockIdx.x;   // cluster or CTA
  const int units = CG == 2 ? (int)(gridDim.x / 2) : (int)gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.stages; ++s) {
      ptx::mbar_init(&full[s], 1);              // the leader's producer (bytes of both)
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 4 * CG);    // every epilogue warp of the pair
    }
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(tile_bar, 128);
    ptx::mbar_init(tile_bar2, 128);
    for (int j = 0; j < kTileRing; ++j) {
      ptx::mbar_init(&ring_full[j], 1);           // the producer
      ptx::mbar_init(&ring_free[j], 1 + 4);       // the MMA thread and the epilogue warps
    }
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  for (int c = threadIdx.x; c < 256; c += kThreads) s_cmax[c] = INT_MIN;
  if (warp == 4 && lane == 0) {
    ptx::tma_prefetch_desc(&tm_w);
    ptx::tma_prefetch_desc(&tm_h);
  }
  if (warp == 0) {
    if (CG == 2) {
      ptx::tmem_alloc_pair(tmem_slot, g.tmem_cols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, g.tmem_cols);
      ptx::tmem_relinquish();
    }
  }
  // Launched as a dependent of the kernel that zeroes the pass's control block: nothing
  // in global memory is read or written before that kernel (hence every earlier one on
  // the stream) has finished.
  pdl_wait();
  // Adaptive block length: an N-tile whose slots all lie at or past every one of its
  // blocks' cuts is not computed (the cuts come from the confidence kernel, launched
  // before this one).  Without cuts, or with more N-tiles than the list holds, all are.
  const bool cut_tiles = g.n_draft && g.n_tiles <= kMaxLiveTiles;
  if (warp == 2) {
    int cnt = 0;
    for (int nt = 0; nt < g.n_tiles; ++nt) {
      bool live = true;
      if (cut_tiles) {
        int i0, ni, bb0, nb;
        ntile_extent(g, nt, i0, ni, bb0, nb);
        bool any = false;
        for (int bl = lane; bl < nb; bl += 32) any |= g.n_draft[bb0 + bl] > i0;
        live = __any_sync(0xFFFFFFFFu, any);
        if (live && lane == 0) s_live[1 + cnt] = nt;
      }
      cnt += live;
    }
    if (lane == 0) s_live[0] = cnt;
  }
  pdl_signal();                                 // the chain's kernels may be scheduled
  ptx::tc_fence_before();
  __syncthreads();
  if (CG == 2) ptx::cluster_sync();             // the peer's barriers are initialised
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_live = s_live[0];
  const int num_tiles = g.v_tiles * n_live;
  // tile t: vocabulary tile t / n_live, N-tile the (t % n_live)-th live one
  auto tile_vt = [&](int t) { return t / n_live; };
  auto tile_nt = [&](int t) { return cut_tiles ? s_live[1 + t % n_live] : t % n_live; };
  // cluster addresses of the leader's full / acc_empty barriers (unused for CG = 1)
  const uint32_t full0 = CG == 2 ? ptx::mapa_shared(ptx::smem_u32(full), 0) : 0;
  const uint32_t acc_empty0 = CG == 2 ? ptx::mapa_shared(ptx::smem_u32(acc_empty), 0) : 0;

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(g.err, kErrTimeout);
  };

  // The tile schedule.  Static: CTA (or pair) `unit` takes tiles unit, unit + units, ...
  // Dynamic (CG = 1 with a claim counter): the producer claims each next tile from the
  // counter as it starts the current one, so that CTAs that stream faster take more
  // tiles, and posts the indices in order through the mailbox ring; the MMA thread and
  // the epilogue warps read them there.  An index past the last tile ends the sequence.
  const bool dyn = CG == 1 && g.tile_ctr != nullptr;
  // a reader's local-th tile (false: the wait gave up)
  auto read_tile = [&](uint32_t local, int& tile) -> bool {
    if (!dyn) {
      tile = unit + (int)local * units;
      return true;
    }
    const uint32_t j = local % kTileRing;
    if (!ptx::mbar_wait(&ring_full[j], (local / kTileRing) & 1, kWaitBudget, abort_flag))
      return false;
    tile = s_ring[j];
    return true;
  };

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const int ni_half = g.Ni / CG;
      const uint32_t tx = CG * (a_stage + (uint32_t)(g.BB * ni_half) * kBlockK * 2 * g.kpb);
      const int num_st = (g.num_kb + g.kpb - 1) / g.kpb;
      uint32_t it = 0, s = 0, ph = 0;          // stages issued; ring slot and phase
      bool ok = true;
      int tile = unit;
      // The lm_head stream is read once (or by the CTAs working on the same vocabulary
      // tile at the same moment): its lines are the first to leave L2, so that it does
      // not push out z, its maxima, the hidden states or the chain's data.  One GB300,
      // against the default policy: Qwen3-8B shape at B=1, GEMM 205 -> 192 us; at B=32,
      // pass 402.5 -> 393-396 us.
      const uint64_t w_pol = ptx::l2_policy_evict_first();
      for (uint32_t local = 0;; ++local) {
        if (dyn) {
          // post the index once every reader has taken the one posted kTileRing ago
          const uint32_t j = local % kTileRing;
          if (!ptx::mbar_wait(&ring_free[j], ((local / kTileRing) & 1) ^ 1, kWaitBudget,
                              abort_flag)) {
            ok = false;
            break;
          }
          s_ring[j] = tile;
          ptx::mbar_arrive(&ring_full[j]);
        }
        if (tile >= num_tiles) break;
        // the next claim goes out now; its answer is needed only after this tile's copies
        const int next = dyn ? units + (int)atomicAdd(g.tile_ctr, 1u) : tile + units;
        const int vt = tile_vt(tile), nt = tile_nt(tile);
        const int row_a = (vt * CG + (int)rank) * kBlockV;
        const int bcol = (nt % g.n_bt) * g.BB;
        const int slot = g.ifp + (nt / g.n_bt) * g.Ni + (int)rank * ni_half;
        for (int st = 0; st < num_st; ++st, ++it) {
          if (!ptx::mbar_wait(&empty[s], ph ^ 1, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* da = sA + (size_t)s * a_stage;
          uint8_t* db = sB + (size_t)s * b_stage;
          if (g.kpb > 1) {
            // K-blocks st * kpb ... as the third (lm_head) / fourth (hidden) map coordinate
            const int kc = st * g.kpb;
            if (CG == 2) {
              const uint32_t bar = full0 + s * 8;
              if (leader) ptx::mbar_arrive_expect_tx(&full[s], tx);
              ptx::tma_load_3d_pair_hint(da, &tm_w, bar, 0, row_a, kc, w_pol);
              ptx::tma_load_4d_pair(db, &tm_h, bar, 0, bcol, slot, kc);
            } else {
              ptx::mbar_arrive_expect_tx(&full[s], tx);
              ptx::tma_load_3d_hint(da, &tm_w, &full[s], 0, row_a, kc, w_pol);
              ptx::tma_load_4d(db, &tm_h, &full[s], 0, bcol, slot, kc);
            }
          } else if (CG == 2) {
            const uint32_t bar = full0 + s * 8;
            if (leader) ptx::mbar_arrive_expect_tx(&full[s], tx);
            ptx::tma_load_2d_pair_hint(da, &tm_w, bar, st * kBlockK, row_a, w_pol);
            ptx::tma_load_3d_pair(db, &tm_h, bar, st * kBlockK, bcol, slot);
          } else {
            ptx::mbar_arrive_expect_tx(&full[s], tx);
            ptx::tma_load_2d_hint(da, &tm_w, &full[s], st * kBlockK, row_a, w_pol);
            ptx::tma_load_3d(db, &tm_h, &full[s], st * kBlockK, bcol, slot);
          }
          if (++s == (uint32_t)g.stages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        tile = next;
      }
      if (!ok) {
        give_up();
        // let the copies already issued land before the CTA can exit
        if (CG == 1) {
          const uint32_t first = it > (uint32_t)g.stages ? it - g.stages : 0;
          for (uint32_t j = first; j < it; ++j)
            ptx::mbar_wait(&full[j % g.stages], (j / g.stages) & 1, kWaitBudget, nullptr);
        } else {
          // a pair's copies count on the leader's barrier: give them time to land
          const long long t0 = clock64();
          while (clock64() - t0 < 1000000) {
          }
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && leader) {
      // The tensor pipe holds only a couple of MMAs ahead of this thread, so whatever
      // the thread does between two stages' MMAs (the barrier wait, the commit, the loop)
      // leaves the pipe idle once it takes longer than those: keep it short, with the
      // ring position counted incrementally and the usual two K-blocks per stage issued
      // as one straight run.
      uint32_t s = 0, ph = 0, local = 0;
      bool ok = true;
      const int num_st = (g.num_kb + g.kpb - 1) / g.kpb;
      const uint32_t a_base = ptx::smem_u32(sA), b_base = ptx::smem_u32(sB);
      for (;; ++local) {
        int tile;
        if (!read_tile(local, tile)) {
          ok = false;
          break;
        }
        if (dyn) ptx::mbar_arrive(&ring_free[local % kTileRing]);
        if (tile >= num_tiles) break;
        int i0, ni, bb0, nb;
        ntile_extent(g, tile_nt(tile), i0, ni, bb0, nb);
        // rows up to the last valid slot (a pair always covers the full tile)
        const int n_mma = CG == 2 ? g.bn_mma : (ni * g.BB + 15) / 16 * 16;
        const uint32_t idesc = ptx::idesc_bf16_f32(kBlockV * CG, n_mma, 0, 0);
        const uint32_t acc = local & 1, aph = (local >> 1) & 1;
        if (!ptx::mbar_wait(&acc_empty[acc], aph ^ 1, kWaitBudget, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * (uint32_t)g.acc_stride;
        // one K-block: a [128 x 64] lm_head tile and a [rows x 64] hidden tile, as four
        // K = 16 MMAs (the descriptors' start addresses advance by 32 bytes = 2 units)
        auto kblock = [&](uint32_t a0, uint32_t b0, bool first) {
          const uint64_t da = ptx::desc_kmajor_sw128(PM ? b0 : a0);
          const uint64_t db = ptx::desc_kmajor_sw128(PM ? a0 : b0);
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k) {
            const uint32_t accum = (first && k == 0) ? 0u : 1u;
            if (CG == 2)
              ptx::mma_f16_pair(d_tmem, da + 2 * k, db + 2 * k, idesc, accum);
            else
              ptx::mma_f16(d_tmem, da + 2 * k, db + 2 * k, idesc, accum);
          }
        };
        for (int st = 0; st < num_st; ++st) {
          if (!ptx::mbar_wait(&full[s], ph, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_st = a_base + s * a_stage, b_st = b_base + s * b_stage;
          const int nk = min(g.kpb, g.num_kb - st * g.kpb);   // past H: nothing to add
          if (nk == 2) {
            kblock(a_st, b_st, st == 0);
            kblock(a_st + kStageA, b_st + b_sub, false);
          } else {
            for (int kc = 0; kc < nk; ++kc)
              kblock(a_st + kc * kStageA, b_st + kc * b_sub, st == 0 && kc == 0);
          }
          if (CG == 2)
            ptx::mma_commit_pair_multicast(&empty[s], 0x3);
          else
            ptx::mma_commit(&empty[s]);
          if (++s == (uint32_t)g.stages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        if (CG == 2)
          ptx::mma_commit_pair_multicast(&acc_full[acc], 0x3);
        else
          ptx::mma_commit(&acc_full[acc]);
      }
      if (!ok) give_up();
      // every MMA issued has finished once this commit lands
      if (CG == 2)
        ptx::mma_commit_pair_multicast(drain, 0x1);
      else
        ptx::mma_commit(drain);
      ptx::mbar_wait(drain, 0, kWaitBudget, nullptr);
    }
  } else if (PM) {
    // ---------------------------------------------------------------- epilogue (PM = 1)
    // Thread = one prediction row of this CTA (its TMEM lane); columns = the pair's 256
    // lm_head rows, 128 per tile maximum.
    //
    // Leaving out tiles of z (zbound_k > 0).  With the Markov term bounded by
    // |markov_w1[p] . markov_w2[:, v]| <= Umax cn[v] (Cauchy-Schwarz), a tile T of this
    // row holds a corrected logit >= lb[T] = zmax[T] - Umax cmax[T] and none above
    // ub[T] = zmax[T] + Umax cmax[T].  Every thread posts lb[T] into one of zbound_k
    // maxima (T mod zbound_k): the smallest of those maxima is a lower bound of
    // zbound_k distinct tiles' lb, hence of the zbound_k-th largest corrected logit.  A
    // tile whose ub stays below it can hold none of the top zbound_k (nor the argmax):
    // its z is not stored, and zwritten says so to the chain.
    uint32_t local = 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int p = warp * 32 + lane;
    const int il = p / g.BB, bl = p - il * g.BB;     // slot and block within this CTA's half
    const size_t oct_step = g.ldb * 8;               // floats between consecutive row octets
    // (a prepared buffer made for another head: its bounds are not read, every tile is
    // stored, and the chain reports the mismatch)
    const int K = (g.zbound_k > 0 && prepared_matches(g.prep, g.prep_want)) ? g.zbound_k : 0;
    const int NB = K <= 8 ? K * kBucketX : K;        // maxima kept per row
    const float umax = K > 0 ? __uint_as_float(*g.w1max) * (1.f + kPrunedRelMargin) : 0.f;
    // a key of the same order as the float, 0 below every float
    auto ukey = [](float f) { return (uint32_t)order_key32(f) ^ 0x80000000u; };
    for (int tile = unit; tile < num_tiles; tile += units, ++local) {
      const int vt = tile_vt(tile);
      int i0, ni, bb0, nb;
      ntile_extent(g, tile_nt(tile), i0, ni, bb0, nb);
      const int islot = (int)rank * (g.Ni / CG) + il;   // slot within the N-tile
      // (rows past their block's cut: not drafted, nothing stored)
      const bool live = islot < ni && bl < nb && (!g.n_draft || i0 + islot < g.n_draft[bb0 + bl]);
      const int i = i0 + islot, b = bb0 + bl;
      const uint32_t acc = local & 1, aph = (local >> 1) & 1;
      const bool ok = __all_sync(0xFFFFFFFFu,
                                 ptx::mbar_wait(&acc_full[acc], aph, kWaitBudget, abort_flag));
      if (!ok) {
        give_up();
        break;
      }
      ptx::tc_fence_after();
      // z_octet_index(i, v, b) = zrow + (v / 8) * oct_step + v % 8
      float* zrow = live ? g.z + ((size_t)i * (g.Vhp / 8) * g.ldb + (size_t)b) * 8 : g.z;
      // this row's maxima sit B apart, so that a warp's consecutive blocks read and
      // update them in whole sectors
      uint32_t* bound = (K > 0 && live) ? g.zbound + (size_t)i * NB * g.B + b : nullptr;
      // the current threshold, read once for both 128-row tiles (first, so that its
      // latency hides behind the TMEM loads; any value read is a valid bound, they only
      // grow)
      uint32_t th = 0;
      if (bound && vt * 2 * kBlockV < g.Vh) {
        if (NB == K) {
          th = 0xFFFFFFFFu;
          for (int j = 0; j < K; ++j) th = min(th, __ldcg(bound + (size_t)j * g.B));
        } else {
          // the K-th largest of the NB maxima (K <= 8): a descending top 8 by insertion
          uint32_t top[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          for (int j = 0; j < NB; ++j) {
            uint32_t x = __ldcg(bound + (size_t)j * g.B);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t hi = max(top[q], x);
              x = min(top[q], x);
              top[q] = hi;
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q == K - 1) th = top[q];
        }
      }
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int rt = vt * 2 + half;               // the 128-row tile of these columns
        const bool tile_in = rt * kBlockV < g.Vh;
        // this tile's maximum, with the bias
        float m = -INFINITY;
#pragma unroll 1
        for (int c0 = half * 128; c0 < half * 128 + 128; c0 += 32) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(tmem + lane_base + acc * (uint32_t)g.acc_stride + c0, r);
          ptx::tmem_ld_wait();
          const int v0 = vt * 256 + c0;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int v = v0 + 8 * q;                 // an octet: all in or all past the head
            if (v >= g.Vh) break;
            float x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(r[8 * q + j]);
            if (g.bias) {
              const float4 b0 = __ldg(reinterpret_cast<const float4*>(g.bias + v));
              const float4 b1 = __ldg(reinterpret_cast<const float4*>(g.bias + v + 4));
              x[0] += b0.x; x[1] += b0.y; x[2] += b0.z; x[3] += b0.w;
              x[4] += b1.x; x[5] += b1.y; x[6] += b1.z; x[7] += b1.w;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) m = fmaxf(m, x[j]);
            if (live && K == 0) ptx::st_global_v8(zrow + (size_t)(v >> 3) * oct_step, x);
          }
        }
        bool store = live && tile_in;
        if (live && tile_in) {
          if (bound) {
            const float d = umax * g.cnmax[rt] * (1.f + kPrunedRelMargin) + kPrunedAbsMargin;
            store = ukey(m + d) >= th;
            atomicMax(bound + (size_t)(rt % NB) * g.B, ukey(m - d));
          }
          if (g.zmax) g.zmax[((size_t)i * g.B + b) * g.zm_tiles + rt] = m;
          if (g.zwritten) g.zwritten[((size_t)i * g.B + b) * g.zm_tiles + rt] = store ? 1 : 0;
        }
        // the stores, from a second read of TMEM (a collective of the warp: every lane
        // takes part when any of them stores)
        if (K > 0 && __any_sync(0xFFFFFFFFu, store)) {
#pragma unroll 1
          for (int c0 = half * 128; c0 < half * 128 + 128; c0 += 32) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(tmem + lane_base + acc * (uint32_t)g.acc_stride + c0, r);
            ptx::tmem_ld_wait();
            const int v0 = vt * 256 + c0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int v = v0 + 8 * q;
              if (v >= g.Vh) break;
              float x[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(r[8 * q + j]);
              if (g.bias) {
                const float4 b0 = __ldg(reinterpret_cast<const float4*>(g.bias + v));
                const float4 b1 = __ldg(reinterpret_cast<const float4*>(g.bias + v + 4));
                x[0] += b0.x; x[1] += b0.y; x[2] += b0.z; x[3] += b0.w;
                x[4] += b1.x; x[5] += b1.y; x[6] += b1.z; x[7] += b1.w;
              }
              if (store) ptx::st_global_v8(zrow + (size_t)(v >> 3) * oct_step, x);
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(acc_empty0 + acc * 8);   // the leader's barrier
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (uint32_t local = 0;; ++local) {
      int tile;
      // the warp leaves together (tcgen05.ld below is a warp-collective instruction)
      if (!__all_sync(0xFFFFFFFFu, read_tile(local, tile))) {
        give_up();
        break;
      }
      if (dyn) {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&ring_free[local % kTileRing]);
      }
      if (tile >= num_tiles) break;
      const int vt = tile_vt(tile);
      const int rt = vt * CG + (int)rank;              // this CTA's 128-row tile
      int i0, ni, bb0, nb;
      ntile_extent(g, tile_nt(tile), i0, ni, bb0, nb);
      const int rows = ni * g.BB;
      const uint32_t acc = local & 1, aph = (local >> 1) & 1;
      // the warp leaves together: tcgen05.ld below is a warp-collective instruction
      const bool ok = __all_sync(0xFFFFFFFFu,
                                 ptx::mbar_wait(&acc_full[acc], aph, kWaitBudget, abort_flag));
      if (!ok) {
        give_up();
        break;
      }
      ptx::tc_fence_after();
      const int v = rt * kBlockV + warp * 32 + lane;
      const bool live = v < g.Vh;
      const float bias_v = (g.bias && live) ? g.bias[v] : 0.f;
      for (int c0 = 0; c0 < rows; c0 += 32) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_base + acc * (uint32_t)g.acc_stride + c0, r);
        ptx::tmem_ld_wait();
        if (g.zmax) {
          // column maxima over this warp's 32 head rows (one warp reduction per column,
          // lane j keeps column j), then over the four warps through shared memory
          int mk = INT_MIN;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = __reduce_max_sync(
                0xFFFFFFFFu, order_key32(live ? __uint_as_float(r[j]) + bias_v : -INFINITY));
            if (lane == j) mk = m;
          }
          if (c0 + lane < rows) atomicMax(&s_cmax[c0 + lane], mk);
        }
        if (!live) continue;
        if (g.octet) {
          // z[slot][row / 8][block][row % 8]: one column's 32 lanes store four 32-byte
          // runs, and the columns of one slot fill a contiguous stretch
          int il = c0 / g.BB, bl = c0 - (c0 / g.BB) * g.BB;
          float* zo = g.z + ((size_t)(i0 + il) * (g.Vhp / 8) + (v >> 3)) * g.ldb * 8 + (v & 7);
          const size_t slot_step = (g.Vhp / 8) * g.ldb * 8;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c0 + j < rows && bl < nb) zo[(size_t)(bb0 + bl) * 8] = __uint_as_float(r[j]) + bias_v;
            if (++bl == g.BB) {
              bl = 0;
              zo += slot_step;
            }
          }
        } else if ((g.BB & 3) == 0) {
          // runs of four consecutive blocks of one slot: 16-byte stores
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const int c = c0 + j, il = c / g.BB, bl = c % g.BB;
            if (c < rows && bl < nb) {
              float4 o = make_float4(__uint_as_float(r[j]) + bias_v,
                                     __uint_as_float(r[j + 1]) + bias_v,
                                     __uint_as_float(r[j + 2]) + bias_v,
                                     __uint_as_float(r[j + 3]) + bias_v);
              *reinterpret_cast<float4*>(
                  &g.z[((size_t)(i0 + il) * g.Vhp + v) * g.ldb + bb0 + bl]) = o;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c = c0 + j, il = c / g.BB, bl = c % g.BB;
            if (c < rows && bl < nb)
              g.z[((size_t)(i0 + il) * g.Vhp + v) * g.ldb + bb0 + bl] =
                  __uint_as_float(r[j]) + bias_v;
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CG == 2)
          ptx::mbar_arrive_cluster(acc_empty0 + acc * 8);   // the leader's barrier
        else
          ptx::mbar_arrive(&acc_empty[acc]);
      }
      if (g.zmax) {
        // the four warps' maxima are in (a bounded wait, so that a warp that gave up
        // cannot strand the others)
        ptx::mbar_arrive(tile_bar);
        if (!ptx::mbar_wait(tile_bar, local & 1, kWaitBudget, abort_flag)) {
          give_up();
          break;
        }
        for (int c = threadIdx.x; c < rows; c += 128) {
          const int il = c / g.BB, bl = c % g.BB;
          if (bl < nb && rt * kBlockV < g.Vh)
            g.zmax[((size_t)(i0 + il) * g.B + bb0 + bl) * g.zm_tiles + rt] =
                order_key32_value(s_cmax[c]);
          s_cmax[c] = INT_MIN;
        }
        // every key is read and reset before any warp adds the next tile's
        ptx::mbar_arrive(tile_bar2);
        if (!ptx::mbar_wait(tile_bar2, local & 1, kWaitBudget, abort_flag)) {
          give_up();
          break;
        }
      }
    }
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (CG == 2) ptx::cluster_sync();             // the pair's MMAs and arrivals are done
  if (warp == 0) {
    ptx::tc_fence_after();
    if (CG == 2)
      ptx::tmem_dealloc_pair(tmem, g.tmem_cols);
    else
      ptx::tmem_dealloc(tmem, g.tmem_cols);
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

constexpr int kMaxDevices = 64;
constexpr int kSmemMax = 227 * 1024;   // opt-in shared memory limit of one CTA

// Once per device and kernel form: allow the largest dynamic shared memory, and find how
// many CTAs (CG = 1) or pairs (CG = 2) can be resident at once, which sizes the
// persistent grid.
template <int CG>
cudaError_t resident_units(int* out) {
  static std::mutex mu;
  static int cached[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] > 0) {
    *out = cached[dev];
    return cudaSuccess;
  }
  auto kern = logits_gemm_tc<CG, 0>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
  if (e != cudaSuccess) return e;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int units = std::max(1, sms / CG);
  if (CG > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * CG);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemMax;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters > 0)
      units = std::min(units, clusters);
    cudaGetLastError();   // an occupancy query that failed leaves the estimate above
  }
  cached[dev] = units;
  *out = units;
  return cudaSuccess;
}

}  // namespace

// Prediction rows on M when the pair's N-tile is exactly 256 of them (z in the octet
// layout, which the PM epilogue writes; 16-byte bias loads).
bool logits_gemm_pm(int B, int N, bool z_octet, const float* lm_bias) {
  const GemmTilePlan tp = plan_logits_gemm(B, N);
  const bool pair = tp.Ni % 2 == 0 && (tp.BB * tp.Ni) % 32 == 0;
  return pair && tp.BB * tp.Ni == 256 && z_octet && ((uintptr_t)lm_bias & 15) == 0;
}

// Tile plan of the lm_head GEMM for B blocks of N prediction slots.
GemmTilePlan plan_logits_gemm(int B, int N) {
  // Candidate widths BB (blocks per tile); for each, slots are split into balanced
  // chunks of at most 256 / BB.  The cost estimate counts MMA instructions per 128 head
  // rows (halved when the tile qualifies for CTA pairs) times the measured time of one
  // 128 x n x 16 MMA, about 108 + 0.078 n clocks: narrow MMAs are expensive per row.
  GemmTilePlan best{};
  double best_cost = 0.0;
  const int widths[] = {256, 128, 64, 32, 16, 8, 4, 2, 1};
  for (int w : widths) {
    const int BB = std::min(B, w);
    if (w < 256 && BB != w) continue;                // each width once
    GemmTilePlan t{};
    t.BB = BB;
    const int ni_max = std::max(1, 256 / BB);
    t.n_it = (N + ni_max - 1) / ni_max;
    t.Ni = (N + t.n_it - 1) / t.n_it;                // balanced slot chunks
    t.n_bt = (B + BB - 1) / BB;
    t.bn_mma = (BB * t.Ni + 15) / 16 * 16;
    const bool pair = t.Ni % 2 == 0 && (BB * t.Ni) % 32 == 0;
    const double cost =
        (double)t.n_it * t.n_bt * (108.0 + 0.078 * t.bn_mma) / (pair ? 2.0 : 1.0);
    if (best.BB == 0 || cost < best_cost - 1e-9) {
      best = t;
      best_cost = cost;
    }
  }
  return best;
}

template <int CG, int PM>
cudaError_t launch_gemm(const CUtensorMap& tm_w, const CUtensorMap& tm_h, const GemmArgs& g,
                        size_t smem, cudaStream_t stream) {
  if (smem > (size_t)kSmemMax) return cudaErrorInvalidValue;
  int resident = 0;
  cudaError_t e = resident_units<CG>(&resident);
  if (e != cudaSuccess) return e;
  const int tiles = g.v_tiles * g.n_tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(std::max(1, std::min(tiles, resident)) * CG);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may be scheduled while the previous kernel runs (the kernel waits for it first)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (PM) {
    // the PM form has the same resources; it needs its own shared-memory opt-in, once
    // per device
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e2 = cudaGetDevice(&dev);
    if (e2 != cudaSuccess) return e2;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      e2 = cudaFuncSetAttribute(logits_gemm_tc<CG, PM>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
      if (e2 != cudaSuccess) return e2;
      done[dev] = true;
    }
  }
  return cudaLaunchKernelEx(&cfg, logits_gemm_tc<CG, PM>, tm_w, tm_h, g);
}

cudaError_t launch_base_logits_tc(const ProposePlan& p) {
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  const GemmTilePlan tp = plan_logits_gemm(p.B, p.N);
  // a CTA pair splits the prediction rows by slot halves: needs an even slot count per
  // tile and 16-row halves (whole swizzle atoms on both sides)
  const int CG = (tp.Ni % 2 == 0 && (tp.BB * tp.Ni) % 32 == 0) ? 2 : 1;
  GemmArgs g{};
  g.z = p.z;
  g.zbound = p.zbound;
  g.zwritten = p.zwritten;
  g.cnmax = p.cnmax;
  g.w1max = p.w1max;
  g.prep = p.prep;
  g.prep_want = p.prep_want;
  g.zbound_k = p.zbound_k;
  // single CTAs claim their tiles as they go (the control block is zeroed per pass)
  g.tile_ctr = CG == 1 ? p.ctrl + kCtrlGemmTiles : nullptr;
  g.n_draft = p.skip_truncated ? p.n_draft : nullptr;
  g.Vhp = p.Vhp;
  g.ldb = p.ldb;
  g.zmax = p.zmax;
  g.octet = p.z_octet ? 1 : 0;
  g.bias = p.lm_bias;
  g.err = p.ctrl;
  g.B = p.B;
  g.N = p.N;
  g.ifp = p.ifp;
  g.Vh = p.Vh;
  g.BB = tp.BB;
  g.Ni = tp.Ni;
  g.n_bt = tp.n_bt;
  g.bn_mma = CG == 2 ? tp.BB * tp.Ni : tp.bn_mma;
  g.n_tiles = tp.n_it * tp.n_bt;
  g.v_tiles = (p.Vh + kBlockV * CG - 1) / (kBlockV * CG);
  g.zm_tiles = (int)(p.Vhp / kBlockV);
  g.num_kb = (p.H + kBlockK - 1) / kBlockK;
  // Two K-blocks per stage when H allows: each operand then arrives in one 32 KB copy
  // per stage instead of two 16 KB ones (a copy has a fixed cost in the TMA unit).
  // (the hidden box must then fill whole 8-row swizzle atoms, so that the second
  // K-block's rows start where the descriptors expect them).  A last stage reaching past
  // H loads zeros there, which add nothing.
  // shared memory: up to 1023 bytes of alignment, the stages, the barriers and tile ring,
  // and the column-maximum keys
  const size_t fixed = 1024 + kBarBytes + (256 + 1 + kMaxLiveTiles) * sizeof(int);
  const int box_rows = g.BB * g.Ni / CG;
  const uint32_t kblock_bytes = kStageA + (uint32_t)(g.bn_mma / CG) * kBlockK * 2;
  g.kpb = 1;
  if (p.H % kBlockK == 0 && box_rows % 8 == 0 && box_rows * CG == g.bn_mma)
    for (int c = kMaxKpb; c > 1; --c)
      if (g.num_kb >= c && ((size_t)kSmemMax - fixed) / (kblock_bytes * c) >= 2) {
        g.kpb = c;
        break;
      }
  const uint32_t stage_bytes = kblock_bytes * (uint32_t)g.kpb;
  g.stages = (int)std::min<size_t>(8, ((size_t)kSmemMax - fixed) / stage_bytes);
  // 32-column TMEM loads may run past the last valid column of an accumulator, so
  // each accumulator owns a multiple of 32 columns
  g.acc_stride = (g.bn_mma + 31) / 32 * 32;
  uint32_t cols = 32;
  while (cols < 2u * (uint32_t)g.acc_stride) cols <<= 1;
  g.tmem_cols = cols;
  const size_t smem = fixed + (size_t)g.stages * stage_bytes;

  CUtensorMap tm_w, tm_h;
  if (g.kpb > 1) {
    // lm_head [V_head, H] seen as (64 columns, row, 64-column chunk), and hidden
    // [B, L_in, H] as (64 columns, block, slot, chunk): a box of kpb chunks lands as kpb
    // consecutive [rows x 64] tiles, the layout of kpb single K-block stages
    {
      cuuint64_t dims[3] = {(cuuint64_t)kBlockK, (cuuint64_t)p.Vh, (cuuint64_t)(p.H / kBlockK)};
      cuuint64_t strides[2] = {(cuuint64_t)p.H * 2, (cuuint64_t)kBlockK * 2};
      cuuint32_t box[3] = {kBlockK, kBlockV, (cuuint32_t)g.kpb};
      cuuint32_t es[3] = {1, 1, 1};
      if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)p.lm_head, dims, strides,
                 box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    {
      cuuint64_t dims[4] = {(cuuint64_t)kBlockK, (cuuint64_t)p.B, (cuuint64_t)p.L_in,
                            (cuuint64_t)(p.H / kBlockK)};
      cuuint64_t strides[3] = {(cuuint64_t)p.L_in * p.H * 2, (cuuint64_t)p.H * 2,
                               (cuuint64_t)kBlockK * 2};
      cuuint32_t box[4] = {kBlockK, (cuuint32_t)g.BB, (cuuint32_t)(g.Ni / CG),
                           (cuuint32_t)g.kpb};
      cuuint32_t es[4] = {1, 1, 1, 1};
      if (encode(&tm_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void*)p.hidden, dims, strides,
                 box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  } else {
  {
    cuuint64_t dims[2] = {(cuuint64_t)p.H, (cuuint64_t)p.Vh};
    cuuint64_t strides[1] = {(cuuint64_t)p.H * 2};
    cuuint32_t box[2] = {kBlockK, kBlockV};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)p.lm_head, dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // hidden [B, L_in, H] viewed as (h, block, slot) so that a box lands slot-major with
    // the blocks of one slot contiguous; a pair member loads half of the tile's slots
    cuuint64_t dims[3] = {(cuuint64_t)p.H, (cuuint64_t)p.B, (cuuint64_t)p.L_in};
    cuuint64_t strides[2] = {(cuuint64_t)p.L_in * p.H * 2, (cuuint64_t)p.H * 2};
    cuuint32_t box[3] = {kBlockK, (cuuint32_t)g.BB, (cuuint32_t)(g.Ni / CG)};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&tm_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)p.hidden, dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  }
  const bool pm = logits_gemm_pm(p.B, p.N, p.z_octet, p.lm_bias);
  // only the PM form leaves tiles out (and writes zwritten)
  if ((p.zbound_k > 0 || p.zwritten) && !pm) return cudaErrorInvalidValue;
  cudaError_t e = CG == 2 ? (pm ? launch_gemm<2, 1>(tm_w, tm_h, g, smem, p.stream)
                                : launch_gemm<2, 0>(tm_w, tm_h, g, smem, p.stream))
                          : launch_gemm<1, 0>(tm_w, tm_h, g, smem, p.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dspark
