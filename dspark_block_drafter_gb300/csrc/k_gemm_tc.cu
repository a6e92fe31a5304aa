// Base logits on the 5th-generation tensor cores (bf16 in, fp32 accumulate in TMEM).
//
//   z[i][v][b] = sum_h hidden[b, ifp + i, h] * lm_head[v, h] + lm_bias[v]
//
// (llama.cpp commit 6fed9f6, "spec: add DSpark speculative decoding": logits(i) of the
// proposal formula.)  The GEMM runs "swap-AB": the MMA's M dimension is the vocabulary
// (128 head rows per tile), its N dimension the prediction rows of Ni slots x BB blocks
// (blocks fastest, up to 256), so a small batch still fills the instruction.  The
// output keeps the blocks of one (slot, head row) contiguous, so each thread stores
// runs of 16 bytes and the chain reads them back the same way.
//
// One persistent CTA per SM, warp-specialised:
//   warp 4      TMA producer: lm_head tile [128 x 64] and hidden tile [Ni, BB, 64] per
//               K-block into a ring of shared-memory stages (128-byte swizzle)
//   warp 5      MMA issuer: 4 x tcgen05.mma (K = 16) per stage into a TMEM accumulator;
//               tcgen05.commit frees the stage, and the accumulator when the tile ends
//   warps 0-3   epilogue: tcgen05.ld of their 32 TMEM lanes (= 32 head rows), + bias,
//               fp32 stores of z (16-byte runs of blocks per thread)
// Two TMEM accumulators alternate so that the epilogue of one tile overlaps the MMAs of
// the next.  Tiles are ordered vocabulary-major: CTAs that run side by side share the
// same lm_head tile through L2, so lm_head streams from HBM once.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
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
constexpr long long kWaitBudget = 2000000000ll;       // ~1 s of SM clocks

struct GemmArgs {
  float* z;
  size_t Vhp, ldb;
  float* zmax;     // [N][B][v_tiles] per-tile maxima of z, or NULL
  const float* bias;
  uint32_t* err;
  int B, N, ifp, Vh;
  int BB, Ni;      // blocks and slots per N-tile
  int n_bt;        // N-tiles along the blocks (the slot index is tile / n_bt)
  int bn_mma;      // MMA N (rows of the B operand per stage), multiple of 16
  int acc_stride;  // TMEM columns between the two accumulators (multiple of 32)
  int n_tiles, v_tiles, num_kb, stages;
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

__global__ void __launch_bounds__(kThreads, 1)
logits_gemm_tc(const __grid_constant__ CUtensorMap tm_w,
               const __grid_constant__ CUtensorMap tm_h, const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t b_stage = (uint32_t)g.bn_mma * kBlockK * 2;
  uint8_t* sA = smem;
  uint8_t* sB = sA + (size_t)g.stages * kStageA;
  uint64_t* full = (uint64_t*)(sB + (size_t)g.stages * b_stage);
  uint64_t* empty = full + g.stages;
  uint64_t* acc_full = empty + g.stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* tile_bar = drain + 1;                         // epilogue warps, per tile
  uint32_t* tmem_slot = (uint32_t*)(tile_bar + 1);
  volatile int* abort_flag = (volatile int*)(tmem_slot + 1);
  // tile maxima: a padded 32 x 32 transpose panel per epilogue warp, and the four
  // warps' column maxima, double-buffered by tile parity
  float* s_panel = (float*)((uint8_t*)smem + g.stages * (kStageA + b_stage) + 256);
  float* s_cmax = s_panel + 4 * 32 * 33;                 // [2][4][256]

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < g.stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&acc_full[a], 1);
      ptx::mbar_init(&acc_empty[a], 128);
    }
    ptx::mbar_init(drain, 1);
    ptx::mbar_init(tile_bar, 128);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    ptx::tma_prefetch_desc(&tm_w);
    ptx::tma_prefetch_desc(&tm_h);
  }
  if (warp == 0) {
    ptx::tmem_alloc(tmem_slot, g.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int num_tiles = g.v_tiles * g.n_tiles;

  auto give_up = [&]() {
    *abort_flag = 1;
    flag_error(g.err, kErrTimeout);
  };

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t tx = kStageA + (uint32_t)(g.BB * g.Ni) * kBlockK * 2;
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        const int vt = tile / g.n_tiles, nt = tile % g.n_tiles;
        for (int kb = 0; kb < g.num_kb; ++kb, ++it) {
          const uint32_t s = it % g.stages, ph = (it / g.stages) & 1;
          if (!ptx::mbar_wait(&empty[s], ph ^ 1, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[s], tx);
          ptx::tma_load_2d(sA + (size_t)s * kStageA, &tm_w, &full[s], kb * kBlockK,
                           vt * kBlockV);
          ptx::tma_load_3d(sB + (size_t)s * b_stage, &tm_h, &full[s], kb * kBlockK,
                           (nt % g.n_bt) * g.BB, g.ifp + (nt / g.n_bt) * g.Ni);
        }
      }
      if (!ok) {
        give_up();
        // let the copies already issued land before the CTA can exit
        const uint32_t first = it > (uint32_t)g.stages ? it - g.stages : 0;
        for (uint32_t j = first; j < it; ++j)
          ptx::mbar_wait(&full[j % g.stages], (j / g.stages) & 1, kWaitBudget, nullptr);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0, local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x, ++local) {
        int i0, ni, bb0, nb;
        ntile_extent(g, tile % g.n_tiles, i0, ni, bb0, nb);
        const int n_mma = (ni * g.BB + 15) / 16 * 16;   // rows up to the last valid slot
        const uint32_t idesc = ptx::idesc_bf16_f32(kBlockV, n_mma, 0, 0);
        const uint32_t acc = local & 1, aph = (local >> 1) & 1;
        if (!ptx::mbar_wait(&acc_empty[acc], aph ^ 1, kWaitBudget, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem + acc * (uint32_t)g.acc_stride;
        for (int kb = 0; kb < g.num_kb; ++kb, ++it) {
          const uint32_t s = it % g.stages, ph = (it / g.stages) & 1;
          if (!ptx::mbar_wait(&full[s], ph, kWaitBudget, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(sA + (size_t)s * kStageA);
          const uint32_t b0 = ptx::smem_u32(sB + (size_t)s * b_stage);
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k)
            ptx::mma_f16(d_tmem, ptx::desc_kmajor_sw128(a0 + k * 32),
                         ptx::desc_kmajor_sw128(b0 + k * 32), idesc, (kb | k) != 0);
          ptx::mma_commit(&empty[s]);
        }
        if (ok) ptx::mma_commit(&acc_full[acc]);
      }
      if (!ok) give_up();
      // every MMA issued has finished once this commit lands
      ptx::mma_commit(drain);
      ptx::mbar_wait(drain, 0, kWaitBudget, nullptr);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    uint32_t local = 0;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const int vt = tile / g.n_tiles;
      int i0, ni, bb0, nb;
      ntile_extent(g, tile % g.n_tiles, i0, ni, bb0, nb);
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
      const int v = vt * kBlockV + warp * 32 + lane;
      const bool live = v < g.Vh;
      const float bias_v = (g.bias && live) ? g.bias[v] : 0.f;
      float* cmax = s_cmax + (local & 1) * 4 * 256;
      for (int c0 = 0; c0 < rows; c0 += 32) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tmem + lane_base + acc * (uint32_t)g.acc_stride + c0, r);
        ptx::tmem_ld_wait();
        if (g.zmax) {
          // column maxima over this warp's 32 head rows, through a transpose panel
          float* panel = s_panel + warp * 32 * 33;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            panel[j * 33 + lane] = live ? __uint_as_float(r[j]) + bias_v : -INFINITY;
          __syncwarp();
          float m = -INFINITY;
#pragma unroll 8
          for (int q = 0; q < 32; ++q) m = fmaxf(m, panel[lane * 33 + q]);
          cmax[warp * 256 + c0 + lane] = m;
          __syncwarp();
        }
        if (!live) continue;
        if ((g.BB & 3) == 0) {
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
      ptx::mbar_arrive(&acc_empty[acc]);
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
          if (bl < nb) {
            const float m = fmaxf(fmaxf(cmax[c], cmax[256 + c]),
                                  fmaxf(cmax[512 + c], cmax[768 + c]));
            g.zmax[((size_t)(i0 + il) * g.B + bb0 + bl) * g.v_tiles + vt] = m;
          }
        }
      }
    }
  }
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
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

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace

// Tile plan of the lm_head GEMM for B blocks of N prediction slots.
GemmTilePlan plan_logits_gemm(int B, int N) {
  GemmTilePlan t{};
  t.BB = B < 256 ? B : 256;
  const int ni_max = std::max(1, 256 / t.BB);
  t.n_it = (N + ni_max - 1) / ni_max;
  t.Ni = (N + t.n_it - 1) / t.n_it;                  // balanced slot chunks
  t.n_bt = (B + t.BB - 1) / t.BB;
  t.bn_mma = (t.BB * t.Ni + 15) / 16 * 16;
  return t;
}

cudaError_t launch_base_logits_tc(const ProposePlan& p) {
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  const GemmTilePlan tp = plan_logits_gemm(p.B, p.N);
  GemmArgs g{};
  g.z = p.z;
  g.Vhp = p.Vhp;
  g.ldb = p.ldb;
  g.zmax = p.zmax;
  g.bias = p.lm_bias;
  g.err = p.ctrl;
  g.B = p.B;
  g.N = p.N;
  g.ifp = p.ifp;
  g.Vh = p.Vh;
  g.BB = tp.BB;
  g.Ni = tp.Ni;
  g.n_bt = tp.n_bt;
  g.bn_mma = tp.bn_mma;
  g.n_tiles = tp.n_it * tp.n_bt;
  g.v_tiles = (p.Vh + kBlockV - 1) / kBlockV;
  g.num_kb = (p.H + kBlockK - 1) / kBlockK;
  const uint32_t stage_bytes = kStageA + (uint32_t)g.bn_mma * kBlockK * 2;
  const size_t smem_budget = 220 * 1024 - (4 * 32 * 33 + 2 * 4 * 256) * sizeof(float);
  g.stages = (int)std::min<size_t>(8, (smem_budget - 1024 - 256) / stage_bytes);
  // 32-column TMEM loads may run past the last valid column of an accumulator, so
  // each accumulator owns a multiple of 32 columns
  g.acc_stride = (g.bn_mma + 31) / 32 * 32;
  uint32_t cols = 32;
  while (cols < 2u * (uint32_t)g.acc_stride) cols <<= 1;
  g.tmem_cols = cols;
  const size_t smem = 1024 + (size_t)g.stages * stage_bytes + 256 +
                      (4 * 32 * 33 + 2 * 4 * 256) * sizeof(float);

  CUtensorMap tm_w, tm_h;
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
    // the blocks of one slot contiguous
    cuuint64_t dims[3] = {(cuuint64_t)p.H, (cuuint64_t)p.B, (cuuint64_t)p.L_in};
    cuuint64_t strides[2] = {(cuuint64_t)p.L_in * p.H * 2, (cuuint64_t)p.H * 2};
    cuuint32_t box[3] = {kBlockK, (cuuint32_t)g.BB, (cuuint32_t)g.Ni};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&tm_h, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)p.hidden, dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(logits_gemm_tc,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int tiles = g.v_tiles * g.n_tiles;
  const int grid = std::min(tiles, sm_count());
  logits_gemm_tc<<<grid, kThreads, smem, p.stream>>>(tm_w, tm_h, g);
  return cudaGetLastError();
}

}  // namespace dspark
