// Internal launch interface between the C ABI layer and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace dspark {

// First bytes of a prepared head buffer: what it was prepared for.  The kernels that
// read a prepared buffer compare it with the head of the call before they read anything
// else in it, and flag kErrPrepared (reading nothing more) when they differ.
struct PreparedHeader {
  uint32_t magic;          // kPreparedMagic once dspark_prepare_head has run
  int32_t V, Vh, r;
  unsigned long long w1, w2;   // device addresses of markov_w1 / markov_w2
};
constexpr uint32_t kPreparedMagic = 0x4B525044u;

__device__ __forceinline__ bool prepared_matches(const PreparedHeader* h,
                                                 const PreparedHeader& want) {
  const PreparedHeader got = *h;
  return got.magic == want.magic && got.V == want.V && got.Vh == want.Vh &&
         got.r == want.r && got.w1 == want.w1 && got.w2 == want.w2;
}

// A head given in the bias form (full-V lm_head, lm_bias marking the rows the draft
// cannot emit) is prepared as a compact head: the first bytes of its prepared buffer
// are a CompactHeader, followed by the sorted emittable rows (the compact head's d2t,
// padded to a multiple of 8), their lm_head rows, markov_w2 columns and biases, and the
// compact head's own prepared data (a PreparedHeader and the rest).
constexpr float kEmitMaskLevel = -1e8f;   // a bias at or below it marks a masked row
struct CompactHeader {
  uint32_t magic;                         // kCompactMagic once dspark_prepare_head has run
  int32_t V, H, r, n_emit, n_pad;
  unsigned long long lm_head, lm_bias, w1, w2;   // the full head's device addresses
};
constexpr uint32_t kCompactMagic = 0x4D435044u;
struct CompactLayout {
  size_t header, list, chunk_count, lm_head, w2, bias, prepared, total;
};
CompactLayout plan_compact(int V, int H, int r, int n_pad);
cudaError_t launch_emit_count(const float* bias, int V, int* count, cudaStream_t stream);
cudaError_t launch_prepare_compact(const void* lm_head, const float* bias, const void* w1,
                                   const void* w2, int V, int H, int r, int n_emit, int n_pad,
                                   void* prepared, cudaStream_t stream);

// Everything a proposal launch needs, resolved by the ABI layer.
struct ProposePlan {
  // sizes
  int B, L_in, N, ifp, H, V, Vh, r, k, topk_markov, dtype;
  float conf_min, b_conf;
  // inputs
  const void* hidden;
  const void* conf_hidden;   // what the confidence head reads: hidden, or a separate input
  const int32_t* anchors;
  const void* lm_head;
  const float* lm_bias;
  const int32_t* d2t;
  const void* w1;
  const void* w2;
  const void* w_conf;
  // outputs
  int32_t* draft;
  int32_t* n_draft;
  int32_t* topk_ids;
  float* topk_vals;
  float* conf;
  float* logits;
  // workspace pieces
  uint32_t* ctrl;       // [0] = error word
  unsigned int* bar;    // grid-barrier counters of the dense chain, one per 16 blocks
  unsigned long long* keys;  // [N][B] order keys of each slot's winner
  float* cand_val;      // dense chain: [N][B][kChainMaxCtas][kDenseLocal] rows of each
  int32_t* cand_id;     //   CTA that reach the slot's top-k bound, their ranked values;
                        //   fp32 chain: [N][B][G][k] each CTA's k best ranked rows
  int32_t* cand_cnt;    //   [N][B][kChainMaxCtas] how many each CTA found
  uint32_t* bucket;     //   [N][B][kDenseBuckets] maxima of the CTAs' best values (order
                        //   keys, zeroed per pass)
  float* zmax;          // per-tile maxima of z [N][B][Vhp / 128], or NULL (dense chain)
  const __nv_bfloat16* w2t;   // prepared head: markov_w2 transposed [Vhp][r], or NULL
  const float* cnorm;   // prepared head: column norms of markov_w2 [Vhp]
  const float* cnmax;   // prepared head: per-tile maxima of cnorm [Vhp / 128]
  const unsigned* w1max;  // prepared head: max row norm of markov_w1 (float bits)
  const PreparedHeader* prep;  // prepared head: its header, or NULL
  PreparedHeader prep_want;    // the header this call's head would have
  int32_t* cand_v;      // pruned chain: candidate head rows of each slot [N][B][cap]
  float* cand_z;        //               their base logits
  int32_t* cand_n;      //               candidate counts [N][B]
  int32_t* prev_v;      //               head rows that can be the previous slot's
                        //               argmax [N][B][cap_a] (slot 0: the anchor)
  int32_t* prev_n;      //               their counts [N][B]
  int32_t* amax;        //               argmax head row given each previous row
                        //               [N][B][cap_a]
  int32_t* tk_id;       //               top-k tokens given each previous row
  float* tk_val;        //               [N][B][cap_a][k], and their values
  uint32_t* zbound;     //               [N][2 zbound_k][B] room for the maxima of the tiles'
                        //               lower bounds (unsigned order keys)
  uint8_t* zwritten;    //               [N][B][Vhp / 128] whether the GEMM stored the
                        //               tile's z (NULL: it stored every tile)
  int zbound_k;         //               0: the GEMM stores every tile
  int32_t* walk_done;   //               [B] table CTAs finished per block (zeroed per pass)
  bool skip_truncated;  // adaptive block length: n_draft is computed before the GEMM and
                        // the slots from it on are not drafted
  float* z;             // base logits: [N][Vhp][ldb] (slot, head row, block fastest), or
                        // [N][Vhp / 8][ldb][8] when z_octet (see z_octet_index)
  bool z_octet;
  size_t Vhp, ldb;      // head rows rounded up to whole 128-row tiles; blocks rounded to 8
  size_t ldz;           // row stride of zc
  float* zc;            // corrected logits of the current slot [B][ldz]
  float* zk;            // fp32 chain, few prediction rows: every slot's ranked values
                        //   [N][B][ldz], or NULL
  float* conf_ws;       // confidences when the caller did not ask for them [B][N]
  cudaStream_t stream;
};

// Index of base logit (slot i, head row v, block b) in the octet layout: eight
// consecutive head rows of one block are contiguous (one 32-byte sector), and the octets
// of all blocks for the same rows follow each other, so the lm_head GEMM writes long
// contiguous stretches while a scan of one block's rows reads whole sectors.
__host__ __device__ __forceinline__ size_t z_octet_index(size_t i, size_t v, size_t b,
                                                         size_t Vhp, size_t ldb) {
  return ((i * (Vhp / 8) + v / 8) * ldb + b) * 8 + (v % 8);
}

// Upper bound on the chain kernel's grid (one CTA per SM).
constexpr int kChainMaxCtas = 256;
// Dense chain: candidate rows kept per (slot, block, CTA) and per (slot, block), and the
// number of maxima that bound the top k.
constexpr int kDenseLocal = 4;
constexpr int kDenseCap = 256;
constexpr int kDenseBuckets = 32;

// Workspace carve-up shared by the size query and the launch.  [ctrl, zero_end) is
// cleared at the start of every call.
struct WorkspaceLayout {
  size_t ctrl, bar, keys, zbound, walk_done, dense_cnt, dense_bucket, zero_end, z, zmax,
      zwritten, cand, zc, zk, conf, dense_val, dense_id, total;
  size_t Vhp, ldb, ldz;
};
WorkspaceLayout plan_workspace(int B, int N, int Vh, int k, int dtype, bool pruned);

// Layout of a prepared head (dspark_prepare_head): a PreparedHeader (256 bytes reserved),
// markov_w2 transposed to [Vhp][r]
// bf16, the fp32 Euclidean norm of every markov_w2 column [Vhp] (0 past V_head), the
// maximum of those norms over each 128-row tile [Vhp / 128], and the largest norm of a
// markov_w1 row (one float).
struct PreparedLayout {
  size_t header, w2t, cnorm, cnmax, w1max, total;
  size_t Vhp, tiles;
};
PreparedLayout plan_prepared(int Vh, int r);
// Candidate lists and tables of the pruned chain; the pieces lie in this order.
struct PrunedLists {
  size_t cand_v, cand_z, cand_n, prev_v, prev_n, amax, tk_id, tk_val, total;
};
PrunedLists plan_pruned_lists(int B, int N, int k);

// Rounding margins of the pruned chain's bounds (relative to the Markov bound, and
// absolute), shared by the chain and the lm_head GEMM, which prunes with the same bounds.
constexpr float kPrunedRelMargin = 1.0f / 1024;
constexpr float kPrunedAbsMargin = 1e-4f;

// Whether the lm_head GEMM runs with the prediction rows on M for these sizes (the form
// that can leave out tiles of z that cannot matter, see logits_gemm_tc).
bool logits_gemm_pm(int B, int N, bool z_octet, const float* lm_bias);
cudaError_t launch_prepare_head(const void* w1, const void* w2, int V, int r, int Vh,
                                void* prepared, cudaStream_t stream);
cudaError_t launch_chain_pruned(const ProposePlan& p);

// Blocking of the lm_head GEMM's N dimension: a tile holds Ni slots x BB blocks of
// prediction rows (blocks fastest; padded to bn_mma, a multiple of 16, at most 256);
// n_it x n_bt such tiles cover all N slots and B blocks.
struct GemmTilePlan {
  int BB, Ni, n_it, n_bt, bn_mma;
};
GemmTilePlan plan_logits_gemm(int B, int N);

cudaError_t launch_conf(const ProposePlan& p);
// Zeroes `bytes` (a multiple of 16, 16-byte aligned) at p; the next kernel on the stream
// may be launched as its dependent (launch_dependent, or the lm_head GEMM).
cudaError_t launch_zero_block(void* p, size_t bytes, cudaStream_t stream);

// Launch `kernel` on `stream` with programmatic stream serialisation, so that it may
// start before the previous kernel on the stream has finished (it calls pdl_wait()
// before reading that kernel's results).
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
cudaError_t launch_base_logits_tc(const ProposePlan& p);
cudaError_t launch_base_logits_simt(const ProposePlan& p);
cudaError_t launch_chain_simt(const ProposePlan& p);
int simt_chain_ctas_max(int Vh);
// Whether the fp32 chain of this shape also evaluates the confidence head and the base
// logits (one launch for the whole proposal).
bool simt_fused(int B, int N, int H, int Vh, int r, bool skip_truncated);
constexpr int kSimtFusedRows = 16;   // prediction rows of a problem small enough to fuse
cudaError_t launch_chain_dense(const ProposePlan& p);
// Blocks per launch of the dense chain for a head of Vh rows on `sms` SMs (32 or 16), or
// 0 when its per-CTA share of the Markov terms does not fit TMEM.
int dense_chain_group(int Vh, int sms);

// Launch facts of the current device, cached across calls (each query costs host time
// that a small problem would otherwise spend with the GPU idle):
//   device_sms: its SM count;
//   blocks_per_sm: resident CTAs per SM of kernel `fn` at `threads` threads and `smem`
//   bytes of dynamic shared memory, after raising the kernel's dynamic shared memory
//   limit to `smem` when that is above the default 48 KB;
//   raise_smem_limit: that limit alone (set only when a larger one is needed).
cudaError_t device_sms(int* sms);
cudaError_t blocks_per_sm(const void* fn, int threads, size_t smem, int* out);
cudaError_t raise_smem_limit(const void* fn, size_t smem);
cudaError_t launch_verify(int B, int N, const int32_t* draft, const int32_t* n_draft,
                          const int32_t* target, int32_t* accepted, int32_t* bonus,
                          int32_t* emitted, cudaStream_t stream);
cudaError_t launch_tree_verify(int B, int N, int k, const int32_t* topk_ids,
                               const int32_t* n_draft, const int32_t* target,
                               int32_t* accepted, int32_t* bonus, int32_t* emitted,
                               int32_t* path, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint32_t* err, long long budget, int pre_abort,
                                 cudaStream_t stream);

}  // namespace dspark
