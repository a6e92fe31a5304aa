// The C ABI: argument validation, workspace carve-up and kernel dispatch.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dspark.h"
#include "common.cuh"
#include "kernels.h"

namespace dspark {

static thread_local std::string g_last_error;

static dspark_status fail(dspark_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

static dspark_status cuda_fail(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return DSPARK_ERR_CUDA;
}

static constexpr size_t kAlign = 256;
// the longest wait the self-test may ask for: the budget of the pipelines' own waits
static constexpr long long kMaxSelftestBudget = 2000000000ll;

cudaError_t device_sms(int* sms) {
  static std::mutex mu;
  static int cached[64];                              // 0: not looked up yet
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (cached[dev] == 0) {
    e = cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      cached[dev] = 0;
      return e;
    }
  }
  *sms = cached[dev];
  return cudaSuccess;
}

cudaError_t raise_smem_limit(const void* fn, size_t smem) {
  struct Entry {
    const void* fn;
    int dev;
    size_t smem;                                      // the limit set so far
  };
  static std::mutex mu;
  static std::vector<Entry> set;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  Entry* found = nullptr;
  for (Entry& x : set)
    if (x.fn == fn && x.dev == dev) found = &x;
  if (found && found->smem >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (found)
    found->smem = smem;
  else if (set.size() < 256)
    set.push_back({fn, dev, smem});
  return cudaSuccess;
}

cudaError_t blocks_per_sm(const void* fn, int threads, size_t smem, int* out) {
  struct Entry {
    const void* fn;
    int dev, threads;
    size_t smem;
    int blocks;
  };
  static std::mutex mu;
  static std::vector<Entry> cache;                   // a few kernels x sizes per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Entry& x : cache)
    if (x.fn == fn && x.dev == dev && x.threads == threads && x.smem == smem) {
      *out = x.blocks;
      return cudaSuccess;
    }
  if (smem > 48 * 1024) {
    e = raise_smem_limit(fn, smem);
    if (e != cudaSuccess) return e;
  }
  int blocks = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, threads, smem);
  if (e != cudaSuccess) return e;
  if (cache.size() < 256) cache.push_back({fn, dev, threads, smem, blocks});
  *out = blocks;
  return cudaSuccess;
}

WorkspaceLayout plan_workspace(int B, int N, int Vh, int k, int dtype, bool pruned) {
  WorkspaceLayout w{};
  w.ldz = align_up((size_t)Vh, 64);
  w.Vhp = align_up((size_t)Vh, 128);
  w.ldb = align_up((size_t)B, 8);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  w.ctrl = take(256);
  w.bar = take(sizeof(unsigned) * (size_t)((B + 15) / 16));   // one per dense-chain launch
  w.keys = take(sizeof(unsigned long long) * (size_t)N * B);
  // the maxima of the lower bounds with which the GEMM leaves tiles of z out start from
  // zero (below every key) in every pass
  if (pruned) {
    w.zbound = take(sizeof(uint32_t) * (size_t)N * B * 2 * k);   // up to two maxima per rank
    w.walk_done = take(sizeof(int32_t) * (size_t)B);
  } else if (dtype != DSPARK_F32) {   // the dense chain's bound maxima
    w.dense_bucket = take(sizeof(uint32_t) * (size_t)N * B * kDenseBuckets);
  }
  w.zero_end = off;
  w.z = take(sizeof(float) * (size_t)N * w.Vhp * w.ldb);
  if (pruned) {
    w.zmax = take(sizeof(float) * (size_t)N * B * (w.Vhp / 128));
    w.zwritten = take((size_t)N * B * (w.Vhp / 128));
    w.cand = take(plan_pruned_lists(B, N, k).total);
  }
  if (dtype == DSPARK_F32) {          // the CUDA-core chain keeps one corrected row per block
    w.zc = take(sizeof(float) * (size_t)B * w.ldz);   // and each CTA's k best of every slot
    if ((size_t)B * N <= (size_t)kSimtFusedRows)      // (or every slot's ranked values)
      w.zk = take(sizeof(float) * (size_t)N * B * w.ldz);
    const size_t per = (size_t)N * B * simt_chain_ctas_max(Vh) * k;
    w.dense_val = take(sizeof(float) * per);
    w.dense_id = take(sizeof(int32_t) * per);
  } else if (!pruned) {               // the dense chain's candidate rows, per CTA
    const size_t per = (size_t)N * B * kChainMaxCtas;
    w.dense_cnt = take(sizeof(int32_t) * per);
    w.dense_val = take(sizeof(float) * per * kDenseLocal);
    w.dense_id = take(sizeof(int32_t) * per * kDenseLocal);
  }
  w.conf = take(sizeof(float) * (size_t)B * N);
  w.total = off;
  return w;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The pruned chain runs for bf16 heads that come with a prepared buffer.
static bool use_pruned(const dspark_config* c, const dspark_head* h) {
  return c->dtype == DSPARK_BF16 && h->prepared != nullptr && c->r % 8 == 0;
}

// Host-side checks; on success fills N and i_first_pred.
static dspark_status validate(const dspark_config* c, const dspark_head* h, int* N,
                              int* ifp) {
  if (!c) return fail(DSPARK_ERR_INVALID_ARG, "config is NULL");
  if (!h) return fail(DSPARK_ERR_INVALID_ARG, "head is NULL");
  if (c->B < 1 || c->L_in < 1 || c->H < 1 || c->V < 1 || c->r < 1)
    return fail(DSPARK_ERR_INVALID_ARG, "B, L_in, H, V and r must all be >= 1");
  if (c->sample_from_anchor != 0 && c->sample_from_anchor != 1)
    return fail(DSPARK_ERR_INVALID_ARG, "sample_from_anchor must be 0 or 1");
  if (c->topk_markov != 0 && c->topk_markov != 1)
    return fail(DSPARK_ERR_INVALID_ARG, "topk_markov must be 0 or 1");
  if (c->skip_truncated != 0 && c->skip_truncated != 1)
    return fail(DSPARK_ERR_INVALID_ARG, "skip_truncated must be 0 or 1");
  if (c->dtype != DSPARK_F32 && c->dtype != DSPARK_BF16)
    return fail(DSPARK_ERR_INVALID_ARG, "dtype must be DSPARK_F32 or DSPARK_BF16");
  if (!c->sample_from_anchor && c->L_in < 2)
    return fail(DSPARK_ERR_INVALID_ARG, "the 1+N bonus-anchor layout needs L_in >= 2");
  if (!(c->conf_min == c->conf_min))
    return fail(DSPARK_ERR_INVALID_ARG, "conf_min is NaN");
  if (!h->lm_head || !h->markov_w1 || !h->markov_w2)
    return fail(DSPARK_ERR_INVALID_ARG, "lm_head, markov_w1 and markov_w2 are required");
  if (h->V_head < 1 || h->V_head > c->V)
    return fail(DSPARK_ERR_INVALID_ARG, "V_head must be in [1, V]");
  if (!h->d2t && h->V_head != c->V)
    return fail(DSPARK_ERR_INVALID_ARG, "without d2t, V_head must equal V");
  if (c->top_k < 1 || c->top_k > 32 || c->top_k > h->V_head)
    return fail(DSPARK_ERR_INVALID_ARG, "top_k must be in [1, min(32, V_head)]");
  if (c->r > 4096) return fail(DSPARK_ERR_UNSUPPORTED, "Markov rank above 4096");
  if ((long long)c->B * c->L_in > (1ll << 30) || (long long)c->V * c->r > (1ll << 40))
    return fail(DSPARK_ERR_UNSUPPORTED, "sizes too large");
  if (c->dtype == DSPARK_BF16) {
    if (c->H % 8 != 0)
      return fail(DSPARK_ERR_UNSUPPORTED, "bf16 path needs H % 8 == 0 (16-byte rows)");
    if (h->V_head % 8 != 0)
      return fail(DSPARK_ERR_UNSUPPORTED, "bf16 path needs V_head % 8 == 0 (16-byte rows)");
    if (!aligned(h->lm_head, 16) || !aligned(h->markov_w2, 16) || !aligned(h->markov_w1, 16))
      return fail(DSPARK_ERR_INVALID_ARG, "bf16 weights must be 16-byte aligned");
  }
  if (c->dtype == DSPARK_BF16 && (c->sample_from_anchor ? c->L_in : c->L_in - 1) > 256)
    return fail(DSPARK_ERR_UNSUPPORTED, "bf16 path takes at most 256 prediction slots");
  if (c->dtype == DSPARK_BF16 && c->r > 512)
    return fail(DSPARK_ERR_UNSUPPORTED, "bf16 path takes a Markov rank of at most 512");
  *N = c->sample_from_anchor ? c->L_in : c->L_in - 1;
  *ifp = c->sample_from_anchor ? 0 : 1;
  return DSPARK_OK;
}

// ------------------------------------------------------------------ compact heads
// A bf16 head in the bias form (full-V lm_head, lm_bias marking the rows the draft cannot
// emit) whose prepared buffer holds its compact form: every proposal then runs on the
// emittable rows only (the d2t form), with the same results.
static bool bias_form(const dspark_config* c, const dspark_head* h) {
  return c->dtype == DSPARK_BF16 && h->lm_bias && !h->d2t && h->V_head == c->V;
}

namespace {
std::mutex g_compact_mu;
struct CompactEntry {
  const void* prepared;
  CompactHeader h;
};
std::vector<CompactEntry> g_compact;   // per prepared buffer, what dspark_prepare_head wrote
}  // namespace

static bool compact_matches(const CompactHeader& h, const dspark_config* c,
                            const dspark_head* hd) {
  return h.magic == kCompactMagic && h.V == c->V && h.H == c->H && h.r == c->r &&
         h.n_emit >= 1 && h.n_pad >= h.n_emit && h.n_pad % 8 == 0 &&
         h.lm_head == (unsigned long long)(uintptr_t)hd->lm_head &&
         h.lm_bias == (unsigned long long)(uintptr_t)hd->lm_bias &&
         h.w1 == (unsigned long long)(uintptr_t)hd->markov_w1 &&
         h.w2 == (unsigned long long)(uintptr_t)hd->markov_w2;
}

static void remember_compact(const void* prepared, const CompactHeader& h) {
  std::lock_guard<std::mutex> lock(g_compact_mu);
  for (CompactEntry& x : g_compact)
    if (x.prepared == prepared) {
      x.h = h;
      return;
    }
  if (g_compact.size() >= 256) g_compact.erase(g_compact.begin());
  g_compact.push_back({prepared, h});
}

// For a bias-form head whose prepared buffer holds its compact form: 1 and the compact
// head in *hc when the call's top_k is within the emittable rows; -1 and, in *hc, the
// full head without the prepared buffer (the dense chain over every row) when it is not.
// 0 for any other head (used as given).  A prepared buffer this process has not
// prepared is read once (synchronously) to learn its row count.
static int resolve_compact(const dspark_config* cfg, const dspark_head* head, dspark_head* hc) {
  if (!bias_form(cfg, head) || !head->prepared) return 0;
  CompactHeader h{};
  bool found = false;
  {
    std::lock_guard<std::mutex> lock(g_compact_mu);
    for (const CompactEntry& x : g_compact)
      if (x.prepared == head->prepared) {
        h = x.h;
        found = true;
      }
  }
  if (!found) {
    if (cudaMemcpy(&h, head->prepared, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    if (!compact_matches(h, cfg, head)) return 0;
    remember_compact(head->prepared, h);
  }
  if (!compact_matches(h, cfg, head)) return 0;
  if (cfg->top_k > h.n_emit) {
    *hc = *head;
    hc->prepared = nullptr;
    return -1;
  }
  const CompactLayout l = plan_compact(cfg->V, cfg->H, cfg->r, h.n_pad);
  const char* base = (const char*)head->prepared;
  *hc = *head;
  hc->lm_head = base + l.lm_head;
  hc->lm_bias = (const float*)(base + l.bias);
  hc->d2t = (const int32_t*)(base + l.list);
  hc->V_head = h.n_pad;
  hc->markov_w2 = base + l.w2;
  hc->prepared = base + l.prepared;
  return 1;
}

// Emittable rows of a bias (bias > -1e8), counted on the device; synchronous.
static __device__ int g_emit_count;
static dspark_status count_emittable(const float* bias, int V, cudaStream_t stream, int* n) {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  void* dev = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&dev, g_emit_count);
  if (e == cudaSuccess) e = launch_emit_count(bias, V, (int*)dev, stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(n, dev, sizeof(int), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "counting the emittable rows");
  return DSPARK_OK;
}

// Workspace of a proposal with this head: enough for the head as given and for its
// compact form, so that one size serves both.
static size_t propose_ws_bytes(const dspark_config* cfg, const dspark_head* head, int N) {
  // (a prepared head runs the dense chain when the logits output is asked for)
  auto both = [&](const dspark_head* h) {
    size_t n = plan_workspace(cfg->B, N, h->V_head, cfg->top_k, cfg->dtype, false).total;
    if (use_pruned(cfg, h))
      n = std::max(n, plan_workspace(cfg->B, N, h->V_head, cfg->top_k, cfg->dtype, true).total);
    return n;
  };
  size_t n = both(head);
  dspark_head hc;
  if (resolve_compact(cfg, head, &hc) != 0) n = std::max(n, both(&hc));
  return n;
}

}  // namespace dspark

using namespace dspark;

static_assert(sizeof(dspark_config) == 44, "dspark_config layout");
static_assert(sizeof(dspark_head) == 72, "dspark_head layout");
static_assert(sizeof(dspark_outputs) == 48, "dspark_outputs layout");

extern "C" {

int32_t dspark_num_slots(const dspark_config* cfg) {
  if (!cfg || cfg->L_in < 1) return 0;
  if (cfg->sample_from_anchor) return cfg->L_in;
  return cfg->L_in >= 2 ? cfg->L_in - 1 : 0;
}

size_t dspark_propose_workspace_size(const dspark_config* cfg, const dspark_head* head) {
  int N, ifp;
  if (validate(cfg, head, &N, &ifp) != DSPARK_OK) return 0;
  return propose_ws_bytes(cfg, head, N);
}

static dspark_status propose_impl(const dspark_config* cfg, const dspark_head* head_in,
                                  const void* hidden, const int32_t* anchors,
                                  const void* conf_hidden, const dspark_outputs* out,
                                  void* workspace,
                                  size_t workspace_bytes, void* stream,
                                  void* const* events) {
  int N, ifp;
  dspark_status st = validate(cfg, head_in, &N, &ifp);
  if (st != DSPARK_OK) return st;
  if (!hidden || !anchors) return fail(DSPARK_ERR_INVALID_ARG, "hidden and anchors are required");
  if (!out || !out->draft || !out->n_draft)
    return fail(DSPARK_ERR_INVALID_ARG, "outputs draft and n_draft are required");
  // a bias-form head prepared in its compact form runs on its emittable rows (unless the
  // logits output, indexed by every head row, is asked for)
  dspark_head hc;
  const dspark_head* head =
      (!out->logits && resolve_compact(cfg, head_in, &hc) != 0) ? &hc : head_in;
  if (cfg->dtype == DSPARK_BF16 && !aligned(hidden, 16))
    return fail(DSPARK_ERR_INVALID_ARG, "bf16 hidden must be 16-byte aligned");
  if (cfg->dtype == DSPARK_BF16 && conf_hidden && !aligned(conf_hidden, 16))
    return fail(DSPARK_ERR_INVALID_ARG, "bf16 conf_hidden must be 16-byte aligned");
  const bool pruned = use_pruned(cfg, head) && !out->logits;
  if (cfg->skip_truncated && !pruned)
    return fail(DSPARK_ERR_UNSUPPORTED,
                "skip_truncated needs the pruned chain: bf16, a prepared head, no logits "
                "output");
  WorkspaceLayout wl = plan_workspace(cfg->B, N, head->V_head, cfg->top_k, cfg->dtype, pruned);
  if (!workspace || !aligned(workspace, 256))
    return fail(DSPARK_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
  if (workspace_bytes < wl.total)
    return fail(DSPARK_ERR_WORKSPACE, "workspace too small: need " +
                                          std::to_string(wl.total) + " bytes");

  char* ws = (char*)workspace;
  ProposePlan p{};
  p.B = cfg->B; p.L_in = cfg->L_in; p.N = N; p.ifp = ifp; p.H = cfg->H; p.V = cfg->V;
  p.Vh = head->V_head; p.r = cfg->r; p.k = cfg->top_k; p.topk_markov = cfg->topk_markov;
  p.dtype = cfg->dtype; p.conf_min = cfg->conf_min; p.b_conf = head->b_conf;
  p.hidden = hidden; p.anchors = anchors; p.lm_head = head->lm_head;
  p.conf_hidden = conf_hidden ? conf_hidden : hidden;
  p.lm_bias = head->lm_bias; p.d2t = head->d2t; p.w1 = head->markov_w1;
  p.w2 = head->markov_w2; p.w_conf = head->w_conf;
  p.draft = out->draft; p.n_draft = out->n_draft; p.topk_ids = out->topk_ids;
  p.topk_vals = out->topk_vals; p.conf = head->w_conf ? out->conf : nullptr;
  p.logits = out->logits;
  p.ctrl = (uint32_t*)(ws + wl.ctrl);
  p.bar = (unsigned*)(ws + wl.bar);
  p.keys = (unsigned long long*)(ws + wl.keys);
  p.z = (float*)(ws + wl.z);
  p.ldz = wl.ldz;
  p.Vhp = wl.Vhp;
  p.ldb = wl.ldb;
  p.zc = (float*)(ws + wl.zc);
  p.zk = wl.zk ? (float*)(ws + wl.zk) : nullptr;
  p.cand_val = (float*)(ws + wl.dense_val);
  p.cand_id = (int32_t*)(ws + wl.dense_id);
  p.cand_cnt = (int32_t*)(ws + wl.dense_cnt);
  p.bucket = (uint32_t*)(ws + wl.dense_bucket);
  p.conf_ws = (float*)(ws + wl.conf);
  p.stream = (cudaStream_t)stream;
  if (pruned) {
    const PreparedLayout pl = plan_prepared(head->V_head, cfg->r);
    const char* pr = (const char*)head->prepared;
    p.zmax = (float*)(ws + wl.zmax);
    p.w2t = (const __nv_bfloat16*)(pr + pl.w2t);
    p.cnorm = (const float*)(pr + pl.cnorm);
    p.cnmax = (const float*)(pr + pl.cnmax);
    p.w1max = (const unsigned*)(pr + pl.w1max);
    p.prep = (const PreparedHeader*)(pr + pl.header);
    p.prep_want.magic = kPreparedMagic;
    p.prep_want.V = cfg->V;
    p.prep_want.Vh = head->V_head;
    p.prep_want.r = cfg->r;
    p.prep_want.w1 = (unsigned long long)(uintptr_t)head->markov_w1;
    p.prep_want.w2 = (unsigned long long)(uintptr_t)head->markov_w2;
    const PrunedLists ll = plan_pruned_lists(cfg->B, N, cfg->top_k);
    char* lists = ws + wl.cand;
    p.cand_v = (int32_t*)(lists + ll.cand_v);
    p.cand_z = (float*)(lists + ll.cand_z);
    p.cand_n = (int32_t*)(lists + ll.cand_n);
    p.prev_v = (int32_t*)(lists + ll.prev_v);
    p.prev_n = (int32_t*)(lists + ll.prev_n);
    p.amax = (int32_t*)(lists + ll.amax);
    p.tk_id = (int32_t*)(lists + ll.tk_id);
    p.tk_val = (float*)(lists + ll.tk_val);
    p.z_octet = true;           // the candidate scans read one block's rows of z
    p.walk_done = (int32_t*)(ws + wl.walk_done);
    p.skip_truncated = cfg->skip_truncated != 0;
    // Tiles of z that provably cannot hold a slot's top k are left out by the GEMM when
    // it runs with the prediction rows on M and the top-k ranks corrected logits.
    const bool want_topk = out->topk_ids || out->topk_vals;
    if (logits_gemm_pm(cfg->B, N, true, head->lm_bias) && (!want_topk || cfg->topk_markov)) {
      p.zbound = (uint32_t*)(ws + wl.zbound);
      p.zwritten = (uint8_t*)(ws + wl.zwritten);
      p.zbound_k = want_topk ? cfg->top_k : 1;
    }
  }

  cudaError_t e;
  auto mark = [&](int s) -> cudaError_t {
    return events ? cudaEventRecord((cudaEvent_t)events[s], p.stream) : cudaSuccess;
  };
  // the control words (error word, barrier counters, winner keys) start from zero
  e = launch_zero_block(ws + wl.ctrl, wl.zero_end - wl.ctrl, p.stream);
  if (e != cudaSuccess) return cuda_fail(e, "control reset");
  if ((e = mark(DSPARK_STAGE_CONF)) != cudaSuccess) return cuda_fail(e, "event record");
  // the pruned chain evaluates the confidence head and truncation in its own kernels,
  // unless the adaptive block length needs the cuts before the GEMM
  // (small fp32 problems: the confidence head and the base logits run inside the chain's
  // single launch)
  const bool simt_one = p.dtype == DSPARK_F32 &&
                        simt_fused(p.B, p.N, p.H, p.Vh, p.r, p.skip_truncated);
  if ((!pruned || p.skip_truncated) && !simt_one && (e = launch_conf(p)) != cudaSuccess)
    return cuda_fail(e, "confidence kernel");
  if ((e = mark(DSPARK_STAGE_LOGITS)) != cudaSuccess) return cuda_fail(e, "event record");
  e = p.dtype == DSPARK_BF16 ? launch_base_logits_tc(p)
                             : (simt_one ? cudaSuccess : launch_base_logits_simt(p));
  if (e != cudaSuccess) return cuda_fail(e, "base logits");
  if ((e = mark(DSPARK_STAGE_CHAIN)) != cudaSuccess) return cuda_fail(e, "event record");
  e = p.dtype == DSPARK_F32 ? launch_chain_simt(p)
                            : (pruned ? launch_chain_pruned(p) : launch_chain_dense(p));
  if (e != cudaSuccess) return cuda_fail(e, "chain");
  if ((e = mark(DSPARK_STAGE_TOPK)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = mark(DSPARK_NUM_STAGES)) != cudaSuccess) return cuda_fail(e, "event record");
  return DSPARK_OK;
}

dspark_status dspark_propose(const dspark_config* cfg, const dspark_head* head,
                             const void* hidden, const int32_t* anchors,
                             const void* conf_hidden, const dspark_outputs* out,
                             void* workspace, size_t workspace_bytes, void* stream) {
  return propose_impl(cfg, head, hidden, anchors, conf_hidden, out, workspace,
                      workspace_bytes, stream, nullptr);
}

dspark_status dspark_propose_timed(const dspark_config* cfg, const dspark_head* head,
                                   const void* hidden, const int32_t* anchors,
                                   const void* conf_hidden, const dspark_outputs* out,
                                   void* workspace, size_t workspace_bytes, void* stream,
                                   void* const* events) {
  if (!events) return fail(DSPARK_ERR_INVALID_ARG, "events is NULL");
  for (int s = 0; s <= DSPARK_NUM_STAGES; ++s)
    if (!events[s]) return fail(DSPARK_ERR_INVALID_ARG, "an event is NULL");
  return propose_impl(cfg, head, hidden, anchors, conf_hidden, out, workspace,
                      workspace_bytes, stream, events);
}

int32_t dspark_propose_kernel_count(const dspark_config* cfg, const dspark_head* head_in,
                                    const dspark_outputs* out) {
  int N, ifp;
  if (validate(cfg, head_in, &N, &ifp) != DSPARK_OK || !out) return -1;
  dspark_head hc;
  const dspark_head* head =
      (!out->logits && resolve_compact(cfg, head_in, &hc) != 0) ? &hc : head_in;
  // every pass starts with the kernel that zeroes the control block
  if (cfg->dtype == DSPARK_F32)                         // confidence, GEMM, chain; or the
    return 1 + (simt_fused(cfg->B, N, cfg->H, head->V_head, cfg->r, cfg->skip_truncated != 0)
                    ? 1                                 // chain alone, for small problems
                    : 3);
  if (use_pruned(cfg, head) && !out->logits)            // GEMM; tables with the walk;
    return 1 + (cfg->skip_truncated ? 3 : 2);           // confidence first when adaptive
  const bool topk = out->topk_ids || out->topk_vals;
  int sms = 0;
  if (device_sms(&sms) != cudaSuccess) {
    cudaGetLastError();
    sms = 152;
  }
  const int group = dense_chain_group(head->V_head, sms);
  const bool merge = topk && (cfg->top_k > 1 || !cfg->topk_markov);
  return 1 /* control block */ + 1 /* confidence */ + 1 /* GEMM */ +
         (cfg->B + group - 1) / std::max(group, 1) /* chain, one launch per group */ +
         (merge ? 1 : 0);
}

// staging for dspark_step_host, placed after dspark_propose's workspace
struct StageLayout {
  size_t hidden, conf_hidden, anchors, target, draft, n_draft, accepted, bonus, tk_ids, tk_vals, total;
};
static StageLayout plan_stage(const dspark_config* c, int N, size_t base, bool conf_input) {
  StageLayout s{};
  size_t es = c->dtype == DSPARK_BF16 ? 2 : 4;
  size_t off = base;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, kAlign); return o; };
  s.hidden = take(es * (size_t)c->B * c->L_in * c->H);
  s.conf_hidden = take(conf_input ? es * (size_t)c->B * c->L_in * c->H : 0);
  s.anchors = take(4 * (size_t)c->B);
  s.target = take(4 * (size_t)c->B * (N + 1));
  s.draft = take(4 * (size_t)c->B * N);
  s.n_draft = take(4 * (size_t)c->B);
  s.accepted = take(4 * (size_t)c->B);
  s.bonus = take(4 * (size_t)c->B);
  s.tk_ids = take(4 * (size_t)c->B * N * c->top_k);
  s.tk_vals = take(4 * (size_t)c->B * N * c->top_k);
  s.total = off;
  return s;
}

size_t dspark_step_host_workspace_size(const dspark_config* cfg, const dspark_head* head) {
  int N, ifp;
  if (validate(cfg, head, &N, &ifp) != DSPARK_OK) return 0;
  // (room for a separate confidence input is always planned, so one size fits both)
  return plan_stage(cfg, N, propose_ws_bytes(cfg, head, N), true).total;
}

dspark_status dspark_step_host(const dspark_config* cfg, const dspark_head* head,
                               const void* hidden_h, const int32_t* anchors_h,
                               const void* conf_hidden_h,
                               const int32_t* target_h, int32_t* draft_h,
                               int32_t* n_draft_h, int32_t* accepted_h, int32_t* bonus_h,
                               int32_t* topk_ids_h, float* topk_vals_h,
                               void* workspace, size_t workspace_bytes, void* stream) {
  int N, ifp;
  dspark_status st = validate(cfg, head, &N, &ifp);
  if (st != DSPARK_OK) return st;
  if (!hidden_h || !anchors_h || !target_h || !draft_h || !n_draft_h || !accepted_h || !bonus_h)
    return fail(DSPARK_ERR_INVALID_ARG, "a required host buffer is NULL");
  size_t base = propose_ws_bytes(cfg, head, N);
  StageLayout s = plan_stage(cfg, N, base, true);
  if (!workspace || !aligned(workspace, 256))
    return fail(DSPARK_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
  if (workspace_bytes < s.total)
    return fail(DSPARK_ERR_WORKSPACE, "workspace too small: need " + std::to_string(s.total) +
                                          " bytes");
  char* ws = (char*)workspace;
  cudaStream_t cs = (cudaStream_t)stream;
  const size_t es = cfg->dtype == DSPARK_BF16 ? 2 : 4;
  const size_t B = cfg->B, k = cfg->top_k;
  cudaError_t e;
  auto h2d = [&](size_t off, const void* src, size_t bytes) {
    return cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, cs);
  };
  auto d2h = [&](void* dst, size_t off, size_t bytes) {
    return cudaMemcpyAsync(dst, ws + off, bytes, cudaMemcpyDeviceToHost, cs);
  };
  // Page-locked host buffers that the GPU can address (cudaHostAlloc / cudaHostRegister
  // with a device mapping) are read and written by the kernels in place: each small copy
  // costs more in fixed overhead than its bytes.  The hidden states, the one large
  // input, still go by copy (the TMA loads of the GEMM need device memory).
  auto device_view = [](const void* h) -> void* {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, h) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
  };
  if ((e = h2d(s.hidden, hidden_h, es * B * cfg->L_in * cfg->H)) != cudaSuccess)
    return cuda_fail(e, "host-to-device copy");
  if (conf_hidden_h &&
      (e = h2d(s.conf_hidden, conf_hidden_h, es * B * cfg->L_in * cfg->H)) != cudaSuccess)
    return cuda_fail(e, "host-to-device copy");
  const int32_t* anchors_d = (const int32_t*)device_view(anchors_h);
  const int32_t* target_d = (const int32_t*)device_view(target_h);
  if (!anchors_d) {
    if ((e = h2d(s.anchors, anchors_h, 4 * B)) != cudaSuccess)
      return cuda_fail(e, "host-to-device copy");
    anchors_d = (const int32_t*)(ws + s.anchors);
  }
  if (!target_d) {
    if ((e = h2d(s.target, target_h, 4 * B * (N + 1))) != cudaSuccess)
      return cuda_fail(e, "host-to-device copy");
    target_d = (const int32_t*)(ws + s.target);
  }
  // outputs: in place when every one of them is addressable, else staged and copied
  void* out_d[6] = {device_view(draft_h), device_view(n_draft_h), device_view(accepted_h),
                    device_view(bonus_h), topk_ids_h ? device_view(topk_ids_h) : nullptr,
                    topk_vals_h ? device_view(topk_vals_h) : nullptr};
  const bool in_place = out_d[0] && out_d[1] && out_d[2] && out_d[3] &&
                        (!topk_ids_h || out_d[4]) && (!topk_vals_h || out_d[5]);
  dspark_outputs o{};
  o.draft = in_place ? (int32_t*)out_d[0] : (int32_t*)(ws + s.draft);
  o.n_draft = in_place ? (int32_t*)out_d[1] : (int32_t*)(ws + s.n_draft);
  o.topk_ids = !topk_ids_h ? nullptr : in_place ? (int32_t*)out_d[4] : (int32_t*)(ws + s.tk_ids);
  o.topk_vals = !topk_vals_h ? nullptr : in_place ? (float*)out_d[5] : (float*)(ws + s.tk_vals);
  int32_t* accepted_d = in_place ? (int32_t*)out_d[2] : (int32_t*)(ws + s.accepted);
  int32_t* bonus_d = in_place ? (int32_t*)out_d[3] : (int32_t*)(ws + s.bonus);
  st = propose_impl(cfg, head, ws + s.hidden, anchors_d,
                    conf_hidden_h ? (const void*)(ws + s.conf_hidden) : nullptr, &o, workspace,
                    base, stream, nullptr);
  if (st != DSPARK_OK) return st;
  st = dspark_verify(cfg->B, N, o.draft, o.n_draft, target_d, accepted_d, bonus_d, nullptr,
                     stream);
  if (st != DSPARK_OK) return st;
  if (in_place) return DSPARK_OK;
  if ((e = d2h(draft_h, s.draft, 4 * B * N)) != cudaSuccess ||
      (e = d2h(n_draft_h, s.n_draft, 4 * B)) != cudaSuccess ||
      (e = d2h(accepted_h, s.accepted, 4 * B)) != cudaSuccess ||
      (e = d2h(bonus_h, s.bonus, 4 * B)) != cudaSuccess)
    return cuda_fail(e, "device-to-host copy");
  if (topk_ids_h && (e = d2h(topk_ids_h, s.tk_ids, 4 * B * N * k)) != cudaSuccess)
    return cuda_fail(e, "device-to-host copy");
  if (topk_vals_h && (e = d2h(topk_vals_h, s.tk_vals, 4 * B * N * k)) != cudaSuccess)
    return cuda_fail(e, "device-to-host copy");
  return DSPARK_OK;
}

dspark_status dspark_verify(int32_t B, int32_t N, const int32_t* draft,
                            const int32_t* n_draft, const int32_t* target,
                            int32_t* accepted, int32_t* bonus, int32_t* emitted,
                            void* stream) {
  if (B < 1 || N < 1) return fail(DSPARK_ERR_INVALID_ARG, "B and N must be >= 1");
  if (!draft || !n_draft || !target || !accepted || !bonus)
    return fail(DSPARK_ERR_INVALID_ARG, "draft, n_draft, target, accepted, bonus are required");
  cudaError_t e = launch_verify(B, N, draft, n_draft, target, accepted, bonus, emitted,
                                (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "verify kernel");
  return DSPARK_OK;
}

dspark_status dspark_tree_verify(int32_t B, int32_t N, int32_t top_k,
                                 const int32_t* topk_ids, const int32_t* n_draft,
                                 const int32_t* target, int32_t* accepted, int32_t* bonus,
                                 int32_t* emitted, int32_t* path, void* stream) {
  if (B < 1 || N < 1) return fail(DSPARK_ERR_INVALID_ARG, "B and N must be >= 1");
  if (top_k < 1 || top_k > 32) return fail(DSPARK_ERR_INVALID_ARG, "top_k must be in [1, 32]");
  if (!topk_ids || !n_draft || !target || !accepted || !bonus)
    return fail(DSPARK_ERR_INVALID_ARG,
                "topk_ids, n_draft, target, accepted and bonus are required");
  cudaError_t e = launch_tree_verify(B, N, top_k, topk_ids, n_draft, target, accepted, bonus,
                                     emitted, path, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "tree verify kernel");
  return DSPARK_OK;
}

dspark_status dspark_device_status(void* workspace, void* stream) {
  if (!workspace) return fail(DSPARK_ERR_INVALID_ARG, "workspace is NULL");
  uint32_t word = 0;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  if (word == 0) return DSPARK_OK;
  e = cudaMemsetAsync(workspace, 0, sizeof(word), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  if (word & kErrTimeout) return fail(DSPARK_ERR_TIMEOUT, "a device-side wait timed out");
  if (word & kErrPrepared)
    return fail(DSPARK_ERR_DEVICE,
                "head->prepared was prepared for other weights or sizes (run "
                "dspark_prepare_head for this head)");
  return fail(DSPARK_ERR_DEVICE, "a kernel saw a token outside [0, V)");
}

dspark_status dspark_pass_stats(void* workspace, void* stream, int32_t* on_the_fly,
                                int32_t* every_row, int32_t* dense_overflow) {
  if (!workspace) return fail(DSPARK_ERR_INVALID_ARG, "workspace is NULL");
  uint32_t w[4] = {0, 0, 0, 0};
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(w, workspace, sizeof(w), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the pass counters");
  if (on_the_fly) *on_the_fly = (int32_t)w[kCtrlOnTheFly];
  if (every_row) *every_row = (int32_t)w[kCtrlEveryRow];
  if (dense_overflow) *dense_overflow = (int32_t)w[kCtrlDenseOver];
  return DSPARK_OK;
}

dspark_status dspark_wait_selftest(void* workspace, size_t workspace_bytes,
                                   int64_t budget_cycles, int32_t pre_abort, void* stream) {
  if (!workspace || !aligned(workspace, 256))
    return fail(DSPARK_ERR_WORKSPACE, "workspace must be non-NULL and 256-byte aligned");
  if (workspace_bytes < 256)
    return fail(DSPARK_ERR_WORKSPACE, "workspace too small: need 256 bytes");
  if (budget_cycles < 1 || budget_cycles > kMaxSelftestBudget)
    return fail(DSPARK_ERR_INVALID_ARG, "budget_cycles must be in [1, 2e9]");
  if (pre_abort != 0 && pre_abort != 1)
    return fail(DSPARK_ERR_INVALID_ARG, "pre_abort must be 0 or 1");
  cudaError_t e = launch_wait_selftest((uint32_t*)workspace, (long long)budget_cycles,
                                       pre_abort, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test kernel");
  return DSPARK_OK;
}

size_t dspark_prepare_head_size(const dspark_config* cfg, const dspark_head* head) {
  int N, ifp;
  if (validate(cfg, head, &N, &ifp) != DSPARK_OK || cfg->dtype != DSPARK_BF16) return 0;
  if (bias_form(cfg, head)) {
    int n = 0;
    if (count_emittable(head->lm_bias, cfg->V, 0, &n) != DSPARK_OK) return 0;
    if (n >= 1 && n < cfg->V)
      return plan_compact(cfg->V, cfg->H, cfg->r, (int)align_up((size_t)n, 8)).total;
  }
  return plan_prepared(head->V_head, cfg->r).total;
}

dspark_status dspark_prepare_head(const dspark_config* cfg, const dspark_head* head,
                                  void* prepared, size_t prepared_bytes, void* stream) {
  int N, ifp;
  dspark_status st = validate(cfg, head, &N, &ifp);
  if (st != DSPARK_OK) return st;
  if (cfg->dtype != DSPARK_BF16)
    return fail(DSPARK_ERR_UNSUPPORTED, "head preparation is for the bf16 path");
  const PreparedLayout pl = plan_prepared(head->V_head, cfg->r);
  if (!prepared || !aligned(prepared, 256))
    return fail(DSPARK_ERR_WORKSPACE, "prepared buffer must be non-NULL and 256-byte aligned");
  if (bias_form(cfg, head)) {
    // the compact form: the emittable rows (counted first, synchronously, to size it)
    int n = 0;
    st = count_emittable(head->lm_bias, cfg->V, (cudaStream_t)stream, &n);
    if (st != DSPARK_OK) return st;
    if (n >= 1 && n < cfg->V) {
      const int n_pad = (int)align_up((size_t)n, 8);
      const CompactLayout cl = plan_compact(cfg->V, cfg->H, cfg->r, n_pad);
      if (prepared_bytes < cl.total)
        return fail(DSPARK_ERR_WORKSPACE,
                    "prepared buffer too small: need " + std::to_string(cl.total) + " bytes");
      cudaError_t e = launch_prepare_compact(head->lm_head, head->lm_bias, head->markov_w1,
                                             head->markov_w2, cfg->V, cfg->H, cfg->r, n, n_pad,
                                             prepared, (cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_fail(e, "head preparation (compact form)");
      CompactHeader h{};
      h.magic = kCompactMagic;
      h.V = cfg->V;
      h.H = cfg->H;
      h.r = cfg->r;
      h.n_emit = n;
      h.n_pad = n_pad;
      h.lm_head = (unsigned long long)(uintptr_t)head->lm_head;
      h.lm_bias = (unsigned long long)(uintptr_t)head->lm_bias;
      h.w1 = (unsigned long long)(uintptr_t)head->markov_w1;
      h.w2 = (unsigned long long)(uintptr_t)head->markov_w2;
      remember_compact(prepared, h);
      return DSPARK_OK;
    }
  }
  if (prepared_bytes < pl.total)
    return fail(DSPARK_ERR_WORKSPACE,
                "prepared buffer too small: need " + std::to_string(pl.total) + " bytes");
  cudaError_t e = launch_prepare_head(head->markov_w1, head->markov_w2, cfg->V, cfg->r,
                                      head->V_head, prepared, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "head preparation");
  {
    // (a buffer prepared in the ordinary form is no longer a compact one)
    std::lock_guard<std::mutex> lock(g_compact_mu);
    for (size_t i = 0; i < g_compact.size(); ++i)
      if (g_compact[i].prepared == prepared) {
        g_compact.erase(g_compact.begin() + i);
        break;
      }
  }
  return DSPARK_OK;
}

const char* dspark_status_string(int32_t s) {
  switch (s) {
    case DSPARK_OK: return "ok";
    case DSPARK_ERR_INVALID_ARG: return "invalid argument";
    case DSPARK_ERR_UNSUPPORTED: return "unsupported configuration";
    case DSPARK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DSPARK_ERR_CUDA: return "CUDA runtime error";
    case DSPARK_ERR_DEVICE: return "device-side data error";
    case DSPARK_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

const char* dspark_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"

// ------------------------------------------------------------------ no-allocation entry
// Scratch for dspark_propose_noalloc: a fixed array in device memory that exists on every
// GPU that loads this library, from the load until the process exits.  Host code must not
// pass `g_noalloc_scratch` itself to a kernel: on the host that name is only a stand-in,
// so its device address is looked up with cudaGetSymbolAddress while the device is
// current.  The address belongs to the CUDA context that is current (a cudaDeviceReset or
// a caller's own driver-API context gives another one), so it is looked up again on
// every call that is not being captured into a graph, and remembered per context for
// calls that are.
static constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kMaxContexts = 64;
std::mutex g_noalloc_mutex;
struct ScratchEntry {
  void* ctx;
  void* ptr;
};
ScratchEntry g_noalloc_seen[kMaxContexts] = {};
int g_noalloc_next = 0;

// The calling thread's current CUDA context (driver API, reached through the runtime's
// entry-point query so that the library needs no link against libcuda).
dspark_status current_context(void** ctx) {
  using GetCurrent = int (*)(void**);
  static GetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (GetCurrent)p;
  });
  if (!fn) return fail(DSPARK_ERR_CUDA, "cuCtxGetCurrent is not available");
  *ctx = nullptr;
  if (fn(ctx) != 0 || !*ctx) return fail(DSPARK_ERR_CUDA, "no current CUDA context");
  return DSPARK_OK;
}

// The device address of the built-in scratch in the current context.
dspark_status noalloc_scratch(void* stream, void** scratch) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing((cudaStream_t)stream, &cap);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  void* ptr = nullptr;
  if (cap == cudaStreamCaptureStatusNone) {
    // (with the device current; this also brings up its context on a first call)
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch");
  }
  void* ctx = nullptr;
  dspark_status st = current_context(&ctx);
  if (st != DSPARK_OK) return st;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  int slot = -1;
  for (int j = 0; j < kMaxContexts; ++j)
    if (g_noalloc_seen[j].ctx == ctx) slot = j;
  if (cap != cudaStreamCaptureStatusNone) {
    if (slot < 0 || !g_noalloc_seen[slot].ptr)
      return fail(DSPARK_ERR_INVALID_ARG,
                  "dspark_propose_noalloc: make one call on this device outside stream "
                  "capture first (it looks up the built-in scratch)");
    *scratch = g_noalloc_seen[slot].ptr;
    return DSPARK_OK;
  }
  if (slot < 0) {
    slot = g_noalloc_next;
    g_noalloc_next = (g_noalloc_next + 1) % kMaxContexts;
  }
  g_noalloc_seen[slot] = {ctx, ptr};
  *scratch = ptr;
  return DSPARK_OK;
}
}  // namespace

extern "C" {

dspark_status dspark_propose_noalloc(const dspark_config* cfg, const dspark_head* head,
                                     const void* hidden, const int32_t* anchors,
                                     const void* conf_hidden, const dspark_outputs* out,
                                     void* stream) {
  const size_t need = dspark_propose_workspace_size(cfg, head);
  if (need == 0) {
    int N, ifp;
    return validate(cfg, head, &N, &ifp);     // sets the message of the failing check
  }
  if (need > kNoAllocScratchBytes)
    return fail(DSPARK_ERR_WORKSPACE,
                "this call needs " + std::to_string(need) +
                    " bytes of scratch; the built-in scratch of dspark_propose_noalloc holds " +
                    std::to_string(kNoAllocScratchBytes) +
                    " bytes (use dspark_propose with a caller workspace)");
  void* scratch = nullptr;
  dspark_status st = noalloc_scratch(stream, &scratch);
  if (st != DSPARK_OK) return st;
  // the control words that must start at zero (the error word among them) are cleared by
  // dspark_propose itself
  return propose_impl(cfg, head, hidden, anchors, conf_hidden, out, scratch,
                      kNoAllocScratchBytes, stream, nullptr);
}

dspark_status dspark_noalloc_device_status(void* stream) {
  void* scratch = nullptr;
  dspark_status st = noalloc_scratch(stream, &scratch);
  if (st != DSPARK_OK) return st;
  return dspark_device_status(scratch, stream);
}

}  // extern "C"
