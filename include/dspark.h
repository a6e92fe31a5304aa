/*
 * dspark.h -- C ABI of the DSpark proposal head and the greedy verify step.
 *
 * The method (llama.cpp commit 6fed9f6, src/models/dflash.cpp, squash log of
 * "spec: add DSpark speculative decoding", the proposal formula):
 *
 *   logits(i)  = h[b, i] . lm_head^T (+ lm_bias)
 *   logits'(i) = logits(i) + markov_w2^T . markov_w1[prev(i)]
 *   prev(0)    = the block's anchor token,  prev(i > 0) = argmax logits'(i - 1)
 *
 * run greedily over the slots of a block and in parallel over the blocks of a batch,
 * followed by DFlash's unchanged greedy verify/accept.  The confidence head
 * conf = sigmoid(h . w_conf + b_conf) truncates each block at its first slot below
 * conf_min ("spec: add confidence-based draft pruning for DSpark").  Block layouts:
 * anchor-first (every slot predicts) and the 1+N bonus-anchor layout of
 * speculators-format drafts (llama.cpp PR #26275, "Format differences": slot 0 holds
 * the bonus token and is not a prediction slot).  Reduced draft vocabularies come in
 * the two forms PR #26275 describes: an lm_head expanded to the full vocabulary with a
 * -1e9 bias on rows the draft cannot emit, or a compact head plus a d2t table of
 * absolute target ids.
 *
 * Conventions shared by every entry point:
 *   - Pointers named "device" must point to device memory of the current device;
 *     "host" pointers to host memory.  The caller owns every buffer; the library keeps
 *     no pointer after a call returns and allocates no device memory.
 *   - Arrays are dense and row-major with the shapes given; element types are the
 *     config's dtype for the tensors marked "dtype", int32 / fp32 otherwise.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) unless stated otherwise.
 *   - dspark_propose and dspark_verify can be captured into a CUDA graph (stream
 *     capture) and replayed; a replay reads the buffers the captured call was given, so
 *     refill them in place between replays.  Make one direct call on the device before
 *     the first capture: it does the library's one-time per-device set-up.
 *   - Argument errors detectable on the host return before anything is launched and
 *     leave every output untouched.  Problems only the device can see (an anchor
 *     outside [0, V), a bounded wait that gave up, a prepared buffer made for another
 *     head) set bits of an error word in the workspace.  Each dspark_propose call clears
 *     that word when it starts, so it describes the latest call on that workspace; read
 *     it with dspark_device_status().
 *   - dspark_last_error() returns a message for the calling thread's last failure.
 */
#ifndef DSPARK_H_
#define DSPARK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dspark_status {
  DSPARK_OK = 0,
  DSPARK_ERR_INVALID_ARG = 1,  /* a NULL required pointer, a bad size, a bad flag */
  DSPARK_ERR_UNSUPPORTED = 2,  /* valid in principle but outside what the kernels take */
  DSPARK_ERR_WORKSPACE = 3,    /* workspace NULL, misaligned or too small */
  DSPARK_ERR_CUDA = 4,         /* a CUDA runtime call failed (message has the details) */
  DSPARK_ERR_DEVICE = 5,       /* a kernel saw bad data (e.g. an anchor outside [0, V)) */
  DSPARK_ERR_TIMEOUT = 6       /* a bounded device-side wait gave up */
} dspark_status;

typedef enum dspark_dtype {
  DSPARK_F32 = 0,   /* fp32 operands, fp32 FMA arithmetic */
  DSPARK_BF16 = 1   /* bf16 operands, fp32 accumulation on the tensor cores */
} dspark_dtype;

/* Sizes and knobs of one call. */
typedef struct dspark_config {
  int32_t B;                  /* blocks in the batch, >= 1 */
  int32_t L_in;               /* slots per block in `hidden`, >= 1 (>= 2 for 1+N) */
  int32_t H;                  /* hidden size, >= 1 (multiple of 8 for bf16) */
  int32_t V;                  /* vocabulary: token ids are in [0, V) */
  int32_t r;                  /* Markov rank, >= 1 */
  int32_t top_k;              /* candidates kept per slot, 1 .. min(32, V_head) */
  int32_t sample_from_anchor; /* 1: anchor-first, N = L_in prediction slots reading
                                 hidden rows 0..L_in-1;
                                 0: 1+N bonus anchor, N = L_in - 1 slots reading
                                 hidden rows 1..L_in-1 (row 0 is the bonus token) */
  int32_t topk_markov;        /* 1: top-k ranks the corrected logits (the lattice
                                 candidates get the Markov bias, lucebox PR #626);
                                 0: top-k ranks the base logits */
  float conf_min;             /* truncate at the first slot with conf < conf_min;
                                 <= 0 disables truncation (n_draft = N) */
  int32_t dtype;              /* dspark_dtype of hidden, lm_head, markov_w1/w2, w_conf */
  int32_t skip_truncated;     /* 0: every slot is drafted; n_draft only marks the cut.
                                 1: adaptive block length -- the confidences and n_draft
                                 are computed first, and the slots of block b from
                                 n_draft[b] on are not drafted: draft and topk_ids read
                                 -1 there, topk_vals NaN (llama.cpp DSpark log,
                                 confidence-based draft pruning: verify reads nothing
                                 past the cut).  bf16 with a prepared head and no logits
                                 output only (DSPARK_ERR_UNSUPPORTED otherwise). */
} dspark_config;

/* The drafter head's weights (device memory, not modified). */
typedef struct dspark_head {
  const void* lm_head;        /* device [V_head, H], dtype */
  const float* lm_bias;       /* device [V_head] fp32, or NULL.  A bias <= -1e8 marks a
                                 row the draft cannot emit (never chosen while any
                                 other row is finite) */
  const int32_t* d2t;         /* device [V_head] int32, strictly increasing token ids in
                                 [0, V): row j of lm_head / column j of markov_w2 is
                                 token d2t[j].  NULL: row j is token j and V_head == V */
  int32_t V_head;             /* rows of lm_head = columns of markov_w2 (multiple of 8
                                 for bf16) */
  const void* markov_w1;      /* device [V, r], dtype; row p is gathered for prev = p */
  const void* markov_w2;      /* device [r, V_head], dtype */
  const void* w_conf;         /* device [H], dtype, or NULL (no confidence head:
                                 conf output is not written, n_draft = N) */
  float b_conf;
  const void* prepared;       /* device buffer filled by dspark_prepare_head() for these
                                 weights, or NULL.  With it (bf16 only), the chain runs
                                 the exact-bound pruned form: same results, the Markov
                                 term evaluated only where it can change them.  Without
                                 it, or when the logits output is requested, the chain
                                 evaluates every head row (dense form). */
} dspark_head;

/* Outputs of dspark_propose (device memory).  N = dspark_num_slots(cfg). */
typedef struct dspark_outputs {
  int32_t* draft;             /* required [B, N]: the greedy chain's tokens; all N slots
                                 are filled and truncation only sets n_draft, except
                                 with skip_truncated = 1 (-1 from n_draft[b] on) */
  int32_t* n_draft;           /* required [B]: truncated draft length, 0..N */
  int32_t* topk_ids;          /* [B, N, top_k] token ids by value descending, ties to
                                 the lower id; or NULL */
  float* topk_vals;           /* [B, N, top_k] the ranked logits of topk_ids; or NULL */
  float* conf;                /* [B, N] confidences; or NULL */
  float* logits;              /* [B, N, V_head] corrected logits (column j = head row
                                 j); or NULL.  Costs a full write; meant for tests */
} dspark_outputs;

/* N, the prediction slots per block (L_in or L_in - 1); 0 on invalid input. */
int32_t dspark_num_slots(const dspark_config* cfg);

/* Bytes of device workspace dspark_propose needs for this config and head; 0 on
   invalid input.  The workspace must be 256-byte aligned.  Its contents need no
   initialisation and are scratch between calls; each call clears the error word that
   dspark_device_status() reads, so that word describes the latest call. */
size_t dspark_propose_workspace_size(const dspark_config* cfg, const dspark_head* head);

/*
 * dspark_propose -- the whole proposal of one batch.
 *
 * hidden  device [B, L_in, H] dtype: the drafter's final hidden states
 * anchors device [B] int32: token 0 of every block (the dedicated anchor input of the
 *         llama.cpp squash log; in the 1+N layout the bonus token), each in [0, V)
 * conf_hidden device [B, L_in, H] dtype, or NULL: a separate input of the confidence
 *         head (lucebox PR #626, summary: a calibrated confidence export taken before
 *         the final norm).  When given, the confidence head reads it in place of
 *         `hidden`, slot for slot; the logits and the chain still read `hidden`.  NULL:
 *         the confidence head reads `hidden`.
 * out     the outputs above
 *
 * Steps, all on the device: (a) emittable-row handling from lm_bias / d2t;
 * (b) base logits of every prediction slot over the head's rows; (c) the confidence
 * head and the truncation length; (d) the Markov-corrected greedy chain over the N
 * slots, vectorised over blocks; (e) top-k per slot.  Not reentrant on one workspace:
 * calls that share a workspace must be ordered on the GPU.
 */
dspark_status dspark_propose(const dspark_config* cfg, const dspark_head* head,
                             const void* hidden, const int32_t* anchors,
                             const void* conf_hidden, const dspark_outputs* out,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * dspark_verify -- DFlash's greedy verify/accept (unchanged by DSpark).
 *
 * draft    device [B, N] int32      n_draft device [B] int32 (values outside [0, N] are
 *                                    clamped to that range)
 * target   device [B, N + 1] int32: the target model's argmax after the anchor and after
 *          each drafted slot
 * accepted device [B] int32: a = the longest prefix j <= n_draft[b] with
 *          draft[b, 0..j-1] == target[b, 0..j-1]
 * bonus    device [B] int32: target[b, a]
 * emitted  device [B, N + 1] int32 or NULL: draft[b, 0..a-1], then the bonus token, then
 *          -1; with greedy decoding this equals the target's own argmax sequence.
 */
dspark_status dspark_verify(int32_t B, int32_t N, const int32_t* draft,
                            const int32_t* n_draft, const int32_t* target,
                            int32_t* accepted, int32_t* bonus, int32_t* emitted,
                            void* stream);

/*
 * dspark_tree_verify -- greedy verify of the top-k candidate lattice (the tree consumer
 * of the per-slot candidates; lucebox PR #626, description: the DDTree's candidate
 * top-k gets the Markov bias; onnxruntime-genai PR #2490, DFlash 2 / DSpark builder
 * commits: the runtime walks the drafter's candidate lattice greedily).
 *
 * The tree is the whole lattice: every candidate of slot i is a child of every candidate
 * of slot i - 1, down to depth n_draft[b] (the pages define no other construction).  A
 * greedy target accepts the child equal to its argmax after the accepted prefix; as that
 * prefix is always the target's own tokens, the argmax at depth i is target[b, i].
 *
 * topk_ids device [B, N, top_k] int32: the candidates of dspark_propose (topk_ids)
 * n_draft  device [B] int32 (clamped to [0, N])
 * target   device [B, N + 1] int32: the target model's argmax tokens along its own
 *          greedy continuation
 * accepted device [B] int32: a = the largest j <= n_draft[b] such that target[b, i] is
 *          among topk_ids[b, i, :] for every i < j
 * bonus    device [B] int32: target[b, a]
 * emitted  device [B, N + 1] int32 or NULL: target[b, 0..a], then -1 (greedy lossless)
 * path     device [B, N] int32 or NULL: for i < a the rank q with
 *          topk_ids[b, i, q] == target[b, i] (the first such q), -1 from a on
 *
 * With top_k = 1 it equals dspark_verify on the greedy draft.  Host-detectable errors
 * (sizes, NULL required pointers) return before any launch.
 */
dspark_status dspark_tree_verify(int32_t B, int32_t N, int32_t top_k,
                                 const int32_t* topk_ids, const int32_t* n_draft,
                                 const int32_t* target, int32_t* accepted, int32_t* bonus,
                                 int32_t* emitted, int32_t* path, void* stream);

/* Bytes of the buffer dspark_prepare_head() fills for this head (bf16 only; 0 on invalid
   input or fp32).  Layout: a 256-byte header recording what the buffer was prepared for
   (V, V_head, r and the markov_w1 / markov_w2 addresses), markov_w2 transposed
   [round_up(V_head, 128)][r] bf16, the fp32 Euclidean norm of every markov_w2 column,
   their maximum over each 128-row tile, and the largest Euclidean norm of a markov_w1
   row.
   A head in the bias form of a reduced draft vocabulary (lm_bias given, d2t NULL,
   V_head == V, and 1 <= n_emit < V rows with bias > -1e8) is prepared in its compact
   form instead (llama.cpp PR #26275, the reduced draft vocabulary as an expanded head
   and as a d2t map): a 256-byte header (V, H, r, n_emit, the padded row count
   n_pad = round_up(n_emit, 8) and the lm_head, lm_bias, markov_w1, markov_w2
   addresses), the emittable rows in increasing order [n_pad] int32 (padded with copies
   of the last), per-chunk counts, their lm_head rows [n_pad][H] bf16, markov_w2
   columns [r][n_pad] bf16 and biases [n_pad] fp32 (padding rows: zero weights, bias
   -1e30), then the layout above for that compact head.  To size it, this call counts
   the emittable rows on the device and waits for the count (current device, default
   stream). */
size_t dspark_prepare_head_size(const dspark_config* cfg, const dspark_head* head);

/*
 * dspark_prepare_head -- one-time preparation of a head's Markov weights for the pruned
 * chain (the weights are constant across calls, like a converted checkpoint).
 *
 * prepared  device buffer of dspark_prepare_head_size() bytes, 256-byte aligned, owned by
 *           the caller; pass it as head->prepared to later dspark_propose calls.  It must
 *           be prepared again whenever markov_w1 or markov_w2 changes, in place or by
 *           address: the pruned chain's bounds come from both (the column norms of
 *           markov_w2 and the largest row norm of markov_w1), and stale bounds can drop
 *           the true argmax or top-k rows without any error.  head->prepared itself is
 *           ignored here.
 *
 * A dspark_propose call whose V, V_head, r, markov_w1 or markov_w2 address differ from
 * those the buffer was prepared for reads nothing past the buffer's header: it drafts
 * nothing and dspark_device_status() then reports DSPARK_ERR_DEVICE with that reason.
 * (Contents changed in place at the same addresses cannot be detected; re-prepare.)
 *
 * Bias form (see dspark_prepare_head_size): the emittable rows are counted (this call
 * waits for the count on `stream`), found and gathered on the device into the compact
 * head; later dspark_propose calls with this head run on those rows only (the GEMM, the
 * chain and the top-k), with the same outputs as over the full head.  That holds while
 * top_k <= n_emit and the logits output is not requested; otherwise a call uses the
 * full head (the dense chain over every row).  It must be prepared again when lm_head or
 * lm_bias changes too.  A process that did not prepare the buffer itself reads its
 * header once, synchronously, on first use: make that first call outside stream
 * capture.
 */
dspark_status dspark_prepare_head(const dspark_config* cfg, const dspark_head* head,
                                  void* prepared, size_t prepared_bytes, void* stream);

/* Stages of dspark_propose, in launch order, for dspark_propose_timed(). */
enum {
  DSPARK_STAGE_CONF = 0,    /* confidence head + truncation length */
  DSPARK_STAGE_LOGITS = 1,  /* base logits of every prediction slot (the lm_head GEMM) */
  DSPARK_STAGE_CHAIN = 2,   /* Markov-corrected greedy chain and per-slot candidates */
  DSPARK_STAGE_TOPK = 3,    /* final top-k ordering */
  DSPARK_NUM_STAGES = 4
};

/* dspark_propose that also records events[s] (cudaEvent_t, created by the caller) on
   `stream` as stage s begins, and events[DSPARK_NUM_STAGES] after the last stage.
   A stage with no kernel for this config records its event right before the next
   one's.  The work done is identical to dspark_propose's. */
dspark_status dspark_propose_timed(const dspark_config* cfg, const dspark_head* head,
                                   const void* hidden, const int32_t* anchors,
                                   const void* conf_hidden, const dspark_outputs* out,
                                   void* workspace, size_t workspace_bytes, void* stream,
                                   void* const* events);

/* Number of kernels one dspark_propose call launches for this config, head and set of
   requested outputs, the kernel that resets the workspace's control block included; -1
   on invalid input. */
int32_t dspark_propose_kernel_count(const dspark_config* cfg, const dspark_head* head,
                                    const dspark_outputs* out);

/* Bytes of device workspace dspark_step_host needs: dspark_propose's plus staging for
   the host inputs and outputs.  256-byte aligned; 0 on invalid input. */
size_t dspark_step_host_workspace_size(const dspark_config* cfg, const dspark_head* head);

/*
 * dspark_step_host -- one draft step from and to HOST memory: copies hidden, anchors
 * and target in, runs dspark_propose and dspark_verify, copies the results out.
 *
 * hidden_h  host [B, L_in, H] dtype      anchors_h host [B] int32
 * conf_hidden_h host [B, L_in, H] dtype, or NULL: the confidence head's separate input
 *           (see dspark_propose); copied in like hidden_h
 * target_h  host [B, N + 1] int32 (the target's argmax tokens for the verify step)
 * draft_h   host [B, N] int32            n_draft_h host [B] int32
 * accepted_h, bonus_h host [B] int32
 * topk_ids_h / topk_vals_h host [B, N, top_k] or NULL
 *
 * hidden_h is copied with cudaMemcpyAsync on `stream`.  The other buffers are read or
 * written by the kernels in place when they are page-locked host memory the device can
 * address (cudaHostAlloc, or cudaHostRegister with a mapping; cudaPointerGetAttributes
 * reports them as host memory with a device pointer); otherwise they too are copied
 * through workspace staging.  Page-locked buffers throughout are the fast case.  The
 * call returns once everything is queued: synchronise `stream` before reading the
 * outputs.
 */
dspark_status dspark_step_host(const dspark_config* cfg, const dspark_head* head,
                               const void* hidden_h, const int32_t* anchors_h,
                               const void* conf_hidden_h,
                               const int32_t* target_h, int32_t* draft_h,
                               int32_t* n_draft_h, int32_t* accepted_h, int32_t* bonus_h,
                               int32_t* topk_ids_h, float* topk_vals_h,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * dspark_propose_noalloc -- dspark_propose for callers that cannot allocate device memory.
 *
 * (No counterpart on the pages: an interface addition of this library.)  Some callers
 * cannot call cudaMalloc or any allocating routine: code that runs inside a host
 * framework owning every allocation, allocator-free plugins, or callers that must not
 * touch the allocator while the device is in use elsewhere.  This entry point takes the
 * same arguments as dspark_propose minus the workspace: its scratch is a fixed 16 MiB
 * array of device memory built into the library, which every GPU that loads the library
 * holds until the process exits.  It allocates nothing itself.
 *
 *   - Calls whose dspark_propose_workspace_size() exceeds 16 MiB return
 *     DSPARK_ERR_WORKSPACE before launching anything (small batches and vocabularies
 *     only; larger ones need dspark_propose and a caller workspace).
 *   - The scratch's device address belongs to the CUDA context current at the call.  A
 *     call that is not being captured looks it up (with the device current) and keeps it
 *     for that context; a call made while `stream` is capturing uses the address kept
 *     for the current context and is refused if there is none.  So make one call on each
 *     device (and again after a cudaDeviceReset) before any stream capture.
 *   - Every call on a device shares the one scratch array, which keeps the contents the
 *     last call left (each call clears what has to start at zero).  Calls that overlap on
 *     the GPU -- on different streams, or from different host threads without ordering --
 *     race on it and give wrong results: order them on one stream.
 *   - Problems only the device can see (an anchor outside [0, V), a bounded wait that
 *     gave up) are recorded in the scratch's error word; read them with
 *     dspark_noalloc_device_status() before the next call on the device clears them.
 */
dspark_status dspark_propose_noalloc(const dspark_config* cfg, const dspark_head* head,
                                     const void* hidden, const int32_t* anchors,
                                     const void* conf_hidden, const dspark_outputs* out,
                                     void* stream);

/* Synchronises `stream`, reads the device error word of a workspace used by
   dspark_propose (it describes the latest call on that workspace), and clears it.
   DSPARK_OK when no kernel flagged anything; DSPARK_ERR_DEVICE or DSPARK_ERR_TIMEOUT
   otherwise, with the reason in dspark_last_error(). */
dspark_status dspark_device_status(void* workspace, void* stream);

/* Synchronises `stream` and reads three counters of the latest dspark_propose call on
   `workspace` (they restart at zero with every call).  Instrumentation of the cost of
   the two chain forms; the method on the pages has no counterpart.  Any output pointer
   may be NULL.
     on_the_fly:     (slot, block) pairs the exact-bound pruned chain could not look up
                     in its tables and evaluated on the fly (loose Cauchy-Schwarz bounds:
                     too many candidate rows or possible previous rows);
     every_row:      of those, the pairs whose candidate list overflowed, so that every
                     head row was evaluated;
     dense_overflow: (slot, block) pairs of the dense chain whose top-k candidate lists
                     overflowed (massive ties) and were recomputed over every head row.
   DSPARK_ERR_INVALID_ARG for a NULL workspace; DSPARK_ERR_CUDA if the read fails. */
dspark_status dspark_pass_stats(void* workspace, void* stream, int32_t* on_the_fly,
                                int32_t* every_row, int32_t* dense_overflow);

/* dspark_device_status() for the built-in scratch of dspark_propose_noalloc() on the
   current device: synchronises `stream`, reads the error word of the latest no-alloc call
   on this device and clears it.  (No counterpart on the pages, like the entry point it
   serves.)  Call it on the stream of that call, outside stream capture. */
dspark_status dspark_noalloc_device_status(void* stream);

/*
 * dspark_wait_selftest -- makes one bounded device-side wait run out, on purpose.
 *
 * (No counterpart on the pages: a test hook of this library's failure detection.)  Every
 * wait inside the library's kernels (a pipeline stage waiting for its copy, the MMA
 * waiting for a free accumulator, a grid barrier) gives up after a clock budget of about
 * one second, raises the timeout bit of the workspace's error word and lets the kernel
 * return, so that the CUDA context stays usable.  This call launches one small kernel that
 * waits, through the same bounded-wait routine, on a barrier that nothing ever completes.
 *
 *   workspace        device, >= 256 bytes, 256-byte aligned; only its first word (the
 *                    error word) is written.  A dspark_propose workspace qualifies.
 *   budget_cycles    SM clock cycles to wait before giving up, in [1, 2e9].
 *   pre_abort        1 = the abort flag is already set, so the wait gives up at its first
 *                    check; 0 = it gives up when the budget runs out.
 *   stream           the CUDA stream (cudaStream_t), may be NULL.
 *
 * Host-detectable errors (above) return before any launch.  Afterwards,
 * dspark_device_status() on the same workspace reports DSPARK_ERR_TIMEOUT and clears it.
 */
dspark_status dspark_wait_selftest(void* workspace, size_t workspace_bytes,
                                   int64_t budget_cycles, int32_t pre_abort, void* stream);

/* Static description of a status code. */
const char* dspark_status_string(int32_t status);

/* Message describing the calling thread's most recent failed call ("" if none). */
const char* dspark_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H_ */
