/*
 * growpage.h -- C ABI of the GrowPage decode hot path on one B300 (sm_103a).
 *
 * What the calls compute comes from the pages titled "GrowPage: On-Demand KV
 * Budgeting for Efficient LLM Reasoning Serving":
 *   - abstract: KV capacity as a runtime resource on top of PagedAttention's
 *     page-level memory; dual-timescale query summaries; at each capacity
 *     boundary either compress KV within the current allocation or acquire
 *     one more physical page; continuous batching and prefix caching kept;
 *   - evolve.pub review, section "Summary": Top-p attention working sets of a
 *     short (beta 0.9) and a long (beta 0.999) exponentially smoothed query
 *     summary, maintained pre-RoPE; a larger recent working set allocates one
 *     extra page, otherwise history is compacted by the maximum of both
 *     importance scores;
 *   - same review, "Frequently asked questions": Top-p, demand threshold tau,
 *     local retention quota, KV block size.
 * The pages define no API; the calls below follow that statement of the
 * problem.  Conventions the pages leave open are stated at each call.
 *
 * Ownership.  The caller owns every byte of device memory: the pool buffer
 * (size from gp_pool_bytes, allocated by the caller, e.g. with torch) and all
 * input/output tensors.  The library never allocates or frees device memory;
 * it keeps only host-side bookkeeping in the gp_pool handle.
 *
 * Streams.  Every call enqueues its work on the pool's stream (set at
 * creation or by gp_set_stream) in call order.  Calls marked SYNC wait for
 * that stream; the others return as soon as the work is enqueued.
 *
 * Errors.  Every call returns an int status (GP_OK = 0).  Invalid arguments
 * are reported before anything is enqueued.  Faults found on the device
 * (a bad slot list, a page id out of range, a wait that timed out) set bits
 * in the device status word and make the offending kernel skip the access;
 * the next SYNC call returns GP_ERR_DEVICE and gp_last_error says which bit.
 * No C++ exception crosses this ABI.  No kernel traps or asserts.
 *
 * Device pointers.  Arguments named *_dev, and q / k / v / out / k_prompt /
 * v_prompt / k_prefix / v_prefix, are device pointers.  All tensors are dense,
 * row-major, 16-byte aligned, of the pool's storage dtype unless stated.
 */
#ifndef GROWPAGE_H
#define GROWPAGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define GP_OK            0
#define GP_ERR_INVALID   1  /* bad argument or call order; nothing enqueued */
#define GP_ERR_NO_PAGES  2  /* add_request / add_prefix: not enough free pages */
#define GP_ERR_CUDA      3  /* a CUDA runtime call failed */
#define GP_ERR_DEVICE    4  /* the device status word is non-zero */

/* ---- device status word bits (gp_ctrl.status) ------------------------ */
#define GP_ST_BAD_SLOTS    0x1u  /* slot list not ascending / not active     */
#define GP_ST_BAD_PAGE     0x2u  /* a block-table entry outside the pool     */
#define GP_ST_TIMEOUT      0x4u  /* a bounded wait gave up                   */
#define GP_ST_STARVED      0x8u  /* not raised: a starved full-KV boundary is
                                    counted in gp_ctrl.starved instead       */
#define GP_ST_BAD_PLAN     0x10u /* inconsistent compaction plan            */
#define GP_ST_POS_RANGE    0x20u /* a request reached max_seq_len            */
#define GP_ST_SMEM_ALIGN   0x40u /* attention kernel skipped: its shared
                                    memory was not 1024-byte aligned         */

/* ---- configuration --------------------------------------------------- */
#define GP_DTYPE_F32   0
#define GP_DTYPE_BF16  1

#define GP_MODE_GROWPAGE 0 /* grow or compact at each boundary            */
#define GP_MODE_FULL_KV  1 /* every boundary grows; no scoring, no compaction */
/* Ablation policies on the same kernels ("GrowPage: On-Demand KV Budgeting
 * for Efficient LLM Reasoning Serving", evolve.pub review: the frequency-
 * matched random policy and the inverted signal of Tables 8-9, and the
 * fixed-budget compressed-paging baseline it compares against).  Scoring,
 * Top-p counts and compaction are those of GP_MODE_GROWPAGE; only the grow
 * decision differs. */
#define GP_MODE_FIXED    2 /* never grow: every boundary compacts          */
#define GP_MODE_INVERSE  3 /* grow iff -Delta > tau (the signal reversed)  */
#define GP_MODE_RANDOM   4 /* grow iff u < random_grow_rate, u uniform in [0,1)
                              from SplitMix64 of (slot << 32 | boundaries
                              seen so far by the request), top 53 bits */
/* The review's SHRINK ablation ("the cost of irreversible shrinking"; the
 * pages give no rule, this is a reading): grow iff Delta > tau as in
 * GP_MODE_GROWPAGE; otherwise release the request's last private page.  The
 * boundary then drops 2P private tokens by the compaction rule (keeping the
 * most recent min(W_r, C - 2P) and the most important older ones), so that
 * the remaining b - 1 pages again hold P free slots.  A page is released
 * only while (b - 2) * P >= W_r; below that the boundary compacts in place.
 * Released pages are pushed on the free stack after every growth of the
 * step has popped, in ascending slot order. */
#define GP_MODE_SHRINK   5

typedef struct gp_config {
  int32_t num_layers;        /* L */
  int32_t num_q_heads;       /* Hq */
  int32_t num_kv_heads;      /* Hk; G = Hq / Hk must be 1, 2 or 4 */
  int32_t head_dim;          /* d: 64 (f32 storage) or 128 (f32 or bf16) */
  int32_t page_size;         /* P tokens per page, a multiple of 16, <= 256 */
  int32_t num_pages;         /* physical pages in the pool */
  int32_t max_requests;      /* request slots 0 .. max_requests-1 */
  int32_t max_pages_per_req; /* cap on a request's private pages */
  int32_t max_prefixes;      /* shared-prefix slots */
  int32_t max_prefix_len;    /* tokens, a multiple of P */
  int32_t max_seq_len;       /* largest absolute position + 1 (RoPE table rows) */
  int32_t dtype;             /* GP_DTYPE_*: K/V pages, q, k, v, out */
  int32_t mode;              /* GP_MODE_* */
  int32_t recent_window;     /* W_r: most recent private tokens always kept */
  float beta_s;              /* short summary smoothing (0.9) */
  float beta_l;              /* long summary smoothing (0.999) */
  float top_p;               /* working-set mass threshold */
  float tau;                 /* grow iff Delta > tau */
  double rope_theta;         /* 0: no rotary embedding */
  int32_t flags;             /* reserved, must be 0 */
  float random_grow_rate;    /* GP_MODE_RANDOM: grow probability in [0, 1] */
} gp_config;

/* ---- device layout of the pool buffer -------------------------------- */
/* Byte offsets from the start of the caller's buffer.  All regions are
 * 256-byte aligned.  Tensors listed as [a][b]... are dense row-major.
 *
 *  kv        [num_pages][L][Hk][2][P][d] dtype   page contents; [..][0] = keys
 *            (rotated to their positions), [..][1] = values
 *  tok_pos   [num_pages][L][Hk][P] int32          absolute position of the token
 *                                                 in each page slot
 *  block     [max_requests][block_width] int32    page ids: prefix pages first,
 *                                                 then private pages in order
 *  req       [max_requests] gp_req_meta
 *  summary   [max_requests][L][Hk][2][d] float32  [..][0] short, [..][1] long,
 *                                                 pre-RoPE
 *  staging   [max_requests][L][Hk][2][d] dtype    the last step's token:
 *                                                 [0] rotated key, [1] value
 *  logits    [max_requests][L][Hk][2][logit_width] float32  summary scores of
 *                                                 the last boundary (GROWPAGE)
 *  wset      [max_requests][L][Hk][2] int32       Top-p working-set sizes of the
 *                                                 last boundary (short, long)
 *  free      [num_pages] int32                    free-page stack, height in ctrl
 *  ctrl      gp_ctrl
 *  prefix    [max_prefixes] gp_prefix_meta; then [max_prefixes][max_prefix_pages]
 *            int32 page ids
 *  rope      [max_seq_len] rows of 16·d bytes, one per position: cos, sin
 *            fp32 [d/2] each (the fp64 values rounded once), their fp32
 *            residuals (fp64 value minus the fp32 value, rounded once), then
 *            cos, sin fp64 [d/2] each
 *  scratch   plan, split-K partials, move lists (internal) */
typedef struct gp_layout {
  uint64_t kv, tok_pos, block, req, summary, staging, logits, wset, free_stack,
      ctrl, prefix, prefix_pages, rope, scratch, total;
  uint64_t page_bytes;       /* one page across all layers and heads */
  int32_t block_width;       /* max_prefix_len / P + max_pages_per_req */
  int32_t logit_width;       /* max_prefix_len + max_pages_per_req * P */
  int32_t max_prefix_pages;
  int32_t num_workers;       /* attention workers (warps) per launch */
} gp_layout;

/* Per-request metadata, one per slot, as stored on the device. */
typedef struct gp_req_meta {
  int32_t active;        /* 1 while the slot holds a request */
  int32_t prefix_id;     /* -1: none */
  int32_t n_pre_pages;   /* prefix pages at the head of the block table */
  int32_t n_pages;       /* private pages held (the current budget b) */
  int32_t seq_priv;      /* private tokens resident (<= n_pages * P) */
  int32_t pos;           /* absolute position of the next token */
  int32_t steps;         /* decode steps done */
  int32_t last_decision; /* 0 none, 1 grow, 2 compact, 3 compact (grow
                            denied), 4 starved (full-KV, no page),
                            5 shrink (GP_MODE_SHRINK: a page released) */
  int64_t delta;         /* sum over layers and kv heads of W_S - W_L at the
                            last boundary */
  int32_t n_boundaries, n_grows, n_compacts, n_denied;
  int32_t n_starved;
  int32_t n_shrinks;     /* pages released (GP_MODE_SHRINK) */
} gp_req_meta; /* 64 bytes */

typedef struct gp_prefix_meta {
  int32_t refs;     /* requests using it + 1 while the creator holds it */
  int32_t n_pages;
  int32_t len;
  int32_t reserved;
} gp_prefix_meta;

/* Pool-wide counters, as stored on the device. */
typedef struct gp_ctrl {
  int32_t free_top;      /* free pages (stack height) */
  uint32_t status;       /* GP_ST_* bits */
  int32_t status_info;   /* first offending slot / page, when known */
  int32_t plan_n;        /* requests in the current step's plan */
  int64_t steps;         /* decode steps planned */
  int64_t tokens_attended;  /* sum over planned steps and requests of the
                               resident tokens R (prefix + private) */
  int64_t boundary_tokens;  /* same, restricted to requests at a boundary */
  int64_t boundaries, grows, compacts, denied, starved, moved_tokens;
  int64_t shrinks;       /* pages released (GP_MODE_SHRINK) */
  int64_t reserved[3];
} gp_ctrl;

typedef struct gp_pool gp_pool; /* opaque host handle */

/* Bytes of device memory a pool with this configuration needs.  Host-only,
 * needs no GPU.  GP_ERR_INVALID if the configuration is unsupported. */
int gp_pool_bytes(const gp_config* cfg, size_t* bytes);

/* Lay the pool out in the caller's buffer (>= gp_pool_bytes, 256-byte
 * aligned) and initialise it on `stream` (a cudaStream_t; NULL = legacy
 * default stream): empty block tables, free stack such that pops return
 * pages 0, 1, 2, ..., RoPE tables built on the host in fp64 with the C
 * library's pow/cos/sin.  SYNC.  *out receives the handle. */
int gp_create_pool(const gp_config* cfg, void* dev_buf, size_t bytes,
                   void* stream, gp_pool** out);

/* Release the host handle.  The device buffer stays the caller's. */
int gp_destroy_pool(gp_pool* pool);

/* Enqueue later calls on another stream. */
int gp_set_stream(gp_pool* pool, void* stream);

/* Offsets of every region of the caller's buffer (see gp_layout). */
int gp_get_layout(const gp_pool* pool, gp_layout* out);

/* Store a shared prefix (prefix caching).  k_prefix, v_prefix: device
 * [L][len][Hk][d], keys not yet rotated; len a multiple of P, <=
 * max_prefix_len.  Pops len/P pages, writes keys rotated to positions
 * 0..len-1 (fp64 rotation, one rounding to the storage dtype) and values.
 * The prefix starts with one reference held by the caller
 * (gp_release_prefix drops it); its pages return to the pool when no request
 * uses it and the caller has released it.  Prefix pages are never compacted.
 * SYNC.  GP_ERR_NO_PAGES if the pool is short of pages. */
int gp_add_prefix(gp_pool* pool, const void* k_prefix, const void* v_prefix,
                  int32_t len, int32_t* prefix_id);
int gp_release_prefix(gp_pool* pool, int32_t prefix_id);

/* Admit a request into an empty slot.  Follows the abstract of "GrowPage:
 * On-Demand KV Budgeting for Efficient LLM Reasoning Serving": requests live
 * on PagedAttention's page-level memory with continuous batching and prefix
 * caching kept, so a request joins between steps with an initial KV budget
 * of physical pages and may share a cached prefix.  Its block
 * table becomes the prefix's pages (prefix_id >= 0) followed by
 * budget_pages freshly popped private pages (the initial KV budget).
 * k_prompt, v_prompt: device [L][prompt_len][Hk][d] (keys not yet
 * rotated; may be NULL when prompt_len == 0), stored at positions
 * prefix_len .. prefix_len + prompt_len - 1.  prompt_len <= budget_pages * P.
 * The summaries start empty: the first decode step sets them to that step's
 * query mean.  SYNC.  GP_ERR_NO_PAGES if fewer than budget_pages are free. */
int gp_add_request(gp_pool* pool, int32_t slot, const void* k_prompt,
                   const void* v_prompt, int32_t prompt_len,
                   int32_t budget_pages, int32_t prefix_id);

/* One layer of one decode step for the n requests in slots_dev (device
 * int32[n], strictly ascending active slots; the same list for every layer
 * of the step).  Follows the evolve.pub review of "GrowPage: On-Demand KV
 * Budgeting for Efficient LLM Reasoning Serving", section "Summary": paged
 * (PagedAttention) decode attention, with the short (beta 0.9) and long
 * (beta 0.999) exponentially smoothed query summaries maintained pre-RoPE,
 * and, at a capacity boundary, the attention scores those summaries induce
 * over the resident keys (their Top-p working sets are taken by
 * gp_boundary).  q, out: [n][Hq][d]; k_new, v_new: [n][Hk][d]; q and k_new
 * are pre-RoPE.  For each request i, kv head g and query head h in
 * [g*G, (g+1)*G):
 *   - stages k_new rotated to the request's position (fp64 rotation, one
 *     rounding to the storage dtype) and v_new;
 *   - folds qbar = mean of the G query heads (fp32, head order) into the
 *     short and the long summary: s <- fl(fl(b*s) + fl((1-b)*qbar));
 *   - out[i][h] = softmax(RoPE(q_h)·K^T / sqrt(d)) · V over the request's
 *     resident tokens (prefix + private) plus the staged token;
 *   - at a boundary step (all private pages full at step start, GROWPAGE
 *     mode): also writes u = RoPE(s, pos)·k_j / sqrt(d) of both updated
 *     summaries for every resident key j into the logits region.
 * Layers must be called 0, 1, ..., L-1, then gp_boundary, once per step.
 * Asynchronous. */
int gp_decode_step(gp_pool* pool, int32_t layer, int32_t n,
                   const int32_t* slots_dev, const void* q, const void* k_new,
                   const void* v_new, void* out);

/* Finish the step for the same n requests.  Follows the abstract of
 * "GrowPage: On-Demand KV Budgeting for Efficient LLM Reasoning Serving" (at
 * each capacity boundary, compress KV within the current allocation or
 * acquire one more physical page) and its evolve.pub review, section
 * "Summary" (compare the Top-p working sets of the two summaries; a larger
 * recent one allocates an extra page, otherwise compact by the maximum of
 * both importance scores) and "Frequently asked questions" (Top-p, demand
 * threshold tau = 0, local retention quota).  For each request at a boundary,
 * softmax of each summary's scores, Top-p working-set sizes W_S, W_L per
 * (layer, kv head), Delta = sum (W_S - W_L); grow by one page iff
 * Delta > tau, a page is free and n_pages < max_pages_per_req (requests
 * served in ascending slot order, so page ids are deterministic); otherwise
 * compact in place: per (layer, kv head) keep the min(W_r, C-P) most recent
 * private tokens plus the best older ones by max(p_S, p_L) (ties: the more
 * recent), C - P in all, and move the survivors of the last page into the
 * freed slots.  Then every request appends its staged token.  Full-KV mode:
 * every boundary grows.  The ablation modes change only the grow decision
 * (GP_MODE_FIXED, GP_MODE_INVERSE, GP_MODE_RANDOM) or, for GP_MODE_SHRINK,
 * replace in-place compaction by a page release (see its definition above).
 * n and slots_dev must be the step's own (those given to gp_decode_step);
 * called before the step's last layer it returns GP_ERR_INVALID.
 * Asynchronous. */
int gp_boundary(gp_pool* pool, int32_t n, const int32_t* slots_dev);

/* gp_boundary with the boundary work made asynchronous.  Follows the
 * evolve.pub review of "GrowPage: On-Demand KV Budgeting for Efficient LLM
 * Reasoning Serving", "Frequently asked questions": GrowPage builds on
 * Zipage's machinery, including its asynchronous compression.  The pages
 * say no more; this is a reading: a request at a boundary sits out the next
 * step while its boundary work runs beside that step.
 *   - on the pool's stream: the requests not at a boundary are finished
 *     (their staged token appended), so the next step can start at once;
 *   - on side_stream (a cudaStream_t other than the pool's): for the
 *     requests at a boundary, everything gp_boundary does for them -- Top-p
 *     working sets, Delta, the grow / compact decision (growth served in
 *     ascending slot order), the compaction moves and the staged token.
 * Results are those of gp_boundary.  The requests that were at a boundary
 * must not be in the next step's slot list (the plan kernel refuses a
 * request whose boundary work is still running: GP_ST_BAD_SLOTS, step
 * dropped); from the step after they may take part again, and that step's
 * first gp_decode_step makes the pool's stream wait for the work on the
 * device (no host sync).  Steps are counted by calls: if no request is left
 * for the next step, call it anyway with n = 0 (every layer, then
 * gp_boundary_async or gp_boundary).  Every other call that reads or changes the pool
 * between steps (admission, gp_free, prefixes, SYNC calls, the read
 * ceiling, gp_set_stream) first makes the pool's stream wait for it too.
 * A later step's boundary work is ordered after an earlier one's, even on
 * another side stream.  Asynchronous. */
int gp_boundary_async(gp_pool* pool, int32_t n, const int32_t* slots_dev, void* side_stream);

/* Release a request: its private pages are pushed in block-table order; a
 * prefix whose last reference goes is pushed too.  Asynchronous. */
int gp_free(gp_pool* pool, int32_t slot);

/* Measurement, not part of the decode path: for each layer in
 * [layer0, layer0 + count), one launch that reads every resident K/V block of
 * that layer for the n requests in slots_dev (same list rules as
 * gp_decode_step) through the same persistent grid, per-warp split and
 * tensor-map copies as the bf16 attention kernel, with no arithmetic.  It
 * gives the bandwidth ceiling of that access pattern.  mode 0: the requests'
 * own pages (the attention kernel's pattern); mode 1: the same number of
 * 8 KiB blocks in address order (tensor-map copies); mode 2: the same bytes
 * in address order with plain 16-byte loads.  sink_dev: device uint32[4],
 * caller-owned; [0] receives an XOR checksum of the data, [2..3] the bytes
 * one launch moved (uint64, little-endian).  Only for bf16 pages with
 * head_dim 128 (GP_ERR_INVALID otherwise) and between steps.  Leaves the
 * pool's state and counters unchanged.  Asynchronous. */
int gp_kv_read_ceiling(gp_pool* pool, int32_t layer0, int32_t count, int32_t mode, int32_t n,
                       const int32_t* slots_dev, uint32_t* sink_dev);

/* gp_kv_read_ceiling without caller scratch.  No counterpart in the paper:
 * it is a convenience of this library for callers that cannot allocate device
 * memory when they call it -- code running inside a memory arena sized
 * once at start-up, or a runtime whose allocator must not be entered at that
 * point -- and for callers that must not disturb the pool's own scratch,
 * which gp_kv_read_ceiling overwrites (so that one may only run between
 * steps).  Same arguments and result as gp_kv_read_ceiling, except:
 *   - it leaves the pool's scratch untouched, so it may also be called
 *     between two layers of a step (after gp_decode_step(layer), before the
 *     next layer): the step's outputs and decisions do not change;
 *   - the per-call scratch (the step plan of the n requests and the start
 *     cursor and first block of every attention worker) lives in a file-scope
 *     device array of this library, about 160 KB, which every GPU that loads the library
 *     keeps until the process exits; nothing of it needs clearing, as each
 *     call writes all the scratch it reads;
 *   - n may not exceed 1024 (GP_ERR_INVALID with a message otherwise);
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the life of the
 *     process: it assumes the device's primary context lives as long, so do
 *     not reset the device (cudaDeviceReset) while the library is used there;
 *   - all calls share the array: two calls whose work overlaps on the GPU
 *     (different streams, or different pools on one device) race.
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 * Asynchronous. */
int gp_kv_read_ceiling_static(gp_pool* pool, int32_t layer0, int32_t count, int32_t mode,
                              int32_t n, const int32_t* slots_dev, uint32_t* sink_dev);

/* Wait for the stream; GP_ERR_DEVICE if the device status word is set.
 * The word stays set (every later gp_sync reports it) until
 * gp_clear_status.  SYNC. */
int gp_sync(gp_pool* pool);

/* Read and clear the device status word: *status_out receives the GP_ST_*
 * bits that were set and *info_out the first offending slot or page (either
 * pointer may be NULL).  What a flagged step left behind:
 *   GP_ST_BAD_SLOTS / GP_ST_POS_RANGE: the plan kernel dropped the whole
 *     step before any state changed (no token staged, no summary folded, no
 *     boundary work, `out` not written); the pool continues as if the step
 *     had not been called;
 *   GP_ST_TIMEOUT: a bounded wait gave up; that step's outputs are
 *     incomplete;
 *   GP_ST_BAD_PAGE: an out-of-range page id was read as page 0; the
 *     affected request's contents are undefined;
 *   GP_ST_SMEM_ALIGN: the attention kernel did not run; that step's
 *     outputs are undefined.
 * SYNC. */
int gp_clear_status(gp_pool* pool, uint32_t* status_out, int32_t* info_out);

/* Copy the pool-wide counters to the host.  SYNC. */
int gp_get_stats(gp_pool* pool, gp_ctrl* out);

/* Copy one request's metadata and its block table (up to cap entries) to
 * the host.  SYNC. */
int gp_get_request(gp_pool* pool, int32_t slot, gp_req_meta* meta,
                   int32_t* block_table, int32_t cap);

/* Host destinations for gp_get_state; any pointer may be NULL (that region
 * is not copied).  Sizes, with the pool's configuration and layout:
 *   req        [max_requests] gp_req_meta
 *   block      [max_requests][block_width] int32 (gp_layout.block_width)
 *   ctrl       one gp_ctrl
 *   wset       [max_requests][num_layers][num_kv_heads][2] int32: W_S, W_L
 *              of each request's last boundary
 *   tok_pos    [num_pages][num_layers][num_kv_heads][page_size] int32: the
 *              absolute position of the token in each page slot
 *   free_stack [num_pages] int32, valid up to ctrl->free_top
 * The caller owns these buffers. */
typedef struct gp_state_view {
  gp_req_meta* req;
  int32_t* block;
  gp_ctrl* ctrl;
  int32_t* wset;
  int32_t* tok_pos;
  int32_t* free_stack;
} gp_state_view;

/* Copy the pool's state (block tables, request metadata with sequence
 * lengths, budgets and the last Delta, working-set sizes, kept positions,
 * counters, the free stack) to the host in one call.  SYNC. */
int gp_get_state(gp_pool* pool, gp_state_view* out);

/* Text of the last error on this handle ("" if none).  Owned by the pool. */
const char* gp_last_error(const gp_pool* pool);

/* Number of kernel launches this handle has enqueued so far. */
int64_t gp_launch_count(const gp_pool* pool);

#ifdef __cplusplus
}
#endif

#endif /* GROWPAGE_H */
