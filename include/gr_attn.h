/*
 * gr_attn.h -- C ABI of libgrattn.so: large-beam decode attention over a
 * shared request context (ContextKV + BeamKV + BeamPath), for NVIDIA GB300
 * (sm_103a).
 *
 * The operation (GR-Inference blog, "system design" and "kernel design";
 * SID-GR Inference README, section 3 "Design Highlights" and section 9
 * "Nsight breakdown"; xGR review, "xAttention", three-stage computation):
 *
 *   For request r, active beam b < W_s at decode step s and query head h
 *   (kv head g = h / G, G = Hq / Hkv), with the ancestor chain
 *       a_s = b,   a_{t-1} = beam_path[r, t, a_t]   (t = s .. 1)
 *   the row attends to the keys/values
 *       ctx_k/ctx_v[r, g, 0 .. ctx_len[r]-1]             (shared stage)
 *       beam_k/beam_v[r, t, a_t, g]  for t = 0 .. s      (unshared stage)
 *   with scores x_j = softmax_scale * <q[r, b, h], k_j>, and the two partial
 *   softmaxes are merged exactly by log-sum-exp (merging stage):
 *       lse[r, b, h] = ln sum_j exp(x_j)
 *       out[r, b, h] = sum_j exp(x_j - lse) * v_j
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller allocates and owns every buffer.  No entry point
 *     here allocates or frees memory, and only gr_get_device_error()
 *     synchronises.
 *   - Execution: device work is enqueued on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and runs asynchronously.  Host-side checks
 *     happen before anything is enqueued; on an error nothing is enqueued.
 *   - Layout: every tensor is dense, row-major, with the shapes below.  bf16
 *     is IEEE bfloat16 stored in 2 bytes.  Device pointers must be 16-byte
 *     aligned.
 *   - Widths are per step and shared by every request in the call
 *     (`widths` is a HOST array of at least step+1 entries).
 *   - The caller appends the step-s K/V of every active beam to beam_k/beam_v
 *     before the call, so each chain holds s+1 tokens (the current token is
 *     attended).
 *   - Preconditions not checked on the hot path (gr_validate_beam_path checks
 *     them on the device): 0 <= ctx_len[r] <= ctx_capacity; beam_path[r, t, b]
 *     in [0, widths[t-1]) for 1 <= t <= s and b < widths[t].  beam_path[r, 0, .]
 *     is never read (step 0 expands from the single prefill row).
 *   - Returns GR_OK (0) or a negative gr_status.
 */
#ifndef GR_ATTN_H
#define GR_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *gr_stream_t; /* a cudaStream_t */
typedef void *gr_event_t;  /* a cudaEvent_t */

typedef enum {
    GR_OK = 0,
    GR_ERR_NULL_ARG = -1,            /* a required pointer is NULL */
    GR_ERR_BAD_SHAPE = -2,           /* inconsistent or out-of-range sizes */
    GR_ERR_UNSUPPORTED = -3,         /* head_dim not 64/128, or no sm_103 device */
    GR_ERR_MISALIGNED = -4,          /* a device pointer is not 16-byte aligned */
    GR_ERR_WORKSPACE_TOO_SMALL = -5, /* workspace_bytes below the size required */
    GR_ERR_CUDA = -6,                /* a CUDA runtime/driver call failed */
    GR_ERR_DEVICE_TIMEOUT = -7,      /* a kernel gave up a bounded wait */
    GR_ERR_BAD_BEAM_PATH = -8        /* a kernel met a parent slot out of range */
} gr_status;

/* Problem geometry.  Every size is a count of elements, not bytes. */
typedef struct {
    int32_t num_requests;  /* R >= 1 */
    int32_t num_q_heads;   /* Hq >= 1 */
    int32_t num_kv_heads;  /* Hkv >= 1, Hq % Hkv == 0, G = Hq / Hkv <= 128 */
    int32_t head_dim;      /* D: 64 or 128 */
    int32_t ctx_capacity;  /* Lc_max >= 0: context slots per (request, kv head) */
    int32_t step_capacity; /* S_max >= 1: decode-step slots in BeamKV/BeamPath */
    int32_t beam_capacity; /* W_max >= 1: beam slots per step */
    float softmax_scale;   /* score scale > 0 (1/sqrt(D) for the Qwen3 heads) */
} gr_attn_shape;

/*
 * Bytes of device workspace gr_decode_attn needs for this geometry, step and
 * width schedule (host array, step+1 entries).  Depends only on the shape,
 * widths[step] and the device's SM count; 0 on a bad argument.
 */
size_t gr_decode_attn_workspace_size(const gr_attn_shape *shape, const int32_t *widths,
                                     int32_t step);

/*
 * Decode attention for all requests at decode step `step`.
 *
 *   q          device bf16 [R, W_s, Hq, D]          W_s = widths[step]
 *   ctx_k      device bf16 [R, Hkv, Lc_max, D]      shared ContextKV
 *   ctx_v      device bf16 [R, Hkv, Lc_max, D]
 *   ctx_len    device int32 [R]                     valid context positions
 *   beam_k     device bf16 [R, S_max, W_max, Hkv, D] BeamKV
 *   beam_v     device bf16 [R, S_max, W_max, Hkv, D]
 *   beam_path  device int32 [R, S_max, W_max]       parent slot at step t-1
 *   widths     HOST int32 [step+1]                  active width per step
 *   out        device bf16 [R, W_s, Hq, D]          written (round to nearest even)
 *   lse        device fp32 [R, W_s, Hq]             written, natural log of the
 *                                                   summed exp of scaled scores
 *   workspace  device scratch of workspace_bytes >= gr_decode_attn_workspace_size()
 *              (16-byte aligned; may be NULL when that size is 0)
 *
 * Context positions >= ctx_len[r] are never used, whatever they hold.
 * Errors: GR_ERR_NULL_ARG, GR_ERR_BAD_SHAPE (step outside [0, S_max),
 * widths[t] outside [1, W_max], ...), GR_ERR_UNSUPPORTED, GR_ERR_MISALIGNED,
 * GR_ERR_WORKSPACE_TOO_SMALL, GR_ERR_CUDA (launch failure).
 */
int gr_decode_attn(const gr_attn_shape *shape, const void *q, const void *ctx_k,
                   const void *ctx_v, const int32_t *ctx_len, const void *beam_k,
                   const void *beam_v, const int32_t *beam_path, const int32_t *widths,
                   int32_t step, void *out, float *lse, void *workspace,
                   size_t workspace_bytes, gr_stream_t stream);

/*
 * Paged ContextKV (SID-GR README, section 10 "TODO and Roadmap": page-backed
 * ContextKV storage and native page tables in decode attention).  The
 * context of request r is a list of pages of a shared pool:
 *     position j of request r  ->  page block_table[r * pages_per_request + j / page_size],
 *                                  offset j % page_size
 *     ctx_k_pool, ctx_v_pool   device bf16 [num_pages, Hkv, page_size, D]
 *     block_table              device int32 [R, pages_per_request]
 * Only the pages that cover positions below ctx_len[r] are read.  A page
 * index outside [0, num_pages) reads zeros (it is not followed out of the
 * pool).  Everything else -- shapes, outputs, workspace (same size as
 * gr_decode_attn for the same shape), errors -- is as for gr_decode_attn, with
 * ctx_capacity <= pages_per_request * page_size.  The CUDA-core cross-check
 * path (GR_ATTN_FORCE_PATH=simt) does not take pages: GR_ERR_UNSUPPORTED.
 */
typedef struct {
    int32_t page_size;          /* positions per page: a positive multiple of 128 */
    int32_t num_pages;          /* pages in the pool, >= 1 */
    int32_t pages_per_request;  /* block-table row length */
} gr_ctx_pages;

int gr_decode_attn_paged(const gr_attn_shape *shape, const gr_ctx_pages *pages, const void *q,
                         const void *ctx_k_pool, const void *ctx_v_pool, const int32_t *ctx_len,
                         const int32_t *block_table, const void *beam_k, const void *beam_v,
                         const int32_t *beam_path, const int32_t *widths, int32_t step, void *out,
                         float *lse, void *workspace, size_t workspace_bytes, gr_stream_t stream);

/*
 * gr_decode_attn with a width per request (SID-GR README, section 10
 * "TODO and Roadmap": per-request beam widths in one batch).  Request r has
 * width W[r][t] at step t:
 *   req_widths_host  HOST int32 [R][step+1]  (row stride step+1)
 *   req_widths       device int32 [R, S_max]  the same values (read by the kernels;
 *                    a value above the step's padded width Wpad_t is taken as Wpad_t)
 * The tensors keep the shared layout with each step's largest width
 * Wpad_t = max_r W[r][t]: q/out [R, Wpad_s, Hq, D], lse [R, Wpad_s, Hq].
 * Rows b < W[r][step] are computed; rows past a request's width hold
 * unspecified values.  Parents are checked against W[r][t-1].  The
 * workspace is gr_decode_attn_workspace_size() with widths Wpad.  Errors as
 * for gr_decode_attn; the CUDA-core cross-check path
 * (GR_ATTN_FORCE_PATH=simt) returns GR_ERR_UNSUPPORTED.
 */
int gr_decode_attn_ragged(const gr_attn_shape *shape, const void *q, const void *ctx_k,
                          const void *ctx_v, const int32_t *ctx_len, const void *beam_k,
                          const void *beam_v, const int32_t *beam_path,
                          const int32_t *req_widths_host, const int32_t *req_widths, int32_t step,
                          void *out, float *lse, void *workspace, size_t workspace_bytes,
                          gr_stream_t stream);

/*
 * Size of the static device scratch gr_decode_attn_noalloc uses: 64 MiB.
 */
#define GR_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * gr_decode_attn for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for callers such as
 * code inside an engine whose memory pool already holds the device memory
 * (so another cudaMalloc fails or breaks its accounting), and
 * latency-critical paths that cannot pay for cudaMalloc's implicit
 * synchronisation.  (A stream callback cannot call it: CUDA allows no CUDA
 * call there at all, kernel launches included.)
 *
 * Same arguments, results and errors as gr_decode_attn, without the
 * workspace: the partial results live in a static device array of
 * GR_NOALLOC_SCRATCH_BYTES inside the library.  Every check gr_decode_attn
 * makes runs first, in the same order, so both report the same error for
 * the same arguments.  Every GPU that loads the
 * library holds that array until the process exits.  The caller still
 * passes every input and output buffer.  This entry point allocates and
 * frees nothing.
 *
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture.
 *   - A call whose plan needs more scratch than GR_NOALLOC_SCRATCH_BYTES
 *     (gr_decode_attn_workspace_size() larger than it) returns
 *     GR_ERR_WORKSPACE_TOO_SMALL and enqueues nothing.
 *   - All calls share the one array and it keeps the last call's contents;
 *     nothing in it needs clearing, since each call writes every scratch
 *     entry before reading it.  Calls that may overlap on the GPU (on
 *     different streams, or from several host threads) race on the array:
 *     order them on one stream or with events.
 */
int gr_decode_attn_noalloc(const gr_attn_shape *shape, const void *q, const void *ctx_k,
                           const void *ctx_v, const int32_t *ctx_len, const void *beam_k,
                           const void *beam_v, const int32_t *beam_path, const int32_t *widths,
                           int32_t step, void *out, float *lse, gr_stream_t stream);

/*
 * gr_decode_attn, plus three CUDA events recorded on `stream`: events[0]
 * before the context-stage kernel, events[1] after it (before the per-beam
 * stage and merge), events[2] after the last kernel.  Elapsed times between
 * them give each kernel's device time without a profiler.  `events` is a
 * HOST array of 3 created events (cudaEventCreate), of which events[1] may
 * be NULL and is then not recorded (on GB300 each record adds about 2 us of
 * device time between its neighbours, so a caller timing a call that runs one
 * kernel leaves it NULL); GR_ERR_NULL_ARG when events, events[0] or events[2]
 * is NULL.  All other arguments and errors are those of gr_decode_attn.
 */
int gr_decode_attn_timed(const gr_attn_shape *shape, const void *q, const void *ctx_k,
                         const void *ctx_v, const int32_t *ctx_len, const void *beam_k,
                         const void *beam_v, const int32_t *beam_path, const int32_t *widths,
                         int32_t step, void *out, float *lse, void *workspace,
                         size_t workspace_bytes, gr_stream_t stream, gr_event_t const *events);

/* How gr_decode_attn will run a given call (filled by gr_decode_attn_plan). */
typedef struct {
    int32_t path;            /* 0: tensor-core context stage, 1: CUDA-core context stage */
    int32_t n_splits;        /* key splits of the context stage (0: no context) */
    int32_t split_len;       /* context positions per split */
    int32_t context_ctas;    /* CTAs of the context-stage kernel */
    int32_t kernels;         /* kernels one call launches */
    int32_t fused_merge;     /* 1 when the context kernel also runs the per-beam stage and merge */
    int32_t persistent;      /* 1 when one persistent kernel (one CTA per SM, 128-row tiles) runs the call */
} gr_plan_info;

/*
 * Fills *info with the plan gr_decode_attn would use for this geometry and
 * step on the current device.  Errors: those of the shape checks, and
 * GR_ERR_CUDA / GR_ERR_UNSUPPORTED when no sm_103 device is current.
 */
int gr_decode_attn_plan(const gr_attn_shape *shape, const int32_t *widths, int32_t step,
                        gr_plan_info *info);

/*
 * The ancestor walk alone (BeamPath parent pointers, GR-Inference blog
 * "system design"): anc[r, b, t] = a_t for b < widths[step], t = 0 .. step.
 *   anc  device int32 [R, W_s, step+1], written.
 * For debugging and tests; the same walk runs inside gr_decode_attn.  An
 * out-of-range parent is not followed: the walk stops there and writes -1
 * for it and for every earlier step.
 */
int gr_resolve_ancestors(const gr_attn_shape *shape, const int32_t *beam_path,
                         const int32_t *widths, int32_t step, int32_t *anc,
                         gr_stream_t stream);

/*
 * Checks gr_decode_attn's unchecked preconditions on the device: counts
 * parents outside [0, widths[t-1]) (1 <= t <= step, b < widths[t]) and
 * ctx_len entries outside [0, Lc_max].  *bad_count (device int32) is
 * overwritten with the count.  Reads nothing out of range itself.
 */
int gr_validate_beam_path(const gr_attn_shape *shape, const int32_t *beam_path,
                          const int32_t *widths, int32_t step, const int32_t *ctx_len,
                          int32_t *bad_count, gr_stream_t stream);

/*
 * Synchronises the current device, then returns and clears the library's
 * device error word: GR_OK; GR_ERR_DEVICE_TIMEOUT when a kernel gave up a
 * bounded wait (its outputs are then incomplete); GR_ERR_BAD_BEAM_PATH when
 * gr_decode_attn met a BeamPath parent outside [0, widths[t-1]) (it reads
 * nothing out of range and writes NaN to the affected rows).  GR_ERR_CUDA
 * when the synchronisation itself fails.
 */
int gr_get_device_error(void);

/*
 * Beam selection after a decode forward (SID-GR Inference README, section 10
 * "TODO and Roadmap": log_softmax + topK + beam selection on the device;
 * xGR review, "xBeam": one size-BW selection over every beam's candidates).
 *
 * For request r, active beam b < W_s with cumulative log-probability
 * beam_scores[r, b] and next-token logits logits[r, b, 0 .. V-1]:
 *     score[r, b, v] = beam_scores[r, b]
 *                    + (logits[r, b, v] - (m_b + ln sum_v' exp(logits[r, b, v'] - m_b)))
 * in fp32, m_b the row maximum.  The next_width candidates (b, v) of largest
 * score are kept, equal scores ordered by the smaller flat index b * V + v,
 * and written in that order:
 *     next_parent[r * parent_stride + j] = b   (the next BeamPath row: pass
 *                                               &beam_path[r0][s+1][0] with
 *                                               parent_stride = S_max * W_max
 *                                               to write it in place)
 *     next_token [r * next_width + j]    = v
 *     next_score [r * next_width + j]    = score[r, b, v]
 * No length penalty or score normalisation is applied (the pages leave them
 * open).  A logit of -inf masks its token; every beam needs at least one
 * finite logit, and no logit may be NaN or +inf (not checked).
 */
#define GR_SELECT_MAX_WIDTH 1024
#define GR_SELECT_MAX_BEAMS 4096

typedef struct {
    int32_t num_requests; /* R >= 1 */
    int32_t width;        /* W_s: 1 <= W_s <= GR_SELECT_MAX_BEAMS active beams per request */
    int32_t vocab;        /* V >= 1: logits per beam; W_s * V < 2^31 */
    int32_t next_width;   /* W': 1 <= W' <= min(GR_SELECT_MAX_WIDTH, W_s * V) */
} gr_select_shape;

/* Bytes of device workspace gr_beam_select needs (0 on a bad shape). */
size_t gr_beam_select_workspace_size(const gr_select_shape *shape);

/*
 *   logits       device fp32 [R, W_s, V]
 *   beam_scores  device fp32 [R, W_s]
 *   next_parent  device int32, R rows of next_width entries, row r at
 *                next_parent + r * parent_stride (parent_stride >= next_width)
 *   next_token   device int32 [R, next_width], written
 *   next_score   device fp32 [R, next_width], written
 *   workspace    device scratch of workspace_bytes >= gr_beam_select_workspace_size()
 * Device pointers must be 16-byte aligned (next_parent's rows need not be).
 * Two kernels on `stream`; nothing is allocated.  Errors: GR_ERR_NULL_ARG,
 * GR_ERR_BAD_SHAPE, GR_ERR_MISALIGNED, GR_ERR_WORKSPACE_TOO_SMALL,
 * GR_ERR_UNSUPPORTED, GR_ERR_CUDA.
 */
int gr_beam_select(const gr_select_shape *shape, const float *logits, const float *beam_scores,
                   int32_t *next_parent, int64_t parent_stride, int32_t *next_token,
                   float *next_score, void *workspace, size_t workspace_bytes,
                   gr_stream_t stream);

/*
 * gr_beam_select, plus three CUDA events recorded on `stream`: events[0]
 * before the per-row kernel, events[1] between it and the per-request merge
 * kernel, events[2] after the merge.  `events` is a HOST array of 3 created
 * events; all other arguments and errors are those of gr_beam_select.
 */
int gr_beam_select_timed(const gr_select_shape *shape, const float *logits,
                         const float *beam_scores, int32_t *next_parent, int64_t parent_stride,
                         int32_t *next_token, float *next_score, void *workspace,
                         size_t workspace_bytes, gr_stream_t stream, gr_event_t const *events);

/*
 * Item-constrained beam selection (GR-Inference blog, "kernel design": the
 * item-constrained fused kernel with the SID trie resident on the device in
 * CSR form, prefix traversal, legal-token gather and a local top-K, and no
 * full-vocabulary mask; xGR review, "xBeam": an item mask on the logits).
 *
 * The trie: node n's edges are k in [trie_offsets[n], trie_offsets[n+1]),
 * each with a token trie_tokens[k] (strictly increasing within a node, in
 * [0, V)) and a child node trie_children[k]; node 0 is the root.  Beam b of
 * request r sits at node beam_node[r, b] (the root at the first step).  Its
 * legal next tokens are its node's edge tokens, and the log_softmax is taken
 * over those only (every other logit masked):
 *     score[r, b, k] = beam_scores[r, b] + logits[r, b, t_k]
 *                      - ln sum_{k' edges of the node} exp(logits[r, b, t_k'])
 * The next_width candidates of largest score are kept exactly as
 * gr_beam_select keeps them (equal scores by the smaller b * V + token), and
 * next_node[r * next_width + j] is the chosen edge's child, so each step
 * advances the traversal one level.  A beam at a leaf has no candidates;
 * slots past a request's candidates get parent -1, token -1, score -inf and
 * node -1.  A node index, edge range or token out of range is skipped
 * (nothing is read out of it).
 */
typedef struct {
    int32_t num_requests; /* R >= 1 */
    int32_t width;        /* W_s: 1 <= W_s <= GR_SELECT_MAX_BEAMS */
    int32_t vocab;        /* V >= 1; W_s * V < 2^31 */
    int32_t next_width;   /* W': 1 <= W' <= GR_SELECT_MAX_WIDTH */
    int32_t num_nodes;    /* N >= 1 trie nodes */
    int32_t num_edges;    /* E >= 0 trie edges */
} gr_trie_select_shape;

/* Bytes of device workspace gr_trie_select needs (0 on a bad shape). */
size_t gr_trie_select_workspace_size(const gr_trie_select_shape *shape);

/*
 *   logits, beam_scores   as for gr_beam_select
 *   beam_node             device int32 [R, W_s]
 *   trie_offsets          device int32 [N + 1]
 *   trie_tokens           device int32 [E]
 *   trie_children         device int32 [E]
 *   next_parent           as for gr_beam_select (row stride parent_stride)
 *   next_token, next_node device int32 [R, next_width], written
 *   next_score            device fp32 [R, next_width], written
 * Device pointers must be 16-byte aligned (trie_tokens / trie_children may be
 * NULL when E = 0).  Two kernels on `stream`; nothing is allocated.  Errors
 * as for gr_beam_select.
 */
int gr_trie_select(const gr_trie_select_shape *shape, const float *logits, const float *beam_scores,
                   const int32_t *beam_node, const int32_t *trie_offsets, const int32_t *trie_tokens,
                   const int32_t *trie_children, int32_t *next_parent, int64_t parent_stride,
                   int32_t *next_token, float *next_score, int32_t *next_node, void *workspace,
                   size_t workspace_bytes, gr_stream_t stream);

/*
 * The per-beam cache reordered along BeamPath, out of place (xGR review,
 * "xAttention": the unshared cache is rearranged after each beam selection
 * instead of being read through parent indices; the review's update formula
 * is garbled, so this takes the plain reading):
 *     out_k/out_v[r, t, b] = beam_k/beam_v[r, t, a_t(b)]  for t = 0..step, b < widths[step]
 *     out_path[r, t, b]    = b for t >= 1 (0 at t = 0)
 * with a_step = b, a_{t-1} = beam_path[r, t, a_t].  gr_decode_attn over
 * (out_k, out_v, out_path) with every width set to widths[step] gives the
 * same rows as over (beam_k, beam_v, beam_path) with `widths`.
 *   out_k, out_v  device bf16 [R, S_max, W_max, Hkv, D], written at the rows above
 *   out_path      device int32 [R, S_max, W_max], written at the entries above
 * out_k/out_v must not be beam_k/beam_v (GR_ERR_BAD_SHAPE).  A parent outside
 * [0, widths[t-1]) is not followed: the lower levels of that beam are not
 * written and the device error word reports GR_ERR_BAD_BEAM_PATH.  Other
 * errors as for gr_resolve_ancestors.
 */
int gr_beam_reorder(const gr_attn_shape *shape, const void *beam_k, const void *beam_v,
                    const int32_t *beam_path, const int32_t *widths, int32_t step, void *out_k,
                    void *out_v, int32_t *out_path, gr_stream_t stream);

/*
 * The same reorder in place (xGR review, "xAttention": the unshared cache
 * updated in place after each beam selection, so that attention reads each
 * beam's chain from its own slots; the review's update formula is garbled,
 * so this takes the plain reading): with the chains as for gr_beam_reorder,
 *     beam_k/beam_v[r, t, b] <- beam_k/beam_v[r, t, a_t(b)]  for t = 0..step-1, b < widths[step]
 *     beam_path[r, t, b]     <- b                            for t = 1..step,   b < widths[step]
 * Level `step` (a_step = b) and beam_path[r, 0, .] are left as they are.
 * Afterwards the caller's width schedule is widths[step] at every level
 * t <= step: gr_decode_attn with those widths gives the rows it gave before
 * with the old cache, path and widths.  The usual call is right after a
 * beam selection has written the parents of step s + 1 (pass step = s + 1,
 * before that step's K/V is appended), so the next attention call reads
 * every chain through slot b.
 *   beam_k, beam_v  device bf16 [R, S_max, W_max, Hkv, D], updated
 *   beam_path       device int32 [R, S_max, W_max], read, then updated
 * One CTA owns each column tile of a (request, level) and stages its source
 * rows in shared memory before it writes, so no read sees a row already
 * overwritten.  A parent outside [0, widths[t-1]) is not followed: the beam's
 * rows below the break keep their old contents and the device error word
 * reports GR_ERR_BAD_BEAM_PATH.  Two kernels on `stream` (none at step 0).
 * Errors: GR_ERR_BAD_SHAPE (as gr_resolve_ancestors, or the three buffers
 * share a byte), GR_ERR_UNSUPPORTED (a level wider than about 14,000 slots
 * cannot be staged), GR_ERR_NULL_ARG, GR_ERR_MISALIGNED, GR_ERR_CUDA.
 */
int gr_beam_reorder_inplace(const gr_attn_shape *shape, void *beam_k, void *beam_v, int32_t *beam_path,
                            const int32_t *widths, int32_t step, gr_stream_t stream);

/*
 * BeamKV append (GR-Inference blog, "system design": BeamKV holds only the
 * short K/V each beam adds at each decode step; SID-GR README, section 3:
 * the per-beam cache grows by one token per step): the K and V that the
 * active beams' current tokens produced go to their own slots of the step's
 * plane, ahead of the attention call that reads them,
 *     beam_k[r, step, b, g, :] = k_new[(r * W_s + b) * src_stride + g * D + (0..D-1)]
 *     beam_v[r, step, b, g, :] = v_new[... same ...]             for b < W_s = widths[step]
 *   k_new, v_new    device bf16, R * W_s rows of Hkv * D values, row i at
 *                   element i * src_stride (src_stride >= Hkv * D, a
 *                   multiple of 8, so a row of a fused QKV output can be
 *                   read where it lies)
 *   beam_k, beam_v  device bf16 [R, S_max, W_max, Hkv, D], written at the
 *                   rows above only
 * One kernel on `stream`.  Errors: GR_ERR_NULL_ARG, GR_ERR_BAD_SHAPE (as
 * gr_decode_attn, src_stride too small, or a source sharing a byte with
 * beam_k/beam_v, or beam_k with beam_v), GR_ERR_MISALIGNED (a pointer, or
 * src_stride not a multiple of 8), GR_ERR_UNSUPPORTED, GR_ERR_CUDA.
 */
int gr_beam_append(const gr_attn_shape *shape, const int32_t *widths, int32_t step, const void *k_new,
                   const void *v_new, int64_t src_stride, void *beam_k, void *beam_v, gr_stream_t stream);

/* Static description of a gr_status code. */
const char *gr_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int gr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GR_ATTN_H */
