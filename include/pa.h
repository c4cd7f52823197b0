/*
 * pa.h -- C ABI of libpagedfp8: paged decode attention over an FP8 (e4m3) KV cache
 * with per-token or scalar K/V scales (and a BF16-KV control), for grouped-query
 * attention with ragged speculative-decode query lengths, split-K over long contexts
 * with a log-sum-exp merge, and a sparse selected-page variant; with the two steps next
 * to it: the per-token FP8 quantise-and-write that fills the cache
 * (pa_kv_quantize_write) and the indexer's page scores and top-k that choose the sparse
 * variant's pages (pa_index_topk); and the log-sum-exp merge that combines the parts of a
 * context split across GPUs (pa_lse_merge).  sm_103a (GB300).
 *
 * Sources of the operation (the pages are pull-request threads):
 *  - ROCm/ATOM PR 2614, "Change": dense max-q-len-1 per-token FP8 decode and sparse
 *    decode share one paged-decode contract; "Validation": the per-token kernel
 *    needs split-K.
 *  - ROCm/ATOM PR 2710, review "Must fix" 1 and "Should fix" 2: scratch is sized
 *    from a bounded set of capacity buckets and reused; an unsupported call is
 *    refused at set-up, not raised mid-run; "Smaller": partition scratch
 *    (exp_sums, max_logits, temporary_output).
 *  - ROCm/ATOM PR 2122 ("fix(minimax-m3): unblock fp8 KV cache and EAGLE3 spec decode
 *    on the vLLM plugin"), section 1: FP8 caches are raw bytes; section 2: a decode
 *    segment must be measured as uniform, rows map to requests through
 *    cu_seqlens_q, and row tok attends positions < seq_len - q_len + tok + 1.
 *  - vLLM PR 52060 ("[ROCm][Perf] Fold scalar KV scales in MiniMax-M3 sparse
 *    attention"), "Suggested Fix": a scalar K scale folds into the score scale and a
 *    scalar V scale is applied once to the normalised fp32 accumulator; per-token
 *    scales stay per token.
 *
 * Conventions for every call:
 *  - Device pointers are caller-owned device memory; the library allocates no device
 *    memory at any time.  Its only scratch is the caller's workspace, sized once per
 *    plan by pa_plan_workspace_size.
 *  - Errors are returned as pa_status_t; no call aborts, throws or prints.
 *  - pa_decode performs no host synchronisation and no allocation, and returns as
 *    soon as its kernel is enqueued on the given stream.
 */
#ifndef PAGEDFP8_PA_H
#define PAGEDFP8_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* a null pointer, a negative size or a value out of range */
  PA_ERR_UNSUPPORTED = 2,   /* a shape or mode this library does not implement */
  PA_ERR_CAPACITY = 3,      /* a call larger than its plan's capacity bucket */
  PA_ERR_RAGGED = 4,        /* a uniform plan given ragged (or miscounted) query rows */
  PA_ERR_ALIGN = 5,         /* a pointer without the required 16-byte alignment */
  PA_ERR_CUDA = 6,          /* a CUDA runtime or driver call failed */
  PA_ERR_DEVICE_DATA = 7,   /* the kernel flagged bad data (see PA_DEV_* flags) */
  PA_ERR_WORKSPACE = 8      /* the workspace is null, misaligned or too small */
} pa_status_t;

enum { PA_KV_FP8_E4M3 = 0, PA_KV_BF16 = 1 };
enum { PA_SCALE_NONE = 0, PA_SCALE_SCALAR = 1, PA_SCALE_PER_TOKEN = 2 };
enum { PA_Q_UNIFORM = 0, PA_Q_RAGGED = 1 };
enum { PA_OUT_BF16 = 0, PA_OUT_F32 = 1 };

/* Device status flags, OR-ed into the plan's workspace by the kernels.  A flagged
 * work item is skipped (its pages are not read); nothing traps.  Read them with
 * pa_plan_get_device_status. */
#define PA_DEV_BAD_PAGE      0x01u  /* a block-table entry outside [0, num_pages) */
#define PA_DEV_BAD_CONTEXT   0x02u  /* context_len < 0, > max_context_len, or more pages than the block-table stride */
#define PA_DEV_BAD_QLEN      0x04u  /* a request's q_len < 0 or > the plan's q_len, or context_len < q_len */
#define PA_DEV_NOT_UNIFORM   0x08u  /* uniform plan, but cu_seqlens_q[r] != r * q_len */
#define PA_DEV_BAD_SELECTED  0x10u  /* num_selected outside [0, selected_stride], or a selected page outside [-1, pages of the request) */
#define PA_DEV_Q_RANGE       0x20u  /* a query value outside the f16 range (|q| > 65504) */
#define PA_DEV_TIMEOUT       0x40u  /* a bounded wait inside a kernel gave up (the output is incomplete) */
#define PA_DEV_DUMP_RANGE    0x80u  /* pa_debug_gather's buffer was too small for the schedule */
#define PA_DEV_BAD_SLOT      0x100u /* pa_kv_quantize_write: a slot >= num_pages * page_size */

/* Plan flags.
 * PA_PLAN_NO_PDL: launch pa_decode as an ordinary kernel.  By default it is launched
 *   with programmatic dependent launch: its CTAs may start while the kernel before it
 *   in the stream is finishing, and read the index inputs (block_table, context_lens,
 *   cu_seqlens_q, selected_pages, num_selected) before that kernel has completed; they
 *   wait for it to complete before reading q, the caches or the scales, and before
 *   writing anything (before the wait they only ask L2 to prefetch the first pages,
 *   which reads nothing into the kernel).  So with PDL on, the kernel enqueued immediately before pa_decode
 *   must not write those index inputs (copies and host writes are unaffected).  Set
 *   this flag if it does. */
#define PA_PLAN_NO_PDL 0x1
/* PA_PLAN_TCGEN05: for an FP8 plan with q_len 1, run the tcgen05 kernel, which feeds the
 *   cache bytes to the tensor core (QK^T and PV as kind::f8f6f4 MMAs with accumulators
 *   in tensor memory), instead of the default mma.sync kernel, which widens e4m3 to f16
 *   on the SM sub-partitions.  Both give the same results within the library's
 *   tolerances.  On GB300 the default kernel is currently the faster of the two; the
 *   flag is ignored for other plans. */
#define PA_PLAN_TCGEN05 0x2

/* Plan descriptor: the capacity bucket and the fixed shape of every call on the plan
 * (ROCm/ATOM PR 2710 review, "Must fix" 1: size the plan by a capacity bucket).
 * Supported: head_dim 128, group_size 16, page_size in {16, 32, 64, 128},
 * kv_dtype FP8 with scale_mode SCALAR or PER_TOKEN, or BF16 with scale_mode NONE;
 * q_len 1..8; max_batch 1..4096. */
typedef struct pa_plan_desc {
  int32_t num_kv_heads;       /* Hkv >= 1; query heads = Hkv * group_size, head j uses KV head j / group_size */
  int32_t group_size;         /* query heads sharing one KV head */
  int32_t head_dim;           /* D */
  int32_t page_size;          /* tokens per page */
  int32_t kv_dtype;           /* PA_KV_* */
  int32_t scale_mode;         /* PA_SCALE_* */
  int32_t q_mode;             /* PA_Q_UNIFORM: every request has q_len rows; PA_Q_RAGGED: rows from cu_seqlens_q */
  int32_t q_len;              /* uniform: rows per request; ragged: the most rows one request may have */
  int32_t max_batch;          /* most requests per call */
  int32_t max_rows;           /* most query rows per call */
  int32_t max_context_len;    /* longest context (tokens, counting the request's own q_len new tokens) */
  int32_t max_selected_pages; /* 0: dense-only plan; else the most selected pages per request in sparse calls */
  int32_t partition_tokens;   /* 0: balanced persistent schedule (one CTA per SM, equal tile counts);
                                 else fixed split-K partitions of this many tokens (multiple of 128) */
  int32_t out_dtype;          /* PA_OUT_BF16 (round to nearest even) or PA_OUT_F32 */
  int32_t num_sms;            /* 0: the current device's SM count; > 0: use this count (sizing without a GPU) */
  int32_t flags;              /* PA_PLAN_* bits */
  int32_t reserved[2];        /* must be 0 */
} pa_plan_desc_t;

/* One decode call.  Layouts are dense row-major; rows = query tokens. */
typedef struct pa_decode_args {
  const void *q;                   /* device bf16 [num_rows, Hkv*group, head_dim], 16-B aligned */
  const void *k_cache;             /* device [num_pages, Hkv, page_size, head_dim]: e4m3 bytes (raw uint8 or
                                      float8_e4m3fn storage, ROCm/ATOM PR 2122 section 1) or bf16; 16-B aligned */
  const void *v_cache;             /* same layout as k_cache */
  const float *k_scale;            /* device fp32 [num_pages, Hkv, page_size]; PER_TOKEN only, 16-B aligned */
  const float *v_scale;            /* same; PER_TOKEN only */
  float k_scale_scalar;            /* SCALAR only: one K scale for the whole cache */
  float v_scale_scalar;            /* SCALAR only: one V scale */
  int64_t num_pages;               /* physical pages in each cache (bounds every block-table entry) */
  const int32_t *block_table;      /* device int32 [num_seqs, block_table_stride]: logical page -> physical page */
  int32_t block_table_stride;      /* entries per block-table row */
  int32_t num_seqs;                /* requests in this call (<= max_batch) */
  const int32_t *context_lens;     /* device int32 [num_seqs]: tokens in each request's cache, own q_len included */
  const int32_t *cu_seqlens_q;     /* device int32 [num_seqs + 1]: request r owns rows [cu[r], cu[r+1]);
                                      required by RAGGED plans, optional for UNIFORM (then checked on device) */
  const int32_t *cu_seqlens_q_host;/* host int32 [num_seqs + 1], optional: validated before launch */
  const int32_t *selected_pages;   /* device int32 [num_seqs, selected_stride] logical page indices, -1 = padding;
                                      NULL for a dense call */
  const int32_t *num_selected;     /* device int32 [num_seqs]: entries used per row of selected_pages */
  int32_t selected_stride;         /* entries per selected_pages row (<= max_selected_pages) */
  int32_t num_rows;                /* query rows in this call (<= max_rows) */
  float sm_scale;                  /* softmax scale, > 0 (1/sqrt(head_dim) for the workloads) */
  int32_t reserved0;               /* must be 0 */
  void *out;                       /* device [num_rows, Hkv*group, head_dim], bf16 or fp32 per the plan; 16-B aligned */
  float *lse;                      /* device fp32 [num_rows, Hkv*group], optional: natural-log sum of exp of the
                                      scores (-inf for an empty key set) */
} pa_decode_args_t;

/* Facts about a created plan (for tests and benchmarks). */
typedef struct pa_plan_info {
  int32_t grid_ctas;          /* CTAs per decode launch (balanced: the SM count) */
  int32_t stages;             /* KV tiles in flight per CTA */
  int32_t threads_per_cta;
  int32_t tile_tokens;        /* tokens per KV tile (128) */
  int64_t smem_bytes;         /* dynamic shared memory per CTA */
  int64_t workspace_bytes;
  int64_t partial_slots;      /* split-K partial (m, l, o) slots in the workspace */
  int32_t kernel;             /* decode kernel of the plan: 0 mma.sync, 1 tcgen05 (PA_PLAN_TCGEN05) */
  int32_t reserved;
} pa_plan_info_t;

typedef struct pa_plan pa_plan_t;

/* Validates a descriptor without touching a GPU.  PA_ERR_UNSUPPORTED for an
 * unimplemented shape or mode, PA_ERR_INVALID_ARG for an out-of-range field. */
pa_status_t pa_plan_validate(const pa_plan_desc_t *desc);

/* Workspace bytes a plan with this descriptor needs (a multiple of 256), or 0 if the
 * descriptor is refused.  Queries the current device when desc->num_sms == 0. */
size_t pa_plan_workspace_size(const pa_plan_desc_t *desc);

/* Creates a plan bound to a caller-owned device workspace of at least
 * pa_plan_workspace_size bytes (256-B aligned).  The workspace holds the split-K
 * partials, per-request merge counters and the device status word; this call
 * zero-fills its control part with a synchronous cudaMemset on the current device.
 * The plan is immutable and reusable by any call within its bucket; calls that share
 * a plan (and so its workspace) must be serialised on one stream.  On error *plan is
 * set to NULL.  With d_workspace == NULL and workspace_bytes == 0 the plan is
 * check-only: it makes no CUDA call, serves pa_decode_check (for refusing a serving
 * configuration at start-up), and pa_decode on it returns PA_ERR_WORKSPACE. */
pa_status_t pa_plan_create(const pa_plan_desc_t *desc, void *d_workspace, size_t workspace_bytes,
                           pa_plan_t **plan);

/* Host-only check of a call against its plan (capacity, mode, pointers, alignment,
 * the host mirror of cu_seqlens_q).  Launches nothing.  pa_decode runs it first. */
pa_status_t pa_decode_check(const pa_plan_t *plan, const pa_decode_args_t *args);

/* Enqueues one decode on `stream` (a cudaStream_t; NULL = the legacy default stream).
 * Refusals (PA_ERR_CAPACITY, PA_ERR_RAGGED, ...) happen before anything is enqueued.
 * Rows of requests with an empty key set are written as zeros (lse -inf).  Data errors
 * found on the device set PA_DEV_* flags instead of faulting. */
pa_status_t pa_decode(pa_plan_t *plan, const pa_decode_args_t *args, void *stream);

/* Synchronises the device, copies the plan's PA_DEV_* flags to *flags and, if clear
 * is non-zero, resets them.  For tests and diagnostics, never on the hot path. */
pa_status_t pa_plan_get_device_status(pa_plan_t *plan, uint32_t *flags, int clear);

pa_status_t pa_plan_get_info(const pa_plan_t *plan, pa_plan_info_t *info);

/* Frees the host-side plan (the workspace stays the caller's).  NULL is a no-op. */
void pa_plan_destroy(pa_plan_t *plan);

/* A static string naming the status. */
const char *pa_status_string(pa_status_t status);

/* Size of the fixed device scratch that pa_decode_noalloc uses (8 MiB per GPU). */
#define PA_NOALLOC_SCRATCH_BYTES (8u << 20)

/* pa_decode for callers that cannot allocate device memory when they set up or run a
 * decode -- for example an engine plugin whose enqueue step must not allocate, or a
 * runtime whose device memory pool is fixed before the first request -- and so cannot
 * hand pa_plan_create a workspace.  No source page has a counterpart of this call: it
 * is a convenience of this library.
 *
 * It takes the plan descriptor directly and runs the same decode as pa_decode, with the
 * split-K scratch in one fixed array of PA_NOALLOC_SCRATCH_BYTES that the library
 * reserves on every GPU that loads it, for the life of the process.  It calls no
 * cudaMalloc, cudaFree or other allocating routine, host or device.
 *  - Descriptors whose workspace (pa_plan_workspace_size) exceeds the array are
 *    refused with PA_ERR_CAPACITY (on 152 SMs a balanced plan fits for q_len <= 3);
 *    other refusals are those of pa_plan_create and pa_decode_check.
 *  - The first call on a device looks up the array's device address and sets the
 *    kernels' shared-memory limit for that device; make that first call before any
 *    stream capture on the device.
 *  - Each call first clears the scratch's status word and arrival counters on `stream`.
 *    All calls on a device share the one array, so calls that may overlap on the GPU
 *    (different streams without ordering between them) race and corrupt each other.
 *  - Device-side data flags (PA_DEV_*) of these calls are not reported. */
pa_status_t pa_decode_noalloc(const pa_plan_desc_t *desc, const pa_decode_args_t *args,
                              void *stream);

/* ---- the producer of the cache: per-token FP8 quantise-and-write ---- */

/* Arguments of pa_kv_quantize_write.  All pointers are device pointers. */
typedef struct pa_kv_write_args {
  const void *k_new;             /* bf16 [num_tokens, num_kv_heads, head_dim], 16-B aligned */
  const void *v_new;             /* bf16, same shape */
  const int64_t *slot_mapping;   /* [num_tokens]: cache slot page * page_size + offset of each
                                    token; a negative slot skips the token */
  void *k_cache;                 /* e4m3 bytes [num_pages, num_kv_heads, page_size, head_dim], 16-B aligned */
  void *v_cache;
  float *k_scale;                /* fp32 [num_pages, num_kv_heads, page_size], 4-B aligned */
  float *v_scale;
  uint32_t *status;              /* nullable; PA_DEV_BAD_SLOT is OR-ed in when a slot is past the cache */
  int64_t num_tokens;            /* >= 0; 0 enqueues nothing */
  int64_t num_pages;
  int32_t num_kv_heads;          /* >= 1 */
  int32_t head_dim;              /* 128 */
  int32_t page_size;             /* 16, 32, 64 or 128 */
  int32_t reserved;              /* 0 */
} pa_kv_write_args_t;

/* Quantises new K and V rows to the per-token FP8 cache that pa_decode reads (ROCm/ATOM
 * PR 2614: MiniMax-M3 writes FP8 KV plus per-token K/V scales, checked by a
 * producer-to-consumer operator test; ROCm/ATOM PR 2710, "Smaller": the cache-write
 * branch).  For every token t with slot s = slot_mapping[t] >= 0 and every KV head h,
 * with row = (s / page_size * num_kv_heads + h) * page_size + s % page_size:
 *   scale = max_d |x[d]| / 448 in fp32 (448 being the largest finite e4m3fn value),
 *   code[d] = x[d] / scale taken as the fp32 product x[d] * (448 / amax), the reciprocal
 *   rounded to fp32 once per row (the fp32 quotient where it overflows), then rounded to
 *   the nearest e4m3fn value (ties to even) and saturated to +-448 (all codes 0 when
 *   amax is 0),
 *   k_scale[row] = scale, k_cache[row][d] = code[d]; V the same.
 * Inputs must be finite (codes of NaN or infinite inputs are unspecified).  Slots past
 * the cache are skipped and reported through *status.  Rows of different tokens must
 * not share a slot.  One kernel launch on `stream`; no host synchronisation, no
 * allocation.  Returns PA_ERR_INVALID_ARG for a missing pointer or a bad size (also
 * num_tokens * num_kv_heads above 2^31 - 1), PA_ERR_ALIGN for a misaligned pointer,
 * PA_ERR_UNSUPPORTED for head_dim or page_size outside the list, PA_ERR_CUDA when the
 * launch fails. */
pa_status_t pa_kv_quantize_write(const pa_kv_write_args_t *args, void *stream);

/* ---- the indexer: block score and top-k page selection for the sparse decode ---- */

#define PA_DEV_BAD_INDEX_ROW 0x200u /* pa_index_topk: q_len < 0 or > max_q_len, context_len < q_len, rows past num_rows, or more pages than the stride (the request's rows are skipped) */

/* Arguments of pa_index_topk.  All pointers are device pointers. */
typedef struct pa_index_args {
  const void *q;                 /* bf16 [num_rows, index_heads, head_dim], 16-B aligned */
  const void *k_cache;           /* index cache, e4m3 bytes [num_pages, page_size, head_dim], 16-B aligned */
  const float *k_scale;          /* fp32 [num_pages, page_size], or NULL: codes read at scale 1 */
  const int32_t *block_table;    /* [num_seqs, block_table_stride] physical page of each logical page */
  const int32_t *context_lens;   /* [num_seqs] */
  const int32_t *cu_seqlens_q;   /* [num_seqs + 1]: rows of request r are [cu[r], cu[r+1]) */
  int32_t *selected;             /* out: [num_rows, topk] logical pages, -1 after num_selected */
  int32_t *num_selected;         /* out: [num_rows] */
  float *scores;                 /* out: [num_rows, block_table_stride] page scores (log2 units),
                                    -inf where a page holds no attended position; 16-B aligned */
  uint32_t *status;              /* nullable: PA_DEV_BAD_PAGE, PA_DEV_BAD_INDEX_ROW are OR-ed in */
  int64_t num_pages;
  int32_t num_seqs;
  int32_t num_rows;
  int32_t index_heads;           /* >= 1; max_q_len * index_heads <= 16 */
  int32_t head_dim;              /* 128 */
  int32_t page_size;             /* 16, 32, 64 or 128 */
  int32_t topk;                  /* 1 .. 1024 */
  int32_t block_table_stride;    /* 1 .. 16384 */
  int32_t max_q_len;             /* bound on any request's q_len, >= 1 */
  float sm_scale;                /* > 0 */
  int32_t reserved;              /* 0 */
} pa_index_args_t;

/* The indexer step before the sparse decode (ROCm/ATOM PR 2122, section 1: the index
 * cache of (num_blocks, 128, 128) e4m3 codes and the block score q . k * sm_scale * log2(e);
 * section 2: rows map to requests through cu_seqlens_q, and row tok of a request with
 * context L and q_len rows attends positions < L - q_len + tok + 1).  For each row:
 *   s[h][p] = sm_scale * log2(e) * sum_d q[row][h][d] * k[p][d] * k_scale[p] over the
 *     attended positions p, where k is the index key at p (through the block table);
 *   scores[row][b] = log2 sum_h sum_{attended p in page b} 2^s[h][p] (-inf if none);
 *   selected[row] = the row's last attended page, then the other candidates by descending
 *     score (equal scores: lower page first), topk entries at most, -1 after.
 * With q_len 1 rows are requests, and selected / num_selected are pa_decode's
 * selected_pages / num_selected.  Inputs must be finite.  Two kernel launches on
 * `stream`; no host synchronisation, no allocation.  PA_ERR_INVALID_ARG for a missing
 * pointer or a value out of range, PA_ERR_ALIGN for a misaligned pointer,
 * PA_ERR_UNSUPPORTED for head_dim, page_size or max_q_len * index_heads outside the
 * limits above, PA_ERR_CUDA when a launch fails. */
pa_status_t pa_index_topk(const pa_index_args_t *args, void *stream);

/* ---- the merge of a context split across GPUs ---- */

/* Arguments of pa_lse_merge.  All pointers are device pointers. */
typedef struct pa_lse_merge_args {
  const float *part_out;   /* fp32 [num_parts, num_rows, num_heads, head_dim]: each part's normalised
                              attention output (pa_decode with PA_OUT_F32), 16-B aligned */
  const float *part_lse;   /* fp32 [num_parts, num_rows, num_heads]: each part's natural-log LSE
                              (pa_decode's lse; -inf where the part attended no position) */
  void *out;               /* [num_rows, num_heads, head_dim], bf16 or fp32 per out_dtype, 16-B aligned */
  float *lse;              /* fp32 [num_rows, num_heads] merged LSE, or NULL */
  int32_t num_parts;       /* 1 .. 64 */
  int32_t num_rows;        /* >= 0; 0 enqueues nothing */
  int32_t num_heads;       /* >= 1 */
  int32_t head_dim;        /* 128 */
  int32_t out_dtype;       /* PA_OUT_BF16 (round to nearest even) or PA_OUT_F32 */
  int32_t reserved;        /* 0 */
} pa_lse_merge_args_t;

/* Merges attention partials computed over disjoint parts of each request's positions: the
 * combine step of a long context split across GPUs (each GPU decodes its own pages with
 * pa_decode, PA_OUT_F32 and an lse; the parts are gathered, then merged here).  It is the
 * merge of the split-K partition triple -- maximum logit, exponential sum and partial
 * output per partition, ROCm/ATOM PR 2710, "Smaller" -- with each part's (max, sum) carried
 * as its lse; MiniMax-M3 is served across four GPUs (ROCm/ATOM PR 2614, "Validation").
 * For every (row, head) v, over the parts i with lse_i > -inf:
 *   M = max_i lse_i, w_i = exp(lse_i - M),
 *   out[v] = sum_i w_i part_out_i[v] / sum_i w_i,   lse[v] = M + log sum_i w_i;
 * no such part gives out = 0 and lse = -inf (an empty part's output is never read).
 * One kernel launch on `stream`; no host synchronisation, no allocation.
 * PA_ERR_INVALID_ARG for a missing pointer or a bad size, PA_ERR_ALIGN for a misaligned
 * pointer, PA_ERR_UNSUPPORTED for head_dim other than 128 or more than 64 parts,
 * PA_ERR_CUDA when the launch fails. */
pa_status_t pa_lse_merge(const pa_lse_merge_args_t *args, void *stream);

/* ---- test hooks: exact integer / byte outputs of the row map and the page gather ---- */

/* For every query row: (request, query token, causal cutoff) as int32 triples into the
 * device buffer row_map [num_rows, 3], computed by the same device code that maps rows
 * in pa_decode (ROCm/ATOM PR 2122, section 2).  Rows no request owns are left as is. */
pa_status_t pa_debug_row_map(pa_plan_t *plan, const pa_decode_args_t *args, int32_t *row_map,
                             void *stream);

/* Bytes per KV tile in pa_debug_gather's output. */
size_t pa_debug_gather_tile_bytes(const pa_plan_t *plan);

/* Runs pa_decode's schedule and page-gather path (block table, selected pages, tile
 * loads into shared memory) and, instead of attending, writes every tile it loaded to
 * `dump` at its global tile index: a 128-byte header of int32 (request, KV head, tile,
 * flags, context_len, q_len, first row, valid pages, then 8 first-positions and 8
 * physical pages, -1 where a page slot is empty), the K tile and the V tile as
 * [128 tokens][head_dim] elements with the swizzle undone, then (FP8 per-token) the
 * 128 K and 128 V scales.  Tiles are numbered request-major, then KV head, then tile;
 * dump must hold (number of tiles) * pa_debug_gather_tile_bytes bytes, given as
 * dump_bytes (tiles past it set PA_DEV_DUMP_RANGE and are skipped). */
pa_status_t pa_debug_gather(pa_plan_t *plan, const pa_decode_args_t *args, void *dump,
                            size_t dump_bytes, void *stream);

/* Launch trace of the mma.sync decode kernel, a diagnostic: the GPU global timer (ns) at
 * fixed points of each CTA's run, kept for each CTA's last 16 launches on the current
 * device.  Copies min(bytes, 2 MiB) of the array uint64 [16 slots][1024 CTAs][16 marks]
 * to host memory; slot = the CTA's launch count mod 16.  Marks: 0 entry, 1 prologue (the
 * schedule) done, 2 producer past the dependency wait, 3 consumers past it, 4 first tile
 * in warp 0, 5 warp 0 through the CTA's range, 6 partial stored, 7 arrival counted,
 * 8 / 9 merge start / end, 10 exit, 11 the CTA's launch count, 12 / 13 its tile range
 * [a, b), 14 merge duty bits; marks a launch does not reach keep older values.  Returns
 * PA_ERR_UNSUPPORTED unless the library was built with tracing (its kernels carry no
 * trace code otherwise), PA_ERR_CUDA if the copy fails. */
pa_status_t pa_debug_trace(void *host, size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDFP8_PA_H */
