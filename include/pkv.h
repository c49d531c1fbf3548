/*
 * pkv.h -- C ABI of pkv: single-token grouped-query decode attention over a
 * block-table paged KV cache, hand-written CUDA for GB300 (sm_103a).
 *
 * The operation is the one "PersistentKV: Page-Aware Decode Scheduling for
 * Long-Context LLM Serving on Commodity GPUs" (gist.science summary) states in
 * its Technical Summary:
 *   - Problem Statement: decode attention is bound by KV-cache movement;
 *   - Methodology section 1 "Native Block-Table Decode Engine": G = Hq/Hkv query
 *     heads share one KV head; attention runs directly over the paged layout
 *     through the block table ("Layout"); the sequence is cut into disjoint
 *     splits whose partial softmax states a merge combines exactly ("Sequence
 *     Splitting"); split ranges follow each row's true length and empty splits
 *     write neutral states ("Row-Local Bounds"); only non-empty
 *     (row, KV head, split) tiles are emitted ("Compact Workqueue");
 *   - Methodology section 2 "Calibrated Adaptive Policy": the route (split,
 *     queue, or a single-pass kernel) is chosen from the batch size and the
 *     longest context.
 * The persistent mode drains the work queue with an atomic counter, as the
 * persistent worker of "GPUOS" (arXiv 2604.17861, section 4.1 "Persistent
 * Kernel Executor") and the resident kernel of "WPK persistent kernel"
 * (dotwave.ai, "What a persistent kernel is") do with their task lists.
 *
 * Definition computed, for row b < B, query head h < Hq, kvh = floor(h / G):
 *     s_t = (1/sqrt(D)) * <q[b][h], K[kvh] of token t>     for t < seq_lens[b]
 *     out[b][h] = sum_t softmax(s)_t * V[kvh] of token t
 *     lse[b][h] = ln sum_t exp(s_t)             (natural log; -inf for an empty row)
 * Token t of row b lives in page block_table[b][t / page_size], slot
 * t % page_size.  An empty row gives out = 0, lse = -inf.
 *
 * Layouts (all row-major, dense, device memory unless stated):
 *   q            bf16  [B][Hq][D]
 *   k_pages      bf16  [num_pages][page_size][Hkv][D]   (v_pages the same)
 *   block_table  int32 [B][max_pages_per_seq]
 *   seq_lens     int32 [B]
 *   out          fp32  [B][Hq][D]
 *   lse          fp32  [B][Hq]
 * Supported shapes: D in {64, 128}; G in {1, 2, 4, 8}; page_size a multiple of
 * 16 up to 256.  Every device pointer must be 16-byte aligned.
 *
 * Ownership: the caller owns every tensor.  The library owns the plan (host
 * queue in pinned memory, device queue, split workspace, counters, status
 * word) and the page pool.  Nothing else is allocated per call.
 *
 * Errors: every call returns a pkv_status_code.  No call aborts, and device
 * code never traps: a bad page id, a plan that does not match the device
 * lengths, or a wait that runs out sets a bit in the plan's device status word
 * (read with pkv_status) and poisons the affected outputs with NaN.
 *
 * Streams: pkv_stream_t is the same type as cudaStream_t; NULL is the legacy
 * default stream.  Calls that take a stream only enqueue work on it.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *pkv_stream_t;

/* Return codes. */
enum pkv_status_code {
    PKV_OK = 0,
    PKV_EINVAL = 1,         /* bad argument: geometry, length, page id, null pointer */
    PKV_ENOMEM = 2,         /* host or device allocation failed */
    PKV_ECUDA = 3,          /* a CUDA runtime call failed (see pkv_last_cuda_error) */
    PKV_EUNSUPPORTED = 4,   /* shape the kernels are not built for */
    PKV_EDEVICE = 5,        /* the device status word is non-zero (pkv_status) */
    PKV_ENOSPACE = 6        /* page pool exhausted / row table full */
};

/* Bits of the device status word. */
enum pkv_device_status_bits {
    PKV_DEV_PAGE_OOB = 1u,       /* a block-table entry outside [0, num_pages) */
    PKV_DEV_PLAN_MISMATCH = 2u,  /* the device seq_lens disagree with the plan */
    PKV_DEV_TIMEOUT = 4u,        /* a bounded wait inside a kernel ran out */
    PKV_DEV_ROW_FULL = 8u        /* an append found no page for a row's new token: the row's
                                    table is full, or its entry for that position is unassigned
                                    (negative); an entry naming a page outside the pool sets
                                    PKV_DEV_PAGE_OOB instead */
};

/* Execution routes (Methodology section 2 of the PersistentKV summary). */
enum pkv_mode {
    PKV_MODE_AUTO = 0,          /* let the policy choose */
    PKV_MODE_DIRECT = 1,        /* one CTA per (row, KV head); no split, no merge */
    PKV_MODE_SPLIT_QUEUE = 2,   /* one CTA per compact-queue tile; exact LSE merge of splits */
    PKV_MODE_SPLIT_PADDED = 3,  /* one CTA per slot of the padded B*Hkv*S_max grid; merge */
    PKV_MODE_PERSISTENT = 4     /* SM-sized grid drains the compact queue; merge */
};

typedef struct {
    int32_t batch;              /* B */
    int32_t num_q_heads;        /* Hq */
    int32_t num_kv_heads;       /* Hkv; Hq % Hkv == 0 */
    int32_t head_dim;           /* D */
    int32_t max_pages_per_seq;  /* row stride of block_table */
    int32_t num_pages;          /* pages in the pool */
} pkv_geom;

/* Planner options.  Zero means "default" for every field, so a zeroed struct
 * (or a NULL pointer) gives the calibrated policy. */
typedef struct {
    int32_t force_mode;          /* pkv_mode; PKV_MODE_AUTO lets the policy choose */
    int32_t num_splits;          /* > 0: split count S, chunk C = ceil(P_max / S) pages */
    int32_t direct_units_per_sm; /* policy: DIRECT when B*Hkv >= this * SMs (default 2); smaller
                                    batches take SPLIT_QUEUE, one split per row if rows are short */
    int32_t target_ctas_per_sm;  /* policy: aim for this many tiles per SM (default 2) */
    int32_t min_chunk_pages;     /* policy: smallest split chunk in pages (default 8) */
    int32_t ctas_per_sm;         /* persistent grid = SMs * this (default: occupancy) */
    int32_t separate_merge;      /* split routes: 1 = merge in its own launch, 0 = the last
                                    arriving split of each (row, KV head) merges (default) */
    int32_t num_sms;             /* SM count to plan for (default: current device) */
    int32_t math;                /* pkv_math: block reduction on tensor cores or CUDA cores */
    int32_t copy;                /* pkv_copy: how K/V pages reach shared memory */
    int32_t merge;               /* pkv_merge: how the fused merge is shared out */
} pkv_plan_opts;

/* How the split routes merge the partial states of a (row, KV head) inside the
 * attention launch (with separate_merge = 0). */
enum pkv_merge {
    PKV_MERGE_AUTO = 0,   /* LAST */
    PKV_MERGE_LAST = 1,   /* the last split to arrive merges all partials; the launch may
                             overlap the previous kernel's tail (programmatic dependent launch) */
    PKV_MERGE_ALL = 2     /* every split waits for the others, then merges a 1/S share of the
                             outputs: a shorter merge, but a cooperative launch, which does not
                             overlap the previous kernel; needs the queue or padded route with
                             a grid that fits on the device at once, else PKV_EUNSUPPORTED */
};

/* How the producer warp moves K/V blocks into shared memory. */
enum pkv_copy {
    PKV_COPY_AUTO = 0,   /* TMA on the direct, split-queue and padded routes; cp.async on the
                            persistent route (the faster of the two on each, as measured) */
    PKV_COPY_LSU = 1,    /* cp.async 16-byte copies issued by all 32 producer lanes */
    PKV_COPY_TMA = 2     /* cp.async.bulk.tensor boxes of 16 tokens x 64 elements */
};

/* How a 16-token block is reduced (results agree to the stated tolerances). */
enum pkv_math {
    PKV_MATH_AUTO = 0,   /* tensor cores */
    PKV_MATH_FMA = 1,    /* fp32 FMA on CUDA cores */
    PKV_MATH_MMA = 2     /* mma.sync bf16 x bf16 -> fp32, P split into bf16 hi + lo */
};

/* One work tile: KV head `kvh` of row `b`, split `split`, pages
 * [page_begin, page_end) of the row (end exclusive). 20 bytes. */
typedef struct {
    int32_t b, kvh, split, page_begin, page_end;
} pkv_work_item;

typedef struct {
    int32_t mode;               /* resolved pkv_mode */
    int32_t chunk_pages;        /* C */
    int32_t max_splits;         /* S_max = ceil(P_max / C) */
    int32_t num_tiles;          /* tiles the attention launch covers */
    int32_t num_work_items;     /* length of the compact queue */
    int32_t empty_tiles;        /* padded-grid slots with no pages */
    int32_t launches_per_step;  /* kernels pkv_decode launches */
    int32_t grid_ctas;          /* CTAs of the attention launch */
    int32_t num_sms;            /* SM count planned for */
    int32_t merge;              /* 0: no split is merged; pkv_merge LAST or ALL; 3: separate launch */
    int64_t kv_bytes;           /* sum_b N_b * Hkv * D * 2 (K and V) * 2 B */
    int64_t workspace_bytes;    /* split partial states written + read per step */
    int64_t table_bytes;        /* block-table entries read per step */
    int32_t copy;               /* the resolved pkv_copy: PKV_COPY_LSU or PKV_COPY_TMA */
} pkv_plan_info;

typedef struct pkv_plan_s *pkv_plan_t;
typedef struct pkv_pool_s *pkv_pool_t;
typedef struct pkv_session_s *pkv_session_t;

/*
 * Build a plan: validate the problem, run the policy, enumerate the work tiles
 * in lexicographic (b, kvh, split) order and size the split workspace.
 *   seq_lens_h     host int32 [B]; 0 <= N_b <= max_pages_per_seq * page_size
 *   block_table_h  host int32 [B][max_pages_per_seq] or NULL; when given, the
 *                  first ceil(N_b / page_size) entries of every row are checked
 *                  to lie in [0, num_pages)
 *   page_size      tokens per page
 *   opts           NULL for defaults
 * Binds to the current CUDA device.  On success *plan owns device memory until
 * pkv_plan_destroy.  The queue reaches the device inside the next pkv_decode,
 * on that call's stream.  Errors: PKV_EINVAL, PKV_EUNSUPPORTED, PKV_ENOMEM,
 * PKV_ECUDA; *plan is left NULL on error.
 */
int pkv_plan(const int32_t *seq_lens_h, const int32_t *block_table_h, int32_t page_size,
             const pkv_geom *geom, const pkv_plan_opts *opts, pkv_plan_t *plan);

/* The planner alone, on the host: validation, policy and tile enumeration with
 * no device touched.  opts->num_sms must be set (> 0); the persistent grid uses
 * opts->ctas_per_sm (default 1).  Fills *info (nullable), copies up to
 * `capacity` tiles (as pkv_plan_queue would) and sets *count. */
int pkv_plan_dry_run(const int32_t *seq_lens_h, const int32_t *block_table_h, int32_t page_size,
                     const pkv_geom *geom, const pkv_plan_opts *opts, pkv_plan_info *info,
                     pkv_work_item *items, int32_t capacity, int32_t *count);

/* Re-plan for new lengths (same geometry, page size and options), reusing the
 * plan's buffers; they grow only when the new tile count needs more room.
 * Waits for the previous upload of the queue to finish before rewriting it.
 * Errors: PKV_EINVAL / PKV_EUNSUPPORTED leave the plan as it was.  After
 * PKV_ENOMEM (or PKV_ECUDA) the plan's buffers may not hold the new tiles: a
 * decode with it returns PKV_ENOMEM and launches nothing until an update
 * succeeds. */
int pkv_plan_update(pkv_plan_t plan, const int32_t *seq_lens_h, const int32_t *block_table_h);

void pkv_plan_destroy(pkv_plan_t plan);

int pkv_plan_get_info(pkv_plan_t plan, pkv_plan_info *info);

/* Copy the plan's tiles to host memory: the compact queue (SPLIT_QUEUE,
 * PERSISTENT), the padded grid with its empty slots (SPLIT_PADDED), or one tile
 * per (row, KV head) (DIRECT).  *count receives the total; at most `capacity`
 * items are written. */
int pkv_plan_queue(pkv_plan_t plan, pkv_work_item *items, int32_t capacity, int32_t *count);

/*
 * Decode attention for every (row, query head); see the definition above.
 *   q, k_pages, v_pages   device bf16 (as uint16 bit patterns or __nv_bfloat16)
 *   block_table_d         device int32 [B][max_pages_per_seq]
 *   seq_lens_d            device int32 [B]; must equal the lengths the plan was built from
 *   out, lse              device fp32 outputs
 * Enqueues 1 or 2 kernels (pkv_plan_info.launches_per_step) on `stream`.
 * Errors: PKV_EINVAL (null pointer, misalignment), PKV_ENOMEM (a plan whose
 * last pkv_plan_update ran out of memory), PKV_ECUDA (launch failure).
 * Device-side faults are reported through pkv_status.
 */
int pkv_decode(const void *q, const void *k_pages, const void *v_pages,
               const int32_t *block_table_d, const int32_t *seq_lens_d, pkv_plan_t plan,
               float *out, float *lse, pkv_stream_t stream);

/*
 * pkv_decode with host buffers: q_h (bf16 [B][Hq][D]) in, out_h / lse_h (fp32)
 * out; synchronises `stream`.  No copy engine is used: pinned host memory
 * (cudaMallocHost, cudaHostAlloc, cudaHostRegister) is mapped into the GPU's
 * address space, and on GB300 the kernel reads q and writes out / lse there
 * directly, over NVLink-C2C.  A buffer that is pageable (or whose mapped
 * address is not 16-byte aligned; 4 for lse_h) goes through pinned staging
 * owned by the plan, with a host memcpy before (q) or after (out, lse) the
 * decode.  A plan re-planned since its last upload is likewise read in place
 * from its pinned host copy.  The other arguments and errors are those of
 * pkv_decode; ENOMEM if the staging cannot be allocated.
 */
int pkv_decode_host(const void *q_h, const void *k_pages, const void *v_pages, const int32_t *block_table_d,
                    const int32_t *seq_lens_d, pkv_plan_t plan, float *out_h, float *lse_h, pkv_stream_t stream);

/*
 * Append one new token per row: for every row b and KV head, write
 * k_new[b][kvh][:] / v_new[b][kvh][:] (device bf16 [B][Hkv][D]) at position
 * seq_lens_d[b] -- page block_table_d[b][pos / page_size], slot
 * pos % page_size -- and then increment seq_lens_d[b].  The page for a new
 * position must already be in the table (see pkv_pool_reserve).  A row whose
 * table is full or whose entry for the position is negative sets
 * PKV_DEV_ROW_FULL, one whose entry is >= num_pages sets PKV_DEV_PAGE_OOB; such
 * a row is left unchanged (no page byte written, length not incremented).
 * Only the plan's geometry and page size are used.  One kernel on `stream`.
 */
int pkv_append(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
               const int32_t *block_table_d, int32_t *seq_lens_d, pkv_plan_t plan,
               pkv_stream_t stream);

/* Read and clear the plan's device status word (synchronises `stream`). */
int pkv_status(pkv_plan_t plan, pkv_stream_t stream, uint32_t *status);

/*
 * Copy the split workspace of the last pkv_decode to host memory (synchronises
 * `stream`): o_h fp32 [n][G][D] normalised partial outputs and lse_h fp32 [n][G]
 * natural-log partial LSEs, one entry per tile in pkv_plan_queue order (SPLIT_*
 * and PERSISTENT modes).  Entries of rows that needed no merge are not written
 * by the kernels and hold stale data.  For tests and diagnostics.
 */
int pkv_read_workspace(pkv_plan_t plan, pkv_stream_t stream, float *o_h, float *lse_h,
                       int32_t capacity, int32_t *count);

/*
 * Failure-detection self-test of the kernels' bounded waits: one thread waits,
 * with the pipeline's own wait routine and a limit of `limit_ns` (at most 2 s),
 * on an mbarrier phase that nothing completes.  The wait must give up, set
 * PKV_DEV_TIMEOUT in *status_h and raise its CTA's abort flag, after which a
 * second wait returns at once.  result_h[3] = {first wait succeeded, abort flag
 * raised, second wait succeeded}.  Synchronises the device; no GPU fault or
 * hang is involved, the context stays usable.
 */
int pkv_selftest_wait(int64_t limit_ns, uint32_t *status_h, int32_t *result_h);

/*
 * Per-CTA timeline of the attention launch, a diagnostic (the debug per-CTA
 * tile counter and phase stamps).  While enabled, every attention launch of
 * pkv_decode / pkv_decode_host writes one row of PKV_TRACE_WORDS uint64 per CTA
 * into a device buffer owned by the plan (grown, synchronously, when a launch
 * has more CTAs than it holds); pkv_trace_read synchronises the device and
 * copies the last traced launch's rows out (row = blockIdx.x; *count = its
 * CTAs; no event is recorded between launches, so tracing leaves the overlap of
 * back-to-back launches as it is).  Word i of a
 * row: 0 tiles the CTA ran; 1 its SM; then %globaltimer ns of 2 kernel entry,
 * 3 grid dependency wait released, 4 consumer warp 0 holds its first block,
 * 5 consumer warp 0 has reduced its last block, 6 the last tile's warp states
 * combined and written, 7 split arrival counted, 8 merge done (only a CTA that
 * merged), 9 CTA done; 10 (b << 40) | (kvh << 20) | split of its last tile;
 * 0 where a phase did not occur.  Rows are written after the grid dependency
 * wait, so back-to-back launches do not mix.  Off: one uniform branch per
 * phase.  Results are unchanged by tracing.
 */
#define PKV_TRACE_WORDS 12
int pkv_trace_enable(pkv_plan_t plan, int32_t enable);
int pkv_trace_read(pkv_plan_t plan, uint64_t *rows_h, int32_t capacity, int32_t *count);

/* Per-launch timing.  While enabled, pkv_decode brackets each kernel it
 * launches with CUDA events; pkv_profile_read waits for them and returns the
 * durations in milliseconds of the last pkv_decode's launches, in launch order. */
int pkv_profile_enable(pkv_plan_t plan, int32_t enable);
int pkv_profile_read(pkv_plan_t plan, float *ms, int32_t capacity, int32_t *count);

/*
 * Host page pool: a FIFO free list of page ids, for callers that grow rows one
 * token at a time (the continuous-session workload).
 *   pkv_pool_create     copies `count` free page ids, handed out in that order
 *                       (PKV_EINVAL for an id outside [0, num_pages) or listed twice)
 *   pkv_pool_reserve    for every row whose next token (position seq_lens_h[b])
 *                       starts a new page whose table entry is still unassigned
 *                       (negative), pops a page into
 *                       block_table_h[b][seq_lens_h[b] / page_size]; writes the
 *                       rows it touched to rows_out (nullable, capacity B) and
 *                       their number to *n_rows.  PKV_ENOSPACE when the pool or
 *                       a row's table runs out (no row is changed then).
 *   pkv_pool_release    returns pages to the back of the free list; PKV_EINVAL
 *                       (and no change) for a page that is already free
 */
int pkv_pool_create(const int32_t *free_pages, int32_t count, int32_t num_pages, pkv_pool_t *pool);
int pkv_pool_reserve(pkv_pool_t pool, const int32_t *seq_lens_h, int32_t *block_table_h,
                     int32_t batch, int32_t max_pages_per_seq, int32_t page_size,
                     int32_t *rows_out, int32_t *n_rows);
int pkv_pool_release(pkv_pool_t pool, const int32_t *pages, int32_t count);
int32_t pkv_pool_free_count(pkv_pool_t pool);
void pkv_pool_destroy(pkv_pool_t pool);

/*
 * pkv_decode_static: decode attention for callers that cannot allocate device
 * memory.  The PersistentKV summary has no counterpart; this is a deployment
 * variant.  Code that runs inside another framework's memory budget, real-time
 * loops that must not touch the allocator, and hosts that forbid cudaMalloc
 * after start-up cannot build a plan (pkv_plan allocates).  This call needs
 * none: it runs the padded split route with fused merge and keeps its split
 * workspace, arrival counters and status word in one fixed device array of
 * PKV_STATIC_SCRATCH_BYTES that the library declares at file scope (every GPU
 * that loads the library holds it until the process exits).  It calls no
 * allocating routine.
 *   q, k_pages, v_pages, block_table_d, seq_lens_d, out, lse: as in pkv_decode
 *   max_seq_len  host bound on seq_lens_d[b] that sizes the split grid: with
 *                P = ceil(max_seq_len / page_size) pages and S splits, the chunk
 *                is C = ceil(P / S) pages (raised if needed so that S_max * G
 *                stays within the merge's 4096-float scratch) and S_max =
 *                ceil(P / C) splits cover S_max * C >= P pages per row.  A row
 *                whose pages fit in S_max * C is decoded exactly, even if it is
 *                a little longer than max_seq_len; a row with more pages than
 *                that (or negative, or longer than max_pages_per_seq *
 *                page_size) reads no KV and gets NaN out and lse
 *   num_splits   S (> 0)
 * Needs B * Hkv * S_max * G * (D + 1) * 4 bytes of workspace plus a few KB of
 * counters within PKV_STATIC_SCRATCH_BYTES; larger problems get PKV_ENOSPACE
 * before anything is enqueued.  The first call with a device current looks the
 * array's device address up with cudaGetSymbolAddress and keeps it for that
 * device's current context (a device reset brings a new context and a new
 * look-up); make that first call before any stream capture.  All calls on a
 * device share the array and it keeps the last call's contents (counters are
 * cleared on `stream` by each call), so calls that overlap on the GPU race:
 * keep them ordered on one stream.  Device-side faults poison outputs with NaN;
 * there is no status read-back.  PKV_ECUDA records the CUDA error for
 * pkv_last_cuda_error.
 */
#define PKV_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)
int pkv_decode_static(const void *q, const void *k_pages, const void *v_pages, const int32_t *block_table_d,
                      const int32_t *seq_lens_d, int32_t page_size, const pkv_geom *geom, int32_t max_seq_len,
                      int32_t num_splits, float *out, float *lse, pkv_stream_t stream);

/*
 * Continuous sessions: B rows that each grow by one token per step, advanced
 * together (the cohort of "WPK persistent kernel", dotwave.ai, "What has to
 * exist instead": fixed arenas, sessions advanced every beat).
 *   pkv_session_create   binds a plan (its geometry and options), a page pool,
 *                        the caller's device table and lengths; copies the host
 *                        lengths and table into pinned mirrors owned by the
 *                        session
 *   pkv_session_step     one step on `stream`: the pool hands a page to every row
 *                        whose next token starts one; the plan is rebuilt for the
 *                        lengths after the append; then two launches: one enters
 *                        the new pages in the device table, moves the plan to
 *                        the device (both read in place from mapped pinned host
 *                        memory, no copy engine) and appends k_new / v_new
 *                        (device bf16 [B][Hkv][D]); then pkv_decode (q, out,
 *                        lse).  The host staging is reused by the next step
 *                        only after the first launch has run.  PKV_EINVAL for
 *                        a null or misaligned pointer, PKV_ENOSPACE when the
 *                        pool or a row runs out (nothing changes or is enqueued
 *                        then).  After PKV_ENOMEM or PKV_ECUDA the host mirrors
 *                        may be a step ahead of the device: destroy the session
 *   pkv_session_lengths / pkv_session_table   copy the host mirrors out
 * The session does not own the plan, the pool or any device memory.
 */
int pkv_session_create(pkv_plan_t plan, pkv_pool_t pool, const int32_t *seq_lens_h, const int32_t *block_table_h,
                       int32_t *block_table_d, int32_t *seq_lens_d, pkv_session_t *session);
int pkv_session_step(pkv_session_t session, const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                     const void *q, float *out, float *lse, pkv_stream_t stream);
int pkv_session_lengths(pkv_session_t session, int32_t *seq_lens_h);
int pkv_session_table(pkv_session_t session, int32_t *block_table_h);
void pkv_session_destroy(pkv_session_t session);

/*
 * Switch a session to device-planned steps (the plan must use the persistent
 * route).  Allocates the device free list (the pool's remaining pages move to
 * it, in order), the device plan buffers and a workspace for the largest plan
 * the table allows; synchronises `stream`.  Afterwards every pkv_session_step
 * only enqueues work: a one-CTA planner kernel (page allocation in row order,
 * queue in (b, kvh, s) order, longest-first hand-out order; see
 * paged_kv_decode_block_gb300/csrc/pkv_devplan.cu), the append, and the
 * persistent decode over the device-built plan -- no host work and no host
 * data per step, so a step can be captured once in a CUDA graph and replayed.
 * The split chunk is fixed at this call (one split per row stays one split).
 * pkv_session_lengths / pkv_session_table then read the device copies
 * (synchronising the device).  Up to 2048 rows.
 */
int pkv_session_device_plan(pkv_session_t session, pkv_stream_t stream);
/* Copy the last device-built plan: its tiles in queue order and the hand-out
 * order (synchronises the device).  *count receives the tile count. */
int pkv_session_device_queue(pkv_session_t session, pkv_work_item *items, int32_t *order, int32_t capacity,
                             int32_t *count);

/*
 * Slot admit / evict at step boundaries.  The rows of a session are fixed
 * slots, as the per-session state of "WPK persistent kernel" (dotwave.ai,
 * "What has to exist instead") lives in fixed arenas whose slots are reset at
 * a beat boundary.  A slot is active (it takes one token per step) or idle:
 * length 0, no pages, skipped by the append and by page allocation, and decoded
 * to the neutral state (out 0, lse -inf).  Every row is active when the session
 * is created.
 *   pkv_session_evict   makes the n listed active rows idle: their pages (every
 *                       non-negative entry of the row's table, in table order,
 *                       rows in the order listed) go to the back of the free
 *                       list, their table entries become -1 and their lengths 0
 *   pkv_session_admit   gives each of the n listed idle rows a new session of
 *                       lens_h[i] >= 0 tokens: ceil(lens_h[i] / page_size) pages
 *                       from the front of the free list (rows in the order
 *                       listed, pages in table order), that length, and its
 *                       prompt's K/V copied into those pages from k_src / v_src
 *                       (device bf16 [sum_i lens_h[i]][Hkv][D], the rows' tokens
 *                       one after another in the order listed)
 * The free list is the session's host pool, or, after pkv_session_device_plan,
 * the device free list, which then lives on the GPU: the requests go to the
 * device through a pinned, mapped slot table and one kernel applies them (a
 * graph-captured step needs no re-capture); an admission the device free list
 * cannot serve sets PKV_DEV_ROW_FULL and leaves that row and the rows listed
 * after it idle.  Both calls enqueue their device work on `stream`, to run
 * between two steps.  Errors (nothing changes): PKV_EINVAL for a row out of
 * range, listed twice, or in the wrong state (evict: not active; admit: not
 * idle), a null or misaligned pointer, a length above max_pages_per_seq *
 * page_size; PKV_ENOSPACE when the host pool holds too few pages; PKV_EINVAL
 * while a resident kernel runs (use pkv_resident_evict / pkv_resident_admit).
 */
int pkv_session_evict(pkv_session_t session, const int32_t *rows_h, int32_t n, pkv_stream_t stream);
int pkv_session_admit(pkv_session_t session, const int32_t *rows_h, const int32_t *lens_h, int32_t n,
                      const void *k_src, const void *v_src, void *k_pages, void *v_pages, pkv_stream_t stream);
/* Copy the session's free list, front first (the host pool, or the device free
 * list in device-plan mode, which synchronises the device); *count receives its
 * length, at most `capacity` ids are written.  active_h (nullable, [B]) receives
 * 1 for an active row, 0 for an idle one. */
int pkv_session_free_pages(pkv_session_t session, int32_t *pages_h, int32_t capacity, int32_t *count,
                           int32_t *active_h);

/*
 * Resident steps (a continuous session kept on the GPU by one launch).
 * pkv_resident_start launches one cooperative kernel over every SM on a stream
 * of its own; the kernel stays resident and runs one step each time the host
 * publishes one through a control block in mapped pinned host memory.  A step
 * is what a device-planned pkv_session_step enqueues -- page allocation and
 * plan (the device planner), the append of k_new / v_new, the persistent
 * decode of q into out / lse -- with one grid-wide barrier (after the plan)
 * instead of launches: each row is marked ready once its token is appended and
 * its tiles wait for that mark, and the last CTA to finish the decode
 * publishes the step; in the spirit of the persistent worker of "GPUOS"
 * (arXiv 2604.17861, section 4.1) and the resident beat of "WPK persistent
 * kernel" (dotwave.ai).  yield_every (the GPUOS host API's set_yield_every,
 * section 4, Table 1) bounds how long the kernel holds the GPU: after that many
 * steps it leaves, and the next pkv_resident_step launches it again (0: it
 * stays until pkv_resident_stop).
 *   pkv_resident_start   session in device-plan mode; k_pages / v_pages the
 *                        pools; q_d, k_new_d, v_new_d, out_d, lse_d device
 *                        buffers of the step's inputs and outputs (caller
 *                        owned, bound for the kernel's life); idle_limit_ns
 *                        (0, 60 s]: the longest the kernel waits for the next
 *                        step before leaving with PKV_DEV_TIMEOUT; times_cap:
 *                        steps whose device start / end times are kept;
 *                        yield_every >= 0 as above.  Synchronises the device
 *                        first.  PKV_EUNSUPPORTED if the kernel cannot be
 *                        resident on this device
 *   pkv_resident_step    copies the host inputs given (pinned host pointers, or
 *                        NULL to keep the device buffer) to the bound buffers,
 *                        publishes the step, waits (at most wait_limit_ns) for
 *                        the kernel to finish it, then copies out / lse to the
 *                        host pointers given.  PKV_EDEVICE if the kernel left
 *                        its loop or the wait ran out (then pkv_resident_stop)
 *   pkv_resident_stop    asks the kernel to leave and waits for it; PKV_EDEVICE
 *                        if it had left on an error (see pkv_status)
 *   pkv_resident_times   after stop: [count][4] globaltimer ns of each kept
 *                        step: the kernel saw it, plan done, append done,
 *                        outputs published (the last times_cap steps, by
 *                        step index modulo times_cap)
 * While a resident kernel runs, the session refuses pkv_session_step and its
 * read-back calls (PKV_EINVAL), and no other kernel should be queued behind it
 * on the device: it holds every SM until it is stopped or yields.  Between a
 * yield and the next step the GPU is free for other work.
 */
typedef struct pkv_resident_s *pkv_resident_t;
int pkv_resident_start(pkv_session_t session, void *k_pages, void *v_pages, void *q_d, void *k_new_d,
                       void *v_new_d, float *out_d, float *lse_d, int64_t idle_limit_ns, int32_t times_cap,
                       int32_t yield_every, pkv_resident_t *resident);
int pkv_resident_step(pkv_resident_t resident, const void *q_h, const void *k_new_h, const void *v_new_h,
                      float *out_h, float *lse_h, int64_t wait_limit_ns);
int pkv_resident_stop(pkv_resident_t resident);
int pkv_resident_times(pkv_resident_t resident, uint64_t *stamps_ns, int32_t capacity, int32_t *count);
/* Launches of the resident kernel so far (1 + the relaunches after yields). */
int pkv_resident_launches(pkv_resident_t resident, int32_t *launches);
void pkv_resident_destroy(pkv_resident_t resident);
/* Slot requests for a running resident kernel, applied at the start of the next
 * pkv_resident_step, before its page allocation and plan: the same evictions and
 * admissions as pkv_session_evict / pkv_session_admit (device free list; k_src /
 * v_src device memory that must stay valid until that step returns).  Up to
 * PKV_RESIDENT_MAX_REQUESTS rows per step; PKV_EINVAL / PKV_ENOSPACE as there. */
#define PKV_RESIDENT_MAX_REQUESTS 64
int pkv_resident_evict(pkv_resident_t resident, const int32_t *rows_h, int32_t n);
int pkv_resident_admit(pkv_resident_t resident, const int32_t *rows_h, const int32_t *lens_h, int32_t n,
                       const void *k_src, const void *v_src);

const char *pkv_strerror(int code);
/* The CUDA error code behind the last PKV_ECUDA on this thread (0 if none). */
int pkv_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
