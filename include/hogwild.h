/*
 * hogwild.h -- C ABI of the GB300 concurrent-attention library (libhogwild.so).
 *
 * The method is Hogwild! Inference ("Parallel LLM Generation via Concurrent Attention";
 * summary at gentlecold.top, cited below by section).  W workers decode in parallel and share
 * one KV cache made of blocks: a common block (prompt and finished paragraphs) and one
 * current block per worker (section 6; section 9 "the Hogwild! cache is split into blocks").
 * Every block stores K/V of all layers at block-local positions 0 .. len-1 (section 9).  Worker
 * w attends over the common history, then the other workers' current blocks, then its own
 * block last (sections 4 and 6); instead of re-rotating stored keys, the query is rotated once
 * per block by (query position - the block's offset in w's view) (section 5, the identity
 * rho(q,i_q)[rho(A,i_A) (+) ...] = [rho(q,i_q - i_A) A (+) ...]).  A step appends each worker's
 * new token, attends, and at the end of a paragraph moves the worker's block to the end of the
 * common history (section 8, inference flow).
 *
 * Conventions shared by every call
 * --------------------------------
 * - P problems, W workers, L layers, H_q query heads, H_kv KV heads (G = H_q / H_kv; query head
 *   h reads KV head h / G), head dimension D in {64, 128}, page size S (a multiple of 128).
 * - All tensors are dense, row-major, and bf16 unless stated otherwise.
 * - "device" pointers are CUDA device memory of the current device; "host" pointers are CPU
 *   memory.  The caller owns every buffer: the library never allocates device memory (its
 *   tables live inside the caller's workspace), it only creates host-side state, pinned
 *   staging buffers, events and one TMA descriptor per layer.
 * - ``stream`` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All work
 *   is enqueued asynchronously on it.  A context is not thread-safe: use one host thread at a
 *   time per context.
 * - RoPE: half-split pairs (x_i, x_{i+D/2}) rotated by p * theta^(-2i/D).  The cos/sin table
 *   is computed on the host in fp64 and stored as fp32.
 * - Errors: arguments are validated on the host before anything is enqueued; on an error
 *   nothing is enqueued and the state is unchanged.  Kernels never trap: an index that fails a
 *   device-side range check is skipped and recorded in a device error word that
 *   hw_check_device_errors() reads back.
 */
#ifndef HOGWILD_H_
#define HOGWILD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum hw_status {
  HW_OK = 0,
  HW_ERR_INVALID_ARG = 1,     /* null pointer, bad size or shape, protocol misuse */
  HW_ERR_OUT_OF_PAGES = 2,    /* the page pool cannot hold this append */
  HW_ERR_CAPACITY = 3,        /* a table (segments, positions, workspace) would overflow */
  HW_ERR_CUDA = 4,            /* a CUDA runtime call failed (see hw_last_cuda_error) */
  HW_ERR_DEVICE_CHECK = 5,    /* a kernel's range check fired (hw_check_device_errors) */
  HW_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device wait gave up (hw_check_device_errors) */
  HW_ERR_UNSUPPORTED = 7      /* shape or device this build does not handle */
} hw_status;

enum { HW_OUT_BF16 = 0, HW_OUT_F32 = 1 };

/*
 * Cache layouts (summary section 6 compares the first three; section 10 adds the no-sync
 * setting): which blocks a worker's view holds, and in what order.  Blocks, commits and pages
 * are the same in every layout; only the views -- and so the query rotations -- differ.
 */
enum {
  HW_LAYOUT_COMBINED = 0,   /* token-wise (the main method): common history in commit order,
                               the other workers' current blocks in ascending id, own block */
  HW_LAYOUT_STEP_WISE = 1,  /* interleaved: common history, own block; the other workers'
                               unfinished blocks are not visible */
  HW_LAYOUT_CONTIGUOUS = 2, /* each worker's output is one run: the prompt, every other
                               worker's committed paragraphs then current block (ascending id),
                               then the worker's own paragraphs and block */
  HW_LAYOUT_NO_SYNC = 3     /* independent workers: the prompt, own committed paragraphs, own
                               block */
};

typedef struct hw_config {
  int32_t num_problems;      /* P >= 1 independent Hogwild! problems */
  int32_t num_workers;       /* W >= 1 workers per problem */
  int32_t num_layers;        /* L >= 1; each layer has its own pages in the pools */
  int32_t num_q_heads;       /* H_q, a multiple of H_kv */
  int32_t num_kv_heads;      /* H_kv >= 1 */
  int32_t head_dim;          /* D: 64 or 128 */
  int32_t page_size;         /* S: tokens per page, a multiple of 128 */
  int32_t contiguous;        /* 0: paged blocks; 1: each block is one page of S tokens */
  int32_t num_pages;         /* pages per layer */
  int32_t max_position;      /* exceeds every view length; rows of the RoPE table */
  int32_t max_segments;      /* segment capacity over all problems (0: P * (1 + 4W)) */
  int32_t max_append_tokens; /* largest sum of n_new in one append (0: num_pages * S) */
  double rope_theta;         /* RoPE base */
  int32_t layout;            /* HW_LAYOUT_* (0: combined).  In the contiguous and no-sync
                                layouts a committed paragraph belongs to the worker that wrote
                                it, and tokens appended to the last common segment belong to
                                that segment's writer (the prompt's when nothing is committed) */
  int32_t reserved;          /* 0 */
} hw_config;

typedef struct hw_ctx hw_ctx;

/* Human-readable name of a status code (static storage). */
const char* hw_status_string(hw_status s);

/* Last CUDA error code and message seen by a call that returned HW_ERR_CUDA (per process). */
int32_t hw_last_cuda_error(const char** message);

/*
 * Bytes of ONE pool (the K pool or the V pool) for cfg: L * num_pages * H_kv * S * D bf16.
 * Layout of a pool: [L][num_pages][H_kv][S][D]; a page holds S consecutive block-local
 * positions of one block, for every KV head (section 9: blocks hold every layer's K/V).
 */
hw_status hw_pool_size(const hw_config* cfg, size_t* bytes);

/* Bytes of device workspace hw_create() needs for cfg (tables, RoPE table, partials). */
hw_status hw_workspace_size(const hw_config* cfg, size_t* bytes);

/*
 * Create a context over caller-owned device buffers.
 *   k_pool, v_pool: device, hw_pool_size() bytes each, 256-byte aligned; zero-filled here.
 *   workspace:      device, >= hw_workspace_size() bytes, 256-byte aligned.
 *   page_order:     host int32[num_pages] (a permutation of 0..num_pages-1) giving the order
 *                   in which physical pages are handed out, or NULL for 0, 1, 2, ...
 * Each problem starts with an empty common block and W empty worker blocks (segment ids:
 * per problem, the common block then workers 0..W-1).  Blocks until the set-up copies are
 * done.  *out receives the handle; release it with hw_destroy().
 */
hw_status hw_create(const hw_config* cfg, void* k_pool, void* v_pool, void* workspace,
                    size_t workspace_bytes, const int32_t* page_order, void* stream,
                    hw_ctx** out);

/* Release the host-side state (never the caller's device buffers).  NULL is a no-op. */
void hw_destroy(hw_ctx* ctx);

/*
 * Append new tokens' K/V of one layer (section 8: each worker appends its token's K/V to its
 * own block before attention; section 9: block-local positions).
 *   n_new: host int32[P][W + 1]; n_new[p][0] tokens go to problem p's common block (the last
 *          common segment), n_new[p][1 + w] to worker w's current block.
 *   k_raw, v_raw: device bf16 [sum n_new][H_kv][D], UNROTATED keys and values, ordered
 *          problem-major, then block 0 (common), 1..W, each in position order; 16-byte
 *          aligned.  They may be read later than this call (see "When the write happens").
 * Key token j of a block is stored as bf16(rho(k, j)) at (page_of(j), j mod S); values are
 * copied.  The first append of a step allocates pages (FIFO from page_order; problems in
 * order, then the common block, then workers in ascending id; a new page whenever j mod S == 0;
 * in contiguous mode one page at j == 0).  Every layer must append once per step with the same
 * n_new.  Attention in the step sees the appended tokens; lengths advance at hw_step_end().
 * When the write happens: with at most 16 tokens per block in the step (decode), this call
 * only records k_raw / v_raw and the layer's hw_concurrent_attention writes the tokens itself,
 * inside its kernel (either attention kernel), before it reads them; if the step ends without that call, hw_step_end writes them.  Otherwise an append
 * kernel is enqueued here.  Either way k_raw and v_raw must keep their contents, in stream
 * order, until the layer's attention call or hw_step_end, whichever comes first.
 * Errors: HW_ERR_INVALID_ARG (bad layer, counts differing from the step's first append, layer
 * appended twice, unaligned k_raw / v_raw), HW_ERR_OUT_OF_PAGES, HW_ERR_CAPACITY (contiguous
 * block full).
 */
hw_status hw_append_kv(hw_ctx* ctx, int32_t layer, const int32_t* n_new, const void* k_raw,
                       const void* v_raw, void* stream);

/*
 * Concurrent attention of one layer (sections 5 and 9).
 *   q:   device bf16 [P][W][H_q][D], UNROTATED queries (one token per worker), 16-byte aligned.
 *   out: device [P][W][H_q][D], bf16 (out_dtype HW_OUT_BF16) or fp32 (HW_OUT_F32), 16-byte
 *        aligned.
 *   lse: device fp32 [P][W][H_q] or NULL: natural-log log-sum-exp of the scaled scores.
 * For worker w of problem p the view is [common segments in commit order] ++ [other workers'
 * blocks, ascending id] ++ [own block]; empty blocks are skipped; i_q = view length - 1.  Each
 * block at view offset o is attended with the query rotated by (i_q - o), scores scaled by
 * 1/sqrt(D), and the per-block softmax partials merged by log-sum-exp.  An empty view gives
 * out = 0 and lse = -inf.  Requires that, if the current step appended tokens, this layer
 * has been appended, and q and out aligned (HW_ERR_INVALID_ARG otherwise).  Scratch: partial
 * results live in the workspace; calls on one context must not overlap on the GPU (use one
 * stream).
 */
hw_status hw_concurrent_attention(hw_ctx* ctx, int32_t layer, const void* q, void* out,
                                  int32_t out_dtype, float* lse, void* stream);

/*
 * Several query tokens per worker, attending causally (summary section 8, step 4: after a
 * commit the worker's new block starts with a paragraph header of several tokens, whose
 * forward pass needs them all; likewise any chunk of tokens a worker appends in one step).
 * Worker w's queries are the last n_q[p][w] tokens of its own block (appended before this call,
 * in this step or earlier), in order.  Query token t sits at view position
 * i_q(w) - (n_q[p][w] - 1 - t) and attends to every token of w's view up to and including its
 * own position: the whole view but the own block, which is last in every layout, and the own
 * block's tokens up to its own.  With n_q = 1 for every worker this is hw_concurrent_attention.
 *   q:     device bf16 [N][H_q][D], N = sum of n_q, rows in order problem, worker, token;
 *          16-byte aligned.  Unrotated, as for hw_concurrent_attention.
 *   n_q:   host int32 [P][W], 0 <= n_q[p][w] <= the worker's own block length (this step's
 *          appended tokens included).
 *   out:   device [N][H_q][D], bf16 or fp32 (out_dtype); lse: device fp32 [N][H_q] or NULL.
 * A problem's query rows, (sum_w n_q[p][w]) * H_q / H_kv, are attended 128 at a time: when
 * they exceed one 128-row tile, each problem's query tokens (workers in order, each worker's
 * tokens in order) are cut into parts of at most 128 rows -- a worker's tokens may straddle
 * parts, each keeping its causal offset -- and part k of every problem goes into the k-th of
 * several attention launches (the K/V are streamed once per launch; every token keeps its row
 * of q / out / lse).  N = 0 enqueues nothing.  The layer's recorded append (hw_append_kv) is
 * written first, by the append kernel.
 * Errors: as hw_concurrent_attention; HW_ERR_INVALID_ARG for a NULL n_q or a count out of
 * range.  An error from a later launch of a split call leaves the earlier launches' rows
 * written.
 */
hw_status hw_concurrent_attention_mq(hw_ctx* ctx, int32_t layer, const void* q,
                                     const int32_t* n_q, void* out, int32_t out_dtype, float* lse,
                                     void* stream);

/*
 * Concurrent attention over a range of KV entries, for splitting one step's attention into
 * parts (summary section 9: the work is split over KV entries and the partial results are
 * reduced afterwards) -- on one GPU, or across GPUs that each take a range and exchange their
 * results.  A problem's entries are numbered in segment order: its common segments in commit
 * order, then the workers' current blocks in ascending worker id (entry e of a segment with
 * first number f is its block-local token e - f).  Every view holds whole segments of that
 * list in its own order, so the numbering is the same for every worker.
 *   q:      as hw_concurrent_attention.
 *   ranges: host int64 [P][2]: problem p's entries [ranges[p][0], ranges[p][1]); 0 <= begin <=
 *           end (an end past the last entry stops there).
 *   out:    device fp32 [P][W][H_q][D], 16-byte aligned: each worker's softmax attention over
 *           the selected entries of its view, each key still at its position in the worker's
 *           view (the query rotation is the full call's), normalised over those keys.
 *   lse:    device fp32 [P][W][H_q] (required): natural-log log-sum-exp of the selected
 *           scaled scores; -inf (and out = 0) where a worker selects nothing.
 * Merging, with hw_merge_attention, the results of ranges that partition every problem's
 * entries gives hw_concurrent_attention's out and lse.  The layer's recorded append is
 * written first, by the append kernel.  Errors: as hw_concurrent_attention; HW_ERR_INVALID_ARG
 * for a NULL ranges or lse, or a range with begin < 0 or end < begin.
 */
hw_status hw_concurrent_attention_range(hw_ctx* ctx, int32_t layer, const void* q,
                                        const int64_t* ranges, float* out, float* lse,
                                        void* stream);

/*
 * Merge of n partial attention results of the same query rows over disjoint sets of keys
 * (summary section 9, "partial result reduction"; section 5: by log-sum-exp):
 *   LSE = log sum_i exp(lse_i),   out = sum_i exp(lse_i - LSE) out_i,
 * parts with lse_i = -inf count as empty; out = 0 and LSE = -inf when every part is.  Needs no
 * context: the parts may come from hw_concurrent_attention_range calls on this GPU, or be
 * gathered from GPUs that attended to other ranges.
 *   n_parts: 1 .. 4096.  rows: query rows per part (P * W * H_q for one query per worker).
 *   head_dim: D, a multiple of 4.
 *   parts_out: device fp32 [n_parts][rows][D], 16-byte aligned; parts_lse: device fp32
 *   [n_parts][rows].  out: device [rows][D], bf16 or fp32 (out_dtype), 16-byte aligned; lse:
 *   device fp32 [rows] or NULL.  One kernel on `stream`.
 * Errors: HW_ERR_INVALID_ARG (counts, NULL or misaligned pointers), HW_ERR_CUDA.
 */
hw_status hw_merge_attention(int32_t n_parts, int64_t rows, int32_t head_dim,
                             const float* parts_out, const float* parts_lse, void* out,
                             int32_t out_dtype, float* lse, void* stream);

/*
 * hw_concurrent_attention for callers that cannot allocate device memory when they call it
 * (no counterpart in the paper; a deployment need).  Same arguments, same result as
 * hw_concurrent_attention; the context's pools, tables and RoPE table are used as usual, but
 * the call's plan and its split-K partial results live in a fixed 16 MiB array in device global
 * memory that the library defines, instead of in the workspace.  Nothing is allocated: no
 * cudaMalloc, cudaFree or allocating library routine is called.
 *   - Speed: it always runs the CUDA-core attention kernel and a separate merge kernel, also
 *     on contexts whose regular call uses the tensor cores (16 or more query rows per KV
 *     head), so it is several times slower there; the regular call remains the fast path.
 *   - Limit: the plan plus one partial result per (problem, KV head) group, i.e.
 *     P * H_kv * rows * (D + 4) * 4 bytes with rows = W * H_q / H_kv, must fit in 16 MiB, else
 *     HW_ERR_CAPACITY and nothing is enqueued.  The KV split adapts to the space left.
 *   - Not on a capturing stream: a call on a stream that is capturing a CUDA graph returns
 *     HW_ERR_UNSUPPORTED with nothing enqueued (the plan is copied from a host staging slot
 *     that later calls reuse).  A capture on another stream is no obstacle.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current).
 *   - Every call, from every context, shares the one array, which keeps the last call's
 *     contents; nothing in it needs to start at zero (each call writes its plan and every
 *     partial before reading them).  Calls whose GPU work overlaps -- on different streams,
 *     or from different contexts -- race on the array: order them on one stream.
 *   - A recorded append of the layer (hw_append_kv) is written first, by the append kernel,
 *     once the call's plan has been checked; on HW_ERR_CAPACITY nothing is enqueued.
 */
hw_status hw_concurrent_attention_noalloc(hw_ctx* ctx, int32_t layer, const void* q, void* out,
                                          int32_t out_dtype, float* lse, void* stream);

/*
 * End the step (section 8): every block's length grows by the tokens appended in this step;
 * then, for each problem and each worker in ascending id with finished[p][w] != 0 and a
 * non-empty block, the worker's block is moved, unchanged, to the end of the common history
 * and the worker starts a new empty block (new segment id).  No K/V byte moves and nothing is
 * re-rotated: the new view offset is absorbed by the query rotation.
 *   finished: host uint8[P][W] or NULL (no commits).
 * Errors: HW_ERR_INVALID_ARG if the step appended some but not all layers; HW_ERR_CAPACITY
 * if the segment table is full.  Enqueues on `stream` only the writes of appended tokens that
 * no attention call of the step has written (see hw_append_kv); nothing otherwise.
 */
hw_status hw_step_end(hw_ctx* ctx, const uint8_t* finished, void* stream);

/*
 * One whole decode step from host memory (section 8's inference flow: every worker appends its
 * token, attends to the shared cache, and the step ends with the commits), for callers whose
 * inputs and outputs are in host memory.  Every layer's K, V and queries go to the device in
 * one host-to-device copy and every layer's output comes back in one device-to-host copy;
 * in between, hw_append_kv for every layer, hw_concurrent_attention for every layer and
 * hw_step_end, all on `stream` -- the step's attention plan too, copied in stream order
 * (the separate calls send it on the library's copy stream, where the kernels check for it).
 *   n_new:    host int32[P][W + 1], as hw_append_kv (the same counts for every layer).
 *   in_host:  host, packed [K][V][Q]: K and V bf16 [L][sum n_new][H_kv][D] each (layer-major;
 *             within a layer as hw_append_kv's k_raw / v_raw), then Q bf16 [L][P][W][H_q][D]
 *             (unrotated, as hw_concurrent_attention's q).
 *   in_bytes: must equal 2 * L * D * (2 * sum(n_new) * H_kv + P * W * H_q).
 *   out_host: host, [L][P][W][H_q][D] of out_dtype (HW_OUT_BF16 or HW_OUT_F32).
 *   finished: host uint8[P][W] or NULL, as hw_step_end.
 *   scratch:  device, >= hw_step_scratch_size() bytes, 256-byte aligned, caller-owned: the
 *             device copies of the inputs and outputs.  Not to be shared with GPU work that
 *             may overlap the step.
 *   sync:     nonzero: return once the step's GPU work and the output copy have completed
 *             (cudaStreamSynchronize); zero: return after enqueueing, and in_host, out_host
 *             and scratch must then stay untouched until the stream has passed the step.
 * Host buffers should be page-locked (cudaHostAlloc or cudaHostRegister) for the copies to be
 * asynchronous.  Between steps only (HW_ERR_INVALID_ARG if a step is open).
 * Errors: HW_ERR_INVALID_ARG (NULL pointer, bad out_dtype, a negative count, in_bytes not as
 * above, unaligned scratch, a step open) and HW_ERR_CAPACITY (scratch too small) with nothing
 * enqueued; otherwise those of hw_append_kv (the first append's errors leave no open step; the
 * input copy into scratch is already enqueued then, nothing else), hw_concurrent_attention
 * (every layer is appended by then: hw_step_end can close the step) and hw_step_end.
 */
hw_status hw_decode_step_host(hw_ctx* ctx, const int32_t* n_new, const void* in_host,
                              size_t in_bytes, void* out_host, int32_t out_dtype,
                              const uint8_t* finished, void* scratch, size_t scratch_bytes,
                              int32_t sync, void* stream);

/* Device scratch bytes hw_decode_step_host needs for the counts n_new (host int32[P][W + 1])
 * and the output type.  Errors: HW_ERR_INVALID_ARG (NULL, bad out_dtype, a negative count). */
hw_status hw_step_scratch_size(const hw_ctx* ctx, const int32_t* n_new, int32_t out_dtype,
                               size_t* bytes);

/*
 * Compaction (summary section 8: a finished block moves to the end of the common history and
 * is "corrected by RoPE offset" -- reading 1 of that correction; hw_step_end does reading 2,
 * an index remap): problem p's common segments first .. first+count-1 (commit order; 0 is
 * the prompt) merge into one segment with one RoPE frame.  Each key is re-rotated from its
 * block-local position j to its position in the merge (j plus the segment's offset in it) and,
 * with its value, copied into fresh pages taken FIFO from the free list; the old pages then
 * return to the end of the free list (segment by segment in commit order, each in page order)
 * and the old segments stay in the table, empty.  Views and attention results do not change
 * (up to the extra bf16 rounding of the re-rotated keys); the segment count and the partial
 * tiles at segment ends go down.  The merged segment's writer (origin) is the segments'
 * common writer, or -1 when they differ.
 *   Between steps only (no hw_append_kv since the last hw_step_end); count >= 2.  Enqueues
 *   one kernel on `stream`, in stream order after every earlier call of the context.
 * Errors: HW_ERR_INVALID_ARG (range, during a step, or writers that differ in the contiguous
 * or no-sync layout, whose views depend on the writer); HW_ERR_OUT_OF_PAGES (nothing changes);
 * HW_ERR_CAPACITY (segment table full, or a contiguous block's capacity).
 */
hw_status hw_compact_segments(hw_ctx* ctx, int32_t problem, int32_t first, int32_t count,
                              void* stream);

/*
 * A compaction policy over hw_compact_segments, between steps: every problem with more than
 * max_paragraphs committed paragraphs (common segments after the prompt) has them merged --
 * in the combined and step-wise layouts all of them into one segment after the prompt; in the
 * contiguous and no-sync layouts, whose views depend on the writer, each run of consecutive
 * paragraphs of one writer.  The prompt is never re-rotated.  Each merge re-rotates and copies
 * the merged tokens of every layer (one kernel), so a larger max_paragraphs compacts less
 * often.  merged (host, or NULL) receives the number of merges enqueued.
 * Errors: HW_ERR_INVALID_ARG (during a step, max_paragraphs < 1), else those of
 * hw_compact_segments; the merges before a failing one stand.
 */
hw_status hw_compact_auto(hw_ctx* ctx, int32_t max_paragraphs, void* stream, int32_t* merged);

/*
 * Synchronise ``stream`` and read the device error word.  Returns HW_OK, or
 * HW_ERR_DEVICE_CHECK / HW_ERR_DEVICE_TIMEOUT if a kernel recorded one (the word is then
 * cleared).  info: host uint32[4] or NULL: {code, kernel id, detail a, detail b}.
 */
hw_status hw_check_device_errors(hw_ctx* ctx, void* stream, uint32_t* info);

/*
 * Fault injection on the host, for tests of the error path: the next `count` plans this
 * context uploads (a step's plan goes up with its first hw_append_kv; an attention call
 * outside a step uploads its own) are announced to the kernels with a sequence number that
 * never arrives.  Every kernel gated on such a plan gives up after its bounded wait (about one
 * second), skips its work, writes empty partials and records a timeout, so that the next
 * hw_check_device_errors returns HW_ERR_DEVICE_TIMEOUT.  Outputs of the affected calls are
 * zero (tensor-core and CUDA-core attention alike), and tokens whose append such a call
 * carried are not written; the host tables are unaffected and the context stays usable.
 * count = 0 cancels what is left.  Errors: HW_ERR_INVALID_ARG (null context, count < 0).
 */
hw_status hw_debug_expire_plans(hw_ctx* ctx, int32_t count);

/* ---- measurement ------------------------------------------------------------------------ */

typedef struct hw_profile {
  int64_t launches;          /* kernels this context launched since the last read */
  int64_t attention_launches;
  int64_t append_launches;
  double attention_ms;       /* summed CUDA-event time of the attention kernels (enabled only) */
  double append_ms;          /* summed CUDA-event time of the append kernels (enabled only) */
  int64_t timed_attention;   /* how many attention launches attention_ms covers */
  int64_t timed_append;
  double merge_ms;           /* summed CUDA-event time of the merge kernels (enabled only) */
  int64_t timed_merge;
} hw_profile;

/*
 * Turn kernel timing on or off.  When on, every attention and append call records a pair of
 * CUDA events on its stream directly around each of its kernels -- the attention kernel, the
 * merge kernel, the append kernel -- (up to 4096 pairs per read); the kernels are then launched
 * without programmatic chaining.  Launch counting is always on.
 */
hw_status hw_profile_enable(hw_ctx* ctx, int32_t enable);

/* Synchronise the recorded events, sum their elapsed times, fill *out and reset. */
hw_status hw_profile_read(hw_ctx* ctx, hw_profile* out);

/* ---- read-back of the host tables (tests; bit-exact comparison with the oracle) ---------- */

/* Number of segments created so far and pages still free. */
hw_status hw_get_counts(const hw_ctx* ctx, int32_t* num_segments, int32_t* free_pages);

/* One segment: problem, origin worker (-1 for the prompt), committed length, tokens pending
 * in the current step, and its physical pages (pages_out: host int32[pages_cap]). */
hw_status hw_get_segment(const hw_ctx* ctx, int32_t seg, int32_t* problem, int32_t* origin,
                         int32_t* length, int32_t* pending, int32_t* num_pages,
                         int32_t* pages_out, int32_t pages_cap);

/* Problem p's common segment ids in commit order (host int32[cap]) and the W current-block
 * segment ids (host int32[W]). */
hw_status hw_get_blocks(const hw_ctx* ctx, int32_t problem, int32_t* common_ids, int32_t cap,
                        int32_t* num_common, int32_t* live_ids);

/* Worker w's view as the attention call will see it: segment ids, view offsets and visible
 * lengths (host int32[cap] each), the entry count and i_q. */
hw_status hw_get_view(const hw_ctx* ctx, int32_t problem, int32_t worker, int32_t* seg_ids,
                      int32_t* view_offsets, int32_t* lengths, int32_t cap, int32_t* n,
                      int32_t* i_q);

#ifdef __cplusplus
}
#endif

#endif /* HOGWILD_H_ */
