/*
 * Batched paged Multi-head Latent Attention (MLA) decode -- C ABI.
 *
 * The operation (problem statement of the FlashInfer page
 * "prims_ts_batch_decode_with_kv_cache_mla", signature and parameter text):
 * for request b with KV length L = seq_lens[b] and q query rows, every query
 * row i and head h attends over the rows of a paged latent cache,
 *
 *   s_j = bmm1_scale * <Q[b,i,h,0:576], K_b[j,0:576]>
 *   O[b,i,h,:] = bmm2_scale * sum_j softmax_j(s) * K_b[j,0:512]
 *   lse[b,i,h] = ln sum_j exp(s_j)                       (natural log)
 *
 * where K_b[j] = kv_cache[block_tables[b][j / page_size]][j % page_size], the
 * 576-wide rows concatenate 512 latent and 64 RoPE dims, and V is the first
 * 512 dims of the same rows (one-copy cache).  Causal masking is bottom-right
 * aligned: row i sees KV rows 0 .. L - q + i; dense masking sees 0 .. L - 1.
 * The natural-log LSE follows the vLLM "FlashInferMLAImpl" page (its LSE
 * contract is base e); the scales are the folded bmm1/bmm2 factors of the
 * FlashInfer pull request "dynamic scale factor interface and one-copy
 * kvcache on trtllm-gen mla" (bmm1 from q/k/softmax scales, bmm2 from v/o).
 *
 * Calling sequence:  mla_decode_plan (host only; before any graph capture)
 * -> mla_decode_run (any number of times; capture-safe) -> mla_decode_destroy.
 *
 * Every tensor argument is a DEVICE pointer owned by the caller (except in
 * mla_decode_run_host, which copies a step's host-side inputs and results
 * itself).  The library allocates no device memory, performs no
 * device-to-host copy (outside mla_decode_run_host) and never synchronises
 * the stream: all per-launch metadata (seq_lens, qo_indptr,
 * block_tables) is read on the device.  Status codes are returned only for
 * what the host can check; violations of the device-side contract below are
 * undefined behaviour, except that out-of-range lengths and offsets are
 * clamped on the device so that no access leaves the given buffers, and a
 * nonzero status word is left in the workspace (mla_decode_status_offset).
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_HEAD_DIM_QK 576 /* 512 latent + 64 RoPE */
#define MLA_HEAD_DIM_V 512  /* V = first 512 dims of each cache row */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,        /* null pointer, negative size, bad enum */
  MLA_ERR_UNSUPPORTED = -2,        /* head count / page size outside the supported set */
  MLA_ERR_WORKSPACE_TOO_SMALL = -3,
  MLA_ERR_ALIGNMENT = -4,          /* a tensor pointer is not 16-byte aligned */
  MLA_ERR_CUDA = -5                /* a CUDA runtime call failed (launch, attribute) */
} mla_status;

typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype;
typedef enum { MLA_MASK_CAUSAL = 0, MLA_MASK_DENSE = 1 } mla_mask;
typedef enum { MLA_Q_BF16 = 0, MLA_Q_FP8_E4M3 = 1 } mla_q_dtype;

/*
 * Static parameters of a launch (the "semantic key" of the problem
 * statement): everything that sizes grids and the workspace.  Runtime
 * lengths live on the device and may change between launches of one plan
 * (and between replays of a captured graph) within these bounds.
 */
typedef struct mla_decode_params {
  int32_t batch;             /* B >= 0 requests */
  int32_t num_heads;         /* H in {16, 32, 64, 128} */
  int32_t max_seq_len_q;     /* fixed launch: the q_len SQ of every request;
                                packed launch: static bound on each q_len (required) */
  int32_t max_seq_len;       /* static bound on every seq_lens[b] (>= 1) */
  int32_t page_size;         /* 32 or 64 rows per page */
  int32_t max_pages_per_req; /* row stride of block_tables (>= ceil(max_seq_len / page_size)) */
  int64_t num_pages;         /* physical pages in kv_cache */
  int32_t packed;            /* 0: query [B, SQ, H, 576]; 1: query [total_q, H, 576] + qo_indptr */
  int64_t max_total_q;       /* packed: bound on total_q (query.shape[0]); fixed: ignored */
  int32_t kv_dtype;          /* mla_kv_dtype */
  int32_t mask;              /* mla_mask */
  int32_t return_lse;        /* nonzero: mla_decode_run writes lse */
  int32_t device;            /* CUDA device ordinal the plan is for */
  int32_t q_dtype;           /* mla_q_dtype: bf16, or e4m3 with the caller's q_scale
                                folded into bmm1 (bmm1 = q_scale * k_scale * softmax scale) */
  int32_t cp_world;          /* decode-context parallelism: ranks the KV sequence is
                                sharded over (0 or 1: off; > 1: run with mla_decode_run_dcp) */
  int32_t cp_rank;           /* this rank, 0 <= cp_rank < cp_world (0 when off) */
  int32_t sparse_top_k;      /* sparse top-k selection: entries k per query token of the
                                position list (0: off; > 0: run with mla_decode_run_sparse;
                                not with cp_world > 1) */
  int32_t e4m3_widen;        /* e4m3 cache only.  0: the e4m3 tiles go straight to the
                                FP8 tensor cores (kind::f8f6f4).  The query enters them
                                as e4m3: an e4m3 query as it is; a bf16 query row
                                scaled by a power of two and split into two e4m3 parts
                                whose sum is the row (exact for every element of at
                                least 2^-9 of the row's largest magnitude, within 2^-17
                                of that magnitude below).  P enters as two e4m3 parts
                                (about 2^-8 relative).  Nonzero: every e4m3 value is
                                widened exactly to bf16 before bf16 MMAs (P in bf16).
                                Sparse top-k always widens. */
} mla_decode_params;

typedef struct mla_plan_s mla_plan_t; /* opaque; host memory only */

/*
 * Validate the static parameters, query the device (SM count, shared memory)
 * and size the workspace.  Host only; not capture-safe (it sets kernel
 * attributes).  On success *plan receives a new plan (free with
 * mla_decode_destroy) and *workspace_bytes the number of bytes the caller must
 * provide to every mla_decode_run of this plan.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_CUDA.
 */
int mla_decode_plan(const mla_decode_params *params, mla_plan_t **plan,
                    size_t *workspace_bytes);

/*
 * Enqueue one decode on `stream` (a cudaStream_t; NULL = legacy default).
 *
 * query        bf16 or fp8-e4m3 (per params.q_dtype), fixed [B, SQ, H, 576] or
 *              packed [total_q, H, 576], contiguous.
 * kv_cache     bf16 or fp8-e4m3 (per params.kv_dtype), [num_pages, page_size, 576]
 *              (a rank-4 [num_pages, 1, page_size, 576] cache is the same memory).
 * block_tables int32 [B, max_pages_per_req]; entries at or past a request's
 *              ceil(seq_lens[b] / page_size) pages are never read.
 * seq_lens     int32 [B]; 1 <= seq_lens[b] <= max_seq_len; for causal masking
 *              q_len(b) <= seq_lens[b].
 * qo_indptr    packed: int32 [B + 1], qo_indptr[0] = 0, strictly increasing,
 *              qo_indptr[B] = total_q, every delta <= max_seq_len_q.
 *              fixed: must be NULL.
 * total_q      packed: query.shape[0] (<= max_total_q); fixed: ignored.
 * bmm1_scale   multiplies the 576-dim dot products (softmax scale and any
 *              q/k dequantisation scales already folded in by the caller);
 *              finite and >= 0, else MLA_ERR_INVALID_ARG.
 * bmm2_scale   multiplies the normalised output (v/o scales folded in).
 * out          bf16, [B, SQ, H, 512] or [total_q, H, 512]; required.
 * lse          fp32, [B * SQ or total_q, H]; required iff params.return_lse.
 * workspace    caller-owned device scratch of >= the planned size, 256-byte
 *              aligned, exclusive to one in-flight launch (or one captured
 *              graph) and not overlapping any other argument.  Needs no
 *              zeroing: every launch re-initialises what it uses.
 *
 * Call with params.device current (the kernels launch on the current
 * device; the plan's launch shapes belong to params.device).
 *
 * Errors (synchronous, nothing enqueued): MLA_ERR_INVALID_ARG (also: another
 * device current, a causal decode-context-parallel plan, which needs
 * mla_decode_run_dcp, or a sparse top-k plan, which needs
 * mla_decode_run_sparse), MLA_ERR_WORKSPACE_TOO_SMALL, MLA_ERR_ALIGNMENT;
 * MLA_ERR_CUDA if a launch fails.
 */
int mla_decode_run(const mla_plan_t *plan, const void *query, const void *kv_cache,
                   const int32_t *block_tables, const int32_t *seq_lens,
                   const int32_t *qo_indptr, int64_t total_q, float bmm1_scale,
                   float bmm2_scale, void *out, float *lse, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * mla_decode_run (or, with sparse_indices non-NULL on a sparse top-k plan,
 * mla_decode_run_sparse), plus two CUDA events (cudaEvent_t, may be NULL)
 * recorded on `stream` immediately before and after the decode kernel, so
 * that a caller can time that kernel alone with cudaEventElapsedTime.  Same
 * arguments, errors and capture rules as those entry points; while the stream
 * is being captured into a CUDA graph the two records become event-record
 * nodes (cudaEventRecordExternal), so every replay re-times the kernel.
 */
int mla_decode_run_profiled(const mla_plan_t *plan, const void *query, const void *kv_cache,
                            const int32_t *block_tables, const int32_t *seq_lens,
                            const int32_t *qo_indptr, int64_t total_q,
                            const int32_t *sparse_indices, float bmm1_scale, float bmm2_scale,
                            void *out, float *lse, void *workspace, size_t workspace_bytes,
                            void *stream, void *event_before_decode, void *event_after_decode);

/*
 * mla_decode_run with bmm1_scale and bmm2_scale read from device memory by
 * the kernels when they run, instead of passed by value.  This is the form a
 * captured CUDA graph needs when the scales change between replays, e.g.
 * when the caller folds per-step q/k/v quantisation scales into them (the
 * FlashInfer pull request "dynamic scale factor interface and one-copy
 * kvcache on trtllm-gen mla", its summary of the device-tensor scale
 * interface).
 *
 * bmm1_scale, bmm2_scale  device pointers to one fp32 each, 4-byte aligned,
 *              non-NULL; written by earlier work on `stream` or before the
 *              launch.  The same meaning as the by-value scales.  bmm1 must
 *              be finite and >= 0: the host cannot check it, so a violation
 *              sets status bit 64 (mla_decode_status_offset) and bmm1 reads
 *              as 0.
 * All other arguments, errors and capture rules as mla_decode_run.
 */
int mla_decode_run_device_scales(const mla_plan_t *plan, const void *query, const void *kv_cache,
                                 const int32_t *block_tables, const int32_t *seq_lens,
                                 const int32_t *qo_indptr, int64_t total_q,
                                 const float *bmm1_scale, const float *bmm2_scale, void *out,
                                 float *lse, void *workspace, size_t workspace_bytes,
                                 void *stream);

/*
 * Size of the library-owned scratch array used by
 * mla_decode_run_static_workspace (48 MiB on every GPU that loads the
 * library, held until the process exits).
 */
#define MLA_STATIC_WORKSPACE_BYTES (48u * 1024u * 1024u)

/*
 * mla_decode_run without a caller-provided workspace.  The source pages have
 * no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory when they enqueue a decode -- for example code that
 * runs while a CUDA graph is being captured (where cudaMalloc is not
 * allowed), or a plug-in inside a runtime that owns all device memory and
 * offers it no allocator.  Its scratch is a fixed array of
 * MLA_STATIC_WORKSPACE_BYTES in the library's own device memory; the call
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library call).
 *
 * Same arguments and errors as mla_decode_run, minus the workspace.  Returns
 * MLA_ERR_WORKSPACE_TOO_SMALL if the plan needs more scratch than
 * MLA_STATIC_WORKSPACE_BYTES.  The array used is the current device's, so
 * call with the plan's device current (else MLA_ERR_INVALID_ARG).  Every call
 * made outside stream capture resolves the array's device address
 * (cudaGetSymbolAddress, with that device current); a call made while its
 * stream is being captured uses the address the last uncaptured call on the
 * device resolved, so make one uncaptured call on each device before any
 * stream capture that includes this entry point (MLA_ERR_CUDA otherwise),
 * and again after a device reset.  All calls on a device share the one
 * array: calls that may overlap on the GPU race, so the caller must order
 * them (one stream, or events).  Nothing needs clearing between calls; each
 * run re-initialises what it uses.
 */
int mla_decode_run_static_workspace(const mla_plan_t *plan, const void *query,
                                    const void *kv_cache, const int32_t *block_tables,
                                    const int32_t *seq_lens, const int32_t *qo_indptr,
                                    int64_t total_q, float bmm1_scale, float bmm2_scale,
                                    void *out, float *lse, void *stream);

/*
 * Device bytes mla_decode_run_host needs for its staging buffer: the query,
 * block_tables, seq_lens, qo_indptr (packed), out and lse (return_lse) of one
 * step, each 256-byte aligned.  total_q as for mla_decode_run (packed: the
 * step's query rows, 0 <= total_q <= max_total_q; fixed: ignored).  Returns 0
 * for a NULL plan or an out-of-range packed total_q.
 */
size_t mla_decode_host_staging_bytes(const mla_plan_t *plan, int64_t total_q);

/*
 * One decode step whose per-step inputs and results live in HOST memory: the
 * query and the metadata are copied host-to-device into `staging`, the decode
 * runs as mla_decode_run, and out (and lse) are copied device-to-host, with
 * one cudaMemcpyAsync per buffer.  Everything is ordered on `stream` except
 * the query's copy, which runs on a stream the plan owns so that it overlaps
 * the partitioner: it starts after `stream`'s earlier work and the decode
 * waits for it (event fork and join, also under stream capture).  The KV
 * cache stays in device memory (the persistent state of a serving loop).
 *
 * This entry point is the exception to the device-pointers rule above: it
 * exists for callers that hold the step's query and metadata on the host.
 * The call returns once everything is enqueued; the host buffers must stay
 * valid (and h_out / h_lse unread) until the stream has passed the copies.
 * Page-locked host buffers keep the copies asynchronous; pageable ones work
 * but make the CUDA runtime stage (and partly synchronise) the copies.
 *
 * h_query, h_block_tables, h_seq_lens, h_qo_indptr, h_out, h_lse
 *              host pointers with the shapes and dtypes of mla_decode_run's
 *              query, block_tables, seq_lens, qo_indptr (packed only; NULL
 *              for a fixed launch), out and lse (return_lse only).
 * kv_cache     device pointer, as for mla_decode_run.
 * staging      caller-owned device buffer of >= mla_decode_host_staging_bytes
 *              bytes, 256-byte aligned, exclusive to this step until the
 *              stream has passed it.
 * workspace    as for mla_decode_run.
 * Errors (nothing enqueued unless stated): MLA_ERR_INVALID_ARG,
 * MLA_ERR_WORKSPACE_TOO_SMALL (staging or workspace), MLA_ERR_ALIGNMENT;
 * MLA_ERR_CUDA if a copy or launch fails (earlier copies may be enqueued).
 * Not for stream capture with pageable host buffers.
 */
int mla_decode_run_host(const mla_plan_t *plan, const void *h_query, const void *kv_cache,
                        const int32_t *h_block_tables, const int32_t *h_seq_lens,
                        const int32_t *h_qo_indptr, int64_t total_q, float bmm1_scale,
                        float bmm2_scale, void *h_out, float *h_lse, void *staging,
                        size_t staging_bytes, void *workspace, size_t workspace_bytes,
                        void *stream);

/* Free a plan (NULL is allowed). */
void mla_decode_destroy(mla_plan_t *plan);

/*
 * One rank's share of a decode under decode-context parallelism (DCP): the
 * vLLM "FlashInferMLAImpl" page (forward_mqa, its dcp_world_size > 1 branch)
 * hands the kernel enable_dcp, cp_world, cp_rank and causal_seqlens_kv_global.
 * The pages do not spell out the shard layout; this library reads it as a
 * round robin of single rows: global KV row g of a request lives on rank
 * g mod cp_world, as that rank's local row g div cp_world.  So, for request b
 * of global length Lg = causal_seqlens_kv_global[b]:
 *   seq_lens[b]      the rank's local row count, the number of g < Lg with
 *                    g mod cp_world == cp_rank (0 is allowed);
 *   block_tables     page the local rows as usual;
 *   causal masking   query row i sees the local rows j whose global position
 *                    j * cp_world + cp_rank is <= Lg - q_len + i;
 *   dense masking    sees every local row (causal_seqlens_kv_global may be NULL).
 * A query row that sees no local row gets out = 0 and lse = -inf, the empty
 * sum, which mla_merge_states ignores.  Merging every rank's (out, lse) with
 * mla_merge_states (bmm2_scale = 1 here, bmm2 there) gives the single pass
 * over the whole sequence.
 *
 * plan         made with params.cp_world > 1 and params.cp_rank.
 * causal_seqlens_kv_global
 *              device int32 [B], 1 <= Lg, q_len(b) <= Lg (causal); required
 *              for causal plans, NULL for dense ones.
 * All other arguments, errors and capture rules as mla_decode_run
 * (return_lse is what makes the result mergeable).  mla_decode_run and the
 * other run entry points refuse a causal DCP plan (MLA_ERR_INVALID_ARG).
 */
int mla_decode_run_dcp(const mla_plan_t *plan, const void *query, const void *kv_cache,
                       const int32_t *block_tables, const int32_t *seq_lens,
                       const int32_t *qo_indptr, int64_t total_q,
                       const int32_t *causal_seqlens_kv_global, float bmm1_scale,
                       float bmm2_scale, void *out, float *lse, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Sparse top-k decode.  The trtllm-gen MLA launcher in the FlashInfer issue
 * "Support cum_seq_lens_q in trtllm_batch_decode_with_kv_cache_mla" takes a
 * sparse_mla_top_k argument; the pages say no more, and this library reads it
 * as a per-token list of KV positions that replaces the mask:
 *
 * sparse_indices  device int32 [tokens, k], k = params.sparse_top_k, row t for
 *                 query token t in the query's row order (fixed: b * SQ + i;
 *                 packed: qo_indptr[b] + i).  Entries are LOGICAL positions of
 *                 the token's own request, resolved through block_tables like
 *                 any other row.  The token attends exactly the listed
 *                 positions j with 0 <= j < seq_lens[b]; any other entry
 *                 (-1 padding, a position past the request's length) is unused
 *                 and never dereferenced; a position listed twice counts twice.
 *                 The plan's mask is not consulted.  A token with no usable
 *                 entry gets out = 0 and lse = -inf.  4-byte aligned.
 *
 * Work items are one token each (its H query rows), so a token's KV tiles are
 * gathered row by row from the list.  plan: made with params.sparse_top_k > 0
 * (and cp_world <= 1).  All other arguments, errors and capture rules as
 * mla_decode_run; the other run entry points refuse a sparse plan and this
 * one refuses any other (MLA_ERR_INVALID_ARG).
 */
int mla_decode_run_sparse(const mla_plan_t *plan, const void *query, const void *kv_cache,
                          const int32_t *block_tables, const int32_t *seq_lens,
                          const int32_t *qo_indptr, int64_t total_q,
                          const int32_t *sparse_indices, float bmm1_scale, float bmm2_scale,
                          void *out, float *lse, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * Merge n partial attention states of the same query rows into one: the
 * exchange step of decode-context parallelism (DCP), where each rank runs
 * mla_decode_run over its own shard of every request's KV rows with
 * return_lse and the ranks all-gather (O, lse) (the vLLM "FlashInferMLAImpl"
 * page merges DCP shards by this natural-log LSE).  For every row r:
 *   lse[r] = ln sum_k exp(lse_k[r]),   out[r] = scale * sum_k exp(lse_k[r] - lse[r]) O_k[r]
 * which equals a single pass over the union of the shards.  A shard with no
 * visible row for r (lse_k = -inf) contributes nothing.
 *
 * o_parts    bf16 [n_parts, rows, 512], each shard's normalised output (run
 *            the shards with bmm2_scale = 1 and pass bmm2 here as `scale`)
 * lse_parts  fp32 [n_parts, rows] natural-log LSEs (mla_decode_run's lse)
 * rows       tokens * H
 * out        bf16 [rows, 512]; lse_out fp32 [rows] or NULL
 * All device pointers; o_parts and out 16-byte aligned.  Enqueued on
 * `stream`, capture-safe, allocates nothing.
 * Errors: MLA_ERR_INVALID_ARG (n_parts < 1, rows < 0 or > 2^40, n_parts * rows
 * > 9e15), MLA_ERR_ALIGNMENT, MLA_ERR_CUDA.
 */
int mla_merge_states(const void *o_parts, const float *lse_parts, int32_t n_parts, int64_t rows,
                     float scale, void *out, float *lse_out, void *stream);

/* Workspace bytes of a plan (the value mla_decode_plan returned). */
size_t mla_decode_workspace_size(const mla_plan_t *plan);

/*
 * Where a run leaves its split-KV work list in the workspace, for tests and
 * tools that check the on-device partition (decoding never needs it).  After
 * a run has completed:
 *   int32 at byte 4             number of work items
 *   items_offset                the items, 10 int32 each: request b, row group
 *                               g (rows [128 g, 128 g + 128) of the request's
 *                               q_len * H rows), KV rows [kv_begin, kv_end),
 *                               partial slot (-1: writes out directly), q_len,
 *                               seq_len, first token, combine entry (-1: none),
 *                               causal mask base
 *   worker_ranges_offset        int32[n_workers + 1]: persistent worker w (a CTA
 *                               pair) runs items [r[w], r[w + 1])
 * Errors: MLA_ERR_INVALID_ARG on a NULL argument.
 */
int mla_decode_work_list_layout(const mla_plan_t *plan, size_t *items_offset,
                                size_t *worker_ranges_offset, int32_t *n_workers);

/*
 * Number of kernels one run of `plan` launches on the caller's stream (a
 * plan property; batch 0 launches none): the partitioner, the decode kernel
 * and the combine kernel, plus, on the FP8 MMA path with a bf16 query (an
 * e4m3 cache, no sparse top-k, e4m3_widen 0), the query split that precedes
 * the decode.  Returns -1 for a NULL plan.
 */
int32_t mla_decode_kernels_per_run(const mla_plan_t *plan);

/*
 * Byte offset, inside the workspace, of the int32 device status word the last
 * run left behind.  0: every device-side value was within the contract.
 * Bits (values are clamped and never read out of bounds):
 *   1  a seq_len out of [1, max_seq_len]
 *   2  a q_len out of [1, max_seq_len_q], or a qo_indptr offset out of range
 *   4  causal masking with q_len > seq_len
 *   8  a workspace capacity exceeded (unreachable within the contract)
 *  16  a block_tables entry of a visible page out of [0, num_pages)
 *  32  an internal wait timed out (the run unwound; results are invalid)
 *  64  a device bmm1 scale negative or not finite (read as 0)
 * Reading it is the caller's choice (a device-to-host copy after the stream
 * syncs).
 */
size_t mla_decode_status_offset(void);

/* Human-readable name of a status code. */
const char *mla_decode_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
