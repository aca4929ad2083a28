/*
 * pkv: batched GQA attention over a paged bf16 KV cache, for GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only.  Device pointers are CUDA device
 * addresses on the current device; host pointers are ordinary process memory.
 * The caller owns every device buffer (q, k/v, out, lse, the KV layer slice, the
 * workspace).  The library allocates no device memory; it owns the opaque handle
 * and the handle's page-locked host staging ring.
 *
 * Cache layout (mstar.engine.resources.attn.wrappers, module docstring): the full
 * cache is [num_layers, max_pages, 2, page_size, num_kv_heads, head_dim] bf16; every
 * call here takes ONE layer slice [max_pages, 2, page_size, num_kv_heads, head_dim]
 * (index 0 of the "2" axis = K, 1 = V), contiguous, 16-byte aligned.
 *
 * Index arrays (mstar.engine.resources.kv.plan, PagedIndptrs): int32
 *   qo_indptr[batch+1]      new-token offsets of each row into q / out
 *   paged_kv_indptr[batch+1] page offsets of each row into paged_kv_indices
 *   paged_kv_indices[nnz]   page ids, in position order within a row
 *   paged_kv_last_page_len[batch] slots filled in each row's last page, 1..page_size
 * They describe the cache AFTER this step's append (the layer writes its K/V before
 * attention runs: DenseAttentionManager.requires_kv_write), so row r holds
 *   L_r = (pages_r - 1) * page_size + last_page_len[r] tokens, of which the last
 *   n_r = qo_indptr[r+1] - qo_indptr[r] are this step's new tokens.
 *
 * Attention (the softmax definition the wrappers compute): new token i of row r sits
 * at position p = L_r - n_r + i; q head h reads kv head h / (num_qo_heads/num_kv_heads);
 * it sees keys j with lo <= j <= p (causal) or lo <= j <= L_r - 1 (non-causal), where
 * lo = max(0, p - window_left) if window_left >= 0, else 0 (FlashInferPrefillWrapper.plan:
 * window_left is the number of preceding positions a query sees, -1 unbounded);
 *   out = softmax(sm_scale * q K^T) V (bf16), lse = natural-log log-sum-exp (fp32).
 *
 * Call order for one step:  pkv_plan (host)  ->  per layer: pkv_kv_append (or
 * pkv_kv_append_planned), then pkv_run_decode / pkv_run_prefill / pkv_run_mixed.  One
 * plan serves every layer until the next plan on that workspace (DensePlan: "once per
 * step and read by each layer run").  run and append calls allocate nothing and never
 * synchronise the host.  A plan reaches its workspace through a copy queued on the
 * plan's stream, so the runs and appends that read it must be queued on that stream, or
 * on one ordered after it (an event); the next plan on the same workspace overwrites it
 * in stream order, so plans may run ahead of the GPU on one stream.
 *
 * Errors: every function returns a pkv_status; validation happens on the host before
 * any launch; pkv_last_error() explains the last failure.  Kernels never trap: a
 * device-side wait that exceeds its iteration limit records an error word in the
 * workspace, which pkv_check_device_error() reads.
 *
 * Threading: one handle per issuing thread.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_handle_s *pkv_handle_t;
typedef void *pkv_stream_t; /* a cudaStream_t; NULL = the legacy default stream */

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,               /* malformed arguments or index arrays */
    PKV_ERR_UNSUPPORTED = 2,           /* a shape this build's kernels do not compute */
    PKV_ERR_WORKSPACE = 3,             /* workspace too small: pkv_last_error names the bytes */
    PKV_ERR_TOO_MANY_PREFILL_ROWS = 4, /* mixed plan with more prompt rows than max_prefill_rows */
    PKV_ERR_NOT_PLANNED = 5,           /* run/append without a matching plan on that workspace */
    PKV_ERR_CUDA = 6,                  /* a CUDA runtime/driver call failed */
    PKV_ERR_DEVICE = 7                 /* a kernel recorded a device-side error (wait limit hit) */
} pkv_status;

enum { PKV_MODE_DECODE = 0, PKV_MODE_PREFILL = 1, PKV_MODE_MIXED = 2, PKV_MODE_DENSE = 3 };
enum { PKV_NON_CAUSAL = 0, PKV_CAUSAL = 1, PKV_CONTEXT_ONLY = 2 };

/*
 * Static configuration, fixed for the life of a handle (the wrappers' constructor
 * arguments: FlashInferDecodeWrapper / FlashInferPrefillWrapper / FlashInferMixedWrapper).
 *   num_qo_heads, num_kv_heads, head_dim, page_size: shape of q and of the cache.
 *   max_batch:        most rows a plan may have.
 *   max_total_tokens: most new tokens a plan may have (prefill and mixed).
 *   max_num_pages:    most entries paged_kv_indices may have.
 *   num_cache_pages:  pages in one layer slice (its first dimension); every page id
 *                     must be below it.
 *   max_prefill_rows: mixed only: most prompt rows (rows with >= 2 new tokens).
 *   sm_count:         SMs the work split targets; 0 = query the current device.
 *   sink_page:        mixed only: a caller-reserved page id holding finite values,
 *                     read (one token) by every non-decode row of the decode pass;
 *                     -1 when no mixed plans are made.
 *   graph_static:     1 = CUDA-graph mode (the wrappers' accelerator_graph): every plan
 *                     uses the workspace layout of the handle's maxima and every kernel is
 *                     launched at the maxima, reading the plan's own counts, causal flag,
 *                     window and scale from the workspace.  pkv_kv_append_planned /
 *                     pkv_run_* calls captured once into a CUDA graph then stay valid for
 *                     every later
 *                     pkv_plan on the same workspace, as long as q, out, lse, k, v and the
 *                     layer slices keep their addresses and q / out / k / v are sized for
 *                     the maxima (max_batch rows for decode, max_total_tokens otherwise).
 *                     Make one uncaptured call of each kind first (it sets kernel
 *                     attributes).  0 = launches sized to each plan.
 *   enable_nvtx:      1 = every call on this handle opens an NVTX range named after it
 *                     ("pkv_plan", "pkv_kv_append", "pkv_run_decode", ...) for its
 *                     host-side duration, so a profiler's timeline shows the plan,
 *                     append and run spans of a step (the wrappers' enable_nvtx).  With
 *                     no profiler attached the ranges cost nothing.  0 = no ranges.
 */
typedef struct {
    int num_qo_heads;
    int num_kv_heads;
    int head_dim;
    int page_size;
    int max_batch;
    int max_total_tokens;
    int max_num_pages;
    int num_cache_pages;
    int max_prefill_rows;
    int sm_count;
    int sink_page;
    int graph_static;
    int enable_nvtx;
} pkv_config;

/*
 * Create a handle.  Host-only apart from the device query when sm_count == 0.
 * Returns PKV_ERR_UNSUPPORTED unless head_dim is 64, 128 or 256, page_size is a power
 * of two from 1 to 1024, num_qo_heads is a multiple of num_kv_heads with a group size
 * g of 1..8 or 16, and num_kv_heads <= 256 (check_flashinfer_head_dim: the pages'
 * kernels likewise reject a head_dim they do not compute exactly).  PKV_ERR_INVALID on
 * non-positive sizes.
 * *out is set only on PKV_OK.
 */
pkv_status pkv_create(const pkv_config *cfg, pkv_handle_t *out);

/* Release the handle and its pinned staging (waits for that staging's copies). */
void pkv_destroy(pkv_handle_t h);

/* Message for the last failure on this handle (never NULL; "" when none).  With
 * h == NULL, the message of the last failed pkv_create on this thread. */
const char *pkv_last_error(pkv_handle_t h);

/*
 * Bytes of device workspace a plan of `mode` needs at the handle's static maxima
 * (the worst case: mstar.engine.resources.attn.workspace, Workspace: what a plan
 * needs depends on rows, segments, heads and the SM count).  Host-only.
 */
pkv_status pkv_workspace_size(pkv_handle_t h, int mode, size_t *bytes);

/*
 * Plan a step (FlashInferDecodeWrapper.plan / FlashInferPrefillWrapper.plan /
 * FlashInferMixedWrapper.plan).  All index arrays are HOST int32 pointers (the pages
 * prefer CPU inputs so planning never waits on the device).  The planner validates
 * them, derives the KV write locations, splits the attention into work tiles sized to
 * the SM count (split-KV partials live in the workspace), for mode MIXED classifies
 * rows and builds the prompt-token permutation and the sink routing, stages the plan
 * in page-locked memory and copies it into `workspace` with one async H2D on `stream`.
 *   mode          PKV_MODE_DECODE: qo_indptr may be NULL (row r's query is token r);
 *                 PKV_MODE_PREFILL / PKV_MODE_MIXED: qo_indptr required.
 *   causal        prefill and mixed (the prefill pass); decode is always "sees its row".
 *                 0 non-causal, 1 causal, 2 (PKV_CONTEXT_ONLY, prefill plans only):
 *                 attention over the stored context alone (mstar.engine.resources.kv.plan,
 *                 context_only_views): the index arrays describe only the context (see
 *                 pkv_context_only_views), query i of row r sits at position L_r + i and
 *                 sees every context key (window_left counted from that position); n_r may
 *                 exceed L_r; a query that sees no key gets out = 0 and lse = -inf.  Such a
 *                 plan appends nothing (pkv_kv_append_planned is a no-op on it).
 *   window_left   -1 unbounded, else >= 0.
 *   sm_scale      0 selects 1/sqrt(head_dim).
 *   workspace     device buffer of workspace_bytes (>= pkv_workspace_size for the
 *                 plan actually made; 256-byte aligned).  A too-small workspace returns
 *                 PKV_ERR_WORKSPACE and pkv_last_error states the bytes required.
 * Host staging is a ring of two page-locked sets fenced by CUDA events
 * (PinnedIndexRing), so a plan may be issued while the previous step still runs.
 */
pkv_status pkv_plan(pkv_handle_t h, int mode, const int32_t *qo_indptr, const int32_t *paged_kv_indptr,
                    const int32_t *paged_kv_indices, const int32_t *paged_kv_last_page_len, int batch,
                    int causal, int window_left, float sm_scale, void *workspace, size_t workspace_bytes,
                    pkv_stream_t stream);

/*
 * Last-page KV append from the index arrays themselves (the KVManager's write before
 * attention: DenseAttentionManager.requires_kv_write; the write location of
 * FlashInferDecodeWrapper.plan).  No plan is needed.  New token t of row r (qo_indptr[r]
 * <= t < qo_indptr[r+1]) sits at position p = L_r - n_r + (t - qo_indptr[r]) of the
 * post-append row and is written to page paged_kv_indices[paged_kv_indptr[r] + p /
 * page_size], slot p % page_size: its K row to [page, 0, slot, :, :] and its V row to
 * [page, 1, slot, :, :] of the layer slice.  Nothing else in the slice is touched.
 *   k, v:           DEVICE bf16 [num_new_tokens, num_kv_heads, head_dim], 16-byte aligned.
 *   num_new_tokens: qo_indptr[batch] (batch when qo_indptr is NULL).
 *   kv_layer:       DEVICE layer slice, written in place.
 *   qo_indptr, paged_kv_indptr, paged_kv_indices, paged_kv_last_page_len: DEVICE int32
 *                   arrays of the post-append state, as in pkv_plan; qo_indptr may be
 *                   NULL (decode: row r's one new token is token r).
 *   batch:          rows (<= max_batch).
 * The host never reads the device arrays, so the kernel checks every token's location
 * before it writes: a token whose row is inconsistent (non-monotone offsets, a fill
 * outside 1..page_size, a position outside the row, a page id outside the cache) is left
 * unwritten, and nothing outside the listed buffers is read or written.  Host-validated
 * appends come from pkv_plan + pkv_kv_append_planned.  Allocates nothing, never
 * synchronises, so it can sit in a captured graph.  PKV_ERR_INVALID on null or misaligned
 * pointers and negative sizes.
 */
pkv_status pkv_kv_append(pkv_handle_t h, const void *k, const void *v, int num_new_tokens, void *kv_layer,
                         const int32_t *qo_indptr, const int32_t *paged_kv_indptr, const int32_t *paged_kv_indices,
                         const int32_t *paged_kv_last_page_len, int batch, pkv_stream_t stream);

/*
 * The same append at the write locations the last pkv_plan on `workspace` computed and
 * validated on the host (FlashInferDecodeWrapper.plan: "compute KV write locations").
 * k, v: device bf16 [T, num_kv_heads, head_dim], T = the planned step's new tokens
 * (decode: batch).  kv_layer: device layer slice, written in place at (page, slot) of
 * each new token; nothing else in the slice is touched.  Must be issued on the stream the
 * plan was made on (or one ordered after it): the plan's copy into the workspace is
 * ordered only on that stream.  PKV_ERR_NOT_PLANNED without a plan on `workspace`; a
 * context-only plan appends nothing.
 */
pkv_status pkv_kv_append_planned(pkv_handle_t h, const void *k, const void *v, void *kv_layer, void *workspace,
                                 pkv_stream_t stream);

/*
 * Batched decode (FlashInferDecodeWrapper.run).  q: device bf16 [batch, Hq, D];
 * out: device bf16 [batch, Hq, D]; lse: device fp32 [batch, Hq] or NULL.
 */
pkv_status pkv_run_decode(pkv_handle_t h, const void *q, const void *kv_layer, void *out, float *lse,
                          void *workspace, pkv_stream_t stream);

/*
 * pkv_kv_append_planned followed by pkv_run_decode, in one kernel launch (same results, the
 * appended slots bit-identical).  Decode plans only (PKV_ERR_NOT_PLANNED otherwise).
 * k, v: device bf16 [batch, num_kv_heads, head_dim], 16-byte aligned; the rest as
 * pkv_run_decode.  The CTA that reads a row's last page writes the row's new token
 * into it and uses it from shared memory, so no other launch orders the two.
 */
pkv_status pkv_run_decode_append(pkv_handle_t h, const void *q, const void *k, const void *v, void *kv_layer,
                                 void *out, float *lse, void *workspace, pkv_stream_t stream);

/*
 * Ragged prefill over a cached prefix (FlashInferPrefillWrapper.run).  q, out: device
 * bf16 [T, Hq, D] in qo_indptr order; lse: device fp32 [T, Hq] or NULL.
 */
pkv_status pkv_run_prefill(pkv_handle_t h, const void *q, const void *kv_layer, void *out, float *lse,
                           void *workspace, pkv_stream_t stream);

/*
 * Mixed step (FlashInferMixedWrapper.run): the decode pass over every row of the
 * plan (non-decode rows read one token of sink_page, their result is dropped) and
 * the prefill pass over the prompt rows (at most max_prefill_rows, padded with empty
 * rows).  q, out: device bf16 [T, Hq, D] in the original qo_indptr order; lse: device
 * fp32 [T, Hq] or NULL.
 */
pkv_status pkv_run_mixed(pkv_handle_t h, const void *q, const void *kv_layer, void *out, float *lse,
                         void *workspace, pkv_stream_t stream);

/*
 * Dense varlen attention (mstar.engine.resources.attn.dense, DenseAttentionManager and
 * DensePlan): one pass over contiguous [frozen prefix | fresh tokens] K/V per segment,
 * no KV write.  pkv_plan_dense takes HOST int32 cu_q[batch+1] (query offsets into q /
 * out) and cu_k[batch+1] (key-row offsets into k / v); segment r's queries are its last
 * n_r = cu_q[r+1]-cu_q[r] keys' tokens (n_r <= L_r = cu_k[r+1]-cu_k[r]), so query i sits at
 * position L_r - n_r + i; causal 0/1 and window_left as for pkv_plan.  Workspace:
 * pkv_workspace_size(PKV_MODE_DENSE).  pkv_run_dense: q / out [cu_q[batch], Hq, D] bf16,
 * k / v [cu_k[batch], Hkv, D] bf16 (device, contiguous, 16-byte aligned), lse
 * [cu_q[batch], Hq] fp32 or NULL.  The pages call this path eager-only; graph_static does
 * not apply to it.
 */
pkv_status pkv_plan_dense(pkv_handle_t h, const int32_t *cu_q, const int32_t *cu_k, int batch, int causal,
                          int window_left, float sm_scale, void *workspace, size_t workspace_bytes,
                          pkv_stream_t stream);
pkv_status pkv_run_dense(pkv_handle_t h, const void *q, const void *k, const void *v, void *out, float *lse,
                         void *workspace, pkv_stream_t stream);

/*
 * Gather a frozen prefix out of the pages (DenseAttentionManager: "gathers the prefix once
 * per (stream, layer)"): positions 0 .. num_tokens-1 of the page list `pages` (DEVICE
 * int32, ceil(num_tokens / page_size) ids) are copied from the layer slice into k_out and
 * v_out ([num_tokens, Hkv, D] bf16, device).  Pure data movement.
 */
pkv_status pkv_gather_kv(pkv_handle_t h, const void *kv_layer, const int32_t *pages, int num_tokens, void *k_out,
                         void *v_out, pkv_stream_t stream);

/*
 * Read and clear the workspace's device error word (synchronises `stream`).
 * PKV_OK when no kernel recorded an error since the last plan on it.
 */
pkv_status pkv_check_device_error(pkv_handle_t h, void *workspace, pkv_stream_t stream, int *code);

/*
 * Self-test of that error path (no counterpart on the pages): one device thread waits,
 * for `polls` polls (1..2^20), on a barrier nothing arrives on, gives up, records error
 * code 4 in the workspace's error word and returns -- no trap, no hang.  A following
 * pkv_check_device_error reports PKV_ERR_DEVICE with code 4 and clears the word; the
 * handle, the workspace and the CUDA context stay usable.  Needs a plan on `workspace`.
 */
pkv_status pkv_selftest_wait_timeout(pkv_handle_t h, void *workspace, int polls, pkv_stream_t stream);

/*
 * Decode that needs no workspace: plan + pkv_run_decode in one call, with the plan and
 * the split-KV partials kept in a 16 MiB scratch array compiled into the library
 * (one per GPU that loads it, held until the process exits).  The pages have no
 * counterpart to this call.  It is for callers that are handed only their inputs,
 * outputs and a stream and may not allocate device memory themselves: plugin hooks of
 * inference runtimes whose host owns every allocation, and latency-critical paths that
 * must not enter an allocator that can synchronise the device or fail.
 *   q, out, lse, kv_layer: as pkv_run_decode.  kv_indptr, kv_indices, last_page_len:
 *   HOST int32 arrays as in pkv_plan (decode: one new token per row).
 * The call plans on the host (ordinary heap memory only), copies the plan from that
 * pageable memory into the scratch on `stream` (so it may wait for work already queued
 * there), and launches the decode and merge kernels; it makes no device or page-locked
 * allocation.  The scratch's device address is resolved once per CUDA context, on the
 * first call made with that device current (again after cudaDeviceReset).
 * Errors: PKV_ERR_WORKSPACE when the decode's plan and partials need more than 16 MiB
 * (pkv_last_error names the bytes); PKV_ERR_INVALID when `stream` is capturing, since
 * the plan is copied from host memory the call frees before returning; otherwise as
 * pkv_plan.  Every call shares the one array and overwrites it: calls that overlap on
 * the GPU (other streams or threads) race; calls on one stream do not.  Device-side
 * wait errors are recorded in the scratch and are not reported.
 */
pkv_status pkv_run_decode_static(pkv_handle_t h, const void *q, const void *kv_layer, void *out, float *lse,
                                 const int32_t *paged_kv_indptr, const int32_t *paged_kv_indices,
                                 const int32_t *paged_kv_last_page_len, int batch, int window_left, float sm_scale,
                                 pkv_stream_t stream);

/* ---- host-only planning queries (no CUDA call; usable on a machine without a GPU) ---- */

/*
 * KV write locations of a step (FlashInferDecodeWrapper.plan: "compute KV write
 * locations"; KVPlanOutput.decode_pages / decode_offsets): for every new token t,
 * pages[t] and slots[t].  Host arrays of the step's token count.
 */
pkv_status pkv_append_slots(int page_size, const int32_t *qo_indptr, const int32_t *paged_kv_indptr,
                            const int32_t *paged_kv_indices, const int32_t *paged_kv_last_page_len, int batch,
                            int32_t *pages, int32_t *slots);

/*
 * The mixed step's two plans (FlashInferMixedWrapper): is_decode[batch], prompt_rows
 * [max_prefill_rows] (-1 padding), perm[T] (perm[k] = original token of permuted token
 * k: prompt tokens first in row order, then the rest in order), pf_qo_indptr
 * [max_prefill_rows+1], the decode pass's dec_kv_indptr[batch+1], dec_kv_indices
 * [<= nnz + batch], dec_last_page_len[batch], dec_q_token[batch], dec_out_token[batch]
 * (-1 = dropped).  *dec_nnz receives the length of dec_kv_indices.
 */
pkv_status pkv_mixed_layout(const int32_t *qo_indptr, const int32_t *paged_kv_indptr,
                            const int32_t *paged_kv_indices, const int32_t *paged_kv_last_page_len, int batch,
                            int max_prefill_rows, int sink_page, int32_t *is_decode, int32_t *prompt_rows,
                            int32_t *perm, int32_t *pf_qo_indptr, int32_t *dec_kv_indptr,
                            int32_t *dec_kv_indices, int32_t *dec_last_page_len, int32_t *dec_q_token,
                            int32_t *dec_out_token, int *dec_nnz);

/*
 * mstar.engine.resources.kv.plan, context_only_views: the views of a step without the
 * tokens it appends.  Row r's length shrinks by its query count n_r = qo_indptr[r+1] -
 * qo_indptr[r]; the pages past the shorter length are dropped; last_page_len is
 * recomputed (0 for a row left without context).  Outputs: out_kv_indptr[batch+1],
 * out_kv_indices (<= input nnz entries), out_last_page_len[batch]; *out_nnz receives the
 * number of indices written.  PKV_ERR_INVALID if a row has more queries than tokens.
 */
pkv_status pkv_context_only_views(int page_size, const int32_t *qo_indptr, const int32_t *paged_kv_indptr,
                                  const int32_t *paged_kv_indices, const int32_t *paged_kv_last_page_len, int batch,
                                  int32_t *out_kv_indptr, int32_t *out_kv_indices, int32_t *out_last_page_len,
                                  int *out_nnz);

/*
 * The decode work split the plan would make: tiles[k] = {row, first visible page,
 * page count, partial slot or -1 for a direct write, cta}.  *num_tiles in: capacity
 * (tiles holds 5 * capacity ints), out: tiles written.  *num_ctas receives the grid.
 */
pkv_status pkv_decode_split(pkv_handle_t h, const int32_t *paged_kv_indptr, const int32_t *paged_kv_last_page_len,
                            int batch, int window_left, int32_t *tiles, int *num_tiles, int *num_ctas);

/*
 * The cache rows (page id * 2 * page_size + slot) of the first 4 16-key chunks of each
 * decode CTA of that split, in the order the CTA reads them, -1 past its last chunk: the
 * values the plan stores beside each CTA's tile range, from which the CTA's first K / V
 * copies are issued without loading its tile and page ids first.  rows holds 4 * capacity
 * ints; *num_ctas in: capacity (CTAs), out: CTAs written.  Host only.  PKV_ERR_INVALID on a
 * null argument or a buffer below the CTA count.
 */
pkv_status pkv_decode_head_rows(pkv_handle_t h, const int32_t *paged_kv_indptr, const int32_t *paged_kv_indices,
                                const int32_t *paged_kv_last_page_len, int batch, int window_left, int32_t *rows,
                                int *num_ctas);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
