/*
 * pagedkv.h -- C ABI of libpagedkv: the data-parallel hot path of a paged
 * KV cache on GB300 (sm_103a).
 *
 * What the library computes comes from four pages:
 *  - "A Paged KV Cache and Sliding-Window Attention" (silicon_compiler_from_
 *    scratch, chapter 15), section "The model": fixed-size pages from a
 *    shared pool, a block table per request, a LIFO free list, reference
 *    counts, fork, lazy copy-on-write and the window trim; Figure 15.1 (the
 *    released pages leave holes at the front of the table).
 *  - "PagedAttention block allocator" (llm-systems-cookbook), section
 *    "Sequence block table": position t lives in logical page t / P at
 *    offset t % P.
 *  - mini-sglang code series, part 4 (jaehun.me): the 6-axis KV buffer
 *    (2, layers, num_pages, page_size, kv_heads, head_dim), store_cache
 *    writing rows at flat token locations ``out_loc``, the raw-location page
 *    table, the page->token expansion and the one-scatter table write, the
 *    dummy request row and dummy page.
 *  - "Week 3 Day 3: Paged KV Cache" (tiny-llm), sections "Tail-Append Logic"
 *    and "Make write cost proportional to the appended slice" (a device write
 *    sized to the new rows) and "Correctness Checkpoint: Gather Pages for
 *    Dense Attention" (attention over the rows gathered in logical order).
 *
 * Conventions for every call
 *  - Return value: KVP_OK (0) or a negative KVP_ERR_* code. No exception or
 *    abort crosses the ABI.
 *  - Host-side argument checks run before any launch; a call that fails them
 *    launches nothing and changes nothing.
 *  - Device pointers (KV buffer, tables, q/k/v, outputs, workspace, the error
 *    word) are OWNED BY THE CALLER; the library never allocates or frees
 *    them. Host pointers are read or written only during the call.
 *  - ``stream`` is a cudaStream_t (NULL = the legacy default stream). Device
 *    calls are asynchronous on it; the caller orders them (page_table_write,
 *    copy_pages, store_cache, then paged_decode_attention for one step).
 *  - Errors found ON THE DEVICE (a negative or out-of-range table entry,
 *    slot or length, or a bounded internal wait that ran out) are recorded in
 *    the pool's device error word (first error wins) and the offending row
 *    is skipped; kvp_sync_error() reads and clears it. Kernels never trap.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVP_OK 0
#define KVP_ERR_INVALID_ARG (-1) /* bad argument; nothing launched            */
#define KVP_ERR_CUDA (-2)        /* a CUDA runtime call failed                */
#define KVP_ERR_OUT_OF_PAGES (-3)/* host bookkeeping: no free page, no change */
#define KVP_ERR_BAD_INDEX (-4)   /* device: table entry/slot/length invalid   */
#define KVP_ERR_TIMEOUT (-5)     /* device: a bounded wait ran out            */

enum kvp_dtype { KVP_F32 = 0, KVP_BF16 = 1 };
enum kvp_table_mode {
  KVP_BLOCK_TABLE = 0,   /* table[row][logical page] = physical page, -1 hole */
  KVP_RAW_LOCATIONS = 1  /* table[row][position] = flat token slot, -1 hole   */
};

typedef struct kvp_pool kvp_pool;

/* ------------------------------------------------------------------------
 * kv_pool_create: describe a caller-owned KV buffer (mini-sglang part 4,
 * section "KV 버퍼는 6축인데, 쓸 때는 3축이다").
 *   kv_buffer   device, (2, num_layers, num_pages, page_size, kv_heads,
 *               head_dim) elements of ``dtype``, C-contiguous; index 0 of
 *               the first axis is K, 1 is V. Must be 16-byte aligned.
 *               A flat token slot s = page * page_size + offset addresses
 *               row s of the (num_pages * page_size, kv_heads, head_dim)
 *               view of one layer's K or V. num_pages counts EVERY page of
 *               the buffer, including a dummy page the caller keeps back.
 *   error_word  device int32, zero-initialised, caller-owned; receives the
 *               first device-detected error of calls on this pool.
 *   out         receives an opaque descriptor (host memory owned by the
 *               library until kv_pool_destroy).
 * kv_heads * head_dim * sizeof(dtype) must be a multiple of 16 bytes.
 * Errors: INVALID_ARG (null pointer, non-positive size, misalignment),
 * CUDA (device query failed).
 * ---------------------------------------------------------------------- */
int kv_pool_create(int num_pages, int page_size, int kv_heads, int head_dim,
                   int dtype, int num_layers, void* kv_buffer,
                   int32_t* error_word, kvp_pool** out);
int kv_pool_destroy(kvp_pool* pool);

/* ------------------------------------------------------------------------
 * store_cache: K[layer][out_loc[i]] = k[i], V[layer][out_loc[i]] = v[i] for
 * i < n (mini-sglang part 4: store_cache(k_cache, v_cache, indices=out_loc,
 * k, v); tiny-llm week 3 day 3: the write covers only the new rows).
 *   k, v     device, [n, kv_heads, head_dim] of the pool's dtype, contiguous.
 *   out_loc  device int32 [n], flat token slots. Duplicate slots within one
 *            call are a caller error except in a dummy page (the last write
 *            is then unspecified).
 * A slot outside [0, num_pages*page_size) sets KVP_ERR_BAD_INDEX on the
 * device and that row is skipped. n == 0 launches nothing.
 * ---------------------------------------------------------------------- */
int store_cache(const kvp_pool* pool, int layer, const void* k, const void* v,
                const int32_t* out_loc, int n, void* stream);

/* ------------------------------------------------------------------------
 * page_table_write: the device-side table write for newly allocated (or
 * released, or copied-on-write) pages (mini-sglang part 4, section "할당은
 * 페이지로, 기록은 토큰으로": host-built (row, position) lists, one scatter;
 * its page->token expansion is done here on the device).
 * For i < n and j < expand:
 *     table[rows[i]][cols[i]*expand + j] = vals[i] < 0 ? -1
 *                                                    : vals[i]*expand + j
 *   expand = 1          block-table mode: cols = logical page, vals = page.
 *   expand = page_size  raw-location mode: cols/vals in PAGE units, written
 *                       as page_size token locations each.
 *   table    device int32 [table_rows_total, table_cols], row-major.
 *   rows, cols, vals  device int32 [n].
 *   error_word        device int32 or NULL; an entry outside the table sets
 *                     KVP_ERR_BAD_INDEX there and is skipped.
 * ---------------------------------------------------------------------- */
int page_table_write(int32_t* table, int table_rows_total, int table_cols,
                     const int32_t* rows, const int32_t* cols,
                     const int32_t* vals, int n, int expand,
                     int32_t* error_word, void* stream);

/* ------------------------------------------------------------------------
 * copy_pages: copy-on-write (chapter 15, section "The model": a shared tail
 * page is copied whole before a private write). For i < n, every layer, K
 * and V: page dst[i] <- page src[i]. src/dst device int32 [n]; a page
 * outside [0, num_pages) sets KVP_ERR_BAD_INDEX and is skipped. Pairs must
 * not overlap (no page is both a source and a destination).
 * ---------------------------------------------------------------------- */
int copy_pages(const kvp_pool* pool, const int32_t* src, const int32_t* dst,
               int n, void* stream);

/* ------------------------------------------------------------------------
 * paged_decode_attention: one decode step of attention for ``batch``
 * requests, one query token each, reading K/V in place through the table.
 * For request b and query head h (GQA: KV head h / (num_q_heads/kv_heads)):
 *     L  = context_lens[b]            (includes the token stored this step)
 *     lo = window > 0 ? max(0, L - (window - sinks)) : 0
 *     se = window > 0 ? min(sinks, lo) : 0
 *     s_t = scale * <q[b][h], K[slot(b,t)][h/G]>  for 0 <= t < se, lo <= t < L
 *     out[b][h] = sum_t softmax(s)_t * V[slot(b,t)][h/G]
 * sinks = 0 is the plain window; sinks > 0 keeps the first ``sinks`` rows
 * in every windowed context (chapter 15, exercise "Attention sinks": the
 * first S rows plus the last W - S). 0 <= sinks < window when window > 0
 * (else KVP_ERR_INVALID_ARG); ignored without a window.
 * slot(b,t): block mode table[r][t/P]*P + t%P, raw mode table[r][t], with
 * r = table_rows ? table_rows[b] : b (the mini-sglang table_idx).
 * Sources: chapter 15, section "The model" (the window: the new token and at
 * most W-1 earlier ones); tiny-llm week 3 day 3, section "Correctness
 * Checkpoint" (dense attention over the gathered rows, here read in place).
 *   q            device [batch, num_q_heads, head_dim], pool dtype.
 *   table        device int32 [table_rows_total, table_cols].
 *   context_lens device int32 [batch]; 1 <= L <= table capacity.
 *   out          device [batch, num_q_heads, head_dim], pool dtype (bf16
 *                results are rounded to nearest even from fp32).
 *   workspace    device, >= paged_decode_attention_workspace_size() bytes,
 *                256-byte aligned; scratch for the work plan and split-K
 *                partials. Its contents need no initialisation and are
 *                clobbered; two calls that may run at the same time on the
 *                GPU need separate workspaces.
 * Device-detected errors (L out of range, hole or out-of-range entry in the
 * attended range) set KVP_ERR_BAD_INDEX; an invalid request's output is
 * zero-filled.
 * ---------------------------------------------------------------------- */
int paged_decode_attention_workspace_size(const kvp_pool* pool, int batch,
                                          int num_q_heads, size_t* bytes);
int paged_decode_attention(const kvp_pool* pool, int layer, const void* q,
                           int batch, int num_q_heads, const int32_t* table,
                           int table_rows_total, int table_cols,
                           int table_mode, const int32_t* table_rows,
                           const int32_t* context_lens, int window,
                           int sinks, float scale, void* out,
                           void* workspace, size_t workspace_bytes,
                           void* stream);

/* ------------------------------------------------------------------------
 * paged_verify_attention: multi-token verify for speculative decoding. The
 * M = num_q_tokens newest tokens of each request (already stored; L =
 * context_lens[b] counts them) are queries at once: query j sits at
 * position p = L - M + j and attends what a one-token step with context
 * p + 1 attends (causal; the same window and sinks), i.e.
 *     out[b][j][h] = paged_decode_attention with context p + 1.
 * "Week 3 Day 3: Paged KV Cache" (tiny-llm) names speculative decoding as
 * the user of rewind(n) (kvp_host_rewind); the verify formula is the
 * decode step's, applied per query position. The K/V rows are read once
 * for all M queries.
 *   q    device [batch, M, num_q_heads, head_dim], pool dtype, 16-byte aligned.
 *   out  device [batch, M, num_q_heads, head_dim], pool dtype.
 *   context_lens  M <= L <= table capacity (else KVP_ERR_BAD_INDEX, zeros).
 *   1 <= M <= 32. Workspace from paged_verify_attention_workspace_size;
 * everything else as paged_decode_attention.
 * ---------------------------------------------------------------------- */
int paged_verify_attention_workspace_size(const kvp_pool* pool, int batch,
                                          int num_q_tokens, int num_q_heads,
                                          size_t* bytes);
int paged_verify_attention(const kvp_pool* pool, int layer, const void* q,
                           int batch, int num_q_tokens, int num_q_heads,
                           const int32_t* table, int table_rows_total,
                           int table_cols, int table_mode,
                           const int32_t* table_rows,
                           const int32_t* context_lens, int window,
                           int sinks, float scale, void* out,
                           void* workspace, size_t workspace_bytes,
                           void* stream);

/* ------------------------------------------------------------------------
 * paged_prefill_attention: chunked prefill. Request b's q_lens[b] newest
 * tokens (NULL: ``chunk`` each; their K/V already stored, L =
 * context_lens[b] counts them) are queries at once; query j sits at
 * position L - q_lens[b] + j and attends what a one-token decode step with
 * that context attends (causal, window and sinks as paged_decode_attention)
 * - the formula of paged_verify_attention for chunks of any length
 * ("Week 3 Day 3: Paged KV Cache" of tiny-llm: chunked prefill appends each
 * chunk to the pages, then attends over them). bf16 pools with head_dim 128,
 * 128 % (num_q_heads / kv_heads) == 0 and scale > 0 run on the tcgen05
 * tensor cores (TMEM accumulators), others on the general kernel. The
 * tcgen05 kernel keeps the pool's tensor map (built on first use) in the
 * pool descriptor; ``q`` is mapped per call. It may read the rows of a
 * request's last page past the attended span (they lie in the same page of
 * the pool); whatever they hold never reaches the output.
 *   q    device [batch, chunk, num_q_heads, head_dim], pool dtype,
 *        16-byte aligned.
 *   out  device, the same shape; rows j >= q_lens[b] are not written.
 *   q_lens  device int32 [batch] with 1 <= q_lens[b] <= min(chunk, L), or NULL.
 * No workspace. Errors as paged_decode_attention (an invalid request's rows
 * are zero-filled).
 * ---------------------------------------------------------------------- */
int paged_prefill_attention(const kvp_pool* pool, int layer, const void* q,
                            int batch, int chunk, int num_q_heads,
                            const int32_t* q_lens, const int32_t* table,
                            int table_rows_total, int table_cols,
                            int table_mode, const int32_t* table_rows,
                            const int32_t* context_lens, int window,
                            int sinks, float scale, void* out, void* stream);

/* ------------------------------------------------------------------------
 * store_cache_and_attention: one layer of a decode step in one launch:
 *     page_table_write(table, tw_rows, tw_cols, tw_vals, n_tw, expand);
 *     store_cache(pool, layer, k, v, out_loc, batch);
 *     paged_decode_attention(pool, layer, q, ...);
 * with expand = page_size for a raw-location table, else 1; the results
 * (table, cache rows, out) are those of the three calls in that order (the
 * mini-sglang code series, part 4: host-built lists, one scatter, then the
 * attention). Not a separate operation of the source pages: it saves two
 * launches and their ramps per step.
 * In one launch the attention cannot wait for the writes, so the call
 * relies on what a decode step guarantees:
 *   - out_loc[b] is the slot of request b's newest position
 *     (context_lens[b] - 1): that position is read from k[b], v[b];
 *   - the table writes touch no entry of an attended position other than
 *     the newest ones (new pages for this step's tokens). Releases of a
 *     sliding window and copy-on-write pages are written before (copy) or
 *     after (release) the call, not through it.
 *   k, v      device [batch, kv_heads, head_dim], pool dtype, 16-byte aligned.
 *   out_loc   device int32 [batch].
 *   tw_*      device int32 [n_tw] (n_tw may be 0; then they may be NULL).
 * Other arguments, the workspace and the errors as for
 * paged_decode_attention and the two writes. Pools without the fused kernel
 * (fp32, head_dim other than 128) run the three operations in sequence.
 * ---------------------------------------------------------------------- */
int store_cache_and_attention(const kvp_pool* pool, int layer, const void* q,
                              const void* k, const void* v,
                              const int32_t* out_loc, int batch,
                              int num_q_heads, int32_t* table,
                              int table_rows_total, int table_cols,
                              int table_mode, const int32_t* table_rows,
                              const int32_t* context_lens,
                              const int32_t* tw_rows, const int32_t* tw_cols,
                              const int32_t* tw_vals, int n_tw, int window,
                              int sinks, float scale, void* out, void* workspace,
                              size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * paged_decode_attention_noalloc: paged_decode_attention for callers that
 * cannot allocate device memory at the point where they run attention (code
 * inside another framework's memory pool or under a budget that forbids new
 * reservations, callers that may not enter an allocator from their thread,
 * plug-in hosts that only receive their input and output buffers). There is
 * no counterpart in the source pages: it is an interface convenience.
 * Same arguments (window and sinks included) and results as
 * paged_decode_attention minus the workspace: the split-K scratch is a fixed
 * 12 MiB array in the library's own device memory, held by every GPU that
 * loads it until the process exits.
 *  - The pool's device must be current. The first call on a device looks up
 *    the array's device address (cudaGetSymbolAddress) and keeps it with the
 *    CUDA context it belongs to; make that first call before any stream
 *    capture. After a device reset a call finds another context current and
 *    looks the address up again (outside a capture, as the first call).
 *  - No allocation of any kind (no cudaMalloc/cudaFree, no library
 *    allocator) happens in any call.
 *  - A shape whose scratch would exceed 12 MiB is rejected with
 *    KVP_ERR_INVALID_ARG and nothing is launched; so is a pool of another
 *    device than the current one.
 *  - Every call on a device shares the one array: calls that overlap on the
 *    GPU (different streams, or different pools on the same device) race and
 *    must be serialised by the caller. The array keeps the last call's
 *    contents; nothing in it needs to start at zero.
 * ---------------------------------------------------------------------- */
int paged_decode_attention_noalloc(const kvp_pool* pool, int layer,
                                   const void* q, int batch, int num_q_heads,
                                   const int32_t* table, int table_rows_total,
                                   int table_cols, int table_mode,
                                   const int32_t* table_rows,
                                   const int32_t* context_lens, int window,
                                   int sinks, float scale, void* out,
                                   void* stream);

/* ------------------------------------------------------------------------
 * gather_indices: the slots paged_decode_attention would read, for
 * bit-exact checks of the index arithmetic ("PagedAttention block
 * allocator", section "Sequence block table"; chapter 15 Figure 15.1).
 * slots_out device int32 [batch, max_tokens]: row b holds the slots of the
 * attended positions in logical order (the se sink rows, then lo..L-1; see
 * paged_decode_attention) and -1 after. More than max_tokens of them, or an
 * invalid entry, sets KVP_ERR_BAD_INDEX (the entry is written as -1).
 * ---------------------------------------------------------------------- */
int gather_indices(const kvp_pool* pool, const int32_t* table,
                   int table_rows_total, int table_cols, int table_mode,
                   const int32_t* table_rows, const int32_t* context_lens,
                   int batch, int window, int sinks, int32_t* slots_out,
                   int max_tokens, void* stream);

/* kvp_sync_error: wait for ``stream``, read the pool's device error word
 * into *err (0 = none) and clear it. */
int kvp_sync_error(const kvp_pool* pool, void* stream, int* err);

/* kvp_selftest_wait: checks, on the device, the bounded wait behind every
 * pipeline wait of the library's kernels (mbarrier try-wait against the
 * global timer, then an error code instead of a hang). One warp waits on a
 * shared-memory mbarrier for at most limit_ns (1 .. 1e9 ns). arrive = 0:
 * nothing arrives, the wait gives up after limit_ns and KVP_ERR_TIMEOUT is
 * recorded in *err (DEVICE int32, first error wins, as the pool's error
 * word). arrive = 1: the barrier is satisfied first and nothing is recorded.
 * Asynchronous on ``stream``; KVP_ERR_INVALID_ARG for a NULL err or a limit
 * or mode out of range. No kernel traps or hangs either way. */
int kvp_selftest_wait(long long limit_ns, int arrive, int32_t* err, void* stream);

/* kvp_pool_set_timing_events: measurement hook. When both events are
 * non-NULL (cudaEvent_t, caller-owned), the next paged_decode_attention call
 * on this pool records ``before`` on its stream just before its main
 * attention kernel and ``after`` just after it, then forgets them; NULL
 * clears the hook. No effect on results. */
int kvp_pool_set_timing_events(kvp_pool* pool, void* before, void* after);

/* ========================================================================
 * Host bookkeeping (pure host C++; no CUDA). Chapter 15, section "The
 * model", restated: LIFO free list, reference counts, block tables indexed
 * by absolute logical page, fork, lazy copy-on-write, window trim, release.
 * Request ids are table rows in [0, max_requests).
 * Every call that can run out of pages checks first and changes nothing on
 * KVP_ERR_OUT_OF_PAGES (chapter 15, section "Tests", item 2).
 * ====================================================================== */
typedef struct kvp_host kvp_host;

/* free_stack: the initial free list as a stack, free_stack[num_pages-1] is
 * handed out first; NULL means num_pages-1 .. 0 (page 0 first). */
int kvp_host_create(int num_pages, int page_size, int max_requests,
                    const int32_t* free_stack, kvp_host** out);
int kvp_host_destroy(kvp_host* h);
int kvp_host_new(kvp_host* h, int rid);
int kvp_host_release(kvp_host* h, int rid);

/* Fork: dst shares every page of src (one more reference each, no data
 * copied). Emits the table writes (dst, logical page, page or -1) that make
 * the device row of dst equal to that of src; capacity tw_cap must cover
 * every logical page of src, count in *n_tw. On a short buffer returns
 * KVP_ERR_INVALID_ARG and changes nothing. */
int kvp_host_fork(kvp_host* h, int src, int dst, int32_t* tw_rows,
                  int32_t* tw_cols, int32_t* tw_vals, int tw_cap, int* n_tw);

/* Append one token to each of rids[0..n) in order (one token per entry; a
 * request may appear several times). Outputs (host arrays):
 *   slots[n]                 flat slot of each new token;
 *   tw_rows/tw_cols/tw_vals  table writes (row, logical page, page) for new
 *                            pages and copy-on-write replacements; capacity
 *                            tw_cap >= n suffices; count in *n_tw;
 *   cow_src/cow_dst          copy-on-write page pairs, capacity >= n; count
 *                            in *n_cow.
 * If the pool cannot serve the whole batch, returns KVP_ERR_OUT_OF_PAGES and
 * changes nothing. */
int kvp_host_append(kvp_host* h, const int32_t* rids, int n, int32_t* slots,
                    int32_t* tw_rows, int32_t* tw_cols, int32_t* tw_vals,
                    int tw_cap, int* n_tw, int32_t* cow_src,
                    int32_t* cow_dst, int* n_cow);

/* Release the front pages of request rid that hold only positions below
 * keep_from (page ``dropped`` goes while (dropped+1)*P <= keep_from). Emits
 * (rid, logical page, -1) table writes; capacity tw_cap, count in *n_tw. */
int kvp_host_trim(kvp_host* h, int rid, int keep_from, int32_t* tw_rows,
                  int32_t* tw_cols, int32_t* tw_vals, int tw_cap, int* n_tw);

/* kvp_host_trim for a window with attention sinks (chapter 15, exercise
 * "Attention sinks": the first S rows stay in every context). The first
 * sp = ceil(sink_rows / P) pages are kept; after them page sp + dropped goes
 * while (sp + dropped + 1) * P <= keep_from. sink_rows = 0 is kvp_host_trim.
 * A request's sink count cannot change once it has released pages
 * (KVP_ERR_INVALID_ARG, nothing changed). */
int kvp_host_trim_sinks(kvp_host* h, int rid, int keep_from, int sink_rows,
                        int32_t* tw_rows, int32_t* tw_cols, int32_t* tw_vals,
                        int tw_cap, int* n_tw);

/* Drop the newest n tokens of request rid ("Week 3 Day 3: Paged KV Cache",
 * tiny-llm: rewind(n) frees the whole pages no longer needed and shortens
 * the valid length of the last page; speculative decoding uses it when
 * drafted tokens are rejected). Pages past ceil((length - n) / P) are let go
 * tail first, so that the free stack hands them back in logical order, and
 * emitted as (rid, logical page, -1) table writes (capacity tw_cap, count in
 * *n_tw). The new length may not reach below the pages a window or its sinks
 * released (KVP_ERR_INVALID_ARG, nothing changed); n > length likewise. */
int kvp_host_rewind(kvp_host* h, int rid, int n, int32_t* tw_rows,
                    int32_t* tw_cols, int32_t* tw_vals, int tw_cap, int* n_tw);

/* ------------------------------------------------------------------------
 * kvp_decode_step: one decode step of the whole path in one call, in the
 * order of chapter 15's host loop ("The model") with the attention after a
 * separate store:
 *   1. host bookkeeping: one token for each request rids[0..n) (request id
 *      = table row; each id at most once); all-or-nothing on exhaustion;
 *   2. one host->device copy of the step's metadata, packed in host_meta
 *      (caller-owned PINNED host memory) and copied to dev_meta (device):
 *      [slots n | table writes 3*w | copy pairs 2*c | lengths n | rows n |
 *       trim writes 3*t];
 *   3. copy_pages, then for each layer l: wait for layer_ready[l] (a
 *      cudaEvent_t, or NULL), store_cache_and_attention(q[l], k[l], v[l]
 *      -> out[l]; layer 0 also applies the step's table writes, or a
 *      separate page_table_write precedes it when the step copies pages),
 *      record layer_done[l] (or NULL); q/k/v/out are per-layer DEVICE
 *      pointers;
 *   4. the window's trim writes (released pages are read by this step):
 *      keep_from = L + 1 - (window - sinks), keeping the first
 *      ceil(sinks / P) pages (kvp_host_trim_sinks); a request's sink count
 *      must stay the same from step to step.
 * meta_cap bounds host_meta/dev_meta in int32 entries (8n plus three per
 * page the window releases suffices); it and every argument are checked
 * before anything changes. host_meta is read asynchronously: reuse it only
 * after the stream has passed this call. ``info`` receives the counts.
 * Errors: as the calls it makes; KVP_ERR_OUT_OF_PAGES leaves the host
 * bookkeeping unchanged and launches nothing.
 * ---------------------------------------------------------------------- */
typedef struct kvp_step_info {
  int n_table_writes;  /* new pages and copy-on-write replacements */
  int n_copies;        /* copy-on-write page pairs */
  int n_trim_writes;   /* pages released by the window */
  int meta_ints;       /* int32 entries copied to the device */
} kvp_step_info;

int kvp_decode_step(kvp_host* h, const kvp_pool* pool, int32_t* table,
                    int table_rows_total, int table_cols, int table_mode,
                    const int32_t* rids, int n, int window, int sinks,
                    int num_q_heads,
                    float scale, const void* const* q, const void* const* k,
                    const void* const* v, void* const* out,
                    void* const* layer_ready, void* const* layer_done,
                    int32_t* host_meta, int32_t* dev_meta, int meta_cap,
                    void* workspace, size_t workspace_bytes, void* stream,
                    kvp_step_info* info);

/* Queries. kvp_host_block_row writes dropped+live entries (-1 for released
 * pages) to out (capacity cap) and the count to *n. */
int kvp_host_used(const kvp_host* h, int* used);
int kvp_host_length(const kvp_host* h, int rid, int* length, int* dropped);
int kvp_host_block_row(const kvp_host* h, int rid, int32_t* out, int cap,
                       int* n);
int kvp_host_refcounts(const kvp_host* h, int32_t* out, int cap);
int kvp_host_free_list(const kvp_host* h, int32_t* out, int cap, int* n);

/* ------------------------------------------------------------------------
 * Device-side page allocation: the block-table bookkeeping of kvp_host_*
 * (chapter 15 "The model": LIFO free list, reference counts, a fresh page
 * on a page boundary, lazy copy-on-write of a shared tail page, window trim
 * with sinks, release) kept in device memory, so that a decode step needs
 * no host decision and no host->device copy of table writes (mini-sglang
 * code series, part 4: allocate by page, record by token, here both on the
 * device). Every decision is taken in the order the host bookkeeping takes
 * it, request after request, so the device state equals kvp_host_*'s for
 * the same operations.
 *   state   caller-owned device buffer of kvp_dev_pages_bytes(), 16-byte
 *           aligned: [top, error word][free stack][ref counts][lengths]
 *           [released pages][sink pages]. The library keeps the pointer.
 *   table   the caller's device table (block: page ids; raw: token slots,
 *           expanded P per page), at least max_requests rows; request id
 *           = table row.
 * Each call is one thread block of up to 1024 requests, asynchronous on
 * ``stream``, and all-or-nothing: a bad request id, a repeated id, a row too
 * short, a full pool (KVP_ERR_OUT_OF_PAGES) or a short output buffer sets
 * the state's error word (kvp_dev_sync_error) and changes nothing.
 * ---------------------------------------------------------------------- */
typedef struct kvp_dev_pages kvp_dev_pages;

int kvp_dev_pages_bytes(int num_pages, int max_requests, size_t* bytes);
int kvp_dev_pages_create(int num_pages, int page_size, int max_requests,
                         void* state, size_t state_bytes, int32_t* table,
                         int table_rows, int table_cols, int table_mode,
                         kvp_dev_pages** out);
int kvp_dev_pages_destroy(kvp_dev_pages* d);
/* Empty pool: the free stack from free_stack (device int32 [num_pages], the
 * end handed out first), or num_pages-1 .. 0 when NULL; counts zero. */
int kvp_dev_pages_init(kvp_dev_pages* d, const int32_t* free_stack,
                       void* stream);
/* Start requests rids[0..n) (device int32) with no rows. */
int kvp_dev_new(kvp_dev_pages* d, const int32_t* rids, int n, void* stream);
/* Append counts[i] rows (NULL: one) to request rids[i] (device int32 [n],
 * n <= 1024, distinct ids): new pages popped in call order, a shared tail
 * page copied first (pairs in cow_src/cow_dst [n], their number in *n_cow,
 * all device; copy them with copy_pages_device_count before storing), the
 * table entries written (expanded for a raw table), the slot of every new
 * row in out_loc (device int32, request-major, at most max_tokens) and, if
 * lens_out is not NULL, each request's new length (device int32 [n], the
 * context_lens of the step's attention). */
int kvp_dev_append(kvp_dev_pages* d, const int32_t* rids,
                   const int32_t* counts, int n, int32_t* out_loc,
                   int max_tokens, int32_t* cow_src, int32_t* cow_dst,
                   int32_t* n_cow, int32_t* lens_out, void* stream);
/* Window trim of requests rids[i] to keep_from[i] (both device int32 [n])
 * keeping the first ceil(sinks / P) pages, as kvp_host_trim_sinks; the
 * released entries become -1. keep_from NULL: each request's own
 * L + 1 - (window - sinks), what its next decode step reads (0 <= sinks <
 * window). At most 4096 pages per call. */
int kvp_dev_trim(kvp_dev_pages* d, const int32_t* rids, const int32_t* keep_from,
                 int n, int window, int sinks, void* stream);
/* End requests rids[0..n): every live page loses a reference (and returns
 * to the free stack at zero), as kvp_host_release. At most 4096 pages. */
int kvp_dev_release(kvp_dev_pages* d, const int32_t* rids, int n,
                    void* stream);
/* Rewind (kvp_host_rewind on the device): request rids[i] drops its newest
 * n_back[i] rows (both device int32 [n], n <= 1024); the pages past the new
 * length go, tail first, and their entries become -1. A rewind below the
 * rows a window or its sinks released, or n_back[i] outside [0, length],
 * sets KVP_ERR_INVALID_ARG in the state's error word and changes nothing. */
int kvp_dev_rewind(kvp_dev_pages* d, const int32_t* rids, const int32_t* n_back,
                   int n, void* stream);
/* Fork: request dst[i] shares every page of src[i] (one more reference
 * each) and takes its length (device int32 [n]); the dst ids must be
 * distinct and none of them a src of the same call. */
int kvp_dev_fork(kvp_dev_pages* d, const int32_t* src, const int32_t* dst,
                 int n, void* stream);
/* Read and clear the state's error word (synchronises the stream). */
int kvp_dev_sync_error(kvp_dev_pages* d, void* stream, int* err);
/* kvp_decode_step with the page bookkeeping on the device: for the n
 * requests rids (DEVICE int32 [n], distinct, ids = table rows),
 *   1. kvp_dev_append: one row each, slots and new lengths into scratch;
 *   2. if may_share (requests can hold shared pages after a fork): the
 *      copy-on-write copies, copy_pages_device_count;
 *   3. for each layer l: wait for layer_ready[l] (or NULL), one
 *      store_cache_and_attention(q[l], k[l], v[l] -> out[l]) (per-layer
 *      DEVICE pointers, as kvp_decode_step), record layer_done[l];
 *   4. with a window: kvp_dev_trim to each request's L + 1 - (window - sinks).
 * scratch: device int32 [4n + 1] (slots, lengths, copy pairs, their count),
 * owned by the caller, in use until the step completes on ``stream``.
 * Nothing is synchronised; device-detected errors go to the state's error
 * word (kvp_dev_sync_error) and the pool's (kvp_sync_error). */
int kvp_decode_step_device(kvp_dev_pages* d, const kvp_pool* pool,
                           int32_t* table, int table_rows_total,
                           int table_cols, int table_mode,
                           const int32_t* rids, int n, int window, int sinks,
                           int num_q_heads, float scale,
                           const void* const* q, const void* const* k,
                           const void* const* v, void* const* out,
                           void* const* layer_ready, void* const* layer_done,
                           int32_t* scratch, int may_share, void* workspace,
                           size_t workspace_bytes, void* stream);
/* kvp_decode_step_device with host buffers: q_host/k_host/v_host (per-layer
 * HOST pointers, [n, Hq, D] / [n, kv_heads, D], pinned for the copies to
 * be asynchronous) are copied into the caller's per-layer device staging
 * q_dev/k_dev/v_dev, the step runs, and each layer's output goes from
 * out_dev back to out_host. Returns once the outputs are on the host (the
 * stream is synchronised). One call per step.
 * The input copies run on a copy stream of the page state, after the work
 * already queued on ``stream``, while the page append runs on ``stream``;
 * layer l's attention waits for layer l's copies only, and layer l's output
 * goes back on a second copy stream as soon as the layer is done. The first
 * call creates the two streams and 2 * num_layers + 1 events;
 * kvp_dev_pages_destroy releases them (no device memory is allocated). */
int kvp_decode_step_device_io(kvp_dev_pages* d, const kvp_pool* pool,
                              int32_t* table, int table_rows_total,
                              int table_cols, int table_mode,
                              const int32_t* rids, int n, int window,
                              int sinks, int num_q_heads, float scale,
                              const void* const* q_host,
                              const void* const* k_host,
                              const void* const* v_host,
                              void* const* out_host, void* const* q_dev,
                              void* const* k_dev, void* const* v_dev,
                              void* const* out_dev, int32_t* scratch,
                              int may_share, void* workspace,
                              size_t workspace_bytes, void* stream);
/* kvp_verify_step_device_io: one speculative-decoding verify step with the
 * page bookkeeping on the device and host buffers ("Week 3 Day 3: Paged KV
 * Cache" of tiny-llm names speculative decoding as the user of rewind(n)):
 *   1. the inputs go to the caller's device staging on the page state's copy
 *      stream: per layer q_host[l] [n, M, Hq, D] -> q_dev[l], k_host[l] and
 *      v_host[l] [n * M, kv_heads, D] (request-major) -> k_dev[l], v_dev[l],
 *      and n_back_host (host int32 [n], 0 <= n_back[i] <= M) into scratch;
 *   2. kvp_dev_append: M rows for each of the n requests rids (DEVICE int32
 *      [n], distinct, ids = table rows); if may_share, the copy-on-write
 *      copies;
 *   3. for each layer, once its inputs are in: store_cache of the n * M
 *      rows, paged_verify_attention(q_dev[l] -> out_dev[l]) with the new
 *      lengths;
 *   4. kvp_dev_rewind of n_back[i] rows per request (the rejected drafts),
 *      then with a window kvp_dev_trim to L + 1 - (window - sinks);
 *   5. out_dev[l] -> out_host[l] on a second copy stream as soon as layer l
 *      is done; returns once the outputs are on the host.
 * scratch: device int32 [n * M + 4 n + 1]; workspace as
 * paged_verify_attention_workspace_size(pool, n, M, Hq). Host buffers
 * should be pinned for the copies to be asynchronous. Errors as the calls
 * it makes; device-detected ones go to the state's and the pool's error
 * words. */
int kvp_verify_step_device_io(kvp_dev_pages* d, const kvp_pool* pool,
                              int32_t* table, int table_rows_total,
                              int table_cols, int table_mode,
                              const int32_t* rids, int n, int num_q_tokens,
                              int window, int sinks, int num_q_heads,
                              float scale, const void* const* q_host,
                              const void* const* k_host,
                              const void* const* v_host,
                              const int32_t* n_back_host,
                              void* const* out_host, void* const* q_dev,
                              void* const* k_dev, void* const* v_dev,
                              void* const* out_dev, int32_t* scratch,
                              int may_share, void* workspace,
                              size_t workspace_bytes, void* stream);
/* copy_pages with the number of pairs read on the device (at most max_n),
 * for the pairs kvp_dev_append emits. */
int copy_pages_device_count(const kvp_pool* pool, const int32_t* src,
                            const int32_t* dst, const int32_t* n_dev,
                            int max_n, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
