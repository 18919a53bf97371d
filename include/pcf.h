/*
 * pcf.h -- C ABI of the position-free KV cache-fusion hot path (GB300, sm_103a).
 *
 * The operation (from the two methods this library implements):
 *   - MiniPIC: Position-Independent Caching ..., section 2.1 "Position-free KV": the cache holds
 *     UNROTATED keys k~_j in shared physical pages; attention applies RoPE on the fly from the
 *     key's per-request logical position pi(j): score(t, j) = (R_t q_t)^T (R_pi(j) k~_j) / sqrt(d),
 *     implemented as a cos/sin table lookup and fused multiply-adds per key element, so one
 *     physical block serves concurrent requests at different offsets (section 1, "concurrency
 *     barrier").
 *   - QCFuse: Query-Centric Cache Fusion ..., section 2B "Critical-layer attention profiling": at
 *     one critical layer the query attends to the key cache only; the attention weights rank the
 *     context tokens and the Top-N guide selective recomputation (section 2C / Phase 4), done by a
 *     sparse attention that keeps causal constraints.
 *
 * Conventions
 *   - Every entry point returns pcf_status (0 = PCF_OK, negative = error) and never allocates
 *     memory: all host and device buffers belong to the caller.
 *   - Device calls are asynchronous on the caller's CUDA stream, passed as `void* stream`
 *     (a cudaStream_t; NULL = legacy default stream).  Arguments are validated on the host before
 *     any launch; an invalid call launches nothing.
 *   - bf16 tensors are passed as `const uint16_t*` (raw bfloat16 bits).  Device pointers must be
 *     16-byte aligned.
 *   - Tensor layouts (row-major, innermost last):
 *       k_pool, v_pool : [n_phys_pages][Hkv][16][d]     cached pages, keys UNROTATED
 *       q_query        : [sum_b T_b][Hq][d]              scoring query, unrotated
 *       q_fresh        : [sum_b rows_b][Hq][d]           rows of request b: its R_b recomputed
 *       k_fresh,v_fresh: [sum_b rows_b][Hkv][d]          tokens (ascending token index) then its
 *       out            : [sum_b rows_b][Hq][d]           T_b query tokens; all unrotated
 *       rope           : [max_pos][d/2][2] fp32          (cos, sin) of p * theta^(-2i/d)
 *     Query head h reads kv head h / (Hq/Hkv).  RoPE pairs dimension i with i + d/2.
 *   - A batch is described once by a "layout": an int32 blob built on the host by
 *     pcf_layout_build and copied by the caller to the device.  Calls take both copies
 *     (pcf_layout.host for launch configuration, pcf_layout.dev for the kernels); they must hold
 *     the same words.
 *   - Device-side faults that the host cannot rule out (a bounded wait that ran out, an index out
 *     of range) set a device error word and the kernel returns early; pcf_check_device_error
 *     reports and clears it.
 */
#ifndef PCF_H
#define PCF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pcf_status;
#define PCF_OK                        0
#define PCF_ERR_INVALID_ARG          -1  /* bad pointer, size, span placement or layout blob */
#define PCF_ERR_UNSUPPORTED          -2  /* head_dim not in {64,128}, group size not a divisor of 128 */
#define PCF_ERR_CUDA                 -3  /* a CUDA runtime/driver call failed */
#define PCF_ERR_DEVICE_TIMEOUT       -4  /* a kernel's bounded wait ran out (reported by check) */
#define PCF_ERR_WORKSPACE_TOO_SMALL  -5
#define PCF_ERR_DEVICE_BOUNDS        -6  /* a kernel met an out-of-range index (reported by check) */
#define PCF_ERR_NO_DEVICE            -7  /* no sm_103 device is current */
#define PCF_ERR_DEVICE_RANGE         -8  /* a rotated query or key left the fp16 operand range
                                            (infinities included; reported by check) */

/* One cached span of a request: n_pages consecutive physical pages starting at phys_first_page,
 * holding tokens at logical positions pos0 .. pos0 + 16*n_pages - 1; k of its tokens are to be
 * recomputed (0 <= k <= 16*n_pages).  MiniPIC section 2.2: spans are padded to page boundaries. */
typedef struct pcf_span_desc {
    int32_t phys_first_page;
    int32_t n_pages;
    int32_t pos0;
    int32_t k;
} pcf_span_desc;

/* One request: its spans in increasing position order, then n_query query tokens at positions
 * query_pos0 .. query_pos0 + n_query - 1 (query_pos0 after the last span token). */
typedef struct pcf_request_desc {
    int32_t n_spans;
    const pcf_span_desc* spans;
    int32_t n_query;
    int32_t query_pos0;
} pcf_request_desc;

typedef struct pcf_dims {
    int32_t n_q_heads;     /* Hq */
    int32_t n_kv_heads;    /* Hkv, divides Hq; g = Hq/Hkv must divide 128 */
    int32_t head_dim;      /* d in {64, 128} */
    int32_t n_phys_pages;  /* pages in the pool */
    int32_t max_pos;       /* rows of the rope table; every position must be < max_pos <= 1<<20 */
    int32_t n_sms;         /* SMs the work lists are balanced over (the device's multiprocessor
                              count); <= 0 selects 152, GB300's count; at most 4096 */
} pcf_dims;

typedef struct pcf_layout {
    const int32_t* host;   /* blob in host memory */
    const int32_t* dev;    /* identical blob in device memory */
} pcf_layout;

/* Header words of a layout blob readable with pcf_layout_query (sizes for the caller). */
enum {
    PCF_L_WORDS = 1, PCF_L_N_REQS = 2, PCF_L_HQ = 3, PCF_L_HKV = 4, PCF_L_D = 5,
    PCF_L_N_PHYS_PAGES = 6, PCF_L_MAX_POS = 7, PCF_L_TOTAL_TOKENS = 8, PCF_L_TOTAL_QUERY = 9,
    PCF_L_TOTAL_ROWS = 10, PCF_L_TOTAL_SEL = 11, PCF_L_TOTAL_PAGES = 12, PCF_L_N_SPANS = 13
};

/* Text for a status code (static storage). */
const char* pcf_status_string(pcf_status s);

/* ceil(pct * span_len / 100) in integer arithmetic; -1 for pct < 0 or span_len < 0. */
int32_t pcf_k_from_percent(int32_t pct, int32_t span_len);

/* Host-only.  Fills table[max_pos][head_dim/2][2] (caller-owned, host memory) with
 * (cos, sin)(p * theta^(-2i/d)) computed in fp64 and rounded to fp32 (MiniPIC 2.1, "cos/sin table
 * lookup").  The caller copies it to the device.  Errors: null table, head_dim not in {64,128},
 * theta <= 0, max_pos < 16 or > 1<<20. */
pcf_status pcf_rope_table_init(float* table, int32_t head_dim, double theta, int32_t max_pos);

/* Host-only.  Number of int32 words of the layout blob for this batch (validates like build). */
pcf_status pcf_layout_words(const pcf_request_desc* reqs, int32_t n_reqs, const pcf_dims* dims,
                            int64_t* n_words);

/* Host-only.  Validates the batch and writes the layout blob (MiniPIC section 1 "concurrency
 * barrier" and section 2.1: per-request logical positions over shared physical pages; section 2.2
 * "Padding": spans start on page boundaries): per request, the block table
 * (logical page -> physical page), the logical position of every page's first token, span
 * records, row/selection offsets and the kernels' work lists.  Errors (PCF_ERR_INVALID_ARG):
 * null pointers, n_reqs < 1, a span outside the pool or with n_pages < 1, positions not strictly
 * increasing inside a request, query_pos0 before the end of the last span, any position >=
 * max_pos, k outside [0, 16*n_pages], n_query < 0, n_words too small.  PCF_ERR_UNSUPPORTED for
 * head_dim not in {64,128} or Hq/Hkv not dividing 128. */
pcf_status pcf_layout_build(const pcf_request_desc* reqs, int32_t n_reqs, const pcf_dims* dims,
                            int32_t* blob, int64_t n_words);

/* Host-only.  Reads one PCF_L_* header word of a built blob into *value. */
pcf_status pcf_layout_query(const int32_t* blob, int32_t field, int64_t* value);

/* Bytes of device workspace pcf_score needs for this layout. */
pcf_status pcf_score_workspace_bytes(const int32_t* layout_host, size_t* bytes);

/* Critical-layer scoring (QCFuse 2B; MiniPIC 2.1 score equation).  For every request b and every
 * cached token j of b:
 *   importance[tok_base_b + j] = sum_{h < Hq} sum_{t < T_b}
 *       softmax_j( (R_{pos(t)} q_{t,h}) . (R_{pi(j)} k~_{j, h/g}) / sqrt(d) )
 * with the softmax over all cached tokens of request b.  Output fp32 [total_tokens].
 * ws: device workspace of >= pcf_score_workspace_bytes bytes, contents need not be initialised
 * (PCF_ERR_WORKSPACE_TOO_SMALL otherwise).  Deterministic (fixed summation order). */
pcf_status pcf_score(const pcf_layout* layout, const uint16_t* q_query, const uint16_t* k_pool,
                     const float* rope, float* importance, void* ws, size_t ws_bytes, void* stream);

/* Importance at every layer instead of one critical layer (QCFuse section 4 "Resultados": the
 * all-layer method QCAll the critical layer is compared with; the last layer alone is QCLast).
 * For each layer l: importance_layers[l][:] = pcf_score of layer l's query q_query_layers[l] over
 * layer l's key pool k_pool_layers[l] (same layout, positions and rope table at every layer);
 * then importance_sum[j] = sum over l of importance_layers[l][j], added in layer order in fp32
 * (the pages name no rule for combining layers; the sum ranks tokens like the mean).
 * q_query_layers / k_pool_layers: host arrays of n_layers (1 .. 4096) device pointers, each laid
 * out as for pcf_score; importance_layers [n_layers][total_tokens] and importance_sum
 * [total_tokens] fp32, device, 16-byte aligned.  ws: the scoring workspace
 * (pcf_score_workspace_bytes), reused layer after layer on `stream`.  Deterministic. */
pcf_status pcf_score_layers(const pcf_layout* layout, int32_t n_layers, const uint16_t* const* q_query_layers,
                            const uint16_t* const* k_pool_layers, const float* rope, float* importance_layers,
                            float* importance_sum, void* ws, size_t ws_bytes, void* stream);

/* Bytes of device workspace pcf_score_paged needs: the rotated query rows, the row LSE and
 * importance partials and counters -- no copy of the cached keys. */
pcf_status pcf_score_paged_workspace_bytes(const int32_t* layout_host, size_t* bytes);

/* The same scoring as pcf_score (same arguments and result within the same tolerance), without any
 * copy of the cached keys: both passes copy each key tile from its pool pages (through the block
 * table) and rotate it in shared memory to the request's positions before the tensor-core
 * contraction (MiniPIC 2.1).  ws: >= pcf_score_paged_workspace_bytes.  The rotation is repeated for
 * every query-tile pair (row LSE) and every pair of 256-row query chunks (importance) that reads a
 * tile, so this takes longer than pcf_score;
 * with pcf_fused_attention_paged it completes a hot path that keeps no per-request copy of the
 * cached keys or values. */
pcf_status pcf_score_paged(const pcf_layout* layout, const uint16_t* q_query, const uint16_t* k_pool,
                           const float* rope, float* importance, void* ws, size_t ws_bytes, void* stream);

/* Per-span Top-k (QCFuse 2B "Top-N tokens", taken per span).  For every span s of request b:
 * the k_s request-local token indices with the largest importance, ties to the lower index,
 * written in ascending order to sel_idx[sel_base_b + offset of s ...].  Also writes
 *   excl[page]     uint16 per logical page (global page index = tok_base_b/16 + page): bit r set
 *                  iff token 16*page + r of that request is recomputed;
 *   row_pos[row]   logical position of every row: the selected tokens' pi(j), then
 *                  query_pos0 + t for the query rows.
 * Comparison is on the fp32 bit patterns (values must not be NaN); bit-exact and deterministic. */
pcf_status pcf_select_topk(const pcf_layout* layout, const float* importance, int32_t* sel_idx,
                           uint16_t* excl, int32_t* row_pos, void* stream);

/* Global Top-N (QCFuse 2B read literally: one selection over all of a request's cached tokens).
 * For every request b: the N_b = sum over its spans of k_s request-local token indices with the
 * largest importance over the whole request, ties to the lower index, in ascending order at
 * sel_idx[sel_base_b ...]; excl and row_pos as for pcf_select_topk.  The budget per request,
 * hence every row count and buffer size, is that of the per-span selection: only where the N_b
 * tokens fall differs.  Bit-exact and deterministic; one block per request (its cached tokens
 * must fit a 48 KB bitmap: at most 393216 of them, else PCF_ERR_UNSUPPORTED). */
pcf_status pcf_select_topn_global(const pcf_layout* layout, const float* importance, int32_t* sel_idx,
                                  uint16_t* excl, int32_t* row_pos, void* stream);

/* Anchor key norms (QCFuse 2A / Phase 1, anchor extraction): norms[t] for every cached token t
 * of the layout (same order as importance) = Euclidean norm of its unrotated key over all Hkv
 * heads and d dimensions, fp32 accumulation of the bf16 squares.  A span's anchors are then its
 * tokens with the largest norms: pcf_select_topk on a layout whose span k's are the anchor
 * counts, fed these norms as the importance.  k_pool as for pcf_score (16-byte aligned). */
pcf_status pcf_key_norms(const pcf_layout* layout, const uint16_t* k_pool, float* norms, void* stream);

/* Anchor pages (QCFuse 2A injection / Phase 2): `layout` is an anchor-selection layout (span k's =
 * anchor counts, every one a multiple of 16, else PCF_ERR_INVALID_ARG) and sel_idx its selection
 * (pcf_select_topk on pcf_key_norms).  Copies anchor i of the batch (selection order) to page
 * i / 16, row i % 16 of k_anchor / v_anchor, [total_sel / 16][Hkv][16][d] bf16, every kv head.
 * The query then attends over them as a prefix with pcf_fused_attention on a second layout whose
 * request b has one span (phys_first_page = sel_base_b / 16, n_pages = anchors_b / 16, pos0 = 0,
 * k = 0) and its query at query_pos0 = anchors_b, pools k_anchor / v_anchor. */
pcf_status pcf_pack_anchor_pages(const pcf_layout* layout, const int32_t* sel_idx, const uint16_t* k_pool,
                                 const uint16_t* v_pool, uint16_t* k_anchor, uint16_t* v_anchor, void* stream);

/* Layer-pipelined pool prefetch (QCFuse 2C / Phase 4: while layer i is reconstructed, layer i+1's
 * cache is loaded; here from host memory, the SSD tier being out of scope).  Copies every physical
 * page the layout's spans reference, each once (spans shared by several requests, or touching,
 * merge into one run), from src_k / src_v to the same page offsets of dst_k / dst_v: one
 * cudaMemcpyAsync per run and pool, queued on `stream` (host sources should be pinned for the
 * copies to overlap kernels).  Pools as for pcf_score, [n_phys][Hkv][16][d] bf16; src_v and dst_v
 * may both be NULL (K only, as the critical-layer scoring needs).  Pages the layout does not
 * reference are not touched. */
pcf_status pcf_prefetch_pool_pages(const pcf_layout* layout, const uint16_t* src_k, const uint16_t* src_v,
                                   uint16_t* dst_k, uint16_t* dst_v, void* stream);

/* Row gather of the recompute batch (QCFuse Phase 4, second summary: the Top-N tokens are recomputed
 * discretely, so their inputs are collected into one dense batch):
 * dst[sel_base_b + i][:] = src[tok_base_b + sel_idx[...]][:]
 * for every selected row; src [total_tokens][row_elems], dst [total_sel][row_elems], bf16;
 * row_elems a positive multiple of 8. */
pcf_status pcf_gather_rows(const pcf_layout* layout, const int32_t* sel_idx, const uint16_t* src,
                           int32_t row_elems, uint16_t* dst, void* stream);

/* Bytes of device workspace pcf_fused_attention needs for this layout. */
pcf_status pcf_attention_workspace_bytes(const int32_t* layout_host, size_t* bytes);

/* Fused prefill attention over the merged cached + fresh KV (QCFuse 2C, Phase 4; MiniPIC 2.1).
 * For each row r of request b (its recomputed tokens then its query tokens) and q head h:
 *   out[r][h] = sum_u softmax_u(s_u) v_u,  s_u = (R_{pos(r)} q_{r,h}) . (R_{pos(u)} k_u) / sqrt(d)
 * over keys u = the cached tokens of b whose excl bit is clear, at pi(j), plus the fresh rows of
 * b at row_pos; u is visible iff pos(u) <= row_pos[r].  The pool stays unrotated and is never
 * written: the cached keys that take part are read from their pages through the block table and
 * rotated to the request's positions by a pass of this call (into ws, with their V rows beside
 * them), which the attention kernel then streams.  ws: >= pcf_attention_workspace_bytes bytes. */
pcf_status pcf_fused_attention(const pcf_layout* layout, const uint16_t* q_fresh,
                               const uint16_t* k_fresh, const uint16_t* v_fresh,
                               const uint16_t* k_pool, const uint16_t* v_pool,
                               const uint16_t* excl, const int32_t* row_pos, const float* rope,
                               uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* Bytes of device workspace pcf_fused_attention_paged needs for this layout: the rotated fresh rows
 * (Q and K), per-page counters and the split-merge partials -- it grows with the batch's rows, not
 * with its cached tokens. */
pcf_status pcf_attention_paged_workspace_bytes(const int32_t* layout_host, size_t* bytes);

/* The same fused attention as pcf_fused_attention (same arguments, result within the same
 * tolerances, same errors), computed without any copy of the cached keys or values (MiniPIC 2.1,
 * "Implementation": the cos/sin lookup and fused multiply-adds sit in the attention kernel;
 * "Benefit": one block serves concurrent requests at different offsets without duplication).
 * The kernel copies each cached tile's pool pages (through the block table) straight into shared
 * memory, rotates the keys there to the request's positions before the tensor-core contraction,
 * and writes each recomputed token's fresh key and value over its stale cached copy in place.
 * ws: >= pcf_attention_paged_workspace_bytes bytes (rotated fresh rows and split partials only),
 * against pcf_attention_workspace_bytes, which also holds a rotated copy of the batch's kept
 * cached keys with their values.  The rotation runs on the SMs' arithmetic units beside the
 * softmax, once per tile and query-tile pair, so the kernel takes about twice as long as the one
 * behind pcf_fused_attention on GB300; it is meant for callers whose device memory cannot hold
 * the per-request copy. */
pcf_status pcf_fused_attention_paged(const pcf_layout* layout, const uint16_t* q_fresh, const uint16_t* k_fresh,
                                     const uint16_t* v_fresh, const uint16_t* k_pool, const uint16_t* v_pool,
                                     const uint16_t* excl, const int32_t* row_pos, const float* rope,
                                     uint16_t* out, void* ws, size_t ws_bytes, void* stream);

/* pcf_fused_attention (paged == 0) or pcf_fused_attention_paged (paged != 0, ws sized by
 * pcf_attention_paged_workspace_bytes) with two caller-created CUDA events (cudaEvent_t, non-NULL,
 * else PCF_ERR_INVALID_ARG) recorded on `stream` right before and right after the attention
 * kernel's launch, for timing that kernel alone (its cudaEventElapsedTime).  An event between two
 * kernels ends their programmatic launch overlap, so a timed call runs slightly slower than an
 * untimed one. */
pcf_status pcf_fused_attention_timed(const pcf_layout* layout, const uint16_t* q_fresh, const uint16_t* k_fresh,
                                     const uint16_t* v_fresh, const uint16_t* k_pool, const uint16_t* v_pool,
                                     const uint16_t* excl, const int32_t* row_pos, const float* rope, uint16_t* out,
                                     void* ws, size_t ws_bytes, void* ev_kernel_start, void* ev_kernel_stop,
                                     int32_t paged, void* stream);

/* Largest scoring workspace pcf_score_noalloc can serve (16 MiB), i.e. the size of the scratch
 * array built into the library. */
#define PCF_SCORE_NOALLOC_MAX_WORKSPACE ((size_t)16 << 20)

/* pcf_score without a caller workspace and without allocating anything.  (The paper has no
 * counterpart: this is an integration aid.)  Same inputs, outputs, result and errors as pcf_score,
 * but its scratch lives in a fixed array of PCF_SCORE_NOALLOC_MAX_WORKSPACE bytes compiled into
 * the library, which every GPU that loads the library keeps until the process exits.
 *   Who needs it: callers that may not call cudaMalloc or any allocating routine on this path --
 *   e.g. a host engine whose memory pool has reserved all device memory up front, code running
 *   under a strict real-time or fixed-memory budget, or plugin hosts whose allocator is not
 *   reachable from the library.
 *   Limit: a batch whose pcf_score_workspace_bytes exceeds the array size is rejected with
 *   PCF_ERR_WORKSPACE_TOO_SMALL before any work is queued.
 *   Set-up: the first call on each device (and again after that device's context was reset)
 *   looks up the array's device address, with that device current; make that first call before
 *   any stream capture.
 *   Sharing: every call on a device uses the same array, which keeps the last call's contents
 *   (the call clears what must start at zero itself).  Calls that overlap on the GPU -- on
 *   different streams, or from different threads -- race on it and must be serialized by the
 *   caller. */
pcf_status pcf_score_noalloc(const pcf_layout* layout, const uint16_t* q_query, const uint16_t* k_pool,
                             const float* rope, float* importance, void* stream);

/* Synchronizes `stream`, then reads and clears the device error word: PCF_OK,
 * PCF_ERR_DEVICE_TIMEOUT, PCF_ERR_DEVICE_BOUNDS or PCF_ERR_DEVICE_RANGE (the first error raised
 * since the last check; PCF_ERR_CUDA if the sync itself failed).  The rotated queries and keys
 * enter the tensor cores as fp16: a value whose magnitude rounds above 65504 (inputs far outside
 * the usual activation range) raises PCF_ERR_DEVICE_RANGE instead of being clamped silently, and
 * the results of that call must be discarded. */
pcf_status pcf_check_device_error(void* stream);

/* Check of the failure-detection path (the pages have no counterpart: a library self-test).
 * Every wait of the library's kernels is bounded; when one runs out, the kernel raises an abort
 * flag and the device error word, drains what it has in flight and returns.  This call launches a
 * one-thread-block kernel whose only work is such a wait, with a limit of `limit_cycles` GPU clock
 * cycles (1000 .. 2e8, about 0.1 s at most), on a barrier that nothing ever arrives on.  The wait
 * gives up, so flag[0] (device int32) becomes 1 and the next pcf_check_device_error returns
 * PCF_ERR_DEVICE_TIMEOUT; the device stays usable.  flag[0] == 2 would mean the wait returned
 * without its arrival.  Errors: PCF_ERR_INVALID_ARG for a limit out of range or a null or
 * misaligned flag; PCF_ERR_NO_DEVICE. */
pcf_status pcf_wait_limit_check(int64_t limit_cycles, int32_t* flag, void* stream);

/* Queues `n` asynchronous copies on `stream`, in order: copy i moves bytes[i] bytes from src[i]
 * to dst[i] with one cudaMemcpyAsync of kind cudaMemcpyDefault (the direction follows from the
 * pointers: device memory or page-locked host memory).  Used by the pipelined host-input step to
 * move a step's inputs and results in one call; the arrays are read before the call returns, the
 * buffers must stay valid until the copies have run.  n == 0 queues nothing.
 * Errors: PCF_ERR_INVALID_ARG if n < 0, or n > 0 and an array is null (nothing queued);
 * PCF_ERR_NO_DEVICE without a usable device; PCF_ERR_CUDA if a copy fails to queue (the copies
 * before it stay queued). */
pcf_status pcf_copy_async(int32_t n, void* const* dst, const void* const* src, const size_t* bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PCF_H */
