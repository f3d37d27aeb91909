/*
 * sel.h -- C ABI of libsel: sparse-attention token selection over a paged KV cache
 * on one GB300 (sm_103a).
 *
 * For each query row of a decode or prefill batch the library scores the row's
 * request's compressed pool keys, keeps the best index_topk / kpool pools, expands
 * them to tokens (plus the trailing incomplete pool), and remaps the tokens through
 * the request's block table to physical KV-cache slots with a per-row valid count.
 *
 * Sources for the operation (vLLM documentation pages and a vLLM-fork pull request):
 *  - "sparse_utils" page, triton_convert_req_index_to_global_index: the remap
 *    slot = block_table[req, t / block_size] * block_stride_rows + t % block_size,
 *    -1 for t == -1 or an out-of-bounds block, valid counts in the same pass;
 *    flat_kv_row_view: block_stride_rows > block_size when other layers' pages sit
 *    between blocks; _remap_tiling: counting without atomics.
 *  - ReVolta PR #59 ("Change"): the request-segmented scorer -- 64-key tiles of the
 *    compressed key cache reached through a per-request page table, loaded once per
 *    segment of rows of one request, 4 heads x 128 dims in fp16, int32 metadata,
 *    segment descriptors built on the device so the call is CUDA-graph safe; the
 *    selection keeps the top-512 pools (index_topk 2048 / kpool 4).
 *  - "flash_maxsim_rerank" page: the MaxSim rerank of a query against documents
 *    packed in one tensor (sel_maxsim_rerank), a second workload on the same
 *    segmented tensor-core scoring.
 *  - "flashinfer_mla_sparse_sm90" page, _kv_lens_host: a row's context is
 *    position + 1; contexts up to index_topk select every token, longer ones keep
 *    index_topk pool-expanded tokens plus the trailing incomplete pool, so the valid
 *    count is ctx if ctx <= index_topk else index_topk + ctx % kpool.
 *
 * Conventions for every entry point:
 *  - All array arguments are DEVICE pointers unless stated otherwise, owned by the
 *    caller, and must stay valid until the work queued on `stream` has finished.
 *    The library allocates no memory; apart from the fixed scratch array of
 *    sel_select_static it keeps no device state between calls.
 *  - Work is queued on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *    No entry point synchronises the device or reads device memory on the host, so
 *    the device entry points can be captured into a CUDA graph. Values baked into a
 *    graph at capture: every pointer, every size in sel_problem, and the key-cache
 *    and query base addresses (they are encoded into TMA descriptors).
 *  - Return value: SEL_OK (0) or a negative SEL_E* code; sel_error_string() gives
 *    a message. On an error nothing has been queued unless the code is SEL_ECUDA.
 *  - Data errors found on the device never trap: they set bits in an optional
 *    device status word (bitwise OR, see SEL_ST_*) and the affected outputs are -1.
 *    The status word is never cleared by the library.
 *  - Sentinel: -1 marks an empty output entry or an out-of-bounds slot.
 */
#ifndef SEL_H
#define SEL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *sel_stream_t; /* same type as cudaStream_t */

/* return codes */
#define SEL_OK 0
#define SEL_EINVAL (-1)        /* a null pointer, a negative size, an inconsistent size */
#define SEL_EUNSUPPORTED (-2)  /* a shape or alignment this build does not implement */
#define SEL_ECUDA (-3)         /* a CUDA call failed (launch or driver entry point) */
#define SEL_EWORKSPACE (-4)    /* the workspace is smaller than the *_workspace_bytes query */

/* device status bits (OR-ed into the optional int32 status word) */
#define SEL_ST_KEYPAGE_OOB 1u     /* a key page id outside [0, num_key_pages): those pools score -inf */
#define SEL_ST_CTX_OVER_BOUND 2u  /* a row's context exceeds max_context: the row is all -1, count 0 */
#define SEL_ST_TIMEOUT 4u         /* a bounded wait inside a kernel expired: outputs are incomplete */
#define SEL_ST_BAD_QSL 8u         /* query_start_loc not non-decreasing within [0, num_rows]: all rows -1 */

/*
 * One selection problem. Host struct, read during the call only.
 *
 * Rows: query rows are grouped by request; request i owns rows
 * [query_start_loc[i], query_start_loc[i+1]). Rows at or past
 * query_start_loc[num_reqs] (up to num_rows) are padding (e.g. CUDA-graph padding):
 * their outputs are all -1 with a count of 0. Row r's context is positions[r] + 1.
 *
 * Compressed keys: pool j of request i (the keys of tokens j*kpool .. j*kpool+kpool-1)
 * is row j % 64 of physical key page key_page_table[i * kpt_ld + j / 64]; a key page
 * is 64 rows x 128 fp16 values, row-major, and physical page p starts at element
 * p * key_page_stride of key_cache. Only complete pools (j < ctx / kpool) are read.
 *
 * KV blocks: token t of request i sits in row
 * block_table[i * bt_ld + t / block_size] * block_stride_rows + t % block_size of the
 * flat KV cache (which the library never touches).
 */
typedef struct sel_problem {
    int32_t num_reqs;              /* >= 0 */
    int32_t num_rows;              /* rows in the batch (>= query_start_loc[num_reqs]) */
    int32_t max_context;           /* host upper bound on every row's context (sizes grids) */
    int32_t max_q_len;             /* host hint: most rows any request has (0 = unknown) */
    int32_t num_heads;             /* must be 4 */
    int32_t head_dim;              /* must be 128 */
    int32_t index_topk;            /* tokens kept per row (2048 in the workloads), multiple of kpool */
    int32_t kpool;                 /* tokens per compressed key (4 in the workloads), >= 1 */
    int32_t key_page_size;         /* keys per key page: must be 64 */
    int32_t block_size;            /* tokens per KV block (64 in the workloads), >= 1 */
    int64_t block_stride_rows;     /* physical rows between consecutive KV blocks, >= block_size */
    int64_t key_page_stride;       /* fp16 elements between physical key pages, >= 64*128, multiple of 8 */
    int32_t num_key_pages;         /* physical key pages addressable through key_cache */
    int32_t num_kv_blocks;         /* physical KV blocks: ids outside [0, num_kv_blocks) map to -1 */
    int32_t max_key_pages_per_req; /* valid columns of key_page_table (<= kpt_ld) */
    int32_t max_blocks_per_req;    /* valid columns of block_table (<= bt_ld); later blocks map to -1 */
    int64_t kpt_ld;                /* row stride of key_page_table, in elements */
    int64_t bt_ld;                 /* row stride of block_table, in elements */
    int64_t q_row_stride;          /* fp16 elements between query rows (>= 512, multiple of 8) */
    int32_t segment_rows;          /* rows of one request scored together (1..64; 0 = automatic) */
    int32_t chunk_rows;            /* rows per score-workspace chunk (0: the library's choice,
                                      four times the SM count, capped so one chunk's fp32
                                      scores at max_context fill at most 3/4 of L2, >= 256) */
    const int32_t *query_start_loc; /* [num_reqs + 1] */
    const int32_t *positions;       /* [num_rows] */
    const void *q;                  /* fp16 [num_rows][4][128] with row stride q_row_stride; 16-B aligned */
    const void *key_cache;          /* fp16 key pages; 16-B aligned */
    const int32_t *key_page_table;  /* [num_reqs][kpt_ld] */
    const int32_t *block_table;     /* [num_reqs][bt_ld] */
} sel_problem;

/* Message for a return code (static storage). */
const char *sel_error_string(int code);

/* ABI version of this header (major * 100 + minor): 102. */
int sel_version(void);

/* Workspace (device bytes, 256-B aligned base) needed by sel_select / sel_score_paged
 * for problem p. Returns 0 if p is invalid. */
size_t sel_workspace_bytes(const sel_problem *p);
size_t sel_score_workspace_bytes(const sel_problem *p);

/*
 * sel_score_paged -- the scoring step alone (ReVolta PR #59, "Change": the request-segmented
 * scorer; rows of one request share the request's key page table and each 64-key page is
 * read once per segment of rows; FP16 queries and keys, 4 heads x 128 dims).
 * scores[r * scores_ld + j] = sum_{h<4} sum_{d<128} q[r][h][d] * key(j)[d]  (fp32)
 * for every row r of a request and every complete pool j < (positions[r] + 1) / kpool
 * (and j < scores_ld); -inf when pool j's key page id is out of range. Other
 * entries are left untouched. Rows past query_start_loc[num_reqs] are skipped.
 * scores: device fp32 [num_rows][scores_ld], scores_ld >= 1.
 * Accumulation is fp32 on the tensor cores in an order of the hardware's choosing
 * (exact for integer-valued inputs whose dot products stay below 2^24).
 * status: optional device int32 word (see SEL_ST_*). ws: 16-B aligned workspace of at
 * least sel_score_workspace_bytes(p) bytes (no initialisation needed).
 */
int sel_score_paged(const sel_problem *p, float *scores, int64_t scores_ld, int32_t *status,
                    void *ws, size_t ws_bytes, sel_stream_t stream);

/*
 * sel_topk_expand -- top-k pools, expansion and trailing pool on given scores (ReVolta
 * PR #59, "Change": the top-512 pools of index_topk 2048 / kpool 4; the
 * "flashinfer_mla_sparse_sm90" page, _kv_lens_host: contexts up to index_topk keep every
 * token, longer ones index_topk pool-expanded tokens plus the trailing incomplete pool).
 * For each row r < num_rows with ctx = positions[r] + 1:
 *   ctx <= 0:          no tokens;
 *   ctx <= index_topk: tokens 0 .. ctx-1;
 *   otherwise:         the K = index_topk / kpool pools of scores[r][0 .. ctx/kpool)
 *                      that are best under (score descending, pool index ascending),
 *                      each expanded to its kpool tokens, then the trailing tokens
 *                      (ctx/kpool)*kpool .. ctx-1.
 * token_idx[r * out_width + c] lists the tokens in ascending order, then -1.
 * valid_counts[r] (optional) = number of tokens. A row whose ctx / kpool exceeds
 * scores_ld is out of bound: all -1, count 0, SEL_ST_CTX_OVER_BOUND.
 * Scores must be finite or -inf; -0.0 ranks equal to +0.0.
 * Requires out_width >= index_topk + kpool - 1 and out_width % 4 == 0, scores_ld % 4 == 0.
 */
int sel_topk_expand(const float *scores, int64_t scores_ld, const int32_t *positions,
                    int32_t num_rows, int32_t index_topk, int32_t kpool, int32_t *token_idx,
                    int32_t out_width, int32_t *valid_counts, int32_t *status,
                    sel_stream_t stream);

/*
 * sel_remap_global -- token indices to physical KV slots (the sparse_utils remap).
 * For row r with request q = req_id[r] and each column c < width, t = token_idx[r*width + c]:
 *   slots[r*width + c] = -1 if t < 0, q outside [0, num_reqs), t / block_size >=
 *   max_blocks_per_req, or the physical block b = block_table[q*bt_ld + t/block_size]
 *   is outside [0, num_kv_blocks); else b * block_stride_rows + t % block_size.
 * valid_counts[r] (optional) = number of entries that are not -1, reduced in
 * registers (no atomics, no zero-initialised counter). Columns keep their positions.
 * Requires width % 4 == 0 and 16-B aligned token_idx / slots (int4 vector access),
 * and (num_kv_blocks - 1) * block_stride_rows + block_size <= INT32_MAX.
 */
int sel_remap_global(const int32_t *req_id, int32_t num_reqs, const int32_t *block_table,
                     int64_t bt_ld, int32_t max_blocks_per_req, int32_t num_kv_blocks,
                     const int32_t *token_idx, int32_t num_rows, int32_t width,
                     int32_t block_size, int64_t block_stride_rows, int32_t *slots,
                     int32_t *valid_counts, sel_stream_t stream);

/*
 * sel_remap_workspace -- the remap with a prefill workspace (the sparse_utils page,
 * triton_convert_req_index_to_global_index with HAS_PREFILL_WORKSPACE: prefill tokens
 * map to workspace offsets instead of global cache slots).
 * ws_req [num_rows]: -1 for a decode row, which takes sel_remap_global's formula, else the
 * row's prefill request w, whose tokens start at ws_starts[w] (ws_starts [num_prefills],
 * 0-indexed). A prefill row writes ws_starts[w] + t for every t >= 0 and -1 for t == -1
 * (reading: the page names the mapping but prints no formula; the plainest one is taken);
 * a w outside [-1, num_prefills) gives an all -1 row. ws_starts[w] + t must fit in int32.
 * valid_counts, columns and the other arguments as in sel_remap_global.
 */
int sel_remap_workspace(const int32_t *req_id, int32_t num_reqs, const int32_t *block_table,
                        int64_t bt_ld, int32_t max_blocks_per_req, int32_t num_kv_blocks,
                        const int32_t *ws_req, const int32_t *ws_starts, int32_t num_prefills,
                        const int32_t *token_idx, int32_t num_rows, int32_t width,
                        int32_t block_size, int64_t block_stride_rows, int32_t *slots,
                        int32_t *valid_counts, sel_stream_t stream);

/*
 * sel_remap_dcp -- one decode-context-parallel rank's slots (the sparse_utils page,
 * triton_filter_and_convert_dcp_index: filter global per-request indices to this rank's
 * local slots; non-owned slots are -1; optionally compacted to a contiguous prefix).
 * Tokens are dealt to the dcp_size ranks in groups of `interleave` consecutive tokens,
 * round robin (reading: the page does not print the formula): token t belongs to rank
 * (t / interleave) % dcp_size at local index (t / (interleave * dcp_size)) * interleave +
 * t % interleave. An owned token's slot is block_table[q * bt_ld + l / block_size] *
 * block_size + l % block_size for its local index l (this rank's dense cache), with the
 * -1 guards of sel_remap_global; tokens of other ranks are -1. compact != 0 moves the
 * row's non -1 slots, in ascending column order, to columns 0 .. count-1 and writes -1 to
 * the rest (the page leaves the prefix order unspecified; no atomics are used here).
 * valid_counts[r] (optional) = number of non -1 slots. Requires 1 <= dcp_size,
 * 0 <= dcp_rank < dcp_size, interleave >= 1 and block_size % interleave == 0 (an
 * interleave group never straddles a block), plus sel_remap_global's requirements.
 */
int sel_remap_dcp(const int32_t *req_id, int32_t num_reqs, const int32_t *block_table,
                  int64_t bt_ld, int32_t max_blocks_per_req, int32_t num_kv_blocks,
                  const int32_t *token_idx, int32_t num_rows, int32_t width, int32_t block_size,
                  int32_t dcp_size, int32_t dcp_rank, int32_t interleave, int32_t compact,
                  int32_t *slots, int32_t *valid_counts, sel_stream_t stream);

/*
 * sel_maxsim_rerank -- MaxSim scores of one query against documents packed in one tensor
 * (vLLM page "flash_maxsim_rerank", _maxsim_rerank_kernel / flash_maxsim_rerank_direct).
 *   q [lq][q_stride] fp16: the query's token embeddings, d used columns per row.
 *   docs [total_tokens][doc_stride] fp16: the packed tensor; document b is rows
 *     doc_offsets[b] .. doc_offsets[b] + doc_lengths[b] - 1 (int32 [num_docs] each; documents
 *     may be scattered, out of order or overlapping; read in place, never copied).
 *   scores [num_docs] fp32 (written): score[b] = sum_{a<lq} max_{j<len_b} q[a] . docs[off_b+j],
 *     each dot product on the tensor cores with fp32 accumulation.
 * The page's masking decides the degenerate cases: a document with doc_lengths[b] <= 0
 * scores -inf; lq == 0 gives 0 for every document (q and docs may then be NULL);
 * num_docs == 0 queues nothing. Rows outside [0, total_tokens) read as zero vectors (no
 * fault; outside the page's contract).
 * Requires 1 <= d <= 1024, q_stride and doc_stride >= d and multiples of 8, q and docs
 * 16-B aligned, total_tokens <= INT32_MAX - 64, and a 4-B aligned device workspace of
 * sel_maxsim_workspace_bytes() bytes, ZERO-FILLED before its first use: it holds the
 * kernel's work counters, and every launch leaves them zero again when it finishes (also
 * after a timeout), so a workspace kept for this entry point needs zeroing only once.
 * Calls sharing one workspace must not overlap on the GPU. Queues one kernel per block of
 * up to 128 query rows (64 for d > 256, 32 for d > 512); later blocks add to scores.
 * status (optional): SEL_ST_TIMEOUT if a bounded wait expired.
 */
size_t sel_maxsim_workspace_bytes(void);
int sel_maxsim_rerank(const void *q, int32_t lq, int32_t d, int64_t q_stride, const void *docs,
                      int64_t total_tokens, int64_t doc_stride, const int32_t *doc_offsets,
                      const int32_t *doc_lengths, int32_t num_docs, float *scores, int32_t *status,
                      void *ws, size_t ws_bytes, sel_stream_t stream);
/* Kernel launches one sel_maxsim_rerank call with this lq and d queues. */
int32_t sel_maxsim_launch_count(int32_t lq, int32_t d);

/*
 * sel_mla_decode -- sparse MLA decode attention over the selected slots (vLLM page
 * "flashinfer_mla_sparse_sm90", _SM90State: the MLA wrapper planned with page size 1, so the
 * selection's slots are the page table, and the exact kv_len of _kv_lens_host). For row r,
 * head h and each entry j < kv_len[r] whose slot s = slots[r][j] lies in [0, num_slots):
 *     logit_j = sm_scale * (q_nope[r][h] . ckv[s] + q_pe[r][h] . kpe[s])
 *     out[r][h] = sum_j softmax(logit)_j * ckv[s_j]      lse[r][h] = ln sum_j exp(logit_j)
 * A -1 or out-of-range slot inside kv_len contributes nothing; entries past kv_len (the -1
 * tail) are never read, nor is the cache row of a bad slot. A row with no such entry gives
 * out = 0 and lse = -inf. kv_len above width counts as width.
 *   q_nope bf16 (uint16 bit patterns) [rows][heads][dc] at qn_row_stride / qn_head_stride
 *     elements; q_pe bf16 [rows][heads][dr] likewise (unused when dr == 0, may be NULL);
 *   ckv bf16: slot s's dc latent dims at s * ckv_stride; kpe bf16: its dr rotary dims at
 *     s * kpe_stride (kpe may alias ckv + dc: one cache row of dc + dr);
 *   slots int32 [rows][width], kv_len int32 [rows];
 *   out fp32 [rows][heads][dc] and lse fp32 [rows][heads] (written, contiguous).
 * Scores and products run on the tensor cores with bf16 operands and fp32 accumulation; the
 * softmax weights enter the second product rounded to bf16 (and are normalised by the sum of
 * the rounded weights), the log-sum-exp uses the unrounded fp32 weights.
 * Requires heads == 16, dc == 512, dr in {0, 64}, 1 <= width <= 8192, num_slots <= INT32_MAX,
 * strides multiples of 8 elements, q_nope / q_pe / ckv / kpe / out 16-B aligned, and a 16-B aligned
 * device workspace of sel_mla_workspace_bytes(rows, width) bytes (needs no initialisation;
 * calls sharing one must not overlap on the GPU). Queues two kernels (sel_mla_launch_count).
 * status (optional): SEL_ST_TIMEOUT if a bounded wait expired.
 */
size_t sel_mla_workspace_bytes(int32_t rows, int32_t width);
int sel_mla_decode(const void *q_nope, int64_t qn_row_stride, int64_t qn_head_stride, const void *q_pe,
                   int64_t qp_row_stride, int64_t qp_head_stride, int32_t rows, int32_t heads, int32_t dc,
                   int32_t dr, const void *ckv, int64_t ckv_stride, const void *kpe, int64_t kpe_stride,
                   int64_t num_slots, const int32_t *slots, int32_t width, const int32_t *kv_len,
                   float sm_scale, float *out, float *lse, int32_t *status, void *ws, size_t ws_bytes,
                   sel_stream_t stream);
int32_t sel_mla_launch_count(int32_t rows);

/*
 * sel_select -- the fused path (ReVolta PR #59, "Change": request segments built on the
 * device, the segmented scorer, the top-512 pools; the "flashinfer_mla_sparse_sm90" page,
 * _kv_lens_host: expansion with the trailing incomplete pool; the "sparse_utils" page,
 * triton_convert_req_index_to_global_index: the remap and the valid counts): segment
 * builder (one launch that plans every chunk of chunk_rows rows), then per chunk the
 * segmented scorer and the top-k with expansion and remap, all queued on `stream`.
 * slots [num_rows][out_width]: the remapped slots of each row's selected tokens in
 * ascending token order, then -1 (an out-of-bounds block gives -1 in place).
 * valid_counts [num_rows]: number of entries of the row that are not -1.
 * token_idx [num_rows][out_width] (optional): the selected token indices.
 * status (optional): device int32 word, see SEL_ST_*.
 * Requires out_width >= index_topk + kpool - 1, out_width % 4 == 0, slots and
 * token_idx 16-B aligned, and a 16-B aligned workspace of sel_workspace_bytes(p) bytes.
 * The workspace (caller-owned device memory) needs no initialisation and carries nothing
 * from one call to the next; calls that share one must not overlap on the GPU.
 */
int sel_select(const sel_problem *p, int32_t *slots, int32_t out_width, int32_t *valid_counts,
               int32_t *token_idx, int32_t *status, void *ws, size_t ws_bytes,
               sel_stream_t stream);

/*
 * sel_select_static -- sel_select without a workspace argument, for callers that cannot
 * allocate device memory per call (a serving engine that has reserved nearly all HBM for
 * its paged KV cache at start-up; a plain C host program with no device allocator). The
 * published method has no counterpart of this entry point.
 * Arguments, layouts, results and the other error codes are those of sel_select. The
 * scratch is one file-scope device array of SEL_STATIC_WS_MAX_BYTES bytes, held by every
 * GPU that loads the library until the process exits (the driver places it when the
 * library's module is loaded on a device; with lazy module loading, at the first call of
 * this entry point there, which therefore adds SEL_STATIC_WS_MAX_BYTES to the device memory
 * in use once); no call allocates or frees device memory. Returns SEL_EWORKSPACE, queueing nothing, when sel_workspace_bytes(p) exceeds
 * SEL_STATIC_WS_MAX_BYTES (a smaller p->chunk_rows lowers that size).
 * Outside stream capture every call looks up the array's address on the current device
 * (so the address stays right after a device reset reloads the module); a call inside a
 * capture uses the address found by the last call on that device outside capture, so make
 * one call on each device before capturing. Every call on a device uses the same array:
 * calls whose work overlaps on the GPU (unordered streams) race and give wrong results.
 * The kernels clear every counter they rely on, so no zeroing is needed between calls.
 */
#define SEL_STATIC_WS_MAX_BYTES (16u << 20)
int sel_select_static(const sel_problem *p, int32_t *slots, int32_t out_width,
                      int32_t *valid_counts, int32_t *token_idx, int32_t *status,
                      sel_stream_t stream);

/*
 * sel_select_host -- sel_select for callers whose per-step inputs and outputs live
 * in HOST memory (ideally pinned). The key cache stays resident on the device
 * (p->key_cache is a device pointer). p's query_start_loc, positions, q,
 * key_page_table and block_table are HOST pointers here; they are copied into the
 * device staging area `stage` (sel_host_stage_bytes(p, out_width) bytes), the
 * selection runs, and slots_host / counts_host (host) receive the results, all
 * asynchronously on `stream`. When every one of these host buffers is pinned and
 * mapped into the device's address space (cudaHostAlloc, cudaHostRegister), one kernel
 * reads all the inputs over the host link and the selection writes slots and counts
 * straight into slots_host / counts_host (one launch per call instead of seven
 * copy-engine transfers); otherwise every buffer is copied by cudaMemcpyAsync. The caller synchronises the stream before reading the
 * outputs. status (optional) is a device word. `stage` and `ws` are device memory, 16-B
 * aligned; ws holds sel_workspace_bytes(p) bytes, as for sel_select.
 */
size_t sel_host_stage_bytes(const sel_problem *p, int32_t out_width);
int sel_select_host(const sel_problem *p, int32_t *slots_host, int32_t out_width,
                    int32_t *counts_host, int32_t *status, void *stage, size_t stage_bytes,
                    void *ws, size_t ws_bytes, sel_stream_t stream);

/*
 * Tracing hook. With n >= 4 events (cudaEvent_t handles, created by the caller with
 * timing enabled), every following sel_select records, on `stream`: events[0] before its
 * segment-builder launch, events[1] after that builder (before the first scorer
 * launch), events[2] after the last scorer launch and events[3] after the last row-select
 * launch (exact top-k, expansion, remap). Inside stream capture the records
 * become external event nodes. n == 0 switches tracing off. Calls to sel_select are
 * serialised while tracing state is read.
 */
int sel_set_trace_events(void *const *events, int32_t n);

/*
 * sel_debug_wait_limit -- failure-detection test hook (the published method has no
 * counterpart). Every later sel_select / sel_score_paged / sel_maxsim_rerank launch gives
 * each of its bounded waits wait_ns nanoseconds (default 1 s) and, with fault_tile >= 0,
 * never loads the data of that work item (the scorer's tile fault_tile; MaxSim's tile
 * fault_tile of each CTA), so the waits on it expire: the launch sets SEL_ST_TIMEOUT, every
 * role of the kernel leaves without touching the missing data, and the work counters of a
 * MaxSim workspace are returned to zero as after any launch. Call with (-1, 1000000000) to
 * restore normal operation. Process-wide and not thread safe: for tests only.
 */
int sel_debug_wait_limit(int32_t fault_tile, int64_t wait_ns);

/* Number of kernel launches sel_select queues for problem p (for launch accounting):
 * one builder, then a scorer and a row select per chunk of chunk_rows rows. */
int32_t sel_select_launch_count(const sel_problem *p);

#ifdef __cplusplus
}
#endif

#endif /* SEL_H */
