// Argument blocks and launchers of the selection kernels. Host and device code both
// include this file; it holds no device code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sel {

// Segment builder: one CTA turns query_start_loc / positions into per-row request
// ids and contexts and a list of request segments (<= seg_rows rows of one request)
// with the exclusive prefix of the 128-pool tiles each must score.
struct BuildArgs {
    const int32_t* qsl;        // [num_reqs + 1]
    const int32_t* positions;  // [num_rows]
    const int32_t* key_page_table;
    int64_t kpt_ld;
    int32_t max_key_pages, num_key_pages;
    int32_t num_reqs, num_rows;
    int32_t row_begin, row_end;  // the rows handled by this launch
    int32_t chunk_rows;          // rows per CTA (one chunk each)
    int64_t plan_stride;         // bytes between consecutive chunks' row_req .. hdr arrays
    int32_t seg_rows;
    int32_t topk, kpool, max_context;
    int32_t score_all;  // 1: score every row's complete pools; 0: only rows with ctx > topk
    int32_t pool_cap;   // no row scores more pools than this (the score row length)
    int32_t max_segs;
    int32_t* row_req;          // [chunk_rows] per chunk
    int32_t* row_ctx;          // [chunk_rows] per chunk; -1 = no output (padding, bad row)
    int4* seg;                 // [max_segs] {req, first row, rows, pools to score}
    int32_t* seg_tile_prefix;  // [max_segs + 1] exclusive prefix of tiles per segment
    int32_t* hdr;              // [0] segments, [1] tiles, [2] scorer's dynamic-tile counter (set to 0)
    int32_t* status;
    // shared-memory staging plan (filled by launch_build)
    int32_t smem_qsl, smem_rows, smem_segs;
    int32_t smem_rows_off, smem_segs_off, smem_prefix_off;
};

// Segmented scorer (TMA + tcgen05): CTAs take static shares of the tiles, then single
// tiles from an atomic counter; each CTA resolves a tile's segment and key pages itself.
// How a scorer launch gets its chunk's plan (segments and tile prefix):
//   kPlanAfterBuilder  it reads the builder's plan after waiting for the builder;
//   kPlanReady         the builder had finished before the preceding grid (the previous chunk's
//                      row select, which reads the score buffer) started: the CTA reads the plan
//                      and fetches its tiles at once, and only its score stores and its draws of
//                      shared tiles wait for the preceding grid;
//   kPlanSelf          every CTA computes the plan itself from query_start_loc and positions (the
//                      builder's rule; small problems only), so it starts fetching tiles while the
//                      builder runs; its epilogue (the builder's row contexts) and its draws of
//                      shared tiles (the builder zeroes their counter) wait for the builder.
constexpr int kPlanAfterBuilder = 0, kPlanReady = 1, kPlanSelf = 2;
constexpr int kSelfPlanMaxReqs = 2048, kSelfPlanMaxRows = 1024;

struct ScoreArgs {
    const int4* seg;
    const int32_t* seg_tile_prefix;  // [segments + 1]
    int32_t* hdr;            // [0] segments, [1] tiles; [2] dynamic-tile counter (zeroed by the builder)
    const int32_t* key_page_table;
    int64_t kpt_ld;
    int32_t max_key_pages, num_key_pages, max_segs;
    const int32_t* row_ctx;  // chunk-local
    int32_t row_begin;
    int32_t topk, kpool, score_all, pool_cap;
    float* scores;           // chunk-local rows
    int64_t scores_ld;
    int32_t as_keys;         // 1: store ordered_key(score) (uint32 bits) instead of the fp32 score
    int32_t plan_mode;       // kPlanAfterBuilder, kPlanReady or kPlanSelf (above)
    // kPlanSelf only: the inputs the chunk's plan is computed from
    const int32_t* qsl;      // [num_reqs + 1]
    const int32_t* positions;
    int32_t num_reqs, num_rows, row_end, seg_rows, max_context;
    int32_t npad_max;        // query lines per q buffer (multiple of 16, <= 256)
    int32_t stages;
    uint32_t tmem_cols;      // TMEM columns allocated (power of two)
    uint32_t acc_cols;       // columns per accumulator buffer
    int32_t* status;
    int32_t fault_tile;      // failure-detection test: this tile's keys are never loaded (-1: none)
    uint64_t wait_ns;        // limit of every bounded wait
};

// Copies between host-mapped and device buffers by a kernel (the host-buffer entry point):
// segment i moves bytes[i] bytes (a multiple of 4, 4-byte aligned ends) from src[i] to dst[i].
constexpr int kStageMaxSegs = 5;
struct StageArgs {
    const void* src[kStageMaxSegs];
    void* dst[kStageMaxSegs];
    int64_t bytes[kStageMaxSegs];
    int32_t nseg;
};
cudaError_t launch_stage_copy(const StageArgs& a, int sms, cudaStream_t s);

// Per-row exact top-k pools, expansion and remap on the scorer's keys (one CTA per row).
struct RowSelectArgs {
    const uint32_t* keys;      // chunk-local rows: ordered_key of every complete pool's score
    int64_t keys_ld;
    const int32_t* row_ctx;    // chunk-local (builder output)
    const int32_t* row_req;    // chunk-local (builder output)
    int32_t stage_cap;         // keys staged in shared memory per row (multiple of 4)
    int32_t bm_words;          // bitmap words per row, >= ceil(max pools / 32)
    int32_t bt_cap;            // block-table entries staged in shared memory per row
    int32_t row_begin;
    int32_t topk, kpool, out_width;
    int32_t kpool_shift;       // log2(kpool) when kpool is a power of two, else -1
    int32_t bs_shift;          // log2(block_size) when block_size is a power of two, else -1
    int32_t* slots;            // [rows][out_width] global rows
    int32_t* token_idx;        // nullable
    int32_t* counts;           // nullable
    const int32_t* block_table;
    int64_t bt_ld;
    int32_t max_blocks, num_kv_blocks, block_size;
    int64_t block_stride_rows;
    int32_t next_chunk;        // 1: another chunk's scorer follows (this grid lets it launch early)
};

// Top-k pools + expansion (+ remap), one CTA per row.
struct TopkArgs {
    const float* scores;       // chunk-local rows
    int64_t scores_ld;
    const int32_t* positions;  // global rows; used when row_ctx is null
    const int32_t* row_ctx;    // chunk-local (builder output) or null
    const int32_t* row_req;    // chunk-local (builder output), needed with remap
    int32_t row_begin;
    int32_t topk, kpool, out_width;
    int64_t max_pools;         // rows with ctx / kpool beyond this are out of bound
    int32_t bt_cap;            // block-table entries staged in shared memory per row
    int32_t* token_idx;        // [rows][out_width] global rows, nullable
    int32_t* slots;            // [rows][out_width] global rows, with remap
    int32_t* counts;           // [rows] global rows, nullable
    const int32_t* block_table;
    int64_t bt_ld;
    int32_t max_blocks, num_kv_blocks, block_size;
    int64_t block_stride_rows;
    int32_t* status;
};

// Stand-alone block-table remap.
struct RemapArgs {
    const int32_t* req_id;
    int32_t num_reqs;
    const int32_t* block_table;
    int64_t bt_ld;
    int32_t max_blocks, num_kv_blocks, block_size;
    int64_t block_stride_rows;
    const int32_t* token_idx;
    int32_t width;
    int32_t* slots;
    int32_t* counts;
    // prefill-workspace mode: ws_req[row] -1 = decode row (global remap), else the row's
    // prefill request, whose tokens map to ws_starts[ws_req[row]] + t
    const int32_t* ws_req;
    const int32_t* ws_starts;
    int32_t num_prefills;
    // decode-context-parallel mode: this rank's tokens only, through its dense block table
    int32_t dcp_size, dcp_rank, interleave, compact;
    // log2 of block_size, interleave and dcp_size when powers of two, else -1 (divisions)
    int32_t bs_shift, il_shift, dcp_shift;
};

enum RemapMode { kRemapGlobal = 0, kRemapWorkspace = 1, kRemapDcp = 2 };

// MaxSim rerank (TMA + tcgen05): one block of up to 128 query rows against documents packed
// in one tensor; CTAs claim documents, the first claim static, the rest through `counter`.
struct MaxsimArgs {
    const int32_t* offsets;  // [num_docs] first row of each document
    const int32_t* lengths;  // [num_docs] rows of each document (<= 0: empty)
    int32_t num_docs;
    int32_t first_claim;     // documents in each CTA's static first claim (1..32)
    int32_t claim_base;      // gridDim.x * first_claim: the first document the counter hands out
    int64_t total_tokens;    // rows of the packed tensor
    float* scores;           // [num_docs]
    int32_t accumulate;      // 1: add to scores (a later block of query rows)
    int32_t q_row0;          // first query row of this block
    int32_t nq;              // valid query rows of this block
    int32_t nq_pad;          // nq rounded up to 32 (<= 128): the query rows held in shared memory
    int32_t kslabs;          // 64-column K slabs (ceil(d / 64))
    int32_t stages;          // K slabs in flight (<= 16)
    uint32_t tmem_cols;      // 256: two 128-column accumulators
    int32_t* counter;        // [2] grab counter and finished-CTA count: zero at the start, zero again at the end
    int32_t* status;
    int32_t fault_tile;      // failure-detection test: each CTA leaves its tile of this index unloaded (-1: none)
    uint64_t wait_ns;        // limit of every bounded wait
};

// Sparse MLA decode attention over selected slots: one launch over all rows' tiles of 64
// entries, each CTA a contiguous run of tiles (a row's tiles may span CTAs), then one merge
// launch that combines the partial results of rows split between CTAs.
struct MlaArgs {
    const uint16_t* q_nope;    // bf16 [rows][16][512] at row / head strides (elements)
    int64_t qn_row, qn_head;
    const uint16_t* q_pe;      // bf16 [rows][16][dr]
    int64_t qp_row, qp_head;
    const uint16_t* ckv;       // bf16, slot s's 512 latent dims at s * ckv_stride
    int64_t ckv_stride;
    const uint16_t* kpe;       // bf16, slot s's dr rotary dims at s * kpe_stride
    int64_t kpe_stride;
    int64_t num_slots;
    const int32_t* slots;      // [rows][width]
    const int32_t* kv_len;     // [rows]
    int32_t width, rows, dr, tiles_per_row;
    int64_t total_tiles;
    float scale_log2;          // sm_scale * log2(e): logits in base-2 units
    float* out;                // fp32 [rows][16][512]
    float* lse;                // fp32 [rows][16], natural logarithm
    uint8_t* part;             // partial results: [2 * grid] slots of kMlaPartBytes
    int32_t* status;
    uint64_t wait_ns;
};
constexpr int kMlaHeads = 16;
constexpr int kMlaDc = 512;
constexpr int kMlaTile = 64;                    // entries per tile
constexpr int kMlaMaxTilesPerRow = 128;         // width <= 8192
constexpr int kMlaThreads = 288;                // warps 0-3 gather, 4 MMA + TMEM, 5-8 softmax
constexpr size_t kMlaPartBytes = 33024;         // O [16][512] fp32, m / l / l_exact [16] fp32
size_t mla_smem_bytes();
cudaError_t launch_mla(const MlaArgs& a, int grid, cudaStream_t s);
cudaError_t launch_mla_merge(const MlaArgs& a, int grid, cudaStream_t s);

constexpr int kBuildThreads = 512;
constexpr int kScoreEpiWarps = 8;    // two per TMEM lane quarter
constexpr int kScoreThreads = 64 + 32 * kScoreEpiWarps;   // warp 0 TMA, warp 1 MMA + TMEM, warps 2-9 epilogue
constexpr int kTopkThreads = 512;
constexpr int kTopkBins = 2048;
constexpr int kTopkListCap = 4096;   // keys at or above the threshold bin listed per row
constexpr int kMaxDevicesTracked = 64;
constexpr int kRemapThreads = 128;
constexpr int kSelectThreads = 1024;    // threads of the row select CTA (512 in its two-per-SM variant)
constexpr int kSelectMaxStage = 32768;  // keys of a row staged in shared memory (128 KiB)
constexpr int kMaxsimThreads = 256;     // warp 1 schedule, 2 MMA + TMEM, 3 TMA, 4-7 epilogue, 0 idle

size_t score_smem_bytes(int stages, int npad_max, int max_segs);
size_t topk_smem_bytes(int bt_cap);

// Launchers. With `pdl` the kernel is a programmatic dependent of the previous kernel
// on the stream: its prologue may overlap that kernel, and it waits (griddepcontrol)
// before reading what that kernel wrote.
cudaError_t launch_build(const BuildArgs& a, bool pdl, cudaStream_t s);
cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_q, int grid,
                         size_t smem, bool pdl, cudaStream_t s);
cudaError_t launch_topk(const TopkArgs& a, bool remap, int rows, size_t smem, bool pdl, cudaStream_t s);
cudaError_t launch_remap(const RemapArgs& a, int rows, RemapMode mode, cudaStream_t s);
size_t select_smem_bytes(int stage_cap, int bm_words, int K, int bt_cap);
// threads: 1024 or 512 (the 512-thread variant is meant to run two CTAs per SM)
cudaError_t launch_select_rows(const RowSelectArgs& a, int rows, size_t smem, bool pdl, cudaStream_t s,
                               int threads);
size_t maxsim_smem_bytes(int stages, int nq_pad, int kslabs);
// Tensor maps of one MaxSim launch: the packed tensor with boxes of 8, 16, 24, 32, 64, 96 and
// 128 rows (64 columns each), and the query block.
constexpr int kMaxsimDocMaps = 7;
constexpr int kMaxsimBoxRows[kMaxsimDocMaps] = {8, 16, 24, 32, 64, 96, 128};
struct MaxsimMaps {
    CUtensorMap d[kMaxsimDocMaps];
    CUtensorMap q;
};
cudaError_t launch_maxsim(const MaxsimArgs& a, const MaxsimMaps& maps, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_fill_f32(float* out, int n, float v, cudaStream_t s);

}  // namespace sel
