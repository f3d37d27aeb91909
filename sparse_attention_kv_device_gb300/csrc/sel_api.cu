// Host side of libsel: argument checks, workspace planning, TMA descriptor encoding
// and the launch sequence behind every entry point of include/sel.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "sel.h"
#include "sel_device.cuh"
#include "sel_kernels.h"

using namespace sel;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSegRows = 64;          // rows x 4 heads <= 256 = the MMA's largest N
constexpr int kMaxChunkRows = 32768;
constexpr int kTopkMaxBtCap = 8192;      // block-table entries a top-k CTA stages at most

// Failure-detection test hook (sel_debug_wait_limit): a tile the next launches leave
// unloaded, and the limit of every bounded wait in them.
int g_fault_tile = -1;
uint64_t g_wait_ns = sel::kWaitLimitNs;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
uint32_t next_pow2(uint32_t x) {
    uint32_t p = 1;
    while (p < x) p <<= 1;
    return p;
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
    int sms = 0;
    int max_smem_optin = 0;
    int smem_per_sm = 0;
    int l2_bytes = 0;
};

int current_device_info(DeviceInfo* out) {
    static DeviceInfo cache[kMaxDevices];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SEL_ECUDA;
    std::lock_guard<std::mutex> g(mu);
    if (cache[dev].sms == 0) {
        int sms = 0, smem = 0, smem_sm = 0, l2 = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            return SEL_ECUDA;
        cache[dev].sms = sms;
        cache[dev].max_smem_optin = smem;
        cache[dev].smem_per_sm = smem_sm;
        cache[dev].l2_bytes = l2;
    }
    *out = cache[dev];
    return SEL_OK;
}

// ------------------------------------------------------------------ TMA descriptors
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// fp16 [pages][64 rows][128] with page stride `page_stride` elements; box = one 64-row x
// 64-dim half page in the 128-byte swizzle layout the tensor-core descriptors expect.
int encode_key_map(CUtensorMap* m, const void* base, int64_t num_pages, int64_t page_stride) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return SEL_ECUDA;
    cuuint64_t dims[3] = {128, 64, static_cast<cuuint64_t>(num_pages)};
    cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(page_stride) * 2};
    cuuint32_t box[3] = {64, 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SEL_OK : SEL_ECUDA;
}

// fp16 [rows][4 heads][128] with row stride `row_stride` elements; box = 4 rows x 4
// heads x 64 dims (16 query lines), same swizzle.
int encode_q_map(CUtensorMap* m, const void* base, int64_t rows, int64_t row_stride) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return SEL_ECUDA;
    cuuint64_t dims[3] = {128, 4, static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(row_stride) * 2};
    cuuint32_t box[3] = {64, 4, 4};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SEL_OK : SEL_ECUDA;
}

// fp16 [rows][>= d] with row stride `row_stride` elements (a multiple of 8); box = `box_rows`
// rows x 64 columns in the 128-byte swizzle layout. Rows past `rows` and columns past `d`
// read as zeros.
int encode_rows_map(CUtensorMap* m, const void* base, int64_t d, int64_t rows, int64_t row_stride, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return SEL_ECUDA;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SEL_OK : SEL_ECUDA;
}

// ------------------------------------------------------------------ planning
struct TopkPlan {
    int bt_cap = 0;
    size_t smem = 0;
};

// Shared-memory plan of the top-k: with remap, a row stages up to kTopkMaxBtCap entries
// of its block-table row (longer rows read the rest from global memory).
int plan_topk(int64_t max_context, int block_size, bool remap, int max_smem, TopkPlan* t) {
    t->bt_cap = remap ? static_cast<int>(std::min<int64_t>(kTopkMaxBtCap, ceil_div(std::max<int64_t>(max_context, 1),
                                                                                   block_size)))
                      : 0;
    t->smem = topk_smem_bytes(t->bt_cap);
    if (t->smem > static_cast<size_t>(max_smem)) return SEL_EUNSUPPORTED;
    return SEL_OK;
}

struct Plan {
    int chunk_rows = 1, seg_rows = 1, max_segs = 1, chunks = 1;
    int64_t max_pools = 0, scores_ld = 4;
    // one plan block per chunk (offsets inside a block, plan_bytes apart), then the scores
    size_t off_hdr = 0, off_row_req = 0, off_row_ctx = 0, off_seg = 0, off_prefix = 0, plan_bytes = 0,
           off_scores = 0;
    size_t ws_score = 0, ws_select = 0;
    int npad_max = 16, stages = 2;
    uint32_t acc_cols = 32, tmem_cols = 64;
    size_t score_smem = 0;
    TopkPlan topk;
    int sms = 0;
    int bm_words = 1;
    int stage_cap = 0;  // keys of a row the select kernel stages in shared memory
    size_t sel_smem = 0;
    // the select kernel's 512-thread variant, two CTAs per SM (chunks with more rows than
    // SMs): its own staging capacity and shared-memory size; sel2_ok when it fits
    bool sel2_ok = false;
    int stage_cap2 = 0;
    size_t sel_smem2 = 0;
};

// log2(v) when v is a power of two, else -1
int log2_if_pow2(int v) {
    if (v < 1 || (v & (v - 1)) != 0) return -1;
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

int check_problem(const sel_problem* p) {
    if (!p) return SEL_EINVAL;
    if (p->num_reqs < 0 || p->num_rows < 0 || p->max_context < 0 || p->max_q_len < 0) return SEL_EINVAL;
    if (p->num_heads != 4 || p->head_dim != 128 || p->key_page_size != 64) return SEL_EUNSUPPORTED;
    if (p->kpool < 1 || p->index_topk < 1 || p->index_topk % p->kpool != 0) return SEL_EINVAL;
    if (p->block_size < 1 || p->block_stride_rows < p->block_size) return SEL_EINVAL;
    if (p->key_page_stride < 64 * 128 || p->q_row_stride < 4 * 128) return SEL_EINVAL;
    if (p->key_page_stride % 8 != 0 || p->q_row_stride % 8 != 0) return SEL_EUNSUPPORTED;
    if (p->num_key_pages < 1 || p->num_kv_blocks < 0) return SEL_EINVAL;
    if (p->max_key_pages_per_req < 0 || p->max_key_pages_per_req > p->kpt_ld) return SEL_EINVAL;
    if (p->max_blocks_per_req < 0 || p->max_blocks_per_req > p->bt_ld) return SEL_EINVAL;
    if (p->segment_rows < 0 || p->segment_rows > kMaxSegRows || p->chunk_rows < 0) return SEL_EINVAL;
    // the key page table must be wide enough for the longest allowed context
    if (ceil_div(p->max_context / p->kpool, 64) > p->max_key_pages_per_req) return SEL_EINVAL;
    // slots are int32
    if (p->num_kv_blocks > 0 &&
        static_cast<int64_t>(p->num_kv_blocks - 1) * p->block_stride_rows + p->block_size > INT32_MAX)
        return SEL_EINVAL;
    if (p->num_rows > 0) {
        if (!p->query_start_loc || !p->positions || !p->q || !p->key_cache || !p->key_page_table ||
            !p->block_table)
            return SEL_EINVAL;
        if (!aligned16(p->q) || !aligned16(p->key_cache)) return SEL_EUNSUPPORTED;
    }
    return SEL_OK;
}

// Rows per chunk when the caller leaves it to the library. The pages bound a logits chunk at
// 256 rows so that its fp32 scores stay in L2; with GB300's L2 a chunk can be larger under the
// same rule. Four times the SM count: two waves of the two-CTAs-per-SM row select, with fewer
// scorer-to-select hand-offs per call (the 4,112-row mixed step: 447 us at 256 rows, 345 us
// at 608). It is capped so one chunk's score rows at max_context fill at most 3/4 of L2 (rounded
// down to whole waves of the row select), and it is never below 256.
int default_chunk_rows(const sel_problem* p, const DeviceInfo& di) {
    const int64_t row_bytes = 4 * ((std::max<int64_t>(p->max_context / p->kpool, 1) + 3) & ~int64_t(3));
    const int64_t fit = static_cast<int64_t>(di.l2_bytes) * 3 / 4 / row_bytes;
    const int wave = 2 * di.sms;
    int64_t c = std::min<int64_t>(4 * static_cast<int64_t>(di.sms), fit);
    if (c > wave) c -= c % wave;
    return static_cast<int>(std::max<int64_t>(256, c));
}

int make_plan(const sel_problem* p, Plan* pl) {
    int rc = check_problem(p);
    if (rc != SEL_OK) return rc;
    DeviceInfo di;
    if ((rc = current_device_info(&di)) != SEL_OK) return rc;
    pl->sms = di.sms;
    const int rows = std::max(1, p->num_rows);
    pl->chunk_rows = std::min(std::min(rows, kMaxChunkRows), p->chunk_rows > 0 ? p->chunk_rows : default_chunk_rows(p, di));
    int sr = p->segment_rows;
    if (sr == 0) sr = p->max_q_len > 0 ? p->max_q_len : rows;
    pl->seg_rows = std::max(1, std::min(sr, kMaxSegRows));
    pl->max_segs = std::min(std::max(p->num_reqs, 1), pl->chunk_rows) +
                   static_cast<int>(ceil_div(pl->chunk_rows, pl->seg_rows)) + 1;
    pl->max_pools = p->max_context / p->kpool;
    pl->scores_ld = (std::max<int64_t>(pl->max_pools, 1) + 3) & ~int64_t(3);
    const int64_t tiles = static_cast<int64_t>(pl->max_segs) * std::max<int64_t>(1, ceil_div(pl->max_pools, 128));
    if (tiles > INT32_MAX / 2) return SEL_EUNSUPPORTED;  // tile ids and the tile counter are int32

    size_t off = 0;
    pl->off_hdr = off;
    off = align256(off + 16 * sizeof(int32_t));
    pl->off_row_req = off;
    off = align256(off + sizeof(int32_t) * pl->chunk_rows);
    pl->off_row_ctx = off;
    off = align256(off + sizeof(int32_t) * pl->chunk_rows);
    pl->off_seg = off;
    off = align256(off + sizeof(int4) * pl->max_segs);
    pl->off_prefix = off;
    off = align256(off + sizeof(int32_t) * (pl->max_segs + 1));
    pl->plan_bytes = off;
    pl->chunks = static_cast<int>(ceil_div(rows, pl->chunk_rows));
    off = pl->plan_bytes * static_cast<size_t>(pl->chunks);
    pl->ws_score = off;
    pl->off_scores = off;
    off = align256(off + sizeof(float) * static_cast<size_t>(pl->chunk_rows) * pl->scores_ld);
    pl->bm_words = static_cast<int>((pl->max_pools + 31) / 32);
    pl->ws_select = off;

    pl->npad_max = ((4 * pl->seg_rows + 15) / 16) * 16;
    pl->acc_cols = std::max<uint32_t>(32, next_pow2(static_cast<uint32_t>(pl->npad_max)));
    pl->tmem_cols = 2 * pl->acc_cols;
    const size_t fixed = score_smem_bytes(0, pl->npad_max, pl->max_segs);
    if (fixed + 2 * 32768 > static_cast<size_t>(di.max_smem_optin)) return SEL_EUNSUPPORTED;
    pl->stages = static_cast<int>(std::min<size_t>(8, (di.max_smem_optin - fixed) / 32768));
    while (pl->stages > 2 && score_smem_bytes(pl->stages, pl->npad_max, pl->max_segs) > static_cast<size_t>(di.max_smem_optin))
        --pl->stages;
    pl->score_smem = score_smem_bytes(pl->stages, pl->npad_max, pl->max_segs);
    if ((rc = plan_topk(p->max_context, p->block_size, true, di.max_smem_optin, &pl->topk)) != SEL_OK) return rc;
    // the select kernel stages as many of a row's keys as fit (longer rows read the rest from L2)
    const int K = p->index_topk / p->kpool;
    pl->stage_cap = static_cast<int>(std::min<int64_t>(kSelectMaxStage, (pl->max_pools + 3) & ~int64_t(3)));
    const size_t fixed_sel = select_smem_bytes(0, pl->bm_words, K, pl->topk.bt_cap);
    if (fixed_sel > static_cast<size_t>(di.max_smem_optin)) return SEL_EUNSUPPORTED;
    const int64_t fit = ((static_cast<int64_t>(di.max_smem_optin) - static_cast<int64_t>(fixed_sel)) / 4) & ~int64_t(3);
    pl->stage_cap = static_cast<int>(std::min<int64_t>(pl->stage_cap, fit));
    pl->sel_smem = select_smem_bytes(pl->stage_cap, pl->bm_words, K, pl->topk.bt_cap);
    // two CTAs per SM: each gets half the SM's shared memory less the 1 KiB the hardware
    // reserves per CTA; worth it only if a useful share of a row still fits
    const int64_t half = static_cast<int64_t>(di.smem_per_sm) / 2 - 1024;
    const int64_t fit2 = ((half - static_cast<int64_t>(fixed_sel)) / 4) & ~int64_t(3);
    pl->stage_cap2 = static_cast<int>(std::min<int64_t>(pl->stage_cap, fit2));
    pl->sel2_ok = fit2 >= 4096;
    pl->sel_smem2 = select_smem_bytes(pl->stage_cap2, pl->bm_words, K, pl->topk.bt_cap);
    return SEL_OK;
}

// ------------------------------------------------------------------ tracing
std::mutex g_trace_mu;
constexpr int kTraceEvents = 4;
cudaEvent_t g_trace[kTraceEvents] = {};
int g_trace_n = 0;

void trace_record(int i, cudaStream_t s) {
    if (g_trace_n < kTraceEvents || !g_trace[i]) return;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(s, &cs);
    if (cs == cudaStreamCaptureStatusActive)
        cudaEventRecordWithFlags(g_trace[i], s, cudaEventRecordExternal);
    else
        cudaEventRecord(g_trace[i], s);
}

// ------------------------------------------------------------------ shared launch path
struct Ws {
    int32_t* hdr;  // chunk 0's plan block; chunk k's is plan_bytes * k further
    int32_t* row_req;
    int32_t* row_ctx;
    int4* seg;
    int32_t* prefix;
    float* scores;
    size_t plan_bytes;
    // the plan block of chunk k
    Ws chunk(int k) const {
        const size_t off = plan_bytes * static_cast<size_t>(k);
        auto at = [off](auto* p) { return reinterpret_cast<decltype(p)>(reinterpret_cast<uint8_t*>(p) + off); };
        Ws w = *this;
        w.hdr = at(hdr);
        w.row_req = at(row_req);
        w.row_ctx = at(row_ctx);
        w.seg = at(seg);
        w.prefix = at(prefix);
        return w;
    }
};

Ws carve_ws(void* ws, const Plan& pl) {
    uint8_t* b = static_cast<uint8_t*>(ws);
    Ws w;
    w.hdr = reinterpret_cast<int32_t*>(b + pl.off_hdr);
    w.row_req = reinterpret_cast<int32_t*>(b + pl.off_row_req);
    w.row_ctx = reinterpret_cast<int32_t*>(b + pl.off_row_ctx);
    w.seg = reinterpret_cast<int4*>(b + pl.off_seg);
    w.prefix = reinterpret_cast<int32_t*>(b + pl.off_prefix);
    w.scores = reinterpret_cast<float*>(b + pl.off_scores);
    w.plan_bytes = pl.plan_bytes;
    return w;
}

// The builder: every chunk's plan in one launch, one CTA per chunk.
int launch_plans(const sel_problem* p, const Plan& pl, const Ws& w, int score_all, int64_t pool_cap,
                 int32_t* status, bool after_stage, cudaStream_t s) {
    BuildArgs b{};
    b.qsl = p->query_start_loc;
    b.positions = p->positions;
    b.key_page_table = p->key_page_table;
    b.kpt_ld = p->kpt_ld;
    b.max_key_pages = p->max_key_pages_per_req;
    b.num_key_pages = p->num_key_pages;
    b.num_reqs = p->num_reqs;
    b.num_rows = p->num_rows;
    b.row_begin = 0;
    b.row_end = p->num_rows;
    b.chunk_rows = pl.chunk_rows;
    b.plan_stride = static_cast<int64_t>(pl.plan_bytes);
    b.seg_rows = pl.seg_rows;
    b.topk = p->index_topk;
    b.kpool = p->kpool;
    b.max_context = p->max_context;
    b.score_all = score_all;
    b.pool_cap = static_cast<int32_t>(std::min<int64_t>(pool_cap, INT32_MAX));
    b.max_segs = pl.max_segs;
    b.row_req = w.row_req;
    b.row_ctx = w.row_ctx;
    b.seg = w.seg;
    b.seg_tile_prefix = w.prefix;
    b.hdr = w.hdr;
    b.status = status;
    if (launch_build(b, after_stage, s) != cudaSuccess) return SEL_ECUDA;
    if (!score_all) trace_record(1, s);
    return SEL_OK;
}

// The scorer for rows [c0, c1), on that chunk's plan block w; scores row k of the chunk at
// scores + k*ld.
int launch_chunk_score(const sel_problem* p, const Plan& pl, const Ws& w, int c0, int c1, int score_all, float* scores,
                       int64_t ld, int64_t pool_cap, int32_t* status, const CUtensorMap& tk,
                       const CUtensorMap& tq, cudaStream_t s) {
    ScoreArgs a{};
    a.seg = w.seg;
    a.hdr = w.hdr;
    a.seg_tile_prefix = w.prefix;
    a.key_page_table = p->key_page_table;
    a.kpt_ld = p->kpt_ld;
    a.max_key_pages = p->max_key_pages_per_req;
    a.num_key_pages = p->num_key_pages;
    a.max_segs = pl.max_segs;
    a.row_ctx = w.row_ctx;
    a.row_begin = c0;
    a.topk = p->index_topk;
    a.kpool = p->kpool;
    a.score_all = score_all;
    a.pool_cap = static_cast<int32_t>(std::min<int64_t>(pool_cap, INT32_MAX));
    a.scores = scores;
    a.scores_ld = ld;
    a.as_keys = score_all ? 0 : 1;  // the fused selection (score_all = 0) works on ordered keys
    // Chunk 0 follows the builder: small problems plan the chunk in the scorer itself, larger
    // ones wait for the builder's plan. Every later chunk follows a grid that started only
    // after the builder had finished (no grid of the chain lets its dependents launch before
    // the builder is done), so its plan is ready.
    if (c0 > 0)
        a.plan_mode = kPlanReady;
    else if (p->num_reqs <= kSelfPlanMaxReqs && c1 - c0 <= kSelfPlanMaxRows)
        a.plan_mode = kPlanSelf;
    else
        a.plan_mode = kPlanAfterBuilder;
    a.qsl = p->query_start_loc;
    a.positions = p->positions;
    a.num_reqs = p->num_reqs;
    a.num_rows = p->num_rows;
    a.row_end = c1;
    a.seg_rows = pl.seg_rows;
    a.max_context = p->max_context;
    a.npad_max = pl.npad_max;
    a.stages = pl.stages;
    a.tmem_cols = pl.tmem_cols;
    a.acc_cols = pl.acc_cols;
    a.status = status;
    a.fault_tile = g_fault_tile;
    a.wait_ns = g_wait_ns;
    if (launch_score(a, tk, tq, pl.sms, pl.score_smem, true, s) != cudaSuccess) return SEL_ECUDA;
    return SEL_OK;
}

// Validates the arguments every remap mode shares and fills them in.
int remap_args(const int32_t* req_id, int32_t num_reqs, const int32_t* block_table, int64_t bt_ld,
               int32_t max_blocks_per_req, int32_t num_kv_blocks, const int32_t* token_idx, int32_t num_rows,
               int32_t width, int32_t block_size, int64_t block_stride_rows, int32_t* slots, int32_t* valid_counts,
               RemapArgs* a) {
    if (num_rows < 0 || width < 0 || num_reqs < 0 || block_size < 1 || block_stride_rows < block_size)
        return SEL_EINVAL;
    if (max_blocks_per_req < 0 || max_blocks_per_req > bt_ld || num_kv_blocks < 0) return SEL_EINVAL;
    if (num_kv_blocks > 0 && static_cast<int64_t>(num_kv_blocks - 1) * block_stride_rows + block_size > INT32_MAX)
        return SEL_EINVAL;
    if (num_rows == 0) return SEL_OK;
    if (!req_id || !block_table || !token_idx || !slots) return SEL_EINVAL;
    if (width % 4 != 0) return SEL_EINVAL;
    if (!aligned16(token_idx) || !aligned16(slots)) return SEL_EUNSUPPORTED;
    a->req_id = req_id;
    a->num_reqs = num_reqs;
    a->block_table = block_table;
    a->bt_ld = bt_ld;
    a->max_blocks = max_blocks_per_req;
    a->num_kv_blocks = num_kv_blocks;
    a->block_size = block_size;
    a->block_stride_rows = block_stride_rows;
    a->token_idx = token_idx;
    a->width = width;
    a->slots = slots;
    a->counts = valid_counts;
    a->dcp_size = 1;
    a->interleave = 1;
    a->bs_shift = log2_if_pow2(block_size);
    a->il_shift = 0;
    a->dcp_shift = 0;
    return SEL_OK;
}

// The device's address of a pinned host buffer mapped into its address space, or null (a
// pageable or device buffer: the caller then uses the copy engine).
template <typename T>
T* device_view(T* host) {
    cudaPointerAttributes at{};
    if (!host || cudaPointerGetAttributes(&at, host) != cudaSuccess) {
        cudaGetLastError();  // an unknown pointer is not an error here
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? static_cast<T*>(at.devicePointer) : nullptr;
}

}  // namespace

extern "C" {

const char* sel_error_string(int code) {
    switch (code) {
        case SEL_OK: return "ok";
        case SEL_EINVAL: return "invalid argument (null pointer, negative or inconsistent size)";
        case SEL_EUNSUPPORTED: return "unsupported shape or alignment (needs 4 heads, 128 dims, 64-key pages, 16-B aligned buffers)";
        case SEL_ECUDA: return "a CUDA call failed";
        case SEL_EWORKSPACE: return "workspace smaller than the size query returned";
        default: return "unknown error";
    }
}

int sel_version(void) { return 102; }

size_t sel_workspace_bytes(const sel_problem* p) {
    Plan pl;
    return make_plan(p, &pl) == SEL_OK ? pl.ws_select : 0;
}

size_t sel_score_workspace_bytes(const sel_problem* p) {
    Plan pl;
    return make_plan(p, &pl) == SEL_OK ? pl.ws_score : 0;
}

int sel_score_paged(const sel_problem* p, float* scores, int64_t scores_ld, int32_t* status, void* ws,
                    size_t ws_bytes, sel_stream_t stream) {
    Plan pl;
    int rc = make_plan(p, &pl);
    if (rc != SEL_OK) return rc;
    if (p->num_rows == 0) return SEL_OK;
    if (!scores || scores_ld < 1 || !ws) return SEL_EINVAL;
    if (!aligned16(ws)) return SEL_EUNSUPPORTED;  // 16-B plan records
    if (ws_bytes < pl.ws_score) return SEL_EWORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap tk, tq;
    if ((rc = encode_key_map(&tk, p->key_cache, p->num_key_pages, p->key_page_stride)) != SEL_OK) return rc;
    if ((rc = encode_q_map(&tq, p->q, p->num_rows, p->q_row_stride)) != SEL_OK) return rc;
    Ws w = carve_ws(ws, pl);
    int32_t* st = status ? status : w.hdr + 8;
    if ((rc = launch_plans(p, pl, w, 1, scores_ld, st, false, s)) != SEL_OK) return rc;
    for (int k = 0, c0 = 0; c0 < p->num_rows; ++k, c0 += pl.chunk_rows) {
        rc = launch_chunk_score(p, pl, w.chunk(k), c0, std::min(p->num_rows, c0 + pl.chunk_rows), 1,
                                scores + static_cast<int64_t>(c0) * scores_ld, scores_ld,
                                scores_ld, st, tk, tq, s);
        if (rc != SEL_OK) return rc;
    }
    return SEL_OK;
}

int sel_topk_expand(const float* scores, int64_t scores_ld, const int32_t* positions, int32_t num_rows,
                    int32_t index_topk, int32_t kpool, int32_t* token_idx, int32_t out_width,
                    int32_t* valid_counts, int32_t* status, sel_stream_t stream) {
    if (num_rows < 0 || kpool < 1 || index_topk < 1 || index_topk % kpool != 0) return SEL_EINVAL;
    if (num_rows == 0) return SEL_OK;
    if (!scores || !positions || !token_idx || scores_ld < 1) return SEL_EINVAL;
    if (out_width < index_topk + kpool - 1 || out_width % 4 != 0 || scores_ld % 4 != 0) return SEL_EINVAL;
    if (!aligned16(scores) || !aligned16(token_idx)) return SEL_EUNSUPPORTED;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != SEL_OK) return rc;
    TopkPlan tp;
    if ((rc = plan_topk(0, 1, false, di.max_smem_optin, &tp)) != SEL_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int c0 = 0; c0 < num_rows; c0 += kMaxChunkRows) {
        const int rows = std::min(kMaxChunkRows, num_rows - c0);
        TopkArgs a{};
        a.scores = scores + static_cast<int64_t>(c0) * scores_ld;
        a.scores_ld = scores_ld;
        a.positions = positions;
        a.row_begin = c0;
        a.topk = index_topk;
        a.kpool = kpool;
        a.out_width = out_width;
        a.max_pools = scores_ld;
        a.bt_cap = 0;
        a.token_idx = token_idx;
        a.counts = valid_counts;
        a.status = status;
        a.block_size = 1;
        if (launch_topk(a, false, rows, tp.smem, false, s) != cudaSuccess) return SEL_ECUDA;
    }
    return SEL_OK;
}

int sel_remap_global(const int32_t* req_id, int32_t num_reqs, const int32_t* block_table, int64_t bt_ld,
                     int32_t max_blocks_per_req, int32_t num_kv_blocks, const int32_t* token_idx,
                     int32_t num_rows, int32_t width, int32_t block_size, int64_t block_stride_rows,
                     int32_t* slots, int32_t* valid_counts, sel_stream_t stream) {
    RemapArgs a{};
    const int rc = remap_args(req_id, num_reqs, block_table, bt_ld, max_blocks_per_req, num_kv_blocks, token_idx,
                              num_rows, width, block_size, block_stride_rows, slots, valid_counts, &a);
    if (rc != SEL_OK || num_rows == 0) return rc;
    return launch_remap(a, num_rows, kRemapGlobal, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SEL_OK
               : SEL_ECUDA;
}

int sel_remap_workspace(const int32_t* req_id, int32_t num_reqs, const int32_t* block_table, int64_t bt_ld,
                        int32_t max_blocks_per_req, int32_t num_kv_blocks, const int32_t* ws_req,
                        const int32_t* ws_starts, int32_t num_prefills, const int32_t* token_idx, int32_t num_rows,
                        int32_t width, int32_t block_size, int64_t block_stride_rows, int32_t* slots,
                        int32_t* valid_counts, sel_stream_t stream) {
    RemapArgs a{};
    const int rc = remap_args(req_id, num_reqs, block_table, bt_ld, max_blocks_per_req, num_kv_blocks, token_idx,
                              num_rows, width, block_size, block_stride_rows, slots, valid_counts, &a);
    if (rc != SEL_OK) return rc;
    if (num_prefills < 0) return SEL_EINVAL;
    if (num_rows == 0) return SEL_OK;
    if (!ws_req || (num_prefills > 0 && !ws_starts)) return SEL_EINVAL;
    a.ws_req = ws_req;
    a.ws_starts = ws_starts;
    a.num_prefills = num_prefills;
    return launch_remap(a, num_rows, kRemapWorkspace, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SEL_OK
               : SEL_ECUDA;
}

int sel_remap_dcp(const int32_t* req_id, int32_t num_reqs, const int32_t* block_table, int64_t bt_ld,
                  int32_t max_blocks_per_req, int32_t num_kv_blocks, const int32_t* token_idx, int32_t num_rows,
                  int32_t width, int32_t block_size, int32_t dcp_size, int32_t dcp_rank, int32_t interleave,
                  int32_t compact, int32_t* slots, int32_t* valid_counts, sel_stream_t stream) {
    RemapArgs a{};
    const int rc = remap_args(req_id, num_reqs, block_table, bt_ld, max_blocks_per_req, num_kv_blocks, token_idx,
                              num_rows, width, block_size, block_size, slots, valid_counts, &a);
    if (rc != SEL_OK) return rc;
    if (dcp_size < 1 || dcp_rank < 0 || dcp_rank >= dcp_size || interleave < 1 || block_size % interleave != 0)
        return SEL_EINVAL;
    if (num_rows == 0) return SEL_OK;
    a.dcp_size = dcp_size;
    a.dcp_rank = dcp_rank;
    a.interleave = interleave;
    a.il_shift = log2_if_pow2(interleave);
    a.dcp_shift = log2_if_pow2(dcp_size);
    a.compact = compact ? 1 : 0;
    return launch_remap(a, num_rows, kRemapDcp, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SEL_OK
               : SEL_ECUDA;
}

// ------------------------------------------------------------------ MaxSim rerank
namespace {

constexpr int kMaxsimMaxD = 1024;
constexpr size_t kMaxsimQBytes = 64 * 1024;  // query slabs resident per CTA
constexpr int kMaxsimMaxStages = 12;

// query rows per launch: a multiple of 32, at most 128 (the MMA's M), with the query's K
// slabs in 64 KiB of shared memory
int maxsim_nq_cap(int d) {
    const int kslabs = (d + 63) / 64;
    return std::min(128, static_cast<int>(kMaxsimQBytes / (static_cast<size_t>(kslabs) * 128)) & ~31);
}

}  // namespace

size_t sel_maxsim_workspace_bytes(void) { return 256; }

int32_t sel_maxsim_launch_count(int32_t lq, int32_t d) {
    if (lq <= 0 || d < 1 || d > kMaxsimMaxD) return lq == 0 ? 1 : 0;
    return static_cast<int32_t>(ceil_div(lq, maxsim_nq_cap(d)));
}

int sel_maxsim_rerank(const void* q, int32_t lq, int32_t d, int64_t q_stride, const void* docs, int64_t total_tokens,
                      int64_t doc_stride, const int32_t* doc_offsets, const int32_t* doc_lengths, int32_t num_docs,
                      float* scores, int32_t* status, void* ws, size_t ws_bytes, sel_stream_t stream) {
    if (lq < 0 || d < 1 || num_docs < 0 || total_tokens < 0) return SEL_EINVAL;
    if (num_docs == 0) return SEL_OK;
    if (!scores || !doc_offsets || !doc_lengths) return SEL_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (lq == 0) return launch_fill_f32(scores, num_docs, 0.0f, s) == cudaSuccess ? SEL_OK : SEL_ECUDA;
    if (!q || !docs || !ws || total_tokens < 1 || q_stride < d || doc_stride < d) return SEL_EINVAL;
    if (d > kMaxsimMaxD || total_tokens > INT32_MAX - 64 || q_stride % 8 != 0 || doc_stride % 8 != 0 ||
        !aligned16(q) || !aligned16(docs) || (reinterpret_cast<uintptr_t>(ws) & 3u) != 0)
        return SEL_EUNSUPPORTED;
    if (ws_bytes < sel_maxsim_workspace_bytes()) return SEL_EWORKSPACE;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != SEL_OK) return rc;

    const int kslabs = (d + 63) / 64;
    const int nq_cap = maxsim_nq_cap(d);
    // each CTA's static first claim: about an eighth of its share of the documents (<= 32)
    const int g0 = std::min(di.sms, num_docs);
    const int first_claim = std::max(1, std::min(32, num_docs / (8 * g0)));
    const int grid = std::min<int>(g0, static_cast<int>(ceil_div(num_docs, first_claim)));
    MaxsimMaps maps;
    for (int i = 0; i < kMaxsimDocMaps; ++i)
        if ((rc = encode_rows_map(&maps.d[i], docs, d, total_tokens, doc_stride, kMaxsimBoxRows[i])) != SEL_OK)
            return rc;
    int32_t* counter = static_cast<int32_t*>(ws);
    for (int q0 = 0; q0 < lq; q0 += nq_cap) {
        const int nq = std::min(nq_cap, lq - q0);
        const int nq_pad = (nq + 31) & ~31;
        int stages = kMaxsimMaxStages;
        while (stages > 2 && maxsim_smem_bytes(stages, nq_pad, kslabs) > static_cast<size_t>(di.max_smem_optin))
            --stages;
        const size_t smem = maxsim_smem_bytes(stages, nq_pad, kslabs);
        if (smem > static_cast<size_t>(di.max_smem_optin)) return SEL_EUNSUPPORTED;
        if ((rc = encode_rows_map(&maps.q, q, d, lq, q_stride, nq_pad)) != SEL_OK) return rc;
        MaxsimArgs a{};
        a.offsets = doc_offsets;
        a.lengths = doc_lengths;
        a.num_docs = num_docs;
        a.first_claim = first_claim;
        a.claim_base = grid * first_claim;
        a.total_tokens = total_tokens;
        a.scores = scores;
        a.accumulate = q0 > 0 ? 1 : 0;
        a.q_row0 = q0;
        a.nq = nq;
        a.nq_pad = nq_pad;
        a.kslabs = kslabs;
        a.stages = stages;
        a.tmem_cols = 256;
        a.counter = counter;
        a.status = status;
        a.fault_tile = g_fault_tile;
        a.wait_ns = g_wait_ns;
        if (launch_maxsim(a, maps, grid, smem, s) != cudaSuccess) return SEL_ECUDA;
    }
    return SEL_OK;
}

// ------------------------------------------------------------------ sparse MLA decode
namespace {
int mla_grid(int32_t rows, int32_t width, int sms, int64_t* total) {
    const int64_t tpr = ceil_div(width, kMlaTile);
    *total = static_cast<int64_t>(rows) * tpr;
    return static_cast<int>(std::min<int64_t>(sms, *total));
}
}  // namespace

size_t sel_mla_workspace_bytes(int32_t rows, int32_t width) {
    if (rows <= 0 || width <= 0) return 0;
    DeviceInfo di;
    if (current_device_info(&di) != SEL_OK) return 0;
    int64_t total = 0;
    const int grid = mla_grid(rows, width, di.sms, &total);
    return static_cast<size_t>(2 * grid) * kMlaPartBytes;
}

int sel_mla_decode(const void* q_nope, int64_t qn_row_stride, int64_t qn_head_stride, const void* q_pe,
                   int64_t qp_row_stride, int64_t qp_head_stride, int32_t rows, int32_t heads, int32_t dc, int32_t dr,
                   const void* ckv, int64_t ckv_stride, const void* kpe, int64_t kpe_stride, int64_t num_slots,
                   const int32_t* slots, int32_t width, const int32_t* kv_len, float sm_scale, float* out, float* lse,
                   int32_t* status, void* ws, size_t ws_bytes, sel_stream_t stream) {
    if (rows < 0 || width < 1 || num_slots < 0) return SEL_EINVAL;
    if (rows == 0) return SEL_OK;
    if (!q_nope || !ckv || !slots || !kv_len || !out || !lse || !ws) return SEL_EINVAL;
    if (dr > 0 && (!q_pe || !kpe)) return SEL_EINVAL;
    if (heads != kMlaHeads || dc != kMlaDc || (dr != 0 && dr != 64)) return SEL_EUNSUPPORTED;
    if (ceil_div(width, kMlaTile) > kMlaMaxTilesPerRow || num_slots > INT32_MAX) return SEL_EUNSUPPORTED;
    if (qn_head_stride < dc || qn_row_stride < static_cast<int64_t>(heads) * qn_head_stride || ckv_stride < dc)
        return SEL_EINVAL;
    if (dr > 0 && (qp_head_stride < dr || qp_row_stride < static_cast<int64_t>(heads) * qp_head_stride || kpe_stride < dr))
        return SEL_EINVAL;
    auto a8 = [](int64_t v) { return v % 8 == 0; };
    if (!a8(qn_row_stride) || !a8(qn_head_stride) || !a8(ckv_stride) || !aligned16(q_nope) || !aligned16(ckv) ||
        !aligned16(out) || (reinterpret_cast<uintptr_t>(ws) & 15u) != 0)
        return SEL_EUNSUPPORTED;
    if (dr > 0 && (!a8(qp_row_stride) || !a8(qp_head_stride) || !a8(kpe_stride) || !aligned16(q_pe) || !aligned16(kpe)))
        return SEL_EUNSUPPORTED;
    DeviceInfo di;
    int rc = current_device_info(&di);
    if (rc != SEL_OK) return rc;
    if (mla_smem_bytes() > static_cast<size_t>(di.max_smem_optin)) return SEL_EUNSUPPORTED;
    int64_t total = 0;
    const int grid = mla_grid(rows, width, di.sms, &total);
    if (ws_bytes < static_cast<size_t>(2 * grid) * kMlaPartBytes) return SEL_EWORKSPACE;
    MlaArgs a{};
    a.q_nope = static_cast<const uint16_t*>(q_nope);
    a.qn_row = qn_row_stride;
    a.qn_head = qn_head_stride;
    a.q_pe = static_cast<const uint16_t*>(q_pe);
    a.qp_row = qp_row_stride;
    a.qp_head = qp_head_stride;
    a.ckv = static_cast<const uint16_t*>(ckv);
    a.ckv_stride = ckv_stride;
    a.kpe = static_cast<const uint16_t*>(kpe);
    a.kpe_stride = kpe_stride;
    a.num_slots = num_slots;
    a.slots = slots;
    a.kv_len = kv_len;
    a.width = width;
    a.rows = rows;
    a.dr = dr;
    a.tiles_per_row = static_cast<int32_t>(ceil_div(width, kMlaTile));
    a.total_tiles = total;
    a.scale_log2 = sm_scale * 1.4426950408889634f;
    a.out = out;
    a.lse = lse;
    a.part = static_cast<uint8_t*>(ws);
    a.status = status;
    a.wait_ns = g_wait_ns;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (launch_mla(a, grid, s) != cudaSuccess) return SEL_ECUDA;
    if (launch_mla_merge(a, grid, s) != cudaSuccess) return SEL_ECUDA;
    return SEL_OK;
}

int32_t sel_mla_launch_count(int32_t rows) { return rows > 0 ? 2 : 0; }

// sel_select's work; after_stage: a staging kernel of the host-buffer entry point directly
// precedes it on the stream, and the builder is launched as its dependent.
static int select_queue(const sel_problem* p, int32_t* slots, int32_t out_width, int32_t* valid_counts,
                        int32_t* token_idx, int32_t* status, void* ws, size_t ws_bytes, sel_stream_t stream,
                        bool after_stage) {
    Plan pl;
    int rc = make_plan(p, &pl);
    if (rc != SEL_OK) return rc;
    if (p->num_rows == 0) return SEL_OK;
    if (!slots || !ws) return SEL_EINVAL;
    if (out_width < p->index_topk + p->kpool - 1 || out_width % 4 != 0) return SEL_EINVAL;
    if (!aligned16(slots) || (token_idx && !aligned16(token_idx)) || !aligned16(ws)) return SEL_EUNSUPPORTED;
    if (ws_bytes < pl.ws_select) return SEL_EWORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap tk, tq;
    if ((rc = encode_key_map(&tk, p->key_cache, p->num_key_pages, p->key_page_stride)) != SEL_OK) return rc;
    if ((rc = encode_q_map(&tq, p->q, p->num_rows, p->q_row_stride)) != SEL_OK) return rc;
    Ws w = carve_ws(ws, pl);
    int32_t* st = status ? status : w.hdr + 8;
    std::lock_guard<std::mutex> g(g_trace_mu);
    trace_record(0, s);
    if ((rc = launch_plans(p, pl, w, 0, pl.scores_ld, st, after_stage, s)) != SEL_OK) return rc;
    for (int k = 0, c0 = 0; c0 < p->num_rows; ++k, c0 += pl.chunk_rows) {
        const int c1 = std::min(p->num_rows, c0 + pl.chunk_rows);
        const bool last = c1 == p->num_rows;
        const Ws wc = w.chunk(k);
        rc = launch_chunk_score(p, pl, wc, c0, c1, 0, w.scores, pl.scores_ld, pl.scores_ld, st, tk, tq, s);
        if (rc != SEL_OK) return rc;
        if (last) trace_record(2, s);
        const uint32_t* keys = reinterpret_cast<const uint32_t*>(w.scores);

        RowSelectArgs ra{};
        ra.keys = keys;
        ra.keys_ld = pl.scores_ld;
        ra.row_ctx = wc.row_ctx;
        ra.row_req = wc.row_req;
        const bool two = pl.sel2_ok && c1 - c0 > pl.sms;  // more rows than SMs: 512 threads, two per SM
        ra.stage_cap = two ? pl.stage_cap2 : pl.stage_cap;
        ra.bm_words = pl.bm_words;
        ra.bt_cap = pl.topk.bt_cap;
        ra.row_begin = c0;
        ra.topk = p->index_topk;
        ra.kpool = p->kpool;
        ra.out_width = out_width;
        ra.kpool_shift = log2_if_pow2(p->kpool);
        ra.bs_shift = log2_if_pow2(p->block_size);
        ra.slots = slots;
        ra.token_idx = token_idx;
        ra.counts = valid_counts;
        ra.block_table = p->block_table;
        ra.bt_ld = p->bt_ld;
        ra.max_blocks = p->max_blocks_per_req;
        ra.num_kv_blocks = p->num_kv_blocks;
        ra.block_size = p->block_size;
        ra.block_stride_rows = p->block_stride_rows;
        ra.next_chunk = last ? 0 : 1;
        if (launch_select_rows(ra, c1 - c0, two ? pl.sel_smem2 : pl.sel_smem, true, s, two ? 512 : 1024) !=
            cudaSuccess)
            return SEL_ECUDA;
        if (last) trace_record(3, s);
    }
    return SEL_OK;
}

int sel_select(const sel_problem* p, int32_t* slots, int32_t out_width, int32_t* valid_counts, int32_t* token_idx,
               int32_t* status, void* ws, size_t ws_bytes, sel_stream_t stream) {
    return select_queue(p, slots, out_width, valid_counts, token_idx, status, ws, ws_bytes, stream, false);
}

int32_t sel_select_launch_count(const sel_problem* p) {
    Plan pl;
    if (make_plan(p, &pl) != SEL_OK || p->num_rows == 0) return 0;
    return static_cast<int32_t>(1 + 2 * ceil_div(p->num_rows, pl.chunk_rows));
}

size_t sel_host_stage_bytes(const sel_problem* p, int32_t out_width) {
    if (check_problem(p) != SEL_OK || out_width < 0) return 0;
    size_t off = 0;
    off = align256(off + sizeof(int32_t) * (p->num_reqs + 1));
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(p->num_rows));
    off = align256(off + 2 * static_cast<size_t>(p->num_rows) * p->q_row_stride);
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(p->num_reqs) * p->kpt_ld);
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(p->num_reqs) * p->bt_ld);
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(p->num_rows) * out_width);
    off = align256(off + sizeof(int32_t) * static_cast<size_t>(p->num_rows));
    return off;
}

int sel_select_host(const sel_problem* p, int32_t* slots_host, int32_t out_width, int32_t* counts_host,
                    int32_t* status, void* stage, size_t stage_bytes, void* ws, size_t ws_bytes,
                    sel_stream_t stream) {
    int rc = check_problem(p);
    if (rc != SEL_OK) return rc;
    if (p->num_rows == 0) return SEL_OK;
    if (!slots_host || !counts_host || !stage || !ws) return SEL_EINVAL;
    // the staged queries are read by tensor copies, the workspace holds 16-byte records: refuse
    // misaligned buffers before any copy is queued
    if (!aligned16(stage) || !aligned16(ws)) return SEL_EUNSUPPORTED;
    if (stage_bytes < sel_host_stage_bytes(p, out_width)) return SEL_EWORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* b = static_cast<uint8_t*>(stage);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* q = b + off;
        off = align256(off + bytes);
        return q;
    };
    const size_t n_qsl = sizeof(int32_t) * (p->num_reqs + 1);
    const size_t n_pos = sizeof(int32_t) * static_cast<size_t>(p->num_rows);
    const size_t n_q = 2 * (static_cast<size_t>(p->num_rows - 1) * p->q_row_stride + 512);
    const size_t n_kpt = p->num_reqs ? sizeof(int32_t) * (static_cast<size_t>(p->num_reqs - 1) * p->kpt_ld +
                                                          p->max_key_pages_per_req)
                                     : 0;
    const size_t n_bt = p->num_reqs ? sizeof(int32_t) * (static_cast<size_t>(p->num_reqs - 1) * p->bt_ld +
                                                         p->max_blocks_per_req)
                                    : 0;
    uint8_t* d_qsl = take(n_qsl);
    uint8_t* d_pos = take(n_pos);
    uint8_t* d_q = take(2 * static_cast<size_t>(p->num_rows) * p->q_row_stride);
    uint8_t* d_kpt = take(sizeof(int32_t) * static_cast<size_t>(p->num_reqs) * p->kpt_ld);
    uint8_t* d_bt = take(sizeof(int32_t) * static_cast<size_t>(p->num_reqs) * p->bt_ld);
    uint8_t* d_slots = take(sizeof(int32_t) * static_cast<size_t>(p->num_rows) * out_width);
    uint8_t* d_counts = take(n_pos);
    DeviceInfo di;
    if ((rc = current_device_info(&di)) != SEL_OK) return rc;
    // Pinned, mapped host buffers are copied by one kernel each way (over the host link);
    // any other host buffer goes through the copy engine, one transfer per buffer.
    StageArgs in{};
    auto add = [](StageArgs& g, const void* src, void* dst, size_t bytes) {
        g.src[g.nseg] = src;
        g.dst[g.nseg] = dst;
        g.bytes[g.nseg] = static_cast<int64_t>(bytes);
        ++g.nseg;
    };
    const void* m_qsl = device_view(p->query_start_loc);
    const void* m_pos = device_view(p->positions);
    const void* m_q = device_view(p->q);
    const void* m_kpt = n_kpt ? device_view(p->key_page_table) : nullptr;
    const void* m_bt = n_bt ? device_view(p->block_table) : nullptr;
    if (m_qsl && m_pos && m_q && (!n_kpt || m_kpt) && (!n_bt || m_bt)) {
        add(in, m_qsl, d_qsl, n_qsl);
        add(in, m_pos, d_pos, n_pos);
        add(in, m_q, d_q, n_q);
        if (n_kpt) add(in, m_kpt, d_kpt, n_kpt);
        if (n_bt) add(in, m_bt, d_bt, n_bt);
        if (launch_stage_copy(in, di.sms, s) != cudaSuccess) return SEL_ECUDA;
    } else {
        const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
        if (cudaMemcpyAsync(d_qsl, p->query_start_loc, n_qsl, h2d, s) != cudaSuccess ||
            cudaMemcpyAsync(d_pos, p->positions, n_pos, h2d, s) != cudaSuccess ||
            cudaMemcpyAsync(d_q, p->q, n_q, h2d, s) != cudaSuccess ||
            (n_kpt && cudaMemcpyAsync(d_kpt, p->key_page_table, n_kpt, h2d, s) != cudaSuccess) ||
            (n_bt && cudaMemcpyAsync(d_bt, p->block_table, n_bt, h2d, s) != cudaSuccess))
            return SEL_ECUDA;
    }
    // results: written by the row select straight into mapped host buffers, else copied back
    const size_t n_slots = sizeof(int32_t) * static_cast<size_t>(p->num_rows) * out_width;
    int32_t* m_slots = device_view(slots_host);
    int32_t* m_counts = device_view(counts_host);
    const bool direct_out = m_slots && m_counts && aligned16(m_slots);
    sel_problem d = *p;
    d.query_start_loc = reinterpret_cast<const int32_t*>(d_qsl);
    d.positions = reinterpret_cast<const int32_t*>(d_pos);
    d.q = d_q;
    d.key_page_table = reinterpret_cast<const int32_t*>(d_kpt);
    d.block_table = reinterpret_cast<const int32_t*>(d_bt);
    rc = select_queue(&d, direct_out ? m_slots : reinterpret_cast<int32_t*>(d_slots), out_width,
                      direct_out ? m_counts : reinterpret_cast<int32_t*>(d_counts), nullptr, status, ws, ws_bytes,
                      stream, in.nseg > 0);
    if (rc != SEL_OK) return rc;
    if (!direct_out) {
        const cudaMemcpyKind d2h = cudaMemcpyDeviceToHost;
        if (cudaMemcpyAsync(slots_host, d_slots, n_slots, d2h, s) != cudaSuccess ||
            cudaMemcpyAsync(counts_host, d_counts, n_pos, d2h, s) != cudaSuccess)
            return SEL_ECUDA;
    }
    return SEL_OK;
}

int sel_debug_wait_limit(int32_t fault_tile, int64_t wait_ns) {
    if (fault_tile < -1 || wait_ns < 1000) return SEL_EINVAL;
    g_fault_tile = fault_tile;
    g_wait_ns = static_cast<uint64_t>(wait_ns);
    return SEL_OK;
}

int sel_set_trace_events(void* const* events, int32_t n) {
    std::lock_guard<std::mutex> g(g_trace_mu);
    if (n == 0) {
        g_trace_n = 0;
        for (int i = 0; i < kTraceEvents; ++i) g_trace[i] = nullptr;
        return SEL_OK;
    }
    if (n < kTraceEvents || !events) return SEL_EINVAL;
    for (int i = 0; i < kTraceEvents; ++i) g_trace[i] = static_cast<cudaEvent_t>(events[i]);
    g_trace_n = kTraceEvents;
    return SEL_OK;
}

}  // extern "C"
