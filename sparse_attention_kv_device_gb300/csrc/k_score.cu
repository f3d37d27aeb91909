// K-b: request-segmented paged scorer on the 5th-generation tensor cores.
//
// What it computes (ReVolta PR #59, "Change"; the score definition is the plain one,
// sum over the 4 heads of q_h . k, accumulated in fp32):
//     scores[r][j] = sum_{h<4} sum_{d<128} q[r][h][d] * key(j)[d]
// for every row r of a segment and every pool j the row may score. The PR's idea is
// kept: the rows of one request share its key page table, so each 64-key page is
// loaded once per segment of rows and multiplied against all of the segment's
// rows x 4 heads at once. The design is GB300's own:
//   * each tile is two key pages (128 pools = the MMA's M); TMA copies the pages
//     (128-byte swizzle, evict-first) into a ring of shared-memory stages;
//   * one thread issues tcgen05.mma (M=128, N = rows*4 padded to 16, K=16, fp16 in,
//     fp32 accumulate) with the keys as A and the segment's queries as B, into one
//     of two TMEM accumulators;
//   * eight epilogue warps (two per TMEM lane quarter, 32 rows each) read the
//     accumulator (one TMEM lane = one pool per thread; a warp's 32 rows in one load),
//     add each row's 4 head columns, and store the row scores coalesced (for the fused
//     selection, the scores' order-preserving 32-bit keys instead);
//   * every CTA takes a static share of the segments' tiles, and the rest through an
//     atomic tile counter (segments may change inside a CTA's work, so the queries are
//     double-buffered too).
// Pools on key pages whose id is out of range score -inf and raise SEL_ST_KEYPAGE_OOB.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

constexpr int kSchedRing = 16;  // tiles published ahead by the producer (> stages + accumulators + 2)

struct ScoreSmem {
    uint8_t* a;          // stages x kTileBytes (keys)
    uint8_t* q;          // 2 x npad_max x 256 B (queries, two K halves each)
    int4* segs;          // [max_segs] the chunk's segments {request, first row, rows, pools}
    int* prefix;         // [max_segs + 1] exclusive prefix of their tiles
    int4* rec_ring;      // [kSchedRing] tile records in the order this CTA processes them
    int* tile_ring;      // [kSchedRing] tile ids (-1: no more tiles)
    uint64_t* full;      // [stages]
    uint64_t* empty;     // [stages]
    uint64_t* tfull;     // [2]
    uint64_t* tempty;    // [2]
    uint64_t* qfull;     // [2]
    uint64_t* qempty;    // [2]
    uint64_t* sfull;     // [kSchedRing] schedule slot published
    uint64_t* sempty;    // [kSchedRing] schedule slot read by the MMA thread and the epilogue warps
    uint64_t* done;      // [1]
    uint32_t* tmem_base;
    int* abort_flag;
    int* oob_flag;
    int* plan_nseg;      // segments of a plan the CTA computed itself
};

__device__ __forceinline__ ScoreSmem carve(uint8_t* raw, int stages, int npad_max, int max_segs) {
    ScoreSmem s;
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + (((base + 1023u) & ~1023u) - base);
    s.a = p;
    p += static_cast<size_t>(stages) * kTileBytes;
    s.q = p;
    p += 2u * static_cast<size_t>(npad_max) * 256u;
    s.segs = reinterpret_cast<int4*>(p);
    p += static_cast<size_t>(max_segs) * sizeof(int4);
    s.prefix = reinterpret_cast<int*>(p);
    p += ((static_cast<size_t>(max_segs) + 1) * sizeof(int) + 15) & ~size_t(15);
    s.rec_ring = reinterpret_cast<int4*>(p);
    p += kSchedRing * sizeof(int4);
    s.tile_ring = reinterpret_cast<int*>(p);
    p += kSchedRing * sizeof(int);
    uint64_t* b = reinterpret_cast<uint64_t*>(p);
    s.full = b;
    s.empty = b + stages;
    s.tfull = b + 2 * stages;
    s.tempty = s.tfull + 2;
    s.qfull = s.tempty + 2;
    s.qempty = s.qfull + 2;
    s.sfull = s.qempty + 2;
    s.sempty = s.sfull + kSchedRing;
    s.done = s.sempty + kSchedRing;
    uint32_t* w = reinterpret_cast<uint32_t*>(s.done + 1);
    s.tmem_base = w;
    s.abort_flag = reinterpret_cast<int*>(w + 1);
    s.oob_flag = reinterpret_cast<int*>(w + 2);
    s.plan_nseg = reinterpret_cast<int*>(w + 3);
    return s;
}

// Pools a row may score: its complete pools, when the row needs scoring.
__device__ __forceinline__ int row_pool_limit(const ScoreArgs& a, int row) {
    const int32_t c = __ldcg(a.row_ctx + row - a.row_begin);
    return (c > 0 && (a.score_all || c > a.topk)) ? min(c / a.kpool, a.pool_cap) : 0;
}

// The chunk's plan computed by the whole CTA from query_start_loc and positions with the
// segment builder's rule (ReVolta PR #59, "Change"; contexts as in _kv_lens_host of the
// flashinfer_mla_sparse_sm90 page): the chunk's rows of each request, cut every seg_rows rows,
// each segment scoring the largest complete-pool count of its rows, then the exclusive prefix
// of its 128-pool tiles. `scratch` holds num_reqs + 1 + rows + 33 words of shared memory that
// nothing else uses before the first key copy. An invalid query_start_loc gives no segments
// (the builder reports it). Ends with a block barrier.
__device__ void plan_self(const ScoreArgs& a, const ScoreSmem& sm, int32_t* scratch) {
    const int tid = threadIdx.x, T = blockDim.x;
    const int nrows = a.row_end - a.row_begin;
    int32_t* qs = scratch;                                       // [num_reqs + 1]
    int32_t* cx = scratch + a.num_reqs + 1;                      // [nrows] contexts, -1 = out of bound
    uint32_t* red = reinterpret_cast<uint32_t*>(cx + nrows);     // [33] scan scratch
    for (int i = tid; i <= a.num_reqs; i += T) qs[i] = __ldg(a.qsl + i);
    for (int k = tid; k < nrows; k += T) {
        const int64_t c64 = static_cast<int64_t>(__ldg(a.positions + a.row_begin + k)) + 1;
        cx[k] = c64 > a.max_context ? -1 : static_cast<int32_t>(c64 > 0 ? c64 : 0);
    }
    __syncthreads();
    int bad = 0;
    for (int i = tid; i < a.num_reqs; i += T) bad |= qs[i] > qs[i + 1];
    if (tid == 0) bad |= (qs[0] < 0) | (qs[a.num_reqs] > a.num_rows);
    bad = __syncthreads_or(bad);
    // segments: request i's rows inside the chunk, cut every seg_rows rows
    uint32_t carry = 0;
    for (int base = 0; !bad && base < a.num_reqs; base += T) {
        const int i = base + tid;
        int lo = 0, hi = 0;
        uint32_t ns = 0;
        if (i < a.num_reqs) {
            lo = max(qs[i], a.row_begin);
            hi = min(qs[i + 1], a.row_end);
            if (hi > lo) ns = (hi - lo + a.seg_rows - 1) / a.seg_rows;
        }
        uint32_t total;
        const uint32_t first = carry + block_excl_scan(ns, red, &total);
        for (uint32_t k = 0; k < ns; ++k) {
            const uint32_t sg = first + k;
            if (sg >= static_cast<uint32_t>(a.max_segs)) break;  // cannot happen with the host bound
            const int row0 = lo + static_cast<int>(k) * a.seg_rows;
            sm.segs[sg] = make_int4(i, row0, min(a.seg_rows, hi - row0), 0);
        }
        carry += total;
        __syncthreads();
    }
    const int nseg = min(static_cast<int>(carry), a.max_segs);
    // pools to score per segment: the largest over its rows, one warp per segment
    {
        const int lane = tid & 31, nwarps = T >> 5;
        for (int sg = tid >> 5; sg < nseg; sg += nwarps) {
            const int4 d = sm.segs[sg];
            int pools = 0;
            for (int rr = lane; rr < d.z; rr += 32) {
                const int32_t c = cx[d.y + rr - a.row_begin];
                if (c > 0 && (a.score_all || c > a.topk)) pools = max(pools, min(c / a.kpool, a.pool_cap));
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) pools = max(pools, __shfl_xor_sync(0xffffffffu, pools, o));
            if (lane == 0) sm.segs[sg] = make_int4(d.x, d.y, d.z, pools);
        }
        __syncthreads();
    }
    // tiles of 128 pools per segment, exclusive prefix
    uint32_t tcarry = 0;
    for (int base = 0; base < nseg; base += T) {
        const int sg = base + tid;
        const uint32_t t = sg < nseg ? static_cast<uint32_t>((sm.segs[sg].w + kTilePools - 1) / kTilePools) : 0u;
        uint32_t total;
        const uint32_t ex = tcarry + block_excl_scan(t, red, &total);
        if (sg < nseg) sm.prefix[sg] = static_cast<int>(ex);
        tcarry += total;
        __syncthreads();
    }
    if (tid == 0) {
        sm.prefix[nseg] = static_cast<int>(tcarry);
        *sm.plan_nseg = nseg;
    }
    fence_proxy_async_smem();  // the scratch (key stage 0) is next written by the tensor copies
    __syncthreads();
}

}  // namespace

// At most 96 registers a thread (320 x 96 = 30,720): a CTA then fits on an SM beside the
// segment builder's CTA (1,024 threads x 32 registers), so every scorer CTA can do its
// prologue while the builder runs.
constexpr int kScoreMaxRegs = 96;

// Tile schedule: CTA g first takes the contiguous static share [g*S, g*S + S) with
// S = floor(31/32 * tiles / grid), then draws single tiles from [S*grid, tiles) through an
// atomic counter, so CTAs that stream faster take more of the tail.
// kMode: how the CTA gets its plan (kPlanAfterBuilder, kPlanReady, kPlanSelf). In the last two
// it runs ahead of the preceding grid's end; each mode is its own instantiation, so the plain
// mode's producer loop carries none of that.
template <int kMode>
__global__ void __maxnreg__(kScoreMaxRegs)
    k_score_segments(const ScoreArgs a, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_q) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ScoreSmem sm = carve(smem_raw, a.stages, a.npad_max, a.max_segs);
    const uint32_t qhalf_bytes = static_cast<uint32_t>(a.npad_max) * 128u;
    constexpr bool kEarly = kMode != kPlanAfterBuilder;

    // ---- prologue (overlaps the segment builder when launched as a dependent grid)
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], kScoreEpiWarps * 32);
            mbar_init(&sm.qfull[i], 1);
            mbar_init(&sm.qempty[i], 1);
        }
        for (int i = 0; i < kSchedRing; ++i) {
            mbar_init(&sm.sfull[i], 1);
            mbar_init(&sm.sempty[i], 1 + kScoreEpiWarps);
        }
        mbar_init(sm.done, 1);
        *sm.abort_flag = 0;
        *sm.oob_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_q);
    }
    if (warp == 1) {
        tmem_alloc(sm.tmem_base, a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_base;
    volatile int* abort_flag = sm.abort_flag;

    // With the plan already complete (every chunk after the first), the CTA fetches its
    // tiles and runs its first products while the preceding grid (the previous chunk's
    // row select, which reads the score buffer) finishes; only the epilogue's stores wait
    // for it. Otherwise the builder's outputs are needed first.
    if constexpr (kMode == kPlanSelf) plan_self(a, sm, reinterpret_cast<int32_t*>(sm.a));
    if constexpr (kMode == kPlanAfterBuilder) pdl_wait();  // the builder's outputs are visible from here on
    // the row-select grid may be scheduled as CTAs retire (with a plan of its own, the CTA lets
    // it launch only once the builder, whose row descriptors it reads, has finished: below)
    if constexpr (kMode != kPlanSelf) pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ scheduler + TMA producer
        // the builder's segments and tile prefix, staged once by the whole warp: every slot
        // up to max_segs is loaded together with the header (entries past the builder's
        // segment count are never used), so the loads overlap
        int nseg;
        if constexpr (kMode == kPlanSelf) {
            nseg = *sm.plan_nseg;
        } else {
            const int nseg_raw = __ldcg(a.hdr + 0);
            for (int i = lane; i < a.max_segs; i += 32) sm.segs[i] = __ldcg(a.seg + i);
            for (int i = lane; i <= a.max_segs; i += 32) sm.prefix[i] = __ldcg(a.seg_tile_prefix + i);
            nseg = min(nseg_raw, a.max_segs);
            __syncwarp();
        }
        const int total = sm.prefix[nseg];
        // a large static share: each shared draw is an atomic round trip in the producer's
        // lookahead (measured: shares of 1/2, 5/8, 3/4, 7/8, 15/16 of the tiles were slower, and
        // so was no shared tail at all)
        const int share = static_cast<int>((static_cast<int64_t>(total) * 31 / 32) / gridDim.x);
        const int dyn0 = share * static_cast<int>(gridDim.x);
        {
            // warm L2 with the page-table entries of this CTA's static share (one line per lane)
            const int t = static_cast<int>(blockIdx.x) * share + lane * 8;
            if (lane * 8 < share && t < total) {
                int s = 0;
                for (int lo = 0, hi = nseg - 1; lo <= hi;) {
                    const int mid = (lo + hi) >> 1;
                    if (sm.prefix[mid] <= t) { s = mid; lo = mid + 1; } else { hi = mid - 1; }
                }
                const int lt = t - sm.prefix[s];
                if (2 * lt < a.max_key_pages)
                    prefetch_l2(a.key_page_table + static_cast<int64_t>(sm.segs[s].x) * a.kpt_ld + 2 * lt);
            }
        }
        if (lane == 0) {
            int s_next = static_cast<int>(blockIdx.x) * share;
            const int s_end = s_next + share;
            // A CTA that started early (beside the preceding grid) takes no shared tile before
            // its epilogue may store, or it would hold the tile while its stores wait: until
            // then a lookahead draw is deferred (kDeferred) and repeated when the tile is due.
            constexpr int kDeferred = -3;
            bool dyn_ok = !kEarly;
            auto grab = [&](bool may_wait) -> int {
                if (s_next < s_end) return s_next++;
                if constexpr (kEarly) {
                    if (!dyn_ok) {
                        if (!may_wait) return kDeferred;
                        pdl_wait();
                        dyn_ok = true;
                    }
                }
                const int t = dyn0 + atomicAdd(a.hdr + 2, 1);
                return t < total ? t : -1;
            };
            // A tile's record {segment, tile in segment, key page 0, key page 1}. Its two
            // page-table loads are issued when the tile is taken (two tiles ahead of its
            // TMA), and checked only when it is issued, so their latency is hidden.
            struct Pending {
                int t, seg, lt;
                int p0, p1;            // raw page-table entries
                bool has0, second, has1;
            };
            int cur_s = 0;  // the static share ascends: the search usually starts here
            auto take = [&](int t) -> Pending {
                Pending r;
                r.t = t;
                r.seg = 0;
                r.lt = 0;
                r.p0 = r.p1 = -1;
                r.has0 = r.second = r.has1 = false;
                if (t < 0) return r;
                int lo = sm.prefix[cur_s] <= t ? cur_s : 0, hi = nseg - 1;
                while (lo < hi) {  // last segment whose first tile is <= t
                    const int mid = (lo + hi + 1) >> 1;
                    if (sm.prefix[mid] <= t) lo = mid; else hi = mid - 1;
                }
                cur_s = lo;
                const int4 d = sm.segs[lo];
                r.seg = lo;
                r.lt = t - sm.prefix[lo];
                const int32_t* kpt_row = a.key_page_table + static_cast<int64_t>(d.x) * a.kpt_ld;
                r.has0 = 2 * r.lt < a.max_key_pages;
                if (r.has0) r.p0 = __ldg(kpt_row + 2 * r.lt);
                r.second = r.lt * kTilePools + kPagePools < d.w;
                r.has1 = r.second && 2 * r.lt + 1 < a.max_key_pages;
                if (r.has1) r.p1 = __ldg(kpt_row + 2 * r.lt + 1);
                return r;
            };
            // -1: page id out of range; -2: the tile has no second page
            auto record = [&](const Pending& r) -> int4 {
                const int pg0 = r.has0 && r.p0 >= 0 && r.p0 < a.num_key_pages ? r.p0 : -1;
                const int pg1 = !r.second ? -2 : (r.has1 && r.p1 >= 0 && r.p1 < a.num_key_pages ? r.p1 : -1);
                return make_int4(r.seg, r.lt, pg0, pg1);
            };
            // two tiles ahead: their ids and page-table entries are in flight while the current one is issued
            Pending t_a = take(grab(false));
            Pending t_b = take(t_a.t >= 0 ? grab(false) : t_a.t);

            const uint64_t pol_k = l2_policy_evict_first();
            const uint64_t pol_q = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            int qb = 1, cur = -1;
            int q_uses0 = 0, q_uses1 = 0;          // segments loaded into query buffer 0 / 1
            uint32_t qe_phase = 0;                 // bit b: parity to wait on query buffer b's release
            uint32_t loaded = 0, last_parity = 0;  // stages holding a load, parity of their last load
            bool ok = true;
            for (int n = 0; ok; ++n) {
                if constexpr (kEarly) {
                    if (t_a.t == kDeferred) {  // the shared tiles are open once the preceding grid is done
                        t_a = take(grab(true));
                        t_b = take(t_a.t >= 0 ? grab(true) : -1);
                    }
                }
                const int t = t_a.t;
                const int4 rec = t >= 0 ? record(t_a) : make_int4(0, 0, 0, 0);
                t_a = t_b;
                t_b = take(t_a.t >= 0 ? grab(false) : t_a.t);
                // publish the tile (or the end) to the MMA thread and the epilogue warps
                const int slot = n & (kSchedRing - 1);
                if (!mbar_wait(&sm.sempty[slot], ((n / kSchedRing) & 1) ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                sm.tile_ring[slot] = t;
                sm.rec_ring[slot] = rec;
                mbar_arrive(&sm.sfull[slot]);
                if (t < 0) break;

                if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                if (t != a.fault_tile) {  // the failure-detection test leaves one tile unloaded
                    const int npages = rec.w == -2 ? 1 : 2;
                    mbar_expect_tx(&sm.full[stage], static_cast<uint32_t>(npages) * kPageBytes);
                    uint8_t* adst = sm.a + static_cast<size_t>(stage) * kTileBytes;
                    loaded |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    for (int h = 0; h < npages; ++h) {
                        const int pg = max(h == 0 ? rec.z : rec.w, 0);  // out-of-range pages: the epilogue writes -inf
                        tma_load_3d(adst + h * kBoxBytes, &tmap_k, &sm.full[stage], 0, 0, pg, pol_k);
                        tma_load_3d(adst + kPageBytes + h * kBoxBytes, &tmap_k, &sm.full[stage], 64, 0, pg, pol_k);
                    }
                }
                if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                if (rec.x != cur) {
                    // the segment's queries, after its first key tile is on its way
                    const int4 sd = sm.segs[rec.x];
                    qb ^= 1;
                    if ((qb ? q_uses1 : q_uses0) > 0) {
                        if (!mbar_wait(&sm.qempty[qb], (qe_phase >> qb) & 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                        qe_phase ^= 1u << qb;
                    }
                    if (qb) ++q_uses1; else ++q_uses0;
                    const int nbox = (sd.z + 3) / 4;
                    mbar_expect_tx(&sm.qfull[qb], static_cast<uint32_t>(nbox) * 2u * kQBoxBytes);
                    uint8_t* qdst = sm.q + qb * 2 * qhalf_bytes;
                    for (int i = 0; i < nbox; ++i) {
                        tma_load_3d(qdst + i * kQBoxBytes, &tmap_q, &sm.qfull[qb], 0, 0, sd.y + 4 * i, pol_q);
                        tma_load_3d(qdst + qhalf_bytes + i * kQBoxBytes, &tmap_q, &sm.qfull[qb], 64, 0,
                                    sd.y + 4 * i, pol_q);
                    }
                    cur = rec.x;
                }
            }
            if (ok) {
                // drain: every stage's last load consumed, every query buffer released
                for (int i = 0; i < a.stages && ok; ++i) {
                    ok = mbar_wait(&sm.empty[stage], phase ^ 1u, abort_flag, a.wait_ns);
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
                if (ok && q_uses0 > 0) ok = mbar_wait(&sm.qempty[0], qe_phase & 1u, abort_flag, a.wait_ns);
                if (ok && q_uses1 > 0) ok = mbar_wait(&sm.qempty[1], (qe_phase >> 1) & 1u, abort_flag, a.wait_ns);
            }
            if (!ok) {
                *abort_flag = 1;
                report(a.status, kStTimeout);
                // let every copy already issued land before the CTA leaves (bounded)
                for (int i = 0; i < a.stages; ++i)
                    if (loaded & (1u << i)) mbar_wait(&sm.full[i], (last_parity >> i) & 1u, nullptr, a.wait_ns);
                if (q_uses0 > 0) mbar_wait(&sm.qfull[0], static_cast<uint32_t>(q_uses0 - 1) & 1u, nullptr, a.wait_ns);
                if (q_uses1 > 0) mbar_wait(&sm.qfull[1], static_cast<uint32_t>(q_uses1 - 1) & 1u, nullptr, a.wait_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            int qb = 1, cur = -1;
            uint32_t qf_phase = 0;  // bit b: parity of query buffer b's next fill
            uint32_t idesc = 0;
            const uint32_t a_base = smem_u32(sm.a);
            const uint32_t q_base = smem_u32(sm.q);
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int slot = n & (kSchedRing - 1);
                if (!mbar_wait(&sm.sfull[slot], (n / kSchedRing) & 1, abort_flag, a.wait_ns)) { ok = false; break; }
                const int t = sm.tile_ring[slot];
                const int4 rec = sm.rec_ring[slot];
                mbar_arrive(&sm.sempty[slot]);
                if (t < 0) break;
                if (rec.x != cur) {
                    // the previous segment's queries are free once its MMAs complete
                    if (cur >= 0) umma_commit(&sm.qempty[qb]);
                    const int4 sd = sm.segs[rec.x];
                    qb ^= 1;
                    if (!mbar_wait(&sm.qfull[qb], (qf_phase >> qb) & 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                    qf_phase ^= 1u << qb;
                    const uint32_t npad = static_cast<uint32_t>(((sd.z + 3) / 4) * 16);
                    idesc = umma_idesc_f16_f32(kTilePools, npad);
                    cur = rec.x;
                }
                if (!mbar_wait(&sm.full[stage], phase, abort_flag, a.wait_ns)) { ok = false; break; }
                if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc) * a.acc_cols;
                const uint32_t abase = a_base + static_cast<uint32_t>(stage) * kTileBytes;
                const uint32_t bbase = q_base + static_cast<uint32_t>(qb) * 2u * qhalf_bytes;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint32_t koff = static_cast<uint32_t>(kk & 3) * 32u;
                    const uint64_t ad = umma_desc_sw128(abase + static_cast<uint32_t>(kk >> 2) * kPageBytes + koff);
                    const uint64_t bd = umma_desc_sw128(bbase + static_cast<uint32_t>(kk >> 2) * qhalf_bytes + koff);
                    umma_f16(d, ad, bd, idesc, kk > 0 ? 1u : 0u);
                }
                umma_commit(&sm.empty[stage]);
                umma_commit(&sm.tfull[acc]);
                if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (ok && cur >= 0) umma_commit(&sm.qempty[qb]);  // the last segment's buffer
            if (!ok) {
                *abort_flag = 1;
                report(a.status, kStTimeout);
            }
            // all issued MMAs finished before teardown
            umma_commit(sm.done);
            mbar_wait(sm.done, 0, nullptr, a.wait_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-9)
        // Warp-local only: each warp waits on its own, holds the segment's per-row
        // pool limits in its lanes, and never waits for the other epilogue warps. Two warps
        // share each TMEM lane quarter (a tile's 128 pools): the first stores the segment's
        // rows 0-31, the second rows 32-63. Where every row of the segment may score all of
        // the warp's 32 pools (on an in-range key page) and the warp has all 32 of its rows,
        // it reads them 16 rows (64 accumulator columns) per TMEM load and stores the rows
        // back to back with no per-row check; otherwise 8 rows at a time, checked.
        if (kEarly) pdl_wait();                   // the preceding grid no longer reads the scores
        if constexpr (kMode == kPlanSelf) pdl_launch_dependents();  // the builder has finished
        const int quarter = warp & 3;             // TMEM lanes this warp may access
        const int r0 = ((warp - 2) >> 2) * 32;    // first row of the segment this warp stores
        int acc = 0;
        uint32_t acc_phase = 0;
        int cur = -1;
        int4 sd = make_int4(0, 0, 0, 0);
        int lim_mine = 0;                         // pools row r0 + lane may score
        int seg_min = 0;                          // the smallest such limit over the segment's rows
        int oob = 0;
        for (int n = 0;; ++n) {
            const int slot = n & (kSchedRing - 1);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&sm.sfull[slot], (n / kSchedRing) & 1, abort_flag, a.wait_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report(a.status, kStTimeout);
                }
                break;
            }
            const int t = sm.tile_ring[slot];
            const int4 rec = sm.rec_ring[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.sempty[slot]);
            if (t < 0) break;
            if (rec.x != cur) {
                sd = sm.segs[rec.x];
                const int lim_lo = lane < sd.z ? row_pool_limit(a, sd.y + lane) : 0;
                const int lim_hi = lane + 32 < sd.z ? row_pool_limit(a, sd.y + lane + 32) : 0;
                lim_mine = r0 == 0 ? lim_lo : lim_hi;
                int m = min(lane < sd.z ? lim_lo : 0x7fffffff, lane + 32 < sd.z ? lim_hi : 0x7fffffff);
#pragma unroll
                for (int o = 16; o; o >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, o));
                seg_min = m;
                cur = rec.x;
            }
            if (lane == 0) ok = mbar_wait(&sm.tfull[acc], acc_phase, abort_flag, a.wait_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    report(a.status, kStTimeout);
                }
                break;
            }
            __syncwarp();
            tc_fence_after();
            const int p_in_tile = quarter * 32 + lane;
            const int j = rec.y * kTilePools + p_in_tile;
            const bool page_ok = (quarter < 2 ? rec.z : rec.w) >= 0;  // the same for the whole warp
            if (!page_ok && j < sd.w) oob = 1;
            const int nr = min(32, sd.z - r0);  // rows of this warp in the segment
            const bool fast = page_ok && rec.y * kTilePools + quarter * 32 + 32 <= seg_min;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc) * a.acc_cols + static_cast<uint32_t>(r0 * 4);
            uint32_t* out = reinterpret_cast<uint32_t*>(a.scores) +
                            static_cast<int64_t>(sd.y + r0 - a.row_begin) * a.scores_ld + j;
            // a row's score from its 4 head columns, as stored: the order-preserving key for
            // the fused selection, else the fp32 bits
            auto word = [&](uint32_t h0, uint32_t h1, uint32_t h2, uint32_t h3) -> uint32_t {
                const float sc = page_ok ? ((__uint_as_float(h0) + __uint_as_float(h1)) + __uint_as_float(h2)) +
                                               __uint_as_float(h3)
                                         : -__int_as_float(0x7f800000);
                return a.as_keys ? ordered_key(sc) : __float_as_uint(sc);
            };
            if (nr == 32 && fast) {
                for (int h = 0; h < 2; ++h) {  // 16 rows (64 columns) per TMEM load
                    uint32_t v[64];
                    __syncwarp();
                    tmem_ld64_sync(taddr + static_cast<uint32_t>(h * 64), v);
                    uint32_t* o = out + static_cast<int64_t>(h * 16) * a.scores_ld;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        o[static_cast<int64_t>(i) * a.scores_ld] = word(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                }
            } else {
                for (int g = 0; g * 8 < nr; ++g) {
                    uint32_t v[32];
                    __syncwarp();
                    tmem_ld32(taddr + static_cast<uint32_t>(g * 32), v);
                    tmem_ld_wait();
#pragma unroll
                    for (int rr = 0; rr < 8; ++rr) {
                        const int i = g * 8 + rr;
                        if (i >= nr) break;  // uniform over the warp
                        const int lim = __shfl_sync(0xffffffffu, lim_mine, i);
                        if (fast || j < lim)
                            out[static_cast<int64_t>(i) * a.scores_ld] = word(v[4 * rr], v[4 * rr + 1], v[4 * rr + 2], v[4 * rr + 3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (__any_sync(0xffffffffu, oob) && lane == 0) *sm.oob_flag = 1;
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, a.tmem_cols);
    }
    if (threadIdx.x == 0 && *sm.oob_flag) report(a.status, kStKeyPageOob);
}

size_t score_smem_bytes(int stages, int npad_max, int max_segs) {
    return 1024 + static_cast<size_t>(stages) * kTileBytes + 2u * static_cast<size_t>(npad_max) * 256u +
           static_cast<size_t>(max_segs) * sizeof(int4) + (((static_cast<size_t>(max_segs) + 1) * sizeof(int) + 15) & ~size_t(15)) +
           kSchedRing * (sizeof(int4) + sizeof(int)) + (2 * static_cast<size_t>(stages) + 9 + 2 * kSchedRing) * 8 + 64;
}

cudaError_t launch_score(const ScoreArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_q, int grid,
                         size_t smem, bool pdl, cudaStream_t s) {
    static size_t configured[3][kMaxDevicesTracked] = {};
    const int m = a.plan_mode;
    if (m < kPlanAfterBuilder || m > kPlanSelf) return cudaErrorInvalidValue;
    auto kernel = m == kPlanSelf ? k_score_segments<kPlanSelf>
                                 : (m == kPlanReady ? k_score_segments<kPlanReady> : k_score_segments<kPlanAfterBuilder>);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevicesTracked && smem > configured[m][dev]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[m][dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kScoreThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, a, tmap_k, tmap_q);
}

}  // namespace sel
