// K-m: MaxSim rerank of one query against documents packed in one tensor, on the
// 5th-generation tensor cores.
//
// What it computes (vLLM page "flash_maxsim_rerank", _maxsim_rerank_kernel):
//     score[b] = sum_{a < lq} max_{j < len_b} q[a] . docs[off_b + j]
// with fp16 inputs and fp32 accumulation; a document with no rows scores -inf (the page's
// running maxima start at -inf). The page runs one program per document over power-of-two
// buckets of rows. The design here is GB300's own:
//   * documents are cut into 32-row chunks and packed, in the order the CTA takes them, four
//     chunks to a 128-row tile (a document may span tiles), so tiles stay full until the
//     CTA's last one;
//   * each tile streams through a ring of 64-column (128-byte swizzle) K slabs; full chunks
//     that continue one another (one document's consecutive rows) are copied by one TMA box
//     of 32, 64, 96 or 128 rows, and a document's partial last chunk by a box of its valid
//     rows rounded up to 8, so a document over-reads at most 7 rows;
//   * one thread issues tcgen05.mma with the query block as A (M = 128: up to 128 query rows,
//     resident in shared memory) and the tile as B (N = 128 document rows, K = 16 per
//     instruction, fp16 in, fp32 accumulate) into one of two TMEM accumulators, so TMEM lane
//     a holds query row a's dot products with the tile's 128 rows;
//   * epilogue warp w reads the lanes of query rows 32w .. 32w + 31: each thread takes the
//     maximum over a chunk's valid rows in registers, folds it into its document's running
//     maximum, and at the document's last chunk the warp sums its 32 rows; with more than 32
//     query rows the warp finishing a tile last adds the warps' sums in a fixed order;
//   * roles: warp 1 schedules (documents -> chunks -> tile records, at most 4 tiles ahead of
//     the copies, so the work a CTA has committed to when the documents run out stays small),
//     warp 3 only issues TMA copies, so the copy engine is never left idle while the schedule
//     is built, and forwards each tile's chunk info to the MMA and epilogue; warp 2 issues the MMAs; warps 4-7 are the epilogue (warp 0 idles so that the
//     busiest epilogue warp has its SM sub-partition to itself);
//   * CTAs claim consecutive documents: each CTA's first claim is static, later ones come from
//     an atomic counter in the caller's workspace (the last CTA to finish sets it back to zero,
//     so no memset is queued), sized ceil(unclaimed / (8 * CTAs)) in [1, 32] documents (guided
//     self-scheduling: fewer round trips early, one-document claims at the end); the next
//     claim is taken when the last document of the current one starts, so a CTA never holds
//     more than one unstarted document. Every document is finished by the CTA that claimed it.
// Rows outside [0, total_tokens) read as zero vectors (the TMA's out-of-bounds fill).
#include <algorithm>

#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

constexpr int kMsRing = 4;                      // tile records the scheduler may publish ahead of the TMA issuer
constexpr int kMsInfo = 8;                      // tiles' chunk info forwarded by the TMA issuer to the MMA / epilogue
constexpr int kMsRec = 16;                      // ints per tile record: {doc, info, first row, box chunks} x 4
constexpr uint32_t kMsChunkBytes = 32 * 128;    // 32 rows x 64 fp16 columns
constexpr uint32_t kMsSlabBytes = 4 * kMsChunkBytes;  // one 128-row K slab of a tile
constexpr int kMsPartBufs = 4;                  // tiles whose per-warp sums may be pending at once

// chunk info word: rows valid (1..32) | first chunk of its document << 6 | last << 7
constexpr int kInfoFirst = 64;
constexpr int kInfoLast = 128;

// Warp roles. A warp issues on SM sub-partition warp % 4, and the epilogue warp of query
// rows 0-31 (the only busy one for up to 32 query rows) must be a warp with warp % 4 == 0
// (TMEM lanes 0-31); the scheduler, MMA and TMA warps sit on sub-partitions 1-3 and warp 0
// idles, so that warp has its sub-partition to itself.
constexpr int kWarpSched = 1;
constexpr int kWarpMma = 2;
constexpr int kWarpTma = 3;
constexpr int kWarpEpi = 4;  // warps 4-7: query rows 32 * (warp % 4) ..

struct MsSmem {
    uint8_t* q;          // kslabs x nq_pad x 128 B (the query block, K slab by K slab)
    uint8_t* a;          // stages x kMsSlabBytes
    int* ring;           // [kMsRing][kMsRec] tile records; chunk c: doc (-1: none), info, first row,
                         // rows in the box starting at c (0: none); word 3 of chunk 0 = -1: end
    float* part;         // [kMsPartBufs][4 chunks][4 warps] per-warp sums of documents ending in a tile
    int* part_cnt;       // [kMsPartBufs] warps done with the tile
    int* qoff;           // [2][32] document offsets of the current and next grab (copied ahead by cp.async)
    int* qlen;           // [2][32] document lengths of the current and next grab
    uint64_t* full;      // [stages]
    uint64_t* empty;     // [stages]
    uint64_t* tfull;     // [2]
    uint64_t* tempty;    // [2]
    int* info;           // [kMsInfo][8] per tile, {doc, info} of chunks 0..3; info of chunk 0 = -1: end
    uint64_t* sfull;     // [kMsRing]
    uint64_t* sempty;    // [kMsRing] read by the TMA thread
    uint64_t* ifull;     // [kMsInfo]
    uint64_t* iempty;    // [kMsInfo] read by the MMA thread and the epilogue warps
    uint64_t* qfull;     // [1]
    uint64_t* done;      // [1]
    uint32_t* tmem_base;
    int* abort_flag;
};

__device__ __forceinline__ MsSmem ms_carve(uint8_t* raw, int stages, int nq_pad, int kslabs) {
    MsSmem s;
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + (((base + 1023u) & ~1023u) - base);
    s.q = p;
    p += static_cast<size_t>(kslabs) * nq_pad * 128u;
    s.a = p;
    p += static_cast<size_t>(stages) * kMsSlabBytes;
    s.ring = reinterpret_cast<int*>(p);
    p += kMsRing * kMsRec * sizeof(int);
    s.info = reinterpret_cast<int*>(p);
    p += kMsInfo * 8 * sizeof(int);
    s.part = reinterpret_cast<float*>(p);
    p += kMsPartBufs * 16 * sizeof(float);
    s.part_cnt = reinterpret_cast<int*>(p);
    p += kMsPartBufs * sizeof(int);
    s.qoff = reinterpret_cast<int*>(p);
    p += 2 * 32 * sizeof(int);
    s.qlen = reinterpret_cast<int*>(p);
    p += 2 * 32 * sizeof(int);
    uint64_t* b = reinterpret_cast<uint64_t*>(p);
    s.full = b;
    s.empty = b + stages;
    s.tfull = b + 2 * stages;
    s.tempty = s.tfull + 2;
    s.sfull = s.tempty + 2;
    s.sempty = s.sfull + kMsRing;
    s.ifull = s.sempty + kMsRing;
    s.iempty = s.ifull + kMsInfo;
    s.qfull = s.iempty + kMsInfo;
    s.done = s.qfull + 1;
    uint32_t* w = reinterpret_cast<uint32_t*>(s.done + 1);
    s.tmem_base = w;
    s.abort_flag = reinterpret_cast<int*>(w + 1);
    return s;
}

// Waits on `bar` with lane 0 polling; every lane learns the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, limit_ns) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Maximum of v[0 .. rows-1] (1 <= rows <= 32), as fp32: a five-level tree (independent
// operations at each level); rows past `rows` are masked only when the chunk is partial.
__device__ __forceinline__ float row_max(const uint32_t (&v)[32], int rows) {
    float x[16];
    if (rows >= 32) {
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = fmaxf(__uint_as_float(v[j]), __uint_as_float(v[j + 16]));
    } else {
        const float ninf = -__int_as_float(0x7f800000);
#pragma unroll
        for (int j = 0; j < 16; ++j)
            x[j] = fmaxf(__uint_as_float(v[j]), j + 16 < rows ? __uint_as_float(v[j + 16]) : ninf);
#pragma unroll
        for (int j = 1; j < 16; ++j)
            if (j >= rows) x[j] = ninf;
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) x[j] = fmaxf(x[j], x[j + w]);
    return x[0];
}

__device__ __forceinline__ float warp_sum(float s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

}  // namespace

__global__ void __launch_bounds__(kMaxsimThreads, 1)
    k_maxsim(const MaxsimArgs a, const __grid_constant__ MaxsimMaps maps) {
    const CUtensorMap* tmap_d = maps.d;
    const CUtensorMap& tmap_q = maps.q;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    MsSmem sm = ms_carve(smem_raw, a.stages, a.nq_pad, a.kslabs);
    const int nwarps = a.nq_pad >> 5;  // epilogue warps with query rows
    // diagnostics: CTA 0 stamps its phases, every CTA its end (300 + CTA)
    // the scheduler's first round trips start before the setup: the offsets/lengths of the
    // CTA's static first claim and the atomic for its second claim
    int pend = 0;  // scheduler warp, lane 0: an atomic's value in flight
    if (warp == kWarpSched) {
        if (lane == 0) pend = atomicAdd(a.counter, a.first_claim);
        const int doc = static_cast<int>(blockIdx.x) * a.first_claim + lane;
        if (lane < a.first_claim && doc < a.num_docs) {
            cp_async_4(&sm.qoff[lane], a.offsets + doc);
            cp_async_4(&sm.qlen[lane], a.lengths + doc);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], 32 * nwarps);
        }
        for (int i = 0; i < kMsRing; ++i) {
            mbar_init(&sm.sfull[i], 1);
            mbar_init(&sm.sempty[i], 1);
        }
        for (int i = 0; i < kMsInfo; ++i) {
            mbar_init(&sm.ifull[i], 1);
            mbar_init(&sm.iempty[i], 1 + nwarps);
        }
        for (int i = 0; i < kMsPartBufs; ++i) sm.part_cnt[i] = 0;
        mbar_init(sm.qfull, 1);
        mbar_init(sm.done, 1);
        *sm.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kWarpTma && lane < kMaxsimDocMaps) tma_prefetch_desc(&tmap_d[lane]);
    if (warp == kWarpTma && lane == kMaxsimDocMaps) tma_prefetch_desc(&tmap_q);
    if (warp == kWarpMma) {
        tmem_alloc(sm.tmem_base, a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_base;
    volatile int* abort_flag = sm.abort_flag;
    const float neg_inf = -__int_as_float(0x7f800000);

    if (warp == kWarpSched) {
        // ------------------------------------------------------------ scheduler: documents -> chunks -> tiles
        // Document source: claims of consecutive documents (guided self-scheduling). The CTA's
        // first claim is static, first_claim documents from blockIdx.x * first_claim; later ones
        // come from an atomic counter (claim_base + its value), each sized from the documents
        // still unclaimed, ceil(remaining / (8 * CTAs)) clamped to [1, 32]: several while much is
        // left (fewer round trips), one document at the end (balanced tails). One atomic is in
        // flight (issued when the previous claim is resolved; a single thread issues them, so
        // their values rise in issue order), and a claim's offsets and lengths are copied by
        // cp.async into a queue slot.
        const int nd = a.num_docs;
        const int G = static_cast<int>(gridDim.x);
        int pend_k = a.first_claim;  // size of the claim in flight
        bool has_pend = true;        // warp-uniform: `pend` holds an atomic in flight
        auto fetch_meta = [&](int s, int start, int cnt) {  // cp.async a claim's offsets and lengths into slot s % 2
            if (lane < cnt) {
                cp_async_4(&sm.qoff[(s & 1) * 32 + lane], a.offsets + start + lane);
                cp_async_4(&sm.qlen[(s & 1) * 32 + lane], a.lengths + start + lane);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        auto resolve = [&](int& start, int& cnt) {  // the next claim (cnt 0: none); warp-uniform
            start = 0;
            cnt = 0;
            if (!has_pend) return;
            const int v = __shfl_sync(0xffffffffu, pend, 0);
            has_pend = false;
            if (v >= nd - a.claim_base) return;  // counter past the end: no claim, no more atomics
            start = a.claim_base + v;
            cnt = min(pend_k, nd - start);
            const int left = nd - start - cnt;
            if (left > 0) {
                pend_k = min(32, max(1, (left + 8 * G - 1) / (8 * G)));
                if (lane == 0) pend = atomicAdd(a.counter, pend_k);
                has_pend = true;
            }
        };
        int start0 = static_cast<int>(blockIdx.x) * a.first_claim;  // its metadata copy started before the setup
        int cnt0 = max(0, min(a.first_claim, nd - start0));
        // the tile being gathered: lane c < nc holds chunk c
        int nc = 0, my_doc = -1, my_info = 0, my_row = 0;
        int n = 0;
        bool ok = true;

        // publishes the gathered tile (nc == 0: the end record)
        auto publish = [&]() -> bool {
            const int slot = n & (kMsRing - 1);
            if (!warp_wait(&sm.sempty[slot], ((n / kMsRing) & 1) ^ 1u, abort_flag, a.wait_ns)) return false;
            int doc[4], row[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                doc[c] = __shfl_sync(0xffffffffu, c < nc ? my_doc : -1, c);
                row[c] = __shfl_sync(0xffffffffu, my_row, c);
            }
            // full chunks that continue one another (one document, consecutive rows) share one
            // box of 32 * run rows; a document's partial last chunk gets its own box of its valid
            // rows rounded up to 8
            int rows[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) rows[c] = __shfl_sync(0xffffffffu, my_info, c) & 63;
            bool cont[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                cont[c] = c > 0 && c < nc && doc[c] == doc[c - 1] && row[c] == row[c - 1] + 32 && rows[c] == 32;
            int box = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                int l = c < nc && !cont[c] ? 1 : 0;
#pragma unroll
                for (int e = c + 1; e < 4; ++e)
                    if (l == e - c && cont[e]) ++l;
                const int h = l == 1 && rows[c] < 32 ? (rows[c] + 7) & ~7 : 32 * l;
                if (c == lane) box = h;
            }
            if (lane < 4) {
                const int4 v = make_int4(lane < nc ? my_doc : -1, my_info, my_row, (nc == 0 && lane == 0) ? -1 : box);
                *reinterpret_cast<int4*>(sm.ring + slot * kMsRec + 4 * lane) = v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.sfull[slot]);
            ++n;
            nc = 0;
            return true;
        };

        // The claim in hand is consumed document by document; the next claim is resolved (and
        // its metadata copy started) only when the last document of this one begins, so a CTA
        // holds at most one document beyond what it is scheduling.
        for (int step = 0; ok; ++step) {
            if (cnt0 == 0) {  // nothing in hand (an empty first claim): resolve one now
                if (!has_pend) break;
                resolve(start0, cnt0);
                fetch_meta(step, start0, cnt0);
                if (cnt0 == 0) break;  // the counter is past the end
            }
            asm volatile("cp.async.wait_group 0;" ::: "memory");  // this claim's metadata
            const int base_doc = start0, ndocs = cnt0;
            int cur_off = 0, cur_len = 0;
            if (lane < ndocs) {  // each lane reads what it copied
                cur_off = sm.qoff[(step & 1) * 32 + lane];
                cur_len = sm.qlen[(step & 1) * 32 + lane];
            }
            cnt0 = 0;
            for (int i = 0; i < ndocs && ok; ++i) {
                if (i == ndocs - 1) {  // the last document: line up the next claim
                    resolve(start0, cnt0);
                    fetch_meta(step + 1, start0, cnt0);
                }
                const int doc = base_doc + i;
                const int off = __shfl_sync(0xffffffffu, cur_off, i);
                const int len = __shfl_sync(0xffffffffu, cur_len, i);
                if (len <= 0) {
                    if (lane == 0) a.scores[doc] = neg_inf;
                    continue;
                }
                const int nch = (len + 31) >> 5;
                for (int k = 0; k < nch; ++k) {
                    if (lane == nc) {
                        // clamp the first row into [-32, total_tokens]: rows outside read as zeros
                        int64_t r = static_cast<int64_t>(off) + 32 * static_cast<int64_t>(k);
                        r = r < -32 ? -32 : (r > a.total_tokens ? a.total_tokens : r);
                        my_doc = doc;
                        my_row = static_cast<int>(r);
                        my_info = min(32, len - 32 * k) | (k == 0 ? kInfoFirst : 0) | (k == nch - 1 ? kInfoLast : 0);
                    }
                    if (++nc == 4 && !(ok = publish())) break;
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        // an atomic still in flight (only after an abort) completes before the counter is reset:
        // storing its value makes this thread wait for it
        if (has_pend && lane == 0) *reinterpret_cast<volatile int*>(sm.qoff) = pend;
        if (ok && nc > 0) ok = publish();
        if (ok) ok = publish();  // the end record
        if (!ok && lane == 0) {
            *abort_flag = 1;
            report(a.status, kStTimeout);
        }
    } else if (warp == kWarpTma) {
        // ------------------------------------------------------------ TMA issuer
        if (lane == 0) {
            const uint64_t pol_d = l2_policy_evict_first();
            const uint32_t qslab = static_cast<uint32_t>(a.nq_pad) * 128u;
            mbar_expect_tx(sm.qfull, static_cast<uint32_t>(a.kslabs) * qslab);
            for (int g = 0; g < a.kslabs; ++g)
                tma_load_2d(sm.q + static_cast<size_t>(g) * qslab, &tmap_q, sm.qfull, g * 64, a.q_row0,
                            l2_policy_evict_last());
            int stage = 0;
            uint32_t phase = 0, loaded = 0, last_parity = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int slot = n & (kMsRing - 1);
                if (!mbar_wait(&sm.sfull[slot], (n / kMsRing) & 1, abort_flag, a.wait_ns)) { ok = false; break; }
                int4 r[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) r[c] = *reinterpret_cast<const int4*>(sm.ring + slot * kMsRec + 4 * c);
                mbar_arrive(&sm.sempty[slot]);
                // forward the chunks' {doc, info} (or the end) to the MMA thread and the epilogue
                const int islot = n & (kMsInfo - 1);
                if (!mbar_wait(&sm.iempty[islot], ((n / kMsInfo) & 1) ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                {
                    int4* dst = reinterpret_cast<int4*>(sm.info + islot * 8);
                    dst[0] = make_int4(r[0].x, r[0].w < 0 ? -1 : r[0].y, r[1].x, r[1].y);
                    dst[1] = make_int4(r[2].x, r[2].y, r[3].x, r[3].y);
                }
                mbar_arrive(&sm.ifull[islot]);
                if (r[0].w < 0) break;
                const uint32_t bytes = static_cast<uint32_t>(max(r[0].w, 0) + max(r[1].w, 0) + max(r[2].w, 0) +
                                                             max(r[3].w, 0)) * 128u;
                for (int g = 0; g < a.kslabs; ++g) {
                    if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                    if (n == a.fault_tile) {  // the failure-detection test leaves this tile unloaded
                        if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                        continue;
                    }
                    mbar_expect_tx(&sm.full[stage], bytes);
                    uint8_t* dst = sm.a + static_cast<size_t>(stage) * kMsSlabBytes;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int h = r[c].w;  // rows in the box starting at chunk c (0: none)
                        if (h > 0) {
                            const CUtensorMap* m = h == 8 ? &tmap_d[0] : h == 16 ? &tmap_d[1] : h == 24 ? &tmap_d[2]
                                                 : h == 32 ? &tmap_d[3] : h == 64 ? &tmap_d[4] : h == 96 ? &tmap_d[5]
                                                 : &tmap_d[6];
                            tma_load_2d(dst + c * kMsChunkBytes, m, &sm.full[stage], g * 64, r[c].z, pol_d);
                        }
                    }
                    loaded |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
            }
            if (ok) {
                // drain: every stage's last copy consumed before the CTA leaves
                for (int i = 0; i < a.stages && ok; ++i) {
                    ok = mbar_wait(&sm.empty[stage], phase ^ 1u, abort_flag, a.wait_ns);
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                report(a.status, kStTimeout);
                for (int i = 0; i < a.stages; ++i)
                    if (loaded & (1u << i)) mbar_wait(&sm.full[i], (last_parity >> i) & 1u, nullptr, a.wait_ns);
                mbar_wait(sm.qfull, 0, nullptr, a.wait_ns);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            const uint32_t idesc = umma_idesc_f16_f32(128, 128);
            const uint32_t a_base = smem_u32(sm.a);
            const uint32_t q_base = smem_u32(sm.q);
            const uint32_t qslab = static_cast<uint32_t>(a.nq_pad) * 128u;
            bool ok = mbar_wait(sm.qfull, 0, abort_flag, a.wait_ns);
            for (int n = 0; ok; ++n) {
                const int islot = n & (kMsInfo - 1);
                if (!mbar_wait(&sm.ifull[islot], (n / kMsInfo) & 1, abort_flag, a.wait_ns)) { ok = false; break; }
                const bool end = sm.info[islot * 8 + 1] < 0;
                mbar_arrive(&sm.iempty[islot]);
                if (end) break;
                if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * 128);
                for (int g = 0; g < a.kslabs; ++g) {
                    if (!mbar_wait(&sm.full[stage], phase, abort_flag, a.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    // A: query rows (rows past nq_pad read what follows in shared memory and only
                    // reach TMEM lanes no warp reads); B: the tile's 128 document rows
                    const uint32_t qb = q_base + static_cast<uint32_t>(g) * qslab;
                    const uint32_t db = a_base + static_cast<uint32_t>(stage) * kMsSlabBytes;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f16(d, umma_desc_sw128(qb + kk * 32u), umma_desc_sw128(db + kk * 32u), idesc,
                                 (g | kk) ? 1u : 0u);
                    umma_commit(&sm.empty[stage]);
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&sm.tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                *abort_flag = 1;
                report(a.status, kStTimeout);
            }
            umma_commit(sm.done);
            mbar_wait(sm.done, 0, nullptr, a.wait_ns);
        }
    } else if (warp >= kWarpEpi && (warp & 3) < nwarps) {
        // ------------------------------------------------------------ epilogue
        // Warp w reads TMEM lanes 32 * (w % 4) .. = query rows qw * 32 + lane of the block.
        const int qw = warp & 3;
        const bool row_ok = qw * 32 + lane < a.nq;
        float run = neg_inf;  // this query row's running maximum over the current document
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int n = 0;; ++n) {
            const int islot = n & (kMsInfo - 1);
            if (!warp_wait(&sm.ifull[islot], (n / kMsInfo) & 1, abort_flag, a.wait_ns)) { ok = false; break; }
            int2 r[4];  // {doc (-1: none), info} of chunks 0..3
#pragma unroll
            for (int c = 0; c < 4; ++c) r[c] = *reinterpret_cast<const int2*>(sm.info + islot * 8 + 2 * c);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.iempty[islot]);
            if (r[0].y < 0) break;
            if (!warp_wait(&sm.tfull[acc], acc_phase, abort_flag, a.wait_ns)) { ok = false; break; }
            tc_fence_after();
            // per chunk: this row's best dot product over the chunk's valid rows
            float m[4];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(qw * 32) << 16) + static_cast<uint32_t>(acc * 128);
            {
                uint32_t v0[32], v1[32], v2[32], v3[32];  // all four chunks in flight, one wait
                tmem_ld32(taddr, v0);
                tmem_ld32(taddr + 32u, v1);
                tmem_ld32(taddr + 64u, v2);
                tmem_ld32(taddr + 96u, v3);
                tmem_ld_wait();
                m[0] = r[0].x >= 0 ? row_max(v0, r[0].y & 63) : neg_inf;
                m[1] = r[1].x >= 0 ? row_max(v1, r[1].y & 63) : neg_inf;
                m[2] = r[2].x >= 0 ? row_max(v2, r[2].y & 63) : neg_inf;
                m[3] = r[3].x >= 0 ? row_max(v3, r[3].y & 63) : neg_inf;
            }
            tc_fence_before();
            mbar_arrive(&sm.tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
            // fold into the documents, in chunk order; a document's sum at its last chunk
            const int pb = n & (kMsPartBufs - 1);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (r[c].x < 0) continue;
                run = (r[c].y & kInfoFirst) ? m[c] : fmaxf(run, m[c]);
                if (r[c].y & kInfoLast) {
                    const float s = warp_sum(row_ok ? run : 0.f);
                    if (lane == 0) {
                        if (nwarps == 1)
                            a.scores[r[c].x] = a.accumulate ? a.scores[r[c].x] + s : s;
                        else
                            sm.part[(pb * 4 + c) * 4 + qw] = s;
                    }
                }
            }
            if (nwarps > 1 && lane == 0) {
                // the warp that finishes the tile last adds the warps' sums in warp order
                __threadfence_block();
                const int before = atomicAdd(&sm.part_cnt[pb], 1);
                if (before == nwarps - 1) {
                    __threadfence_block();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (r[c].x >= 0 && (r[c].y & kInfoLast)) {
                            float s = 0.f;
                            for (int w = 0; w < nwarps; ++w) s += sm.part[(pb * 4 + c) * 4 + w];
                            a.scores[r[c].x] = a.accumulate ? a.scores[r[c].x] + s : s;
                        }
                    }
                    sm.part_cnt[pb] = 0;
                }
            }
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            report(a.status, kStTimeout);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) {
        __syncwarp();
        tmem_dealloc(tmem, a.tmem_cols);
    }
    if (threadIdx.x == 0) {
        // the last CTA to finish returns the grab counter and this done count to zero, so the
        // workspace is ready for the next launch (every CTA's atomics have completed by now)
        __threadfence();
        if (atomicAdd(a.counter + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            atomicExch(a.counter, 0);
            atomicExch(a.counter + 1, 0);
        }
    }
}

// Scores of a query with no rows: every document sums nothing.
__global__ void k_fill_f32(float* out, int n, float v) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) out[i] = v;
}

size_t maxsim_smem_bytes(int stages, int nq_pad, int kslabs) {
    return 1024 + static_cast<size_t>(kslabs) * nq_pad * 128u + static_cast<size_t>(stages) * kMsSlabBytes +
           kMsRing * kMsRec * sizeof(int) + kMsInfo * 8 * sizeof(int) + kMsPartBufs * (16 * sizeof(float) + sizeof(int)) +
           2 * 2 * 32 * sizeof(int) + (2 * static_cast<size_t>(stages) + 4 + 2 * kMsRing + 2 * kMsInfo + 2) * 8 + 16;
}

cudaError_t launch_maxsim(const MaxsimArgs& a, const MaxsimMaps& maps, int grid, size_t smem, cudaStream_t s) {
    static size_t configured[kMaxDevicesTracked] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevicesTracked && smem > configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_maxsim, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = smem;
    }
    k_maxsim<<<grid, kMaxsimThreads, smem, s>>>(a, maps);
    return cudaGetLastError();
}

cudaError_t launch_fill_f32(float* out, int n, float v, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int grid = static_cast<int>(std::min<int64_t>(1024, (static_cast<int64_t>(n) + 255) / 256));
    k_fill_f32<<<grid, 256, 0, s>>>(out, n, v);
    return cudaGetLastError();
}

}  // namespace sel
