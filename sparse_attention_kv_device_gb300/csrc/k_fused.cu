// The fused selection, one persistent kernel per chunk of rows: request segments,
// tensor-core scoring, exact top-k pools, expansion with the trailing pool, and the
// block-table remap.
//
// What it computes (the sources' statement of the problem):
//   * ReVolta PR #59 ("Change"): rows of one request form segments that share the
//     request's key page table, so each 64-key page is read once per segment and
//     multiplied against all of the segment's rows x 4 heads; segment descriptors are
//     built on the device so the call stays CUDA-graph safe. The score of pool j for
//     row r is sum_{h<4} q[r][h] . key(j), accumulated in fp32.
//   * vLLM flashinfer_mla_sparse_sm90 page (_kv_lens_host): row context = position + 1;
//     a row with context <= index_topk keeps every token; a longer one keeps the
//     index_topk / kpool best complete pools (score descending, lower pool first),
//     expanded to tokens, plus the trailing incomplete pool.
//   * vLLM sparse_utils page (triton_convert_req_index_to_global_index): slot =
//     block_table[req][t / block_size] * block_stride_rows + t % block_size, -1 for empty
//     entries and out-of-bounds blocks, valid counts in the same pass without atomics.
//
// How (GB300): a cooperative grid of one CTA per SM; every CTA plans the chunk itself
// from query_start_loc and positions (no separate builder launch). Roles by warp:
//   warp 0      tile scheduler + TMA producer (key pages into a ring of stages, queries
//               of the segment into a double buffer);
//   warp 1      tcgen05.mma issuer (M = 128 pools, N = rows x 4 heads, fp16 in, fp32 in TMEM);
//   warps 2-5   epilogue: per pool and row the 4-head sum, stored as an order-preserving
//               32-bit key, and per row and 32-pool group the two largest keys (with the
//               lane of the largest) -- the group records;
//   warp 6      signal: when a tile's keys are stored it counts the tile against its
//               segment (release at GPU scope); the CTA that stores a segment's last tile
//               publishes the segment's rows as select jobs;
//   warps 7-14  select: claim rows from a job counter (rows needing no scoring first), and
//               for each row take the index_topk / kpool best pools exactly:
//                 T = a lower bound on the K-th key from the group records (their K-th
//                     largest value: each is a key of a distinct pool),
//                 candidates = every key >= T: directly from a record when the group's
//                     second key is below T, else by reading the group's 32 keys,
//                 a radix select over the candidates (bits below the prefix that T and the
//                     row's largest key share), the lowest pool index winning ties,
//                 then ascending order by a bitmap scan, expansion, remap and count.
//               A row whose candidates exceed their buffer is selected over all its keys.
// Rows are selected while later tiles are still being scored. Every wait is bounded and
// reports SEL_ST_TIMEOUT. The counter words in the workspace must be zero when the launch
// starts; the last CTA to finish returns them to zero.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

constexpr int kSchedRing = 16;
constexpr int T_ALL = kFusedThreads;
constexpr int NTS = kFusedSelThreads;
constexpr int kSelWarp0 = kFusedSelWarp0;
constexpr int kSignalWarp = kFusedSignalWarp;
constexpr int kHistBins = 2048;
constexpr int kScanCap = 1024;       // groups read in full per row (more: the row is selected over all its keys)
constexpr int kWarpPlanReqs = 2048;  // batches with more requests are planned by the whole CTA
constexpr int kMaxPlanRows = kFusedMaxChunkRows;
static_assert(T_ALL == 32 * (kSelWarp0 + NTS / 32), "warp roles cover the CTA");
static_assert(NTS == 256, "select helpers assume 8 warps");

// counter block (int32 words at a.ctr)
constexpr int kCtrTile = 0;    // dynamic tile counter
constexpr int kCtrJobHead = 1; // jobs claimed
constexpr int kCtrJobTail = 2; // jobs published
constexpr int kCtrExit = 3;    // CTAs finished
constexpr int kCtrAbort = 4;   // a wait expired somewhere in the grid

struct Smem {
    uint8_t* a;          // stages x kTileBytes
    uint8_t* q;          // 2 x npad_max x 256 B
    int4* segs;          // [max_segs] {request, first row, rows, pools}
    int* prefix;         // [max_segs + 1]
    int4* rec_ring;      // [kSchedRing]
    int* tile_ring;      // [kSchedRing]
    uint64_t *full, *empty, *tfull, *tempty, *qfull, *qempty, *sfull, *sempty, *tdone, *done;
    int* words;          // [16]
    int32_t *p_ctx, *p_req, *p_lim, *p_triv;  // [chunk_cap] each
    int32_t* btab;       // select: [bt_cap]
    uint32_t* hist;      // select: [kHistBins]; also the list of groups to scan
    uint32_t* ckey;      // select: [cand_cap]
    int32_t* cidx;       // select: [cand_cap]
    uint2* rec;          // select: [gcap] group records; later the kept / equal bitmaps
    uint32_t* kbm;       // = rec (words [0, gcap))
    uint32_t* ebm;       // = rec + gcap words
    int32_t* list;       // select: [K]
    uint32_t* small_key; // select: [64] keys of a last, small range
    int32_t* small_idx;  // select: [64]
    uint32_t* scan_mask; // select: [kScanCap] keys >= T of each group read in full
    int32_t* scan_off;   // select: [kScanCap] their first place in the candidate list
    uint32_t* scratch;   // select: [64]
};

// word slots in Smem::words
constexpr int kWTmem = 0, kWAbort = 1, kWOob = 2, kWNseg = 3, kWNtiles = 4, kWNtriv = 5, kWBad = 6, kWJob = 7,
              kWCand = 8, kWScan = 9, kWSmall = 10, kWCount = 11;

__device__ __forceinline__ Smem carve(uint8_t* raw, const FusedArgs& a) {
    const uint32_t base = smem_u32(raw);
    uint8_t* p = raw + (((base + 1023u) & ~1023u) - base);
    const FusedLayout& L = a.lay;
    Smem s;
    s.a = p + L.a;
    s.q = p + L.q;
    s.segs = reinterpret_cast<int4*>(p + L.segs);
    s.prefix = reinterpret_cast<int*>(p + L.prefix);
    s.rec_ring = reinterpret_cast<int4*>(p + L.rec_ring);
    s.tile_ring = reinterpret_cast<int*>(p + L.tile_ring);
    uint64_t* b = reinterpret_cast<uint64_t*>(p + L.bars);
    s.full = b;
    s.empty = b + a.stages;
    s.tfull = b + 2 * a.stages;
    s.tempty = s.tfull + 2;
    s.qfull = s.tempty + 2;
    s.qempty = s.qfull + 2;
    s.sfull = s.qempty + 2;
    s.sempty = s.sfull + kSchedRing;
    s.tdone = s.sempty + kSchedRing;
    s.done = s.tdone + kSchedRing;
    s.words = reinterpret_cast<int*>(p + L.words);
    s.p_ctx = reinterpret_cast<int32_t*>(p + L.p_ctx);
    s.p_req = reinterpret_cast<int32_t*>(p + L.p_req);
    s.p_lim = reinterpret_cast<int32_t*>(p + L.p_lim);
    s.p_triv = reinterpret_cast<int32_t*>(p + L.p_triv);
    s.btab = reinterpret_cast<int32_t*>(p + L.s_btab);
    s.hist = reinterpret_cast<uint32_t*>(p + L.s_hist);
    s.ckey = reinterpret_cast<uint32_t*>(p + L.s_ckey);
    s.cidx = reinterpret_cast<int32_t*>(p + L.s_cidx);
    s.rec = reinterpret_cast<uint2*>(p + L.s_rec);
    s.kbm = reinterpret_cast<uint32_t*>(p + L.s_rec);
    s.ebm = s.kbm + a.gcap;
    s.list = reinterpret_cast<int32_t*>(p + L.s_list);
    s.small_key = reinterpret_cast<uint32_t*>(p + L.s_small);
    s.small_idx = reinterpret_cast<int32_t*>(p + L.s_small + 256);
    s.scan_mask = reinterpret_cast<uint32_t*>(p + L.s_scan);
    s.scan_off = reinterpret_cast<int32_t*>(p + L.s_scan + 4 * kScanCap);
    s.scratch = reinterpret_cast<uint32_t*>(p + L.s_scratch);
    return s;
}

// ------------------------------------------------------------------ select-group helpers
// The select warps synchronise among themselves with named barrier 1. Every helper below
// ends its use of the scratch words with at least one barrier and alternates between two
// scratch areas (the caller's `ph`), so consecutive helpers never race on them.
__device__ __forceinline__ void sbar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan over the 256 select threads (one barrier); the total goes to *total.
__device__ __forceinline__ uint32_t s_scan(uint32_t v, uint32_t* scratch, uint32_t* total, int gt, int& ph) {
    const int lane = gt & 31, w = gt >> 5;
    const uint32_t incl = warp_incl_scan(v);
    uint32_t* buf = scratch + 8 * ph;
    ph ^= 1;
    if (lane == 31) buf[w] = incl;
    sbar();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < NTS / 32; ++i) {
        const uint32_t x = buf[i];
        before += i < w ? x : 0u;
        tot += x;
    }
    *total = tot;
    return before + incl - v;
}

// Minimum and maximum over the select threads (one barrier).
__device__ __forceinline__ void s_minmax(uint32_t& mn, uint32_t& mx, uint32_t* scratch, int gt, int& ph) {
    mn = __reduce_min_sync(0xffffffffu, mn);
    mx = __reduce_max_sync(0xffffffffu, mx);
    uint32_t* buf = scratch + 32 + 16 * ph;
    ph ^= 1;
    if ((gt & 31) == 0) {
        buf[gt >> 5] = mn;
        buf[8 + (gt >> 5)] = mx;
    }
    sbar();
    mn = buf[0];
    mx = buf[8];
#pragma unroll
    for (int i = 1; i < NTS / 32; ++i) {
        mn = min(mn, buf[i]);
        mx = max(mx, buf[8 + i]);
    }
}

// Among nb histogram bins (nb <= 2048), the bin, counted from the top, in which the
// cumulative count first reaches `need`; `above` = keys in higher bins, `cnt` = the bin's
// (two barriers).
__device__ __forceinline__ void s_find_bin(const uint32_t* hist, int nb, uint32_t need, uint32_t* scratch, int gt,
                                           int& ph, uint32_t& bin, uint32_t& above, uint32_t& cnt) {
    const int per = (nb + NTS - 1) / NTS;  // <= 8
    const int hi = nb - 1 - gt * per;
    uint32_t h[8];
    uint32_t local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int b = hi - i;
        h[i] = (i < per && b >= 0) ? hist[b] : 0u;
        local += h[i];
    }
    if (gt == 0) {
        scratch[16] = 0u;
        scratch[17] = 0u;
        scratch[18] = need;
    }
    uint32_t tot;
    const uint32_t ab = s_scan(local, scratch, &tot, gt, ph);
    if (ab < need && need <= ab + local) {
        uint32_t acc = ab;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (acc < need && acc + h[i] >= need) {
                scratch[16] = static_cast<uint32_t>(hi - i);
                scratch[17] = acc;
                scratch[18] = h[i];
            }
            acc += h[i];
        }
    }
    sbar();
    bin = scratch[16];
    above = scratch[17];
    cnt = scratch[18];
}

// A range of keys [lo, lo + 2^shift) that holds the need-th largest key of a source;
// cnt = the source's keys inside it (known after a level).
struct Range {
    uint32_t lo;
    int shift;       // 0..32
    uint32_t need;   // keys still to take from inside the range (all keys above it are kept)
    uint32_t cnt;
};

__device__ __forceinline__ bool in_range(uint32_t k, uint32_t lo, int shift) {
    return k >= lo && static_cast<uint64_t>(k - lo) < (1ull << shift);
}

// One radix level: counts the range's keys by the next (up to) 11 bits below `shift`
// (the histogram must be zero on entry), and narrows the range to the bin holding the
// need-th largest key.
template <class Visit>
__device__ __forceinline__ void s_level(Visit visit, Range& R, uint32_t* hist, uint32_t* scratch, int gt, int& ph) {
    const int b = R.shift < 11 ? R.shift : 11;
    const int ns = R.shift - b;
    const uint32_t lo = R.lo;
    const int sh = R.shift;
    visit([&](uint32_t k, int) {
        if (in_range(k, lo, sh)) atomicAdd(&hist[(k - lo) >> ns], 1u);
    });
    sbar();
    uint32_t bin, above, cnt;
    s_find_bin(hist, 1 << b, R.need, scratch, gt, ph, bin, above, cnt);
    R.lo = lo + (bin << ns);
    R.shift = ns;
    R.need -= above;
    R.cnt = cnt;
}

__device__ __forceinline__ int bitlen(uint32_t x) { return x ? 32 - __clz(x) : 0; }

__device__ __forceinline__ int32_t slot_of(const FusedArgs& a, const int32_t* btab, int nblk, const int32_t* bt_row,
                                           int32_t t) {
    if (t < 0) return -1;
    const int32_t b = a.bs_shift >= 0 ? (t >> a.bs_shift) : t / a.block_size;
    int32_t ph;
    if (b < nblk) {
        ph = btab[b];
    } else {
        if (b >= a.max_blocks) return -1;
        ph = __ldg(bt_row + b);
    }
    if (ph < 0 || ph >= a.num_kv_blocks) return -1;
    return static_cast<int32_t>(static_cast<int64_t>(ph) * a.block_stride_rows + (t - b * a.block_size));
}

// Warp-aggregated append: lane items j < N with take[j] get consecutive slots of the
// counter, one shared-memory atomic per warp for the whole batch; emit(j, slot) stores item j.
template <int N, class Emit>
__device__ __forceinline__ void warp_append_n(const bool (&take)[N], int* counter, Emit emit) {
    uint32_t m[N];
    int tot = 0;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        m[j] = __ballot_sync(0xffffffffu, take[j]);
        tot += __popc(m[j]);
    }
    int base = 0;
    if ((threadIdx.x & 31) == 0 && tot) base = atomicAdd(counter, tot);
    base = __shfl_sync(0xffffffffu, base, 0);
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int j = 0; j < N; ++j) {
        if (take[j]) emit(j, base + __popc(m[j] & lt));
        base += __popc(m[j]);
    }
}

__device__ __forceinline__ void set_bit(uint32_t* bm, int p) { atomicOr(bm + (p >> 5), 1u << (p & 31)); }

// Marks the `need` best keys of a source in the kept bitmap, given a range that holds the
// need-th largest key: every key above the range is kept; inside it, the keys are either
// all kept (cnt == need), ranked one by one when few (the lower pool index first among
// equal keys), or narrowed further level by level down to one value, whose equal keys are
// then taken in ascending pool order.
template <class Visit>
__device__ __forceinline__ void s_take_best(Visit visit, Range R, const Smem& sm, int nw, int gt, int& ph) {
    constexpr uint32_t kSmall = 64;
    for (;;) {
        const uint64_t hi = static_cast<uint64_t>(R.lo) + (1ull << R.shift);  // keys >= hi are kept
        if (R.cnt == R.need) {
            const uint32_t lo = R.lo;
            visit([&](uint32_t k, int p) {
                if (k >= lo) set_bit(sm.kbm, p);
            });
            sbar();
            return;
        }
        if (R.cnt <= kSmall) {
            const uint32_t lo = R.lo;
            const int sh = R.shift;
            int* ns = sm.words + kWSmall;
            visit([&](uint32_t k, int p) {
                if (static_cast<uint64_t>(k) >= hi) {
                    set_bit(sm.kbm, p);
                } else if (in_range(k, lo, sh)) {
                    const int i = atomicAdd(ns, 1);
                    if (i < static_cast<int>(kSmall)) {
                        sm.small_key[i] = k;
                        sm.small_idx[i] = p;
                    }
                }
            });
            sbar();
            const int m = min(*ns, static_cast<int>(kSmall));
            if (gt < m) {
                const uint32_t kj = sm.small_key[gt];
                const int ij = sm.small_idx[gt];
                uint32_t rank = 0;
                for (int i = 0; i < m; ++i) {
                    const uint32_t ki = sm.small_key[i];
                    rank += (ki > kj || (ki == kj && sm.small_idx[i] < ij)) ? 1u : 0u;
                }
                if (rank < R.need) set_bit(sm.kbm, ij);
            }
            sbar();
            return;
        }
        if (R.shift == 0) {
            // one value with more equal keys than needed: the lowest pool indices win
            const uint32_t thr = R.lo;
            visit([&](uint32_t k, int p) {
                if (k > thr) set_bit(sm.kbm, p);
                else if (k == thr) set_bit(sm.ebm, p);
            });
            sbar();
            const int per = (nw + NTS - 1) / NTS;
            const int w0 = gt * per, w1 = min(nw, w0 + per);
            uint32_t eqc = 0;
            for (int w = w0; w < w1; ++w) eqc += __popc(sm.ebm[w]);
            uint32_t tot;
            uint32_t before = s_scan(eqc, sm.scratch, &tot, gt, ph);
            for (int w = w0; w < w1; ++w) {
                const uint32_t e = sm.ebm[w];
                uint32_t take_mask = 0;
                if (before < R.need && e) {
                    uint32_t take = min(static_cast<uint32_t>(__popc(e)), R.need - before);
                    uint32_t rest = e;
                    while (take--) {
                        const uint32_t lowest = rest & (0u - rest);
                        take_mask |= lowest;
                        rest ^= lowest;
                    }
                }
                before += __popc(e);
                if (take_mask) atomicOr(sm.kbm + w, take_mask);
            }
            sbar();
            return;
        }
        for (int i = gt; i < kHistBins; i += NTS) sm.hist[i] = 0u;
        sbar();
        s_level(visit, R, sm.hist, sm.scratch, gt, ph);
    }
}

// Marks (with the sign bit of cidx) the `need` best keys of a candidate list that is in
// ascending pool order, given a range [R.lo, R.lo + 2^R.shift) that holds the need-th
// largest key: every candidate above the range is kept; inside it the keys are all kept
// (cnt == need), ranked one by one when few (the lower pool index first among equal keys),
// or narrowed level by level down to one value, whose first equal keys in list order (the
// lowest pool indices) are kept.
__device__ __forceinline__ void s_take_best_list(int nc, Range R, const Smem& sm, int gt, int& ph) {
    constexpr uint32_t kSmall = 64;
    auto cand = [&](auto f) {
        for (int i = gt; i < nc; i += NTS) f(sm.ckey[i], i);
    };
    for (;;) {
        const uint64_t hi = static_cast<uint64_t>(R.lo) + (1ull << R.shift);
        const uint32_t lo = R.lo;
        const int sh = R.shift;
        if (R.cnt == R.need) {
            for (int i = gt; i < nc; i += NTS)
                if (sm.ckey[i] >= lo) sm.cidx[i] |= static_cast<int32_t>(0x80000000u);
            sbar();
            return;
        }
        if (R.cnt <= kSmall) {
            int* ns = sm.words + kWSmall;
            for (int i = gt; i < nc; i += NTS) {
                const uint32_t k = sm.ckey[i];
                if (static_cast<uint64_t>(k) >= hi) {
                    sm.cidx[i] |= static_cast<int32_t>(0x80000000u);
                } else if (in_range(k, lo, sh)) {
                    const int j = atomicAdd(ns, 1);
                    if (j < static_cast<int>(kSmall)) sm.small_idx[j] = i;
                }
            }
            sbar();
            const int m = min(*ns, static_cast<int>(kSmall));
            if (gt < m) {
                const int ij = sm.small_idx[gt];
                const uint32_t kj = sm.ckey[ij];
                uint32_t rank = 0;
                for (int j = 0; j < m; ++j) {
                    const int ii = sm.small_idx[j];
                    const uint32_t ki = sm.ckey[ii];
                    rank += (ki > kj || (ki == kj && ii < ij)) ? 1u : 0u;  // list order = pool order
                }
                if (rank < R.need) sm.cidx[ij] |= static_cast<int32_t>(0x80000000u);
            }
            sbar();
            return;
        }
        if (sh == 0) {
            // one value with more equal keys than needed: the first ones in list order
            const int per = (nc + NTS - 1) / NTS;
            const int i0 = gt * per, i1 = min(nc, i0 + per);
            uint32_t eqc = 0;
            for (int i = i0; i < i1; ++i) {
                const uint32_t k = sm.ckey[i];
                if (k > lo) sm.cidx[i] |= static_cast<int32_t>(0x80000000u);
                eqc += k == lo;
            }
            uint32_t tot;
            uint32_t before = s_scan(eqc, sm.scratch, &tot, gt, ph);
            for (int i = i0; i < i1; ++i)
                if (sm.ckey[i] == lo) {
                    if (before < R.need) sm.cidx[i] |= static_cast<int32_t>(0x80000000u);
                    ++before;
                }
            sbar();
            return;
        }
        for (int i = gt; i < kHistBins; i += NTS) sm.hist[i] = 0u;
        sbar();
        s_level(cand, R, sm.hist, sm.scratch, gt, ph);
    }
}

// One row of the chunk: select (when it was scored), expand, remap, count.
__device__ void select_row(const FusedArgs& a, const Smem& sm, int rl, int gt) {
    const int r = a.row_begin + rl;
    const int32_t c = sm.p_ctx[rl];
    const int req = sm.p_req[rl];
    const bool valid = c >= 0 && req >= 0;
    const int64_t ctx = valid ? c : 0;
    const int P = sm.p_lim[rl];  // > 0: the row was scored (ctx > index_topk)
    const int K = a.topk / a.kpool;
    int ph = 0;
    const int32_t* bt_row = a.block_table + static_cast<int64_t>(valid ? req : 0) * a.bt_ld;
    int nblk = 0;
    if (valid) {
        int64_t need = (ctx + a.block_size - 1) / a.block_size;
        if (need > a.max_blocks) need = a.max_blocks;
        nblk = static_cast<int>(need < a.bt_cap ? need : a.bt_cap);
        if ((reinterpret_cast<uintptr_t>(bt_row) & 15u) == 0) {
            const int n4 = nblk >> 2;
            for (int i = gt; i < n4; i += NTS) cp_async_16(sm.btab + 4 * i, bt_row + 4 * i);
            for (int i = 4 * n4 + gt; i < nblk; i += NTS) cp_async_4(sm.btab + i, bt_row + i);
        } else {
            for (int i = gt; i < nblk; i += NTS) cp_async_4(sm.btab + i, bt_row + i);
        }
    }
    if (gt == 0) {
        sm.words[kWSmall] = 0;
        sm.words[kWCount] = 0;
    }
    int64_t run_from = 0;
    int col_run = 0;
    if (P > 0) {
        const uint32_t* krow = a.keys + static_cast<int64_t>(rl) * a.keys_ld;
        const int G = (P + 31) >> 5;
        const bool use_rec = 2 * G >= K;
        if (use_rec) {
            const uint4* src = reinterpret_cast<const uint4*>(a.grp + static_cast<int64_t>(rl) * a.grp_ld);
            uint4* dst = reinterpret_cast<uint4*>(sm.rec);
            for (int i = gt; i < (G + 1) / 2; i += NTS) cp_async_16(dst + i, src + i);
        }
        for (int i = gt; i < kHistBins; i += NTS) sm.hist[i] = 0u;
        cp_async_wait_all();
        sbar();
        uint32_t T = 0, vmax = 0;
        bool overflow = false;
        int nc = 0;
        if (use_rec) {
            // ---- T: the lower edge of the histogram bin that holds the K-th largest record
            //      value (m1 and m2 rounded down; each a key of a distinct pool)
            uint32_t mn = 0xffffffffu, mx = 0;
            for (int g = gt; g < G; g += NTS) {
                const uint2 v = sm.rec[g];
                mx = max(mx, v.x);
                mn = min(mn, K <= G ? v.x : min(v.x, v.y & ~31u));  // with K <= G the K-th is >= every m1's minimum
            }
            s_minmax(mn, mx, sm.scratch, gt, ph);
            vmax = mx;
            T = mx;
            if (mx != mn) {
                Range R{mn, bitlen(mx - mn), static_cast<uint32_t>(K), 0u};
                s_level(
                    [&](auto f) {
                        for (int g = gt; g < G; g += NTS) {
                            const uint2 v = sm.rec[g];
                            f(v.x, 0);
                            f(v.y & ~31u, 0);
                        }
                    },
                    R, sm.hist, sm.scratch, gt, ph);
                T = R.lo;
            }
            // ---- candidates = every key >= T, in ascending pool order. Each thread owns a
            //      contiguous run of groups; a group whose second key is below T gives its
            //      first key, the others are read in full.
            const int gpt = (G + NTS - 1) / NTS;
            const int g0 = gt * gpt, g1 = min(G, g0 + gpt);
            uint32_t nsc = 0;
            for (int g = g0; g < g1; ++g) {
                const uint2 v = sm.rec[g];
                nsc += (v.x >= T && ((v.y & ~31u) | 31u) >= T) ? 1u : 0u;
            }
            uint32_t nscan;
            const uint32_t sbase = s_scan(nsc, sm.scratch, &nscan, gt, ph);
            int32_t* scan_g = reinterpret_cast<int32_t*>(sm.hist);  // the histogram is free again
            overflow = nscan > static_cast<uint32_t>(kScanCap);
            if (!overflow) {
                uint32_t e = sbase;
                for (int g = g0; g < g1; ++g) {
                    const uint2 v = sm.rec[g];
                    if (v.x >= T && ((v.y & ~31u) | 31u) >= T) scan_g[e++] = g;
                }
            }
            sbar();
            const int w = gt >> 5, lane = gt & 31;
            const int ns = overflow ? 0 : static_cast<int>(nscan);
            // the listed groups' keys: warp w reads entries w, w + 8, ... (one key per lane);
            // up to 16 entries per warp stay in registers for the write below
            uint32_t kreg[16];
            for (int e0 = 0; e0 < ns; e0 += 128) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int e = e0 + w + 8 * u;
                    const int p = e < ns ? scan_g[e] * 32 + lane : P;
                    kreg[u] = p < P ? __ldcg(krow + p) : 0u;
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int e = e0 + w + 8 * u;
                    const uint32_t m = __ballot_sync(0xffffffffu, kreg[u] >= T && e < ns &&
                                                                      scan_g[e] * 32 + lane < P);
                    if (lane == 0 && e < ns) sm.scan_mask[e] = m;
                }
            }
            sbar();
            // per-thread candidate counts over its groups, then their places in the list
            uint32_t cnt = 0;
            {
                uint32_t e = sbase;
                for (int g = g0; g < g1; ++g) {
                    const uint2 v = sm.rec[g];
                    if (v.x >= T) {
                        if (((v.y & ~31u) | 31u) >= T) cnt += overflow ? 0u : __popc(sm.scan_mask[e++]);
                        else cnt += 1;
                    }
                }
            }
            uint32_t total;
            uint32_t off = s_scan(cnt, sm.scratch, &total, gt, ph);
            overflow = overflow || total > static_cast<uint32_t>(a.cand_cap);
            if (!overflow) {
                uint32_t e = sbase;
                for (int g = g0; g < g1; ++g) {
                    const uint2 v = sm.rec[g];
                    if (v.x >= T) {
                        if (((v.y & ~31u) | 31u) >= T) {
                            sm.scan_off[e] = static_cast<int>(off);
                            off += __popc(sm.scan_mask[e++]);
                        } else {
                            sm.ckey[off] = v.x;
                            sm.cidx[off] = g * 32 + static_cast<int>(v.y & 31u);
                            ++off;
                        }
                    }
                }
            }
            sbar();
            if (!overflow) {
                const uint32_t lt = lanemask_lt();
                for (int e0 = 0; e0 < ns; e0 += 128) {
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int e = e0 + w + 8 * u;
                        if (e < ns) {
                            const int p = scan_g[e] * 32 + lane;
                            const uint32_t k = ns <= 128 ? kreg[u] : (p < P ? __ldcg(krow + p) : 0u);
                            const uint32_t m = sm.scan_mask[e];
                            if ((m >> lane) & 1u) {
                                const int at = sm.scan_off[e] + __popc(m & lt);
                                sm.ckey[at] = k;
                                sm.cidx[at] = p;
                            }
                        }
                    }
                }
            }
            sbar();
            nc = static_cast<int>(total);
        } else if (P <= a.cand_cap) {
            // every key is a candidate
            for (int p = gt; p < P; p += NTS) {
                const uint32_t k = __ldcg(krow + p);
                sm.ckey[p] = k;
                sm.cidx[p] = p;
                vmax = max(vmax, k);
            }
            uint32_t mn = 0;
            s_minmax(mn, vmax, sm.scratch, gt, ph);
            nc = P;
        } else {
            overflow = true;
        }
        if (P == K) {
            // every pool is kept (marked in the bitmap below)
        } else if (!overflow) {
            // candidates: every key >= T, ascending pool order; start from the range [T, vmax]
            for (int i = gt; i < kHistBins; i += NTS) sm.hist[i] = 0u;
            sbar();
            auto cand = [&](auto f) {
                for (int i = gt; i < nc; i += NTS) f(sm.ckey[i], i);
            };
            Range R{T, bitlen(vmax - T), static_cast<uint32_t>(K), static_cast<uint32_t>(nc)};
            if (R.shift > 0) s_level(cand, R, sm.hist, sm.scratch, gt, ph);
            s_take_best_list(nc, R, sm, gt, ph);
        }
        if (P == K || overflow) {
            // every key of the row, read from L2: kept pools marked in a bitmap
            const int nw = G;
            for (int i = gt; i < nw; i += NTS) {
                sm.kbm[i] = 0u;
                sm.ebm[i] = 0u;
            }
            for (int i = gt; i < kHistBins; i += NTS) sm.hist[i] = 0u;
            sbar();
            if (P == K) {
                for (int p = gt; p < P; p += NTS) set_bit(sm.kbm, p);
                sbar();
            } else {
                auto all_keys = [&](auto f) {
                    const uint4* k4 = reinterpret_cast<const uint4*>(krow);
                    const int full4 = P >> 2;
                    for (int base = gt; base < full4; base += 4 * NTS) {
                        uint4 v[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int i4 = base + j * NTS;
                            v[j] = i4 < full4 ? __ldcg(k4 + i4) : make_uint4(0u, 0u, 0u, 0u);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int i4 = base + j * NTS;
                            if (i4 < full4) {
                                f(v[j].x, 4 * i4);
                                f(v[j].y, 4 * i4 + 1);
                                f(v[j].z, 4 * i4 + 2);
                                f(v[j].w, 4 * i4 + 3);
                            }
                        }
                    }
                    for (int p = 4 * full4 + gt; p < P; p += NTS) f(__ldcg(krow + p), p);
                };
                Range R{0u, 32, static_cast<uint32_t>(K), static_cast<uint32_t>(P)};
                s_level(all_keys, R, sm.hist, sm.scratch, gt, ph);
                s_take_best(all_keys, R, sm, nw, gt, ph);
            }
            // kept pools in ascending order from the bitmap
            const int per = (nw + NTS - 1) / NTS;
            const int w0 = gt * per, w1 = min(nw, w0 + per);
            uint32_t keptc = 0;
            for (int w = w0; w < w1; ++w) keptc += __popc(sm.kbm[w]);
            uint32_t tot;
            uint32_t pos = s_scan(keptc, sm.scratch, &tot, gt, ph);
            for (int w = w0; w < w1; ++w) {
                uint32_t kept = sm.kbm[w];
                while (kept) {
                    const int bit = __ffs(kept) - 1;
                    kept &= kept - 1;
                    if (pos < static_cast<uint32_t>(K)) sm.list[pos] = w * 32 + bit;
                    ++pos;
                }
            }
        } else {
            // kept candidates in list order (ascending pools)
            const int per = (nc + NTS - 1) / NTS;
            const int i0 = gt * per, i1 = min(nc, i0 + per);
            uint32_t keptc = 0;
            for (int i = i0; i < i1; ++i) keptc += sm.cidx[i] < 0 ? 1u : 0u;
            uint32_t tot;
            uint32_t pos = s_scan(keptc, sm.scratch, &tot, gt, ph);
            for (int i = i0; i < i1; ++i) {
                const int32_t ci = sm.cidx[i];
                if (ci < 0) {
                    if (pos < static_cast<uint32_t>(K)) sm.list[pos] = ci & 0x7fffffff;
                    ++pos;
                }
            }
        }
        run_from = static_cast<int64_t>(P) * a.kpool;
        col_run = K * a.kpool;
    }
    cp_async_wait_all();  // the block-table entries
    sbar();

    // ---- one column per thread: kept pools' tokens, trailing tokens (for a short row,
    //      every token), then -1; remapped; the valid count
    int32_t* slot_row = a.slots + static_cast<int64_t>(r) * a.out_width;
    int32_t* tok_row = a.token_idx ? a.token_idx + static_cast<int64_t>(r) * a.out_width : nullptr;
    uint32_t vcount = 0;
#pragma unroll 4
    for (int col = gt; col < a.out_width; col += NTS) {
        int32_t t;
        if (col < col_run) {
            const int qq = a.kpool_shift >= 0 ? (col >> a.kpool_shift) : col / a.kpool;
            t = sm.list[qq] * a.kpool + (col - qq * a.kpool);
        } else {
            const int64_t tt = run_from + (col - col_run);
            t = valid && tt < ctx ? static_cast<int32_t>(tt) : -1;
        }
        const int32_t s = slot_of(a, sm.btab, nblk, bt_row, t);
        slot_row[col] = s;
        if (tok_row) tok_row[col] = t;
        vcount += s != -1;
    }
    vcount = __reduce_add_sync(0xffffffffu, vcount);
    if ((gt & 31) == 0) atomicAdd(sm.words + kWCount, static_cast<int>(vcount));
    sbar();
    if (gt == 0 && a.counts) a.counts[r] = sm.words[kWCount];
}

// The plan of a chunk by every thread of the CTA (batches with many requests).
__device__ __forceinline__ void plan_cta(const FusedArgs& a, const Smem& sm, int tid) {
    const int rb = a.row_begin;
    const int nchunk = a.row_end - a.row_begin;
    int* words = sm.words;
    for (int r = tid; r < nchunk; r += T_ALL) {
        const int64_t c64 = static_cast<int64_t>(__ldg(a.positions + rb + r)) + 1;
        sm.p_ctx[r] = c64 > 0x7fffffff ? 0x7fffffff : (c64 < 0 ? 0 : static_cast<int32_t>(c64));
        sm.p_req[r] = -1;
    }
    int bad = 0;
    if (tid == 0) bad = (__ldg(a.qsl) < 0) | (__ldg(a.qsl + a.num_reqs) > a.num_rows);
    __syncthreads();
    {
        uint32_t carry = 0;
        for (int base = 0; base < a.num_reqs; base += T_ALL) {
            const int i = base + tid;
            int lo = 0, hi = 0;
            uint32_t ns = 0;
            if (i < a.num_reqs) {
                const int x = __ldg(a.qsl + i), y = __ldg(a.qsl + i + 1);
                bad |= x > y;
                lo = max(x, a.row_begin);
                hi = min(y, a.row_end);
                if (hi > lo) ns = static_cast<uint32_t>((hi - lo + a.seg_rows - 1) / a.seg_rows);
            }
            uint32_t total;
            const uint32_t first = carry + block_excl_scan(ns, reinterpret_cast<uint32_t*>(sm.hist), &total);
            for (uint32_t k = 0; k < ns; ++k) {
                const uint32_t s = first + k;
                if (s >= static_cast<uint32_t>(a.max_segs)) break;  // bounded by the host's max_segs
                const int row0 = lo + static_cast<int>(k) * a.seg_rows;
                sm.segs[s] = make_int4(i, row0, min(a.seg_rows, hi - row0), 0);
            }
            for (int r = lo; r < hi; ++r) sm.p_req[r - rb] = i;
            carry += total;
            __syncthreads();
        }
        bad = __syncthreads_or(bad);
        if (tid == 0) {
            words[kWNseg] = bad ? 0 : min(static_cast<int>(carry), a.max_segs);
            words[kWBad] = bad;
        }
    }
    __syncthreads();
    const int nseg = words[kWNseg];
    for (int r = tid; r < nchunk; r += T_ALL) {
        int32_t c = sm.p_ctx[r];
        int req = bad ? -1 : sm.p_req[r];
        if (req >= 0 && c > a.max_context) {
            if (blockIdx.x == 0) report(a.status, kStCtxOverBound);
            req = -1;
        }
        if (req < 0) c = -1;
        sm.p_req[r] = req;
        sm.p_ctx[r] = c;
        sm.p_lim[r] = (c > 0 && (a.score_all ? c >= a.kpool : c > a.topk)) ? min(c / a.kpool, a.pool_cap) : 0;
    }
    if (bad && tid == 0 && blockIdx.x == 0) report(a.status, kStBadQsl);
    __syncthreads();
    for (int s = tid; s < nseg; s += T_ALL) {
        const int4 d = sm.segs[s];
        int pools = 0;
        for (int rr = 0; rr < d.z; ++rr) pools = max(pools, sm.p_lim[d.y + rr - rb]);
        sm.segs[s].w = pools;
    }
    __syncthreads();
    {
        uint32_t carry = 0;
        for (int base = 0; base < nseg; base += T_ALL) {
            const int s = base + tid;
            const uint32_t t = s < nseg ? static_cast<uint32_t>((sm.segs[s].w + kTilePools - 1) / kTilePools) : 0u;
            uint32_t total;
            const uint32_t ex = carry + block_excl_scan(t, reinterpret_cast<uint32_t*>(sm.hist), &total);
            if (s < nseg) sm.prefix[s] = static_cast<int>(ex);
            carry += total;
            __syncthreads();
        }
        if (tid == 0) {
            sm.prefix[nseg] = static_cast<int>(carry);
            words[kWNtiles] = static_cast<int>(carry);
        }
        carry = 0;
        for (int base = 0; base < nchunk; base += T_ALL) {
            const int r = base + tid;
            const uint32_t t = (r < nchunk && sm.p_lim[r] == 0) ? 1u : 0u;
            uint32_t total;
            const uint32_t ex = carry + block_excl_scan(t, reinterpret_cast<uint32_t*>(sm.hist), &total);
            if (t) sm.p_triv[ex] = r;
            carry += total;
            __syncthreads();
        }
        if (tid == 0) words[kWNtriv] = static_cast<int>(carry);
    }
}

// The plan of a chunk by one warp: every input load is issued first, then warp scans.
__device__ __forceinline__ void plan_warp(const FusedArgs& a, const Smem& sm, int lane) {
    const int rb = a.row_begin, re = a.row_end;
    const int nchunk = re - rb;
    int* words = sm.words;
    // the plan's first loads, issued together: one memory round trip for a chunk of up to
    // 512 rows and the first 32 requests
    static_assert(kMaxPlanRows <= 16 * 32, "positions held in registers");
    int32_t pos[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int r = lane + 32 * j;
        pos[j] = r < nchunk ? __ldg(a.positions + rb + r) : 0;
    }
    const int q_lo = __ldg(a.qsl + min(lane, a.num_reqs));
    const int q_hi = __ldg(a.qsl + min(lane + 1, a.num_reqs));
    const int q_end = __ldg(a.qsl + a.num_reqs);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int r = lane + 32 * j;
        if (r < nchunk) {
            const int64_t c64 = static_cast<int64_t>(pos[j]) + 1;
            sm.p_ctx[r] = c64 > 0x7fffffff ? 0x7fffffff : (c64 < 0 ? 0 : static_cast<int32_t>(c64));
            sm.p_req[r] = -1;
        }
    }
    int bad = 0;
    if (lane == 0) bad = (q_lo < 0) | (q_end > a.num_rows);
    __syncwarp();
    int nseg = 0;
    for (int base = 0; base < a.num_reqs; base += 32) {
        const int i = base + lane;
        int lo = 0, hi = 0;
        uint32_t ns = 0;
        if (i < a.num_reqs) {
            const int x = base == 0 ? q_lo : __ldg(a.qsl + i), y = base == 0 ? q_hi : __ldg(a.qsl + i + 1);
            bad |= x > y;
            lo = max(x, rb);
            hi = min(y, re);
            if (hi > lo) ns = static_cast<uint32_t>((hi - lo + a.seg_rows - 1) / a.seg_rows);
        }
        const uint32_t incl = warp_incl_scan(ns);
        const int first = nseg + static_cast<int>(incl - ns);
        nseg += static_cast<int>(__shfl_sync(0xffffffffu, incl, 31));
        for (uint32_t k = 0; k < ns; ++k) {
            const int sidx = first + static_cast<int>(k);
            if (sidx >= a.max_segs) break;  // bounded by the host's max_segs
            const int row0 = lo + static_cast<int>(k) * a.seg_rows;
            sm.segs[sidx] = make_int4(i, row0, min(a.seg_rows, hi - row0), 0);
        }
        // the rows of the 32 requests of this round, the warp's lanes side by side
        for (int j = 0; j < 32; ++j) {
            const int lj = __shfl_sync(0xffffffffu, lo, j), hj = __shfl_sync(0xffffffffu, hi, j);
            for (int r = lj + lane; r < hj; r += 32) sm.p_req[r - rb] = base + j;
        }
    }
    __syncwarp();
    bad = __any_sync(0xffffffffu, bad);
    nseg = bad ? 0 : min(nseg, a.max_segs);
    for (int r = lane; r < nchunk; r += 32) {
        int32_t c = sm.p_ctx[r];
        int req = bad ? -1 : sm.p_req[r];
        if (req >= 0 && c > a.max_context) {
            if (blockIdx.x == 0) report(a.status, kStCtxOverBound);
            req = -1;
        }
        if (req < 0) c = -1;
        sm.p_req[r] = req;
        sm.p_ctx[r] = c;
        sm.p_lim[r] = (c > 0 && (a.score_all ? c >= a.kpool : c > a.topk)) ? min(c / a.kpool, a.pool_cap) : 0;
    }
    if (bad && lane == 0 && blockIdx.x == 0) report(a.status, kStBadQsl);
    __syncwarp();
    int tiles = 0;
    for (int base = 0; base < nseg; base += 32) {
        const int sidx = base + lane;
        uint32_t t = 0;
        if (sidx < nseg) {
            const int4 d = sm.segs[sidx];
            int pools = 0;
            for (int rr = 0; rr < d.z; ++rr) pools = max(pools, sm.p_lim[d.y + rr - rb]);
            sm.segs[sidx].w = pools;
            t = static_cast<uint32_t>((pools + kTilePools - 1) / kTilePools);
        }
        const uint32_t incl = warp_incl_scan(t);
        if (sidx < nseg) sm.prefix[sidx] = tiles + static_cast<int>(incl - t);
        tiles += static_cast<int>(__shfl_sync(0xffffffffu, incl, 31));
    }
    int ntriv = 0;
    for (int base = 0; base < nchunk; base += 32) {
        const int r = base + lane;
        const uint32_t t = (r < nchunk && sm.p_lim[r] == 0) ? 1u : 0u;
        const uint32_t incl = warp_incl_scan(t);
        if (t) sm.p_triv[ntriv + static_cast<int>(incl) - 1] = r;
        ntriv += static_cast<int>(__shfl_sync(0xffffffffu, incl, 31));
    }
    if (lane == 0) {
        sm.prefix[nseg] = tiles;
        words[kWNseg] = nseg;
        words[kWNtiles] = tiles;
        words[kWNtriv] = ntriv;
        words[kWBad] = bad;
    }
}

}  // namespace

__global__ void __launch_bounds__(kFusedThreads, 1)
    k_select_fused(const FusedArgs a, const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    Smem sm = carve(smem_raw, a);
    const int rb = a.row_begin;
    const int nchunk = a.row_end - a.row_begin;
    const uint32_t qhalf_bytes = static_cast<uint32_t>(a.npad_max) * 128u;
    int* words = sm.words;
    volatile int* abort_flag = words + kWAbort;
    int32_t* seg_done = a.ctr + kFusedCtrHeader;
    int32_t* jobs = seg_done + a.max_segs;

    // ---- set-up: barriers, TMEM, descriptor prefetch; page-table lines warmed into L2
    if (tid == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.tfull[i], 1);
            mbar_init(&sm.tempty[i], 4 * 32);
            mbar_init(&sm.qfull[i], 1);
            mbar_init(&sm.qempty[i], 1);
        }
        for (int i = 0; i < kSchedRing; ++i) {
            mbar_init(&sm.sfull[i], 1);
            mbar_init(&sm.sempty[i], a.select ? 1 + 4 + 1 : 1 + 4);
            mbar_init(&sm.tdone[i], 4);
        }
        mbar_init(sm.done, 1);
        for (int i = 1; i < 16; ++i) words[i] = 0;  // word 0 receives the TMEM address from warp 1
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_k);
        tma_prefetch_desc(&tmap_q);
    }
    if (warp == 1) {
        tmem_alloc(reinterpret_cast<uint32_t*>(words + kWTmem), a.tmem_cols);
        tmem_relinquish();
    }
    {
        // the key page table is small next to the keys: its first lines, spread over the
        // grid, are requested now so the producer's first look-ups hit L2
        const int64_t row_lines = (static_cast<int64_t>(a.max_key_pages) * 4 + 127) / 128;
        const int64_t lines = row_lines * a.num_reqs;
        if (tid < 8) {
            const int64_t l = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(tid) * gridDim.x;
            if (l < lines && row_lines > 0) {
                const int64_t i = l / row_lines, li = l % row_lines;
                prefetch_l2(a.key_page_table + i * a.kpt_ld + li * 32);
            }
        }
    }

    // ---- plan: row contexts, request runs, segments, tile prefix, trivial rows (one warp
    //      when the batch has few requests, the whole CTA otherwise)
    if (a.num_reqs <= kWarpPlanReqs) {
        if (warp == 0) plan_warp(a, sm, lane);
    } else {
        plan_cta(a, sm, tid);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(words[kWTmem]);
    const int nseg = words[kWNseg];
    const int total_tiles = words[kWNtiles];
    const int n_triv = words[kWNtriv];
    const uint64_t wait_ns = a.wait_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ scheduler + TMA producer
        const int share = static_cast<int>((static_cast<int64_t>(total_tiles) * 3 / 4) / gridDim.x);
        const int dyn0 = share * static_cast<int>(gridDim.x);
        if (lane == 0) {
            int s_next = static_cast<int>(blockIdx.x) * share;
            const int s_end = s_next + share;
            auto grab = [&]() -> int {
                if (s_next < s_end) return s_next++;
                const int t = dyn0 + atomicAdd(a.ctr + kCtrTile, 1);
                return t < total_tiles ? t : -1;
            };
            struct Pending {
                int t, seg, lt;
                int p0, p1;
                bool has0, second, has1;
            };
            int cur_s = 0;
            auto take = [&](int t) -> Pending {
                Pending r;
                r.t = t;
                r.seg = 0;
                r.lt = 0;
                r.p0 = r.p1 = -1;
                r.has0 = r.second = r.has1 = false;
                if (t < 0) return r;
                int lo = sm.prefix[cur_s] <= t ? cur_s : 0, hi = nseg - 1;
                while (lo < hi) {
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
            Pending t_a = take(grab());
            Pending t_b = take(t_a.t >= 0 ? grab() : -1);

            const uint64_t pol_k = l2_policy_evict_first();
            const uint64_t pol_q = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            int qb = 1, cur = -1;
            int q_uses0 = 0, q_uses1 = 0;
            uint32_t qe_phase = 0;
            uint32_t loaded = 0, last_parity = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int t = t_a.t;
                const int4 rec = t >= 0 ? record(t_a) : make_int4(0, 0, 0, 0);
                t_a = t_b;
                t_b = take(t_a.t >= 0 ? grab() : -1);
                const int slot = n & (kSchedRing - 1);
                if (!mbar_wait(&sm.sempty[slot], ((n / kSchedRing) & 1) ^ 1u, abort_flag, wait_ns)) { ok = false; break; }
                sm.tile_ring[slot] = t;
                sm.rec_ring[slot] = rec;
                mbar_arrive(&sm.sfull[slot]);
                if (t < 0) break;

                if (!mbar_wait(&sm.empty[stage], phase ^ 1u, abort_flag, wait_ns)) { ok = false; break; }
                if (t != a.fault_tile) {  // the failure-detection test leaves one tile unloaded
                    const int npages = rec.w == -2 ? 1 : 2;
                    mbar_expect_tx(&sm.full[stage], static_cast<uint32_t>(npages) * kPageBytes);
                    uint8_t* adst = sm.a + static_cast<size_t>(stage) * kTileBytes;
                    loaded |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    for (int h = 0; h < npages; ++h) {
                        const int pg = max(h == 0 ? rec.z : rec.w, 0);  // out-of-range pages: -inf in the epilogue
                        tma_load_3d(adst + h * kBoxBytes, &tmap_k, &sm.full[stage], 0, 0, pg, pol_k);
                        tma_load_3d(adst + kPageBytes + h * kBoxBytes, &tmap_k, &sm.full[stage], 64, 0, pg, pol_k);
                    }
                }
                if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                if (rec.x != cur) {
                    const int4 sd = sm.segs[rec.x];
                    qb ^= 1;
                    if ((qb ? q_uses1 : q_uses0) > 0) {
                        if (!mbar_wait(&sm.qempty[qb], (qe_phase >> qb) & 1u, abort_flag, wait_ns)) { ok = false; break; }
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
                for (int i = 0; i < a.stages && ok; ++i) {
                    ok = mbar_wait(&sm.empty[stage], phase ^ 1u, abort_flag, wait_ns);
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
                if (ok && q_uses0 > 0) ok = mbar_wait(&sm.qempty[0], qe_phase & 1u, abort_flag, wait_ns);
                if (ok && q_uses1 > 0) ok = mbar_wait(&sm.qempty[1], (qe_phase >> 1) & 1u, abort_flag, wait_ns);
            }
            if (!ok) {
                *abort_flag = 1;
                st_relaxed_gpu(a.ctr + kCtrAbort, 1);
                report(a.status, kStTimeout);
                // every copy already issued lands before the CTA leaves (bounded)
                for (int i = 0; i < a.stages; ++i)
                    if (loaded & (1u << i)) mbar_wait(&sm.full[i], (last_parity >> i) & 1u, nullptr, wait_ns);
                if (q_uses0 > 0) mbar_wait(&sm.qfull[0], static_cast<uint32_t>(q_uses0 - 1) & 1u, nullptr, wait_ns);
                if (q_uses1 > 0) mbar_wait(&sm.qfull[1], static_cast<uint32_t>(q_uses1 - 1) & 1u, nullptr, wait_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            int qb = 1, cur = -1;
            uint32_t qf_phase = 0;
            uint32_t idesc = 0;
            const uint32_t a_base = smem_u32(sm.a);
            const uint32_t q_base = smem_u32(sm.q);
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int slot = n & (kSchedRing - 1);
                if (!mbar_wait(&sm.sfull[slot], (n / kSchedRing) & 1, abort_flag, wait_ns)) { ok = false; break; }
                const int t = sm.tile_ring[slot];
                const int4 rec = sm.rec_ring[slot];
                mbar_arrive(&sm.sempty[slot]);
                if (t < 0) break;
                if (rec.x != cur) {
                    if (cur >= 0) umma_commit(&sm.qempty[qb]);
                    const int4 sd = sm.segs[rec.x];
                    qb ^= 1;
                    if (!mbar_wait(&sm.qfull[qb], (qf_phase >> qb) & 1u, abort_flag, wait_ns)) { ok = false; break; }
                    qf_phase ^= 1u << qb;
                    const uint32_t npad = static_cast<uint32_t>(((sd.z + 3) / 4) * 16);
                    idesc = umma_idesc_f16_f32(kTilePools, npad);
                    cur = rec.x;
                }
                if (!mbar_wait(&sm.full[stage], phase, abort_flag, wait_ns)) { ok = false; break; }
                if (!mbar_wait(&sm.tempty[acc], acc_phase ^ 1u, abort_flag, wait_ns)) { ok = false; break; }
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
            if (ok && cur >= 0) umma_commit(&sm.qempty[qb]);
            if (!ok) {
                *abort_flag = 1;
                st_relaxed_gpu(a.ctr + kCtrAbort, 1);
                report(a.status, kStTimeout);
            }
            umma_commit(sm.done);
            mbar_wait(sm.done, 0, nullptr, wait_ns);
        }
    } else if (warp < kSignalWarp) {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int quarter = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        int cur = -1;
        int4 sd = make_int4(0, 0, 0, 0);
        int lim_lo = 0, lim_hi = 0;
        int oob = 0;
        for (int n = 0;; ++n) {
            const int slot = n & (kSchedRing - 1);
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&sm.sfull[slot], (n / kSchedRing) & 1, abort_flag, wait_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    st_relaxed_gpu(a.ctr + kCtrAbort, 1);
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
                lim_lo = lane < sd.z ? sm.p_lim[sd.y - rb + lane] : 0;
                lim_hi = lane + 32 < sd.z ? sm.p_lim[sd.y - rb + lane + 32] : 0;
                cur = rec.x;
            }
            if (lane == 0) ok = mbar_wait(&sm.tfull[acc], acc_phase, abort_flag, wait_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *abort_flag = 1;
                    st_relaxed_gpu(a.ctr + kCtrAbort, 1);
                    report(a.status, kStTimeout);
                }
                break;
            }
            __syncwarp();
            tc_fence_after();
            const int p_in_tile = quarter * 32 + lane;
            const int j = rec.y * kTilePools + p_in_tile;
            const int g = rec.y * (kTilePools / 32) + quarter;  // this warp's 32-pool group
            const bool page_ok = (p_in_tile < kPagePools ? rec.z : rec.w) >= 0;
            if (!page_ok && j < sd.w) oob = 1;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc) * a.acc_cols;
            const int64_t row0 = sd.y - rb;
            for (int rg = 0; rg * 8 < sd.z; ++rg) {
                uint32_t v[32];
                __syncwarp();
                tmem_ld32(taddr + static_cast<uint32_t>(rg * 32), v);
                tmem_ld_wait();
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const int r = rg * 8 + rr;
                    if (r >= sd.z) break;  // uniform over the warp
                    const int lim = __shfl_sync(0xffffffffu, r < 32 ? lim_lo : lim_hi, r & 31);
                    const bool okp = j < lim;
                    const float h0 = __uint_as_float(v[4 * rr + 0]);
                    const float h1 = __uint_as_float(v[4 * rr + 1]);
                    const float h2 = __uint_as_float(v[4 * rr + 2]);
                    const float h3 = __uint_as_float(v[4 * rr + 3]);
                    const float sc = page_ok ? ((h0 + h1) + h2) + h3 : -__int_as_float(0x7f800000);
                    if (a.select) {
                        const uint32_t k = okp ? ordered_key(sc) : 0u;
                        if (okp) a.keys[(row0 + r) * a.keys_ld + j] = k;
                        if (g * 32 < lim) {  // uniform: the group holds a pool of this row
                            const uint32_t m1 = __reduce_max_sync(0xffffffffu, k);
                            const uint32_t eqm = __ballot_sync(0xffffffffu, k == m1);
                            const int l1 = __ffs(eqm) - 1;
                            const uint32_t m2 = __reduce_max_sync(0xffffffffu, lane == l1 ? 0u : k);
                            if (lane == 0)
                                a.grp[(row0 + r) * a.grp_ld + g] =
                                    make_uint2(m1, (m2 & ~31u) | static_cast<uint32_t>(l1));
                        }
                    } else if (okp) {
                        a.scores[(row0 + r) * a.scores_ld + j] = sc;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&sm.tempty[acc]);
            if (a.select) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.tdone[slot]);  // this warp's stores of the tile are done
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (__any_sync(0xffffffffu, oob) && lane == 0) words[kWOob] = 1;
    } else if (warp == kSignalWarp) {
        // ------------------------------------------------------------ tile completion -> jobs
        // Tiles are counted against their segment in runs (one GPU-scope release per run of
        // consecutive tiles of one segment): the CTA whose count completes a segment
        // publishes the segment's rows that need selecting as jobs.
        if (a.select && lane == 0) {
            int cur = -1, cnt = 0;
            auto flush = [&]() {
                if (cnt == 0) return;
                const int sg = cur;
                const int ntile = sm.prefix[sg + 1] - sm.prefix[sg];
                // the keys and records of these tiles, stored by the epilogue warps, are
                // ordered before this count at GPU scope
                if (atom_add_acq_rel_gpu(seg_done + sg, cnt) + cnt == ntile) {
                    const int4 d = sm.segs[sg];
                    int njob = 0;
                    for (int rr = 0; rr < d.z; ++rr) njob += sm.p_lim[d.y - rb + rr] > 0;
                    int base = atomicAdd(a.ctr + kCtrJobTail, njob);
                    if (base < 0 || base + njob > nchunk - n_triv) {
                        report(a.status, kStBadWorkspace);  // counters not zero at launch
                    } else {
                        for (int rr = 0; rr < d.z; ++rr) {
                            const int rl = d.y - rb + rr;
                            if (sm.p_lim[rl] > 0) st_release_gpu(jobs + base++, rl + 1);
                        }
                    }
                }
                cnt = 0;
            };
            for (int n = 0;; ++n) {
                const int slot = n & (kSchedRing - 1);
                const uint32_t par = (n / kSchedRing) & 1;
                if (!mbar_wait(&sm.sfull[slot], par, abort_flag, wait_ns)) break;
                const int t = sm.tile_ring[slot];
                const int4 rec = sm.rec_ring[slot];
                if (t < 0) {
                    mbar_arrive(&sm.sempty[slot]);
                    flush();
                    break;
                }
                if (!mbar_wait(&sm.tdone[slot], par, abort_flag, wait_ns)) break;
                mbar_arrive(&sm.sempty[slot]);
                if (rec.x != cur) {
                    flush();
                    cur = rec.x;
                }
                ++cnt;
            }
        }
    } else {
        // ------------------------------------------------------------ select (warps 7-14)
        if (a.select) {
            const int gt = tid - kSelWarp0 * 32;
            {
                // the block-table rows of the chunk's requests, spread over the grid, are
                // requested into L2 now: the rows' remaps read them at the end
                const int64_t bt_need = (static_cast<int64_t>(a.max_context) + a.block_size - 1) / a.block_size;
                const int lines = static_cast<int>(
                    (min(static_cast<int64_t>(a.max_blocks), bt_need) * 4 + 127) / 128);
                const int64_t total = static_cast<int64_t>(nseg) * lines;
                for (int64_t e = blockIdx.x + static_cast<int64_t>(gridDim.x) * gt; e < total;
                     e += static_cast<int64_t>(gridDim.x) * NTS) {
                    const int sg = static_cast<int>(e / lines), l = static_cast<int>(e % lines);
                    prefetch_l2(a.block_table + static_cast<int64_t>(sm.segs[sg].x) * a.bt_ld + l * 32);
                }
            }
            for (;;) {
                if (gt == 0) {
                    int row = -1;
                    const int i = atomicAdd(a.ctr + kCtrJobHead, 1);
                    if (i < 0) {
                        row = -2;
                        report(a.status, kStBadWorkspace);
                    } else if (i < n_triv) {
                        row = sm.p_triv[i];
                    } else if (i < nchunk) {
                        const int32_t* slotp = jobs + (i - n_triv);
                        int32_t v = ld_acquire_gpu(slotp);
                        if (v == 0) {
                            const uint64_t t0 = global_timer_ns();
                            while (true) {
                                __nanosleep(64);
                                v = ld_acquire_gpu(slotp);
                                if (v != 0) break;
                                if (ld_relaxed_gpu(a.ctr + kCtrAbort) != 0 || global_timer_ns() - t0 > wait_ns) break;
                            }
                        }
                        if (v > 0 && v <= nchunk) {
                            row = v - 1;
                        } else {
                            // no job in time, or a slot that no launch of this chunk wrote (the
                            // workspace did not start zero-filled): stop without touching memory
                            row = -2;
                            st_relaxed_gpu(a.ctr + kCtrAbort, 1);
                            report(a.status, v == 0 ? kStTimeout : kStBadWorkspace);
                        }
                    }
                    words[kWJob] = row;
                }
                sbar();
                const int row = words[kWJob];
                if (row < 0) break;
                select_row(a, sm, row, gt);
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, a.tmem_cols);
    }
    if (tid == 0) {
        if (words[kWOob]) report(a.status, kStKeyPageOob);
        // the last CTA to leave returns the counter words to zero for the next launch
        if (atom_add_acq_rel_gpu(a.ctr + kCtrExit, 1) == static_cast<int>(gridDim.x) - 1) {
            for (int i = 0; i < kFusedCtrHeader; ++i) a.ctr[i] = 0;
            for (int s = 0; s < nseg; ++s) seg_done[s] = 0;
            for (int i = 0; i < nchunk - n_triv; ++i) jobs[i] = 0;
        }
    }
}

FusedLayout fused_layout(int stages, int npad_max, int max_segs, int chunk_cap, int bt_cap, int cand_cap, int gcap,
                         int K) {
    auto up = [](size_t x, size_t al) { return (x + al - 1) & ~(al - 1); };
    FusedLayout L{};
    size_t off = 0;
    L.a = static_cast<uint32_t>(off);
    off += static_cast<size_t>(stages) * kTileBytes;
    L.q = static_cast<uint32_t>(off);
    off += 2u * static_cast<size_t>(npad_max) * 256u;
    L.segs = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(max_segs) * 16, 16);
    L.prefix = static_cast<uint32_t>(off);
    off = up(off + (static_cast<size_t>(max_segs) + 1) * 4, 16);
    L.rec_ring = static_cast<uint32_t>(off);
    off += kSchedRing * 16;
    L.tile_ring = static_cast<uint32_t>(off);
    off = up(off + kSchedRing * 4, 8);
    L.bars = static_cast<uint32_t>(off);
    off += (2 * static_cast<size_t>(stages) + 8 + 3 * kSchedRing + 1) * 8;
    L.words = static_cast<uint32_t>(off);
    off = up(off + 16 * 4, 16);
    L.p_ctx = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(chunk_cap) * 4, 16);
    L.p_req = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(chunk_cap) * 4, 16);
    L.p_lim = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(chunk_cap) * 4, 16);
    L.p_triv = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(chunk_cap) * 4, 16);
    L.s_btab = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(bt_cap) * 4, 16);
    L.s_hist = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(kHistBins) * 4, 16);
    L.s_ckey = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(cand_cap) * 4, 16);
    L.s_cidx = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(cand_cap) * 4, 16);
    L.s_rec = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(gcap) * 8, 16);  // records, later two bitmaps of gcap words
    L.s_list = static_cast<uint32_t>(off);
    off = up(off + static_cast<size_t>(K) * 4, 16);
    L.s_small = static_cast<uint32_t>(off);
    off += 512;
    L.s_scan = static_cast<uint32_t>(off);
    off += K > 0 ? 8 * kScanCap : 0;
    L.s_scratch = static_cast<uint32_t>(off);
    off = up(off + 64 * 4, 16);
    L.total = static_cast<uint32_t>(off + 1024);  // + alignment slack of the 1024-B base
    return L;
}

cudaError_t launch_fused(const FusedArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_q, int grid,
                         cudaStream_t s) {
    static size_t configured[kMaxDevicesTracked] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = a.lay.total;
    if (dev >= 0 && dev < kMaxDevicesTracked && smem > configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_select_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // the CTAs wait on one another: all must be resident
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_select_fused, a, tmap_k, tmap_q);
}

}  // namespace sel
