// K-c: per-row top-k over pool scores, fused with expansion, the trailing incomplete
// pool and (optionally) the block-table remap.
//
// Semantics (vLLM flashinfer_mla_sparse_sm90 page, _kv_lens_host; ReVolta PR #59):
// a row with ctx = position + 1 <= index_topk selects tokens 0..ctx-1; otherwise the
// K = index_topk / kpool best of its P = ctx / kpool complete pools (score descending,
// lower pool index first on ties) are expanded to their kpool tokens each, followed by
// the trailing tokens P*kpool..ctx-1; tokens ascend, the rest of the row is -1. With
// remap, each token goes through the sparse_utils formula
// block_table[req, t / block_size] * block_stride_rows + t % block_size (-1 guarded), and
// the valid count is the number of non -1 slots, reduced on chip without atomics.
//
// GB300 design: one thread-block cluster (1..8 CTAs) per row. Each CTA takes an even
// slice of the row; thread t of a CTA owns a contiguous run of the slice, staged once
// as order-preserving 32-bit keys in shared memory in a transposed layout (key i of
// thread t at i * threads + t, so every pass is bank-conflict free) together with the
// block-table entries the slice's tokens need. A first radix level over the top 11
// key bits finds the bin b1 holding the K-th largest key: each CTA builds a local
// histogram, the owner of every bin range sums it across the cluster through
// distributed shared memory and pushes the totals to all CTAs, and every CTA scans
// them. The keys of bin b1 (a few hundred for real scores) are then gathered from all
// CTAs in index order and every CTA finishes the select on that small set alone (two
// local radix levels over the remaining 21 bits). When the bin is too crowded
// (massive ties), the two levels run cluster-wide instead. Keys equal to the threshold
// are kept lowest index first across the cluster. The kept pools are placed by one
// block scan over the per-thread counts, so each pass over the slice costs a few
// instructions per key.
#include <cooperative_groups.h>

#include "sel_device.cuh"
#include "sel_kernels.h"

namespace cg = cooperative_groups;

namespace sel {

SEL_PHASE_TABLE(topk)

namespace {

struct TopkSmem {
    uint32_t* keys;     // [slice_cap] key i of thread t at i * kTopkThreads + t
    uint32_t* hist;     // [kTopkBins] local histogram
    uint32_t* tot;      // [kTopkBins] cluster totals
    uint2* cand;        // [kTopkCandCap] this CTA's keys of bin b1: (key, pool index), index order
    uint2* merged;      // [kTopkCandCap] every CTA's candidates, index order
    int32_t* btab;      // [bt_cap] block-table entries covering this CTA's tokens
    uint32_t* scratch;  // [64]
    uint32_t* xch;      // [32]: 0..7 candidates, 8..15 keys above b1, 16..23 valid slots (per CTA)
    uint32_t* cnt;      // [32]: 0..7 keys > thr, 8..15 keys == thr, 16..23 candidates, 24..31 above b1
    uint32_t* res;      // [8]
};

__device__ __forceinline__ TopkSmem carve(uint32_t* base, int slice_cap, int bt_cap) {
    TopkSmem s;
    s.keys = base;
    s.hist = base + slice_cap;
    s.tot = s.hist + kTopkBins;
    s.cand = reinterpret_cast<uint2*>(s.tot + kTopkBins);
    s.merged = s.cand + kTopkCandCap;
    s.btab = reinterpret_cast<int32_t*>(s.merged + kTopkCandCap);
    s.scratch = reinterpret_cast<uint32_t*>(s.btab + ((bt_cap + 3) & ~3));
    s.xch = s.scratch + 64;
    s.cnt = s.xch + 32;
    s.res = s.cnt + 32;
    return s;
}

// Local: the bin (of `nbins`, counted from the top) that holds the Kc-th largest key
// counted in `hist`, and Kc minus the keys in the bins above it.
__device__ __forceinline__ void block_find_bin(const uint32_t* hist, const TopkSmem& sm, int nbins, uint32_t Kc,
                                               uint32_t& bin, uint32_t& krem) {
    const int tid = threadIdx.x;
    const int per = nbins / kTopkThreads;
    uint32_t local = 0;
    for (int i = 0; i < per; ++i) local += hist[nbins - 1 - (tid * per + i)];
    uint32_t total;
    const uint32_t above = block_excl_scan(local, sm.scratch, &total);
    if (above < Kc && Kc <= above + local) {
        uint32_t acc = above;
        for (int i = 0; i < per; ++i) {
            const int b = nbins - 1 - (tid * per + i);
            if (acc + hist[b] >= Kc) {
                sm.res[0] = static_cast<uint32_t>(b);
                sm.res[1] = Kc - acc;
                break;
            }
            acc += hist[b];
        }
    }
    __syncthreads();
    bin = sm.res[0];
    krem = sm.res[1];
}

// Cluster-wide: sums every CTA's local histogram into `tot` (each CTA owns a bin
// range, adds it over the cluster and pushes the totals to every CTA), then finds the
// bin of the Kc-th largest key locally.
__device__ __forceinline__ void cluster_find_bin(cg::cluster_group& cluster, uint32_t C, uint32_t crank,
                                                 const TopkSmem& sm, int nbins, uint32_t Kc, uint32_t& bin,
                                                 uint32_t& krem) {
    cluster.sync();  // every local histogram is complete
    const int lo = static_cast<int>(crank) * nbins / static_cast<int>(C);
    const int hi = static_cast<int>(crank + 1) * nbins / static_cast<int>(C);
    for (int b = lo + static_cast<int>(threadIdx.x); b < hi; b += blockDim.x) {
        uint32_t v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = c < static_cast<int>(C) ? cluster.map_shared_rank(sm.hist, c)[b] : 0u;
        uint32_t s = 0;
#pragma unroll
        for (int c = 0; c < 8; ++c) s += v[c];
#pragma unroll
        for (int c = 0; c < 8; ++c)
            if (c < static_cast<int>(C)) cluster.map_shared_rank(sm.tot, c)[b] = s;
    }
    cluster.sync();  // every CTA holds the totals of all bins
    block_find_bin(sm.tot, sm, nbins, Kc, bin, krem);
}

struct RowMap {  // how a token reaches its slot
    const int32_t* bt_row;  // global block-table row
    const int32_t* btab;    // shared-memory copy of entries [blk0, blk0 + nblk), or null
    int64_t blk0;
    int32_t nblk;
};

__device__ __forceinline__ int32_t slot_of(const TopkArgs& a, const RowMap& m, int32_t t) {
    if (t < 0) return -1;
    const int32_t b = t / a.block_size;
    int32_t ph;
    if (m.btab && b >= m.blk0 && b < m.blk0 + m.nblk) {
        ph = m.btab[b - m.blk0];  // entries past max_blocks were stored as -1
    } else {
        if (b >= a.max_blocks) return -1;
        ph = __ldg(m.bt_row + b);
    }
    if (ph < 0 || ph >= a.num_kv_blocks) return -1;
    return static_cast<int32_t>(static_cast<int64_t>(ph) * a.block_stride_rows + (t - b * a.block_size));
}

// Writes kpool consecutive tokens starting at token t0 into columns col..col+kpool-1.
template <bool REMAP>
__device__ __forceinline__ uint32_t emit_pool(const TopkArgs& a, const RowMap& m, int32_t* tok_row,
                                              int32_t* slot_row, int64_t col, int32_t t0) {
    uint32_t valid = 0;
    if (a.kpool == 4 && (a.block_size & 3) == 0) {
        if (tok_row) *reinterpret_cast<int4*>(tok_row + col) = make_int4(t0, t0 + 1, t0 + 2, t0 + 3);
        if (REMAP) {
            const int32_t s0 = slot_of(a, m, t0);  // the 4 tokens share one block
            const int4 s = s0 < 0 ? make_int4(-1, -1, -1, -1) : make_int4(s0, s0 + 1, s0 + 2, s0 + 3);
            *reinterpret_cast<int4*>(slot_row + col) = s;
            valid = s0 < 0 ? 0u : 4u;
        } else {
            valid = 4u;
        }
    } else {
        for (int u = 0; u < a.kpool; ++u) {
            const int32_t t = t0 + u;
            if (tok_row) tok_row[col + u] = t;
            if (REMAP) {
                const int32_t s = slot_of(a, m, t);
                slot_row[col + u] = s;
                valid += s != -1;
            } else {
                valid += 1;
            }
        }
    }
    return valid;
}

// Columns [c_begin, W): tokens `first`, `first`+1, ... up to `last` (exclusive), then -1.
template <bool REMAP>
__device__ __forceinline__ uint32_t emit_run(const TopkArgs& a, const RowMap& m, int32_t* tok_row,
                                             int32_t* slot_row, int c_begin, int64_t first, int64_t last) {
    uint32_t valid = 0;
    for (int c = c_begin + threadIdx.x; c < a.out_width; c += blockDim.x) {
        const int64_t tt = first + (c - c_begin);
        const int32_t t = tt < last ? static_cast<int32_t>(tt) : -1;
        if (tok_row) tok_row[c] = t;
        if (REMAP) {
            const int32_t s = slot_of(a, m, t);
            slot_row[c] = s;
            valid += s != -1;
        } else {
            valid += t != -1;
        }
    }
    return valid;
}

}  // namespace

template <bool REMAP>
__global__ void __launch_bounds__(kTopkThreads, 2) k_topk_expand(const TopkArgs a) {
    extern __shared__ __align__(16) uint32_t tk_smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t C = cluster.num_blocks();
    const uint32_t crank = cluster.block_rank();
    const int tid = threadIdx.x;
    constexpr int T = kTopkThreads;
    const int rl = blockIdx.y;
    const int r = a.row_begin + rl;
    TopkSmem sm = carve(tk_smem, a.slice_cap, a.bt_cap);
    // diagnostics: CTA rank 0 of rows 0 and gridDim.y/2 stamp their phases (bases 0, 256)
    const int tb = crank != 0 ? -1 : (rl == 0 ? 0 : (rl == static_cast<int>(gridDim.y) / 2 ? 256 : -1));
    (void)tb;
#define TK_PHASE(i) do { if (tb >= 0 && tid == 0) SEL_PHASE(tb + (i)); } while (0)
    TK_PHASE(0);

    pdl_wait();  // scores and row descriptors come from the preceding kernels
    TK_PHASE(1);

    // ---- the row: context, request, mode (identical in every CTA of the cluster)
    bool valid = true;
    int64_t ctx;
    if (a.row_ctx) {
        const int32_t c = a.row_ctx[rl];
        valid = c >= 0;
        ctx = c;
    } else {
        ctx = static_cast<int64_t>(a.positions[r]) + 1;
    }
    int req = 0;
    if (REMAP) {
        req = a.row_req[rl];
        valid = valid && req >= 0;
    }
    int64_t P = 0;
    const int K = a.topk / a.kpool;
    int64_t L = 0;
    int R = 0;  // keys per thread (multiple of 4)
    if (valid && ctx > a.topk) {
        P = ctx / a.kpool;
        L = ((P + C - 1) / C + 3) & ~int64_t(3);
        R = static_cast<int>(((L + T - 1) / T + 3) & ~int64_t(3));
        if (P > a.max_pools || static_cast<int64_t>(R) * T > a.slice_cap) {
            valid = false;
            if (crank == 0 && tid == 0) report(a.status, kStCtxOverBound);
        }
    }
    int32_t* tok_row = a.token_idx ? a.token_idx + static_cast<int64_t>(r) * a.out_width : nullptr;
    int32_t* slot_row = REMAP ? a.slots + static_cast<int64_t>(r) * a.out_width : nullptr;
    RowMap map{(REMAP && valid) ? a.block_table + static_cast<int64_t>(req) * a.bt_ld : nullptr, nullptr, 0, 0};

    if (!valid || ctx <= a.topk) {
        // every token of a short row, or nothing: no selection, the first CTA writes the row
        if (crank != 0) return;
        const int64_t n = valid && ctx > 0 ? ctx : 0;
        const uint32_t v = emit_run<REMAP>(a, map, tok_row, slot_row, 0, 0, n);
        const uint32_t cnt = block_sum(v, sm.scratch);
        if (tid == 0 && a.counts) a.counts[r] = static_cast<int32_t>(cnt);
        return;
    }

    // ---- this CTA's slice [beg, beg + n); thread t owns [t*R, t*R + R) of it
    const int64_t beg = static_cast<int64_t>(crank) * L;
    const int64_t rem = P - beg < L ? P - beg : L;
    const int n = rem > 0 ? static_cast<int>(rem) : 0;
    const int my0 = tid * R;                      // first slice index of this thread
    const int my_n = max(0, min(R, n - my0));     // valid keys of this thread
    if (REMAP && n > 0) {
        const int64_t b0 = beg * a.kpool / a.block_size;
        const int64_t b1e = ((beg + n) * a.kpool - 1) / a.block_size + 1;
        if (b1e - b0 <= a.bt_cap) {
            map.btab = sm.btab;
            map.blk0 = b0;
            map.nblk = static_cast<int32_t>(b1e - b0);
            for (int i = tid; i < map.nblk; i += blockDim.x)
                sm.btab[i] = b0 + i < a.max_blocks ? __ldg(map.bt_row + b0 + i) : -1;
        }
    }
    for (int b = tid; b < kTopkBins; b += blockDim.x) sm.hist[b] = 0;
    __syncthreads();

    // ---- stage the run as keys (loads issued 4 float4 at a time); level-1 histogram
    //      locally unless the scorer already counted it
    const bool local_hist = a.hist == nullptr;
    {
        const float4* src = reinterpret_cast<const float4*>(a.scores + static_cast<int64_t>(rl) * a.scores_ld +
                                                            beg + my0);
        for (int q0 = 0; q0 < R; q0 += 16) {
            float4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (q0 + 4 * j < my_n) v[j] = __ldcg(src + (q0 >> 2) + j);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = q0 + 4 * j;
                if (i < my_n) {
                    const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t k = i + u < my_n ? ordered_key(f[u]) : 0u;
                        sm.keys[(i + u) * T + tid] = k;
                        if (local_hist && i + u < my_n) atomicAdd(&sm.hist[k >> 21], 1u);
                    }
                }
            }
        }
    }
    TK_PHASE(2);
    uint32_t b1, k1, b2, k2, b3, k3;
    if (local_hist) {
        cluster_find_bin(cluster, C, crank, sm, 2048, static_cast<uint32_t>(K), b1, k1);
    } else {
        const uint32_t* hrow = a.hist + static_cast<int64_t>(rl) * kTopkBins;
        for (int b = tid; b < kTopkBins; b += blockDim.x) sm.tot[b] = __ldcg(hrow + b);
        __syncthreads();
        block_find_bin(sm.tot, sm, 2048, static_cast<uint32_t>(K), b1, k1);
    }
    TK_PHASE(3);
    const uint32_t m_all = sm.tot[b1];  // keys of bin b1 in the whole row
    uint32_t thr, need_eq;

    if (m_all <= static_cast<uint32_t>(kTopkCandCap)) {
        // ---- local candidates (keys of bin b1) in index order, and keys above bin b1
        uint32_t nc = 0, na = 0;
        for (int i = 0; i < my_n; ++i) {
            const uint32_t bk = sm.keys[i * T + tid] >> 21;
            nc += bk == b1;
            na += bk > b1;
        }
        uint32_t tot_packed;
        const uint32_t pre = block_excl_scan(nc | (na << 16), sm.scratch, &tot_packed);
        uint32_t pos = pre & 0xffffu;
        if (nc) {
            for (int i = 0; i < my_n; ++i) {
                const uint32_t k = sm.keys[i * T + tid];
                if ((k >> 21) == b1) sm.cand[pos++] = make_uint2(k, static_cast<uint32_t>(beg + my0 + i));
            }
        }
        if (tid == 0) {
            sm.xch[crank] = tot_packed & 0xffffu;
            sm.xch[8 + crank] = tot_packed >> 16;
        }
        TK_PHASE(4);
        cluster.sync();  // every CTA's candidate list and counts are published
        TK_PHASE(5);

        // ---- gather all candidates in index order (CTA order, then each list's order)
        if (tid < static_cast<int>(C)) {
            const uint32_t* px = cluster.map_shared_rank(sm.xch, static_cast<unsigned>(tid));
            sm.cnt[16 + tid] = px[tid];      // candidates of CTA tid
            sm.cnt[24 + tid] = px[8 + tid];  // keys above bin b1 in CTA tid
        }
        if (tid < 16) sm.cnt[tid] = 0;  // per-CTA counts of keys > thr / == thr, filled below
        __syncthreads();
        for (uint32_t g = tid; g < m_all; g += blockDim.x) {  // all DSMEM loads in flight at once
            uint32_t c = 0, base = 0;
            while (g >= base + sm.cnt[16 + c]) base += sm.cnt[16 + c++];
            sm.merged[g] = cluster.map_shared_rank(sm.cand, c)[g - base];
        }
        for (int b = tid; b < kTopkBins; b += blockDim.x) sm.hist[b] = 0;
        __syncthreads();
        TK_PHASE(6);

        // ---- exact select of the k1-th largest among the candidates, locally
        for (uint32_t i = tid; i < m_all; i += blockDim.x) atomicAdd(&sm.hist[(sm.merged[i].x >> 10) & 2047u], 1u);
        __syncthreads();
        block_find_bin(sm.hist, sm, 2048, k1, b2, k2);
        const uint32_t pre22 = (b1 << 11) | b2;
        for (int b = tid; b < 1024; b += blockDim.x) sm.tot[b] = 0;
        __syncthreads();
        for (uint32_t i = tid; i < m_all; i += blockDim.x) {
            const uint32_t k = sm.merged[i].x;
            if ((k >> 10) == pre22) atomicAdd(&sm.tot[k & 1023u], 1u);
        }
        __syncthreads();
        block_find_bin(sm.tot, sm, 1024, k2, b3, k3);
        thr = (pre22 << 10) | b3;
        need_eq = k3;
        TK_PHASE(7);

        // ---- per-CTA counts of keys > thr and == thr (from the candidates + keys above b1)
        for (uint32_t i = tid; i < m_all; i += blockDim.x) {
            const uint32_t k = sm.merged[i].x;
            uint32_t c = 0, end = sm.cnt[16];
            while (i >= end) end += sm.cnt[16 + ++c];
            if (k > thr) atomicAdd(&sm.cnt[c], 1u);
            else if (k == thr) atomicAdd(&sm.cnt[8 + c], 1u);
        }
        __syncthreads();
        if (tid < static_cast<int>(C)) sm.cnt[tid] += sm.cnt[24 + tid];
        __syncthreads();
    } else {
        // ---- crowded bin (massive ties): levels 2 and 3 over the whole cluster
        for (int b = tid; b < kTopkBins; b += blockDim.x) sm.hist[b] = 0;
        __syncthreads();
        for (int i = 0; i < my_n; ++i) {
            const uint32_t k = sm.keys[i * T + tid];
            if ((k >> 21) == b1) atomicAdd(&sm.hist[(k >> 10) & 2047u], 1u);
        }
        cluster_find_bin(cluster, C, crank, sm, 2048, k1, b2, k2);
        const uint32_t pre22 = (b1 << 11) | b2;
        for (int b = tid; b < kTopkBins; b += blockDim.x) sm.hist[b] = 0;
        __syncthreads();
        for (int i = 0; i < my_n; ++i) {
            const uint32_t k = sm.keys[i * T + tid];
            if ((k >> 10) == pre22) atomicAdd(&sm.hist[k & 1023u], 1u);
        }
        cluster_find_bin(cluster, C, crank, sm, 1024, k2, b3, k3);
        thr = (pre22 << 10) | b3;
        need_eq = k3;
        uint32_t g = 0, e = 0;
        for (int i = 0; i < my_n; ++i) {
            const uint32_t k = sm.keys[i * T + tid];
            g += k > thr;
            e += k == thr;
        }
        uint32_t ge;
        block_excl_scan(g | (e << 16), sm.scratch, &ge);
        if (tid < static_cast<int>(C)) {
            uint32_t* peer = cluster.map_shared_rank(sm.xch, static_cast<unsigned>(tid));
            peer[crank] = ge & 0xffffu;
            peer[8 + crank] = ge >> 16;
        }
        cluster.sync();
        if (tid < static_cast<int>(C)) {
            sm.cnt[tid] = sm.xch[tid];
            sm.cnt[8 + tid] = sm.xch[8 + tid];
        }
        __syncthreads();
    }
    TK_PHASE(8);

    // ---- this CTA's share of the kept pools: keys > thr, then the first equal ones
    uint32_t sel_before = 0, my_take = 0, eq_seen = 0;
    for (uint32_t c = 0; c < C; ++c) {
        const uint32_t e = sm.cnt[8 + c];
        const uint32_t take = need_eq > eq_seen ? min(e, need_eq - eq_seen) : 0u;
        eq_seen += e;
        if (c < crank) sel_before += sm.cnt[c] + take;
        if (c == crank) my_take = take;
    }

    // ---- per-thread counts, one block scan, then each thread writes its kept pools in order
    uint32_t gt = 0, eq = 0;
    for (int i = 0; i < my_n; ++i) {
        const uint32_t k = sm.keys[i * T + tid];
        gt += k > thr;
        eq += k == thr;
    }
    uint32_t unused;
    const uint32_t pre2 = block_excl_scan(gt | (eq << 16), sm.scratch, &unused);
    const uint32_t gt_pre = pre2 & 0xffffu, eq_pre = pre2 >> 16;
    TK_PHASE(9);
    uint32_t vcount = 0;
    if (gt | eq) {
        uint32_t pos = sel_before + gt_pre + min(eq_pre, my_take);
        uint32_t eq_run = eq_pre;
        for (int i = 0; i < my_n; ++i) {
            const uint32_t k = sm.keys[i * T + tid];
            bool keep = k > thr;
            if (k == thr) keep = eq_run++ < my_take;
            if (keep) {
                const int32_t t0 = static_cast<int32_t>((beg + my0 + i) * a.kpool);
                vcount += emit_pool<REMAP>(a, map, tok_row, slot_row, static_cast<int64_t>(pos) * a.kpool, t0);
                ++pos;
            }
        }
    }
    TK_PHASE(10);

    // ---- trailing incomplete pool and -1 padding (first CTA), valid count
    if (crank == 0) vcount += emit_run<REMAP>(a, map, tok_row, slot_row, K * a.kpool, P * a.kpool, ctx);
    const uint32_t vcta = block_sum(vcount, sm.scratch);
    if (tid == 0) cluster.map_shared_rank(sm.xch, 0u)[16 + crank] = vcta;
    cluster.sync();  // also: no CTA leaves while a peer may still read its shared memory
    if (crank == 0 && tid == 0 && a.counts) {
        uint32_t total = 0;
        for (uint32_t c = 0; c < C; ++c) total += sm.xch[16 + c];
        a.counts[r] = static_cast<int32_t>(total);
    }
    TK_PHASE(11);
#undef TK_PHASE
}

size_t topk_smem_bytes(int slice_cap, int bt_cap) {
    return static_cast<size_t>(slice_cap) * 4 + 2 * kTopkBins * 4 + 2 * kTopkCandCap * 8 +
           static_cast<size_t>((bt_cap + 3) & ~3) * 4 + (64 + 32 + 32 + 8) * 4;
}

cudaError_t launch_topk(const TopkArgs& a, bool remap, int cluster, int rows, size_t smem, bool pdl,
                        cudaStream_t s) {
    static size_t configured[2][kMaxDevicesTracked] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const void* fn = remap ? reinterpret_cast<const void*>(&k_topk_expand<true>)
                           : reinterpret_cast<const void*>(&k_topk_expand<false>);
    if (dev >= 0 && dev < kMaxDevicesTracked && smem > configured[remap ? 1 : 0][dev]) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[remap ? 1 : 0][dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster), static_cast<unsigned>(rows), 1);
    cfg.blockDim = dim3(kTopkThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    if (remap) return cudaLaunchKernelEx(&cfg, k_topk_expand<true>, a);
    return cudaLaunchKernelEx(&cfg, k_topk_expand<false>, a);
}

}  // namespace sel
