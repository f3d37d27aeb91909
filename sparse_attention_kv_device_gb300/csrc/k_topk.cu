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
// GB300 design: one 512-thread CTA per row; no cluster, no distributed shared memory.
// The row is read in chunks of 32 x 512 pools; in a chunk thread t holds the
// order-preserving 32-bit keys of pools t, t + 512, ... (32 registers, coalesced loads). An exact three-level radix
// select (11 + 11 + 10 key bits) finds the K-th largest key:
//   level 1: the bin b1 holding it, from the row's histogram of the top 11 bits;
//   list:    the row's keys with bin >= b1 (the keys above the threshold bin and the
//            threshold bin itself: about K plus a few hundred for real scores) are
//            compacted, in index order, into a shared-memory list by one block scan;
//   levels 2, 3: on the list's bin-b1 keys only.
// The kept pools are then the list entries above the threshold plus the first equal ones;
// one packed block scan over the list gives each its output column. The block-table row
// is staged in shared memory while the keys load. A crowded threshold bin (massive ties,
// list overflow) takes a slower path that re-reads the row for levels 2, 3 and output.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

constexpr int T = kTopkThreads;
constexpr int kChunk = 32;  // keys a thread holds in registers at a time

struct TopkSmem {
    uint32_t* cnt;      // [T] per (key slot, warp) counts of a chunk, then their prefix
    uint32_t* hist;     // [kTopkBins]
    uint2* list;        // [kTopkListCap] (key, pool) with bin >= b1, index order
    int32_t* btab;      // [bt_cap] the row's block-table entries
    uint32_t* scratch;  // [64]
    uint32_t* res;      // [8]
};

__device__ __forceinline__ TopkSmem carve(uint32_t* base, int bt_cap) {
    TopkSmem s;
    s.cnt = base;
    s.hist = base + T;
    s.list = reinterpret_cast<uint2*>(s.hist + kTopkBins);
    s.btab = reinterpret_cast<int32_t*>(s.list + kTopkListCap);
    s.scratch = reinterpret_cast<uint32_t*>(s.btab + ((bt_cap + 3) & ~3));
    s.res = s.scratch + 64;
    return s;
}

// The bin (of `nbins`, counted from the top) that holds the Kc-th largest key counted in
// `hist`, and Kc minus the keys in the bins above it.
__device__ __forceinline__ void block_find_bin(const uint32_t* hist, const TopkSmem& sm, int nbins, uint32_t Kc,
                                               uint32_t& bin, uint32_t& krem) {
    const int tid = threadIdx.x;
    const int per = (nbins + T - 1) / T;
    uint32_t local = 0;
    for (int i = 0; i < per; ++i) {
        const int b = nbins - 1 - (tid * per + i);
        if (b >= 0) local += hist[b];
    }
    uint32_t total;
    const uint32_t above = block_excl_scan(local, sm.scratch, &total);
    if (above < Kc && Kc <= above + local) {
        uint32_t acc = above;
        for (int i = 0; i < per; ++i) {
            const int b = nbins - 1 - (tid * per + i);
            if (b < 0) break;
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

struct RowMap {  // how a token reaches its slot
    const int32_t* bt_row;  // global block-table row
    const int32_t* btab;    // shared-memory copy of entries [0, nblk), or null
    int32_t nblk;
};

__device__ __forceinline__ int32_t slot_of(const TopkArgs& a, const RowMap& m, int32_t t) {
    if (t < 0) return -1;
    const int32_t b = t / a.block_size;
    int32_t ph;
    if (m.btab && b < m.nblk) {
        ph = m.btab[b];  // entries past max_blocks were stored as -1
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

// Chunk c of a row is pools [c*kChunkPools, (c+1)*kChunkPools); its key i held by thread
// tid is pool c*kChunkPools + i*T + tid, so every warp load reads one contiguous 128-byte
// line. Keys are loaded first, then converted in place to order-preserving keys; pools
// past P become 0, below every real key.
constexpr int kChunkPools = T * kChunk;

__device__ __forceinline__ void load_chunk(const float* row, int64_t c, int64_t P, uint32_t (&k)[kChunk]) {
    const int64_t base = c * kChunkPools + threadIdx.x;
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
        k[i] = base + static_cast<int64_t>(i) * T < P ? __float_as_uint(__ldcg(row + base + static_cast<int64_t>(i) * T)) : 0u;
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
        k[i] = base + static_cast<int64_t>(i) * T < P ? ordered_key(__uint_as_float(k[i])) : 0u;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    return (1u << (threadIdx.x & 31)) - 1u;
}

}  // namespace

template <bool REMAP>
__global__ void __launch_bounds__(kTopkThreads, 1) k_topk_expand(const TopkArgs a) {
    extern __shared__ __align__(16) uint32_t tk_smem[];
    const int tid = threadIdx.x;
    const int rl = blockIdx.x;
    const int r = a.row_begin + rl;
    TopkSmem sm = carve(tk_smem, a.bt_cap);
    // diagnostics: rows 0 and gridDim.x/2 stamp their phases (bases 0, 256)

    pdl_wait();  // scores, row descriptors and histograms come from the preceding kernels

    // ---- the row: context, request, mode
    bool valid = true;
    int64_t ctx;
    if (a.row_ctx) {
        const int32_t c = __ldcg(a.row_ctx + rl);
        valid = c >= 0;
        ctx = c;
    } else {
        ctx = static_cast<int64_t>(a.positions[r]) + 1;
    }
    int req = 0;
    if (REMAP) {
        req = __ldcg(a.row_req + rl);
        valid = valid && req >= 0;
    }
    const int K = a.topk / a.kpool;
    int64_t P = 0;
    if (valid && ctx > a.topk) {
        P = ctx / a.kpool;
        if (P > a.max_pools) {
            valid = false;
            if (tid == 0) report(a.status, kStCtxOverBound);
        }
    }
    int32_t* tok_row = a.token_idx ? a.token_idx + static_cast<int64_t>(r) * a.out_width : nullptr;
    int32_t* slot_row = REMAP ? a.slots + static_cast<int64_t>(r) * a.out_width : nullptr;
    RowMap map{(REMAP && valid) ? a.block_table + static_cast<int64_t>(req) * a.bt_ld : nullptr, nullptr, 0};

    if (!valid || ctx <= a.topk) {
        // every token of a short row, or nothing: no selection
        const int64_t n = valid && ctx > 0 ? ctx : 0;
        const uint32_t v = emit_run<REMAP>(a, map, tok_row, slot_row, 0, 0, n);
        const uint32_t cnt = block_sum(v, sm.scratch);
        if (tid == 0 && a.counts) a.counts[r] = static_cast<int32_t>(cnt);
        return;
    }

    // ---- the row's scores, read chunk by chunk (see load_chunk)
    const float* row = a.scores + static_cast<int64_t>(rl) * a.scores_ld;
    const int64_t nchunks = (P + kChunkPools - 1) / kChunkPools;
    const int warp = tid >> 5;

    // the block table is copied asynchronously into shared memory while the first keys load
    int nblk = 0;
    if (REMAP) {
        int64_t need = (ctx + a.block_size - 1) / a.block_size;
        if (need > a.max_blocks) need = a.max_blocks;
        if (need <= a.bt_cap) nblk = static_cast<int>(need);
        for (int i = tid; i < nblk; i += T) cp_async_4(sm.btab + i, map.bt_row + i);
    }
    uint32_t key[kChunk];
    load_chunk(row, 0, P, key);

    // ---- level 1: the bin b1 (top 11 key bits) of the K-th largest key
    for (int b = tid; b < kTopkBins; b += T) sm.hist[b] = 0;
    __syncthreads();
    for (int64_t c = 0; c < nchunks; ++c) {
        if (c > 0) load_chunk(row, c, P, key);
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            if (c * kChunkPools + static_cast<int64_t>(i) * T + tid < P) atomicAdd(&sm.hist[key[i] >> 21], 1u);
    }
    if (nchunks > 1) load_chunk(row, 0, P, key);
    cp_async_wait_all();
    __syncthreads();
    uint32_t b1, k1;
    block_find_bin(sm.hist, sm, kTopkBins, static_cast<uint32_t>(K), b1, k1);
    const uint32_t m_list = static_cast<uint32_t>(K) - k1 + sm.hist[b1];  // keys with bin >= b1
    if (nblk > 0) {
        map.btab = sm.btab;
        map.nblk = nblk;
    }

    uint32_t vcount = 0;
    if (m_list <= static_cast<uint32_t>(kTopkListCap)) {
        // ---- ordered list of the keys with bin >= b1: per chunk, warp ballots counted per
        //      (key slot, warp), one block scan over those counts, then the writes
        uint32_t listed = 0;
        for (int64_t c = 0; c < nchunks; ++c) {
            if (c > 0) load_chunk(row, c, P, key);
            const int64_t cbase = c * kChunkPools + tid;  // pool of key[0]; key[i] is pool cbase + i*T
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const uint32_t m = __ballot_sync(0xffffffffu, cbase + i * T < P && (key[i] >> 21) >= b1);
                if ((tid & 31) == 0) sm.cnt[i * (T / 32) + warp] = __popc(m);
            }
            __syncthreads();
            uint32_t total;
            const uint32_t ex = block_excl_scan(sm.cnt[tid], sm.scratch, &total);
            sm.cnt[tid] = ex;  // slot (i, warp) at index i * (T/32) + warp: index order
            __syncthreads();
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const bool sel = cbase + i * T < P && (key[i] >> 21) >= b1;
                const uint32_t m = __ballot_sync(0xffffffffu, sel);
                if (sel) {
                    const uint32_t pos = listed + sm.cnt[i * (T / 32) + warp] + __popc(m & lanemask_lt());
                    if (pos < static_cast<uint32_t>(kTopkListCap))
                        sm.list[pos] = make_uint2(key[i], static_cast<uint32_t>(c * kChunkPools + i * T + tid));
                }
            }
            listed += total;
            __syncthreads();  // sm.cnt is reused by the next chunk
        }
        for (int b = tid; b < kTopkBins; b += T) sm.hist[b] = 0;
        __syncthreads();
        const uint32_t n_list = min(listed, static_cast<uint32_t>(kTopkListCap));

        // ---- levels 2 and 3 among the list's keys of bin b1
        for (uint32_t g = tid; g < n_list; g += T) {
            const uint32_t k = sm.list[g].x;
            if ((k >> 21) == b1) atomicAdd(&sm.hist[(k >> 10) & 2047u], 1u);
        }
        __syncthreads();
        uint32_t b2, k2, b3, k3;
        block_find_bin(sm.hist, sm, 2048, k1, b2, k2);
        const uint32_t pre22 = (b1 << 11) | b2;
        for (int b = tid; b < 1024; b += T) sm.hist[b] = 0;
        __syncthreads();
        for (uint32_t g = tid; g < n_list; g += T) {
            const uint32_t k = sm.list[g].x;
            if ((k >> 10) == pre22) atomicAdd(&sm.hist[k & 1023u], 1u);
        }
        __syncthreads();
        block_find_bin(sm.hist, sm, 1024, k2, b3, k3);
        const uint32_t thr = (pre22 << 10) | b3;  // the K-th largest key of the row
        const uint32_t need_eq = k3;              // keys equal to thr that are kept (lowest index first)

        // ---- kept entries: keys > thr and the first need_eq keys == thr; one packed scan
        //      gives each its output column
        const uint32_t per = (n_list + T - 1) / T;
        const uint32_t g0 = tid * per, g1 = min(n_list, g0 + per);
        uint32_t gt = 0, eq = 0;
        for (uint32_t g = g0; g < g1; ++g) {
            const uint32_t k = sm.list[g].x;
            gt += k > thr;
            eq += k == thr;
        }
        uint32_t unused;
        const uint32_t pre2 = block_excl_scan(gt | (eq << 16), sm.scratch, &unused);
        uint32_t gt_run = pre2 & 0xffffu, eq_run = pre2 >> 16;
        for (uint32_t g = g0; g < g1; ++g) {
            const uint2 e = sm.list[g];
            const uint32_t out = gt_run + min(eq_run, need_eq);
            const bool keep = e.x > thr || (e.x == thr && eq_run < need_eq);
            gt_run += e.x > thr;
            eq_run += e.x == thr;
            if (keep)
                vcount += emit_pool<REMAP>(a, map, tok_row, slot_row, static_cast<int64_t>(out) * a.kpool,
                                           static_cast<int32_t>(static_cast<int64_t>(e.y) * a.kpool));
        }
    } else {
        // ---- crowded threshold bin (massive ties): levels 2 and 3 and the output re-read the row
        uint32_t pre = b1, shift = 21, krem = k1;
        for (int lvl = 0; lvl < 2; ++lvl) {
            const uint32_t nb = lvl == 0 ? 2048u : 1024u;
            const uint32_t sh = lvl == 0 ? 10u : 0u;
            for (int b = tid; b < kTopkBins; b += T) sm.hist[b] = 0;
            __syncthreads();
            for (int64_t c = 0; c < nchunks; ++c) {
                load_chunk(row, c, P, key);
#pragma unroll
                for (int i = 0; i < kChunk; ++i)
                    if (c * kChunkPools + i * T + tid < P && (key[i] >> shift) == pre)
                    atomicAdd(&sm.hist[(key[i] >> sh) & (nb - 1)], 1u);
            }
            __syncthreads();
            uint32_t bb, kk;
            block_find_bin(sm.hist, sm, static_cast<int>(nb), krem, bb, kk);
            pre = (pre << (lvl == 0 ? 11 : 10)) | bb;
            shift = sh;
            krem = kk;
        }
        const uint32_t thr = pre;
        const uint32_t need_eq = krem;
        // per chunk: counts of keys > thr and == thr per (key slot, warp), two block scans,
        // then each kept key's column = (keys > thr before it) + min(keys == thr before it, need_eq)
        uint32_t gt_base = 0, eq_base = 0;
        uint32_t* gcnt = sm.hist;          // [T]
        uint32_t* ecnt = sm.hist + T;      // [T]
        for (int64_t c = 0; c < nchunks; ++c) {
            load_chunk(row, c, P, key);
            const int64_t cbase = c * kChunkPools + tid;
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const bool in = cbase + i * T < P;
                const uint32_t mg = __ballot_sync(0xffffffffu, in && key[i] > thr);
                const uint32_t me = __ballot_sync(0xffffffffu, in && key[i] == thr);
                if ((tid & 31) == 0) {
                    gcnt[i * (T / 32) + warp] = __popc(mg);
                    ecnt[i * (T / 32) + warp] = __popc(me);
                }
            }
            __syncthreads();
            uint32_t gtot, etot;
            const uint32_t gex = block_excl_scan(gcnt[tid], sm.scratch, &gtot);
            __syncthreads();
            const uint32_t eex = block_excl_scan(ecnt[tid], sm.scratch, &etot);
            gcnt[tid] = gex;
            ecnt[tid] = eex;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const bool in = cbase + i * T < P;
                const bool g = in && key[i] > thr;
                const bool e = in && key[i] == thr;
                const uint32_t mg = __ballot_sync(0xffffffffu, g);
                const uint32_t me = __ballot_sync(0xffffffffu, e);
                const uint32_t gb = gt_base + gcnt[i * (T / 32) + warp] + __popc(mg & lanemask_lt());
                const uint32_t eb = eq_base + ecnt[i * (T / 32) + warp] + __popc(me & lanemask_lt());
                if (g || (e && eb < need_eq))
                    vcount += emit_pool<REMAP>(a, map, tok_row, slot_row,
                                               static_cast<int64_t>(gb + min(eb, need_eq)) * a.kpool,
                                               static_cast<int32_t>((c * kChunkPools + i * T + tid) * a.kpool));
            }
            gt_base += gtot;
            eq_base += etot;
            __syncthreads();
        }
    }

    // ---- trailing incomplete pool and -1 padding, valid count
    vcount += emit_run<REMAP>(a, map, tok_row, slot_row, K * a.kpool, P * a.kpool, ctx);
    const uint32_t total_valid = block_sum(vcount, sm.scratch);
    if (tid == 0 && a.counts) a.counts[r] = static_cast<int32_t>(total_valid);
}

size_t topk_smem_bytes(int bt_cap) {
    return (static_cast<size_t>(T) + kTopkBins) * 4 + static_cast<size_t>(kTopkListCap) * 8 +
           static_cast<size_t>((bt_cap + 3) & ~3) * 4 + (64 + 8) * 4;
}

cudaError_t launch_topk(const TopkArgs& a, bool remap, int rows, size_t smem, bool pdl, cudaStream_t s) {
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
    cfg.gridDim = dim3(static_cast<unsigned>(rows), 1, 1);
    cfg.blockDim = dim3(kTopkThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (remap) return cudaLaunchKernelEx(&cfg, k_topk_expand<true>, a);
    return cudaLaunchKernelEx(&cfg, k_topk_expand<false>, a);
}

}  // namespace sel
