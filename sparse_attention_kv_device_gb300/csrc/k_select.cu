// K-c1: the per-row tail of the fused selection: exact top-k pools, expansion and remap.
//
// Semantics as in k_topk.cu (vLLM flashinfer_mla_sparse_sm90 page, _kv_lens_host; ReVolta
// PR #59; remap from the vLLM sparse_utils page): keep the K = index_topk / kpool best
// complete pools of each row (score descending, lower pool index first), expand them and
// the trailing incomplete pool to ascending tokens, remap through the block table, -1 pad,
// count the non -1 slots.
//
// Input: the scorer's order-preserving 32-bit key of every complete pool of each row
// (ordered_key of the fp32 score).
//
// One 1024-thread CTA per row:
//   before the dependency wait: the row's descriptors (made by the segment builder, which
//       has completed before this grid can start) and its block-table entries, copied into
//       shared memory with cp.async; the histograms and bitmaps are cleared;
//   after it: the row's keys are copied into shared memory (cp.async, up to stage_cap of
//       them; longer rows read the rest from L2) and counted by their top 11 bits (level
//       1), which gives the bin b1 that holds the K-th largest key. One sweep over the keys
//       (one compare for each key below bin b1, about 97% of them) sets the bit of every
//       pool above b1 in a kept bitmap and of every pool in b1 in a second bitmap, and
//       counts bin b1's keys by bits 20..10 (level 2), with fire-and-forget shared-memory
//       atomics only. Level 3 (bits 9..0) and the marks at the exact threshold key visit
//       only the bin-b1 bits, each thread on its own run of bitmap words. One block scan
//       over the words then ranks the kept pools in ascending order into a list, which is
//       written out one column per thread (coalesced), expanded and remapped. Massive ties
//       take the same path.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {


struct SelSmem {
    uint32_t* keys;     // [stage_cap] the row's keys
    uint32_t* hist1;    // [kTopkBins] level-1 counts
    uint32_t* hist;     // [kTopkBins] level-2 counts
    uint32_t* hist3;    // [1024] level-3 counts
    uint32_t* gbm;      // [bm_words] pools whose key is above the threshold
    uint32_t* ebm;      // [bm_words] pools whose key equals it
    int32_t* list;      // [K] kept pools, ascending
    int32_t* btab;      // [bt_cap] the row's block-table entries
    uint32_t* scratch;  // [64]
    uint32_t* res;      // [8]
};

__device__ __forceinline__ int pad4(int n) { return (n + 3) & ~3; }

__device__ __forceinline__ SelSmem carve_sel(uint32_t* base, int stage_cap, int bm_words, int K, int bt_cap) {
    SelSmem s;
    s.keys = base;
    s.hist1 = s.keys + pad4(stage_cap);
    s.hist = s.hist1 + kTopkBins;
    s.hist3 = s.hist + kTopkBins;
    s.gbm = s.hist3 + 1024;
    s.ebm = s.gbm + pad4(bm_words);
    s.list = reinterpret_cast<int32_t*>(s.ebm + pad4(bm_words));
    s.btab = s.list + pad4(K);
    s.scratch = reinterpret_cast<uint32_t*>(s.btab + pad4(bt_cap));
    s.res = s.scratch + 64;
    return s;
}

// Given this thread's `n` counts of consecutive bins in descending order (thread 0 holds
// the highest bins; `first_bin` is this thread's highest), the bin holding the Kc-th
// largest key and Kc minus the keys above that bin.
template <int n>
__device__ __forceinline__ void find_bin_desc(const uint32_t (&h)[n], uint32_t first_bin, uint32_t Kc,
                                              const SelSmem& sm, uint32_t& bin, uint32_t& krem) {
    uint32_t local = 0;
#pragma unroll
    for (int i = 0; i < n; ++i) local += h[i];
    uint32_t total;
    const uint32_t above = block_excl_scan(local, sm.scratch, &total);
    if (above < Kc && Kc <= above + local) {
        uint32_t acc = above;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            if (acc < Kc && acc + h[i] >= Kc) {
                sm.res[0] = first_bin - i;
                sm.res[1] = Kc - acc;
            }
            acc += h[i];
        }
    }
    __syncthreads();
    bin = sm.res[0];
    krem = sm.res[1];
}

__device__ __forceinline__ uint32_t key_at(const SelSmem& sm, const uint32_t* krow, int p, int ns4) {
    return p < 4 * ns4 ? sm.keys[p] : __ldcg(krow + p);
}

__device__ __forceinline__ int32_t slot_of(const RowSelectArgs& a, const int32_t* btab, int nblk, const int32_t* bt_row,
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

}  // namespace

// T threads per row: 1,024 (one CTA per SM; rows up to the SM count) or 512 (two CTAs per SM,
// for chunks with more rows than SMs, so a chunk's rows run in one wave).
template <int T>
__global__ void __launch_bounds__(T, T == 512 ? 2 : 1) k_select_rows(const RowSelectArgs a) {
    constexpr int B1 = kTopkBins / T;  // level-1 / level-2 bins per thread
    constexpr int B3 = 1024 / T;       // level-3 bins per thread
    static_assert(B1 * T == kTopkBins && B3 * T == 1024, "the histograms split evenly over the threads");
    extern __shared__ __align__(16) uint32_t ssm[];
    const int tid = threadIdx.x;
    const int rl = blockIdx.x;
    const int r = a.row_begin + rl;
    const int K = a.topk / a.kpool;
    SelSmem sm = carve_sel(ssm, a.stage_cap, a.bm_words, K, a.bt_cap);
    // the next chunk's scorer may launch once every CTA of this grid is resident: it fetches
    // its tiles meanwhile and stores no score before this grid has finished
    if (a.next_chunk) pdl_launch_dependents();

    // ---- before the wait: only inputs and data of grids that completed before this one
    //      could start (row descriptors from the segment builder, keys from the scorer)
    const int32_t c = __ldcg(a.row_ctx + rl);
    const int req = __ldcg(a.row_req + rl);
    const bool valid = c >= 0 && req >= 0;
    const int64_t ctx = valid ? c : 0;
    const bool selects = valid && ctx > a.topk;
    const int P = selects ? static_cast<int>(ctx / a.kpool) : 0;
    const int32_t* bt_row = a.block_table + static_cast<int64_t>(valid ? req : 0) * a.bt_ld;
    const uint32_t* krow = a.keys + static_cast<int64_t>(rl) * a.keys_ld;

    int nblk = 0;
    if (valid) {
        int64_t need = (ctx + a.block_size - 1) / a.block_size;
        if (need > a.max_blocks) need = a.max_blocks;
        nblk = static_cast<int>(need < a.bt_cap ? need : a.bt_cap);
        for (int i = tid; i < nblk; i += T) cp_async_4(sm.btab + i, bt_row + i);
    }
    // full key vectors [0, ns4) are staged in shared memory; keys past them (a longer row's
    // rest, the last partial vector) are read from global memory
    const int ns4 = (P >> 2) < (a.stage_cap >> 2) ? (P >> 2) : (a.stage_cap >> 2);
    const int nwords = (P + 31) >> 5;
    if (selects) {
        for (int i = tid; i < kTopkBins; i += T) {
            sm.hist1[i] = 0;
            sm.hist[i] = 0;
        }
        for (int i = tid; i < 1024; i += T) sm.hist3[i] = 0;
        for (int w = tid; w < nwords; w += T) {
            sm.gbm[w] = 0;
            sm.ebm[w] = 0;
        }
    }

    pdl_wait();  // the scorer's keys are complete
    __syncthreads();  // every histogram and bitmap word is cleared before any thread counts into it

    uint32_t vcount = 0;
    int64_t run_from = 0;  // columns [col_run, out_width) get tokens run_from .. ctx-1, then -1
    int col_run = 0;
    if (selects) {
        const int full4 = P >> 2;
        const uint4* ks = reinterpret_cast<const uint4*>(sm.keys);
        const uint4* kg = reinterpret_cast<const uint4*>(krow);
        // level 1: the row's keys, eight vectors per thread loaded together into registers,
        // stored into shared memory (the first ns4 vectors) and counted by bits 31..21 with
        // fire-and-forget shared atomics
        uint4* ksw = reinterpret_cast<uint4*>(sm.keys);
        auto count1 = [&sm](uint32_t k) { atomicAdd(&sm.hist1[k >> 21], 1u); };
        for (int base = 0; base < full4; base += 8 * T) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i4 = base + j * T + tid;
                v[j] = i4 < full4 ? __ldcg(kg + i4) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i4 = base + j * T + tid;
                if (i4 < full4) {
                    if (i4 < ns4) ksw[i4] = v[j];
                    count1(v[j].x);
                    count1(v[j].y);
                    count1(v[j].z);
                    count1(v[j].w);
                }
            }
        }
        {
            // the last partial vector: its keys are read from global memory wherever needed
            const int tail = P - 4 * full4;
            if (tid < tail) count1(__ldcg(krow + 4 * full4 + tid));
        }
        cp_async_wait_all();  // the block-table entries
        __syncthreads();
        uint32_t h1[B1];
#pragma unroll
        for (int i = 0; i < B1; ++i) h1[i] = sm.hist1[kTopkBins - 1 - B1 * tid - i];
        uint32_t b1, k1;
        find_bin_desc<B1>(h1, kTopkBins - 1 - B1 * tid, static_cast<uint32_t>(K), sm, b1, k1);

        // ---- the one full sweep: keys below bin b1 (nearly all of them) cost a compare each.
        //      A thread first records which of its next 32 keys are at or above b1 in a mask,
        //      then visits those few together with the other lanes (not one lane at a time):
        //      a key above b1 sets its pool's bit in the kept bitmap, a key in b1 sets its
        //      bit in the bin-b1 bitmap (ebm, until the marks below) and counts by bits 20..10.
        const uint32_t lo1 = b1 << 21;
        {
            for (int base = 0; base < full4; base += 8 * T) {
                uint32_t hits = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int i4 = base + j * T + tid;
                    if (i4 < full4) {
                        const uint4 v = i4 < ns4 ? ks[i4] : __ldcg(kg + i4);
                        hits |= ((v.x >= lo1 ? 1u : 0u) | (v.y >= lo1 ? 2u : 0u) | (v.z >= lo1 ? 4u : 0u) |
                                 (v.w >= lo1 ? 8u : 0u))
                                << (4 * j);
                    }
                }
                while (hits) {
                    const int h = __ffs(hits) - 1;
                    hits &= hits - 1;
                    const int p = 4 * (base + (h >> 2) * T + tid) + (h & 3);
                    const uint32_t k = key_at(sm, krow, p, ns4);
                    const bool in_b1 = (k >> 21) == b1;
                    atomicOr((in_b1 ? sm.ebm : sm.gbm) + (p >> 5), 1u << (p & 31));
                    if (in_b1) atomicAdd(&sm.hist[(k >> 10) & 2047u], 1u);
                }
            }
            const int tail = P - 4 * full4;
            if (tid < tail) {
                const int p = 4 * full4 + tid;
                const uint32_t k = key_at(sm, krow, p, ns4);
                if (k >= lo1) {
                    const bool in_b1 = (k >> 21) == b1;
                    atomicOr((in_b1 ? sm.ebm : sm.gbm) + (p >> 5), 1u << (p & 31));
                    if (in_b1) atomicAdd(&sm.hist[(k >> 10) & 2047u], 1u);
                }
            }
        }
        __syncthreads();
        uint32_t b2, k2;
        {
            uint32_t h2[B1];
#pragma unroll
            for (int i = 0; i < B1; ++i) h2[i] = sm.hist[kTopkBins - 1 - B1 * tid - i];
            find_bin_desc<B1>(h2, kTopkBins - 1 - B1 * tid, k1, sm, b2, k2);
        }

        // ---- level 3 and the marks at the threshold, on the bin-b1 keys of the bitmap words
        //      this thread also ranks below (a contiguous run of words per thread)
        const int per = (nwords + T - 1) / T;
        const int w0 = tid * per, w1 = min(nwords, w0 + per);
        const uint32_t pre22 = (b1 << 11) | b2;
        for (int w = w0; w < w1; ++w) {
            uint32_t m = sm.ebm[w];
            while (m) {
                const int p = w * 32 + __ffs(m) - 1;
                m &= m - 1;
                const uint32_t k = key_at(sm, krow, p, ns4);
                if ((k >> 10) == pre22) atomicAdd(&sm.hist3[k & 1023u], 1u);
            }
        }
        __syncthreads();
        uint32_t b3, need_eq;
        {
            uint32_t h3[B3];
#pragma unroll
            for (int i = 0; i < B3; ++i) h3[i] = sm.hist3[1023 - B3 * tid - i];
            find_bin_desc<B3>(h3, 1023u - B3 * tid, k2, sm, b3, need_eq);
        }
        const uint32_t thr = (pre22 << 10) | b3;
        const uint32_t n_eq = sm.hist3[b3];
        for (int w = w0; w < w1; ++w) {
            uint32_t m = sm.ebm[w], gt = 0, eq = 0;
            while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1;
                const uint32_t k = key_at(sm, krow, w * 32 + bit, ns4);
                if (k > thr) gt |= 1u << bit;
                else if (k == thr) eq |= 1u << bit;
            }
            sm.gbm[w] |= gt;
            sm.ebm[w] = eq;  // from here on: the pools equal to the threshold
        }
        __syncthreads();

        // ---- kept pools in ascending order: all above the threshold and the first need_eq
        //      equal ones
        uint32_t tot;
        if (n_eq > need_eq) {  // ties at the threshold: rank the equal keys (uniform branch)
            uint32_t eqc = 0;
            for (int w = w0; w < w1; ++w) eqc += __popc(sm.ebm[w]);
            uint32_t eq_before = block_excl_scan(eqc, sm.scratch, &tot);
            for (int w = w0; w < w1; ++w) {
                const uint32_t e = sm.ebm[w];
                uint32_t take_mask = 0;
                if (eq_before < need_eq && e) {
                    uint32_t take = min(static_cast<uint32_t>(__popc(e)), need_eq - eq_before);
                    uint32_t rest = e;
                    while (take--) {
                        const uint32_t lowest = rest & (0u - rest);
                        take_mask |= lowest;
                        rest ^= lowest;
                    }
                }
                eq_before += __popc(e);
                sm.ebm[w] = take_mask;
            }
            __syncthreads();
        }
        uint32_t keptc = 0;
        for (int w = w0; w < w1; ++w) keptc += __popc(sm.gbm[w] | sm.ebm[w]);
        uint32_t pos = block_excl_scan(keptc, sm.scratch, &tot);
        for (int w = w0; w < w1; ++w) {
            uint32_t kept = sm.gbm[w] | sm.ebm[w];
            while (kept) {
                const int bit = __ffs(kept) - 1;
                kept &= kept - 1;
                if (pos < static_cast<uint32_t>(K)) sm.list[pos] = w * 32 + bit;
                ++pos;
            }
        }
        __syncthreads();
        run_from = static_cast<int64_t>(P) * a.kpool;
        col_run = K * a.kpool;
    } else {
        cp_async_wait_all();
        __syncthreads();
    }

    // ---- one column per thread: the kept pools' tokens, then the trailing tokens (for a
    //      short row, every token), then -1; remapped; the valid count
    int32_t* slot_row = a.slots + static_cast<int64_t>(r) * a.out_width;
    int32_t* tok_row = a.token_idx ? a.token_idx + static_cast<int64_t>(r) * a.out_width : nullptr;
    for (int col = tid; col < a.out_width; col += T) {
        int32_t t;
        if (col < col_run) {
            const int q = a.kpool_shift >= 0 ? (col >> a.kpool_shift) : col / a.kpool;
            t = sm.list[q] * a.kpool + (col - q * a.kpool);
        } else {
            const int64_t tt = run_from + (col - col_run);
            t = valid && tt < ctx ? static_cast<int32_t>(tt) : -1;
        }
        const int32_t s = slot_of(a, sm.btab, nblk, bt_row, t);
        slot_row[col] = s;
        if (tok_row) tok_row[col] = t;
        vcount += s != -1;
    }
    const uint32_t total = block_sum(vcount, sm.scratch);
    if (tid == 0 && a.counts) a.counts[r] = static_cast<int32_t>(total);
}

size_t select_smem_bytes(int stage_cap, int bm_words, int K, int bt_cap) {
    auto p4 = [](int64_t n) { return static_cast<size_t>((n + 3) & ~int64_t(3)); };
    return 4 * (p4(stage_cap) + 2 * kTopkBins + 1024 + 2 * p4(bm_words) +
                p4(K) + p4(bt_cap) + 64 + 8);
}

cudaError_t launch_select_rows(const RowSelectArgs& a, int rows, size_t smem, bool pdl, cudaStream_t s,
                               int threads) {
    static size_t configured[2][kMaxDevicesTracked] = {};
    const int v = threads == 512 ? 1 : 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevicesTracked && smem > configured[v][dev]) {
        cudaError_t e = v ? cudaFuncSetAttribute(k_select_rows<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem))
                          : cudaFuncSetAttribute(k_select_rows<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[v][dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(v ? 512 : 1024), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return v ? cudaLaunchKernelEx(&cfg, k_select_rows<512>, a) : cudaLaunchKernelEx(&cfg, k_select_rows<1024>, a);
}

}  // namespace sel
