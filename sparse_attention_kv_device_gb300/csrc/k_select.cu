// K-c1, K-c2: the wide tail of the radix top-k used by the fused selection.
//
// Semantics as in k_topk.cu (vLLM flashinfer_mla_sparse_sm90 page, _kv_lens_host; ReVolta
// PR #59; remap from the vLLM sparse_utils page): keep the K = index_topk / kpool best
// complete pools of each row (score descending, lower pool index first), expand them and
// the trailing incomplete pool to ascending tokens, remap through the block table, -1 pad,
// count the non -1 slots.
//
// After the histogram kernel has counted every row's keys by their top 11 bits:
//   k_collect (CTA = 2048 pools of one row): reads the row's histogram, finds the bin b1
//       holding the K-th largest key, and appends its keys with bin >= b1 (about K plus a
//       few hundred) to the row's candidate buffer: warp ballots place them, one global
//       atomic per warp reserves room. The order of the buffer does not matter.
//   k_finalize (CTA = one row): finds the exact K-th largest key among the candidates of
//       bin b1 (two local radix levels over the remaining 21 bits), marks the kept pools
//       in a bitmap over the row (keys above the threshold, and the lowest-index ones equal
//       to it), and writes them in ascending pool order from one scan over the bitmap
//       words, expanded and remapped. If a row's candidates overflow the buffer (massive
//       ties), it re-reads the row's scores for levels 2 and 3 instead; the bitmap output
//       is the same.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

SEL_PHASE_TABLE(select)

namespace {

constexpr int kCT = kCollectThreads;
constexpr int kFT = kFinalizeThreads;
static_assert(kCT * 8 == kTopkBins, "k_collect holds 8 histogram bins per thread");

// Suffix search over a 2048-bin histogram held 8 bins per thread in descending order
// (thread t holds bins 2047-8t .. 2040-8t): the bin of the Kc-th largest key and Kc minus
// the keys above it. `scratch` >= 33 words, `res` >= 2 words of shared memory.
__device__ __forceinline__ void find_bin_desc8(const uint32_t (&h)[8], uint32_t Kc, uint32_t* scratch, uint32_t* res,
                                               uint32_t& bin, uint32_t& krem) {
    uint32_t local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) local += h[i];
    uint32_t total;
    const uint32_t above = block_excl_scan(local, scratch, &total);
    if (above < Kc && Kc <= above + local) {
        uint32_t acc = above;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (acc < Kc && acc + h[i] >= Kc) {
                res[0] = 2047u - (8u * threadIdx.x + i);
                res[1] = Kc - acc;
            }
            acc += h[i];
        }
    }
    __syncthreads();
    bin = res[0];
    krem = res[1];
}

}  // namespace

__global__ void __launch_bounds__(kCollectThreads) k_collect(const CollectArgs a) {
    __shared__ uint32_t scratch[40];
    __shared__ uint32_t res[2];
    pdl_wait();               // the row histograms are complete
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31;
    const int rl = blockIdx.y;
    const int32_t c = a.row_ctx[rl];
    if (c <= a.topk) return;
    const int64_t P = c / a.kpool;
    const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kHistSlice;
    if (s0 >= P) return;
    const int n = static_cast<int>(P - s0 < kHistSlice ? P - s0 : kHistSlice);

    // histogram bins 2047-8t .. 2040-8t and this CTA's scores, loaded together
    const uint4* hrow = reinterpret_cast<const uint4*>(a.hist + static_cast<int64_t>(rl) * kTopkBins);
    const uint4 hA = __ldcg(hrow + (2040 - 8 * tid) / 4 + 1);  // bins 2044-8t .. 2047-8t
    const uint4 hB = __ldcg(hrow + (2040 - 8 * tid) / 4);      // bins 2040-8t .. 2043-8t
    const float4* src = reinterpret_cast<const float4*>(a.scores + static_cast<int64_t>(rl) * a.scores_ld + s0);
    constexpr int kVec = kHistSlice / 4 / kCT;
    float4 v[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const int i4 = tid + j * kCT;
        v[j] = 4 * i4 < n ? __ldcg(src + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const uint32_t h[8] = {hA.w, hA.z, hA.y, hA.x, hB.w, hB.z, hB.y, hB.x};
    uint32_t b1, k1;
    find_bin_desc8(h, static_cast<uint32_t>(a.topk / a.kpool), scratch, res, b1, k1);
    if (blockIdx.x == 0 && tid == 0) a.row_sel[rl] = make_int2(static_cast<int>(b1), static_cast<int>(k1));

    // keys with bin >= b1: a warp's ballots give each its place, one atomic per warp reserves room
    uint32_t key[4 * kVec];
    bool sel[4 * kVec];
    uint32_t mine = 0;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const int i = 4 * (tid + j * kCT);
        const float f[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            key[4 * j + u] = ordered_key(f[u]);
            sel[4 * j + u] = i + u < n && (key[4 * j + u] >> 21) >= b1;
            mine += sel[4 * j + u];
        }
    }
    const uint32_t incl = warp_incl_scan(mine);
    const uint32_t wtotal = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t base = 0;
    if (lane == 31 && wtotal) base = atomicAdd(a.row_count + rl, wtotal);
    base = __shfl_sync(0xffffffffu, base, 31);
    uint32_t pos = base + incl - mine;
    uint2* out = a.cand + static_cast<int64_t>(rl) * a.cand_cap;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const int i = 4 * (tid + j * kCT);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (sel[4 * j + u]) {
                if (pos < static_cast<uint32_t>(a.cand_cap))
                    out[pos] = make_uint2(key[4 * j + u], static_cast<uint32_t>(s0 + i + u));
                ++pos;
            }
        }
    }
    const int cta = blockIdx.y * gridDim.x + blockIdx.x;
    (void)cta;
    if (tid == 0 && cta < 256) SEL_PHASE(cta);  // diagnostics: collect CTA end
}

namespace {

struct FinSmem {
    uint2* cand;       // [cand_cap]
    uint32_t* hist;    // [kTopkBins]
    uint32_t* gbm;     // [bm_words] pools whose key is above the threshold
    uint32_t* ebm;     // [bm_words] pools whose key equals the threshold
    int32_t* btab;     // [bt_cap]
    uint32_t* scratch; // [64]
    uint32_t* res;     // [8]
};

__device__ __forceinline__ FinSmem carve_fin(uint32_t* base, int cand_cap, int bm_words, int bt_cap) {
    FinSmem s;
    s.cand = reinterpret_cast<uint2*>(base);
    s.hist = reinterpret_cast<uint32_t*>(s.cand + cand_cap);
    s.gbm = s.hist + kTopkBins;
    s.ebm = s.gbm + bm_words;
    s.btab = reinterpret_cast<int32_t*>(s.ebm + bm_words);
    s.scratch = reinterpret_cast<uint32_t*>(s.btab + ((bt_cap + 3) & ~3));
    s.res = s.scratch + 64;
    return s;
}

// The bin (of `nbins`, counted from the top) holding the Kc-th largest key counted in
// `hist` (shared), and Kc minus the keys above it.
__device__ __forceinline__ void fin_find_bin(const uint32_t* hist, const FinSmem& sm, int nbins, uint32_t Kc,
                                             uint32_t& bin, uint32_t& krem) {
    const int per = nbins / kFT;
    uint32_t local = 0;
    for (int i = 0; i < per; ++i) local += hist[nbins - 1 - (threadIdx.x * per + i)];
    uint32_t total;
    const uint32_t above = block_excl_scan(local, sm.scratch, &total);
    if (above < Kc && Kc <= above + local) {
        uint32_t acc = above;
        for (int i = 0; i < per; ++i) {
            const int b = nbins - 1 - (threadIdx.x * per + i);
            if (acc < Kc && acc + hist[b] >= Kc) {
                sm.res[0] = static_cast<uint32_t>(b);
                sm.res[1] = Kc - acc;
            }
            acc += hist[b];
        }
    }
    __syncthreads();
    bin = sm.res[0];
    krem = sm.res[1];
}

__device__ __forceinline__ int32_t fin_slot(const FinalizeArgs& a, const int32_t* btab, int nblk,
                                            const int32_t* bt_row, int32_t t) {
    if (t < 0) return -1;
    const int32_t b = t / a.block_size;
    int32_t ph;
    if (btab && b < nblk) {
        ph = btab[b];
    } else {
        if (b >= a.max_blocks) return -1;
        ph = __ldg(bt_row + b);
    }
    if (ph < 0 || ph >= a.num_kv_blocks) return -1;
    return static_cast<int32_t>(static_cast<int64_t>(ph) * a.block_stride_rows + (t - b * a.block_size));
}

}  // namespace

__global__ void __launch_bounds__(kFinalizeThreads, 1) k_finalize(const FinalizeArgs a) {
    extern __shared__ __align__(16) uint32_t fsm[];
    const int tid = threadIdx.x;
    const int rl = blockIdx.x;
    const int r = a.row_begin + rl;
    FinSmem sm = carve_fin(fsm, a.cand_cap, a.bm_words, a.bt_cap);
    pdl_wait();  // candidates, histograms and row descriptors are complete

    const int32_t c = a.row_ctx[rl];
    const int req = a.row_req[rl];
    const bool valid = c >= 0 && req >= 0;
    const int64_t ctx = valid ? c : 0;
    const int K = a.topk / a.kpool;
    int32_t* slot_row = a.slots + static_cast<int64_t>(r) * a.out_width;
    int32_t* tok_row = a.token_idx ? a.token_idx + static_cast<int64_t>(r) * a.out_width : nullptr;
    const int32_t* bt_row = a.block_table + static_cast<int64_t>(valid ? req : 0) * a.bt_ld;

    // the row's block-table entries, copied asynchronously while the rest loads
    int nblk = 0;
    if (valid) {
        int64_t need = (ctx + a.block_size - 1) / a.block_size;
        if (need > a.max_blocks) need = a.max_blocks;
        if (need <= a.bt_cap) nblk = static_cast<int>(need);
        for (int i = tid; i < nblk; i += kFT) cp_async_4(sm.btab + i, bt_row + i);
    }
    const int32_t* btab = nblk > 0 ? sm.btab : nullptr;

    uint32_t vcount = 0;
    int64_t run_from = 0;   // columns [col_run, W) get tokens run_from .. ctx-1, then -1
    int col_run = 0;
    if (valid && ctx > a.topk) {
        const int64_t P = ctx / a.kpool;
        const int nwords = static_cast<int>((P + 31) / 32);
        const uint32_t n_cand = min(a.row_count[rl], static_cast<uint32_t>(0x7fffffff));
        const int2 bk = a.row_sel[rl];
        const uint32_t b1 = static_cast<uint32_t>(bk.x), k1 = static_cast<uint32_t>(bk.y);
        for (int w = tid; w < nwords; w += kFT) {
            sm.gbm[w] = 0;
            sm.ebm[w] = 0;
        }
        for (int b = tid; b < kTopkBins; b += kFT) sm.hist[b] = 0;
        uint32_t thr, need_eq;
        if (n_cand <= static_cast<uint32_t>(a.cand_cap)) {
            const uint2* cr = a.cand + static_cast<int64_t>(rl) * a.cand_cap;
            for (uint32_t g = tid; g < n_cand; g += kFT) sm.cand[g] = __ldcg(cr + g);
            __syncthreads();
            // levels 2 and 3 among the candidates of bin b1
            for (uint32_t g = tid; g < n_cand; g += kFT) {
                const uint32_t k = sm.cand[g].x;
                if ((k >> 21) == b1) atomicAdd(&sm.hist[(k >> 10) & 2047u], 1u);
            }
            __syncthreads();
            uint32_t b2, k2, b3, k3;
            fin_find_bin(sm.hist, sm, 2048, k1, b2, k2);
            const uint32_t pre22 = (b1 << 11) | b2;
            for (int b = tid; b < 1024; b += kFT) sm.hist[b] = 0;
            __syncthreads();
            for (uint32_t g = tid; g < n_cand; g += kFT) {
                const uint32_t k = sm.cand[g].x;
                if ((k >> 10) == pre22) atomicAdd(&sm.hist[k & 1023u], 1u);
            }
            __syncthreads();
            fin_find_bin(sm.hist, sm, 1024, k2, b3, k3);
            thr = (pre22 << 10) | b3;
            need_eq = k3;
            for (uint32_t g = tid; g < n_cand; g += kFT) {
                const uint2 e = sm.cand[g];
                if (e.x > thr) atomicOr(&sm.gbm[e.y >> 5], 1u << (e.y & 31));
                else if (e.x == thr) atomicOr(&sm.ebm[e.y >> 5], 1u << (e.y & 31));
            }
        } else {
            // crowded threshold bin: levels 2 and 3 from the row's scores
            const float* row = a.scores + static_cast<int64_t>(rl) * a.scores_ld;
            __syncthreads();
            uint32_t pre = b1, shift = 21, krem = k1;
            for (int lvl = 0; lvl < 2; ++lvl) {
                const uint32_t nb = lvl == 0 ? 2048u : 1024u;
                const uint32_t sh = lvl == 0 ? 10u : 0u;
                for (int64_t p = tid; p < P; p += kFT) {
                    const uint32_t k = ordered_key(__ldcg(row + p));
                    if ((k >> shift) == pre) atomicAdd(&sm.hist[(k >> sh) & (nb - 1)], 1u);
                }
                __syncthreads();
                uint32_t bb, kk;
                fin_find_bin(sm.hist, sm, static_cast<int>(nb), krem, bb, kk);
                pre = (pre << (lvl == 0 ? 11 : 10)) | bb;
                shift = sh;
                krem = kk;
                for (int b = tid; b < kTopkBins; b += kFT) sm.hist[b] = 0;
                __syncthreads();
            }
            thr = pre;
            need_eq = krem;
            for (int64_t p = tid; p < P; p += kFT) {
                const uint32_t k = ordered_key(__ldcg(row + p));
                if (k > thr) atomicOr(&sm.gbm[p >> 5], 1u << (p & 31));
                else if (k == thr) atomicOr(&sm.ebm[p >> 5], 1u << (p & 31));
            }
        }
        cp_async_wait_all();
        __syncthreads();

        // ---- kept pools in ascending order: every key above the threshold and the first
        //      need_eq equal ones; thread t scans a contiguous range of bitmap words
        const int per = (nwords + kFT - 1) / kFT;
        const int w0 = tid * per, w1 = min(nwords, w0 + per);
        uint32_t eqc = 0;
        for (int w = w0; w < w1; ++w) eqc += __popc(sm.ebm[w]);
        uint32_t tot;
        uint32_t eq_before = block_excl_scan(eqc, sm.scratch, &tot);
        uint32_t keptc = 0;
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
            sm.ebm[w] = take_mask;  // from here on: the equal keys that are kept
            keptc += __popc(sm.gbm[w] | take_mask);
        }
        __syncthreads();
        uint32_t pos = block_excl_scan(keptc, sm.scratch, &tot);
        for (int w = w0; w < w1; ++w) {
            uint32_t kept = sm.gbm[w] | sm.ebm[w];
            while (kept) {
                const int bit = __ffs(kept) - 1;
                kept &= kept - 1;
                const int32_t t0 = static_cast<int32_t>((static_cast<int64_t>(w) * 32 + bit) * a.kpool);
                const int64_t col = static_cast<int64_t>(pos++) * a.kpool;
                for (int u = 0; u < a.kpool; ++u) {
                    const int32_t s = fin_slot(a, btab, nblk, bt_row, t0 + u);
                    slot_row[col + u] = s;
                    if (tok_row) tok_row[col + u] = t0 + u;
                    vcount += s != -1;
                }
            }
        }
        run_from = P * a.kpool;
        col_run = K * a.kpool;
    } else {
        cp_async_wait_all();
        __syncthreads();
    }

    // ---- short rows (every token), the trailing incomplete pool, -1 padding; valid count
    for (int col = col_run + tid; col < a.out_width; col += kFT) {
        const int64_t tt = run_from + (col - col_run);
        const int32_t t = valid && tt < ctx ? static_cast<int32_t>(tt) : -1;
        const int32_t s = fin_slot(a, btab, nblk, bt_row, t);
        slot_row[col] = s;
        if (tok_row) tok_row[col] = t;
        vcount += s != -1;
    }
    const uint32_t total = block_sum(vcount, sm.scratch);
    if (tid == 0 && a.counts) a.counts[r] = static_cast<int32_t>(total);
    if (tid == 0 && rl < 256) SEL_PHASE(256 + rl);  // diagnostics: finalize row end
}

size_t finalize_smem_bytes(int cand_cap, int bm_words, int bt_cap) {
    return static_cast<size_t>(cand_cap) * 8 + kTopkBins * 4 + 2 * static_cast<size_t>(bm_words) * 4 +
           static_cast<size_t>((bt_cap + 3) & ~3) * 4 + (64 + 8) * 4;
}

cudaError_t launch_collect(const CollectArgs& a, int rows, int64_t max_pools, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    const int64_t gx = (max_pools + kHistSlice - 1) / kHistSlice;
    cfg.gridDim = dim3(static_cast<unsigned>(gx > 0 ? gx : 1), static_cast<unsigned>(rows), 1);
    cfg.blockDim = dim3(kCollectThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_collect, a);
}

cudaError_t launch_finalize(const FinalizeArgs& a, int rows, size_t smem, bool pdl, cudaStream_t s) {
    static size_t configured[kMaxDevicesTracked] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevicesTracked && smem > configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_finalize, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows), 1, 1);
    cfg.blockDim = dim3(kFinalizeThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_finalize, a);
}

}  // namespace sel
