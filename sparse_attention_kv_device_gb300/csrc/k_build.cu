// K-a: device-side request-segment builder.
//
// ReVolta PR #59 ("Change") builds the segment descriptors on the device so the
// selection call stays CUDA-graph safe; row contexts follow _kv_lens_host on the
// vLLM flashinfer_mla_sparse_sm90 page (context = position + 1). One launch plans
// every chunk of a call, one CTA per chunk of chunk_rows rows, each into its own plan
// block (plan_stride bytes apart), so the chunks' scorers and selects run back to back
// with no builder between them. A CTA reads query_start_loc and positions for its
// chunk and writes:
//   row_req / row_ctx  per row (-1 ctx = no output: padding, out of bound, bad table)
//   seg[]              {request, first row, rows (<= seg_rows), pools to score}
//   seg_tile_prefix[]  exclusive prefix of ceil(pools / 128) over segments
//   hdr                {segments, tiles, 0 (the scorer's tile counter)}
// The inputs are staged in shared memory when they fit (generic pointers fall back
// to the global workspace copies otherwise), so the CTA pays few memory round trips.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

__device__ __forceinline__ int last_le(const int32_t* v, int n, int x) {
    // largest i in [0, n) with v[i] <= x (v non-decreasing, v[0] <= x)
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (v[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace

__global__ void __launch_bounds__(kBuildThreads) k_build_segments(const BuildArgs in) {
    extern __shared__ __align__(16) uint8_t bsm[];
    __shared__ uint32_t scratch[40];
    // Launched as a dependent (the host-buffer entry point's staging kernel precedes it), the
    // builder waits for its inputs here; otherwise the wait returns at once. The scorer, which
    // reads query_start_loc and positions before any wait of its own, may start after this.
    pdl_wait();
    pdl_launch_dependents();
    // this CTA's chunk and plan block
    BuildArgs a = in;
    {
        a.row_begin = in.row_begin + static_cast<int>(blockIdx.x) * in.chunk_rows;
        a.row_end = min(in.row_end, a.row_begin + in.chunk_rows);
        const int64_t off = static_cast<int64_t>(blockIdx.x) * in.plan_stride;
        auto at = [off](auto* p) { return reinterpret_cast<decltype(p)>(reinterpret_cast<uint8_t*>(p) + off); };
        a.row_req = at(in.row_req);
        a.row_ctx = at(in.row_ctx);
        a.seg = at(in.seg);
        a.seg_tile_prefix = at(in.seg_tile_prefix);
        a.hdr = at(in.hdr);
    }
    const int tid = threadIdx.x;
    const int nchunk = a.row_end - a.row_begin;

    // shared-memory staging (host decided what fits); generic pointers either way
    int32_t* qsl = a.smem_qsl ? reinterpret_cast<int32_t*>(bsm) : const_cast<int32_t*>(a.qsl);
    int32_t* ctx = a.smem_rows ? reinterpret_cast<int32_t*>(bsm + a.smem_rows_off) : a.row_ctx;
    int4* seg = a.smem_segs ? reinterpret_cast<int4*>(bsm + a.smem_segs_off) : a.seg;
    int32_t* prefix = a.smem_segs ? reinterpret_cast<int32_t*>(bsm + a.smem_prefix_off) : a.seg_tile_prefix;

    // every input load of the kernel is issued here, before the first barrier
    if (a.smem_qsl)
        for (int i = tid; i <= a.num_reqs; i += blockDim.x) qsl[i] = a.qsl[i];
    int32_t pos_reg[4];  // positions of rows tid, tid + kBuildThreads, ... (the first 4 x kBuildThreads rows)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int k = tid + j * kBuildThreads;
        pos_reg[j] = k < nchunk ? __ldg(a.positions + a.row_begin + k) : 0;
    }
    __syncthreads();

    // 1. query_start_loc must be non-decreasing inside [0, num_rows].
    int bad = 0;
    for (int i = tid; i < a.num_reqs; i += blockDim.x) bad |= qsl[i] > qsl[i + 1];
    if (tid == 0) bad |= (qsl[0] < 0) | (qsl[a.num_reqs] > a.num_rows);
    bad = __syncthreads_or(bad);
    if (bad) {
        for (int r = tid; r < nchunk; r += blockDim.x) {
            a.row_req[r] = -1;
            a.row_ctx[r] = -1;
        }
        if (tid == 0) {
            report(a.status, kStBadQsl);
            a.hdr[0] = 0;
            a.hdr[1] = 0;
            a.hdr[2] = 0;
            a.seg_tile_prefix[0] = 0;
        }
        return;
    }

    // 2. per row: request (binary search in qsl) and context.
    for (int k = tid; k < nchunk; k += blockDim.x) {
        const int r = a.row_begin + k;
        int req = -1;
        if (a.num_reqs > 0 && qsl[0] <= r) {
            const int i = last_le(qsl, a.num_reqs + 1, r);
            if (i < a.num_reqs && r < qsl[i + 1]) req = i;
        }
        const int j = (k - tid) / kBuildThreads;
        const int64_t c64 = static_cast<int64_t>(j < 4 ? pos_reg[j] : __ldg(a.positions + r)) + 1;
        int32_t c = -1;
        if (req >= 0) {
            if (c64 > a.max_context) {
                report(a.status, kStCtxOverBound);
                req = -1;
            } else {
                c = c64 > 0 ? static_cast<int32_t>(c64) : 0;
            }
        }
        a.row_req[k] = req;
        ctx[k] = c;
        if (a.smem_rows) a.row_ctx[k] = c;
    }
    __syncthreads();

    // 3. segments: request i's rows inside the chunk, cut every seg_rows rows.
    uint32_t carry = 0;
    for (int base = 0; base < a.num_reqs; base += blockDim.x) {
        const int i = base + tid;
        int lo = 0, hi = 0;
        uint32_t ns = 0;
        if (i < a.num_reqs) {
            lo = max(qsl[i], a.row_begin);
            hi = min(qsl[i + 1], a.row_end);
            if (hi > lo) ns = (hi - lo + a.seg_rows - 1) / a.seg_rows;
        }
        uint32_t total;
        const uint32_t first = carry + block_excl_scan(ns, scratch, &total);
        for (uint32_t k = 0; k < ns; ++k) {
            const uint32_t s = first + k;
            if (s >= static_cast<uint32_t>(a.max_segs)) break;  // cannot happen with the host bound
            const int row0 = lo + static_cast<int>(k) * a.seg_rows;
            seg[s] = make_int4(i, row0, min(a.seg_rows, hi - row0), 0);  // pools: below
        }
        carry += total;
        __syncthreads();
    }
    const int nseg = min(static_cast<int>(carry), a.max_segs);

    // 3b. pools to score per segment: the largest over its rows, one warp per segment
    //     (a segment has at most 64 rows: two per lane)
    {
        const int lane = tid & 31, nwarps = blockDim.x >> 5;
        for (int s = tid >> 5; s < nseg; s += nwarps) {
            const int4 d = seg[s];
            int pools = 0;
            for (int rr = lane; rr < d.z; rr += 32) {
                const int32_t c = ctx[d.y + rr - a.row_begin];
                if (c > 0 && (a.score_all || c > a.topk)) pools = max(pools, min(c / a.kpool, a.pool_cap));
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) pools = max(pools, __shfl_xor_sync(0xffffffffu, pools, o));
            if (lane == 0) {
                const int4 e = make_int4(d.x, d.y, d.z, pools);
                seg[s] = e;
                if (a.smem_segs) a.seg[s] = e;
            }
        }
        __syncthreads();
    }

    // 4. tiles of 128 pools per segment, exclusive prefix.
    uint32_t tcarry = 0;
    for (int base = 0; base < nseg; base += blockDim.x) {
        const int s = base + tid;
        const uint32_t t = s < nseg ? static_cast<uint32_t>((seg[s].w + kTilePools - 1) / kTilePools) : 0u;
        uint32_t total;
        const uint32_t ex = tcarry + block_excl_scan(t, scratch, &total);
        if (s < nseg) {
            prefix[s] = static_cast<int32_t>(ex);
            if (a.smem_segs) a.seg_tile_prefix[s] = static_cast<int32_t>(ex);
        }
        tcarry += total;
        __syncthreads();
    }
    const int ntiles = static_cast<int>(tcarry);
    if (tid == 0) {
        prefix[nseg] = static_cast<int32_t>(tcarry);
        if (a.smem_segs) a.seg_tile_prefix[nseg] = static_cast<int32_t>(tcarry);
        a.hdr[0] = nseg;
        a.hdr[1] = ntiles;
        a.hdr[2] = 0;
    }
}

size_t build_smem_bytes(const BuildArgs& a, BuildArgs* layout) {
    // qsl, then row contexts, then segments and their tile prefix; each only if it fits
    size_t off = 0;
    const size_t budget = 160 * 1024;
    const size_t qsl_b = (static_cast<size_t>(a.num_reqs) + 1) * 4;
    layout->smem_qsl = qsl_b <= 64 * 1024;
    if (layout->smem_qsl) off += (qsl_b + 15) & ~size_t(15);
    const size_t rows_b = static_cast<size_t>(a.chunk_rows < a.row_end - a.row_begin ? a.chunk_rows : a.row_end - a.row_begin) * 4;
    layout->smem_rows = off + rows_b <= budget;
    layout->smem_rows_off = static_cast<int32_t>(off);
    if (layout->smem_rows) off += (rows_b + 15) & ~size_t(15);
    const size_t seg_b = static_cast<size_t>(a.max_segs) * 16;
    const size_t pre_b = (static_cast<size_t>(a.max_segs) + 1) * 4;
    layout->smem_segs = off + seg_b + pre_b <= budget;
    layout->smem_segs_off = static_cast<int32_t>(off);
    layout->smem_prefix_off = static_cast<int32_t>(off + seg_b);
    if (layout->smem_segs) off += seg_b + pre_b;
    return off;
}

cudaError_t launch_build(const BuildArgs& in, bool pdl, cudaStream_t s) {
    BuildArgs a = in;
    const size_t smem = build_smem_bytes(in, &a);
    static int configured[kMaxDevicesTracked] = {};
    static bool carved[kMaxDevicesTracked] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevicesTracked && !carved[dev]) {
        // the SM's largest shared-memory configuration, the one the scorer runs in: with a
        // smaller one the SM holding the builder could take no scorer CTA until it is done
        cudaError_t e = cudaFuncSetAttribute(k_build_segments, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
        if (e != cudaSuccess) return e;
        carved[dev] = true;
    }
    if (dev >= 0 && dev < kMaxDevicesTracked && static_cast<int>(smem) > configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_build_segments, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = static_cast<int>(smem);
    }
    const int chunks = (a.row_end - a.row_begin + a.chunk_rows - 1) / a.chunk_rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(chunks), 1, 1);
    cfg.blockDim = dim3(kBuildThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_build_segments, a);
}

}  // namespace sel
