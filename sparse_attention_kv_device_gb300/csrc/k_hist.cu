// K-c0: level-1 histograms for the radix top-k.
//
// For every row that selects pools (ctx > index_topk), counts its complete pools' scores
// by the top 11 bits of their order-preserving 32-bit keys (the scorer stores the keys).
// CTA (x, y) takes kHistSlice consecutive pools of row y, counts them with shared-memory
// atomics, then adds each non-zero bin to the row's global counters (zeroed by the
// segment builder). The row select kernel that follows reads the finished histogram and
// goes straight to the bin that holds the K-th largest score.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

SEL_PHASE_TABLE(hist)

__global__ void __launch_bounds__(kHistThreads) k_row_histogram(const HistArgs a) {
    __shared__ uint32_t h[kTopkBins];
    const int cta = blockIdx.y * gridDim.x + blockIdx.x;
    (void)cta;
    if (threadIdx.x == 0 && cta < 128) SEL_PHASE(cta);                 // diagnostics: CTA start
    pdl_wait();               // scores come from the scorer
    pdl_launch_dependents();  // the top-k may start its prologue
    if (threadIdx.x == 0 && cta < 128) SEL_PHASE(128 + cta);           // diagnostics: dependency met
    const int tid = threadIdx.x;
    const int rl = blockIdx.y;
    const int32_t c = __ldcg(a.row_ctx + rl);
    if (c <= a.topk) return;  // short rows and rows without output select no pools
    const int64_t P = c / a.kpool;
    const int64_t s0 = static_cast<int64_t>(blockIdx.x) * kHistSlice;
    if (s0 >= P) return;
    const int n = static_cast<int>(P - s0 < kHistSlice ? P - s0 : kHistSlice);
    for (int b = tid; b < kTopkBins; b += kHistThreads) h[b] = 0;
    const uint4* src = reinterpret_cast<const uint4*>(a.keys + static_cast<int64_t>(rl) * a.keys_ld + s0);
    constexpr int kVec = kHistSlice / 4 / kHistThreads;
    uint4 v[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const int i4 = tid + j * kHistThreads;
        if (4 * i4 < n) v[j] = __ldcg(src + i4);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        const int i = 4 * (tid + j * kHistThreads);
        if (i < n) {
            atomicAdd(&h[v[j].x >> 21], 1u);
            if (i + 1 < n) atomicAdd(&h[v[j].y >> 21], 1u);
            if (i + 2 < n) atomicAdd(&h[v[j].z >> 21], 1u);
            if (i + 3 < n) atomicAdd(&h[v[j].w >> 21], 1u);
        }
    }
    __syncthreads();
    uint32_t* g = a.hist + static_cast<int64_t>(rl) * kTopkBins;
    for (int b = tid; b < kTopkBins; b += kHistThreads) {
        const uint32_t x = h[b];
        if (x) atomicAdd(g + b, x);
    }
    if (threadIdx.x == 0 && cta < 128) SEL_PHASE(256 + cta);           // diagnostics: CTA end
}

cudaError_t launch_hist(const HistArgs& a, int rows, int64_t max_pools, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    const int64_t gx = (max_pools + kHistSlice - 1) / kHistSlice;
    cfg.gridDim = dim3(static_cast<unsigned>(gx > 0 ? gx : 1), static_cast<unsigned>(rows), 1);
    cfg.blockDim = dim3(kHistThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_row_histogram, a);
}

}  // namespace sel
