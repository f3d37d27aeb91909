// Host <-> device staging for the host-buffer entry point. When every host buffer of a call is
// pinned and mapped into the device's address space, one kernel pulls all of a step's inputs
// into the device staging area, and one pushes the results back, over the host link, instead of
// one copy-engine transfer per buffer (each of which carries a few microseconds of fixed cost).
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

// one word per thread and step; 16-byte words where both ends and the length allow it
__global__ void __launch_bounds__(256) k_stage_copy(const StageArgs a) {
    pdl_launch_dependents();  // the builder may take its place; it waits for this grid's end
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (int s = 0; s < a.nseg; ++s) {
        const uint8_t* src = static_cast<const uint8_t*>(a.src[s]);
        uint8_t* dst = static_cast<uint8_t*>(a.dst[s]);
        const int64_t n = a.bytes[s];
        const bool wide = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | n) & 15) == 0;
        if (wide) {
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
            uint4* d4 = reinterpret_cast<uint4*>(dst);
            for (int64_t i = tid; i < n / 16; i += stride) d4[i] = s4[i];
        } else {  // the entry point's buffers are int32 arrays (4-byte aligned, lengths of 4)
            const uint32_t* s1 = reinterpret_cast<const uint32_t*>(src);
            uint32_t* d1 = reinterpret_cast<uint32_t*>(dst);
            for (int64_t i = tid; i < n / 4; i += stride) d1[i] = s1[i];
        }
    }
}

}  // namespace

cudaError_t launch_stage_copy(const StageArgs& a, int sms, cudaStream_t s) {
    int64_t words = 0;
    for (int i = 0; i < a.nseg; ++i) words += a.bytes[i] / 4;
    const int64_t want = (words + 255) / 256;
    const int grid = static_cast<int>(want < 1 ? 1 : (want > 2 * sms ? 2 * sms : want));
    k_stage_copy<<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace sel
