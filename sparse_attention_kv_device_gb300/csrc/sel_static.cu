// sel_select_static: the fused selection with its workspace in a file-scope device array.
//
// Some callers cannot allocate device memory for a call:
//   - a serving engine that reserves nearly all free HBM for its paged KV cache when it
//     starts, so no room is left, and no allocator may be called, between decode steps;
//   - a plain C host program that links this library and has no device allocator of its
//     own to hand out a workspace.
// This entry point takes no workspace argument: the scratch sel_select needs lives in
// `g_static_ws` below, a fixed SEL_STATIC_WS_MAX_BYTES array that every GPU which loads
// this module holds until the process exits. Nothing here calls cudaMalloc, cudaFree or
// any other allocating routine.
//
// Set-up: a call looks up the array's device address on the current device with
// cudaGetSymbolAddress (host code never uses the array's name as a device address). Outside
// stream capture the look-up is repeated on every call, so that a module reloaded after a
// device reset is found at its new address; inside a capture the address found by the last
// call on that device outside capture is used, so make one call on each device before
// capturing.
//
// Zeroing: the launch sequence clears every counter it relies on before use (the segment
// builder resets the tile header and counter of each chunk; the row kernel clears its own
// shared-memory histograms), so the array needs no clearing between calls.
//
// Sharing: all calls on one device share the one array. Two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on it and give wrong results;
// order them on one stream, or through events.
#include <mutex>

#include "sel.h"
#include "sel_kernels.h"

namespace {

constexpr size_t kStaticWsBytes = static_cast<size_t>(SEL_STATIC_WS_MAX_BYTES);

static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_static_mu;
void* g_static_ptr[sel::kMaxDevicesTracked] = {};

// Device address of g_static_ws on the current device.
int static_workspace(cudaStream_t stream, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return SEL_ECUDA;
    if (dev < 0 || dev >= sel::kMaxDevicesTracked) return SEL_EUNSUPPORTED;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return SEL_ECUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (cs == cudaStreamCaptureStatusNone || !g_static_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || !ptr) return SEL_ECUDA;
        g_static_ptr[dev] = ptr;
    }
    *out = g_static_ptr[dev];
    return SEL_OK;
}

}  // namespace

extern "C" int sel_select_static(const sel_problem* p, int32_t* slots, int32_t out_width, int32_t* valid_counts,
                                 int32_t* token_idx, int32_t* status, sel_stream_t stream) {
    if (!p) return SEL_EINVAL;
    void* ws = nullptr;
    int rc = static_workspace(reinterpret_cast<cudaStream_t>(stream), &ws);
    if (rc != SEL_OK) return rc;
    // sel_workspace_bytes is 0 for a problem sel_select rejects; sel_select then reports why
    if (sel_workspace_bytes(p) > kStaticWsBytes) return SEL_EWORKSPACE;
    return sel_select(p, slots, out_width, valid_counts, token_idx, status, ws, kStaticWsBytes, stream);
}
