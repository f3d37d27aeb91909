// K-d: token indices -> physical KV-cache slots (vLLM "sparse_utils" page,
// triton_convert_req_index_to_global_index):
//     slot = block_table[req, t / block_size] * block_stride_rows + t % block_size
// with -1 for t == -1 and for out-of-bounds blocks, columns kept in place, and the
// per-row count of valid slots computed in the same pass. The page's _remap_tiling
// notes that counting is the only reason column tiles would need to cooperate; here
// one warp owns a whole row, so the count is a register reduction plus one store
// (no atomics, no zero-initialised counter), and every access is an int4 (16 B).
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

__global__ void __launch_bounds__(kRemapThreads) k_remap_rows(const RemapArgs a, int rows) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (kRemapThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;  // whole warp
    const int req = a.req_id[row];
    const bool req_ok = req >= 0 && req < a.num_reqs;
    const int32_t* bt_row = a.block_table + static_cast<int64_t>(req_ok ? req : 0) * a.bt_ld;
    const int4* src = reinterpret_cast<const int4*>(a.token_idx + static_cast<int64_t>(row) * a.width);
    int4* dst = reinterpret_cast<int4*>(a.slots + static_cast<int64_t>(row) * a.width);
    const int n4 = a.width >> 2;
    uint32_t cnt = 0;
    for (int v = lane; v < n4; v += 32) {
        const int4 t = __ldg(src + v);
        int4 s = make_int4(-1, -1, -1, -1);
        if (req_ok) {
            s.x = remap_token(t.x, bt_row, a.max_blocks, a.num_kv_blocks, a.block_size, a.block_stride_rows);
            s.y = remap_token(t.y, bt_row, a.max_blocks, a.num_kv_blocks, a.block_size, a.block_stride_rows);
            s.z = remap_token(t.z, bt_row, a.max_blocks, a.num_kv_blocks, a.block_size, a.block_stride_rows);
            s.w = remap_token(t.w, bt_row, a.max_blocks, a.num_kv_blocks, a.block_size, a.block_stride_rows);
        }
        dst[v] = s;
        cnt += (s.x != -1) + (s.y != -1) + (s.z != -1) + (s.w != -1);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0 && a.counts) a.counts[row] = static_cast<int32_t>(cnt);
}

cudaError_t launch_remap(const RemapArgs& a, int rows, cudaStream_t s) {
    const int rows_per_cta = kRemapThreads / 32;
    const int grid = (rows + rows_per_cta - 1) / rows_per_cta;
    k_remap_rows<<<grid, kRemapThreads, 0, s>>>(a, rows);
    return cudaGetLastError();
}

}  // namespace sel
