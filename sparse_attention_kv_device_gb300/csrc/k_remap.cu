// K-d: token indices -> physical KV-cache slots (vLLM "sparse_utils" page,
// triton_convert_req_index_to_global_index):
//     slot = block_table[req, t / block_size] * block_stride_rows + t % block_size
// with -1 for t == -1 and for out-of-bounds blocks, columns kept in place, and the
// per-row count of valid slots computed in the same pass. The page's _remap_tiling
// notes that counting is the only reason column tiles would need to cooperate; here
// one warp owns a whole row, so the count is a register reduction plus one store
// (no atomics, no zero-initialised counter), and every load is an int4 (16 B).
//
// The page's two other modes of the same conversion:
//   prefill workspace (HAS_PREFILL_WORKSPACE): a row of prefill request w maps t to
//       ws_starts[w] + t; decode rows (w == -1) take the global remap;
//   decode context parallelism (triton_filter_and_convert_dcp_index): the tokens this
//       rank owns under a round-robin interleave of `interleave` tokens go through its
//       dense block table, the rest become -1; with compaction the owned slots move to a
//       contiguous prefix of the row. The page's kernel uses an atomic slot allocator and
//       leaves the prefix order unspecified; here the warp places them with a prefix sum
//       over its lanes, in ascending column order, without atomics.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

// q / d and q % d for q >= 0, by shift and mask when d = 2^shift (shift >= 0).
__device__ __forceinline__ int32_t div_by(int32_t q, int32_t d, int32_t shift) { return shift >= 0 ? q >> shift : q / d; }
__device__ __forceinline__ int32_t mod_by(int32_t q, int32_t d, int32_t shift) {
    return shift >= 0 ? q & (d - 1) : q % d;
}

// block_table row entry of token t (>= 0 or -1) -> slot, with the remap's -1 guards.
__device__ __forceinline__ int32_t remap_fast(int32_t t, const RemapArgs& a, const int32_t* bt_row, int64_t stride) {
    if (t < 0) return -1;
    const int32_t b = div_by(t, a.block_size, a.bs_shift);
    if (b >= a.max_blocks) return -1;
    const int32_t ph = __ldg(bt_row + b);
    if (ph < 0 || ph >= a.num_kv_blocks) return -1;
    return static_cast<int32_t>(static_cast<int64_t>(ph) * stride) + mod_by(t, a.block_size, a.bs_shift);
}

// This rank's local index of token t, or -1 (t == -1, or another rank owns t).
__device__ __forceinline__ int32_t dcp_local(int32_t t, const RemapArgs& a) {
    if (t < 0) return -1;
    const int32_t group = div_by(t, a.interleave, a.il_shift);
    if (mod_by(group, a.dcp_size, a.dcp_shift) != a.dcp_rank) return -1;
    return div_by(group, a.dcp_size, a.dcp_shift) * a.interleave + mod_by(t, a.interleave, a.il_shift);
}

template <int MODE>
__device__ __forceinline__ int32_t slot_of(int32_t t, const RemapArgs& a, const int32_t* bt_row, bool req_ok,
                                           int32_t ws_start, int ws_state) {
    if (MODE == kRemapWorkspace && ws_state != 0) {
        // ws_state 1: a prefill row (start + t); 2: a prefill request id out of range
        return ws_state == 1 && t >= 0 ? ws_start + t : -1;
    }
    if (!req_ok) return -1;
    if (MODE == kRemapDcp) return remap_fast(dcp_local(t, a), a, bt_row, a.block_size);
    return remap_fast(t, a, bt_row, a.block_stride_rows);
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kRemapThreads) k_remap_rows(const RemapArgs a, int rows) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (kRemapThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;  // whole warp
    const int req = a.req_id[row];
    const bool req_ok = req >= 0 && req < a.num_reqs;
    const int32_t* bt_row = a.block_table + static_cast<int64_t>(req_ok ? req : 0) * a.bt_ld;
    int32_t ws_start = 0;
    int ws_state = 0;  // 0: global remap, 1: prefill workspace row, 2: bad prefill id
    if (MODE == kRemapWorkspace) {
        const int32_t w = a.ws_req[row];
        if (w != -1) {
            ws_state = (w >= 0 && w < a.num_prefills) ? 1 : 2;
            if (ws_state == 1) ws_start = a.ws_starts[w];
        }
    }
    const int4* src = reinterpret_cast<const int4*>(a.token_idx + static_cast<int64_t>(row) * a.width);
    int32_t* out = a.slots + static_cast<int64_t>(row) * a.width;
    const int n4 = a.width >> 2;
    const bool compact = MODE == kRemapDcp && a.compact;
    constexpr int U = 4;  // token vectors each lane has in flight before it uses any
    uint32_t cnt = 0;
    for (int base = 0; base < n4; base += 32 * U) {  // warp-uniform trip count
        int4 t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = base + u * 32 + lane;
            t[u] = v < n4 ? __ldg(src + v) : make_int4(-1, -1, -1, -1);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = base + u * 32 + lane;
            int4 s;
            s.x = slot_of<MODE>(t[u].x, a, bt_row, req_ok, ws_start, ws_state);
            s.y = slot_of<MODE>(t[u].y, a, bt_row, req_ok, ws_start, ws_state);
            s.z = slot_of<MODE>(t[u].z, a, bt_row, req_ok, ws_start, ws_state);
            s.w = slot_of<MODE>(t[u].w, a, bt_row, req_ok, ws_start, ws_state);
            const uint32_t mine = (s.x != -1) + (s.y != -1) + (s.z != -1) + (s.w != -1);
            if (!compact) {
                if (v < n4) reinterpret_cast<int4*>(out)[v] = s;
                cnt += mine;
            } else {
                // this lane's valid slots go to [cnt + slots of the lanes before it, ...): the
                // row's columns are visited in ascending order, 128 at a time
                uint32_t incl = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                uint32_t pos = cnt + incl - mine;
                if (s.x != -1) out[pos++] = s.x;
                if (s.y != -1) out[pos++] = s.y;
                if (s.z != -1) out[pos++] = s.z;
                if (s.w != -1) out[pos++] = s.w;
                cnt += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
    }
    if (compact) {
        for (int c = static_cast<int>(cnt) + lane; c < a.width; c += 32) out[c] = -1;
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    }
    if (lane == 0 && a.counts) a.counts[row] = static_cast<int32_t>(cnt);
}

cudaError_t launch_remap(const RemapArgs& a, int rows, RemapMode mode, cudaStream_t s) {
    const int rows_per_cta = kRemapThreads / 32;
    const int grid = (rows + rows_per_cta - 1) / rows_per_cta;
    switch (mode) {
        case kRemapWorkspace: k_remap_rows<kRemapWorkspace><<<grid, kRemapThreads, 0, s>>>(a, rows); break;
        case kRemapDcp: k_remap_rows<kRemapDcp><<<grid, kRemapThreads, 0, s>>>(a, rows); break;
        default: k_remap_rows<kRemapGlobal><<<grid, kRemapThreads, 0, s>>>(a, rows); break;
    }
    return cudaGetLastError();
}

}  // namespace sel
