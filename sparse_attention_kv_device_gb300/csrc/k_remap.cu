// K-d: token indices -> physical KV-cache slots (vLLM "sparse_utils" page,
// triton_convert_req_index_to_global_index):
//     slot = block_table[req, t / block_size] * block_stride_rows + t % block_size
// with -1 for t == -1 and for out-of-bounds blocks, columns kept in place, and the
// per-row count of valid slots computed in the same pass. The page's _remap_tiling
// notes that counting is the only reason column tiles would need to cooperate; here
// one CTA owns a whole row, so the count is a block reduction plus one store (no atomics,
// no zero-initialised counter); every load is an int4 (16 B), and a thread loads all its
// vectors of the row before it uses any.
//
// The page's two other modes of the same conversion:
//   prefill workspace (HAS_PREFILL_WORKSPACE): a row of prefill request w maps t to
//       ws_starts[w] + t; decode rows (w == -1) take the global remap;
//   decode context parallelism (triton_filter_and_convert_dcp_index): the tokens this
//       rank owns under a round-robin interleave of `interleave` tokens go through its
//       dense block table, the rest become -1; with compaction the owned slots move to a
//       contiguous prefix of the row. The page's kernel uses an atomic slot allocator and
//       leaves the prefix order unspecified; here the CTA places them with block prefix
//       sums, in ascending column order, without atomics.
#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

// q / d and q % d for q >= 0, by shift and mask when d = 2^shift (shift >= 0). P2: every
// divisor of the launch is a power of two, so only the shift form is compiled (the division
// sequences, unrolled over a thread's twenty tokens, otherwise overflow the instruction cache).
template <bool P2>
__device__ __forceinline__ int32_t div_by(int32_t q, int32_t d, int32_t shift) {
    if constexpr (P2) return q >> shift;
    else return shift >= 0 ? q >> shift : q / d;
}
template <bool P2>
__device__ __forceinline__ int32_t mod_by(int32_t q, int32_t d, int32_t shift) {
    if constexpr (P2) return q & (d - 1);
    else return shift >= 0 ? q & (d - 1) : q % d;
}

// block_table row entry of token t (>= 0 or -1) -> slot, with the remap's -1 guards.
template <bool P2>
__device__ __forceinline__ int32_t remap_fast(int32_t t, const RemapArgs& a, const int32_t* bt_row, int64_t stride) {
    if (t < 0) return -1;
    const int32_t b = div_by<P2>(t, a.block_size, a.bs_shift);
    if (b >= a.max_blocks) return -1;
    const int32_t ph = __ldg(bt_row + b);
    if (ph < 0 || ph >= a.num_kv_blocks) return -1;
    return static_cast<int32_t>(static_cast<int64_t>(ph) * stride) + mod_by<P2>(t, a.block_size, a.bs_shift);
}

// This rank's local index of token t, or -1 (t == -1, or another rank owns t).
template <bool P2>
__device__ __forceinline__ int32_t dcp_local(int32_t t, const RemapArgs& a) {
    if (t < 0) return -1;
    const int32_t group = div_by<P2>(t, a.interleave, a.il_shift);
    if (mod_by<P2>(group, a.dcp_size, a.dcp_shift) != a.dcp_rank) return -1;
    return div_by<P2>(group, a.dcp_size, a.dcp_shift) * a.interleave + mod_by<P2>(t, a.interleave, a.il_shift);
}

template <int MODE, bool P2>
__device__ __forceinline__ int32_t slot_of(int32_t t, const RemapArgs& a, const int32_t* bt_row, bool req_ok,
                                           int32_t ws_start, int ws_state) {
    if (MODE == kRemapWorkspace && ws_state != 0) {
        // ws_state 1: a prefill row (start + t); 2: a prefill request id out of range
        return ws_state == 1 && t >= 0 ? ws_start + t : -1;
    }
    if (!req_ok) return -1;
    if (MODE == kRemapDcp) return remap_fast<P2>(dcp_local<P2>(t, a), a, bt_row, a.block_size);
    return remap_fast<P2>(t, a, bt_row, a.block_stride_rows);
}

// The slots of one int4 of tokens. Four consecutive tokens in one block (what the selection
// writes: a pool of 4 consecutive tokens starts at a multiple of 4) take one block-table load
// for the four, with consecutive slots; anything else goes token by token. The results are
// those of slot_of for each token.
template <int MODE, bool P2>
__device__ __forceinline__ int4 slots4(int4 t, const RemapArgs& a, const int32_t* bt_row, bool req_ok,
                                      int32_t ws_start, int ws_state) {
    // (the DCP mode keeps the token-by-token path: its local indices are consecutive only with
    // an interleave of 4 or more, and the extra code costs its latency-bound loop registers)
    if (MODE != kRemapDcp && ws_state == 0 && req_ok) {
        const uint32_t x = static_cast<uint32_t>(t.x);
        if (t.x >= 0 && x <= 0x7ffffffcu && static_cast<uint32_t>(t.y) == x + 1u &&
            static_cast<uint32_t>(t.z) == x + 2u && static_cast<uint32_t>(t.w) == x + 3u) {
            const int32_t b = div_by<P2>(t.x, a.block_size, a.bs_shift);
            if (div_by<P2>(t.w, a.block_size, a.bs_shift) == b) {
                if (b >= a.max_blocks) return make_int4(-1, -1, -1, -1);
                const int32_t ph = __ldg(bt_row + b);
                if (ph < 0 || ph >= a.num_kv_blocks) return make_int4(-1, -1, -1, -1);
                const int32_t s0 = static_cast<int32_t>(static_cast<int64_t>(ph) * a.block_stride_rows) +
                                   mod_by<P2>(t.x, a.block_size, a.bs_shift);
                return make_int4(s0, s0 + 1, s0 + 2, s0 + 3);
            }
        }
    }
    if constexpr (MODE == kRemapDcp && P2) {
        // an interleave of 4 or more (a power of two): four consecutive tokens from a multiple of
        // 4 share one interleave group, so one rank owns all four (or none) at consecutive local
        // indices; in one block they take one table load
        const uint32_t x = static_cast<uint32_t>(t.x);
        if (a.il_shift >= 2 && req_ok && t.x >= 0 && (x & 3u) == 0u && x <= 0x7ffffffcu &&
            static_cast<uint32_t>(t.y) == x + 1u && static_cast<uint32_t>(t.z) == x + 2u &&
            static_cast<uint32_t>(t.w) == x + 3u) {
            const int32_t e0 = dcp_local<P2>(t.x, a);
            if (e0 < 0) return make_int4(-1, -1, -1, -1);
            const int32_t b = e0 >> a.bs_shift;
            if (((e0 + 3) >> a.bs_shift) == b) {
                if (b >= a.max_blocks) return make_int4(-1, -1, -1, -1);
                const int32_t ph = __ldg(bt_row + b);
                if (ph < 0 || ph >= a.num_kv_blocks) return make_int4(-1, -1, -1, -1);
                const int32_t s0 = ph * a.block_size + (e0 & (a.block_size - 1));
                return make_int4(s0, s0 + 1, s0 + 2, s0 + 3);
            }
        }
    }
    if (MODE != kRemapDcp)  // token by token (the fewest registers: occupancy wins here)
        return make_int4(slot_of<MODE, P2>(t.x, a, bt_row, req_ok, ws_start, ws_state),
                         slot_of<MODE, P2>(t.y, a, bt_row, req_ok, ws_start, ws_state),
                         slot_of<MODE, P2>(t.z, a, bt_row, req_ok, ws_start, ws_state),
                         slot_of<MODE, P2>(t.w, a, bt_row, req_ok, ws_start, ws_state));
    // DCP, token by token: the guards first, then the four table loads together (a load only
    // where its guard passes), so their latencies overlap instead of adding up (the local-index
    // arithmetic otherwise keeps them apart)
    const int32_t tt[4] = {t.x, t.y, t.z, t.w};
    int32_t e[4], b[4], ph[4], r[4];
    bool ok[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        e[i] = MODE == kRemapDcp ? dcp_local<P2>(tt[i], a) : tt[i];
        ok[i] = req_ok && e[i] >= 0;
        b[i] = ok[i] ? div_by<P2>(e[i], a.block_size, a.bs_shift) : 0;
        ok[i] = ok[i] && b[i] < a.max_blocks;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) ph[i] = ok[i] ? __ldg(bt_row + b[i]) : -1;
    const int64_t stride = MODE == kRemapDcp ? a.block_size : a.block_stride_rows;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        r[i] = ok[i] && ph[i] >= 0 && ph[i] < a.num_kv_blocks
                   ? static_cast<int32_t>(static_cast<int64_t>(ph[i]) * stride) + mod_by<P2>(e[i], a.block_size, a.bs_shift)
                   : -1;
    return make_int4(r[0], r[1], r[2], r[3]);
}

}  // namespace

constexpr int kCompactStage = 4096;  // columns of a compacted row assembled in shared memory

template <int MODE, bool P2>
__global__ void __launch_bounds__(kRemapThreads, MODE == kRemapDcp ? 10 : 16) k_remap_rows(const RemapArgs a, int rows) {
    __shared__ uint32_t scratch[64];
    __shared__ __align__(16) int32_t stage[MODE == kRemapDcp ? kCompactStage : 4];
    const int tid = threadIdx.x;
    const int row = blockIdx.x;
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
    // a compacted row is assembled in shared memory and written out with 16-byte stores
    const bool staged = compact && a.width <= kCompactStage;
    int32_t* cdst = staged ? stage : out;
    // every thread has all its vectors of a round in flight before it uses any: one round
    // covers a row of up to kRemapThreads * U vectors (2,560 tokens)
    constexpr int U = 5;
    uint32_t cnt = 0;  // non-compact: this thread's valid slots; compact: the row's so far
    for (int base = 0; base < n4; base += kRemapThreads * U) {  // block-uniform trip count
        // vector of (round position u, thread): strided across the threads, so each load
        // instruction of a warp reads 512 contiguous bytes
        auto vec = [&](int u) { return base + u * kRemapThreads + tid; };
        int4 t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = vec(u);
            t[u] = v < n4 ? __ldg(src + v) : make_int4(-1, -1, -1, -1);
        }
        if (compact) {
            // kept slots in column order: position u comes before u + 1, and within it the
            // threads in order. Each warp scans its lanes' counts per position with shuffles and
            // publishes the warp totals (one buffer per round parity); after one barrier every
            // thread adds up the totals ahead of it.
            constexpr int kW = kRemapThreads / 32;
            uint32_t* wt = scratch + ((base / (kRemapThreads * U)) & 1) * (U * kW);
            const int lane = tid & 31, warp = tid >> 5;
            int4 sl[U];
            uint32_t excl[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                sl[u] = slots4<MODE, P2>(t[u], a, bt_row, req_ok, ws_start, ws_state);
                const uint32_t m = (sl[u].x != -1) + (sl[u].y != -1) + (sl[u].z != -1) + (sl[u].w != -1);
                const uint32_t incl = warp_incl_scan(m);
                excl[u] = incl - m;
                if (lane == 31) wt[u * kW + warp] = incl;
            }
            __syncthreads();
            uint32_t pre = cnt;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                uint32_t before = 0, all = 0;
#pragma unroll
                for (int w = 0; w < kW; ++w) {
                    const uint32_t x = wt[u * kW + w];
                    before += w < warp ? x : 0u;
                    all += x;
                }
                uint32_t pos = pre + before + excl[u];
                if (sl[u].x != -1) cdst[pos++] = sl[u].x;
                if (sl[u].y != -1) cdst[pos++] = sl[u].y;
                if (sl[u].z != -1) cdst[pos++] = sl[u].z;
                if (sl[u].w != -1) cdst[pos++] = sl[u].w;
                pre += all;
            }
            cnt = pre;
            continue;
        }
        if constexpr (MODE == kRemapDcp) {
            // every vector's slots first (their table loads all in flight), then the stores
            int4 sl[U];
#pragma unroll
            for (int u = 0; u < U; ++u) sl[u] = slots4<MODE, P2>(t[u], a, bt_row, req_ok, ws_start, ws_state);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = vec(u);
                if (v < n4) reinterpret_cast<int4*>(out)[v] = sl[u];
                cnt += (sl[u].x != -1) + (sl[u].y != -1) + (sl[u].z != -1) + (sl[u].w != -1);
            }
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = vec(u);
                const int4 sl = slots4<MODE, P2>(t[u], a, bt_row, req_ok, ws_start, ws_state);
                if (v < n4) reinterpret_cast<int4*>(out)[v] = sl;
                cnt += (sl.x != -1) + (sl.y != -1) + (sl.z != -1) + (sl.w != -1);
            }
        }
    }
    if (compact) {
        for (int c = static_cast<int>(cnt) + tid; c < a.width; c += kRemapThreads) cdst[c] = -1;
        if (staged) {
            __syncthreads();
            for (int v = tid; v < n4; v += kRemapThreads)
                reinterpret_cast<int4*>(out)[v] = reinterpret_cast<const int4*>(stage)[v];
        }
    } else {
        cnt = block_sum(cnt, scratch);
    }
    if (tid == 0 && a.counts) a.counts[row] = static_cast<int32_t>(cnt);
}

cudaError_t launch_remap(const RemapArgs& a, int rows, RemapMode mode, cudaStream_t s) {
    const int grid = rows;  // one CTA per row
    const bool p2 = a.bs_shift >= 0 && (mode != kRemapDcp || (a.il_shift >= 0 && a.dcp_shift >= 0));
    switch (mode) {
        case kRemapWorkspace:
            if (p2) k_remap_rows<kRemapWorkspace, true><<<grid, kRemapThreads, 0, s>>>(a, rows);
            else k_remap_rows<kRemapWorkspace, false><<<grid, kRemapThreads, 0, s>>>(a, rows);
            break;
        case kRemapDcp:
            if (p2) k_remap_rows<kRemapDcp, true><<<grid, kRemapThreads, 0, s>>>(a, rows);
            else k_remap_rows<kRemapDcp, false><<<grid, kRemapThreads, 0, s>>>(a, rows);
            break;
        default:
            if (p2) k_remap_rows<kRemapGlobal, true><<<grid, kRemapThreads, 0, s>>>(a, rows);
            else k_remap_rows<kRemapGlobal, false><<<grid, kRemapThreads, 0, s>>>(a, rows);
            break;
    }
    return cudaGetLastError();
}

}  // namespace sel
