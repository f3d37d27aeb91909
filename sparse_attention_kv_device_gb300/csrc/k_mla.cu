// K-e: sparse MLA decode attention over the selected slots (vLLM page
// "flashinfer_mla_sparse_sm90", _SM90State: FlashInfer's MLA wrapper planned with page size 1,
// so the selection's slots are the page table, and the exact kv_len of _kv_lens_host).
//
// For row r and head h, over the entries j < kv_len[r] whose slot s = slots[r][j] lies in
// [0, num_slots) (a -1 or out-of-range slot inside kv_len contributes nothing, and nothing
// past kv_len is read):
//   logit_j = sm_scale * (q_nope[r][h] . ckv[s] + q_pe[r][h] . kpe[s])
//   out[r][h] = sum_j softmax(logit)_j * ckv[s_j],   lse[r][h] = log sum_j exp(logit_j)
// with 16 heads, 512 latent and 0 or 64 rotary dims, bf16 inputs, fp32 outputs.
//
// The rows' tiles of 64 entries are laid end to end and cut into one contiguous run per CTA,
// so the job spreads evenly over the SMs even for a handful of rows. Per tile:
//   warps 0-3 (eight lanes per 128-byte box row, four entries per warp-wide copy) read the
//     entries' slots and gather their 576 dims from the cache with 16-byte cp.async into
//     64-dim boxes in the 128-byte swizzle layout: the latent boxes in pairs (a ring of 11
//     pairs, 2.75 tiles) that stay until the tile's output product, the rotary box in a ring
//     of 2; meanwhile the next tile's rows are prefetched into L2 by the TMA engine. An
//     entry past kv_len or with a bad slot is zero-filled without touching the cache;
//   warp 4 (one thread) issues, for tile k, S^T = K . Q^T on the tensor cores into TMEM
//     (kind::f16, bf16 operands, fp32 accumulation in four interleaved partial sums; M = 64,
//     the tile's entries, whose results sit in lanes 0-15 of each TMEM lane quarter), then
//     tile k-1's O^T[512 x 16] += V^T . P^T, the same latent boxes read as an MN-major
//     operand (a latent row is both key and value);
//   warps 5-8 (one entry per lane 0-15 of each warp) read the tile's logits from TMEM, keep
//     the running maximum per head -- raised only when a logit exceeds it by more than 2^8,
//     which then rescales O in TMEM --, and write p = 2^(logit - max) rounded to bf16 for
//     the output product; the sums of p are kept per thread and reduced once per row.
// A row whose tiles all ran in one CTA is normalised and written by that CTA; a row split
// between CTAs leaves one partial (unnormalised O, maximum, sums) per CTA, and k_mla_merge
// combines them.
#include <cuda_bf16.h>

#include "sel_device.cuh"
#include "sel_kernels.h"

namespace sel {

namespace {

constexpr int kPairSlots = 11;                 // latent pair buffers (boxes 2k, 2k+1 of one tile)
constexpr int kRopeSlots = 2;
constexpr uint32_t kBoxBytes16 = 64 * 128;     // 64 dims x 64 entries, bf16
constexpr uint32_t kPairBytes = 2 * kBoxBytes16;
constexpr uint32_t kQBox = 16 * 128;           // 16 heads x 64 dims
constexpr uint32_t kPBuf = 16 * 128;           // 16 heads x 64 entries
constexpr uint32_t kOffRope = kPairSlots * kPairBytes;
constexpr uint32_t kOffQ = kOffRope + kRopeSlots * kBoxBytes16;
constexpr uint32_t kOffP = kOffQ + 9 * kQBox;
constexpr uint32_t kOffBar = kOffP + 2 * kPBuf;
// barriers
constexpr int kBPairFull = 0, kBPairEmpty = kBPairFull + kPairSlots, kBRopeFull = kBPairEmpty + kPairSlots,
              kBRopeEmpty = kBRopeFull + kRopeSlots, kBQFull = kBRopeEmpty + kRopeSlots, kBQEmpty = kBQFull + 1,
              kBSFull = kBQEmpty + 1, kBSEmpty = kBSFull + 2, kBPFull = kBSEmpty + 2, kBPEmpty = kBPFull + 2,
              kBOFull = kBPEmpty + 2, kBOEmpty = kBOFull + 2, kBODone = kBOEmpty + 2, kBDone = kBODone + 2,
              kNumBars = kBDone + 1;
constexpr uint32_t kOffWords = kOffBar + kNumBars * 8;       // tmem base, abort flag
constexpr uint32_t kOffRed = kOffWords + 16;                  // 2 x 4 warps x 16 floats
constexpr uint32_t kSmemUsed = kOffRed + 2 * 4 * 16 * 4;
// TMEM columns: S = 2 buffers x 4 partial accumulators x 16 heads (the score product's K
// steps alternate between four accumulators so consecutive MMAs do not depend on each other;
// the softmax adds the four), then O = 2 buffers x 4 dim-blocks x 16 heads.
constexpr uint32_t kColS = 0, kColO = 128, kTmemCols = 256;
constexpr float kRaise = 8.0f;                                // log2 of the largest p kept unscaled
constexpr int kSoftBar = 1;                                   // named barrier of the softmax warps

struct Seg {
    int row, tin_a, tin_b;  // tiles tin_a..tin_b of the row
    int n_act;              // tiles holding an entry below kv_len (a prefix of the segment)
    int kvl;                // the row's kv_len, clamped to [0, width]
};

__device__ __forceinline__ Seg segment_of(const MlaArgs& a, int64_t t0, int64_t t1, int row) {
    Seg s;
    s.row = row;
    const int64_t r0 = static_cast<int64_t>(row) * a.tiles_per_row;
    const int64_t lo = t0 > r0 ? t0 : r0, hi = t1 < r0 + a.tiles_per_row ? t1 : r0 + a.tiles_per_row;
    s.tin_a = static_cast<int>(lo - r0);
    s.tin_b = static_cast<int>(hi - 1 - r0);
    int kvl = __ldg(a.kv_len + row);
    kvl = max(0, min(kvl, a.width));
    s.kvl = kvl;
    const int tiles = (kvl + kMlaTile - 1) / kMlaTile;
    s.n_act = max(0, min(s.tin_b + 1, tiles) - s.tin_a);
    return s;
}

// Walks the CTA's tiles that hold an entry below kv_len, row by row (rows without any are
// skipped): the gather and MMA roles step through the same sequence.
struct ActIter {
    int row, row_b, tt;
    Seg sg;
    bool valid;
    __device__ __forceinline__ void skip(const MlaArgs& a, int64_t t0, int64_t t1) {
        while (row <= row_b && sg.n_act == 0) {
            ++row;
            if (row <= row_b) sg = segment_of(a, t0, t1, row);
        }
        valid = row <= row_b;
    }
    __device__ __forceinline__ void start(const MlaArgs& a, int64_t t0, int64_t t1, int ra, int rb) {
        row = ra;
        row_b = rb;
        tt = 0;
        sg = segment_of(a, t0, t1, row);
        skip(a, t0, t1);
    }
    __device__ __forceinline__ void next(const MlaArgs& a, int64_t t0, int64_t t1) {
        if (++tt == sg.n_act) {
            tt = 0;
            ++row;
            if (row <= row_b) sg = segment_of(a, t0, t1, row);
            skip(a, t0, t1);
        }
    }
    __device__ __forceinline__ int entry0() const { return (sg.tin_a + tt) * kMlaTile; }
};

// The slot of entry e of a row with (clamped) kv_len kvl, or -1 (past kv_len, or a bad slot).
// One load, predicated on e < kvl: its result is only needed by the caller's next step.
__device__ __forceinline__ int raw_slot(const MlaArgs& a, int row, int kvl, int e) {
    return e < kvl ? __ldg(a.slots + static_cast<int64_t>(row) * a.width + e) : -1;
}
__device__ __forceinline__ int checked_slot(const MlaArgs& a, int s) {
    return (s >= 0 && s < a.num_slots) ? s : -1;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Max (op 0) or sum (op 1) per head over the 128 softmax threads; `red` alternates between
// two halves so back-to-back reductions need one barrier each.
template <int op>
__device__ __forceinline__ void soft_reduce(float (&v)[16], float* red, int& half, int sw, int lane) {
    float* r = red + half * 64;
    half ^= 1;
#pragma unroll
    for (int h = 0; h < 16; ++h) {
        const float x = op == 0 ? warp_max(v[h]) : warp_sum(v[h]);
        if (lane == 0) r[sw * 16 + h] = x;
    }
    named_bar_sync(kSoftBar, 128);
#pragma unroll
    for (int h = 0; h < 16; ++h) {
        const float a0 = r[h], a1 = r[16 + h], a2 = r[32 + h], a3 = r[48 + h];
        v[h] = op == 0 ? fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) : (a0 + a1) + (a2 + a3);
    }
}

}  // namespace

__global__ void __launch_bounds__(kMlaThreads, 1) k_mla_decode(const MlaArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffBar);
    uint32_t* words = reinterpret_cast<uint32_t*>(sm + kOffWords);
    float* red = reinterpret_cast<float*>(sm + kOffRed);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * a.total_tiles / G;
    const int64_t t1 = static_cast<int64_t>(blockIdx.x + 1) * a.total_tiles / G;
    const int row_a = static_cast<int>(t0 / a.tiles_per_row);
    const int row_b = static_cast<int>((t1 - 1) / a.tiles_per_row);
    const int nbox_r = a.dr > 0 ? 1 : 0;  // rotary boxes per tile

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPairSlots; ++i) {
            mbar_init(&bar[kBPairFull + i], 128);
            mbar_init(&bar[kBPairEmpty + i], 1);
        }
        for (int i = 0; i < kRopeSlots; ++i) {
            mbar_init(&bar[kBRopeFull + i], 128);
            mbar_init(&bar[kBRopeEmpty + i], 1);
        }
        mbar_init(&bar[kBQFull], 128);
        mbar_init(&bar[kBQEmpty], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar[kBSFull + i], 1);
            mbar_init(&bar[kBSEmpty + i], 4);
            mbar_init(&bar[kBPFull + i], 4);
            mbar_init(&bar[kBPEmpty + i], 1);
            mbar_init(&bar[kBOEmpty + i], 4);
            mbar_init(&bar[kBOFull + i], 1);
        }
        mbar_init(&bar[kBODone], 1);
        mbar_init(&bar[kBODone + 1], 1);
        mbar_init(&bar[kBDone], 1);
        words[1] = 0;  // abort flag
        mbar_fence_init();
    }
    if (warp == 4) {
        tmem_alloc(&words[0], kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();  // the merge grid may take its places now (it waits for this grid's end)
    const uint32_t tmem = words[0];
    volatile int* abort_flag = reinterpret_cast<volatile int*>(&words[1]);
    auto fail = [&]() {
        *abort_flag = 1;
        report(a.status, kStTimeout);
    };

    if (warp < 4) {
        // ------------------------------------------------------------ gather
        // Thread i copies 16-byte chunk (i & 7) of the 128-byte box rows of entries
        // (i >> 3) + 16 r, r < 4: eight consecutive lanes cover one entry's whole box row, so
        // each warp-wide copy reads four full 128-byte lines. Per tile k: its four latent
        // pairs and its rotary box go to shared memory; then tile k+1's rows are brought
        // into L2 by bulk prefetches (TMA engine), and tile k+2's slot indices are loaded.
        const int i = threadIdx.x;
        const int c = i & 7, eg = i >> 3;
        auto load_raw = [&](const ActIter& t, int (&raw)[4]) {
#pragma unroll
            for (int r = 0; r < 4; ++r) raw[r] = t.valid ? raw_slot(a, t.row, t.sg.kvl, t.entry0() + eg + 16 * r) : -1;
        };
        auto prefetch_rows = [&](const int (&raw)[4]) {
            if (c != 0) return;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int sl = checked_slot(a, raw[r]);
                if (sl >= 0) {
                    bulk_prefetch_l2(a.ckv + static_cast<int64_t>(sl) * a.ckv_stride, kMlaDc * 2);
                    if (nbox_r) bulk_prefetch_l2(a.kpe + static_cast<int64_t>(sl) * a.kpe_stride, 128);
                }
            }
        };
        ActIter it;
        it.start(a, t0, t1, row_a, row_b);
        ActIter it1 = it;
        if (it1.valid) it1.next(a, t0, t1);
        int cur_raw[4], nxt_raw[4], far_raw[4];
        load_raw(it, cur_raw);
        load_raw(it1, nxt_raw);
        int64_t seq = 0, k = 0;
        int q_loads = 0;
        bool ok = true;
        while (ok && it.valid) {
            ActIter it2 = it1;
            if (it2.valid) it2.next(a, t0, t1);
            load_raw(it2, far_raw);
            if (it.tt == 0) {
                // the row's queries: 16 heads x 9 boxes of 64 dims, K-major swizzle layout
                if (!mbar_wait(&bar[kBQEmpty], (q_loads & 1) ^ 1u, abort_flag, a.wait_ns)) { ok = false; break; }
                const int h = i >> 3;
                const uint16_t* qn = a.q_nope + static_cast<int64_t>(it.row) * a.qn_row + h * a.qn_head;
                uint8_t* qd = sm + kOffQ + h * 128 + ((c ^ (h & 7)) << 4);
#pragma unroll
                for (int b = 0; b < 8; ++b) cp_async_16(qd + b * kQBox, qn + 64 * b + 8 * c);
                if (a.dr > 0)
                    cp_async_16(qd + 8 * kQBox,
                                a.q_pe + static_cast<int64_t>(it.row) * a.qp_row + h * a.qp_head + 8 * c);
                cp_async_mbar_arrive(&bar[kBQFull]);
                ++q_loads;
            }
            const uint16_t* src[4];
            uint32_t nb[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int sl = checked_slot(a, cur_raw[r]);
                src[r] = a.ckv + (sl >= 0 ? static_cast<int64_t>(sl) * a.ckv_stride : 0) + 8 * c;
                nb[r] = sl >= 0 ? 16u : 0u;
            }
            for (int pr = 0; pr < 4; ++pr, ++seq) {
                const int ps = static_cast<int>(seq % kPairSlots);
                if (!mbar_wait(&bar[kBPairEmpty + ps], static_cast<uint32_t>((seq / kPairSlots) & 1) ^ 1u, abort_flag,
                               a.wait_ns)) { ok = false; break; }
                uint8_t* dst = sm + ps * kPairBytes;
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int e = eg + 16 * r;
                        cp_async_16_zfill(dst + half * kBoxBytes16 + e * 128 + ((c ^ (e & 7)) << 4),
                                          src[r] + (2 * pr + half) * 64, nb[r]);
                    }
                cp_async_mbar_arrive(&bar[kBPairFull + ps]);
            }
            if (!ok) break;
            if (nbox_r) {
                const int rs = static_cast<int>(k % kRopeSlots);
                if (!mbar_wait(&bar[kBRopeEmpty + rs], static_cast<uint32_t>((k / kRopeSlots) & 1) ^ 1u, abort_flag,
                               a.wait_ns)) { ok = false; break; }
                uint8_t* dst = sm + kOffRope + rs * kBoxBytes16;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int e = eg + 16 * r;
                    const int sl = checked_slot(a, cur_raw[r]);
                    const uint16_t* srp = a.kpe + (sl >= 0 ? static_cast<int64_t>(sl) * a.kpe_stride : 0) + 8 * c;
                    cp_async_16_zfill(dst + e * 128 + ((c ^ (e & 7)) << 4), srp, nb[r]);
                }
                cp_async_mbar_arrive(&bar[kBRopeFull + rs]);
            }
            prefetch_rows(nxt_raw);
            it = it1;
            it1 = it2;
            ++k;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                cur_raw[r] = nxt_raw[r];
                nxt_raw[r] = far_raw[r];
            }
        }
        if (!ok) fail();
        cp_async_wait_all();  // nothing lands in shared memory after the CTA leaves
    } else if (warp == 4) {
        // ------------------------------------------------------------ MMA issuer
        // Step k: tile k's scores S^T = K . Q^T (latent pairs, then the rotary box),
        // committed; then tile k-1's output O^T += V^T . P^T once the softmax has written
        // P(k-1), which frees tile k-1's pairs. The commit of S(k) covers every product of
        // tile k-2; O_DONE[t & 1] marks tile t's output products.
        if (lane == 0) {
            // the score product: M = 64 entries (a tile), so only the tile's own rows are read;
            // its result rows land in TMEM lanes 0-15 of each 32-lane quarter
            const uint32_t idesc_s = umma_idesc_bf16_f32(kMlaTile, kMlaHeads, 0);
            const uint32_t idesc_o = umma_idesc_bf16_f32(128, kMlaHeads, 1);
            const uint32_t base = smem_u32(sm);
            ActIter it;
            it.start(a, t0, t1, row_a, row_b);
            bool have_prev = false, prev_first = false, prev_last = false;
            int prev_ob = 0, prev_seg = 0, o_segs = 0, q_loads = 0;
            int64_t k = 0;
            bool ok = true;
            while (ok && (it.valid || have_prev)) {
                const bool have_cur = it.valid;
                const bool cur_first = have_cur && it.tt == 0;
                const bool cur_last = have_cur && it.tt == it.sg.n_act - 1;
                const int sb = static_cast<int>(k & 1);
                const int pb = static_cast<int>((k - 1) & 1);
                if (have_cur) {
                    if (cur_first) {
                        if (!mbar_wait(&bar[kBQFull], q_loads & 1, abort_flag, a.wait_ns)) { ok = false; break; }
                        ++q_loads;
                    }
                    if (!mbar_wait(&bar[kBSEmpty + sb], static_cast<uint32_t>((k >> 1) & 1) ^ 1u, abort_flag,
                                   a.wait_ns)) { ok = false; break; }
                    const uint32_t d_s = tmem + kColS + 64u * sb;  // + 16 * accumulator
                    for (int pr = 0; pr < 4; ++pr) {
                        const int64_t seq = 4 * k + pr;
                        const int ps = static_cast<int>(seq % kPairSlots);
                        if (!mbar_wait(&bar[kBPairFull + ps], static_cast<uint32_t>((seq / kPairSlots) & 1), abort_flag,
                                       a.wait_ns)) { ok = false; break; }
                        fence_proxy_async_smem();
                        tc_fence_after();
                        const uint32_t pair = base + ps * kPairBytes;
#pragma unroll
                        for (int half = 0; half < 2; ++half)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                umma_f16(d_s + 16u * kk, umma_desc_sw128(pair + half * kBoxBytes16 + 32u * kk),
                                         umma_desc_sw128(base + kOffQ + (2 * pr + half) * kQBox + 32u * kk), idesc_s,
                                         (pr | half) ? 1u : 0u);
                    }
                    if (!ok) break;
                    if (nbox_r) {
                        const int rs = static_cast<int>(k % kRopeSlots);
                        if (!mbar_wait(&bar[kBRopeFull + rs], static_cast<uint32_t>((k / kRopeSlots) & 1), abort_flag,
                                       a.wait_ns)) { ok = false; break; }
                        fence_proxy_async_smem();
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f16(d_s + 16u * kk, umma_desc_sw128(base + kOffRope + rs * kBoxBytes16 + 32u * kk),
                                     umma_desc_sw128(base + kOffQ + 8 * kQBox + 32u * kk), idesc_s, 1u);
                        umma_commit(&bar[kBRopeEmpty + rs]);
                    }
                    umma_commit(&bar[kBSFull + sb]);
                    if (cur_last) umma_commit(&bar[kBQEmpty]);  // the row's queries are free
                }
                if (have_prev) {
                    // tile k-1's P, and for a row's first tile its O buffer free again
                    if (!mbar_wait(&bar[kBPFull + pb], static_cast<uint32_t>(((k - 1) >> 1) & 1), abort_flag,
                                   a.wait_ns)) { ok = false; break; }
                    if (prev_first && !mbar_wait(&bar[kBOEmpty + prev_ob], static_cast<uint32_t>((prev_seg >> 1) & 1) ^ 1u,
                                                 abort_flag, a.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t p_base = base + kOffP + pb * kPBuf;
                    // pair by pair, each freed as soon as its products finish
                    for (int pr = 0; pr < 4; ++pr) {
                        const int ps = static_cast<int>((4 * (k - 1) + pr) % kPairSlots);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_f16(tmem + kColO + 64u * prev_ob + 16u * pr,
                                     umma_desc_sw128_mn(base + ps * kPairBytes + 2048u * kk, kBoxBytes16),
                                     umma_desc_sw128(p_base + 32u * kk), idesc_o, (prev_first && kk == 0) ? 0u : 1u);
                        umma_commit(&bar[kBPairEmpty + ps]);
                    }
                    umma_commit(&bar[kBPEmpty + pb]);
                    umma_commit(&bar[kBODone + pb]);  // tile k-1's output products, by tile parity
                    if (prev_last) umma_commit(&bar[kBOFull + prev_ob]);  // the row's O is complete
                }
                // tile k becomes the previous one
                if (have_cur) {
                    if (cur_first) {
                        prev_seg = o_segs;
                        prev_ob = o_segs & 1;
                        ++o_segs;
                    }
                    prev_first = cur_first;
                    prev_last = cur_last;
                    it.next(a, t0, t1);
                    ++k;
                }
                have_prev = have_cur;
            }
            if (!ok) fail();
            umma_commit(&bar[kBDone]);  // every MMA issued has finished before teardown
            mbar_wait(&bar[kBDone], 0, nullptr, a.wait_ns);
        }
    } else {
        // ------------------------------------------------------------ softmax + output
        const int sw = warp - 5;             // softmax warp 0..3
        const int quarter = warp & 3;        // TMEM lanes this warp may access
        const int j = quarter * 32 + lane;   // dim within an O block (TMEM lane of the output product)
        // entry of the tile: the M = 64 score product puts entry 16q + i in lane i < 16 of quarter q
        const bool has_entry = lane < 16;
        const int je = quarter * 16 + lane;
        int64_t tile_no = 0;
        int o_segs = 0, half = 0;
        bool ok = true;
        for (int row = row_a; row <= row_b && ok; ++row) {
            const Seg sg = segment_of(a, t0, t1, row);
            const bool whole = sg.tin_a == 0 && sg.tin_b == a.tiles_per_row - 1;
            float m_run[16], l_bf[16], l_ex[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                m_run[h] = -INFINITY;
                l_bf[h] = 0.0f;
                l_ex[h] = 0.0f;
            }
            const int ob = o_segs & 1;
            for (int tt = 0; tt < sg.n_act; ++tt, ++tile_no) {
                const int sb = static_cast<int>(tile_no & 1);
                const uint32_t use = static_cast<uint32_t>((tile_no >> 1) & 1);
                const int e = (sg.tin_a + tt) * kMlaTile + je;
                const int sraw = has_entry ? raw_slot(a, row, sg.kvl, e) : -1;  // lanes 16-31: no entry
                int okw = 1;
                if (lane == 0) okw = mbar_wait(&bar[kBSFull + sb], use, abort_flag, a.wait_ns) ? 1 : 0;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (bar_red_or(!okw, kSoftBar, 128)) { ok = false; break; }  // the four warps leave together
                tc_fence_after();
                uint32_t raw[16];
                {
                    const uint32_t ts = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kColS + 64u * sb;
                    uint32_t r0[16], r1[16], r2[16], r3[16];
                    tmem_ld16(ts, r0);
                    tmem_ld16(ts + 16, r1);
                    tmem_ld16(ts + 32, r2);
                    tmem_ld16(ts + 48, r3);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 16; ++h)
                        raw[h] = __float_as_uint((__uint_as_float(r0[h]) + __uint_as_float(r1[h])) +
                                                 (__uint_as_float(r2[h]) + __uint_as_float(r3[h])));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kBSEmpty + sb]);
                const bool valid = checked_slot(a, sraw) >= 0;
                float x[16];
                bool need = tt == 0;
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    x[h] = valid ? __uint_as_float(raw[h]) * a.scale_log2 : -INFINITY;
                    need |= x[h] > m_run[h] + kRaise;
                }
                need = bar_red_or(need, kSoftBar, 128);
                if (need) {
                    float t[16];
#pragma unroll
                    for (int h = 0; h < 16; ++h) t[h] = x[h];
                    soft_reduce<0>(t, red, half, sw, lane);
                    float alpha[16];
                    bool grow = false;
#pragma unroll
                    for (int h = 0; h < 16; ++h) {
                        const float mn = fmaxf(m_run[h], t[h]);
                        alpha[h] = mn > m_run[h] ? exp2f(m_run[h] - mn) : 1.0f;
                        grow |= mn > m_run[h];
                        m_run[h] = mn;
                    }
                    if (grow && tt > 0) {
                        // the previous tile's output products must finish first: completion
                        // (t-1) >> 1 of O_DONE[(t-1) & 1]. That barrier's previous completion
                        // (tile t-3) was committed before this tile's scores, and its next one
                        // (tile t+1) needs a P not yet written, so the parity names one phase.
                        int okd = 1;
                        if (lane == 0)
                            okd = mbar_wait(&bar[kBODone + ((tile_no - 1) & 1)],
                                            static_cast<uint32_t>(((tile_no - 1) >> 1) & 1), abort_flag, a.wait_ns)
                                      ? 1 : 0;
                        okd = __shfl_sync(0xffffffffu, okd, 0);
                        if (bar_red_or(!okd, kSoftBar, 128)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int h = 0; h < 16; ++h) {
                            l_bf[h] *= alpha[h];
                            l_ex[h] *= alpha[h];
                        }
                        for (int mb = 0; mb < 4; ++mb) {
                            const uint32_t ta = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kColO + 64u * ob +
                                                16u * mb;
                            uint32_t ov[16];
                            tmem_ld16(ta, ov);
                            tmem_ld_wait();
#pragma unroll
                            for (int h = 0; h < 16; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
                            tmem_st16(ta, ov);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                    }
                }
                // p = 2^(x - max), rounded to bf16 for the product; both sums kept per thread
                uint16_t pb[16];
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const float p = x[h] == -INFINITY ? 0.0f : exp2f(x[h] - m_run[h]);
                    const __nv_bfloat16 b = __float2bfloat16_rn(p);
                    pb[h] = __bfloat16_as_ushort(b);
                    l_bf[h] += __bfloat162float(b);
                    l_ex[h] += p;
                }
                if (lane == 0) okw = mbar_wait(&bar[kBPEmpty + sb], use ^ 1u, abort_flag, a.wait_ns) ? 1 : 0;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (bar_red_or(!okw, kSoftBar, 128)) { ok = false; break; }
                if (has_entry) {
                    uint8_t* pbase = sm + kOffP + sb * kPBuf + (je & 7) * 2;
                    const uint32_t chunk = static_cast<uint32_t>(je >> 3);
#pragma unroll
                    for (int h = 0; h < 16; ++h)
                        *reinterpret_cast<uint16_t*>(pbase + h * 128 + ((chunk ^ (h & 7)) << 4)) = pb[h];
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kBPFull + sb]);
            }
            if (!ok) break;
            // ---- the row's (or partial row's) result
            soft_reduce<1>(l_bf, red, half, sw, lane);
            soft_reduce<1>(l_ex, red, half, sw, lane);
            const int pslot = 2 * static_cast<int>(blockIdx.x) + (row == row_a ? 0 : 1);
            float* part = reinterpret_cast<float*>(a.part + static_cast<size_t>(pslot) * kMlaPartBytes);
            if (sg.n_act > 0) {
                int okw = 1;
                if (lane == 0) okw = mbar_wait(&bar[kBOFull + ob], static_cast<uint32_t>((o_segs >> 1) & 1), abort_flag,
                                               a.wait_ns) ? 1 : 0;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (bar_red_or(!okw, kSoftBar, 128)) { ok = false; break; }
                tc_fence_after();
                for (int mb = 0; mb < 4; ++mb) {
                    uint32_t ov[16];
                    tmem_ld16(tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kColO + 64u * ob + 16u * mb, ov);
                    tmem_ld_wait();
                    const int d = mb * 128 + j;
                    if (whole) {
                        float* o = a.out + static_cast<int64_t>(row) * (kMlaHeads * kMlaDc) + d;
#pragma unroll
                        for (int h = 0; h < 16; ++h)
                            o[h * kMlaDc] = l_bf[h] > 0.0f ? __uint_as_float(ov[h]) / l_bf[h] : 0.0f;
                    } else {
#pragma unroll
                        for (int h = 0; h < 16; ++h) part[h * kMlaDc + d] = __uint_as_float(ov[h]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[kBOEmpty + ob]);
                ++o_segs;
            } else if (whole) {
                for (int d = j; d < kMlaDc; d += 128) {
                    float* o = a.out + static_cast<int64_t>(row) * (kMlaHeads * kMlaDc) + d;
#pragma unroll
                    for (int h = 0; h < 16; ++h) o[h * kMlaDc] = 0.0f;
                }
            }
            // one thread per head: the row's log-sum-exp, or the partial's maximum and sums
            if (sw == 0 && lane < 16) {
                float mh = 0.0f, lb = 0.0f, le = 0.0f;
#pragma unroll
                for (int h = 0; h < 16; ++h)
                    if (h == lane) {
                        mh = m_run[h];
                        lb = l_bf[h];
                        le = l_ex[h];
                    }
                if (whole) {
                    a.lse[static_cast<int64_t>(row) * kMlaHeads + lane] =
                        le > 0.0f ? (mh + log2f(le)) * 0.69314718055994531f : -INFINITY;
                } else {
                    part[kMlaHeads * kMlaDc + lane] = le > 0.0f ? mh : -INFINITY;
                    part[kMlaHeads * kMlaDc + 16 + lane] = lb;
                    part[kMlaHeads * kMlaDc + 32 + lane] = le;
                }
            }
        }
        if (!ok) fail();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 4) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// One CTA per (row, head): a row whose tiles ran in more than one CTA gets the weighted
// combination of their partials (weights 2^(m_c - max_c m_c)); other rows were written whole.
// A row has at most kMlaMaxTilesPerRow tiles (the host checks), so at most that many
// partials. Every thread loads its four dims of each partial together with the partials'
// maxima and sums (one round of loads, no block barrier) and computes the weights itself.
__global__ void __launch_bounds__(128) k_mla_merge(const MlaArgs a, int grid) {
    // launched as a dependent grid: its CTAs are in place when the decode kernel ends, and wait
    // here for its partials and outputs
    pdl_wait();
    const int row = blockIdx.x, h = blockIdx.y;
    const int64_t tpr = a.tiles_per_row, total = a.total_tiles, G = grid;
    const int64_t first = static_cast<int64_t>(row) * tpr, last = first + tpr - 1;
    // CTA c runs tiles [c * total / G, (c + 1) * total / G): the CTA of tile t is the last c
    // whose first tile is <= t
    const int c_lo = static_cast<int>(((first + 1) * G - 1) / total);
    const int c_hi = static_cast<int>(((last + 1) * G - 1) / total);
    if (c_lo == c_hi) return;
    const int n = c_hi - c_lo + 1;
    const int t = threadIdx.x;
    auto part_of = [&](int i) {
        const int c = c_lo + i;
        const int slot = 2 * c + ((c * total / G) < first ? 1 : 0);
        return reinterpret_cast<const float*>(a.part + static_cast<size_t>(slot) * kMlaPartBytes);
    };
    float mx = -INFINITY, lb = 0.0f, le = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    constexpr int kB = 8;  // partials whose loads are in flight together
    for (int i0 = 0; i0 < n; i0 += kB) {
        float m[kB], b[kB], e[kB];
        float4 v[kB];
#pragma unroll
        for (int k = 0; k < kB; ++k) {
            if (i0 + k < n) {
                const float* p = part_of(i0 + k);
                m[k] = __ldcg(p + kMlaHeads * kMlaDc + h);
                b[k] = __ldcg(p + kMlaHeads * kMlaDc + 16 + h);
                e[k] = __ldcg(p + kMlaHeads * kMlaDc + 32 + h);
                v[k] = __ldcg(reinterpret_cast<const float4*>(p + h * kMlaDc) + t);
            } else {
                m[k] = -INFINITY;
            }
        }
#pragma unroll
        for (int k = 0; k < kB; ++k) {
            if (m[k] == -INFINITY) continue;  // a partial without entries: its values were never written
            // a running maximum: rescale what was summed so far when it rises
            if (m[k] > mx) {
                const float r = mx == -INFINITY ? 0.0f : exp2f(mx - m[k]);
                lb *= r;
                le *= r;
                acc.x *= r;
                acc.y *= r;
                acc.z *= r;
                acc.w *= r;
                mx = m[k];
            }
            const float w = exp2f(m[k] - mx);
            lb += w * b[k];
            le += w * e[k];
            acc.x += w * v[k].x;
            acc.y += w * v[k].y;
            acc.z += w * v[k].z;
            acc.w += w * v[k].w;
        }
    }
    const float inv = lb > 0.0f ? 1.0f / lb : 0.0f;
    reinterpret_cast<float4*>(a.out + (static_cast<int64_t>(row) * kMlaHeads + h) * kMlaDc)[t] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (t == 0)
        a.lse[static_cast<int64_t>(row) * kMlaHeads + h] =
            le > 0.0f ? (mx + log2f(le)) * 0.69314718055994531f : -INFINITY;
}

size_t mla_smem_bytes() { return kSmemUsed + 1024; }

cudaError_t launch_mla(const MlaArgs& a, int grid, cudaStream_t s) {
    static size_t configured[kMaxDevicesTracked] = {};
    const size_t smem = mla_smem_bytes();
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevicesTracked && smem > configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_mla_decode, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = smem;
    }
    k_mla_decode<<<grid, kMlaThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_mla_merge(const MlaArgs& a, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.rows), kMlaHeads, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_mla_merge, a, grid);
}

}  // namespace sel
