// Pieces shared by the attention kernels: launch parameters, the device
// error word, bounded mbarrier waits, the cp.async tile loader and small
// conversions.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "gqa_attn.h"
#include "sm103_ptx.cuh"

namespace gqa {

constexpr int kBM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;  // key/value rows per tile

// Error word of this library on each device, and the sequence number of the
// launch that gave up (so that its remaining CTAs exit at once).
__device__ int g_error_code;
__device__ unsigned int g_abort_seq;

// Key tiles a causal query tile visits: every tile up to the one holding the
// last key visible to its last valid row (row < Nq).
__device__ __forceinline__ int causal_kv_tiles(int row0, int Nq, int causal_off, int n_kv_tiles) {
    const int last_row = (row0 + kBM - 1 < Nq - 1) ? row0 + kBM - 1 : Nq - 1;
    const int n = (last_row + causal_off) / kBN + 1;
    return n < n_kv_tiles ? n : n_kv_tiles;
}

struct Params {
    const uint8_t *q;  // [B*Hq, Nq, D] elements of 2 bytes
    const uint8_t *k;  // [B*Hkv, Nk, D]
    const uint8_t *v;  // [B*Hkv, Nk, D]
    void *o;
    float *lse;
    int Nq;          // query rows per head
    int Nk;          // keys per head
    int causal_off;  // Nk - Nq: under the causal mask query row i sees keys j <= i + causal_off
    int group;       // Hq / Hkv
    int n_qtiles;    // ceil(Nq / kBM)
    int n_kv_tiles;  // ceil(Nk / kBN)
    int BHq;         // B * Hq
    int n_qblocks;   // ceil(Nq / 256): work items of the persistent kernel per head
    int n_items;     // BHq * n_qblocks
    float scale_log2;  // scale * log2(e)
    unsigned int seq;
    unsigned long long timeout_ns;
    int inject_stall;  // test hook: the producer never loads Q
    int item_order;    // persistent kernel: 0 head-fastest, 1 kv-group major
    // persistent kernel, key-split work units (attn_fwd_kv_split): units [0, n_whole)
    // are whole items; every item from n_whole on is cut into n_parts key ranges
    int n_units;       // n_whole + (n_items - n_whole) * n_parts
    int n_whole;
    int n_parts;
    float *part_o;     // [split items][n_parts][2 tiles][128 rows][D] partial outputs (O / l)
    float *part_lse;   // [split items][n_parts][2 tiles][128 rows] partial log-sum-exp
    unsigned int *part_count;  // [split items][2 tiles][4 warps] arrivals, tagged with the launch
    // packed short-query path (attn_fwd_decode)
    int rows_per_kv;   // Hq / Hkv * Nq query rows share one kv head (contiguous in Q)
    int n_mtiles;      // ceil(rows_per_kv / kBM)
    int n_splits;      // key splits per (kv head, row tile)
    int split_tiles;   // key tiles per split
    int total_rows;    // B * Hq * Nq
    float *ws_o;       // [n_splits, total_rows, D] partial outputs (n_splits > 1)
    float *ws_lse;     // [n_splits, total_rows] partial log-sum-exp
};

// Bounded wait on an mbarrier phase.  Spins on try_wait alone; every 256
// spins it checks this CTA's abort flag, and once a millisecond has passed it
// also checks whether another CTA of the launch gave up and whether timeout_ns
// has run out (then it records ATTN_ERR_TIMEOUT and returns false).  Keeping
// the global-memory check out of the tight loop matters: a waiting warp that
// stalls on a global load notices the phase change late.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Params &p,
                                         volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 255u) == 0) {
            if (*abort_flag) return false;
            const uint64_t dt = global_timer_ns() - t0;
            if (dt > 1000000ull) {
                if (*reinterpret_cast<volatile unsigned int *>(&g_abort_seq) == p.seq) {
                    *abort_flag = 1;
                    return false;
                }
                if (dt > p.timeout_ns) {
                    *abort_flag = 1;
                    atomicCAS(&g_error_code, 0, static_cast<int>(ATTN_ERR_TIMEOUT));
                    atomicExch(&g_abort_seq, p.seq);
                    return false;
                }
            }
        }
    }
}

// Bounded wait used while shutting down: ignores the abort flag.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, const Params &p) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > p.timeout_ns) {
            atomicCAS(&g_error_code, 0, static_cast<int>(ATTN_ERR_TIMEOUT));
            return;
        }
    }
}

constexpr int kLoaderThreads = 64;  // warps 2 and 3 of the per-tile cross-check kernel
constexpr int kAtomBytes = 128 * 128;  // 128 rows x 128 B: one 128-byte swizzle atom column

// Copies rows [row0, row0 + 128) of one head ([N, D], 2-byte elements, D
// fastest) into a shared-memory tile in the UMMA K-major 128-byte-swizzle
// layout: columns [64a, 64a + 64) of row r sit in atom a at r * 128 bytes, and
// 16-byte chunk c of that 128-byte row is stored at chunk c ^ (r % 8).  Rows
// at or past N are zero-filled.  Each of the 64 loader threads owns one
// 16-byte column chunk and every (64 / chunks-per-row)-th row, so a warp
// reads 512 contiguous bytes per instruction.
template <int D>
__device__ __forceinline__ void load_tile(uint32_t dst, const uint8_t *head, int row0, int N, int ltid) {
    constexpr int kChunksPerRow = D / 8;
    constexpr int kRowStep = kLoaderThreads / kChunksPerRow;  // rows between a thread's copies
    constexpr int kIters = 128 / kRowStep;
    const int cc = ltid % kChunksPerRow;
    const int r0 = ltid / kChunksPerRow;  // < kRowStep <= 8
    const uint32_t col = (cc >> 3) * kAtomBytes;
    // Row r0 + i*kRowStep has swizzle phase (r0 + i*kRowStep) % 8: constant when the
    // step is 8, alternating between two values when it is 4.
    const uint32_t d_even = dst + col + r0 * 128 + (((cc & 7) ^ (r0 & 7)) << 4);
    const uint32_t d_odd = dst + col + r0 * 128 + (((cc & 7) ^ ((r0 + kRowStep) & 7)) << 4);
    const uint8_t *src = head + static_cast<size_t>(row0 + r0) * (D * 2) + cc * 16;
    if (row0 + 128 <= N) {
        // whole tile in range: every copy is a base plus a compile-time offset
#pragma unroll
        for (int i = 0; i < kIters; ++i)
            cp_async_16(((i & 1) ? d_odd : d_even) + i * kRowStep * 128, src + i * kRowStep * (D * 2), 16u);
    } else {
        const uint8_t *row_zero = head + cc * 16;  // any valid address for zero-filled rows
#pragma unroll 4
        for (int i = 0; i < kIters; ++i) {
            const bool in = row0 + r0 + i * kRowStep < N;
            cp_async_16(((i & 1) ? d_odd : d_even) + i * kRowStep * 128,
                        in ? src + i * kRowStep * (D * 2) : row_zero, in ? 16u : 0u);
        }
    }
}

// Completion protocol of the loader threads: each committed cp.async group is
// announced one group late (wait for all but the newest group, make the data
// visible to the tensor core's async proxy, then arrive on its barriers), so
// that copies of consecutive tiles overlap.
struct LoadSignal {
    uint32_t bar_a = 0, bar_b = 0;  // barriers of the newest, not yet announced group
    template <bool kAll>
    __device__ __forceinline__ void announce() {
        if (bar_a == 0) return;
        if (kAll) cp_async_wait<0>(); else cp_async_wait<1>();
        fence_proxy_async_smem();
        mbar_arrive(bar_a);
        if (bar_b != 0) mbar_arrive(bar_b);
        bar_a = bar_b = 0;
    }
    // Commit the group just issued; announce the one before it.
    __device__ __forceinline__ void commit(uint32_t a, uint32_t b = 0) {
        cp_async_commit();
        announce<false>();
        bar_a = a;
        bar_b = b;
    }
};

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (kBF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

// The two halves of a packed pair as floats (exact).
template <bool kBF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (kBF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    } else {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        return __half22float2(h);
    }
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

}  // namespace gqa
