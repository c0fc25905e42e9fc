// Pieces shared by the attention kernels: launch parameters, the device
// error word, bounded mbarrier waits and small conversions.
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

struct Params {
    void *o;
    float *lse;
    int N;
    int group;       // Hq / Hkv
    int n_qtiles;    // ceil(N / kBM)
    int n_kv_tiles;  // ceil(N / kBN)
    int BHq;         // B * Hq
    int n_qblocks;   // ceil(N / 256): work items of the persistent kernel per head
    int n_items;     // BHq * n_qblocks
    float scale_log2;  // scale * log2(e)
    unsigned int seq;
    unsigned long long timeout_ns;
    int inject_stall;  // test hook: the producer never loads Q
};

// Bounded wait on an mbarrier phase.  Gives up (returns false) when this CTA
// or another CTA of the same launch has given up, or after timeout_ns; the
// first to give up records ATTN_ERR_TIMEOUT.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Params &p,
                                         volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (*reinterpret_cast<volatile unsigned int *>(&g_abort_seq) == p.seq) {
            *abort_flag = 1;
            return false;
        }
        if (global_timer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            atomicCAS(&g_error_code, 0, static_cast<int>(ATTN_ERR_TIMEOUT));
            atomicExch(&g_abort_seq, p.seq);
            return false;
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

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

}  // namespace gqa
