// Short query blocks over long key sequences (decode steps, small chunks):
// grouped-query packing and split keys.
//
// Packing.  The G = Hq/Hkv query heads that share a kv head are adjacent, and
// each has Nq contiguous rows, so the G*Nq query rows of one kv head form one
// contiguous block of the flattened [B*Hq*Nq, D] query matrix (and of O and
// LSE).  A 128-row tile of that block is an ordinary row range: packed row m
// is query position i = m % Nq of head m / Nq, and the causal mask keeps key
// j <= i + Nk - Nq.  Every K/V tile is then read once per kv head instead of
// once per query head.
//
// Split keys.  With few kv heads the (kv head, row tile) pairs cannot fill the
// GPU, so the key range is cut into n_splits pieces of split_tiles 128-key
// tiles, one CTA each.  A CTA writes its rows' partial output (already divided
// by its own running sum) and partial log-sum-exp to a workspace; a second
// kernel merges the pieces of a row with weights exp(lse_s - lse), where lse
// is the log-sum-exp over the pieces.  This is the online-softmax merge of the
// page "从零开始写Qwen3" (deepseek.csdn.net/6a3201f8..., section "在线softmax")
// applied across CTAs instead of across the tiles of one CTA.  With one split
// the first kernel writes O and LSE itself and no workspace is used.
//
// Roles (256 threads): warp 2 lane 0 loads (TMA, 4-stage ring), warp 1 issues
// the MMAs (S = Q K^T and O += P V into TMEM), warps 4-7 run the softmax of
// one row each and stage P through shared memory.  S has two TMEM buffers and
// P two shared-memory buffers, so the tensor core computes S(j+1) while the
// softmax works on S(j), and the softmax waits for P(j-1) V only when it must
// rescale O.  The O accumulator is rescaled whenever a row's max grows, so the
// largest weight of a row is exactly 1 and near one-hot rows keep their
// ratios through P's rounding.
#pragma once
#include <cuda.h>  // CUtensorMap

#include "kernel_common.cuh"

namespace gqa {

constexpr int kDecStages = 4;
constexpr int kDecThreads = 256;
constexpr uint32_t kDecTmemCols = 512;  // S0 [0, 128), S1 [128, 256), O [256, 256 + D)
constexpr uint32_t kDecTmemO = 256;
constexpr int kPBytes = 2 * kAtomBytes;  // one P buffer: 128 x 128 halves

template <int D>
struct DecLayout {
    static constexpr int kTileBytes = (D / 64) * kAtomBytes;
    static constexpr int kQ = 0;
    static constexpr int kKV = kQ + kTileBytes;
    static constexpr int kP = kKV + kDecStages * kTileBytes;  // P0, P1
    static constexpr int kBar = kP + 2 * kPBytes;
    // q_full, kv_full[S], kv_empty[S], s_full[2], p_full, o_done[2], mma_done
    static constexpr int kNumBars = 1 + 2 * kDecStages + 2 + 1 + 2 + 1;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kAlloc = kAbort + 4 + 1024;  // slack to align the base to 1024 B
};

// Smallest and largest query position i = m % Nq among the packed rows
// [m0, min(m0 + 128, rows)) of one kv head.
struct PosRange {
    int lo, hi;
};
__device__ __forceinline__ PosRange tile_positions(int m0, int rows, int Nq) {
    const int last = (m0 + kBM < rows ? m0 + kBM : rows) - 1;
    if (last - m0 + 1 >= Nq) return {0, Nq - 1};
    const int a = m0 % Nq, b = last % Nq;
    return a <= b ? PosRange{a, b} : PosRange{0, Nq - 1};
}

// tmQ: 3-D tensor map (D, rows_per_kv, B*Hkv) of Q seen as [B*Hkv, G*Nq, D] (the
// packed rows of each kv head); tmK, tmV: (D, Nk, B*Hkv).  Box 64 x 128 x 1 with the
// 128-byte swizzle; rows past the end of a kv head's block read as zeros.
template <int D, bool kBF16, bool kCausal>
__global__ void __launch_bounds__(kDecThreads, 1)
    attn_fwd_decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const Params p) {
    using L = DecLayout<D>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = static_cast<int>(blockIdx.x % p.n_splits);
    const int tile = static_cast<int>(blockIdx.x / p.n_splits);
    const int mt = tile % p.n_mtiles;
    const int bkv = tile / p.n_mtiles;  // b*Hkv + kv head
    const int m0 = mt * kBM;
    const size_t base_row = static_cast<size_t>(bkv) * p.rows_per_kv;  // flattened row of packed row 0
    const PosRange pos = tile_positions(m0, p.rows_per_kv, p.Nq);
    const int kt0 = split * p.split_tiles;
    int kt1 = kt0 + p.split_tiles < p.n_kv_tiles ? kt0 + p.split_tiles : p.n_kv_tiles;
    if (kCausal) {
        const int last = (pos.hi + p.causal_off) / kBN + 1;  // past the last key any row sees
        kt1 = kt1 < last ? kt1 : last;
    }
    const int n_kv = kt1 > kt0 ? kt1 - kt0 : 0;
    const bool partial = p.n_splits > 1;

    // This kernel and the merge are launched as programmatic dependents: let the
    // next one start launching now (it waits for this grid before touching
    // memory), and touch global memory only after the grid before this one is
    // done (a previous call's merge may still read the workspace).
    grid_launch_dependents();
    if (n_kv == 0) {
        // No key of this split is visible to these rows (only with several splits):
        // an empty piece, weight zero in the merge.
        grid_dependency_wait();
        if (warp >= 4) {
            const int m = m0 + (warp - 4) * 32 + lane;
            if (m < p.rows_per_kv) {
                const size_t R = static_cast<size_t>(split) * p.total_rows + base_row + m;
                float4 *dst = reinterpret_cast<float4 *>(p.ws_o + R * D);
#pragma unroll
                for (int d = 0; d < D / 4; ++d) dst[d] = make_float4(0.f, 0.f, 0.f, 0.f);
                p.ws_lse[R] = -INFINITY;
            }
        }
        return;
    }

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sQ = base + L::kQ, sKV = base + L::kKV, sP = base + L::kP;
    const uint32_t bar0 = base + L::kBar;
    const uint32_t q_full = bar0;
    auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return bar0 + 8u * (1 + kDecStages + s); };
    auto s_full = [&](int b) { return bar0 + 8u * (1 + 2 * kDecStages + b); };
    const uint32_t p_full = bar0 + 8u * (3 + 2 * kDecStages);
    auto o_done = [&](int b) { return bar0 + 8u * (4 + 2 * kDecStages + b); };  // P_b V finished
    const uint32_t mma_done = bar0 + 8u * (6 + 2 * kDecStages);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbort);

    if (threadIdx.x == 0) {
        *abort_flag = (*reinterpret_cast<volatile unsigned int *>(&g_abort_seq) == p.seq) ? 1 : 0;
        mbar_init(q_full, 1);
        for (int s = 0; s < kDecStages; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        mbar_init(s_full(0), 1);
        mbar_init(s_full(1), 1);
        mbar_init(p_full, kBM);
        mbar_init(o_done(0), 1);
        mbar_init(o_done(1), 1);
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (*abort_flag) return;  // another CTA of this launch already gave up
    if (warp == 1) {
        tmem_alloc(base + L::kTmemSlot, kDecTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();  // the set-up above overlapped the previous kernel's tail

    if (warp == 2) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            // One tile = D/64 boxes of 128 rows x 64 columns (x = 64a: a multiple of
            // 16 bytes); its full barrier expects all of its bytes.
            auto load_tile_tma = [&](uint32_t dst, const CUtensorMap *tm, int row, uint32_t bar) {
                mbar_arrive_expect_tx(bar, L::kTileBytes);
#pragma unroll
                for (int a = 0; a < D / 64; ++a) tma_load_3d(dst + a * kAtomBytes, tm, 64 * a, row, bkv, bar);
            };
            const bool q_loaded = !p.inject_stall;
            if (q_loaded) load_tile_tma(sQ, &tmQ, m0, q_full);
            int stage = 0, loads = 0;
            uint32_t phase = 0;
            auto load = [&](const CUtensorMap *tm, int j) -> bool {
                if (!wait_bar(kv_empty(stage), phase ^ 1u, p, abort_flag)) return false;
                load_tile_tma(sKV + stage * L::kTileBytes, tm, (kt0 + j) * kBN, kv_full(stage));
                ++loads;
                if (++stage == kDecStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                return true;
            };
            // the MMA warp's order: K_0, K_1, then V_j, K_{j+2} for each j
            bool ok = load(&tmK, 0) && (n_kv < 2 || load(&tmK, 1));
            for (int j = 0; j < n_kv && ok; ++j) ok = load(&tmV, j) && (j + 2 >= n_kv || load(&tmK, j + 2));
            // Every copy has landed before the CTA exits (also after a timeout).  The
            // ring is filled in order, so stage st last received a copy in the current
            // lap (phase) if st < stage, else in the lap before.
#pragma unroll
            for (int st = 0; st < kDecStages; ++st)
                if (loads > st) drain_bar(kv_full(st), st < stage ? phase : phase ^ 1u, p);
            if (q_loaded) drain_bar(q_full, 0, p);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            constexpr uint32_t idesc_qk = idesc_f16_f32acc(kBF16, kBM, kBN, false);
            constexpr uint32_t idesc_pv = idesc_f16_f32acc(kBF16, kBM, D, true);
            const uint32_t tO = tmem + kDecTmemO;
            bool ok = wait_bar(q_full, 0, p, abort_flag);
            tc_fence_after();
            int stage = 0;
            uint32_t phase = 0;
            auto next_stage = [&]() -> uint32_t {
                const uint32_t st = sKV + stage * L::kTileBytes;
                if (++stage == kDecStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                return st;
            };
            // S_b = Q K^T into TMEM buffer b (A = Q, B = K: both K-major, 128-byte swizzle)
            auto qk = [&](int b) -> bool {
                if (!wait_bar(kv_full(stage), phase, p, abort_flag)) return false;
                tc_fence_after();
                const int ks = stage;
                const uint32_t sK = next_stage();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
                    mma_f16_ss(tmem + 128u * b, sdesc_sw128(sQ + koff, 16, 1024),
                               sdesc_sw128(sK + koff, 16, 1024), idesc_qk, kk > 0);
                }
                mma_commit(s_full(b));
                mma_commit(kv_empty(ks));
                return true;
            };
            ok = ok && qk(0) && (n_kv < 2 || qk(1));
            for (int j = 0; j < n_kv && ok; ++j) {
                // O += P_b V_j   (A = P: K-major; B = V: MN-major, 64-wide chunks of D at
                // LBO = one atom, 8-row groups of keys at SBO = 1024 B)
                const int b = j & 1;
                if (!(ok = wait_bar(p_full, j & 1, p, abort_flag))) break;
                tc_fence_after();
                if (!(ok = wait_bar(kv_full(stage), phase, p, abort_flag))) break;
                tc_fence_after();
                const int vs = stage;
                const uint32_t sV = next_stage();
                const uint32_t sPb = sP + b * kPBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint32_t poff = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
                    mma_f16_ss(tO, sdesc_sw128(sPb + poff, 16, 1024),
                               sdesc_sw128(sV + kk * 2048, kAtomBytes, 1024), idesc_pv,
                               (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(o_done(b));
                mma_commit(kv_empty(vs));
                // S_b is free: its softmax read it before P_b was ready
                if (j + 2 < n_kv) ok = qk(b);
            }
            mma_commit(mma_done);
            drain_bar(mma_done, 0, p);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------- softmax rows
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // row within the tile == TMEM lane
        const int m = m0 + r;          // packed row
        const bool valid = m < p.rows_per_kv;
        const int key_last = kCausal ? (valid ? m % p.Nq : 0) + p.causal_off : p.Nk - 1;
        // A key tile needs a mask when some row of the tile does not see all of it.
        const int tile_key_last = kCausal ? pos.lo + p.causal_off : p.Nk - 1;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tO = tmem + kDecTmemO + lane_off;
        const float c = p.scale_log2;
        float mrow = -INFINITY, l = 0.f;
        bool ok = true;
        const uint32_t prow = sP + (r >> 3) * 1024 + (r & 7) * 128;
        for (int j = 0; j < n_kv; ++j) {
            const int b = j & 1;  // S, P buffer of this tile
            if (!__all_sync(0xffffffffu, wait_bar(s_full(b), (j >> 1) & 1, p, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            __syncwarp();
            const int kv0 = (kt0 + j) * kBN;
            const uint32_t tS = tmem + 128u * b + lane_off;
            uint32_t s[128];
            float mt;
            if (kv0 + kBN - 1 <= tile_key_last) {
                float mq[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tmem_ld32_max(tS + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * q]), mq[q]);
                tmem_ld_wait(s, mq);
                mt = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tmem_ld32(tS + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * q]));
                tmem_ld_wait(s);
                const int lim = key_last - kv0;  // keep keys c <= lim of this tile
#pragma unroll
                for (int cc = 0; cc < 128; ++cc)
                    if (cc > lim) s[cc] = __float_as_uint(-INFINITY);
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = fmaxf(u2f(s[2 * k]), u2f(s[2 * k + 1]));
#pragma unroll
                for (int cc = 16; cc < 128; cc += 16)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mx[k] = fmax3(mx[k], u2f(s[cc + 2 * k]), u2f(s[cc + 2 * k + 1]));
                mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
            }
            const float m_new = fmaxf(mrow, mt);
            // a row that has seen no key of this split yet keeps reference 0, so no
            // -inf - -inf appears; its weights are then exactly 0
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = ex2_approx((mrow - m_use) * c);  // 0 while nothing was seen
            if (j >= 2) {
                // P_b is free once P_b V_{j-2} is done
                if (!__all_sync(0xffffffffu, wait_bar(o_done(b), ((j - 2) >> 1) & 1, p, abort_flag))) {
                    ok = false;
                    break;
                }
            }
            if (j > 0 && __any_sync(0xffffffffu, m_new > mrow)) {
                // rescale O: P V_{j-1} must have finished writing it
                if (!__all_sync(0xffffffffu, wait_bar(o_done(b ^ 1), ((j - 1) >> 1) & 1, p, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                {
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * q, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(u2f(o[t]) * alpha);
                        tmem_st32(tO + 32 * q, o);
                    }
                    tmem_st_wait();
                }
            }
            mrow = m_new;
            const float2 c2 = make_float2(c, c);
            const float2 nmc2 = make_float2(-m_use * c, -m_use * c);
            float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int cc = ch * 8 + 2 * t;
                    float2 e = ffma2(make_float2(u2f(s[cc]), u2f(s[cc + 1])), c2, nmc2);
                    e.x = ex2_approx(e.x);
                    e.y = ex2_approx(e.y);
                    acc[t & 1] = fadd2(acc[t & 1], e);
                    w[t] = pack2<kBF16>(e.x, e.y);
                }
                const uint32_t addr = prow + b * kPBytes + (ch >> 3) * kAtomBytes + (((ch & 7) ^ (r & 7)) << 4);
                st_shared_v4(addr, w[0], w[1], w[2], w[3]);
            }
            const float2 sum2 = fadd2(acc[0], acc[1]);
            l = l * alpha + (sum2.x + sum2.y);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        // ---------------------------------------------------- epilogue
        if (ok && __all_sync(0xffffffffu,
                             wait_bar(o_done((n_kv - 1) & 1), ((n_kv - 1) >> 1) & 1, p, abort_flag))) {
            tc_fence_after();
            __syncwarp();
            const size_t R = base_row + m;  // flattened (b*Hq + hq)*Nq + i
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
            const float lse = l > 0.f ? ((mrow * c + log2f(l)) * 0.6931471805599453f) : -INFINITY;
            uint8_t *orow = static_cast<uint8_t *>(p.o) + R * (D * 2);
            float *wrow = p.ws_o + (static_cast<size_t>(split) * p.total_rows + R) * D;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(tO + 32 * q, o);
                tmem_ld_wait(o);
                if (!valid) continue;
                if (partial) {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        st_global_v4(wrow + q * 32 + v * 4, __float_as_uint(u2f(o[4 * v]) * inv_l),
                                     __float_as_uint(u2f(o[4 * v + 1]) * inv_l),
                                     __float_as_uint(u2f(o[4 * v + 2]) * inv_l),
                                     __float_as_uint(u2f(o[4 * v + 3]) * inv_l));
                } else {
                    uint32_t w[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        w[t] = pack2<kBF16>(u2f(o[2 * t]) * inv_l, u2f(o[2 * t + 1]) * inv_l);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        st_global_v4(orow + q * 64 + v * 16, w[4 * v], w[4 * v + 1], w[4 * v + 2],
                                     w[4 * v + 3]);
                }
            }
            if (valid) {
                if (partial)
                    p.ws_lse[static_cast<size_t>(split) * p.total_rows + R] = lse;
                else if (p.lse != nullptr)
                    p.lse[R] = lse;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kDecTmemCols);
    }
}

// Merges the n_splits pieces of every row: lse = log sum_s exp(lse_s) and
// O = sum_s exp(lse_s - lse) * O_s.  One warp per row and D/32 columns per
// lane; pieces go in batches of 16 whose log-sum-exps and partial rows are all
// requested at once, with the running max and sum rebased between batches (the
// same online merge), so up to 16 pieces cost one round trip to memory.  Launched as a
// programmatic dependent of the split kernel: it waits for that grid's results
// before reading them, so its launch overlaps the split kernel's tail.
template <int D, bool kBF16>
__global__ void __launch_bounds__(128) attn_combine_kernel(const Params p) {
    grid_launch_dependents();  // the next call's split kernel may begin its set-up
    grid_dependency_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long R = static_cast<long long>(blockIdx.x) * 4 + warp;
    if (R >= p.total_rows) return;
    constexpr int kPer = D / 32;
    if (*reinterpret_cast<volatile unsigned int *>(&g_abort_seq) == p.seq) {
        // The split kernel of this call gave up on a wait, so some pieces were
        // never written (with a shared buffer they would be an earlier call's):
        // mark the row as undefined instead of merging stale partials.
        uint8_t *dst = static_cast<uint8_t *>(p.o) + (static_cast<size_t>(R) * D + lane * kPer) * 2;
        const uint32_t nan2 = kBF16 ? 0x7FC07FC0u : 0x7E007E00u;
        if constexpr (kPer == 4)
            *reinterpret_cast<uint2 *>(dst) = make_uint2(nan2, nan2);
        else
            *reinterpret_cast<uint32_t *>(dst) = nan2;
        if (p.lse != nullptr && lane == 0) p.lse[R] = __int_as_float(0x7FC00000);
        return;
    }
    constexpr int kBatch = 16;  // pieces whose loads are in flight together
    const int S = p.n_splits;
    const size_t stride = static_cast<size_t>(p.total_rows);
    const float *col = p.ws_o + static_cast<size_t>(R) * D + lane * kPer;  // piece 0's columns
    float acc[kPer];
#pragma unroll
    for (int d = 0; d < kPer; ++d) acc[d] = 0.f;
    float mx = -INFINITY, sum = 0.f;  // running max and sum (lane-local weights, merged below)
    for (int s0 = 0; s0 < S; s0 += kBatch) {
        const int n = S - s0 < kBatch ? S - s0 : kBatch;
        // the batch's log-sum-exps (lane t < n holds piece s0 + t) and partial rows,
        // all requested before any of them is used
        const float ls = lane < n ? p.ws_lse[(s0 + lane) * stride + R] : -INFINITY;
        float v[kBatch][kPer];
#pragma unroll
        for (int t = 0; t < kBatch; ++t)
            if (t < n) {
                const float *q = col + static_cast<size_t>(s0 + t) * stride * D;
#pragma unroll
                for (int d = 0; d < kPer; ++d) v[t][d] = q[d];
            }
        float bm = ls;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
        // rebase what was accumulated so far onto the new max (split 0 sees key 0,
        // so the max is finite from the first batch on)
        const float m_new = fmaxf(mx, bm);
        const float scale_old = mx == -INFINITY ? 0.f : expf(mx - m_new);
#pragma unroll
        for (int d = 0; d < kPer; ++d) acc[d] *= scale_old;
        sum *= scale_old;
        mx = m_new;
        const float wl = ls == -INFINITY ? 0.f : expf(ls - mx);
        sum += wl;
#pragma unroll
        for (int t = 0; t < kBatch; ++t) {
            const float w = __shfl_sync(0xffffffffu, wl, t);
            if (t < n) {
#pragma unroll
                for (int d = 0; d < kPer; ++d) acc[d] += w * v[t][d];
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = 1.f / sum;
    uint32_t w[kPer / 2];
#pragma unroll
    for (int t = 0; t < kPer / 2; ++t) w[t] = pack2<kBF16>(acc[2 * t] * inv, acc[2 * t + 1] * inv);
    uint8_t *dst = static_cast<uint8_t *>(p.o) + (static_cast<size_t>(R) * D + lane * kPer) * 2;
    if constexpr (kPer == 4)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    else
        *reinterpret_cast<uint32_t *>(dst) = w[0];
    if (p.lse != nullptr && lane == 0) p.lse[R] = mx + logf(sum);
}

}  // namespace gqa
