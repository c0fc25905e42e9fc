// Persistent, warp-specialised fused GQA attention forward for sm_103a.
//
// A work item is a 256-row query block of one (batch, query head): two
// 128-row query tiles Q0, Q1 that share every K/V tile the producer brings
// in.  The online-softmax update is the one of the page "从零开始写Qwen3"
// (deepseek.csdn.net/6a3201f8..., sections "在线softmax" and "FlashAttention").
//
// Roles (384 threads):
//   warp 2        TMA producer (one lane): K_0, (Q0, Q1), V_0, K_1, V_1, ... as
//                 128-row boxes of 64 columns with the 128-byte swizzle, into a
//                 ring of kStagesWs tiles (full / empty mbarriers).  A unit's
//                 first K tile completes its own full barrier; V_j and K_{j+1}
//                 complete V_j's together (its transaction count is both tiles'
//                 bytes), so the MMA warp waits once per key tile.
//   warp 1        allocates and frees the 512 TMEM columns.
//   warp 0        MMA issuer (one lane):  S0 = Q0 K_0^T, S1 = Q1 K_0^T, then per
//                 key tile j:  O0 += P0 V_j,  S0 = Q0 K_{j+1}^T,  O1 += P1 V_j,
//                 S1 = Q1 K_{j+1}^T.  While softmax warpgroup 0 works on S0 the
//                 tensor core runs tile 1's products, and the other way round.
//   warps 4-7     softmax warpgroup 0 (rows of Q0, one row per thread = TMEM lane)
//   warps 8-11    softmax warpgroup 1 (rows of Q1)
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D).
// P_i (the probabilities, rounded to the input type, two per 32-bit column)
// overwrites the first 64 columns of S_i and is the TMEM A operand of P_i V_j,
// so P never goes through shared memory.  The commit that signals S_i(j+1)
// also covers P_i V_j (tcgen05.commit tracks every earlier MMA), so when a
// softmax thread sees S_i(j+1) its O_i row is stable and can be rescaled.
// The epilogue stages each warp's rows through shared memory so that every
// global store instruction writes whole 64-byte row segments.
//
// Work items are ordered longest causal row block first and dealt to the
// persistent CTAs in a snake order (CTA c takes item r*G + c on even rounds and
// r*G + G-1-c on odd rounds), which evens out the linearly shrinking causal
// work; the heads of one GQA group are adjacent so their K/V reads share L2
// (page "从零开始写Qwen3", deepseek.csdn.net/6a31faef..., "改进1-使用正确的grid").
// A second order (kv-group major: every block of one (batch, kv head) group
// before the next group) keeps one group's K/V in L2 at a time; measured, it
// is slower on causal problems, so it is not the default.
// Causal tiles above the diagonal are never loaded and only diagonal tiles are
// masked (same page, "改进2-KV只读取下三角", "改进3-两阶段计算").
#pragma once
#include <cuda.h>  // CUtensorMap

#include "kernel_common.cuh"

namespace gqa {

constexpr int kWsThreads = 384;
constexpr int kStagesWs = 4;
constexpr uint32_t kWsTmemCols = 512;
// A warp's 32 rows of probabilities are split into two input-type terms
// (P_hi + P_lo) when some row's running sum, in units of its largest weight,
// is below this.
constexpr float kSplitL = 4.f;
// The probabilities are referenced to a stale row max until the true max
// exceeds it by more than this many powers of two (P <= 2^8 meanwhile).
constexpr float kRescaleLog2 = 8.f;
// at most this many key ranges per cut item (attn_fwd_kv_split)
constexpr int kMaxPartsWs = 8;
constexpr uint32_t kRegsLow = 104;   // warps 0-3 after the hand-off
constexpr uint32_t kRegsHigh = 200;  // softmax warpgroups after the hand-off (128*104 + 256*200 <= 384*168)

template <int D>
struct WsLayout {
    static constexpr int kAtoms = D / 64;
    static constexpr int kTileBytes = kAtoms * kAtomBytes;
    static constexpr int kQ = 0;  // Q0, Q1
    static constexpr int kKV = kQ + 2 * kTileBytes;
    // epilogue staging: 32 rows x 64 bytes for each of the 8 softmax warps
    static constexpr int kStageBytes = 32 * 64;
    static constexpr int kStage = kKV + kStagesWs * kTileBytes;
    static constexpr int kBar = kStage + 8 * kStageBytes;
    // q_full[2], q_empty, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2], mma_done
    static constexpr int kNumBars = 2 + 1 + 2 * kStagesWs + 2 + 2 + 2 + 1;
    static constexpr int kFlags = kBar + kNumBars * 8;  // split flags [2 tiles][4 warps]
    static constexpr int kTmemSlot = kFlags + 32;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kUsed = kAbort + 4;
    // at least half of the SM's shared memory, so that one CTA (which takes all
    // 512 TMEM columns) is resident per SM
    static constexpr int kAlloc = (kUsed + 1024) > 118 * 1024 ? (kUsed + 1024) : 118 * 1024;
};

// Position in the K/V ring.
struct Ring {
    int s = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next() {
        if (++s == kStagesWs) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// Work item of round r for this CTA (snake order), or false past the end.
//   item_order 0: longest row block first over all heads, the heads of a block
//                 level adjacent (t -> qb = last - t / BHq, bh = t % BHq);
//   item_order 1: kv-group major: all blocks of one (batch, kv head) group
//                 before the next, longest first within the group, the group's
//                 query heads adjacent.
//
// A work unit is a whole item, or (attn_fwd_kv_split) one of n_parts key ranges of
// an item: units [0, n_whole) are the first n_whole items, and the items after them
// (the last round of a schedule of equal-length items) are cut into n_parts units
// each, so that the last round has more, shorter units.  part = -1 for a whole item;
// x numbers the cut items.
__device__ __forceinline__ bool ws_item(const Params &p, int r, int &bh, int &qb, int &part, int &x) {
    // 32-bit arithmetic throughout: the host guarantees n_units <= INT_MAX, and
    // 64-bit divisions here cost the softmax loop around them measurably.
    const unsigned G = gridDim.x;
    const unsigned c = (r & 1) ? (G - 1u - blockIdx.x) : blockIdx.x;
    const unsigned u = static_cast<unsigned>(r) * G + c;
    if (u >= static_cast<unsigned>(p.n_units)) return false;
    unsigned t = u;
    part = -1;
    x = 0;
    if (u >= static_cast<unsigned>(p.n_whole)) {
        const unsigned v = u - static_cast<unsigned>(p.n_whole), np = static_cast<unsigned>(p.n_parts);
        const unsigned xx = v / np;
        part = static_cast<int>(v - xx * np);
        x = static_cast<int>(xx);
        t = static_cast<unsigned>(p.n_whole) + xx;
    }
    const unsigned nqb = static_cast<unsigned>(p.n_qblocks);
    if (p.item_order == 0) {
        const unsigned bhq = static_cast<unsigned>(p.BHq);
        qb = static_cast<int>(nqb - 1u - t / bhq);
        bh = static_cast<int>(t % bhq);
    } else {
        const unsigned grp = static_cast<unsigned>(p.group), per_group = grp * nqb;
        const unsigned g = t / per_group, rr = t - g * per_group;
        qb = static_cast<int>(nqb - 1u - rr / grp);
        bh = static_cast<int>(g * grp + rr % grp);
    }
    return true;
}

// Key tiles visited by query tile i (0, 1) of block qb (never fewer for i = 1).
template <bool kCausal>
__device__ __forceinline__ int ws_tiles(const Params &p, int qb, int i) {
    if (!kCausal) return p.n_kv_tiles;
    return causal_kv_tiles(qb * 256 + 128 * i, p.Nq, p.causal_off, p.n_kv_tiles);
}

// Key tiles of a unit: query tile 0 visits [k0, e0), query tile 1 [k0, e1).  A whole
// item starts at 0; part s of n_parts of an item takes tiles [s n0 / np, (s+1) n0 / np)
// of query tile 0's n0, the same range for query tile 1, and the last part also query
// tile 1's tiles past n0.  The host keeps np small enough that every part starts with
// a tile that no row masks.
struct KeyRange {
    int k0, e0, e1;
};
template <bool kCausal>
__device__ __forceinline__ KeyRange ws_range(const Params &p, int qb, int part) {
    const int n0 = ws_tiles<kCausal>(p, qb, 0), n1 = ws_tiles<kCausal>(p, qb, 1);
    if (part < 0) return {0, n0, n1};
    const int k0 = part * n0 / p.n_parts, e0 = (part + 1) * n0 / p.n_parts;
    return {k0, e0, part == p.n_parts - 1 ? n1 : e0};
}

// Counts one arrival on a counter that keeps the launch's sequence number in its
// upper 24 bits, so that a value left by another launch (or never written) counts as
// no arrival.  Returns true for the arrival that brings the count to n, which also
// puts the counter back at zero arrivals of this launch (ready for a graph replay).
__device__ __forceinline__ bool arrive_last(unsigned int *ctr, unsigned int seq, int n) {
    const unsigned int tag = (seq & 0xFFFFFFu) << 8;
    unsigned int old = *reinterpret_cast<volatile unsigned int *>(ctr);
    for (;;) {
        const unsigned int cnt = ((old & ~0xFFu) == tag) ? (old & 0xFFu) : 0u;
        const bool last = cnt + 1u == static_cast<unsigned int>(n);
        const unsigned int prev = atomicCAS(ctr, old, last ? tag : (tag | (cnt + 1u)));
        if (prev == old) return last;
        old = prev;
    }
}

// tmQ, tmK, tmV: 3-D tensor maps (D, rows, heads) of Q [B*Hq, Nq, D] and
// K, V [B*Hkv, Nk, D], box 64 x 128 x 1 with the 128-byte swizzle; rows past
// the end of a head read as zeros.
template <int D, bool kBF16, bool kCausal>
__global__ void __launch_bounds__(kWsThreads, 1)
    attn_fwd_ws_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Params p) {
    using L = WsLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sQ = base + L::kQ, sKV = base + L::kKV;
    const uint32_t bar0 = base + L::kBar;
    auto q_full = [&](int i) { return bar0 + 8u * i; };
    const uint32_t q_empty = bar0 + 8u * 2;
    auto kv_full = [&](int s) { return bar0 + 8u * (3 + s); };
    auto kv_empty = [&](int s) { return bar0 + 8u * (3 + kStagesWs + s); };
    auto s_full = [&](int i) { return bar0 + 8u * (3 + 2 * kStagesWs + i); };
    auto p_full = [&](int i) { return bar0 + 8u * (5 + 2 * kStagesWs + i); };
    auto o_full = [&](int i) { return bar0 + 8u * (7 + 2 * kStagesWs + i); };
    const uint32_t mma_done = bar0 + 8u * (9 + 2 * kStagesWs);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbort);
    volatile uint32_t *flags = reinterpret_cast<volatile uint32_t *>(smem + L::kFlags);
    auto split_flag = [&](int i, int w) -> volatile uint32_t & { return flags[4 * i + w]; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 64) {
        // the producer's tensor maps: fetch the descriptors while the CTA sets up
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
    }
    if (threadIdx.x == 0) {
        // No global read on the way to the first copy: a CTA that starts after
        // another one of this launch gave up learns of it in its first bounded
        // wait (after a millisecond), like every other CTA.
        *abort_flag = 0;
        mbar_init(q_full(0), 1);
        mbar_init(q_full(1), 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < kStagesWs; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full(i), 1);
            mbar_init(p_full(i), 4);  // one arrival per softmax warp
            mbar_init(o_full(i), 1);
        }
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 1) {
        tmem_alloc(base + L::kTmemSlot, kWsTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
        regs_dec<kRegsLow>();
        if (warp == 2 && lane == 0) {
            // ---------------------------------------------------- TMA producer
            Ring ring;
            int items = 0;
            bool ok = true;
            // One tile = D/64 boxes of 128 rows x 64 columns (128 bytes, x = 64a:
            // a multiple of 16 bytes); the full barrier expects all of its bytes.
            auto load_tile_tma = [&](uint32_t dst, const CUtensorMap *tm, int row, int head, uint32_t bar) {
                mbar_arrive_expect_tx(bar, L::kTileBytes);
#pragma unroll
                for (int a = 0; a < L::kAtoms; ++a) tma_load_3d(dst + a * kAtomBytes, tm, 64 * a, row, head, bar);
            };
            // Full barriers: the first K tile of a unit completes its own stage's
            // barrier; V_j and K_{j+1} both complete V_j's, so the MMA warp waits once
            // per key tile.  Stages are then not armed once per lap, so each keeps its
            // own phase bit (fph), as the MMA warp does.
            uint32_t fph = 0, armed = 0;
            auto issue = [&](uint32_t dst, const CUtensorMap *tm, int row, int head, uint32_t bar) {
#pragma unroll
                for (int a = 0; a < L::kAtoms; ++a) tma_load_3d(dst + a * kAtomBytes, tm, 64 * a, row, head, bar);
            };
            auto load_k_first = [&](int row, int head) -> bool {
                if (!wait_bar(kv_empty(ring.s), ring.ph ^ 1u, p, abort_flag)) return false;
                mbar_arrive_expect_tx(kv_full(ring.s), L::kTileBytes);
                armed |= 1u << ring.s;
                fph ^= 1u << ring.s;
                issue(sKV + ring.s * L::kTileBytes, &tmK, row, head, kv_full(ring.s));
                ring.next();
                return true;
            };
            // V_j, and K_{j+1} when `pair`, on V_j's barrier
            auto load_vk = [&](int j, bool pair, int head) -> bool {
                const int vs = ring.s;
                if (!wait_bar(kv_empty(vs), ring.ph ^ 1u, p, abort_flag)) return false;
                Ring nr = ring;
                nr.next();
                if (pair && !wait_bar(kv_empty(nr.s), nr.ph ^ 1u, p, abort_flag)) return false;
                mbar_arrive_expect_tx(kv_full(vs), L::kTileBytes * (pair ? 2u : 1u));
                armed |= 1u << vs;
                fph ^= 1u << vs;
                issue(sKV + vs * L::kTileBytes, &tmV, j * kBN, head, kv_full(vs));
                ring.next();
                if (pair) {
                    issue(sKV + ring.s * L::kTileBytes, &tmK, (j + 1) * kBN, head, kv_full(vs));
                    ring.next();
                }
                return true;
            };
            int q_loads = 0;
            for (int r = 0; ok && static_cast<long long>(r) * gridDim.x < p.n_units; ++r) {
                int bh, qb, part, x;
                if (!ws_item(p, r, bh, qb, part, x)) continue;
                const int kvh = bh / p.group;
                const int q0 = qb * 256;
                const KeyRange kr = ws_range<kCausal>(p, qb, part);
                // The first K tile may land while the previous unit still runs; the Q
                // buffers are free once every S MMA of the previous unit is done.
                if (!(ok = load_k_first(kr.k0 * kBN, kvh))) break;
                if (!(ok = wait_bar(q_empty, (items & 1) ^ 1u, p, abort_flag))) break;
                if (!p.inject_stall) {
                    load_tile_tma(sQ, &tmQ, q0, bh, q_full(0));
                    load_tile_tma(sQ + L::kTileBytes, &tmQ, q0 + 128, bh, q_full(1));
                    ++q_loads;
                }
                ++items;
                // The next item's query rows are read from DRAM once; start bringing
                // them into L2 now, so that their load after this item hits L2.
                int nbh, nqb, npart, nx;
                if (ws_item(p, r + 1, nbh, nqb, npart, nx)) {
#pragma unroll
                    for (int a = 0; a < L::kAtoms; ++a) {
                        tma_prefetch_l2_3d(&tmQ, 64 * a, nqb * 256, nbh);
                        tma_prefetch_l2_3d(&tmQ, 64 * a, nqb * 256 + 128, nbh);
                    }
                }
                for (int j = kr.k0; j < kr.e1 && ok; ++j) ok = load_vk(j, j + 1 < kr.e1, kvh);
            }
            // Every copy has landed before the CTA exits (also after a timeout): wait for
            // the last armed phase of every stage's full barrier.
#pragma unroll
            for (int st = 0; st < kStagesWs; ++st)
                if ((armed >> st) & 1u) drain_bar(kv_full(st), ((fph >> st) & 1u) ^ 1u, p);
            if (q_loads > 0) {
                drain_bar(q_full(0), (q_loads - 1) & 1, p);
                drain_bar(q_full(1), (q_loads - 1) & 1, p);
            }
        } else if (warp == 0 && lane == 0) {
            // ---------------------------------------------------- MMA issuer
            constexpr uint32_t idesc_qk = idesc_f16_f32acc(kBF16, 128, kBN, false);
            constexpr uint32_t idesc_pv = idesc_f16_f32acc(kBF16, 128, D, true);
            Ring ring;
            uint32_t fph = 0;  // per-stage phase of the full barriers, as the producer arms them
            auto wait_full = [&](int st) -> bool {
                const bool r = wait_bar(kv_full(st), (fph >> st) & 1u, p, abort_flag);
                fph ^= 1u << st;
                return r;
            };
            uint32_t pcount[2] = {0, 0};
            int items = 0;
            bool ok = true;
            // Descriptors are built once per operand tile; stepping K by 16 moves
            // the start address by 32 B within a swizzle atom (+2 in the 16-byte
            // address field) and by one 16 KB atom every 4 steps (+1024).
            const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
            const uint64_t dkv0 = sdesc_sw128(sKV, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sKV, kAtomBytes, 1024);
            auto qk = [&](int i, int kstage) {
                uint64_t a = dq0 + static_cast<uint64_t>(i * (L::kTileBytes >> 4));
                uint64_t b = dkv0 + static_cast<uint64_t>(kstage * (L::kTileBytes >> 4));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (kk >> 2) * (kAtomBytes >> 4) + (kk & 3) * 2;
                    mma_f16_ss(tmem + 128u * i, a + off, b + off, idesc_qk, kk > 0);
                }
            };
            // O_i (+)= P_i V: P_hi from the first 64 columns of S_i, and, when a
            // softmax warp split this tile, P_lo from the next 64.  The P_lo pass
            // writes only the lanes of the warps that split: the other warps'
            // columns 64..127 still hold scores, which must not reach O.
            auto pv = [&](int i, int vstage, bool acc) {
                const uint64_t b0 = dv0 + static_cast<uint64_t>(vstage * (L::kTileBytes >> 4));
                const uint32_t ta = tmem + 128u * i, td = tmem + 256u + 128u * i;
                // lanes 32w..32w+31 belong to softmax warp w of the tile
                uint32_t lo_off[4];
                bool split = false;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const bool sw = split_flag(i, w) != 0;
                    lo_off[w] = sw ? 0u : ~0u;
                    split |= sw;
                }
                const int passes = split ? 2 : 1;
#pragma unroll 1
                for (int h = 0; h < passes; ++h) {
                    const uint32_t off[4] = {h ? lo_off[0] : 0u, h ? lo_off[1] : 0u, h ? lo_off[2] : 0u,
                                             h ? lo_off[3] : 0u};
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_f16_ts_lanes(td, ta + 64u * h + 8u * kk, b0 + kk * (2048 >> 4), idesc_pv, off,
                                         (acc || kk > 0 || h > 0) ? 1u : 0u);
                }
            };
            for (int r = 0; ok && static_cast<long long>(r) * gridDim.x < p.n_units; ++r) {
                int bh, qb, part, x;
                if (!ws_item(p, r, bh, qb, part, x)) continue;
                const KeyRange kr = ws_range<kCausal>(p, qb, part);
                const int k0 = kr.k0, n0 = kr.e0, n1 = kr.e1;  // tiles [k0, n0) and [k0, n1)
                const uint32_t ip = items & 1;
                if (!(ok = wait_bar(q_full(0), ip, p, abort_flag))) break;
                if (!(ok = wait_full(ring.s))) break;
                tc_fence_after();
                qk(0, ring.s);
                mma_commit(s_full(0));
                if (!(ok = wait_bar(q_full(1), ip, p, abort_flag))) break;
                tc_fence_after();
                qk(1, ring.s);
                mma_commit(s_full(1));
                mma_commit(kv_empty(ring.s));
                ring.next();
                for (int j = k0; j < n1; ++j) {
                    const int vs = ring.s;
                    if (!(ok = wait_full(vs))) break;  // V_j, and K_{j+1} if any
                    tc_fence_after();
                    ring.next();
                    if (j < n0) {
                        if (!(ok = wait_bar(p_full(0), pcount[0] & 1u, p, abort_flag))) break;
                        ++pcount[0];
                        tc_fence_after();
                        pv(0, vs, j > k0);
                        if (j == n0 - 1) mma_commit(o_full(0));
                    }
                    const bool more = j + 1 < n1;
                    const int ks = ring.s;
                    if (more) {
                        if (j + 1 < n0) {
                            qk(0, ks);
                            mma_commit(s_full(0));
                        }
                    }
                    if (!(ok = wait_bar(p_full(1), pcount[1] & 1u, p, abort_flag))) break;
                    ++pcount[1];
                    tc_fence_after();
                    pv(1, vs, j > k0);
                    if (j == n1 - 1) mma_commit(o_full(1));
                    mma_commit(kv_empty(vs));
                    if (more) {
                        qk(1, ks);
                        mma_commit(s_full(1));
                        mma_commit(kv_empty(ks));
                        ring.next();
                    }
                }
                if (!ok) break;
                mma_commit(q_empty);  // this item's S MMAs no longer read Q0, Q1
                ++items;
            }
            // TMEM and shared memory stay alive until every issued MMA is done.
            mma_commit(mma_done);
            drain_bar(mma_done, 0, p);
        }
        __syncwarp();
    } else {
        regs_inc<kRegsHigh>();
        // -------------------------------------------------------- softmax
        const int i = (warp - 4) >> 2;  // query tile of this warpgroup
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // row within the tile == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + 128u * i + lane_off;  // S_i, and P_i in its first 64 columns
        const uint32_t tO = tmem + 256u + 128u * i + lane_off;
        const float c = p.scale_log2;
        uint32_t scount = 0;
        int items = 0;
        bool ok = true;
        for (int rr = 0; ok && static_cast<long long>(rr) * gridDim.x < p.n_units; ++rr) {
            int bh, qb, part, x;
            if (!ws_item(p, rr, bh, qb, part, x)) continue;
            const KeyRange kr = ws_range<kCausal>(p, qb, part);
            const int jend = i ? kr.e1 : kr.e0;   // key tiles [kr.k0, jend) of this query tile
            const int row0 = qb * 256 + 128 * i;  // first query row of this tile
            // Causal: key tile j needs a mask unless its last key is visible to
            // row0, i.e. from tile (row0 + Nk - Nq + 1) / 128 on.
            const int first_masked = (row0 + p.causal_off + 1) / kBN;
            // m_ref: the max the probabilities are taken against (updated lazily);
            // m_top: the true running row max; l: running sum in units of 2^(m_ref*c).
            float m_ref = -INFINITY, m_top = -INFINITY, l = 0.f;
            for (int j = kr.k0; j < jend; ++j) {
                if (!__all_sync(0xffffffffu, wait_bar(s_full(i), scount & 1u, p, abort_flag))) {
                    ok = false;
                    break;
                }
                ++scount;
                tc_fence_after();
                __syncwarp();
                uint32_t s[128];
                const bool masked = kCausal ? (j >= first_masked) : ((j + 1) * kBN > p.Nk);
                if (!masked) {
                    // Interior tile: each load also returns the max of its 32 columns.
                    float mq[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld32_max(tS + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * q]), mq[q]);
                    tmem_ld_wait(s, mq);
                    m_top = fmaxf(m_top, fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3])));
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld32(tS + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * q]));
                    tmem_ld_wait(s);
                    if (kCausal) {  // tile on the causal boundary: row r keeps keys c <= lim
                        const int lim = r + row0 + p.causal_off - j * kBN;
#pragma unroll
                        for (int cc = 0; cc < 128; ++cc)
                            if (cc > lim) s[cc] = __float_as_uint(-INFINITY);
                    } else {  // ragged last tile: keys >= Nk are absent
                        const int lim = p.Nk - j * kBN;
#pragma unroll
                        for (int cc = 0; cc < 128; ++cc)
                            if (cc >= lim) s[cc] = __float_as_uint(-INFINITY);
                    }
                    float mx[8];  // eight independent chains of 3-input max
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx[k] = fmaxf(u2f(s[2 * k]), u2f(s[2 * k + 1]));
#pragma unroll
                    for (int cc = 16; cc < 128; cc += 16)
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            mx[k] = fmax3(mx[k], u2f(s[cc + 2 * k]), u2f(s[cc + 2 * k + 1]));
                    m_top = fmaxf(m_top, fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                               fmaxf(mx[6], mx[7])));
                }
                // Re-reference only when the max has grown by more than kRescaleLog2
                // (in log2 units) since the last reference; otherwise P may exceed 1.
                float alpha = 1.f;
                bool rescale = false;
                if (m_ref == -INFINITY) {
                    m_ref = m_top;  // first tile: the accumulator is still empty
                } else if ((m_top - m_ref) * c > kRescaleLog2) {
                    alpha = ex2_approx((m_ref - m_top) * c);
                    m_ref = m_top;
                    rescale = true;
                }
                const float2 c2 = make_float2(c, c);
                const float2 nmc2 = make_float2(-m_ref * c, -m_ref * c);
                float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int cc = 0; cc < 128; cc += 2) {
                    float2 e = ffma2(make_float2(u2f(s[cc]), u2f(s[cc + 1])), c2, nmc2);
                    e.x = ex2_approx(e.x);
                    e.y = ex2_approx(e.y);
                    acc[(cc >> 1) & 1] = fadd2(acc[(cc >> 1) & 1], e);
                    s[cc] = __float_as_uint(e.x);
                    s[cc + 1] = __float_as_uint(e.y);
                }
                const float2 sum2 = fadd2(acc[0], acc[1]);
                l = l * alpha + (sum2.x + sum2.y);
                // Split P = P_hi + P_lo for a warp's 32 rows when one of them has its
                // weight on few keys: its running sum relative to its largest weight
                // 2^((m_top - m_ref) c) is below kSplitL.
                const bool need = l * ex2_approx((m_ref - m_top) * c) < kSplitL;
                // No warpgroup-wide agreement: each warp decides for its 32 rows, and
                // the MMA warp's P_lo pass writes only the lanes of warps that split.
                const bool split = __any_sync(0xffffffffu, need);
                if (lane == 0) split_flag(i, wq) = split ? 1u : 0u;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pk[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) pk[t] = pack2<kBF16>(u2f(s[32 * q + 2 * t]), u2f(s[32 * q + 2 * t + 1]));
                    tmem_st16(tS + 16 * q, pk);
                    if (split) {
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const float2 h = unpack2<kBF16>(pk[t]);
                            pk[t] = pack2<kBF16>(u2f(s[32 * q + 2 * t]) - h.x, u2f(s[32 * q + 2 * t + 1]) - h.y);
                        }
                        tmem_st16(tS + 64 + 16 * q, pk);
                    }
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // O_i holds P_i V_{j-1} already (covered by the S_i(j) commit).
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
                }
                tmem_st_wait();
                tc_fence_before();
                // one arrival per warp once every lane's TMEM stores are done: 4 instead
                // of 128 atomics on the barrier the MMA warp is waiting for
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(i));
            }
            if (!ok) break;
            // ---------------------------------------------------- epilogue
            if (!__all_sync(0xffffffffu, wait_bar(o_full(i), items & 1, p, abort_flag))) {
                ok = false;
                break;
            }
            ++items;
            tc_fence_after();
            __syncwarp();
            const int row = row0 + r;
            // 32 columns at a time: each thread puts its row's 64 bytes into the
            // warp's staging rows (16-byte chunk c of row t at chunk c ^ ((t >> 1) & 3),
            // so neither the writes nor the reads conflict on banks), then lanes
            // 4k..4k+3 write the 64 bytes of one row: 8 whole row segments per store.
            const uint32_t stage = base + L::kStage + static_cast<uint32_t>(warp - 4) * L::kStageBytes;
            const int rd_row = lane >> 2, rd_c = lane & 3;  // + 8 s for s = 0..3
            uint8_t *ohead = static_cast<uint8_t *>(p.o) + static_cast<size_t>(bh) * p.Nq * (D * 2);
            const int wrow0 = row0 + wq * 32;  // first row of this warp
            auto store_cols = [&](int q, const uint32_t (&w)[16]) {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    st_shared_v4(stage + lane * 64 + ((v ^ ((lane >> 1) & 3)) << 4), w[4 * v], w[4 * v + 1],
                                 w[4 * v + 2], w[4 * v + 3]);
                __syncwarp();
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const int t = 8 * s4 + rd_row;  // row within the warp
                    const uint4 xv = ld_shared_v4(stage + t * 64 + ((rd_c ^ ((t >> 1) & 3)) << 4));
                    if (wrow0 + t < p.Nq)
                        st_global_v4(ohead + static_cast<size_t>(wrow0 + t) * (D * 2) + q * 64 + rd_c * 16, xv.x,
                                     xv.y, xv.z, xv.w);
                }
                __syncwarp();
            };
            if (part < 0) {
                const float inv_l = 1.f / l;  // l is in units of 2^(m_ref * c)
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * q, o);
                    tmem_ld_wait(o);
                    uint32_t w[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t)
                        w[t] = pack2<kBF16>(u2f(o[2 * t]) * inv_l, u2f(o[2 * t + 1]) * inv_l);
                    store_cols(q, w);
                }
                if (p.lse != nullptr && row < p.Nq)
                    p.lse[static_cast<size_t>(bh) * p.Nq + row] = (m_ref * c + log2f(l)) * 0.6931471805599453f;
            } else {
                // One key range of a cut item: this warp's rows of O / l (fp32) and their
                // log-sum-exp go to the workspace; the warp that brings the last of the
                // n_parts pieces of these rows merges them, with weights
                // exp(lse_s - lse), lse = log sum_s exp(lse_s) (the online-softmax
                // update of page "从零开始写Qwen3", deepseek.csdn.net/6a3201f8...,
                // section "在线softmax", applied across CTAs).
                // Pieces are stored column-major per (cut item, part, tile): element (d, r)
                // at d * 128 + r, so that a warp's row-per-thread accesses are 128
                // contiguous bytes.
                const size_t tile_stride = static_cast<size_t>(2) * 128;  // lse entries per part
                const size_t lse0 = (static_cast<size_t>(x) * p.n_parts * 2 + i) * 128 + r;  // part 0
                const float *po0 = p.part_o + (static_cast<size_t>(x) * p.n_parts * 2 + i) * 128 * D + r;
                const size_t part_stride = tile_stride * D;  // floats between parts' pieces
                float *po = p.part_o + ((static_cast<size_t>(x) * p.n_parts + part) * 2 + i) * 128 * D + r;
                const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * q, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int t = 0; t < 32; ++t) po[(32 * q + t) * 128] = u2f(o[t]) * inv_l;
                }
                p.part_lse[lse0 + part * tile_stride] = l > 0.f ? (m_ref * c + log2f(l)) * 0.6931471805599453f : -INFINITY;
                __threadfence();  // this warp's pieces are visible before its arrival counts
                __syncwarp();
                unsigned int last = 0;
                if (lane == 0)
                    last = arrive_last(p.part_count + (static_cast<size_t>(x) * 2 + i) * 4 + wq, p.seq, p.n_parts)
                               ? 1u : 0u;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();  // every piece arrived before this: read them from L2
                    // weights exp(lse_s - lse) once, in registers (kMaxParts bounds the parts)
                    float wgt[kMaxPartsWs];
                    float mx = -INFINITY;
#pragma unroll
                    for (int sp = 0; sp < kMaxPartsWs; ++sp) {
                        wgt[sp] = sp < p.n_parts ? __ldcg(p.part_lse + lse0 + sp * tile_stride) : -INFINITY;
                        mx = fmaxf(mx, wgt[sp]);
                    }
                    float sum = 0.f;
#pragma unroll
                    for (int sp = 0; sp < kMaxPartsWs; ++sp) {
                        wgt[sp] = wgt[sp] == -INFINITY ? 0.f : expf(wgt[sp] - mx);
                        sum += wgt[sp];
                    }
                    const float lse_all = mx + logf(sum), inv_sum = 1.f / sum;
#pragma unroll 1
                    for (int q = 0; q < D / 32; ++q) {
                        float acc[32];
#pragma unroll
                        for (int t = 0; t < 32; ++t) acc[t] = 0.f;
#pragma unroll
                        for (int sp = 0; sp < kMaxPartsWs; ++sp) {
                            if (sp < p.n_parts) {
                                const float *src = po0 + sp * part_stride + static_cast<size_t>(32 * q) * 128;
                                const float ww = wgt[sp] * inv_sum;
#pragma unroll
                                for (int t = 0; t < 32; ++t) acc[t] += ww * __ldcg(src + t * 128);
                            }
                        }
                        uint32_t w[16];
#pragma unroll
                        for (int t = 0; t < 16; ++t) w[t] = pack2<kBF16>(acc[2 * t], acc[2 * t + 1]);
                        store_cols(q, w);
                    }
                    if (p.lse != nullptr && row < p.Nq) p.lse[static_cast<size_t>(bh) * p.Nq + row] = lse_all;
                }
            }
            // O_i is read; the next item's first P_i V MMA waits for this warpgroup's p_full.
            tc_fence_before();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kWsTmemCols);
    }
}

}  // namespace gqa
