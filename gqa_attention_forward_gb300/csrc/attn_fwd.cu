// Fused grouped-query attention forward for GB300 (sm_103a).
//
// O = softmax(mask(Q K^T * scale)) V with the online-softmax update of the
// page "从零开始写Qwen3" (deepseek.csdn.net/6a3201f8..., sections "在线softmax"
// and "FlashAttention"): each CTA owns one 128-row query tile, streams the
// key/value tiles it needs, keeps a running row max m and row sum l in fp32,
// rescales the output accumulator when m grows and normalises once at the
// end.  The score matrix never leaves the SM.
//
// Hardware mapping:
//   * warps 2-3: loaders.  Q once; then K_j, V_j alternately, with 16-byte
//     cp.async into a kStages-deep ring of 128-byte-swizzled shared-memory
//     tiles guarded by full / empty mbarriers.
//   * warp 1 (one lane): tcgen05 MMA issuer.  S = Q K_j^T into TMEM columns
//     [0, 128); O += P V_j into TMEM columns [128, 128 + D).  Completion is
//     signalled with tcgen05.commit onto mbarriers.
//   * warps 4-7: softmax.  Thread t owns query row t (TMEM lane t): it reads
//     its 128 scores with tcgen05.ld, applies the causal / tail mask, updates
//     m and l, writes P (rounded to the input type) into shared memory in the
//     UMMA K-major swizzled layout, and rescales its O row in TMEM when m
//     grows.  Finally it normalises O, stores it and the log-sum-exp.
//
// Causal tiles above the diagonal are never visited and only the diagonal
// tile is masked (page "从零开始写Qwen3", deepseek.csdn.net/6a31faef..., sections
// "改进2-KV只读取下三角" and "改进3-两阶段计算").  The exponent uses exp2 with
// scale*log2(e) folded into one FMA (same page, "优化点6-使用exp2而不是exp").
// Query tiles of one (batch, head) are adjacent in launch order so their K/V
// reads hit L2 (same page, "改进1-使用正确的grid").
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "attn_fwd_decode.cuh"
#include "attn_fwd_ws.cuh"
#include "gqa_attn.h"
#include "kernel_common.cuh"
#include "sm103_ptx.cuh"

namespace gqa {

constexpr int kStages = 4;     // K/V tiles in flight
constexpr int kThreads = 256;  // warps 2-3 loaders, warp 1 MMA, warps 4..7 softmax
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kTmemO = 128;  // first TMEM column of the O accumulator

template <int D>
struct Layout {
    static constexpr int kAtoms = D / 64;           // 64 halfs = one 128-byte swizzle row
    static constexpr int kTileBytes = kAtoms * kAtomBytes;
    static constexpr int kQ = 0;
    static constexpr int kKV = kQ + kTileBytes;
    static constexpr int kP = kKV + kStages * kTileBytes;
    static constexpr int kPBytes = 2 * kAtomBytes;  // P tile: 128 x 128 halfs
    static constexpr int kBar = kP + kPBytes;
    static constexpr int kNumBars = 1 + 2 * kStages + 4;
    static constexpr int kTmemSlot = kBar + kNumBars * 8;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kUsed = kAbort + 4;
    static constexpr int kAlloc = kUsed + 1024;  // slack to align the base to 1024 B
};

template <int D, bool kBF16, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const Params p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const uint32_t sQ = base + L::kQ, sKV = base + L::kKV, sP = base + L::kP;
    const uint32_t bar0 = base + L::kBar;
    const uint32_t q_full = bar0;
    auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto kv_empty = [&](int s) { return bar0 + 8u * (1 + kStages + s); };
    const uint32_t s_full = bar0 + 8u * (1 + 2 * kStages);
    const uint32_t p_full = bar0 + 8u * (2 + 2 * kStages);
    const uint32_t o_full = bar0 + 8u * (3 + 2 * kStages);
    const uint32_t mma_done = bar0 + 8u * (4 + 2 * kStages);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kAbort);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Query tiles of one (b, hq) are adjacent; within it the longest causal
    // rows come first.
    const int q_tile = p.n_qtiles - 1 - static_cast<int>(blockIdx.x % p.n_qtiles);
    const int bh = static_cast<int>(blockIdx.x / p.n_qtiles);  // b*Hq + hq
    const int kvh = bh / p.group;                               // b*Hkv + hq/(Hq/Hkv)
    const int q0 = q_tile * kBM;
    const int n_kv = kCausal ? causal_kv_tiles(q0, p.Nq, p.causal_off, p.n_kv_tiles) : p.n_kv_tiles;

    if (threadIdx.x == 0) {
        *abort_flag = (*reinterpret_cast<volatile unsigned int *>(&g_abort_seq) == p.seq) ? 1 : 0;
        mbar_init(q_full, kLoaderThreads);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(kv_full(s), kLoaderThreads);
            mbar_init(kv_empty(s), 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_full, kBM);
        mbar_init(o_full, 1);
        mbar_init(mma_done, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (*abort_flag) return;  // another CTA of this launch already gave up
    if (warp == 1) {
        tmem_alloc(base + L::kTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 2 && warp < 4) {
        // ---------------------------------------------------- loaders (warps 2, 3)
        const int ltid = threadIdx.x - 64;
        const size_t kv_head_bytes = static_cast<size_t>(p.Nk) * D * 2;
        const uint8_t *kh = p.k + static_cast<size_t>(kvh) * kv_head_bytes;
        const uint8_t *vh = p.v + static_cast<size_t>(kvh) * kv_head_bytes;
        LoadSignal sig;
        if (!p.inject_stall) {
            load_tile<D>(sQ, p.q + static_cast<size_t>(bh) * p.Nq * D * 2, q0, p.Nq, ltid);
            sig.commit(q_full);
        }
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int j = 0; j < n_kv && ok; ++j) {
            for (int t = 0; t < 2; ++t) {
                if (!wait_bar(kv_empty(stage), phase ^ 1u, p, abort_flag)) {
                    ok = false;
                    break;
                }
                load_tile<D>(sKV + stage * L::kTileBytes, t ? vh : kh, j * kBN, p.Nk, ltid);
                sig.commit(kv_full(stage));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Announce the last group; every copy has landed before the CTA exits.
        sig.announce<true>();
        cp_async_wait<0>();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            constexpr uint32_t idesc_qk = idesc_f16_f32acc(kBF16, kBM, kBN, false);
            constexpr uint32_t idesc_pv = idesc_f16_f32acc(kBF16, kBM, D, true);
            const uint32_t tS = tmem, tO = tmem + kTmemO;
            bool ok = wait_bar(q_full, 0, p, abort_flag);
            tc_fence_after();
            int stage = 0;
            uint32_t phase = 0;
            for (int j = 0; j < n_kv && ok; ++j) {
                // S = Q K_j^T   (A = Q, B = K: both K-major, 128-byte swizzle)
                if (!wait_bar(kv_full(stage), phase, p, abort_flag)) break;
                tc_fence_after();
                const uint32_t sK = sKV + stage * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
                    mma_f16_ss(tS, sdesc_sw128(sQ + koff, 16, 1024), sdesc_sw128(sK + koff, 16, 1024),
                               idesc_qk, kk > 0);
                }
                mma_commit(s_full);
                mma_commit(kv_empty(stage));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
                // O += P V_j   (A = P: K-major; B = V: MN-major, 64-wide chunks
                // of D at LBO = one atom, 8-row groups of keys at SBO = 1024 B)
                if (!wait_bar(p_full, j & 1, p, abort_flag)) break;
                tc_fence_after();
                if (!wait_bar(kv_full(stage), phase, p, abort_flag)) break;
                tc_fence_after();
                const uint32_t sV = sKV + stage * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint32_t poff = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
                    mma_f16_ss(tO, sdesc_sw128(sP + poff, 16, 1024),
                               sdesc_sw128(sV + kk * 2048, kAtomBytes, 1024), idesc_pv,
                               (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(o_full);
                mma_commit(kv_empty(stage));
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // TMEM and shared memory stay alive until every issued MMA is done.
            mma_commit(mma_done);
            drain_bar(mma_done, 0, p);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------------------------------------------- softmax rows
        const int wq = warp & 3;
        const int r = wq * 32 + lane;  // row within the tile == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + lane_off, tO = tmem + kTmemO + lane_off;
        const float c = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        const uint32_t prow = sP + (r >> 3) * 1024 + (r & 7) * 128;
        for (int j = 0; j < n_kv; ++j) {
            if (!__all_sync(0xffffffffu, wait_bar(s_full, j & 1, p, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            __syncwarp();
            uint32_t s[128];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                tmem_ld32(tS + 32 * q, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * q]));
            tmem_ld_wait(s);
            const int kv0 = j * kBN;
            if (kCausal) {
                const int lim0 = q0 + p.causal_off - kv0;  // row r sees keys c <= r + lim0 here
                if (lim0 < kBN - 1) {
                    const int lim = r + lim0;
#pragma unroll
                    for (int cc = 0; cc < 128; ++cc)
                        if (cc > lim) s[cc] = __float_as_uint(-INFINITY);
                }
            } else if (kv0 + kBN > p.Nk) {  // ragged last tile: keys >= Nk are absent
                const int lim = p.Nk - kv0;
#pragma unroll
                for (int cc = 0; cc < 128; ++cc)
                    if (cc >= lim) s[cc] = __float_as_uint(-INFINITY);
            }
            float mt = u2f(s[0]);
#pragma unroll
            for (int cc = 1; cc < 128; ++cc) mt = fmaxf(mt, u2f(s[cc]));
            const float m_new = fmaxf(m, mt);
            const float alpha = ex2_approx((m - m_new) * c);  // 0 on the first tile
            if (j > 0) {
                // P V_{j-1} must be done: it reads the P buffer and writes O.
                if (!__all_sync(0xffffffffu, wait_bar(o_full, (j - 1) & 1, p, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, m_new > m)) {
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32 * q, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(u2f(o[i]) * alpha);
                        tmem_st32(tO + 32 * q, o);
                    }
                    tmem_st_wait();
                }
            }
            m = m_new;
            l *= alpha;
            const float mc = m * c;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                float e[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    e[t] = ex2_approx(fmaf(u2f(s[ch * 8 + t]), c, -mc));
                    l += e[t];
                }
                const uint32_t addr = prow + (ch >> 3) * kAtomBytes + (((ch & 7) ^ (r & 7)) << 4);
                st_shared_v4(addr, pack2<kBF16>(e[0], e[1]), pack2<kBF16>(e[2], e[3]),
                             pack2<kBF16>(e[4], e[5]), pack2<kBF16>(e[6], e[7]));
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        // ---------------------------------------------------- epilogue
        if (ok && __all_sync(0xffffffffu, wait_bar(o_full, (n_kv - 1) & 1, p, abort_flag))) {
            tc_fence_after();
            __syncwarp();
            const int row = q0 + r;
            const float inv_l = 1.f / l;
            uint8_t *orow = static_cast<uint8_t *>(p.o) + (static_cast<size_t>(bh) * p.Nq + row) * (D * 2);
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t o[32];
                tmem_ld32(tO + 32 * q, o);
                tmem_ld_wait(o);
                if (row < p.Nq) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack2<kBF16>(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        st_global_v4(orow + q * 64 + v * 16, w[4 * v], w[4 * v + 1], w[4 * v + 2],
                                     w[4 * v + 3]);
                }
            }
            if (p.lse != nullptr && row < p.Nq)
                p.lse[static_cast<size_t>(bh) * p.Nq + row] = (m * c + log2f(l)) * 0.6931471805599453f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace gqa

// =================================================================== host
namespace {

thread_local char t_last_cuda_error[256] = "";

// Scratch of attn_fwd_decode_noalloc: part of this module's device memory, so
// no call allocates it.  Its address is looked up once per device.
static __device__ __align__(256) float g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES / sizeof(float)];
std::atomic<unsigned int> g_launch_seq{1};
std::atomic<unsigned long long> g_timeout_ns{4000000000ull};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_force_splits{0};  // test hook: key splits of the packed kernel (0 = chosen)

void note_cuda_error(cudaError_t e, const char *where) {
    std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s: %s", where, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_dev_state[kMaxDevices];      // 0 unknown, 1 sm_103, -1 other
int g_dev_sms[kMaxDevices];        // multiprocessor count
unsigned g_dev_smem_set[kMaxDevices];  // bit per kernel instantiation
void *g_dev_scratch[kMaxDevices];      // address of g_noalloc_scratch on the device

// Streams and events of attn_fwd_host, created on the first call on a device and
// kept for the life of the process (no memory is allocated per call).
constexpr int kMaxChunks = 8;
struct HostPipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kMaxChunks] = {}, out[kMaxChunks] = {};
    bool ready = false;
};
std::mutex g_pipe_mu;  // serialises the enqueueing of attn_fwd_host calls
HostPipe g_pipe[kMaxDevices];
std::atomic<int> g_kernel_choice{0};   // 0 persistent warp-specialised, 1 one CTA per query tile
std::atomic<int> g_item_order{0};      // work-item order of the persistent kernel (0 or 1)

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Tensor map of a [heads, rows, D] array of 2-byte elements viewed as the 3-D
// tensor (D, rows, heads): a box of 64 columns x 128 rows x 1 head lands in
// shared memory in the 128-byte swizzle, and rows past `rows` read as zeros,
// so a box never reaches into the next head.
bool encode_rows_map(CUtensorMap *map, const void *base, bool bf16, int D, int rows, long long heads) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(heads)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(rows) * D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

attn_status_t check_device(int *dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaGetDevice");
        return ATTN_ERR_NODEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NODEVICE;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_dev_state[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            note_cuda_error(cudaGetLastError(), "cudaDeviceGetAttribute");
            return ATTN_ERR_NODEVICE;
        }
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        g_dev_sms[dev] = sms > 0 ? sms : 1;
        g_dev_state[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    *dev_out = dev;
    return g_dev_state[dev] == 1 ? ATTN_OK : ATTN_ERR_NODEVICE;
}

// The first launch of a kernel instantiation on a device raises its dynamic
// shared-memory limit (bit `kid` of the device's mask records it).
template <typename K>
attn_status_t set_smem_limit(int dev, int kid, K kern, int smem) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!(g_dev_smem_set[dev] >> kid & 1u)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            note_cuda_error(e, "cudaFuncSetAttribute");
            return ATTN_ERR_LAUNCH;
        }
        g_dev_smem_set[dev] |= 1u << kid;
    }
    return ATTN_OK;
}

template <int D, bool BF16, bool CAUSAL>
attn_status_t launch(int dev, int kid, const gqa::Params &prm, cudaStream_t stream) {
    if (g_kernel_choice.load() == 0) {
        // persistent kernel: one CTA per SM (or per item when there are fewer), TMA loads
        auto kern = gqa::attn_fwd_ws_kernel<D, BF16, CAUSAL>;
        constexpr int smem = gqa::WsLayout<D>::kAlloc;
        if (attn_status_t st = set_smem_limit(dev, kid + 8, kern, smem); st != ATTN_OK) return st;
        CUtensorMap tq, tk, tv;
        const long long BHkv = prm.BHq / prm.group;
        if (!encode_rows_map(&tq, prm.q, BF16, D, prm.Nq, prm.BHq) ||
            !encode_rows_map(&tk, prm.k, BF16, D, prm.Nk, BHkv) ||
            !encode_rows_map(&tv, prm.v, BF16, D, prm.Nk, BHkv)) {
            std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "cuTensorMapEncodeTiled failed");
            return ATTN_ERR_LAUNCH;
        }
        const int sms = g_dev_sms[dev];
        const unsigned grid = static_cast<unsigned>(prm.n_units < sms ? prm.n_units : sms);
        kern<<<grid, gqa::kWsThreads, smem, stream>>>(tq, tk, tv, prm);
    } else {
        auto kern = gqa::attn_fwd_kernel<D, BF16, CAUSAL>;
        constexpr int smem = gqa::Layout<D>::kAlloc;
        if (attn_status_t st = set_smem_limit(dev, kid, kern, smem); st != ATTN_OK) return st;
        const unsigned grid = static_cast<unsigned>(static_cast<long long>(prm.BHq) * prm.n_qtiles);
        kern<<<grid, gqa::kThreads, smem, stream>>>(prm);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        note_cuda_error(e, "kernel launch");
        return ATTN_ERR_LAUNCH;
    }
    return ATTN_OK;
}

// Packed short-query kernel (one CTA per kv head, row tile and key split), then
// the merge of the splits when there are several.
template <int D, bool BF16, bool CAUSAL>
attn_status_t launch_decode(int dev, int kid, const gqa::Params &prm, cudaStream_t stream) {
    auto kern = gqa::attn_fwd_decode_kernel<D, BF16, CAUSAL>;
    constexpr int smem = gqa::DecLayout<D>::kAlloc;
    if (attn_status_t st = set_smem_limit(dev, 16 + kid, kern, smem); st != ATTN_OK) return st;
    // Both kernels wait inside (griddepcontrol.wait) for the grid before them
    // before touching global memory, so they are launched as programmatic
    // dependents: their launch and set-up overlap the previous kernel's tail.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(prm.BHq / prm.group) * prm.n_mtiles *
                                             prm.n_splits));
    cfg.blockDim = dim3(gqa::kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Q as [B*Hkv, G*Nq, D]: the packed rows of one kv head are one block
    CUtensorMap tq, tk, tv;
    const long long BHkv = prm.BHq / prm.group;
    if (!encode_rows_map(&tq, prm.q, BF16, D, prm.rows_per_kv, BHkv) ||
        !encode_rows_map(&tk, prm.k, BF16, D, prm.Nk, BHkv) || !encode_rows_map(&tv, prm.v, BF16, D, prm.Nk, BHkv)) {
        std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "cuTensorMapEncodeTiled failed");
        return ATTN_ERR_LAUNCH;
    }
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, prm);
    if (e == cudaSuccess && prm.n_splits > 1) {
        cfg.gridDim = dim3(static_cast<unsigned>((prm.total_rows + 3) / 4));
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, gqa::attn_combine_kernel<D, BF16>, prm);
    }
    if (e != cudaSuccess) {
        note_cuda_error(e, "kernel launch");
        return ATTN_ERR_LAUNCH;
    }
    return ATTN_OK;
}

// Argument checks shared by the entry points and the fields of Params they
// fill.  *empty is set for a problem with nothing to compute (B, Hq or Nq 0).
attn_status_t prepare(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                      int Hkv, int Nq, int Nk, int D, float scale, int causal, attn_dtype_t dtype,
                      gqa::Params &prm, int &dev, bool &empty) {
    empty = false;
    if (B < 0 || Hq < 0 || Nq < 0 || Nk < 0 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_SHAPE;
    if (!(std::isfinite(scale) && scale > 0.f)) return ATTN_ERR_SHAPE;
    if (D != 64 && D != 128) return ATTN_ERR_HEADDIM;
    if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
    if (B == 0 || Hq == 0 || Nq == 0) {
        empty = true;
        return ATTN_OK;
    }
    if (Nk == 0 || (causal && Nq > Nk)) return ATTN_ERR_SHAPE;  // a query row would see no key
    if (!q || !k || !v || !o) return ATTN_ERR_NULL;
    auto misaligned = [](const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0; };
    if (misaligned(q, 16) || misaligned(k, 16) || misaligned(v, 16) || misaligned(o, 16) ||
        (lse && misaligned(lse, 4)))
        return ATTN_ERR_ALIGN;
    const long long BHq = static_cast<long long>(B) * Hq;
    const int n_qtiles = (Nq + gqa::kBM - 1) / gqa::kBM;
    if (BHq * n_qtiles > INT_MAX || BHq * Nq > INT_MAX) return ATTN_ERR_SHAPE;

    attn_status_t st = check_device(&dev);
    if (st != ATTN_OK) return st;

    prm = gqa::Params{};
    prm.q = static_cast<const uint8_t *>(q);
    prm.k = static_cast<const uint8_t *>(k);
    prm.v = static_cast<const uint8_t *>(v);
    prm.o = o;
    prm.lse = lse;
    prm.Nq = Nq;
    prm.Nk = Nk;
    prm.causal_off = Nk - Nq;
    prm.group = Hq / Hkv;
    prm.n_qtiles = n_qtiles;
    prm.n_kv_tiles = (Nk + gqa::kBN - 1) / gqa::kBN;
    prm.BHq = static_cast<int>(BHq);
    prm.n_qblocks = (Nq + 255) / 256;
    prm.n_items = static_cast<int>(BHq * prm.n_qblocks);
    prm.n_units = prm.n_items;  // whole items only unless a split plan says otherwise
    prm.n_whole = prm.n_items;
    prm.n_parts = 1;
    prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    prm.seq = g_launch_seq.fetch_add(1);
    prm.timeout_ns = g_timeout_ns.load();
    prm.inject_stall = g_inject_stall.load();
    prm.item_order = g_item_order.load();
    prm.rows_per_kv = prm.group * Nq;
    prm.n_mtiles = (prm.rows_per_kv + gqa::kBM - 1) / gqa::kBM;
    prm.total_rows = static_cast<int>(BHq * Nq);
    prm.n_splits = 1;
    prm.split_tiles = prm.n_kv_tiles;
    return ATTN_OK;
}

// Key splits of the packed kernel: enough (kv head, row tile, split) CTAs for one
// per SM, at least one key tile per split, and no more splits than `cap` (the
// workspace's capacity in splits).  Fills n_splits and split_tiles.
void plan_splits(gqa::Params &prm, int sms, long long cap) {
    const long long tiles = static_cast<long long>(prm.BHq / prm.group) * prm.n_mtiles;
    long long want = tiles >= sms ? 1 : sms / tiles;
    if (const int forced = g_force_splits.load(); forced > 0) want = forced;
    if (want > prm.n_kv_tiles) want = prm.n_kv_tiles;
    if (want > cap) want = cap;
    if (want < 1) want = 1;
    prm.split_tiles = static_cast<int>((prm.n_kv_tiles + want - 1) / want);
    prm.n_splits = (prm.n_kv_tiles + prm.split_tiles - 1) / prm.split_tiles;
}

size_t split_bytes(const gqa::Params &prm, int D) {
    return static_cast<size_t>(prm.total_rows) * (D + 1) * sizeof(float);
}

// Launches the packed kernel (and the merge) with the splits planned in prm;
// workspace holds the partial results when there are several.
attn_status_t run_decode(gqa::Params &prm, int dev, int D, attn_dtype_t dtype, int causal, void *workspace,
                         cudaStream_t s) {
    if (prm.n_splits > 1) {
        prm.ws_o = static_cast<float *>(workspace);
        prm.ws_lse = prm.ws_o + static_cast<size_t>(prm.n_splits) * prm.total_rows * D;
    }
    const bool bf16 = dtype == ATTN_BF16;
    const int kid = (D == 128 ? 4 : 0) + (bf16 ? 2 : 0) + (causal ? 1 : 0);
    switch (kid) {
        case 0: return launch_decode<64, false, false>(dev, kid, prm, s);
        case 1: return launch_decode<64, false, true>(dev, kid, prm, s);
        case 2: return launch_decode<64, true, false>(dev, kid, prm, s);
        case 3: return launch_decode<64, true, true>(dev, kid, prm, s);
        case 4: return launch_decode<128, false, false>(dev, kid, prm, s);
        case 5: return launch_decode<128, false, true>(dev, kid, prm, s);
        case 6: return launch_decode<128, true, false>(dev, kid, prm, s);
        default: return launch_decode<128, true, true>(dev, kid, prm, s);
    }
}

// Key-split plan of the persistent kernel (attn_fwd_kv_split).  Items are dealt in
// rounds of `grid` = min(items, SMs); when the last round holds at most half a round,
// each of its R items is cut into n_parts = SMs / R key ranges (at most kMaxParts), so
// that round runs more, shorter units.  Every range must start with a key tile that no
// row of the item masks: n_parts is at most the number of such tiles of the item
// (causal: tiles before the first one masked for the item's first query tile;
// non-causal: the full tiles).  Fills n_whole / n_parts / n_units; returns the number
// of cut items (0: no split).
constexpr int kMaxParts = gqa::kMaxPartsWs;
int plan_last_round(gqa::Params &prm, int sms, int causal) {
    const long long G = prm.n_items < sms ? prm.n_items : sms;
    const long long rounds = (prm.n_items + G - 1) / G;
    const long long R = prm.n_items - (rounds - 1) * G;  // items of the last round
    if (R <= 0 || 2 * R > sms) return 0;
    int np = static_cast<int>(sms / R);
    if (np > kMaxParts) np = kMaxParts;
    // The cut items are the last R of the item order.  Part s of np takes the key
    // tiles [s n0 / np, (s+1) n0 / np) of the item's first query tile (n0 of them):
    // np is lowered until, for every cut item, each part has a tile and starts before
    // the first tile that a row of the item masks.
    auto fits = [&](int parts) {
        for (long long t = prm.n_items - R; t < prm.n_items; ++t) {
            int qb;
            if (prm.item_order == 0) {
                qb = prm.n_qblocks - 1 - static_cast<int>(t / prm.BHq);
            } else {
                const long long per_group = static_cast<long long>(prm.group) * prm.n_qblocks;
                qb = prm.n_qblocks - 1 - static_cast<int>((t % per_group) / prm.group);
            }
            const int row0 = qb * 256;
            int n0 = prm.n_kv_tiles, first_masked = prm.Nk / gqa::kBN;
            if (causal) {
                const int last_row = row0 + gqa::kBM - 1 < prm.Nq - 1 ? row0 + gqa::kBM - 1 : prm.Nq - 1;
                n0 = (last_row + prm.causal_off) / gqa::kBN + 1;
                if (n0 > prm.n_kv_tiles) n0 = prm.n_kv_tiles;
                first_masked = (row0 + prm.causal_off + 1) / gqa::kBN;
            }
            if (n0 < parts || static_cast<long long>(parts - 1) * n0 / parts >= first_masked) return false;
        }
        return true;
    };
    while (np >= 2 && !fits(np)) --np;
    if (np < 2) return 0;
    prm.n_parts = np;
    prm.n_whole = static_cast<int>(prm.n_items - R);
    prm.n_units = static_cast<int>(prm.n_whole + R * np);
    return static_cast<int>(R);
}

// Workspace layout of a split plan with `cut` items: partial outputs, then partial
// log-sum-exps, then the arrival counters (each part 256-byte aligned).
size_t split_ws_bytes(int cut, int parts, int D, size_t *off_lse, size_t *off_cnt) {
    auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
    const size_t rows = static_cast<size_t>(cut) * parts * 2 * gqa::kBM;
    const size_t o = up(rows * D * sizeof(float));
    const size_t l = up(rows * sizeof(float));
    const size_t c = up(static_cast<size_t>(cut) * 2 * 4 * sizeof(unsigned int));
    if (off_lse) *off_lse = o;
    if (off_cnt) *off_cnt = o + l;
    return o + l + c;
}

attn_status_t host_pipe(int dev, HostPipe *&pipe) {
    HostPipe &hp = g_pipe[dev];
    if (!hp.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming);
        for (int c = 0; c < kMaxChunks && e == cudaSuccess; ++c) {
            e = cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&hp.out[c], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) {
            note_cuda_error(e, "attn_fwd_host set-up");
            return ATTN_ERR_LAUNCH;
        }
        hp.ready = true;
    }
    pipe = &hp;
    return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                          int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                          attn_dtype_t dtype, void *stream) {
    gqa::Params prm;
    int dev = 0;
    bool empty = false;
    attn_status_t st = prepare(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, prm, dev, empty);
    if (st != ATTN_OK || empty) return st;
    const bool bf16 = dtype == ATTN_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int kid = (D == 128 ? 4 : 0) + (bf16 ? 2 : 0) + (causal ? 1 : 0);
    switch (kid) {
        case 0: return launch<64, false, false>(dev, kid, prm, s);
        case 1: return launch<64, false, true>(dev, kid, prm, s);
        case 2: return launch<64, true, false>(dev, kid, prm, s);
        case 3: return launch<64, true, true>(dev, kid, prm, s);
        case 4: return launch<128, false, false>(dev, kid, prm, s);
        case 5: return launch<128, false, true>(dev, kid, prm, s);
        case 6: return launch<128, true, false>(dev, kid, prm, s);
        default: return launch<128, true, true>(dev, kid, prm, s);
    }
}

attn_status_t attn_fwd_kv_split_workspace(int B, int Hq, int Hkv, int Nq, int Nk, int D, int causal,
                                          size_t *bytes) {
    if (bytes == nullptr) return ATTN_ERR_NULL;
    *bytes = 0;
    static const uint8_t dummy[16] = {};
    gqa::Params prm;
    int dev = 0;
    bool empty = false;
    // validate with stand-in pointers: only the sizes matter here
    const void *fake = reinterpret_cast<const void *>((reinterpret_cast<uintptr_t>(dummy) + 15) & ~uintptr_t(15));
    attn_status_t st = prepare(fake, fake, fake, const_cast<void *>(fake), nullptr, B, Hq, Hkv, Nq, Nk, D, 1.f,
                               causal, ATTN_BF16, prm, dev, empty);
    if (st != ATTN_OK || empty) return st;
    const int cut = plan_last_round(prm, g_dev_sms[dev], causal);
    *bytes = cut > 0 ? split_ws_bytes(cut, prm.n_parts, D, nullptr, nullptr) : 0;
    return ATTN_OK;
}

attn_status_t attn_fwd_kv_split(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                                int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                                attn_dtype_t dtype, void *workspace, size_t workspace_bytes, void *stream) {
    if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_ALIGN;
    gqa::Params prm;
    int dev = 0;
    bool empty = false;
    attn_status_t st = prepare(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, prm, dev, empty);
    if (st != ATTN_OK || empty) return st;
    if (workspace != nullptr && g_kernel_choice.load() == 0) {
        gqa::Params plan = prm;
        const int cut = plan_last_round(plan, g_dev_sms[dev], causal);
        size_t off_lse = 0, off_cnt = 0;
        if (cut > 0 && split_ws_bytes(cut, plan.n_parts, D, &off_lse, &off_cnt) <= workspace_bytes) {
            prm = plan;
            uint8_t *w = static_cast<uint8_t *>(workspace);
            prm.part_o = reinterpret_cast<float *>(w);
            prm.part_lse = reinterpret_cast<float *>(w + off_lse);
            prm.part_count = reinterpret_cast<unsigned int *>(w + off_cnt);
        }
    }
    const bool bf16 = dtype == ATTN_BF16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int kid = (D == 128 ? 4 : 0) + (bf16 ? 2 : 0) + (causal ? 1 : 0);
    switch (kid) {
        case 0: return launch<64, false, false>(dev, kid, prm, s);
        case 1: return launch<64, false, true>(dev, kid, prm, s);
        case 2: return launch<64, true, false>(dev, kid, prm, s);
        case 3: return launch<64, true, true>(dev, kid, prm, s);
        case 4: return launch<128, false, false>(dev, kid, prm, s);
        case 5: return launch<128, false, true>(dev, kid, prm, s);
        case 6: return launch<128, true, false>(dev, kid, prm, s);
        default: return launch<128, true, true>(dev, kid, prm, s);
    }
}

attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                       int Hkv, int N, int D, float scale, int causal, attn_dtype_t dtype, void *stream) {
    return attn_fwd_kv(q, k, v, o, lse, B, Hq, Hkv, N, N, D, scale, causal, dtype, stream);
}

attn_status_t attn_fwd_decode_workspace(int B, int Hq, int Hkv, int Nq, int Nk, int D, size_t *bytes) {
    if (bytes == nullptr) return ATTN_ERR_NULL;
    *bytes = 0;
    static const uint8_t dummy[16] = {};
    gqa::Params prm;
    int dev = 0;
    bool empty = false;
    // validate with stand-in pointers: only the sizes matter here
    const void *fake = reinterpret_cast<const void *>((reinterpret_cast<uintptr_t>(dummy) + 15) & ~uintptr_t(15));
    attn_status_t st = prepare(fake, fake, fake, const_cast<void *>(fake), nullptr, B, Hq, Hkv, Nq, Nk, D,
                               1.f, 0, ATTN_BF16, prm, dev, empty);
    if (st != ATTN_OK || empty) return st;
    plan_splits(prm, g_dev_sms[dev], LLONG_MAX);
    *bytes = prm.n_splits > 1 ? split_bytes(prm, D) * prm.n_splits : 0;
    return ATTN_OK;
}

attn_status_t attn_fwd_decode(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                              int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                              attn_dtype_t dtype, void *workspace, size_t workspace_bytes, void *stream) {
    if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return ATTN_ERR_ALIGN;
    gqa::Params prm;
    int dev = 0;
    bool empty = false;
    attn_status_t st = prepare(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, prm, dev, empty);
    if (st != ATTN_OK || empty) return st;
    const long long cap = workspace == nullptr ? 1 : static_cast<long long>(workspace_bytes / split_bytes(prm, D));
    plan_splits(prm, g_dev_sms[dev], cap);
    return run_decode(prm, dev, D, dtype, causal, workspace, static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_decode_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                      int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
                                      int causal, attn_dtype_t dtype, void *stream) {
    gqa::Params prm;
    int dev = 0;
    bool empty = false;
    attn_status_t st = prepare(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, prm, dev, empty);
    if (st != ATTN_OK || empty) return st;
    plan_splits(prm, g_dev_sms[dev], LLONG_MAX);
    if (prm.n_splits > 1 && split_bytes(prm, D) * prm.n_splits > ATTN_NOALLOC_SCRATCH_BYTES)
        return ATTN_ERR_SCRATCH;
    // Every call that gets this far looks the buffer up on its first use on the
    // device, whether or not this plan splits, so that any one successful call
    // made before a stream capture has done the (non-stream) lookup.
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (g_dev_scratch[dev] == nullptr) {
            cudaError_t e = cudaGetSymbolAddress(&g_dev_scratch[dev], g_noalloc_scratch);
            if (e != cudaSuccess) {
                note_cuda_error(e, "cudaGetSymbolAddress");
                g_dev_scratch[dev] = nullptr;
                return ATTN_ERR_LAUNCH;
            }
        }
        scratch = g_dev_scratch[dev];
    }
    return run_decode(prm, dev, D, dtype, causal, prm.n_splits > 1 ? scratch : nullptr,
                      static_cast<cudaStream_t>(stream));
}

attn_status_t attn_fwd_host(const void *q_h, const void *k_h, const void *v_h, void *o_h, float *lse_h,
                            void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d, int B, int Hq,
                            int Hkv, int Nq, int Nk, int D, float scale, int causal, attn_dtype_t dtype,
                            void *stream) {
    const bool non_empty = B > 0 && Hq > 0 && Nq > 0;
    if (non_empty && (!q_h || !k_h || !v_h || !o_h || (lse_h == nullptr) != (lse_d == nullptr)))
        return ATTN_ERR_NULL;
    gqa::Params prm;
    int dev = 0;
    bool empty = false;
    attn_status_t st = prepare(q_d, k_d, v_d, o_d, lse_d, B, Hq, Hkv, Nq, Nk, D, scale, causal, dtype, prm,
                               dev, empty);
    if (st != ATTN_OK || empty) return st;

    // Chunks of consecutive (b, kv head) groups: each group's query heads, keys,
    // values, outputs and log-sum-exps are contiguous, so a chunk is five plain
    // copies and one attn_fwd_kv call over B' = groups, Hq' = G, Hkv' = 1.
    const int G = Hq / Hkv;
    const int groups = B * Hkv;
    const long long items = static_cast<long long>(B) * Hq * ((Nq + 255) / 256);
    long long want = items / (2LL * g_dev_sms[dev]);  // keep every chunk's launch a full GPU or more
    if (want > kMaxChunks) want = kMaxChunks;
    if (want > groups) want = groups;
    if (want < 1) want = 1;
    const int per = static_cast<int>((groups + want - 1) / want);
    const int chunks = (groups + per - 1) / per;
    const size_t qb = static_cast<size_t>(G) * Nq * D * 2;  // bytes of one group's Q (and O)
    const size_t kb = static_cast<size_t>(Nk) * D * 2;      // bytes of one group's K (and V)
    const size_t lb = static_cast<size_t>(G) * Nq * sizeof(float);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    auto at = [](const void *base, size_t off) { return static_cast<const uint8_t *>(base) + off; };
    auto atw = [](void *base, size_t off) { return static_cast<uint8_t *>(base) + off; };

    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe *hp = nullptr;
    if ((st = host_pipe(dev, hp)) != ATTN_OK) return st;
    cudaError_t e = cudaEventRecord(hp->start, cs);  // after the caller's earlier work
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->h2d, hp->start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->start, 0);
    for (int c = 0; c < chunks && e == cudaSuccess && st == ATTN_OK; ++c) {
        const int g0 = c * per, ng = (groups - g0 < per) ? groups - g0 : per;
        // copy in on h2d
        e = cudaMemcpyAsync(atw(q_d, g0 * qb), at(q_h, g0 * qb), ng * qb, cudaMemcpyHostToDevice, hp->h2d);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(atw(k_d, g0 * kb), at(k_h, g0 * kb), ng * kb, cudaMemcpyHostToDevice, hp->h2d);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(atw(v_d, g0 * kb), at(v_h, g0 * kb), ng * kb, cudaMemcpyHostToDevice, hp->h2d);
        if (e == cudaSuccess) e = cudaEventRecord(hp->in[c], hp->h2d);
        // compute on the caller's stream
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, hp->in[c], 0);
        if (e != cudaSuccess) break;
        st = attn_fwd_kv(at(q_d, g0 * qb), at(k_d, g0 * kb), at(v_d, g0 * kb), atw(o_d, g0 * qb),
                         lse_d ? reinterpret_cast<float *>(atw(lse_d, g0 * lb)) : nullptr, ng, G, 1, Nq, Nk, D,
                         scale, causal, dtype, stream);
        if (st != ATTN_OK) break;
        e = cudaEventRecord(hp->out[c], cs);
        // copy out on d2h
        if (e == cudaSuccess) e = cudaStreamWaitEvent(hp->d2h, hp->out[c], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(atw(o_h, g0 * qb), at(o_d, g0 * qb), ng * qb, cudaMemcpyDeviceToHost, hp->d2h);
        if (e == cudaSuccess && lse_h)
            e = cudaMemcpyAsync(atw(lse_h, g0 * lb), at(lse_d, g0 * lb), ng * lb, cudaMemcpyDeviceToHost,
                                hp->d2h);
    }
    // the caller's stream resumes after the last copy out, also after an error above
    cudaError_t e2 = cudaEventRecord(hp->done, hp->d2h);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(cs, hp->done, 0);
    if (e == cudaSuccess) e = e2;
    if (e != cudaSuccess) {
        note_cuda_error(e, "attn_fwd_host copies");
        return ATTN_ERR_LAUNCH;
    }
    return st;
}

const char *attn_status_str(attn_status_t status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_NULL: return "null pointer";
        case ATTN_ERR_SHAPE: return "invalid shape or scale";
        case ATTN_ERR_HEADDIM: return "unsupported head dimension (64 or 128)";
        case ATTN_ERR_DTYPE: return "unsupported dtype";
        case ATTN_ERR_ALIGN: return "misaligned pointer";
        case ATTN_ERR_LAUNCH: return "CUDA launch or driver call failed";
        case ATTN_ERR_TIMEOUT: return "in-kernel wait timed out";
        case ATTN_ERR_NODEVICE: return "no sm_103 device is current";
        case ATTN_ERR_SCRATCH: return "problem needs more scratch than the fixed device buffer holds";
    }
    return "unknown status";
}

attn_status_t attn_last_device_error(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaStreamSynchronize");
        return ATTN_ERR_LAUNCH;
    }
    int code = 0;
    e = cudaMemcpyFromSymbol(&code, gqa::g_error_code, sizeof(int));
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaMemcpyFromSymbol");
        return ATTN_ERR_LAUNCH;
    }
    if (code != 0) {
        // Clear the error and the abort mark of the launch that gave up: a CUDA
        // graph replays its launches with the sequence number they were captured
        // with, and a stale mark would make every later replay exit at once.
        const int zero = 0;
        const unsigned int no_seq = 0;  // sequence numbers start at 1
        e = cudaMemcpyToSymbol(gqa::g_error_code, &zero, sizeof(int));
        if (e == cudaSuccess) e = cudaMemcpyToSymbol(gqa::g_abort_seq, &no_seq, sizeof(unsigned int));
        if (e != cudaSuccess) note_cuda_error(e, "cudaMemcpyToSymbol");
    }
    return static_cast<attn_status_t>(code);
}

const char *attn_last_cuda_error(void) { return t_last_cuda_error; }

int attn_version(void) { return 0x000100; }

void attn_test_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns.store(ns ? ns : 4000000000ull); }

void attn_test_inject_stall(int enable) { g_inject_stall.store(enable ? 1 : 0); }

void attn_test_select_kernel(int which) { g_kernel_choice.store(which == 1 ? 1 : 0); }

void attn_test_force_splits(int n_splits) { g_force_splits.store(n_splits > 0 ? n_splits : 0); }

void attn_test_set_item_order(int order) { g_item_order.store(order == 1 ? 1 : 0); }

}  // extern "C"
