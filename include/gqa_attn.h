/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) fused grouped-query attention
 * forward library (libgqa_attn.so).
 *
 * The operation is the fused attention forward of the page "从零开始写Qwen3"
 * (deepseek.csdn.net/6a3201f8..., section "FlashAttention": O_i is the sum over
 * key blocks j of softmax(mask(Q_i K_j^T / sqrt(D))) V_j, computed with the
 * online-softmax update of section "在线softmax" so that no N x N score matrix
 * is ever stored), with
 *   - grouped-query heads: query head hq reads key/value head
 *     hq / (Hq / Hkv) of the same batch entry (same section's kernel: the
 *     flattened (b, q_head) index divided by the group count);
 *   - the optional causal mask j <= i on absolute row indices (same section:
 *     positions with offsets_qm >= offsets_kk are kept); with Nq query rows
 *     over Nk keys (attn_fwd_kv and the calls built on it) the query rows are
 *     the last Nq positions, so row i keeps keys j <= i + Nk - Nq;
 *   - the natural-log log-sum-exp of each masked, scaled score row,
 *     lse = max_j s_ij + ln(sum_j exp(s_ij - max_j s_ij)), written as fp32.
 *
 * Arithmetic: Q K^T and P V on the tensor cores with fp32 accumulation;
 * running max, running sum and the output accumulator in fp32 (page
 * "从零开始写Qwen3", deepseek.csdn.net/6a31faef..., section "改进点4-去掉多余的
 * 转换"); the probabilities P are rounded to the input type before the P V
 * product; O is rounded once, to nearest even, at the end.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of q, k, v and o. */
typedef enum {
    ATTN_F16 = 0,  /* IEEE binary16 */
    ATTN_BF16 = 1  /* bfloat16 */
} attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,     /* q, k, v or o is NULL while the problem is non-empty */
    ATTN_ERR_SHAPE = 2,    /* negative size, Hkv < 1, Hq % Hkv != 0, a size too
                              large for 32-bit tile coordinates, or scale not
                              finite and > 0 */
    ATTN_ERR_HEADDIM = 3,  /* D is not 64 or 128 */
    ATTN_ERR_DTYPE = 4,    /* dtype is not ATTN_F16 / ATTN_BF16 */
    ATTN_ERR_ALIGN = 5,    /* q, k, v or o not 16-byte aligned, or lse not 4-byte aligned */
    ATTN_ERR_LAUNCH = 6,   /* a CUDA runtime / driver call failed (see attn_last_cuda_error) */
    ATTN_ERR_TIMEOUT = 7,  /* a bounded in-kernel wait ran out (reported by
                              attn_last_device_error) */
    ATTN_ERR_NODEVICE = 8, /* no CUDA device of compute capability 10.3 is current */
    ATTN_ERR_SCRATCH = 9   /* attn_fwd_decode_noalloc: the problem needs more scratch
                              than the library's fixed device buffer holds */
} attn_status_t;

/*
 * attn_fwd -- O = softmax(mask(Q K^T * scale)) V and LSE, one kernel launch.
 *
 * q    device pointer, [B, Hq,  N, D] contiguous (row-major, D fastest), dtype
 * k    device pointer, [B, Hkv, N, D] contiguous, dtype
 * v    device pointer, [B, Hkv, N, D] contiguous, dtype
 * o    device pointer, [B, Hq,  N, D] contiguous, dtype (written)
 * lse  device pointer, [B, Hq, N] fp32 (written), or NULL to skip it
 * B, Hq, Hkv, N   batch, query heads, key/value heads (Hq % Hkv == 0), sequence
 *                 length (keys and queries have the same length N)
 * D      head dimension, 64 or 128
 * scale  logit scale, finite and > 0 (1/sqrt(D) for standard attention)
 * causal nonzero: keep only keys j <= i for query row i (top-left aligned)
 * dtype  ATTN_F16 or ATTN_BF16 for q, k, v and o
 * stream CUDA stream (cudaStream_t) the kernel is launched on; NULL = legacy
 *        default stream
 *
 * Ownership: the caller owns every buffer; the library allocates no device
 * memory per call and keeps no pointer after the call returns.  o must not
 * overlap q, k or v.
 * Asynchrony: returns after the launch is queued on `stream`; results are
 * ready when the stream reaches that point.  The call never synchronises.
 * CUDA graphs: a call can be captured into a CUDA graph (one kernel node; the
 * node keeps the pointers, sizes and scale of the captured call).  The first
 * call of each (D, dtype, causal) variant on a device sets the kernel's shared
 * memory limit, which is not a stream operation: make one such call before
 * capturing, as with any library that configures itself on first use.
 * Errors: argument errors are returned before anything is launched and leave
 * o and lse untouched.  An empty problem (B, Hq or N equal to 0) launches
 * nothing and returns ATTN_OK.  A wait inside the kernel that runs out of time
 * makes the kernel stop early and record ATTN_ERR_TIMEOUT, which
 * attn_last_device_error reports; o and lse are then undefined.
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int Hq, int Hkv, int N, int D, float scale, int causal,
                       attn_dtype_t dtype, void *stream);

/*
 * attn_fwd_kv -- as attn_fwd, for Nq query rows attending over Nk keys (a
 * block of new tokens over a longer key/value sequence, e.g. a chunk of a
 * prefill or a decode step over a cache).  The derivation page's kernel
 * ("从零开始写Qwen3", deepseek.csdn.net/6a3201f8..., section "FlashAttention")
 * keeps the query and key lengths apart; this call does too.
 *
 * q, o   [B, Hq,  Nq, D];  k, v  [B, Hkv, Nk, D];  lse  [B, Hq, Nq] or NULL
 * causal nonzero: the query rows are the last Nq positions of the Nk-long
 *        sequence (bottom-right alignment): row i keeps keys j <= i + Nk - Nq.
 *        With Nq == Nk this is attn_fwd's mask j <= i.
 * Errors: as attn_fwd, plus ATTN_ERR_SHAPE when Nk == 0 while Nq > 0, or when
 *        causal and Nq > Nk (some query row would see no key).  Nq == 0 is an
 *        empty problem (nothing launched, ATTN_OK).
 * attn_fwd(..., N, ...) is attn_fwd_kv(..., N, N, ...).
 */
attn_status_t attn_fwd_kv(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
                          int causal, attn_dtype_t dtype, void *stream);

/*
 * attn_fwd_kv_split -- attn_fwd_kv with a caller workspace that lets the library
 * balance the last round of its schedule.
 *
 * The persistent kernel deals 256-row items to one CTA per SM in rounds.  When
 * every item has the same length (no mask, or a chunk of queries over a much
 * longer key sequence) and the last round holds at most half a round of items,
 * each of those items is cut into up to 8 key ranges; the pieces (the partial
 * O / l in fp32 and the partial log-sum-exp of every row) go to the workspace,
 * and the warp that computes the last piece of its rows merges them:
 * lse = log sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s -- the online-softmax
 * update of page "从零开始写Qwen3" (deepseek.csdn.net/6a3201f8..., section
 * "在线softmax"), applied across CTAs.  The result equals attn_fwd_kv's up to
 * rounding.
 *
 * Arguments, layout, masks and errors: as attn_fwd_kv, plus
 * workspace        device pointer, 256-byte aligned, or NULL; workspace_bytes its
 *                  size.  attn_fwd_kv_split_workspace gives the size the plan needs
 *                  (0 when nothing is cut, e.g. causal problems with Nq == Nk,
 *                  whose items already differ in length).  With a NULL or smaller
 *                  workspace, or when nothing is cut, the call is attn_fwd_kv.
 * Contents: the workspace needs no initial value; its counters carry the launch's
 *   sequence number, so stale contents are recognised.  A captured call replays
 *   correctly as long as no replay of it has timed out (ATTN_ERR_TIMEOUT); after a
 *   timeout, capture the call again or clear the workspace.
 * Races: calls that can run at the same time must not share a workspace.
 * ATTN_ERR_ALIGN also when workspace is not 256-byte aligned.
 */
attn_status_t attn_fwd_kv_split_workspace(int B, int Hq, int Hkv, int Nq, int Nk, int D, int causal,
                                          size_t *bytes);
attn_status_t attn_fwd_kv_split(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
                                int causal, attn_dtype_t dtype, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * attn_fwd_decode -- the same function as attn_fwd_kv, computed by a kernel
 * for short query blocks over long key sequences (decode steps, small chunks).
 *
 * The Hq / Hkv query heads that share a kv head have adjacent rows, so their
 * Hq/Hkv * Nq query rows are stacked into 128-row tiles and every K/V tile is
 * read once per kv head (grouped-query packing).  The key range is cut into
 * splits, one CTA each, so that few kv heads still fill the GPU; the splits'
 * partial results are merged through their log-sum-exp by a second kernel
 * (the online-softmax merge of the derivation page "从零开始写Qwen3",
 * deepseek.csdn.net/6a3201f8..., section "在线softmax", applied across CTAs).
 *
 * Arguments as attn_fwd_kv, plus:
 * workspace        device pointer, 16-byte aligned, or NULL; scratch for the
 *                  partial results, owned by the caller, used by the two
 *                  kernels this call queues on `stream` and free again once
 *                  the stream has passed them.  Nothing in it needs to start
 *                  at any value.
 * workspace_bytes  its size.  The call uses as many splits as it wants and
 *                  the workspace holds (attn_fwd_decode_workspace gives the
 *                  size for all it wants); with NULL or too little for two
 *                  splits it runs one split, which needs no workspace.
 * Two calls that run at the same time must not share a workspace.
 * Errors: as attn_fwd_kv; ATTN_ERR_ALIGN also for a misaligned workspace.
 */
attn_status_t attn_fwd_decode(const void *q, const void *k, const void *v, void *o, float *lse,
                              int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale,
                              int causal, attn_dtype_t dtype, void *workspace,
                              size_t workspace_bytes, void *stream);

/*
 * Workspace bytes attn_fwd_decode uses for this problem on the current device
 * when given enough (0 when it would run one split).  Writes *bytes; returns
 * argument errors as attn_fwd_kv, ATTN_ERR_NULL for bytes == NULL and
 * ATTN_ERR_NODEVICE without an sm_103 device.
 */
attn_status_t attn_fwd_decode_workspace(int B, int Hq, int Hkv, int Nq, int Nk, int D,
                                        size_t *bytes);

/*
 * attn_fwd_decode_noalloc -- attn_fwd_decode for callers that cannot allocate
 * device memory (an allocator-free runtime, a captured graph that must not own
 * buffers, a call site that only receives q, k, v, o and lse).  The pages have
 * no counterpart: their kernels keep everything on chip and need no scratch;
 * the key splits of attn_fwd_decode do.
 *
 * Instead of a caller workspace the call uses a buffer that the library
 * itself holds in device memory: ATTN_NOALLOC_SCRATCH_BYTES (16 MiB) per
 * device, a static array of this library's module, so nothing is allocated
 * on any call.  The split plan is the one attn_fwd_decode chooses with an
 * unlimited workspace, so both calls give the same bits.  That plan needs at
 * most (number of SMs) * 128 * (D + 1) * 4 bytes (10 MB on 152 SMs), so the
 * buffer covers every problem on devices with up to 254 SMs; a plan that needs
 * more (e.g. one forced by attn_test_force_splits) returns ATTN_ERR_SCRATCH
 * before anything is launched.
 *
 * Arguments, layout, masks and errors: as attn_fwd_kv.
 * Setup: the first call on a device that passes argument validation looks
 *   up the buffer's address (not a stream operation), whether or not its plan
 *   splits the keys; make one such call on each device before capturing calls
 *   into a CUDA graph.
 * Contents: nothing in the buffer needs to start at any value; each call
 *   writes every part it reads.
 * Races: all calls on one device share the buffer.  Calls queued on one
 *   stream are ordered and safe; calls that can run at the same time (other
 *   streams, concurrently replayed graphs) race on it and give undefined
 *   results.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (16u << 20)
attn_status_t attn_fwd_decode_noalloc(const void *q, const void *k, const void *v, void *o,
                                      float *lse, int B, int Hq, int Hkv, int Nq, int Nk, int D,
                                      float scale, int causal, attn_dtype_t dtype, void *stream);

/*
 * attn_fwd_host -- attn_fwd_kv for inputs and outputs in host memory: copies Q,
 * K, V in, computes, copies O and LSE out, overlapping the three.
 *
 * The B * Hkv (batch, kv head) groups are contiguous in every tensor (a group's
 * Hq / Hkv query heads are adjacent), so the call cuts them into up to 8 chunks
 * of consecutive groups: chunk c + 1 is copied in on one library stream while
 * chunk c is computed on `stream` and chunk c - 1 is copied out on another.
 * The pages have no counterpart (their benchmarks start from device tensors).
 *
 * q_h, k_h, v_h       host inputs, layouts as attn_fwd_kv; page-locked memory
 *                     makes the copies asynchronous (pageable memory works but
 *                     serialises them)
 * o_h, lse_h          host outputs (lse_h NULL exactly when lse_d is NULL)
 * q_d ... lse_d       device buffers of the same sizes, owned by the caller;
 *                     they hold the inputs and results when the call is done
 * stream              the call is ordered after earlier work on `stream`, and
 *                     later work on `stream` waits for its last copy out; the
 *                     call returns without waiting.  Host outputs are valid
 *                     once `stream` has passed that point.
 * Set-up: the first call on a device creates the library's two copy streams
 *   and its events (not memory; kept for the life of the process).
 * Errors: as attn_fwd_kv; ATTN_ERR_NULL for a missing host pointer.
 */
attn_status_t attn_fwd_host(const void *q_h, const void *k_h, const void *v_h, void *o_h,
                            float *lse_h, void *q_d, void *k_d, void *v_d, void *o_d, float *lse_d,
                            int B, int Hq, int Hkv, int Nq, int Nk, int D, float scale, int causal,
                            attn_dtype_t dtype, void *stream);

/* Static, human-readable name of a status code. */
const char *attn_status_str(attn_status_t status);

/*
 * Synchronises `stream`, then returns and clears the error word that kernels
 * of this library set on the current device (ATTN_OK if none), together with
 * the mark that makes the other CTAs of a launch that gave up exit early.  A
 * CUDA error raised by the synchronisation itself is returned as
 * ATTN_ERR_LAUNCH.  Call it while no other launch of this library is running
 * on the device.
 */
attn_status_t attn_last_device_error(void *stream);

/* Text of the last CUDA error this library saw on the calling thread ("" if none). */
const char *attn_last_cuda_error(void);

/* Library version, e.g. 0x000100 for 0.1.0. */
int attn_version(void);

/*
 * Test hooks for the failure path (process-wide, affect later launches).
 *
 * attn_test_set_wait_timeout_ns: limit of every bounded in-kernel wait, in
 *   nanoseconds; 0 restores the default (4 s).
 * attn_test_inject_stall: nonzero makes later launches skip the load of the
 *   query tile, so the MMA warp's wait on it can only end by running out; the
 *   kernel then records ATTN_ERR_TIMEOUT, drains its own copies in flight,
 *   frees its TMEM and returns.  0 restores normal launches.
 * Neither hook faults, traps or hangs the GPU.
 */
void attn_test_set_wait_timeout_ns(unsigned long long ns);
void attn_test_inject_stall(int enable);

/*
 * attn_test_select_kernel: 0 (default) = persistent warp-specialised kernel
 *   (two 128-row query tiles per work item, P kept in TMEM); 1 = the simpler
 *   kernel with one CTA per 128-row query tile and P staged in shared memory.
 *   Both compute the same operation; the second exists to cross-check the first.
 */
void attn_test_select_kernel(int which);

/* attn_test_force_splits: n > 0 makes attn_fwd_decode and attn_fwd_decode_noalloc
 * use n key splits (as far as the key tiles and the workspace allow); 0 restores
 * their own choice. */
void attn_test_force_splits(int n_splits);

/* attn_test_set_item_order: work-item order of the persistent kernel (the
 * default one of attn_fwd / attn_fwd_kv).  0 (default) = the longest causal
 * row blocks first across all heads, the query heads of a GQA group adjacent;
 * 1 = kv-group major: every row block of one (batch, kv head) group, longest
 * first, before the next group, so that one group's K/V is live in L2 at a
 * time (the grid order of page "从零开始写Qwen3", deepseek.csdn.net/6a31faef...,
 * section "改进1-使用正确的grid").  Both orders compute every item once and give
 * the same bits; the hook exists to measure one against the other. */
void attn_test_set_item_order(int order);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
