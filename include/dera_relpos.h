/*
 * dera_relpos — global self-attention with decomposed relative-position bias
 * (the DeepEncoder / SAM-style "rel-pos" attention), on GB300 (sm_103a).
 *
 * Source of the operation: vLLM PR #55629 page ("为 DeepEncoder 全局注意力融合
 * 相对位置偏置到 Triton 内核").
 *   - Section 关键源码片段 (key source excerpt): RelPosAttention.forward calls
 *     add_decomposed_rel_pos(q, rel_pos_h, rel_pos_w, (H,W), (H,W)) and then
 *     either the fused launcher deepencoder_rel_pos_attention(q, k, v,
 *     rel_h.squeeze(-1), rel_w.squeeze(-2), W, scale) or SDPA with the
 *     materialised bias (rel_h + rel_w).view(B, heads, HW, H*W).  The SDPA
 *     call defines the result:
 *         out[n] = sum_m softmax_m(scale * q_n.k_m + rel_h[n, kh(m)] + rel_w[n, kw(m)]) v_m
 *     with tokens n = qh*W + qw and keys m = kh*W + kw.
 *   - The body of add_decomposed_rel_pos is not printed; this library takes
 *     the SAM-style reading rel_h[n, kh] = q_n . rel_pos_h[qh - kh + H - 1] and
 *     rel_w[n, kw] = q_n . rel_pos_w[qw - kw + W - 1] (unscaled q).
 *   - Section 实现拆解 (implementation breakdown) item 1: the fused kernel
 *     streams keys/values with an online softmax and adds the bias slice per
 *     key block, never building the HW x HW bias.
 *   - Section 风险与影响 (risks): fp32 accumulation, exp2; fast path only for
 *     FP16/BF16 with head_dim 64.
 *   - Section 评论区精华 (review discussion): all five launcher inputs must be
 *     device tensors on the same device.
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers on the current CUDA device, except
 *     where an argument says otherwise.  The caller owns every buffer; the
 *     library allocates nothing, never synchronises, and enqueues all work on
 *     `stream` (a cudaStream_t passed as void*; NULL = legacy default stream).
 *   - Layouts are contiguous, row-major:
 *       q, k, v, out : [BH, N, head_dim], N = H*W, token n = qh*W + qw
 *       rel_pos_h    : [2H-1, head_dim]      rel_pos_w : [2W-1, head_dim]
 *       rel_h        : [BH, N, H]            rel_w     : [BH, N, W]
 *   - head_dim is 64 or 128 (the pages' kernel fixes 64; 128 is this
 *     library's extension).  q, k, v, tables share one dtype: DERA_F16 or
 *     DERA_BF16.  1 <= H, W <= 64.  BH >= 0 (BH == 0 is a no-op).
 *   - Buffer lengths are the caller's precondition: the ABI takes no length
 *     arguments, so a table must hold exactly 2H-1 (2W-1) rows and every
 *     tensor the elements its layout above implies.  A shorter buffer is read
 *     or written past its end; nothing here can detect it.
 *   - Every pointer must be 16-byte aligned (TMA operands).  With BH == 0
 *     the call returns DERA_OK before looking at any pointer.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and returned as a status; nothing falls back to another backend.
 *   - DERA_ERR_CUDA: a CUDA call made by the library failed (launch error,
 *     invalid device pointer query).  The sticky CUDA error, if any, is left
 *     for the caller to inspect.
 *   - A kernel that exceeds its internal bounded-wait budget (about one
 *     second per wait) stops early and records DERA_ERR_TIMEOUT in the
 *     library's device status word; read it with dera_relpos_device_status().
 *     Its output is then undefined.
 *   - All entry points are stream-ordered and allocation-free, so they can be
 *     captured in a CUDA graph.
 *   - DERA_ERR_ALIGN also covers a workspace that is not 256-byte aligned.
 */
#ifndef DERA_RELPOS_H
#define DERA_RELPOS_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DERA_RELPOS_ABI_VERSION 3

#if defined(__GNUC__)
#define DERA_API __attribute__((visibility("default")))
#else
#define DERA_API
#endif

typedef enum dera_status {
  DERA_OK = 0,
  DERA_ERR_NULL = 1,        /* a required pointer is NULL */
  DERA_ERR_SHAPE = 2,       /* H, W, BH out of range, or N overflow */
  DERA_ERR_DTYPE = 3,       /* dtype not supported for that argument */
  DERA_ERR_HEAD_DIM = 4,    /* head_dim is neither 64 nor 128 */
  DERA_ERR_ALIGN = 5,       /* a pointer is not 16-byte aligned */
  DERA_ERR_DEVICE = 6,      /* a pointer is not device memory of the current device */
  DERA_ERR_TIMEOUT = 7,     /* (device status only) a bounded wait expired */
  DERA_ERR_CUDA = 8,        /* a CUDA runtime/driver call failed */
  DERA_ERR_SCRATCH = 9      /* (dera_relpos_fused_noalloc) the problem needs more scratch than its static buffer */
} dera_status;

typedef enum dera_dtype { DERA_F16 = 0, DERA_BF16 = 1, DERA_F32 = 2 } dera_dtype;

/*
 * A1 — decomposed rel-pos projection (add_decomposed_rel_pos; page section
 * 关键源码片段, and the squeeze to the compact [.., HW, H] / [.., HW, W] form
 * of section 实现拆解 item 2):
 *     rel_h[b, n, kh] = sum_c q[b, n, c] * rel_pos_h[qh(n) - kh + H - 1, c]
 *     rel_w[b, n, kw] = sum_c q[b, n, c] * rel_pos_w[qw(n) - kw + W - 1, c]
 * in:  q [BH,N,head_dim], rel_pos_h [2H-1,head_dim], rel_pos_w [2W-1,head_dim], all in_dtype
 *      (DERA_F16 | DERA_BF16).
 * out: rel_h [BH,N,H], rel_w [BH,N,W] in bias_dtype (DERA_F32, or
 *      DERA_BF16/DERA_F16, rounded to nearest from the fp32 accumulator).
 */
DERA_API dera_status dera_relpos_project(const void* q, const void* rel_pos_h, const void* rel_pos_w, void* rel_h,
                                void* rel_w, int BH, int H, int W, int head_dim, dera_dtype in_dtype,
                                dera_dtype bias_dtype, void* stream);

/*
 * A2..A7 — attention with a compact bias (deepencoder_rel_pos_attention;
 * page sections 关键源码片段 and 实现拆解 item 1):
 *     out[b, n] = sum_m softmax_m(scale * q[b,n].k[b,m] + rel_h[b,n,kh(m)] + rel_w[b,n,kw(m)]) v[b,m]
 * in:  q, k, v [BH,N,head_dim] in_dtype (DERA_F16 | DERA_BF16);
 *      rel_h [BH,N,H], rel_w [BH,N,W] in bias_dtype (DERA_F32 | DERA_BF16 | DERA_F16).
 * out: out [BH,N,head_dim] in out_dtype (DERA_F32, or in_dtype).
 * workspace / workspace_bytes: optional scratch, see dera_relpos_workspace_size.
 * Softmax runs in base 2 with fp32 accumulation; P is rounded to fp16 for the
 * P.V product (for bf16 inputs, V tiles are converted to fp16 on chip, so
 * |v| must stay below 65504).  The rounding of P moves each output by at most
 * (2^-11 + 2^-9) max|v|: a tile whose row sums show less is computed again
 * before anything is stored.
 */
DERA_API dera_status dera_relpos_attention(const void* q, const void* k, const void* v, const void* rel_h,
                                  const void* rel_w, void* out, int BH, int H, int W, int head_dim, float scale,
                                  dera_dtype in_dtype, dera_dtype bias_dtype, dera_dtype out_dtype,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * A1..A7 fused — projection computed inside the attention kernel (tensor-core
 * q.rel_pos^T products, skewed on chip), so neither the dense HW x HW bias
 * nor the compact rel_h / rel_w ever reaches global memory.
 * in:  q, k, v [BH,N,head_dim], rel_pos_h [2H-1,head_dim], rel_pos_w [2W-1,head_dim], in_dtype.
 * out: out [BH,N,head_dim] in out_dtype (DERA_F32, or in_dtype).
 * workspace / workspace_bytes: optional scratch, see dera_relpos_workspace_size.
 */
DERA_API dera_status dera_relpos_fused(const void* q, const void* k, const void* v, const void* rel_pos_h,
                              const void* rel_pos_w, void* out, int BH, int H, int W, int head_dim, float scale,
                              dera_dtype in_dtype, dera_dtype out_dtype, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Scratch needed by dera_relpos_attention / dera_relpos_fused for a problem
 * size on the current device, written to *bytes (host pointer); 0 when the
 * work splits evenly over the device or the units are too short to be worth
 * cutting (no scratch used).
 *
 * Scheduling (no counterpart on the pages, which give no kernel schedule):
 * the work unit is a pair of 128-row query tiles of one head.  When the
 * number of units is not a whole number of waves of one CTA per SM and a
 * unit spans at least 4 key tiles (grids of at least 4 x 16 or so), the
 * kernel runs one persistent CTA per SM over equal shares of the
 * (unit, key tile) iteration space and cuts some units between two CTAs; the
 * partial results (unnormalised O, row max, row sum, fp32) and two 8-byte
 * arrival counters per unit (one per query tile) live in the caller's
 * `workspace`.  A NULL workspace, or one smaller than this size, selects
 * whole units taken round-robin by one CTA per SM instead (same result, no
 * scratch, less even load).  The
 * workspace must be device memory, 256-byte aligned, owned by the caller, and
 * not used by another call in flight.  Its contents need no initialisation
 * and are never cleared: each launch marks its arrivals with a 64-bit tag that
 * no earlier launch of the process used, so whatever an earlier call (or one
 * that stopped early) left behind is ignored.
 */
DERA_API dera_status dera_relpos_workspace_size(int BH, int H, int W, int head_dim, size_t* bytes);

/*
 * Training forward: dera_relpos_fused that also writes, for every row, the
 * base-2 log-sum-exp of its logits, lse[b, n] = log2(sum_m exp(Z[b, n, m])) with
 * Z = scale q k^T + rel_h + rel_w (vLLM PR #55629 page, section 实现拆解 item 1:
 * the online softmax's row maximum and row sum, combined).  lse: [BH, N] fp32,
 * device memory, 16-byte aligned.  Every other argument, error and the output
 * are as for dera_relpos_fused.  The backward needs lse.
 */
DERA_API dera_status dera_relpos_fused_lse(const void* q, const void* k, const void* v, const void* rel_pos_h,
                                  const void* rel_pos_w, void* out, float* lse, int BH, int H, int W,
                                  int head_dim, float scale, dera_dtype in_dtype, dera_dtype out_dtype,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * Scratch needed by dera_relpos_fused_backward (bytes, written to *bytes):
 * 4 * (BH N (H + W + 1) + BH ceil(N / 128) (128 H + 64 (2H - 1 + 2W - 1)))
 * plus alignment: the compact bias, one term per row, the rel_h term of the
 * exponent laid out by key grid row, and per-query-tile table-gradient
 * partials, all fp32.  head_dim must be 64.
 */
DERA_API dera_status dera_relpos_backward_workspace_size(int BH, int H, int W, int head_dim, size_t* bytes);

/*
 * Backward of dera_relpos_fused (training use; the pages print no backward:
 * this is the chain-rule gradient of the forward's definition).  With
 * Z = scale q k^T + rel_h + rel_w, P = softmax(Z), an upstream gradient dout
 * and D[n] = dout[n] . out[n], dZ = P * (dout v^T - D):
 *   dv = P^T dout, dk = scale dZ^T q,
 *   dq = scale dZ k + sum_kh drel_h[n, kh] rel_pos_h[qh - kh + H - 1] + sum_kw (same for w),
 *   drel_pos_h[i] = sum over (b, n, kh) with qh - kh + H - 1 = i of drel_h[b, n, kh] q[b, n] (same for w),
 * where drel_h[n, kh] = sum_kw dZ[n, kh W + kw] and drel_w[n, kw] = sum_kh dZ[n, kh W + kw].
 * in:  q, k, v [BH,N,64] and rel_pos_h [2H-1,64], rel_pos_w [2W-1,64] in in_dtype
 *      (as given to the forward); out [BH,N,64] (the forward's output) in out_dtype
 *      (DERA_F32 or in_dtype); lse [BH,N] fp32 from dera_relpos_fused_lse; dout
 *      [BH,N,64] in in_dtype.
 * out: dq, dk, dv [BH,N,64] in grad_dtype (DERA_F32 or in_dtype); drel_pos_h
 *      [2H-1,64] and drel_pos_w [2W-1,64] fp32 (summed over every batch and head).
 * workspace: device memory of at least dera_relpos_backward_workspace_size bytes,
 *      256-byte aligned, owned by the caller, not used by another call in flight;
 *      its contents need no initialisation.
 * Precision: P is recomputed from lse in fp32; dZ, P and the bias gradients
 *      (drel_h, drel_w) enter the tensor-core products rounded to in_dtype (relative
 *      2^-9 for bf16, 2^-11 for fp16), with fp32 accumulation; the per-tile table
 *      gradients are added in fp32.
 *      Nothing is accumulated with atomics: the result is the same on every run.
 * Errors: DERA_ERR_HEAD_DIM unless head_dim is 64; DERA_ERR_SCRATCH if the
 *      workspace is NULL or smaller than the size above; otherwise as for
 *      dera_relpos_fused.  With BH = 0 only drel_pos_h and drel_pos_w are
 *      read (as pointers) and written, with zeros; the other pointers may be NULL.
 */
DERA_API dera_status dera_relpos_fused_backward(const void* q, const void* k, const void* v, const void* rel_pos_h,
                                       const void* rel_pos_w, const void* out, const float* lse,
                                       const void* dout, void* dq, void* dk, void* dv, float* drel_pos_h,
                                       float* drel_pos_w, int BH, int H, int W, int head_dim, float scale,
                                       dera_dtype in_dtype, dera_dtype out_dtype, dera_dtype grad_dtype,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Allocation-free variant of dera_relpos_fused (the pages have no
 * counterpart: it exists for callers of this library that are not allowed
 * to allocate device memory).  Some callers cannot call cudaMalloc at all:
 * plug-ins living inside a host engine that owns every byte of device memory
 * and forbids allocations after start-up, or latency-critical code that must
 * never hit the implicit device synchronisation an allocation can cause.
 * Such a caller still passes its own inputs and output, but cannot hand over
 * the scratch workspace that dera_relpos_fused uses when it splits work
 * units between CTAs.
 *
 * This entry point computes exactly what dera_relpos_fused computes (same
 * arguments minus the workspace) and takes its scratch from a buffer
 * compiled into the library: a file-scope device array of
 * DERA_NOALLOC_SCRATCH_BYTES (48 MiB) that every GPU which loads the library
 * holds until the process exits.  It calls no cudaMalloc/cudaFree and no
 * allocating library routine.
 *   - Set-up: the first call on each device looks up the device address of
 *     that buffer (cudaGetSymbolAddress) with the device current and caches
 *     it; make that first call on a device before any stream capture.
 *   - Limit: problems whose split schedule needs more scratch than the
 *     buffer holds are rejected with DERA_ERR_SCRATCH before anything is
 *     enqueued.  The need is what dera_relpos_workspace_size reports: on a
 *     152-SM GB300, 20 545 536 bytes of partial-result slots (40 468 480 with
 *     head_dim 128) plus 16 bytes per work unit (a pair of 128-row query
 *     tiles of one head), so problems of up to about 1.8 million units (600 000
 *     with head_dim 128) fit.  Problems that need no scratch always run.
 *   - Sharing: every call on a device uses the same buffer and leaves its
 *     contents behind; like a caller's workspace, the buffer needs no
 *     clearing between calls (see dera_relpos_workspace_size).  Calls that overlap on
 *     the GPU (for example on two streams) race on the buffer and give wrong
 *     results: serialise them.
 * Other arguments, layouts and errors: as dera_relpos_fused.
 */
#define DERA_NOALLOC_SCRATCH_BYTES (48u * 1024u * 1024u)
DERA_API dera_status dera_relpos_fused_noalloc(const void* q, const void* k, const void* v, const void* rel_pos_h,
                                               const void* rel_pos_w, void* out, int BH, int H, int W,
                                               int head_dim, float scale, dera_dtype in_dtype, dera_dtype out_dtype,
                                               void* stream);

/* Human-readable name of a status code (static storage, never NULL). */
DERA_API const char* dera_status_string(dera_status status);

/*
 * Reads the device status word of the current device into *status (host
 * pointer) and, if reset != 0, clears it.  Synchronises the current device.
 * Returns DERA_ERR_NULL for a NULL status pointer, DERA_ERR_CUDA if the copy
 * fails.  *status is DERA_OK or DERA_ERR_TIMEOUT.
 */
DERA_API dera_status dera_relpos_device_status(int* status, int reset);

/*
 * Self-test of the bounded wait: launches one CTA that waits on an mbarrier
 * that nothing ever arrives on, with a budget of `budget_cycles` SM cycles
 * (clamped to [1e3, 4e9]).  The kernel gives up, writes DERA_ERR_TIMEOUT to
 * the device status word and exits normally; the host reads it back with
 * dera_relpos_device_status().  Used by tests to show that an expired wait
 * ends in an error status rather than a hang.
 */
DERA_API dera_status dera_relpos_selftest_wait_timeout(long long budget_cycles, void* stream);

/* ABI version of the loaded library (DERA_RELPOS_ABI_VERSION; 2 added the workspace arguments, 3 the
 * training forward and the backward). */
DERA_API int dera_relpos_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DERA_RELPOS_H */
