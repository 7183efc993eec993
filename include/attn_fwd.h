/*
 * attn_fwd.h -- C ABI of the GB300 (sm_103a) exact attention-forward library.
 *
 * The operation (page "Hardware Acceleration & Custom Kernels", section 2
 * "FlashAttention: SRAM Tiling & Online Softmax"): for every batch b, head h
 * and query row i,
 *
 *     O[b,h,i,:] = softmax_j( scale * Q[b,h,i,:] . K[b,h,j,:] ) V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp( scale * Q[b,h,i,:] . K[b,h,j,:] )
 *
 * with j over [0, N), or over [0, i] when `causal` is set.  The kernels walk
 * K and V in tiles and keep a running row maximum and row sum (the online
 * normalisation identity of the same section), so the N x N score matrix is
 * never written to device memory.
 *
 * Conventions shared by every entry point:
 *   - Tensors are dense row-major [B, H, N, d] with d contiguous (element
 *     (b,h,i,c) at offset ((b*H + h)*N + i)*d + c); Q, K and V share N.
 *   - All tensor pointers are DEVICE pointers (cudaMalloc or managed memory
 *     on the current device), 16-byte aligned.  The caller owns them; the
 *     library keeps no reference after the call returns.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous on that stream: a return of ATTN_OK
 *     means the work was validated and enqueued, not that it finished.
 *   - Arguments are validated on the host before anything is launched; on any
 *     error nothing is launched and the outputs are untouched.
 *   - The first call on a device sets up per-device state (a 256-byte device
 *     status word, kernel attributes); make it before capturing a stream into
 *     a CUDA graph.  No call allocates device memory after that.
 */
#ifndef ATTN_FWD_GB300_H
#define ATTN_FWD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum attn_status {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,           /* a required pointer is NULL */
    ATTN_ERR_SHAPE = 2,          /* B, H or N < 1, or a size overflows the kernels' index range */
    ATTN_ERR_DTYPE = 3,          /* dtype is not an attn_dtype value */
    ATTN_ERR_HEADDIM = 4,        /* d is not 64 or 128 */
    ATTN_ERR_ALIGN = 5,          /* a tensor pointer is not 16-byte aligned */
    ATTN_ERR_ARCH = 6,           /* current device is not compute capability 10.3 (sm_103) */
    ATTN_ERR_LAUNCH = 7,         /* the kernel launch itself failed */
    ATTN_ERR_DEVICE_TIMEOUT = 8, /* a kernel's bounded wait ran out (reported by attn_device_status) */
    ATTN_ERR_NOT_DEVICE = 9,     /* a pointer is not device-accessible memory of the current device */
    ATTN_ERR_CUDA = 10,          /* a CUDA runtime call failed during set-up or status read-back */
    ATTN_ERR_SCALE = 11,         /* scale is NaN, infinite, or larger than 2e38 in magnitude */
    ATTN_ERR_DEVICE_BOUNDS = 12  /* bounds-checking debug build only: a kernel found an index or
                                    TMA coordinate out of range and skipped the access
                                    (reported by attn_device_status) */
} attn_status;

typedef enum attn_dtype {
    ATTN_F32 = 0,  /* fp32 in/out; exact fp32 FMA on CUDA cores (no TF32) */
    ATTN_BF16 = 1  /* bf16 in/out; tcgen05 tensor-core products, fp32 accumulation */
} attn_dtype;

/*
 * attn_fwd -- O = softmax(scale * Q K^T [+ causal mask]) V and the row LSE.
 *
 *   q, k, v  [B,H,N,d] inputs in `dtype` (device, read only).
 *   o        [B,H,N,d] output in `dtype` (device, fully overwritten).  Must
 *            not overlap q, k or v.
 *   lse      [B,H,N] fp32 output, natural-log log-sum-exp of the scaled
 *            logits of each row (device, fully overwritten), or NULL to skip.
 *   B, H, N  batch, heads, sequence length; each >= 1, N < 2^31 and
 *            B*H*N*d < 2^62.  ATTN_BF16 also needs N <= 8388480 (65535*128,
 *            a tested-range cap, not an index limit) and
 *            B*H*ceil(N/256) < 2^31 (the kernels' 1-D grid of 256-row
 *            items); ATTN_F32 needs B*H <= 65535.
 *   d        head dimension: 64 or 128.
 *   scale    multiplier applied to Q.K before the softmax (1/sqrt(d) usually).
 *            Any finite value with |scale| <= 2e38: positive, negative (the
 *            softmax then favours the smallest dot products) or zero (every
 *            visible key weighs the same).  NaN, infinities and larger values
 *            return ATTN_ERR_SCALE.
 *   causal   0: every key is visible; non-zero: key j visible to row i iff j <= i.
 *   dtype    an attn_dtype value.
 *   stream   cudaStream_t (as void*).
 *
 * Returns ATTN_OK or the first validation / launch error.  Faults inside a
 * kernel are never used for signalling: a kernel whose internal wait runs out
 * records ATTN_ERR_DEVICE_TIMEOUT in the device status word and returns; read
 * it with attn_device_status().
 */
attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                     int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                     int dtype, void *stream);

/*
 * attn_fwd_noalloc -- attn_fwd for callers that must never allocate device
 * memory: for example a server whose own allocator owns every byte of the GPU,
 * or code running where a device allocation is forbidden or would synchronise
 * the device.  The pages have no counterpart; this is an interface addition.
 *
 * Arguments, results and validation are exactly those of attn_fwd, and it
 * runs the same kernels.  The one difference is where the kernels' scratch
 * memory lives.  attn_fwd obtains a device status word with cudaMalloc on its
 * first call per device.  This entry point uses a 256-byte file-scope
 * __device__ array that the library's CUDA module carries; every GPU that
 * loads the library holds it until the process exits.  The kernels need
 * 4 bytes of it (the status word) whatever B, H, N and d are, so no problem
 * size exceeds it.  No call makes a cudaMalloc, cudaFree or other allocating
 * call.
 *
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  Make that first call
 *     before capturing a stream into a CUDA graph.
 *   - Every call shares the one array and clears its status word (an
 *     asynchronous memset on `stream`) before launching.  Calls that overlap
 *     on the GPU (different streams, no ordering between them) race on it.
 *   - A bounded-wait timeout inside the kernel ends that launch early, and its
 *     outputs are then undefined.  The timeout is recorded only in this
 *     array, not in the word attn_device_status reads: read it with
 *     attn_fwd_noalloc_status, which allocates nothing either.
 */
attn_status attn_fwd_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                             int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                             int causal, int dtype, void *stream);

/*
 * attn_fwd_noalloc_status -- synchronise `stream`, then return and clear the
 * status word of attn_fwd_noalloc on the current device (word 0 of its static
 * array): ATTN_OK, or ATTN_ERR_DEVICE_TIMEOUT if a kernel launched by
 * attn_fwd_noalloc gave up a bounded wait since the word was last cleared.
 * ATTN_ERR_CUDA if synchronising or reading back failed.  Like
 * attn_fwd_noalloc it allocates no device memory: the word is copied into
 * host stack memory.  Because attn_fwd_noalloc clears the word at the start
 * of each call, read it after the call to be checked and before the next one.
 */
attn_status attn_fwd_noalloc_status(void *stream);

/*
 * attn_fwd_host_workspace_bytes -- bytes of device workspace attn_fwd_host
 * needs for this problem: room for Q, K, V and O in `dtype` and LSE in fp32,
 * each rounded up to 256 bytes.  0 when the arguments are invalid for
 * attn_fwd.
 */
size_t attn_fwd_host_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d, int dtype);

/*
 * attn_fwd_host -- attn_fwd from and to host memory.  Q, K and V are copied to
 * the device, the forward runs, and O and LSE are copied back.  The problem
 * is cut into chunks of consecutive (batch, head) pairs (up to 8, each about
 * 16 MB of copies or more).  Copying chunk c+1 in, computing chunk c and
 * copying chunk c-1 out run at the same time: the library keeps two copy
 * streams per device beside `stream`, ordered with events, and issues one
 * cudaMemcpyAsync per tensor and chunk.
 *
 *   q, k, v    [B,H,N,d] inputs in `dtype`, read only.  Host memory: page-locked
 *              (pinned) memory lets the copies overlap; pageable memory works,
 *              but its copies do not overlap.  Any pointer the CUDA runtime can
 *              copy from with cudaMemcpyDefault is accepted.
 *   o          [B,H,N,d] output in `dtype`, host memory as above, fully
 *              overwritten.
 *   lse        [B,H,N] fp32 output in host memory, or NULL to skip it.
 *   workspace  device memory of the current device, 256-byte aligned, at least
 *              attn_fwd_host_workspace_bytes(B,H,N,d,dtype) bytes.  The caller
 *              owns it; the call holds no reference once the work is done.
 *   workspace_bytes  its size.
 *   B, H, N, d, scale, causal, dtype, stream   as attn_fwd.
 *
 * Asynchronous like attn_fwd.  The work is ordered after what `stream` already
 * holds, and everything the call enqueues, the last copy out included, is
 * ordered before later work on `stream`.  The outputs are on the host once
 * `stream` has been synchronised.  The first call on a device creates the two
 * copy streams and 18 events.  Calls from several host threads are
 * serialised while they enqueue.  No device memory is allocated.
 * Returns ATTN_OK or the first validation / launch error: ATTN_ERR_NULL for a
 * NULL q, k, v, o or workspace; ATTN_ERR_SHAPE also for a workspace that is
 * too small; ATTN_ERR_ALIGN for a workspace that is not 256-byte aligned.
 */
attn_status attn_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                          int64_t B, int64_t H, int64_t N, int64_t d, float scale, int causal,
                          int dtype, void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_row_softmax -- row softmax of a [rows, width] fp32 matrix in one pass
 * over the row with a running maximum and sum (page "14. Triton and kernel
 * fusion", section "Fusion", and its exercise on rows too long for one
 * block; the online identity of the attention page, section 2).
 *
 *   x     [rows, width] fp32 input (device, read only), rows contiguous.
 *   y     [rows, width] fp32 output (device, fully overwritten), may equal x.
 *   lse   [rows] fp32 natural-log log-sum-exp per row, or NULL.
 *   rows, width >= 1, rows*width < 2^62.  Any width is accepted.
 *   -inf entries get probability 0; a row of -inf only gets all zeros and
 *   LSE = -inf.  A few very long rows (more than 12288 floats, fewer rows than twice
 *   the SM count, 16-byte aligned) are split over a thread-block cluster of
 *   up to 8 CTAs per row.
 * Returns ATTN_OK or a validation / launch error (as attn_fwd).
 */
attn_status attn_row_softmax(const float *x, float *y, float *lse, int64_t rows,
                             int64_t width, void *stream);

/*
 * attn_bwd -- gradients of attn_fwd: dQ, dK, dV from Q, K, V, the forward's O
 * and LSE, and dO.  The pages give no attention backward; this is the exact
 * derivative of the forward formula:
 *     P_ij = exp(scale q_i.k_j - LSE_i) (0 for masked keys),  D_i = dO_i . O_i,
 *     dS_ij = P_ij (dO_i . v_j - D_i),
 *     dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
 * No atomics: one pass over key blocks for dK and dV, one over query blocks
 * for dQ.  ATTN_F32: exact fp32 arithmetic on CUDA cores.  ATTN_BF16: tcgen05
 * tensor cores, S and dP recomputed per block pair, P and dS rounded to bf16
 * for the products, every sum accumulated in fp32, outputs rounded once.
 *
 *   q, k, v, o, dout   [B,H,N,d] in `dtype` (device, read only); o is the
 *                      forward's output.
 *   lse                [B,H,N] fp32 from the forward (device, read only).
 *   delta              [B,H,N] fp32 workspace owned by the caller (device,
 *                      overwritten with D); the call allocates nothing.
 *   dq, dk, dv         [B,H,N,d] outputs in `dtype` (device, fully overwritten).
 *   B, H, N, d, scale, causal, dtype, stream   as attn_fwd; B*H <= 65535
 *                      (any finite scale, as attn_fwd).
 * All pointers 16-byte aligned.  Returns ATTN_OK or a validation / launch error.
 */
attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                     const void *dout, const float *lse, float *delta, void *dq, void *dk,
                     void *dv, int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                     int causal, int dtype, void *stream);

/*
 * attn_add_rmsnorm -- fused residual add + RMSNorm (page "14. Triton and
 * kernel fusion", section "Fused residual add + RMSNorm"; the RMSNorm formula
 * of page "TritonForge"):
 *
 *     h       = x + residual          (h = x when residual is NULL)
 *     out     = h / sqrt(mean_c h_c^2 + eps) * weight
 *     res_out = h                     (written only with a residual)
 *
 *   x, residual   [rows, width] inputs in `dtype` (device, read only);
 *                 residual may be NULL.
 *   weight        [width] scale in `dtype` (device, read only).
 *   out           [rows, width] output in `dtype` (device, fully overwritten).
 *   res_out       [rows, width] output in `dtype`, required with a residual,
 *                 ignored without one.  out and res_out must not overlap the
 *                 inputs.
 *   rows, width   >= 1, width < 2^31.  eps >= 0 added to the mean square.
 *   dtype         ATTN_F32 or ATTN_BF16; arithmetic is fp32 either way and bf16
 *                 outputs are rounded (nearest even) once, on store.
 * All pointers 16-byte aligned device memory.  Returns ATTN_OK or a
 * validation / launch error (as attn_fwd).
 */
attn_status attn_add_rmsnorm(const void *x, const void *residual, const void *weight, void *out,
                             void *res_out, int64_t rows, int64_t width, float eps, int dtype,
                             void *stream);

/*
 * attn_device_status -- synchronise `stream`, then return and clear the
 * current device's status word: ATTN_OK, or ATTN_ERR_DEVICE_TIMEOUT if any
 * kernel of this library gave up a bounded wait since the last read.
 * ATTN_ERR_CUDA if synchronising or reading back failed.  In the
 * bounds-checking debug build (the same sources compiled with
 * -DATTN_DEBUG_BOUNDS into a library of its own) the forward kernels check
 * every global index and TMA coordinate against B*H, N and d before use; a
 * failed check skips the access and this call then returns
 * ATTN_ERR_DEVICE_BOUNDS.
 */
attn_status attn_device_status(void *stream);

/*
 * attn_selftest_wait_timeout -- launch one tiny kernel that waits, with the
 * library's bounded wait, on a barrier that nothing ever signals, using a
 * limit of `timeout_ns` nanoseconds (clamped to [1e3, 5e9]).  The kernel
 * gives up, records the timeout and returns; this call then returns what
 * attn_device_status() reads (ATTN_ERR_DEVICE_TIMEOUT when the error path
 * works).  Exists to test failure detection without faulting or hanging a GPU.
 */
attn_status attn_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/*
 * attn_last_cuda_error -- the CUDA runtime's message for the most recent CUDA
 * error this thread's calls into the library saw (for example why a launch was
 * rejected), or "no error".  Static string, never NULL.
 */
const char *attn_last_cuda_error(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *attn_status_string(int status);

/* Library ABI version: major*10000 + minor*100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_GB300_H */
