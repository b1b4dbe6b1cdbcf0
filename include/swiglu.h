/*
 * swiglu.h -- C ABI of libswiglu, the fused gate-up SwiGLU for GB300 (sm_103a).
 *
 * The operation (Liger-Kernel Megatron SwiGLU page, §Background): Megatron's
 * linear_fc1 produces a single [s, b, 2n] (or [tokens, 2n]) buffer x whose
 * columns [0, n) hold the gate g and columns [n, 2n) the up projection u.  The
 * fused kernels read both halves of each row through a column offset into that
 * one buffer -- no chunk, copy or concatenation.  3D inputs are passed as
 * rows = s * b rows of one common row stride (§Megatron feature compatibility:
 * 2D and 3D inputs).
 *
 *   forward   y[r, j]      = silu(g) * u,  silu(g) = g * sigmoid(g)
 *   backward  dx[r, j]     = dy[r, j] * u * s * (1 + g * (1 - s))    (d gate)
 *             dx[r, n + j] = dy[r, j] * g * s                        (d up)
 *   with g = x[r, j], u = x[r, n + j], s = sigmoid(g), 0 <= j < n.
 *
 * The backward recomputes the sigmoid from the saved fc1 buffer and may write
 * its result over that buffer (§Optional: in_place=True).  The page prints no
 * backward formula; the one above is the analytic derivative of silu(g) * u.
 * The plain entry points take no bias (§Scope: bias=None); the bias and
 * per-token-weight variants further down are the page's named follow-ups.
 *
 * Conventions shared by every entry point:
 *   - All pointers are DEVICE pointers owned by the caller (the *_host
 *     arguments of swiglu_gateup_fwd_bwd_host excepted).  No call allocates
 *     or frees memory, and no state survives a call; the one piece of device
 *     memory the library itself holds is the fixed scratch array of
 *     swiglu_gateup_bias_bwd_noalloc (below), part of the loaded module.
 *   - Sizes and row strides are counted in ELEMENTS of the dtype; within a row
 *     elements are contiguous.  Row r of x starts at x + r * x_row_stride.
 *   - Every pointer is aligned to its element size: 2 bytes for bf16, 4 for
 *     fp32 and for the fp32 per-token weights and their gradient (else
 *     SWIGLU_ERR_STRIDE, before anything is launched).
 *   - All tensors of one call share one dtype.  Arithmetic is fp32; each result
 *     is rounded once to the dtype (round to nearest even).
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and runs
 *     asynchronously; the call returns after the launch.  The current CUDA
 *     device must be the one that owns the pointers.
 *   - No call synchronises, allocates or waits on the host -- except the
 *     host-buffer pipeline swiglu_gateup_fwd_bwd_host, which by design returns
 *     once its results are in host memory -- so every other entry point can
 *     be captured into a CUDA graph (stream capture) and replayed; the first
 *     call on a device caches a few device attributes, which is best done once
 *     eagerly before capturing.
 *   - Every argument is checked on the host before anything is launched; on
 *     any error nothing is written and nothing is launched.  rows == 0 or
 *     n == 0 is a valid empty call (returns SWIGLU_OK, touches nothing, and
 *     accepts NULL pointers).
 */
#ifndef LIBSWIGLU_SWIGLU_H
#define LIBSWIGLU_SWIGLU_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream (a pointer to the CUDA driver's stream
 * object), declared here so that this header does not need the CUDA headers. */
typedef struct CUstream_st *swiglu_stream_t;

typedef enum {
    SWIGLU_F32 = 0,  /* IEEE binary32 */
    SWIGLU_BF16 = 1  /* bfloat16: top 16 bits of a binary32 */
} swiglu_dtype_t;

typedef enum {
    SWIGLU_OK = 0,
    SWIGLU_ERR_NULL = -1,   /* a required pointer is NULL                       */
    SWIGLU_ERR_DTYPE = -2,  /* dtype is not a swiglu_dtype_t value              */
    SWIGLU_ERR_SHAPE = -3,  /* rows or n negative, or n > SWIGLU_MAX_N, or the
                               byte extent of a tensor overflows int64          */
    SWIGLU_ERR_STRIDE = -4, /* a row stride is shorter than its row, or a
                               pointer is not aligned to its element size      */
    SWIGLU_ERR_ALIAS = -5,  /* an output overlaps an input it must not overlap  */
    SWIGLU_ERR_CUDA = -6,   /* the CUDA runtime reported an error; see
                               swiglu_last_cuda_error()                         */
    SWIGLU_ERR_WORKSPACE = -7 /* workspace smaller than required, or not
                                 16-byte aligned                                */
} swiglu_status_t;

/* Largest supported n (columns per half). */
#define SWIGLU_MAX_N ((int64_t)1 << 30)

/*
 * Forward: y[r, j] = silu(x[r, j]) * x[r, n + j] for r < rows, j < n.
 *   x  [rows, 2n], row stride x_row_stride >= 2n   (read only)
 *   y  [rows, n],  row stride y_row_stride >= n    (written)
 * The byte range spanned by y must not overlap the one spanned by x
 * (SWIGLU_ERR_ALIAS).
 */
swiglu_status_t swiglu_gateup_fwd(const void *x, void *y, int64_t rows, int64_t n,
                                  int64_t x_row_stride, int64_t y_row_stride,
                                  swiglu_dtype_t dtype, swiglu_stream_t stream);

/*
 * Backward: dx[r, j] = d gate, dx[r, n + j] = d up (formulas above).
 *   dy [rows, n],  row stride dy_row_stride >= n   (read only)
 *   x  [rows, 2n], row stride x_row_stride >= 2n   (the saved fc1 buffer)
 *   dx [rows, 2n], row stride dx_row_stride >= 2n  (written)
 * in_place == 0: dx must not overlap x or dy (SWIGLU_ERR_ALIAS).
 * in_place != 0: the gradient is written over x.  dx must be NULL or equal to
 *   x (else SWIGLU_ERR_ALIAS) and dx_row_stride must be 0 or equal to
 *   x_row_stride (else SWIGLU_ERR_STRIDE); dy must not overlap x
 *   (SWIGLU_ERR_ALIAS).  The in-place result is bit-identical to the
 *   out-of-place one.  Afterwards x no longer holds the forward input: a second
 *   backward over the same buffer computes garbage, which the library cannot
 *   detect (the caller must guard against it, as the page's known issue 1 says).
 */
swiglu_status_t swiglu_gateup_bwd(const void *dy, const void *x, void *dx, int64_t rows,
                                  int64_t n, int64_t dy_row_stride, int64_t x_row_stride,
                                  int64_t dx_row_stride, swiglu_dtype_t dtype, int in_place,
                                  swiglu_stream_t stream);

/*
 * Two-tensor form (Liger-Kernel Megatron SwiGLU page, §Background: the gate
 * and the up projection arrive as two separate tensors a and b, as HuggingFace
 * models produce them).  Same arithmetic as the fused form:
 *   c[r, j]  = silu(a[r, j]) * b[r, j]
 *   da[r, j] = dc * b * s * (1 + a * (1 - s)),  db[r, j] = dc * a * s
 * for r < rows, j < n; every tensor is [rows, n] with its own row stride
 * (>= n, elements).  a and b may overlap each other (they are only read).
 *   forward:  c must not overlap a or b (SWIGLU_ERR_ALIAS).
 *   backward: da may be exactly a (same pointer and stride) and db exactly b,
 *             giving the in-place form (bit-identical to the out-of-place one);
 *             apart from that an output may overlap no input and not the other
 *             output (SWIGLU_ERR_ALIAS).
 * For the fused [rows, 2n] layout use swiglu_gateup_*: its halves interleave
 * row by row, which these byte-range overlap rules would reject.
 */
swiglu_status_t swiglu_silu_mul_fwd(const void *a, const void *b, void *c, int64_t rows, int64_t n,
                                    int64_t a_row_stride, int64_t b_row_stride,
                                    int64_t c_row_stride, swiglu_dtype_t dtype,
                                    swiglu_stream_t stream);

swiglu_status_t swiglu_silu_mul_bwd(const void *dc, const void *a, const void *b, void *da,
                                    void *db, int64_t rows, int64_t n, int64_t dc_row_stride,
                                    int64_t a_row_stride, int64_t b_row_stride,
                                    int64_t da_row_stride, int64_t db_row_stride,
                                    swiglu_dtype_t dtype, swiglu_stream_t stream);

/*
 * Per-token weights (Liger-Kernel Megatron SwiGLU page, §Known issues 2: MoE
 * routed experts scale each token's activation by its routing weight and need a
 * per_token_scale-aware kernel).  w and dw are fp32 vectors of `rows` floats
 * (unit stride); everything else is as in swiglu_gateup_fwd / _bwd.
 *   forward   y[r, j]  = w[r] * silu(g) * u
 *   backward  dx       = the plain backward with dy[r, :] scaled by w[r]
 *             dw[r]    = sum_j dy[r, j] * silu(g[r, j]) * u[r, j]   (fp32)
 * y / dx / dw may not overlap w; dw may overlap nothing.  dw[r] is summed in
 * fp32 in a fixed order (deterministic).  With n == 0 the backward sets dw to
 * zero.
 */
swiglu_status_t swiglu_gateup_weighted_fwd(const void *x, const float *w, void *y, int64_t rows,
                                           int64_t n, int64_t x_row_stride, int64_t y_row_stride,
                                           swiglu_dtype_t dtype, swiglu_stream_t stream);

swiglu_status_t swiglu_gateup_weighted_bwd(const void *dy, const void *x, const float *w, void *dx,
                                           float *dw, int64_t rows, int64_t n,
                                           int64_t dy_row_stride, int64_t x_row_stride,
                                           int64_t dx_row_stride, swiglu_dtype_t dtype,
                                           int in_place, swiglu_stream_t stream);

/*
 * Bias (Liger-Kernel Megatron SwiGLU page, §Scope: Megatron's bias_swiglu_impl
 * adds a [2n] bias before the activation; the page's kernels fall back when a
 * bias is given).  bias and dbias are contiguous [2n] vectors of x's dtype:
 *   forward   y[r, j]  = silu(g + bias[j]) * (u + bias[n + j])
 *   backward  dx       = the plain backward at (g + bias[j], u + bias[n + j])
 *             dbias[k] = sum_r dx[r, k] for k < 2n (fp32 sum of the unrounded
 *                        fp32 gradients, rounded once; fixed order)
 * The backward needs a caller-provided device workspace of at least
 * swiglu_gateup_bias_bwd_workspace_size(rows, n) bytes, 16-byte aligned; it
 * holds per-row-group column sums and is overwritten (no state survives the
 * call).  The size depends on the current device's SM count.  y / dx / dbias
 * / workspace may not overlap bias, and dbias and the workspace overlap
 * nothing.  With rows == 0 (and n > 0) the backward sets dbias to zero.
 */
swiglu_status_t swiglu_gateup_bias_fwd(const void *x, const void *bias, void *y, int64_t rows,
                                       int64_t n, int64_t x_row_stride, int64_t y_row_stride,
                                       swiglu_dtype_t dtype, swiglu_stream_t stream);

swiglu_status_t swiglu_gateup_bias_bwd_workspace_size(int64_t rows, int64_t n, size_t *bytes);

swiglu_status_t swiglu_gateup_bias_bwd(const void *dy, const void *x, const void *bias, void *dx,
                                       void *dbias, void *workspace, size_t workspace_bytes,
                                       int64_t rows, int64_t n, int64_t dy_row_stride,
                                       int64_t x_row_stride, int64_t dx_row_stride,
                                       swiglu_dtype_t dtype, int in_place,
                                       swiglu_stream_t stream);

/*
 * Per-token weights and bias together (Liger-Kernel Megatron SwiGLU page,
 * §Scope and §Known issues 2: the MoE routed experts' weighted_bias_swiglu_impl
 * takes both).  bias / dbias as in swiglu_gateup_bias_*, w / dw as in
 * swiglu_gateup_weighted_*:
 *   forward   y[r, j]  = w[r] * silu(g + bias[j]) * (u + bias[n + j])
 *   backward  dx       = the bias backward with dy[r, :] scaled by w[r]
 *             dbias[k] = sum_r dx[r, k]                      (as for the bias form)
 *             dw[r]    = sum_j dy[r, j] * silu(g + bias[j]) * (u + bias[n + j])
 * Both sums run in fp32 in a fixed order (deterministic).  The backward needs
 * a device workspace of at least
 * swiglu_gateup_weighted_bias_bwd_workspace_size(rows, n) bytes, 16-byte
 * aligned: the bias form's column sums plus one fp32 partial of dw per row and
 * column tile (tiles of 2048 columns, or 1024 when the operands allow no pack
 * wider than 4 bytes; the size covers both).  Aliasing: y / dx / dbias / dw / workspace may overlap
 * neither bias nor w; dbias, dw and the workspace overlap nothing.
 * With rows == 0 (n > 0) the backward sets dbias to zero; with n == 0
 * (rows > 0) it sets dw to zero.
 */
swiglu_status_t swiglu_gateup_weighted_bias_fwd(const void *x, const void *bias, const float *w,
                                                void *y, int64_t rows, int64_t n,
                                                int64_t x_row_stride, int64_t y_row_stride,
                                                swiglu_dtype_t dtype, swiglu_stream_t stream);

swiglu_status_t swiglu_gateup_weighted_bias_bwd_workspace_size(int64_t rows, int64_t n,
                                                               size_t *bytes);

swiglu_status_t swiglu_gateup_weighted_bias_bwd(
    const void *dy, const void *x, const void *bias, const float *w, void *dx, void *dbias,
    float *dw, void *workspace, size_t workspace_bytes, int64_t rows, int64_t n,
    int64_t dy_row_stride, int64_t x_row_stride, int64_t dx_row_stride, swiglu_dtype_t dtype,
    int in_place, swiglu_stream_t stream);

/*
 * Allocation-free bias backward.  The page has no counterpart: this is an
 * addition for callers that cannot hand the library any device memory -- for
 * example code running under an engine that plans all device memory ahead of
 * time and forbids allocation during a step, plugin interfaces whose host owns
 * the allocator and exposes none to the plugin, or latency-bound paths that
 * cannot afford cudaMalloc's implicit synchronisation.
 *
 * Same arguments, results and checks as swiglu_gateup_bias_bwd minus the
 * workspace: the column-sum scratch lives in a fixed file-scope device array
 * of SWIGLU_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.  The call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *   - A problem whose scratch need (swiglu_gateup_bias_bwd_workspace_size)
 *     exceeds SWIGLU_NOALLOC_SCRATCH_BYTES is rejected with
 *     SWIGLU_ERR_WORKSPACE before anything is launched.  For any rows and n
 *     the need is at most max(2 * SMs * 2048 * 8, 8 n) bytes, SMs being the
 *     device's multiprocessor count (4.75 MiB on a 152-SM GB300, so every
 *     n <= 2^21 fits); it reaches 8 n only when one row group spans the
 *     whole matrix (n above 2 * SMs * 2048).
 *   - The first call in a CUDA context (per device, and again after a
 *     cudaDeviceReset) looks up the array's device address with that device
 *     current (cudaGetSymbolAddress); make that first call before any stream
 *     capture.
 *   - All calls share the one array, which keeps the last call's contents (the
 *     kernels overwrite every scratch value they later read, so nothing needs
 *     to start at zero).  Calls that overlap on the GPU -- on different streams,
 *     or from different threads without ordering -- race on it: serialise them.
 */
#define SWIGLU_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

swiglu_status_t swiglu_gateup_bias_bwd_noalloc(const void *dy, const void *x, const void *bias,
                                               void *dx, void *dbias, int64_t rows, int64_t n,
                                               int64_t dy_row_stride, int64_t x_row_stride,
                                               int64_t dx_row_stride, swiglu_dtype_t dtype,
                                               int in_place, swiglu_stream_t stream);

/*
 * linear_fc1 with the activation fused into its epilogue (tensor cores).
 * Megatron's MLP produces the [tokens, 2n] buffer as fc1 = X W^T
 * (Liger-Kernel Megatron SwiGLU page, §Background: linear_fc1 is one
 * ColumnParallelLinear whose output holds gate and up side by side); this call
 * computes
 *   y[m, j] = silu(fc1[m, j]) * fc1[m, n + j],   fc1 = X W^T (fp32 accumulate)
 * directly from the fp32 accumulators, without writing fc1 to memory unless
 * x_out is given (then fc1, rounded to bf16, is stored there too, as a training
 * step saves it for swiglu_gateup_bwd).  bias-free, bf16 only.
 *   X     [M, K]  bf16, row-major, contiguous         (read)
 *   W     [2n, K] bf16, row-major (nn.Linear weight: rows [0, n) gate,
 *                 rows [n, 2n) up), contiguous         (read)
 *   y     [M, n]  bf16, contiguous                     (written)
 *   x_out [M, 2n] bf16, contiguous, or NULL            (written)
 * Requirements: n and K multiples of 8, K >= 8, M, K, 2n below 2^31 and
 * ceil(M / 256) * ceil(n / 128) (the tile count) below 2^30 (else
 * SWIGLU_ERR_SHAPE); all pointers 16-byte aligned
 * (else SWIGLU_ERR_STRIDE); outputs overlap no input and each other
 * (SWIGLU_ERR_ALIAS); dtype SWIGLU_BF16 (else SWIGLU_ERR_DTYPE).  M == 0 or
 * n == 0 is an empty call.  The launch holds one 2-CTA cluster per tile; the
 * pairs that fit run and take the other tiles by cancelling launches that
 * have not started, so the result does not depend on how many SMs other
 * streams' work leaves free.  Each CTA bounds its internal waits; a wait that
 * times out, or a cancellation answer that names no tile of the grid, raises
 * the flag read by swiglu_fc1_timeout_flag (results of that call are then
 * undefined).
 */
swiglu_status_t swiglu_fc1_fwd(const void *x_in, const void *w, void *y, void *x_out, int64_t M,
                               int64_t n, int64_t K, swiglu_dtype_t dtype, swiglu_stream_t stream);

/* *flag = 1 if any swiglu_fc1_fwd launch so far gave up on an internal wait,
 * else 0.  Synchronises with the current device. */
swiglu_status_t swiglu_fc1_timeout_flag(int *flag);

/*
 * Forward and backward over HOST buffers, end to end.  The page has no
 * counterpart (its kernels take device tensors); this serves callers whose fc1
 * buffer and incoming gradient live in host memory -- offloaded activations,
 * or tensors kept on the CPU side of the Grace-Blackwell link -- with the same
 * results as swiglu_gateup_fwd followed by the out-of-place swiglu_gateup_bwd:
 *   y_host  = forward(x_host),  dx_host = backward(dy_host, x_host)
 *   x_host  [rows, 2n], dy_host [rows, n]   host memory, read
 *   y_host  [rows, n],  dx_host [rows, 2n]  host memory, written
 * All four are contiguous (row strides 2n / n), may overlap none of the others,
 * and should be page-locked (cudaHostAlloc / cudaHostRegister): pageable
 * memory gives the same results without the overlap.
 * Rows go through the device in chunks of chunk_rows (>= 1), `depth` chunks
 * (1 ... 8) in flight: chunk i is copied in on stream h2d, computed on stream
 * compute (forward, then the backward in place over the staged x, which is
 * bit-identical to the out-of-place one) and copied out on stream d2h, so
 * copies in, kernels and copies out of different chunks overlap.  The three
 * streams may be the same stream (then nothing overlaps).
 *   staging  caller-owned DEVICE memory of at least
 *            swiglu_gateup_fwd_bwd_host_staging_size(chunk_rows, n, dtype,
 *            depth, &bytes) bytes, 256-byte aligned (else SWIGLU_ERR_WORKSPACE);
 *            its contents on return are unspecified.
 * The call allocates no device memory; it creates and destroys 3 * depth CUDA
 * events, and it blocks until every result is in host memory (it waits on
 * the three streams), so it cannot be captured into a CUDA graph.  One
 * memcpy per tensor per chunk; no batched copies.
 */
swiglu_status_t swiglu_gateup_fwd_bwd_host_staging_size(int64_t chunk_rows, int64_t n,
                                                        swiglu_dtype_t dtype, int depth,
                                                        size_t *bytes);

swiglu_status_t swiglu_gateup_fwd_bwd_host(const void *x_host, const void *dy_host, void *y_host,
                                           void *dx_host, int64_t rows, int64_t n,
                                           swiglu_dtype_t dtype, void *staging,
                                           size_t staging_bytes, int64_t chunk_rows, int depth,
                                           swiglu_stream_t h2d, swiglu_stream_t compute,
                                           swiglu_stream_t d2h);

/* Static English text for a status code; never NULL. */
const char *swiglu_status_string(swiglu_status_t status);

/* The cudaError_t value behind the calling thread's most recent
 * SWIGLU_ERR_CUDA (0 if there was none). */
int swiglu_last_cuda_error(void);

/* ABI version: incremented when a signature or a convention above changes. */
int swiglu_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBSWIGLU_SWIGLU_H */
