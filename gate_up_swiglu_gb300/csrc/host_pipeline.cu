// host_pipeline.cu -- forward + backward over host buffers, streamed through
// caller-provided device staging memory (swiglu_gateup_fwd_bwd_host).
//
// For callers whose fc1 buffer and incoming gradient live in host memory
// (offloaded activations, or data kept on the CPU side of the Grace-Blackwell
// link): instead of copying everything in, computing and copying everything
// out -- which leaves the link idle while the kernels run and the GPU idle
// while the link works -- row chunks go through a ring of `depth` staging
// slots on three streams, so the copy-in of one chunk, the kernels of another
// and the copy-out of a third overlap, and both link directions are busy at
// once.  Each slot holds a chunk's x (overwritten by its gradient: the
// backward runs in place, which gives the out-of-place result bit for bit),
// dy and y.  Every element is computed by swiglu_gateup_fwd /
// swiglu_gateup_bwd; this file only orders copies and launches.
#include <cuda_runtime.h>

#include <cstdint>

#include "abi_internal.h"
#include "swiglu.h"

namespace {

constexpr int kMaxDepth = 8;
constexpr size_t kSlotAlign = 256;

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Byte sizes of one slot's x, dy and y regions (each rounded to kSlotAlign),
// false on overflow.
bool slot_layout(int64_t chunk_rows, int64_t n, int eb, size_t &bx, size_t &bdy, size_t &slot) {
    size_t row_x, rows_x;
    if (__builtin_mul_overflow((size_t)(2 * n), (size_t)eb, &row_x)) return false;
    if (__builtin_mul_overflow(row_x, (size_t)chunk_rows, &rows_x)) return false;
    bx = round_up(rows_x, kSlotAlign);
    bdy = round_up(rows_x / 2, kSlotAlign);
    return !__builtin_add_overflow(bx, 2 * bdy, &slot);
}

int elem_bytes(swiglu_dtype_t dt) { return dt == SWIGLU_F32 ? 4 : dt == SWIGLU_BF16 ? 2 : 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + nb && pb < pa + na;
}

}  // namespace

extern "C" swiglu_status_t swiglu_gateup_fwd_bwd_host_staging_size(int64_t chunk_rows, int64_t n,
                                                                    swiglu_dtype_t dtype, int depth,
                                                                    size_t *bytes) {
    if (bytes == nullptr) return SWIGLU_ERR_NULL;
    const int eb = elem_bytes(dtype);
    if (eb == 0) return SWIGLU_ERR_DTYPE;
    if (chunk_rows < 1 || n < 1 || n > SWIGLU_MAX_N || depth < 1 || depth > kMaxDepth)
        return SWIGLU_ERR_SHAPE;
    size_t bx, bdy, slot, total;
    if (!slot_layout(chunk_rows, n, eb, bx, bdy, slot)) return SWIGLU_ERR_SHAPE;
    if (__builtin_mul_overflow(slot, (size_t)depth, &total)) return SWIGLU_ERR_SHAPE;
    *bytes = total;
    return SWIGLU_OK;
}

extern "C" swiglu_status_t swiglu_gateup_fwd_bwd_host(
    const void *x_host, const void *dy_host, void *y_host, void *dx_host, int64_t rows, int64_t n,
    swiglu_dtype_t dtype, void *staging, size_t staging_bytes, int64_t chunk_rows, int depth,
    swiglu_stream_t h2d, swiglu_stream_t compute, swiglu_stream_t d2h) {
    const int eb = elem_bytes(dtype);
    if (eb == 0) return SWIGLU_ERR_DTYPE;
    if (rows < 0 || n < 0 || n > SWIGLU_MAX_N) return SWIGLU_ERR_SHAPE;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    if (x_host == nullptr || dy_host == nullptr || y_host == nullptr || dx_host == nullptr ||
        staging == nullptr)
        return SWIGLU_ERR_NULL;
    if (chunk_rows < 1 || depth < 1 || depth > kMaxDepth) return SWIGLU_ERR_SHAPE;
    if (chunk_rows > rows) chunk_rows = rows;
    size_t bx, bdy, slot, need;
    if (!slot_layout(chunk_rows, n, eb, bx, bdy, slot) ||
        __builtin_mul_overflow(slot, (size_t)depth, &need))
        return SWIGLU_ERR_SHAPE;
    if (staging_bytes < need || (uintptr_t)staging % kSlotAlign != 0) return SWIGLU_ERR_WORKSPACE;
    // whole host tensors: x, dx [rows, 2n]; dy, y [rows, n]
    size_t hx, hy;
    if (__builtin_mul_overflow((size_t)rows, (size_t)(2 * n) * eb, &hx)) return SWIGLU_ERR_SHAPE;
    hy = hx / 2;
    if (overlap(y_host, hy, x_host, hx) || overlap(y_host, hy, dy_host, hy) ||
        overlap(dx_host, hx, x_host, hx) || overlap(dx_host, hx, dy_host, hy) ||
        overlap(y_host, hy, dx_host, hx))
        return SWIGLU_ERR_ALIAS;

    cudaStream_t s_in = reinterpret_cast<cudaStream_t>(h2d);
    cudaStream_t s_k = reinterpret_cast<cudaStream_t>(compute);
    cudaStream_t s_out = reinterpret_cast<cudaStream_t>(d2h);
    cudaEvent_t loaded[kMaxDepth] = {}, done[kMaxDepth] = {}, drained[kMaxDepth] = {};
    cudaError_t e = cudaSuccess;
    swiglu_status_t st = SWIGLU_OK;
    for (int i = 0; i < depth && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&loaded[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&done[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&drained[i], cudaEventDisableTiming);
    }
    const char *xh = static_cast<const char *>(x_host);
    const char *dyh = static_cast<const char *>(dy_host);
    char *yh = static_cast<char *>(y_host);
    char *dxh = static_cast<char *>(dx_host);
    const size_t row_x = (size_t)(2 * n) * eb, row_y = (size_t)n * eb;
    int64_t chunk = 0;
    for (int64_t r0 = 0; r0 < rows && e == cudaSuccess && st == SWIGLU_OK; r0 += chunk_rows, ++chunk) {
        const int64_t m = rows - r0 < chunk_rows ? rows - r0 : chunk_rows;
        const int s = (int)(chunk % depth);
        char *sx = static_cast<char *>(staging) + (size_t)s * slot;
        char *sdy = sx + bx;
        char *sy = sdy + bdy;
        // a slot is refilled only once its previous results have left for the host
        if (chunk >= depth) e = cudaStreamWaitEvent(s_in, drained[s], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(sx, xh + (size_t)r0 * row_x, (size_t)m * row_x, cudaMemcpyHostToDevice, s_in);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(sdy, dyh + (size_t)r0 * row_y, (size_t)m * row_y, cudaMemcpyHostToDevice,
                                s_in);
        if (e == cudaSuccess) e = cudaEventRecord(loaded[s], s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_k, loaded[s], 0);
        if (e != cudaSuccess) break;
        st = swiglu_gateup_fwd(sx, sy, m, n, 2 * n, n, dtype, compute);
        if (st == SWIGLU_OK)
            st = swiglu_gateup_bwd(sdy, sx, nullptr, m, n, n, 2 * n, 0, dtype, 1, compute);
        if (st != SWIGLU_OK) break;
        e = cudaEventRecord(done[s], s_k);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, done[s], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(yh + (size_t)r0 * row_y, sy, (size_t)m * row_y, cudaMemcpyDeviceToHost, s_out);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dxh + (size_t)r0 * row_x, sx, (size_t)m * row_x, cudaMemcpyDeviceToHost, s_out);
        if (e == cudaSuccess) e = cudaEventRecord(drained[s], s_out);
    }
    // results are in host memory once the copy-out stream drains; on an error
    // every stream is drained before the events go
    cudaError_t e2 = cudaStreamSynchronize(s_out);
    if (e != cudaSuccess || st != SWIGLU_OK) {
        cudaStreamSynchronize(s_in);
        cudaStreamSynchronize(s_k);
    }
    for (int i = 0; i < depth; ++i) {
        if (loaded[i]) cudaEventDestroy(loaded[i]);
        if (done[i]) cudaEventDestroy(done[i]);
        if (drained[i]) cudaEventDestroy(drained[i]);
    }
    if (st != SWIGLU_OK) return st;
    if (e == cudaSuccess) e = e2;
    if (e != cudaSuccess) {
        swiglu_abi::record_cuda_error((int)e);
        return SWIGLU_ERR_CUDA;
    }
    return SWIGLU_OK;
}
