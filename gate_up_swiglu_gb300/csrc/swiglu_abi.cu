// swiglu_abi.cu -- host side of libswiglu: argument checks, pack-width and
// grid selection, launches.  The C declarations and their contract are in
// include/swiglu.h; the kernels are in swiglu_kernels.cuh.
//
// Every argument is checked before any CUDA call is made, so a rejected call
// launches nothing, writes nothing and needs no GPU.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>

#include "swiglu.h"
#include "swiglu_kernels.cuh"

namespace {

constexpr int kMaxDevices = 64;
thread_local int g_last_cuda_error = 0;

swiglu_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return SWIGLU_ERR_CUDA;
}

int elem_bytes(swiglu_dtype_t dt) {
    switch (dt) {
        case SWIGLU_F32: return 4;
        case SWIGLU_BF16: return 2;
    }
    return 0;
}

// Byte extent [lo, hi) of a [rows, cols] tensor with the given row stride.
struct Span {
    uintptr_t lo, hi;
};

bool span_of(const void *p, int64_t rows, int64_t cols, int64_t stride, int eb, Span &s) {
    // (rows - 1) * stride + cols elements, times eb bytes, must fit int64
    int64_t last, elems, bytes;
    if (__builtin_mul_overflow(rows - 1, stride, &last)) return false;
    if (__builtin_add_overflow(last, cols, &elems)) return false;
    if (__builtin_mul_overflow(elems, (int64_t)eb, &bytes)) return false;
    uintptr_t lo = (uintptr_t)p;
    if (lo + (uintptr_t)bytes < lo) return false;
    s.lo = lo;
    s.hi = lo + (uintptr_t)bytes;
    return true;
}

bool overlaps(const Span &a, const Span &b) { return a.lo < b.hi && b.lo < a.hi; }

// Widest pack (at most max_bytes: 32, 16, 8, 4 or 2 bytes) that divides n,
// every row stride and every base address; returns the elements per pack.
int pick_vec(int eb, int max_bytes, int64_t n, const int64_t *strides, int ns,
             const void *const *ptrs, int np) {
    for (int bytes = max_bytes; bytes > eb; bytes /= 2) {
        const int vec = bytes / eb;
        bool ok = (n % vec) == 0;
        for (int i = 0; ok && i < ns; ++i) ok = (strides[i] % vec) == 0;
        for (int i = 0; ok && i < np; ++i) ok = ((uintptr_t)ptrs[i] % (uintptr_t)bytes) == 0;
        if (ok) return vec;
    }
    return 1;
}

// Launch policy, chosen by sweeping pack width, unroll and resident CTAs per
// SM over the Megatron-shape, large-FFN and Llama-like bf16 workloads on a
// GB300: the forward is fastest with one 32-byte pack per operand in flight
// and 4 CTAs of 256 threads per SM, both backward forms with two 16-byte packs
// and 3 CTAs per SM.  Filling the SM with more CTAs lost 5-10 %.
struct Policy {
    int max_pack_bytes;
    int max_ctas_per_sm;
};
constexpr Policy kFwdPolicy = {32, 4};
constexpr Policy kBwdPolicy = {16, 3};

// Packs in flight per operand per thread: one 32-byte pack, two 16-byte
// packs, four 8-byte packs, else eight.
constexpr int unroll_for(int pack_bytes) {
    return pack_bytes >= 32 ? 1 : (pack_bytes >= 16 ? 2 : (pack_bytes >= 8 ? 4 : 8));
}

// Cache behaviour: inputs of the out-of-place kernels go through the
// read-only path without L1 allocation; the in-place backward reads what it
// writes, so it uses coherent loads.  Outputs are streaming stores.
constexpr int kLoadOutOfPlace = swiglu::kLdNC;
constexpr int kLoadInPlace = swiglu::kLdNoAlloc;
constexpr int kStore = swiglu::kStStream;

struct Device {
    int id;
    int sms;
};

cudaError_t current_device(Device &d) {
    static std::atomic<int> sm_cache[kMaxDevices];
    cudaError_t e = cudaGetDevice(&d.id);
    if (e != cudaSuccess) return e;
    if (d.id < 0 || d.id >= kMaxDevices) {
        return cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, d.id);
    }
    int sms = sm_cache[d.id].load(std::memory_order_relaxed);
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d.id);
        if (e != cudaSuccess) return e;
        sm_cache[d.id].store(sms, std::memory_order_relaxed);
    }
    d.sms = sms;
    return cudaSuccess;
}

// Resident CTAs per SM of `kernel` at kThreads threads, cached per device in
// the caller-provided table (one table per kernel instantiation).
template <typename K>
cudaError_t ctas_per_sm(K kernel, const Device &d, std::atomic<int> *cache, int &out) {
    int v = (d.id >= 0 && d.id < kMaxDevices) ? cache[d.id].load(std::memory_order_relaxed) : 0;
    if (v == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, swiglu::kThreads, 0);
        if (e != cudaSuccess) return e;
        if (v < 1) v = 1;
        if (d.id >= 0 && d.id < kMaxDevices) cache[d.id].store(v, std::memory_order_relaxed);
    }
    out = v;
    return cudaSuccess;
}

// Persistent grid: never more CTAs than there are units of U * kThreads packs,
// never more than fill every SM with resident CTAs.
template <int U>
int64_t grid_for(int64_t total_packs, const Device &d, int per_sm) {
    const int64_t per_cta = (int64_t)U * swiglu::kThreads;
    int64_t need = (total_packs + per_cta - 1) / per_cta;
    int64_t full = (int64_t)d.sms * per_sm;
    return need < full ? need : full;
}

template <typename E, int VEC>
swiglu_status_t launch_fwd(const void *x, void *y, int64_t rows, int64_t n, int64_t sx,
                           int64_t sy, cudaStream_t stream) {
    constexpr int U = unroll_for(E::kBytes * VEC);
    static std::atomic<int> occ[kMaxDevices];
    auto kernel = swiglu::swiglu_fwd_kernel<E, VEC, U, kLoadOutOfPlace, kStore>;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    int per_sm = 0;
    e = ctas_per_sm(kernel, d, occ, per_sm);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm > kFwdPolicy.max_ctas_per_sm) per_sm = kFwdPolicy.max_ctas_per_sm;
    const int64_t nvec = n / VEC;
    const int64_t grid = grid_for<U>(rows * nvec, d, per_sm);
    const int64_t step = grid * U * swiglu::kThreads;
    swiglu::FwdParams p;
    p.x = x;
    p.y = y;
    p.rows = rows;
    p.x_stride = sx / VEC;
    p.y_stride = sy / VEC;
    p.step_q = step / nvec;
    p.nvec = (int32_t)nvec;
    p.step_r = (int32_t)(step % nvec);
    kernel<<<(unsigned)grid, swiglu::kThreads, 0, stream>>>(p);
    e = cudaGetLastError();
    return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
}

template <typename E, int VEC, bool IN_PLACE>
swiglu_status_t launch_bwd(const void *dy, const void *x, void *dx, int64_t rows, int64_t n,
                           int64_t sdy, int64_t sx, int64_t sdx, cudaStream_t stream) {
    constexpr int U = unroll_for(E::kBytes * VEC);
    static std::atomic<int> occ[kMaxDevices];
    auto kernel = swiglu::swiglu_bwd_kernel<E, VEC, U, IN_PLACE,
                                            IN_PLACE ? kLoadInPlace : kLoadOutOfPlace, kStore>;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    int per_sm = 0;
    e = ctas_per_sm(kernel, d, occ, per_sm);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm > kBwdPolicy.max_ctas_per_sm) per_sm = kBwdPolicy.max_ctas_per_sm;
    const int64_t nvec = n / VEC;
    const int64_t grid = grid_for<U>(rows * nvec, d, per_sm);
    const int64_t step = grid * U * swiglu::kThreads;
    swiglu::BwdParams p;
    p.dy = dy;
    p.x = x;
    p.dx = dx;
    p.rows = rows;
    p.dy_stride = sdy / VEC;
    p.x_stride = sx / VEC;
    p.dx_stride = sdx / VEC;
    p.step_q = step / nvec;
    p.nvec = (int32_t)nvec;
    p.step_r = (int32_t)(step % nvec);
    kernel<<<(unsigned)grid, swiglu::kThreads, 0, stream>>>(p);
    e = cudaGetLastError();
    return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
}

// pick_vec never returns more than max_pack_bytes / kBytes elements, so only
// those pack widths are instantiated.
template <typename E>
swiglu_status_t dispatch_fwd(int vec, const void *x, void *y, int64_t rows, int64_t n, int64_t sx,
                             int64_t sy, cudaStream_t st) {
    constexpr int kMaxVec = kFwdPolicy.max_pack_bytes / E::kBytes;
    if constexpr (kMaxVec >= 16) if (vec == 16) return launch_fwd<E, 16>(x, y, rows, n, sx, sy, st);
    if constexpr (kMaxVec >= 8) if (vec == 8) return launch_fwd<E, 8>(x, y, rows, n, sx, sy, st);
    if (vec == 4) return launch_fwd<E, 4>(x, y, rows, n, sx, sy, st);
    if (vec == 2) return launch_fwd<E, 2>(x, y, rows, n, sx, sy, st);
    return launch_fwd<E, 1>(x, y, rows, n, sx, sy, st);
}

template <typename E, bool IP>
swiglu_status_t dispatch_bwd(int vec, const void *dy, const void *x, void *dx, int64_t rows,
                             int64_t n, int64_t sdy, int64_t sx, int64_t sdx, cudaStream_t st) {
    constexpr int kMaxVec = kBwdPolicy.max_pack_bytes / E::kBytes;
    if constexpr (kMaxVec >= 16)
        if (vec == 16) return launch_bwd<E, 16, IP>(dy, x, dx, rows, n, sdy, sx, sdx, st);
    if constexpr (kMaxVec >= 8)
        if (vec == 8) return launch_bwd<E, 8, IP>(dy, x, dx, rows, n, sdy, sx, sdx, st);
    if (vec == 4) return launch_bwd<E, 4, IP>(dy, x, dx, rows, n, sdy, sx, sdx, st);
    if (vec == 2) return launch_bwd<E, 2, IP>(dy, x, dx, rows, n, sdy, sx, sdx, st);
    return launch_bwd<E, 1, IP>(dy, x, dx, rows, n, sdy, sx, sdx, st);
}

// Checks shared by both directions: shape range and the int64 byte extents.
swiglu_status_t check_shape(int64_t rows, int64_t n) {
    if (rows < 0 || n < 0 || n > SWIGLU_MAX_N) return SWIGLU_ERR_SHAPE;
    return SWIGLU_OK;
}

}  // namespace

extern "C" {

swiglu_status_t swiglu_gateup_fwd(const void *x, void *y, int64_t rows, int64_t n,
                                  int64_t x_row_stride, int64_t y_row_stride,
                                  swiglu_dtype_t dtype, swiglu_stream_t stream) {
    const int eb = elem_bytes(dtype);
    if (eb == 0) return SWIGLU_ERR_DTYPE;
    swiglu_status_t st = check_shape(rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    if (x == nullptr || y == nullptr) return SWIGLU_ERR_NULL;
    if (x_row_stride < 2 * n || y_row_stride < n) return SWIGLU_ERR_STRIDE;
    Span sxs, sys;
    if (!span_of(x, rows, 2 * n, x_row_stride, eb, sxs) || !span_of(y, rows, n, y_row_stride, eb, sys))
        return SWIGLU_ERR_SHAPE;
    if (overlaps(sxs, sys)) return SWIGLU_ERR_ALIAS;

    const int64_t strides[2] = {x_row_stride, y_row_stride};
    const void *ptrs[2] = {x, y};
    const int vec = pick_vec(eb, kFwdPolicy.max_pack_bytes, n, strides, 2, ptrs, 2);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == SWIGLU_F32)
        return dispatch_fwd<swiglu::F32>(vec, x, y, rows, n, x_row_stride, y_row_stride, s);
    return dispatch_fwd<swiglu::BF16>(vec, x, y, rows, n, x_row_stride, y_row_stride, s);
}

swiglu_status_t swiglu_gateup_bwd(const void *dy, const void *x, void *dx, int64_t rows,
                                  int64_t n, int64_t dy_row_stride, int64_t x_row_stride,
                                  int64_t dx_row_stride, swiglu_dtype_t dtype, int in_place,
                                  swiglu_stream_t stream) {
    const int eb = elem_bytes(dtype);
    if (eb == 0) return SWIGLU_ERR_DTYPE;
    swiglu_status_t st = check_shape(rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    if (in_place) {
        if (dx == nullptr) dx = const_cast<void *>(x);
        if (dx_row_stride == 0) dx_row_stride = x_row_stride;
    }
    if (dy == nullptr || x == nullptr || dx == nullptr) return SWIGLU_ERR_NULL;
    if (dy_row_stride < n || x_row_stride < 2 * n || dx_row_stride < 2 * n) return SWIGLU_ERR_STRIDE;
    Span sdys, sxs, sdxs;
    if (!span_of(dy, rows, n, dy_row_stride, eb, sdys) ||
        !span_of(x, rows, 2 * n, x_row_stride, eb, sxs) ||
        !span_of(dx, rows, 2 * n, dx_row_stride, eb, sdxs))
        return SWIGLU_ERR_SHAPE;
    if (in_place) {
        if (dx != x) return SWIGLU_ERR_ALIAS;
        if (dx_row_stride != x_row_stride) return SWIGLU_ERR_STRIDE;
        if (overlaps(sdys, sxs)) return SWIGLU_ERR_ALIAS;
    } else {
        if (overlaps(sdxs, sxs) || overlaps(sdxs, sdys)) return SWIGLU_ERR_ALIAS;
    }

    const int64_t strides[3] = {dy_row_stride, x_row_stride, dx_row_stride};
    const void *ptrs[3] = {dy, x, dx};
    const int vec = pick_vec(eb, kBwdPolicy.max_pack_bytes, n, strides, 3, ptrs, 3);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == SWIGLU_F32) {
        if (in_place)
            return dispatch_bwd<swiglu::F32, true>(vec, dy, x, dx, rows, n, dy_row_stride,
                                                   x_row_stride, dx_row_stride, s);
        return dispatch_bwd<swiglu::F32, false>(vec, dy, x, dx, rows, n, dy_row_stride,
                                                x_row_stride, dx_row_stride, s);
    }
    if (in_place)
        return dispatch_bwd<swiglu::BF16, true>(vec, dy, x, dx, rows, n, dy_row_stride,
                                                x_row_stride, dx_row_stride, s);
    return dispatch_bwd<swiglu::BF16, false>(vec, dy, x, dx, rows, n, dy_row_stride, x_row_stride,
                                             dx_row_stride, s);
}

const char *swiglu_status_string(swiglu_status_t status) {
    switch (status) {
        case SWIGLU_OK: return "success";
        case SWIGLU_ERR_NULL: return "a required pointer is NULL";
        case SWIGLU_ERR_DTYPE: return "unsupported dtype";
        case SWIGLU_ERR_SHAPE: return "rows or n out of range, or tensor extent overflows int64";
        case SWIGLU_ERR_STRIDE: return "row stride shorter than the row (or in-place stride mismatch)";
        case SWIGLU_ERR_ALIAS: return "output overlaps an input it must not overlap";
        case SWIGLU_ERR_CUDA: return "CUDA runtime error (see swiglu_last_cuda_error)";
    }
    return "unknown status";
}

int swiglu_last_cuda_error(void) { return g_last_cuda_error; }

int swiglu_abi_version(void) { return 1; }

}  // extern "C"
