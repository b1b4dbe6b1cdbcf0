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
#include <mutex>
#include <utility>

#include "abi_internal.h"
#include "swiglu.h"
#include "swiglu_kernels.cuh"

namespace {

// Launch with programmatic stream serialization (pdl): the kernel may launch
// while the previous kernel in the stream finishes; it waits for that
// kernel's completion itself (await_previous_grid, at the top of every kernel
// here).  pdl = false launches it after the previous kernel, as usual.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}


constexpr int kMaxDevices = 64;
thread_local int g_last_cuda_error = 0;

swiglu_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return SWIGLU_ERR_CUDA;
}

}  // namespace

void swiglu_abi::record_cuda_error(int err) { g_last_cuda_error = err; }

namespace {

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

// Launch policy, chosen by sweeping pack width, unroll, resident CTAs per SM
// and grid size on a GB300 (back-to-back launches timed by CUDA events).
// Forward: with one 32-byte pack per operand and thread, a one-pass grid (a
// CTA per 256 packs, launched in order) beats every persistent grid -- large
// FFN 225.6 us against 238.5 us at 4 CTAs per SM, Llama-like 101.9 against
// 105.5, Megatron shape 31.9 against 34.0: CTAs that start in address order
// keep the DRAM access window compact, where persistent CTAs drift apart.
// With 16-byte packs (two in flight) 6 CTAs per SM did best.  The forward
// variants with a bias or row weights: see kFwdBiasPolicy.  Backward, plain
// form: one-pass as well (see kBwdPolicy; at 3 CTAs per SM the large FFN ran
// 399-418 us against 386 on one pass, before the 32-byte packs).  Narrow
// packs (4 bytes or less: odd n, misaligned rows) of the plain and two-tensor
// forms go to the row-segment kernels (SegShape below); for the bias and
// per-token-weight forms they want persistent CTAs with more threads: four
// packs in flight and 8 (forward) / 6 (backward) CTAs per SM.
struct Policy {
    int max_pack_bytes;
    int ctas_wide;    // 32-byte packs; 0 = a one-pass grid
    int ctas_16;      // 16-byte packs
    int ctas_8;       // 8-byte packs
    int ctas_narrow;  // packs of 4 bytes or less
};
// 8-byte packs (bf16 n = 4 mod 8, fp32 n = 2 mod 4): the plain forward runs
// one pass (bf16 [8192, 2 x 14340] 0.925 -> 0.945 of the copy rate, fp32
// [8192, 2 x 4098] 0.917 -> 0.967 against 6 CTAs per SM), the weighted forward
// 6 CTAs per SM (0.822 -> 0.945, 0.805 -> 0.930 against 4); the bias forms
// were no faster at 6 and slower on one pass, and every form was slower with
// eight packs in flight instead of four.
constexpr Policy kFwdPolicy = {32, 0, 6, 0, 8};
// Bias or row weights alone: one pass as well (large FFN 225.4 / 223.3 us
// against 258.0 / 254.3 us at 4 CTAs per SM; Llama-like 101.4 / 100.2 against
// 109.5 / 108.9).  Both together: persistent at 4 CTAs per SM (234.8 us
// against 249.9 on one pass of 256-thread CTAs and 325.8 of 128-thread ones).
// The bias forward on 8-byte packs: 8 CTAs per SM with two packs in flight
// (bf16 [8192, 2 x 14340] 0.817 -> 0.848 of the copy rate, fp32 [8192, 2 x
// 4098] 0.842 -> 0.851, against 4 CTAs with four packs; with both the weights
// + bias forward fell from 0.82 to 0.74 and keeps 4 with four).
constexpr Policy kFwdBiasPolicy = {32, 0, 4, 8, 8};
constexpr Policy kFwdWeightPolicy = {32, 0, 4, 6, 8};
constexpr Policy kFwdBiasWeightPolicy = {32, 4, 4, 4, 8};
// Forward outputs below this size (the Megatron ffn-4096 shape's 67 MB among
// them) use 16-byte packs at 6 CTAs per SM: 29.4 us against 33.1 us on the
// one-pass 32-byte grid; the Llama-like (235 MB) and large-FFN shapes are
// faster on the one-pass grid.
constexpr int64_t kFwdSmallBytes = (int64_t)128 << 20;
// Backward, plain form: 32-byte packs, one per thread, on a one-pass grid of
// 128-thread CTAs (16-byte packs: two per thread): Megatron shape 51.1 us
// against 53.0 us with two 16-byte packs per thread on 256-thread CTAs,
// Llama-like 165.3 against 168.0, large FFN 373 against 378 (256-thread CTAs
// with one 32-byte pack: 54.3 / 176.2 / 394.8).  The bias and per-token-weight
// forms stay at 16-byte packs (their tile and row kernels are built on them).
constexpr Policy kBwdPolicy = {32, 0, 0, 0, 6};
constexpr int kBwdModeMaxPack = 16;
// The per-token-weighted backward is one CTA per row, persistent over rows.
constexpr Policy kRowPolicy = {16, 3, 3, 3, 6};
// The bias tile kernel is launched as one wave of per_sm CTAs per SM, each
// covering tile_cols columns of each half, with its registers held to
// min_ctas CTAs per SM; the workspace size follows from it.  Packs of 8 and
// 16 bytes: swept with the cp.async ring (bias_stages) over 1.5 - 6 CTAs per
// SM on the large-FFN and Llama-like shapes, the bias form did best at 2
// (407.6 / 189.0 us against 424.7 / 196.7 us for the ring-less kernel at 3),
// the weights + bias form at 3 (429.0 / 202.7 us against 475.2 / 221.1; 466 /
// 215 at 2).  Single-element packs (fp32 4 bytes, bf16 2 bytes; no ring): with
// that shape the kernel waits on its loads (2 CTAs per SM: 23 % of the warps
// active, issue 46 %, fp32 odd-width bias form), and at 4 CTAs per SM its 2048
// columns spill.  1024-column tiles at 4 CTAs per SM (53-63 registers) did
// best, in fractions of the copy rate (bias / weights + bias form):
//   shape (columns, CTAs/SM, register bound)   fp32 3000 x 5503   bf16 8192 x 14335
//   2048, 2 (bias) / 3, 3                      0.62 / 0.56        0.55 / 0.44
//   2048, 3, 3                                 0.70 / 0.56        0.67 / 0.44
//   2048, 4, 4                                 0.38 / 0.37        0.46 / 0.41
//   1024, 4, 4                                 0.72 / 0.69        0.68 / 0.62
//   1024, 5, 5                                 0.72 / 0.59        0.68 / 0.44
//   1024, 6, 6                                 0.59 / 0.51        0.53 / 0.41
//   512, 5, 5 / 512, 6, 6 / 512, 8, 8          0.69-0.74 / 0.62-0.66   0.60-0.64 / 0.42-0.53
// (equal-width tiles, for the ragged last tile, added nothing).
struct BiasShape {
    int tile_cols, per_sm, min_ctas;
};
constexpr BiasShape kBiasWide = {swiglu::kBiasTileCols, 2, 3};
constexpr BiasShape kWeightedBiasWide = {swiglu::kBiasTileCols, 3, 3};
constexpr BiasShape kBiasNarrow = {1024, 4, 4};
constexpr BiasShape kWeightedBiasNarrow = {1024, 4, 4};
// 8-byte packs: bf16 [8192, 2 x 14340] / fp32 [8192, 2 x 4098], bias / weights
// + bias form, fractions of the copy rate:
//   2048-column shape, no ring      0.662 / 0.691    0.619 / 0.639
//   2048-column shape, 2-row ring   0.880 / 0.783    0.734 / 0.518
//   1024 x 4, no ring               0.815 / 0.714    0.768 / 0.722
//   1024 x 4, 2-row ring            0.872 / 0.727    0.794 / 0.707
// so bf16 takes the ring on the 2048-column shape, fp32 the 1024-column shape
// (with the ring for the bias form only).  bf16 on 4-byte packs (two elements)
// also takes the ring on the 2048-column shape (bf16 [8192, 2 x 14334]: 0.708
// -> 0.775 / 0.661 -> 0.703; the ring on the 1024-column shape: 0.711 /
// 0.667).
// The 1024-column shape: single-element packs, and fp32 pairs (8 bytes).
template <typename E>
constexpr bool bias_narrow(int pack_bytes) {
    return E::kBytes == 2 ? pack_bytes <= 2 : pack_bytes <= 8;
}
template <typename E>
constexpr BiasShape bias_shape(bool weighted, int pack_bytes) {
    return bias_narrow<E>(pack_bytes) ? (weighted ? kWeightedBiasNarrow : kBiasNarrow)
                                      : (weighted ? kWeightedBiasWide : kBiasWide);
}

// Resident CTAs per SM to launch with, 0 for a one-pass grid.
constexpr int ctas_cap(const Policy &p, int pack_bytes) {
    return pack_bytes >= 32 ? p.ctas_wide
                             : pack_bytes >= 16 ? p.ctas_16 : pack_bytes >= 8 ? p.ctas_8 : p.ctas_narrow;
}

// Packs in flight per operand per thread: one 32-byte pack, two 16-byte
// packs, else four.
constexpr int unroll_for(int pack_bytes) {
    return pack_bytes >= 32 ? 1 : (pack_bytes >= 16 ? 2 : 4);
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

// Resident CTAs per SM of `kernel` at `threads` threads per CTA and `smem`
// bytes of dynamic shared memory, cached per device in the caller-provided
// table (one table per kernel instantiation and launch shape).
template <typename K>
cudaError_t ctas_per_sm(K kernel, int threads, const Device &d, std::atomic<int> *cache, int &out,
                        size_t smem = 0) {
    int v = (d.id >= 0 && d.id < kMaxDevices) ? cache[d.id].load(std::memory_order_relaxed) : 0;
    if (v == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, threads, smem);
        if (e != cudaSuccess) return e;
        if (v < 1) v = 1;
        if (d.id >= 0 && d.id < kMaxDevices) cache[d.id].store(v, std::memory_order_relaxed);
    }
    out = v;
    return cudaSuccess;
}

// Dynamic shared memory of a one-wave launch planned at per_sm CTAs per SM.
// The kernel uses `need` bytes.  When more than per_sm CTAs would fit, the
// launch asks for enough unused shared memory that no SM can hold more than
// per_sm of them.  Launched early beside the previous grid's last CTAs, such a
// plan is then still spread evenly (left free, an SM may take one CTA more than
// the plan and another one less: the bias form ran 7 % slower on the large FFN
// that way, so those launches used to wait for the previous grid instead).
// Raises the kernel's dynamic shared memory limit as needed.  `fit` is the
// CTAs per SM that `bytes` allows; both are cached per device.
struct HeldSmem {
    int bytes, fit;
};

template <typename K>
cudaError_t held_smem(K kernel, int threads, const Device &d, int per_sm, int need,
                      std::atomic<long long> *cache, HeldSmem &out) {
    const bool cacheable = d.id >= 0 && d.id < kMaxDevices;
    const long long v = cacheable ? cache[d.id].load(std::memory_order_relaxed) : 0;
    if (v != 0) {
        out.bytes = (int)(v >> 8);
        out.fit = (int)(v & 0xff);
        return cudaSuccess;
    }
    cudaError_t e = cudaSuccess;
    if (need > 0 && (e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, need)) !=
                        cudaSuccess)
        return e;
    int fit = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, kernel, threads, (size_t)need)) != cudaSuccess)
        return e;
    out.bytes = need;
    out.fit = fit < 1 ? 1 : fit;
    if (fit > per_sm) {
        cudaFuncAttributes fa;
        int sm_bytes = 0, reserved = 0, optin = 0;
        if ((e = cudaFuncGetAttributes(&fa, kernel)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d.id)) !=
            cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, d.id)) != cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d.id)) != cudaSuccess)
            return e;
        // per_sm + 1 CTAs of (pad + static + reserved) bytes overflow the SM
        long long pad = sm_bytes / (per_sm + 1) + 1 - (long long)fa.sharedSizeBytes - reserved;
        pad = (pad + 127) / 128 * 128;
        if (pad > need && pad + (long long)fa.sharedSizeBytes <= optin) {
            if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pad)) !=
                cudaSuccess)
                return e;
            int held = 0;
            if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&held, kernel, threads, (size_t)pad)) !=
                cudaSuccess)
                return e;
            if (held == per_sm) {  // else keep the unpadded launch
                out.bytes = (int)pad;
                out.fit = held;
            }
        }
    }
    if (cacheable) cache[d.id].store(((long long)out.bytes << 8) | out.fit, std::memory_order_relaxed);
    return cudaSuccess;
}

// Persistent grid: never more CTAs than there are units of U * T packs,
// never more than fill every SM with resident CTAs.
template <int U, int T = swiglu::kThreads>
int64_t grid_for(int64_t total_packs, const Device &d, int per_sm) {
    const int64_t per_cta = (int64_t)U * T;
    int64_t need = (total_packs + per_cta - 1) / per_cta;
    // per_sm == 0: one pass (bounded by the launch limit; the kernels' grid
    // stride covers anything beyond it)
    int64_t full = per_sm > 0 ? (int64_t)d.sms * per_sm : (int64_t)INT32_MAX;
    return need < full ? need : full;
}

// Multiplier and shift of swiglu::fast_div for the divisor d >= 1 (the
// smallest l with 2^l >= d, m = ceil(2^(63 + l) / d)).
swiglu::FastDiv make_fast_div(uint64_t d) {
    if (d <= 1) return {0, -1};
    int l = 0;
    while (l < 63 && ((uint64_t)1 << l) < d) ++l;
    const unsigned __int128 num = (unsigned __int128)1 << (63 + l);
    return {(uint64_t)((num + d - 1) / d), l - 1};
}

// One operand of a launch: base pointer and row stride in elements.
struct Operand {
    const void *p;
    int64_t stride;
};

struct FwdArgs {
    Operand g, u, y;
    int64_t rows, n;
    int mode = swiglu::kPlain;
    const void *bias_g = nullptr, *bias_u = nullptr;  // kBias
    const float *w = nullptr;                          // kWeight
};

struct BwdArgs {
    Operand dy, g, u, dg, du;
    int64_t rows, n;
    int mode = swiglu::kPlain;
    const void *bias_g = nullptr, *bias_u = nullptr;  // kBias
    void *dbias = nullptr;
    float *partial = nullptr;                          // kBias workspace
    const float *w = nullptr;                          // kWeight
    float *dw = nullptr;
    float *partial_dw = nullptr;                       // kBiasWeight workspace
};

// Row groups of the bias backward: enough (column tile, row group) CTAs to
// fill every SM with the shape's per_sm of them, once.
struct BiasPlan {
    int64_t tiles, groups, rows_per_group;
    size_t workspace_bytes;  // the column sums: groups x 2n fp32
};

BiasPlan bias_plan(int64_t rows, int64_t n, int sms, const BiasShape &s) {  // rows, n >= 1
    BiasPlan b;
    b.tiles = (n + s.tile_cols - 1) / s.tile_cols;
    int64_t groups = ((int64_t)sms * s.per_sm) / b.tiles;
    if (groups < 1) groups = 1;
    if (groups > rows) groups = rows;
    b.rows_per_group = (rows + groups - 1) / groups;
    b.groups = (rows + b.rows_per_group - 1) / b.rows_per_group;
    b.workspace_bytes = (size_t)b.groups * (size_t)(2 * n) * sizeof(float);
    return b;
}

// Workspace of the bias backward: the column sums from the start and, with
// weights, one fp32 dw partial per (row, column tile) from dw_offset (a 16-byte
// boundary).  The pack width, which picks the shape, depends on the pointers,
// so the size covers both shapes of the form.  False when the size does not
// fit size_t.
bool bias_workspace(int64_t rows, int64_t n, int sms, bool weighted, size_t &dw_offset,
                    size_t &bytes) {
    const BiasPlan w = bias_plan(rows, n, sms, weighted ? kWeightedBiasWide : kBiasWide);
    const BiasPlan v = bias_plan(rows, n, sms, weighted ? kWeightedBiasNarrow : kBiasNarrow);
    bytes = w.workspace_bytes > v.workspace_bytes ? w.workspace_bytes : v.workspace_bytes;
    dw_offset = 0;
    if (!weighted) return true;
    dw_offset = (bytes + 15) / 16 * 16;
    const int64_t tiles = w.tiles > v.tiles ? w.tiles : v.tiles;
    size_t cells, dw_bytes;
    if (__builtin_mul_overflow((size_t)rows, (size_t)tiles, &cells)) return false;
    if (__builtin_mul_overflow(cells, sizeof(float), &dw_bytes)) return false;
    return !__builtin_add_overflow(dw_offset, dw_bytes, &bytes);
}

template <typename E, int VEC, int MODE>
swiglu_status_t launch_fwd(const FwdArgs &a, cudaStream_t stream) {
    constexpr int U = MODE == swiglu::kBias && E::kBytes * VEC == 8 ? 2 : unroll_for(E::kBytes * VEC);
    constexpr int cap = ctas_cap(MODE == swiglu::kPlain        ? kFwdPolicy
                                 : MODE == swiglu::kBiasWeight ? kFwdBiasWeightPolicy
                                 : MODE == swiglu::kBias       ? kFwdBiasPolicy
                                                               : kFwdWeightPolicy,
                                 E::kBytes * VEC);
    // the one-pass grid runs 128-thread CTAs: 0.5-1.7 % faster than 256 on the
    // large-FFN and Llama-like shapes
    constexpr int T = cap == 0 ? 128 : swiglu::kThreads;
    static std::atomic<int> occ[kMaxDevices];
    auto kernel = swiglu::swiglu_fwd_kernel<E, VEC, U, kLoadOutOfPlace, kStore, MODE, T>;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    int per_sm = 0;
    if (cap > 0) {
        e = ctas_per_sm(kernel, T, d, occ, per_sm);
        if (e != cudaSuccess) return cuda_fail(e);
        if (per_sm > cap) per_sm = cap;
    }
    const int64_t nvec = a.n / VEC;
    const int64_t grid = grid_for<U, T>(a.rows * nvec, d, per_sm);
    const int64_t step = grid * U * T;
    swiglu::FwdParams p;
    p.g = a.g.p;
    p.u = a.u.p;
    p.y = const_cast<void *>(a.y.p);
    p.bias_g = a.bias_g;
    p.bias_u = a.bias_u;
    p.w = a.w;
    p.rows = a.rows;
    p.g_stride = a.g.stride / VEC;
    p.u_stride = a.u.stride / VEC;
    p.y_stride = a.y.stride / VEC;
    p.step_q = step / nvec;
    p.div_nvec = make_fast_div((uint64_t)nvec);
    p.nvec = (int32_t)nvec;
    p.step_r = (int32_t)(step % nvec);
    e = launch_pdl(true, kernel, (unsigned)grid, T, 0, stream, p);
    return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
}

// Row-segment kernels (swiglu_rowseg_kernel) for narrow packs: K columns per
// thread, T threads per CTA, resident CTAs per SM (0 = a one-pass grid).
// Swept over K in {2, 4, 8, 16}, T in {128, 256, 512} and grids of 4 / 8
// CTAs per SM or one pass on the fp32 odd-width workload and a bf16
// [8192, 2 * 14335] case: one pass with 128-thread CTAs did best -- fp32
// forward 32.3 us (K = 8; 33.1 at K = 8, T = 256; 34.8 at 8 CTAs per SM),
// backward 53.3 us (K = 8; 55.3 at T = 256), bf16 forward 135.2 us at K = 16
// (141.4 at K = 8), backward 219.6 us at K = 8.  The per-element walk these
// kernels replace took 44.5 / 62.4 us on the fp32 workload.
// The forward of the bias forms keeps K = 8 for bf16 too (the bias values of
// 16 columns took the kernel to 101 registers and half the speed).
template <typename E, int MODE, int FMODE = swiglu::kPlain, int PV = 1>
struct SegShape {
    static constexpr int K = 8, T = 128, per_sm = 0;
};
template <>
struct SegShape<swiglu::BF16, swiglu::kSegFwd, swiglu::kPlain> {
    static constexpr int K = 16, T = 128, per_sm = 0;
};
template <>
struct SegShape<swiglu::BF16, swiglu::kSegFwd, swiglu::kWeight> {
    static constexpr int K = 16, T = 128, per_sm = 0;
};

// Operands: fwd in = {g, u}, out = {y}; bwd in = {dy, g, u}, out = {dg, du}.
// FMODE: the forward's variant; bias_g / bias_u / w as in FwdArgs.
// PV: elements per pack, 2 for bf16 whose operands all allow 4-byte packs.
template <typename E, int MODE, bool IN_PLACE, int FMODE = swiglu::kPlain, int PV = 1>
swiglu_status_t launch_rowseg(const Operand *in, const Operand *out, int64_t rows, int64_t n,
                              cudaStream_t stream, const void *bias_g = nullptr,
                              const void *bias_u = nullptr, const float *w = nullptr) {
    using Sh = SegShape<E, MODE, FMODE, PV>;
    constexpr int NIN = MODE == swiglu::kSegFwd ? 2 : 3;
    constexpr int NOUT = MODE == swiglu::kSegFwd ? 1 : 2;
    auto kernel = swiglu::swiglu_rowseg_kernel<E, MODE, Sh::K, Sh::T,
                                               IN_PLACE ? kLoadInPlace : kLoadOutOfPlace, FMODE, PV>;
    static std::atomic<int> occ[kMaxDevices];
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    n /= PV;  // packs per row from here on
    const int64_t chunks = (n + Sh::K * Sh::T - 1) / (Sh::K * Sh::T);
    const int64_t segments = rows * chunks;
    int64_t grid = segments;
    if (Sh::per_sm > 0) {
        int per_sm = 0;
        e = ctas_per_sm(kernel, Sh::T, d, occ, per_sm);
        if (e != cudaSuccess) return cuda_fail(e);
        if (per_sm > Sh::per_sm) per_sm = Sh::per_sm;
        if (grid > (int64_t)d.sms * per_sm) grid = (int64_t)d.sms * per_sm;
    }
    if (grid > INT32_MAX) grid = INT32_MAX;  // the segment loop covers the rest
    swiglu::SegParams p;
    for (int x = 0; x < 3; ++x) {
        p.in[x] = x < NIN ? static_cast<const char *>(in[x].p) : nullptr;
        p.in_stride[x] = x < NIN ? in[x].stride * E::kBytes : 0;
    }
    for (int x = 0; x < 2; ++x) {
        p.out[x] = x < NOUT ? static_cast<char *>(const_cast<void *>(out[x].p)) : nullptr;
        p.out_stride[x] = x < NOUT ? out[x].stride * E::kBytes : 0;
    }
    p.bias_g = static_cast<const char *>(bias_g);
    p.bias_u = static_cast<const char *>(bias_u);
    p.w = w;
    p.n = n;
    p.segments = segments;
    p.div_chunks = make_fast_div((uint64_t)chunks);
    p.chunks = (int32_t)chunks;
    e = launch_pdl(true, kernel, (unsigned)grid, Sh::T, 0, stream, p);
    return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
}

// Calls whose operands share no pack wider than this many bytes take the
// row-segment kernels (the forward of every form, the plain and two-tensor
// backward; the bias and per-token-weight backward keep their tile and row
// kernels).
constexpr int kSegMaxPackBytes = 4;

swiglu::BwdParams bwd_params(const BwdArgs &a, int vec) {
    swiglu::BwdParams p;
    p.dy = a.dy.p;
    p.g = a.g.p;
    p.u = a.u.p;
    p.dg = const_cast<void *>(a.dg.p);
    p.du = const_cast<void *>(a.du.p);
    p.bias_g = a.bias_g;
    p.bias_u = a.bias_u;
    p.w = a.w;
    p.dw = a.dw;
    p.partial = a.partial;
    p.partial_dw = a.partial_dw;
    p.rows = a.rows;
    p.dy_stride = a.dy.stride / vec;
    p.g_stride = a.g.stride / vec;
    p.u_stride = a.u.stride / vec;
    p.dg_stride = a.dg.stride / vec;
    p.du_stride = a.du.stride / vec;
    p.nvec = (int32_t)(a.n / vec);
    p.div_nvec = make_fast_div((uint64_t)(a.n / vec));
    p.step_q = 0;
    p.step_r = 0;
    return p;
}

template <typename E, int VEC, bool IN_PLACE>
swiglu_status_t launch_bwd_plain(const BwdArgs &a, cudaStream_t stream) {
    constexpr int U = unroll_for(E::kBytes * VEC);
    constexpr int cap = ctas_cap(kBwdPolicy, E::kBytes * VEC);
    // one-pass grids run 128-thread CTAs, persistent ones kThreads
    constexpr int T = cap == 0 ? 128 : swiglu::kThreads;
    static std::atomic<int> occ[kMaxDevices];
    auto kernel = swiglu::swiglu_bwd_kernel<E, VEC, U, IN_PLACE,
                                            IN_PLACE ? kLoadInPlace : kLoadOutOfPlace, kStore, T>;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    int per_sm = 0;
    if (cap > 0) {
        e = ctas_per_sm(kernel, T, d, occ, per_sm);
        if (e != cudaSuccess) return cuda_fail(e);
        if (per_sm > cap) per_sm = cap;
    }
    const int64_t nvec = a.n / VEC;
    const int64_t grid = grid_for<U, T>(a.rows * nvec, d, per_sm);
    const int64_t step = grid * U * T;
    swiglu::BwdParams p = bwd_params(a, VEC);
    p.step_q = step / nvec;
    p.step_r = (int32_t)(step % nvec);
    e = launch_pdl(true, kernel, (unsigned)grid, T, 0, stream, p);
    return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
}

template <typename E, int VEC, bool IN_PLACE, int ROWS, int MINB>
swiglu_status_t launch_bwd_weighted_rows(const BwdArgs &a, cudaStream_t stream) {
    // single bf16 elements (odd n) keep eight in flight per operand and
    // thread (bf16 [8192, 2 x 14335]: 0.665 -> 0.688 of the copy rate; sixteen:
    // 0.561)
    constexpr int U = E::kBytes * VEC <= 2 ? 8 : unroll_for(E::kBytes * VEC);
    static std::atomic<int> occ[kMaxDevices];
    auto kernel = swiglu::swiglu_bwd_weighted_kernel<E, VEC, U, IN_PLACE,
                                                     IN_PLACE ? kLoadInPlace : kLoadOutOfPlace,
                                                     kStore, ROWS, MINB>;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    int per_sm = 0;
    e = ctas_per_sm(kernel, swiglu::kThreads, d, occ, per_sm);
    if (e != cudaSuccess) return cuda_fail(e);
    static_assert(ctas_cap(kRowPolicy, E::kBytes * VEC) > 0, "the row kernel is persistent");
    const int fit = per_sm;
    if (per_sm > ctas_cap(kRowPolicy, E::kBytes * VEC)) per_sm = ctas_cap(kRowPolicy, E::kBytes * VEC);
    int64_t grid = (int64_t)d.sms * per_sm;
    if (grid > a.rows) grid = a.rows;
    // a fixed number of row-walking CTAs per SM, as in the bias tile kernel:
    // launched early only when that fills every SM (below that, 4.5 % slower).
    // Holding the SMs to the plan with padded shared memory (held_smem) and
    // launching early was slower still here (large FFN 0.980 -> 0.926 of the
    // copy rate, Llama-like 0.934 -> 0.893), unlike the bias tile kernel.
    e = launch_pdl(per_sm >= fit, kernel, (unsigned)grid, swiglu::kThreads, 0, stream, bwd_params(a, VEC));
    return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
}

// Rows per pass of the per-token-weighted row kernel and the CTAs per SM its
// registers are held to.  16-byte packs take two rows per pass; fractions of
// the copy rate, one row / two rows at 127 registers (2 CTAs per SM) / two
// rows held to 3 CTAs per SM (80 registers):
//   ffn-4096 [8192, 2 x 4096] bf16       0.831 / 0.880 / 0.915
//   Llama-like [8192, 2 x 14336] bf16    0.931 / 0.950 / 0.965
//   large FFN [8192, 2 x 32768] bf16     0.979 / 0.988 / 0.948
//   odd width [6000, 2 x 5000] bf16      0.723 / 0.763 / 0.823
// so rows of at most kWeightedShortRowPacks packs take the held form and
// longer rows the unbounded one.  Narrow packs keep one row per pass (fp32
// odd width: 0.818 / 0.725 / 0.718).
constexpr int64_t kWeightedShortRowPacks = 2048;

template <typename E, int VEC, bool IN_PLACE>
swiglu_status_t launch_bwd_weighted(const BwdArgs &a, cudaStream_t stream) {
    if constexpr (E::kBytes * VEC == 16) {
        if (a.n / VEC <= kWeightedShortRowPacks) return launch_bwd_weighted_rows<E, VEC, IN_PLACE, 2, 3>(a, stream);
        return launch_bwd_weighted_rows<E, VEC, IN_PLACE, 2, 0>(a, stream);
    }
    return launch_bwd_weighted_rows<E, VEC, IN_PLACE, 1, 0>(a, stream);
}

// Rows in flight through the bias tile kernel's cp.async ring (0: plain
// register loads); see swiglu_bwd_bias_kernel.  16-byte packs: 2.  8-byte
// packs: 2 but for fp32 with weights (see bias_shape).  4-byte packs: 2 for
// bf16 (two elements a pack), none for fp32 (one element; odd n: a 2-row ring
// ran 139 us against 97 us without on the odd-width workload's bias
// backward).  Narrower packs: none.
template <typename E, bool WEIGHTED>
constexpr int bias_stages(int pack_bytes) {
    return pack_bytes == 16                                     ? 2
           : pack_bytes == 8 && !(E::kBytes == 4 && WEIGHTED) ? 2
           : pack_bytes == 4 && E::kBytes == 2                 ? 2
                                                               : 0;
}
// Rows of dw partial sums the weights + bias tile kernel batches per barrier
// (16 leaves room for the ring at 3 CTAs per SM; same speed as 32).
constexpr int kDwBatch = 16;

template <typename E, int VEC, bool IN_PLACE, bool WEIGHTED>
swiglu_status_t launch_bwd_bias(const BwdArgs &a, cudaStream_t stream) {
    constexpr int STAGES = bias_stages<E, WEIGHTED>(E::kBytes * VEC);
    constexpr BiasShape S = bias_shape<E>(WEIGHTED, E::kBytes * VEC);
    constexpr int ring = swiglu::swiglu_bias_ring_bytes<VEC, E::kBytes, STAGES, S.tile_cols>();
    auto kernel = swiglu::swiglu_bwd_bias_kernel<E, VEC, IN_PLACE,
                                                 IN_PLACE ? kLoadInPlace : kLoadOutOfPlace, kStore,
                                                 WEIGHTED, STAGES, kDwBatch, S.tile_cols, S.min_ctas>;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    const BiasPlan b = bias_plan(a.rows, a.n, d.sms, S);
    // The plan is one wave of a fixed number of CTAs per SM, each walking its
    // rows, and the SM's issue bounds them.  The launch holds every SM to the
    // plan (held_smem: the bias form's 2 CTAs per SM would otherwise leave room
    // for 3; with that, 0.848 -> 0.860 of the copy rate on ffn-4096, 0.960 ->
    // 0.973 Llama-like, 0.991 -> 0.996 large FFN) and launches early when it
    // does.
    static std::atomic<long long> held[kMaxDevices];
    HeldSmem hs;
    e = held_smem(kernel, swiglu::kThreads, d, S.per_sm, ring, held, hs);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_pdl(S.per_sm >= hs.fit, kernel, (unsigned)(b.tiles * b.groups), swiglu::kThreads,
                   (size_t)hs.bytes, stream, bwd_params(a, VEC), (int32_t)b.tiles, b.rows_per_group);
    if (e != cudaSuccess) return cuda_fail(e);
    // the reductions: kReduceCols columns of dbias per CTA, then (with
    // weights) kReduceThreads rows of dw per CTA, in one launch
    constexpr int64_t RC = swiglu::kReduceCols, RT = swiglu::kReduceThreads, kCap = 8;
    int64_t col_ctas = (2 * a.n + RC - 1) / RC;
    if (col_ctas > (int64_t)d.sms * kCap) col_ctas = (int64_t)d.sms * kCap;
    int64_t dw_ctas = WEIGHTED ? (a.rows + RT - 1) / RT : 0;
    if (dw_ctas > (int64_t)d.sms * kCap) dw_ctas = (int64_t)d.sms * kCap;
    e = launch_pdl(true, swiglu::swiglu_bias_reduce_kernel<E>, (unsigned)(col_ctas + dw_ctas), (unsigned)RT, 0,
                   stream, a.partial, b.groups, 2 * a.n, a.dbias, col_ctas, a.partial_dw,
                   WEIGHTED ? a.rows : 0, (int32_t)b.tiles, a.dw);
    return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
}

template <typename E, int VEC, bool IN_PLACE>
swiglu_status_t launch_bwd(const BwdArgs &a, cudaStream_t stream) {
    // packs wider than kBwdModeMaxPack only ever reach here for the plain form
    if constexpr (E::kBytes * VEC <= kBwdModeMaxPack) {
        if (a.mode == swiglu::kWeight) return launch_bwd_weighted<E, VEC, IN_PLACE>(a, stream);
        if (a.mode == swiglu::kBias) return launch_bwd_bias<E, VEC, IN_PLACE, false>(a, stream);
        if (a.mode == swiglu::kBiasWeight) return launch_bwd_bias<E, VEC, IN_PLACE, true>(a, stream);
    }
    return launch_bwd_plain<E, VEC, IN_PLACE>(a, stream);
}

template <typename E, int VEC>
swiglu_status_t launch_fwd_mode(const FwdArgs &a, cudaStream_t st) {
    if (a.mode == swiglu::kWeight) return launch_fwd<E, VEC, swiglu::kWeight>(a, st);
    if (a.mode == swiglu::kBias) return launch_fwd<E, VEC, swiglu::kBias>(a, st);
    if (a.mode == swiglu::kBiasWeight) return launch_fwd<E, VEC, swiglu::kBiasWeight>(a, st);
    return launch_fwd<E, VEC, swiglu::kPlain>(a, st);
}

// The forward of every form on the row-segment kernels, PV elements per pack.
template <typename E, int PV>
swiglu_status_t rowseg_fwd(const FwdArgs &a, cudaStream_t st) {
    const Operand in[2] = {a.g, a.u};
    switch (a.mode) {
        case swiglu::kBias:
            return launch_rowseg<E, swiglu::kSegFwd, false, swiglu::kBias, PV>(in, &a.y, a.rows, a.n, st,
                                                                               a.bias_g, a.bias_u);
        case swiglu::kWeight:
            return launch_rowseg<E, swiglu::kSegFwd, false, swiglu::kWeight, PV>(in, &a.y, a.rows, a.n, st,
                                                                                 nullptr, nullptr, a.w);
        case swiglu::kBiasWeight:
            return launch_rowseg<E, swiglu::kSegFwd, false, swiglu::kBiasWeight, PV>(
                in, &a.y, a.rows, a.n, st, a.bias_g, a.bias_u, a.w);
        default:
            return launch_rowseg<E, swiglu::kSegFwd, false, swiglu::kPlain, PV>(in, &a.y, a.rows, a.n, st);
    }
}

// The widest pack every operand (bias halves included) allows; pick_vec never
// returns more than max_pack_bytes / kBytes elements, so only those widths are
// instantiated.
template <typename E>
swiglu_status_t dispatch_fwd(const FwdArgs &a, cudaStream_t st) {
    const int64_t strides[3] = {a.g.stride, a.u.stride, a.y.stride};
    const void *ptrs[5] = {a.g.p, a.u.p, a.y.p, a.bias_g, a.bias_u};
    const int np = (a.mode & swiglu::kBias) ? 5 : 3;
    // below kFwdSmallBytes of output the plain forward does better with 16-byte
    // packs on a persistent grid than with the one-pass 32-byte grid
    const bool small = a.mode == swiglu::kPlain && a.rows * a.n * E::kBytes < kFwdSmallBytes;
    const int vec = pick_vec(E::kBytes, small ? 16 : kFwdPolicy.max_pack_bytes, a.n, strides, 3,
                             ptrs, np);
    if (vec * E::kBytes <= kSegMaxPackBytes) {
        if constexpr (E::kBytes == 2)
            if (vec == 2) return rowseg_fwd<E, 2>(a, st);
        return rowseg_fwd<E, 1>(a, st);
    }
    constexpr int kMaxVec = kFwdPolicy.max_pack_bytes / E::kBytes;
    if constexpr (kMaxVec >= 16) if (vec == 16) return launch_fwd_mode<E, 16>(a, st);
    if constexpr (kMaxVec >= 8) if (vec == 8) return launch_fwd_mode<E, 8>(a, st);
    if (vec == 4) return launch_fwd_mode<E, 4>(a, st);
    if (vec == 2) return launch_fwd_mode<E, 2>(a, st);
    return launch_fwd_mode<E, 1>(a, st);
}

template <typename E, bool IP>
swiglu_status_t dispatch_bwd(const BwdArgs &a, cudaStream_t st) {
    const int64_t strides[5] = {a.dy.stride, a.g.stride, a.u.stride, a.dg.stride, a.du.stride};
    const void *ptrs[7] = {a.dy.p, a.g.p, a.u.p, a.dg.p, a.du.p, a.bias_g, a.bias_u};
    const int np = (a.mode & swiglu::kBias) ? 7 : 5;
    const int max_pack = a.mode == swiglu::kPlain ? kBwdPolicy.max_pack_bytes : kBwdModeMaxPack;
    const int vec = pick_vec(E::kBytes, max_pack, a.n, strides, 5, ptrs, np);
    if (a.mode == swiglu::kPlain && vec * E::kBytes <= kSegMaxPackBytes) {
        const Operand in[3] = {a.dy, a.g, a.u};
        const Operand out[2] = {a.dg, a.du};
        if constexpr (E::kBytes == 2)
            if (vec == 2) return launch_rowseg<E, swiglu::kSegBwd, IP, swiglu::kPlain, 2>(in, out, a.rows, a.n, st);
        return launch_rowseg<E, swiglu::kSegBwd, IP>(in, out, a.rows, a.n, st);
    }
    constexpr int kMaxVec = kBwdPolicy.max_pack_bytes / E::kBytes;
    if constexpr (kMaxVec >= 16) if (vec == 16) return launch_bwd<E, 16, IP>(a, st);
    if constexpr (kMaxVec >= 8) if (vec == 8) return launch_bwd<E, 8, IP>(a, st);
    if (vec == 4) return launch_bwd<E, 4, IP>(a, st);
    if (vec == 2) return launch_bwd<E, 2, IP>(a, st);
    return launch_bwd<E, 1, IP>(a, st);
}

// The kernels load and store whole elements, so every pointer must sit on a
// multiple of its element size.
bool on_element(const void *p, int bytes) { return (uintptr_t)p % (uintptr_t)bytes == 0; }

swiglu_status_t run_fwd(swiglu_dtype_t dtype, const FwdArgs &a, swiglu_stream_t stream) {
    const int eb = dtype == SWIGLU_F32 ? 4 : 2;
    if (!on_element(a.g.p, eb) || !on_element(a.u.p, eb) || !on_element(a.y.p, eb) ||
        !on_element(a.bias_g, eb) || !on_element(a.bias_u, eb) || !on_element(a.w, 4))
        return SWIGLU_ERR_STRIDE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == SWIGLU_F32) return dispatch_fwd<swiglu::F32>(a, s);
    return dispatch_fwd<swiglu::BF16>(a, s);
}

swiglu_status_t run_bwd(swiglu_dtype_t dtype, bool in_place, const BwdArgs &a,
                        swiglu_stream_t stream) {
    const int eb = dtype == SWIGLU_F32 ? 4 : 2;
    if (!on_element(a.dy.p, eb) || !on_element(a.g.p, eb) || !on_element(a.u.p, eb) ||
        !on_element(a.dg.p, eb) || !on_element(a.du.p, eb) || !on_element(a.bias_g, eb) ||
        !on_element(a.bias_u, eb) || !on_element(a.dbias, eb) || !on_element(a.w, 4) ||
        !on_element(a.dw, 4))
        return SWIGLU_ERR_STRIDE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == SWIGLU_F32)
        return in_place ? dispatch_bwd<swiglu::F32, true>(a, s) : dispatch_bwd<swiglu::F32, false>(a, s);
    return in_place ? dispatch_bwd<swiglu::BF16, true>(a, s) : dispatch_bwd<swiglu::BF16, false>(a, s);
}

// Checks shared by every entry point: dtype and shape range.
swiglu_status_t check_common(swiglu_dtype_t dtype, int64_t rows, int64_t n) {
    if (elem_bytes(dtype) == 0) return SWIGLU_ERR_DTYPE;
    if (rows < 0 || n < 0 || n > SWIGLU_MAX_N) return SWIGLU_ERR_SHAPE;
    return SWIGLU_OK;
}

// Validates the fused backward's dy / x / dx (with the in-place contract) and
// fills `a` with the fused layout's operands; sp[] = spans of dy, x, dx.
swiglu_status_t gateup_bwd_args(const void *dy, const void *x, void *dx, int64_t rows, int64_t n,
                                int64_t dy_row_stride, int64_t x_row_stride,
                                int64_t dx_row_stride, swiglu_dtype_t dtype, int in_place,
                                BwdArgs &a, Span sp[3]) {
    const int eb = elem_bytes(dtype);
    if (in_place) {
        if (dx == nullptr) dx = const_cast<void *>(x);
        if (dx_row_stride == 0) dx_row_stride = x_row_stride;
    }
    if (dy == nullptr || x == nullptr || dx == nullptr) return SWIGLU_ERR_NULL;
    if (dy_row_stride < n || x_row_stride < 2 * n || dx_row_stride < 2 * n) return SWIGLU_ERR_STRIDE;
    if (!span_of(dy, rows, n, dy_row_stride, eb, sp[0]) ||
        !span_of(x, rows, 2 * n, x_row_stride, eb, sp[1]) ||
        !span_of(dx, rows, 2 * n, dx_row_stride, eb, sp[2]))
        return SWIGLU_ERR_SHAPE;
    if (in_place) {
        if (dx != x) return SWIGLU_ERR_ALIAS;
        if (dx_row_stride != x_row_stride) return SWIGLU_ERR_STRIDE;
        if (overlaps(sp[0], sp[1])) return SWIGLU_ERR_ALIAS;
    } else {
        if (overlaps(sp[2], sp[1]) || overlaps(sp[2], sp[0])) return SWIGLU_ERR_ALIAS;
    }
    const char *xb = static_cast<const char *>(x);
    char *dxb = static_cast<char *>(dx);
    a.dy = {dy, dy_row_stride};
    a.g = {x, x_row_stride};
    a.u = {xb + n * eb, x_row_stride};
    a.dg = {dx, dx_row_stride};
    a.du = {dxb + n * eb, dx_row_stride};
    a.rows = rows;
    a.n = n;
    return SWIGLU_OK;
}

// The bias backward, with per-token weights when w != nullptr (then dw is
// written too and the workspace also holds the dw partials).
swiglu_status_t bias_bwd_impl(const void *dy, const void *x, const void *bias, const float *w,
                              void *dx, void *dbias, float *dw, void *workspace,
                              size_t workspace_bytes, int64_t rows, int64_t n,
                              int64_t dy_row_stride, int64_t x_row_stride, int64_t dx_row_stride,
                              swiglu_dtype_t dtype, int in_place, swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (n == 0 && rows == 0) return SWIGLU_OK;
    const int eb = elem_bytes(dtype);
    const bool weighted = w != nullptr;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) {  // every row sums nothing
        if (!weighted) return SWIGLU_OK;
        Span sws, sdws;
        if (!span_of(w, 1, rows, rows, 4, sws) || !span_of(dw, 1, rows, rows, 4, sdws))
            return SWIGLU_ERR_SHAPE;
        if (overlaps(sws, sdws)) return SWIGLU_ERR_ALIAS;
        cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)rows * sizeof(float), cs);
        return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
    }
    if (bias == nullptr || dbias == nullptr) return SWIGLU_ERR_NULL;
    Span sbs, sdbs;
    if (!span_of(bias, 1, 2 * n, 2 * n, eb, sbs) || !span_of(dbias, 1, 2 * n, 2 * n, eb, sdbs))
        return SWIGLU_ERR_SHAPE;
    if (overlaps(sbs, sdbs)) return SWIGLU_ERR_ALIAS;
    if (rows == 0) {  // the sum over no rows
        cudaError_t e = cudaMemsetAsync(dbias, 0, (size_t)(2 * n) * eb, cs);
        return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
    }
    if (workspace == nullptr) return SWIGLU_ERR_NULL;
    BwdArgs a;
    Span sp[3];
    st = gateup_bwd_args(dy, x, dx, rows, n, dy_row_stride, x_row_stride, dx_row_stride, dtype,
                         in_place, a, sp);
    if (st != SWIGLU_OK) return st;
    Span sws;
    if (!span_of(workspace, 1, (int64_t)workspace_bytes, (int64_t)workspace_bytes, 1, sws))
        return SWIGLU_ERR_SHAPE;
    // dbias and the workspace are written: they overlap nothing; bias is read
    // while dx is written
    for (int i = 0; i < 3; ++i)
        if (overlaps(sdbs, sp[i]) || overlaps(sws, sp[i])) return SWIGLU_ERR_ALIAS;
    if (overlaps(sws, sbs) || overlaps(sws, sdbs) || overlaps(sbs, sp[2])) return SWIGLU_ERR_ALIAS;
    if (weighted) {
        // dw is written: it overlaps nothing; w is read while dx, dbias and
        // the workspace are written
        Span sw, sdw;
        if (!span_of(w, 1, rows, rows, 4, sw) || !span_of(dw, 1, rows, rows, 4, sdw))
            return SWIGLU_ERR_SHAPE;
        for (int i = 0; i < 3; ++i)
            if (overlaps(sdw, sp[i])) return SWIGLU_ERR_ALIAS;
        if (overlaps(sdw, sw) || overlaps(sdw, sbs) || overlaps(sdw, sdbs) || overlaps(sdw, sws))
            return SWIGLU_ERR_ALIAS;
        if (overlaps(sw, sp[2]) || overlaps(sw, sdbs) || overlaps(sw, sws)) return SWIGLU_ERR_ALIAS;
    }
    if ((uintptr_t)workspace % 16 != 0) return SWIGLU_ERR_WORKSPACE;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    size_t need = 0, dw_offset = 0;
    if (!bias_workspace(rows, n, d.sms, weighted, dw_offset, need)) return SWIGLU_ERR_SHAPE;
    if (workspace_bytes < need) return SWIGLU_ERR_WORKSPACE;
    a.mode = weighted ? swiglu::kBiasWeight : swiglu::kBias;
    a.bias_g = bias;
    a.bias_u = static_cast<const char *>(bias) + n * eb;
    a.dbias = dbias;
    a.partial = static_cast<float *>(workspace);
    if (weighted) {
        a.w = w;
        a.dw = dw;
        a.partial_dw = reinterpret_cast<float *>(static_cast<char *>(workspace) + dw_offset);
    }
    return run_bwd(dtype, in_place != 0, a, stream);
}

}  // namespace

extern "C" {

swiglu_status_t swiglu_gateup_fwd(const void *x, void *y, int64_t rows, int64_t n,
                                  int64_t x_row_stride, int64_t y_row_stride,
                                  swiglu_dtype_t dtype, swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    const int eb = elem_bytes(dtype);
    if (x == nullptr || y == nullptr) return SWIGLU_ERR_NULL;
    if (x_row_stride < 2 * n || y_row_stride < n) return SWIGLU_ERR_STRIDE;
    Span sxs, sys;
    if (!span_of(x, rows, 2 * n, x_row_stride, eb, sxs) || !span_of(y, rows, n, y_row_stride, eb, sys))
        return SWIGLU_ERR_SHAPE;
    if (overlaps(sxs, sys)) return SWIGLU_ERR_ALIAS;
    const char *xb = static_cast<const char *>(x);
    FwdArgs a{{x, x_row_stride}, {xb + n * eb, x_row_stride}, {y, y_row_stride}, rows, n};
    return run_fwd(dtype, a, stream);
}

swiglu_status_t swiglu_gateup_bwd(const void *dy, const void *x, void *dx, int64_t rows,
                                  int64_t n, int64_t dy_row_stride, int64_t x_row_stride,
                                  int64_t dx_row_stride, swiglu_dtype_t dtype, int in_place,
                                  swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    BwdArgs a;
    Span sp[3];
    st = gateup_bwd_args(dy, x, dx, rows, n, dy_row_stride, x_row_stride, dx_row_stride, dtype,
                         in_place, a, sp);
    if (st != SWIGLU_OK) return st;
    return run_bwd(dtype, in_place != 0, a, stream);
}

swiglu_status_t swiglu_gateup_weighted_fwd(const void *x, const float *w, void *y, int64_t rows,
                                           int64_t n, int64_t x_row_stride, int64_t y_row_stride,
                                           swiglu_dtype_t dtype, swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    const int eb = elem_bytes(dtype);
    if (x == nullptr || y == nullptr || w == nullptr) return SWIGLU_ERR_NULL;
    if (x_row_stride < 2 * n || y_row_stride < n) return SWIGLU_ERR_STRIDE;
    Span sxs, sys, sws;
    if (!span_of(x, rows, 2 * n, x_row_stride, eb, sxs) ||
        !span_of(y, rows, n, y_row_stride, eb, sys) || !span_of(w, 1, rows, rows, 4, sws))
        return SWIGLU_ERR_SHAPE;
    if (overlaps(sxs, sys) || overlaps(sws, sys)) return SWIGLU_ERR_ALIAS;
    const char *xb = static_cast<const char *>(x);
    FwdArgs a{{x, x_row_stride}, {xb + n * eb, x_row_stride}, {y, y_row_stride}, rows, n};
    a.mode = swiglu::kWeight;
    a.w = w;
    return run_fwd(dtype, a, stream);
}

swiglu_status_t swiglu_gateup_weighted_bwd(const void *dy, const void *x, const float *w, void *dx,
                                           float *dw, int64_t rows, int64_t n,
                                           int64_t dy_row_stride, int64_t x_row_stride,
                                           int64_t dx_row_stride, swiglu_dtype_t dtype,
                                           int in_place, swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0) return SWIGLU_OK;
    if (w == nullptr || dw == nullptr) return SWIGLU_ERR_NULL;
    Span sws, sdws;
    if (!span_of(w, 1, rows, rows, 4, sws) || !span_of(dw, 1, rows, rows, 4, sdws))
        return SWIGLU_ERR_SHAPE;
    if (overlaps(sws, sdws)) return SWIGLU_ERR_ALIAS;
    if (n == 0) {  // every row sums nothing
        cudaError_t e = cudaMemsetAsync(dw, 0, (size_t)rows * sizeof(float),
                                        reinterpret_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? SWIGLU_OK : cuda_fail(e);
    }
    BwdArgs a;
    Span sp[3];
    st = gateup_bwd_args(dy, x, dx, rows, n, dy_row_stride, x_row_stride, dx_row_stride, dtype,
                         in_place, a, sp);
    if (st != SWIGLU_OK) return st;
    // dw may overlap nothing; w may not overlap the written dx
    for (int i = 0; i < 3; ++i)
        if (overlaps(sdws, sp[i])) return SWIGLU_ERR_ALIAS;
    if (overlaps(sws, sp[2])) return SWIGLU_ERR_ALIAS;
    a.mode = swiglu::kWeight;
    a.w = w;
    a.dw = dw;
    return run_bwd(dtype, in_place != 0, a, stream);
}

swiglu_status_t swiglu_gateup_bias_fwd(const void *x, const void *bias, void *y, int64_t rows,
                                       int64_t n, int64_t x_row_stride, int64_t y_row_stride,
                                       swiglu_dtype_t dtype, swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    const int eb = elem_bytes(dtype);
    if (x == nullptr || y == nullptr || bias == nullptr) return SWIGLU_ERR_NULL;
    if (x_row_stride < 2 * n || y_row_stride < n) return SWIGLU_ERR_STRIDE;
    Span sxs, sys, sbs;
    if (!span_of(x, rows, 2 * n, x_row_stride, eb, sxs) ||
        !span_of(y, rows, n, y_row_stride, eb, sys) || !span_of(bias, 1, 2 * n, 2 * n, eb, sbs))
        return SWIGLU_ERR_SHAPE;
    if (overlaps(sxs, sys) || overlaps(sbs, sys)) return SWIGLU_ERR_ALIAS;
    const char *xb = static_cast<const char *>(x);
    FwdArgs a{{x, x_row_stride}, {xb + n * eb, x_row_stride}, {y, y_row_stride}, rows, n};
    a.mode = swiglu::kBias;
    a.bias_g = bias;
    a.bias_u = static_cast<const char *>(bias) + n * eb;
    return run_fwd(dtype, a, stream);
}

swiglu_status_t swiglu_gateup_bias_bwd_workspace_size(int64_t rows, int64_t n, size_t *bytes) {
    if (bytes == nullptr) return SWIGLU_ERR_NULL;
    if (rows < 0 || n < 0 || n > SWIGLU_MAX_N) return SWIGLU_ERR_SHAPE;
    *bytes = 0;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    size_t off;
    if (!bias_workspace(rows, n, d.sms, false, off, *bytes)) return SWIGLU_ERR_SHAPE;
    return SWIGLU_OK;
}

swiglu_status_t swiglu_gateup_bias_bwd(const void *dy, const void *x, const void *bias, void *dx,
                                       void *dbias, void *workspace, size_t workspace_bytes,
                                       int64_t rows, int64_t n, int64_t dy_row_stride,
                                       int64_t x_row_stride, int64_t dx_row_stride,
                                       swiglu_dtype_t dtype, int in_place,
                                       swiglu_stream_t stream) {
    return bias_bwd_impl(dy, x, bias, nullptr, dx, dbias, nullptr, workspace, workspace_bytes, rows,
                         n, dy_row_stride, x_row_stride, dx_row_stride, dtype, in_place, stream);
}

swiglu_status_t swiglu_gateup_weighted_bias_fwd(const void *x, const void *bias, const float *w,
                                                void *y, int64_t rows, int64_t n,
                                                int64_t x_row_stride, int64_t y_row_stride,
                                                swiglu_dtype_t dtype, swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    const int eb = elem_bytes(dtype);
    if (x == nullptr || y == nullptr || bias == nullptr || w == nullptr) return SWIGLU_ERR_NULL;
    if (x_row_stride < 2 * n || y_row_stride < n) return SWIGLU_ERR_STRIDE;
    Span sxs, sys, sbs, sws;
    if (!span_of(x, rows, 2 * n, x_row_stride, eb, sxs) ||
        !span_of(y, rows, n, y_row_stride, eb, sys) || !span_of(bias, 1, 2 * n, 2 * n, eb, sbs) ||
        !span_of(w, 1, rows, rows, 4, sws))
        return SWIGLU_ERR_SHAPE;
    if (overlaps(sxs, sys) || overlaps(sbs, sys) || overlaps(sws, sys)) return SWIGLU_ERR_ALIAS;
    const char *xb = static_cast<const char *>(x);
    FwdArgs a{{x, x_row_stride}, {xb + n * eb, x_row_stride}, {y, y_row_stride}, rows, n};
    a.mode = swiglu::kBiasWeight;
    a.bias_g = bias;
    a.bias_u = static_cast<const char *>(bias) + n * eb;
    a.w = w;
    return run_fwd(dtype, a, stream);
}

swiglu_status_t swiglu_gateup_weighted_bias_bwd_workspace_size(int64_t rows, int64_t n,
                                                               size_t *bytes) {
    if (bytes == nullptr) return SWIGLU_ERR_NULL;
    if (rows < 0 || n < 0 || n > SWIGLU_MAX_N) return SWIGLU_ERR_SHAPE;
    *bytes = 0;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    size_t off;
    if (!bias_workspace(rows, n, d.sms, true, off, *bytes)) return SWIGLU_ERR_SHAPE;
    return SWIGLU_OK;
}

swiglu_status_t swiglu_gateup_weighted_bias_bwd(
    const void *dy, const void *x, const void *bias, const float *w, void *dx, void *dbias,
    float *dw, void *workspace, size_t workspace_bytes, int64_t rows, int64_t n,
    int64_t dy_row_stride, int64_t x_row_stride, int64_t dx_row_stride, swiglu_dtype_t dtype,
    int in_place, swiglu_stream_t stream) {
    if (w == nullptr || dw == nullptr) {  // the rest is checked in bias_bwd_impl
        swiglu_status_t st = check_common(dtype, rows, n);
        if (st != SWIGLU_OK) return st;
        return rows == 0 ? bias_bwd_impl(dy, x, bias, nullptr, dx, dbias, nullptr, workspace,
                                         workspace_bytes, rows, n, dy_row_stride, x_row_stride,
                                         dx_row_stride, dtype, in_place, stream)
                         : SWIGLU_ERR_NULL;
    }
    return bias_bwd_impl(dy, x, bias, w, dx, dbias, dw, workspace, workspace_bytes, rows, n,
                         dy_row_stride, x_row_stride, dx_row_stride, dtype, in_place, stream);
}

swiglu_status_t swiglu_silu_mul_fwd(const void *a, const void *b, void *c, int64_t rows, int64_t n,
                                    int64_t a_row_stride, int64_t b_row_stride,
                                    int64_t c_row_stride, swiglu_dtype_t dtype,
                                    swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    const int eb = elem_bytes(dtype);
    if (a == nullptr || b == nullptr || c == nullptr) return SWIGLU_ERR_NULL;
    if (a_row_stride < n || b_row_stride < n || c_row_stride < n) return SWIGLU_ERR_STRIDE;
    Span sa, sb, sc;
    if (!span_of(a, rows, n, a_row_stride, eb, sa) || !span_of(b, rows, n, b_row_stride, eb, sb) ||
        !span_of(c, rows, n, c_row_stride, eb, sc))
        return SWIGLU_ERR_SHAPE;
    if (overlaps(sc, sa) || overlaps(sc, sb)) return SWIGLU_ERR_ALIAS;
    FwdArgs args{{a, a_row_stride}, {b, b_row_stride}, {c, c_row_stride}, rows, n};
    return run_fwd(dtype, args, stream);
}

swiglu_status_t swiglu_silu_mul_bwd(const void *dc, const void *a, const void *b, void *da,
                                    void *db, int64_t rows, int64_t n, int64_t dc_row_stride,
                                    int64_t a_row_stride, int64_t b_row_stride,
                                    int64_t da_row_stride, int64_t db_row_stride,
                                    swiglu_dtype_t dtype, swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0) return SWIGLU_OK;
    const int eb = elem_bytes(dtype);
    if (dc == nullptr || a == nullptr || b == nullptr || da == nullptr || db == nullptr)
        return SWIGLU_ERR_NULL;
    if (dc_row_stride < n || a_row_stride < n || b_row_stride < n || da_row_stride < n ||
        db_row_stride < n)
        return SWIGLU_ERR_STRIDE;
    Span sdc, sa, sb, sda, sdb;
    if (!span_of(dc, rows, n, dc_row_stride, eb, sdc) || !span_of(a, rows, n, a_row_stride, eb, sa) ||
        !span_of(b, rows, n, b_row_stride, eb, sb) ||
        !span_of(da, rows, n, da_row_stride, eb, sda) ||
        !span_of(db, rows, n, db_row_stride, eb, sdb))
        return SWIGLU_ERR_SHAPE;
    // an output may be exactly its own input (same pointer and stride);
    // otherwise it may overlap no input and not the other output
    const bool da_is_a = da == a && da_row_stride == a_row_stride;
    const bool db_is_b = db == b && db_row_stride == b_row_stride;
    if (overlaps(sda, sdb)) return SWIGLU_ERR_ALIAS;
    if (overlaps(sda, sdc) || overlaps(sda, sb) || (!da_is_a && overlaps(sda, sa)))
        return SWIGLU_ERR_ALIAS;
    if (overlaps(sdb, sdc) || overlaps(sdb, sa) || (!db_is_b && overlaps(sdb, sb)))
        return SWIGLU_ERR_ALIAS;
    BwdArgs args{{dc, dc_row_stride}, {a, a_row_stride},   {b, b_row_stride},
                 {da, da_row_stride}, {db, db_row_stride}, rows, n};
    return run_bwd(dtype, da_is_a || db_is_b, args, stream);
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
        case SWIGLU_ERR_WORKSPACE: return "workspace too small or not 16-byte aligned";
    }
    return "unknown status";
}

int swiglu_last_cuda_error(void) { return g_last_cuda_error; }

int swiglu_abi_version(void) { return 5; }

}  // extern "C"

// ------------------------------------------------ allocation-free variant ---
// swiglu_gateup_bias_bwd_noalloc: the bias backward with its column-sum
// scratch in a fixed file-scope device array instead of a caller workspace,
// for callers that have no way to obtain device memory of their own.  Every
// GPU that loads this library holds the array until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SWIGLU_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of g_noalloc_scratch in each CUDA context, looked up on the
// first call made with that context current (host code cannot use the
// array's name as a device address).  The cache is keyed on the context's
// process-unique id, not only on the device: after cudaDeviceReset the
// device's next primary context loads the module afresh and the array may sit
// at another address.
struct NoallocSlot {
    unsigned long long ctx_id;  // 0: empty
    void *addr;
};
std::mutex g_noalloc_mu;
NoallocSlot g_noalloc_slot[kMaxDevices];

// The CUDA driver's cuCtxGetCurrent / cuCtxGetId, reached through the
// runtime's entry-point query (the library links no driver library).
using CtxGetCurrentFn = int (*)(void **);
using CtxGetIdFn = int (*)(void *, unsigned long long *);

// Process-unique id of the current context, 0 when there is none or the
// driver cannot say (then nothing is cached).
unsigned long long current_context_id() {
    static const std::pair<CtxGetCurrentFn, CtxGetIdFn> fns = [] {
        void *cur = nullptr, *id = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &cur, 12000, cudaEnableDefault,
                                             &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess)
            cur = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &id, 12000, cudaEnableDefault, &q2) !=
                cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess)
            id = nullptr;
        return std::make_pair(reinterpret_cast<CtxGetCurrentFn>(cur),
                              reinterpret_cast<CtxGetIdFn>(id));
    }();
    if (fns.first == nullptr || fns.second == nullptr) return 0;
    void *ctx = nullptr;
    unsigned long long id = 0;
    if (fns.first(&ctx) != 0 || ctx == nullptr) return 0;
    if (fns.second(ctx, &id) != 0) return 0;
    return id;
}

cudaError_t noalloc_scratch(int dev, void **out) {
    const bool cacheable = dev >= 0 && dev < kMaxDevices;
    if (cacheable) {
        const unsigned long long id = current_context_id();
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (id != 0 && g_noalloc_slot[dev].ctx_id == id) {
            *out = g_noalloc_slot[dev].addr;
            return cudaSuccess;
        }
    }
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (cacheable) {
        // the lookup above has made the device's context current
        const unsigned long long id = current_context_id();
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        g_noalloc_slot[dev] = {id, p};
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" swiglu_status_t swiglu_gateup_bias_bwd_noalloc(
    const void *dy, const void *x, const void *bias, void *dx, void *dbias, int64_t rows, int64_t n,
    int64_t dy_row_stride, int64_t x_row_stride, int64_t dx_row_stride, swiglu_dtype_t dtype,
    int in_place, swiglu_stream_t stream) {
    swiglu_status_t st = check_common(dtype, rows, n);
    if (st != SWIGLU_OK) return st;
    if (rows == 0 || n == 0)  // no scratch needed
        return swiglu_gateup_bias_bwd(dy, x, bias, dx, dbias, nullptr, 0, rows, n, dy_row_stride,
                                      x_row_stride, dx_row_stride, dtype, in_place, stream);
    Device d;
    cudaError_t e = current_device(d);
    if (e != cudaSuccess) return cuda_fail(e);
    size_t off, need;
    if (!bias_workspace(rows, n, d.sms, false, off, need) || need > SWIGLU_NOALLOC_SCRATCH_BYTES)
        return SWIGLU_ERR_WORKSPACE;
    void *scratch = nullptr;
    e = noalloc_scratch(d.id, &scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    return swiglu_gateup_bias_bwd(dy, x, bias, dx, dbias, scratch, SWIGLU_NOALLOC_SCRATCH_BYTES,
                                  rows, n, dy_row_stride, x_row_stride, dx_row_stride, dtype,
                                  in_place, stream);
}
