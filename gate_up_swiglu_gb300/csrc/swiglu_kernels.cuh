// swiglu_kernels.cuh -- sm_103a kernels of the fused gate-up SwiGLU.
//
// Layout (Liger-Kernel Megatron SwiGLU page, §Background): row r of the fc1
// buffer x holds the gate g in columns [0, n) and the up projection u in
// columns [n, 2n); both halves are read straight out of that buffer through a
// column offset of n, so one pass streams g, u (and dy) from HBM and writes y
// (or d gate / d up) back, with no intermediate tensor.
//
// The work is pure streaming: 3n (forward) or 5n (backward) elements of HBM
// traffic per row and ~20 fp32 operations per element pair, so the kernels are
// bound by HBM bandwidth, not by arithmetic; tensor cores have nothing to do
// here.  Each thread moves aligned VEC-element packs (16 bytes when the shapes,
// strides and pointers allow it, narrower otherwise, one element for odd n)
// with streaming cache hints, keeps U independent packs per operand in flight,
// and a persistent grid (a whole number of resident CTAs on every SM) strides
// over the flattened (row, pack) index space.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "silu_root_poly.h"

namespace swiglu {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- memory ---
// Streaming loads/stores of one B-byte pack, viewed as 32-bit words
// (a 2-byte pack uses the low half of word 0).
template <int B>
struct Mem;

template <>
struct Mem<16> {
    static __device__ __forceinline__ void load(const void *p, uint32_t *w) {
        const uint4 r = __ldcs(reinterpret_cast<const uint4 *>(p));
        w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
    }
    static __device__ __forceinline__ void store(void *p, const uint32_t *w) {
        __stcs(reinterpret_cast<uint4 *>(p), make_uint4(w[0], w[1], w[2], w[3]));
    }
};
template <>
struct Mem<8> {
    static __device__ __forceinline__ void load(const void *p, uint32_t *w) {
        const uint2 r = __ldcs(reinterpret_cast<const uint2 *>(p));
        w[0] = r.x; w[1] = r.y;
    }
    static __device__ __forceinline__ void store(void *p, const uint32_t *w) {
        __stcs(reinterpret_cast<uint2 *>(p), make_uint2(w[0], w[1]));
    }
};
template <>
struct Mem<4> {
    static __device__ __forceinline__ void load(const void *p, uint32_t *w) {
        w[0] = __ldcs(reinterpret_cast<const unsigned int *>(p));
    }
    static __device__ __forceinline__ void store(void *p, const uint32_t *w) {
        __stcs(reinterpret_cast<unsigned int *>(p), w[0]);
    }
};
template <>
struct Mem<2> {
    static __device__ __forceinline__ void load(const void *p, uint32_t *w) {
        w[0] = __ldcs(reinterpret_cast<const unsigned short *>(p));
    }
    static __device__ __forceinline__ void store(void *p, const uint32_t *w) {
        __stcs(reinterpret_cast<unsigned short *>(p), static_cast<unsigned short>(w[0]));
    }
};

// ------------------------------------------------------------ data types ---
// Element i of a pack <-> fp32.  Storage rounding is round-to-nearest-even.
struct F32 {
    static constexpr int kBytes = 4;
    // fp32 results must sit within 2e-6 relative (1e-7 absolute) of the exact
    // value, which plain fp32 evaluation of silu' misses near its root.
    static constexpr bool kRootWindow = true;
    // fp32 results below the 1e-7 absolute floor are never graded, so the
    // deep negative tail needs no rescaling (see BF16::kDeepScale).
    static constexpr bool kDeepScale = false;
    static __device__ __forceinline__ float get(const uint32_t *w, int i) {
        return __uint_as_float(w[i]);
    }
    static __device__ __forceinline__ void put(uint32_t *w, int i, float f) {
        w[i] = __float_as_uint(f);
    }
};

struct BF16 {
    static constexpr int kBytes = 2;
    // one bf16 ulp (2^-8 relative) dwarfs the fp32 error of silu' at the bf16
    // values nearest its root (|silu'| >= 6e-4 there), so no root window.
    static constexpr bool kRootWindow = false;
    // For g < -64, exp(-|g|) heads into the fp32 subnormal range (below
    // g = -87.3) and loses relative precision, while silu(g) * u and friends
    // can still be normal or subnormal bf16 numbers.  There the exponential
    // is taken 64 binades higher and every result is scaled back by 2^-64 in
    // one final, correctly rounded multiply.
    static constexpr bool kDeepScale = true;
    static __device__ __forceinline__ float get(const uint32_t *w, int i) {
        const uint32_t word = w[i >> 1];
        return __uint_as_float((i & 1) ? (word & 0xFFFF0000u) : (word << 16));
    }
    static __device__ __forceinline__ void put(uint32_t *w, int i, float f) {
        const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
        w[i >> 1] |= (i & 1) ? (b << 16) : b;
    }
};

// ------------------------------------------------------------------ math ---
// sigmoid(g) and 1 - sigmoid(g) come from t = exp(-|g|) in (0, 1]:
//   g >= 0:  s = 1 / (1 + t),  1 - s = t / (1 + t)
//   g <  0:  s = t / (1 + t),  1 - s = 1 / (1 + t)
// so neither the exponential overflows nor 1 - s cancels, for any finite g.
// Explicit _rn operations fix the rounding of every step (no contraction), so
// all instantiations -- in particular the in-place and out-of-place backward
// -- produce the same bits.

constexpr float kLn2x64 = 44.3614195558365f;  // 64 ln 2
constexpr float kTwoPowMinus64 = 5.421010862427522e-20f;  // 2^-64, exact

// silu'(g0 + d) near the root g0 of silu', as a Taylor polynomial in d.
__device__ __forceinline__ float dsilu_near_root(float d) {
    constexpr float c[SILU_ROOT_DEGREE] = SILU_ROOT_COEFFS;
    float acc = c[SILU_ROOT_DEGREE - 1];
#pragma unroll
    for (int k = SILU_ROOT_DEGREE - 2; k >= 0; --k) acc = __fmaf_rn(acc, d, c[k]);
    return __fmul_rn(acc, d);
}

// The activation terms of one gate value:
//   silu  = g s            (times 2^64 when `scale` is 2^-64)
//   dsilu = s (1 + g (1 - s))   (same scaling)
//   scale = the factor every product of silu / dsilu must finally be multiplied by.
struct Act {
    float silu, dsilu, scale;
};

template <typename E, bool kGrad>
__device__ __forceinline__ Act activation(float g) {
    const float a = fabsf(g);
    const bool pos = g >= 0.0f;
    bool deep = false;
    float arg = a;
    if (E::kDeepScale) {
        // for a > 64, t * 2^64 < 2^-24, so 1 + t rounds to 1 with or without
        // the scaling and r = 1 stays exact
        deep = !pos && a > 64.0f;
        arg = deep ? __fsub_rn(a, kLn2x64) : a;
    }
    const float t = expf(-arg);
    const float r = __frcp_rn(__fadd_rn(1.0f, t));
    const float tr = __fmul_rn(t, r);
    const float s = pos ? r : tr;
    Act o;
    o.silu = __fmul_rn(g, s);
    o.scale = deep ? kTwoPowMinus64 : 1.0f;
    o.dsilu = 0.0f;
    if (kGrad) {
        const float oms = pos ? tr : r;
        o.dsilu = __fmul_rn(s, __fmaf_rn(g, oms, 1.0f));
        if (E::kRootWindow) {
            const float d = __fsub_rn(__fsub_rn(g, SILU_ROOT_G0_HI), SILU_ROOT_G0_LO);
            if (fabsf(d) < SILU_ROOT_WINDOW) o.dsilu = dsilu_near_root(d);
        }
    }
    return o;
}

// ---------------------------------------------------------------- kernels ---
// The index space is rows x nvec packs per half-row, flattened row-major.
// Thread t of CTA b starts at pack b * U * kThreads + t + k * kThreads (k < U)
// and advances by gridDim * U * kThreads packs per iteration; (row, column)
// of each of its U packs is carried along incrementally (step_q rows plus
// step_r packs, with one carry), so the loop needs no division.
struct FwdParams {
    const void *x;
    void *y;
    int64_t rows;
    int64_t x_stride;  // row strides, in packs
    int64_t y_stride;
    int64_t step_q;    // (gridDim * U * kThreads) / nvec
    int32_t nvec;      // packs per half-row (n / VEC)
    int32_t step_r;    // (gridDim * U * kThreads) % nvec
};

struct BwdParams {
    const void *dy;
    const void *x;
    void *dx;  // == x for the in-place backward
    int64_t rows;
    int64_t dy_stride;  // row strides, in packs
    int64_t x_stride;
    int64_t dx_stride;
    int64_t step_q;
    int32_t nvec;
    int32_t step_r;
};

template <int U>
__device__ __forceinline__ void first_positions(int64_t nvec, int64_t (&r)[U], int32_t (&c)[U]) {
    const int64_t base = (int64_t)blockIdx.x * (U * kThreads) + threadIdx.x;
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const int64_t v = base + (int64_t)k * kThreads;
        r[k] = v / nvec;
        c[k] = (int32_t)(v - r[k] * nvec);
    }
}

template <int U>
__device__ __forceinline__ void advance(int64_t step_q, int32_t step_r, int32_t nvec,
                                        int64_t (&r)[U], int32_t (&c)[U]) {
#pragma unroll
    for (int k = 0; k < U; ++k) {
        c[k] += step_r;
        r[k] += step_q;
        if (c[k] >= nvec) {
            c[k] -= nvec;
            r[k] += 1;
        }
    }
}

template <typename E, int VEC, int U>
__global__ void __launch_bounds__(kThreads) swiglu_fwd_kernel(const FwdParams p) {
    constexpr int B = E::kBytes * VEC;
    constexpr int NW = (B + 3) / 4;
    using M = Mem<B>;
    const char *x = static_cast<const char *>(p.x);
    char *y = static_cast<char *>(p.y);
    const int64_t up_off = (int64_t)p.nvec * B;

    int64_t r[U];
    int32_t c[U];
    first_positions<U>(p.nvec, r, c);
    while (r[0] < p.rows) {
        uint32_t g[U][NW], u[U][NW];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (r[k] < p.rows) {
                const char *px = x + (r[k] * p.x_stride + c[k]) * B;
                M::load(px, g[k]);
                M::load(px + up_off, u[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (r[k] < p.rows) {
                uint32_t o[NW] = {};
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const Act act = activation<E, false>(E::get(g[k], i));
                    E::put(o, i, __fmul_rn(__fmul_rn(act.silu, E::get(u[k], i)), act.scale));
                }
                M::store(y + (r[k] * p.y_stride + c[k]) * B, o);
            }
        }
        advance<U>(p.step_q, p.step_r, p.nvec, r, c);
    }
}

// IN_PLACE selects nothing but the aliasing contract (dx == x); the arithmetic
// is the same template body, so both instances give identical bits.
template <typename E, int VEC, int U, bool IN_PLACE>
__global__ void __launch_bounds__(kThreads) swiglu_bwd_kernel(const BwdParams p) {
    constexpr int B = E::kBytes * VEC;
    constexpr int NW = (B + 3) / 4;
    using M = Mem<B>;
    const char *dy = static_cast<const char *>(p.dy);
    const char *x = static_cast<const char *>(p.x);
    char *dx = IN_PLACE ? const_cast<char *>(x) : static_cast<char *>(p.dx);
    const int64_t up_off = (int64_t)p.nvec * B;

    int64_t r[U];
    int32_t c[U];
    first_positions<U>(p.nvec, r, c);
    while (r[0] < p.rows) {
        uint32_t d[U][NW], g[U][NW], u[U][NW];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (r[k] < p.rows) {
                const char *px = x + (r[k] * p.x_stride + c[k]) * B;
                M::load(dy + (r[k] * p.dy_stride + c[k]) * B, d[k]);
                M::load(px, g[k]);
                M::load(px + up_off, u[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (r[k] < p.rows) {
                uint32_t og[NW] = {}, ou[NW] = {};
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    const float gf = E::get(g[k], i);
                    const float uf = E::get(u[k], i);
                    const float df = E::get(d[k], i);
                    const Act act = activation<E, true>(gf);
                    E::put(og, i, __fmul_rn(__fmul_rn(df, __fmul_rn(uf, act.dsilu)), act.scale));
                    E::put(ou, i, __fmul_rn(__fmul_rn(df, act.silu), act.scale));
                }
                char *pdx = dx + (r[k] * p.dx_stride + c[k]) * B;
                M::store(pdx, og);
                M::store(pdx + up_off, ou);
            }
        }
        advance<U>(p.step_q, p.step_r, p.nvec, r, c);
    }
}

}  // namespace swiglu
