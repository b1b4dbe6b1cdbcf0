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
// here.  Each thread moves aligned VEC-element packs (32 or 16 bytes when the
// shapes, strides and pointers allow it, narrower otherwise) with streaming
// cache hints and keeps U independent packs per operand in flight; the grid
// strides over the flattened (row, pack) index space, either in one pass (a
// CTA per U * T packs, T threads per CTA) or as a persistent grid of a few
// resident CTAs per SM, as the host's launch policy decides.  Shapes whose
// operands share no pack wider than 4 bytes (odd n, misaligned rows) go to
// the row-segment kernels further down (the forward of every form and the
// plain backward).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "silu_root_poly.h"

namespace swiglu {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- memory ---
// Loads and stores of one B-byte pack (B = 32, 16, 8, 4 or 2), viewed as
// 32-bit words (a 2-byte pack uses the low half of word 0).  32-byte packs use
// the 256-bit global accesses of sm_100-class GPUs.  The cache behaviour is a
// template parameter:
//   loads   kLdStream      ld.global.cs            evict-first, coherent
//           kLdNoAlloc     ld.global.L1::no_allocate                  coherent
//           kLdNoAlloc256  ... .L2::256B           + 256-byte L2 prefetch
//           kLdNC          ld.global.nc.L1::no_allocate   read-only path
//           kLdNC256       ... .L2::256B           + 256-byte L2 prefetch
//           kLdCached      ld.global.nc            read-only, cached in L1 (bias
//                                                  vectors reread by every row)
//   stores  kStStream      st.global.cs            evict-first
//           kStNoAlloc     st.global.L1::no_allocate
//           kStPlain       st.global
// The read-only (.nc) kinds are only legal when no thread of the kernel writes
// the loaded memory, i.e. never for the in-place backward.
enum : int { kLdStream = 0, kLdNoAlloc = 1, kLdNoAlloc256 = 2, kLdNC = 3, kLdNC256 = 4, kLdCached = 5 };
enum : int { kStStream = 0, kStNoAlloc = 1, kStPlain = 2 };

template <int B, int KIND>
struct Ld;
template <int B, int KIND>
struct St;

#define SWIGLU_DEFINE_LD(KIND, QUAL)                                                           \
    template <>                                                                                \
    struct Ld<32, KIND> {                                                                      \
        static __device__ __forceinline__ void run(const void *p, uint32_t *w) {               \
            asm(QUAL ".v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"                          \
                : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),       \
                  "=r"(w[6]), "=r"(w[7])                                                       \
                : "l"(p));                                                                     \
        }                                                                                      \
    };                                                                                         \
    template <>                                                                                \
    struct Ld<16, KIND> {                                                                      \
        static __device__ __forceinline__ void run(const void *p, uint32_t *w) {               \
            asm(QUAL ".v4.b32 {%0, %1, %2, %3}, [%4];"                                          \
                : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])                                \
                : "l"(p));                                                                     \
        }                                                                                      \
    };                                                                                         \
    template <>                                                                                \
    struct Ld<8, KIND> {                                                                       \
        static __device__ __forceinline__ void run(const void *p, uint32_t *w) {               \
            asm(QUAL ".v2.b32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));              \
        }                                                                                      \
    };                                                                                         \
    template <>                                                                                \
    struct Ld<4, KIND> {                                                                       \
        static __device__ __forceinline__ void run(const void *p, uint32_t *w) {               \
            asm(QUAL ".b32 %0, [%1];" : "=r"(w[0]) : "l"(p));                                   \
        }                                                                                      \
    };                                                                                         \
    template <>                                                                                \
    struct Ld<2, KIND> {                                                                       \
        static __device__ __forceinline__ void run(const void *p, uint32_t *w) {               \
            unsigned short h;                                                                  \
            asm(QUAL ".b16 %0, [%1];" : "=h"(h) : "l"(p));                                      \
            w[0] = h;                                                                          \
        }                                                                                      \
    };

SWIGLU_DEFINE_LD(kLdStream, "ld.global.cs")
SWIGLU_DEFINE_LD(kLdNoAlloc, "ld.global.L1::no_allocate")
SWIGLU_DEFINE_LD(kLdNoAlloc256, "ld.global.L1::no_allocate.L2::256B")
SWIGLU_DEFINE_LD(kLdNC, "ld.global.nc.L1::no_allocate")
SWIGLU_DEFINE_LD(kLdNC256, "ld.global.nc.L1::no_allocate.L2::256B")
SWIGLU_DEFINE_LD(kLdCached, "ld.global.nc")
#undef SWIGLU_DEFINE_LD

#define SWIGLU_DEFINE_ST(KIND, QUAL)                                                           \
    template <>                                                                                \
    struct St<32, KIND> {                                                                      \
        static __device__ __forceinline__ void run(void *p, const uint32_t *w) {               \
            asm volatile(QUAL ".v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),       \
                         "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),       \
                         "r"(w[6]), "r"(w[7]));                                                 \
        }                                                                                      \
    };                                                                                         \
    template <>                                                                                \
    struct St<16, KIND> {                                                                      \
        static __device__ __forceinline__ void run(void *p, const uint32_t *w) {               \
            asm volatile(QUAL ".v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(w[0]), "r"(w[1]), \
                         "r"(w[2]), "r"(w[3]));                                                 \
        }                                                                                      \
    };                                                                                         \
    template <>                                                                                \
    struct St<8, KIND> {                                                                       \
        static __device__ __forceinline__ void run(void *p, const uint32_t *w) {               \
            asm volatile(QUAL ".v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(w[0]), "r"(w[1]));        \
        }                                                                                      \
    };                                                                                         \
    template <>                                                                                \
    struct St<4, KIND> {                                                                       \
        static __device__ __forceinline__ void run(void *p, const uint32_t *w) {               \
            asm volatile(QUAL ".b32 [%0], %1;" ::"l"(p), "r"(w[0]));                            \
        }                                                                                      \
    };                                                                                         \
    template <>                                                                                \
    struct St<2, KIND> {                                                                       \
        static __device__ __forceinline__ void run(void *p, const uint32_t *w) {               \
            asm volatile(QUAL ".b16 [%0], %1;" ::"l"(p), "h"((unsigned short)w[0]));            \
        }                                                                                      \
    };

SWIGLU_DEFINE_ST(kStStream, "st.global.cs")
SWIGLU_DEFINE_ST(kStNoAlloc, "st.global.L1::no_allocate")
SWIGLU_DEFINE_ST(kStPlain, "st.global")
#undef SWIGLU_DEFINE_ST

// Asynchronous 16-byte copies from global into shared memory (cached in L2
// only), grouped by commit_group and awaited by wait_group: the issuing
// thread may read its own copies once the wait returns.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
// 4- and 8-byte copies (cached in L1 as well: the L2-only form takes 16 bytes)
template <int B>
__device__ __forceinline__ void cp_async_small(void *smem_dst, const void *gsrc) {
    static_assert(B == 4 || B == 8, "cp.async copies 4, 8 or 16 bytes");
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;" ::"r"(d), "l"(gsrc), "n"(B) : "memory");
}
template <int B>
__device__ __forceinline__ void cp_async_pack(void *smem_dst, const void *gsrc) {
    if constexpr (B == 16)
        cp_async16(smem_dst, gsrc);
    else
        cp_async_small<B>(smem_dst, gsrc);
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

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
    // accurate expf and IEEE reciprocal: the fp32 tolerance needs them
    static constexpr bool kFastExp = false;
    static __device__ __forceinline__ float get(const uint32_t *w, int i) {
        return __uint_as_float(w[i]);
    }
    static __device__ __forceinline__ void put(uint32_t *w, int i, float f) {
        w[i] = __float_as_uint(f);
    }
    static __device__ __forceinline__ void put2(uint32_t *w, int i, float f0, float f1) {
        w[i] = __float_as_uint(f0);
        w[i + 1] = __float_as_uint(f1);
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
    // The hardware base-2 exponential and reciprocal (relative errors near
    // 2^-22) are far inside one bf16 step (2^-8).  With the deep-tail scaling
    // above, the exponential's result is never subnormal where it matters, so
    // their flush-to-zero of subnormal results is harmless.
    static constexpr bool kFastExp = true;
    static __device__ __forceinline__ float get(const uint32_t *w, int i) {
        const uint32_t word = w[i >> 1];
        return __uint_as_float((i & 1) ? (word & 0xFFFF0000u) : (word << 16));
    }
    static __device__ __forceinline__ void put(uint32_t *w, int i, float f) {
        const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
        w[i >> 1] |= (i & 1) ? (b << 16) : b;
    }
    // elements i (even) and i + 1 in one packed conversion, both RNE
    static __device__ __forceinline__ void put2(uint32_t *w, int i, float f0, float f1) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);
        w[i >> 1] = (uint32_t)__bfloat16_as_ushort(h.x) | ((uint32_t)__bfloat16_as_ushort(h.y) << 16);
    }
};

// ------------------------------------------- programmatic dependent launch ---
// The host launches every streaming kernel so that the next kernel in the
// stream may launch while this one's last CTAs still run (sm_90 and later).
// Each kernel therefore first waits until the grid before it in the stream has
// completed and its writes are visible -- before any global memory access,
// read or write -- and later lets the next one launch: once every CTA of a
// grid has done so, the next grid's CTAs are placed on SMs as room appears and
// start the moment this grid completes, instead of after a full launch.
// Every kernel lets it go at the top: for a grid of many waves that happens
// once its last wave has started.
__device__ __forceinline__ void await_previous_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ math ---
// fp32 (and the deep bf16 tail): sigmoid(g) and 1 - sigmoid(g) come from
// t = exp(-|g|) in (0, 1]:
//   g >= 0:  s = 1 / (1 + t),  1 - s = t / (1 + t)
//   g <  0:  s = t / (1 + t),  1 - s = 1 / (1 + t)
// so neither the exponential overflows nor 1 - s cancels, for any finite g.
// bf16 with g >= -64 takes a shorter form that one bf16 step tolerates (see
// activation below).  Explicit _rn operations fix the rounding of every step
// (no contraction), so all instantiations -- in particular the in-place and
// out-of-place backward -- produce the same bits.

constexpr float kLn2x64 = 44.3614195558365f;  // 64 ln 2
constexpr float kTwoPowMinus64 = 5.421010862427522e-20f;  // 2^-64, exact
constexpr float kLog2e = 1.4426950408889634f;

// exp(x) = 2^(x log2 e) with the hardware base-2 exponential (PTX
// ex2.approx.ftz), and the hardware reciprocal (PTX rcp.approx.ftz).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two fp32 lanes per instruction (PTX .f32x2 arithmetic, sm_100 and later):
// each lane rounds to nearest even exactly as the scalar operation does.
__device__ __forceinline__ uint64_t x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void x2_split(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul_x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t add_x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub_x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma_x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

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

// Knuth's TwoSum: s = fl(a + b) and the exact rounding error e, a + b = s + e.
__device__ __forceinline__ float two_sum(float a, float b, float &e) {
    const float s = __fadd_rn(a, b);
    const float bv = __fsub_rn(s, a);
    const float av = __fsub_rn(s, bv);
    e = __fadd_rn(__fsub_rn(a, av), __fsub_rn(b, bv));
    return s;
}

// g_lo: a correction the exact gate value carries beyond the fp32 g (the
// rounding error of g + bias); only the root window of silu' is sensitive
// enough to need it.
// kMayDeep = false: the caller knows g >= -64 (or NaN), so the deep-tail
// scaling is left out (scale is exactly 1; same bits as the general form).
//
// Storage types with the hardware exponential (bf16), g >= -64 or NaN: with
// t = e^-g <= e^64 nothing overflows, so
//   s = 1 / (1 + t),  1 - s = 1 - s (rounded),  silu' = s (1 + g (1 - s))
// without |g|, a sign test or selects.  Error, relative to one bf16 step
// (2^-8): t carries the rounding of its exponent argument (at most 2^-18 ln 2
// relative, at |g| = 64) and ex2.approx / rcp.approx their ~2^-22, so s is
// within ~3e-6 relative; 1 - s adds an absolute 2^-24, which only matters
// where 1 + g (1 - s) is small: at the bf16 gates nearest silu's root
// (|1 + g (1 - s)| >= 0.0028) it stays below 1e-4 relative, and for large
// positive g the term g (1 - s) is below 1e-6 against 1.  So every result is
// within a small fraction of a bf16 step of the exact value before its single
// rounding.  g < -64 takes the scaled form below.
template <typename E, bool kGrad, bool kMayDeep = true>
__device__ __forceinline__ Act activation(float g, float g_lo = 0.0f) {
    if (E::kFastExp && !(E::kDeepScale && kMayDeep && g < -64.0f)) {
        const float s = rcp_approx(__fadd_rn(1.0f, ex2_approx(__fmul_rn(g, -kLog2e))));
        Act o;
        o.silu = __fmul_rn(g, s);
        o.scale = 1.0f;
        o.dsilu = kGrad ? __fmul_rn(s, __fmaf_rn(g, __fsub_rn(1.0f, s), 1.0f)) : 0.0f;
        return o;
    }
    const float a = fabsf(g);
    const bool pos = g >= 0.0f;
    // deep: for g < -64, t * 2^64 < 2^-24, so 1 + t rounds to 1 with or
    // without the scaling and r = 1 stays exact
    const bool deep = E::kDeepScale && kMayDeep && g < -64.0f;
    float t;
    if (E::kFastExp) {
        // t = 2^(-|g| log2 e (+ 64 when deep))
        t = ex2_approx(__fmaf_rn(a, -kLog2e, deep ? 64.0f : 0.0f));
    } else {
        t = expf(-(deep ? __fsub_rn(a, kLn2x64) : a));
    }
    const float r = E::kFastExp ? rcp_approx(__fadd_rn(1.0f, t)) : __frcp_rn(__fadd_rn(1.0f, t));
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
            const float d = __fadd_rn(__fsub_rn(g, SILU_ROOT_G0_HI), __fsub_rn(g_lo, SILU_ROOT_G0_LO));
            if (fabsf(d) < SILU_ROOT_WINDOW) o.dsilu = dsilu_near_root(d);
        }
    }
    return o;
}

// True when some gate of the pack is below -64, where the storage type needs
// the deep-tail scaling (never for fp32).  NaN gates do not count, as in the
// scalar test.
template <typename E, int VEC>
__device__ __forceinline__ bool pack_has_deep(const uint32_t *g) {
    if (!E::kDeepScale) return false;
    float m = E::get(g, 0);
#pragma unroll
    for (int i = 1; i < VEC; ++i) m = fminf(m, E::get(g, i));
    return m < -64.0f;
}

// pack_has_deep for the gates shifted by their bias (rounded as bwd_pair
// rounds them).
template <typename E, int VEC>
__device__ __forceinline__ bool pack_has_deep_biased(const uint32_t *g, const uint32_t *bg) {
    if (!E::kDeepScale) return false;
    float m = __fadd_rn(E::get(g, 0), E::get(bg, 0));
#pragma unroll
    for (int i = 1; i < VEC; ++i) m = fminf(m, __fadd_rn(E::get(g, i), E::get(bg, i)));
    return m < -64.0f;
}

// Round VEC fp32 results into the words of one pack (pairs at a time when
// there are pairs).
template <typename E, int VEC>
__device__ __forceinline__ void store_pack(uint32_t *w, const float *v) {
    if (VEC == 1) {
        E::put(w, 0, v[0]);
    } else {
#pragma unroll
        for (int i = 0; i < VEC; i += 2) E::put2(w, i, v[i], v[i + 1]);
    }
}

// ------------------------------------------------ division by an invariant ---
// v / d for 0 <= v < 2^63 and a divisor d fixed per launch, by one high
// multiplication and a shift (Granlund and Montgomery, "Division by invariant
// integers using multiplication", PLDI 1994, Theorem 4.2, with N = 63):
// with l = ceil(log2 d) and m = ceil(2^(63 + l) / d), m < 2^64 and
// v / d = floor(v m / 2^(63 + l)) = (high 64 bits of v m) >> (l - 1).
// d == 1 is marked by shift < 0.  The host computes m and the shift.
struct FastDiv {
    uint64_t m;
    int32_t shift;  // l - 1, or -1 when d == 1
};

__device__ __forceinline__ int64_t fast_div(int64_t v, const FastDiv &f) {
    return f.shift < 0 ? v : (int64_t)(__umul64hi((uint64_t)v, f.m) >> f.shift);
}

// ---------------------------------------------------------------- kernels ---
// The index space is rows x nvec packs per half-row, flattened row-major.
// Thread t of CTA b (T threads per CTA) starts at pack b * U * T + t + k * T
// (k < U) and advances by gridDim * U * T packs per iteration; (row, column)
// of each of its U packs is found once by a division by the invariant nvec and
// then carried along incrementally (step_q rows plus step_r packs, with one
// carry), so the loop itself needs no division.
// The gate and up operands are addressed separately (base pointer and row
// stride each), which covers both the fused [rows, 2n] buffer (up = gate + n,
// same stride) and two separate tensors.
// Variants of the activation:
//   kPlain   silu(g) * u
//   kBias    silu(g + bias_g[j]) * (u + bias_u[j])
//   kWeight  w[r] * silu(g) * u            (w: fp32 per row)
//   kBiasWeight  both: w[r] * silu(g + bias_g[j]) * (u + bias_u[j])
enum : int { kPlain = 0, kBias = 1, kWeight = 2, kBiasWeight = 3 };  // bit flags

struct FwdParams {
    const void *g;
    const void *u;
    void *y;
    const void *bias_g;  // kBias: [n] bias of the gate half
    const void *bias_u;  // kBias: [n] bias of the up half
    const float *w;      // kWeight: [rows]
    int64_t rows;
    int64_t g_stride;  // row strides, in packs
    int64_t u_stride;
    int64_t y_stride;
    int64_t step_q;    // (gridDim * U * T) / nvec
    FastDiv div_nvec;  // division by nvec
    int32_t nvec;      // packs per row of each operand (n / VEC)
    int32_t step_r;    // (gridDim * U * T) % nvec
};

struct BwdParams {
    const void *dy;
    const void *g;
    const void *u;
    void *dg;  // == g for the in-place backward
    void *du;  // == u for the in-place backward
    const void *bias_g;  // kBias
    const void *bias_u;
    const float *w;      // kWeight: [rows]
    float *dw;           // kWeight: [rows]
    float *partial;      // kBias: [groups, 2n] fp32 column sums per row group
    float *partial_dw;   // kBiasWeight: [rows, tiles] fp32 row sums per column tile
    int64_t rows;
    int64_t dy_stride;  // row strides, in packs
    int64_t g_stride;
    int64_t u_stride;
    int64_t dg_stride;
    int64_t du_stride;
    int64_t step_q;
    FastDiv div_nvec;
    int32_t nvec;
    int32_t step_r;
};

template <int U, int T = kThreads>
__device__ __forceinline__ void first_positions(int64_t nvec, const FastDiv &div, int64_t (&r)[U],
                                                int32_t (&c)[U]) {
    const int64_t base = (int64_t)blockIdx.x * (U * T) + threadIdx.x;
#pragma unroll
    for (int k = 0; k < U; ++k) {
        const int64_t v = base + (int64_t)k * T;
        r[k] = fast_div(v, div);
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

// One pack of the forward into yv.
template <typename E, int VEC, int MODE, bool kMayDeep>
__device__ __forceinline__ void fwd_pack(const uint32_t *g, const uint32_t *u, const uint32_t *bg,
                                         const uint32_t *bu, float wr, float *yv) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        float gf = E::get(g, i), uf = E::get(u, i);
        if (MODE & kBias) {
            gf = __fadd_rn(gf, E::get(bg, i));
            uf = __fadd_rn(uf, E::get(bu, i));
        }
        const Act act = activation<E, false, kMayDeep>(gf);
        float v = __fmul_rn(act.silu, uf);
        if (MODE & kWeight) v = __fmul_rn(v, wr);
        if (kMayDeep) v = __fmul_rn(v, act.scale);
        yv[i] = v;
    }
}

// T: threads per CTA (kThreads unless the launch policy picks another).
// SPLIT: test each pack for the deep tail and run the common case without
// the per-element test (same bits either way).
template <typename E, int VEC, int U, int LD, int ST, int MODE = kPlain, int T = kThreads,
          bool SPLIT = true>
__global__ void __launch_bounds__(T, MODE == kBiasWeight ? 4 : 0) swiglu_fwd_kernel(const FwdParams p) {
    await_previous_grid();
    allow_next_grid();
    constexpr int B = E::kBytes * VEC;
    constexpr int NW = (B + 3) / 4;
    using L = Ld<B, LD>;
    using S = St<B, ST>;
    const char *gp = static_cast<const char *>(p.g);
    const char *up = static_cast<const char *>(p.u);
    char *y = static_cast<char *>(p.y);

    int64_t r[U];
    int32_t c[U];
    first_positions<U, T>(p.nvec, p.div_nvec, r, c);
    while (r[0] < p.rows) {
        uint32_t g[U][NW], u[U][NW];
        uint32_t bg[U][NW], bu[U][NW];
        float wr[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            wr[k] = 1.0f;
            if (r[k] < p.rows) {
                L::run(gp + (r[k] * p.g_stride + c[k]) * B, g[k]);
                L::run(up + (r[k] * p.u_stride + c[k]) * B, u[k]);
                if (MODE & kBias) {
                    Ld<B, kLdCached>::run(static_cast<const char *>(p.bias_g) + (int64_t)c[k] * B, bg[k]);
                    Ld<B, kLdCached>::run(static_cast<const char *>(p.bias_u) + (int64_t)c[k] * B, bu[k]);
                }
                if (MODE & kWeight) wr[k] = __ldg(p.w + r[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (r[k] < p.rows) {
                uint32_t o[NW] = {};
                float yv[VEC];
                // packs with no gate below -64 (all but the deep tail) take
                // the activation without the deep-tail test (same bits)
                const bool deep = !SPLIT ? true
                                  : (MODE & kBias) ? pack_has_deep_biased<E, VEC>(g[k], bg[k])
                                                   : pack_has_deep<E, VEC>(g[k]);
                if (deep)
                    fwd_pack<E, VEC, MODE, true>(g[k], u[k], bg[k], bu[k], wr[k], yv);
                else
                    fwd_pack<E, VEC, MODE, false>(g[k], u[k], bg[k], bu[k], wr[k], yv);
                store_pack<E, VEC>(o, yv);
                S::run(y + (r[k] * p.y_stride + c[k]) * B, o);
            }
        }
        advance<U>(p.step_q, p.step_r, p.nvec, r, c);
    }
}

// The backward of one pack: dgate and dup in fp32.
template <typename E, int VEC, bool kMayDeep>
__device__ __forceinline__ void bwd_pack(const uint32_t *d, const uint32_t *g, const uint32_t *u,
                                         float *gv, float *uv) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const float gf = E::get(g, i);
        const float uf = E::get(u, i);
        const float df = E::get(d, i);
        const Act act = activation<E, true, kMayDeep>(gf);
        float a = __fmul_rn(df, __fmul_rn(uf, act.dsilu));
        float b = __fmul_rn(df, act.silu);
        if (kMayDeep) {
            a = __fmul_rn(a, act.scale);
            b = __fmul_rn(b, act.scale);
        }
        gv[i] = a;
        uv[i] = b;
    }
}

// IN_PLACE selects nothing but the aliasing contract (an output may be the
// very buffer of the matching input, so LD must be a coherent kind); the
// arithmetic is the same template body, so both instances give identical bits.
template <typename E, int VEC, int U, bool IN_PLACE, int LD, int ST, int T = kThreads>
__global__ void __launch_bounds__(T) swiglu_bwd_kernel(const BwdParams p) {
    await_previous_grid();
    allow_next_grid();
    static_assert(!IN_PLACE || (LD != kLdNC && LD != kLdNC256),
                  "the in-place backward writes what it reads: no read-only loads");
    constexpr int B = E::kBytes * VEC;
    constexpr int NW = (B + 3) / 4;
    using L = Ld<B, LD>;
    using S = St<B, ST>;
    const char *dy = static_cast<const char *>(p.dy);
    const char *gp = static_cast<const char *>(p.g);
    const char *up = static_cast<const char *>(p.u);
    char *dg = static_cast<char *>(p.dg);
    char *du = static_cast<char *>(p.du);

    int64_t r[U];
    int32_t c[U];
    first_positions<U, T>(p.nvec, p.div_nvec, r, c);
    while (r[0] < p.rows) {
        uint32_t d[U][NW], g[U][NW], u[U][NW];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (r[k] < p.rows) {
                L::run(dy + (r[k] * p.dy_stride + c[k]) * B, d[k]);
                L::run(gp + (r[k] * p.g_stride + c[k]) * B, g[k]);
                L::run(up + (r[k] * p.u_stride + c[k]) * B, u[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (r[k] < p.rows) {
                uint32_t og[NW] = {}, ou[NW] = {};
                float gv[VEC], uv[VEC];
                if (pack_has_deep<E, VEC>(g[k]))
                    bwd_pack<E, VEC, true>(d[k], g[k], u[k], gv, uv);
                else
                    bwd_pack<E, VEC, false>(d[k], g[k], u[k], gv, uv);
                store_pack<E, VEC>(og, gv);
                store_pack<E, VEC>(ou, uv);
                S::run(dg + (r[k] * p.dg_stride + c[k]) * B, og);
                S::run(du + (r[k] * p.du_stride + c[k]) * B, ou);
            }
        }
        advance<U>(p.step_q, p.step_r, p.nvec, r, c);
    }
}

// ----------------------------------------------------- row-segment kernels ---
// When the operands of a call share no pack wider than 4 bytes -- odd n, or
// rows and base pointers misaligned to one another, as in the fp32 odd-width
// workload, where the gate and up of one column sit 12 bytes apart mod 16 and
// rows 8 bytes apart -- the flattened (row, pack) walk above spends most of
// its instructions on per-element 64-bit index arithmetic.  These kernels
// take one segment of K * T columns of one row at a time instead: each thread
// forms its operand pointers once per segment and reaches its K columns
// (t, t + T, ..., so a warp touches consecutive elements) through constant
// offsets, loading all of them before computing any.  The arithmetic is
// fwd_pack / bwd_pack on one-element packs, split on the deep tail like the
// pack kernels, so the bits equal those of every other kernel; each column is
// read and written by one thread, so the in-place backward is the same kernel
// with coherent loads.
enum : int { kSegFwd = 0, kSegBwd = 1 };

struct SegParams {
    const char *in[3];      // fwd: g, u; bwd: dy, g, u (address of row 0, column 0)
    int64_t in_stride[3];   // row strides in bytes
    char *out[2];           // fwd: y; bwd: dg, du
    int64_t out_stride[2];
    const char *bias_g;     // forward with kBias: [n] bias of each half (column 0)
    const char *bias_u;
    const float *w;         // forward with kWeight: [rows]
    int64_t n;
    int64_t segments;       // rows * chunks
    FastDiv div_chunks;     // division by chunks
    int32_t chunks;         // segments per row: ceil(n / (K * T))
};

// FMODE: the forward's variant (kPlain, kBias, kWeight, kBiasWeight); the
// backward is the plain form only.  PV: elements per pack (2 for bf16 whose
// operands all allow 4-byte packs; p.n then counts packs).
template <typename E, int MODE, int K, int T, int LD, int FMODE = kPlain, int PV = 1>
__global__ void __launch_bounds__(T) swiglu_rowseg_kernel(const SegParams p) {
    await_previous_grid();
    allow_next_grid();
    static_assert(PV == 1 || (PV == 2 && E::kBytes == 2), "packs of one element, or two bf16");
    constexpr int EB = E::kBytes * PV;
    constexpr int NIN = MODE == kSegFwd ? 2 : 3;
    constexpr int NOUT = MODE == kSegFwd ? 1 : 2;
    static_assert(MODE == kSegFwd || FMODE == kPlain, "the backward row segments are the plain form");
    for (int64_t seg = blockIdx.x; seg < p.segments; seg += gridDim.x) {
        const int64_t r = fast_div(seg, p.div_chunks);
        const int64_t c = (seg - r * p.chunks) * (int64_t)(K * T) + threadIdx.x;
        // columns of this thread in the segment: c + i * T for i < live
        const int64_t left = p.n - c;
        const int live = left <= 0 ? 0 : (left >= (int64_t)(K - 1) * T + 1 ? K : (int)((left + T - 1) / T));
        const char *ip[NIN];
#pragma unroll
        for (int x = 0; x < NIN; ++x) ip[x] = p.in[x] + r * p.in_stride[x] + c * EB;
        uint32_t w[NIN][K];
        uint32_t bgw[K], buw[K];  // kBias: the bias of each column (reread by every row: L1)
#pragma unroll
        for (int i = 0; i < K; ++i) {
            if (i < live) {
#pragma unroll
                for (int x = 0; x < NIN; ++x) Ld<EB, LD>::run(ip[x] + i * T * EB, &w[x][i]);
                if (FMODE & kBias) {
                    Ld<EB, kLdCached>::run(p.bias_g + (c + i * T) * EB, &bgw[i]);
                    Ld<EB, kLdCached>::run(p.bias_u + (c + i * T) * EB, &buw[i]);
                }
            }
        }
        const float wr = (FMODE & kWeight) ? __ldg(p.w + r) : 1.0f;
        char *op[NOUT];
#pragma unroll
        for (int x = 0; x < NOUT; ++x) op[x] = p.out[x] + r * p.out_stride[x] + c * EB;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            if (i < live) {
                if (MODE == kSegFwd) {
                    float yv[PV];
                    const bool deep = (FMODE & kBias) ? pack_has_deep_biased<E, PV>(&w[0][i], &bgw[i])
                                                      : pack_has_deep<E, PV>(&w[0][i]);
                    if (deep)
                        fwd_pack<E, PV, FMODE, true>(&w[0][i], &w[1][i], &bgw[i], &buw[i], wr, yv);
                    else
                        fwd_pack<E, PV, FMODE, false>(&w[0][i], &w[1][i], &bgw[i], &buw[i], wr, yv);
                    uint32_t o[1] = {0u};
                    store_pack<E, PV>(o, yv);
                    St<EB, kStStream>::run(op[0] + i * T * EB, o);
                } else {
                    float gv[PV], uv[PV];
                    if (pack_has_deep<E, PV>(&w[1][i]))
                        bwd_pack<E, PV, true>(&w[0][i], &w[1][i], &w[2][i], gv, uv);
                    else
                        bwd_pack<E, PV, false>(&w[0][i], &w[1][i], &w[2][i], gv, uv);
                    uint32_t og[1] = {0u}, ou[1] = {0u};
                    store_pack<E, PV>(og, gv);
                    store_pack<E, PV>(ou, uv);
                    St<EB, kStStream>::run(op[0] + i * T * EB, og);
                    St<EB, kStStream>::run(op[1] + i * T * EB, ou);
                }
            }
        }
    }
}

// ------------------------------------------------ backward with reductions ---

// Sum of v over the CTA (kThreads threads), in a fixed order; every thread
// gets the result.  `red` is shared scratch of kThreads / 32 floats.
__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red may still be read from the previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int k = 0; k < kThreads / 32; ++k) t = __fadd_rn(t, red[k]);
    return t;
}

// One element pair of the backward: dy scaled by the row weight when there is
// one, gate and up shifted by their bias when there is one.
template <typename E, int MODE>
struct BwdPair {
    float dg, du, dw_term;
};

template <typename E, int MODE, bool kMayDeep = true>
__device__ __forceinline__ BwdPair<E, MODE> bwd_pair(float df, float gf, float uf, float bgf,
                                                     float buf, float wr) {
    float g_lo = 0.0f;
    if (MODE & kBias) {
        if (E::kRootWindow)
            gf = two_sum(gf, bgf, g_lo);
        else
            gf = __fadd_rn(gf, bgf);
        uf = __fadd_rn(uf, buf);
    }
    const Act act = activation<E, true, kMayDeep>(gf, g_lo);
    BwdPair<E, MODE> o;
    o.dw_term = 0.0f;
    if (MODE & kWeight) {
        // dw[r] sums dy * silu(g) * u over the row; dy * w drives the gradient
        o.dw_term = __fmul_rn(__fmul_rn(df, act.silu), uf);
        if (kMayDeep) o.dw_term = __fmul_rn(o.dw_term, act.scale);
        df = __fmul_rn(df, wr);
    }
    o.dg = __fmul_rn(df, __fmul_rn(uf, act.dsilu));
    o.du = __fmul_rn(df, act.silu);
    if (kMayDeep) {
        o.dg = __fmul_rn(o.dg, act.scale);
        o.du = __fmul_rn(o.du, act.scale);
    }
    return o;
}

// bwd_pair of two elements at once (d2, g2, u2: dy, the gate with its bias
// added, and up, one element per lane), for storage types with the hardware
// exponential and no gate below -64: the same operations in the same order,
// each lane rounded as the scalar operation rounds, so the same bits as
// bwd_pair<E, MODE, false>; the exponential and the reciprocal stay one per
// element.  The dw terms come back apart, for the caller to add in element
// order.
template <int MODE>
__device__ __forceinline__ void bwd_pair_x2(uint64_t d2, uint64_t g2, uint64_t u2, uint64_t w2,
                                            uint64_t &dg2, uint64_t &du2, float &dw0, float &dw1) {
    const uint64_t one = x2(1.0f, 1.0f);
    float t0, t1, q0, q1;
    x2_split(mul_x2(g2, x2(-kLog2e, -kLog2e)), t0, t1);
    x2_split(add_x2(one, x2(ex2_approx(t0), ex2_approx(t1))), q0, q1);
    const uint64_t s2 = x2(rcp_approx(q0), rcp_approx(q1));
    const uint64_t silu2 = mul_x2(g2, s2);
    const uint64_t dsilu2 = mul_x2(s2, fma_x2(g2, sub_x2(one, s2), one));
    if (MODE & kWeight) {
        x2_split(mul_x2(mul_x2(d2, silu2), u2), dw0, dw1);
        d2 = mul_x2(d2, w2);
    }
    dg2 = mul_x2(d2, mul_x2(u2, dsilu2));
    du2 = mul_x2(d2, silu2);
}

// Packs of two elements or more in the branch-free bf16 form of the weights
// + bias backward take bwd_pair_x2 pair by pair: the same bits, fewer
// instructions for that issue-bound kernel (fractions of the copy rate: 8-byte
// packs 0.783 -> 0.812, bf16 [6000, 2 x 5000] 0.677 -> 0.704, ffn-4096 and
// the large FFN +0.4 %).  The bias form (0.2-0.5 % slower) and the weighted
// row kernel (2-7 % slower at its register bound) keep the scalar form.
template <typename E, int VEC, int MODE, bool kMayDeep>
constexpr bool kPairwise = MODE == kBiasWeight && E::kFastExp && !kMayDeep && VEC % 2 == 0;

// Weighted backward: one CTA per row (persistent over rows), so dw[r] is a
// fixed-order reduction inside the CTA: no scratch, deterministic.
template <typename E, int VEC, bool kMayDeep>
__device__ __forceinline__ void weighted_pack(const uint32_t *d, const uint32_t *g, const uint32_t *u,
                                              float wr, float &acc, float *gv, float *uv) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const BwdPair<E, kWeight> o = bwd_pair<E, kWeight, kMayDeep>(E::get(d, i), E::get(g, i),
                                                                     E::get(u, i), 0.0f, 0.0f, wr);
        acc = __fadd_rn(acc, o.dw_term);
        gv[i] = o.dg;
        uv[i] = o.du;
    }
}

// Two sums over the CTA, each added in block_sum's fixed order (the same bits
// as two block_sum calls), behind one pair of barriers.
__device__ __forceinline__ float2 block_sum2(float a, float b, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, o));
        b = __fadd_rn(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red may still be read from the previous call
    if (lane == 0) {
        red[warp] = a;
        red[kThreads / 32 + warp] = b;
    }
    __syncthreads();
    float ta = 0.0f, tb = 0.0f;
#pragma unroll
    for (int k = 0; k < kThreads / 32; ++k) {
        ta = __fadd_rn(ta, red[k]);
        tb = __fadd_rn(tb, red[kThreads / 32 + k]);
    }
    return make_float2(ta, tb);
}

// ROWS rows per pass (1 or 2): with 2, a CTA takes rows r and r + gridDim.x
// together, issues both rows' loads before computing either, and finishes
// both dw values behind one pair of barriers, so twice the bytes are in flight
// per CTA and a row's barriers are shared.  Each row's sum keeps its order.
// MINB: CTAs per SM the registers are held to (0: no bound).
template <typename E, int VEC, int U, bool IN_PLACE, int LD, int ST, int ROWS = 1, int MINB = 0>
__global__ void __launch_bounds__(kThreads, MINB) swiglu_bwd_weighted_kernel(const BwdParams p) {
    await_previous_grid();
    allow_next_grid();
    static_assert(!IN_PLACE || (LD != kLdNC && LD != kLdNC256), "in place: coherent loads only");
    static_assert(ROWS == 1 || ROWS == 2, "one or two rows per pass");
    constexpr int B = E::kBytes * VEC;
    constexpr int NW = (B + 3) / 4;
    using L = Ld<B, LD>;
    using S = St<B, ST>;
    __shared__ float red[ROWS * kThreads / 32];
    for (int64_t r0 = blockIdx.x; r0 < p.rows; r0 += ROWS * (int64_t)gridDim.x) {
        // row h of the pass is r0 + h * gridDim.x; live[h]: it exists
        bool live[ROWS];
        const char *dyr[ROWS], *gr[ROWS], *ur[ROWS];
        char *dgr[ROWS], *dur[ROWS];
        float wr[ROWS], acc[ROWS];
#pragma unroll
        for (int h = 0; h < ROWS; ++h) {
            live[h] = r0 + h * (int64_t)gridDim.x < p.rows;
            const int64_t r = live[h] ? r0 + h * (int64_t)gridDim.x : r0;
            dyr[h] = static_cast<const char *>(p.dy) + r * p.dy_stride * B;
            gr[h] = static_cast<const char *>(p.g) + r * p.g_stride * B;
            ur[h] = static_cast<const char *>(p.u) + r * p.u_stride * B;
            dgr[h] = static_cast<char *>(p.dg) + r * p.dg_stride * B;
            dur[h] = static_cast<char *>(p.du) + r * p.du_stride * B;
            wr[h] = __ldg(p.w + r);
            acc[h] = 0.0f;
        }
        for (int32_t c0 = threadIdx.x; c0 < p.nvec; c0 += U * kThreads) {
            uint32_t d[ROWS][U][NW], g[ROWS][U][NW], u[ROWS][U][NW];
#pragma unroll
            for (int h = 0; h < ROWS; ++h) {
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const int32_t c = c0 + k * kThreads;
                    if (live[h] && c < p.nvec) {
                        L::run(dyr[h] + (int64_t)c * B, d[h][k]);
                        L::run(gr[h] + (int64_t)c * B, g[h][k]);
                        L::run(ur[h] + (int64_t)c * B, u[h][k]);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < ROWS; ++h) {
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const int32_t c = c0 + k * kThreads;
                    if (live[h] && c < p.nvec) {
                        uint32_t og[NW] = {}, ou[NW] = {};
                        float gv[VEC], uv[VEC];
                        if (pack_has_deep<E, VEC>(g[h][k]))
                            weighted_pack<E, VEC, true>(d[h][k], g[h][k], u[h][k], wr[h], acc[h], gv, uv);
                        else
                            weighted_pack<E, VEC, false>(d[h][k], g[h][k], u[h][k], wr[h], acc[h], gv, uv);
                        store_pack<E, VEC>(og, gv);
                        store_pack<E, VEC>(ou, uv);
                        S::run(dgr[h] + (int64_t)c * B, og);
                        S::run(dur[h] + (int64_t)c * B, ou);
                    }
                }
            }
        }
        if constexpr (ROWS == 2) {
            const float2 t = block_sum2(acc[0], acc[1], red);
            if (threadIdx.x == 0) {
                p.dw[r0] = t.x;
                if (live[1]) p.dw[r0 + gridDim.x] = t.y;
            }
        } else {
            const float t = block_sum(acc[0], red);
            if (threadIdx.x == 0) p.dw[r0] = t;
        }
    }
}

// Bias backward, first pass: CTA (tile, group) covers TILE_COLS columns of
// each half (kBiasTileCols unless the launch picks a narrower tile) for the
// rows of its row group (see below), writes dx and leaves the column sums of
// its rows, in fp32, in partial[group][0, 2n).
constexpr int kBiasTileCols = 2048;

// One pack of the bias backward: dgate / dup into gv / uv, added to the
// column sums ag / au, and (with weights) the dw terms added to rowsum.
template <typename E, int VEC, int MODE, bool kMayDeep>
__device__ __forceinline__ void bias_pack(const uint32_t *d, const uint32_t *g, const uint32_t *u,
                                          const uint32_t *bg, const uint32_t *bu, float wr,
                                          float *ag, float *au, float &rowsum, float *gv,
                                          float *uv) {
    static_assert(MODE & kBias, "the bias forms");
    if constexpr (kPairwise<E, VEC, MODE, kMayDeep>) {
        const uint64_t w2 = x2(wr, wr);
#pragma unroll
        for (int i = 0; i < VEC; i += 2) {
            // the biased gate and up, as bwd_pair forms them without a root window
            const uint64_t g2 = add_x2(x2(E::get(g, i), E::get(g, i + 1)), x2(E::get(bg, i), E::get(bg, i + 1)));
            const uint64_t u2 = add_x2(x2(E::get(u, i), E::get(u, i + 1)), x2(E::get(bu, i), E::get(bu, i + 1)));
            uint64_t dg2, du2;
            float a0 = 0.0f, a1 = 0.0f;
            bwd_pair_x2<MODE>(x2(E::get(d, i), E::get(d, i + 1)), g2, u2, w2, dg2, du2, a0, a1);
            if (MODE & kWeight) {
                rowsum = __fadd_rn(rowsum, a0);
                rowsum = __fadd_rn(rowsum, a1);
            }
            x2_split(add_x2(x2(ag[i], ag[i + 1]), dg2), ag[i], ag[i + 1]);
            x2_split(add_x2(x2(au[i], au[i + 1]), du2), au[i], au[i + 1]);
            x2_split(dg2, gv[i], gv[i + 1]);
            x2_split(du2, uv[i], uv[i + 1]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            const BwdPair<E, MODE> o = bwd_pair<E, MODE, kMayDeep>(
                E::get(d, i), E::get(g, i), E::get(u, i), E::get(bg, i), E::get(bu, i), wr);
            if (MODE & kWeight) rowsum = __fadd_rn(rowsum, o.dw_term);
            ag[i] = __fadd_rn(ag[i], o.dg);
            au[i] = __fadd_rn(au[i], o.du);
            gv[i] = o.dg;
            uv[i] = o.du;
        }
    }
}

// With WEIGHTED (per-token weights as well), each row's dw terms over the
// tile's columns are summed across the CTA into partial_dw[row, tile]: every
// thread parks its row sum in shared memory, and once per kDwBatch rows, after
// one barrier, each warp finishes rows of the batch: a lane adds the sums of
// threads lane, lane + 32, ... in order, then a shuffle tree adds the lanes.
// The row loop itself carries no cross-thread step.
//
// STAGES > 0 (16-byte packs; the ring also works with 4 and 8): instead of loading each row's packs into
// registers and waiting for them, every thread copies its own packs of the
// next STAGES - 1 rows into a private slice of a shared-memory ring with
// cp.async and reads each row back from there when it computes it.  Loads in
// flight then hold no registers, so more rows are in flight at the occupancy
// the registers allow; no barrier is needed, since a thread only ever reads
// the ring slots it filled itself (cp.async.wait_group orders them).  Ring:
// STAGES x 3 operands x PPT packs x kThreads threads x one pack of dynamic
// shared memory (swiglu_bias_ring_bytes); consecutive threads own consecutive
// slots, so the reads back are free of bank conflicts.
template <int VEC, int E_BYTES, int STAGES, int TILE_COLS = kBiasTileCols>
constexpr int swiglu_bias_ring_bytes() {
    return STAGES * 3 * (TILE_COLS / (kThreads * VEC)) * kThreads * E_BYTES * VEC;
}

// MINB: the CTAs per SM the register allocation is held to (launch bounds).
template <typename E, int VEC, bool IN_PLACE, int LD, int ST, bool WEIGHTED = false, int STAGES = 0,
          int DW_BATCH = 32, int TILE_COLS = kBiasTileCols, int MINB = 3>
__global__ void __launch_bounds__(kThreads, MINB) swiglu_bwd_bias_kernel(const BwdParams p, int32_t tiles,
                                                                         int64_t rows_per_group) {
    await_previous_grid();
    allow_next_grid();
    constexpr int MODE = WEIGHTED ? kBiasWeight : kBias;
    constexpr int kDwBatch = DW_BATCH;
    __shared__ float wpart[WEIGHTED ? kDwBatch : 1][WEIGHTED ? kThreads : 1];
    static_assert(!IN_PLACE || (LD != kLdNC && LD != kLdNC256), "in place: coherent loads only");
    constexpr int B = E::kBytes * VEC;
    constexpr int NW = (B + 3) / 4;
    constexpr int PPT = TILE_COLS / (kThreads * VEC);  // packs per thread per row and half
    static_assert(PPT >= 1 && PPT * kThreads * VEC == TILE_COLS, "tile / pack mismatch");
    static_assert(STAGES == 0 || ((B == 4 || B == 8 || B == 16) && STAGES >= 2),
                  "the cp.async ring moves 4-, 8- or 16-byte packs");
    // rows whose loads are issued together: keeps about as many bytes in flight
    // per thread as the streaming backward (the ring keeps STAGES - 1 rows in
    // flight instead)
    constexpr int RU = STAGES > 0 ? 1 : (PPT >= 2 ? 1 : 2);
    extern __shared__ __align__(16) unsigned char bias_ring[];
    using L = Ld<B, LD>;
    using S = St<B, ST>;
    const int32_t tile = blockIdx.x % tiles;
    // The bias form's row group g takes rows g, g + G, g + 2G, ... (G groups):
    // the CTAs of a column tile then walk one compact band of neighbouring
    // rows together instead of each streaming its own distant block (0.9-2.6 %
    // faster on the large-FFN, Llama-like and ffn-4096 shapes).  With weights
    // the contiguous blocks measured faster (the interleaved layout lost 3-6 %),
    // so that form keeps them.  Either way a group's column sums run over its
    // rows in order.
    constexpr bool kInterleave = !WEIGHTED;
    const int64_t group = blockIdx.x / tiles;
    const int64_t rs = kInterleave ? gridDim.x / tiles : 1;
    const int64_t r0 = kInterleave ? group : group * rows_per_group;
    const int64_t r1 = kInterleave ? p.rows : min(p.rows, r0 + rows_per_group);
    int32_t c[PPT];
    // the bias stays in its packed storage form (half the registers for bf16)
    // and is widened where it is used
    uint32_t bg[PPT][NW], bu[PPT][NW];
    float ag[PPT][VEC], au[PPT][VEC];
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        c[k] = tile * (TILE_COLS / VEC) + k * kThreads + threadIdx.x;
#pragma unroll
        for (int i = 0; i < NW; ++i) bg[k][i] = bu[k][i] = 0u;
        if (c[k] < p.nvec) {
            Ld<B, kLdCached>::run(static_cast<const char *>(p.bias_g) + (int64_t)c[k] * B, bg[k]);
            Ld<B, kLdCached>::run(static_cast<const char *>(p.bias_u) + (int64_t)c[k] * B, bu[k]);
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i) ag[k][i] = au[k][i] = 0.0f;
    }
    // Byte address of pack k of row r of an operand: one multiply-add per row
    // and operand (r * stride + c[0]), then a constant offset per k (c[k] =
    // c[0] + k * kThreads), which the loads and stores take as an immediate.
    const int64_t c0 = c[0];
    auto at = [&](const void *base, int64_t stride, int64_t r, int k) -> const char * {
        return static_cast<const char *>(base) + (r * stride + c0) * B + (int64_t)k * kThreads * B;
    };
    // ring slot of (stage, operand, pack) for this thread
    auto ring_at = [&](int st, int x, int k) -> unsigned char * {
        return bias_ring + ((size_t)((st * 3 + x) * PPT + k) * kThreads + threadIdx.x) * B;
    };
    // start the copies of row r's packs into ring stage st
    auto ring_fill = [&](int64_t r, int st) {
        if constexpr (STAGES > 0) {
#pragma unroll
            for (int k = 0; k < PPT; ++k) {
                if (c[k] < p.nvec) {
                    cp_async_pack<B>(ring_at(st, 0, k), at(p.dy, p.dy_stride, r, k));
                    cp_async_pack<B>(ring_at(st, 1, k), at(p.g, p.g_stride, r, k));
                    cp_async_pack<B>(ring_at(st, 2, k), at(p.u, p.u_stride, r, k));
                }
            }
        }
    };
    // the NW words of a ring slot
    auto ring_read = [&](const unsigned char *slot, uint32_t *w) {
        if constexpr (B == 16) {
            const uint4 q = *reinterpret_cast<const uint4 *>(slot);
            w[0] = q.x;
            w[1] = q.y;
            w[2] = q.z;
            w[3] = q.w;
        } else if constexpr (B == 8) {
            const uint2 q = *reinterpret_cast<const uint2 *>(slot);
            w[0] = q.x;
            w[1] = q.y;
        } else {
            w[0] = *reinterpret_cast<const uint32_t *>(slot);
        }
    };
    int stage = 0;  // ring stage of the current row
    if (STAGES > 0) {
#pragma unroll
        for (int st = 0; st < (STAGES > 0 ? STAGES - 1 : 0); ++st) {
            if (r0 + st * rs < r1) ring_fill(r0 + st * rs, st);
            cp_async_commit();
        }
    }
    int slot = 0;  // rows of the current dw batch held in wpart
    for (int64_t rb = r0; rb < r1; rb += RU * rs) {
        uint32_t d[RU][PPT][NW], g[RU][PPT][NW], u[RU][PPT][NW];
        if (STAGES > 0) {
            // refill the stage the previous row used, then wait for this row
            const int64_t ahead = rb + (STAGES > 0 ? STAGES - 1 : 0) * rs;
            if (ahead < r1) ring_fill(ahead, stage == 0 ? STAGES - 1 : stage - 1);
            cp_async_commit();
            cp_async_wait<(STAGES > 0 ? STAGES - 1 : 0)>();
#pragma unroll
            for (int k = 0; k < PPT; ++k) {
                if (c[k] < p.nvec) {
                    ring_read(ring_at(stage, 0, k), d[0][k]);
                    ring_read(ring_at(stage, 1, k), g[0][k]);
                    ring_read(ring_at(stage, 2, k), u[0][k]);
                }
            }
            stage = stage + 1 == STAGES ? 0 : stage + 1;
        } else {
#pragma unroll
            for (int q = 0; q < RU; ++q) {
                const int64_t r = rb + q * rs;
#pragma unroll
                for (int k = 0; k < PPT; ++k) {
                    if (r < r1 && c[k] < p.nvec) {
                        L::run(at(p.dy, p.dy_stride, r, k), d[q][k]);
                        L::run(at(p.g, p.g_stride, r, k), g[q][k]);
                        L::run(at(p.u, p.u_stride, r, k), u[q][k]);
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < RU; ++q) {
            const int64_t r = rb + q * rs;
            const float wr = (WEIGHTED && r < r1) ? __ldg(p.w + r) : 1.0f;
            float rowsum = 0.0f;
#pragma unroll
            for (int k = 0; k < PPT; ++k) {
                if (r < r1 && c[k] < p.nvec) {
                    uint32_t og[NW] = {}, ou[NW] = {};
                    float gv[VEC], uv[VEC];
                    if (pack_has_deep_biased<E, VEC>(g[q][k], bg[k]))
                        bias_pack<E, VEC, MODE, true>(d[q][k], g[q][k], u[q][k], bg[k], bu[k], wr,
                                                      ag[k], au[k], rowsum, gv, uv);
                    else
                        bias_pack<E, VEC, MODE, false>(d[q][k], g[q][k], u[q][k], bg[k], bu[k], wr,
                                                       ag[k], au[k], rowsum, gv, uv);
                    store_pack<E, VEC>(og, gv);
                    store_pack<E, VEC>(ou, uv);
                    S::run(const_cast<char *>(at(p.dg, p.dg_stride, r, k)), og);
                    S::run(const_cast<char *>(at(p.du, p.du_stride, r, k)), ou);
                }
            }
            if (WEIGHTED && r < r1) {  // r is the same for every thread of the CTA
                wpart[slot][threadIdx.x] = rowsum;
                if (slot == kDwBatch - 1 || r + rs >= r1) {  // a full batch, or the CTA's last row
                    __syncthreads();
                    const int lane = threadIdx.x & 31;
                    for (int q = threadIdx.x >> 5; q <= slot; q += kThreads / 32) {
                        float t = 0.0f;
#pragma unroll
                        for (int k = 0; k < kThreads / 32; ++k) t = __fadd_rn(t, wpart[q][lane + 32 * k]);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1)
                            t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, o));
                        if (lane == 0) p.partial_dw[(r - (slot - q) * rs) * tiles + tile] = t;
                    }
                    __syncthreads();  // wpart is refilled by the next batch
                    slot = -1;
                }
                ++slot;
            }
        }
    }
    if (STAGES > 0) cp_async_wait<0>();
    const int64_t n = (int64_t)p.nvec * VEC;
    // The column sums go out as whole vectors: a thread's VEC sums per half
    // are consecutive, and one scalar store per sum left each warp store
    // touching 32 separate sectors (ffn-4096 weights + bias backward: 0.789
    // -> 0.847 of the copy rate with the vector stores, bias 0.882 -> 0.899).
    // The workspace is 16-byte aligned (32-byte stores when it is 32-byte
    // aligned), and n is a multiple of VEC, so every vector below is aligned.
    float *part = p.partial + group * 2 * n;
    const bool part32 = (reinterpret_cast<uintptr_t>(p.partial) & 31) == 0;
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
        if (c[k] < p.nvec) {
            float *pg = part + (int64_t)c[k] * VEC, *pu = pg + n;
            if (VEC == 8 && part32) {
                uint32_t wg[8], wu[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    wg[i] = __float_as_uint(ag[k][i % VEC]);
                    wu[i] = __float_as_uint(au[k][i % VEC]);
                }
                St<32, kStPlain>::run(pg, wg);
                St<32, kStPlain>::run(pu, wu);
            } else if constexpr (VEC % 4 == 0) {
#pragma unroll
                for (int i = 0; i < VEC; i += 4) {
                    *reinterpret_cast<float4 *>(pg + i) = make_float4(ag[k][i], ag[k][i + 1], ag[k][i + 2], ag[k][i + 3]);
                    *reinterpret_cast<float4 *>(pu + i) = make_float4(au[k][i], au[k][i + 1], au[k][i + 2], au[k][i + 3]);
                }
            } else if constexpr (VEC == 2) {
                *reinterpret_cast<float2 *>(pg) = make_float2(ag[k][0], ag[k][1]);
                *reinterpret_cast<float2 *>(pu) = make_float2(au[k][0], au[k][1]);
            } else {
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    pg[i] = ag[k][i];
                    pu[i] = au[k][i];
                }
            }
        }
    }
}

// Bias backward, second pass.  dbias[k] = the sum over row groups of
// partial[group][k], rounded once to the storage type: a CTA takes
// kReduceCols consecutive columns (one per lane, so each group's row is one
// coalesced load per warp), its kReduceSegs warps sum contiguous segments of
// the groups in group order, and warp 0 adds the segment sums in segment
// order -- a fixed tree, so the result does not depend on timing, and the
// chain behind each value is about groups / kReduceSegs + kReduceSegs long
// instead of `groups`.  With dw (the weights + bias form), the CTAs after the
// column CTAs also form dw[r] = the sum over column tiles of partial_dw[r][tile],
// in tile order, so both reductions take one launch.
constexpr int kReduceCols = 32;
constexpr int kReduceSegs = 8;
constexpr int kReduceThreads = kReduceCols * kReduceSegs;

// Sum of the `count` floats at p, p + stride, ..., added in that order.  The
// loads go out sixteen at a time (the last batch only up to count) from one
// walking pointer, so a chain waits on one load latency per sixteen terms and
// holds no address per term: the ffn-4096 bias backward's 19-group segments
// took two load rounds instead of two plus three single loads (0.827 -> 0.853
// of the copy rate; the earlier form loaded eight at a time).
__device__ __forceinline__ float ordered_sum(const float *p, int64_t count, int64_t stride) {
    constexpr int kBatch = 16;
    float s = 0.0f;
    for (int64_t q = 0; q < count; q += kBatch) {
        const int live = count - q < kBatch ? (int)(count - q) : kBatch;
        float v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            v[i] = 0.0f;
            if (i < live) v[i] = *p;
            p += stride;
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
            if (i < live) s = __fadd_rn(s, v[i]);
    }
    return s;
}

template <typename E>
__global__ void __launch_bounds__(kReduceThreads)
    swiglu_bias_reduce_kernel(const float *partial, int64_t groups, int64_t two_n, void *dbias,
                              int64_t col_ctas, const float *partial_dw, int64_t rows, int32_t tiles,
                              float *dw) {
    await_previous_grid();
    allow_next_grid();
    if ((int64_t)blockIdx.x >= col_ctas) {  // dw rows (whole CTAs, so no barrier diverges)
        for (int64_t r = ((int64_t)blockIdx.x - col_ctas) * kReduceThreads + threadIdx.x; r < rows;
             r += ((int64_t)gridDim.x - col_ctas) * kReduceThreads)
            dw[r] = ordered_sum(partial_dw + r * tiles, tiles, 1);
        return;
    }
    __shared__ float seg[kReduceSegs][kReduceCols];
    const int lane = threadIdx.x % kReduceCols, warp = threadIdx.x / kReduceCols;
    const int64_t per = (groups + kReduceSegs - 1) / kReduceSegs;
    const int64_t g0 = warp * per;
    const int64_t cnt = g0 < groups ? (groups - g0 < per ? groups - g0 : per) : 0;
    for (int64_t c0 = (int64_t)blockIdx.x * kReduceCols; c0 < two_n; c0 += col_ctas * kReduceCols) {
        const int64_t k = c0 + lane;
        seg[warp][lane] = k < two_n ? ordered_sum(partial + g0 * two_n + k, cnt, two_n) : 0.0f;
        __syncthreads();
        if (warp == 0 && k < two_n) {
            float t = seg[0][lane];
#pragma unroll
            for (int w = 1; w < kReduceSegs; ++w) t = __fadd_rn(t, seg[w][lane]);
            uint32_t word[1] = {0};
            E::put(word, 0, t);
            if (E::kBytes == 4)
                static_cast<uint32_t *>(dbias)[k] = word[0];
            else
                static_cast<unsigned short *>(dbias)[k] = (unsigned short)word[0];
        }
        __syncthreads();
    }
}

}  // namespace swiglu
