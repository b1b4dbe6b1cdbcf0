// fc1_swiglu.cu -- linear_fc1 with the SwiGLU activation fused into its
// epilogue, on the sm_100-class tensor cores (tcgen05, TMEM, TMA, CTA pairs).
//
// Megatron's MLP computes fc1 = X W^T (W: [2n, K], rows [0, n) the gate
// projection, [n, 2n) the up projection) and then silu(fc1[:, :n]) *
// fc1[:, n:] (Liger-Kernel Megatron SwiGLU page, §Background).  Here a cluster
// of two CTAs owns a 256-row x 128-column tile of y.  Its tensor-core
// accumulator (one 128 x 256 fp32 block per CTA, in tensor memory) holds in
// columns [0, 128) the gate dot products for output columns j0 .. j0 + 127 and
// in columns [128, 256) the matching up dot products (W rows n + j0 ..), so the
// epilogue forms y from the fp32 accumulators directly and [M, 2n] never has
// to pass through HBM unless the caller asks for it (x_out, the buffer a
// training step saves).
//
// One CTA per SM, in pairs.  The grid holds one cluster per tile, but only as
// many pairs as fit the SMs start: each takes further tiles by cancelling the
// launch of clusters that have not started (cluster launch control), so a pair
// runs until no tile is left, and faster pairs take more tiles.  Roles (192
// threads per CTA): warp 0 lane 0 of each CTA TMA-loads that CTA's 128 rows
// of X and its half of the W slab (64 bf16 of K, 128-byte swizzle) into a
// 6-stage, 192 KiB ring (the leader's also schedules the tiles); warp 1
// of each CTA takes part in allocating all 512 TMEM columns (two
// accumulators), and lane 0 of the leader's warp 1 issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16, bf16 in, fp32
// accumulate) for both SMs, multicasting each stage's release and each
// finished accumulator to both CTAs; warps 2-5 of each CTA read their CTA's
// accumulator with tcgen05.ld (each warp its own 32-lane quarter), hand it
// back to the leader and store y while the tensor cores fill the other one.
//
// Every wait on an mbarrier gives up after kTimeoutNs of %globaltimer time,
// raises the sticky flag g_fc1_timeout and lets the pair drain and free its
// tensor memory, so a fault in the pipeline cannot hang the GPU.
#include <cuda.h>  // CUtensorMap and its encoding enums (the encoder is fetched at run time)
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "abi_internal.h"
#include "swiglu.h"
#include "swiglu_kernels.cuh"

namespace fc1 {

constexpr int BM = 128;           // rows of X per tile (MMA M)
constexpr int BN = 128;           // output columns per tile
constexpr int UMMA_N = 2 * BN;    // accumulator columns: gate then up
// K per stage: 64 bf16 = one 128-byte swizzle row.  (BK = 32 with the
// 64-byte swizzle and twice the stages measured 25 % slower on GB300.)
constexpr int BK = 64;
constexpr int SWZ_BYTES = BK * 2;             // bytes per swizzled row
constexpr int UMMA_K = 16;                    // K per tcgen05.mma of kind::f16
constexpr int A_BYTES = BM * BK * 2;          // this CTA's 128 rows of X
static_assert(SWZ_BYTES == 64 || SWZ_BYTES == 128, "64- or 128-byte swizzle");
constexpr int TMEM_COLS = 2 * UMMA_N;  // two accumulators
constexpr int kThreads = 192;
constexpr int kBarrierBytes = 256;
constexpr int RING_BYTES = 192 * 1024;
constexpr int SMEM_BYTES = RING_BYTES + kBarrierBytes + 1024;  // ring + barriers + alignment slack
constexpr unsigned long long kTimeoutNs = 2000000000ull;                  // 2 s

__device__ int g_fc1_timeout = 0;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// kCluster: acquire at cluster scope, for data another CTA of the cluster
// wrote before its release arrive on this barrier.
template <bool kCluster>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    if (kCluster)
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n"
            "}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n"
            "}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity; false (and the timeout
// flag raised) if it does not complete within kTimeoutNs.
template <bool kCluster = false>
__device__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    while (!mbar_try_wait<kCluster>(bar, parity)) {
        if (now_ns() - t0 > kTimeoutNs) {
            atomicExch(&g_fc1_timeout, 1);
            return false;
        }
    }
    return true;
}

// Shared-memory matrix descriptor of a K-major operand laid out by TMA with
// the SWZ_BYTES swizzle: rows of SWZ_BYTES bytes, 8-row groups 8 * SWZ_BYTES
// apart (stride byte offset), descriptor version 1 (bits 46-47), layout type
// in bits 61-63 (2 = 128-byte swizzle, 4 = 64-byte swizzle).  The leading
// byte offset is unused in the swizzled K-major layouts.
__device__ __forceinline__ uint64_t smem_desc_swizzled(uint32_t saddr) {
    constexpr uint64_t layout = SWZ_BYTES == 128 ? 2 : 4;
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;
    d |= (uint64_t)((8u * SWZ_BYTES) >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= layout << 61;
    return d;
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 accumulator columns of this warp's 32 TMEM lanes (one
// lane = one row per thread).
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),
          "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),
          "=r"(v[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// outputs are written once and not reread here: evict-first, so they do not
// push the reused X and W tiles out of L2
__device__ __forceinline__ void store16(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}
// 32 bytes (sm_100-class 256-bit store): a whole sector
__device__ __forceinline__ void store32(void *p, const uint32_t *w) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// The 16 words of 32 output columns of one row, from column `col` on (n % 8
// == 0, so a 16-byte piece is all inside or all outside the row): as two
// 32-byte stores when `wide` (rows and base 32-byte aligned), else four.
__device__ __forceinline__ void store_row_chunk(__nv_bfloat16 *p, const uint32_t (&w)[16], int col, int n,
                                                bool wide) {
    if (wide) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (col + 16 * q < n) store32(p + 16 * q, w + 8 * q);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (col + 8 * q < n) store16(p + 8 * q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
}

// Two fp32 lanes per instruction: swiglu::x2 and friends (.f32x2 arithmetic,
// each lane rounded as the scalar operation rounds).
using swiglu::add_x2;
using swiglu::mul_x2;
using swiglu::x2;
using swiglu::x2_split;

// y for 32 accumulator columns of one row: silu(g) * u from the fp32 gate and
// up dot products, rounded once to bf16, in pairs.  kMayDeep = false when no
// gate of the chunk is below -64: then each pair takes the streaming kernels'
// branch-free form, s = 1 / (1 + 2^(-g log2 e)), silu = g s, y = silu u, with
// the multiplications and the addition done on both lanes at once (the same
// operations and roundings per element, so the same bits).  The epilogue
// shares its SM with the tensor pipe, and the fewer FP32 instructions it
// issues the fewer cycles the pipe loses to it.
template <bool kMayDeep>
__device__ __forceinline__ void activate_chunk(const uint32_t (&gv)[32], const uint32_t (&uv)[32],
                                               uint32_t (&out)[16]) {
    if constexpr (!kMayDeep) {
        const uint64_t neg_log2e = x2(-swiglu::kLog2e, -swiglu::kLog2e), one = x2(1.0f, 1.0f);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const uint64_t g2 = x2(__uint_as_float(gv[i]), __uint_as_float(gv[i + 1]));
            const uint64_t u2 = x2(__uint_as_float(uv[i]), __uint_as_float(uv[i + 1]));
            float t0, t1, d0, d1, r0, r1;
            x2_split(mul_x2(g2, neg_log2e), t0, t1);
            x2_split(add_x2(one, x2(swiglu::ex2_approx(t0), swiglu::ex2_approx(t1))), d0, d1);
            const uint64_t s2 = x2(swiglu::rcp_approx(d0), swiglu::rcp_approx(d1));
            x2_split(mul_x2(mul_x2(g2, s2), u2), r0, r1);
            swiglu::BF16::put2(out, i, r0, r1);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            float r2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float g = __uint_as_float(gv[i + h]);
                const float u = __uint_as_float(uv[i + h]);
                const swiglu::Act act = swiglu::activation<swiglu::BF16, false, true>(g);
                r2[h] = __fmul_rn(__fmul_rn(act.silu, u), act.scale);
            }
            swiglu::BF16::put2(out, i, r2[0], r2[1]);
        }
    }
}

// Tile order: groups of kGroupM row tiles; within a group the row tile varies
// fastest.  A wave of co-resident CTA pairs then covers about kGroupM row tiles
// x (pairs / kGroupM) column tiles, so its X rows stay in L2 across the whole
// group and each W tile is fetched from HBM once per group instead of once per
// wave (waves spanning every row tile read 10x the input bytes from HBM).
constexpr int kGroupM = 16;

// ------------------------------------------------------ the CTA-pair kernel ---
// A cluster of two CTAs computes a 256-row tile with
// tcgen05.mma.cta_group::2: each CTA loads its own 128 rows of X and one half
// of the W slab (the leader the 128 gate rows, the peer the 128 up rows), the
// leader's single MMA thread drives both SMs' tensor cores, and each CTA's
// tensor memory receives the accumulator of its own 128 rows (gate columns
// [0, 128), up columns [128, 256)).  A CTA's stage is 32 KiB, so six stages
// fit a 192 KiB ring.  With one CTA per 128 x 256 tile the stage was 48 KiB,
// four stages hid too little latency and the tensor pipe idled a quarter of
// the time (1.05 ms against 0.99 ms for the Llama-3-8B fc1 shape).
constexpr int PAIR_M = 2 * BM;
constexpr int B2_BYTES = BN * BK * 2;                 // this CTA's half of the W slab
constexpr int STAGE2_BYTES = A_BYTES + B2_BYTES;      // 32 KiB
constexpr int STAGES2 = RING_BYTES / STAGE2_BYTES;     // 6
static_assert(STAGES2 * STAGE2_BYTES == RING_BYTES, "the ring fills its bytes");
// Tile scheduling by cluster launch control: the grid has one cluster per
// tile; a running pair takes further tiles by cancelling the launch of
// clusters that have not started, so pairs that run faster take more tiles
// and all finish within about one tile of each other.  The leader's producer
// thread publishes each tile id in a ring of kTileSlots slots in both CTAs,
// read by the peer's producer, the MMA thread and the eight epilogue warps.
constexpr int kTileSlots = 4;
constexpr int kTileReaders = 1 + 1 + 2 * 4;  // peer producer, MMA thread, epilogue warps
// the next tile is asked for this many K blocks before the current one's last load
constexpr int kAskAhead = 16;
// byte offsets in the region after the ring
constexpr int OFF_FULL = 0;                                   // full[STAGES2]
constexpr int OFF_EMPTY = OFF_FULL + 8 * STAGES2;             // empty[STAGES2]
constexpr int OFF_ACC_FULL = OFF_EMPTY + 8 * STAGES2;         // acc_full[2]
constexpr int OFF_ACC_EMPTY = OFF_ACC_FULL + 16;              // acc_empty[2]
constexpr int OFF_MMA_DONE = OFF_ACC_EMPTY + 16;              // mma_done
constexpr int OFF_TILE_FULL = OFF_MMA_DONE + 8;               // tile_full[kTileSlots]
constexpr int OFF_TILE_EMPTY = OFF_TILE_FULL + 8 * kTileSlots;  // tile_empty[kTileSlots]
constexpr int OFF_CLC_BAR = OFF_TILE_EMPTY + 8 * kTileSlots;  // the cancel answer's barrier
constexpr int OFF_CLC_RESP = (OFF_CLC_BAR + 8 + 15) / 16 * 16;  // the 16-byte answer
constexpr int OFF_TILE_ID = OFF_CLC_RESP + 16;                // tile_id[kTileSlots]
constexpr int OFF_TMEM = OFF_TILE_ID + 4 * kTileSlots;        // the TMEM base address
constexpr int OFF_ABORT = OFF_TMEM + 4;                       // the abort flag
static_assert(OFF_ABORT + 4 <= kBarrierBytes, "barriers and state fit their region");
// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 =
// 0), N / 8 in bits 17-22, M / 16 in bits 24-28 (M = 256 across the pair).
constexpr uint32_t kInstrDesc2 = (1u << 4) | (1u << 7) | (1u << 10) |
                                 ((uint32_t)(UMMA_N >> 3) << 17) | ((uint32_t)(PAIR_M >> 4) << 24);

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of this CTA's shared variable `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA (the leader's).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
        : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(kInstrDesc2), "r"(acc)
        : "memory");
}

// Arrive on the mbarrier at this offset in both CTAs once the pair MMAs issued
// so far are done.
__device__ __forceinline__ void mma_commit_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
}

__device__ __forceinline__ void mma_commit_local_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
                 : "memory");
}

// Cluster launch control: ask to cancel the launch of a cluster of this grid
// that has not started; the 16-byte answer is written at `resp` (this CTA's
// shared memory) and completes 16 bytes of transaction on `bar`.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
            resp),
        "r"(bar)
        : "memory");
}

// The x index of the first CTA of the cluster whose launch was cancelled, or
// -1 when the request failed (no cluster was left to take).
__device__ __forceinline__ int clc_cancelled_cta(uint32_t resp) {
    uint32_t ok, x = 0;
    asm volatile(
        "{\n"
        ".reg .b128 r;\n"
        ".reg .pred p;\n"
        "ld.shared.b128 r, [%2];\n"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n"
        "}\n"
        : "=r"(ok), "=r"(x)
        : "r"(resp)
        : "memory");
    return ok ? (int)x : -1;
}

// Write a tile id (-1: none left) into slot `slot` of both CTAs' tile rings
// and release it with an arrive on each CTA's tile_full barrier.
__device__ __forceinline__ void publish_tile(uint32_t ids, uint32_t tile_full0, int slot, int tile) {
#pragma unroll
    for (uint32_t r = 0; r < 2; ++r) {
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(map_to_rank(ids + 4 * slot, r)), "r"(tile)
                     : "memory");
        mbar_arrive_cluster(map_to_rank(tile_full0 + 8 * slot, r));
    }
}

__device__ __forceinline__ void pair_tile_coords(int t, int tiles_m2, int tiles_n, int &m0, int &j0) {
    const int per_group = kGroupM * tiles_n;
    const int g = t / per_group;
    const int first = g * kGroupM;
    const int gm = min(kGroupM, tiles_m2 - first);
    const int local = t - g * per_group;
    m0 = (first + local % gm) * PAIR_M;
    j0 = (local / gm) * BN;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fc1_swiglu_pair_kernel(const __grid_constant__ CUtensorMap tm_x,
                           const __grid_constant__ CUtensorMap tm_wg,
                           const __grid_constant__ CUtensorMap tm_wu, __nv_bfloat16 *__restrict__ y,
                           __nv_bfloat16 *__restrict__ x_out, int M, int n, int K) {
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sa = smem_addr(smem);
    const uint32_t sb = sa + STAGES2 * A_BYTES;
    unsigned char *state = smem + RING_BYTES;
    const uint32_t st0 = smem_addr(state);
    const uint32_t full0 = st0 + OFF_FULL, empty0 = st0 + OFF_EMPTY;
    const uint32_t acc_full0 = st0 + OFF_ACC_FULL, acc_empty0 = st0 + OFF_ACC_EMPTY;
    const uint32_t mma_done = st0 + OFF_MMA_DONE;
    const uint32_t tile_full0 = st0 + OFF_TILE_FULL, tile_empty0 = st0 + OFF_TILE_EMPTY;
    const uint32_t clc_bar = st0 + OFF_CLC_BAR, clc_resp = st0 + OFF_CLC_RESP;
    const uint32_t tile_ids_addr = st0 + OFF_TILE_ID;
    volatile int *tile_ids = reinterpret_cast<volatile int *>(state + OFF_TILE_ID);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(state + OFF_TMEM);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(state + OFF_ABORT);

    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kblocks = (K + BK - 1) / BK;
    const int tiles_m2 = (M + PAIR_M - 1) / PAIR_M;
    const int tiles_n = (n + BN - 1) / BN;  // the last column tile may be ragged
    const int tiles = tiles_m2 * tiles_n;
    const uint32_t tile_empty_leader0 = map_to_rank(tile_empty0, 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES2; ++s) {
            mbar_init(full0 + 8 * s, 1);   // the leader's producer (plus both CTAs' bytes)
            mbar_init(empty0 + 8 * s, 1);  // the leader's commit, multicast to both CTAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full0 + 8 * a, 1);   // the leader's commit, multicast
            mbar_init(acc_empty0 + 8 * a, 8);  // the epilogue warps of both CTAs (leader's copy)
        }
        mbar_init(mma_done, 1);
        for (int i = 0; i < kTileSlots; ++i) {
            mbar_init(tile_full0 + 8 * i, 1);              // the leader's producer
            mbar_init(tile_empty0 + 8 * i, kTileReaders);  // leader's copy only
        }
        mbar_init(clc_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_wg)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_wu)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched early (programmatic dependent launch): the setup above ran
    // beside the previous grid's last CTAs; from here on every role may touch
    // global memory, so wait until that grid has completed and its writes are
    // visible.  The next grid may launch now: its CTAs take SMs as this
    // grid's pairs leave.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0 && lane == 0) {
        // ---- producer (both CTAs): this CTA's X rows and its half of the W
        // slab for each tile.  The leader's producer also schedules: it
        // publishes each tile id in both CTAs' tile rings (its own tile
        // first) and asks for the next by cancelling a pending cluster.
        // the gate and up halves of W have tensor maps of their own, each n
        // rows long, so a ragged last column tile reads zeros past row n
        // instead of rows of the other half
        const CUtensorMap *wmap = leader ? &tm_wg : &tm_wu;
        int it = 0, asks = 0;
        int tile = (int)(blockIdx.x >> 1);
        for (int k = 0;; ++k) {
            const int slot = k % kTileSlots;
            if (leader) {
                if (!mbar_wait<true>(tile_empty0 + 8 * slot, ((k / kTileSlots) & 1) ^ 1)) {
                    *abort_flag = 1;
                    tile = -1;
                }
                publish_tile(tile_ids_addr, tile_full0, slot, tile);
            } else {
                tile = mbar_wait<true>(tile_full0 + 8 * slot, (k / kTileSlots) & 1) ? tile_ids[slot] : -1;
                mbar_arrive_cluster(tile_empty_leader0 + 8 * slot);
            }
            if (tile < 0) break;
            int m0, j0;
            pair_tile_coords(tile, tiles_m2, tiles_n, m0, j0);
            const int my_m0 = m0 + BM * (int)rank;
            const int ask_at = kblocks > kAskAhead ? kblocks - kAskAhead : 0;
            bool asked = false;
            for (int kb = 0; kb < kblocks && !*abort_flag; ++kb, ++it) {
                if (leader && kb == ask_at) {
                    mbar_arrive_expect_tx(clc_bar, 16);
                    clc_try_cancel(clc_resp, clc_bar);
                    asked = true;
                }
                const int s = it % STAGES2;
                if (!mbar_wait(empty0 + 8 * s, ((it / STAGES2) & 1) ^ 1)) {
                    *abort_flag = 1;
                    break;
                }
                const uint32_t full_leader = map_to_rank(full0 + 8 * s, 0);
                if (leader) mbar_arrive_expect_tx(full0 + 8 * s, 2 * STAGE2_BYTES);
                tma_load_2d_pair(sa + s * A_BYTES, &tm_x, full_leader, kb * BK, my_m0);
                tma_load_2d_pair(sb + s * B2_BYTES, wmap, full_leader, kb * BK, j0);
            }
            if (leader) {
                // the answer is waited for even after an abort, so it never
                // lands in shared memory the CTA has left
                int next = -1;
                if (asked && mbar_wait<true>(clc_bar, asks++ & 1)) {
                    const int x = clc_cancelled_cta(clc_resp);
                    if (x >= 0) {
                        next = x >> 1;
                        if ((x & 1) != 0 || next >= tiles) {  // not a cluster's first CTA of this grid
                            *abort_flag = 1;
                            atomicExch(&g_fc1_timeout, 1);
                            next = -1;
                        }
                    }
                }
                tile = *abort_flag ? -1 : next;
            }
        }
        // the leader's full barriers count both CTAs' bytes: once their last
        // phases complete, every load of the pair has landed
        if (leader)
            for (int k = it > STAGES2 ? it - STAGES2 : 0; k < it; ++k)
                mbar_wait(full0 + 8 * (k % STAGES2), (k / STAGES2) & 1);
    } else if (warp == 1 && lane == 0 && leader) {
        // ---- MMA issuer (leader only): drives the tensor cores of both SMs
        int it = 0, lt = 0;
        for (int k = 0;; ++k, ++lt) {
            const int slot = k % kTileSlots;
            const int tile = mbar_wait<true>(tile_full0 + 8 * slot, (k / kTileSlots) & 1) ? tile_ids[slot] : -1;
            mbar_arrive_cluster(tile_empty_leader0 + 8 * slot);
            if (tile < 0 || *abort_flag) break;
            const int acc = lt & 1;
            if (!mbar_wait(acc_empty0 + 8 * acc, ((lt >> 1) & 1) ^ 1)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * UMMA_N);
            bool ok = true;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES2;
                if (!mbar_wait(full0 + 8 * s, (it / STAGES2) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                    const uint64_t a = smem_desc_swizzled(sa + s * A_BYTES + kk * UMMA_K * 2);
                    const uint64_t b = smem_desc_swizzled(sb + s * B2_BYTES + kk * UMMA_K * 2);
                    mma_bf16_pair(d, a, b, (kb | kk) != 0 ? 1u : 0u);
                }
                mma_commit_both(empty0 + 8 * s);
            }
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            mma_commit_both(acc_full0 + 8 * acc);
        }
        mma_commit_local_pair(mma_done);
        mbar_wait(mma_done, 0);
    } else if (warp >= 2) {
        // ---- epilogue (both CTAs): this CTA's 128 rows of the accumulator
        const int quarter = warp & 3;
        const uint32_t acc_empty_leader0 = map_to_rank(acc_empty0, 0);
        // 32-byte stores when every output row starts on a 32-byte boundary
        const bool wide = n % 16 == 0 && reinterpret_cast<uintptr_t>(y) % 32 == 0 &&
                          reinterpret_cast<uintptr_t>(x_out) % 32 == 0;
        int lt = 0;
        // the warp leaves the loop as one (its body has warp-wide .sync.aligned
        // instructions), so the tile id, the abort flag and the waits' outcome
        // are warp-uniform
        for (int k = 0;; ++k, ++lt) {
            const int slot = k % kTileSlots;
            int tile = -1;
            if (lane == 0) {
                if (mbar_wait<true>(tile_full0 + 8 * slot, (k / kTileSlots) & 1)) tile = tile_ids[slot];
                mbar_arrive_cluster(tile_empty_leader0 + 8 * slot);
            }
            tile = __shfl_sync(0xffffffffu, tile, 0);
            if (tile < 0 || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            const int acc = lt & 1;
            int m0, j0;
            pair_tile_coords(tile, tiles_m2, tiles_n, m0, j0);
            const int row = m0 + BM * (int)rank + 32 * quarter + lane;
            if (!__all_sync(0xffffffffu, mbar_wait(acc_full0 + 8 * acc, (lt >> 1) & 1))) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(acc * UMMA_N);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t gv[32], uv[32];
                tmem_load32(tbase + c, gv);
                tmem_load32(tbase + BN + c, uv);
                tmem_wait_ld();
                if (c + 32 == BN) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(acc_empty_leader0 + 8 * acc);
                }
                if (row < M) {
                    uint32_t out[16];
                    // gates below -64 need the scaled deep-tail form; a chunk
                    // without any takes the branch-free form (the same bits
                    // per element) with a much shorter instruction stream
                    float gmin = __uint_as_float(gv[0]);
#pragma unroll
                    for (int i = 1; i < 32; ++i) gmin = fminf(gmin, __uint_as_float(gv[i]));
                    if (!(gmin < -64.0f))
                        activate_chunk<false>(gv, uv, out);
                    else
                        activate_chunk<true>(gv, uv, out);
                    store_row_chunk(y + (int64_t)row * n + j0 + c, out, j0 + c, n, wide);
                    if (x_out != nullptr) {
                        uint32_t pg[16], pu[16];
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            swiglu::BF16::put2(pg, i, __uint_as_float(gv[i]), __uint_as_float(gv[i + 1]));
                            swiglu::BF16::put2(pu, i, __uint_as_float(uv[i]), __uint_as_float(uv[i + 1]));
                        }
                        __nv_bfloat16 *xg = x_out + (int64_t)row * 2 * n + j0 + c;
                        store_row_chunk(xg, pg, j0 + c, n, wide);
                        store_row_chunk(xg + n, pu, j0 + c, n, wide);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the other may still signal it
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::atomic<EncodeTiled> g_encode{nullptr};

swiglu_status_t fail(cudaError_t e) {
    swiglu_abi::record_cuda_error((int)e);
    return SWIGLU_ERR_CUDA;
}

cudaError_t encoder(EncodeTiled &fn) {
    fn = g_encode.load();
    if (fn != nullptr) return cudaSuccess;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || p == nullptr) return cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiled>(p);
    g_encode.store(fn);
    return cudaSuccess;
}

// [rows, K] bf16, row-major: a box of BK K-elements (SWZ_BYTES bytes) by 128
// rows with the matching swizzle, zero fill outside the tensor.
bool make_map(EncodeTiled enc, CUtensorMap *map, const void *base, int64_t rows, int64_t K) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, 128};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               SWZ_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace fc1

extern "C" {

swiglu_status_t swiglu_fc1_fwd(const void *x_in, const void *w, void *y, void *x_out, int64_t M,
                               int64_t n, int64_t K, swiglu_dtype_t dtype, swiglu_stream_t stream) {
    using namespace fc1;
    if (dtype != SWIGLU_BF16) return SWIGLU_ERR_DTYPE;
    if (M < 0 || n < 0 || K < 0) return SWIGLU_ERR_SHAPE;
    if (M == 0 || n == 0) return SWIGLU_OK;
    if (K == 0 || n % 8 != 0 || K % 8 != 0 || M > INT32_MAX || K > INT32_MAX || 2 * n > INT32_MAX)
        return SWIGLU_ERR_SHAPE;
    if (x_in == nullptr || w == nullptr || y == nullptr) return SWIGLU_ERR_NULL;
    if (((uintptr_t)x_in | (uintptr_t)w | (uintptr_t)y | (uintptr_t)x_out) % 16 != 0)
        return SWIGLU_ERR_STRIDE;
    const size_t bx = (size_t)M * K * 2, bw = (size_t)2 * n * K * 2, by = (size_t)M * n * 2,
                 bo = (size_t)M * 2 * n * 2;
    if (overlap(y, by, x_in, bx) || overlap(y, by, w, bw)) return SWIGLU_ERR_ALIAS;
    if (x_out != nullptr && (overlap(x_out, bo, x_in, bx) || overlap(x_out, bo, w, bw) ||
                             overlap(x_out, bo, y, by)))
        return SWIGLU_ERR_ALIAS;

    EncodeTiled enc;
    cudaError_t e = encoder(enc);
    if (e != cudaSuccess) return fail(e);
    CUtensorMap tm_x, tm_wg, tm_wu;
    const char *w_up = static_cast<const char *>(w) + (size_t)n * K * 2;
    if (!make_map(enc, &tm_x, x_in, M, K) || !make_map(enc, &tm_wg, w, n, K) ||
        !make_map(enc, &tm_wu, w_up, n, K))
        return fail(cudaErrorInvalidValue);
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(e);
    // the shared-memory opt-in is a per-device function attribute
    constexpr int kMaxDevices = 64;
    static std::atomic<bool> attr_set[kMaxDevices];
    const bool cached = dev >= 0 && dev < kMaxDevices && attr_set[dev].load();
    if (!cached) {
        e = cudaFuncSetAttribute(fc1_swiglu_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES);
        if (e != cudaSuccess) return fail(e);
        if (dev >= 0 && dev < kMaxDevices) attr_set[dev].store(true);
    }
    const int64_t tiles = ((M + PAIR_M - 1) / PAIR_M) * ((n + BN - 1) / BN);  // 256 x 128 tiles
    if (tiles > INT32_MAX / 2) return SWIGLU_ERR_SHAPE;
    // one cluster per tile; the pairs that start take the others' tiles
    // (cluster launch control), so only as many run as fit on the SMs
    const dim3 grid((unsigned)(2 * tiles));
    // programmatic stream serialization: the grid may launch while the
    // previous kernel in the stream finishes (the kernel waits for it before
    // its first global memory access)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, fc1_swiglu_pair_kernel, tm_x, tm_wg, tm_wu, static_cast<__nv_bfloat16 *>(y),
                           static_cast<__nv_bfloat16 *>(x_out), (int)M, (int)n, (int)K);
    return e == cudaSuccess ? SWIGLU_OK : fail(e);
}

swiglu_status_t swiglu_fc1_timeout_flag(int *flag) {
    if (flag == nullptr) return SWIGLU_ERR_NULL;
    cudaError_t e = cudaMemcpyFromSymbol(flag, fc1::g_fc1_timeout, sizeof(int));
    return e == cudaSuccess ? SWIGLU_OK : fc1::fail(e);
}

}  // extern "C"
