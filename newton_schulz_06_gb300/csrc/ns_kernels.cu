// Tensor-core stages of one Newton-Schulz iteration on sm_103a:
//
//   OP_SYRK_X   A  = X X^T                (symmetric rank-k update, K = n)
//   OP_SYRK_A   B  = b A + c A A^T         (A symmetric, so A A^T = A A;
//                                           the b A + c (.) combination is
//                                           fused into the epilogue, K = m)
//   OP_GEMM_BX  X' = a X + B X            (axpy fused into the epilogue)
//
// "Advancing Emerging Optimizers for Accelerated LLM Training", section
// "SYRK and fused all-reduce": the first two of the three products of an
// iteration are symmetric rank-k updates; only upper-triangle tiles are
// computed (tiles on the diagonal in full) and the full matrix is written,
// not a packed triangle.  Here the lower triangle is written by mirroring
// each computed element, so A and B are exactly symmetric.
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: 128B-swizzled {64 x 64} boxes into a 4-stage
//               shared-memory ring, completion tracked by mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32
//               accumulators) and issues tcgen05.mma (bf16 x bf16 -> fp32)
//               from one thread; tcgen05.commit releases ring slots and
//               hands finished accumulators to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld rows of the accumulator, apply the
//               stage's combination, store bf16 (and the mirrored element).
// The two accumulators let the epilogue of one tile overlap the main loop
// of the next.  Tiles come from a cost-sorted list (largest K first) and CTA
// i takes tiles i, i+grid, ...; every output tile is produced by exactly one
// CTA in a fixed K order, so results do not depend on grouping.
//
// Every wait is bounded: after `wait_limit_ns` a waiting thread records
// DEV_ERR_TIMEOUT in the device error word, raises a CTA-wide abort flag and
// all roles leave their loops; the CTA then waits (bounded) for its own TMA
// copies and MMAs in flight, frees its TMEM and exits.
#include "muon_internal.h"

namespace muon {
namespace {

constexpr int A_STAGE_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_STAGE_BYTES = BN * BK * 2;        // 32 KB
constexpr int BOX_BYTES = 64 * 64 * 2;            // one {64,64} TMA box
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
constexpr int SMEM_BYTES = STAGES * (A_STAGE_BYTES + B_STAGE_BYTES) + 1024 +
                           256;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar),
                 "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase of parity `parity` to complete.  Returns false
// if the CTA aborted (or this wait timed out and raised the abort).
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag, int* err,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicCAS(err, 0, DEV_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap,
                                            uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx"
        "::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2),
// descriptor version 1, base offset 0.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo,
                                              uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), M = 128, N = n.
__device__ __forceinline__ uint32_t instr_desc(int n, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) |
           (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc,
                                         uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster."
        "b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
          "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
          "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
}

__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p,
                                           float (&v)[8]) {
    uint4 q = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float2 f = __bfloat1622float2(h[e]);
        v[2 * e] = f.x;
        v[2 * e + 1] = f.y;
    }
}

__device__ __forceinline__ void store8_bf16(__nv_bfloat16* p,
                                            const float (&v)[8]) {
    uint4 q;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
    for (int e = 0; e < 4; ++e)
        h[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
    *reinterpret_cast<uint4*>(p) = q;
}

template <int OP>
__device__ __forceinline__ int k_extent(const NsUnit& U) {
    return OP == OP_SYRK_X ? U.n : U.m;
}

// ---------------------------------------------------------------------------
// Epilogue of one 32-column chunk for the row `gi` owned by this thread.
//   SYRK stages: element (gi, gc) is stored if gc >= gi and mirrored to
//   (gc, gi) if gc > gi; elements below the diagonal (only inside diagonal
//   blocks) are dropped, so each element of the m x m result is written once.
template <int OP>
__device__ __forceinline__ void epilogue_chunk(const NsUnit& U, int src,
                                               float alpha_a, float coef_b,
                                               float coef_c, int gi, int gc0,
                                               float (&v)[32]) {
    if (OP == OP_GEMM_BX) {
        const int n = U.n;
        if (gi >= U.m || gc0 >= n) return;
        const __nv_bfloat16* xin = U.x[src] + static_cast<int64_t>(gi) * U.ld_x;
        __nv_bfloat16* xout = U.x[src ^ 1] + static_cast<int64_t>(gi) * U.ld_x;
        if (gc0 + 32 <= n) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float xv[8], o[8];
                load8_bf16(xin + gc0 + 8 * q, xv);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    o[e] = fmaf(alpha_a, xv[e], v[8 * q + e]);
                store8_bf16(xout + gc0 + 8 * q, o);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int gc = gc0 + e;
                if (gc < n) {
                    const float xv = __bfloat162float(xin[gc]);
                    xout[gc] = __float2bfloat16_rn(fmaf(alpha_a, xv, v[e]));
                }
            }
        }
        return;
    }
    const int m = U.m;
    if (gi >= m || gc0 >= m) return;
    if (gc0 + 31 < gi) return;                       // wholly below diagonal
    __nv_bfloat16* out = (OP == OP_SYRK_X) ? U.a : U.b;
    const int64_t ld = U.ld_mm;
    if (OP == OP_SYRK_A) {
        const __nv_bfloat16* ain = U.a + static_cast<int64_t>(gi) * ld;
        if (gc0 + 32 <= m) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float av[8];
                load8_bf16(ain + gc0 + 8 * q, av);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[8 * q + e] = fmaf(coef_b, av[e], coef_c * v[8 * q + e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int gc = gc0 + e;
                const float av = gc < m ? __bfloat162float(ain[gc]) : 0.f;
                v[e] = fmaf(coef_b, av, coef_c * v[e]);
            }
        }
    }
    __nv_bfloat16* row = out + static_cast<int64_t>(gi) * ld;
    if (gc0 > gi && gc0 + 32 <= m) {
        // strictly above the diagonal: vector row store + mirrored column
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = v[8 * q + e];
            store8_bf16(row + gc0 + 8 * q, o);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e)
            out[static_cast<int64_t>(gc0 + e) * ld + gi] =
                __float2bfloat16_rn(v[e]);
    } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int gc = gc0 + e;
            if (gc < m && gc >= gi) {
                const __nv_bfloat16 h = __float2bfloat16_rn(v[e]);
                row[gc] = h;
                if (gc > gi) out[static_cast<int64_t>(gc) * ld + gi] = h;
            }
        }
    }
}

template <int OP>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ns_kernel(const __grid_constant__ NsLaunch p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_STAGE_BYTES);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + STAGES;
    uint64_t* tfull_bar = bars + 2 * STAGES;
    uint64_t* tempty_bar = bars + 2 * STAGES + 2;
    uint64_t* drain_bar = bars + 2 * STAGES + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), 4);
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], "
            "%1;" ::"r"(smem_u32(tmem_slot)),
            "r"(TMEM_COLS)
            : "memory");
        asm volatile(
            "tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_dependency_wait();
    allow_dependent_launch();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t limit = p.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            // phase (+1) of the last load issued into each slot, for drain
            int issued[STAGES];
            for (int s = 0; s < STAGES; ++s) issued[s] = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < p.num_tiles;
                 it += gridDim.x) {
                const TileItem t = p.tiles[it];
                const NsUnit* U = p.units + t.unit;
                const void* tmA;
                const void* tmB;
                if (OP == OP_SYRK_X) { tmA = &U->tm_x[p.src]; tmB = tmA; }
                else if (OP == OP_SYRK_A) { tmA = &U->tm_a; tmB = tmA; }
                else { tmA = &U->tm_b; tmB = &U->tm_x[p.src]; }
                const int kblocks = (k_extent<OP>(*U) + BK - 1) / BK;
                int b_parts;     // SYRK: 128-row halves; GEMM: 64-col boxes
                int b_first;
                if (OP == OP_GEMM_BX) {
                    b_parts = (t.n_len + 63) / 64;
                    b_first = 0;
                } else {
                    b_parts = t.n_len / 128;
                    b_first = t.n_off / 128;
                }
                const uint32_t bytes =
                    A_STAGE_BYTES +
                    (OP == OP_GEMM_BX ? b_parts * BOX_BYTES
                                      : b_parts * 2 * BOX_BYTES);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1,
                                      abort_flag, p.err, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full_bar[stage]);
                    mbar_expect_tx(fb, bytes);
                    const uint32_t a_dst = smem_u32(sA + stage * A_STAGE_BYTES);
                    const uint32_t b_dst = smem_u32(sB + stage * B_STAGE_BYTES);
                    const int k0 = kb * BK;
                    const int r0 = t.ti * BM;
                    tma_load_2d(a_dst, tmA, fb, k0, r0);
                    tma_load_2d(a_dst + BOX_BYTES, tmA, fb, k0, r0 + 64);
                    if (OP == OP_GEMM_BX) {
                        const int c0 = t.tj * BN;
                        for (int j = 0; j < b_parts; ++j)
                            tma_load_2d(b_dst + j * BOX_BYTES, tmB, fb,
                                        c0 + 64 * j, k0);
                    } else {
                        for (int h = b_first; h < b_first + b_parts; ++h) {
                            const int rb = t.tj * BN + h * 128;
                            tma_load_2d(b_dst + h * 2 * BOX_BYTES, tmB, fb,
                                        k0, rb);
                            tma_load_2d(b_dst + (h * 2 + 1) * BOX_BYTES, tmB,
                                        fb, k0, rb + 64);
                        }
                    }
                    issued[stage] = static_cast<int>(phase) + 1;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // drain: wait (bounded) for every load this thread issued
                for (int s = 0; s < STAGES; ++s) {
                    if (issued[s] == 0) continue;
                    const uint32_t par = static_cast<uint32_t>(issued[s] - 1);
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(smem_u32(&full_bar[s]), par) &&
                           global_ns() - t0 < limit) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            bool any = false;
            for (int it = blockIdx.x; ok && it < p.num_tiles;
                 it += gridDim.x, ++local) {
                const TileItem t = p.tiles[it];
                const NsUnit* U = p.units + t.unit;
                const int kblocks = (k_extent<OP>(*U) + BK - 1) / BK;
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!wait_bounded(smem_u32(&tempty_bar[acc]), acc_phase ^ 1,
                                  abort_flag, p.err, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem =
                    tmem_base + acc * BN + (OP == OP_GEMM_BX ? 0 : t.n_off);
                const uint32_t idesc =
                    instr_desc(t.n_len, OP == OP_GEMM_BX ? 1 : 0);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_bounded(smem_u32(&full_bar[stage]), phase,
                                      abort_flag, p.err, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + stage * A_STAGE_BYTES);
                    const uint32_t b_base = smem_u32(sB + stage * B_STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = smem_desc(a_base + kk * 32, 16, 1024);
                        uint64_t bd;
                        if (OP == OP_GEMM_BX)
                            bd = smem_desc(b_base + kk * 2048, BOX_BYTES, 1024);
                        else
                            bd = smem_desc(b_base + (t.n_off / 128) * 2 *
                                                        BOX_BYTES + kk * 32,
                                           16, 1024);
                        mma_bf16(d_tmem, ad, bd, idesc,
                                 (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    any = true;
                    mma_commit(smem_u32(&empty_bar[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                mma_commit(smem_u32(&tfull_bar[acc]));
            }
            if (!ok && any) {
                // drain: all MMAs issued by this thread must finish before
                // the accumulator memory is released
                mma_commit(smem_u32(drain_bar));
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(smem_u32(drain_bar), 0) &&
                       global_ns() - t0 < limit) {
                }
            }
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int lg = warp & 3;              // TMEM lane group of this warp
        const int row = lg * 32 + lane;
        int local = 0;
        for (int it = blockIdx.x; it < p.num_tiles; it += gridDim.x, ++local) {
            const TileItem t = p.tiles[it];
            const NsUnit& U = p.units[t.unit];
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            // warp-uniform decision: tcgen05.ld below needs all 32 lanes
            const bool ok = wait_bounded(smem_u32(&tfull_bar[acc]), acc_phase,
                                         abort_flag, p.err, limit);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int gi = t.ti * BM + row;
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + acc * BN;
            const int c_begin = (OP == OP_GEMM_BX) ? 0 : t.n_off;
            const int c_end = c_begin + t.n_len;
            for (int c = c_begin; c < c_end; c += 32) {
                float v[32];
                tmem_ld32(tbase + c, v);
                epilogue_chunk<OP>(U, p.src, p.a, p.b, p.c, gi, t.tj * BN + c,
                                   v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty_bar[acc]));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile(
            "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                tmem_base),
            "r"(TMEM_COLS)
            : "memory");
    }
}

template <int OP>
cudaError_t launch_op(const NsLaunch& p, int grid, cudaStream_t s) {
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(
            ns_kernel<OP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
            SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    return launch_kernel(ns_kernel<OP>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, p);
}

}  // namespace

size_t ns_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_ns(NsOp op, const NsLaunch& p, int grid, cudaStream_t s) {
    switch (op) {
        case OP_SYRK_X: return launch_op<OP_SYRK_X>(p, grid, s);
        case OP_SYRK_A: return launch_op<OP_SYRK_A>(p, grid, s);
        case OP_GEMM_BX: return launch_op<OP_GEMM_BX>(p, grid, s);
        case OP_CHAIN: break;                  // chained launches run on CTA pairs only
    }
    return cudaErrorInvalidValue;
}

}  // namespace muon
