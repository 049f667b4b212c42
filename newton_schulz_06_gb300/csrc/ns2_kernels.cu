// Tensor-core stages of one Newton-Schulz iteration on CTA pairs
// (tcgen05 cta_group::2): the same three operations as the single-CTA
// kernels (A = X X^T; B = b A + c A A^T; X' = a X + B X), computed on
// 256 x 256 output tiles by two CTAs of a cluster sharing one MMA.
//
// Why pairs: at full tensor rate a single CTA with 128 x 256 tiles consumes
// 48 KB of operands per 512 cycles, and four 48 KB stages do not cover the
// TMA round trip under load.  In a pair each CTA stages only its 128 rows of
// A and its half (128 rows or columns) of B, 32 KB per k-block, so six
// stages fit in shared memory and the L2-to-SM traffic per FLOP drops by a
// third.  The even CTA of the pair (the leader) issues
// tcgen05.mma.cta_group::2 with M = 256, N = 256: rows 0-127 of A and the
// first half of B come from its shared memory, rows 128-255 and the second
// half of B from the peer's, and each CTA's TMEM receives its own 128 rows of
// the accumulator.  Both CTAs load with TMA; completion of both is counted on
// the leader's barrier.  The leader's commits multicast to both CTAs.  Both
// CTAs' epilogues drain their TMEM rows and release the accumulator on the
// leader's barrier.
//
// Symmetric stages compute tiles (ti, tj) with ti <= tj on the 256 grid
// ("Advancing Emerging Optimizers for Accelerated LLM Training", section
// "SYRK and fused all-reduce": upper-triangle tiles, diagonal tiles in full,
// the full matrix written) and mirror every element above the diagonal.
//
// Every wait is bounded as in the single-CTA kernels.
#include "tc_ptx.cuh"

namespace muon {
namespace {

using namespace ptx;

constexpr int P_STAGES = 6;
constexpr int P_HALF = 128;                        // rows per CTA
constexpr int P_A_BYTES = P_HALF * BK * 2;         // 16 KB
constexpr int P_B_BYTES = P_HALF * BK * 2;         // 16 KB
constexpr int P_BOX = 64 * 64 * 2;                 // one {64,64} box
constexpr int P_TMEM_COLS = 512;
constexpr int P_THREADS = 192;
constexpr int P_SMEM = P_STAGES * (P_A_BYTES + P_B_BYTES) + 1024 + 256;
constexpr uint32_t P_TX_BYTES = 2 * (P_A_BYTES + P_B_BYTES);   // both CTAs

__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once the leader's MMAs issued so far complete) on the barrier at
// the same shared-memory offset in both CTAs of the pair.
__device__ __forceinline__ void commit_pair_multicast(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster."
        "multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void commit_pair_local(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            bar)
        : "memory");
}

template <int OP>
__device__ __forceinline__ int k_extent(const NsUnit& U) {
    return OP == OP_SYRK_X ? U.n : U.m;
}

// Epilogue of one 32-column chunk of row `gi` (same rules as the
// single-CTA kernels: symmetric stages store (gi, gc) when gc >= gi and
// mirror to (gc, gi) when gc > gi).
template <int OP>
__device__ __forceinline__ void epilogue_chunk(const NsUnit& U, int src, float alpha_a,
                                               float coef_b, float coef_c, int gi, int gc0,
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
                for (int e = 0; e < 8; ++e) o[e] = fmaf(alpha_a, xv[e], v[8 * q + e]);
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
    if (gc0 + 31 < gi) return;
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
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = v[8 * q + e];
            store8_bf16(row + gc0 + 8 * q, o);
        }
#pragma unroll
        for (int e = 0; e < 32; ++e)
            out[static_cast<int64_t>(gc0 + e) * ld + gi] = __float2bfloat16_rn(v[e]);
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
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
    ns2_kernel(const __grid_constant__ NsLaunch p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + P_STAGES * P_A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + P_STAGES * P_B_BYTES);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + P_STAGES;
    uint64_t* tfull_bar = bars + 2 * P_STAGES;
    uint64_t* tempty_bar = bars + 2 * P_STAGES + 2;
    uint64_t* drain_bar = bars + 2 * P_STAGES + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * P_STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();         // 0: leader, 1: peer
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull_bar[a]), 1);
            mbar_init(smem_u32(&tempty_bar[a]), 8);
        }
        mbar_init(smem_u32(drain_bar), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_u32(tmem_slot)),
            "r"(P_TMEM_COLS)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::
                         : "memory");
    }
    tc_fence_before();
    cluster_sync_all();      // peer barriers initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t limit = p.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued[P_STAGES];
            for (int s = 0; s < P_STAGES; ++s) issued[s] = 0;
            bool ok = true;
            for (int it = pair; ok && it < p.num_tiles; it += npairs) {
                const TileItem t = p.tiles[it];
                const NsUnit* U = p.units + t.unit;
                const void* tmA;
                const void* tmB;
                if (OP == OP_SYRK_X) { tmA = &U->tm_x[p.src]; tmB = tmA; }
                else if (OP == OP_SYRK_A) { tmA = &U->tm_a; tmB = tmA; }
                else { tmA = &U->tm_b; tmB = &U->tm_x[p.src]; }
                const int kblocks = (k_extent<OP>(*U) + BK - 1) / BK;
                const int r0 = t.ti * 256 + static_cast<int>(rank) * P_HALF;
                const int b0 = t.tj * 256 + static_cast<int>(rank) * P_HALF;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag,
                                      p.err, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full_bar[stage]);
                    if (rank == 0) mbar_expect_tx(fb_local, P_TX_BYTES);
                    const uint32_t fb = map_to_rank(fb_local, 0);
                    const uint32_t a_dst = smem_u32(sA + stage * P_A_BYTES);
                    const uint32_t b_dst = smem_u32(sB + stage * P_B_BYTES);
                    const int k0 = kb * BK;
                    tma_load_2d_pair(a_dst, tmA, fb, k0, r0);
                    tma_load_2d_pair(a_dst + P_BOX, tmA, fb, k0, r0 + 64);
                    if (OP == OP_GEMM_BX) {
                        tma_load_2d_pair(b_dst, tmB, fb, b0, k0);
                        tma_load_2d_pair(b_dst + P_BOX, tmB, fb, b0 + 64, k0);
                    } else {
                        tma_load_2d_pair(b_dst, tmB, fb, k0, b0);
                        tma_load_2d_pair(b_dst + P_BOX, tmB, fb, k0, b0 + 64);
                    }
                    issued[stage] = static_cast<int>(phase) + 1;
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && rank == 0) {
                // the leader's barriers count both CTAs' loads: wait for them
                for (int s = 0; s < P_STAGES; ++s)
                    if (issued[s])
                        wait_quiet(smem_u32(&full_bar[s]),
                                   static_cast<uint32_t>(issued[s] - 1), limit);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA (leader only)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            bool any = false;
            const uint32_t idesc = instr_desc(256, 256, OP == OP_GEMM_BX ? 1 : 0);
            for (int it = pair; ok && it < p.num_tiles; it += npairs, ++local) {
                const TileItem t = p.tiles[it];
                const NsUnit* U = p.units + t.unit;
                const int kblocks = (k_extent<OP>(*U) + BK - 1) / BK;
                const int acc = local & 1;
                const uint32_t acc_phase = (local >> 1) & 1;
                if (!wait_bounded(smem_u32(&tempty_bar[acc]), acc_phase ^ 1, abort_flag,
                                  p.err, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * 256;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, p.err,
                                      limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + stage * P_A_BYTES);
                    const uint32_t b_base = smem_u32(sB + stage * P_B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = smem_desc(a_base + kk * 32, 16, 1024);
                        const uint64_t bd =
                            (OP == OP_GEMM_BX) ? smem_desc(b_base + kk * 2048, P_BOX, 1024)
                                               : smem_desc(b_base + kk * 32, 16, 1024);
                        mma_pair(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    any = true;
                    commit_pair_multicast(smem_u32(&empty_bar[stage]));
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                commit_pair_multicast(smem_u32(&tfull_bar[acc]));
            }
            if (!ok && any) {
                commit_pair_local(smem_u32(drain_bar));
                wait_quiet(smem_u32(drain_bar), 0, limit);
            }
        }
    } else {
        // -------------------------------------------- epilogue (both CTAs)
        const int lg = warp & 3;
        const int row = lg * 32 + lane;
        uint32_t tempty_leader[2];
        tempty_leader[0] = map_to_rank(smem_u32(&tempty_bar[0]), 0);
        tempty_leader[1] = map_to_rank(smem_u32(&tempty_bar[1]), 0);
        int local = 0;
        for (int it = pair; it < p.num_tiles; it += npairs, ++local) {
            const TileItem t = p.tiles[it];
            const NsUnit& U = p.units[t.unit];
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const bool ok = wait_bounded(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag,
                                         p.err, limit);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int gi = t.ti * 256 + static_cast<int>(rank) * P_HALF + row;
            const uint32_t tbase =
                tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + acc * 256;
#pragma unroll 1
            for (int c = 0; c < 256; c += 32) {
                float v[32];
                tmem_ld32(tbase + c, v);
                epilogue_chunk<OP>(U, p.src, p.a, p.b, p.c, gi, t.tj * 256 + c, v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader[acc]);
        }
    }

    tc_fence_before();
    cluster_sync_all();      // no CTA leaves while its pair may still touch it
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(P_TMEM_COLS)
                     : "memory");
    }
}

template <int OP>
cudaError_t launch_pair_op(const NsLaunch& p, int pairs, cudaStream_t s) {
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(
            ns2_kernel<OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    ns2_kernel<OP><<<2 * pairs, P_THREADS, P_SMEM, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int ns_pair_max_clusters() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev]) return cached[dev];
    cudaError_t e = cudaFuncSetAttribute(ns2_kernel<OP_GEMM_BX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    if (e != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(P_THREADS, 1, 1);
    cfg.dynamicSmemBytes = P_SMEM;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, ns2_kernel<OP_GEMM_BX>, &cfg);
    if (e != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = sms / 2;
    }
    cached[dev] = n;
    return n;
}

cudaError_t launch_ns_pair(NsOp op, const NsLaunch& p, int pairs, cudaStream_t s) {
    switch (op) {
        case OP_SYRK_X: return launch_pair_op<OP_SYRK_X>(p, pairs, s);
        case OP_SYRK_A: return launch_pair_op<OP_SYRK_A>(p, pairs, s);
        case OP_GEMM_BX: return launch_pair_op<OP_GEMM_BX>(p, pairs, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace muon
