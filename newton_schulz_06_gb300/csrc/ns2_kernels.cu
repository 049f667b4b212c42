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
#include "../../include/muon.h"
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
constexpr int P_EPI_WARPS = 8;                     // 2 per TMEM lane group
constexpr int P_THREADS = 64 + 32 * P_EPI_WARPS;
constexpr int T_PITCH = 40;                        // bf16 per transpose row
constexpr int P_EPI_BYTES = P_EPI_WARPS * 32 * T_PITCH * 2;  // 32x32 per warp
constexpr int P_SMEM = P_STAGES * (P_A_BYTES + P_B_BYTES) + 1024 + 256 + P_EPI_BYTES;
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

// 32 consecutive bf16 of one row, as four 16-byte words; zeros where the
// row is invalid or the columns run past `limit`.
__device__ __forceinline__ void load_row32(const __nv_bfloat16* row, int c0, int limit,
                                           bool row_ok, uint4 (&q)[4]) {
    if (row_ok && c0 + 32 <= limit) {
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = *reinterpret_cast<const uint4*>(row + c0 + 8 * k);
    } else {
        __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(q);
#pragma unroll
        for (int e = 0; e < 32; ++e)
            h[e] = (row_ok && c0 + e < limit) ? row[c0 + e] : __float2bfloat16_rn(0.f);
    }
}

__device__ __forceinline__ float bf16_at(const uint4 (&q)[4], int e) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(q)[e]);
}

// Tile-constant fields of a unit, copied into registers once per tile (the
// kernels store through pointers the compiler cannot tell apart from the
// tables, so fields read from the tables would be reloaded after every
// store).
struct EpiUnit {
    int m, n;
    int64_t ld_x, ld_mm;
    const __nv_bfloat16* xin;    // GEMM: current iterate
    __nv_bfloat16* xout;         // GEMM: next iterate
    const __nv_bfloat16* ain;    // SYRK-2: A
    __nv_bfloat16* out;          // SYRK: A or B
    // last iteration: the weight update
    void* w;
    float* w_dbg;
    __nv_bfloat16* o_dbg;
    int64_t ld_w, ld_dbg;
    int w_f32, vec16, transposed;
    float step;
};

template <int OP>
__device__ __forceinline__ EpiUnit load_epi_unit(const NsLaunch& p, int unit) {
    const NsUnit* U = p.units + unit;
    EpiUnit e;
    e.m = U->m;
    e.n = U->n;
    e.ld_x = U->ld_x;
    e.ld_mm = U->ld_mm;
    e.xin = U->x[p.src];
    e.xout = U->x[p.src ^ 1];
    e.ain = U->a;
    e.out = (OP == OP_SYRK_X) ? U->a : U->b;
    e.w = nullptr;
    e.w_dbg = nullptr;
    e.o_dbg = nullptr;
    e.ld_w = e.ld_dbg = 0;
    e.w_f32 = e.vec16 = e.transposed = 0;
    e.step = 0.f;
    if (OP == OP_GEMM_BX && p.last) {
        const EwUnit* E = p.ew + unit;
        e.w = E->w;
        e.w_dbg = E->w_dbg;
        e.o_dbg = E->o_dbg;
        e.ld_w = E->ld_w;
        e.ld_dbg = E->ld_dbg;
        e.w_f32 = E->w_dtype == MUON_F32;
        e.vec16 = E->vec16;
        e.transposed = E->transposed;
        e.step = p.lr * E->shape_scale;
    }
    return e;
}

// Loads W[row, c0 .. c0+7] (count valid) as fp32.
__device__ __forceinline__ void w_load8(const EpiUnit& u, int64_t row, int c0, int count,
                                        float (&w)[8]) {
    const int64_t off = row * u.ld_w + c0;
    if (u.vec16 && count == 8) {
        if (u.w_f32) {
            const float4* pw = reinterpret_cast<const float4*>(static_cast<const float*>(u.w) + off);
            const float4 a = pw[0], b = pw[1];
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        } else {
            const uint4 q =
                *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(u.w) + off);
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(h[k]);
                w[2 * k] = f.x;
                w[2 * k + 1] = f.y;
            }
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        w[k] = 0.f;
        if (k < count)
            w[k] = u.w_f32 ? static_cast<const float*>(u.w)[off + k]
                           : __bfloat162float(static_cast<const __nv_bfloat16*>(u.w)[off + k]);
    }
}

// Stores the updated W[row, c0 .. c0+7] and the optional exports.
__device__ __forceinline__ void w_store8(const EpiUnit& u, int64_t row, int c0, int count,
                                         const float (&w)[8], const float (&o)[8]) {
    const int64_t off = row * u.ld_w + c0;
    if (u.vec16 && count == 8) {
        if (u.w_f32) {
            float4* pw = reinterpret_cast<float4*>(static_cast<float*>(u.w) + off);
            pw[0] = make_float4(w[0], w[1], w[2], w[3]);
            pw[1] = make_float4(w[4], w[5], w[6], w[7]);
        } else {
            uint4 q;
            __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
            for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(w[2 * k], w[2 * k + 1]);
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(u.w) + off) = q;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k >= count) continue;
            if (u.w_f32) static_cast<float*>(u.w)[off + k] = w[k];
            else static_cast<__nv_bfloat16*>(u.w)[off + k] = __float2bfloat16_rn(w[k]);
        }
    }
    if (u.w_dbg || u.o_dbg) {
        const int64_t doff = row * u.ld_dbg + c0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k >= count) continue;
            if (u.w_dbg) u.w_dbg[doff + k] = w[k];
            if (u.o_dbg) u.o_dbg[doff + k] = __float2bfloat16_rn(o[k]);
        }
    }
}

// Symmetric stages, one 32 x 32 block: this warp's rows r0w.., columns
// gc0..; lane = row.  Element (gi, gc) is stored when gc >= gi and mirrored
// to (gc, gi) when gc > gi, so each element of the m x m result is written
// once and the result is exactly symmetric.  The mirror goes through a
// shared-memory transpose so that its global stores are 16-byte vectors
// covering whole 64-byte row segments.
template <int OP>
__device__ __forceinline__ void syrk_block(const EpiUnit& u, const NsLaunch& p, float scale,
                                           int r0w, int gc0, int lane, float (&v)[32],
                                           const uint4 (&ain)[4], __nv_bfloat16* sT) {
    const int m = u.m;
    const int gi = r0w + lane;
    const int64_t ld = u.ld_mm;
#pragma unroll
    for (int e = 0; e < 32; ++e)
        v[e] = (OP == OP_SYRK_A) ? fmaf(p.b, bf16_at(ain, e), p.c * v[e]) : v[e] * scale;
    if (gc0 >= m || r0w >= m || gc0 + 31 < r0w) return;      // warp-uniform
    if (gi < m && gc0 + 31 >= gi) {
        __nv_bfloat16* row = u.out + static_cast<int64_t>(gi) * ld;
        if (gc0 >= gi && gc0 + 32 <= m) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = v[8 * q + e];
                store8_bf16(row + gc0 + 8 * q, o);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int gc = gc0 + e;
                if (gc < m && gc >= gi) row[gc] = __float2bfloat16_rn(v[e]);
            }
        }
    }
    if (gc0 + 31 <= r0w) return;                              // nothing to mirror
#pragma unroll
    for (int e = 0; e < 32; ++e) sT[e * T_PITCH + lane] = __float2bfloat16_rn(v[e]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int jj = 8 * i + (lane >> 2);
        const int R = gc0 + jj;
        const int C0 = r0w + (lane & 3) * 8;
        const uint4 q = *reinterpret_cast<const uint4*>(sT + jj * T_PITCH + (lane & 3) * 8);
        __nv_bfloat16* dst = u.out + static_cast<int64_t>(R) * ld + C0;
        if (R < m && C0 + 8 <= m && R > C0 + 7) {
            *reinterpret_cast<uint4*>(dst) = q;
        } else if (R < m) {
            const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&q);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (C0 + k < m && R > C0 + k) dst[k] = h[k];
        }
    }
    __syncwarp();
}

// GEMM stage, one 32 x 32 block: X' = scale * (a X + D); in the last
// iteration O = bf16(scale * (a X + D)) is applied to W instead of stored:
// W <- W - lr * shape_scale * O (W in its own orientation).
__device__ __forceinline__ void gemm_block(const EpiUnit& u, const NsLaunch& p, float scale,
                                           int r0w, int gc0, int lane, const float (&v)[32],
                                           const uint4 (&xin)[4], __nv_bfloat16* sT) {
    const int m = u.m, n = u.n;
    const int gi = r0w + lane;
    const bool row_ok = gi < m;
    float o[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = scale * fmaf(p.a, bf16_at(xin, e), v[e]);
    if (!p.last) {
        if (!row_ok || gc0 >= n) return;
        __nv_bfloat16* xout = u.xout + static_cast<int64_t>(gi) * u.ld_x;
        if (gc0 + 32 <= n) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float t[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) t[e] = o[8 * q + e];
                store8_bf16(xout + gc0 + 8 * q, t);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (gc0 + e < n) xout[gc0 + e] = __float2bfloat16_rn(o[e]);
        }
        return;
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __bfloat162float(__float2bfloat16_rn(o[e]));
    if (gc0 >= n || r0w >= m) return;                         // warp-uniform
    if (!u.transposed) {
        if (!row_ok) return;
        // all four W loads of the chunk in flight before any store
        float w[4][8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c0 = gc0 + 8 * q;
            w_load8(u, gi, c0, c0 < n ? min(8, n - c0) : 0, w[q]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int c0 = gc0 + 8 * q;
            if (c0 >= n) break;
            float t[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                t[e] = o[8 * q + e];
                w[q][e] = fmaf(-u.step, t[e], w[q][e]);
            }
            w_store8(u, gi, c0, min(8, n - c0), w[q], t);
        }
        return;
    }
    // transposed unit: W[gc][gi]; transpose O through shared memory
#pragma unroll
    for (int e = 0; e < 32; ++e) sT[e * T_PITCH + lane] = __float2bfloat16_rn(o[e]);
    __syncwarp();
    float w[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int R = gc0 + 8 * i + (lane >> 2);   // W row  = X column
        const int C0 = r0w + (lane & 3) * 8;       // W cols = X rows
        const int cnt = (R < n && C0 < m) ? min(8, m - C0) : 0;
        w_load8(u, R, C0, cnt, w[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int jj = 8 * i + (lane >> 2);
        const int R = gc0 + jj;
        const int C0 = r0w + (lane & 3) * 8;
        if (R < n && C0 < m) {
            const uint4 q = *reinterpret_cast<const uint4*>(sT + jj * T_PITCH + (lane & 3) * 8);
            const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&q);
            float t[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                t[k] = __bfloat162float(h[k]);
                w[i][k] = fmaf(-u.step, t[k], w[i][k]);
            }
            w_store8(u, R, C0, min(8, m - C0), w[i], t);
        }
    }
    __syncwarp();
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
            mbar_init(smem_u32(&tempty_bar[a]), 2 * P_EPI_WARPS);
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
        // warps 2..9: lane group warp % 4 (TMEM rounds), column half
        // (warp - 2) / 4 (chunks 4h .. 4h + 3 of the 256 columns)
        const int lg = warp & 3;
        const int half = (warp - 2) >> 2;
        __nv_bfloat16* sT = reinterpret_cast<__nv_bfloat16*>(
                                reinterpret_cast<uint8_t*>(bars) + 256) +
                            (warp - 2) * 32 * T_PITCH;
        uint32_t tempty_leader[2];
        tempty_leader[0] = map_to_rank(smem_u32(&tempty_bar[0]), 0);
        tempty_leader[1] = map_to_rank(smem_u32(&tempty_bar[1]), 0);
        int local = 0;
        for (int it = pair; it < p.num_tiles; it += npairs, ++local) {
            const TileItem t = p.tiles[it];
            const EpiUnit u = load_epi_unit<OP>(p, t.unit);
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const int r0w = t.ti * 256 + static_cast<int>(rank) * P_HALF + lg * 32;
            const int gi = r0w + lane;
            const int col0 = t.tj * 256 + half * 128;
            float scale = 1.f;
            if (p.first && OP != OP_SYRK_A) {
                const float inv = p.inv_norm[t.unit];
                scale = (OP == OP_SYRK_X) ? inv * inv : inv;
            }
            // epilogue input rows (GEMM: X; SYRK-2: A), prefetched a chunk
            // ahead; the first chunk is in flight while the main loop runs
            const __nv_bfloat16* in_row =
                (OP == OP_GEMM_BX) ? u.xin + static_cast<int64_t>(gi) * u.ld_x
                                   : u.ain + static_cast<int64_t>(gi) * u.ld_mm;
            const int in_limit = (OP == OP_GEMM_BX) ? u.n : u.m;
            const bool row_ok = gi < u.m;
            uint4 pre[2][4];
            if (OP != OP_SYRK_X) load_row32(in_row, col0, in_limit, row_ok, pre[0]);
            const bool ok = wait_bounded(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag,
                                         p.err, limit);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) +
                                   acc * 256 + half * 128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (OP != OP_SYRK_X && c + 1 < 4)
                    load_row32(in_row, col0 + 32 * (c + 1), in_limit, row_ok, pre[(c + 1) & 1]);
                float v[32];
                tmem_ld32(tbase + 32 * c, v);
                if (OP == OP_GEMM_BX)
                    gemm_block(u, p, scale, r0w, col0 + 32 * c, lane, v, pre[c & 1], sT);
                else
                    syrk_block<OP>(u, p, scale, r0w, col0 + 32 * c, lane, v, pre[c & 1], sT);
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
