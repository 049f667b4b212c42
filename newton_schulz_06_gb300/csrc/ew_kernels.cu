// Element-wise stages of the Muon step: momentum + sum of squares, the
// per-unit Frobenius norm, normalisation into the short-side-first iterate
// X0, and the weight update.  All four are bound by HBM bandwidth.
//
// Each CTA walks 64 x 64 tiles of a unit.  A tile is read in the weight's
// orientation (coalesced, 16-byte vectors when aligned), staged in shared
// memory, and processed in the X orientation (short side first), so that a
// matrix and its transpose are reduced in exactly the same order and give
// bit-identical norms and iterates.
//
// Readings (the pages, "Advancing Emerging Optimizers for Accelerated LLM
// Training", name the momentum buffer and the orthogonalisation but not the
// formulas): M <- beta*M + G; U = G + beta*M (Nesterov) else U = M;
// X0 = U / (||U||_F + eps); W <- W - lr*scale*O.
#include "muon_internal.h"
#include "tc_ptx.cuh"
#include "../../include/muon.h"

namespace muon {
namespace {

// Unit of tile t: binary search in the compact tile_base array (a few cache
// lines, L1-resident after the first tiles).
__device__ __forceinline__ int find_unit(const int64_t* __restrict__ tile_base, int n,
                                         int64_t t) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(tile_base + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Loads `nval` (0..4) consecutive elements of type `dtype`; zero elsewhere.
__device__ __forceinline__ void ld4(const void* base, int dtype, int64_t off,
                                    int nval, bool vec, float (&v)[4]) {
    if (dtype == MUON_F32) {
        const float* p = static_cast<const float*>(base) + off;
        if (vec && nval == 4) {
            float4 q = *reinterpret_cast<const float4*>(p);
            v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = e < nval ? p[e] : 0.f;
        }
    } else {
        const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(base) + off;
        if (vec && nval == 4) {
            uint2 q = *reinterpret_cast<const uint2*>(p);
            __nv_bfloat162 lo = *reinterpret_cast<__nv_bfloat162*>(&q.x);
            __nv_bfloat162 hi = *reinterpret_cast<__nv_bfloat162*>(&q.y);
            float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
            v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                v[e] = e < nval ? __bfloat162float(p[e]) : 0.f;
        }
    }
}

__device__ __forceinline__ void st4(void* base, int dtype, int64_t off,
                                    int nval, bool vec, const float (&v)[4]) {
    if (dtype == MUON_F32) {
        float* p = static_cast<float*>(base) + off;
        if (vec && nval == 4) {
            *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) if (e < nval) p[e] = v[e];
        }
    } else {
        __nv_bfloat16* p = static_cast<__nv_bfloat16*>(base) + off;
        if (vec && nval == 4) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
            uint2 q;
            q.x = *reinterpret_cast<uint32_t*>(&lo);
            q.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(p) = q;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nval) p[e] = __float2bfloat16_rn(v[e]);
        }
    }
}

struct TileGeom {
    int u;
    int xr0, xc0;     // tile origin in X orientation
    int wr0, wc0;     // tile origin in W orientation
};

__device__ __forceinline__ TileGeom tile_geom(const EwUnit& U, int u,
                                              int64_t t) {
    TileGeom g;
    g.u = u;
    int64_t local = t - U.tile_base;
    int tr = static_cast<int>(local / U.tiles_n);
    int tc = static_cast<int>(local - static_cast<int64_t>(tr) * U.tiles_n);
    g.xr0 = tr * EW_TILE;
    g.xc0 = tc * EW_TILE;
    g.wr0 = U.transposed ? g.xc0 : g.xr0;
    g.wc0 = U.transposed ? g.xr0 : g.xc0;
    return g;
}

// Tile-constant fields of a unit in registers (the kernels store through
// pointers the compiler cannot tell apart from the unit table).
struct EwU {
    void* w;
    const void* g;
    float* mom;
    float* w_dbg;
    __nv_bfloat16* o_dbg;
    __nv_bfloat16* x[2];
    int64_t ld_w, ld_g, ld_m, ld_dbg, tile_base, tile_end;
    int rows, cols, m, n, ld_x, w_dtype, g_dtype, transposed, vec, tiles_n;
    float shape_scale;
};

__device__ __forceinline__ EwU load_ewu(const EwUnit* __restrict__ P) {
    EwU u;
    u.w = P->w; u.g = P->g; u.mom = P->mom; u.w_dbg = P->w_dbg; u.o_dbg = P->o_dbg;
    u.x[0] = P->x[0]; u.x[1] = P->x[1];
    u.ld_w = P->ld_w; u.ld_g = P->ld_g; u.ld_m = P->ld_m; u.ld_dbg = P->ld_dbg;
    u.tile_base = P->tile_base; u.tile_end = P->tile_base + P->tile_count;
    u.rows = P->rows; u.cols = P->cols; u.m = P->m; u.n = P->n; u.ld_x = P->ld_x;
    u.w_dtype = P->w_dtype; u.g_dtype = P->g_dtype; u.transposed = P->transposed;
    u.vec = P->vec_ok; u.tiles_n = P->tiles_n; u.shape_scale = P->shape_scale;
    return u;
}

__device__ __forceinline__ TileGeom geom_of(const EwU& U, int64_t t) {
    TileGeom g;
    g.u = 0;
    const int64_t local = t - U.tile_base;
    const int tr = static_cast<int>(local / U.tiles_n);
    const int tc = static_cast<int>(local - static_cast<int64_t>(tr) * U.tiles_n);
    g.xr0 = tr * EW_TILE;
    g.xc0 = tc * EW_TILE;
    g.wr0 = U.transposed ? g.xc0 : g.xr0;
    g.wc0 = U.transposed ? g.xr0 : g.xc0;
    return g;
}

// Pass 1: M <- beta*M + G; U as above; per tile and warp one fp32 sum of U^2
// taken in the X orientation (short side first) in a fixed order, so that a
// matrix and its transpose give the same sums.  With write_x the
// unnormalised iterate bf16(U) is stored in the X orientation as well.
// Thread (i, j4) owns rows i + 16k (k = 0..3), columns j4 .. j4 + 3 of a
// 64 x 64 tile; only transposed units go through shared memory.
__global__ void __launch_bounds__(EW_THREADS, 4)
ew_momentum_kernel(const EwLaunch p) {
    grid_dependency_wait();
    allow_dependent_launch();
    __shared__ float sU[EW_TILE][EW_TILE + 1];
    __shared__ float red[2][EW_THREADS / 32];
    const int i = threadIdx.x >> 4;          // 0..15
    const int j4 = (threadIdx.x & 15) * 4;   // 0..60
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x >= p.num_tiles) return;
    int u = find_unit(p.tile_base, p.num_units, blockIdx.x);
    EwU U = load_ewu(p.units + u);
    int parity = 0;
    // grid-stride: concurrent blocks work on neighbouring tiles
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, parity ^= 1) {
        while (t >= U.tile_end) U = load_ewu(p.units + (++u));
        const TileGeom g = geom_of(U, t);
        float uv[4][4];
        float mv[4][4], gv[4][4];
        int nval[4];
        const bool interior =
            U.vec && g.wr0 + EW_TILE <= U.rows && g.wc0 + EW_TILE <= U.cols;  // block-uniform
        if (interior) {
            // branch-free: the thread's four 16-byte M loads and four G loads
            // are issued back to back; M and G are streamed (touched once)
            const int64_t r0 = g.wr0 + i;
            const float* mp = U.mom + r0 * U.ld_m + g.wc0 + j4;
            float4 mq[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mq[k] = __ldcs(reinterpret_cast<const float4*>(mp + 16 * k * U.ld_m));
            if (U.g_dtype == MUON_BF16) {
                const __nv_bfloat16* gp =
                    static_cast<const __nv_bfloat16*>(U.g) + r0 * U.ld_g + g.wc0 + j4;
                uint2 gq[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    gq[k] = __ldcs(reinterpret_cast<const uint2*>(gp + 16 * k * U.ld_g));
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 lo = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&gq[k].x));
                    const float2 hi = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&gq[k].y));
                    gv[k][0] = lo.x; gv[k][1] = lo.y; gv[k][2] = hi.x; gv[k][3] = hi.y;
                }
            } else {
                const float* gp = static_cast<const float*>(U.g) + r0 * U.ld_g + g.wc0 + j4;
                float4 gq[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    gq[k] = __ldcs(reinterpret_cast<const float4*>(gp + 16 * k * U.ld_g));
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    gv[k][0] = gq[k].x; gv[k][1] = gq[k].y; gv[k][2] = gq[k].z; gv[k][3] = gq[k].w;
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mv[k][0] = mq[k].x; mv[k][1] = mq[k].y; mv[k][2] = mq[k].z; mv[k][3] = mq[k].w;
                nval[k] = 4;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int wr = g.wr0 + i + 16 * k, wc = g.wc0 + j4;
                nval[k] = max((wr < U.rows) ? min(4, U.cols - wc) : 0, 0);
                ld4(U.mom, MUON_F32, wr * U.ld_m + wc, nval[k], U.vec, mv[k]);
                ld4(U.g, U.g_dtype, wr * U.ld_g + wc, nval[k], U.vec, gv[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int wr = g.wr0 + i + 16 * k, wc = g.wc0 + j4;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                mv[k][e] = fmaf(p.beta, mv[k][e], gv[k][e]);
                uv[k][e] = e < nval[k] ? (p.nesterov ? fmaf(p.beta, mv[k][e], gv[k][e])
                                                     : mv[k][e])
                                       : 0.f;
            }
            if (interior)
                __stcs(reinterpret_cast<float4*>(U.mom + static_cast<int64_t>(wr) * U.ld_m + wc),
                       make_float4(mv[k][0], mv[k][1], mv[k][2], mv[k][3]));
            else
                st4(U.mom, MUON_F32, wr * U.ld_m + wc, nval[k], U.vec, mv[k]);
        }
        if (U.transposed) {            // block-uniform
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) sU[i + 16 * k][j4 + e] = uv[k][e];
            __syncthreads();
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) uv[k][e] = sU[j4 + e][i + 16 * k];
            __syncthreads();
        }
        // uv now holds X(i + 16k, j4 + e) of this tile
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc = fmaf(uv[k][e], uv[k][e], acc);
            if (p.write_x) {
                const int gr = g.xr0 + i + 16 * k, gc = g.xc0 + j4;
                int nx = (gr < U.m) ? min(4, U.n - gc) : 0;
                nx = max(nx, 0);
                st4(U.x[0], MUON_BF16, static_cast<int64_t>(gr) * U.ld_x + gc, nx, true,
                    uv[k]);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) red[parity][warp] = acc;
        __syncthreads();
        if (threadIdx.x == 0) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < EW_THREADS / 32; ++w) s += red[parity][w];
            p.partial[t] = s;
        }
    }
}

// The same pass with M and G streamed into shared memory by TMA: one
// thread loads tile j + S - 1 of the CTA's walk while all threads process
// tile j from an S-stage ring, so each CTA keeps S - 1 tiles of loads in
// flight with few registers (two CTAs per SM).  The thread-to-element map,
// the arithmetic, the masked stores and the order of the sum of squares are
// those of ew_momentum_kernel, so both passes give identical bits.  Tiles
// past the matrix edge read zeros (TMA fill), which add nothing to the sum.
// GB: bytes of the largest gradient element (stage size); NS stages; CPS:
// CTAs per SM the launch is sized for.  The transposed units' transpose
// goes through the stage's momentum block once its values are in registers,
// with column c of row r at (c + r) mod 64 (two-way bank conflicts at most).
template <int GB, int NS>
struct EwtCfg {
    static constexpr int M_BYTES = EW_TILE * EW_TILE * 4;
    static constexpr int G_BYTES = EW_TILE * EW_TILE * GB;
    static constexpr int STAGE = M_BYTES + G_BYTES;
    static constexpr int S = NS;
    static constexpr int SMEM = S * STAGE + 2 * (EW_THREADS / 32) * 4 + S * 8 + 128;
};

template <int GB, int NS, int CPS>
__global__ void __launch_bounds__(EW_THREADS, CPS)
ew_momentum_tma_kernel(const EwLaunch p) {
    using C = EwtCfg<GB, NS>;
    extern __shared__ uint8_t ewt_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(ewt_raw) + 127) & ~uintptr_t(127));
    float* red = reinterpret_cast<float*>(smem + C::S * C::STAGE);
    uint64_t* full = reinterpret_cast<uint64_t*>(red + 2 * (EW_THREADS / 32));
    __shared__ int abort_flag;
    const int i = threadIdx.x >> 4;          // 0..15
    const int j4 = (threadIdx.x & 15) * 4;   // 0..60
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int k = 0; k < C::S; ++k) ptx::mbar_init(ptx::smem_u32(&full[k]), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    grid_dependency_wait();
    allow_dependent_launch();
    const int64_t nj = p.num_tiles > blockIdx.x
                           ? (p.num_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    // thread 0: loads of the CTA's j-th tile into stage j % S
    int pu = 0;                              // producer's unit cursor
    auto issue = [&](int64_t j) {
        const int64_t t = blockIdx.x + j * gridDim.x;
        while (t >= __ldg(p.tile_base + pu + 1)) ++pu;
        const EwUnit& U = p.units[pu];
        const int64_t local = t - U.tile_base;
        const int tr = static_cast<int>(local / U.tiles_n);
        const int tc = static_cast<int>(local - static_cast<int64_t>(tr) * U.tiles_n);
        const int wr0 = U.transposed ? tc * EW_TILE : tr * EW_TILE;
        const int wc0 = U.transposed ? tr * EW_TILE : tc * EW_TILE;
        const int st = static_cast<int>(j % C::S);
        uint8_t* dst = smem + st * C::STAGE;
        const uint32_t bar = ptx::smem_u32(&full[st]);
        ptx::fence_proxy_async_smem();       // earlier reads of the stage first
        ptx::mbar_expect_tx(bar, C::M_BYTES + EW_TILE * EW_TILE *
                                     (U.g_dtype == MUON_F32 ? 4 : 2));
        ptx::tma_load_2d(ptx::smem_u32(dst), &p.maps[pu].m, bar, wc0, wr0);
        ptx::tma_load_2d(ptx::smem_u32(dst + C::M_BYTES), &p.maps[pu].g, bar, wc0, wr0);
    };
    if (threadIdx.x == 0)
        for (int64_t j = 0; j < C::S - 1 && j < nj; ++j) issue(j);
    int u = nj ? find_unit(p.tile_base, p.num_units, blockIdx.x) : 0;
    EwU U = load_ewu(p.units + u);
    int parity = 0;
    int64_t j = 0;
    for (; j < nj; ++j, parity ^= 1) {
        const int64_t t = blockIdx.x + j * gridDim.x;
        if (threadIdx.x == 0 && j + C::S - 1 < nj) issue(j + C::S - 1);
        while (t >= U.tile_end) U = load_ewu(p.units + (++u));
        const TileGeom g = geom_of(U, t);
        const int st = static_cast<int>(j % C::S);
        const uint32_t ph = static_cast<uint32_t>((j / C::S) & 1);
        if (!ptx::wait_bounded(ptx::smem_u32(&full[st]), ph, &abort_flag, p.err,
                               p.wait_limit_ns))
            break;
        const float* sm = reinterpret_cast<const float*>(smem + st * C::STAGE);
        const uint8_t* sg = smem + st * C::STAGE + C::M_BYTES;
        const bool interior =
            U.vec && g.wr0 + EW_TILE <= U.rows && g.wc0 + EW_TILE <= U.cols;  // block-uniform
        float uv[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = i + 16 * k;
            const float4 mq = *reinterpret_cast<const float4*>(sm + r * EW_TILE + j4);
            float gv[4];
            if (U.g_dtype == MUON_BF16) {
                const uint2 q = *reinterpret_cast<const uint2*>(
                    reinterpret_cast<const __nv_bfloat16*>(sg) + r * EW_TILE + j4);
                const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
                const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
                gv[0] = lo.x; gv[1] = lo.y; gv[2] = hi.x; gv[3] = hi.y;
            } else {
                const float4 q = *reinterpret_cast<const float4*>(
                    reinterpret_cast<const float*>(sg) + r * EW_TILE + j4);
                gv[0] = q.x; gv[1] = q.y; gv[2] = q.z; gv[3] = q.w;
            }
            float mv[4] = {mq.x, mq.y, mq.z, mq.w};
            const int wr = g.wr0 + r, wc = g.wc0 + j4;
            const int nval = interior ? 4 : max((wr < U.rows) ? min(4, U.cols - wc) : 0, 0);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                mv[e] = fmaf(p.beta, mv[e], gv[e]);
                uv[k][e] = e < nval ? (p.nesterov ? fmaf(p.beta, mv[e], gv[e]) : mv[e]) : 0.f;
            }
            if (interior)
                __stcs(reinterpret_cast<float4*>(U.mom + static_cast<int64_t>(wr) * U.ld_m + wc),
                       make_float4(mv[0], mv[1], mv[2], mv[3]));
            else
                st4(U.mom, MUON_F32, static_cast<int64_t>(wr) * U.ld_m + wc, nval, U.vec, mv);
        }
        if (U.transposed) {            // block-uniform
            float* sT = const_cast<float*>(sm);
            __syncthreads();           // every thread's M values are in registers
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = i + 16 * k, c = j4 + e;
                    sT[r * EW_TILE + ((c + r) & (EW_TILE - 1))] = uv[k][e];
                }
            __syncthreads();
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = j4 + e, c = i + 16 * k;
                    uv[k][e] = sT[r * EW_TILE + ((c + r) & (EW_TILE - 1))];
                }
        }
        // uv now holds X(i + 16k, j4 + e) of this tile
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc = fmaf(uv[k][e], uv[k][e], acc);
            if (p.write_x) {
                const int gr = g.xr0 + i + 16 * k, gc = g.xc0 + j4;
                int nx = (gr < U.m) ? min(4, U.n - gc) : 0;
                nx = max(nx, 0);
                st4(U.x[0], MUON_BF16, static_cast<int64_t>(gr) * U.ld_x + gc, nx, true,
                    uv[k]);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) red[parity * (EW_THREADS / 32) + warp] = acc;
        __syncthreads();               // also: every read of this stage is done
        if (threadIdx.x == 0) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < EW_THREADS / 32; ++w) sum += red[parity * (EW_THREADS / 32) + w];
            p.partial[t] = sum;
        }
    }
    if (j < nj && threadIdx.x == 0) {
        // a wait ran out: let the loads still in flight land before leaving
        for (int64_t q = j; q < nj && q < j + C::S - 1; ++q)
            ptx::wait_quiet(ptx::smem_u32(&full[q % C::S]),
                            static_cast<uint32_t>((q / C::S) & 1), p.wait_limit_ns);
    }
}

// Per unit: ||U||_F from its tile sums in a fixed order (fp64), then
// inv_norm = 1 / (||U|| + eps).  One block per unit: thread k sums tiles
// k, k + 256, ... in order, then a fixed tree combines the 256 sums.
// Unit u's sum of its tile sums in that order, by one block of 256 threads;
// the result in thread 0 (red: 256 doubles of shared memory).
__device__ __forceinline__ double unit_sum_squares(const EwLaunch& p, int u, double* red) {
    const EwUnit& U = p.units[u];
    const int64_t base = U.tile_base * EW_PARTIALS_PER_TILE;
    const int64_t count = U.tile_count * EW_PARTIALS_PER_TILE;
    double s = 0.0;
    for (int64_t k = threadIdx.x; k < count; k += 256)
        s += static_cast<double>(p.partial[base + k]);
    red[threadIdx.x] = s;
    __syncthreads();
#pragma unroll
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    return red[0];
}

__global__ void __launch_bounds__(256) ew_norm_kernel(const EwLaunch p) {
    grid_dependency_wait();
    allow_dependent_launch();
    __shared__ double red[256];
    const int u = blockIdx.x;
    const double ss = unit_sum_squares(p, u, red);
    if (threadIdx.x == 0)
        p.inv_norm[u] = static_cast<float>(1.0 / (sqrt(ss) + (double)p.eps));
}

// Distributed mode across ranks: the slice's sum of squares itself, summed
// over the group by the caller; the norm follows in dist_convert_kernel with
// the same arithmetic as ew_norm_kernel.
__global__ void __launch_bounds__(256) ew_sumsq_kernel(const EwLaunch p, double* out) {
    grid_dependency_wait();
    allow_dependent_launch();
    __shared__ double red[256];
    const double ss = unit_sum_squares(p, 0, red);
    if (threadIdx.x == 0) *out = ss;
}

// Distributed mode across ranks: the group's summed fp32 partial products to
// the bf16 A buffer the second product reads, on and above the 256-tile
// diagonal (what the symmetric products' consumers read), times inv^2 in
// iteration 1: A = bf16(sum * scale), the first product's epilogue rounding
// of a one-GPU step.  One thread per 4 consecutive columns of a row.
__global__ void __launch_bounds__(256) dist_convert_kernel(const DistLaunch p) {
    grid_dependency_wait();
    allow_dependent_launch();
    float scale = 1.f;
    if (p.first) {
        const float inv = static_cast<float>(1.0 / (sqrt(*p.sumsq_total) + (double)p.eps));
        scale = inv * inv;
        if (blockIdx.x == 0 && threadIdx.x == 0) *p.inv_norm = inv;
    }
    const int64_t q4 = (p.m + 3) / 4;              // 4-column groups per row
    const int64_t total = static_cast<int64_t>(p.m) * q4;
    for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int i = static_cast<int>(g / q4);
        const int j0 = static_cast<int>(g - static_cast<int64_t>(i) * q4) * 4;
        if ((j0 >> 8) < (i >> 8)) continue;          // below the diagonal tiles
        const float* src = p.a32 + static_cast<int64_t>(i) * p.lda32 + j0;
        __nv_bfloat16* dst = p.a16 + static_cast<int64_t>(i) * p.ld_mm + j0;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (j0 + e < p.m) dst[e] = __float2bfloat16_rn(src[e] * scale);
    }
}

// Pass 2: X0 = bf16(U * inv_norm) in the X orientation.
__global__ void __launch_bounds__(EW_THREADS)
ew_normalise_kernel(const EwLaunch p) {
    grid_dependency_wait();
    allow_dependent_launch();
    __shared__ float sU[EW_TILE][EW_TILE + 1];
    const int i = threadIdx.x >> 4;
    const int j4 = (threadIdx.x & 15) * 4;
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        const int u = find_unit(p.tile_base, p.num_units, t);
        const EwUnit& U = p.units[u];
        const TileGeom g = tile_geom(U, u, t);
        const bool vec = U.vec_ok != 0;
        const float inv = p.inv_norm[u];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = i + 16 * k;
            const int wr = g.wr0 + r, wc = g.wc0 + j4;
            int nval = (wr < U.rows) ? min(4, U.cols - wc) : 0;
            nval = max(nval, 0);
            float mv[4], gv[4];
            ld4(U.mom, MUON_F32, wr * U.ld_m + wc, nval, vec, mv);
            ld4(U.g, U.g_dtype, wr * U.ld_g + wc, nval, vec, gv);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float uv = p.nesterov ? fmaf(p.beta, mv[e], gv[e]) : mv[e];
                sU[r][j4 + e] = uv;
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int xr = i + 16 * k;
            const int gr = g.xr0 + xr, gc = g.xc0 + j4;
            int nval = (gr < U.m) ? min(4, U.n - gc) : 0;
            nval = max(nval, 0);
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int xc = j4 + e;
                v[e] = (U.transposed ? sU[xc][xr] : sU[xr][xc]) * inv;
            }
            st4(U.x[0], MUON_BF16, static_cast<int64_t>(gr) * U.ld_x + gc,
                nval, true, v);
        }
        __syncthreads();
    }
}

// Update: W <- W - lr*scale*O with O read from the final iterate.
__global__ void __launch_bounds__(EW_THREADS)
ew_update_kernel(const EwLaunch p) {
    grid_dependency_wait();
    allow_dependent_launch();
    __shared__ float sX[EW_TILE][EW_TILE + 1];
    const int i = threadIdx.x >> 4;
    const int j4 = (threadIdx.x & 15) * 4;
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        const int u = find_unit(p.tile_base, p.num_units, t);
        const EwUnit& U = p.units[u];
        const TileGeom g = tile_geom(U, u, t);
        const bool vec = U.vec_ok != 0;
        const __nv_bfloat16* X = U.x[p.src];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int xr = i + 16 * k;
            const int gr = g.xr0 + xr, gc = g.xc0 + j4;
            int nval = (gr < U.m) ? min(4, U.n - gc) : 0;
            nval = max(nval, 0);
            float v[4];
            ld4(X, MUON_BF16, static_cast<int64_t>(gr) * U.ld_x + gc, nval,
                true, v);
#pragma unroll
            for (int e = 0; e < 4; ++e) sX[xr][j4 + e] = v[e];
        }
        __syncthreads();
        const float step = p.lr * U.shape_scale;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = i + 16 * k;
            const int wr = g.wr0 + r, wc = g.wc0 + j4;
            int nval = (wr < U.rows) ? min(4, U.cols - wc) : 0;
            nval = max(nval, 0);
            float w[4], o[4];
            ld4(U.w, U.w_dtype, wr * U.ld_w + wc, nval, vec, w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = j4 + e;
                o[e] = U.transposed ? sX[c][r] : sX[r][c];
                w[e] = fmaf(-step, o[e], w[e]);
            }
            st4(U.w, U.w_dtype, wr * U.ld_w + wc, nval, vec, w);
            if (U.w_dbg)
                st4(U.w_dbg, MUON_F32, wr * U.ld_dbg + wc, nval, false, w);
            if (U.o_dbg)
                st4(U.o_dbg, MUON_BF16, wr * U.ld_dbg + wc, nval, false, o);
        }
        __syncthreads();
    }
}

}  // namespace

namespace {
bool g_programmatic = true;
}
void set_programmatic_launch(bool on) { g_programmatic = on; }
bool programmatic_launch() { return g_programmatic; }

cudaError_t launch_ew_momentum(const EwLaunch& p, int grid, cudaStream_t s) {
    return launch_kernel(ew_momentum_kernel, dim3(grid), dim3(EW_THREADS), 0, s, p);
}

template <int GB, int NS, int CPS>
cudaError_t launch_ewt(const EwLaunch& p, int grid, cudaStream_t s) {
    static int attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    auto kern = ew_momentum_tma_kernel<GB, NS, CPS>;
    const int smem = EwtCfg<GB, NS>::SMEM;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    return launch_kernel(kern, dim3(grid), dim3(EW_THREADS), smem, s, p);
}

// Two CTAs per SM, four stages (three for fp32 gradients).  Measured on
// GB300 against three CTAs with three stages, eight alternating runs of the
// Qwen3-30B-A3B block: the pass alone the same or 1% slower, but the step
// 1.0% faster (7.24 against 7.31 ms; the products that follow start sooner),
// the 48-layer set the same.
cudaError_t launch_ew_momentum_tma(const EwLaunch& p, int grid, bool g_f32, cudaStream_t s) {
    return g_f32 ? launch_ewt<4, 3, EWT_CTAS_PER_SM>(p, grid, s)
                 : launch_ewt<2, 4, EWT_CTAS_PER_SM>(p, grid, s);
}

cudaError_t launch_ew_norm(const EwLaunch& p, cudaStream_t s) {
    return launch_kernel(ew_norm_kernel, dim3(p.num_units), dim3(256), 0, s, p);
}

cudaError_t launch_ew_sumsq(const EwLaunch& p, double* out, cudaStream_t s) {
    return launch_kernel(ew_sumsq_kernel, dim3(1), dim3(256), 0, s, p, out);
}

cudaError_t launch_dist_convert(const DistLaunch& p, int grid, cudaStream_t s) {
    return launch_kernel(dist_convert_kernel, dim3(grid), dim3(256), 0, s, p);
}

cudaError_t launch_ew_normalise(const EwLaunch& p, int grid, cudaStream_t s) {
    return launch_kernel(ew_normalise_kernel, dim3(grid), dim3(EW_THREADS), 0, s, p);
}

cudaError_t launch_ew_update(const EwLaunch& p, int grid, cudaStream_t s) {
    return launch_kernel(ew_update_kernel, dim3(grid), dim3(EW_THREADS), 0, s, p);
}

}  // namespace muon
