// Tensor-core stages of one Newton-Schulz iteration on CTA pairs
// (tcgen05 cta_group::2): the three products of the single-CTA kernels
// (A = X X^T; B = b A + c A A^T; X' = a X + B X), computed on 256 x 256
// output tiles by two CTAs of a cluster sharing one MMA.  Here the second
// product stores B + a I (a added on the diagonal in its epilogue), so the
// third is the single product X' = (B + a I) X: the same iteration, with
// an X update that reads no input block in its epilogue.
//
// Why pairs: at full tensor rate a single CTA with 128 x 256 tiles consumes
// 48 KB of operands per 512 cycles, and four 48 KB stages do not cover the
// TMA round trip under load.  In a pair each CTA stages only its 128 rows of
// A and its half (128 rows or columns) of B, 32 KB per k-block, so five
// stages fit in shared memory beside the epilogue's buffers (six where the
// epilogue reads no input) and the L2-to-SM traffic per FLOP drops by a
// third.  The even CTA of the pair (the leader) issues
// tcgen05.mma.cta_group::2 with M = 256, N = 256: rows 0-127 of A and the
// first half of B come from its shared memory, rows 128-255 and the second
// half of B from the peer's, and each CTA's TMEM receives its own 128 rows of
// the accumulator.  Both CTAs load with TMA; completion of both is counted on
// the leader's barrier.  The leader's commits multicast to both CTAs.  Both
// CTAs' epilogues drain their TMEM rows and release the accumulator on the
// leader's barrier.
//
// The producer and MMA threads' per-k-block loops are on the critical path
// (a few added instructions there cost several percent): both test their
// barrier inline and call the bounded wait only when the stage is not ready,
// and the MMA thread adds offsets to precomputed descriptors.
//
// A chained launch (OP_CHAIN) runs all of a step's products (iterations
// 1 .. ns, the weight update folded into the last X update) as one tile
// list per pair, walked once per iteration.  Each 256-wide K chunk of a tile
// is loaded once the tiles it reads are complete: epilogue warps count
// finished tiles on per-tile counters (after their TMA stores complete),
// and an eleventh warp per CTA polls the counters of the producer's coming
// chunks and publishes how many are ready through shared memory, so the
// producer's loop never waits on global memory.  The last CTA to leave
// zeroes the counters, so every launch (a replay of a captured graph too)
// starts from zero.
//
// Distributed mode's first product (SL = 1) runs each tile's K slices in
// turn on the same pair and sums them in tensor memory (accumulator 0 holds
// the running sum, accumulator 1 the newest slice).
//
// Symmetric stages compute tiles (ti, tj) with ti <= tj on the 256 grid
// ("Advancing Emerging Optimizers for Accelerated LLM Training", section
// "SYRK and fused all-reduce": upper-triangle tiles, diagonal tiles in
// full) and store them as computed; nothing below the diagonal tiles is
// written.  Consumers read the k-blocks left of an operand's diagonal tile
// from the stored transpose.  On a diagonal tile both operands are the same
// rows, so its K-major k-blocks are loaded once and read as A and as B.
//
// Every wait is bounded as in the single-CTA kernels.
#include "../../include/muon.h"
#include "tc_ptx.cuh"

namespace muon {
namespace {

using namespace ptx;

constexpr int P_STAGES_MAX = 6;
constexpr int P_HALF = 128;                        // rows per CTA
constexpr int P_A_BYTES = P_HALF * BK * 2;         // 16 KB
constexpr int P_B_BYTES = P_HALF * BK * 2;         // 16 KB
constexpr int P_BOX = 64 * 64 * 2;                 // one {64,64} box
// a diagonal tile's B descriptor steps through A's stages with B's stride
static_assert(P_A_BYTES == P_B_BYTES, "A and B stages of one size");
// K-major operands (A of every product, B of the symmetric ones) come in as
// one {64, 128} box per CTA and k-block rather than two {64, 64} boxes
constexpr bool P_WIDE_BOX = true;
constexpr int P_TMEM_COLS = 512;
constexpr int P_EPI_WARPS = 8;                     // 2 per TMEM lane group
constexpr int P_THREADS = 64 + 32 * P_EPI_WARPS;
// chained launches add one warp that watches the tile counters
template <int OP> __host__ __device__ constexpr int p_threads() {
    return P_THREADS + (OP == OP_CHAIN ? 32 : 0);
}
constexpr int P_BLK = 32 * 32 * 2;                 // one 32x32 bf16 block
// Per epilogue warp: two input slots (an A block for the second product, a
// W block when the weight update is folded into the last X update; the X
// update itself reads no input: a X + B X is computed as (B + a I) X, with
// a I added to B by the second product) and two staging blocks, so a block
// is staged while the previous one's TMA store still reads its own.  Inputs
// arrive two blocks ahead.
// Kernels whose epilogue reads nothing (the first product; the X update
// without the folded weight update) have no input slots, which leaves room
// for a sixth pipeline stage.
constexpr int P_IN_SLOTS_MAX = 2;
template <int OP, int FW> __host__ __device__ constexpr int p_in_slots() {
    return (OP == OP_SYRK_X || (OP == OP_GEMM_BX && FW == 0)) ? 0 : 2;
}
template <int FW> __host__ __device__ constexpr int p_in_blk() { return P_BLK; }
template <int OP, int FW> __host__ __device__ constexpr int p_epi_warp_bytes() {
    return p_in_slots<OP, FW>() * p_in_blk<FW>() + 2 * P_BLK;
}
template <int OP, int FW> __host__ __device__ constexpr int p_epi_bytes() {
    return P_EPI_WARPS * p_epi_warp_bytes<OP, FW>();
}
// Shared memory of a kernel with ST pipeline stages.
template <int ST> __host__ __device__ constexpr int p_epi_off() { return ST * (P_A_BYTES + P_B_BYTES) + 1024; }
template <int OP, int ST, int FW> __host__ __device__ constexpr int p_smem() {
    return p_epi_off<ST>() + p_epi_bytes<OP, FW>() + 1024;
}

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

// The operation of tile t in a launch of OP (per tile only for OP_CHAIN).
template <int OP>
__device__ __forceinline__ int tile_op(const TileItem& t) {
    if (OP != OP_CHAIN) return OP;
    return t.flags & TILE_OP_MASK;
}

// The X buffer holding the iterate that a tile of iteration s reads (s
// counts from 1 within a chained launch; other launches run one iteration).
template <int OP>
__device__ __forceinline__ int tile_src(const NsLaunch& p, int s) {
    return OP == OP_CHAIN ? (p.src ^ ((s - 1) & 1)) : p.src;
}

// A tile of a chained launch that is the last iteration's X update with
// the weight update folded in.
template <int OP>
__device__ __forceinline__ bool chain_update_tile(const NsLaunch& p, int op, int s) {
    return OP == OP_CHAIN && p.chain_last && op == OP_GEMM_BX && s == p.iters;
}

// 256-column blocks of n (X-update tiles per 256-row block of X').
__device__ __forceinline__ int row_tiles(const NsUnit& U) { return (U.n + 255) / 256; }
// 256-row blocks of m.
__device__ __forceinline__ int row_blocks(const NsUnit& U) { return (U.m + 255) / 256; }

// Tile counters of a chained launch (layout in NsUnit::tile_cnt).
__device__ __forceinline__ int32_t* x_cnt(const NsUnit& U, int ti, int cj) {
    return U.tile_cnt + ti * row_tiles(U) + cj;
}
__device__ __forceinline__ int32_t* ab_cnt(const NsUnit& U, int which_b, int i, int j) {
    const int T = row_blocks(U);
    const int lo = i < j ? i : j, hi = i < j ? j : i;
    return U.tile_cnt + T * row_tiles(U) + which_b * T * T + lo * T + hi;
}

// Chunk c (256 of K) of tile t of iteration s in a chained launch: the two
// counters it waits for (equal for an X-update tile) and their target.
struct ChunkDeps {
    const int32_t* c0;
    const int32_t* c1;
    int32_t target;
};
__device__ __forceinline__ ChunkDeps chunk_deps(const NsLaunch& p, const NsUnit& U,
                                                const TileItem& t, int op, int s, int c) {
    ChunkDeps d;
    if (op == OP_SYRK_X) {
        d.c0 = x_cnt(U, t.ti, c);
        d.c1 = x_cnt(U, t.tj, c);
        d.target = PAIR_EPI_WARPS * (p.ep_x + s - 1);
    } else if (op == OP_SYRK_A) {
        d.c0 = ab_cnt(U, 0, t.ti, c);
        d.c1 = ab_cnt(U, 0, t.tj, c);
        d.target = PAIR_EPI_WARPS * (p.ep_a + s);
    } else {
        d.c0 = d.c1 = ab_cnt(U, 1, t.ti, c);
        d.target = PAIR_EPI_WARPS * (p.ep_b + s);
    }
    return d;
}

// Does a tile of a chained launch wait for anything?  (The first product of
// iteration 1 reads X from before the launch.)
template <int OP>
__device__ __forceinline__ bool tile_waits(int op, int s) {
    return OP == OP_CHAIN && !(op == OP_SYRK_X && s == 1);
}

// Producer of a chained tile: waits until the watcher warp has published,
// for this CTA's tile number tno, more than c ready chunks; returns how
// many, or -1 when the wait ran out or the CTA aborts.
__device__ __noinline__ int wait_published(const uint64_t* slot, uint32_t tno, uint32_t c,
                                           volatile int* abort_flag, int* err, uint64_t limit) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        const uint64_t v = ld_acquire_cta_u64(slot);
        if (static_cast<uint32_t>(v >> 32) == tno && static_cast<uint32_t>(v) > c)
            return static_cast<int>(static_cast<uint32_t>(v));
        if ((i & 15) == 15) {
            if (*abort_flag) return -1;
            if (global_ns() - t0 > limit) {
                *abort_flag = 1;
                atomicCAS(err, 0, DEV_ERR_TIMEOUT);
                return -1;
            }
        }
    }
}

// Epilogue input block of a chained tile: the counter of the tile it comes
// from (second product: the A tile (ti, tj)); false if it waits for nothing
// (the X update reads no X block; a weight-update tile's W blocks are
// written by nothing in the launch).
__device__ __forceinline__ bool input_dep(const NsLaunch& p, const NsUnit& U, const TileItem& t,
                                          int op, int s, const int32_t** c, int32_t* target) {
    if (op == OP_SYRK_A) {
        *c = ab_cnt(U, 0, t.ti, t.tj);
        *target = PAIR_EPI_WARPS * (p.ep_a + s);
        return true;
    }
    return false;
}

// After a tile of a chained launch: this warp's stores of the tile are
// complete; count them on the tile's counter.
__device__ __forceinline__ void release_tile(const NsUnit& U, const TileItem& t, int op) {
    bulk_wait_all0();
    fence_proxy_async_global();
    count_release(op == OP_GEMM_BX ? x_cnt(U, t.ti, t.tj)
                                   : ab_cnt(U, op == OP_SYRK_A ? 1 : 0, t.ti, t.tj));
}

// Tile-constant fields of a unit, copied into registers once per tile (the
// kernels store through pointers the compiler cannot tell apart from the
// tables, so fields read from the tables would be reloaded after every
// store).
struct EpiUnit {
    const CUtensorMap* te_in;    // epilogue input blocks of SYRK-2 (A)
    const CUtensorMap* te_out;   // output blocks (A, B or X')
    const CUtensorMap* te_w;     // weight blocks (update folded into the last GEMM)
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

// op: the tile's operation (OP itself unless OP == OP_CHAIN); src: the X
// buffer it reads; last: the update is folded into this X update.
__device__ __forceinline__ EpiUnit load_epi_unit(const NsLaunch& p, int unit, int op, int src,
                                                 bool last) {
    const NsUnit* U = p.units + unit;
    EpiUnit e;
    e.te_in = (op == OP_GEMM_BX) ? &U->te_x[src] : &U->te_a;
    e.te_out = (op == OP_SYRK_X) ? &U->te_a : (op == OP_SYRK_A) ? &U->te_b : &U->te_x[src ^ 1];
    e.te_w = &U->te_w;
    e.m = U->m;
    e.n = U->n;
    e.ld_x = U->ld_x;
    e.ld_mm = U->ld_mm;
    e.xin = U->x[src];
    e.xout = U->x[src ^ 1];
    e.ain = U->a;
    e.out = (op == OP_SYRK_X) ? U->a : U->b;
    e.w = nullptr;
    e.w_dbg = nullptr;
    e.o_dbg = nullptr;
    e.ld_w = e.ld_dbg = 0;
    e.w_f32 = e.vec16 = e.transposed = 0;
    e.step = 0.f;
    if (op == OP_GEMM_BX && last) {
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

// Byte offset of 16-byte chunk q of row r in a 32 x 32 bf16 block laid out
// with the TMA's 64-byte swizzle (64-byte rows; chunk index XOR (r / 2) % 4).
__device__ __forceinline__ uint32_t sw64(int r, int q) {
    return static_cast<uint32_t>(r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void st_row_bf16(uint8_t* blk, int r, const float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
        for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(v[8 * q + 2 * k], v[8 * q + 2 * k + 1]);
        *reinterpret_cast<uint4*>(blk + sw64(r, q)) = w;
    }
}

__device__ __forceinline__ void ld_row_bf16(const uint8_t* blk, int r, float (&v)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 w = *reinterpret_cast<const uint4*>(blk + sw64(r, q));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(h[k]);
            v[8 * q + 2 * k] = f.x;
            v[8 * q + 2 * k + 1] = f.y;
        }
    }
}

// Column `c` of the block written from this lane's row values: element
// (row e, column c) = v[e], i.e. the transpose of the lane-per-row block.
__device__ __forceinline__ void st_col_bf16(uint8_t* blk, int c, const float (&v)[32]) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
        *reinterpret_cast<__nv_bfloat16*>(blk + sw64(e, c >> 3) + (c & 7) * 2) =
            __float2bfloat16_rn(v[e]);
}

// GEMM last iteration with the update fused (optional path): O in bf16,
// W <- W - lr * shape_scale * O in W's orientation, through global memory.
__device__ __forceinline__ void gemm_update_block(const EpiUnit& u, int r0w, int gc0, int lane,
                                                  const float (&o_in)[32], uint8_t* stage) {
    const int m = u.m, n = u.n;
    const int gi = r0w + lane;
    const bool row_ok = gi < m;
    float o[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = __bfloat162float(__float2bfloat16_rn(o_in[e]));
    if (gc0 >= n || r0w >= m) return;                         // warp-uniform
    if (!u.transposed) {
        if (!row_ok) return;
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
    st_col_bf16(stage, lane, o);
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
            const uint4 q = *reinterpret_cast<const uint4*>(stage + sw64(jj, lane & 3));
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

// Issues (lane 0) the TMA store of the staged 32 x 32 block at (x, y) after
// every lane's shared-memory writes are ordered before it.
__device__ __forceinline__ void store_block(const CUtensorMap* tm, uint8_t* stage, int x, int y,
                                            int lane) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tm, smem_u32(stage), x, y);
        bulk_commit();
    }
}

// Before staging new data: lane 0 waits until the previous TMA store has
// read the staging block.
__device__ __forceinline__ void stage_free(int lane) {
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
}

// The next of the warp's two staging blocks.  Every use ends with exactly
// one TMA store (one bulk group), so the buffers alternate with the groups:
// once at most one group (the other buffer's) still reads shared memory,
// this buffer is free.
__device__ __forceinline__ uint8_t* next_stage(uint8_t* st0, uint32_t& st_seq, int lane) {
    if (lane == 0) bulk_wait_read1();
    __syncwarp();
    return st0 + (st_seq++ & 1u) * P_BLK;
}

// The 32 x 32 blocks one epilogue warp handles in one tile: which of its
// four column blocks are needed, in order, where they are, and where their
// input blocks come from.  Built for the next tile while the current one is
// drained, so its first inputs can be requested early.
struct InPlan {
    const CUtensorMap* te_in;    // the input blocks: A (second product) or W
    int transposed;              // W blocks: the weight is the iterate's transpose
    int r0w, col0;               // first row, first column of the warp's part
    int n;                       // needed blocks
    int uses_in;                 // the tile reads one input block per needed block
    // chained launches: may its input blocks be loaded (1), not known yet
    // (0: the rows they come from are tested once, then waited for), or
    // tested and not complete (-1: the blocks wait until the tile starts)
    int ready;
    uint32_t order;              // their column-block indices, 2 bits each
    __device__ __forceinline__ int block(int k) const {
        return static_cast<int>((order >> (2 * k)) & 3u);
    }
};

template <int OP, int FW>
__device__ __forceinline__ InPlan plan_blocks(const NsLaunch& p, const TileItem& t, int s,
                                              uint32_t rank, int lg, int half) {
    const NsUnit* U = p.units + t.unit;
    const int op = tile_op<OP>(t);
    InPlan q;
    // the X update reads W blocks where the weight update is folded in
    // through TMA (FW; a chained launch's last X updates), nothing otherwise
    const bool w_in = op == OP_GEMM_BX &&
                      ((OP != OP_CHAIN && FW && p.last) || chain_update_tile<OP>(p, op, s));
    q.te_in = w_in ? &U->te_w : &U->te_a;
    q.transposed = w_in ? p.ew[t.unit].transposed : 0;
    q.uses_in = op == OP_SYRK_A || w_in;
    q.ready = (OP == OP_CHAIN && op == OP_SYRK_A) ? 0 : 1;
    q.r0w = t.ti * 256 + static_cast<int>(rank) * P_HALF + lg * 32;
    q.col0 = t.tj * 256 + half * 128;
    const int m = U->m;
    const int lim_c = (op == OP_GEMM_BX) ? U->n : m;
    q.n = 0;
    q.order = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int gc0 = q.col0 + 32 * c;
        const int rel = half * 128 + 32 * c;          // column within the tile
        // every block of the tile (a symmetric product's diagonal tile is
        // stored whole, each warp storing what its TMEM lanes computed)
        const bool nd = q.r0w < m && gc0 < lim_c && rel >= t.n_off && rel < t.n_off + t.n_len;
        if (nd) q.order |= static_cast<uint32_t>(c) << (2 * q.n++);
    }
    return q;
}

// Input items of plan q: one per needed block.
__device__ __forceinline__ int in_items(const InPlan& q) { return q.n; }

// Lane 0: TMA load of input item j of plan q (the input block of needed
// block j: an A block, or a W block) into input slot `slot`, on the slot's
// barrier.  W blocks sit at (x, y) in the weight's orientation, or (y, x)
// for a transposed unit.
__device__ __forceinline__ void issue_inputs(const InPlan& q, int j, uint8_t* slot,
                                             uint32_t bar) {
    const int x = q.col0 + 32 * q.block(j), y = q.r0w;
    fence_proxy_async_smem();
    mbar_expect_tx(bar, P_BLK);
    if (q.transposed) tma_load_2d(smem_u32(slot), q.te_in, bar, y, x);
    else tma_load_2d(smem_u32(slot), q.te_in, bar, x, y);
}

// The update folded into the last GEMM, one 32 x 32 block: O = bf16(v) (the
// final iterate), W <- W - lr * shape_scale * O in W's own orientation, the
// new W staged in `stage` and TMA-stored.  Same arithmetic as the separate
// update pass (fp32 fma on the bf16 O, stored with round-to-nearest-even).
// DBG: the optional fp32 W / bf16 O exports are written (the FW == 2
// instantiation, used while exports are registered).
template <bool DBG>
__device__ __forceinline__ void fused_update_block(const EpiUnit& u, int r0w, int gc0, int lane,
                                                   const float (&v)[32], const uint8_t* s_w,
                                                   uint8_t* stage) {
    if constexpr (!DBG) {
        // the same arithmetic, eight elements at a time (fewer live
        // registers): O = bf16(v), through the stage as O^T when the unit is
        // transposed (then each lane reads and rewrites only its own row)
        if (u.transposed) {
            st_col_bf16(stage, lane, v);
            __syncwarp();
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float o8[8], w8[8];
            if (u.transposed) {
                const uint4 ob = *reinterpret_cast<const uint4*>(stage + sw64(lane, q));
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&ob);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __bfloat1622float2(h[k]);
                    o8[2 * k] = f.x;
                    o8[2 * k + 1] = f.y;
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    o8[k] = __bfloat162float(__float2bfloat16_rn(v[8 * q + k]));
            }
            const uint4 wb = *reinterpret_cast<const uint4*>(s_w + sw64(lane, q));
            const __nv_bfloat162* hw = reinterpret_cast<const __nv_bfloat162*>(&wb);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(hw[k]);
                w8[2 * k] = f.x;
                w8[2 * k + 1] = f.y;
            }
            uint4 out;
            __nv_bfloat162* ho = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                ho[k] = __floats2bfloat162_rn(fmaf(-u.step, o8[2 * k], w8[2 * k]),
                                              fmaf(-u.step, o8[2 * k + 1], w8[2 * k + 1]));
            *reinterpret_cast<uint4*>(stage + sw64(lane, q)) = out;
        }
        store_block(u.te_w, stage, u.transposed ? r0w : gc0, u.transposed ? gc0 : r0w, lane);
    } else {
        float o[32], w[32];
    #pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
        int wrow, wcol0, wrows, wcols;      // this lane's W row segment
        if (!u.transposed) {
            ld_row_bf16(s_w, lane, w);
            wrow = r0w + lane;
            wcol0 = gc0;
            wrows = u.m;
            wcols = u.n;
        } else {
            // O^T through the stage: lane jj then owns W row gc0 + jj
            st_col_bf16(stage, lane, o);
            __syncwarp();
            ld_row_bf16(stage, lane, o);
            ld_row_bf16(s_w, lane, w);
            __syncwarp();                   // all reads of the stage are done
            wrow = gc0 + lane;
            wcol0 = r0w;
            wrows = u.n;
            wcols = u.m;
        }
    #pragma unroll
        for (int e = 0; e < 32; ++e) w[e] = fmaf(-u.step, o[e], w[e]);
        st_row_bf16(stage, lane, w);
        if ((u.w_dbg || u.o_dbg) && wrow < wrows) {
            const int64_t doff = static_cast<int64_t>(wrow) * u.ld_dbg + wcol0;
    #pragma unroll
            for (int e = 0; e < 32; ++e) {
                if (wcol0 + e >= wcols) break;
                if (u.w_dbg) u.w_dbg[doff + e] = w[e];
                if (u.o_dbg) u.o_dbg[doff + e] = __float2bfloat16_rn(o[e]);
            }
        }
        store_block(u.te_w, stage, u.transposed ? r0w : gc0, u.transposed ? gc0 : r0w, lane);
    }
}

// The tiles of pair `pair`: a planner-built range, or a stride over all.
struct TileRange {
    int begin, end, step;
};
__device__ __forceinline__ TileRange tile_range(const NsLaunch& p, int pair, int npairs) {
    TileRange r;
    if (p.pair_off) {
        r.begin = p.pair_off[pair];
        r.end = p.pair_off[pair + 1];
        r.step = 1;
    } else {
        r.begin = pair;
        r.end = p.num_tiles;
        r.step = npairs;
    }
    return r;
}

// A pair's walk over its tiles: the range once, or in a chained launch once
// per iteration s = 1 .. iters, the last time up to pair_end_last.
template <int OP>
struct TileCursor {
    int it, end, step, s;
    int begin, end_all, end_last, iters;
    __device__ __forceinline__ bool valid() const { return it < end; }
    __device__ __forceinline__ void next() {
        it += step;
        if (OP == OP_CHAIN && it >= end && s < iters) {
            ++s;
            it = begin;
            end = (s == iters) ? end_last : end_all;
        }
    }
};
template <int OP>
__device__ __forceinline__ TileCursor<OP> tile_cursor(const NsLaunch& p, int pair, int npairs) {
    const TileRange r = tile_range(p, pair, npairs);
    TileCursor<OP> c;
    c.it = c.begin = r.begin;
    c.end_all = c.end_last = r.end;
    c.step = r.step;
    c.s = 1;
    c.iters = 1;
    if (OP == OP_CHAIN && r.begin < r.end) {
        c.iters = p.iters;
        c.end_last = p.chain_last ? r.end : p.pair_end_last[pair];
    }
    c.end = (c.iters == 1) ? c.end_last : c.end_all;
    return c;
}

// FW: the last X update with the weight update folded in through TMA-loaded
// W blocks (1; 2 also writes the validation exports); for the first
// product, 3 = distributed mode across ranks (fp32 partial product out).
// SL: distributed mode's first product (K in p.shards slices, OP_SYRK_X).
template <int OP, int P_STAGES, int FW, int SL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(p_threads<OP>(), 1)
    ns2_kernel(const __grid_constant__ NsLaunch p) {
    static_assert(!SL || (OP == OP_SYRK_X && !FW), "slices: first product only");
    constexpr int P_EPI_OFF = p_epi_off<P_STAGES>();
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
    constexpr int NS_SLOTS = p_in_slots<OP, FW>();
    constexpr int NS = NS_SLOTS > 0 ? NS_SLOTS : 1;   // ring arithmetic (unused if 0)
    uint64_t* in_bar = bars + 2 * P_STAGES + 5;    // NS per epilogue warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(in_bar + P_IN_SLOTS_MAX * P_EPI_WARPS);
    static_assert(p_smem<OP, P_STAGES, FW>() <= 232448, "shared memory per CTA");
    static_assert((2 * P_STAGES + 5 + P_IN_SLOTS_MAX * P_EPI_WARPS) * 8 + 8 + 24 + 8 <= 1024,
                  "barrier area");
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // chained launches: the watcher warp's ready chunks of tile number tno
    // (tno << 32 | chunks) in dep_slot[tno & 1]; the producer's tile number
    // in prod_seq
    uint64_t* dep_slot = reinterpret_cast<uint64_t*>(tmem_slot + 2);
    uint64_t* prod_seq = dep_slot + 2;
    // chained launches: is this CTA the last to leave?
    volatile int* leave_last = reinterpret_cast<volatile int*>(prod_seq + 1);

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
        for (int w = 0; w < NS * P_EPI_WARPS; ++w) mbar_init(smem_u32(&in_bar[w]), 1);
        *abort_flag = 0;
        dep_slot[0] = dep_slot[1] = 0;
        *prod_seq = 0;
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
    // everything above overlaps the previous kernel's tail; from here on the
    // kernel reads what earlier kernels wrote
    grid_dependency_wait();
    allow_dependent_launch();
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
            TileCursor<OP> cur = tile_cursor<OP>(p, pair, npairs);
            // the next tile's record is fetched while this tile streams
            TileItem t_next = cur.valid() ? p.tiles[cur.it] : TileItem{};
            int s_next = cur.s;
            uint32_t tno = 0;        // chained launches: this tile's number
            while (ok && cur.valid()) {
                const TileItem t = t_next;
                const int s_it = s_next;
                if (OP == OP_CHAIN) st_release_cta_u64(prod_seq, ++tno);
                cur.next();
                if (cur.valid()) {
                    t_next = p.tiles[cur.it];
                    s_next = cur.s;
                    // the next tile's operand maps, while this tile streams
                    // (tiles of a grouped launch change matrix every time)
                    if (t_next.unit != t.unit) {
                        const NsUnit* Un = p.units + t_next.unit;
                        const int opn = tile_op<OP>(t_next);
                        const int srcn = tile_src<OP>(p, s_next);
                        if (opn == OP_SYRK_X) {
                            prefetch_tmap(&Un->tk_x[srcn]);
                        } else if (opn == OP_SYRK_A) {
                            prefetch_tmap(&Un->tk_a);
                            prefetch_tmap(&Un->tm_a);
                        } else {
                            prefetch_tmap(&Un->tk_b);
                            prefetch_tmap(&Un->tm_b);
                            prefetch_tmap(&Un->tm_x[srcn]);
                        }
                    }
                }
                const NsUnit* U = p.units + t.unit;
                const int op = tile_op<OP>(t);
                const int src = tile_src<OP>(p, s_it);
                const void* tmA;
                const void* tmB;
                if (P_WIDE_BOX) {
                    if (op == OP_SYRK_X) { tmA = &U->tk_x[src]; tmB = tmA; }
                    else if (op == OP_SYRK_A) { tmA = &U->tk_a; tmB = tmA; }
                    else { tmA = &U->tk_b; tmB = &U->tm_x[src]; }
                } else {
                    if (op == OP_SYRK_X) { tmA = &U->tm_x[src]; tmB = tmA; }
                    else if (op == OP_SYRK_A) { tmA = &U->tm_a; tmB = tmA; }
                    else { tmA = &U->tm_b; tmB = &U->tm_x[src]; }
                }
                const int kblocks = t.k_blocks;
                // chained launches: K in 256-wide chunks (4 k-blocks), chunk
                // c loaded once the tiles it reads are complete; chunks below
                // ready_c are known to be
                const int nchunks = (kblocks + 3) >> 2;
                int ready_c = tile_waits<OP>(op, s_it) ? 0 : nchunks;
                const int r0 = t.ti * 256 + static_cast<int>(rank) * P_HALF;
                // N = n_len columns split evenly over the pair (64 or 128 each)
                const int hb = t.n_len >> 1;
                const int b0 = t.tj * 256 + t.n_off + static_cast<int>(rank) * hb;
                // a symmetric product's diagonal tile: each CTA's half of B
                // is its own rows of A, so A's stage serves as both operands
                // (K-major k-blocks only: with both operands MN-major from
                // one buffer the second product ran 5% slower on GB300)
                const bool same = op != OP_GEMM_BX && t.ti == t.tj && t.n_off == 0;
                const uint32_t tx_mn = 2u * (P_A_BYTES + hb * BK * 2);
                const uint32_t tx_bytes = same ? 2u * P_A_BYTES : tx_mn;
                if (P_WIDE_BOX && op != OP_GEMM_BX && hb != 128) {
                    // a K-major B half is one 128-row box: full-width tiles only
                    atomicCAS(p.err, 0, DEV_ERR_BAD_TILE);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                // A and B (the symmetric products' outputs) hold only tiles
                // on or above the diagonal: the k-blocks left of an
                // operand's row block come from the stored transpose, as an
                // MN-major operand (two {64, 64} boxes).  They come first
                // in a loop of their own; the loop over the rest is the
                // plain one.
                const void* tmT = (op == OP_SYRK_A) ? &U->tm_a : &U->tm_b;
                const int kb_at = (op == OP_SYRK_X) ? 0 : 4 * t.ti;
                const int kb_bt = (op == OP_SYRK_A) ? 4 * t.tj : 0;
                const int kb_t = kb_at > kb_bt ? kb_at : kb_bt;
                int kb = 0;
                for (; kb < kb_t; ++kb) {
                    if (OP == OP_CHAIN && (kb >> 2) >= ready_c) {
                        // the watcher warp publishes how many leading chunks
                        // of this tile may be loaded
                        const uint64_t v = ld_acquire_cta_u64(&dep_slot[tno & 1]);
                        if (static_cast<uint32_t>(v >> 32) == tno &&
                            static_cast<int>(static_cast<uint32_t>(v)) > (kb >> 2))
                            ready_c = static_cast<int>(static_cast<uint32_t>(v));
                        else
                            ready_c = wait_published(&dep_slot[tno & 1], tno, kb >> 2,
                                                     abort_flag, p.err, limit);
                        if (ready_c < 0) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_global();    // TMA reads after the acquire
                    }
                    if (!mbar_try_wait(smem_u32(&empty_bar[stage]), phase ^ 1) &&
                        !wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag,
                                      p.err, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full_bar[stage]);
                    if (rank == 0) mbar_expect_tx(fb_local, tx_mn);
                    const uint32_t fb = map_to_rank(fb_local, 0);
                    const uint32_t a_dst = smem_u32(sA + stage * P_A_BYTES);
                    const uint32_t b_dst = smem_u32(sB + stage * P_B_BYTES);
                    const int k0 = kb * BK;
                    if (kb < kb_at) {
                        tma_load_2d_pair(a_dst, tmT, fb, r0, k0);
                        tma_load_2d_pair(a_dst + P_BOX, tmT, fb, r0 + 64, k0);
                    } else {
                        tma_load_2d_pair(a_dst, tmA, fb, k0, r0);
                    }
                    if (op == OP_GEMM_BX) {
                        tma_load_2d_pair(b_dst, tmB, fb, b0, k0);
                        if (hb > 64) tma_load_2d_pair(b_dst + P_BOX, tmB, fb, b0 + 64, k0);
                    } else if (kb < kb_bt) {
                        tma_load_2d_pair(b_dst, tmT, fb, b0, k0);
                        tma_load_2d_pair(b_dst + P_BOX, tmT, fb, b0 + 64, k0);
                    } else {
                        tma_load_2d_pair(b_dst, tmB, fb, k0, b0);
                    }
                    issued[stage] = static_cast<int>(phase) + 1;
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                for (; kb < kblocks; ++kb) {
                    if (OP == OP_CHAIN && (kb >> 2) >= ready_c) {
                        // the watcher warp publishes how many leading chunks
                        // of this tile may be loaded
                        const uint64_t v = ld_acquire_cta_u64(&dep_slot[tno & 1]);
                        if (static_cast<uint32_t>(v >> 32) == tno &&
                            static_cast<int>(static_cast<uint32_t>(v)) > (kb >> 2))
                            ready_c = static_cast<int>(static_cast<uint32_t>(v));
                        else
                            ready_c = wait_published(&dep_slot[tno & 1], tno, kb >> 2,
                                                     abort_flag, p.err, limit);
                        if (ready_c < 0) {
                            ok = false;
                            break;
                        }
                        fence_proxy_async_global();    // TMA reads after the acquire
                    }
                    if (!mbar_try_wait(smem_u32(&empty_bar[stage]), phase ^ 1) &&
                        !wait_bounded(smem_u32(&empty_bar[stage]), phase ^ 1, abort_flag,
                                      p.err, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full_bar[stage]);
                    if (rank == 0) mbar_expect_tx(fb_local, tx_bytes);
                    const uint32_t fb = map_to_rank(fb_local, 0);
                    const uint32_t a_dst = smem_u32(sA + stage * P_A_BYTES);
                    const uint32_t b_dst = smem_u32(sB + stage * P_B_BYTES);
                    const int k0 = kb * BK;
                    tma_load_2d_pair(a_dst, tmA, fb, k0, r0);
                    if (!P_WIDE_BOX) tma_load_2d_pair(a_dst + P_BOX, tmA, fb, k0, r0 + 64);
                    if (op == OP_GEMM_BX) {
                        tma_load_2d_pair(b_dst, tmB, fb, b0, k0);
                        if (hb > 64) tma_load_2d_pair(b_dst + P_BOX, tmB, fb, b0 + 64, k0);
                    } else if (!same) {
                        tma_load_2d_pair(b_dst, tmB, fb, k0, b0);
                        if (!P_WIDE_BOX && hb > 64)
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
            // distributed mode's first product: slices of K in turn, slice 0
            // into accumulator 0, later slices into accumulator 1 (u0, u1:
            // uses of each so far)
            constexpr bool sliced = SL != 0;
            uint32_t u0 = 0, u1 = 0;
            const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, 1024);
            // an operand read from a symmetric input's stored transpose is
            // MN-major: two 64-wide halves P_BOX apart, K rows of 128 bytes,
            // 16 K rows (2048 bytes) per MMA step
            const uint64_t a_desc_mn = smem_desc(smem_u32(sA), P_BOX, 1024);
            // B operand: MN-major for the GEMM (X), K-major otherwise
            const uint64_t b_desc_mn = smem_desc(smem_u32(sB), P_BOX, 1024);
            const uint64_t b_desc_k = smem_desc(smem_u32(sB), 16, 1024);
            TileCursor<OP> cur = tile_cursor<OP>(p, pair, npairs);
            TileItem t_next = cur.valid() ? p.tiles[cur.it] : TileItem{};
            for (; ok && cur.valid(); ++local) {
                const TileItem t = t_next;
                cur.next();
                if (cur.valid()) t_next = p.tiles[cur.it];
                const int op = tile_op<OP>(t);
                const uint32_t idesc = instr_desc(256, t.n_len, op == OP_GEMM_BX ? 1 : 0);
                // a symmetric product's diagonal tile reads B from A's stage
                // in its K-major k-blocks
                const bool same = op != OP_GEMM_BX && t.ti == t.tj && t.n_off == 0;
                const uint64_t b_desc0 = (op == OP_GEMM_BX) ? b_desc_mn : same ? a_desc0 : b_desc_k;
                const uint32_t b_kstep = (op == OP_GEMM_BX) ? (2048 >> 4) : (32 >> 4);
                const int kblocks = t.k_blocks;
                const int kslice = sliced ? kblocks / p.shards : kblocks;
                const int acc = sliced ? 0 : (local & 1);
                const uint32_t acc_phase = sliced ? (u0++ & 1) : ((local >> 1) & 1);
                if (!wait_bounded(smem_u32(&tempty_bar[acc]), acc_phase ^ 1, abort_flag,
                                  p.err, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t d_tmem = tmem_base + acc * 256 + t.n_off;
                int kin = 0;                              // step within the slice
                // k-blocks read from a symmetric input's stored transpose
                // (MN-major operands) first, in a loop of their own
                const int kb_at = (op == OP_SYRK_X) ? 0 : 4 * t.ti;
                const int kb_bt = (op == OP_SYRK_A) ? 4 * t.tj : 0;
                const int kb_t = sliced ? 0 : (kb_at > kb_bt ? kb_at : kb_bt);
                int kb = 0;
                for (; kb < kb_t; ++kb) {
                    if (!mbar_try_wait(smem_u32(&full_bar[stage]), phase) &&
                        !wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, p.err,
                                      limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const bool at = kb < kb_at, bt = kb < kb_bt;
                    const uint64_t ad0 = (at ? a_desc_mn : a_desc0) +
                                         static_cast<uint64_t>(stage) * (P_A_BYTES >> 4);
                    const uint64_t bd0 = (bt ? b_desc_mn : b_desc0) +
                                         static_cast<uint64_t>(stage) * (P_B_BYTES >> 4);
                    const uint32_t a_step = at ? (2048 >> 4) : (32 >> 4);
                    const uint32_t b_step = bt ? (2048 >> 4) : b_kstep;
                    const uint32_t id = idesc | (at ? (1u << 15) : 0u) | (bt ? (1u << 16) : 0u);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_pair(d_tmem, ad0 + static_cast<uint64_t>(kk * a_step),
                                 bd0 + static_cast<uint64_t>(kk * b_step), id,
                                 (kb > 0 || kk > 0) ? 1u : 0u);
                    any = true;
                    commit_pair_multicast(smem_u32(&empty_bar[stage]));
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                for (; kb < kblocks; ++kb) {
                    if (sliced && kin == 0 && kb > 0) {
                        // a new slice into accumulator 1, once the epilogue
                        // has taken the previous one out
                        if (!wait_bounded(smem_u32(&tempty_bar[1]), (u1++ & 1) ^ 1, abort_flag,
                                          p.err, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        d_tmem = tmem_base + 256 + t.n_off;
                    }
                    // this thread issues every MMA of the pair: the common
                    // case (stage already full) stays inline, descriptors
                    // are the stage-0 ones plus offsets (start address in
                    // 16-byte units; shared memory stays below 256 KB, so
                    // the 14-bit field never carries)
                    if (!mbar_try_wait(smem_u32(&full_bar[stage]), phase) &&
                        !wait_bounded(smem_u32(&full_bar[stage]), phase, abort_flag, p.err,
                                      limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad0 = a_desc0 + static_cast<uint64_t>(stage) * (P_A_BYTES >> 4);
                    const uint64_t bd0 = b_desc0 + static_cast<uint64_t>(stage) * (P_B_BYTES >> 4);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = ad0 + static_cast<uint64_t>(kk * 2);
                        const uint64_t bd = bd0 + static_cast<uint64_t>(kk * b_kstep);
                        mma_pair(d_tmem, ad, bd, idesc,
                             ((sliced ? kin : kb) > 0 || kk > 0) ? 1u : 0u);
                    }
                    any = true;
                    commit_pair_multicast(smem_u32(&empty_bar[stage]));
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                    // a finished later slice is handed to the epilogue
                    if (sliced && kb >= kslice && kin == kslice - 1)
                        commit_pair_multicast(smem_u32(&tfull_bar[1]));
                    if (sliced && ++kin == kslice) kin = 0;
                }
                if (!ok) break;
                if (!sliced) commit_pair_multicast(smem_u32(&tfull_bar[acc]));
            }
            if (!ok && any) {
                commit_pair_local(smem_u32(drain_bar));
                wait_quiet(smem_u32(drain_bar), 0, limit);
            }
        }
    } else if (OP == OP_CHAIN && warp == 2 + P_EPI_WARPS) {
        // ------------------------------ counter watcher (chained launches)
        // Walks this CTA's tiles as the producer does.  For a tile that
        // waits, each lane polls one chunk (relaxed loads of its counters);
        // the complete leading chunks are published, after an acquire
        // fence, in dep_slot[tno & 1] (the producer has left tile tno - 2,
        // the slot's previous user, once it works on tile tno - 1).
        TileCursor<OP> cur = tile_cursor<OP>(p, pair, npairs);
        uint32_t tno = 0;
        bool ok = true;
        while (ok && cur.valid()) {
            const TileItem t = p.tiles[cur.it];
            const int s_it = cur.s;
            cur.next();
            ++tno;
            const int op = tile_op<OP>(t);
            if (!tile_waits<OP>(op, s_it)) continue;
            const NsUnit& U = p.units[t.unit];
            const int nch = (t.k_blocks + 3) >> 2;
            uint64_t t0 = global_ns();
            while (ld_acquire_cta_u64(prod_seq) + 1 < tno) {
                const bool stop = lane == 0 && (*abort_flag || global_ns() - t0 > limit);
                if (__any_sync(0xffffffffu, stop)) {
                    ok = false;
                    break;
                }
                __nanosleep(64);
            }
            if (!ok) break;
            t0 = global_ns();
            for (int c = 0; c < nch;) {
                int ready = 1;
                if (lane < nch - c) {
                    const ChunkDeps d = chunk_deps(p, U, t, op, s_it, c + lane);
                    ready = load_relaxed(d.c0) >= d.target && load_relaxed(d.c1) >= d.target;
                }
                const uint32_t mask = __ballot_sync(0xffffffffu, ready);
                int lead = (mask == 0xffffffffu) ? 32 : __ffs(~mask) - 1;
                if (lead > nch - c) lead = nch - c;
                if (lead > 0) {
                    fence_acq_rel_gpu();
                    __syncwarp();
                    c += lead;
                    if (lane == 0)
                        st_release_cta_u64(&dep_slot[tno & 1],
                                           (static_cast<uint64_t>(tno) << 32) | uint32_t(c));
                    t0 = global_ns();
                } else {
                    bool stop = false;
                    if (lane == 0) {
                        if (*abort_flag) {
                            stop = true;
                        } else if (global_ns() - t0 > limit) {
                            *abort_flag = 1;
                            atomicCAS(p.err, 0, DEV_ERR_TIMEOUT);
                            stop = true;
                        }
                    }
                    if (__any_sync(0xffffffffu, stop)) {
                        ok = false;
                        break;
                    }
                    __nanosleep(64);
                }
            }
        }
    } else {
        // -------------------------------------------- epilogue (both CTAs)
        // warps 2..9: lane group warp % 4 (TMEM rows), column half
        // (warp - 2) / 4 (chunks 4h .. 4h + 3 of the 256 columns).  Blocks of
        // 32 x 32 go out through two alternating swizzled shared-memory
        // stages and TMA stores (which also clip at the matrix edge); the
        // epilogue's input blocks (A for SYRK-2; W where the weight update is
        // folded into the last X update) come in by TMA two blocks ahead,
        // the first two of a tile while its main loop still runs.  The X
        // update reads no input otherwise.
        const int ew = warp - 2;
        const int lg = warp & 3;
        const int half = ew >> 2;
        uint8_t* epi = smem + P_EPI_OFF + ew * p_epi_warp_bytes<OP, FW>();
        uint8_t* s_in = epi;                                   // NS slots
        uint8_t* s_st = epi + NS_SLOTS * p_in_blk<FW>();       // two staging blocks
        uint32_t in_seq = 0;     // input loads issued by this warp
        uint32_t in_use = 0;     // input loads consumed
        uint32_t st_seq = 0;     // staging blocks used
        constexpr bool sliced = SL != 0;
        uint32_t f1 = 0;         // sliced: slices taken from accumulator 1
        uint32_t tempty_leader[2];
        tempty_leader[0] = map_to_rank(smem_u32(&tempty_bar[0]), 0);
        tempty_leader[1] = map_to_rank(smem_u32(&tempty_bar[1]), 0);
        int local = 0;
        bool ok = true;
        TileCursor<OP> tc = tile_cursor<OP>(p, pair, npairs);
        TileItem t_next = tc.valid() ? p.tiles[tc.it] : TileItem{};
        int s_next = tc.s;
        // input blocks stream through the slots in tile order, across tile
        // boundaries: cur is this tile's plan, nxt the next tile's
        InPlan cur{}, nxt{};
        if (tc.valid()) cur = plan_blocks<OP, FW>(p, t_next, s_next, rank, lg, half);
        int cur_issued = 0, nxt_issued = 0;
        auto issue_from = [&](const InPlan& q, int k) {
            const uint32_t sl = in_seq % NS;
            if (lane == 0)
                issue_inputs(q, k, s_in + sl * p_in_blk<FW>(), smem_u32(&in_bar[NS * ew + sl]));
            ++in_seq;
        };
        // chained launches: the tile a tile's input blocks come from is
        // complete (lane 0 issues the loads: its acquire, then its proxy
        // fence).  Blocking at a tile's start; a single test for the next
        // tile, which must not wait while this one holds work others need.
        auto input_ready = [&](const TileItem& tt, int ss, bool block) -> bool {
            const int32_t* c;
            int32_t target;
            int r = 1;
            if (lane == 0 && input_dep(p, p.units[tt.unit], tt, tile_op<OP>(tt), ss, &c, &target)) {
                r = block ? wait_count(c, target, abort_flag, p.err, limit)
                          : count_reached(c, target);
                if (r) fence_proxy_async_global();
            }
            return __shfl_sync(0xffffffffu, r, 0) != 0;
        };
        while (ok && tc.valid()) {
            const TileItem t = t_next;
            const int s_it = s_next;
            tc.next();
            const bool has_next = tc.valid();
            if (has_next) {
                t_next = p.tiles[tc.it];
                s_next = tc.s;
                // the next tile's output and input maps (one warp per CTA)
                if (ew == 0 && lane == 0 && t_next.unit != t.unit) {
                    const NsUnit* Un = p.units + t_next.unit;
                    const int opn = tile_op<OP>(t_next);
                    if (opn == OP_SYRK_X) {
                        prefetch_tmap(&Un->te_a);
                    } else if (opn == OP_SYRK_A) {
                        prefetch_tmap(&Un->te_b);
                        prefetch_tmap(&Un->te_a);
                    } else {
                        prefetch_tmap(&Un->te_x[tile_src<OP>(p, s_next) ^ 1]);
                        if (FW || OP == OP_CHAIN) prefetch_tmap(&Un->te_w);
                    }
                }
            }
            if (OP == OP_CHAIN && cur.uses_in && cur.ready != 1) {
                if (!input_ready(t, s_it, true)) {
                    ok = false;
                    break;
                }
                cur.ready = 1;
            }
            if (cur.uses_in)
                while (cur_issued < in_items(cur) && in_seq - in_use < static_cast<uint32_t>(NS))
                    issue_from(cur, cur_issued++);
            nxt.n = 0;
            nxt_issued = 0;
            if (has_next) nxt = plan_blocks<OP, FW>(p, t_next, s_next, rank, lg, half);
            const int op = tile_op<OP>(t);
            const bool uses_in = cur.uses_in;
            // a chained weight-update tile: W read and written, no X' stored
            const bool upd = chain_update_tile<OP>(p, op, s_it);
            const EpiUnit u = load_epi_unit(p, t.unit, op, tile_src<OP>(p, s_it),
                                            (OP != OP_CHAIN && p.last) || upd);
            const int acc = local & 1;
            const uint32_t acc_phase = (local >> 1) & 1;
            const int r0w = cur.r0w;
            const int col0 = cur.col0;
            float scale = 1.f;
            // iteration 1 scales by the norm
            if (p.first && op != OP_SYRK_A && s_it == 1) {
                const float inv = p.inv_norm[t.unit];
                scale = (op == OP_SYRK_X) ? inv * inv : inv;
            }
            // the blocks this warp stores (warp-uniform), in order
            const int n_need = cur.n;
            // this warp's TMEM lanes and columns; sliced tiles keep the sum
            // in accumulator 0 and the newest slice in accumulator 1
            const uint32_t tlane = tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + half * 128;
            if (sliced) {
                for (int sl = 1; ok && sl < p.shards; ++sl) {
                    ok = wait_bounded(smem_u32(&tfull_bar[1]), f1++ & 1u, abort_flag, p.err,
                                      limit);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    if (sl == p.shards - 1) break;       // the last slice: output below
#pragma unroll 1
                    for (int k = 0; k < n_need; ++k) {
                        const int c = cur.block(k);
                        float s0[32], s1[32];
                        tmem_ld32(tlane + 32 * c, s0);
                        tmem_ld32(tlane + 256 + 32 * c, s1);
#pragma unroll
                        for (int e = 0; e < 32; ++e) s0[e] = s0[e] + s1[e];
                        tmem_st32(tlane + 32 * c, s0);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(tempty_leader[1]);
                }
                if (!ok) break;
            } else {
                ok = wait_bounded(smem_u32(&tfull_bar[acc]), acc_phase, abort_flag, p.err, limit);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
            }
            const uint32_t tbase = tlane + (sliced ? 0 : acc * 256);
#pragma unroll 1
            for (int k = 0; k < n_need; ++k) {
                const int c = cur.block(k);
                const int gc0 = col0 + 32 * c;
                float v[32];
                tmem_ld32(tbase + 32 * c, v);
                if (sliced) {
                    // ((p_0 + p_1) + ...) + p_{P-1}
                    float last[32];
                    tmem_ld32(tbase + 256 + 32 * c, last);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = v[e] + last[e];
                }
                if (uses_in) {
                    const uint32_t sl = in_use % NS;
                    const uint8_t* slot = s_in + sl * p_in_blk<FW>();
                    const bool got = wait_bounded(smem_u32(&in_bar[NS * ew + sl]),
                                                  (in_use / NS) & 1u, abort_flag, p.err, limit);
                    if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                    ++in_use;
                    // an X update's input is its W block: the weight update
                    // is folded in (no X' output)
                    const bool fold = op == OP_GEMM_BX;
                    if (fold) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= scale;
                        fused_update_block<FW == 2>(u, r0w, gc0, lane, v, slot,
                                                    next_stage(s_st, st_seq, lane));
                    } else {
                        // second product: b A + c A A, plus a on the
                        // diagonal, so that the X update's single product
                        // (B + a I) X is a X + B X
                        float x[32];
                        ld_row_bf16(slot, lane, x);
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = fmaf(p.b, x[e], p.c * v[e]);
                        if (gc0 == r0w) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (e == lane) v[e] += p.a;
                        }
                    }
                    __syncwarp();      // every lane's reads of the slots are done
                    // refill the free slots: this tile's next items, else the
                    // next tile's first
                    while (in_seq - in_use < static_cast<uint32_t>(NS)) {
                        if (cur_issued < in_items(cur)) {
                            issue_from(cur, cur_issued++);
                        } else if (nxt.uses_in && nxt_issued < in_items(nxt)) {
                            if (OP == OP_CHAIN && nxt.ready == 0)
                                nxt.ready = input_ready(t_next, s_next, false) ? 1 : -1;
                            if (OP == OP_CHAIN && nxt.ready != 1) break;
                            issue_from(nxt, nxt_issued++);
                        } else {
                            break;
                        }
                    }
                    if (fold) continue;
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= scale;
                }
                if (OP != OP_CHAIN && op == OP_GEMM_BX && p.last) {   // a chain never holds the last
                    stage_free(lane);
                    gemm_update_block(u, r0w, gc0, lane, v, s_st + (st_seq & 1u) * P_BLK);
                } else if (OP == OP_SYRK_X && FW == 3) {
                    // distributed mode across ranks: this rank's fp32 partial
                    // product, to be summed over the group before use
                    const int row = r0w + lane;
                    if (row < u.m) {
                        float* dst = p.a32 + static_cast<int64_t>(row) * p.lda32 + gc0;
                        const bool vec = gc0 + 32 <= u.m && (p.lda32 & 3) == 0 &&
                                         (reinterpret_cast<uintptr_t>(p.a32) & 15) == 0;
                        if (vec) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                *reinterpret_cast<float4*>(dst + 4 * q) =
                                    make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (gc0 + e < u.m) dst[e] = v[e];
                        }
                    }
                } else {
                    // every block as computed: X', and the symmetric
                    // products' tiles on or above the diagonal, where a
                    // diagonal tile comes out whole (its pair computes both
                    // triangles; consumers read whole rows of it)
                    uint8_t* st = next_stage(s_st, st_seq, lane);
                    st_row_bf16(st, lane, v);
                    store_block(u.te_out, st, gc0, r0w, lane);
                }
            }
            if (!__all_sync(0xffffffffu, ok)) break;
            cur = nxt;
            cur_issued = nxt_issued;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (sliced) {
                    mbar_arrive_cluster_relaxed(tempty_leader[0]);
                    mbar_arrive_cluster_relaxed(tempty_leader[1]);
                } else {
                    mbar_arrive_cluster_relaxed(tempty_leader[acc]);
                }
                // chained launches: once this warp's stores of the tile are
                // complete, count them for the rows they belong to
                if (OP == OP_CHAIN && !upd) release_tile(p.units[t.unit], t, op);
            }
            __syncwarp();
            ++local;
        }
        // after an abort: let input loads in flight land before leaving
        for (uint32_t q = in_use; q != in_seq; ++q)
            wait_quiet(smem_u32(&in_bar[NS * ew + q % NS]), (q / NS) & 1u, limit);
        if (lane == 0) bulk_wait_all0();
    }

    tc_fence_before();
    cluster_sync_all();      // no CTA leaves while its pair may still touch it
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(P_TMEM_COLS)
                     : "memory");
    }
    if (OP == OP_CHAIN) {
        // the last CTA to leave (every counter read and raise of the launch
        // done) zeroes the group's counters for the next launch
        if (threadIdx.x == 0) {
            fence_acq_rel_gpu();
            *leave_last = count_fetch_add(p.cnt_block) == static_cast<int32_t>(gridDim.x) - 1;
        }
        __syncthreads();
        if (*leave_last)
            for (int i = threadIdx.x; i < p.cnt_words; i += blockDim.x) p.cnt_block[i] = 0;
    }
}

template <int OP, int ST, int FW, int SL = 0>
cudaError_t launch_pair_st(const NsLaunch& p, int pairs, cudaStream_t s) {
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(ns2_kernel<OP, ST, FW, SL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             p_smem<OP, ST, FW>());
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    // A chained launch's tiles wait on tiles of other pairs, so all of its
    // pairs must be resident together: it is launched cooperatively, and a
    // grid that cannot be co-resident is refused instead of left to stall.
    return launch_kernel_attr(ns2_kernel<OP, ST, FW, SL>, dim3(2 * pairs),
                              dim3(p_threads<OP>()), p_smem<OP, ST, FW>(), s, OP == OP_CHAIN, p);
}

template <int OP>
cudaError_t launch_pair_op(const NsLaunch& p, int pairs, int stages, cudaStream_t s) {
    if (OP == OP_SYRK_X && p.shards > 1) return launch_pair_st<OP_SYRK_X, 5, 0, 1>(p, pairs, s);
    switch (stages) {
        case 4: return launch_pair_st<OP, 4, 0>(p, pairs, s);
        case 5: return launch_pair_st<OP, 5, 0>(p, pairs, s);
        default:
            // six stages where the epilogue has no input slots
            if constexpr (OP == OP_SYRK_A) return launch_pair_st<OP, 5, 0>(p, pairs, s);
            else return launch_pair_st<OP, 6, 0>(p, pairs, s);
    }
}

}  // namespace

int ns_pair_max_clusters() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev]) return cached[dev];
    cudaError_t e = cudaFuncSetAttribute(ns2_kernel<OP_GEMM_BX, P_STAGES_MAX, 0, 0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         p_smem<OP_GEMM_BX, P_STAGES_MAX, 0>());
    if (e != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(P_THREADS, 1, 1);
    cfg.dynamicSmemBytes = p_smem<OP_GEMM_BX, P_STAGES_MAX, 0>();
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, ns2_kernel<OP_GEMM_BX, P_STAGES_MAX, 0, 0>, &cfg);
    if (e != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = sms / 2;
    }
    cached[dev] = n;
    return n;
}

cudaError_t launch_ns_pair(NsOp op, const NsLaunch& p, int pairs, int stages,
                           cudaStream_t s) {
    switch (op) {
        case OP_SYRK_X: return launch_pair_op<OP_SYRK_X>(p, pairs, stages, s);
        case OP_SYRK_A: return launch_pair_op<OP_SYRK_A>(p, pairs, stages, s);
        case OP_GEMM_BX: return launch_pair_op<OP_GEMM_BX>(p, pairs, stages, s);
        case OP_CHAIN: return launch_pair_st<OP_CHAIN, 5, 0>(p, pairs, s);
    }
    return cudaErrorInvalidValue;
}

// Distributed mode across ranks: the first product's unscaled fp32 partial
// (its epilogue reads no input, so six pipeline stages).
cudaError_t launch_ns_pair_gram32(const NsLaunch& p, int pairs, cudaStream_t s) {
    return launch_pair_st<OP_SYRK_X, 6, 3>(p, pairs, s);
}

// The last GEMM with the update folded in through TMA-loaded W blocks (W
// blocks in the epilogue's input slots, five pipeline stages).
cudaError_t launch_ns_pair_update(const NsLaunch& p, int pairs, bool exports, cudaStream_t s) {
    return exports ? launch_pair_st<OP_GEMM_BX, 5, 2>(p, pairs, s)
                   : launch_pair_st<OP_GEMM_BX, 5, 1>(p, pairs, s);
}

}  // namespace muon

// ---------------------------------------------------------------------------
// Failure-path check of the bounded wait: one thread waits on an mbarrier
// that nothing ever arrives at; after `limit_ns` the wait records
// DEV_ERR_TIMEOUT in *err and returns, leaving the context usable.
namespace muon {
namespace {

__global__ void wait_timeout_kernel(int* err, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // phase 0 never completes: no thread arrives
    ptx::wait_bounded(ptx::smem_u32(&bar), 0, &abort_flag, err, limit_ns);
}

}  // namespace

cudaError_t launch_wait_timeout_check(int* err, unsigned long long limit_ns, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace muon
