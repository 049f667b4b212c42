// Internal data structures shared by the host planner and the kernels.
// Nothing here is part of the public C ABI (include/muon.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace muon {

// Tile edge of the element-wise stages (momentum, normalise, update).
constexpr int EW_TILE = 64;
constexpr int EW_THREADS = 256;
// The momentum pass writes one fp32 sum of squares per tile.
constexpr int EW_PARTIALS_PER_TILE = 1;

// Tensor-core stages: one CTA computes a BM x BN output tile, K in BK steps.
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;            // 64 bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;

// Device error word codes (first error wins).
constexpr int DEV_ERR_TIMEOUT = 1;
constexpr int DEV_ERR_BAD_TILE = 2;

// One unit of work: a whole matrix (full mode) or one column block of a
// matrix (blockwise mode), seen by the element-wise stages.  All pointers are
// already offset to the unit's first element.  X is the unit oriented short
// side first: m x n with m = min(rows, cols); if `transposed`, X = W-block^T.
struct EwUnit {
    void* w;
    const void* g;
    float* mom;
    float* w_dbg;            // optional fp32 export of the updated weight
    __nv_bfloat16* o_dbg;    // optional bf16 export of O (W orientation)
    __nv_bfloat16* x[2];     // iteration ping-pong buffers (m x ld_x)
    int64_t ld_w, ld_g, ld_m, ld_dbg;
    int32_t rows, cols;      // unit shape in the weight's orientation
    int32_t m, n, ld_x;
    int32_t w_dtype, g_dtype;
    int32_t transposed;
    int32_t vec_ok;          // 16-byte vector path allowed
    int32_t tiles_n;         // 64-tiles along n (X orientation)
    int64_t tile_base;       // first global element-wise tile of the unit
    int64_t tile_count;
    int32_t vec16;           // W rows allow 16-byte vector access
    float shape_scale;
};

// One unit as seen by the tensor-core stages.  Tensor maps come first and
// are 64-byte aligned (TMA reads them from global memory).
struct alignas(128) NsUnit {
    CUtensorMap tm_x[2];     // X ping/pong: dims {n, m}, box {64, 64}
    CUtensorMap tm_a;        // A = X X^T : dims {m, m}, box {64, 64}
    CUtensorMap tm_b;        // B = bA+cAA: dims {m, m}, box {64, 64}
    // X, A and B with {64, 128} boxes: a CTA's 128 rows of a K-major
    // operand in one load (CTA-pair kernels)
    CUtensorMap tk_x[2];
    CUtensorMap tk_a;
    CUtensorMap tk_b;
    // The same four matrices with {32, 32} boxes and 64-byte swizzle, for the
    // epilogue's TMA loads (A, X) and TMA stores (A, B, X').
    CUtensorMap te_x[2];
    CUtensorMap te_a;
    CUtensorMap te_b;
    // The unit's weight W (bf16, W orientation, {32, 32} boxes, 64-byte
    // swizzle) when the update is folded into the last GEMM (else unused).
    CUtensorMap te_w;
    __nv_bfloat16* x[2];
    __nv_bfloat16* a;
    __nv_bfloat16* b;
    // Chained launches: per 256 x 256 output tile, the epilogue warps that
    // finished storing their part of it (PAIR_EPI_WARPS per tile and round):
    // X tiles (ti, cj) at tile_cnt[ti * RT + cj], then A tiles (i <= j) at
    // tile_cnt[T * RT + i * T + j] and B tiles at tile_cnt[T * RT + T * T +
    // i * T + j]; T = 256-row blocks of m, RT = 256-column blocks of n.
    // Zero at the start of every launch (see NsLaunch::cnt_block).
    int32_t* tile_cnt;
    int32_t m, n, ld_x, ld_mm;
};

// One output tile of a tensor-core stage.
//   symmetric stages: rows [128*ti, +128) x cols [256*tj + n_off, +n_len)
//   GEMM stage:       rows [128*ti, +128) x cols [256*tj, +n_len)
struct TileItem {
    int32_t unit;
    int16_t ti, tj;
    int16_t n_off, n_len;
    int32_t k_blocks;        // number of BK steps (cost, also used by LPT)
    int32_t flags;           // TILE_*
};

// In a launch of OP_CHAIN the low two bits of TileItem::flags give the
// tile's operation (OP_SYRK_X, OP_SYRK_A or OP_GEMM_BX).
constexpr int TILE_OP_MASK = 3;
// epilogue warps of a CTA pair (each counts once per finished tile and row)
constexpr int PAIR_EPI_WARPS = 16;
// header words of a group's counter block (NsLaunch::cnt_block)
constexpr int CNT_HEADER_WORDS = 64;

// OP_CHAIN: iterations 1 .. iters of Newton-Schulz in one launch, every
// product but the last X update.  Each pair walks its one-iteration list
// (first-product tiles, then second-product tiles, then X-update tiles)
// once per iteration, the last time without the X-update tiles.  The K
// range of a tile comes in 256-wide chunks; chunk c is loaded once the
// tiles it reads are complete (tile counters):
//   first product (s > 1): X tiles (ti, c), (tj, c), from the X update of s-1;
//   second product:        A tiles {ti, c}, {tj, c}, from the first product of s;
//   X update:              B tile {ti, c}, from the second product of s (which
//                          implies X row c of iteration s is complete).
// The waits also order the overwrites: every tile that still reads the
// buffer a tile writes (A, B, the other X) is done before the tile's first
// chunk may load.  Each pair's walk is in stage order and a tile waits only
// on earlier stages, so no wait depends on a tile that waits on it.
enum NsOp { OP_SYRK_X = 0, OP_SYRK_A = 1, OP_GEMM_BX = 2, OP_CHAIN = 3 };

struct NsLaunch {
    const NsUnit* units;
    const TileItem* tiles;
    int32_t num_tiles;
    int32_t src;             // which X buffer is the current iterate
    float a, b, c;
    unsigned long long wait_limit_ns;
    int* err;                // device error word
    // Fused first and last iterations (CTA-pair kernels only).
    //   first: X holds the unnormalised bf16(U); inv_norm[unit] = 1/(||U||+eps)
    //          scales the SYRK-1 result by inv^2 and the GEMM result by inv;
    //   last:  the GEMM does not store X; it applies the update to W using
    //          ew[unit] (W pointers, orientation, shape scale) and lr.
    const float* inv_norm;
    const EwUnit* ew;
    int32_t first, last;
    float lr;
    // CTA-pair kernels: pair p processes tiles [pair_off[p], pair_off[p+1])
    // (a cost-balanced schedule built by the planner); nullptr = pair p takes
    // tiles p, p + pairs, ...
    const int32_t* pair_off;
    // OP_CHAIN: iterations in the launch; pair_end_last[p]: end of pair p's
    // list without its X-update tiles (the last iteration's walk); ep_x,
    // ep_a, ep_b: rounds the X, A and B counters held when the launch began
    // (the counters are zero at launch, so 0; the A rounds carry a test
    // skew when muon_debug_set_chain_test asks for one).  An X tile read in
    // iteration s is complete once its counter reaches PAIR_EPI_WARPS *
    // (ep_x + s - 1), an A tile once PAIR_EPI_WARPS * (ep_a + s), a B tile
    // once PAIR_EPI_WARPS * (ep_b + s).
    int32_t iters;
    const int32_t* pair_end_last;
    // OP_CHAIN: 1 = the last iteration's X-update tiles run too, with the
    // weight update folded in (W read and written by TMA; no X' stored)
    int32_t chain_last;
    int32_t ep_x, ep_a, ep_b;
    // Distributed mode across ranks, first product (FW == 3): the unscaled
    // fp32 partial product goes to a32 (leading dimension lda32) instead of
    // the bf16 A buffer.
    float* a32;
    int64_t lda32;
    // OP_CHAIN: the group's counter block (cnt_words words: a header of 64
    // words, word 0 counting the CTAs that have left the launch, then every
    // unit's tile_cnt block).  The last CTA to leave zeroes the block, so
    // the next launch finds it zero (the uploaded plan starts it at zero).
    int32_t* cnt_block;
    int32_t cnt_words;
    // Distributed mode, first product (CTA-pair kernels): the K range of
    // every tile is `shards` equal slices.  The pair runs them in turn, slice
    // 0 into accumulator 0 and each later slice into accumulator 1, which
    // the epilogue adds into accumulator 0 (slices 1 .. P-2) or to it (slice
    // P-1, for the output): ((p_0 + p_1) + ...) + p_{P-1}, a fixed order.
    int32_t shards;
};

// Tensor maps of one unit's momentum (fp32) and gradient, in the weight's
// orientation with {64, 64} boxes and no swizzle, for the TMA-fed momentum
// pass (groups whose every unit allows them).
struct alignas(128) EwMaps {
    CUtensorMap m;
    CUtensorMap g;
};

struct EwLaunch {
    const EwUnit* units;
    // per-unit momentum and gradient maps (nullptr: the plain-load pass)
    const EwMaps* maps;
    int* err;                // device error word (bounded waits)
    unsigned long long wait_limit_ns;
    const int64_t* tile_base;   // units' first tiles, num_units + 1 entries
    int32_t write_x;         // momentum pass also stores bf16(U) into x[0]
    int32_t num_units;
    int64_t num_tiles;       // total element-wise tiles of the group
    float* partial;          // one fp32 sum of squares per tile
    float* inv_norm;         // one fp32 1/(||U||+eps) per unit
    float beta;
    int32_t nesterov;
    float lr;
    int32_t src;             // X buffer holding the final iterate (update)
    float eps;
};

// Distributed mode across ranks: the group's summed fp32 partial products
// a32 (m x m, leading dimension lda32; tiles on or above the diagonal of the
// 256 grid) into the bf16 A buffer a16 (leading dimension ld_mm) that the
// second product reads, times scale = inv^2 in iteration 1, where inv =
// 1 / (sqrt(*sumsq_total) + eps) is also stored to *inv_norm for the X
// update.
struct DistLaunch {
    const float* a32;
    int64_t lda32;
    __nv_bfloat16* a16;
    int64_t ld_mm;
    int32_t m;
    int32_t first;
    const double* sumsq_total;
    float* inv_norm;
    float eps;
};

// Programmatic dependent launch: kernels are launched so that they may start
// while the previous kernel in the stream finishes; each kernel waits
// (griddepcontrol.wait) before it touches memory that kernel wrote.
void set_programmatic_launch(bool on);
bool programmatic_launch();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel_attr(void (*kern)(KArgs...), dim3 grid, dim3 block,
                                      size_t smem, cudaStream_t s, bool cooperative,
                                      Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (programmatic_launch()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cooperative) {
        // every block of the grid resident at once, or the launch is refused
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, Args&&... args) {
    return launch_kernel_attr(kern, grid, block, smem, s, false, std::forward<Args>(args)...);
}

#ifdef __CUDACC__
// Waits until the grids this kernel depends on have completed and their
// writes are visible (no-op without programmatic launch).
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel in the stream start launching its blocks.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// Launch wrappers (defined in the .cu files).  Return cudaGetLastError().
cudaError_t launch_ew_momentum(const EwLaunch& p, int grid, cudaStream_t s);
// The TMA-fed momentum pass (p.maps set): persistent grid of `grid` CTAs,
// EWT_CTAS_PER_SM per SM; g_f32: some unit's gradient is fp32 (larger ring
// stages).
constexpr int EWT_CTAS_PER_SM = 2;
cudaError_t launch_ew_momentum_tma(const EwLaunch& p, int grid, bool g_f32, cudaStream_t s);
cudaError_t launch_ew_norm(const EwLaunch& p, cudaStream_t s);
// the group's single unit: its sum of squares (the norm pass's order) -> *out
cudaError_t launch_ew_sumsq(const EwLaunch& p, double* out, cudaStream_t s);
cudaError_t launch_dist_convert(const DistLaunch& p, int grid, cudaStream_t s);
cudaError_t launch_ew_normalise(const EwLaunch& p, int grid, cudaStream_t s);
cudaError_t launch_ew_update(const EwLaunch& p, int grid, cudaStream_t s);
cudaError_t launch_ns(NsOp op, const NsLaunch& p, int grid, cudaStream_t s);
size_t ns_smem_bytes();
// CTA-pair (cta_group::2) kernels on 256 x 256 tiles; `pairs` clusters of 2.
cudaError_t launch_ns_pair(NsOp op, const NsLaunch& p, int pairs, int stages, cudaStream_t s);
// First product of distributed mode across ranks: unscaled fp32 partial
// product to p.a32 (tiles as in p.tiles, one stride over the pairs).
cudaError_t launch_ns_pair_gram32(const NsLaunch& p, int pairs, cudaStream_t s);
// Last GEMM with W <- W - lr*scale*O folded in (W blocks by TMA; bf16 W).
cudaError_t launch_ns_pair_update(const NsLaunch& p, int pairs, bool exports, cudaStream_t s);
int ns_pair_max_clusters();
// One-block kernel whose bounded wait must run out (failure-path check).
cudaError_t launch_wait_timeout_check(int* err, unsigned long long limit_ns, cudaStream_t s);

}  // namespace muon
