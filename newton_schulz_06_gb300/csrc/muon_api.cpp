// Host runtime of libmuon: parameter registry, planner (units, groups,
// cost-sorted tile lists, tensor maps, workspace layout), launch sequence,
// stage timing and error reporting behind the C ABI of include/muon.h.
//
// Work decomposition.  Every registered matrix (full mode) or each of its nb
// equal column blocks (blockwise mode, "Advancing Emerging Optimizers for
// Accelerated LLM Training", section "Blockwise mode") is one unit with its
// own norm, iteration and shape scale.  All units of a group go through each
// stage in ONE launch: the single-GPU counterpart of the pages' layer-wise
// distribution (section "Layer-wise distributed optimizer"), with tiles
// ordered by estimated cost rather than round-robin (section "Load
// balancing").  Groups exist only when the caller's workspace cannot hold
// every unit's intermediates at once; they run one after another.
#include <algorithm>
#include <cmath>
#include <map>
#include <tuple>
#include <queue>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/muon.h"
#include "muon_internal.h"

using namespace muon;

namespace {

constexpr size_t HEADER_BYTES = 256;
constexpr float NORM_EPS = 1e-7f;
constexpr int64_t MAX_DIM = int64_t(1) << 20;
constexpr int64_t MAX_SHORT = 32768;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

enum Stage { ST_MOMENTUM, ST_NORM, ST_NORMALISE, ST_SYRK1, ST_SYRK2,
             ST_GEMM, ST_UPDATE, ST_CHAIN };

struct UnitDesc {
    int param = 0, block = 0;
    int64_t rows = 0, cols = 0, col_off = 0;
    int m = 0, n = 0, ld_x = 0, ld_mm = 0;
    bool transposed = false;
    float scale = 1.f;
    size_t x_bytes = 0, mm_bytes = 0, buf_bytes = 0;
    size_t cnt_bytes = 0;       // chained launches: one counter per X, A and B tile
    int shards = 1;             // distributed mode: slices of the long side
    int64_t ew_tiles = 0;
    size_t need = 0;   // scratch bytes of this unit inside a group
};

struct GroupDesc {
    int u0 = 0, u1 = 0;                      // unit range [u0, u1)
    size_t ew_off = 0, ns_off = 0;           // metadata offsets in ws
    size_t tb_off = 0;                       // int64 tile_base[units + 1]
    size_t em_off = 0;                       // EwMaps[units] (TMA-fed momentum)
    bool ew_tma = false;                     // every unit's M and G suit TMA
    bool g_f32 = false;                      // some unit's gradient is fp32
    bool w_tma = true;                       // every unit's W fits te_w
    size_t t_sx_off = 0, t_sa_off = 0, t_g_off = 0;
    int n_sx = 0, n_sa = 0, n_g = 0;
    // CTA-pair schedules: per-pair offsets into the tile lists
    size_t o_sx_off = 0, o_sa_off = 0, o_g_off = 0;
    int p_sx = 0, p_sa = 0, p_g = 0;
    // chained launch (every product of iterations 1 .. ns but the last X
    // update): one iteration's tiles per pair, pair offsets, and each pair's
    // end without its X-update tiles
    size_t t_c_off = 0, o_c_off = 0, e_c_off = 0;
    int n_c = 0, p_c = 0;
    bool chain_ok = false;
    // this group's tile counters (chained launches): in the metadata region
    // (never aliased by a group's scratch), zeroed by the chained launch's
    // last CTA, so a step's launches carry no state from earlier steps (a
    // step captured in a CUDA graph replays correctly)
    size_t rc_off = 0, rc_bytes = 0;
    // distributed mode across ranks: the first product's tiles in row-block
    // order (in the chained launch's space, unused then), and where each
    // 256-row block's tiles start (T + 1 entries)
    size_t t_d_off = 0;
    std::vector<int> d_band;
    int64_t ew_tiles = 0;
    int shards = 1;                          // distributed mode: P
};

struct Plan {
    bool valid = false;
    int mode = -1, nb = 0;
    // groups also cut (at matrix boundaries) every ~chunk_elems elements, so
    // that muon_step_host can overlap one group's copies with another's
    // compute (0: groups only where the workspace requires them)
    int64_t chunk_elems = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    std::vector<UnitDesc> units;
    std::vector<GroupDesc> groups;
    size_t scratch_off = 0;                  // start of the group scratch
    // distributed mode across ranks (one unit): its bf16 A buffer
    __nv_bfloat16* d_a16 = nullptr;
    int64_t syrk_tiles = 0, gemm_tiles = 0, ew_tiles = 0;
    int64_t useful_flops_iter = 0, executed_flops_iter = 0;
};

struct LaunchRec {
    int stage;
    cudaEvent_t start, stop;
};

}  // namespace

struct muon_ctx {
    int device = 0;
    cudaStream_t stream = nullptr;
    int num_sms = 0;
    std::vector<muon_param> params;
    std::vector<float*> exp_w;
    std::vector<void*> exp_o;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    std::string err;
    Plan plan;
    bool profiling = false;
    std::vector<cudaEvent_t> event_pool;
    std::vector<LaunchRec> launches;
    int last_launch_count = 0;
    unsigned long long wait_limit_ns = 2000000000ull;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    bool pair = true;          // CTA-pair kernels (256 x 256 tiles)
    bool fuse = true;          // pair mode: normalisation fused into iteration 1
    // pair mode: 0 = separate update pass, 1 = update folded into the last
    // GEMM through registers, 2 = folded in through TMA-loaded W blocks
    // (groups whose weights are all bf16 and 16-byte aligned; else pass 0)
    int fuse_update = 2;
    // pair mode: TMA pipeline depth (4, 5, or 6: six where the kernel's
    // epilogue has no input slots, five for the second product)
    int stages = 6;
    bool fuse_stages = true;   // pair mode: iterations chained in one launch where it pays
    int chain_max_tiles = 8;   // X-update tiles per CTA pair up to which groups chain
    int chain_min_tiles = -1;  // X-update tiles from which groups chain (-1: one per pair)
    bool chain_last = true;    // a chain also runs the last X update (weight update folded in)
    // failure test only (muon_debug_set_chain_test): rounds added to what a
    // chained launch's second products wait for, so their waits run out
    int debug_chain_skew = 0;
    int max_pairs = 0;
    // muon_step_host: copy streams (gradients in, weights out) and events,
    // created on first use
    cudaStream_t s_in = nullptr, s_out = nullptr;
    std::vector<cudaEvent_t> host_events;
    // groups muon_step_host aims for (at matrix boundaries); measured on GB300
    // (pipelined step, G in and W out): the Qwen3-30B-A3B block 12.55 / 11.14 /
    // 10.52 / 10.61 ms and the Kimi-K2 layer 58.3 / 54.3 / 53.4 / 56.7 ms with
    // 4 / 8 / 16 / 32 groups
    int host_chunks = 16;
    // momentum pass fed by TMA: 1 = where the group's maps allow it and its
    // units are small (EWT_MAX_TILES_PER_UNIT), 2 = wherever the maps allow
    // it, 0 = never
    int ew_tma = 1;
    // distributed mode across ranks (muon_dist_configure): the one
    // registered parameter is a rank's slice of a matrix whose orientation
    // (dist_transposed) and shape scale (dist_scale) it takes
    bool dist = false;
    int dist_transposed = 0;
    float dist_scale = 1.f;
    // the phases' progress: momentum done, grams queued this iteration, the
    // X buffer holding the iterate
    bool dist_ready = false;
    int dist_grams = 0;
    int dist_cur = 0;
};

namespace {

std::string g_create_err;

int fail(muon_ctx* h, int code, const std::string& msg) {
    if (h) h->err = msg; else g_create_err = msg;
    return code;
}

int cuda_fail(muon_ctx* h, cudaError_t e, const char* what) {
    return fail(h, MUON_ERR_CUDA,
                std::string(what) + ": " + cudaGetErrorString(e));
}

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
            cudaSetDevice(prev);
    }
};

size_t elem_size(int dtype) { return dtype == MUON_F32 ? 4 : 2; }

// Per-unit work counts shared by planning and plan statistics.
//   single-CTA tiles: 128 x 256 (symmetric: 128-column halves below the
//   diagonal or past m skipped); CTA-pair tiles: 256 x 256 (symmetric:
//   ti <= tj on the 256 grid).
void unit_tiles(const UnitDesc& u, bool pair, int64_t* syrk, int64_t* gemm,
                int64_t* useful, int64_t* executed) {
    const int64_t m = u.m, n = u.n;
    const int64_t kn = ceil_div(n, BK) * BK, km = ceil_div(m, BK) * BK;
    int64_t s = 0, g = 0, ex = 0;
    if (pair) {
        const int64_t T2 = ceil_div(m, 256);
        s = T2 * (T2 + 1) / 2;
        g = T2 * ceil_div(n, 256);
        ex = s * 2 * 256 * 256 * (kn + km) + g * 2 * 256 * 256 * km;
    } else {
        const int64_t T = ceil_div(m, BM);
        for (int64_t ti = 0; ti < T; ++ti)
            for (int64_t tj = 0; tj < ceil_div(T, 2); ++tj) {
                const int64_t bl = 2 * tj, br = 2 * tj + 1;
                const int nl = (bl < T && bl >= ti) + (br < T && br >= ti);
                if (!nl) continue;
                ++s;
                ex += 2 * BM * 128 * nl * (kn + km);
            }
        g = T * ceil_div(n, BN);
        for (int64_t tj = 0; tj < ceil_div(n, BN); ++tj) {
            const int64_t nl = std::min<int64_t>(BN, align_up(n - tj * BN, 16));
            ex += T * 2 * BM * nl * km;
        }
    }
    *syrk = s;
    *gemm = g;
    *useful = m * (m + 1) * n + m * (m + 1) * m + 2 * m * m * n;
    *executed = ex;
}

int build_units(muon_ctx* h, int mode, int nb, std::vector<UnitDesc>* out) {
    out->clear();
    if (mode != MUON_FULL && mode != MUON_BLOCKWISE && mode != MUON_DISTRIBUTED)
        return fail(h, MUON_ERR_INVALID_ARG,
                    "mode must be MUON_FULL, MUON_BLOCKWISE or MUON_DISTRIBUTED");
    const int nblk = (mode == MUON_BLOCKWISE) ? nb : 1;
    const int shards = (mode == MUON_DISTRIBUTED) ? nb : 1;
    if (nblk < 1 || shards < 1) return fail(h, MUON_ERR_INVALID_ARG, "nb must be >= 1");
    if (shards > 1 && !h->pair)
        return fail(h, MUON_ERR_UNSUPPORTED, "distributed mode needs the CTA-pair kernels");
    if (h->dist && (mode != MUON_FULL || h->params.size() != 1 || !h->pair))
        return fail(h, MUON_ERR_UNSUPPORTED,
                    "a rank's slice (muon_dist_configure) runs alone, in full mode, on the "
                    "CTA-pair kernels");
    for (size_t i = 0; i < h->params.size(); ++i) {
        const muon_param& p = h->params[i];
        if (p.cols % nblk != 0)
            return fail(h, MUON_ERR_UNSUPPORTED,
                        "nb=" + std::to_string(nblk) + " does not divide cols=" +
                            std::to_string(p.cols) + " of parameter " +
                            std::to_string(i));
        const int64_t bc = p.cols / nblk;
        for (int j = 0; j < nblk; ++j) {
            UnitDesc u;
            u.param = static_cast<int>(i);
            u.block = j;
            u.rows = p.rows;
            u.cols = bc;
            u.col_off = j * bc;
            u.transposed = p.rows > bc;
            u.m = static_cast<int>(std::min(p.rows, bc));
            u.n = static_cast<int>(std::max(p.rows, bc));
            if (u.m > MAX_SHORT)
                return fail(h, MUON_ERR_UNSUPPORTED,
                            "short side above 32768 in parameter " + std::to_string(i));
            u.ld_x = static_cast<int>(align_up(u.n, 64));
            u.ld_mm = static_cast<int>(align_up(u.m, 64));
            u.scale = static_cast<float>(
                std::sqrt(std::max(1.0, double(p.rows) / double(bc))));
            if (h->dist) {
                // a rank's slice: the whole matrix's orientation and scale
                u.transposed = h->dist_transposed != 0;
                u.m = static_cast<int>(u.transposed ? bc : p.rows);
                u.n = static_cast<int>(u.transposed ? p.rows : bc);
                u.scale = h->dist_scale;
                if (u.m > MAX_SHORT)
                    return fail(h, MUON_ERR_UNSUPPORTED, "short side above 32768");
                u.ld_x = static_cast<int>(align_up(u.n, 64));
                u.ld_mm = static_cast<int>(align_up(u.m, 64));
            }
            u.x_bytes = align_up(size_t(u.m) * u.ld_x * 2, 1024);
            u.mm_bytes = align_up(size_t(u.m) * u.ld_mm * 2, 1024);
            u.shards = shards;
            if (shards > 1 && (u.n % shards != 0 || (u.n / shards) % BK != 0))
                return fail(h, MUON_ERR_UNSUPPORTED,
                            std::to_string(shards) + " slices of n=" + std::to_string(u.n) +
                                " (parameter " + std::to_string(i) +
                                ") are not equal multiples of 64");
            {
                const size_t T = size_t(ceil_div(u.m, 256)), RT = size_t(ceil_div(u.n, 256));
                u.cnt_bytes = align_up((T * RT + 2 * T * T) * 4, 256);
            }
            u.buf_bytes = 2 * u.x_bytes + 2 * u.mm_bytes;
            u.ew_tiles = ceil_div(u.m, EW_TILE) * ceil_div(u.n, EW_TILE);
            u.need = u.buf_bytes + size_t(u.ew_tiles) * 4 * EW_PARTIALS_PER_TILE + 4;
            out->push_back(u);
        }
    }
    return MUON_OK;
}

size_t meta_bound(const std::vector<UnitDesc>& units) {
    size_t b = 0;
    for (const UnitDesc& u : units) {
        // the larger of the two tilings bounds either
        int64_t s, g, x, y, s2, g2;
        unit_tiles(u, false, &s, &g, &x, &y);
        unit_tiles(u, true, &s2, &g2, &x, &y);
        s = std::max(s, s2);
        g = std::max(g, g2);
        // tile lists (room for twice the tiles, as if every tile were split in
        // halves) and pair offsets
        // (per unit: 256-byte alignment of 8 tables, and room for a group's
        // counter header, as if every unit were a group)
        b += sizeof(EwUnit) + sizeof(NsUnit) + sizeof(EwMaps) + 9 * 256 + u.cnt_bytes +
             2 * size_t(2 * s + g) * sizeof(TileItem) + 3 * 4 * 1024;
    }
    return align_up(b, 1024);
}

constexpr size_t GROUP_SLACK = 4096;
// groups whose units average fewer 64 x 64 tiles than this use the TMA-fed
// momentum pass
constexpr int64_t EWT_MAX_TILES_PER_UNIT = 1024;

void sizes_for(const std::vector<UnitDesc>& units, size_t* min_b, size_t* full_b) {
    const size_t fixed = align_up(HEADER_BYTES + meta_bound(units), 1024) + GROUP_SLACK;
    size_t mx = 0, sum = 0;
    for (const UnitDesc& u : units) {
        mx = std::max(mx, u.need);
        sum += u.need;
    }
    *min_b = align_up(fixed + mx, 1024);
    *full_b = align_up(fixed + sum, 1024);
}

// Greedy grouping in registration order within the scratch budget.
bool make_groups(const std::vector<UnitDesc>& units, size_t scratch,
                 std::vector<GroupDesc>* groups, int64_t chunk_elems = 0) {
    groups->clear();
    size_t acc = 0;
    int64_t elems = 0;
    GroupDesc g;
    g.u0 = 0;
    for (size_t i = 0; i < units.size(); ++i) {
        const size_t need = units[i].need;
        if (need + GROUP_SLACK > scratch) return false;
        const bool full = acc + need + GROUP_SLACK > scratch;
        // chunk cuts only where a matrix starts (its blocks stay together)
        const bool chunk = chunk_elems > 0 && elems >= chunk_elems && units[i].block == 0;
        if ((full || chunk) && i > static_cast<size_t>(g.u0)) {
            g.u1 = static_cast<int>(i);
            groups->push_back(g);
            g = GroupDesc();
            g.u0 = static_cast<int>(i);
            acc = 0;
            elems = 0;
        }
        acc += need;
        elems += units[i].rows * units[i].cols;
    }
    g.u1 = static_cast<int>(units.size());
    if (g.u1 > g.u0) groups->push_back(g);
    return true;
}

int encode_map(muon_ctx* h, CUtensorMap* tm, void* base, int64_t inner,
               int64_t outer, int64_t ld, uint32_t box = 64, uint32_t box_rows = 0) {
    cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
    cuuint32_t boxd[2] = {box, box_rows ? box_rows : box};
    cuuint32_t es[2] = {1, 1};
    // {64, 64} boxes: 128-byte rows, 128-byte swizzle (operand tiles);
    // {32, 32} boxes: 64-byte rows, 64-byte swizzle (epilogue blocks)
    const CUtensorMapSwizzle sw =
        box == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = h->encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                           strides, boxd, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(h, MUON_ERR_CUDA,
                    "cuTensorMapEncodeTiled failed with code " + std::to_string(int(r)));
    return MUON_OK;
}

// A {64, 64}-box, unswizzled map of a rows x cols matrix in the weight's
// orientation (fp32 momentum or a gradient) for the TMA-fed momentum pass;
// false if its base or row pitch does not suit TMA (16-byte multiples).
bool encode_ew_map(muon_ctx* h, CUtensorMap* tm, const void* base, int dtype, int64_t rows,
                   int64_t cols, int64_t ld) {
    const size_t es = elem_size(dtype);
    if (reinterpret_cast<uintptr_t>(base) % 16 != 0 || (size_t(ld) * es) % 16 != 0)
        return false;
    cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(ld) * es};
    cuuint32_t boxd[2] = {EW_TILE, EW_TILE};
    cuuint32_t el[2] = {1, 1};
    const CUresult r = h->encode(
        tm, dtype == MUON_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
        2, const_cast<void*>(base), dims, strides, boxd, el, CU_TENSOR_MAP_INTERLEAVE_NONE,
        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

void sort_tiles(std::vector<TileItem>* v) {
    std::stable_sort(v->begin(), v->end(), [](const TileItem& a, const TileItem& b) {
        const int64_t ca = int64_t(a.k_blocks) * a.n_len;
        const int64_t cb = int64_t(b.k_blocks) * b.n_len;
        return ca > cb;
    });
}

// Within each unit, tiles in bands of TILE_BAND row blocks, each band column
// by column (row blocks inside a column), instead of row by row.  Tiles of
// equal cost reach the pairs round-robin, so the pairs run consecutive tiles
// of this order together: a band of 8 rows and about 74 / 8 columns, whose
// operands (8 row blocks of one operand, ~9 column blocks of the other) stay
// in L2 however large the unit.  Row by row, a 7168 x 8192 unit's X update
// ran 3 row blocks against all 32 column blocks at once (~128 MB, the size of
// L2) and read its operands from DRAM 1.75 times over.  Stable, so units keep
// their order.
constexpr int TILE_BAND = 8;
void band_tiles(std::vector<TileItem>* v) {
    std::stable_sort(v->begin(), v->end(), [](const TileItem& a, const TileItem& b) {
        if (a.unit != b.unit) return a.unit < b.unit;
        const int ba = a.ti / TILE_BAND, bb = b.ti / TILE_BAND;
        if (ba != bb) return ba < bb;
        if (a.tj != b.tj) return a.tj < b.tj;
        return a.ti < b.ti;
    });
}

// Longest-processing-time schedule of tiles over `P` CTA pairs: the costliest
// remaining tile goes to the least-loaded pair.  With allow_split, a
// full-width tile that would push that pair past the average load is split
// into two 128-column halves (each output element is still computed by one
// pair in one K order, so a split changes no result); measured on GB300 the
// halves run too slowly for this to pay (they need 1.5x the operand traffic
// per FLOP), so the planner does not split.  Rewrites *v in pair-major
// order; off[p] .. off[p + 1] are pair p's tiles.
void lpt_schedule(std::vector<TileItem>* v, int P, bool allow_split,
                  std::vector<int32_t>* off) {
    struct It {
        TileItem t;
        int64_t cost, seq;
    };
    auto cost_of = [](const TileItem& t) { return int64_t(t.k_blocks) * t.n_len; };
    auto cmp = [](const It& a, const It& b) {
        return a.cost != b.cost ? a.cost < b.cost : a.seq > b.seq;
    };
    std::priority_queue<It, std::vector<It>, decltype(cmp)> q(cmp);
    int64_t seq = 0, total = 0;
    for (const TileItem& t : *v) {
        q.push({t, cost_of(t), seq++});
        total += cost_of(t);
    }
    const double target = P > 0 ? double(total) / P : 0.0;
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> loads;
    for (int p = 0; p < P; ++p) loads.push({0, p});
    std::vector<std::vector<TileItem>> lists(P);
    while (!q.empty()) {
        const It it = q.top();
        q.pop();
        const Load l = loads.top();
        if (allow_split && it.t.n_len == 256 && double(l.first + it.cost) > target * 1.001) {
            TileItem a = it.t, b = it.t;
            a.n_len = b.n_len = 128;
            b.n_off = static_cast<int16_t>(it.t.n_off + 128);
            q.push({a, it.cost / 2, seq++});
            q.push({b, it.cost / 2, seq++});
            continue;
        }
        loads.pop();
        lists[l.second].push_back(it.t);
        loads.push({l.first + it.cost, l.second});
    }
    v->clear();
    off->assign(P + 1, 0);
    for (int p = 0; p < P; ++p) {
        (*off)[p] = static_cast<int32_t>(v->size());
        v->insert(v->end(), lists[p].begin(), lists[p].end());
    }
    (*off)[P] = static_cast<int32_t>(v->size());
}

// Groups with at least one X-update tile per CTA pair and at most
// chain_max_tiles of them per pair (8 unless MUON_CHAIN_MAX_TILES says
// otherwise) chain their iterations in one launch.  Chaining pays where
// stage tails are a large share of a launch (a few full waves, as for one
// large matrix: 3072^2 -28%, 2048 x 8192 -10%).  Below one wave every stage
// is a short dependent hop either way and separate launches are slightly
// faster (256 x 512 up to 2048^2: 2-5%); with many short tiles per pair the
// store completion the epilogue waits for before counting a tile costs more
// than the tails (a 388-matrix group: +9..20%).  MUON_CHAIN_MIN_TILES
// overrides the lower bound (tiles, not per pair).
bool chain_eligible(const muon_ctx* h, int shards, int64_t gemm_tiles) {
    const int64_t pairs = std::max(1, h->max_pairs);
    const int64_t lo = h->chain_min_tiles >= 0 ? h->chain_min_tiles : pairs;
    return h->pair && h->fuse_stages && shards == 1 && gemm_tiles > 0 && gemm_tiles >= lo &&
           gemm_tiles <= int64_t(h->chain_max_tiles) * pairs;
}

// Schedule of a chained launch over P CTA pairs.  A list-scheduling
// simulation runs the stages in order (first product, second product, X
// update; costs k-blocks x columns, K in 256-wide chunks).  Chunk c of a
// tile is ready when the tiles it reads end: X tiles (ti, c), (tj, c) for
// the first product, A tiles {ti, c}, {tj, c} for the second, B tile
// {ti, c} for the X update.  Within a stage the tiles go in the order their
// first chunk is ready (ties: the natural order, column-major for the X
// update so that column 0 of X', which the next first products read first,
// comes first), each to the pair that is free first; a tile runs its chunks
// in order, each no earlier than it is ready.  Three iterations are
// simulated; the last one's per-pair lists are the template every iteration
// walks.  Each list is in stage order, so a waiting tile only waits on
// tiles of earlier stages.  end_last[p]: the end of pair p's list without
// its X-update tiles.
void lpt_schedule_chain(const std::vector<TileItem>& sx, const std::vector<TileItem>& sa,
                        std::vector<TileItem> gm, int P, std::vector<TileItem>* v,
                        std::vector<int32_t>* off, std::vector<int32_t>* end_last) {
    using Key = std::tuple<int32_t, int, int>;            // unit, tile row, tile column
    using Load = std::pair<int64_t, int>;
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> free_at;
    for (int p = 0; p < P; ++p) free_at.push({0, p});
    std::map<Key, int64_t> x_end, a_end, b_end;
    auto sym = [](int32_t u, int i, int j) { return Key{u, std::min(i, j), std::max(i, j)}; };
    std::vector<std::vector<TileItem>> lists(P);
    std::vector<int32_t> mid(P, 0);
    // ready time of chunk c of tile t of stage op
    auto chunk_ready = [&](const TileItem& t, int op, int c) -> int64_t {
        if (op == OP_SYRK_X) {
            auto e0 = x_end.find(Key{t.unit, t.ti, c}), e1 = x_end.find(Key{t.unit, t.tj, c});
            return std::max(e0 == x_end.end() ? 0 : e0->second,
                            e1 == x_end.end() ? 0 : e1->second);
        }
        if (op == OP_SYRK_A) return std::max(a_end[sym(t.unit, t.ti, c)], a_end[sym(t.unit, t.tj, c)]);
        return b_end[sym(t.unit, t.ti, c)];
    };
    auto stage = [&](const std::vector<TileItem>& tiles, int op, std::map<Key, int64_t>* out) {
        std::vector<int64_t> r0(tiles.size());
        for (size_t i = 0; i < tiles.size(); ++i) r0[i] = chunk_ready(tiles[i], op, 0);
        std::vector<size_t> order(tiles.size());
        for (size_t i = 0; i < order.size(); ++i) order[i] = i;
        std::stable_sort(order.begin(), order.end(),
                         [&](size_t a, size_t b) { return r0[a] < r0[b]; });
        std::map<Key, int64_t> ends;
        for (size_t i : order) {
            TileItem t = tiles[i];
            const Load l = free_at.top();
            free_at.pop();
            const int nch = static_cast<int>(ceil_div(t.k_blocks, 4));
            const int64_t per = int64_t(t.k_blocks) * t.n_len / std::max(1, nch);
            int64_t now = l.first;
            for (int c = 0; c < nch; ++c) now = std::max(now, chunk_ready(t, op, c)) + per;
            free_at.push({now, l.second});
            t.flags = (t.flags & ~TILE_OP_MASK) | op;
            lists[l.second].push_back(t);
            ends[op == OP_GEMM_BX ? Key{t.unit, t.ti, t.tj} : sym(t.unit, t.ti, t.tj)] = now;
        }
        *out = std::move(ends);
    };
    // the X update's natural order: column-major
    std::stable_sort(gm.begin(), gm.end(), [](const TileItem& a, const TileItem& b) {
        return a.unit != b.unit ? a.unit < b.unit : a.tj != b.tj ? a.tj < b.tj : a.ti < b.ti;
    });
    for (int iter = 0; iter < 3; ++iter) {
        for (auto& l : lists) l.clear();
        if (iter == 0) x_end.clear();        // X from before the launch
        stage(sx, OP_SYRK_X, &a_end);
        stage(sa, OP_SYRK_A, &b_end);
        for (int p = 0; p < P; ++p) mid[p] = static_cast<int32_t>(lists[p].size());
        stage(gm, OP_GEMM_BX, &x_end);
    }
    v->clear();
    off->assign(P + 1, 0);
    end_last->assign(P, 0);
    for (int p = 0; p < P; ++p) {
        (*off)[p] = static_cast<int32_t>(v->size());
        (*end_last)[p] = (*off)[p] + mid[p];
        v->insert(v->end(), lists[p].begin(), lists[p].end());
    }
    (*off)[P] = static_cast<int32_t>(v->size());
}

// The tiles of one unit (local index li) for the three products: symmetric
// tiles (ti <= tj) of the first and second product, X-update tiles.
void append_unit_tiles(const UnitDesc& u, int li, bool pair, std::vector<TileItem>* tsx,
                       std::vector<TileItem>* tsa, std::vector<TileItem>* tg) {
    const int kx = static_cast<int>(ceil_div(u.n, BK));
    const int km = static_cast<int>(ceil_div(u.m, BK));
    if (pair) {
        const int64_t T2 = ceil_div(u.m, 256);
        for (int64_t ti = 0; ti < T2; ++ti)
            for (int64_t tj = ti; tj < T2; ++tj) {
                TileItem t{};
                t.unit = li;
                t.ti = static_cast<int16_t>(ti);
                t.tj = static_cast<int16_t>(tj);
                t.n_off = 0;
                t.n_len = 256;
                t.k_blocks = kx;
                tsx->push_back(t);
                t.k_blocks = km;
                tsa->push_back(t);
            }
        for (int64_t ti = 0; ti < T2; ++ti)
            for (int64_t tj = 0; tj < ceil_div(u.n, 256); ++tj) {
                TileItem t{};
                t.unit = li;
                t.ti = static_cast<int16_t>(ti);
                t.tj = static_cast<int16_t>(tj);
                t.n_off = 0;
                t.n_len = 256;
                t.k_blocks = km;
                tg->push_back(t);
            }
    } else {
        const int64_t T = ceil_div(u.m, BM);
        for (int64_t ti = 0; ti < T; ++ti)
            for (int64_t tj = 0; tj < ceil_div(T, 2); ++tj) {
                const int64_t bl = 2 * tj, br = 2 * tj + 1;
                const bool lneed = bl < T && bl >= ti;
                const bool rneed = br < T && br >= ti;
                if (!lneed && !rneed) continue;
                TileItem t{};
                t.unit = li;
                t.ti = static_cast<int16_t>(ti);
                t.tj = static_cast<int16_t>(tj);
                t.n_off = lneed ? 0 : 128;
                t.n_len = static_cast<int16_t>(128 * (int(lneed) + int(rneed)));
                t.k_blocks = kx;
                tsx->push_back(t);
                t.k_blocks = km;
                tsa->push_back(t);
            }
        for (int64_t ti = 0; ti < T; ++ti)
            for (int64_t tj = 0; tj < ceil_div(u.n, BN); ++tj) {
                TileItem t{};
                t.unit = li;
                t.ti = static_cast<int16_t>(ti);
                t.tj = static_cast<int16_t>(tj);
                t.n_off = 0;
                t.n_len = static_cast<int16_t>(
                    std::min<int64_t>(BN, align_up(u.n - tj * BN, 16)));
                t.k_blocks = km;
                tg->push_back(t);
            }
    }
}

int build_plan(muon_ctx* h, int mode, int nb, int64_t chunk_elems = 0) {
    Plan& P = h->plan;
    P = Plan();
    P.chunk_elems = chunk_elems;
    int rc = build_units(h, mode, nb, &P.units);
    if (rc) return rc;
    if (!h->ws) return fail(h, MUON_ERR_NO_WORKSPACE, "no workspace set (muon_set_workspace)");
    size_t min_b, full_b;
    sizes_for(P.units, &min_b, &full_b);
    if (h->ws_bytes < min_b)
        return fail(h, MUON_ERR_NO_WORKSPACE,
                    "workspace of " + std::to_string(h->ws_bytes) + " bytes is below the minimum " +
                        std::to_string(min_b));
    const size_t meta_b = meta_bound(P.units);
    P.scratch_off = align_up(HEADER_BYTES + meta_b, 1024);
    const size_t scratch = h->ws_bytes - P.scratch_off;
    if (!make_groups(P.units, scratch, &P.groups, chunk_elems))
        return fail(h, MUON_ERR_NO_WORKSPACE, "a unit does not fit the workspace");

    // host image of header + metadata
    std::vector<uint8_t> meta(P.scratch_off, 0);
    size_t off = HEADER_BYTES;
    char* ws = static_cast<char*>(h->ws);
    for (GroupDesc& g : P.groups) {
        const int nu = g.u1 - g.u0;
        // scratch layout of this group: inv | partials | buffers
        const size_t inv_off = P.scratch_off;
        int64_t tiles = 0;
        for (int i = g.u0; i < g.u1; ++i) tiles += P.units[i].ew_tiles;
        g.ew_tiles = tiles;
        const size_t part_off = align_up(inv_off + size_t(nu) * 4, 256);
        size_t buf_off = align_up(part_off + size_t(tiles) * 4 * EW_PARTIALS_PER_TILE, 1024);

        off = align_up(off, 256);
        g.tb_off = off;
        off += sizeof(int64_t) * (nu + 1);
        off = align_up(off, 256);
        g.ew_off = off;
        off += sizeof(EwUnit) * nu;
        off = align_up(off, 256);
        g.em_off = off;
        off += sizeof(EwMaps) * nu;
        // the TMA-fed momentum pass hides the per-tile unit lookups that the
        // plain pass stalls on when units are small (measured on GB300: the
        // Qwen3-30B-A3B block, 392 tiles per unit, 1.35 -> 1.23 ms); units
        // of thousands of tiles stream as fast or faster with plain loads
        // (the Kimi-K2 layer, 3600 per unit: 4.30 against 4.64 ms)
        g.ew_tma = h->ew_tma == 2 ||
                   (h->ew_tma == 1 && tiles < EWT_MAX_TILES_PER_UNIT * int64_t(nu));
        g.g_f32 = false;
        off = align_up(off, 256);
        g.ns_off = off;
        off += sizeof(NsUnit) * nu;
        g.shards = P.units[g.u0].shards;
        // tile counters of chained launches (a header, then every unit's),
        // zero in the uploaded image
        off = align_up(off, 256);
        g.rc_off = off;
        off += CNT_HEADER_WORDS * 4;
        for (int i = g.u0; i < g.u1; ++i) off += P.units[i].cnt_bytes;
        g.rc_bytes = off - g.rc_off;
        size_t rc_next = g.rc_off + CNT_HEADER_WORDS * 4;
        std::vector<TileItem> tsx, tsa, tg;
        int64_t tile_base = 0;
        for (int i = g.u0; i < g.u1; ++i) {
            const UnitDesc& u = P.units[i];
            const muon_param& pr = h->params[u.param];
            char* xb0 = ws + buf_off;
            char* xb1 = xb0 + u.x_bytes;
            char* ab = xb1 + u.x_bytes;
            char* bb = ab + u.mm_bytes;
            buf_off += u.buf_bytes;

            EwUnit e;
            std::memset(&e, 0, sizeof(e));
            e.w = static_cast<char*>(pr.w) + u.col_off * elem_size(pr.w_dtype);
            e.g = static_cast<const char*>(pr.g) + u.col_off * elem_size(pr.g_dtype);
            e.mom = pr.m + u.col_off;
            const bool have_w = u.param < int(h->exp_w.size()) && h->exp_w[u.param];
            const bool have_o = u.param < int(h->exp_o.size()) && h->exp_o[u.param];
            e.w_dbg = have_w ? h->exp_w[u.param] + u.col_off : nullptr;
            e.o_dbg = have_o ? static_cast<__nv_bfloat16*>(h->exp_o[u.param]) + u.col_off
                             : nullptr;
            e.x[0] = reinterpret_cast<__nv_bfloat16*>(xb0);
            e.x[1] = reinterpret_cast<__nv_bfloat16*>(xb1);
            e.ld_w = pr.ld_w;
            e.ld_g = pr.ld_g;
            e.ld_m = pr.ld_m;
            e.ld_dbg = pr.cols;
            e.rows = static_cast<int32_t>(u.rows);
            e.cols = static_cast<int32_t>(u.cols);
            e.m = u.m;
            e.n = u.n;
            e.ld_x = u.ld_x;
            e.w_dtype = pr.w_dtype;
            e.g_dtype = pr.g_dtype;
            e.transposed = u.transposed ? 1 : 0;
            auto al = [](const void* p, size_t a) {
                return (reinterpret_cast<uintptr_t>(p) % a) == 0;
            };
            const size_t wa = pr.w_dtype == MUON_F32 ? 16 : 8;
            const size_t ga = pr.g_dtype == MUON_F32 ? 16 : 8;
            e.vec_ok = (u.cols % 4 == 0) && (pr.ld_w % 4 == 0) && (pr.ld_g % 4 == 0) &&
                       (pr.ld_m % 4 == 0) && al(e.w, wa) && al(e.g, ga) && al(e.mom, 16);
            e.vec16 = al(e.w, 16) && ((pr.ld_w * elem_size(pr.w_dtype)) % 16 == 0);
            e.tiles_n = static_cast<int32_t>(ceil_div(u.n, EW_TILE));
            e.tile_base = tile_base;
            e.tile_count = u.ew_tiles;
            reinterpret_cast<int64_t*>(meta.data() + g.tb_off)[i - g.u0] = tile_base;
            reinterpret_cast<int64_t*>(meta.data() + g.tb_off)[i - g.u0 + 1] =
                tile_base + u.ew_tiles;
            e.shape_scale = u.scale;
            tile_base += u.ew_tiles;
            std::memcpy(meta.data() + g.ew_off + sizeof(EwUnit) * (i - g.u0), &e, sizeof(e));
            if (g.ew_tma) {
                EwMaps em;
                std::memset(&em, 0, sizeof(em));
                g.ew_tma = encode_ew_map(h, &em.m, e.mom, MUON_F32, u.rows, u.cols, pr.ld_m) &&
                           encode_ew_map(h, &em.g, e.g, pr.g_dtype, u.rows, u.cols, pr.ld_g);
                g.g_f32 = g.g_f32 || pr.g_dtype == MUON_F32;
                std::memcpy(meta.data() + g.em_off + sizeof(EwMaps) * (i - g.u0), &em,
                            sizeof(em));
            }

            NsUnit ns;
            std::memset(&ns, 0, sizeof(ns));
            if ((rc = encode_map(h, &ns.tm_x[0], xb0, u.n, u.m, u.ld_x))) return rc;
            if ((rc = encode_map(h, &ns.tm_x[1], xb1, u.n, u.m, u.ld_x))) return rc;
            if ((rc = encode_map(h, &ns.tm_a, ab, u.m, u.m, u.ld_mm))) return rc;
            if ((rc = encode_map(h, &ns.tm_b, bb, u.m, u.m, u.ld_mm))) return rc;
            if ((rc = encode_map(h, &ns.tk_x[0], xb0, u.n, u.m, u.ld_x, 64, 128))) return rc;
            if ((rc = encode_map(h, &ns.tk_x[1], xb1, u.n, u.m, u.ld_x, 64, 128))) return rc;
            if ((rc = encode_map(h, &ns.tk_a, ab, u.m, u.m, u.ld_mm, 64, 128))) return rc;
            if ((rc = encode_map(h, &ns.tk_b, bb, u.m, u.m, u.ld_mm, 64, 128))) return rc;
            if ((rc = encode_map(h, &ns.te_x[0], xb0, u.n, u.m, u.ld_x, 32))) return rc;
            if ((rc = encode_map(h, &ns.te_x[1], xb1, u.n, u.m, u.ld_x, 32))) return rc;
            if ((rc = encode_map(h, &ns.te_a, ab, u.m, u.m, u.ld_mm, 32))) return rc;
            if ((rc = encode_map(h, &ns.te_b, bb, u.m, u.m, u.ld_mm, 32))) return rc;
            {
                const bool ok = pr.w_dtype == MUON_BF16 && al(e.w, 16) && (pr.ld_w % 8 == 0);
                if (ok) {
                    if ((rc = encode_map(h, &ns.te_w, e.w, u.cols, u.rows, pr.ld_w, 32)))
                        return rc;
                } else {
                    g.w_tma = false;
                }
            }
            ns.x[0] = e.x[0];
            ns.x[1] = e.x[1];
            ns.a = reinterpret_cast<__nv_bfloat16*>(ab);
            if (h->dist) P.d_a16 = reinterpret_cast<__nv_bfloat16*>(ab);
            ns.b = reinterpret_cast<__nv_bfloat16*>(bb);
            ns.tile_cnt = reinterpret_cast<int32_t*>(ws + rc_next);
            rc_next += u.cnt_bytes;
            ns.m = u.m;
            ns.n = u.n;
            ns.ld_x = u.ld_x;
            ns.ld_mm = u.ld_mm;
            std::memcpy(meta.data() + g.ns_off + sizeof(NsUnit) * (i - g.u0), &ns, sizeof(ns));

            // tile lists
            append_unit_tiles(u, i - g.u0, h->pair, &tsx, &tsa, &tg);
            int64_t s, gg, us, ex;
            unit_tiles(u, h->pair, &s, &gg, &us, &ex);
            P.useful_flops_iter += us;
            P.executed_flops_iter += ex;
        }
        sort_tiles(&tsx);
        sort_tiles(&tsa);
        sort_tiles(&tg);
        const std::vector<TileItem> tsx0 = tsx, tsa0 = tsa, tg0 = tg;   // before put() reorders
        // separate launches: banded order within units, still costliest first
        for (std::vector<TileItem>* v : {&tsx, &tsa, &tg}) {
            band_tiles(v);
            sort_tiles(v);
        }
        const int64_t base_sx = static_cast<int64_t>(tsx.size());
        const int64_t base_g = static_cast<int64_t>(tg.size());
        auto put = [&](std::vector<TileItem>& v, size_t* o, int* n, size_t* oo, int* np) {
            *oo = 0;
            *np = 0;
            if (h->pair) {
                const int pairs = std::max(1, std::min(h->max_pairs,
                                                       static_cast<int>(v.size())));
                std::vector<int32_t> offs;
                lpt_schedule(&v, pairs, false, &offs);
                off = align_up(off, 256);
                *oo = off;
                *np = pairs;
                std::memcpy(meta.data() + off, offs.data(), offs.size() * sizeof(int32_t));
                off += offs.size() * sizeof(int32_t);
            }
            off = align_up(off, 256);
            *o = off;
            *n = static_cast<int>(v.size());
            if (!v.empty()) std::memcpy(meta.data() + off, v.data(), v.size() * sizeof(TileItem));
            off += v.size() * sizeof(TileItem);
        };
        put(tsx, &g.t_sx_off, &g.n_sx, &g.o_sx_off, &g.p_sx);
        put(tsa, &g.t_sa_off, &g.n_sa, &g.o_sa_off, &g.p_sa);
        put(tg, &g.t_g_off, &g.n_g, &g.o_g_off, &g.p_g);
        g.chain_ok = !h->dist && chain_eligible(h, g.shards, static_cast<int64_t>(tg0.size()));
        if (h->dist) {
            // a rank's slice: the first product's tiles by row block, in the
            // space a chained launch would use
            std::vector<TileItem> vd = tsx0;
            std::stable_sort(vd.begin(), vd.end(), [](const TileItem& x, const TileItem& y) {
                return x.ti != y.ti ? x.ti < y.ti : x.tj < y.tj;
            });
            const int T = static_cast<int>(ceil_div(P.units[g.u0].m, 256));
            g.d_band.assign(T + 1, static_cast<int>(vd.size()));
            for (int k = static_cast<int>(vd.size()) - 1; k >= 0; --k) g.d_band[vd[k].ti] = k;
            for (int b = T - 1; b >= 0; --b) g.d_band[b] = std::min(g.d_band[b], g.d_band[b + 1]);
            off = align_up(off, 256);
            g.t_d_off = off;
            std::memcpy(meta.data() + off, vd.data(), vd.size() * sizeof(TileItem));
            off += vd.size() * sizeof(TileItem);
        }
        if (g.chain_ok) {
            const int pairs = std::max(
                1, std::min(h->max_pairs,
                            static_cast<int>(tg0.size() + tsx0.size() + tsa0.size())));
            std::vector<TileItem> vc;
            std::vector<int32_t> offs, ends;
            lpt_schedule_chain(tsx0, tsa0, tg0, pairs, &vc, &offs, &ends);
            off = align_up(off, 256);
            g.o_c_off = off;
            g.p_c = pairs;
            std::memcpy(meta.data() + off, offs.data(), offs.size() * sizeof(int32_t));
            off += offs.size() * sizeof(int32_t);
            off = align_up(off, 256);
            g.e_c_off = off;
            std::memcpy(meta.data() + off, ends.data(), ends.size() * sizeof(int32_t));
            off += ends.size() * sizeof(int32_t);
            off = align_up(off, 256);
            g.t_c_off = off;
            g.n_c = static_cast<int>(vc.size());
            std::memcpy(meta.data() + off, vc.data(), vc.size() * sizeof(TileItem));
            off += vc.size() * sizeof(TileItem);
        }
        P.syrk_tiles += base_sx;
        P.gemm_tiles += base_g;
        P.ew_tiles += g.ew_tiles;
        if (off > P.scratch_off)
            return fail(h, MUON_ERR_STATE, "internal: metadata exceeds its bound");
        // stash scratch offsets in the group (reuse fields via locals below)
        (void)part_off;
    }
    // pageable source: the copy is staged before cudaMemcpyAsync returns,
    // so `meta` may go out of scope; stream order protects earlier steps
    cudaError_t e = cudaMemcpyAsync(h->ws, meta.data(), meta.size(),
                                    cudaMemcpyHostToDevice, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "metadata upload");
    P.mode = mode;
    P.nb = (mode == MUON_FULL) ? 1 : nb;
    P.ws = h->ws;
    P.ws_bytes = h->ws_bytes;
    P.valid = true;
    return MUON_OK;
}

cudaEvent_t pool_event(muon_ctx* h, size_t idx) {
    while (h->event_pool.size() <= idx) {
        cudaEvent_t ev;
        if (cudaEventCreate(&ev) != cudaSuccess) return nullptr;
        h->event_pool.push_back(ev);
    }
    return h->event_pool[idx];
}

}  // namespace

extern "C" {

int muon_create(muon_handle* out, int device, void* cuda_stream) {
    if (!out) return fail(nullptr, MUON_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    const char* cg = std::getenv("MUON_CTA_GROUP");
    const bool pair = !(cg && std::string(cg) == "1");
    const char* fz = std::getenv("MUON_FUSE");
    const bool fuse = !(fz && std::string(fz) == "0");
    const char* fu = std::getenv("MUON_FUSE_UPDATE");
    int fuse_update = 2;
    if (fu) fuse_update = std::atoi(fu);
    if (fuse_update < 0 || fuse_update > 2) fuse_update = 2;
    if (!fuse) fuse_update = 0;
    if (device == MUON_HOST_ONLY) {
        muon_ctx* h = new muon_ctx();
        h->device = MUON_HOST_ONLY;
        h->num_sms = 152;
        h->max_pairs = 76;
        h->pair = pair;
        *out = h;
        return MUON_OK;
    }
    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) return fail(nullptr, MUON_ERR_CUDA, cudaGetErrorString(e));
    if (device < 0 || device >= ndev)
        return fail(nullptr, MUON_ERR_INVALID_ARG, "device index out of range");
    DeviceGuard guard(device);
    muon_ctx* h = new muon_ctx();
    h->device = device;
    h->stream = static_cast<cudaStream_t>(cuda_stream);
    cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device);
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    if (major != 10 || minor != 3) {
        delete h;
        return fail(nullptr, MUON_ERR_UNSUPPORTED,
                    "libmuon is built for sm_103a (GB300); device has compute capability " +
                        std::to_string(major) + "." + std::to_string(minor));
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
        delete h;
        return fail(nullptr, MUON_ERR_CUDA, "cuTensorMapEncodeTiled not available");
    }
    h->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    h->pair = pair;
    h->fuse = fuse;
    h->fuse_update = fuse_update;
    if (const char* pd = std::getenv("MUON_PDL")) set_programmatic_launch(std::string(pd) != "0");
    if (const char* fs = std::getenv("MUON_FUSE_STAGES")) h->fuse_stages = std::string(fs) != "0";
    if (const char* cl = std::getenv("MUON_CHAIN_LAST")) h->chain_last = std::string(cl) != "0";
    if (const char* cn = std::getenv("MUON_CHAIN_MIN_TILES")) h->chain_min_tiles = std::atoi(cn);
    if (const char* cm = std::getenv("MUON_CHAIN_MAX_TILES")) {
        const int v = std::atoi(cm);
        if (v >= 0) h->chain_max_tiles = v;
    }
    if (const char* et = std::getenv("MUON_EW_TMA")) {
        const int v = std::atoi(et);
        if (v >= 0 && v <= 2) h->ew_tma = v;
    }
    if (const char* st = std::getenv("MUON_STAGES")) {
        const int v = std::atoi(st);
        if (v >= 4 && v <= 6) h->stages = v;
    }
    if (pair) {
        h->max_pairs = ns_pair_max_clusters();
        if (h->max_pairs < 1) {
            delete h;
            return fail(nullptr, MUON_ERR_CUDA, "no CTA pair fits on the device");
        }
    }
    if (const char* s = std::getenv("MUON_WAIT_LIMIT_MS")) {
        const long long ms = std::atoll(s);
        if (ms > 0) h->wait_limit_ns = static_cast<unsigned long long>(ms) * 1000000ull;
    }
    *out = h;
    return MUON_OK;
}

int muon_set_stream(muon_handle h, void* cuda_stream) {
    if (!h) return MUON_ERR_INVALID_ARG;
    h->stream = static_cast<cudaStream_t>(cuda_stream);
    return MUON_OK;
}

int muon_register_params(muon_handle h, int n, const muon_param* params) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (n < 1 || !params) return fail(h, MUON_ERR_INVALID_ARG, "need n >= 1 parameters");
    for (int i = 0; i < n; ++i) {
        const muon_param& p = params[i];
        const std::string who = "parameter " + std::to_string(i) + ": ";
        if (!p.w || !p.g || !p.m) return fail(h, MUON_ERR_INVALID_ARG, who + "NULL pointer");
        if (p.rows < 1 || p.cols < 1 || p.rows > MAX_DIM || p.cols > MAX_DIM)
            return fail(h, MUON_ERR_INVALID_ARG, who + "rows/cols out of range");
        if (p.ld_w < p.cols || p.ld_g < p.cols || p.ld_m < p.cols)
            return fail(h, MUON_ERR_INVALID_ARG, who + "leading dimension below cols");
        if ((p.w_dtype != MUON_F32 && p.w_dtype != MUON_BF16) ||
            (p.g_dtype != MUON_F32 && p.g_dtype != MUON_BF16))
            return fail(h, MUON_ERR_UNSUPPORTED, who + "dtype must be MUON_F32 or MUON_BF16");
        if (std::min(p.rows, p.cols) > MAX_SHORT)
            return fail(h, MUON_ERR_UNSUPPORTED, who + "short side above 32768");
    }
    h->params.assign(params, params + n);
    h->exp_w.clear();
    h->exp_o.clear();
    h->plan.valid = false;
    h->err.clear();
    return MUON_OK;
}

int muon_workspace_size(muon_handle h, int mode, int nb, size_t* min_bytes,
                        size_t* full_bytes) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (!min_bytes || !full_bytes) return fail(h, MUON_ERR_INVALID_ARG, "NULL output");
    if (h->params.empty()) return fail(h, MUON_ERR_STATE, "no parameters registered");
    std::vector<UnitDesc> units;
    int rc = build_units(h, mode, nb, &units);
    if (rc) return rc;
    sizes_for(units, min_bytes, full_bytes);
    return MUON_OK;
}

int muon_set_workspace(muon_handle h, void* dptr, size_t bytes) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (!dptr || bytes == 0) return fail(h, MUON_ERR_INVALID_ARG, "NULL or empty workspace");
    if (reinterpret_cast<uintptr_t>(dptr) % 1024 != 0)
        return fail(h, MUON_ERR_INVALID_ARG, "workspace must be 1024-byte aligned");
    h->ws = dptr;
    h->ws_bytes = bytes;
    h->plan.valid = false;
    return MUON_OK;
}

}  // extern "C"

namespace {

// muon_step_host's buffers: gradients in and weights out, per parameter.
struct HostIO {
    const void* const* g_host;
    void* const* w_host;
};

// Elements per group muon_step_host plans for: about 1/host_chunks of the
// registered set, at least 32 M elements (so that a chunk's copies stay long
// against the per-group launch overhead); 0 when no cut would result.
int64_t host_chunk_elems(const muon_ctx* h) {
    int64_t total = 0;
    for (const muon_param& p : h->params) total += p.rows * p.cols;
    const int64_t c = std::max<int64_t>(int64_t(32) << 20, total / std::max(1, h->host_chunks));
    return (h->params.size() > 1 && c < total) ? c : 0;
}

cudaEvent_t host_event(muon_ctx* h, size_t idx) {
    while (h->host_events.size() <= idx) {
        cudaEvent_t ev;
        if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        h->host_events.push_back(ev);
    }
    return h->host_events[idx];
}

int step_impl(muon_ctx* h, float lr, float beta, int nesterov, int ns_steps, float a, float b,
              float c, int mode, int nb, const HostIO* io) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (h->device == MUON_HOST_ONLY) return fail(h, MUON_ERR_STATE, "host-only handle");
    if (h->params.empty()) return fail(h, MUON_ERR_STATE, "no parameters registered");
    if (h->dist)
        return fail(h, MUON_ERR_STATE, "a rank's slice steps through the muon_dist_* phases");
    if (ns_steps < 1 || ns_steps > 64)
        return fail(h, MUON_ERR_INVALID_ARG, "ns_steps must be in 1..64");
    if (!std::isfinite(lr) || !std::isfinite(beta) || !std::isfinite(a) ||
        !std::isfinite(b) || !std::isfinite(c))
        return fail(h, MUON_ERR_INVALID_ARG, "non-finite hyper-parameter");
    if (mode != MUON_FULL && mode != MUON_BLOCKWISE && mode != MUON_DISTRIBUTED)
        return fail(h, MUON_ERR_INVALID_ARG,
                    "mode must be MUON_FULL, MUON_BLOCKWISE or MUON_DISTRIBUTED");
    if (mode != MUON_FULL && nb < 1) return fail(h, MUON_ERR_INVALID_ARG, "nb must be >= 1");
    DeviceGuard guard(h->device);
    const int want_nb = (mode == MUON_FULL) ? 1 : nb;
    Plan& P = h->plan;
    // muon_step runs any valid plan; muon_step_host wants one cut into
    // chunks (the same bits either way: groups do not change results)
    const int64_t want_chunk = io ? host_chunk_elems(h) : P.chunk_elems;
    // while the stream is captured into a CUDA graph: no plan build (its
    // table upload reads host memory that the graph would read again on
    // every replay) and no stage-timing events
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (h->stream && cudaStreamIsCapturing(h->stream, &cap) != cudaSuccess)
        return fail(h, MUON_ERR_CUDA, "stream capture query");
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    if (capturing && h->profiling)
        return fail(h, MUON_ERR_STATE, "stage profiling is not allowed while capturing");
    if (!P.valid || P.mode != mode || P.nb != want_nb || P.ws != h->ws ||
        P.ws_bytes != h->ws_bytes || (io && P.chunk_elems != want_chunk)) {
        if (capturing)
            return fail(h, MUON_ERR_STATE,
                        "the plan must be built before stream capture: run one step first");
        const int rc = build_plan(h, mode, nb, P.valid || io ? want_chunk : 0);
        if (rc) {
            P.valid = false;
            return rc;
        }
    }
    char* ws = static_cast<char*>(h->ws);
    int* err_word = reinterpret_cast<int*>(ws);
    // muon_step_host: parameter i's gradient goes in before the first group
    // holding one of its units, its weight comes out after the last
    const int ngroups = static_cast<int>(P.groups.size());
    std::vector<int> first_g, last_g;
    cudaEvent_t ev_start = nullptr, ev_end = nullptr;
    if (io) {
        if (!h->s_in &&
            cudaStreamCreateWithFlags(&h->s_in, cudaStreamNonBlocking) != cudaSuccess)
            return fail(h, MUON_ERR_CUDA, "copy stream create");
        if (!h->s_out &&
            cudaStreamCreateWithFlags(&h->s_out, cudaStreamNonBlocking) != cudaSuccess)
            return fail(h, MUON_ERR_CUDA, "copy stream create");
        ev_start = host_event(h, 0);
        ev_end = host_event(h, 1);
        if (!ev_start || !ev_end || !host_event(h, 1 + 2 * size_t(ngroups)))
            return fail(h, MUON_ERR_CUDA, "event create");
        first_g.assign(h->params.size(), -1);
        last_g.assign(h->params.size(), -1);
        for (int gi = 0; gi < ngroups; ++gi)
            for (int i = P.groups[gi].u0; i < P.groups[gi].u1; ++i) {
                const int prm = P.units[i].param;
                if (first_g[prm] < 0) first_g[prm] = gi;
                last_g[prm] = gi;
            }
        // gradients in, group by group, after everything queued so far
        cudaError_t e = cudaEventRecord(ev_start, h->stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_in, ev_start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_out, ev_start, 0);
        for (int gi = 0; gi < ngroups && e == cudaSuccess; ++gi) {
            for (size_t i = 0; i < h->params.size() && e == cudaSuccess; ++i) {
                if (first_g[i] != gi) continue;
                const muon_param& pr = h->params[i];
                const size_t es = elem_size(pr.g_dtype);
                e = cudaMemcpy2DAsync(const_cast<void*>(pr.g), size_t(pr.ld_g) * es,
                                      io->g_host[i], size_t(pr.cols) * es,
                                      size_t(pr.cols) * es, size_t(pr.rows),
                                      cudaMemcpyHostToDevice, h->s_in);
            }
            if (e == cudaSuccess) e = cudaEventRecord(h->host_events[2 + 2 * gi], h->s_in);
        }
        if (e != cudaSuccess) return cuda_fail(h, e, "gradient copy to the device");
    }
    h->launches.clear();
    size_t ev_idx = 0;
    int count = 0;
    auto begin = [&](int stage) -> bool {
        ++count;
        if (!h->profiling) return true;
        LaunchRec r;
        r.stage = stage;
        r.start = pool_event(h, ev_idx++);
        r.stop = pool_event(h, ev_idx++);
        if (!r.start || !r.stop) return false;
        cudaEventRecord(r.start, h->stream);
        h->launches.push_back(r);
        return true;
    };
    auto end = [&]() {
        if (h->profiling) cudaEventRecord(h->launches.back().stop, h->stream);
    };
    const int ew_grid_cap = h->num_sms * 8;
    for (int gi = 0; gi < ngroups; ++gi) {
        GroupDesc& g = P.groups[gi];
        if (io) {
            const cudaError_t we = cudaStreamWaitEvent(h->stream, h->host_events[2 + 2 * gi], 0);
            if (we != cudaSuccess) return cuda_fail(h, we, "wait for the gradient copies");
        }
        const int nu = g.u1 - g.u0;
        const size_t inv_off = P.scratch_off;
        const size_t part_off = align_up(inv_off + size_t(nu) * 4, 256);
        EwLaunch ew{};
        ew.units = reinterpret_cast<const EwUnit*>(ws + g.ew_off);
        ew.tile_base = reinterpret_cast<const int64_t*>(ws + g.tb_off);
        ew.num_units = nu;
        ew.num_tiles = g.ew_tiles;
        ew.partial = reinterpret_cast<float*>(ws + part_off);
        ew.inv_norm = reinterpret_cast<float*>(ws + inv_off);
        ew.beta = beta;
        ew.nesterov = nesterov ? 1 : 0;
        ew.lr = lr;
        ew.src = 0;
        ew.eps = NORM_EPS;
        ew.maps = g.ew_tma ? reinterpret_cast<const EwMaps*>(ws + g.em_off) : nullptr;
        ew.err = err_word;
        ew.wait_limit_ns = h->wait_limit_ns;
        // grid-stride over the tiles with the same number of tiles per block
        // (no part-empty last round)
        const int64_t ew_per_block =
            std::max<int64_t>(1, ceil_div(g.ew_tiles, int64_t(ew_grid_cap)));
        const int ew_grid = static_cast<int>(ceil_div(g.ew_tiles, ew_per_block));
        const bool fused = h->pair && h->fuse;
        ew.write_x = fused ? 1 : 0;
        cudaError_t e;
        if (!begin(ST_MOMENTUM)) return fail(h, MUON_ERR_CUDA, "event create");
        if (ew.maps)   // persistent CTAs, TMA-fed ring
            e = launch_ew_momentum_tma(
                ew,
                static_cast<int>(std::min<int64_t>(g.ew_tiles,
                                                   int64_t(EWT_CTAS_PER_SM) * h->num_sms)),
                g.g_f32, h->stream);
        else
            e = launch_ew_momentum(ew, ew_grid, h->stream);
        end();
        if (e != cudaSuccess) return cuda_fail(h, e, "momentum launch");
        if (!begin(ST_NORM)) return fail(h, MUON_ERR_CUDA, "event create");
        e = launch_ew_norm(ew, h->stream);
        end();
        if (e != cudaSuccess) return cuda_fail(h, e, "norm launch");
        if (!fused) {
            if (!begin(ST_NORMALISE)) return fail(h, MUON_ERR_CUDA, "event create");
            e = launch_ew_normalise(ew, ew_grid, h->stream);
            end();
            if (e != cudaSuccess) return cuda_fail(h, e, "normalise launch");
        }
        NsLaunch L{};
        L.units = reinterpret_cast<const NsUnit*>(ws + g.ns_off);
        L.a = a;
        L.b = b;
        L.c = c;
        L.wait_limit_ns = h->wait_limit_ns;
        L.err = err_word;
        L.inv_norm = ew.inv_norm;
        L.ew = ew.units;
        L.lr = lr;
        int cur = 0;
        // chained groups: one launch holds every product of iterations
        // 1 .. ns_steps, the last X update too when the weight update folds
        // into it through TMA (and no validation exports are registered: the
        // chained kernel does not write them); else that one runs alone
        const bool chain = g.chain_ok;
        const bool exports_on =
            std::any_of(h->exp_w.begin(), h->exp_w.end(), [](float* q) { return q != nullptr; }) ||
            std::any_of(h->exp_o.begin(), h->exp_o.end(), [](void* q) { return q != nullptr; });
        const bool chain_last = chain && h->chain_last && fused && h->fuse_update == 2 &&
                                g.w_tma && !exports_on;
        if (chain) {
            L.src = 0;
            L.first = fused ? 1 : 0;
            L.last = 0;
            L.chain_last = chain_last ? 1 : 0;
            L.tiles = reinterpret_cast<const TileItem*>(ws + g.t_c_off);
            L.num_tiles = g.n_c;
            L.pair_off = reinterpret_cast<const int32_t*>(ws + g.o_c_off);
            L.pair_end_last = reinterpret_cast<const int32_t*>(ws + g.e_c_off);
            L.iters = ns_steps;
            L.ep_x = 0;
            L.ep_a = h->debug_chain_skew;
            L.ep_b = 0;
            L.shards = 1;
            L.cnt_block = reinterpret_cast<int32_t*>(ws + g.rc_off);
            L.cnt_words = static_cast<int32_t>(g.rc_bytes / 4);
            if (!begin(ST_CHAIN)) return fail(h, MUON_ERR_CUDA, "event create");
            e = launch_ns_pair(OP_CHAIN, L, g.p_c, h->stages, h->stream);
            end();
            if (e != cudaSuccess) {
                P.valid = false;              // rebuilt (and re-uploaded) next step
                return cuda_fail(h, e, "chained launch");
            }
            cur = (ns_steps - 1) & 1;
            if (chain_last) cur ^= 1;
        }
        const int s_begin = chain_last ? ns_steps : chain ? ns_steps - 1 : 0;
        for (int s = s_begin; s < ns_steps; ++s) {
            L.src = cur;
            L.first = (fused && s == 0) ? 1 : 0;
            const bool last = s == ns_steps - 1;
            const bool upd_regs = fused && h->fuse_update == 1;
            const bool upd_tma = fused && h->fuse_update == 2 && g.w_tma;
            L.last = (last && (upd_regs || upd_tma)) ? 1 : 0;
            struct Q { NsOp op; size_t off; int n; int st; size_t oo; int np; };
            Q seq[3];
            int nq = 0;
            if (!chain) {
                seq[nq++] = {OP_SYRK_X, g.t_sx_off, g.n_sx, ST_SYRK1, g.o_sx_off, g.p_sx};
                seq[nq++] = {OP_SYRK_A, g.t_sa_off, g.n_sa, ST_SYRK2, g.o_sa_off, g.p_sa};
            }
            seq[nq++] = {OP_GEMM_BX, g.t_g_off, g.n_g, ST_GEMM, g.o_g_off, g.p_g};
            for (int qi = 0; qi < nq; ++qi) {
                const Q& q = seq[qi];
                L.tiles = reinterpret_cast<const TileItem*>(ws + q.off);
                L.num_tiles = q.n;
                L.pair_off = h->pair ? reinterpret_cast<const int32_t*>(ws + q.oo) : nullptr;
                L.pair_end_last = nullptr;
                L.iters = 1;
                L.chain_last = 0;
                L.shards = g.shards;
                if (!begin(q.st)) return fail(h, MUON_ERR_CUDA, "event create");
                if (h->pair && q.op == OP_GEMM_BX && L.last && upd_tma)
                    e = launch_ns_pair_update(L, q.np, exports_on, h->stream);
                else if (h->pair)
                    e = launch_ns_pair(q.op, L, q.np, h->stages, h->stream);
                else
                    e = launch_ns(q.op, L, std::min(q.n, h->num_sms), h->stream);
                end();
                if (e != cudaSuccess) {
                    P.valid = false;          // rebuilt (and re-uploaded) next step
                    return cuda_fail(h, e, "tensor-core stage launch");
                }
            }
            cur ^= 1;
        }
        const bool update_folded =
            fused && (h->fuse_update == 1 || (h->fuse_update == 2 && g.w_tma));
        if (!update_folded) {
            ew.src = cur;
            if (!begin(ST_UPDATE)) return fail(h, MUON_ERR_CUDA, "event create");
            e = launch_ew_update(ew, ew_grid, h->stream);
            end();
            if (e != cudaSuccess) return cuda_fail(h, e, "update launch");
        }
        if (io) {
            // this group's weights out, once its update is done
            cudaEvent_t done = h->host_events[3 + 2 * gi];
            e = cudaEventRecord(done, h->stream);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(h->s_out, done, 0);
            for (size_t i = 0; i < h->params.size() && e == cudaSuccess; ++i) {
                if (last_g[i] != gi || !io->w_host[i]) continue;
                const muon_param& pr = h->params[i];
                const size_t es = elem_size(pr.w_dtype);
                e = cudaMemcpy2DAsync(io->w_host[i], size_t(pr.cols) * es, pr.w,
                                      size_t(pr.ld_w) * es, size_t(pr.cols) * es,
                                      size_t(pr.rows), cudaMemcpyDeviceToHost, h->s_out);
            }
            if (e != cudaSuccess) return cuda_fail(h, e, "weight copy to the host");
        }
    }
    if (io) {
        // the handle's stream (and so muon_sync) covers the copies
        cudaError_t e = cudaEventRecord(ev_end, h->s_out);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(h->stream, ev_end, 0);
        if (e != cudaSuccess) return cuda_fail(h, e, "join of the copy streams");
    }
    h->last_launch_count = count;
    return MUON_OK;
}

// Distributed mode across ranks: checks shared by the phases, and the plan
// (full mode, the one slice) built on first use.
int dist_prepare(muon_ctx* h) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (h->device == MUON_HOST_ONLY) return fail(h, MUON_ERR_STATE, "host-only handle");
    if (!h->dist) return fail(h, MUON_ERR_STATE, "muon_dist_configure has not been called");
    if (h->params.size() != 1)
        return fail(h, MUON_ERR_STATE, "a rank's slice handle holds exactly one parameter");
    Plan& P = h->plan;
    if (!P.valid || P.mode != MUON_FULL || P.nb != 1 || P.ws != h->ws ||
        P.ws_bytes != h->ws_bytes) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (h->stream && cudaStreamIsCapturing(h->stream, &cap) != cudaSuccess)
            return fail(h, MUON_ERR_CUDA, "stream capture query");
        if (cap != cudaStreamCaptureStatusNone)
            return fail(h, MUON_ERR_STATE, "the plan must be built before stream capture");
        const int rc = build_plan(h, MUON_FULL, 1, 0);
        if (rc) {
            P.valid = false;
            return rc;
        }
        h->dist_ready = false;
    }
    if (P.groups.size() != 1)
        return fail(h, MUON_ERR_STATE, "internal: a rank's slice plan has one group");
    return MUON_OK;
}

// The NsLaunch fields every phase's tensor-core launch shares.
NsLaunch dist_launch(muon_ctx* h, float ca, float cb, float cc, float lr) {
    Plan& P = h->plan;
    const GroupDesc& g = P.groups[0];
    char* ws = static_cast<char*>(h->ws);
    NsLaunch L{};
    L.units = reinterpret_cast<const NsUnit*>(ws + g.ns_off);
    L.a = ca;
    L.b = cb;
    L.c = cc;
    L.wait_limit_ns = h->wait_limit_ns;
    L.err = reinterpret_cast<int*>(ws);
    L.inv_norm = reinterpret_cast<float*>(ws + P.scratch_off);
    L.ew = reinterpret_cast<const EwUnit*>(ws + g.ew_off);
    L.lr = lr;
    L.iters = 1;
    L.shards = 1;
    return L;
}

// The element-wise launch fields of the slice's group.
EwLaunch dist_ew(muon_ctx* h) {
    Plan& P = h->plan;
    const GroupDesc& g = P.groups[0];
    char* ws = static_cast<char*>(h->ws);
    EwLaunch ew{};
    ew.units = reinterpret_cast<const EwUnit*>(ws + g.ew_off);
    ew.tile_base = reinterpret_cast<const int64_t*>(ws + g.tb_off);
    ew.num_units = 1;
    ew.num_tiles = g.ew_tiles;
    ew.partial = reinterpret_cast<float*>(ws + align_up(P.scratch_off + 4, 256));
    ew.inv_norm = reinterpret_cast<float*>(ws + P.scratch_off);
    ew.eps = NORM_EPS;
    ew.err = reinterpret_cast<int*>(ws);
    ew.wait_limit_ns = h->wait_limit_ns;
    return ew;
}

int dist_ew_grid(muon_ctx* h) {
    const int64_t tiles = h->plan.groups[0].ew_tiles;
    const int64_t per_block = std::max<int64_t>(1, ceil_div(tiles, int64_t(h->num_sms) * 8));
    return static_cast<int>(ceil_div(tiles, per_block));
}

int dist_momentum(muon_ctx* h, float beta, int nesterov, double* sumsq) {
    if (int rc = dist_prepare(h)) return rc;
    if (!sumsq) return fail(h, MUON_ERR_INVALID_ARG, "sumsq is null");
    if (!std::isfinite(beta)) return fail(h, MUON_ERR_INVALID_ARG, "non-finite beta");
    DeviceGuard guard(h->device);
    const GroupDesc& g = h->plan.groups[0];
    char* ws = static_cast<char*>(h->ws);
    EwLaunch ew = dist_ew(h);
    ew.beta = beta;
    ew.nesterov = nesterov ? 1 : 0;
    ew.src = 0;
    ew.maps = g.ew_tma ? reinterpret_cast<const EwMaps*>(ws + g.em_off) : nullptr;
    ew.write_x = 1;
    cudaError_t e;
    if (ew.maps)
        e = launch_ew_momentum_tma(
            ew, static_cast<int>(std::min<int64_t>(g.ew_tiles, int64_t(EWT_CTAS_PER_SM) *
                                                                   h->num_sms)),
            g.g_f32, h->stream);
    else
        e = launch_ew_momentum(ew, dist_ew_grid(h), h->stream);
    if (e == cudaSuccess) e = launch_ew_sumsq(ew, sumsq, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "momentum phase launch");
    h->dist_ready = true;
    h->dist_grams = 0;
    h->dist_cur = 0;
    return MUON_OK;
}

int dist_gram(muon_ctx* h, float* a, int64_t lda, int band_begin, int band_end) {
    if (int rc = dist_prepare(h)) return rc;
    if (!h->dist_ready)
        return fail(h, MUON_ERR_STATE, "muon_dist_gram before muon_dist_momentum");
    const Plan& P = h->plan;
    const GroupDesc& g = P.groups[0];
    const int m = P.units[g.u0].m;
    const int T = static_cast<int>(g.d_band.size()) - 1;
    if (!a || lda < m) return fail(h, MUON_ERR_INVALID_ARG, "a is null or lda < m");
    if (band_end < 0) band_end = T;
    if (band_begin < 0 || band_begin > band_end || band_end > T)
        return fail(h, MUON_ERR_INVALID_ARG, "band outside the 256-row blocks of A");
    DeviceGuard guard(h->device);
    const int t0 = g.d_band[band_begin], t1 = g.d_band[band_end];
    h->dist_grams += 1;
    if (t1 == t0) return MUON_OK;
    NsLaunch L = dist_launch(h, 0.f, 0.f, 0.f, 0.f);
    char* ws = static_cast<char*>(h->ws);
    L.tiles = reinterpret_cast<const TileItem*>(ws + g.t_d_off) + t0;
    L.num_tiles = t1 - t0;
    L.pair_off = nullptr;
    L.src = h->dist_cur;
    L.first = 0;                 // scaled after the group's sum
    L.last = 0;
    L.a32 = a;
    L.lda32 = lda;
    const int pairs = std::max(1, std::min(h->max_pairs, t1 - t0));
    const cudaError_t e = launch_ns_pair_gram32(L, pairs, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "first product launch");
    return MUON_OK;
}

int dist_update(muon_ctx* h, const float* a, int64_t lda, int first, int last,
                const double* sumsq_total, float lr, float ca, float cb, float cc) {
    if (int rc = dist_prepare(h)) return rc;
    if (!h->dist_ready || h->dist_grams == 0)
        return fail(h, MUON_ERR_STATE, "muon_dist_update before this iteration's muon_dist_gram");
    if (!std::isfinite(lr) || !std::isfinite(ca) || !std::isfinite(cb) || !std::isfinite(cc))
        return fail(h, MUON_ERR_INVALID_ARG, "non-finite hyper-parameter");
    Plan& P = h->plan;
    const GroupDesc& g = P.groups[0];
    const UnitDesc& u = P.units[g.u0];
    if (!a || lda < u.m) return fail(h, MUON_ERR_INVALID_ARG, "a is null or lda < m");
    if (first && !sumsq_total) return fail(h, MUON_ERR_INVALID_ARG, "sumsq_total is null");
    DeviceGuard guard(h->device);
    char* ws = static_cast<char*>(h->ws);
    DistLaunch d{};
    d.a32 = a;
    d.lda32 = lda;
    d.a16 = P.d_a16;
    d.ld_mm = u.ld_mm;
    d.m = u.m;
    d.first = first ? 1 : 0;
    d.sumsq_total = sumsq_total;
    d.inv_norm = reinterpret_cast<float*>(ws + P.scratch_off);
    d.eps = NORM_EPS;
    cudaError_t e = launch_dist_convert(d, h->num_sms * 4, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "conversion launch");
    NsLaunch L = dist_launch(h, ca, cb, cc, lr);
    L.src = h->dist_cur;
    L.first = 0;
    L.last = 0;
    // the second product: B' = b A + c A A + a I
    L.tiles = reinterpret_cast<const TileItem*>(ws + g.t_sa_off);
    L.num_tiles = g.n_sa;
    L.pair_off = reinterpret_cast<const int32_t*>(ws + g.o_sa_off);
    e = launch_ns_pair(OP_SYRK_A, L, g.p_sa, h->stages, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "second product launch");
    // the X update, scaled by inv in iteration 1, with the weight update
    // folded in on the last iteration where the weights allow it
    const bool upd_regs = last && h->fuse_update == 1;
    const bool upd_tma = last && h->fuse_update == 2 && g.w_tma;
    L.first = first ? 1 : 0;
    L.last = (upd_regs || upd_tma) ? 1 : 0;
    L.tiles = reinterpret_cast<const TileItem*>(ws + g.t_g_off);
    L.num_tiles = g.n_g;
    L.pair_off = reinterpret_cast<const int32_t*>(ws + g.o_g_off);
    const bool exports_on =
        std::any_of(h->exp_w.begin(), h->exp_w.end(), [](float* q) { return q != nullptr; }) ||
        std::any_of(h->exp_o.begin(), h->exp_o.end(), [](void* q) { return q != nullptr; });
    if (upd_tma)
        e = launch_ns_pair_update(L, g.p_g, exports_on, h->stream);
    else
        e = launch_ns_pair(OP_GEMM_BX, L, g.p_g, h->stages, h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "X update launch");
    h->dist_cur ^= 1;
    h->dist_grams = 0;
    if (last && !L.last) {
        // the weight update as a pass of its own (fp32 or unaligned weights)
        EwLaunch ew = dist_ew(h);
        ew.lr = lr;
        ew.src = h->dist_cur;
        e = launch_ew_update(ew, dist_ew_grid(h), h->stream);
        if (e != cudaSuccess) return cuda_fail(h, e, "update launch");
    }
    if (last) h->dist_ready = false;
    return MUON_OK;
}

}  // namespace

extern "C" {

int muon_step(muon_handle h, float lr, float beta, int nesterov, int ns_steps,
              float a, float b, float c, int mode, int nb) {
    return step_impl(h, lr, beta, nesterov, ns_steps, a, b, c, mode, nb, nullptr);
}

int muon_step_host(muon_handle h, int n, const void* const* g_host, void* const* w_host,
                   float lr, float beta, int nesterov, int ns_steps, float a, float b, float c,
                   int mode, int nb) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (h->device == MUON_HOST_ONLY) return fail(h, MUON_ERR_STATE, "host-only handle");
    if (n != static_cast<int>(h->params.size()))
        return fail(h, MUON_ERR_INVALID_ARG,
                    "n=" + std::to_string(n) + " but " + std::to_string(h->params.size()) +
                        " parameters are registered");
    if (!g_host || !w_host) return fail(h, MUON_ERR_INVALID_ARG, "NULL host pointer array");
    for (int i = 0; i < n; ++i)
        if (!g_host[i])
            return fail(h, MUON_ERR_INVALID_ARG, "g_host[" + std::to_string(i) + "] is NULL");
    const HostIO io{g_host, w_host};
    return step_impl(h, lr, beta, nesterov, ns_steps, a, b, c, mode, nb, &io);
}

int muon_dist_configure(muon_handle h, int transposed, float shape_scale) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (!std::isfinite(shape_scale) || shape_scale < 1.f)
        return fail(h, MUON_ERR_INVALID_ARG, "shape_scale must be finite and >= 1");
    h->dist = true;
    h->dist_transposed = transposed ? 1 : 0;
    h->dist_scale = shape_scale;
    h->dist_ready = false;
    h->plan.valid = false;
    return MUON_OK;
}

int muon_dist_momentum(muon_handle h, float beta, int nesterov, double* sumsq) {
    return dist_momentum(h, beta, nesterov, sumsq);
}

int muon_dist_gram(muon_handle h, float* a, int64_t lda, int band_begin, int band_end) {
    return dist_gram(h, a, lda, band_begin, band_end);
}

int muon_dist_update(muon_handle h, const float* a, int64_t lda, int first, int last,
                     const double* sumsq_total, float lr, float ca, float cb, float cc) {
    return dist_update(h, a, lda, first, last, sumsq_total, lr, ca, cb, cc);
}

int muon_sync(muon_handle h) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (h->device == MUON_HOST_ONLY) return fail(h, MUON_ERR_STATE, "host-only handle");
    DeviceGuard guard(h->device);
    cudaError_t e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "stream synchronize");
    if (h->ws) {
        int word = 0;
        e = cudaMemcpy(&word, h->ws, sizeof(int), cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(h, e, "error word read");
        if (word != 0) {
            const int zero = 0;
            cudaMemcpy(h->ws, &zero, sizeof(int), cudaMemcpyHostToDevice);
            h->plan.valid = false;    // the next step rebuilds and re-uploads it
            if (word == DEV_ERR_TIMEOUT)
                return fail(h, MUON_ERR_TIMEOUT, "a bounded wait on the GPU ran out");
            return fail(h, MUON_ERR_CUDA, "device error word " + std::to_string(word));
        }
    }
    return MUON_OK;
}

int muon_destroy(muon_handle h) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (h->device != MUON_HOST_ONLY) {
        DeviceGuard guard(h->device);
        for (cudaEvent_t ev : h->event_pool) cudaEventDestroy(ev);
        for (cudaEvent_t ev : h->host_events) cudaEventDestroy(ev);
        if (h->s_in) cudaStreamDestroy(h->s_in);
        if (h->s_out) cudaStreamDestroy(h->s_out);
    }
    delete h;
    return MUON_OK;
}

const char* muon_last_error(muon_handle h) {
    return h ? h->err.c_str() : g_create_err.c_str();
}

int muon_set_profiling(muon_handle h, int on) {
    if (!h) return MUON_ERR_INVALID_ARG;
    h->profiling = on != 0;
    return MUON_OK;
}

int muon_stage_times(muon_handle h, float* ms, int* launches, int n) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (h->device == MUON_HOST_ONLY) return fail(h, MUON_ERR_STATE, "host-only handle");
    if (!ms || n < 0) return fail(h, MUON_ERR_INVALID_ARG, "NULL output");
    DeviceGuard guard(h->device);
    const int k = std::min(n, MUON_N_STAGES);
    for (int i = 0; i < k; ++i) {
        ms[i] = 0.f;
        if (launches) launches[i] = 0;
    }
    for (const LaunchRec& r : h->launches) {
        float t = 0.f;
        cudaError_t e = cudaEventSynchronize(r.stop);
        if (e != cudaSuccess) return cuda_fail(h, e, "event synchronize");
        e = cudaEventElapsedTime(&t, r.start, r.stop);
        if (e != cudaSuccess) return cuda_fail(h, e, "event elapsed time");
        if (r.stage < k) {
            ms[r.stage] += t;
            if (launches) launches[r.stage] += 1;
        }
    }
    return k;
}

int muon_last_launch_count(muon_handle h) { return h ? h->last_launch_count : 0; }

int muon_debug_set_exports(muon_handle h, int n, float* const* w_f32, void* const* o_bf16) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (n < 0 || n > static_cast<int>(h->params.size()))
        return fail(h, MUON_ERR_INVALID_ARG, "n out of range");
    h->exp_w.assign(h->params.size(), nullptr);
    h->exp_o.assign(h->params.size(), nullptr);
    for (int i = 0; i < n; ++i) {
        if (w_f32) h->exp_w[i] = w_f32[i];
        if (o_bf16) h->exp_o[i] = o_bf16[i];
    }
    h->plan.valid = false;
    return MUON_OK;
}

int muon_debug_set_chain_test(muon_handle h, int skew_rounds) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (skew_rounds < 0 || skew_rounds > (1 << 20))
        return fail(h, MUON_ERR_INVALID_ARG, "skew_rounds must be in 0..2^20");
    h->debug_chain_skew = skew_rounds;
    return MUON_OK;
}

int muon_debug_wait_timeout(muon_handle h, int* err_word, int limit_ms) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (h->device == MUON_HOST_ONLY) return fail(h, MUON_ERR_STATE, "host-only handle");
    if (!err_word || limit_ms < 1 || limit_ms > 10000)
        return fail(h, MUON_ERR_INVALID_ARG, "need an error word and 1 <= limit_ms <= 10000");
    DeviceGuard guard(h->device);
    cudaError_t e = cudaMemsetAsync(err_word, 0, sizeof(int), h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "error word clear");
    e = launch_wait_timeout_check(err_word, static_cast<unsigned long long>(limit_ms) * 1000000ull,
                                  h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "wait check launch");
    e = cudaStreamSynchronize(h->stream);
    if (e != cudaSuccess) return cuda_fail(h, e, "wait check sync");
    int word = 0;
    e = cudaMemcpy(&word, err_word, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(h, e, "wait check read");
    if (word == DEV_ERR_TIMEOUT) return fail(h, MUON_ERR_TIMEOUT, "bounded wait ran out (expected)");
    return fail(h, MUON_ERR_STATE, "the bounded wait did not report a timeout");
}

int muon_get_plan_info(muon_handle h, int mode, int nb, muon_plan_info* out) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (!out) return fail(h, MUON_ERR_INVALID_ARG, "NULL output");
    if (h->params.empty()) return fail(h, MUON_ERR_STATE, "no parameters registered");
    std::vector<UnitDesc> units;
    int rc = build_units(h, mode, nb, &units);
    if (rc) return rc;
    std::memset(out, 0, sizeof(*out));
    out->units = static_cast<int64_t>(units.size());
    for (const UnitDesc& u : units) {
        int64_t s, g, us, ex;
        unit_tiles(u, h->pair, &s, &g, &us, &ex);
        out->syrk_tiles += s;
        out->gemm_tiles += g;
        out->ew_tiles += u.ew_tiles;
        out->useful_flops += us;
        out->executed_flops += ex;
    }
    std::vector<GroupDesc> groups;
    size_t min_b, full_b;
    sizes_for(units, &min_b, &full_b);
    if (h->ws && h->ws_bytes >= min_b) {
        const size_t scratch = h->ws_bytes - align_up(HEADER_BYTES + meta_bound(units), 1024);
        make_groups(units, scratch, &groups);
    } else {
        GroupDesc g;
        g.u0 = 0;
        g.u1 = static_cast<int>(units.size());
        groups.push_back(g);
    }
    out->groups = static_cast<int64_t>(groups.size());
    for (const GroupDesc& g : groups) {
        int64_t gemm = 0;
        for (int i = g.u0; i < g.u1; ++i) {
            int64_t s, gg, us, ex;
            unit_tiles(units[i], h->pair, &s, &gg, &us, &ex);
            gemm += gg;
        }
        if (chain_eligible(h, units[g.u0].shards, gemm)) ++out->chained_groups;
    }
    return MUON_OK;
}

int muon_debug_check_chain_schedule(muon_handle h, int mode, int nb) {
    if (!h) return MUON_ERR_INVALID_ARG;
    if (h->params.empty()) return fail(h, MUON_ERR_STATE, "no parameters registered");
    if (!h->pair) return MUON_OK;                 // chains run on CTA pairs only
    std::vector<UnitDesc> units;
    int rc = build_units(h, mode, nb, &units);
    if (rc) return rc;
    std::vector<GroupDesc> groups;
    size_t min_b, full_b;
    sizes_for(units, &min_b, &full_b);
    if (h->ws && h->ws_bytes >= min_b) {
        make_groups(units, h->ws_bytes - align_up(HEADER_BYTES + meta_bound(units), 1024),
                    &groups);
    } else {
        GroupDesc g;
        g.u0 = 0;
        g.u1 = static_cast<int>(units.size());
        groups.push_back(g);
    }
    for (size_t gi = 0; gi < groups.size(); ++gi) {
        const GroupDesc& g = groups[gi];
        std::vector<TileItem> tsx, tsa, tg;
        for (int i = g.u0; i < g.u1; ++i)
            append_unit_tiles(units[i], i - g.u0, true, &tsx, &tsa, &tg);
        sort_tiles(&tsx);
        sort_tiles(&tsa);
        sort_tiles(&tg);
        const int pairs = std::max(
            1, std::min(h->max_pairs, static_cast<int>(tsx.size() + tsa.size() + tg.size())));
        std::vector<TileItem> v;
        std::vector<int32_t> offs, ends;
        lpt_schedule_chain(tsx, tsa, tg, pairs, &v, &offs, &ends);
        const std::string where = "group " + std::to_string(gi) + ": ";
        // every tile of the three products exactly once
        using Key = std::tuple<int, int32_t, int, int, int>;
        std::map<Key, int> want;
        for (const TileItem& t : tsx) ++want[Key{OP_SYRK_X, t.unit, t.ti, t.tj, t.n_off}];
        for (const TileItem& t : tsa) ++want[Key{OP_SYRK_A, t.unit, t.ti, t.tj, t.n_off}];
        for (const TileItem& t : tg) ++want[Key{OP_GEMM_BX, t.unit, t.ti, t.tj, t.n_off}];
        for (const TileItem& t : v)
            --want[Key{t.flags & TILE_OP_MASK, t.unit, t.ti, t.tj, t.n_off}];
        for (const auto& kv : want)
            if (kv.second != 0)
                return fail(h, MUON_ERR_STATE, where + "a tile is missing or repeated");
        if (static_cast<int>(offs.size()) != pairs + 1 || offs[0] != 0 ||
            offs[pairs] != static_cast<int32_t>(v.size()) ||
            static_cast<int>(ends.size()) != pairs)
            return fail(h, MUON_ERR_STATE, where + "pair offsets do not cover the list");
        for (int p = 0; p < pairs; ++p) {
            if (offs[p] > offs[p + 1])
                return fail(h, MUON_ERR_STATE, where + "pair offsets decrease");
            // stage order: first products, second products, X updates
            int prev = OP_SYRK_X, first_gemm = offs[p + 1];
            for (int k = offs[p]; k < offs[p + 1]; ++k) {
                const int op = v[k].flags & TILE_OP_MASK;
                if (op < prev)
                    return fail(h, MUON_ERR_STATE,
                                where + "pair " + std::to_string(p) + " is not in stage order");
                if (op == OP_GEMM_BX && first_gemm == offs[p + 1]) first_gemm = k;
                prev = op;
            }
            if (ends[p] != first_gemm)
                return fail(h, MUON_ERR_STATE,
                            where + "pair " + std::to_string(p) + ": wrong end before X updates");
        }
    }
    return MUON_OK;
}

}  // extern "C"

namespace muon {

// One full-mode step of one matrix with the plan tables and intermediates in
// a caller-supplied device region (used by the no-workspace entry point).
// Same planner, kernels and launch sequence as muon_step, so the results are
// bit-identical to a handle-based step of the same matrix.  Needs the region
// to hold the matrix in a single group; allocates nothing.
int step_in_region(const muon_param& prm, float lr, float beta, int nesterov, int ns_steps,
                   float a, float b, float c, void* region, size_t region_bytes,
                   cudaStream_t stream, std::string* err) {
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) {
        *err = cudaGetErrorString(ce);
        return MUON_ERR_CUDA;
    }
    muon_handle h = nullptr;
    int rc = muon_create(&h, dev, stream);
    if (rc) {
        *err = muon_last_error(nullptr);
        return rc;
    }
    rc = muon_register_params(h, 1, &prm);
    size_t mn = 0, full = 0;
    if (!rc) rc = muon_workspace_size(h, MUON_FULL, 1, &mn, &full);
    if (!rc && full > region_bytes) {
        rc = fail(h, MUON_ERR_UNSUPPORTED,
                  "matrix " + std::to_string(prm.rows) + "x" + std::to_string(prm.cols) +
                      " needs " + std::to_string(full) +
                      " bytes of scratch; the fixed scratch of muon_step_noalloc holds " +
                      std::to_string(region_bytes) +
                      " bytes (use muon_step with a workspace instead)");
    }
    if (!rc) rc = muon_set_workspace(h, region, region_bytes);
    if (!rc) rc = muon_step(h, lr, beta, nesterov, ns_steps, a, b, c, MUON_FULL, 1);
    if (rc) *err = h->err;
    muon_destroy(h);
    return rc;
}

}  // namespace muon
