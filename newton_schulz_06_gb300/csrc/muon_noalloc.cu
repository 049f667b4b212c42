// muon_step_noalloc: one Muon step on one matrix with every intermediate in
// a fixed, file-scope device array instead of a caller-provided workspace.
//
// Who needs this: callers that cannot call cudaMalloc themselves or hand the
// library a buffer.  Examples are a plugin whose host application owns all
// device memory through its own pool and does not expose it, a caching
// allocator that has already reserved the device so a raw cudaMalloc fails
// or fragments it, and a latency-critical loop that cannot pay for
// cudaMalloc's implicit device synchronisation.  They pass W, G and M as
// usual; the plan tables, partial sums, the two iterates X and the m x m
// matrices A and B live in `g_noalloc_scratch` below.
//
// The array is NOALLOC_SCRATCH_BYTES (32 MiB).  It exists once per device
// that loads this code and stays until the process exits; with CUDA's lazy
// module loading that happens at the first call of this entry point on the
// device.  Every call shares it, so two calls whose GPU work overlaps (on two
// streams, or from two threads) race and corrupt each other's results.  The
// kernels are the same ones muon_step launches.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/muon.h"
#include "muon_internal.h"

using namespace muon;

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(32) << 20;
constexpr size_t NA_HEADER = 256;
constexpr int NA_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

struct NoallocDevice {
    bool ready = false;
    char* scratch = nullptr;   // device address of g_noalloc_scratch
    int num_sms = 0;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};

NoallocDevice g_dev[NA_MAX_DEVICES];
std::mutex g_dev_mutex;

size_t na_align(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t na_ceil(int64_t a, int64_t b) { return (a + b - 1) / b; }

int na_fail(char* err, size_t len, int code, const std::string& msg) {
    if (err && len) {
        std::snprintf(err, len, "%s", msg.c_str());
    }
    return code;
}

// Once per device, with that device current: resolve the array's device
// address (the host-side name is only a stand-in) and the TMA encoder.
int na_setup(int dev, NoallocDevice** out, char* err, size_t len) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    NoallocDevice& d = g_dev[dev];
    if (!d.ready) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return na_fail(err, len, MUON_ERR_CUDA,
                           std::string("cudaGetSymbolAddress(scratch): ") +
                               cudaGetErrorString(e));
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return na_fail(err, len, MUON_ERR_UNSUPPORTED,
                           "libmuon is built for sm_103a (GB300)");
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return na_fail(err, len, MUON_ERR_CUDA, "cuTensorMapEncodeTiled not available");
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        d.scratch = static_cast<char*>(p);
        d.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        d.ready = true;
    }
    *out = &d;
    return MUON_OK;
}

bool na_map(NoallocDevice* d, CUtensorMap* tm, void* base, int64_t inner,
            int64_t outer, int64_t ld) {
    cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
    cuuint32_t box[2] = {64, 64};
    cuuint32_t es[2] = {1, 1};
    return d->encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                     es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void na_sort(std::vector<TileItem>* v) {
    std::stable_sort(v->begin(), v->end(), [](const TileItem& a, const TileItem& b) {
        return int64_t(a.k_blocks) * a.n_len > int64_t(b.k_blocks) * b.n_len;
    });
}

}  // namespace

extern "C" MUON_API int muon_step_noalloc(const muon_param* prm, float lr, float beta,
                                          int nesterov, int ns_steps, float a, float b,
                                          float c, void* cuda_stream, char* err,
                                          size_t err_len) {
    if (err && err_len) err[0] = '\0';
    if (!prm) return na_fail(err, err_len, MUON_ERR_INVALID_ARG, "param is NULL");
    const muon_param& p = *prm;
    if (!p.w || !p.g || !p.m)
        return na_fail(err, err_len, MUON_ERR_INVALID_ARG, "NULL w, g or m");
    if (p.rows < 1 || p.cols < 1 || p.ld_w < p.cols || p.ld_g < p.cols || p.ld_m < p.cols)
        return na_fail(err, err_len, MUON_ERR_INVALID_ARG, "bad rows, cols or leading dimension");
    if ((p.w_dtype != MUON_F32 && p.w_dtype != MUON_BF16) ||
        (p.g_dtype != MUON_F32 && p.g_dtype != MUON_BF16))
        return na_fail(err, err_len, MUON_ERR_UNSUPPORTED, "dtype must be MUON_F32 or MUON_BF16");
    if (ns_steps < 1 || ns_steps > 64)
        return na_fail(err, err_len, MUON_ERR_INVALID_ARG, "ns_steps must be in 1..64");

    // sizes of one unit (the whole matrix, short side first)
    const bool transposed = p.rows > p.cols;
    const int64_t m = transposed ? p.cols : p.rows;
    const int64_t n = transposed ? p.rows : p.cols;
    if (m > 32768 || n > (int64_t(1) << 20))
        return na_fail(err, err_len, MUON_ERR_UNSUPPORTED, "matrix too large");
    const int64_t ld_x = int64_t(na_align(size_t(n), 64));
    const int64_t ld_mm = int64_t(na_align(size_t(m), 64));
    const size_t x_bytes = na_align(size_t(m) * ld_x * 2, 1024);
    const size_t mm_bytes = na_align(size_t(m) * ld_mm * 2, 1024);
    const int64_t T = na_ceil(m, BM);
    const int64_t ew_tiles = na_ceil(m, EW_TILE) * na_ceil(n, EW_TILE);

    std::vector<TileItem> tsx, tsa, tg;
    const int kx = int(na_ceil(n, BK)), km = int(na_ceil(m, BK));
    for (int64_t ti = 0; ti < T; ++ti)
        for (int64_t tj = 0; tj < na_ceil(T, 2); ++tj) {
            const bool l = 2 * tj < T && 2 * tj >= ti;
            const bool r = 2 * tj + 1 < T && 2 * tj + 1 >= ti;
            if (!l && !r) continue;
            TileItem t;
            t.unit = 0;
            t.ti = int16_t(ti);
            t.tj = int16_t(tj);
            t.n_off = l ? 0 : 128;
            t.n_len = int16_t(128 * (int(l) + int(r)));
            t.k_blocks = kx;
            tsx.push_back(t);
            t.k_blocks = km;
            tsa.push_back(t);
        }
    for (int64_t ti = 0; ti < T; ++ti)
        for (int64_t tj = 0; tj < na_ceil(n, BN); ++tj) {
            TileItem t;
            t.unit = 0;
            t.ti = int16_t(ti);
            t.tj = int16_t(tj);
            t.n_off = 0;
            t.n_len = int16_t(std::min<int64_t>(BN, int64_t(na_align(size_t(n - tj * BN), 16))));
            t.k_blocks = km;
            tg.push_back(t);
        }
    na_sort(&tsx);
    na_sort(&tsa);
    na_sort(&tg);

    // layout inside the fixed array
    size_t off = NA_HEADER;
    const size_t ew_off = na_align(off, 256);
    off = ew_off + sizeof(EwUnit);
    const size_t ns_off = na_align(off, 256);
    off = ns_off + sizeof(NsUnit);
    const size_t sx_off = na_align(off, 256);
    off = sx_off + tsx.size() * sizeof(TileItem);
    const size_t sa_off = na_align(off, 256);
    off = sa_off + tsa.size() * sizeof(TileItem);
    const size_t g_off = na_align(off, 256);
    off = g_off + tg.size() * sizeof(TileItem);
    const size_t meta_bytes = off;
    const size_t inv_off = na_align(off, 256);
    const size_t part_off = na_align(inv_off + 4, 256);
    const size_t x0_off = na_align(part_off + size_t(ew_tiles) * 4, 1024);
    const size_t x1_off = x0_off + x_bytes;
    const size_t a_off = x1_off + x_bytes;
    const size_t b_off = a_off + mm_bytes;
    const size_t need = b_off + mm_bytes;
    if (need > NOALLOC_SCRATCH_BYTES)
        return na_fail(err, err_len, MUON_ERR_UNSUPPORTED,
                       "matrix " + std::to_string(p.rows) + "x" + std::to_string(p.cols) +
                           " needs " + std::to_string(need) +
                           " bytes of scratch; the fixed scratch of muon_step_noalloc holds " +
                           std::to_string(NOALLOC_SCRATCH_BYTES) +
                           " bytes (use muon_step with a workspace instead)");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return na_fail(err, err_len, MUON_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= NA_MAX_DEVICES)
        return na_fail(err, err_len, MUON_ERR_UNSUPPORTED, "device index above 63");
    NoallocDevice* d = nullptr;
    int rc = na_setup(dev, &d, err, err_len);
    if (rc) return rc;
    char* base = d->scratch;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);

    // host image of header + tables (the header's error word starts at 0)
    std::vector<unsigned char> meta(meta_bytes, 0);
    EwUnit eu;
    std::memset(&eu, 0, sizeof(eu));
    eu.w = p.w;
    eu.g = p.g;
    eu.mom = p.m;
    eu.x[0] = reinterpret_cast<__nv_bfloat16*>(base + x0_off);
    eu.x[1] = reinterpret_cast<__nv_bfloat16*>(base + x1_off);
    eu.ld_w = p.ld_w;
    eu.ld_g = p.ld_g;
    eu.ld_m = p.ld_m;
    eu.ld_dbg = p.cols;
    eu.rows = int32_t(p.rows);
    eu.cols = int32_t(p.cols);
    eu.m = int32_t(m);
    eu.n = int32_t(n);
    eu.ld_x = int32_t(ld_x);
    eu.w_dtype = p.w_dtype;
    eu.g_dtype = p.g_dtype;
    eu.transposed = transposed ? 1 : 0;
    auto al = [](const void* q, size_t k) { return reinterpret_cast<uintptr_t>(q) % k == 0; };
    eu.vec_ok = (p.cols % 4 == 0) && (p.ld_w % 4 == 0) && (p.ld_g % 4 == 0) &&
                (p.ld_m % 4 == 0) && al(p.w, p.w_dtype == MUON_F32 ? 16 : 8) &&
                al(p.g, p.g_dtype == MUON_F32 ? 16 : 8) && al(p.m, 16);
    eu.tiles_n = int32_t(na_ceil(n, EW_TILE));
    eu.tile_base = 0;
    eu.tile_count = ew_tiles;
    eu.shape_scale = float(std::sqrt(std::max(1.0, double(p.rows) / double(p.cols))));
    std::memcpy(meta.data() + ew_off, &eu, sizeof(eu));

    NsUnit nu;
    std::memset(&nu, 0, sizeof(nu));
    if (!na_map(d, &nu.tm_x[0], base + x0_off, n, m, ld_x) ||
        !na_map(d, &nu.tm_x[1], base + x1_off, n, m, ld_x) ||
        !na_map(d, &nu.tm_a, base + a_off, m, m, ld_mm) ||
        !na_map(d, &nu.tm_b, base + b_off, m, m, ld_mm))
        return na_fail(err, err_len, MUON_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    nu.x[0] = eu.x[0];
    nu.x[1] = eu.x[1];
    nu.a = reinterpret_cast<__nv_bfloat16*>(base + a_off);
    nu.b = reinterpret_cast<__nv_bfloat16*>(base + b_off);
    nu.m = int32_t(m);
    nu.n = int32_t(n);
    nu.ld_x = int32_t(ld_x);
    nu.ld_mm = int32_t(ld_mm);
    std::memcpy(meta.data() + ns_off, &nu, sizeof(nu));
    std::memcpy(meta.data() + sx_off, tsx.data(), tsx.size() * sizeof(TileItem));
    std::memcpy(meta.data() + sa_off, tsa.data(), tsa.size() * sizeof(TileItem));
    std::memcpy(meta.data() + g_off, tg.data(), tg.size() * sizeof(TileItem));
    // pageable source: the copy is staged before the call returns
    e = cudaMemcpyAsync(base, meta.data(), meta.size(), cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return na_fail(err, err_len, MUON_ERR_CUDA,
                       std::string("table upload: ") + cudaGetErrorString(e));

    EwLaunch ew;
    ew.units = reinterpret_cast<const EwUnit*>(base + ew_off);
    ew.num_units = 1;
    ew.num_tiles = ew_tiles;
    ew.partial = reinterpret_cast<float*>(base + part_off);
    ew.inv_norm = reinterpret_cast<float*>(base + inv_off);
    ew.beta = beta;
    ew.nesterov = nesterov ? 1 : 0;
    ew.lr = lr;
    ew.src = 0;
    ew.eps = 1e-7f;
    const int ew_grid = int(std::min<int64_t>(ew_tiles, int64_t(d->num_sms) * 8));
    if ((e = launch_ew_momentum(ew, ew_grid, stream)) != cudaSuccess ||
        (e = launch_ew_norm(ew, stream)) != cudaSuccess ||
        (e = launch_ew_normalise(ew, ew_grid, stream)) != cudaSuccess)
        return na_fail(err, err_len, MUON_ERR_CUDA, cudaGetErrorString(e));
    NsLaunch L;
    L.units = reinterpret_cast<const NsUnit*>(base + ns_off);
    L.a = a;
    L.b = b;
    L.c = c;
    L.wait_limit_ns = 2000000000ull;
    L.err = reinterpret_cast<int*>(base);
    int cur = 0;
    for (int s = 0; s < ns_steps; ++s) {
        L.src = cur;
        const struct { NsOp op; size_t off; size_t n; } seq[3] = {
            {OP_SYRK_X, sx_off, tsx.size()}, {OP_SYRK_A, sa_off, tsa.size()},
            {OP_GEMM_BX, g_off, tg.size()}};
        for (const auto& q : seq) {
            L.tiles = reinterpret_cast<const TileItem*>(base + q.off);
            L.num_tiles = int32_t(q.n);
            e = launch_ns(q.op, L, std::min(int(q.n), d->num_sms), stream);
            if (e != cudaSuccess)
                return na_fail(err, err_len, MUON_ERR_CUDA, cudaGetErrorString(e));
        }
        cur ^= 1;
    }
    ew.src = cur;
    if ((e = launch_ew_update(ew, ew_grid, stream)) != cudaSuccess)
        return na_fail(err, err_len, MUON_ERR_CUDA, cudaGetErrorString(e));
    return MUON_OK;
}
