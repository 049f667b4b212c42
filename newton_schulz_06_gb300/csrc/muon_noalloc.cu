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
// device.  Its device address is resolved at that first call (set-up, with
// the device current) and cached; it is resolved again only if the device's
// context was replaced since (after cudaDeviceReset the module is loaded
// anew, possibly elsewhere).  Every call shares the array, so two calls
// whose GPU work overlaps (on two streams, or from two threads) race and
// corrupt each other's results.  The
// planner, kernels and launch sequence are the ones muon_step uses (the
// tables are rebuilt and uploaded on every call), so a matrix gets the same
// bits from either entry point.
#include <cstdio>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

#include "../../include/muon.h"
#include "muon_internal.h"

namespace muon {
int step_in_region(const muon_param& prm, float lr, float beta, int nesterov, int ns_steps,
                   float a, float b, float c, void* region, size_t region_bytes,
                   cudaStream_t stream, std::string* err);
}  // namespace muon

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(32) << 20;
constexpr int NA_MAX_DEVICES = 64;

// 1 KiB of slack so that a 1024-byte aligned window of the full stated size
// always fits (the planner wants 1024-byte aligned buffers).
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES + 1024];

struct NoallocDevice {
    bool ready = false;
    void* scratch = nullptr;        // device address of g_noalloc_scratch
    unsigned long long ctx_id = 0;  // the context it was resolved in
};

NoallocDevice g_dev[NA_MAX_DEVICES];
std::mutex g_dev_mutex;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

int na_fail(char* err, size_t len, int code, const std::string& msg) {
    if (err && len) std::snprintf(err, len, "%s", msg.c_str());
    return code;
}

// The unique id of the calling thread's current context (0 if none is
// current yet).  Driver functions are resolved once through the runtime.
bool current_ctx_id(unsigned long long* id) {
    *id = 0;
    if (!g_ctx_current || !g_ctx_id) {
        void* f0 = nullptr;
        void* f1 = nullptr;
        cudaDriverEntryPointQueryResult q0, q1;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 4000, cudaEnableDefault,
                                             &q0) != cudaSuccess ||
            q0 != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault,
                                             &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || !f0 || !f1)
            return false;
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f0);
        g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f1);
    }
    CUcontext c = nullptr;
    if (g_ctx_current(&c) != CUDA_SUCCESS) return false;
    if (!c) return true;
    return g_ctx_id(c, id) == CUDA_SUCCESS;
}

// Set-up, once per device with that device current: resolve the array's
// device address (in host code its name is only a stand-in, not a device
// address).  Resolved again only if the device's context was replaced.
int na_setup(int dev, void** out, char* err, size_t len) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    NoallocDevice& d = g_dev[dev];
    unsigned long long id = 0;
    if (!current_ctx_id(&id))
        return na_fail(err, len, MUON_ERR_CUDA, "cannot query the current CUDA context");
    if (!d.ready || id == 0 || id != d.ctx_id) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return na_fail(err, len, MUON_ERR_CUDA,
                           std::string("cudaGetSymbolAddress(scratch): ") +
                               cudaGetErrorString(e));
        const uintptr_t base = (reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023);
        d.scratch = reinterpret_cast<void*>(base);
        // the lookup made the device's primary context current if it was not
        if (!current_ctx_id(&id))
            return na_fail(err, len, MUON_ERR_CUDA, "cannot query the current CUDA context");
        d.ctx_id = id;
        d.ready = id != 0;
    }
    *out = d.scratch;
    return MUON_OK;
}

}  // namespace

extern "C" MUON_API int muon_step_noalloc(const muon_param* prm, float lr, float beta,
                                          int nesterov, int ns_steps, float a, float b,
                                          float c, void* cuda_stream, char* err,
                                          size_t err_len) {
    if (err && err_len) err[0] = '\0';
    if (!prm) return na_fail(err, err_len, MUON_ERR_INVALID_ARG, "param is NULL");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return na_fail(err, err_len, MUON_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= NA_MAX_DEVICES)
        return na_fail(err, err_len, MUON_ERR_UNSUPPORTED, "device index above 63");
    void* region = nullptr;
    int rc = na_setup(dev, &region, err, err_len);
    if (rc) return rc;
    std::string msg;
    rc = muon::step_in_region(*prm, lr, beta, nesterov, ns_steps, a, b, c, region,
                              NOALLOC_SCRATCH_BYTES, static_cast<cudaStream_t>(cuda_stream),
                              &msg);
    if (rc) return na_fail(err, err_len, rc, msg);
    return MUON_OK;
}
