// rowops_online_softmax_noalloc: the split-row online softmax for callers that
// cannot allocate device memory.
//
// Some callers only ever hold the input and output buffers: a plugin that a
// host framework calls with device pointers but no allocator or workspace
// hook, or code on a latency-critical path where a cudaMalloc (which can
// synchronise the device) is not acceptable. For them the chunk partials live
// in a fixed array of device memory that belongs to the library itself, so the
// call needs nothing but x, y and the shape.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds these kNoallocScratchBytes until the process exits. On the host
// its name is only a stand-in for the symbol, not a device address, so the
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) and that pointer is what the kernels receive.
#include <cstdlib>
#include <mutex>
#include <vector>

#include "online_softmax_kernels.cuh"
#include "rowops.h"
#include "rowops_launch.h"

namespace rowops {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(1) << 20;  // 1 MiB: 256-byte header + partials
constexpr int64_t kNoallocMinChunk = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct NoallocDevice {
    int device;
    unsigned long long ctx;  // the context the address belongs to (current_context_id)
    void* scratch;  // device address of g_noalloc_scratch on this device
    int num_sms;
    int max_smem_optin;
};

std::mutex g_noalloc_mu;
std::vector<NoallocDevice> g_noalloc_devices;

// Look up (once per device and context, with that device current) the device
// address of the scratch array and the SM count. A new context on the device
// (after cudaDeviceReset) has a new id, so the address is looked up again:
// the array of a context that is gone is never handed to a kernel.
cudaError_t noalloc_device(int dev, NoallocDevice* out) {
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    for (const auto& d : g_noalloc_devices)
        if (d.device == dev && d.ctx == ctx && ctx != 0) {
            *out = d;
            return cudaSuccess;
        }
    NoallocDevice d{dev, 0, nullptr, 0, 0};
    cudaError_t e = cudaGetSymbolAddress(&d.scratch, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    d.ctx = current_context_id();  // (the symbol lookup made a context current if none was)
    bool replaced = false;
    for (auto& old : g_noalloc_devices)
        if (old.device == dev) {
            old = d;
            replaced = true;
        }
    if (!replaced) g_noalloc_devices.push_back(d);
    *out = d;
    return cudaSuccess;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

rowops_status_t noalloc_check(const void* x, const void* y, int64_t M, int64_t N, int64_t ld,
                              rowops_dtype_t dt, int64_t chunk) {
    if ((dt != ROWOPS_F32 && dt != ROWOPS_BF16) || M < 0 || N < 1 || ld < N) return ROWOPS_ERR_INVALID_VALUE;
    if (N >= (int64_t(1) << 31)) return ROWOPS_ERR_UNSUPPORTED;
    if (chunk != 0 && (chunk < kNoallocMinChunk || chunk > (int64_t(1) << 30) || chunk % 16 != 0))
        return ROWOPS_ERR_INVALID_VALUE;
    if (M == 0) return ROWOPS_OK;
    if (!x || !y) return ROWOPS_ERR_INVALID_VALUE;
    const int es = dt == ROWOPS_F32 ? 4 : 2;
    if (!is_aligned(x, es) || !is_aligned(y, es)) return ROWOPS_ERR_INVALID_VALUE;
    const int64_t lim = INT64_MAX / es - N;
    if (M - 1 > lim / ld) return ROWOPS_ERR_UNSUPPORTED;
    if (x != y) {
        const uintptr_t span = uintptr_t(((M - 1) * ld + N) * es);
        const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(y);
        if (a < b + span && b < a + span) return ROWOPS_ERR_INVALID_VALUE;
    }
    return ROWOPS_OK;
}

}  // namespace
}  // namespace rowops

using namespace rowops;

extern "C" rowops_status_t rowops_online_softmax_noalloc(const void* x, void* y, int64_t M, int64_t N,
                                                         int64_t ld, rowops_dtype_t dtype, int64_t chunk,
                                                         cudaStream_t stream) {
    rowops_status_t st = noalloc_check(x, y, M, N, ld, dtype, chunk);
    if (st != ROWOPS_OK || M == 0) return st;
    const int64_t max_partials = int64_t((kNoallocScratchBytes - kWorkspaceHeader) / 8);
    const int64_t n16 = (N + 15) / 16 * 16;
    if (chunk != 0) {  // an explicit chunk fixes the partial count: reject before any CUDA call
        const int64_t c = chunk > n16 ? (n16 < kNoallocMinChunk ? kNoallocMinChunk : n16) : chunk;
        if ((N + c - 1) / c > max_partials / M) return ROWOPS_ERR_WORKSPACE;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return ROWOPS_ERR_CUDA;
    }
    NoallocDevice nd;
    if (noalloc_device(dev, &nd) != cudaSuccess) {
        cudaGetLastError();
        return ROWOPS_ERR_CUDA;
    }
    const int es = dtype == ROWOPS_F32 ? 4 : 2;
    // the same chunk choice as rowops_online_softmax
    if (chunk == 0) {
        chunk = split_step_cols(es);
        while (chunk > kNoallocMinChunk && M * ((N + chunk - 1) / chunk) < int64_t(4) * nd.num_sms) chunk /= 2;
    }
    if (chunk > n16) chunk = n16 < kNoallocMinChunk ? kNoallocMinChunk : n16;
    const int64_t nchunks = (N + chunk - 1) / chunk;
    // the whole problem's partials must fit the built-in scratch
    if (nchunks > max_partials / M) return ROWOPS_ERR_WORKSPACE;
    LaunchCfg cfg;
    cfg.stream = stream;
    cfg.device = dev;
    cfg.ctx = nd.ctx;
    cfg.num_sms = nd.num_sms;
    cfg.max_smem_optin = nd.max_smem_optin;
    cfg.ctas_per_sm = 0;
    cfg.dev_error = nullptr;  // the split-row kernels have no device-side waits
    cfg.cooperative = false;
    cfg.persist_lookahead = 0;
    cfg.persist_l2 = false;
    cfg.persist_prefetch = 0;
    cfg.wait_ns = 2000000000ull;
    cfg.stall_row = -1;
    // Nothing in the scratch has to start at zero: the first kernel writes the
    // status word and every partial before the second kernel reads them.
    SplitLaunch fn = dtype == ROWOPS_F32 ? split_softmax_f32() : split_softmax_bf16();
    const cudaError_t e = fn(x, y, M, N, ld, chunk, nchunks, nd.scratch, cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return ROWOPS_ERR_CUDA;
    }
    return ROWOPS_OK;
}
