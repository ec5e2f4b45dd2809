// Status word, version, error strings and per-device host state of
// libspecverify.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

// One status word per device that loads the library: kernels OR SPEC_DEV_*
// bits into it; spec_get_status reads and clears it.
__device__ int g_spec_status;

namespace sv {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];

// Default pipeline wait limit (~1 s of SM clock), as kTimeoutCycles.
constexpr long long kDefaultWaitCycles = 2000000000ll;
std::atomic<long long> g_wait_cycles{kDefaultWaitCycles};

// Kernels whose dynamic shared-memory limit has been raised, per device and
// context (the attribute belongs to the device current when it is set).
struct SmemAttr {
    const void *func;
    int dev;
    void *ctx;
};
constexpr int kMaxSmemAttrs = 256;
SmemAttr g_smem_attrs[kMaxSmemAttrs];
int g_n_smem_attrs = 0;
}  // namespace

void *current_context() {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    });
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return reinterpret_cast<void *>(c);
}

spec_status_t symbol_address(DeviceSymbolCache &cache, const void *symbol, void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
    if (dev < 0 || dev >= DeviceSymbolCache::kDevices) return SPEC_ERR_UNSUPPORTED;
    // (before the runtime has made a context current this is NULL, and the
    // next call resolves the address once more)
    void *ctx = current_context();
    std::lock_guard<std::mutex> lk(cache.mu);
    if (!cache.addr[dev] || cache.ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return SPEC_ERR_CUDA;
        cache.addr[dev] = p;
        cache.ctx[dev] = ctx;
    }
    *out = cache.addr[dev];
    return SPEC_OK;
}

int *status_ptr() {
    static DeviceSymbolCache cache;
    void *p = nullptr;
    if (symbol_address(cache, reinterpret_cast<const void *>(&g_spec_status), &p) != SPEC_OK)
        return nullptr;
    return static_cast<int *>(p);
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        g_sms[dev] = n;
    }
    return g_sms[dev];
}

long long wait_limit() { return g_wait_cycles.load(std::memory_order_relaxed); }

spec_status_t set_smem_limit(const void *func, size_t bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
    void *ctx = current_context();
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_n_smem_attrs; ++i)
        if (g_smem_attrs[i].func == func && g_smem_attrs[i].dev == dev && g_smem_attrs[i].ctx == ctx)
            return SPEC_OK;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess)
        return SPEC_ERR_CUDA;
    // a full table only means the attribute is set again on later calls
    if (g_n_smem_attrs < kMaxSmemAttrs) g_smem_attrs[g_n_smem_attrs++] = SmemAttr{func, dev, ctx};
    return SPEC_OK;
}

}  // namespace sv

extern "C" int spec_version(void) { return SPECVERIFY_VERSION; }

extern "C" const char *spec_status_string(spec_status_t s) {
    switch (s) {
        case SPEC_OK: return "ok";
        case SPEC_ERR_INVALID_ARG: return "invalid argument";
        case SPEC_ERR_UNSUPPORTED: return "unsupported dtype or shape";
        case SPEC_ERR_BAD_TREE: return "bad tree";
        case SPEC_ERR_CAPACITY: return "capacity exceeded";
        case SPEC_ERR_CUDA: return "CUDA runtime error";
        case SPEC_ERR_DEVICE: return "device-detected error (see status bits)";
        default: return "unknown status";
    }
}

extern "C" long long spec_set_wait_limit(long long cycles) {
    const long long v = cycles < 0 ? sv::kDefaultWaitCycles : cycles;
    return sv::g_wait_cycles.exchange(v);
}

extern "C" spec_status_t spec_get_status(void *stream, int32_t *out) {
    if (!out) return SPEC_ERR_INVALID_ARG;
    cudaStream_t s = sv::as_stream(stream);
    int *addr = sv::status_ptr();
    if (!addr) return SPEC_ERR_CUDA;
    int host = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
    if (cudaMemcpyAsync(&host, addr, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
    if (host != 0) {
        if (cudaMemsetAsync(addr, 0, sizeof(int), s) != cudaSuccess) return SPEC_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
    }
    *out = host;
    return host ? SPEC_ERR_DEVICE : SPEC_OK;
}
