// Status word, version and error strings of libspecverify.
#include <mutex>

#include "common.cuh"

// One status word per device that loads the library: kernels OR SPEC_DEV_*
// bits into it; spec_get_status reads and clears it.
__device__ int g_spec_status;

namespace sv {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int *g_status_addr[kMaxDevices];
int g_sms[kMaxDevices];
}  // namespace

int *status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_spec_status) != cudaSuccess) return nullptr;
        g_status_addr[dev] = static_cast<int *>(p);
    }
    return g_status_addr[dev];
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
