// spec_verify_attn_noalloc: spec_verify_attn for callers that cannot
// allocate device memory.
//
// Some callers of this library are not in a position to hand it a workspace:
// a serving engine that has carved all of the GPU's memory into its own
// KV-cache pool up front and allows no further allocation, or a plugin hook
// whose host framework owns the device memory and forbids allocating while
// it runs (cudaMalloc may also synchronise the whole device, which such
// paths must avoid).  For them this entry point runs the same attention with
// its split partials in a fixed array that is part of the library itself.
//
// The scratch is a file-scope __device__ array of SPEC_NOALLOC_SCRATCH_BYTES:
// every GPU on which the library's kernels are loaded holds it until the
// process exits.  Host code only sees a stand-in symbol for it, so its device
// address is resolved with cudaGetSymbolAddress, once per device, with that
// device current, on the first call made on that device.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device.
spec_status_t scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SPEC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SPEC_OK;
}

}  // namespace

extern "C" spec_status_t spec_verify_attn_noalloc(const spec_attn_desc *attn, const void *q,
                                                  const spec_kv_desc *cache, const void *kb,
                                                  const void *vb, const void *soft_k,
                                                  const void *soft_v, const int32_t *seq_len,
                                                  const uint32_t *vis, const uint8_t *row_flags,
                                                  void *o, float *lse, void *stream) {
    size_t need = 0;
    spec_status_t st = spec_verify_attn_workspace_size(attn, cache, &need);
    if (st != SPEC_OK) return st;
    if (need > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_CAPACITY;
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != SPEC_OK) return st;
    // The attention writes every partial it later reads, so the scratch
    // needs no clearing between calls.
    return spec_verify_attn(attn, q, cache, kb, vb, soft_k, soft_v, seq_len, vis, row_flags, o,
                            lse, scratch, (size_t)SPEC_NOALLOC_SCRATCH_BYTES, stream);
}
