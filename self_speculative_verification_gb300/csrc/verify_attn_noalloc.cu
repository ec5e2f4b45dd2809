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
// The scratch is a file-scope __device__ array of SPEC_NOALLOC_SCRATCH_BYTES.
// Host code only sees a stand-in symbol for it, so its device address is
// looked up with cudaGetSymbolAddress with the device current: on the first
// call made on each device, and again when that device's context has
// changed (after a cudaDeviceReset, say).  Under lazy module loading (the
// CUDA default) that first lookup is also what loads the module holding the
// array, so the 64 MiB are taken from the device then, not when the library
// is opened: a caller must make its first call on each device before it
// reserves the rest of that device's memory (and before any stream capture).
// From then on the array stays on the device until the process exits.
#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

sv::DeviceSymbolCache g_scratch;

}  // namespace

extern "C" spec_status_t spec_verify_attn_noalloc(const spec_attn_desc *attn, const void *q,
                                                  const spec_kv_desc *cache, const void *kb,
                                                  const void *vb, const void *soft_k,
                                                  const void *soft_v, const int32_t *seq_len,
                                                  const uint32_t *vis, const uint8_t *row_flags,
                                                  void *o, float *lse, void *stream) {
    // the address first, so that any call (even one rejected below) does the
    // per-device set-up
    void *scratch = nullptr;
    spec_status_t st =
        sv::symbol_address(g_scratch, reinterpret_cast<const void *>(g_attn_scratch), &scratch);
    if (st != SPEC_OK) return st;
    size_t need = 0;
    st = spec_verify_attn_workspace_size(attn, cache, &need);
    if (st != SPEC_OK) return st;
    if (need > (size_t)SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_CAPACITY;
    // The attention writes every partial it later reads, so the scratch
    // needs no clearing between calls.
    return spec_verify_attn(attn, q, cache, kb, vb, soft_k, soft_v, seq_len, vis, row_flags, o,
                            lse, scratch, (size_t)SPEC_NOALLOC_SCRATCH_BYTES, stream);
}
