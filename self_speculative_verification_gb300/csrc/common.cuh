// Shared helpers of libspecverify's CUDA sources (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>

#include "specverify.h"

namespace sv {

// Device address of the per-device status word (SPEC_DEV_* bits) for the
// current device; nullptr if it cannot be resolved.
int *status_ptr();

// The current CUDA context (driver handle), or nullptr.
void *current_context();

// Device addresses of one __device__ symbol, per device and context: host
// code sees only a stand-in for such a symbol, and the address it has on a
// device is looked up (cudaGetSymbolAddress) with that device current.  A
// new context on a device (after cudaDeviceReset, say) is looked up again.
struct DeviceSymbolCache {
    static constexpr int kDevices = 64;
    std::mutex mu;
    void *addr[kDevices] = {};
    void *ctx[kDevices] = {};
};
spec_status_t symbol_address(DeviceSymbolCache &cache, const void *symbol, void **out);

// Limit, in SM cycles, that kernel launches give their pipeline waits
// (spec_set_wait_limit; default ~1 s).
long long wait_limit();

// Raise `func`'s dynamic shared-memory limit to `bytes` on the current
// device (once per device and context: the attribute applies to the device
// current when it is set).
spec_status_t set_smem_limit(const void *func, size_t bytes);

// Number of SMs of the current device (cached per device).
int num_sms();

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline spec_status_t launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation, so its launch is processed while
// the kernel before it in the stream finishes and its blocks are scheduled
// as that kernel's blocks exit; it first waits (pdl_wait) until that kernel
// has completed and its writes are visible.  No kernel triggers its
// successor early: blocks of a heavy successor waiting on the SMs slowed the
// running kernel (back-to-back vocabulary reductions 20 % slower).  A no-op
// for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// kernel<<<grid, block, smem, stream>>>(args...) with the attribute above;
// returns the launch's status.
template <typename... KArgs, typename... Args>
inline spec_status_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...) == cudaSuccess
               ? SPEC_OK
               : SPEC_ERR_CUDA;
}

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

__device__ __forceinline__ void raise_status(int *st, int bits) {
    if (st) atomicOr(st, bits);
}

__device__ __forceinline__ float load_f(const float *p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__device__ __forceinline__ void store_f(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_f(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace sv
