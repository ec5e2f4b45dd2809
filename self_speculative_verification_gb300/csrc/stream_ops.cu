// spec_stream_rotate_values and spec_future_gather.
//
// Value rotation ("Speculative Streaming" Eq. 7): the value vector of
// stream s of node j is node j's value vector times e^{i eps s}, with
// consecutive pairs (v[2i], v[2i+1]) as real and imaginary parts.  The
// stream rows of the block's V are written from their node rows before the
// verify attention reads them; one CTA per (request, KV head), each thread
// rotates four pairs (16 bytes of bf16) per step.
//
// Future-token gather ("ConFu" key design 1): the output of the
// contemplate token attached to the last accepted node -- block row
// row_offset + last_node -- is copied out for the next round's draft.
#include <math.h>

#include "common.cuh"

namespace sv {
namespace {

constexpr int kThreads = 256;

struct RotateParams {
    int B, R, Hkv, d, gamma;
    float eps;
    const int32_t *n_nodes;
    void *vb;
    int *status;
};

constexpr int kMaxGamma = 64;

// 8 consecutive elements (4 pairs) at p as floats / back to storage.
__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void st8(__nv_bfloat16 *p, const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&v);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void ld8(const float *p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0];
    const float4 b = reinterpret_cast<const float4 *>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void st8(float *p, const float (&x)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}

// One CTA per (request, KV head); a thread rotates 4 pairs (8 elements) of
// one stream row per step; cos / sin of eps * s are computed once per CTA.
template <typename T>
__global__ void __launch_bounds__(kThreads) rotate_kernel(RotateParams P) {
    pdl_wait();
    __shared__ float s_cos[kMaxGamma], s_sin[kMaxGamma];
    const int b = blockIdx.x / P.Hkv, h = blockIdx.x % P.Hkv;
    const int T_b = P.n_nodes[b];
    if (T_b < 0 || (long long)T_b * (1 + P.gamma) > P.R) {
        if (h == 0 && threadIdx.x == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
        return;
    }
    if (threadIdx.x < P.gamma) sincosf(P.eps * (float)(threadIdx.x + 1), &s_sin[threadIdx.x],
                                       &s_cos[threadIdx.x]);
    __syncthreads();
    T *v = static_cast<T *>(P.vb) + ((size_t)b * P.Hkv + h) * P.R * P.d;
    const int chunks = P.d / 8;
    const int work = T_b * P.gamma * chunks;
    for (int w = threadIdx.x; w < work; w += kThreads) {
        const int ch = w % chunks, q = w / chunks;       // q = j * gamma + (s - 1)
        const int j = q / P.gamma, si = q % P.gamma;
        const float c = s_cos[si], sn = s_sin[si];
        float x[8], y[8];
        ld8(v + (size_t)j * P.d + ch * 8, x);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            y[2 * i] = fmaf(x[2 * i], c, -x[2 * i + 1] * sn);
            y[2 * i + 1] = fmaf(x[2 * i], sn, x[2 * i + 1] * c);
        }
        st8(v + (size_t)(T_b + q) * P.d + ch * 8, y);
    }
}

struct GatherParams {
    int B, R, row_bytes, row_offset;
    const int32_t *last_node;
    const uint8_t *o;
    uint8_t *out;
    int *status;
};

__global__ void __launch_bounds__(kThreads) gather_kernel(GatherParams P) {
    pdl_wait();
    const int b = blockIdx.x;
    const int ln = P.last_node[b];
    const int row = P.row_offset + ln;
    const bool ok = ln >= 0 && row < P.R;
    if (!ok && threadIdx.x == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
    uint8_t *dst = P.out + (size_t)b * P.row_bytes;
    const uint8_t *src = P.o + ((size_t)b * P.R + (ok ? row : 0)) * P.row_bytes;
    // rows are whole multiples of 16 bytes (checked on the host)
    for (int i = threadIdx.x; i < P.row_bytes / 16; i += kThreads)
        reinterpret_cast<uint4 *>(dst)[i] =
            ok ? reinterpret_cast<const uint4 *>(src)[i] : make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace
}  // namespace sv

extern "C" spec_status_t spec_stream_rotate_values(const spec_rotate_desc *d,
                                                   const int32_t *n_nodes, void *vb,
                                                   void *stream) {
    using namespace sv;
    if (!d) return SPEC_ERR_INVALID_ARG;
    if (d->batch < 0 || d->n_rows <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 ||
        d->gamma <= 0 || !(d->eps == d->eps))
        return SPEC_ERR_INVALID_ARG;
    if (d->head_dim % 8 != 0 || d->gamma > kMaxGamma) return SPEC_ERR_UNSUPPORTED;
    if (d->dtype != SPEC_F32 && d->dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    if (d->batch == 0) return SPEC_OK;
    if (!n_nodes || !vb) return SPEC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(vb) % 16 != 0) return SPEC_ERR_INVALID_ARG;
    if ((long long)d->batch * d->n_kv_heads > 2147483647ll) return SPEC_ERR_UNSUPPORTED;
    RotateParams P{};
    P.B = d->batch;
    P.R = d->n_rows;
    P.Hkv = d->n_kv_heads;
    P.d = d->head_dim;
    P.gamma = d->gamma;
    P.eps = d->eps;
    P.n_nodes = n_nodes;
    P.vb = vb;
    P.status = status_ptr();
    if (!P.status) return SPEC_ERR_CUDA;
    const int grid = d->batch * d->n_kv_heads;
    const spec_status_t ls =
        d->dtype == SPEC_BF16
            ? launch(rotate_kernel<__nv_bfloat16>, dim3(grid), dim3(kThreads), 0, as_stream(stream), P)
            : launch(rotate_kernel<float>, dim3(grid), dim3(kThreads), 0, as_stream(stream), P);
    if (ls != SPEC_OK) return ls;
    return launch_status();
}

extern "C" spec_status_t spec_future_gather(int batch, int n_rows, int row_elems, int dtype,
                                            const void *o, const int32_t *last_node,
                                            int row_offset, void *out, void *stream) {
    using namespace sv;
    if (batch < 0 || n_rows <= 0 || row_elems <= 0 || row_offset < 0) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    const long long row_bytes = (long long)row_elems * (dtype == SPEC_BF16 ? 2 : 4);
    if (row_bytes % 16 != 0 || row_bytes > 2147483647ll) return SPEC_ERR_UNSUPPORTED;
    if (batch == 0) return SPEC_OK;
    if (!o || !last_node || !out) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(out)) % 16 != 0)
        return SPEC_ERR_INVALID_ARG;
    GatherParams P{};
    P.B = batch;
    P.R = n_rows;
    P.row_bytes = (int)row_bytes;
    P.row_offset = row_offset;
    P.last_node = last_node;
    P.o = static_cast<const uint8_t *>(o);
    P.out = static_cast<uint8_t *>(out);
    P.status = status_ptr();
    if (!P.status) return SPEC_ERR_CUDA;
    if (launch(gather_kernel, dim3(batch), dim3(kThreads), 0, as_stream(stream), P) != SPEC_OK)
        return SPEC_ERR_CUDA;
    return launch_status();
}
