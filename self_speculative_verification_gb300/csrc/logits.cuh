// Loads of logit rows (fp32 or bf16) as floats, and the exp2 used by the
// vocabulary reductions.
#pragma once

#include "common.cuh"

namespace sv {

// 2^x by the hardware approximation (relative error ~2^-22); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const float *p, float *out) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16 *p, float *out) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

// 8 consecutive logits (16-byte aligned) as floats.
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&out)[8]) {
    Vec<__nv_bfloat16>::load(p, out);
}
__device__ __forceinline__ void load8(const float *p, float (&out)[8]) {
    float a[4], c[4];
    Vec<float>::load(p, a);
    Vec<float>::load(p + 4, c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[i] = a[i];
        out[4 + i] = c[i];
    }
}

}  // namespace sv
