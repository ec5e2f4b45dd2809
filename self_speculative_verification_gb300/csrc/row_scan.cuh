// Row reductions over logits shared by the vocabulary reduction and the
// draft-tree edge test: a running (max, lowest index of the max, sum of
// exp(c (z - max))) per thread, packed arithmetic for bf16 batches, and a
// bulk-copy stream of a bf16 row slice through shared memory.
#pragma once

#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "logits.cuh"
#include "ptx_sm103.cuh"

namespace sv {
namespace {

struct Best {
    float m;     // running max
    int idx;     // lowest index attaining it
    float s;     // sum of exp(z - m)
};

// inv_t: 1 / temperature (the sums are of exp(z / T)).
__device__ __forceinline__ void best_push(Best &b, float z, int i, float inv_t) {
    if (z > b.m) {
        b.s = b.s * __expf((b.m - z) * inv_t) + 1.f;
        b.m = z;
        b.idx = i;
    } else {
        b.s += __expf((z - b.m) * inv_t);
        if (z == b.m && i < b.idx) b.idx = i;
    }
}

__device__ __forceinline__ Best best_merge(Best a, Best b, float inv_t) {
    if (b.m > a.m || (b.m == a.m && b.idx < a.idx)) {
        Best t = a;
        a = b;
        b = t;
    }
    // a has the larger max (or equal max with the lower index)
    if (b.m != -INFINITY) a.s += b.s * __expf((b.m - a.m) * inv_t);
    return a;
}

// bf16 batches without a ragged end take packed arithmetic: the batch max
// on bf16 pairs (exact: a max selects one of its inputs), the exponent
// arguments and the sums on fp32 pairs, so per element about one ex2 and
// three other instructions issue.
constexpr int kUnroll = 4;

struct Bf16Batch {
    uint32_t w[kUnroll][4];     // kUnroll x 8 bf16, pairs in 32-bit words
};

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Running (max, index, sum) over one full batch of kUnroll 8-element
// vectors; vector u starts at element (i0 + u * kStride) * 8.
template <int kStride>
__device__ __forceinline__ void push_bf16_batch(Best &best, const Bf16Batch &x, int i0, float c2) {
    uint32_t m2 = x.w[0][0];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int q = 0; q < 4; ++q) m2 = bf16x2_max(m2, x.w[u][q]);
    const float bm = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xffff0000u));
    if (bm > best.m) {
        int bi = INT_MAX;
#pragma unroll
        for (int u = kUnroll - 1; u >= 0; --u)
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                const uint32_t wq = x.w[u][j >> 1];
                const float v = __uint_as_float((j & 1) ? (wq & 0xffff0000u) : (wq << 16));
                if (v == bm) bi = (i0 + u * kStride) * 8 + j;
            }
        best.s *= ex2((best.m - bm) * c2);
        best.m = bm;
        best.idx = bi;
    }
    const uint64_t c22 = pair(c2, c2);
    const float nmb = -best.m * c2;
    const uint64_t nmb2 = pair(nmb, nmb);
    uint64_t acc[4] = {pair(0.f, 0.f), pair(0.f, 0.f), pair(0.f, 0.f), pair(0.f, 0.f)};
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t wq = x.w[u][q];
            float t0, t1;
            unpair(fma2(pair(__uint_as_float(wq << 16), __uint_as_float(wq & 0xffff0000u)), c22,
                        nmb2),
                   t0, t1);
            acc[q] = add2(acc[q], pair(ex2(t0), ex2(t1)));
        }
    float a0, a1, a2, a3, a4, a5, a6, a7;
    unpair(acc[0], a0, a1);
    unpair(acc[1], a2, a3);
    unpair(acc[2], a4, a5);
    unpair(acc[3], a6, a7);
    best.s += ((a0 + a1) + (a2 + a3)) + ((a4 + a5) + (a6 + a7));
}


__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Chunk of the bulk row stream: kThreads x kUnroll 16-byte vectors.
template <int kThreads>
constexpr int bulk_chunk() { return kThreads * kUnroll * 8; }

// Shared memory the stream of a kThreads-thread CTA with kStages stages takes.
template <int kThreads, int kStages>
constexpr int bulk_smem() { return kStages * bulk_chunk<kThreads>() * 2; }

// Folds a bf16 slice (16-byte aligned, n_el elements, a multiple of 8) into
// every thread's `best`: thread 0 issues bulk copies (cp.async.bulk, L2
// evict-first) of bulk_chunk<kThreads>() elements into kStages buffers of
// `stage` (dynamic shared memory, bulk_smem<kThreads, kStages>() bytes, full[]
// kStages mbarriers of its own) ahead of the others, who sleep in the block
// barrier rather than spin; after it every thread tests the completed phase
// once (its own acquire of the bytes) and reduces its kUnroll vectors of the
// chunk.  The slice's element e is element 8 v0 + e of its row (the index
// kept for the max).  c2 = log2(e) / temperature.  Returns false if a copy had
// not landed within `wait` cycles; the CTA has then waited for its other
// copies (default limit) and `best` holds a partial result.  Call with the
// whole CTA.
template <int kThreads, int kStages>
__device__ bool bulk_row_scan(const __nv_bfloat16 *slice, int n_el, int v0, float c2, Best &best,
                              uint8_t *stage, uint64_t *full, long long wait) {
    constexpr int kChunk = bulk_chunk<kThreads>();
    const int n_chunks = (n_el + kChunk - 1) / kChunk;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int ch) {        // thread 0: chunk ch into its stage
        const int b = ch % kStages;
        const uint32_t bytes = (uint32_t)min(kChunk, n_el - ch * kChunk) * 2u;
        mbar_arrive_expect_tx(&full[b], bytes);
        bulk_load(stage + b * (kChunk * 2), slice + (size_t)ch * kChunk, bytes, &full[b], pol);
    };
    if (threadIdx.x == 0)
        for (int ch = 0; ch < n_chunks && ch < kStages; ++ch) issue(ch);
    int ch = 0;
    bool failed = false;
    for (; ch < n_chunks; ++ch) {
        const int b = ch % kStages;
        const uint32_t parity = (uint32_t)((ch / kStages) & 1);
        const bool got = threadIdx.x != 0 || mbar_wait(&full[b], parity, wait);
        if (__syncthreads_or(!got)) {
            failed = true;
            break;
        }
        (void)mbar_test_wait(&full[b], parity);
        const uint4 *sv = reinterpret_cast<const uint4 *>(stage + b * (kChunk * 2));
        const int i0 = v0 + ch * (kChunk / 8) + (int)threadIdx.x;   // vector index in the row
        const int nvec = min(kChunk, n_el - ch * kChunk) / 8;
        if ((int)threadIdx.x + (kUnroll - 1) * kThreads < nvec) {
            Bf16Batch x;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint4 v = sv[threadIdx.x + u * kThreads];
                x.w[u][0] = v.x;
                x.w[u][1] = v.y;
                x.w[u][2] = v.z;
                x.w[u][3] = v.w;
            }
            push_bf16_batch<kThreads>(best, x, i0, c2);
        } else if ((int)threadIdx.x < nvec) {
            // a batch that runs past the end of the slice
            float xs[kUnroll][8];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int iv = (int)threadIdx.x + u * kThreads;
                if (iv < nvec) {
                    const uint4 v = sv[iv];
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        xs[u][2 * j] = __uint_as_float(w[j] << 16);
                        xs[u][2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) xs[u][j] = -INFINITY;
                }
            }
            float bm = xs[0][0];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j) bm = fmaxf(bm, xs[u][j]);
            if (bm > best.m) {
                int bi = INT_MAX;
#pragma unroll
                for (int u = kUnroll - 1; u >= 0; --u)
#pragma unroll
                    for (int j = 7; j >= 0; --j)
                        if (xs[u][j] == bm) bi = (i0 + u * kThreads) * 8 + j;
                best.s *= ex2((best.m - bm) * c2);
                best.m = bm;
                best.idx = bi;
            }
            const float mb = best.m * c2;
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] += ex2(fmaf(xs[u][j], c2, -mb));
#pragma unroll
            for (int j = 1; j < 8; ++j) acc[0] += acc[j];
            best.s += acc[0];
        }
        __syncthreads();                 // every thread is done with this stage
        if (threadIdx.x == 0 && ch + kStages < n_chunks) issue(ch + kStages);
    }
    if (failed) {
        // do not leave while copies into this CTA's shared memory are in
        // flight
        if (threadIdx.x == 0)
            for (int c = ch; c < n_chunks && c < ch + kStages; ++c)
                if (!mbar_wait(&full[c % kStages], (uint32_t)((c / kStages) & 1))) break;
        __syncthreads();
    }
    return !failed;
}

}  // namespace
}  // namespace sv
