// spec_vocab_reduce and spec_accept.
//
// Vocab reduce: per judged row, the greedy token (argmax, lowest index on
// ties), ln sum exp(z) and the proposal's logit -- what "Lookahead
// Attention" sec. 2.4 (proposal probability against a threshold) and
// "Speculative Streaming"'s verification step (hard matching against the
// greedy token) need.
//
// Accept: the LA threshold longest prefix, or the greedy walk down the draft
// tree ("Speculative Streaming", verification step; "ConFu" tree verify).
#include <limits.h>
#include <math.h>

#include "common.cuh"

namespace sv {
namespace {

constexpr int kReduceThreads = 256;

struct Best {
    float m;     // running max
    int idx;     // lowest index attaining it
    float s;     // sum of exp(z - m)
};

__device__ __forceinline__ void best_push(Best &b, float z, int i) {
    if (z > b.m) {
        b.s = b.s * __expf(b.m - z) + 1.f;
        b.m = z;
        b.idx = i;
    } else {
        b.s += __expf(z - b.m);
        if (z == b.m && i < b.idx) b.idx = i;
    }
}

__device__ __forceinline__ Best best_merge(Best a, Best b) {
    if (b.m > a.m || (b.m == a.m && b.idx < a.idx)) {
        Best t = a;
        a = b;
        b = t;
    }
    // a has the larger max (or equal max with the lower index)
    if (b.m != -INFINITY) a.s += b.s * __expf(b.m - a.m);
    return a;
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

// One CTA per row, 16-byte loads, one pass with a running (max, index, sum).
template <typename T>
__global__ void __launch_bounds__(kReduceThreads)
vocab_reduce_kernel(const T *__restrict__ logits, int V, const int32_t *__restrict__ proposal,
                    int32_t *__restrict__ argmax, float *__restrict__ lse,
                    float *__restrict__ zprop) {
    const int row = blockIdx.x;
    const T *z = logits + (size_t)row * V;
    Best best{-INFINITY, INT_MAX, 0.f};
    constexpr int N = Vec<T>::N;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(z) & 15) == 0);
    int done = 0;
    if (vec_ok) {
        const int nv = V / N;
        for (int i = threadIdx.x; i < nv; i += kReduceThreads) {
            float x[N];
            Vec<T>::load(z + (size_t)i * N, x);
            float vm = x[0];
            int vi = 0;
#pragma unroll
            for (int j = 1; j < N; ++j)
                if (x[j] > vm) { vm = x[j]; vi = j; }
            if (vm > best.m) {
                best.s = best.s * __expf(best.m - vm);
                best.m = vm;
                best.idx = i * N + vi;
            } else if (vm == best.m && i * N + vi < best.idx) {
                best.idx = i * N + vi;
            }
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < N; ++j) acc += __expf(x[j] - best.m);
            best.s += acc;
        }
        done = nv * N;
    }
    for (int i = done + threadIdx.x; i < V; i += kReduceThreads) best_push(best, load_f(z + i), i);

    // block reduction: warps, then across warps
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Best other;
        other.m = __shfl_xor_sync(0xffffffffu, best.m, o);
        other.idx = __shfl_xor_sync(0xffffffffu, best.idx, o);
        other.s = __shfl_xor_sync(0xffffffffu, best.s, o);
        best = best_merge(best, other);
    }
    __shared__ Best sb[kReduceThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sb[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        Best r = sb[0];
        for (int w = 1; w < kReduceThreads / 32; ++w) r = best_merge(r, sb[w]);
        argmax[row] = r.idx == INT_MAX ? 0 : r.idx;
        lse[row] = r.m + logf(r.s);
        if (proposal && zprop) {
            const int pidx = proposal[row];
            zprop[row] = (pidx >= 0 && pidx < V) ? load_f(z + pidx) : NAN;
        }
    }
}

struct AcceptParams {
    int mode;
    float log_tau;
    int B, Rj, N, path_cap;
    const int32_t *tokens, *tree_parent, *row_of, *n_nodes;
    const int32_t *argmax;
    const float *lse, *zprop;
    int32_t *acc_len, *path, *next_token, *last_node;
    int *status;
};

// One warp per request.
__global__ void __launch_bounds__(128) accept_kernel(AcceptParams P) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (b >= P.B) return;
    int n = P.n_nodes[b];
    const int n_lim = P.mode == SPEC_ACCEPT_THRESH_CHAIN ? min(P.N, P.Rj) : P.N;
    if (n < 0 || n > n_lim) {
        if (lane == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
        n = n < 0 ? 0 : n_lim;
    }
    int32_t *pth = P.path + (size_t)b * P.path_cap;
    int len = 0, next = -1, last = -1;
    if (P.mode == SPEC_ACCEPT_THRESH_CHAIN) {
        // L = first i < n whose proposal probability is below tau.
        int L = n;
        for (int base = 0; base < n; base += 32) {
            const int i = base + lane;
            bool fail = false;
            if (i < n) {
                const size_t k = (size_t)b * P.Rj + i;
                fail = !(P.zprop[k] - P.lse[k] >= P.log_tau);
            }
            const unsigned bal = __ballot_sync(0xffffffffu, fail);
            if (bal) {
                L = base + __ffs(bal) - 1;
                break;
            }
        }
        if (L > P.path_cap) {
            if (lane == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
            L = P.path_cap;
        }
        len = L;
        next = L < n ? P.argmax[(size_t)b * P.Rj + L] : -1;
        last = L - 1;
        for (int i = lane; i < P.path_cap; i += 32) pth[i] = i < L ? i : -1;
    } else {
        const int32_t *par = P.tree_parent + (size_t)b * P.N;
        const int32_t *tok = P.tokens + (size_t)b * P.N;
        int cur = 0;
        if (n == 0 || P.path_cap == 0) {
            if (lane == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
        } else {
            len = 1;
            if (lane == 0) pth[0] = 0;
            while (true) {
                const int row = P.row_of ? P.row_of[(size_t)b * P.N + cur] : cur;
                if (row < 0 || row >= P.Rj) {
                    if (lane == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
                    next = -1;
                    break;
                }
                const int want = P.argmax[(size_t)b * P.Rj + row];
                next = want;
                // children have larger indices than their parent
                int found = -1;
                for (int base = cur + 1; base < n; base += 32) {
                    const int c = base + lane;
                    const bool hit = c < n && par[c] == cur && tok[c] == want;
                    const unsigned bal = __ballot_sync(0xffffffffu, hit);
                    if (bal) {
                        found = base + __ffs(bal) - 1;
                        break;
                    }
                }
                if (found < 0) break;
                if (len >= P.path_cap) {
                    if (lane == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
                    break;
                }
                if (lane == 0) pth[len] = found;
                ++len;
                cur = found;
            }
            last = cur;
        }
        __syncwarp();
        for (int i = len + lane; i < P.path_cap; i += 32) pth[i] = -1;
    }
    if (lane == 0) {
        P.acc_len[b] = len;
        P.next_token[b] = next;
        P.last_node[b] = last;
    }
}

spec_status_t launch_vocab_reduce(const void *logits, int dtype, int n_rows, int V,
                                  const int32_t *proposal, int32_t *argmax, float *lse,
                                  float *zprop, cudaStream_t s) {
    if (dtype == SPEC_BF16)
        vocab_reduce_kernel<__nv_bfloat16><<<n_rows, kReduceThreads, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(logits), V, proposal, argmax, lse, zprop);
    else
        vocab_reduce_kernel<float><<<n_rows, kReduceThreads, 0, s>>>(
            static_cast<const float *>(logits), V, proposal, argmax, lse, zprop);
    return launch_status();
}

}  // namespace
}  // namespace sv

extern "C" spec_status_t spec_vocab_reduce(const void *logits, int dtype, int n_rows, int vocab,
                                           const int32_t *proposal, int32_t *argmax, float *lse,
                                           float *zprop, void *stream) {
    if (n_rows < 0 || vocab <= 0) return SPEC_ERR_INVALID_ARG;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    if (n_rows == 0) return SPEC_OK;
    if (!logits || !argmax || !lse || (proposal && !zprop)) return SPEC_ERR_INVALID_ARG;
    if (n_rows > 2147483647 / 1) return SPEC_ERR_UNSUPPORTED;
    return sv::launch_vocab_reduce(logits, dtype, n_rows, vocab, proposal, argmax, lse, zprop,
                                   sv::as_stream(stream));
}

extern "C" spec_status_t spec_accept(const spec_accept_desc *d, const void *logits,
                                     const int32_t *tokens, const int32_t *tree_parent,
                                     const int32_t *row_of, const int32_t *n_nodes,
                                     int32_t *argmax, float *lse, float *zprop, int32_t *acc_len,
                                     int32_t *path, int32_t *next_token, int32_t *last_node,
                                     void *stream) {
    if (!d) return SPEC_ERR_INVALID_ARG;
    if (d->mode != SPEC_ACCEPT_THRESH_CHAIN && d->mode != SPEC_ACCEPT_GREEDY_TREE)
        return SPEC_ERR_INVALID_ARG;
    if (d->batch < 0 || d->n_judge_rows <= 0 || d->max_nodes <= 0 || d->path_cap < 0)
        return SPEC_ERR_INVALID_ARG;
    if (d->batch == 0) return SPEC_OK;
    if (!tokens || !n_nodes || !argmax || !lse || !acc_len || !path || !next_token || !last_node)
        return SPEC_ERR_INVALID_ARG;
    const bool chain = d->mode == SPEC_ACCEPT_THRESH_CHAIN;
    if (chain) {
        if (row_of || !zprop) return SPEC_ERR_INVALID_ARG;
        if (!(d->tau > 0.f) || d->tau > 1.f) return SPEC_ERR_INVALID_ARG;
        if (logits && d->max_nodes != d->n_judge_rows) return SPEC_ERR_INVALID_ARG;
    } else if (!tree_parent) {
        return SPEC_ERR_INVALID_ARG;
    }
    cudaStream_t s = sv::as_stream(stream);
    if (logits) {
        if (d->vocab <= 0) return SPEC_ERR_INVALID_ARG;
        if (d->logit_dtype != SPEC_F32 && d->logit_dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
        const long long rows = (long long)d->batch * d->n_judge_rows;
        if (rows > 2147483647ll) return SPEC_ERR_UNSUPPORTED;
        spec_status_t st = sv::launch_vocab_reduce(logits, d->logit_dtype, (int)rows, d->vocab,
                                                   chain ? tokens : nullptr, argmax, lse,
                                                   chain ? zprop : nullptr, s);
        if (st != SPEC_OK) return st;
    }
    sv::AcceptParams P{};
    P.mode = d->mode;
    P.log_tau = chain ? logf(d->tau) : 0.f;
    P.B = d->batch;
    P.Rj = d->n_judge_rows;
    P.N = d->max_nodes;
    P.path_cap = d->path_cap;
    P.tokens = tokens;
    P.tree_parent = tree_parent;
    P.row_of = row_of;
    P.n_nodes = n_nodes;
    P.argmax = argmax;
    P.lse = lse;
    P.zprop = zprop;
    P.acc_len = acc_len;
    P.path = path;
    P.next_token = next_token;
    P.last_node = last_node;
    P.status = sv::status_ptr();
    if (!P.status) return SPEC_ERR_CUDA;
    sv::accept_kernel<<<sv::ceil_div(P.B, 4), 128, 0, s>>>(P);
    return sv::launch_status();
}
