// spec_draft_tree and spec_prune_tree: the next step's draft tree
// ("Speculative Streaming": tree draft construction, parallel tree pruning,
// batching with streams).
//
// Draft: the top-k tokens of each of the gamma stream logit rows at the
// accepted position (largest logit first, ties to the lower token id) make
// a complete k-ary tree of depth gamma, flattened breadth-first: node 0 is
// the root (the correction token), level g holds k^g nodes, node
// off(g) + m has parent off(g-1) + m / k and token top_g[m % k].  One CTA
// per (stream, request) finds its stream's top-k and writes its level.
//
// Prune: edge (p, c) survives iff softmax(early-exit logits at p)[token c]
// >= threshold; a node survives iff its edge and its parent survive.  One
// CTA per (node, request) computes the node's ln sum exp and tests its
// children; one CTA per request then compacts the survivors in order.
//
// Both can also write the parent pointers of the flattened block that
// spec_mask_build takes: rows 0..n-1 the nodes, row n + j*gamma + (s-1)
// stream s of node j (stream 1 under node j, stream s > 1 under stream
// s-1), padding after.
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "logits.cuh"

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxK = 8;
constexpr int kMaxPruneNodes = 1024;

// vparent row(s) of node j in a tree of n nodes with gamma streams per node
__device__ __forceinline__ void write_block_rows(int32_t *vp, int n, int gamma, int j, int par) {
    vp[j] = par < 0 ? SPEC_VP_ROOT : par;
    for (int s = 1; s <= gamma; ++s) {
        const int r = n + j * gamma + (s - 1);
        vp[r] = s == 1 ? j : r - 1;
    }
}

struct DraftParams {
    int B, rows, gamma, k, V, max_nodes, vp_rows, n_full;
    const void *logits;
    const int32_t *stream_row, *root_token;
    int32_t *tokens, *parent, *n_nodes, *vparent;
    int *status;
};

// (a, ia) comes before (b, ib) in top-k order: larger value, then lower id.
__device__ __forceinline__ bool before(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

// The best (value, id) of a warp, every lane gets it (ids unique or INT_MAX).
__device__ __forceinline__ void warp_best(float &v, int &id) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, id, o);
        if (oi != INT_MAX && (id == INT_MAX || before(ov, oi, v, id))) {
            v = ov;
            id = oi;
        }
    }
}

constexpr int kDraftThreads = 1024;
constexpr int kMaxCand = 2048;

// Top-k of one stream row in two passes.  Pass 1: every thread's maximum;
// the k-th largest of those maxima, T, bounds the k-th largest logit from
// below (k threads each hold a logit >= T).  Pass 2: the logits >= T are
// collected; warp 0 picks the k first in top-k order.  When ties at T
// overflow the candidate buffer, k rounds of "the best entry after the
// previous pick" over the whole row decide instead.
template <typename T>
__global__ void __launch_bounds__(kDraftThreads) draft_tree_kernel(DraftParams P) {
    pdl_wait();
    __shared__ float s_max[kDraftThreads];
    __shared__ float s_cv[kMaxCand];
    __shared__ int s_ci[kMaxCand];
    __shared__ int s_nc;
    __shared__ float s_thr;
    __shared__ int s_top[kMaxK];
    __shared__ float s_wv[kDraftThreads / 32];
    __shared__ int s_wi[kDraftThreads / 32];
    const int j = blockIdx.x, b = blockIdx.y;
    const int k = P.k;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int row = (P.stream_row ? P.stream_row[b] : 0) + j;
    if (row < 0 || row >= P.rows) {
        if (threadIdx.x == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
        row = -1;
    }
    const T *z = row >= 0 ? static_cast<const T *>(P.logits) + ((size_t)b * P.rows + row) * P.V
                          : nullptr;
    const int V = row >= 0 ? P.V : 0;
    const int nv = (reinterpret_cast<uintptr_t>(z) & 15) == 0 ? V / 8 : 0;
    // visits every logit of this thread: f(x, id)
    auto scan = [&](auto f) {
        constexpr int U = 2;
        for (int c0 = threadIdx.x; c0 < nv; c0 += U * kDraftThreads) {
            float x[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kDraftThreads;
                if (c < nv) {
                    load8(z + (size_t)c * 8, x[u]);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[u][e] = -INFINITY;
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * kDraftThreads;
                if (c < nv) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f(x[u][e], c * 8 + e);
                }
            }
        }
        for (int v = nv * 8 + threadIdx.x; v < V; v += kDraftThreads) f(load_f(z + v), v);
    };
    // pass 1
    float m = -INFINITY;
    scan([&](float x, int) { m = fmaxf(m, x); });
    s_max[threadIdx.x] = m;
    if (threadIdx.x == 0) s_nc = 0;
    __syncthreads();
    if (warp == 0) {
        // k-th largest thread maximum (by value; ties count separately)
        float tv[kDraftThreads / 32];
#pragma unroll
        for (int i = 0; i < kDraftThreads / 32; ++i) tv[i] = s_max[i * 32 + lane];
        float thr = -INFINITY;
        for (int r = 0; r < k; ++r) {
            float v = -INFINITY;
            int pos = INT_MAX;
#pragma unroll
            for (int i = 0; i < kDraftThreads / 32; ++i)
                if (pos == INT_MAX || tv[i] > v) {
                    v = tv[i];
                    pos = i * 32 + lane;
                }
            warp_best(v, pos);
            thr = v;
            if ((pos & 31) == lane) {
#pragma unroll
                for (int i = 0; i < kDraftThreads / 32; ++i)
                    if (i == (pos >> 5)) tv[i] = -INFINITY;
            }
        }
        if (lane == 0) s_thr = thr;
    }
    __syncthreads();
    // pass 2: the candidates
    const float thr = s_thr;
    scan([&](float x, int v) {
        if (x >= thr) {
            const int slot = atomicAdd(&s_nc, 1);
            if (slot < kMaxCand) {
                s_cv[slot] = x;
                s_ci[slot] = v;
            }
        }
    });
    __syncthreads();
    const int nc = s_nc;
    if (nc <= kMaxCand) {
        if (warp == 0) {
            float pv = INFINITY;
            int pi = -1;
            for (int r = 0; r < k; ++r) {
                float bv = -INFINITY;
                int bi = INT_MAX;
                for (int c = lane; c < nc; c += 32) {
                    const float cv = s_cv[c];
                    const int ci = s_ci[c];
                    if (before(pv, pi, cv, ci) && (bi == INT_MAX || before(cv, ci, bv, bi))) {
                        bv = cv;
                        bi = ci;
                    }
                }
                warp_best(bv, bi);
                if (lane == 0) s_top[r] = bi == INT_MAX ? 0 : bi;
                pv = bv;
                pi = bi;
            }
        }
    } else {
        // ties overflowed: k rounds over the row
        float pv = INFINITY;
        int pi = -1;
        for (int r = 0; r < k; ++r) {
            float bv = -INFINITY;
            int bi = INT_MAX;
            scan([&](float x, int v) {
                if (before(pv, pi, x, v) && (bi == INT_MAX || before(x, v, bv, bi))) {
                    bv = x;
                    bi = v;
                }
            });
            warp_best(bv, bi);
            if (lane == 0) {
                s_wv[warp] = bv;
                s_wi[warp] = bi;
            }
            __syncthreads();
            if (warp == 0) {
                bv = s_wv[lane];
                bi = s_wi[lane];
                warp_best(bv, bi);
                if (lane == 0) s_top[r] = bi == INT_MAX ? 0 : bi;
                if (lane == 0) {
                    s_wv[0] = bv;
                    s_wi[0] = bi;
                }
            }
            __syncthreads();
            pv = s_wv[0];
            pi = s_wi[0];
            __syncthreads();
        }
    }
    __syncthreads();
    // level g = j + 1: k^g nodes after the off(g) nodes of the levels above
    int off = 0, cnt = 1;
    for (int g = 0; g <= j; ++g) {
        off += cnt;
        cnt *= k;
    }
    const int prev_off = off - cnt / k;
    const size_t nb = (size_t)b * P.max_nodes;
    int32_t *vp = P.vparent ? P.vparent + (size_t)b * P.vp_rows : nullptr;
    for (int m = threadIdx.x; m < cnt; m += kDraftThreads) {
        const int node = off + m, par = prev_off + m / k;
        P.tokens[nb + node] = s_top[m % k];
        P.parent[nb + node] = par;
        if (vp) write_block_rows(vp, P.n_full, P.gamma, node, par);
    }
    if (j == 0) {
        if (threadIdx.x == 0) {
            P.tokens[nb] = P.root_token[b];
            P.parent[nb] = -1;
            P.n_nodes[b] = P.n_full;
            if (vp) write_block_rows(vp, P.n_full, P.gamma, 0, -1);
        }
        for (int c = P.n_full + threadIdx.x; c < P.max_nodes; c += kDraftThreads) {
            P.tokens[nb + c] = -1;
            P.parent[nb + c] = -1;
        }
        if (vp)
            for (int r = P.n_full * (1 + P.gamma) + threadIdx.x; r < P.vp_rows; r += kDraftThreads)
                vp[r] = SPEC_VP_PAD;
    }
}

struct PruneParams {
    int B, N, V, gamma, vp_rows;
    float threshold;
    const int32_t *tokens, *parent, *n_nodes;
    const void *early;
    int32_t *keep, *tokens_out, *parent_out, *n_out, *vparent;
    int *status;
};

__device__ __forceinline__ int clamp_nodes(const PruneParams &P, int b, bool report) {
    int n = P.n_nodes[b];
    if (n < 0 || n > P.N) {
        if (report) raise_status(P.status, SPEC_DEV_BAD_INDEX);
        n = n < 0 ? 0 : P.N;
    }
    return n;
}

// Exclusive prefix sum over a kT-thread block of one count per thread
// (every thread calls it); *s_total receives the sum.
template <int kT>
__device__ __forceinline__ int block_exclusive_scan(int cnt, int *s_wsum, int *s_total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kT / 32 ? s_wsum[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        if (lane < kT / 32) s_wsum[lane] = wi - w;
        if (lane == kT / 32 - 1) *s_total = wi;
    }
    __syncthreads();
    return s_wsum[warp] + incl - cnt;
}

// ln sum exp of one row of V logits (every thread calls it): a running
// (max, sum) per thread over 16-byte vectors (kEdgeLoads loads in flight),
// then the warp, then the block.  s_m / s_s: one slot per warp.
constexpr int kEdgeLoads = 4;
template <typename T>
__device__ float row_lse(const T *z, int V, float *s_m, float *s_s) {
    float m = -INFINITY, s = 0.f;
    const bool vec = (reinterpret_cast<uintptr_t>(z) & 15) == 0;
    const int nv = vec ? V / 8 : 0;
    constexpr int U = kEdgeLoads;
    for (int i0 = threadIdx.x; i0 < nv; i0 += U * kThreads) {
        float x[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * kThreads;
            if (i < nv) {
                load8(z + (size_t)i * 8, x[u]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) x[u][e] = -INFINITY;
            }
        }
        float bm = x[0][0];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int e = 0; e < 8; ++e) bm = fmaxf(bm, x[u][e]);
        if (bm > m) {
            s *= ex2((m - bm) * kLog2e);
            m = bm;
        }
        const float mb = m * kLog2e;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int e = 0; e < 8; ++e) s += ex2(fmaf(x[u][e], kLog2e, -mb));
    }
    for (int v = nv * 8 + threadIdx.x; v < V; v += kThreads) {
        const float x = load_f(z + v);
        if (x > m) {
            s = s * ex2((m - x) * kLog2e) + 1.f;
            m = x;
        } else {
            s += ex2((x - m) * kLog2e);
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const float os = __shfl_xor_sync(0xffffffffu, s, o);
        const float nm = fmaxf(m, om);
        s = (m == -INFINITY ? 0.f : s * ex2((m - nm) * kLog2e)) +
            (om == -INFINITY ? 0.f : os * ex2((om - nm) * kLog2e));
        m = nm;
    }
    if (lane == 0) {
        s_m[warp] = m;
        s_s[warp] = s;
    }
    __syncthreads();
    float M = -INFINITY, S = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const float nm = fmaxf(M, s_m[w]);
        S = (M == -INFINITY ? 0.f : S * ex2((M - nm) * kLog2e)) +
            (s_m[w] == -INFINITY ? 0.f : s_s[w] * ex2((s_m[w] - nm) * kLog2e));
        M = nm;
    }
    __syncthreads();                     // s_m / s_s free for the next row
    return M + logf(S);
}

// A request's tree takes ceil(N / kEdgeNodesPerPart) edge-test CTAs.
constexpr int kEdgeNodesPerPart = 4;

// The edge test of child c of node p: keep[c] = 1 iff its token's
// probability under p's logits (z[token] given, lse the row's) reaches the
// threshold.
__device__ __forceinline__ void edge_keep(const PruneParams &P, size_t nb, int c, int x, float zx,
                                          float lse) {
    int keep = 0;
    if (x < 0 || x >= P.V) raise_status(P.status, SPEC_DEV_BAD_INDEX);
    else keep = __expf(zx - lse) >= P.threshold;
    P.keep[nb + c] = keep;
}

// CTA (part, b): request b's inner nodes (those with a child), in index
// order, every gridDim.x-th from the part-th; for each such node p, the LSE
// of p's early-exit row, and each child keeps its edge iff its token's
// probability under p's logits reaches the threshold (keep[c] = 1 / 0; the
// root's entry is left to the compaction).  A child counts only when its
// parent index precedes it (the compaction reports the others).  The
// request's parents and tokens come in with one round of loads, and a
// thread's first child's logit is loaded before the row, so that only the
// row's loads remain in line.
// (five CTAs per SM, 760 resident: 32 requests x 22 parts of 85-node trees
// fit in one wave)
template <typename T>
__global__ void __launch_bounds__(kThreads, 5) prune_edge_kernel(PruneParams P) {
    pdl_wait();
    constexpr int kPer = kMaxPruneNodes / kThreads;
    __shared__ int s_par[kMaxPruneNodes], s_tok[kMaxPruneNodes], s_inner[kMaxPruneNodes];
    __shared__ uint8_t s_has[kMaxPruneNodes];
    __shared__ int s_wsum[kThreads / 32];
    __shared__ int s_ni;
    __shared__ float s_m[kThreads / 32], s_s[kThreads / 32];
    const int part = blockIdx.x, b = blockIdx.y;
    const int n = clamp_nodes(P, b, part == 0 && threadIdx.x == 0);
    const size_t nb = (size_t)b * P.N;
    for (int c = threadIdx.x; c < n; c += kThreads) {
        s_par[c] = P.parent[nb + c];
        s_tok[c] = P.tokens[nb + c];
        s_has[c] = 0;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < n; c += kThreads) {
        const int a = s_par[c];
        if (a >= 0 && a < c) s_has[a] = 1;
    }
    __syncthreads();
    // the inner nodes numbered in index order (this thread: nodes
    // t * kPer .. t * kPer + kPer - 1)
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = threadIdx.x * kPer + i;
        cnt += (c < n && s_has[c]) ? 1 : 0;
    }
    int idx = block_exclusive_scan<kThreads>(cnt, s_wsum, &s_ni);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = threadIdx.x * kPer + i;
        if (c < n && s_has[c]) s_inner[idx++] = c;
    }
    __syncthreads();
    const int ni = s_ni;
    for (int i = part; i < ni; i += gridDim.x) {
        const int p = s_inner[i];
        const T *z = static_cast<const T *>(P.early) + (nb + p) * P.V;
        // this thread's first candidate child and its token's logit
        const int c0 = p + 1 + threadIdx.x;
        const bool kid0 = c0 < n && s_par[c0] == p;
        const int x0 = kid0 ? s_tok[c0] : -1;
        const float z0 = (x0 >= 0 && x0 < P.V) ? load_f(z + x0) : 0.f;
        const float lse = row_lse(z, P.V, s_m, s_s);
        if (kid0) edge_keep(P, nb, c0, x0, z0, lse);
        for (int c = c0 + kThreads; c < n; c += kThreads) {
            if (s_par[c] != p) continue;
            const int x = s_tok[c];
            edge_keep(P, nb, c, x, (x >= 0 && x < P.V) ? load_f(z + x) : 0.f, lse);
        }
    }
}

// One CTA per request: keep[c] becomes c's new index (or -1) in order, and
// the survivors are written compacted.  Node c survives iff every edge on
// its path to the root survived: each thread walks its nodes' ancestor
// chains in shared memory (parents precede children, so a chain ends), then
// a block scan numbers the survivors.
__global__ void __launch_bounds__(kThreads) prune_compact_kernel(PruneParams P) {
    pdl_wait();
    constexpr int kPer = kMaxPruneNodes / kThreads;
    __shared__ int s_par[kMaxPruneNodes], s_idx[kMaxPruneNodes];
    __shared__ uint8_t s_edge[kMaxPruneNodes];
    __shared__ int s_wsum[kThreads / 32];
    __shared__ int s_cnt;
    const int b = blockIdx.x;
    const int n = clamp_nodes(P, b, false);
    const size_t nb = (size_t)b * P.N;
    for (int c = threadIdx.x; c < n; c += kThreads) {
        s_par[c] = P.parent[nb + c];
        s_edge[c] = c == 0 ? 1 : (P.keep[nb + c] == 1);
    }
    __syncthreads();
    // survival of this thread's nodes [t * kPer, t * kPer + kPer)
    int ok[kPer], cnt = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = threadIdx.x * kPer + i;
        bool alive = c < n;
        int x = c;
        while (alive && x > 0) {
            const int a = s_par[x];
            if (a < 0 || a >= x) {
                bad = true;
                alive = false;
            } else if (!s_edge[x]) {
                alive = false;
            } else {
                x = a;
            }
        }
        if (alive && s_par[0] >= 0) {
            bad = true;
            alive = false;
        }
        ok[i] = alive;
        cnt += alive;
    }
    if (bad) raise_status(P.status, SPEC_DEV_BAD_TREE);
    int idx = block_exclusive_scan<kThreads>(cnt, s_wsum, &s_cnt);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int c = threadIdx.x * kPer + i;
        if (c < n) s_idx[c] = ok[i] ? idx++ : -1;
    }
    __syncthreads();
    const int total = s_cnt;
    int32_t *vp = P.vparent ? P.vparent + (size_t)b * P.vp_rows : nullptr;
    for (int c = threadIdx.x; c < n; c += kThreads) {
        const int i = s_idx[c];
        P.keep[nb + c] = i;
        if (i >= 0) {
            const int np = c == 0 ? -1 : s_idx[s_par[c]];
            P.tokens_out[nb + i] = P.tokens[nb + c];
            P.parent_out[nb + i] = np;
            if (vp) write_block_rows(vp, total, P.gamma, i, np);
        }
    }
    for (int c = n + threadIdx.x; c < P.N; c += kThreads) P.keep[nb + c] = -1;
    for (int i = total + threadIdx.x; i < P.N; i += kThreads) {
        P.tokens_out[nb + i] = -1;
        P.parent_out[nb + i] = -1;
    }
    if (vp)
        for (int r = total * (1 + P.gamma) + threadIdx.x; r < P.vp_rows; r += kThreads)
            vp[r] = SPEC_VP_PAD;
    if (threadIdx.x == 0) P.n_out[b] = total;
}

}  // namespace
}  // namespace sv

extern "C" spec_status_t spec_draft_tree(const spec_draft_desc *d, const void *stream_logits,
                                         const int32_t *stream_row, const int32_t *root_token,
                                         int32_t *tokens, int32_t *tree_parent, int32_t *n_nodes,
                                         int32_t *vparent, void *stream) {
    using namespace sv;
    if (!d) return SPEC_ERR_INVALID_ARG;
    if (d->batch < 0 || d->n_stream_rows <= 0 || d->gamma <= 0 || d->k <= 0 || d->vocab <= 0 ||
        d->max_nodes <= 0 || d->vparent_rows < 0)
        return SPEC_ERR_INVALID_ARG;
    if (d->k > kMaxK || d->k > d->vocab) return SPEC_ERR_UNSUPPORTED;
    if (d->logit_dtype != SPEC_F32 && d->logit_dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    long long n_full = 1, level = 1;
    for (int g = 1; g <= d->gamma; ++g) {
        level *= d->k;
        n_full += level;
        if (n_full > (1 << 20)) return SPEC_ERR_UNSUPPORTED;
    }
    if (n_full > d->max_nodes) return SPEC_ERR_CAPACITY;
    if (vparent && n_full * (1 + d->gamma) > d->vparent_rows) return SPEC_ERR_CAPACITY;
    if (d->batch == 0) return SPEC_OK;
    if (!stream_logits || !root_token || !tokens || !tree_parent || !n_nodes)
        return SPEC_ERR_INVALID_ARG;
    DraftParams P{};
    P.B = d->batch;
    P.rows = d->n_stream_rows;
    P.gamma = d->gamma;
    P.k = d->k;
    P.V = d->vocab;
    P.max_nodes = d->max_nodes;
    P.vp_rows = d->vparent_rows;
    P.n_full = (int)n_full;
    P.logits = stream_logits;
    P.stream_row = stream_row;
    P.root_token = root_token;
    P.tokens = tokens;
    P.parent = tree_parent;
    P.n_nodes = n_nodes;
    P.vparent = vparent;
    P.status = status_ptr();
    if (!P.status) return SPEC_ERR_CUDA;
    dim3 grid(d->gamma, d->batch);
    cudaStream_t s = as_stream(stream);
    const spec_status_t ls =
        d->logit_dtype == SPEC_BF16
            ? launch(draft_tree_kernel<__nv_bfloat16>, grid, dim3(kDraftThreads), 0, s, P)
            : launch(draft_tree_kernel<float>, grid, dim3(kDraftThreads), 0, s, P);
    if (ls != SPEC_OK) return ls;
    return launch_status();
}

extern "C" spec_status_t spec_prune_tree(const spec_prune_desc *d, const int32_t *tokens,
                                         const int32_t *tree_parent, const int32_t *n_nodes,
                                         const void *early_logits, int32_t *keep_map,
                                         int32_t *tokens_out, int32_t *parent_out, int32_t *n_out,
                                         int32_t *vparent, void *stream) {
    using namespace sv;
    if (!d) return SPEC_ERR_INVALID_ARG;
    if (d->batch < 0 || d->max_nodes <= 0 || d->vocab <= 0 || d->gamma < 0 ||
        d->vparent_rows < 0 || !(d->threshold == d->threshold))
        return SPEC_ERR_INVALID_ARG;
    if (d->max_nodes > kMaxPruneNodes) return SPEC_ERR_UNSUPPORTED;
    if (d->logit_dtype != SPEC_F32 && d->logit_dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    if (vparent && (long long)d->max_nodes * (1 + d->gamma) > d->vparent_rows)
        return SPEC_ERR_CAPACITY;
    if (d->batch == 0) return SPEC_OK;
    if (!tokens || !tree_parent || !n_nodes || !early_logits || !keep_map || !tokens_out ||
        !parent_out || !n_out)
        return SPEC_ERR_INVALID_ARG;
    PruneParams P{};
    P.B = d->batch;
    P.N = d->max_nodes;
    P.V = d->vocab;
    P.gamma = d->gamma;
    P.vp_rows = d->vparent_rows;
    P.threshold = d->threshold;
    P.tokens = tokens;
    P.parent = tree_parent;
    P.n_nodes = n_nodes;
    P.early = early_logits;
    P.keep = keep_map;
    P.tokens_out = tokens_out;
    P.parent_out = parent_out;
    P.n_out = n_out;
    P.vparent = vparent;
    P.status = status_ptr();
    if (!P.status) return SPEC_ERR_CUDA;
    cudaStream_t s = as_stream(stream);
    dim3 grid(ceil_div(d->max_nodes, kEdgeNodesPerPart), d->batch);
    const spec_status_t ls =
        d->logit_dtype == SPEC_BF16
            ? launch(prune_edge_kernel<__nv_bfloat16>, grid, dim3(kThreads), 0, s, P)
            : launch(prune_edge_kernel<float>, grid, dim3(kThreads), 0, s, P);
    if (ls != SPEC_OK) return ls;
    spec_status_t st = launch_status();
    if (st != SPEC_OK) return st;
    if (launch(prune_compact_kernel, dim3(d->batch), dim3(kThreads), 0, s, P) != SPEC_OK)
        return SPEC_ERR_CUDA;
    return launch_status();
}
