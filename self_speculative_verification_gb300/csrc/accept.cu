// spec_vocab_reduce and spec_accept.
//
// Vocab reduce: per judged row, the greedy token (argmax, lowest index on
// ties), ln sum exp(z) and the proposal's logit -- what "Lookahead
// Attention" sec. 2.4 (proposal probability against a threshold) and
// "Speculative Streaming"'s verification step (hard matching against the
// greedy token) need.
//
// Accept: the LA threshold longest prefix, or the greedy walk down the draft
// tree ("Speculative Streaming", verification step; "ConFu" tree verify);
// spec_accept_soft: the soft-matching walk and the residual draw.
#include <atomic>
#include <cooperative_groups.h>
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "logits.cuh"
#include "ptx_sm103.cuh"
#include "row_scan.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kReduceThreads = 256;

// One thread-block cluster per row: CTA `rank` of the cluster reduces slice
// `rank` of the row, kUnroll 16-byte loads in flight per thread, one pass
// with a running (max, index, sum of exp).  Per batch of kUnroll * N
// elements: the batch max first; the index search and the rescale of the
// running sum only when the max rises (a thread visits its indices in
// increasing order, so an equal later value never wins a tie); then one
// FFMA + one ex2 per element.  Rank 0 merges the CTAs' results through
// distributed shared memory.
// bf16 batches without a ragged end take the packed arithmetic of
// push_bf16_batch.
template <typename T>
__global__ void __launch_bounds__(kReduceThreads)
vocab_reduce_kernel(const T *__restrict__ logits, int V, const int32_t *__restrict__ proposal,
                    int32_t *__restrict__ argmax, float *__restrict__ lse,
                    float *__restrict__ zprop, float inv_t) {
    pdl_wait();
    const float c2 = kLog2e * inv_t;
    cg::cluster_group cluster = cg::this_cluster();
    const int nc = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int row = blockIdx.x / nc;
    const T *z = logits + (size_t)row * V;
    Best best{-INFINITY, INT_MAX, 0.f};
    constexpr int N = Vec<T>::N;
    if ((reinterpret_cast<uintptr_t>(z) & 15) == 0) {
        const int nv = V / N;
        const int lo = (int)((long long)nv * rank / nc), hi = (int)((long long)nv * (rank + 1) / nc);
        int i0 = lo + threadIdx.x;
        if constexpr (N == 8) {
            // full batches
            const uint4 *zv = reinterpret_cast<const uint4 *>(z);
            for (; i0 + (kUnroll - 1) * kReduceThreads < hi; i0 += kReduceThreads * kUnroll) {
                Bf16Batch x;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const uint4 v = zv[i0 + u * kReduceThreads];
                    x.w[u][0] = v.x;
                    x.w[u][1] = v.y;
                    x.w[u][2] = v.z;
                    x.w[u][3] = v.w;
                }
                push_bf16_batch<kReduceThreads>(best, x, i0, c2);
            }
        }
        // the ragged last batch (all batches for fp32)
        for (; i0 < hi; i0 += kReduceThreads * kUnroll) {
            float x[kUnroll][N];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * kReduceThreads;
                if (i < hi) {
                    Vec<T>::load(z + (size_t)i * N, x[u]);
                } else {
#pragma unroll
                    for (int j = 0; j < N; ++j) x[u][j] = -INFINITY;
                }
            }
            float bm = x[0][0];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int j = 0; j < N; ++j) bm = fmaxf(bm, x[u][j]);
            if (bm > best.m) {
                int bi = INT_MAX;
#pragma unroll
                for (int u = kUnroll - 1; u >= 0; --u)
#pragma unroll
                    for (int j = N - 1; j >= 0; --j)
                        if (x[u][j] == bm) bi = (i0 + u * kReduceThreads) * N + j;
                best.s *= ex2((best.m - bm) * c2);
                best.m = bm;
                best.idx = bi;
            }
            const float mb = best.m * c2;
            float acc[N];
#pragma unroll
            for (int j = 0; j < N; ++j) acc[j] = 0.f;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int j = 0; j < N; ++j) acc[j] += ex2(fmaf(x[u][j], c2, -mb));
#pragma unroll
            for (int j = 1; j < N; ++j) acc[0] += acc[j];
            best.s += acc[0];
        }
        if (rank == nc - 1)
            for (int i = nv * N + threadIdx.x; i < V; i += kReduceThreads)
                best_push(best, load_f(z + i), i, inv_t);
    } else {
        const int lo = (int)((long long)V * rank / nc), hi = (int)((long long)V * (rank + 1) / nc);
        for (int i = lo + threadIdx.x; i < hi; i += kReduceThreads)
            best_push(best, load_f(z + i), i, inv_t);
    }

    // block reduction: warps, then across warps
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Best other;
        other.m = __shfl_xor_sync(0xffffffffu, best.m, o);
        other.idx = __shfl_xor_sync(0xffffffffu, best.idx, o);
        other.s = __shfl_xor_sync(0xffffffffu, best.s, o);
        best = best_merge(best, other, inv_t);
    }
    __shared__ Best sb[kReduceThreads / 32];
    __shared__ Best cta_best;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sb[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        Best r = sb[0];
        for (int w = 1; w < kReduceThreads / 32; ++w) r = best_merge(r, sb[w], inv_t);
        cta_best = r;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0) {
        Best r = cta_best;
        for (int i = 1; i < nc; ++i)
            r = best_merge(r, *cluster.map_shared_rank(&cta_best, i), inv_t);
        if (argmax) argmax[row] = r.idx == INT_MAX ? 0 : r.idx;
        lse[row] = r.m * inv_t + logf(r.s);
        if (proposal && zprop) {
            const int pidx = proposal[row];
            zprop[row] = (pidx >= 0 && pidx < V) ? load_f(z + pidx) : NAN;
        }
    }
    cluster.sync();     // peers' shared memory stays alive until rank 0 has read it
}

// The same reduction for bf16 rows whose start is 16-byte aligned, with the
// row slice streamed through shared memory (bulk_row_scan: thread 0 keeps
// kBulkStages chunks of bulk copies in flight ahead of the reducing
// threads).  CTAs are small (kBulkThreads threads, kBulkStages x 8 KB of
// shared memory) so that many fit on an SM: the host picks the CTAs per row
// so that every CTA is resident at once and the SMs' shares of the bytes are
// even (bulk_cluster_size).  A copy that has not landed within the bounded
// wait sets SPEC_DEV_TIMEOUT; the CTA then writes nothing.
constexpr int kBulkThreads = 128;
constexpr int kBulkStages = 3;
constexpr int kBulkSmem = bulk_smem<kBulkThreads, kBulkStages>();

__global__ void __launch_bounds__(kBulkThreads)
vocab_reduce_bulk_kernel(const __nv_bfloat16 *__restrict__ logits, int V,
                         const int32_t *__restrict__ proposal, int32_t *__restrict__ argmax,
                         float *__restrict__ lse, float *__restrict__ zprop, float inv_t,
                         int *status, long long wait) {
    pdl_wait();
    const float c2 = kLog2e * inv_t;
    cg::cluster_group cluster = cg::this_cluster();
    const int nc = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int row = blockIdx.x / nc;
    const __nv_bfloat16 *z = logits + (size_t)row * V;
    extern __shared__ __align__(128) uint8_t stage[];
    __shared__ uint64_t full[kBulkStages];
    Best best{-INFINITY, INT_MAX, 0.f};
    // this CTA's slice: 8-element vectors [lo, hi) of the row
    const int nv = V / 8;
    const int lo = (int)((long long)nv * rank / nc), hi = (int)((long long)nv * (rank + 1) / nc);
    const int n_el = (hi - lo) * 8;
    const bool failed = !bulk_row_scan<kBulkThreads, kBulkStages>(z + (size_t)lo * 8, n_el, lo, c2,
                                                                   best, stage, full, wait);
    if (failed && threadIdx.x == 0) raise_status(status, SPEC_DEV_TIMEOUT);
    if (rank == nc - 1)
        for (int i = nv * 8 + threadIdx.x; i < V; i += kBulkThreads)
            best_push(best, load_f(z + i), i, inv_t);

    // block reduction: warps, then across warps
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Best other;
        other.m = __shfl_xor_sync(0xffffffffu, best.m, o);
        other.idx = __shfl_xor_sync(0xffffffffu, best.idx, o);
        other.s = __shfl_xor_sync(0xffffffffu, best.s, o);
        best = best_merge(best, other, inv_t);
    }
    __shared__ Best sb[kBulkThreads / 32];
    __shared__ Best cta_best;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sb[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        Best r = sb[0];
        for (int w = 1; w < kBulkThreads / 32; ++w) r = best_merge(r, sb[w], inv_t);
        cta_best = r;
    }
    cluster.sync();
    if (rank == 0 && threadIdx.x == 0 && !failed) {
        Best r = cta_best;
        for (int i = 1; i < nc; ++i)
            r = best_merge(r, *cluster.map_shared_rank(&cta_best, i), inv_t);
        if (argmax) argmax[row] = r.idx == INT_MAX ? 0 : r.idx;
        lse[row] = r.m * inv_t + logf(r.s);
        if (proposal && zprop) {
            const int pidx = proposal[row];
            zprop[row] = (pidx >= 0 && pidx < V) ? load_f(z + pidx) : NAN;
        }
    }
    cluster.sync();     // peers' shared memory stays alive until rank 0 has read it
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
    pdl_wait();
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
        // Node c's parent, token and judge row's argmax live in lane c % 32,
        // slot c / 32; the walk is then shuffles and ballots only.
        constexpr int kSlots = SPEC_MAX_ROWS / 32;
        int par[kSlots], tok[kSlots], am[kSlots];   // am = -1: judge row out of range
#pragma unroll
        for (int k = 0; k < kSlots; ++k) {
            const int c = k * 32 + lane;
            par[k] = -3;
            tok[k] = 0;
            am[k] = -1;
            if (c < n) {
                par[k] = P.tree_parent[(size_t)b * P.N + c];
                tok[k] = P.tokens[(size_t)b * P.N + c];
                const int row = P.row_of ? P.row_of[(size_t)b * P.N + c] : c;
                if (row >= 0 && row < P.Rj) am[k] = P.argmax[(size_t)b * P.Rj + row];
            }
        }
        int cur = 0;
        if (n == 0 || P.path_cap == 0) {
            if (lane == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
        } else {
            len = 1;
            if (lane == 0) pth[0] = 0;
            while (true) {
                // argmax of the current node's judge row, from its lane
                int want = 0;
#pragma unroll
                for (int k = 0; k < kSlots; ++k)
                    if (k == (cur >> 5)) want = __shfl_sync(0xffffffffu, am[k], cur & 31);
                if (want < 0) {           // judge row out of range
                    if (lane == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
                    next = -1;
                    break;
                }
                next = want;
                // lowest-index child of cur carrying the wanted token
                int found = -1;
#pragma unroll
                for (int k = 0; k < kSlots; ++k) {
                    const unsigned bal = __ballot_sync(0xffffffffu, par[k] == cur && tok[k] == want &&
                                                                         k * 32 + lane > cur);
                    if (found < 0 && bal) found = k * 32 + __ffs(bal) - 1;
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

// CTAs per row: the smallest power of two giving at least two CTAs per SM
// (at most 8, each slice at least 16 KB).  Measured on GB300 (bf16, L2
// cold, CUDA-graph timing): 512 x 50272 logits take 15.8 us with one CTA
// per row against 22.3 us with four; 96 rows need four to fill the GPU.
int cluster_size(int n_rows, int V, int dtype) {
    const long long row_bytes = (long long)V * (dtype == SPEC_BF16 ? 2 : 4);
    int nc = 1;
    while (nc < 8 && row_bytes / (2 * nc) >= 16384 && (long long)n_rows * nc < 2ll * num_sms())
        nc *= 2;
    return nc;
}

// Resident bulk-kernel CTAs per SM on the current device (cached).
int bulk_ctas_per_sm() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const int slot = dev & 63;
    int n = cached[slot].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (set_smem_limit(reinterpret_cast<const void *>(vocab_reduce_bulk_kernel), kBulkSmem) !=
            SPEC_OK ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, vocab_reduce_bulk_kernel, kBulkThreads,
                                                      kBulkSmem) != cudaSuccess ||
        n < 1) {
        (void)cudaGetLastError();
        return 1;
    }
    cached[slot].store(n, std::memory_order_relaxed);
    return n;
}

// CTAs per row for the bulk kernel: among the cluster sizes 1, 2, 4, 8 whose
// CTAs are all resident at once (rows x nc <= resident CTAs per SM x SMs;
// slices of at least 16 KB), the one whose busiest SM streams the fewest
// bytes, ceil(rows x nc / SMs) slices of row/nc bytes each; the smaller on
// ties.  With one CTA per row, 480 rows on 152 SMs leave 24 SMs four rows
// and the rest three: the last quarter of the kernel ran on those 24 alone.
int bulk_cluster_size(int n_rows, int V) {
    const long long row_bytes = 2ll * V;
    const long long sms = num_sms();
    const long long slots = sms * bulk_ctas_per_sm();
    int best = 1;
    long long best_busy = ceil_div_ll(n_rows, sms);     // slices on the busiest SM, nc = 1
    for (int nc = 2; nc <= 8; nc *= 2) {
        if (row_bytes / nc < 16384 || (long long)n_rows * nc > slots) break;
        const long long busy = ceil_div_ll((long long)n_rows * nc, sms);
        if (busy * best < best_busy * nc) {      // busy / nc < best_busy / best
            best = nc;
            best_busy = busy;
        }
    }
    return best;
}

template <typename T>
spec_status_t launch_vocab_cluster(const void *logits, int n_rows, int V, int nc,
                                   const int32_t *proposal, int32_t *argmax, float *lse,
                                   float *zprop, float inv_t, cudaStream_t s) {
    // bf16 rows that start on 16-byte boundaries stream through shared
    // memory (vocab_reduce_bulk_kernel)
    const bool bulk = sizeof(T) == 2 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0 &&
                      (V % 8) == 0;
    int *status = nullptr;
    if (bulk) {
        status = status_ptr();
        if (!status) return SPEC_ERR_CUDA;
        if (set_smem_limit(reinterpret_cast<const void *>(vocab_reduce_bulk_kernel), kBulkSmem) !=
            SPEC_OK)
            return SPEC_ERR_CUDA;
        nc = bulk_cluster_size(n_rows, V);
    }
    if ((long long)n_rows * nc > 2147483647ll) return SPEC_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)((long long)n_rows * nc), 1, 1);
    cfg.blockDim = dim3(bulk ? kBulkThreads : kReduceThreads, 1, 1);
    cfg.dynamicSmemBytes = bulk ? kBulkSmem : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = nc;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e =
        bulk ? cudaLaunchKernelEx(&cfg, vocab_reduce_bulk_kernel,
                                  static_cast<const __nv_bfloat16 *>(logits), V, proposal, argmax,
                                  lse, zprop, inv_t, status, wait_limit())
             : cudaLaunchKernelEx(&cfg, vocab_reduce_kernel<T>, static_cast<const T *>(logits), V,
                                  proposal, argmax, lse, zprop, inv_t);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t launch_vocab_reduce(const void *logits, int dtype, int n_rows, int V,
                                  const int32_t *proposal, int32_t *argmax, float *lse,
                                  float *zprop, cudaStream_t s, float inv_t = 1.f) {
    const int nc = cluster_size(n_rows, V, dtype);
    if ((long long)n_rows * nc > 2147483647ll) return SPEC_ERR_UNSUPPORTED;
    if (dtype == SPEC_BF16)
        return launch_vocab_cluster<__nv_bfloat16>(logits, n_rows, V, nc, proposal, argmax, lse,
                                                   zprop, inv_t, s);
    return launch_vocab_cluster<float>(logits, n_rows, V, nc, proposal, argmax, lse, zprop, inv_t,
                                       s);
}

// ------------------------------------------------------------ soft matching
//
// "Speculative Streaming", verification step with soft matching: a drafted
// token x (child of the current node) is accepted with probability
// min(1, p(x) / q(x)), decided as u_x * q(x) < p(x); children are tried in
// index order and the first accepted one is followed.  At the stop node one
// correction token is drawn from the normalised residual max(0, p - q) (from
// p when the node has no drafted children or the residual has no mass), as
// the smallest v whose cumulative mass exceeds u_b times the total.
// p = softmax(z / T) of the node's judge row, q = softmax(z_d / T) of the
// draft row its children were drafted from.

constexpr int kSoftThreads = 512;
constexpr int kSoftTile = 256;             // vocab entries per tile: 8 per lane
constexpr int kMaxSoftTiles = 4096;        // vocab <= 1,048,576

struct SoftParams {
    int B, Rj, Rd, N, V, path_cap;
    float inv_t;
    const void *logits, *draft;
    const int32_t *tokens, *tree_parent, *row_of, *child_draft_row, *n_nodes;
    const float *u_accept, *u_sample, *lse_t, *lse_d;
    int32_t *acc_len, *path, *next_token, *last_node;
    int *status;
};

template <typename T>
__device__ __forceinline__ float prob_at(const T *row, int v, float lse, float inv_t) {
    return __expf(fmaf(load_f(row + v), inv_t, -lse));
}

// One CTA per request.  Every node's test against its parent's rows is
// independent of the walk, so all threads evaluate them at once; thread 0
// then walks the tree in shared memory, and the CTA draws the correction
// token (tile sums, a scan over tiles, a scan inside the tile).
template <typename T>
__global__ void __launch_bounds__(kSoftThreads) soft_accept_kernel(SoftParams P) {
    pdl_wait();
    __shared__ float s_tile[kMaxSoftTiles];
    __shared__ int s_par[SPEC_MAX_ROWS];
    __shared__ uint8_t s_acc[SPEC_MAX_ROWS];
    __shared__ int s_row, s_drow;
    __shared__ float s_total;
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const T *Z = static_cast<const T *>(P.logits);
    const T *ZD = static_cast<const T *>(P.draft);
    const size_t nb = (size_t)b * P.N;

    int n = P.n_nodes[b];
    if (n < 0 || n > P.N) {
        if (threadIdx.x == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
        n = n < 0 ? 0 : P.N;
    }
    // row / draft row of node c's judge distribution (-1 / -2: malformed)
    auto rows_of = [&](int c, int &row, int &drow) {
        row = P.row_of ? P.row_of[nb + c] : c;
        if (row < 0 || row >= P.Rj) row = -1;
        drow = P.child_draft_row ? P.child_draft_row[nb + c] : -1;
        if (drow < -1 || drow >= P.Rd) drow = -2;
    };
    // 1. node c (token x, parent a) is accepted iff u_c q_a(x) < p_a(x)
    for (int c = threadIdx.x; c < n; c += kSoftThreads) {
        const int a = P.tree_parent[nb + c];
        s_par[c] = a;
        uint8_t acc = 0;
        if (c > 0 && a >= 0 && a < c) {
            int row, drow;
            rows_of(a, row, drow);
            const int x = P.tokens[nb + c];
            if (row < 0 || drow == -2 || x < 0 || x >= P.V) {
                raise_status(P.status, SPEC_DEV_BAD_INDEX);
            } else {
                const float p = prob_at(Z + ((size_t)b * P.Rj + row) * P.V, x,
                                        P.lse_t[(size_t)b * P.Rj + row], P.inv_t);
                const float q = drow >= 0 ? prob_at(ZD + ((size_t)b * P.Rd + drow) * P.V, x,
                                                    P.lse_d[(size_t)b * P.Rd + drow], P.inv_t)
                                          : 0.f;
                acc = P.u_accept[nb + c] * q < p;
            }
        }
        s_acc[c] = acc;
    }
    __syncthreads();
    // 2. the walk: the lowest-index accepted child of the current node
    if (threadIdx.x == 0) {
        int32_t *pth = P.path + (size_t)b * P.path_cap;
        int len = 0, cur = 0, row = -1, drow = -1;
        if (n == 0 || P.path_cap == 0) {
            raise_status(P.status, SPEC_DEV_BAD_INDEX);
        } else {
            len = 1;
            pth[0] = 0;
            while (true) {
                int found = -1;
                for (int c = cur + 1; c < n; ++c)
                    if (s_par[c] == cur && s_acc[c]) {
                        found = c;
                        break;
                    }
                if (found < 0) break;
                if (len >= P.path_cap) {
                    raise_status(P.status, SPEC_DEV_BAD_INDEX);
                    break;
                }
                pth[len++] = found;
                cur = found;
            }
            rows_of(cur, row, drow);
            if (row < 0 || drow == -2) {
                raise_status(P.status, SPEC_DEV_BAD_INDEX);
                drow = -1;
            }
        }
        for (int i = len; i < P.path_cap; ++i) pth[i] = -1;
        P.acc_len[b] = len;
        P.last_node[b] = len > 0 ? cur : -1;
        s_row = row;
        s_drow = drow;
    }
    __syncthreads();
    const int row = s_row;
    if (row < 0) {
        if (threadIdx.x == 0) P.next_token[b] = -1;
        return;
    }
    // 3. the correction token
    const int drow = s_drow;
    const T *zt = Z + ((size_t)b * P.Rj + row) * P.V;
    const float lt = P.lse_t[(size_t)b * P.Rj + row];
    const T *zd = drow >= 0 ? ZD + ((size_t)b * P.Rd + drow) * P.V : nullptr;
    const float ld = drow >= 0 ? P.lse_d[(size_t)b * P.Rd + drow] : 0.f;
    const int ntiles = (P.V + kSoftTile - 1) / kSoftTile;
    const bool vec = (reinterpret_cast<uintptr_t>(zt) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(zd) & 15) == 0;
    bool resid = zd != nullptr;
    const float c2 = P.inv_t * kLog2e, lt2 = lt * kLog2e, ld2 = ld * kLog2e;
    // masses of the 8 entries v0 .. v0 + 7 (0 past the vocabulary)
    auto mass8 = [&](int v0, float (&m)[8]) {
        float a[8], q[8];
        if (vec && v0 + 8 <= P.V) {
            load8(zt + v0, a);
            if (resid) load8(zd + v0, q);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                a[e] = v0 + e < P.V ? load_f(zt + v0 + e) : -INFINITY;
                q[e] = (resid && v0 + e < P.V) ? load_f(zd + v0 + e) : -INFINITY;
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float p = ex2(fmaf(a[e], c2, -lt2));
            m[e] = resid ? fmaxf(0.f, p - ex2(fmaf(q[e], c2, -ld2))) : p;
        }
    };
    constexpr int kWarps = kSoftThreads / 32;
    for (int pass = 0; pass < 2; ++pass) {
        for (int t = warp; t < ntiles; t += 2 * kWarps) {
            const int t2 = t + kWarps;
            float m0[8], m1[8];
            mass8(t * kSoftTile + lane * 8, m0);
            if (t2 < ntiles) {
                mass8(t2 * kSoftTile + lane * 8, m1);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) m1[e] = 0.f;
            }
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                s0 += m0[e];
                s1 += m1[e];
            }
            s0 = warp_sum(s0);
            s1 = warp_sum(s1);
            if (lane == 0) {
                s_tile[t] = s0;
                if (t2 < ntiles) s_tile[t2] = s1;
            }
        }
        __syncthreads();
        if (warp == 0) {
            float acc = 0.f;
            for (int t = lane; t < ntiles; t += 32) acc += s_tile[t];
            acc = warp_sum(acc);
            if (lane == 0) s_total = acc;
        }
        __syncthreads();
        if (s_total > 0.f || !resid) break;
        resid = false;           // p <= q everywhere: draw from p
        __syncthreads();
    }
    if (warp != 0) return;
    // the tile holding the target: lane l scans tiles [l K, (l + 1) K)
    const float total = s_total;
    const float target = P.u_sample[b] * total;
    const int K = (ntiles + 31) / 32;
    const int t0 = min(lane * K, ntiles), t1 = min(t0 + K, ntiles);
    float lsum = 0.f;
    for (int t = t0; t < t1; ++t) lsum += s_tile[t];
    float incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned hitl = __ballot_sync(0xffffffffu, incl > target && t0 < t1);
    int tile = -1;
    float base = 0.f;
    if (hitl) {
        const int L = __ffs(hitl) - 1;
        if (lane == L) {
            float run = incl - lsum;
            for (int t = t0; t < t1; ++t) {
                if (run + s_tile[t] > target) {
                    tile = t;
                    break;
                }
                run += s_tile[t];
            }
            if (tile < 0) tile = t1 - 1;
            base = run;
        }
        tile = __shfl_sync(0xffffffffu, tile, L);
        base = __shfl_sync(0xffffffffu, base, L);
    } else {
        // rounding put the target at the very end: the last tile with mass
        int last = -1;
        for (int t = lane; t < ntiles; t += 32)
            if (s_tile[t] > 0.f) last = t;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
        tile = last < 0 ? 0 : last;
        base = -INFINITY;        // take the last element with mass below
    }
    // inside the tile: lane l holds entries [l * 8, l * 8 + 8)
    const int v0 = tile * kSoftTile + lane * 8;
    float m[8], part = 0.f;
    mass8(v0, m);
#pragma unroll
    for (int e = 0; e < 8; ++e) part += m[e];
    float ip = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, ip, o);
        if (lane >= o) ip += y;
    }
    int mine = -1, lastpos = -1;
    float run = base + (ip - part);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        run += m[e];
        if (mine < 0 && m[e] > 0.f && run > target) mine = v0 + e;
        if (m[e] > 0.f) lastpos = v0 + e;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, mine >= 0);
    int tok;
    if (hit) {
        tok = __shfl_sync(0xffffffffu, mine, __ffs(hit) - 1);
    } else {
        tok = lastpos;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tok = max(tok, __shfl_xor_sync(0xffffffffu, tok, o));
        if (tok < 0) tok = 0;
    }
    if (lane == 0) P.next_token[b] = tok;
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
    } else {
        if (!tree_parent) return SPEC_ERR_INVALID_ARG;
        if (d->max_nodes > SPEC_MAX_ROWS) return SPEC_ERR_UNSUPPORTED;   // walk keeps nodes in registers
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
    if (sv::launch(sv::accept_kernel, dim3(sv::ceil_div(P.B, 4)), dim3(128), 0, s, P) != SPEC_OK)
        return SPEC_ERR_CUDA;
    return sv::launch_status();
}

extern "C" spec_status_t spec_accept_soft(const spec_soft_desc *d, const void *logits,
                                          const void *draft_logits, const int32_t *tokens,
                                          const int32_t *tree_parent, const int32_t *row_of,
                                          const int32_t *child_draft_row, const int32_t *n_nodes,
                                          const float *u_accept, const float *u_sample,
                                          float *lse_t, float *lse_d, int32_t *acc_len,
                                          int32_t *path, int32_t *next_token, int32_t *last_node,
                                          void *stream) {
    using namespace sv;
    if (!d) return SPEC_ERR_INVALID_ARG;
    if (d->batch < 0 || d->n_judge_rows <= 0 || d->n_draft_rows < 0 || d->vocab <= 0 ||
        d->max_nodes <= 0 || d->path_cap < 0 || !(d->temperature > 0.f) ||
        !(d->temperature < INFINITY))
        return SPEC_ERR_INVALID_ARG;
    if (d->logit_dtype != SPEC_F32 && d->logit_dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    if ((d->vocab + kSoftTile - 1) / kSoftTile > kMaxSoftTiles) return SPEC_ERR_UNSUPPORTED;
    if (d->max_nodes > SPEC_MAX_ROWS) return SPEC_ERR_UNSUPPORTED;
    if (d->batch == 0) return SPEC_OK;
    if (!logits || !tokens || !tree_parent || !n_nodes || !u_accept || !u_sample || !lse_t ||
        !acc_len || !path || !next_token || !last_node)
        return SPEC_ERR_INVALID_ARG;
    if (d->n_draft_rows > 0 && (!draft_logits || !lse_d || !child_draft_row))
        return SPEC_ERR_INVALID_ARG;
    const long long rows = (long long)d->batch * d->n_judge_rows;
    const long long drows = (long long)d->batch * d->n_draft_rows;
    if (rows > 2147483647ll || drows > 2147483647ll) return SPEC_ERR_UNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    const float inv_t = 1.f / d->temperature;
    spec_status_t st = launch_vocab_reduce(logits, d->logit_dtype, (int)rows, d->vocab, nullptr,
                                           nullptr, lse_t, nullptr, s, inv_t);
    if (st != SPEC_OK) return st;
    if (drows > 0) {
        st = launch_vocab_reduce(draft_logits, d->logit_dtype, (int)drows, d->vocab, nullptr,
                                 nullptr, lse_d, nullptr, s, inv_t);
        if (st != SPEC_OK) return st;
    }
    SoftParams P{};
    P.B = d->batch;
    P.Rj = d->n_judge_rows;
    P.Rd = d->n_draft_rows;
    P.N = d->max_nodes;
    P.V = d->vocab;
    P.path_cap = d->path_cap;
    P.inv_t = inv_t;
    P.logits = logits;
    P.draft = d->n_draft_rows > 0 ? draft_logits : nullptr;
    P.tokens = tokens;
    P.tree_parent = tree_parent;
    P.row_of = row_of;
    P.child_draft_row = d->n_draft_rows > 0 ? child_draft_row : nullptr;
    P.n_nodes = n_nodes;
    P.u_accept = u_accept;
    P.u_sample = u_sample;
    P.lse_t = lse_t;
    P.lse_d = lse_d;
    P.acc_len = acc_len;
    P.path = path;
    P.next_token = next_token;
    P.last_node = last_node;
    P.status = status_ptr();
    if (!P.status) return SPEC_ERR_CUDA;
    const spec_status_t ls =
        d->logit_dtype == SPEC_BF16
            ? launch(soft_accept_kernel<__nv_bfloat16>, dim3(P.B), dim3(kSoftThreads), 0, s, P)
            : launch(soft_accept_kernel<float>, dim3(P.B), dim3(kSoftThreads), 0, s, P);
    if (ls != SPEC_OK) return ls;
    return launch_status();
}
