// kv_commit: append the accepted block rows to the committed cache.
//
// "Lookahead Attention" sec. 3.2: speculative K/V lives only for the current
// pass; "Speculative Streaming": the cache holds main-stream tokens only and
// pruned entries are removed after the step.  Here the block K/V sits in its
// own buffer, so dropping the rejected rows costs nothing: only the accepted
// rows are copied, in path order, to positions seq_len[b], seq_len[b]+1, ...
//
// Two launches: the copy kernel reads the old bookkeeping (seq_len, page
// table, free_head) and writes the K/V bytes; the finalize kernel then
// updates the bookkeeping.  Page allocation is deterministic: requests in
// ascending order, each first fills its partly used last page, then takes
// pages from the free list in order.
#include "common.cuh"

namespace sv {
namespace {

struct CommitParams {
    char *kc, *vc;                 // cache K/V (bytes)
    const char *kb, *vb;           // block K/V (bytes)
    int32_t *page_table;
    const int32_t *path, *acc_len;
    int32_t *seq_len;
    const int32_t *free_pages;
    int32_t *free_head;
    int n_free;
    int B, Hkv, R, path_cap, row_bytes;
    int blk_bytes, vec_per_blk;    // paged: bytes / 16-byte vectors of a 64-element block
    int paged, max_seq, page_size, max_pages, n_pages, capacity;
    int *status;
};

// Accepted rows of request b that will be written (0 when the request is
// skipped), with the reason bits for a skip.
__device__ __forceinline__ int effective_acc(const CommitParams &P, int b, int *bits) {
    const int a = P.acc_len[b];
    const int S = P.seq_len[b];
    if (a < 0 || a > P.path_cap) {
        *bits |= SPEC_DEV_BAD_INDEX;
        return 0;
    }
    if (S < 0 || S > P.capacity) {
        *bits |= SPEC_DEV_SEQ_OVERFLOW;
        return 0;
    }
    if ((long long)S + a > P.capacity) {
        *bits |= SPEC_DEV_CAPACITY;
        return 0;
    }
    return a;
}

__device__ __forceinline__ int pages_for(int tokens, int ps) { return (tokens + ps - 1) / ps; }

__device__ __forceinline__ int new_pages(const CommitParams &P, int b) {
    int bits = 0;
    const int a = effective_acc(P, b, &bits);
    const int S = P.seq_len[b];
    return a ? pages_for(S + a, P.page_size) - pages_for(S, P.page_size) : 0;
}

// Block-wide sums over requests: pages taken by requests before b and by all.
__device__ void page_prefix(const CommitParams &P, int b, int *before, int *total) {
    __shared__ int s_before[32], s_total[32];
    int mb = 0, mt = 0;
    for (int i = threadIdx.x; i < P.B; i += blockDim.x) {
        const int n = new_pages(P, i);
        mt += n;
        if (i < b) mb += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mb += __shfl_xor_sync(0xffffffffu, mb, o);
        mt += __shfl_xor_sync(0xffffffffu, mt, o);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        s_before[warp] = mb;
        s_total[warp] = mt;
    }
    __syncthreads();
    int tb = 0, tt = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        tb += s_before[w];
        tt += s_total[w];
    }
    __syncthreads();
    *before = tb;
    *total = tt;
}

// One CTA per (request, KV head): copies every accepted row, K and V.
__global__ void __launch_bounds__(128) kv_commit_copy_kernel(CommitParams P) {
    pdl_wait();
    const int b = blockIdx.x / P.Hkv, h = blockIdx.x % P.Hkv;
    int before = 0, total = 0;
    int head = 0;
    if (P.paged) {
        page_prefix(P, b, &before, &total);
        head = *P.free_head;
        if (head < 0 || (long long)head + total > P.n_free) {
            if (blockIdx.x == 0 && threadIdx.x == 0) raise_status(P.status, SPEC_DEV_CAPACITY);
            return;
        }
    }
    int bits = 0;
    const int a = effective_acc(P, b, &bits);
    if (bits && h == 0 && threadIdx.x == 0) raise_status(P.status, bits);
    if (a == 0) return;
    const int S = P.seq_len[b];
    const int used = P.paged ? pages_for(S, P.page_size) : 0;
    const int vec_per_row = P.row_bytes / 16;
    const int work = a * vec_per_row;
    for (int w = threadIdx.x; w < work; w += blockDim.x) {
        const int i = w / vec_per_row, v = w % vec_per_row;
        const int row = P.path[(size_t)b * P.path_cap + i];
        if (row < 0 || row >= P.R) {
            if (v == 0) raise_status(P.status, SPEC_DEV_BAD_INDEX);
            continue;
        }
        const int pos = S + i;
        size_t dst;
        if (!P.paged) {
            dst = (((size_t)b * P.Hkv + h) * P.max_seq + pos) * P.row_bytes + (size_t)v * 16;
        } else {
            const int j = pos / P.page_size;
            const int page = j < used ? P.page_table[(size_t)b * P.max_pages + j]
                                      : P.free_pages[head + before + (j - used)];
            if (page < 0 || page >= P.n_pages) {
                if (v == 0) raise_status(P.status, SPEC_DEV_BAD_PAGE);
                continue;
            }
            // [page][head][d / 64][page_size][64]: 16-byte vector v of the row
            // lies in 64-element block v / vec_per_blk
            const int blk = v / P.vec_per_blk, vin = v % P.vec_per_blk;
            dst = (((size_t)page * P.Hkv + h) * (P.row_bytes / P.blk_bytes) + blk) *
                      P.page_size * P.blk_bytes +
                  (size_t)(pos % P.page_size) * P.blk_bytes + (size_t)vin * 16;
        }
        const size_t src = (((size_t)b * P.Hkv + h) * P.R + row) * P.row_bytes;
        const uint4 kx = reinterpret_cast<const uint4 *>(P.kb + src)[v];
        const uint4 vx = reinterpret_cast<const uint4 *>(P.vb + src)[v];
        *reinterpret_cast<uint4 *>(P.kc + dst) = kx;
        *reinterpret_cast<uint4 *>(P.vc + dst) = vx;
    }
}

// One CTA: new page-table entries, seq_len += accepted, free_head += taken.
__global__ void __launch_bounds__(256) kv_commit_finalize_kernel(CommitParams P) {
    pdl_wait();
    int head = 0, total = 0;
    if (P.paged) {
        int dummy = 0;
        page_prefix(P, 0, &dummy, &total);
        head = *P.free_head;
        if (head < 0 || (long long)head + total > P.n_free) return;
    }
    __syncthreads();   // every thread has read free_head
    // exclusive prefix of new pages over requests, in chunks of blockDim
    __shared__ int s_scan[256];
    int carry = 0;
    for (int base = 0; base < P.B; base += blockDim.x) {
        const int b = base + threadIdx.x;
        int bits = 0;
        const int a = b < P.B ? effective_acc(P, b, &bits) : 0;
        const int S = b < P.B ? P.seq_len[b] : 0;
        const int n = (P.paged && a) ? pages_for(S + a, P.page_size) - pages_for(S, P.page_size) : 0;
        s_scan[threadIdx.x] = n;
        __syncthreads();
        for (int o = 1; o < (int)blockDim.x; o <<= 1) {
            const int x = threadIdx.x >= o ? s_scan[threadIdx.x - o] : 0;
            __syncthreads();
            s_scan[threadIdx.x] += x;
            __syncthreads();
        }
        const int excl = carry + s_scan[threadIdx.x] - n;
        const int chunk_total = s_scan[blockDim.x - 1];
        __syncthreads();
        if (b < P.B && a > 0) {
            if (P.paged) {
                const int used = pages_for(S, P.page_size);
                for (int k = 0; k < n; ++k)
                    P.page_table[(size_t)b * P.max_pages + used + k] = P.free_pages[head + excl + k];
            }
            P.seq_len[b] = S + a;
        }
        carry += chunk_total;
    }
    if (P.paged && threadIdx.x == 0) *P.free_head = head + total;
}

}  // namespace
}  // namespace sv

extern "C" spec_status_t kv_commit(const spec_kv_desc *cache, int batch, int n_rows,
                                   const void *kb, const void *vb, int path_cap,
                                   const int32_t *path, const int32_t *acc_len, int32_t *seq_len,
                                   const int32_t *free_pages, int n_free, int32_t *free_head,
                                   void *stream) {
    if (!cache || batch < 0 || n_rows <= 0 || path_cap < 0) return SPEC_ERR_INVALID_ARG;
    if (cache->dtype != SPEC_F32 && cache->dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    if (cache->n_kv_heads <= 0 || cache->head_dim <= 0 || cache->batch < batch)
        return SPEC_ERR_INVALID_ARG;
    const int es = cache->dtype == SPEC_BF16 ? 2 : 4;
    const int row_bytes = cache->head_dim * es;
    if (row_bytes % 16 != 0) return SPEC_ERR_UNSUPPORTED;
    if (cache->kind == SPEC_KV_PAGED && cache->head_dim % 64 != 0) return SPEC_ERR_UNSUPPORTED;
    if (batch == 0) return SPEC_OK;
    if (!kb || !vb || !path || !acc_len || !seq_len || !cache->k || !cache->v)
        return SPEC_ERR_INVALID_ARG;
    if ((long long)batch * cache->n_kv_heads > 2147483647ll) return SPEC_ERR_UNSUPPORTED;
    sv::CommitParams P{};
    P.kc = static_cast<char *>(cache->k);
    P.vc = static_cast<char *>(cache->v);
    P.kb = static_cast<const char *>(kb);
    P.vb = static_cast<const char *>(vb);
    P.path = path;
    P.acc_len = acc_len;
    P.seq_len = seq_len;
    P.B = batch;
    P.Hkv = cache->n_kv_heads;
    P.R = n_rows;
    P.path_cap = path_cap;
    P.row_bytes = row_bytes;
    P.blk_bytes = 64 * es;
    P.vec_per_blk = 64 * es / 16;
    if (cache->kind == SPEC_KV_CONTIGUOUS) {
        if (cache->max_seq < 0) return SPEC_ERR_INVALID_ARG;
        P.paged = 0;
        P.max_seq = cache->max_seq;
        P.capacity = cache->max_seq;
    } else if (cache->kind == SPEC_KV_PAGED) {
        if (cache->page_size <= 0 || cache->max_pages_per_seq <= 0 || cache->n_pages <= 0 ||
            !cache->page_table || !free_pages || !free_head || n_free < 0)
            return SPEC_ERR_INVALID_ARG;
        if ((long long)cache->max_pages_per_seq * cache->page_size > (1ll << 30))
            return SPEC_ERR_UNSUPPORTED;
        P.paged = 1;
        P.page_size = cache->page_size;
        P.max_pages = cache->max_pages_per_seq;
        P.n_pages = cache->n_pages;
        P.capacity = cache->max_pages_per_seq * cache->page_size;
        P.page_table = cache->page_table;
        P.free_pages = free_pages;
        P.free_head = free_head;
        P.n_free = n_free;
    } else {
        return SPEC_ERR_INVALID_ARG;
    }
    P.status = sv::status_ptr();
    if (!P.status) return SPEC_ERR_CUDA;
    cudaStream_t s = sv::as_stream(stream);
    if (sv::launch(sv::kv_commit_copy_kernel, dim3(batch * P.Hkv), dim3(128), 0, s, P) != SPEC_OK)
        return SPEC_ERR_CUDA;
    spec_status_t st = sv::launch_status();
    if (st != SPEC_OK) return st;
    if (sv::launch(sv::kv_commit_finalize_kernel, dim3(1), dim3(256), 0, s, P) != SPEC_OK)
        return SPEC_ERR_CUDA;
    return sv::launch_status();
}
