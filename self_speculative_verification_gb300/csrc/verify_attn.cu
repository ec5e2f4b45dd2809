// spec_verify_attn: masked attention of the speculative rows over
// (committed prefix || soft prompt || block), split-KV, plus the combine.
//
// What is computed ("Speculative Streaming" Eq. 1-2 and Eq. 4; "Lookahead
// Attention" sec. 3.1; "ConFu" key design 1): for every valid row r and
// query head h, O = softmax(q K^T * scale + mask) V over the visible columns
// and LSE = ln sum exp(q k * scale).  Masked columns are excluded, not added
// as -inf arithmetic.
//
// This file holds the host planning, the CUDA-core kernel (fp32 inputs, and
// any shape the tensor-core kernel does not take) and the combine kernel.
#include <math.h>

#include "attn_common.cuh"
#include "attn_tc.cuh"

namespace sv {
namespace {

constexpr int kSimtRows = 16;   // packed rows per CTA (4 warps x 4 rows)
constexpr int kSimtCols = 32;   // columns per tile (one per lane)

// First element of token t's K (or V) row for head h; element k of the row
// is at row + (k / 64) * block_stride(P) + k % 64 (paged caches split the
// head dimension into 64-element blocks of page_size rows).
template <typename T>
__device__ __forceinline__ const T *prefix_row(const AttnParams &P, const T *base, int b, int h,
                                               int t, bool *bad) {
    if (!P.paged) return base + (((size_t)b * P.Hkv + h) * P.max_seq + t) * P.d;
    const int page = P.page_table[(size_t)b * P.max_pages + t / P.page_size];
    if (page < 0 || page >= P.n_pages) {
        *bad = true;
        return nullptr;
    }
    return base + ((size_t)page * P.Hkv + h) * P.page_size * P.d + (t % P.page_size) * 64;
}

__device__ __forceinline__ int block_stride(const AttnParams &P, int kind_prefix) {
    return (kind_prefix && P.paged) ? P.page_size * 64 : 64;
}

// Column kinds of a tile.
enum { kColPrefix = 0, kColSoft = 1, kColBlock = 2 };

template <typename T, int D>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnParams P) {
    pdl_wait();
    __shared__ float sq[kSimtRows][D];
    __shared__ float sk[kSimtCols][D + 1];
    __shared__ float sv_[kSimtCols][D];
    __shared__ uint32_t svis[kSimtRows][SPEC_MAX_ROWS / 32];
    __shared__ uint8_t sflags[kSimtRows];

    const int split = blockIdx.x;
    const int h = blockIdx.y / P.n_rb;
    const int rb = blockIdx.y % P.n_rb;
    const int b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const int S = clamp_seq(P, b, split == 0 && blockIdx.y == 0 && tid == 0);
    const int nsp = n_splits_of(P, S);
    if (split >= nsp) return;
    const int t0 = split * P.chunk;
    const int t1 = min(S, t0 + P.chunk);
    const bool last = split == nsp - 1;
    const int row0 = rb * kSimtRows;

    const T *q = static_cast<const T *>(P.q);
    {
        // the block's queries: every load in flight before the stores
        constexpr int kPerQ = kSimtRows * D / 128;
        float xs[kPerQ];
#pragma unroll
        for (int it = 0; it < kPerQ; ++it) {
            const int i = tid + it * 128;
            const int pr = i / D, k = i % D, p = row0 + pr;
            float x = 0.f;
            if (p < P.M) {
                const int r = p / P.G, hq = h * P.G + p % P.G;
                x = load_f(q + (((size_t)b * P.R + r) * P.Hq + hq) * D + k) * P.scale_log2;
            }
            xs[it] = x;
        }
#pragma unroll
        for (int it = 0; it < kPerQ; ++it) {
            const int i = tid + it * 128;
            sq[i / D][i % D] = xs[it];
        }
    }
    for (int i = tid; i < kSimtRows * P.W; i += blockDim.x) {
        const int pr = i / P.W, w = i % P.W, p = row0 + pr;
        svis[pr][w] = p < P.M ? P.vis[((size_t)b * P.R + p / P.G) * P.W + w] : 0u;
    }
    if (tid < kSimtRows) {
        const int p = row0 + tid;
        sflags[tid] = p < P.M ? P.row_flags[(size_t)b * P.R + p / P.G] : 0;
    }

    float m[4], l[4], acc[4][D / 32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) acc[i][j] = 0.f;
    }

    const T *kc = static_cast<const T *>(P.kc);
    const T *vc = static_cast<const T *>(P.vc);
    const T *kbp = static_cast<const T *>(P.kb);
    const T *vbp = static_cast<const T *>(P.vb);
    const T *skp = static_cast<const T *>(P.soft_k);
    const T *svp = static_cast<const T *>(P.soft_v);

    const int n_prefix_tiles = ceil_div(t1 - t0, kSimtCols);
    const int n_soft_tiles = last ? ceil_div(P.n_soft, kSimtCols) : 0;
    const int n_block_tiles = last ? ceil_div(P.R, kSimtCols) : 0;
    const int n_tiles = n_prefix_tiles + n_soft_tiles + n_block_tiles;

    for (int tile = 0; tile < n_tiles; ++tile) {
        int kind, base, ncols;
        if (tile < n_prefix_tiles) {
            kind = kColPrefix;
            base = t0 + tile * kSimtCols;
            ncols = min(kSimtCols, t1 - base);
        } else if (tile < n_prefix_tiles + n_soft_tiles) {
            kind = kColSoft;
            base = (tile - n_prefix_tiles) * kSimtCols;
            ncols = min(kSimtCols, P.n_soft - base);
        } else {
            kind = kColBlock;
            base = (tile - n_prefix_tiles - n_soft_tiles) * kSimtCols;
            ncols = min(kSimtCols, P.R - base);
        }
        __syncthreads();   // previous tile fully consumed (and sq/svis ready)
        // every load of the tile in flight before the first store (the
        // per-element loop of loads and stores waited one round trip each)
        constexpr int kPer = kSimtCols * D / 128;
        float kxs[kPer], vxs[kPer];
#pragma unroll
        for (int it = 0; it < kPer; ++it) {
            const int i = tid + it * 128;
            const int j = i / D, k = i % D;
            float kx = 0.f, vx = 0.f;
            if (j < ncols) {
                const T *kr = nullptr, *vr = nullptr;
                const int c = base + j;
                if (kind == kColPrefix) {
                    bool bad = false;
                    kr = prefix_row(P, kc, b, h, c, &bad);
                    vr = prefix_row(P, vc, b, h, c, &bad);
                    if (bad && k == 0) raise_status(P.status, SPEC_DEV_BAD_PAGE);
                } else if (kind == kColSoft) {
                    kr = skp + ((size_t)h * P.n_soft + c) * D;
                    vr = svp + ((size_t)h * P.n_soft + c) * D;
                } else {
                    kr = kbp + (((size_t)b * P.Hkv + h) * P.R + c) * D;
                    vr = vbp + (((size_t)b * P.Hkv + h) * P.R + c) * D;
                }
                if (kr) {
                    const int off = (k >> 6) * block_stride(P, kind == kColPrefix) + (k & 63);
                    kx = load_f(kr + off);
                    vx = load_f(vr + off);
                }
            }
            kxs[it] = kx;
            vxs[it] = vx;
        }
#pragma unroll
        for (int it = 0; it < kPer; ++it) {
            const int i = tid + it * 128;
            sk[i / D][i % D] = kxs[it];
            sv_[i / D][i % D] = vxs[it];
        }
        __syncthreads();

#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int pr = warp * 4 + i;
            const uint8_t fl = sflags[pr];
            bool visible = false;
            if (lane < ncols && (fl & SPEC_ROW_VALID)) {
                if (kind == kColPrefix) visible = true;
                else if (kind == kColSoft) visible = (fl & SPEC_ROW_SEES_SOFT) != 0;
                else {
                    const int c = base + lane;
                    visible = (svis[pr][c >> 5] >> (c & 31)) & 1u;
                }
            }
            float s = -INFINITY;
            if (visible) {
                float dot = 0.f;
#pragma unroll 8
                for (int k = 0; k < D; ++k) dot = fmaf(sq[pr][k], sk[lane][k], dot);
                s = dot;
            }
            const float mn = fmaxf(m[i], warp_max(s));
            if (mn == -INFINITY) continue;     // nothing visible yet (warp-uniform)
            const float alpha = exp2f(m[i] - mn);
            const float p = visible ? exp2f(s - mn) : 0.f;
            l[i] = l[i] * alpha + warp_sum(p);
#pragma unroll
            for (int j = 0; j < D / 32; ++j) acc[i][j] *= alpha;
            for (int jj = 0; jj < ncols; ++jj) {
                const float pj = __shfl_sync(0xffffffffu, p, jj);
                if (pj != 0.f) {
#pragma unroll
                    for (int j = 0; j < D / 32; ++j) acc[i][j] = fmaf(pj, sv_[jj][lane + 32 * j], acc[i][j]);
                }
            }
            m[i] = mn;
        }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int p = row0 + warp * 4 + i;
        if (p >= P.M) continue;
        const size_t idx = part_index(P, b, h, split, p);
#pragma unroll
        for (int j = 0; j < D / 32; ++j) P.part_o[idx * D + lane + 32 * j] = acc[i][j];
        if (lane == 0) {
            P.part_ml[idx * 2] = m[i];
            P.part_ml[idx * 2 + 1] = l[i];
        }
    }
}

// Merge the splits of every (request, KV head, packed row): one warp per
// packed row.  O = sum_s 2^(m_s - m*) o_s / sum_s 2^(m_s - m*) l_s.
template <typename T, int D>
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnParams P) {
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int p = blockIdx.x * 4 + warp;
    const int h = blockIdx.y, b = blockIdx.z;
    if (p >= P.M) return;
    const int S = clamp_seq(P, b, false);
    const int nsp = n_splits_of(P, S);
    float mstar = -INFINITY;
    for (int s = 0; s < nsp; ++s) mstar = fmaxf(mstar, P.part_ml[part_index(P, b, h, s, p) * 2]);
    const int r = p / P.G, hq = h * P.G + p % P.G;
    T *o = static_cast<T *>(P.o) + (((size_t)b * P.R + r) * P.Hq + hq) * D;
    float out[D / 32];
    float lse;
    if (mstar == -INFINITY) {
#pragma unroll
        for (int j = 0; j < D / 32; ++j) out[j] = 0.f;
        lse = -INFINITY;
    } else {
        float L = 0.f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) out[j] = 0.f;
        for (int s = 0; s < nsp; ++s) {
            const size_t idx = part_index(P, b, h, s, p);
            const float ms = P.part_ml[idx * 2];
            if (ms == -INFINITY) continue;
            const float w = exp2f(ms - mstar);
            L = fmaf(w, P.part_ml[idx * 2 + 1], L);
#pragma unroll
            for (int j = 0; j < D / 32; ++j) out[j] = fmaf(w, P.part_o[idx * D + lane + 32 * j], out[j]);
        }
        const float inv = 1.f / L;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) out[j] *= inv;
        lse = (mstar + log2f(L)) * kLn2;
    }
#pragma unroll
    for (int j = 0; j < D / 32; ++j) store_f(o + lane + 32 * j, out[j]);
    if (lane == 0) P.lse[((size_t)b * P.Hq + hq) * P.R + r] = lse;
}

// ---------------------------------------------------------------- planning

struct Plan {
    AttnParams P;
    size_t off_ml;      // byte offset of part_ml in the workspace
    size_t ws_bytes;
    bool use_tc;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

spec_status_t make_plan(const spec_attn_desc *a, const spec_kv_desc *c, Plan *out) {
    if (!a || !c) return SPEC_ERR_INVALID_ARG;
    if (a->batch < 0 || a->n_rows <= 0 || a->n_q_heads <= 0 || a->n_kv_heads <= 0 ||
        a->n_q_heads % a->n_kv_heads != 0 || a->n_soft < 0 || a->split_tokens < 0)
        return SPEC_ERR_INVALID_ARG;
    if (a->n_rows > SPEC_MAX_ROWS || a->n_soft > 64) return SPEC_ERR_UNSUPPORTED;
    if (a->head_dim != 64 && a->head_dim != 128) return SPEC_ERR_UNSUPPORTED;
    if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED;
    if (c->dtype != a->dtype || c->n_kv_heads != a->n_kv_heads || c->head_dim != a->head_dim ||
        c->batch < a->batch)
        return SPEC_ERR_INVALID_ARG;
    if (a->split_tokens % 64 != 0) return SPEC_ERR_INVALID_ARG;
    if (a->batch > 65535) return SPEC_ERR_UNSUPPORTED;
    AttnParams P{};
    P.B = a->batch;
    P.R = a->n_rows;
    P.Hq = a->n_q_heads;
    P.Hkv = a->n_kv_heads;
    P.G = a->n_q_heads / a->n_kv_heads;
    P.d = a->head_dim;
    P.M = P.R * P.G;
    P.W = ceil_div(P.R, 32);
    P.n_soft = a->n_soft;
    if (c->kind == SPEC_KV_CONTIGUOUS) {
        if (c->max_seq < 0) return SPEC_ERR_INVALID_ARG;
        P.paged = 0;
        P.max_seq = c->max_seq;
        P.capacity = c->max_seq;
        P.cache_rows = (long long)c->batch * c->n_kv_heads * c->max_seq;
    } else if (c->kind == SPEC_KV_PAGED) {
        if (c->page_size <= 0 || c->max_pages_per_seq <= 0 || c->n_pages <= 0) return SPEC_ERR_INVALID_ARG;
        if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64) return SPEC_ERR_UNSUPPORTED;
        if ((long long)c->max_pages_per_seq * c->page_size > (1ll << 30)) return SPEC_ERR_UNSUPPORTED;
        P.paged = 1;
        P.page_size = c->page_size;
        P.max_pages = c->max_pages_per_seq;
        P.n_pages = c->n_pages;
        P.capacity = c->max_pages_per_seq * c->page_size;
        P.cache_rows = (long long)c->n_pages * c->n_kv_heads * c->page_size;
    } else {
        return SPEC_ERR_INVALID_ARG;
    }
    const float scale = a->scale != 0.f ? a->scale : 1.f / sqrtf((float)a->head_dim);
    P.scale_log2 = scale * kLog2e;

    Plan plan{};
    // TMA coordinates are 32-bit: the tensor-core path takes caches and
    // blocks with fewer than 2^31 rows of head_dim elements.
    plan.use_tc = tc_supported(P, a->dtype) && P.cache_rows * (P.d / 64) < (1ll << 31) &&
                  (long long)P.B * P.Hkv * P.R < (1ll << 31) &&
                  (long long)P.Hkv * P.n_soft < (1ll << 31);
    P.rb_rows = plan.use_tc ? tc_rows_per_block(P) : kSimtRows;
    P.n_rb = ceil_div(P.M, P.rb_rows);
    if (a->split_tokens > 0) {
        P.chunk = a->split_tokens;
    } else {
        // Aim at ~8 work items per SM for prefixes at half the capacity.
        const long long units = (long long)P.B * P.Hkv * P.n_rb;
        const long long half = P.capacity / 2 > 64 ? P.capacity / 2 : 64;
        const long long target = 8ll * num_sms();
        long long chunk = (units * half + target - 1) / target;
        chunk = (chunk + 63) / 64 * 64;
        if (chunk < 512) chunk = 512;
        if (chunk > 16384) chunk = 16384;
        P.chunk = (int)chunk;
    }
    P.max_splits = P.capacity > 0 ? ceil_div(P.capacity, P.chunk) : 1;
    if (P.max_splits < 1) P.max_splits = 1;
    if (plan.use_tc) {
        plan.ws_bytes = tc_workspace_bytes(P, &plan.off_ml);
    } else {
        const size_t nrow = (size_t)P.B * P.Hkv * P.max_splits * P.M;
        plan.off_ml = align256(nrow * P.d * sizeof(float));
        plan.ws_bytes = plan.off_ml + align256(nrow * 2 * sizeof(float));
    }
    plan.P = P;
    *out = plan;
    return SPEC_OK;
}

template <typename T>
spec_status_t launch_simt(const AttnParams &P, cudaStream_t s) {
    dim3 grid(P.max_splits, P.Hkv * P.n_rb, P.B);
    const spec_status_t ls = P.d == 64 ? launch(attn_simt_kernel<T, 64>, grid, dim3(128), 0, s, P)
                                       : launch(attn_simt_kernel<T, 128>, grid, dim3(128), 0, s, P);
    if (ls != SPEC_OK) return ls;
    return launch_status();
}

template <typename T>
spec_status_t launch_combine(const AttnParams &P, cudaStream_t s) {
    dim3 grid(ceil_div(P.M, 4), P.Hkv, P.B);
    const spec_status_t ls = P.d == 64 ? launch(attn_combine_kernel<T, 64>, grid, dim3(128), 0, s, P)
                                       : launch(attn_combine_kernel<T, 128>, grid, dim3(128), 0, s, P);
    if (ls != SPEC_OK) return ls;
    return launch_status();
}

}  // namespace
}  // namespace sv

extern "C" spec_status_t spec_verify_attn_workspace_size(const spec_attn_desc *attn,
                                                         const spec_kv_desc *cache,
                                                         size_t *bytes) {
    if (!bytes) return SPEC_ERR_INVALID_ARG;
    sv::Plan plan;
    spec_status_t st = sv::make_plan(attn, cache, &plan);
    if (st != SPEC_OK) return st;
    *bytes = plan.ws_bytes;
    return SPEC_OK;
}

extern "C" spec_status_t spec_verify_attn(const spec_attn_desc *attn, const void *q,
                                          const spec_kv_desc *cache, const void *kb,
                                          const void *vb, const void *soft_k,
                                          const void *soft_v, const int32_t *seq_len,
                                          const uint32_t *vis, const uint8_t *row_flags,
                                          void *o, float *lse, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    sv::Plan plan;
    spec_status_t st = sv::make_plan(attn, cache, &plan);
    if (st != SPEC_OK) return st;
    sv::AttnParams &P = plan.P;
    if (P.B == 0) return SPEC_OK;
    if (!q || !kb || !vb || !seq_len || !vis || !row_flags || !o || !lse || !workspace)
        return SPEC_ERR_INVALID_ARG;
    if (P.capacity > 0 && (!cache->k || !cache->v)) return SPEC_ERR_INVALID_ARG;
    if (P.paged && !cache->page_table) return SPEC_ERR_INVALID_ARG;
    if (P.n_soft > 0 && (!soft_k || !soft_v)) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return SPEC_ERR_INVALID_ARG;
    if (workspace_bytes < plan.ws_bytes) return SPEC_ERR_CAPACITY;
    P.status = sv::status_ptr();
    if (!P.status) return SPEC_ERR_CUDA;
    P.q = q;
    P.kc = cache->k;
    P.vc = cache->v;
    P.page_table = cache->page_table;
    P.kb = kb;
    P.vb = vb;
    P.soft_k = soft_k;
    P.soft_v = soft_v;
    P.seq_len = seq_len;
    P.vis = vis;
    P.row_flags = row_flags;
    P.o = o;
    P.lse = lse;
    P.part_o = static_cast<float *>(workspace);
    P.part_ml = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.off_ml);
    cudaStream_t s = sv::as_stream(stream);
    if (attn->dtype == SPEC_BF16) {
        if (plan.use_tc) return sv::launch_attn_tc(P, s);
        st = sv::launch_simt<__nv_bfloat16>(P, s);
        if (st != SPEC_OK) return st;
        return sv::launch_combine<__nv_bfloat16>(P, s);
    }
    st = sv::launch_simt<float>(P, s);
    if (st != SPEC_OK) return st;
    return sv::launch_combine<float>(P, s);
}
