// Work decomposition shared by the verify-attention kernels.
//
// Packed rows: for KV head h, the G = Hq/Hkv query heads h*G .. h*G+G-1 of
// every speculative row r are processed together as packed row p = r*G + g,
// so one pass over a K/V tile serves R*G query rows (GQA packing).
//
// Splits: request b's prefix [0, S_b) is cut into n_splits(b) =
// max(1, ceil(S_b / chunk)) ranges of `chunk` tokens.  The last split of a
// request also takes the soft-prompt columns and the block's own columns.
// Each (request, KV head, split, row block) writes, per packed row, the
// running max m (log2 domain), the sum l and the unnormalised output
// o[d] (fp32) to the workspace; the combine kernel merges the splits.
#pragma once

#include "common.cuh"

namespace sv {

struct AttnParams {
    const void *q;
    const void *kc;          // cache K (contiguous or pages)
    const void *vc;
    const int32_t *page_table;
    const void *kb;          // block K/V
    const void *vb;
    const void *soft_k;
    const void *soft_v;
    const int32_t *seq_len;
    const uint32_t *vis;
    const uint8_t *row_flags;
    void *o;
    float *lse;
    float *part_o;           // [B][Hkv][max_splits][M][d]
    float *part_ml;          // [B][Hkv][max_splits][M][2]
    int *status;
    int B, R, Hq, Hkv, G, d, M, W, n_soft;
    int paged, max_seq, page_size, max_pages, n_pages, capacity;
    long long cache_rows;    // rows of the cache viewed as [rows][d]
    int chunk, max_splits;
    int n_rb, rb_rows;       // row blocks of packed rows per (request, KV head)
    float scale_log2;        // softmax scale * log2(e)
};

// Clamp seq_len to [0, capacity]; report overflow once per request.
__device__ __forceinline__ int clamp_seq(const AttnParams &P, int b, bool report) {
    int S = P.seq_len[b];
    if (S < 0 || S > P.capacity) {
        if (report) raise_status(P.status, SPEC_DEV_SEQ_OVERFLOW);
        S = S < 0 ? 0 : P.capacity;
    }
    return S;
}

__device__ __forceinline__ int n_splits_of(const AttnParams &P, int S) {
    int n = ceil_div(S, P.chunk);
    return n < 1 ? 1 : n;
}

__device__ __forceinline__ size_t part_index(const AttnParams &P, int b, int h, int split, int p) {
    return (((size_t)b * P.Hkv + h) * P.max_splits + split) * P.M + p;
}

}  // namespace sv
