// spec_mask_build: visibility bitmask of the speculative block.
//
// "Lookahead Attention", sec. 3.1 (verify form: a lookahead row sees the
// prefix and itself), "Speculative Streaming" Eq. 2 (stream j sees streams
// <= j of its node) and Eq. 4 with the sentence after it (a tree node sees
// all its ancestors), "ConFu" key design 1 (a contemplate token sees its
// node's view plus itself and the soft prompt).  Every such view is the
// closure of one parent pointer per row: vis(r) = {r} U vis(vparent[r]).
#include "common.cuh"

namespace {

constexpr int kMaxWords = SPEC_MAX_ROWS / 32;

// One CTA per request, one thread per row.  Each thread walks its own
// parent chain (strictly decreasing row indices, so at most r steps).
__global__ void mask_build_kernel(const int32_t *__restrict__ vparent,
                                  const uint8_t *__restrict__ soft_flags, int R, int W,
                                  uint32_t *__restrict__ vis, uint8_t *__restrict__ row_flags,
                                  int *status) {
    sv::pdl_wait();
    __shared__ int32_t svp[SPEC_MAX_ROWS];
    const int b = blockIdx.x;
    for (int r = threadIdx.x; r < R; r += blockDim.x) svp[r] = vparent[(size_t)b * R + r];
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        uint32_t words[kMaxWords];
#pragma unroll
        for (int w = 0; w < kMaxWords; ++w) words[w] = 0u;
        uint8_t flags = 0;
        const int p0 = svp[r];
        if (p0 != SPEC_VP_PAD) {
            bool ok = true;
            int c = r;
            // c is a valid row index here; its parent must be -1 or an
            // earlier row that is not padding.
            while (true) {
#pragma unroll
                for (int w = 0; w < kMaxWords; ++w)
                    if (w == (c >> 5)) words[w] |= 1u << (c & 31);
                const int p = svp[c];
                if (p == SPEC_VP_ROOT) break;
                if (p < 0 || p >= c || svp[p] == SPEC_VP_PAD) {
                    ok = false;
                    break;
                }
                c = p;
            }
            if (ok) {
                flags = SPEC_ROW_VALID;
                if (soft_flags && soft_flags[(size_t)b * R + r]) flags |= SPEC_ROW_SEES_SOFT;
            } else {
                sv::raise_status(status, SPEC_DEV_BAD_TREE);
#pragma unroll
                for (int w = 0; w < kMaxWords; ++w) words[w] = 0u;
            }
        }
        uint32_t *dst = vis + ((size_t)b * R + r) * W;
#pragma unroll
        for (int w = 0; w < kMaxWords; ++w)
            if (w < W) dst[w] = words[w];
        row_flags[(size_t)b * R + r] = flags;
    }
}

}  // namespace

extern "C" spec_status_t spec_mask_build(const int32_t *vparent, const uint8_t *soft_flags,
                                         int batch, int n_rows, uint32_t *vis,
                                         uint8_t *row_flags, void *stream) {
    if (batch < 0 || n_rows <= 0) return SPEC_ERR_INVALID_ARG;
    if (n_rows > SPEC_MAX_ROWS) return SPEC_ERR_UNSUPPORTED;
    if (batch == 0) return SPEC_OK;
    if (!vparent || !vis || !row_flags) return SPEC_ERR_INVALID_ARG;
    int *st = sv::status_ptr();
    if (!st) return SPEC_ERR_CUDA;
    const int W = sv::ceil_div(n_rows, 32);
    const int threads = n_rows <= 128 ? 128 : 256;
    if (sv::launch(mask_build_kernel, dim3(batch), dim3(threads), 0, sv::as_stream(stream), vparent,
               soft_flags, n_rows, W, vis, row_flags, st) != SPEC_OK)
        return SPEC_ERR_CUDA;
    return sv::launch_status();
}
