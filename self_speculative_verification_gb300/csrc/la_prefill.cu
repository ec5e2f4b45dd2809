// spec_la_prefill_attn: the prefill form of Lookahead Attention
// ("Lookahead Attention", sec. 3.1).  All n + k positions of a request
// attend in one pass under the full (n + k) x (n + k) mask M_LA: original
// position i sees originals 0..i (causal); lookahead position n + j sees
// every original and itself, and no other lookahead position.
//
// Design (GB300, tcgen05):
// * A unit is one 128-row query tile m of one (request, query head); it
//   needs key tiles 0..m.  Units are paired (NM-1-p, p), so every work item
//   costs NM + 1 key tiles (NM: query tiles per head), and the persistent
//   grid (one CTA per SM) takes the items round-robin.  Items are numbered
//   (request, head)-major with heads of one KV group adjacent, so the CTAs
//   working on one KV head at a time read the same K/V tiles at about the
//   same time and share them through L2.
// * Warp roles: warp 4 issues TMA loads (each unit's Q tile into one of two
//   Q buffers; K and V tiles into a five-slot ring), warp 5 issues the MMAs
//   from one thread, warps 0-3 run the softmax with one query row per
//   thread.
// * S = Q K^T: both operands K-major in shared memory (128-byte swizzle),
//   fp32 result in TMEM, double-buffered so S(t+1) is computed while the
//   softmax works on S(t).  P (bf16) goes back to TMEM; O += P V takes P
//   from TMEM and V (MN-major) from shared memory, accumulating in TMEM.
// * The mask is evaluated only on key tiles that reach the diagonal or hold
//   keys >= n; every other tile is wholly visible.  The running max is
//   raised only when it grows by more than 2^8 (then O and l are rescaled
//   in place).
// * Every wait is bounded; on expiry the kernel sets SPEC_DEV_TIMEOUT,
//   stops issuing work, waits (bounded) for its own copies and MMAs, frees
//   its TMEM and returns.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace sv {
namespace {

namespace lap {

constexpr int kD = 128;                  // head_dim
constexpr int kM = 128;                  // query rows per unit (MMA M)
constexpr int kN = 128;                  // keys per key tile (MMA N of S)
constexpr int kHalf = 128 * 128;         // one 128-row x 64-element bf16 box
constexpr int kTileBytes = 2 * kHalf;    // one Q, K or V tile: 32 KB
constexpr int kSlots = 5;                // K/V ring slots
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kTmemCols = 512;
constexpr int kColO = 0;                 // O: columns [0, 128)
constexpr int kColS = 128;               // S buffer b: [128 + 128 b, 256 + 128 b)
constexpr int kColP = 384;               // P buffer b: [384 + 64 b, 448 + 64 b), bf16 pairs
constexpr float kRescale = 8.f;          // log2 growth allowed before rescaling

struct Params {
    int B, L, n;          // requests, positions per request (n + k), originals
    int Hq, Hkv, G;       // query heads, KV heads, Hq / Hkv
    int NM, NP, n_items;  // query tiles per head, items per head, total items
    float scale_log2;     // softmax scale * log2(e)
    __nv_bfloat16 *o;
    float *lse;
    int *status;
};

struct Shared {
    uint64_t q_full[2], q_empty[2];
    uint64_t full[kSlots], empty[kSlots];
    uint64_t s_full[2], p_full[2], o_upd[2];
    uint64_t o_free;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = 2 * (size_t)kTileBytes + kSlots * (size_t)kTileBytes +
                              sizeof(Shared) + 1024;

struct Unit {
    int b, hq, m;
};

// The units of item w: query tiles NM-1-p and p of one (request, head).
__device__ __forceinline__ int units_of(const Params &P, int w, Unit (&u)[2]) {
    const int bh = w / P.NP, p = w % P.NP;
    const int b = bh / P.Hq, hq = bh % P.Hq;
    u[0] = Unit{b, hq, P.NM - 1 - p};
    u[1] = Unit{b, hq, p};
    return (P.NM - 1 - p == p) ? 1 : 2;
}

}  // namespace lap

__global__ void __launch_bounds__(lap::kThreads, 1)
la_prefill_kernel(const __grid_constant__ lap::Params P, const __grid_constant__ CUtensorMap mq,
                  const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv) {
    using namespace lap;
    using namespace tc5;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qbuf = smem;                          // 2 Q tiles
    uint8_t *ring = smem + 2 * kTileBytes;         // kSlots K / V tiles
    Shared &sh = *reinterpret_cast<Shared *>(ring + kSlots * kTileBytes);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == kProducerWarp * 32) {
        const CUtensorMap *maps[3] = {&mq, &mk, &mv};
        for (int i = 0; i < 3; ++i)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(maps[i]))
                         : "memory");
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sh.q_full[b], 1);
            mbar_init(&sh.q_empty[b], 1);
            mbar_init(&sh.s_full[b], 1);
            mbar_init(&sh.p_full[b], kSoftmaxWarps);
            mbar_init(&sh.o_upd[b], 1);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.o_free, kSoftmaxWarps);
        mbar_init(&sh.drain, 1);
        sh.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sh.tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = sh.tmem_base;
    volatile int *abort = &sh.abort;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_q = policy_evict_first();
            const uint64_t pol_kv = policy_evict_last();
            long long ld = 0;          // K/V loads issued
            int nq = 0;                // Q loads issued
            bool ok = true;
            for (int w = blockIdx.x; w < P.n_items && ok; w += gridDim.x) {
                Unit u[2];
                const int nu = units_of(P, w, u);
                for (int s = 0; s < nu && ok; ++s) {
                    const Unit &U = u[s];
                    const int qb = nq & 1;
                    if (*abort || !mbar_wait(&sh.q_empty[qb], (uint32_t)(((nq >> 1) & 1) ^ 1))) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sh.q_full[qb], (uint32_t)kTileBytes);
                    for (int hh = 0; hh < 2; ++hh)
                        tma_load_4d(qbuf + qb * kTileBytes + hh * kHalf, &mq, hh * 64, U.hq,
                                    U.m * kM, U.b, &sh.q_full[qb], pol_q);
                    ++nq;
                    const int hk = U.hq / P.G;
                    for (int j = 0; j <= U.m && ok; ++j) {
                        for (int kv = 0; kv < 2; ++kv) {
                            const int slot = (int)(ld % kSlots);
                            if (*abort ||
                                !mbar_wait(&sh.empty[slot], (uint32_t)(((ld / kSlots) & 1) ^ 1))) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&sh.full[slot], (uint32_t)kTileBytes);
                            for (int hh = 0; hh < 2; ++hh)
                                tma_load_4d(ring + slot * kTileBytes + hh * kHalf, kv ? &mv : &mk,
                                            hh * 64, hk, j * kN, U.b, &sh.full[slot], pol_kv);
                            ++ld;
                        }
                    }
                }
            }
            if (!ok) {
                raise_status(P.status, SPEC_DEV_TIMEOUT);
                *abort = 1;
            }
            // do not leave while copies into this CTA's shared memory are in
            // flight (earlier loads were consumed, hence complete)
            for (long long i = ld - 1; i >= 0 && i >= ld - kSlots; --i)
                if (!mbar_wait(&sh.full[i % kSlots], (uint32_t)((i / kSlots) & 1))) {
                    raise_status(P.status, SPEC_DEV_TIMEOUT);
                    break;
                }
            for (int i = nq - 1; i >= 0 && i >= nq - 2; --i)
                if (!mbar_wait(&sh.q_full[i & 1], (uint32_t)((i >> 1) & 1))) {
                    raise_status(P.status, SPEC_DEV_TIMEOUT);
                    break;
                }
        }
    } else if (warp == kMmaWarp) {
        // --------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc(kM, kN, false, false);
            const uint32_t id_pv = idesc(kM, kD, false, true);
            long long k = 0, ld = 0;   // key tiles processed, K/V loads consumed
            int un = 0;                // units started
            bool ok = true;
            // PV of the previous key tile: its V slot / load index, whether
            // it starts its unit, and that unit's number
            long long pv_ld = 0;
            bool pv_first = false;
            int pv_un = 0;
            auto issue_pv = [&](long long t) -> bool {
                const int b = (int)(t & 1);
                const int vslot = (int)(pv_ld % kSlots);
                if (!mbar_wait(&sh.p_full[b], (uint32_t)((t >> 1) & 1))) return false;
                if (!mbar_wait(&sh.full[vslot], (uint32_t)((pv_ld / kSlots) & 1))) return false;
                // a unit's first PV overwrites O: the previous unit's
                // epilogue must have read it
                if (pv_first && pv_un > 0 &&
                    !mbar_wait(&sh.o_free, (uint32_t)((pv_un - 1) & 1)))
                    return false;
                fence_after();
                const uint64_t vd = smem_desc(smem_u32(ring + vslot * kTileBytes), kHalf, 1024);
                const uint32_t a_p = tmem + kColP + (uint32_t)b * (kN / 2);
#pragma unroll
                for (int ks = 0; ks < kN / 16; ++ks)
                    mma(tmem + kColO, a_p + ks * 8, vd + (uint64_t)((ks * 2048) >> 4), id_pv,
                        (ks > 0 || !pv_first) ? 1u : 0u);
                commit(&sh.o_upd[b]);
                commit(&sh.empty[vslot]);
                return true;
            };
            for (int w = blockIdx.x; w < P.n_items && ok; w += gridDim.x) {
                Unit u[2];
                const int nu = units_of(P, w, u);
                for (int s = 0; s < nu && ok; ++s, ++un) {
                    const int m = u[s].m;
                    const int qb = un & 1;
                    if (*abort || !mbar_wait(&sh.q_full[qb], (uint32_t)((un >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    const uint64_t qd = smem_desc(smem_u32(qbuf + qb * kTileBytes), 16, 1024);
                    for (int j = 0; j <= m; ++j) {
                        const int kslot = (int)(ld % kSlots);
                        if (!mbar_wait(&sh.full[kslot], (uint32_t)((ld / kSlots) & 1))) {
                            ok = false;
                            break;
                        }
                        fence_after();
                        // S(k) = Q K^T into S buffer k % 2 (free: PV(k-2),
                        // issued last iteration, waited for its softmax)
                        const uint64_t kd = smem_desc(smem_u32(ring + kslot * kTileBytes), 16, 1024);
                        const uint32_t s_col = tmem + kColS + (uint32_t)(k & 1) * kN;
#pragma unroll
                        for (int ks = 0; ks < kD / 16; ++ks) {
                            const uint64_t off = (uint64_t)((((ks >> 2) * kHalf) + (ks & 3) * 32) >> 4);
                            mma_ss(s_col, qd + off, kd + off, id_s, ks > 0 ? 1u : 0u);
                        }
                        commit(&sh.s_full[k & 1]);
                        commit(&sh.empty[kslot]);
                        if (j == m) commit(&sh.q_empty[qb]);
                        if (k > 0 && !issue_pv(k - 1)) {
                            ok = false;
                            break;
                        }
                        pv_ld = ld + 1;
                        pv_first = j == 0;
                        pv_un = un;
                        ld += 2;
                        ++k;
                    }
                }
            }
            if (ok && k > 0) ok = issue_pv(k - 1);
            if (!ok) {
                raise_status(P.status, SPEC_DEV_TIMEOUT);
                *abort = 1;
            }
            // every MMA issued above has completed before TMEM is released
            commit(&sh.drain);
            if (!mbar_wait(&sh.drain, 0)) raise_status(P.status, SPEC_DEV_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------ softmax
        const int r = warp * 32 + lane;                 // row of the query tile
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float sc = P.scale_log2;
        long long k = 0;
        bool ok = true;
        for (int w = blockIdx.x; w < P.n_items && ok; w += gridDim.x) {
            Unit u[2];
            const int nu = units_of(P, w, u);
            for (int s = 0; s < nu && ok; ++s) {
                const Unit &U = u[s];
                const int i = U.m * kM + r;              // this thread's position
                float m_used = -INFINITY, l = 0.f;
                for (int j = 0; j <= U.m; ++j, ++k) {
                    if (*abort || !mbar_wait(&sh.s_full[k & 1], (uint32_t)((k >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    fence_after();
                    float x[kN];
                    {
                        const uint32_t sa = tmem + lane_base + kColS + (uint32_t)(k & 1) * kN;
#pragma unroll
                        for (int c = 0; c < kN / 32; ++c) {
                            uint32_t v[32];
                            ld32(sa + c * 32, v);
                            wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[e]);
                        }
                    }
                    // key c is visible iff c <= i and (c < n or c == i)
                    if (j == U.m || (j + 1) * kN > P.n) {
                        const int c0 = j * kN;
#pragma unroll
                        for (int e = 0; e < kN; ++e) {
                            const int c = c0 + e;
                            const bool vis = c <= i && (c < P.n || c == i);
                            x[e] = vis ? x[e] : -INFINITY;
                        }
                    }
                    float tmv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) tmv[e] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < kN; ++e) tmv[e & 7] = fmaxf(tmv[e & 7], x[e]);
                    const float traw = fmaxf(fmaxf(fmaxf(tmv[0], tmv[1]), fmaxf(tmv[2], tmv[3])),
                                             fmaxf(fmaxf(tmv[4], tmv[5]), fmaxf(tmv[6], tmv[7])));
                    const float tm = traw == -INFINITY ? -INFINITY : traw * sc;
                    // raise the reference max only when it grew by more than 2^8
                    if (tm > m_used + kRescale || (m_used == -INFINITY && tm != -INFINITY)) {
                        const float alpha = (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - tm);
                        if (j > 0 && m_used != -INFINITY) {
                            // O holds PV(k-1): wait for it, then scale this row
                            if (!mbar_wait(&sh.o_upd[(k - 1) & 1], (uint32_t)(((k - 1) >> 1) & 1))) {
                                ok = false;
                                break;
                            }
                            fence_after();
#pragma unroll
                            for (int c32 = 0; c32 < kD / 32; ++c32) {
                                uint32_t v[32];
                                const uint32_t oa = tmem + lane_base + kColO + c32 * 32;
                                ld32(oa, v);
                                wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                                st32(oa, v);
                            }
                            wait_st();
                        }
                        l *= alpha;
                        m_used = tm;
                    }
                    const float mu = m_used == -INFINITY ? 0.f : m_used;
                    // P buffer k % 2 was last read by PV(k-2)
                    if (k >= 2 && !mbar_wait(&sh.o_upd[k & 1], (uint32_t)(((k - 2) >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    float rsv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) rsv[e] = 0.f;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t pw[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float p0 = fast_exp2(fmaf(x[h * 64 + 2 * e], sc, -mu));
                            const float p1 = fast_exp2(fmaf(x[h * 64 + 2 * e + 1], sc, -mu));
                            rsv[e & 7] += p0 + p1;
                            pw[e] = pack_bf16(p0, p1);
                        }
                        st32(tmem + lane_base + kColP + (uint32_t)(k & 1) * (kN / 2) + h * 32, pw);
                    }
                    l += ((rsv[0] + rsv[1]) + (rsv[2] + rsv[3])) + ((rsv[4] + rsv[5]) + (rsv[6] + rsv[7]));
                    wait_st();
                    fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.p_full[k & 1]);
                }
                if (!ok) break;
                // epilogue: O / l (bf16) and the LSE of this row
                if (!mbar_wait(&sh.o_upd[(k - 1) & 1], (uint32_t)(((k - 1) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                fence_after();
                const bool row_ok = i < P.L;
                const float inv = l > 0.f ? 1.f / l : 0.f;
                uint4 *dst = reinterpret_cast<uint4 *>(
                    P.o + (((size_t)U.b * P.L + (row_ok ? i : 0)) * P.Hq + U.hq) * kD);
#pragma unroll
                for (int c32 = 0; c32 < kD / 32; ++c32) {
                    uint32_t v[32];
                    ld32(tmem + lane_base + kColO + c32 * 32, v);
                    wait_ld();
                    if (!row_ok) continue;
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        dst[(c32 * 32 + e) / 8] = make_uint4(
                            pack_bf16(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv),
                            pack_bf16(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv),
                            pack_bf16(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv),
                            pack_bf16(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv));
                }
                if (row_ok)
                    P.lse[((size_t)U.b * P.Hq + U.hq) * P.L + i] =
                        l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.o_free);
            }
        }
        if (!ok) {
            raise_status(P.status, SPEC_DEV_TIMEOUT);
            *abort = 1;
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

// 4-D bf16 map over [B][L][H][128] with a (64, 1, 128, 1) box: one
// 128-position x 64-element block of one head, 128-byte swizzle.  Positions
// past L read as zeros.
bool make_map_4d(CUtensorMap *map, const void *base, int H, int L, int B) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    constexpr int D = lap::kD;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)L * H * D * 2};
    cuuint32_t box[4] = {64u, 1u, (cuuint32_t)lap::kM, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace sv

extern "C" spec_status_t spec_la_prefill_attn(const spec_prefill_desc *desc, const void *q,
                                              const void *k, const void *v, void *o, float *lse,
                                              void *stream) {
    using namespace sv;
    if (!desc) return SPEC_ERR_INVALID_ARG;
    const int B = desc->batch, n = desc->n_orig, nl = desc->n_look;
    const int Hq = desc->n_q_heads, Hkv = desc->n_kv_heads;
    if (B < 0 || n < 1 || nl < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || desc->scale < 0.f)
        return SPEC_ERR_INVALID_ARG;
    if (desc->dtype != SPEC_BF16 || desc->head_dim != lap::kD) return SPEC_ERR_UNSUPPORTED;
    const long long L = (long long)n + nl;
    if (L > (1ll << 30)) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!q || !k || !v || !o || !lse) return SPEC_ERR_INVALID_ARG;
    // tensor copies start on 16-byte boundaries
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
         reinterpret_cast<uintptr_t>(v)) % 16 != 0)
        return SPEC_ERR_INVALID_ARG;
    int *st = status_ptr();
    if (!st) return SPEC_ERR_CUDA;

    lap::Params P{};
    P.B = B;
    P.L = (int)L;
    P.n = n;
    P.Hq = Hq;
    P.Hkv = Hkv;
    P.G = Hq / Hkv;
    P.NM = (int)ceil_div_ll(L, lap::kM);
    P.NP = (P.NM + 1) / 2;
    const long long items = (long long)B * Hq * P.NP;
    if (items > 0x7fffffffll) return SPEC_ERR_UNSUPPORTED;
    P.n_items = (int)items;
    const float scale = desc->scale > 0.f ? desc->scale : 1.f / sqrtf((float)lap::kD);
    P.scale_log2 = scale * kLog2e;
    P.o = static_cast<__nv_bfloat16 *>(o);
    P.lse = lse;
    P.status = st;

    CUtensorMap maps[3];
    if (!make_map_4d(&maps[0], q, Hq, (int)L, B) || !make_map_4d(&maps[1], k, Hkv, (int)L, B) ||
        !make_map_4d(&maps[2], v, Hkv, (int)L, B))
        return SPEC_ERR_CUDA;

    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(la_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)lap::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return SPEC_ERR_CUDA;
    const int grid = (int)std::min<long long>(num_sms(), items);
    la_prefill_kernel<<<grid, lap::kThreads, lap::kSmemBytes, as_stream(stream)>>>(
        P, maps[0], maps[1], maps[2]);
    return launch_status();
}
