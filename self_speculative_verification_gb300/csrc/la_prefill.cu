// spec_la_prefill_attn: the prefill form of Lookahead Attention
// ("Lookahead Attention", sec. 3.1).  All n + k positions of a request
// attend in one pass under the full (n + k) x (n + k) mask M_LA: original
// position i sees originals 0..i (causal); lookahead position n + j sees
// every original and itself, and no other lookahead position.
//
// Design (GB300, tcgen05):
// * A unit is a pair of consecutive 128-row query tiles A = 2t and
//   B = 2t + 1 of one (request, query head); they share the K/V tiles
//   0..2t (B also takes tile 2t + 1, its diagonal).  Units are paired
//   (NB-1-p, p) so every work item costs about the same; the persistent
//   grid (one CTA per SM) takes the items round-robin.  Items are numbered
//   (request, head)-major with heads of one KV group adjacent, so the CTAs
//   working on one KV head at a time share its K/V tiles through L2.
// * Warp roles: warps 0-3 run the softmax of tile A and warps 4-7 that of
//   tile B (one query row per thread), warp 8 issues TMA loads (the unit's
//   two Q tiles; K and V tiles into a five-slot ring), warp 9 issues the
//   MMAs from one thread.
// * Per tile, TMEM holds O (128 fp32 columns) and S (128 fp32 columns);
//   P (bf16) is written over the first 64 columns of S, which the next S
//   MMA of the same tile overwrites only after the PV MMA that reads it
//   (tcgen05 MMAs of one thread run in issue order).  The MMA thread
//   interleaves the tiles -- PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) -- so the
//   tensor core works on one tile while the other tile's softmax runs.
// * Softmax of a tile row: the whole S row in registers (four TMEM loads in
//   flight), the masked maximum, then P = exp2(s - m) written chunk by chunk.
//   The running max is raised only when it grows by more than 2^8 (then O
//   and l are rescaled in place); O holds every earlier PV of the tile by
//   then, since the S MMA the softmax waits for was issued after them.
// * The mask is evaluated only on key tiles that reach the diagonal or hold
//   keys >= n; every other tile is wholly visible.
// * Every wait is bounded; on expiry the kernel sets SPEC_DEV_TIMEOUT,
//   stops issuing work, waits (bounded) for its own copies and MMAs, frees
//   its TMEM and returns.
#include <algorithm>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace sv {
namespace {

namespace lap {

constexpr int kD = 128;                  // head_dim
constexpr int kM = 128;                  // query rows per tile (MMA M)
constexpr int kN = 128;                  // keys per key tile (MMA N of S)
constexpr int kHalf = 128 * 128;         // one 128-row x 64-element bf16 box
constexpr int kTileBytes = 2 * kHalf;    // one Q, K or V tile: 32 KB
constexpr int kSlots = 5;                // K/V ring slots
constexpr int kGroupWarps = 4;           // softmax warps per query tile
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;              // warps 10, 11 complete the third warpgroup
constexpr int kThreads = 12 * 32;
// Registers a thread, split by setmaxnreg: the launch gives every thread
// kLaunchRegs (the most a 384-thread CTA can have); the two softmax
// warpgroups raise theirs to kSoftmaxRegs and the third lowers to
// kOtherRegs: 8 * 32 * 184 + 4 * 32 * 128 = 63488 <= 384 * 168 = 64512.
// The split must fit the launch allocation, or the raise would wait
// forever.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 184;
constexpr int kOtherRegs = 128;
static_assert(8 * 32 * kSoftmaxRegs + 4 * 32 * kOtherRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kTmemCols = 512;
// TMEM columns of tile x (0 = A, 1 = B): O at [256 x, 256 x + 128), S at
// [256 x + 128, 256 x + 256), P over the first 64 columns of S
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u * (uint32_t)x; }
__host__ __device__ constexpr uint32_t col_s(int x) { return 256u * (uint32_t)x + 128u; }
constexpr float kRescale = 8.f;          // log2 growth allowed before rescaling

struct Params {
    int B, L, n;          // requests, positions per request (n + k), originals
    int Hq, Hkv, G;       // query heads, KV heads, Hq / Hkv
    int NM, NB, NP;       // query tiles, tile pairs, items per head
    int n_items;
    float scale_log2;     // softmax scale * log2(e)
    __nv_bfloat16 *o;
    float *lse;
    int *status;
    long long wait;       // limit of every pipeline wait, in SM cycles
};

struct Shared {
    uint64_t q_full, q_empty;
    uint64_t full[kSlots], empty[kSlots];
    uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = 2 * (size_t)kTileBytes + kSlots * (size_t)kTileBytes +
                              sizeof(Shared) + 1024;

// Unit: query tiles 2t (A) and 2t + 1 (B, if it exists) of (b, hq).
struct Unit {
    int b, hq, t;
};

__device__ __forceinline__ int units_of(const Params &P, int w, Unit (&u)[2]) {
    const int bh = w / P.NP, p = w % P.NP;
    const int b = bh / P.Hq, hq = bh % P.Hq;
    u[0] = Unit{b, hq, P.NB - 1 - p};
    u[1] = Unit{b, hq, p};
    return (P.NB - 1 - p == p) ? 1 : 2;
}

// last key tile of query tile X of unit t, or -1 if the tile does not exist
__device__ __forceinline__ int last_tile(const Params &P, int t, int X) {
    const int m = 2 * t + X;
    return m < P.NM ? m : -1;
}

// The units each CTA works on, in order: v[c] .. v[c + 1] index CTA c's run
// of unit ids (b * Hq + hq) * NB + t stored from v[grid + 1] on.  Built on
// the host (longest unit first onto the least-loaded CTA, a few heads at a
// time) and passed by value with the launch; n == 0 means no table, and the
// CTAs then take the paired items round-robin.
constexpr int kSchedCap = 8192;
struct Sched {
    int n;
    uint16_t v[kSchedCap];
};

struct Cursor {
    int w, s, e, end;
};

__device__ __forceinline__ Cursor cursor_begin(const Sched &S) {
    Cursor c{(int)blockIdx.x, 0, 0, 0};
    if (S.n) {
        c.e = S.v[blockIdx.x];
        c.end = S.v[blockIdx.x + 1];
    }
    return c;
}

// the CTA's next unit; false when it has none left
__device__ __forceinline__ bool next_unit(const Params &P, const Sched &S, Cursor &c, Unit &U) {
    if (S.n) {
        if (c.e >= c.end) return false;
        const int id = S.v[gridDim.x + 1 + c.e++];
        const int bh = id / P.NB;
        U = Unit{bh / P.Hq, bh % P.Hq, id % P.NB};
        return true;
    }
    while (c.w < P.n_items) {
        Unit u[2];
        const int nus = units_of(P, c.w, u);
        if (c.s < nus) {
            U = u[c.s++];
            return true;
        }
        c.w += gridDim.x;
        c.s = 0;
    }
    return false;
}

}  // namespace lap

__global__ void __launch_bounds__(lap::kThreads, 1)
la_prefill_kernel(const __grid_constant__ lap::Params P, const __grid_constant__ CUtensorMap mq,
                  const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv,
                  const __grid_constant__ lap::Sched S) {
    pdl_wait();
    using namespace lap;
    using namespace tc5;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qbuf = smem;                          // Q tiles A and B
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
        mbar_init(&sh.q_full, 1);
        mbar_init(&sh.q_empty, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(&sh.s_full[x], 1);
            mbar_init(&sh.p_full[x], kGroupWarps);
            mbar_init(&sh.o_done[x], 1);
            mbar_init(&sh.o_free[x], kGroupWarps);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], 1);
        }
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

    if (warp >= kProducerWarp) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
        if (warp == kProducerWarp) {
            // ------------------------------------------------------ producer
            if (lane == 0) {
                const uint64_t pol_q = policy_evict_first();
                const uint64_t pol_kv = policy_evict_last();
                long long ld = 0;          // K/V loads issued
                int nu = 0;                // units (Q loads) issued
                bool ok = true;
                Cursor cur = cursor_begin(S);
                Unit U;
                while (ok && next_unit(P, S, cur, U)) {
                    const int mA = last_tile(P, U.t, 0), mB = last_tile(P, U.t, 1);
                    const int jmax = mB >= 0 ? mB : mA;
                    if (*abort || !mbar_wait(&sh.q_empty, (uint32_t)((nu & 1) ^ 1), P.wait)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sh.q_full, (uint32_t)(mB >= 0 ? 2 : 1) * kTileBytes);
                    for (int x = 0; x < (mB >= 0 ? 2 : 1); ++x)
                        for (int hh = 0; hh < 2; ++hh)
                            tma_load_4d(qbuf + x * kTileBytes + hh * kHalf, &mq, hh * 64, U.hq,
                                        (2 * U.t + x) * kM, U.b, &sh.q_full, pol_q);
                    ++nu;
                    const int hk = U.hq / P.G;
                    for (int j = 0; j <= jmax && ok; ++j) {
                        for (int kv = 0; kv < 2; ++kv) {
                            const int slot = (int)(ld % kSlots);
                            if (*abort ||
                                !mbar_wait(&sh.empty[slot], (uint32_t)(((ld / kSlots) & 1) ^ 1), P.wait)) {
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
                if (nu > 0 && !mbar_wait(&sh.q_full, (uint32_t)((nu - 1) & 1)))
                    raise_status(P.status, SPEC_DEV_TIMEOUT);
            }
        } else if (warp == kMmaWarp) {
            // --------------------------------------------------- MMA issuer
            if (lane == 0) {
                const uint32_t id_s = idesc(kM, kN, false, false);
                const uint32_t id_pv = idesc(kM, kD, false, true);
                int slot = 0;                  // ring slot of the next K/V load to consume
                uint32_t ph = 0;               // and the parity of its fill
                int nu = 0;                    // units started
                int np[2] = {0, 0};            // P hand-offs taken, per tile
                int nact[2] = {0, 0};          // units in which the tile took part
                bool ok = true;
                const uint64_t qd[2] = {smem_desc(smem_u32(qbuf), 16, 1024),
                                        smem_desc(smem_u32(qbuf + kTileBytes), 16, 1024)};
                // descriptors of ring slot 0 (K: K-major, V: MN-major); a slot is
                // kTileBytes further, i.e. kTileBytes >> 4 in the address field
                const uint64_t kd0 = smem_desc(smem_u32(ring), 16, 1024);
                const uint64_t vd0 = smem_desc(smem_u32(ring), kHalf, 1024);
                auto advance = [&]() {
                    if (++slot == kSlots) {
                        slot = 0;
                        ph ^= 1u;
                    }
                };
                auto issue_s = [&](int x, int ks_slot) {
                    const uint64_t kd = kd0 + (uint64_t)(ks_slot * (kTileBytes >> 4));
    #pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks) {
                        const uint64_t off = (uint64_t)((((ks >> 2) * kHalf) + (ks & 3) * 32) >> 4);
                        mma_ss(tmem + col_s(x), qd[x] + off, kd + off, id_s, ks > 0 ? 1u : 0u);
                    }
                    commit(&sh.s_full[x]);
                };
                // O_x += P_x V(j); the tile's first PV of a unit overwrites O_x,
                // after the previous unit's epilogue of that tile read it
                auto issue_pv = [&](int x, int v_slot, bool first) -> bool {
                    if (!mbar_wait(&sh.p_full[x], (uint32_t)(np[x] & 1), P.wait)) return false;
                    ++np[x];
                    if (first && nact[x] > 0 &&
                        !mbar_wait(&sh.o_free[x], (uint32_t)((nact[x] - 1) & 1), P.wait))
                        return false;
                    fence_after();
                    const uint64_t vd = vd0 + (uint64_t)(v_slot * (kTileBytes >> 4));
    #pragma unroll
                    for (int ks = 0; ks < kN / 16; ++ks)
                        mma(tmem + col_o(x), tmem + col_s(x) + ks * 8,
                            vd + (uint64_t)((ks * 2048) >> 4), id_pv, (ks > 0 || !first) ? 1u : 0u);
                    return true;
                };
                Cursor cur = cursor_begin(S);
                Unit U;
                while (ok && next_unit(P, S, cur, U)) {
                    // tile A always exists (2t < NM); tile B may not
                    const int mA = last_tile(P, U.t, 0), mB = last_tile(P, U.t, 1);
                    const int jmax = mB >= 0 ? mB : mA;
                    if (*abort || !mbar_wait(&sh.q_full, (uint32_t)(nu & 1), P.wait) ||
                        !mbar_wait(&sh.full[slot], ph, P.wait)) {
                        ok = false;
                        break;
                    }
                    // S(0) of both tiles
                    issue_s(0, slot);
                    if (mB >= 0) issue_s(1, slot);
                    commit(&sh.empty[slot]);
                    if (jmax == 0) commit(&sh.q_empty);
                    advance();
                    for (int j = 0; j <= jmax; ++j) {
                        const int vslot = slot;
                        if (!mbar_wait(&sh.full[vslot], ph, P.wait)) {
                            ok = false;
                            break;
                        }
                        advance();
                        const bool next = j < jmax;
                        const int kslot = slot;
                        if (next && !mbar_wait(&sh.full[kslot], ph, P.wait)) {
                            ok = false;
                            break;
                        }
                        if (j <= mA) {
                            if (!issue_pv(0, vslot, j == 0)) {
                                ok = false;
                                break;
                            }
                            if (j == mA) commit(&sh.o_done[0]);
                            if (j < mA) issue_s(0, kslot);
                        }
                        if (mB >= 0) {     // j <= mB == jmax
                            if (!issue_pv(1, vslot, j == 0)) {
                                ok = false;
                                break;
                            }
                            if (j == mB) commit(&sh.o_done[1]);
                            commit(&sh.empty[vslot]);
                            if (next) issue_s(1, kslot);
                        } else {
                            commit(&sh.empty[vslot]);
                        }
                        if (next) {
                            commit(&sh.empty[kslot]);
                            if (j + 1 == jmax) commit(&sh.q_empty);
                            advance();
                        }
                    }
                    ++nact[0];
                    if (mB >= 0) ++nact[1];
                    ++nu;
                }
                if (!ok) {
                    raise_status(P.status, SPEC_DEV_TIMEOUT);
                    *abort = 1;
                }
                // every MMA issued above has completed before TMEM is released
                commit(&sh.drain);
                if (!mbar_wait(&sh.drain, 0)) raise_status(P.status, SPEC_DEV_TIMEOUT);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
        // ------------------------------------------------------ softmax
        const int x = warp / kGroupWarps;               // query tile A (0) or B (1)
        const int r = (warp % kGroupWarps) * 32 + lane; // row of the tile
        const uint32_t lane_base = (uint32_t)((warp % kGroupWarps) * 32) << 16;
        const uint32_t tS = tmem + lane_base + col_s(x), tO = tmem + lane_base + col_o(x);
        const float sc = P.scale_log2;
        int ns = 0, nact = 0;      // S hand-offs taken; units this tile took part in
        bool ok = true;
        Cursor cur = cursor_begin(S);
        Unit U;
        while (ok && next_unit(P, S, cur, U)) {
            const int mX = last_tile(P, U.t, x);
            if (mX < 0) continue;
            const int i = mX * kM + r;               // this thread's position
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j <= mX; ++j) {
                if (__any_sync(0xffffffffu, *abort != 0) ||
                    !mbar_wait_warp(&sh.s_full[x], (uint32_t)(ns & 1), P.wait)) {
                    ok = false;
                    break;
                }
                ++ns;
                fence_after();
                const bool masked = j == mX || (j + 1) * kN > P.n;
                const int c0 = j * kN;
                // visibility of keys lo .. lo + 31 for this row: key c is
                // visible iff c <= i and (c < n or c == i)
                auto vis_bits = [&](int lo) -> uint32_t {
                    if (!masked) return 0xffffffffu;
                    const int di = i - lo, dn = P.n - lo;
                    const uint32_t le = di < 0 ? 0u : di >= 31 ? 0xffffffffu
                                                               : (2u << di) - 1u;
                    const uint32_t lt = dn <= 0 ? 0u : dn >= 32 ? 0xffffffffu
                                                                : (1u << dn) - 1u;
                    const uint32_t self = (di >= 0 && di < 32) ? (1u << di) : 0u;
                    return (le & lt) | self;
                };
                // the S row: four TMEM loads in flight, one wait (each
                // wait_ld ties its registers; the later ones return at once)
                uint32_t v[kN / 32][32];
#pragma unroll
                for (int c = 0; c < kN / 32; ++c) ld32(tS + c * 32, v[c]);
#pragma unroll
                for (int c = 0; c < kN / 32; ++c) wait_ld(v[c]);
                // masked tiles: invisible scores become -inf in place
                if (masked) {
#pragma unroll
                    for (int c = 0; c < kN / 32; ++c) {
                        const uint32_t vm = vis_bits(c0 + c * 32);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[c][e] = ((vm >> e) & 1u) ? v[c][e] : 0xff800000u;
                    }
                }
                // the row maximum (three-input max, four chains)
                float tmv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < kN / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            tmv[q] = max3(tmv[q], __uint_as_float(v[c][e + 2 * q]),
                                          __uint_as_float(v[c][e + 2 * q + 1]));
                const float traw = fmaxf(fmaxf(tmv[0], tmv[1]), fmaxf(tmv[2], tmv[3]));
                const float tm = traw == -INFINITY ? -INFINITY : traw * sc;
                const bool raise = tm > m_used + kRescale || (m_used == -INFINITY && tm != -INFINITY);
                const float alpha =
                    !raise ? 1.f : (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - tm);
                // O holds every earlier PV of this tile (issued before the S
                // just waited for): rescale the rows that raised their max
                // (TMEM loads and stores are warp-collective: the whole warp
                // takes part, the other rows scaled by exactly 1)
                const bool scale_o = raise && j > 0 && m_used != -INFINITY;
                if (__any_sync(0xffffffffu, scale_o)) {
                    const float a = scale_o ? alpha : 1.f;
#pragma unroll 1
                    for (int c = 0; c < kD / 32; ++c) {
                        uint32_t o[32];
                        ld32(tO + c * 32, o);
                        wait_ld(o);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
                        st32(tO + c * 32, o);
                    }
                }
                if (raise) {
                    l *= alpha;
                    m_used = tm;
                }
                const float mu = m_used == -INFINITY ? 0.f : m_used;
                // P = exp2(s * scale - mu) (pairs: one f32x2 FMA, two ex2,
                // one f32x2 add, one pack) over the first 64 columns of S
                const uint64_t sc2 = pair(sc, sc), nmu2 = pair(-mu, -mu);
                uint64_t rs2[2] = {pair(0.f, 0.f), pair(0.f, 0.f)};
#pragma unroll
                for (int c = 0; c < kN / 32; ++c) {
                    uint32_t pw[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float t0, t1;
                        unpair(fma2(pair(__uint_as_float(v[c][2 * e]),
                                         __uint_as_float(v[c][2 * e + 1])),
                                    sc2, nmu2),
                               t0, t1);
                        const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
                        rs2[e & 1] = add2(rs2[e & 1], pair(p0, p1));
                        pw[e] = pack_bf16(p0, p1);
                    }
                    st16(tS + c * 16, pw);
                }
                float rs[4];
                unpair(rs2[0], rs[0], rs[1]);
                unpair(rs2[1], rs[2], rs[3]);
                l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
                wait_st();
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.p_full[x]);
            }
            if (!ok) break;
            // epilogue: O / l (bf16) and the LSE of this row
            if (!mbar_wait_warp(&sh.o_done[x], (uint32_t)(nact & 1), P.wait)) {
                ok = false;
                break;
            }
            fence_after();
            const bool row_ok = i < P.L;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(
                P.o + (((size_t)U.b * P.L + (row_ok ? i : 0)) * P.Hq + U.hq) * kD);
#pragma unroll 1
            for (int c = 0; c < kD / 32; ++c) {
                uint32_t v[32];
                ld32(tO + c * 32, v);
                wait_ld(v);
                if (!row_ok) continue;
#pragma unroll
                for (int e = 0; e < 32; e += 8)
                    dst[(c * 32 + e) / 8] = make_uint4(
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
            if (lane == 0) mbar_arrive(&sh.o_free[x]);
            ++nact;
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

// Unit schedule for `grid` CTAs: heads are taken kSchedHeads at a time (a
// multiple of the KV group, so the CTAs at work share few K/V sets in L2),
// and within such a window the longest unit goes first onto the CTA with the
// least work so far (cost of a unit: its key tiles plus a fixed allowance
// for the Q load and the epilogue).  Returns false when the table does not
// fit; the result depends only on the arguments and is cached.
constexpr int kSchedHeads = 8;
constexpr int kUnitOverhead = 2;

bool build_schedule(int BH, int G, int NB, int NM, int grid, lap::Sched &out) {
    const long long n_units = (long long)BH * NB;
    if (n_units >= 65536 || n_units + grid + 1 > lap::kSchedCap) return false;
    using Key = std::tuple<int, int, int, int, int>;
    static std::mutex mu;
    static std::map<Key, std::vector<uint16_t>> cache;
    const Key key{BH, G, NB, NM, grid};
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it == cache.end()) {
        const int W = ((kSchedHeads + G - 1) / G) * G;
        std::vector<std::vector<uint16_t>> lists(grid);
        using Slot = std::pair<long long, int>;           // (work so far, CTA)
        std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
        for (int c = 0; c < grid; ++c) heap.push({0, c});
        for (int h0 = 0; h0 < BH; h0 += W) {
            const int h1 = std::min(BH, h0 + W);
            for (int t = NB - 1; t >= 0; --t) {
                const int jmax = 2 * t + 1 < NM ? 2 * t + 1 : 2 * t;
                for (int bh = h0; bh < h1; ++bh) {
                    Slot sl = heap.top();
                    heap.pop();
                    lists[sl.second].push_back((uint16_t)(bh * NB + t));
                    heap.push({sl.first + jmax + 1 + kUnitOverhead, sl.second});
                }
            }
        }
        std::vector<uint16_t> v(grid + 1 + n_units);
        int e = 0;
        for (int c = 0; c < grid; ++c) {
            v[c] = (uint16_t)e;
            for (uint16_t id : lists[c]) v[grid + 1 + e++] = id;
        }
        v[grid] = (uint16_t)e;
        it = cache.emplace(key, std::move(v)).first;
    }
    out.n = (int)it->second.size();
    std::copy(it->second.begin(), it->second.end(), out.v);
    return true;
}

// 4-D bf16 map over [B][L][H][128] with a (64, 1, 128, 1) box: one
// 128-position x 64-element block of one head, 128-byte swizzle.  Positions
// past L read as zeros.
bool make_map_4d(CUtensorMap *map, const void *base, int H, int L, int B) {
    constexpr int D = lap::kD;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                   (cuuint64_t)L * H * D * 2};
    const cuuint32_t box[4] = {64u, 1u, (cuuint32_t)lap::kM, 1u};
    return encode_bf16_map(map, base, 4, dims, strides, box);
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
    P.NB = (P.NM + 1) / 2;
    P.NP = (P.NB + 1) / 2;
    const long long items = (long long)B * Hq * P.NP;
    if (items > 0x7fffffffll) return SPEC_ERR_UNSUPPORTED;
    P.n_items = (int)items;
    const float scale = desc->scale > 0.f ? desc->scale : 1.f / sqrtf((float)lap::kD);
    P.scale_log2 = scale * kLog2e;
    P.o = static_cast<__nv_bfloat16 *>(o);
    P.lse = lse;
    P.status = st;
    P.wait = wait_limit();

    CUtensorMap maps[3];
    if (!make_map_4d(&maps[0], q, Hq, (int)L, B) || !make_map_4d(&maps[1], k, Hkv, (int)L, B) ||
        !make_map_4d(&maps[2], v, Hkv, (int)L, B))
        return SPEC_ERR_CUDA;

    if (set_smem_limit(reinterpret_cast<const void *>(la_prefill_kernel), lap::kSmemBytes) !=
        SPEC_OK)
        return SPEC_ERR_CUDA;
    const long long n_units = (long long)B * Hq * P.NB;
    static thread_local lap::Sched sched;   // 16 KB: kept off the stack
    int grid = (int)std::min<long long>(num_sms(), n_units);
    if (!build_schedule(B * Hq, P.G, P.NB, P.NM, grid, sched)) {
        sched.n = 0;
        grid = (int)std::min<long long>(num_sms(), items);
    }
    if (launch(la_prefill_kernel, dim3(grid), dim3(lap::kThreads), lap::kSmemBytes,
               as_stream(stream), P, maps[0], maps[1], maps[2], sched) != SPEC_OK)
        return SPEC_ERR_CUDA;
    return launch_status();
}
