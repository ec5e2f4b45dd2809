// Work schedule shared by the tensor-core verify-attention kernels of
// attn_tc.cu (the mma.sync and tcgen05 kernels): the linear step space, the
// split into CTA ranges, the cursor, the boundary records for the combine,
// and the tcgen05 kernel's step producer.
//
// Work is one linear space of steps over segments: a segment is one unit of
// a kernel (mma.sync: a (request, KV head, row block); tcgen05: see the
// kernels), its steps its prefix tiles, then its soft-prompt tiles, then its
// block tiles (64 tokens each, or pairs of them).  A persistent grid cuts
// the space into contiguous CTA ranges of equal cost; a CTA writes one fp32
// partial (m, l, O) per segment it shares with another CTA, and a combine
// kernel merges those.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_tc.cuh"
#include "ptx_sm103.cuh"

namespace sv {

constexpr int kTile = 64;                 // tokens per tile
constexpr int kHalfBytes = kTile * 128;   // one 64-token x 64-element bf16 box

// A split segment, as the CTA holding its first boundary between CTA
// ranges records it (tcgen05 attention kernel) for the combine; seg < 0 in
// every other CTA's record.
struct BoundaryRec {
    long long s0, s1;    // the segment's tiles
    int seg;             // (b * seg_h + h) * seg_rb + rb
    int first, last;     // CTAs whose ranges meet [s0, s1)
    uint32_t parts;      // bit j: CTA first + j holds a part (when last - first < 32)
};

struct TcParams {
    AttnParams a;
    int n_ctas;
    int soft_tiles;      // ceil(n_soft / 64)
    int tail;            // soft_tiles + ceil(R / 64)
    int box_rows;        // rows per cache box: 64 (contiguous) or NH * page_size
    int page_log2;       // log2(page_size) (paged)
    int seg_cost;        // what a segment start costs, in tiles, for the split
    long long *bounds;   // first tile of each CTA's range, [n_ctas + 1] (workspace),
                         // written by the attention kernel for the combine
    BoundaryRec *recs;   // tcgen05 kernel: per CTA, the split segment it merges
                         // (workspace, [n_ctas])
    long long wait;      // limit of every pipeline wait, in SM cycles
    // segments of a request: seg_h x seg_rb, numbered h * seg_rb + rb (the
    // mma.sync kernel: KV heads x row blocks; the tcgen05 kernels: their
    // units)
    int seg_h, seg_rb;
    // tcgen05 kernel: um_merged: a unit is two KV heads, their rows in one
    // query block (the second at lanes 64..127), else one row block;
    // um_act[x]: softmax warps of sub-tile x that take part (bit q: lane
    // quarter q)
    int um_merged;
    unsigned um_act[2];
    int pair_steps;      // a schedule step covers two 64-token tiles (tcgen05 kernels)
};

namespace {

// -------------------------------------------------------------- schedule

__device__ __forceinline__ int req_seq(const TcParams &P, int b) {
    int S = P.a.seq_len[b];
    return S < 0 ? 0 : (S > P.a.capacity ? P.a.capacity : S);
}

// Schedule steps of a segment with prefix S: its 64-token tiles (prefix,
// soft prompt, block), or pairs of them.
__device__ __forceinline__ int seg_tiles(const TcParams &P, int S) {
    const int n = ceil_div(S, kTile) + P.tail;
    return P.pair_steps ? (n + 1) >> 1 : n;
}

// The split.  CTAs take equal parts of a cost space in which every segment
// counts its tiles plus P.seg_cost for its start (epilogue, query block,
// row flags), so a CTA whose range holds many short segments gets fewer
// tiles.  Segment s of request b occupies costs [Cb + s u, Cb + (s + 1) u),
// u = tiles + seg_cost; the first seg_cost + 1 of them map to its first tile.
// A CTA's range is the tiles its part of the cost space maps to.
//
// A warp reads the prefix lengths once (WarpSched): lane l holds requests
// [lo, hi), ceil(B / 32) of them, with their tile and cost sums and the
// exclusive prefix sums of both over the lanes before it.  Every lookup
// below is then a ballot and a few shuffles (and, with more than 32
// requests, a walk over one lane's requests).
struct WarpSched {
    long long T, C;          // total tiles and cost
    long long et, ec;        // tiles and cost of the requests before lo
    long long st, sc;        // tiles and cost of requests lo .. hi - 1
    int lo, hi;
    int s_lo;                // prefix length of request lo (lo < hi)
};

__device__ WarpSched warp_sched(const TcParams &P) {
    const int lane = threadIdx.x & 31;
    const int B = P.a.B, per = ceil_div(B, 32);
    const long long units = (long long)P.seg_h * P.seg_rb;
    WarpSched w;
    w.lo = min(B, lane * per);
    w.hi = min(B, w.lo + per);
    w.st = w.sc = 0;
    w.s_lo = 0;
    for (int b = w.lo; b < w.hi; ++b) {
        const int S = req_seq(P, b);
        if (b == w.lo) w.s_lo = S;
        const long long n = (long long)seg_tiles(P, S) * units;
        w.st += n;
        w.sc += n + (long long)P.seg_cost * units;
    }
    long long it = w.st, ic = w.sc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long vt = __shfl_up_sync(0xffffffffu, it, o);
        const long long vc = __shfl_up_sync(0xffffffffu, ic, o);
        if (lane >= o) {
            it += vt;
            ic += vc;
        }
    }
    w.et = it - w.st;
    w.ec = ic - w.sc;
    w.T = __shfl_sync(0xffffffffu, it, 31);
    w.C = __shfl_sync(0xffffffffu, ic, 31);
    return w;
}

// Request b holding position x (< the total) of the tile space (by_cost =
// false) or of the cost space (true), with the tiles and cost of the
// requests before it and its prefix length (warp-collective).
__device__ void sched_locate(const TcParams &P, const WarpSched &w, long long x, bool by_cost,
                             int &b, long long &t0, long long &c0, int &S) {
    const long long e = by_cost ? w.ec : w.et, n = by_cost ? w.sc : w.st;
    const unsigned m = __ballot_sync(0xffffffffu, w.lo < w.hi && x >= e && x < e + n);
    const int src = m ? __ffs(m) - 1 : 0;
    b = __shfl_sync(0xffffffffu, w.lo, src);
    const int hi = __shfl_sync(0xffffffffu, w.hi, src);
    t0 = __shfl_sync(0xffffffffu, w.et, src);
    c0 = __shfl_sync(0xffffffffu, w.ec, src);
    S = __shfl_sync(0xffffffffu, w.s_lo, src);
    const long long units = (long long)P.seg_h * P.seg_rb;
    while (b < hi - 1) {            // more than 32 requests: walk the lane's
        const long long nt = (long long)seg_tiles(P, S) * units;
        const long long nc = nt + (long long)P.seg_cost * units;
        if (x < (by_cost ? c0 + nc : t0 + nt)) break;
        t0 += nt;
        c0 += nc;
        S = req_seq(P, ++b);
    }
}

// Request b's prefix length and the tiles and cost of the requests before
// it (warp-collective).
__device__ void sched_request(const TcParams &P, const WarpSched &w, int b, int &S,
                              long long &t0, long long &c0) {
    const int per = ceil_div(P.a.B, 32), src = b / per;
    t0 = __shfl_sync(0xffffffffu, w.et, src);
    c0 = __shfl_sync(0xffffffffu, w.ec, src);
    S = __shfl_sync(0xffffffffu, w.s_lo, src);
    const long long units = (long long)P.seg_h * P.seg_rb;
    for (int i = src * per; i < b; ++i) {      // more than 32 requests
        const long long nt = (long long)seg_tiles(P, S) * units;
        t0 += nt;
        c0 += nt + (long long)P.seg_cost * units;
        S = req_seq(P, i + 1);
    }
}

// First tile of CTA i's range (warp-collective).
__device__ long long sched_range_lo(const TcParams &P, const WarpSched &w, int i) {
    if (i <= 0) return 0;
    if (i >= P.n_ctas) return w.T;
    if (P.seg_cost == 0) return w.T * i / P.n_ctas;    // plain tile split
    const long long c = w.C * i / P.n_ctas;
    int b, S;
    long long t0, c0;
    sched_locate(P, w, c, true, b, t0, c0, S);
    const int nt = seg_tiles(P, S);
    const long long u = nt + P.seg_cost;
    const long long seg = (c - c0) / u, off = (c - c0) % u;
    return t0 + seg * nt + (off > P.seg_cost ? off - P.seg_cost : 0);
}

// CTA whose range holds a tile, from the tile's last position x in the
// cost space (C in total): CTA i's range starts at the tile that position
// C i / n maps to, so it is the last i with C i / n <= x.  For tile j of a
// segment whose costs start at cs, x = cs + seg_cost + j.
__device__ __forceinline__ int cost_split_cta(long long C, int n, long long x) {
    const long long i = ((long long)n * (x + 1) + C - 1) / C - 1;
    return (int)(i < 0 ? 0 : (i >= n ? n - 1 : i));
}

// CTA whose range holds tile t, from the bounds the attention kernel wrote:
// the last CTA whose range starts at or before t (empty ranges share their
// start with the next one).
__device__ __forceinline__ int cta_holding(const TcParams &P, long long t) {
    int lo = 0, hi = P.n_ctas - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P.bounds[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

struct Cursor {
    int b, h, rb;
    int S, n_prefix, n_tiles;   // prefix tokens, its 64-token tiles, the segment's steps
    int tile;                   // step within the segment
};

// The cursor at tile t (< the total; warp-collective).
__device__ void cursor_init(const TcParams &P, const WarpSched &w, long long t, Cursor &c) {
    long long start, c0;
    sched_locate(P, w, t, false, c.b, start, c0, c.S);
    c.n_prefix = ceil_div(c.S, kTile);
    c.n_tiles = seg_tiles(P, c.S);
    const long long local = t - start;
    const int seg = (int)(local / c.n_tiles);
    c.tile = (int)(local % c.n_tiles);
    c.h = seg / P.seg_rb;
    c.rb = seg % P.seg_rb;
}

__device__ __forceinline__ void cursor_next(const TcParams &P, Cursor &c) {
    if (++c.tile < c.n_tiles) return;
    c.tile = 0;
    if (++c.rb < P.seg_rb) return;
    c.rb = 0;
    if (++c.h < P.seg_h) return;
    c.h = 0;
    if (++c.b < P.a.B) {
        c.S = req_seq(P, c.b);
        c.n_prefix = ceil_div(c.S, kTile);
        c.n_tiles = seg_tiles(P, c.S);
    }
}

enum { kPrefix = 0, kSoft = 1, kBlock = 2 };

struct TileInfo {
    int kind, base, nvalid, j;
};

// 64-token tile t of the cursor's segment (0 <= t < n_prefix + tail).
__device__ __forceinline__ TileInfo tile_at(const TcParams &P, const Cursor &c, int t) {
    TileInfo ti;
    if (t < c.n_prefix) {
        ti.kind = kPrefix;
        ti.j = t;
        ti.base = t * kTile;
        ti.nvalid = min(kTile, c.S - ti.base);
    } else if (t - c.n_prefix < P.soft_tiles) {
        ti.kind = kSoft;
        ti.j = t - c.n_prefix;
        ti.base = ti.j * kTile;
        ti.nvalid = min(kTile, P.a.n_soft - ti.base);
    } else {
        ti.kind = kBlock;
        ti.j = t - c.n_prefix - P.soft_tiles;
        ti.base = ti.j * kTile;
        ti.nvalid = min(kTile, P.a.R - ti.base);
    }
    return ti;
}

// The tile of the cursor's step (segments of one tile per step).
__device__ __forceinline__ TileInfo tile_info(const TcParams &P, const Cursor &c) {
    return tile_at(P, c, c.tile);
}

__device__ __forceinline__ size_t slot_row(const TcParams &P, int seg, int cta, int wc, int wcn,
                                           int row) {
    return ((size_t)(seg + cta) * wcn + wc) * P.a.rb_rows + row;
}

__device__ __forceinline__ void check_seq_len(const AttnParams &A, int b) {
    const int S_raw = A.seq_len[b];
    if (S_raw < 0 || S_raw > A.capacity) raise_status(A.status, SPEC_DEV_SEQ_OVERFLOW);
}

// The record this CTA writes for the combine (warp-collective): when its
// range starts inside a unit and the ranges between the unit's first CTA
// and this one are empty (this is the unit's first boundary), the unit and
// the CTAs sharing it; otherwise seg = -1.
__device__ BoundaryRec warp_boundary_record(const TcParams &P, const WarpSched &w, int cta,
                                            long long t_begin, long long t_end) {
    BoundaryRec rec{0, 0, -1, 0, 0, 0};
    if (t_begin >= t_end) return rec;
    Cursor c;
    cursor_init(P, w, t_begin, c);
    if (c.tile == 0) return rec;
    rec.s0 = t_begin - c.tile;
    rec.s1 = rec.s0 + c.n_tiles;
    bool first_boundary = true;
    int f = cta - 1, l = cta;
    for (;; --f) {
        const long long lo = sched_range_lo(P, w, f);
        if (lo <= rec.s0 || f == 0) break;
        if (lo < t_begin) first_boundary = false;   // a part starts in between
    }
    while (l + 1 < P.n_ctas && sched_range_lo(P, w, l + 1) < rec.s1) ++l;
    if (!first_boundary) return rec;
    rec.seg = (c.b * P.seg_h + c.h) * P.seg_rb + c.rb;
    rec.first = f;
    rec.last = l;
    if (l - f < 32) {
        long long lo = sched_range_lo(P, w, f);
        for (int j = f; j <= l; ++j) {
            const long long hi = sched_range_lo(P, w, j + 1);
            if (max(lo, rec.s0) < min(hi, rec.s1)) rec.parts |= 1u << (j - f);
            lo = hi;
        }
    }
    return rec;
}

// ------------------------------------------------ tcgen05 kernels' steps

namespace tcs {

constexpr int kRows = 128;              // rows per tile (MMA M)
// A slot holds the K (or V) of one step: two 64-token sub-tiles x 128 head
// dimensions, as two 64-element halves hh, each 128 rows of 128 bytes
// (sub-tile x at rows 64 x ..), 128-byte swizzled: token t of sub-tile x,
// elements 64 hh .. 64 hh + 63 at byte hh * kHalf + (64 x + t) * 128.
constexpr int kHalf = 2 * 64 * 128;
constexpr int kSlotBytes = 2 * kHalf;   // 32 KB
constexpr int kSlots = 5;               // ring: K and V of a step in consecutive slots
constexpr int kQHalf = kRows * 128;     // one 64-element half of a query block
constexpr int kQBytes = 2 * kQHalf;     // one query block: 128 rows x 128

// The producer's buffers and barriers: a ring of kSlots slots (the K and V
// of step n in slots 2n and 2n + 1 modulo kSlots, full / empty per slot)
// and the query staging (q_full: loaded; q_empty: its unit is done with it).
struct ProducerIO {
    uint8_t *ring, *qbuf;
    uint64_t *full, *empty, *q_full, *q_empty;
};

// One sub-tile of a step: the KV head whose keys it holds and its 64-token
// tile, or absent (merged: an odd last head; rows mode: past the last tile).
struct Sub {
    int head;
    TileInfo ti;
    bool present;
};

// Whether the cursor's step has sub-tile 1.
__device__ __forceinline__ bool has_sub1(const TcParams &P, const Cursor &c) {
    return P.um_merged ? 2 * c.h + 1 < P.a.Hkv : 2 * c.tile + 1 < c.n_prefix + P.tail;
}

// Sub-tile x of the cursor's step.
__device__ __forceinline__ Sub sub_tile(const TcParams &P, const Cursor &c, int x) {
    Sub u;
    if (P.um_merged) {
        u.head = 2 * c.h + x;
        u.present = u.head < P.a.Hkv;
        u.ti = tile_at(P, c, c.tile);
    } else {
        u.head = c.h;
        const int t = 2 * c.tile + x;
        u.present = t < c.n_prefix + P.tail;
        u.ti = tile_at(P, c, u.present ? t : 0);
    }
    return u;
}

// Producer warp: for each step of [t_begin, t_end), its K and V (both
// sub-tiles) into consecutive ring slots, and each unit's query block ahead
// of its first step.  Every lane owns one box of a step -- lane
// 16 kv + 8 x + 2 i + hh: K (kv = 0) or V, sub-tile x, page i (paged prefix
// tiles: boxes of page_size rows; other tiles: i = 0, boxes of 64 rows),
// half hh -- so that one warp-wide TMA instruction issues the whole step and
// every sub-tile has the same layout.
__device__ void run_step_producer(const TcParams &P, const CUtensorMap &mk, const CUtensorMap &mv,
                                  const CUtensorMap &mkb, const CUtensorMap &mvb,
                                  const CUtensorMap &msk, const CUtensorMap &msv,
                                  const CUtensorMap &mq, const ProducerIO &io,
                                  const WarpSched &w, long long t_begin, long long t_end) {
    uint8_t *ring = io.ring, *qbuf = io.qbuf;
    constexpr int NH = 2;
    const AttnParams &A = P.a;
    const int lane = threadIdx.x & 31;
    const int kv = lane >> 4, x = (lane >> 3) & 1, pi = (lane >> 1) & 3, hh = lane & 1;
    const uint64_t pol_keep = policy_evict_last();
    // a prefix is read by one unit unless several row blocks share its head
    const uint64_t pol_stream =
        (P.um_merged || A.n_rb == 1) ? policy_evict_first() : pol_keep;
    const int ps = A.paged ? A.page_size : kTile;
    const int ppt = kTile / ps;          // pages per 64-token tile (paged)

    long long ld = 0;                    // slot loads issued
    int nq = 0;                          // query blocks issued
    bool ok = true;
    Cursor c;
    cursor_init(P, w, t_begin, c);       // warp-collective
    for (long long t = t_begin; t < t_end; ++t) {
        if (t == t_begin || c.tile == 0) {
            // the unit's query block, once the previous unit's block has
            // been copied to TMEM (q_empty): 128 packed rows of one head
            // (lane hh issuing half hh), or 64 of each of the unit's two
            // heads (merged, lane 2 x + hh issuing head 2u + x's half hh)
            bool got = true;
            if (lane == 0) got = nq == 0 || mbar_wait(io.q_empty, (uint32_t)((nq - 1) & 1), P.wait);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                ok = false;
                break;
            }
            if (P.um_merged) {
                const int nh = 2 * c.h + 1 < A.Hkv ? 2 : 1;
                if (lane == 0) mbar_arrive_expect_tx(io.q_full, (uint32_t)nh * (kQBytes / 2));
                __syncwarp();
                if (lane < 2 * nh)
                    tma_load_4d(qbuf + (lane & 1) * kQHalf + (lane >> 1) * (kQHalf / 2), &mq,
                                (lane & 1) * 64, 0, 2 * c.h + (lane >> 1), c.b * A.R, io.q_full,
                                pol_keep);
            } else {
                if (lane == 0) mbar_arrive_expect_tx(io.q_full, (uint32_t)kQBytes);
                __syncwarp();
                if (lane < NH)
                    tma_load_4d(qbuf + lane * kQHalf, &mq, lane * 64, 0, c.h,
                                c.b * A.R + c.rb * (kRows / A.G), io.q_full, pol_keep);
            }
            ++nq;
        }
        // this lane's box of the step
        const Sub u = sub_tile(P, c, x);
        const CUtensorMap *map = nullptr;
        int bx = 0, by = 0;
        uint32_t bytes = 0;
        uint64_t pol = pol_keep;
        if (u.present) {
            const TileInfo &ti = u.ti;
            if (ti.kind == kPrefix && A.paged) {
                const int tok = ti.base + pi * ps;
                if (pi < ppt && tok < c.S) {
                    const int pg = A.page_table[(size_t)c.b * A.max_pages + tok / ps];
                    if (pg < 0 || pg >= A.n_pages) {
                        raise_status(A.status, SPEC_DEV_BAD_PAGE);
                    } else {
                        map = kv ? &mv : &mk;
                        by = ((pg * A.Hkv + u.head) * NH + hh) * ps;
                        bytes = (uint32_t)ps * 128u;
                        pol = pol_stream;
                    }
                }
            } else if (pi == 0) {
                bx = hh * 64;
                bytes = (uint32_t)kTile * 128u;
                if (ti.kind == kPrefix) {
                    map = kv ? &mv : &mk;
                    by = (c.b * A.Hkv + u.head) * A.max_seq + ti.base;
                    pol = pol_stream;
                } else if (ti.kind == kSoft) {
                    map = kv ? &msv : &msk;
                    by = u.head * A.n_soft + ti.base;
                } else {
                    map = kv ? &mvb : &mkb;
                    by = (c.b * A.Hkv + u.head) * A.R + ti.base;
                }
            }
        }
        const uint32_t bytes_k = __reduce_add_sync(0xffffffffu, kv == 0 ? bytes : 0u);
        const uint32_t bytes_v = __reduce_add_sync(0xffffffffu, kv == 1 ? bytes : 0u);
        const int ks = (int)(ld % kSlots), vs = (int)((ld + 1) % kSlots);
        bool got = true;
        if (lane == 0)
            got = mbar_wait(&io.empty[ks], (uint32_t)(((ld / kSlots) & 1) ^ 1), P.wait) &&
                  mbar_wait(&io.empty[vs], (uint32_t)((((ld + 1) / kSlots) & 1) ^ 1), P.wait);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
            ok = false;
            break;
        }
        if (lane == 0) {
            mbar_arrive_expect_tx(&io.full[ks], bytes_k);
            mbar_arrive_expect_tx(&io.full[vs], bytes_v);
        }
        __syncwarp();
        const int slot = kv ? vs : ks;
        if (bytes)
            tma_load_2d(ring + slot * kSlotBytes + hh * kHalf + (x * kTile + pi * ps) * 128, map, bx,
                        by, &io.full[slot], pol);
        ld += 2;
        cursor_next(P, c);
    }
    if (lane == 0) {
        if (!ok) raise_status(A.status, SPEC_DEV_TIMEOUT);
        // do not leave while copies into this CTA's shared memory are in
        // flight (the default limit: these copies were issued and complete)
        for (long long i = ld - 1; i >= 0 && i >= ld - kSlots; --i)
            if (!mbar_wait(&io.full[i % kSlots], (uint32_t)((i / kSlots) & 1))) {
                raise_status(A.status, SPEC_DEV_TIMEOUT);
                break;
            }
        if (nq > 0 && !mbar_wait(io.q_full, (uint32_t)((nq - 1) & 1)))
            raise_status(A.status, SPEC_DEV_TIMEOUT);
    }
}

}  // namespace tcs

}  // namespace
}  // namespace sv
