"""Seeded synthetic workloads for the self-speculative verification step.

Every input of the verification step -- query rows, committed KV prefix, the
speculative block's own K/V, soft-prompt KV, parent-pointer arrays, draft
trees, proposals and logits -- is drawn here from ``numpy.random.Generator``
(PCG64) with an explicit seed, so that x86 and Arm hosts produce the same
bits.  Both the CUDA path and the CPU oracle read these arrays; this module
holds none of the verification arithmetic (no attention, no acceptance).

Floating-point tensors are returned as ``float32`` arrays whose values are
exactly representable in the workload's storage type (bf16 values are
rounded here, round-to-nearest-even), so a bf16 device copy and an fp64 host
copy hold the same numbers.

Workload shapes follow the pages' settings:

* Lookahead Attention (LA) verify, "Lookahead Attention" sec. 2-3: ``k``
  lookahead rows that see the committed prefix and themselves, padded per
  request to one length (sec. 3.3), judged by a probability threshold
  (sec. 2.4).
* ConFu tree verify ("ConFu" notes, key design 1): ``T`` draft-tree nodes plus
  one contemplate token per node, 16 soft-prompt KV entries seen only by the
  contemplate tokens, judged by a greedy walk.
* Speculative Streaming multi-stream verify ("Speculative Streaming",
  Eq. 2 and Eq. 4, batching with streams): ``T`` tree nodes each with
  ``gamma`` stream rows.

Where a workload plants its logits (so that acceptance is decided by a wide
margin and never by rounding), the planted expectation is recorded as
``expect_acc_len`` / ``expect_path``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# --------------------------------------------------------------------------
# configuration table
# --------------------------------------------------------------------------

#: The five verification workloads (name -> parameters).  ``seq`` is either a
#: tuple of fixed prefix lengths or ``("uniform", lo, hi)``.
CONFIGS = {
    "tiny_la": dict(mode="la", B=2, Hq=4, Hkv=2, d=64, dtype="f32",
                    seq=(128, 200), k_choices=(4,), R=4, V=1000,
                    paged=False),
    "la7b": dict(mode="la", B=16, Hq=32, Hkv=32, d=128, dtype="bf16",
                 seq=("uniform", 512, 4096), k_choices=(2, 4, 8), R=8,
                 V=32000, paged=False),
    "confu": dict(mode="confu", B=8, Hq=32, Hkv=8, d=128, dtype="bf16",
                  seq=("uniform", 256, 2048), T=60, max_depth=8, branch=4,
                  n_soft=16, V=128256, paged=False),
    "ss": dict(mode="ss", B=32, Hq=32, Hkv=32, d=128, dtype="bf16",
               seq=("uniform", 128, 1024), T=16, gamma=3, branch=4,
               V=50272, paged=False),
    # the SS workload verified with soft matching ("Speculative Streaming",
    # verification step; T = 1 as in the page's top-k sampling runs)
    "ss_soft": dict(mode="ss", B=32, Hq=32, Hkv=32, d=128, dtype="bf16",
                    seq=("uniform", 128, 1024), T=16, gamma=3, branch=4,
                    V=50272, paged=False, soft=True, temperature=1.0),
    # the SS workload with stream values by rotation ("Speculative Streaming"
    # Eq. 7): eps at the page's upper bound pi / (2N), N = max sequence + streams
    "ss_rot": dict(mode="ss", B=32, Hq=32, Hkv=32, d=128, dtype="bf16",
                   seq=("uniform", 128, 1024), T=16, gamma=3, branch=4,
                   V=50272, paged=False, value_rotation=True),
    "long_paged": dict(mode="la", B=64, Hq=32, Hkv=8, d=128, dtype="bf16",
                       seq=("uniform", 16384, 32768), k_choices=(8,), R=8,
                       V=32000, paged=True),
}

TAU = 0.3            # LA acceptance threshold on the proposal probability
PAGE_SIZE = 16       # tokens per KV page (paged layout)
VALUE_SCALE = 1.0 / 8.0   # q, K, V ~ N(0, 1) / 8
MATCH_P = 0.8        # proposals / walk steps that match the target argmax
GREEDY_MARGIN = 0.5  # planted argmax margin for greedy (tree) workloads

# vparent codes for rows of the speculative block
VP_ROOT = -1   # row sees the committed prefix and itself only
VP_PAD = -2    # padding row: sees nothing, produces nothing


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even).

    Returned as float32 holding exactly representable bf16 numbers.
    NaN inputs stay NaN.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    nan = np.isnan(x)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) \
        & np.uint32(0xFFFF0000)
    out = r.view(np.float32).copy()
    out[nan] = np.float32(np.nan)
    return out


def _to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    return round_bf16(x) if dtype == "bf16" else x


def _normal(rng: np.random.Generator, shape, scale: float, dtype: str):
    x = rng.standard_normal(shape, dtype=np.float32) * np.float32(scale)
    return _to_storage(x, dtype)


# --------------------------------------------------------------------------
# the workload record
# --------------------------------------------------------------------------

@dataclass
class Workload:
    """All inputs of one verification step, plus planted expectations."""

    name: str
    mode: str                 # "la" (threshold chain) or "tree" (greedy walk)
    layout: str               # "la", "confu" or "ss": how block rows are laid out
    seed: int
    B: int
    R: int                    # padded speculative rows per request
    Hq: int
    Hkv: int
    d: int
    dtype: str                # "f32" or "bf16" (q, K, V, O storage)
    logit_dtype: str
    V: int                    # vocabulary
    Rj: int                   # judged rows per request (rows carrying logits)
    N: int                    # max nodes / proposals per request
    path_cap: int
    n_soft: int
    tau: float
    paged: bool
    seq_len: np.ndarray       # int32 [B]
    q: np.ndarray             # [B][R][Hq][d]
    kb: np.ndarray            # [B][Hkv][R][d]  speculative block K
    vb: np.ndarray            # [B][Hkv][R][d]  speculative block V
    soft_k: Optional[np.ndarray]   # [Hkv][n_soft][d]
    soft_v: Optional[np.ndarray]
    vparent: np.ndarray       # int32 [B][R]
    soft_flags: np.ndarray    # uint8 [B][R]
    tokens: np.ndarray        # int32 [B][N] draft tokens / proposals
    tree_parent: np.ndarray   # int32 [B][N] (-1 for the root / chain rows)
    n_nodes: np.ndarray       # int32 [B]
    logits: np.ndarray        # [B][Rj][V]
    expect_acc_len: np.ndarray   # int32 [B]
    expect_path: np.ndarray      # int32 [B][path_cap], -1 padded
    node_depth: np.ndarray = field(default=None)   # int32 [B][N]
    # soft matching (tree workloads with ``soft``): draft distributions,
    # draft row of each node's children (-1: none), the uniforms
    draft_logits: Optional[np.ndarray] = None     # [B][Rd][V]
    child_draft_row: Optional[np.ndarray] = None  # int32 [B][N]
    u_accept: Optional[np.ndarray] = None         # float32 [B][N]
    u_sample: Optional[np.ndarray] = None         # float32 [B]
    temperature: float = 1.0
    # stream values by rotation (SS layout): angle per stream index, or None
    rotation_eps: Optional[float] = None
    gamma: int = 0
    # contiguous cache capacity / paged bookkeeping
    max_seq: int = 0
    page_size: int = PAGE_SIZE
    n_pages: int = 0
    max_pages: int = 0
    page_table: Optional[np.ndarray] = None   # int32 [B][max_pages], -1 unused
    free_pages: Optional[np.ndarray] = None   # int32 [n_free]

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def soft(self) -> bool:
        return self.draft_logits is not None

    def prefix_kv(self, b: int):
        """The committed K/V prefix of request ``b``: two [Hkv][S_b][d] arrays.

        Drawn from its own seed stream so any request can be regenerated
        alone (used for sampled checks at full size).
        """
        S = int(self.seq_len[b])
        rng = np.random.Generator(np.random.PCG64(
            np.random.SeedSequence([self.seed, 0x4B56, b])))
        k = _normal(rng, (self.Hkv, S, self.d), VALUE_SCALE, self.dtype)
        v = _normal(rng, (self.Hkv, S, self.d), VALUE_SCALE, self.dtype)
        return k, v

    def verified_tokens(self) -> int:
        """Candidate tokens judged in one step (sum of n_nodes)."""
        return int(self.n_nodes.sum())

    def contiguous_cache(self, fill=np.nan):
        """K, V as [B][Hkv][max_seq][d] float32; slots past S_b hold ``fill``."""
        shape = (self.B, self.Hkv, self.max_seq, self.d)
        K = np.full(shape, fill, dtype=np.float32)
        Vc = np.full(shape, fill, dtype=np.float32)
        for b in range(self.B):
            k, v = self.prefix_kv(b)
            S = k.shape[1]
            K[b, :, :S] = k
            Vc[b, :, :S] = v
        return K, Vc

    def paged_cache(self, fill=np.nan):
        """K, V pages as [n_pages][Hkv][d // 64][page][64] (the paged layout:
        per head, the head dimension in 64-element blocks of page rows);
        unused slots hold ``fill``."""
        assert self.paged
        shape = (self.n_pages, self.Hkv, self.d // 64, self.page_size, 64)
        K = np.full(shape, fill, dtype=np.float32)
        Vc = np.full(shape, fill, dtype=np.float32)
        for b in range(self.B):
            k, v = self.prefix_kv(b)
            place_request_pages(self, b, k, v, K, Vc)
        return K, Vc


def place_request_pages(wl: Workload, b: int, k, v, Kp, Vp):
    """Scatter request ``b``'s logical prefix [Hkv][S][d] into page arrays
    [n_pages][Hkv][d // 64][page][64]."""
    S = k.shape[1]
    ps = wl.page_size
    for j in range((S + ps - 1) // ps):
        p = int(wl.page_table[b, j])
        t0, t1 = j * ps, min(S, (j + 1) * ps)
        for blk in range(wl.d // 64):
            Kp[p, :, blk, : t1 - t0] = k[:, t0:t1, blk * 64:(blk + 1) * 64]
            Vp[p, :, blk, : t1 - t0] = v[:, t0:t1, blk * 64:(blk + 1) * 64]


# --------------------------------------------------------------------------
# draft trees
# --------------------------------------------------------------------------

def random_tree(rng, T: int, max_depth: int, branch: int):
    """Random draft tree with ``T`` nodes (node 0 = root, parent < child).

    Each new node attaches to a uniformly chosen existing node whose depth is
    below ``max_depth`` and which has fewer than ``branch`` children.
    """
    parent = np.full(T, -1, dtype=np.int32)
    depth = np.zeros(T, dtype=np.int32)
    nchild = np.zeros(T, dtype=np.int32)
    for i in range(1, T):
        cand = [j for j in range(i) if depth[j] < max_depth and nchild[j] < branch]
        if not cand:
            raise ValueError("tree parameters admit no further node")
        p = cand[int(rng.integers(len(cand)))]
        parent[i] = p
        depth[i] = depth[p] + 1
        nchild[p] += 1
    return parent, depth


def full_tree(k: int, gamma: int):
    """The complete k-ary draft tree of depth ``gamma`` in breadth-first order.

    "Speculative Streaming", tree draft construction: top-k tokens per stream,
    stream-j tokens are parents of stream-(j+1) tokens.
    """
    parent = [-1]
    depth = [0]
    frontier = [0]
    for g in range(1, gamma + 1):
        nxt = []
        for p in frontier:
            for _ in range(k):
                parent.append(p)
                depth.append(g)
                nxt.append(len(parent) - 1)
        frontier = nxt
    return np.array(parent, dtype=np.int32), np.array(depth, dtype=np.int32)


def _distinct_child_tokens(rng, parent, V):
    """Tokens for tree nodes with siblings holding distinct tokens."""
    T = len(parent)
    tok = np.zeros(T, dtype=np.int32)
    tok[0] = int(rng.integers(V))
    used = {}
    for i in range(1, T):
        s = used.setdefault(int(parent[i]), set())
        while True:
            t = int(rng.integers(V))
            if t not in s:
                break
        s.add(t)
        tok[i] = t
    return tok


def tree_block_rows(layout: str, parent: np.ndarray, gamma: int = 0):
    """vparent and soft flags for the flattened block of a tree workload.

    ``confu``: rows 0..T-1 are the nodes, row T+j the contemplate token of
    node j (its vparent is node j; it alone sees the soft prompt).
    ``ss``: rows 0..T-1 are the nodes (main stream), row T + j*gamma + (s-1)
    is stream s of node j; stream 1's vparent is node j, stream s>1's is
    stream s-1 of the same node.
    ``tree``: nodes only.
    """
    T = len(parent)
    if layout == "confu":
        R = 2 * T
    elif layout == "ss":
        R = T * (1 + gamma)
    else:
        R = T
    vp = np.full(R, VP_PAD, dtype=np.int32)
    soft = np.zeros(R, dtype=np.uint8)
    for j in range(T):
        vp[j] = VP_ROOT if parent[j] < 0 else parent[j]
    if layout == "confu":
        for j in range(T):
            vp[T + j] = j
            soft[T + j] = 1
    elif layout == "ss":
        for j in range(T):
            for s in range(1, gamma + 1):
                r = T + j * gamma + (s - 1)
                vp[r] = j if s == 1 else r - 1
    return vp, soft


# --------------------------------------------------------------------------
# logits with planted decisions
# --------------------------------------------------------------------------

def _plant_threshold_row(rng, V, dtype, target, p):
    """Logit row whose softmax puts probability ~p on ``target``.

    Other logits ~ N(0,1); the target logit is set so that
    e^{z_t} / (e^{z_t} + sum_{j != t} e^{z_j}) = p before storage rounding.
    """
    z = _to_storage(rng.standard_normal(V, dtype=np.float32), dtype)
    others = np.delete(z.astype(np.float64), target)
    mo = others.max()
    log_rest = mo + math.log(np.exp(others - mo).sum())
    z[target] = math.log(p / (1.0 - p)) + log_rest
    return _to_storage(z, dtype)


def _plant_margin_row(rng, V, dtype, target, margin):
    """Logit row whose argmax is ``target`` by at least ``margin``."""
    z = _to_storage(rng.standard_normal(V, dtype=np.float32), dtype)
    z[target] = -np.inf
    mo = float(z.max())
    val = mo + margin + float(rng.random())
    z[target] = val
    z = _to_storage(z, dtype)
    assert z[target] - mo >= margin - 0.125
    return z


def _plant_probs_row(rng, V, dtype, probs):
    """Logit row whose softmax puts probability probs[t] on each token t of
    ``probs`` (their sum below 1) before storage rounding; other logits
    ~ N(0, 1)."""
    z = _to_storage(rng.standard_normal(V, dtype=np.float32), dtype).astype(np.float64)
    if probs:
        mask = np.ones(V, dtype=bool)
        mask[list(probs)] = False
        rest = z[mask]
        mo = rest.max()
        log_rest = mo + math.log(np.exp(rest - mo).sum())
        s = sum(probs.values())
        assert s < 1.0
        for t, p in probs.items():
            z[t] = math.log(p / (1.0 - s)) + log_rest
    return _to_storage(z.astype(np.float32), dtype)


def _plant_soft(rng, tree_parent, node_depth, tokens, D, V, dtype, path_cap):
    """Soft-matching decisions planted with a wide margin around each
    uniform.  Along the planted walk, the tested children of the current
    node get draft probabilities q ~ U[0.01, 0.04] and target probabilities
    p = ratio * q with ratio >= 1.6 u (accepted child) or ratio <= 0.6 u
    (rejected ones), so storage rounding (a few percent on p and q) never
    flips a decision.  Returns target logits [B][T][V], draft logits
    [B][D][V] (row g: the distribution of depth-(g+1) candidates),
    child_draft_row, u_accept, u_sample and the planted paths."""
    B, T = tree_parent.shape
    child_draft_row = np.where(node_depth < D, node_depth, -1).astype(np.int32)
    u_accept = rng.random((B, T), dtype=np.float32)
    u_sample = rng.random(B, dtype=np.float32)
    logits = np.empty((B, T, V), dtype=np.float32)
    draft = np.empty((B, D, V), dtype=np.float32)
    expect_len = np.zeros(B, dtype=np.int32)
    expect_path = np.full((B, path_cap), -1, dtype=np.int32)
    for b in range(B):
        par = tree_parent[b]
        p_plant, q_plant = {}, {}
        cur, path = 0, [0]
        while True:
            kids = [int(c) for c in np.nonzero(par == cur)[0]]
            if not kids:
                break
            acc_i = int(rng.integers(len(kids))) if rng.random() < MATCH_P else -1
            tested = kids if acc_i < 0 else kids[: acc_i + 1]
            pp = p_plant.setdefault(cur, {})
            qq = q_plant.setdefault(int(child_draft_row[b, cur]), {})
            for i, c in enumerate(tested):
                x, u = int(tokens[b, c]), float(u_accept[b, c])
                qx = float(rng.uniform(0.01, 0.04))
                if i == acc_i:
                    ratio = max(1.6 * u, float(rng.uniform(0.3, 2.5)))
                else:
                    ratio = u * float(rng.uniform(0.1, 0.6))
                qq[x] = qx
                pp[x] = ratio * qx
            if acc_i < 0:
                break
            cur = kids[acc_i]
            path.append(cur)
        for j in range(T):
            logits[b, j] = _plant_probs_row(rng, V, dtype, p_plant.get(j, {}))
        for g in range(D):
            draft[b, g] = _plant_probs_row(rng, V, dtype, q_plant.get(g, {}))
        expect_len[b] = len(path)
        expect_path[b, : len(path)] = path
    return logits, draft, child_draft_row, u_accept, u_sample, expect_len, expect_path


# --------------------------------------------------------------------------
# builders
# --------------------------------------------------------------------------

def _seq_lengths(rng, spec, B):
    if spec[0] == "uniform":
        return rng.integers(spec[1], spec[2] + 1, size=B).astype(np.int32)
    assert len(spec) == B
    return np.array(spec, dtype=np.int32)


def make_workload(name: str, seed: int = 0, *, B=None, seq=None, V=None,
                  q_scale: float = 1.0, T=None, k_choices=None,
                  paged=None, n_soft=None, slack_pages=None,
                  page_order: str = "shuffled", d=None, page_size=None,
                  dtype=None, Hq=None, Hkv=None) -> Workload:
    """Build one seeded workload; keyword overrides shrink it for tests."""
    cfg = dict(CONFIGS[name])
    if Hq is not None:
        cfg["Hq"] = Hq
    if Hkv is not None:
        cfg["Hkv"] = Hkv
    if B is not None:
        cfg["B"] = B
    if seq is not None:
        cfg["seq"] = seq
    if V is not None:
        cfg["V"] = V
    if T is not None:
        cfg["T"] = T
    if k_choices is not None:
        cfg["k_choices"] = k_choices
    if paged is not None:
        cfg["paged"] = paged
    if n_soft is not None:
        cfg["n_soft"] = n_soft
    if d is not None:
        cfg["d"] = d
    if dtype is not None:
        cfg["dtype"] = dtype
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x5EC])))
    B, Hq, Hkv, d, dt, Vv = (cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["d"],
                             cfg["dtype"], cfg["V"])
    seq_len = _seq_lengths(rng, cfg["seq"], B)
    layout = cfg["mode"]

    soft = {}
    if layout == "la":
        R = cfg["R"]
        k_b = rng.choice(np.array(cfg["k_choices"]), size=B).astype(np.int32)
        assert k_b.max() <= R
        vparent = np.full((B, R), VP_PAD, dtype=np.int32)
        for b in range(B):
            vparent[b, : k_b[b]] = VP_ROOT
        soft_flags = np.zeros((B, R), dtype=np.uint8)
        N = Rj = R
        path_cap = R
        n_nodes = k_b.copy()
        tree_parent = np.full((B, N), -1, dtype=np.int32)
        node_depth = np.zeros((B, N), dtype=np.int32)
        tokens = np.zeros((B, N), dtype=np.int32)
        logits = np.empty((B, Rj, Vv), dtype=np.float32)
        expect_len = np.zeros(B, dtype=np.int32)
        expect_path = np.full((B, path_cap), -1, dtype=np.int32)
        for b in range(B):
            stopped = False
            for r in range(R):
                a = int(rng.integers(Vv))
                p = float(rng.uniform(0.40, 0.95))
                logits[b, r] = _plant_threshold_row(rng, Vv, dt, a, p)
                if r < k_b[b]:
                    if rng.random() < MATCH_P:
                        tokens[b, r] = a
                    else:
                        t = int(rng.integers(Vv - 1))
                        tokens[b, r] = t if t < a else t + 1
                    if not stopped and tokens[b, r] == a:
                        expect_path[b, expect_len[b]] = r
                        expect_len[b] += 1
                    else:
                        stopped = True
        mode = "la"
        n_soft = 0
    else:
        T = cfg["T"]
        if layout == "confu":
            gamma = 0
            max_depth = cfg["max_depth"]
            n_soft = cfg["n_soft"]
        else:
            gamma = cfg["gamma"]
            max_depth = gamma
            n_soft = 0
        branch = cfg["branch"]
        N = Rj = T
        path_cap = T
        tree_parent = np.empty((B, T), dtype=np.int32)
        node_depth = np.empty((B, T), dtype=np.int32)
        tokens = np.empty((B, T), dtype=np.int32)
        vps = []
        softs = []
        for b in range(B):
            par, dep = random_tree(rng, T, max_depth, branch)
            tree_parent[b] = par
            node_depth[b] = dep
            tokens[b] = _distinct_child_tokens(rng, par, Vv)
            vp, sf = tree_block_rows(layout, par, gamma)
            vps.append(vp)
            softs.append(sf)
        vparent = np.stack(vps)
        soft_flags = np.stack(softs)
        R = vparent.shape[1]
        n_nodes = np.full(B, T, dtype=np.int32)
        soft = {}
        if cfg.get("soft"):
            (logits, draft, cdr, u_acc, u_smp, expect_len,
             expect_path) = _plant_soft(rng, tree_parent, node_depth, tokens, max_depth, Vv, dt,
                                        path_cap)
            soft = dict(draft_logits=draft, child_draft_row=cdr, u_accept=u_acc,
                        u_sample=u_smp, temperature=float(cfg.get("temperature", 1.0)))
        else:
            # plant the accepted path: from the root, with prob MATCH_P make the
            # target argmax equal to one (uniformly chosen) child's token.
            argtok = np.empty((B, T), dtype=np.int64)
            expect_len = np.zeros(B, dtype=np.int32)
            expect_path = np.full((B, path_cap), -1, dtype=np.int32)
            for b in range(B):
                par = tree_parent[b]
                planted = np.zeros(T, dtype=bool)
                cur = 0
                expect_path[b, 0] = 0
                expect_len[b] = 1
                while True:
                    kids = np.nonzero(par == cur)[0]
                    planted[cur] = True
                    if len(kids) and rng.random() < MATCH_P:
                        c = int(kids[int(rng.integers(len(kids)))])
                        argtok[b, cur] = tokens[b, c]
                        cur = c
                        expect_path[b, expect_len[b]] = c
                        expect_len[b] += 1
                    else:
                        kid_tok = set(int(t) for t in tokens[b, kids])
                        while True:
                            t = int(rng.integers(Vv))
                            if t not in kid_tok:
                                break
                        argtok[b, cur] = t
                        break
                for j in range(T):
                    if not planted[j]:
                        argtok[b, j] = int(rng.integers(Vv))
            logits = np.empty((B, Rj, Vv), dtype=np.float32)
            for b in range(B):
                for j in range(T):
                    logits[b, j] = _plant_margin_row(rng, Vv, dt, int(argtok[b, j]),
                                                     GREEDY_MARGIN)
        mode = "tree"

    q = _normal(rng, (B, R, Hq, d), VALUE_SCALE * q_scale, dt)
    kb = _normal(rng, (B, Hkv, R, d), VALUE_SCALE, dt)
    vb = _normal(rng, (B, Hkv, R, d), VALUE_SCALE, dt)
    if n_soft:
        soft_k = _normal(rng, (Hkv, n_soft, d), VALUE_SCALE, dt)
        soft_v = _normal(rng, (Hkv, n_soft, d), VALUE_SCALE, dt)
    else:
        soft_k = soft_v = None

    wl = Workload(
        name=name, mode=mode, layout=layout, seed=seed, B=B, R=R, Hq=Hq,
        Hkv=Hkv, d=d, dtype=dt, logit_dtype=dt, V=Vv, Rj=Rj, N=N,
        path_cap=path_cap, n_soft=n_soft, tau=TAU, paged=bool(cfg["paged"]),
        seq_len=seq_len, q=q, kb=kb, vb=vb, soft_k=soft_k, soft_v=soft_v,
        vparent=vparent, soft_flags=soft_flags, tokens=tokens,
        tree_parent=tree_parent, n_nodes=n_nodes, logits=logits,
        expect_acc_len=expect_len, expect_path=expect_path,
        node_depth=node_depth, **soft,
    )
    wl.max_seq = int(seq_len.max()) + R if B else R
    if layout == "ss":
        wl.gamma = gamma
        if cfg.get("value_rotation"):
            wl.rotation_eps = math.pi / (2.0 * (wl.max_seq + gamma))
    if page_size is not None:
        wl.page_size = page_size
    if wl.paged:
        ps = wl.page_size
        used = [(int(s) + ps - 1) // ps for s in seq_len]
        need = [(int(s) + R + ps - 1) // ps for s in seq_len]
        slack = B if slack_pages is None else slack_pages
        P = int(sum(need)) + slack
        perm = rng.permutation(P).astype(np.int32)
        if page_order == "sequential":
            perm = np.arange(P, dtype=np.int32)
        wl.max_pages = max(need) if B else 1
        wl.page_table = np.full((B, wl.max_pages), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            wl.page_table[b, : used[b]] = perm[off: off + used[b]]
            off += used[b]
        wl.free_pages = perm[off:].copy()
        wl.n_pages = P
    return wl


def config_names():
    return list(CONFIGS)


# --------------------------------------------------------------------------
# prefill form of Lookahead Attention
# --------------------------------------------------------------------------

#: Prefill-form LA ("Lookahead Attention" sec. 3.1, the full (n + k) mask):
#: n prompt positions plus k lookahead positions per request, with the
#: LLaMA-7B attention shape of the LA verify workload (32 heads MHA,
#: head_dim 128, bf16).  n = 4096 is the top of that workload's prefix range
#: and k = 8 its largest lookahead count.
PREFILL_CONFIGS = {
    "la_prefill": dict(B=4, n=4096, k=8, Hq=32, Hkv=32, d=128),
}


@dataclass
class PrefillWorkload:
    """Inputs of one prefill-form LA call (bf16-representable float32)."""

    B: int
    n: int
    k: int
    Hq: int
    Hkv: int
    d: int
    q: np.ndarray      # [B][n + k][Hq][d]
    kk: np.ndarray     # [B][n + k][Hkv][d]
    v: np.ndarray      # [B][n + k][Hkv][d]

    @property
    def L(self) -> int:
        return self.n + self.k


def make_prefill(seed: int = 0, *, B: int, n: int, k: int, Hq: int, Hkv: int,
                 d: int = 128, q_scale: float = 1.0) -> PrefillWorkload:
    """q, K, V ~ N(0, 1) / 8 (q times ``q_scale``), rounded to bf16."""
    rng = np.random.Generator(np.random.PCG64(seed))
    L = n + k
    q = _normal(rng, (B, L, Hq, d), VALUE_SCALE * q_scale, "bf16")
    kk = _normal(rng, (B, L, Hkv, d), VALUE_SCALE, "bf16")
    v = _normal(rng, (B, L, Hkv, d), VALUE_SCALE, "bf16")
    return PrefillWorkload(B, n, k, Hq, Hkv, d, q, kk, v)


# --------------------------------------------------------------------------
# tree draft construction and pruning ("Speculative Streaming")
# --------------------------------------------------------------------------

#: The next step's draft for the SS workload: gamma = 3 streams, top-k = 4
#: per stream (the page sweeps gamma in {3, 4} and k from 1 up), OPT-6.7B's
#: vocabulary, pruning threshold 0.05 (the page gives none).
DRAFT_CONFIGS = {
    "ss_draft": dict(B=32, gamma=3, k=4, V=50272, dtype="bf16", threshold=0.05),
}


@dataclass
class DraftWorkload:
    """Inputs of one draft construction + pruning, with planted outcomes."""

    B: int
    gamma: int
    k: int
    V: int
    dtype: str
    threshold: float
    stream_logits: np.ndarray    # [B][gamma][V]
    root_token: np.ndarray       # int32 [B]
    early_logits: np.ndarray     # [B][N][V]: early-exit logits at each node
    expect_top: np.ndarray       # int32 [B][gamma][k]: planted top-k per stream
    expect_keep: np.ndarray      # bool [B][N]: planted survivors

    @property
    def N(self) -> int:
        return 1 + sum(self.k ** g for g in range(1, self.gamma + 1))


def make_draft(seed: int = 0, *, B=32, gamma=3, k=4, V=50272, dtype="bf16",
               threshold=0.05, keep_p=0.7) -> DraftWorkload:
    """Stream rows ~ N(0, 1) with k planted winners (logits 10 - 0.5 i, the
    middle two tied so the lower id must come first); early-exit rows
    ~ N(0, 1) with, at every inner node, each child token planted at a
    probability >= 1.6 x threshold (kept, with prob keep_p) or <= 0.6 x
    threshold (pruned)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xD7A])))
    parent, depth = full_tree(k, gamma)
    N = len(parent)
    stream = np.empty((B, gamma, V), dtype=np.float32)
    top = np.empty((B, gamma, k), dtype=np.int32)
    for b in range(B):
        for j in range(gamma):
            z = rng.standard_normal(V, dtype=np.float32)
            ids = rng.choice(V, size=k, replace=False)
            vals = [10.0 - 0.5 * i for i in range(k)]
            if k >= 3:
                vals[2] = vals[1]                      # a tie at ranks 1 and 2
            for t, val in zip(ids, vals):
                z[t] = val
            order = sorted(range(k), key=lambda i: (-vals[i], int(ids[i])))
            top[b, j] = [int(ids[i]) for i in order]
            stream[b, j] = _to_storage(z, dtype)
    root = rng.integers(0, V, B).astype(np.int32)
    early = np.empty((B, N, V), dtype=np.float32)
    keep = np.zeros((B, N), dtype=bool)
    for b in range(B):
        keep[b, 0] = True
        edge = {}
        for p in range(N):
            probs = {}
            if depth[p] < gamma:
                kids = np.nonzero(parent == p)[0]
                for i, c in enumerate(kids):
                    ok = rng.random() < keep_p
                    edge[int(c)] = ok
                    lo, hi = (1.6, 4.0) if ok else (0.1, 0.6)
                    probs[int(top[b, depth[p], i])] = threshold * float(rng.uniform(lo, hi))
            early[b, p] = _plant_probs_row(rng, V, dtype, probs)
        for c in range(1, N):
            keep[b, c] = keep[b, parent[c]] and edge[c]
    return DraftWorkload(B, gamma, k, V, dtype, threshold, stream, root, early, top, keep)
