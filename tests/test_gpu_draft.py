"""GPU parity of draft-tree construction and pruning ("Speculative
Streaming": tree draft construction, parallel tree pruning, batching with
streams) against the oracle.  Everything here is integer output decided by
exact comparisons of stored logits (top-k) or by planted margins (pruning),
so it must match bit for bit."""

import numpy as np
import pytest
import torch

import gpu_helpers as gh
import oracle
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300 import workloads as W
from self_speculative_verification_gb300.workloads import round_bf16

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
I32 = torch.int32


@pytest.fixture(autouse=True)
def _gpu():
    gh.require_gpu()


def _logits(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(DEV, dtype)


def run_draft(stream, root, k, gamma, stream_row=None, dtype=torch.bfloat16, slack=3):
    B, rows, V = stream.shape
    n = 1 + sum(k ** g for g in range(1, gamma + 1))
    N = n + slack
    R = N * (1 + gamma)
    tok = torch.full((B, N), 7, dtype=I32, device=DEV)
    par = torch.full((B, N), 7, dtype=I32, device=DEV)
    nn = torch.zeros(B, dtype=I32, device=DEV)
    vp = torch.full((B, R), 7, dtype=I32, device=DEV)
    sr = None if stream_row is None else torch.tensor(stream_row, dtype=I32, device=DEV)
    d = bn.DraftDesc(B, rows, gamma, k, V, bn.SPEC_BF16 if dtype == torch.bfloat16 else bn.SPEC_F32,
                     N, R)
    bn.spec_draft_tree(d, _logits(stream, dtype), sr, torch.tensor(root, dtype=I32, device=DEV),
                       tok, par, nn, vp)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    return tok.cpu().numpy(), par.cpu().numpy(), nn.cpu().numpy(), vp.cpu().numpy(), N, R


def check_draft(stream, root, k, gamma, tok, par, nn, vp, N, R, stream_row=None):
    for b in range(stream.shape[0]):
        r0 = 0 if stream_row is None else stream_row[b]
        t, p, _ = oracle.draft_tree(stream[b, r0:r0 + gamma], k, root[b])
        n = len(t)
        assert nn[b] == n
        assert tok[b, :n].tolist() == t.tolist()
        assert par[b, :n].tolist() == p.tolist()
        assert np.all(tok[b, n:] == -1) and np.all(par[b, n:] == -1)
        assert vp[b].tolist() == oracle.ss_block_vparent(p, gamma, R).tolist()


@pytest.mark.parametrize("k,gamma,dtype", [(4, 3, torch.bfloat16), (1, 4, torch.bfloat16),
                                           (8, 2, torch.float32), (3, 3, torch.float32)])
def test_draft_random_logits(k, gamma, dtype):
    rng = np.random.Generator(np.random.PCG64(k * 100 + gamma))
    B, V = 5, 3001
    stream = rng.standard_normal((B, gamma, V)).astype(np.float32)
    if dtype == torch.bfloat16:
        stream = W.round_bf16(stream)
    root = rng.integers(0, V, B)
    out = run_draft(stream, root, k, gamma, dtype=dtype)
    check_draft(stream, root, k, gamma, *out)


def test_draft_ties_go_to_lower_ids():
    rng = np.random.Generator(np.random.PCG64(3))
    B, V, k, gamma = 4, 5000, 8, 2
    stream = rng.integers(-2, 3, (B, gamma, V)).astype(np.float32)   # massive ties
    root = rng.integers(0, V, B)
    out = run_draft(stream, root, k, gamma)
    check_draft(stream, root, k, gamma, *out)


def test_draft_stream_row_offsets():
    rng = np.random.Generator(np.random.PCG64(4))
    B, rows, V, k, gamma = 3, 10, 2000, 2, 3
    stream = W.round_bf16(rng.standard_normal((B, rows, V)).astype(np.float32))
    root = rng.integers(0, V, B)
    sr = [0, 4, 7]
    out = run_draft(stream, root, k, gamma, stream_row=sr)
    check_draft(stream, root, k, gamma, *out, stream_row=sr)


def run_prune(dw, tok, par, nn, N, R):
    B = dw.B
    early = _logits(dw.early_logits, torch.bfloat16)
    keep = torch.full((B, N), 9, dtype=I32, device=DEV)
    t2 = torch.full((B, N), 9, dtype=I32, device=DEV)
    p2 = torch.full((B, N), 9, dtype=I32, device=DEV)
    n2 = torch.zeros(B, dtype=I32, device=DEV)
    vp = torch.full((B, R), 9, dtype=I32, device=DEV)
    d = bn.PruneDesc(B, N, dw.V, bn.SPEC_BF16, dw.threshold, dw.gamma, R)
    bn.spec_prune_tree(d, tok, par, nn, early, keep, t2, p2, n2, vp)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    return [x.cpu().numpy() for x in (keep, t2, p2, n2, vp)]


@pytest.mark.parametrize("seed,B,V", [(0, 3, 2000), (1, 6, 4000), (2, 32, 50272)])
def test_draft_then_prune(seed, B, V):
    dw = W.make_draft(seed, B=B, V=V)
    N = dw.N
    R = N * (1 + dw.gamma)
    stream = _logits(dw.stream_logits, torch.bfloat16)
    tok = torch.zeros((B, N), dtype=I32, device=DEV)
    par = torch.zeros((B, N), dtype=I32, device=DEV)
    nn = torch.zeros(B, dtype=I32, device=DEV)
    d = bn.DraftDesc(B, dw.gamma, dw.gamma, dw.k, V, bn.SPEC_BF16, N, R)
    bn.spec_draft_tree(d, stream, None, torch.from_numpy(dw.root_token).to(DEV), tok, par, nn)
    keep, t2, p2, n2, vp = run_prune(dw, tok, par, nn, N, R)
    tok_h, par_h = tok.cpu().numpy(), par.cpu().numpy()
    for b in range(B):
        t, p, _ = oracle.draft_tree(dw.stream_logits[b], dw.k, dw.root_token[b])
        assert tok_h[b].tolist() == t.tolist() and par_h[b].tolist() == p.tolist()
        rt, rp, km = oracle.prune_tree(t, p, dw.early_logits[b], dw.threshold)
        assert np.array_equal(km >= 0, dw.expect_keep[b])
        assert keep[b].tolist() == km.tolist()
        m = len(rt)
        assert n2[b] == m
        assert t2[b, :m].tolist() == rt.tolist() and p2[b, :m].tolist() == rp.tolist()
        assert np.all(t2[b, m:] == -1) and np.all(p2[b, m:] == -1)
        assert vp[b].tolist() == oracle.ss_block_vparent(rp, dw.gamma, R).tolist()



@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [777, 4096, 50272])
def test_prune_irregular_trees(dtype, V):
    """Trees that are not full: random recursive parents mixed with chains,
    requests of 1, 2, 57 and 200 nodes, so that an edge-test CTA takes
    several inner rows (the row stream's barriers carried from one row to
    the next) and some rows take the plain-load path (odd V)."""
    rng = np.random.Generator(np.random.PCG64(V * 2 + (dtype == "f32")))
    sizes = [1, 2, 57, 200]
    B, N, gamma, thr = len(sizes), max(sizes), 2, 0.05
    R = N * (1 + gamma)
    par = np.full((B, N), -1, np.int32)
    tok = np.full((B, N), -1, np.int32)
    early = rng.standard_normal((B, N, V), dtype=np.float32)
    for b, n in enumerate(sizes):
        for c in range(1, n):
            par[b, c] = rng.integers(0, c) if rng.random() < 0.7 else c - 1
        tok[b, :n] = rng.integers(0, V, size=n)
        # most edges far above the threshold (their tokens' logit 12 against
        # N(0, 1) elsewhere), the others far below it
        for c in range(1, n):
            if rng.random() < 0.85:
                early[b, par[b, c], tok[b, c]] = 12.0
    if dtype == "bf16":
        early = round_bf16(early)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    keep = torch.full((B, N), 9, dtype=I32, device=DEV)
    t2 = torch.full((B, N), 9, dtype=I32, device=DEV)
    p2 = torch.full((B, N), 9, dtype=I32, device=DEV)
    n2 = torch.zeros(B, dtype=I32, device=DEV)
    vp = torch.full((B, R), 9, dtype=I32, device=DEV)
    d = bn.PruneDesc(B, N, V, bn.SPEC_BF16 if dtype == "bf16" else bn.SPEC_F32, thr, gamma, R)
    nn = torch.tensor(sizes, dtype=I32, device=DEV)
    bn.spec_prune_tree(d, torch.from_numpy(tok).to(DEV), torch.from_numpy(par).to(DEV), nn,
                       _logits(early, tdt), keep, t2, p2, n2, vp)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    keep, t2, p2, n2, vp = (x.cpu().numpy() for x in (keep, t2, p2, n2, vp))
    for b, n in enumerate(sizes):
        rt, rp, km = oracle.prune_tree(tok[b, :n], par[b, :n], early[b, :n].astype(np.float64), thr)
        assert keep[b, :n].tolist() == km.tolist() and np.all(keep[b, n:] == -1)
        m = len(rt)
        assert n2[b] == m
        assert t2[b, :m].tolist() == rt.tolist() and p2[b, :m].tolist() == rp.tolist()
        assert np.all(t2[b, m:] == -1) and np.all(p2[b, m:] == -1)
        assert vp[b].tolist() == oracle.ss_block_vparent(rp, gamma, R).tolist()

def test_pruned_block_feeds_mask_build():
    """draft -> prune -> spec_mask_build gives the oracle's visibility."""
    dw = W.make_draft(5, B=4, V=3000)
    N = dw.N
    R = N * (1 + dw.gamma)
    assert R <= 256 * 2
    k, gamma = dw.k, dw.gamma
    stream = _logits(dw.stream_logits, torch.bfloat16)
    tok = torch.zeros((dw.B, N), dtype=I32, device=DEV)
    par = torch.zeros((dw.B, N), dtype=I32, device=DEV)
    nn = torch.zeros(dw.B, dtype=I32, device=DEV)
    bn.spec_draft_tree(bn.DraftDesc(dw.B, gamma, gamma, k, dw.V, bn.SPEC_BF16, N, R), stream,
                       None, torch.from_numpy(dw.root_token).to(DEV), tok, par, nn)
    keep, t2, p2, n2, vp = run_prune(dw, tok, par, nn, N, R)
    # the mask takes at most 256 rows: keep the first 256 of each block
    rows = min(R, 256)
    vp_dev = torch.from_numpy(np.ascontiguousarray(vp[:, :rows])).to(DEV)
    if rows < R:
        assert np.all(n2 * (1 + gamma) <= rows), "pruned blocks fit the mask"
    vis = torch.zeros((dw.B, rows, (rows + 31) // 32), dtype=I32, device=DEV)
    flags = torch.zeros((dw.B, rows), dtype=torch.uint8, device=DEV)
    bn.spec_mask_build(vp_dev, None, vis, flags)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    want, valid, _ = oracle.mask_build(vp[:, :rows])
    assert np.array_equal(gh.unpack_vis(vis.cpu().numpy(), rows), want)
    assert np.array_equal((flags.cpu().numpy() & 1) != 0, valid)


def test_draft_and_prune_reject_bad_arguments():
    z = torch.zeros((1, 3, 100), dtype=torch.bfloat16, device=DEV)
    root = torch.zeros(1, dtype=I32, device=DEV)
    buf = torch.zeros((1, 400), dtype=I32, device=DEV)
    n = torch.zeros(1, dtype=I32, device=DEV)
    cases = [
        (bn.DraftDesc(1, 3, 3, 9, 100, bn.SPEC_BF16, 400, 400), bn.SPEC_ERR_UNSUPPORTED),  # k > 8
        (bn.DraftDesc(1, 3, 3, 4, 100, bn.SPEC_BF16, 20, 400), bn.SPEC_ERR_CAPACITY),      # 85 > 20
        (bn.DraftDesc(1, 3, 0, 4, 100, bn.SPEC_BF16, 400, 400), bn.SPEC_ERR_INVALID_ARG),
        (bn.DraftDesc(1, 3, 3, 4, 100, bn.SPEC_BF16, 100, 100), bn.SPEC_ERR_CAPACITY),     # vparent
    ]
    for d, code in cases:
        with pytest.raises(bn.SpecError) as e:
            bn.spec_draft_tree(d, z, None, root, buf, buf, n, buf)
        assert e.value.code == code
    pd = bn.PruneDesc(1, 2000, 100, bn.SPEC_BF16, 0.1, 3, 8000)
    with pytest.raises(bn.SpecError) as e:
        bn.spec_prune_tree(pd, buf, buf, n, z, buf, buf, buf, n, None)
    assert e.value.code == bn.SPEC_ERR_UNSUPPORTED
