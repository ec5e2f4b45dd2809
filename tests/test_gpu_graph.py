"""The step's calls can be captured in a CUDA graph (no host synchronisation,
no allocation, launch shapes fixed by the descriptors): a replayed graph
gives bit-identical results to direct calls."""

import numpy as np
import pytest
import torch

import gpu_helpers as gh
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300 import workloads as W
from self_speculative_verification_gb300.device import DeviceStep

pytestmark = pytest.mark.gpu

OUTS = ("o", "lse", "acc_len", "path", "next_token", "last_node", "k_cache", "v_cache",
        "seq_len")


def _bits(t):
    """Storage bits (unused cache slots hold NaN, which never equals itself)."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16)
    if t.dtype == torch.float32:
        return t.view(torch.int32)
    return t


def _snapshot(ds):
    return {n: _bits(getattr(ds, n)).clone() for n in OUTS}


@pytest.mark.parametrize("name,kw", [
    ("la7b", dict(B=3, seq=("uniform", 100, 700), V=4000)),
    ("long_paged", dict(B=3, seq=("uniform", 300, 1100), V=4000)),
    ("ss", dict(B=3, seq=("uniform", 100, 500), V=5000)),
    ("ss_soft", dict(B=3, seq=("uniform", 100, 500), V=5000)),
    ("ss_rot", dict(B=3, seq=("uniform", 100, 500), V=5000)),
    ("confu", dict(B=2, seq=("uniform", 150, 600), V=5000)),
])
def test_step_graph_replay_matches_direct(name, kw):
    gh.require_gpu()
    wl = W.make_workload(name, 3, **kw)
    ds = DeviceStep(wl)
    ds.reset_state()
    ds.run()                      # first calls (one-time setup) outside the capture
    torch.cuda.synchronize()
    ds.reset_state(page_table=True)
    ds.run()
    torch.cuda.synchronize()
    want = _snapshot(ds)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ds.reset_state(page_table=True)
        ds.run()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert bn.spec_get_status() == 0
        for n, t in want.items():
            assert torch.equal(_bits(getattr(ds, n)), t), n


def test_prefill_graph_replay_matches_direct():
    gh.require_gpu()
    wl = W.make_prefill(4, B=1, n=500, k=8, Hq=2, Hkv=1)
    dev = torch.device("cuda", 0)
    q = torch.from_numpy(wl.q).to(dev, torch.bfloat16)
    k = torch.from_numpy(wl.kk).to(dev, torch.bfloat16)
    v = torch.from_numpy(wl.v).to(dev, torch.bfloat16)
    o = torch.zeros_like(q)
    lse = torch.zeros((1, 2, wl.L), dtype=torch.float32, device=dev)
    d = bn.prefill_desc(1, wl.n, wl.k, 2, 1, 128)
    bn.spec_la_prefill_attn(d, q, k, v, o, lse)
    torch.cuda.synchronize()
    o0, l0 = o.clone(), lse.clone()
    o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bn.spec_la_prefill_attn(d, q, k, v, o, lse)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o0) and torch.equal(lse, l0)


def test_draft_and_prune_graph_replay_matches_direct():
    """The draft tree and its pruning (two entry points, five launches)
    captured together replay to the same trees as direct calls."""
    gh.require_gpu()
    dw = W.make_draft(5, B=4, V=5000)
    dev = torch.device("cuda", 0)
    B, N, g = dw.B, dw.N, dw.gamma
    R = N * (1 + g)
    i32 = torch.int32
    stream_l = torch.from_numpy(dw.stream_logits).to(dev, torch.bfloat16)
    early = torch.from_numpy(dw.early_logits).to(dev, torch.bfloat16)
    root = torch.from_numpy(dw.root_token).to(dev)
    tok, par, t2, p2, keep = (torch.zeros((B, N), dtype=i32, device=dev) for _ in range(5))
    nn, n2 = torch.zeros(B, dtype=i32, device=dev), torch.zeros(B, dtype=i32, device=dev)
    vp_full, vp = (torch.zeros((B, R), dtype=i32, device=dev) for _ in range(2))
    ddesc = bn.DraftDesc(B, g, g, dw.k, dw.V, bn.SPEC_BF16, N, R)
    pdesc = bn.PruneDesc(B, N, dw.V, bn.SPEC_BF16, dw.threshold, g, R)
    outs = (tok, par, nn, vp_full, keep, t2, p2, n2, vp)

    def calls():
        bn.spec_draft_tree(ddesc, stream_l, None, root, tok, par, nn, vp_full)
        bn.spec_prune_tree(pdesc, tok, par, nn, early, keep, t2, p2, n2, vp)

    calls()
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    want = [t.clone() for t in outs]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()
    for t in outs:
        t.fill_(-7)
    graph.replay()
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    for t, w in zip(outs, want):
        assert torch.equal(t, w)
