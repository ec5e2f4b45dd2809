"""GPU parity of spec_la_prefill_attn -- the prefill form of Lookahead
Attention ("Lookahead Attention", sec. 3.1: all n + k positions under the
full M_LA mask) -- against the float64 oracle, element by element.

Shapes span several 128-row query tiles with a ragged last tile, lookahead
rows that straddle a tile boundary, GQA groups, a single-tile request, pure
causal prefill (k = 0), and sharp score distributions that make the running
max grow across key tiles.  The full LLaMA-7B-shaped size is checked on
whole (request, head) slices.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, f64, require_gpu
from self_speculative_verification_gb300 import binding as bd
from self_speculative_verification_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def run_gpu(wl, scale=0.0):
    dev = torch.device("cuda", 0)
    q = torch.from_numpy(wl.q).to(dev, torch.bfloat16)
    k = torch.from_numpy(wl.kk).to(dev, torch.bfloat16)
    v = torch.from_numpy(wl.v).to(dev, torch.bfloat16)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((wl.B, wl.Hq, wl.L), float("nan"), dtype=torch.float32, device=dev)
    bd.spec_la_prefill_attn(bd.prefill_desc(wl.B, wl.n, wl.k, wl.Hq, wl.Hkv, wl.d, scale=scale),
                            q, k, v, o, lse)
    torch.cuda.synchronize()
    assert bd.spec_get_status() == 0
    return f64(o), lse.cpu().numpy().astype(np.float64)


def check(wl, O, LSE, pairs=None, scale=None):
    """Compare the (request, head) slices in ``pairs`` (all by default)."""
    tol = TOL["bf16"]
    G = wl.Hq // wl.Hkv
    if pairs is None:
        pairs = [(b, h) for b in range(wl.B) for h in range(wl.Hq)]
    worst = 0.0
    for b, h in pairs:
        Or, Lr = oracle.la_prefill_attention(wl.q[b, :, h], wl.kk[b, :, h // G],
                                             wl.v[b, :, h // G], wl.n, scale=scale)
        Og, Lg = O[b, :, h], LSE[b, h]
        assert np.isfinite(Og).all() and np.isfinite(Lg).all()
        err = np.abs(Og - Or)
        assert err.max() <= tol["o_abs"], f"(b={b}, h={h}) max abs err {err.max()}"
        assert np.linalg.norm(Og - Or) / np.linalg.norm(Or) <= tol["o_rel_norm"]
        rel = np.abs(Lg - Lr) / np.abs(Lr)
        assert rel.max() <= tol["lse_rel"], f"(b={b}, h={h}) LSE rel err {rel.max()}"
        worst = max(worst, err.max())
    return worst


@pytest.mark.parametrize("B,n,k,Hq,Hkv", [
    (1, 1, 1, 1, 1),        # two positions
    (1, 127, 1, 2, 2),      # exactly one query tile
    (2, 200, 8, 4, 2),      # two tiles, ragged, GQA 2
    (1, 120, 16, 2, 1),     # lookahead rows straddle the tile boundary
    (2, 600, 8, 4, 1),      # five tiles (paired 4+0, 3+1, middle 2), GQA 4
    (1, 256, 0, 2, 2),      # k = 0: causal prefill of the originals
    (3, 1000, 7, 3, 3),     # eight tiles, ragged, more items than pairs
])
def test_prefill_parity(B, n, k, Hq, Hkv):
    require_gpu()
    wl = W.make_prefill(seed=n * 31 + k, B=B, n=n, k=k, Hq=Hq, Hkv=Hkv)
    O, LSE = run_gpu(wl)
    check(wl, O, LSE)


@pytest.mark.parametrize("q_scale", [16.0, 64.0])
def test_prefill_sharp_scores(q_scale):
    """Large queries: peaked softmax, the running max moves across tiles."""
    require_gpu()
    wl = W.make_prefill(seed=7, B=1, n=700, k=8, Hq=2, Hkv=1, q_scale=q_scale)
    O, LSE = run_gpu(wl)
    check(wl, O, LSE)


def test_prefill_explicit_scale():
    require_gpu()
    wl = W.make_prefill(seed=3, B=1, n=300, k=4, Hq=2, Hkv=2)
    O, LSE = run_gpu(wl, scale=0.2)
    check(wl, O, LSE, scale=0.2)


def test_prefill_many_items():
    """More work items than SMs: every CTA takes several item rounds."""
    require_gpu()
    wl = W.make_prefill(seed=11, B=8, n=1500, k=8, Hq=16, Hkv=4)
    O, LSE = run_gpu(wl)
    check(wl, O, LSE, pairs=[(0, 0), (3, 5), (7, 15), (5, 8)])


def test_prefill_without_unit_table():
    """More (request, head, tile pair) units than the launch's unit table
    holds: the CTAs fall back to taking the paired items round-robin."""
    require_gpu()
    wl = W.make_prefill(seed=13, B=64, n=5, k=3, Hq=128, Hkv=16)     # 8192 units
    O, LSE = run_gpu(wl)
    check(wl, O, LSE, pairs=[(b, h) for b in range(0, 64, 7) for h in range(0, 128, 5)])


def test_prefill_full_size_slices():
    """The LLaMA-7B-shaped prefill workload, whole (request, head) slices."""
    require_gpu()
    cfg = W.PREFILL_CONFIGS["la_prefill"]
    wl = W.make_prefill(seed=0, **cfg)
    O, LSE = run_gpu(wl)
    check(wl, O, LSE, pairs=[(0, 0), (1, 17), (3, 31)])


def test_prefill_rejects_bad_shapes():
    require_gpu()
    dev = torch.device("cuda", 0)
    q = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16, device=dev)
    o = torch.zeros_like(q)
    lse = torch.zeros(1, 2, 8, dtype=torch.float32, device=dev)
    cases = [
        (bd.prefill_desc(1, 0, 8, 2, 2, 128), bd.SPEC_ERR_INVALID_ARG),     # n = 0
        (bd.prefill_desc(1, 4, -1, 2, 2, 128), bd.SPEC_ERR_INVALID_ARG),    # k < 0
        (bd.prefill_desc(1, 4, 4, 3, 2, 128), bd.SPEC_ERR_INVALID_ARG),     # Hq % Hkv
        (bd.prefill_desc(1, 4, 4, 2, 2, 64), bd.SPEC_ERR_UNSUPPORTED),      # head_dim
        (bd.prefill_desc(1, 4, 4, 2, 2, 128, dtype=bd.SPEC_F32), bd.SPEC_ERR_UNSUPPORTED),
        (bd.prefill_desc(1, 4, 4, 2, 2, 128, scale=-1.0), bd.SPEC_ERR_INVALID_ARG),
    ]
    for desc, code in cases:
        with pytest.raises(bd.SpecError) as e:
            bd.spec_la_prefill_attn(desc, q, kv, kv, o, lse)
        assert e.value.code == code
    # an empty batch launches nothing
    bd.spec_la_prefill_attn(bd.prefill_desc(0, 4, 4, 2, 2, 128), q, kv, kv, o, lse)
    assert bd.spec_get_status() == 0
