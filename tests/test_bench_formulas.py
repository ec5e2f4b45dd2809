"""The numerators of the bench's roofline figures, checked by counting on
small cases instead of by the closed forms bench.py uses: visible
(query, key) pairs of the LA prefill mask, inner nodes of the draft trees
the oracle builds, the page-table entries a paged prefix touches, and the
verify attention's bytes rebuilt from the arrays the oracle reads."""

from types import SimpleNamespace

import numpy as np
import pytest

import bench
import oracle
from self_speculative_verification_gb300 import workloads as W


@pytest.mark.parametrize("n,k", [(1, 0), (1, 3), (5, 3), (17, 4), (64, 8)])
def test_prefill_flops_count_the_mask(n, k):
    """4 d FLOPs (QK^T and PV) per visible pair and head ("Lookahead
    Attention" sec. 3.1 mask), nothing for masked pairs."""
    wl = SimpleNamespace(n=n, k=k, d=128, B=3, Hq=5)
    pairs = int(oracle.la_prefill_mask(n, k).sum())
    assert bench.prefill_flops(wl) == 4 * wl.d * pairs * wl.B * wl.Hq


@pytest.mark.parametrize("gamma,k", [(1, 3), (2, 2), (3, 4)])
def test_draft_bytes_count_inner_nodes(gamma, k):
    """The early-exit rows read are those of nodes with a child in the trees
    the oracle builds ("Speculative Streaming", tree draft pruning)."""
    dw = W.make_draft(3, B=2, gamma=gamma, k=k, V=64)
    inner = 0
    for b in range(dw.B):
        _, parent, _ = oracle.draft_tree(dw.stream_logits[b], k, dw.root_token[b])
        inner += len({int(p) for p in parent if p >= 0})
    e = 2 if dw.dtype == "bf16" else 4
    arrays = dw.B * dw.N * 4 * (2 + 2 + 1 + 2 * (1 + gamma))
    assert bench.draft_algorithmic_bytes(dw) == (dw.B * gamma + inner) * dw.V * e + arrays


def test_paged_attention_bytes_count_touched_pages():
    """The page-table entries counted are the pages that a request's prefix
    positions actually fall in."""
    wl = W.make_workload("long_paged", 2, B=3, seq=("uniform", 40, 300), V=64)
    assert wl.paged
    touched = 0
    for b in range(wl.B):
        S = int(wl.seq_len[b])
        touched += len({int(wl.page_table[b, t // wl.page_size]) for t in range(S)})
    base = bench.attn_algorithmic_bytes(wl)
    wl.paged = False
    assert base - bench.attn_algorithmic_bytes(wl) == touched * 4


@pytest.mark.parametrize("name,kw", [
    ("confu", dict(B=2, seq=("uniform", 50, 200), V=64)),
    ("long_paged", dict(B=2, seq=("uniform", 40, 200), V=64)),
])
def test_attention_bytes_count_the_arrays(name, kw):
    """spec_verify_attn's algorithmic bytes rebuilt from the arrays the
    oracle's attention reads: each request's prefix K and V (gathered from
    the paged cache where there is one), the block and soft-prompt K/V, q
    and an O of its size, LSE, and the integer inputs (lengths, the packed
    visibility words of the oracle's mask, row flags, touched pages)."""
    wl = W.make_workload(name, 4, **kw)
    e = 2 if wl.dtype == "bf16" else 4
    if wl.paged:
        Kp, Vp = wl.paged_cache(fill=0.0)
        ks = oracle.gather_paged(Kp, wl.page_table, wl.seq_len, wl.page_size)
        vs = oracle.gather_paged(Vp, wl.page_table, wl.seq_len, wl.page_size)
        prefix = sum(k.size + v.size for k, v in zip(ks, vs))
        pages = sum(len({int(wl.page_table[b, t // wl.page_size])
                         for t in range(int(wl.seq_len[b]))}) for b in range(wl.B))
    else:
        prefix = sum(sum(x.size for x in wl.prefix_kv(b)) for b in range(wl.B))
        pages = 0
    soft = (wl.soft_k.size + wl.soft_v.size) if wl.n_soft > 0 else 0
    vis, _, _ = oracle.mask_build(wl.vparent, wl.soft_flags)
    words = vis.shape[0] * vis.shape[1] * ((vis.shape[2] + 31) // 32)
    ints = wl.seq_len.size * 4 + words * 4 + wl.B * wl.R + pages * 4
    lse = wl.B * wl.Hq * wl.R * 4
    want = (prefix + wl.kb.size + wl.vb.size + soft + 2 * wl.q.size) * e + lse + ints
    assert bench.attn_algorithmic_bytes(wl) == want
