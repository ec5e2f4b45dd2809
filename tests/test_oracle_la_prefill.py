"""Pins of the prefill form of Lookahead Attention ("Lookahead Attention",
sec. 3.1: the full (n + k) x (n + k) mask M_LA)."""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _sdpa(q, k, v, causal=False):
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))[None, None]
    return F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal)[0, 0].numpy()


@pytest.mark.parametrize("n,k", [(1, 1), (4, 3), (9, 8), (30, 2)])
def test_prefill_rows(n, k):
    rng = np.random.Generator(np.random.PCG64(n * 10 + k))
    d = 16
    q, kk, v = (rng.standard_normal((n + k, d)) for _ in range(3))
    O, LSE = oracle.la_prefill_attention(q, kk, v, n)
    # original rows: causal attention over the originals only (never see lookahead)
    np.testing.assert_allclose(O[:n], _sdpa(q[:n], kk[:n], v[:n], causal=True), atol=1e-12)
    # lookahead row j: attention over all originals plus itself
    for j in range(n, n + k):
        K = np.concatenate([kk[:n], kk[j:j + 1]])
        V = np.concatenate([v[:n], v[j:j + 1]])
        np.testing.assert_allclose(O[j], _sdpa(q[j:j + 1], K, V)[0], atol=1e-12)


@pytest.mark.parametrize("n,k", [(1, 1), (4, 3), (17, 8), (120, 8)])
def test_prefill_vparent_closure_is_m_la(n, k):
    vis, valid, _ = oracle.mask_build(oracle.la_prefill_vparent(n, k)[None])
    assert valid.all()
    assert np.array_equal(vis[0], oracle.la_prefill_mask(n, k))
