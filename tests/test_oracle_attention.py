"""Pins of the oracle's masked verify attention.

Each pin ties the oracle to something other than itself:

* a chain mask is standard causal attention over the concatenated sequence
  ("Speculative Streaming", Eq. 1) -- checked against
  ``torch.nn.functional.scaled_dot_product_attention(is_causal=True)``;
* an LA lookahead row is plain attention over the prefix plus its own K/V
  ("Lookahead Attention", sec. 3.1) -- checked against unmasked SDPA;
* closed forms: one visible key -> O = v, LSE = s; n equal keys ->
  O = mean(v), LSE = s + ln n;
* brute force with scalar Python loops on tiny inputs;
* GQA head mapping against MHA with repeated K/V;
* soft-prompt and block-column visibility by perturbation ("ConFu" key
  design 1: only contemplate tokens see the soft prompt).
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from self_speculative_verification_gb300 import workloads as W


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _sdpa(q, k, v, causal=False):
    """Library attention in float64: q [L][d], k/v [S][d] -> [L][d]."""
    qt = torch.from_numpy(np.asarray(q, np.float64))[None, None]
    kt = torch.from_numpy(np.asarray(k, np.float64))[None, None]
    vt = torch.from_numpy(np.asarray(v, np.float64))[None, None]
    return F.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)[0, 0].numpy()


def _run(q, pk, pv, kb, vb, vparent, soft_flags=None, sk=None, sv=None, scale=None):
    vis, valid, sees = oracle.mask_build(vparent, soft_flags)
    return oracle.verify_attention(q, pk, pv, kb, vb, vis, valid, sees,
                                   soft_k=sk, soft_v=sv, scale=scale)


def test_chain_equals_causal_attention():
    rng = _rng(1)
    S, R, d = 7, 5, 16
    x_q = rng.standard_normal((S + R, d))
    x_k = rng.standard_normal((S + R, d))
    x_v = rng.standard_normal((S + R, d))
    q = x_q[S:][None, :, None, :]
    pk = [x_k[:S][None]]
    pv = [x_v[:S][None]]
    kb = x_k[S:][None, None]
    vb = x_v[S:][None, None]
    vp = np.arange(-1, R - 1)[None]
    O, LSE = _run(q, pk, pv, kb, vb, vp)
    ref = _sdpa(x_q, x_k, x_v, causal=True)[S:]
    np.testing.assert_allclose(O[0, :, 0], ref, rtol=1e-12, atol=1e-12)


def test_la_row_equals_attention_over_prefix_and_self():
    rng = _rng(2)
    S, k, d = 11, 4, 8
    pk = rng.standard_normal((1, S, d))
    pv = rng.standard_normal((1, S, d))
    kb = rng.standard_normal((1, 1, k, d))
    vb = rng.standard_normal((1, 1, k, d))
    q = rng.standard_normal((1, k, 1, d))
    O, _ = _run(q, [pk], [pv], kb, vb, np.full((1, k), -1))
    for i in range(k):
        K = np.concatenate([pk[0], kb[0, 0, i:i + 1]])
        V = np.concatenate([pv[0], vb[0, 0, i:i + 1]])
        ref = _sdpa(q[0, i, 0][None], K, V)[0]
        np.testing.assert_allclose(O[0, i, 0], ref, rtol=1e-12, atol=1e-12)


def test_single_visible_key():
    rng = _rng(3)
    d = 32
    q = rng.standard_normal((1, 1, 1, d))
    kb = rng.standard_normal((1, 1, 1, d))
    vb = rng.standard_normal((1, 1, 1, d))
    empty = [np.zeros((1, 0, d))]
    O, LSE = _run(q, empty, empty, kb, vb, np.array([[-1]]))
    np.testing.assert_allclose(O[0, 0, 0], vb[0, 0, 0], rtol=1e-13)
    s = float(q[0, 0, 0] @ kb[0, 0, 0]) / math.sqrt(d)
    assert abs(LSE[0, 0, 0] - s) < 1e-12


def test_equal_keys_closed_form():
    rng = _rng(4)
    d, S = 16, 9
    key = rng.standard_normal(d)
    pk = [np.tile(key, (1, S, 1))]
    pv = [rng.standard_normal((1, S, d))]
    kb = np.tile(key, (1, 1, 1, 1))
    vb = rng.standard_normal((1, 1, 1, d))
    q = rng.standard_normal((1, 1, 1, d))
    O, LSE = _run(q, pk, pv, kb, vb, np.array([[-1]]))
    s = float(q[0, 0, 0] @ key) / math.sqrt(d)
    n = S + 1
    assert abs(LSE[0, 0, 0] - (s + math.log(n))) < 1e-12
    mean_v = (pv[0][0].sum(0) + vb[0, 0, 0]) / n
    np.testing.assert_allclose(O[0, 0, 0], mean_v, rtol=1e-12, atol=1e-13)


def test_brute_force_tiny():
    """Scalar-loop attention over an explicitly listed column set."""
    rng = _rng(5)
    B, R, Hq, Hkv, d, nsoft = 2, 5, 4, 2, 3, 2
    S = [3, 0]
    vp = np.array([[-1, 0, 1, 0, -2], [-1, -1, 1, 2, 0]])
    soft = np.array([[0, 1, 0, 1, 1], [1, 0, 0, 1, 0]], dtype=np.uint8)
    q = rng.standard_normal((B, R, Hq, d))
    pk = [rng.standard_normal((Hkv, s, d)) for s in S]
    pv = [rng.standard_normal((Hkv, s, d)) for s in S]
    kb = rng.standard_normal((B, Hkv, R, d))
    vb = rng.standard_normal((B, Hkv, R, d))
    sk = rng.standard_normal((Hkv, nsoft, d))
    sv = rng.standard_normal((Hkv, nsoft, d))
    O, LSE = _run(q, pk, pv, kb, vb, vp, soft, sk, sv)

    def visible_block(b, r):
        out = []
        c = r
        while c >= 0:
            out.append(c)
            c = int(vp[b, c])
        return out

    for b in range(B):
        for r in range(R):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                if vp[b, r] == -2:
                    assert LSE[b, h, r] == -math.inf
                    assert not O[b, r, h].any()
                    continue
                keys, vals = [], []
                for t in range(S[b]):
                    keys.append(pk[b][g, t]); vals.append(pv[b][g, t])
                if soft[b, r]:
                    for t in range(nsoft):
                        keys.append(sk[g, t]); vals.append(sv[g, t])
                for c in visible_block(b, r):
                    keys.append(kb[b, g, c]); vals.append(vb[b, g, c])
                sc = []
                for kk in keys:
                    acc = 0.0
                    for i in range(d):
                        acc += q[b, r, h, i] * kk[i]
                    sc.append(acc / math.sqrt(d))
                tot = 0.0
                for s in sc:
                    tot += math.exp(s)
                lse = math.log(tot)
                assert abs(LSE[b, h, r] - lse) < 1e-12
                for i in range(d):
                    o = 0.0
                    for s, vv in zip(sc, vals):
                        o += math.exp(s) / tot * vv[i]
                    assert abs(O[b, r, h, i] - o) < 1e-12


def test_gqa_mapping_matches_repeated_mha():
    rng = _rng(6)
    B, R, Hq, Hkv, d = 1, 3, 8, 2, 8
    G = Hq // Hkv
    q = rng.standard_normal((B, R, Hq, d))
    pk = [rng.standard_normal((Hkv, 6, d))]
    pv = [rng.standard_normal((Hkv, 6, d))]
    kb = rng.standard_normal((B, Hkv, R, d))
    vb = rng.standard_normal((B, Hkv, R, d))
    vp = np.array([[-1, 0, 0]])
    O, LSE = _run(q, pk, pv, kb, vb, vp)
    rep = lambda a, ax: np.repeat(a, G, axis=ax)
    O2, LSE2 = _run(q, [rep(pk[0], 0)], [rep(pv[0], 0)], rep(kb, 1), rep(vb, 1), vp)
    np.testing.assert_allclose(O, O2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(LSE, LSE2, rtol=1e-13)


def test_soft_prompt_only_changes_contemplate_rows():
    wl = W.make_workload("confu", 7, B=1, seq=("uniform", 20, 40), V=300, T=6)
    pk, pv = zip(*[wl.prefix_kv(b) for b in range(wl.B)])
    vis, valid, sees = oracle.mask_build(wl.vparent, wl.soft_flags)
    args = (wl.q, pk, pv, wl.kb, wl.vb, vis, valid, sees)
    O1, L1 = oracle.verify_attention(*args, soft_k=wl.soft_k, soft_v=wl.soft_v)
    O2, L2 = oracle.verify_attention(*args, soft_k=wl.soft_k * 3 + 0.1,
                                     soft_v=wl.soft_v - 0.5)
    changed = np.abs(O1 - O2).max(axis=(2, 3)) > 0
    assert np.array_equal(changed[0], sees[0])
    # a contemplate row equals SDPA over prefix || soft || its visible block
    T = 6
    r = T + 3
    h = 5
    g = h // wl.G
    cols = np.nonzero(vis[0, r])[0]
    K = np.concatenate([pk[0][g], wl.soft_k[g], wl.kb[0, g, cols]])
    V = np.concatenate([pv[0][g], wl.soft_v[g], wl.vb[0, g, cols]])
    ref = _sdpa(wl.q[0, r, h].astype(np.float64)[None], K, V)[0]
    np.testing.assert_allclose(O1[0, r, h], ref, rtol=1e-10, atol=1e-12)


def test_block_column_perturbation_hits_exactly_its_viewers():
    wl = W.make_workload("ss", 8, B=1, seq=("uniform", 10, 20), V=300)
    pk, pv = zip(*[wl.prefix_kv(b) for b in range(wl.B)])
    vis, valid, sees = oracle.mask_build(wl.vparent, wl.soft_flags)
    base, _ = oracle.verify_attention(wl.q, pk, pv, wl.kb, wl.vb, vis, valid, sees)
    for c in (0, 3, wl.R - 1):
        vb2 = wl.vb.copy()
        vb2[0, :, c] += 1.0
        O2, _ = oracle.verify_attention(wl.q, pk, pv, wl.kb, vb2, vis, valid, sees)
        changed = np.abs(O2 - base).max(axis=(2, 3))[0] > 0
        assert np.array_equal(changed, vis[0, :, c])


def test_paged_gather_roundtrip():
    wl = W.make_workload("long_paged", 9, B=3, seq=("uniform", 17, 70), V=100)
    Kp, Vp = wl.paged_cache()
    got = oracle.gather_paged(Kp, wl.page_table, wl.seq_len, wl.page_size)
    for b in range(wl.B):
        k, _ = wl.prefix_kv(b)
        assert np.array_equal(got[b], k)


@pytest.mark.parametrize("scale", [None, 0.3])
def test_scale_argument(scale):
    rng = _rng(10)
    d = 4
    q = rng.standard_normal((1, 2, 1, d))
    kb = rng.standard_normal((1, 1, 2, d))
    vb = rng.standard_normal((1, 1, 2, d))
    empty = [np.zeros((1, 0, d))]
    O, LSE = _run(q, empty, empty, kb, vb, np.array([[-1, 0]]), scale=scale)
    sc = 1 / math.sqrt(d) if scale is None else scale
    s = np.array([q[0, 0, 0] @ kb[0, 0, 0]]) * sc
    assert abs(LSE[0, 0, 0] - s[0]) < 1e-12
