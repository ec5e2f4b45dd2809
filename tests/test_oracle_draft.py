"""Pins of the draft-tree oracle ("Speculative Streaming": tree draft
construction, parallel tree pruning, batching with streams).

* top-k against a brute-force sort (ties to the lower id);
* the tree's size 1 + sum_g k^g, k children per inner node, the tokens of
  each level equal to the stream's top-k in order, and the same shape as
  the generator's independent complete-tree builder;
* the SS block's parent pointers give, through mask_build, exactly the
  visibility of Eq. 2 and Eq. 4 (ancestors walked independently), and
  match the generator's block layout;
* pruning: a hand-worked case, closure under parents, the threshold
  limits (0 keeps all, above 1 keeps only the root).
"""

import numpy as np
import pytest

import oracle
from self_speculative_verification_gb300 import workloads as W


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("k", [1, 3, 8])
def test_topk_brute_force(seed, k):
    rng = np.random.Generator(np.random.PCG64(seed))
    z = rng.integers(-5, 5, 300).astype(np.float64)      # many ties
    want = sorted(range(len(z)), key=lambda v: (-z[v], v))[:k]
    assert oracle.topk_tokens(z, k).tolist() == want


@pytest.mark.parametrize("k,gamma", [(1, 3), (2, 3), (4, 3), (3, 4)])
def test_draft_tree_shape(k, gamma):
    rng = np.random.Generator(np.random.PCG64(k * 10 + gamma))
    V = 200
    z = rng.integers(-3, 3, (gamma, V)).astype(np.float64)
    tok, par, dep = oracle.draft_tree(z, k, root_token=17)
    n = 1 + sum(k ** g for g in range(1, gamma + 1))
    assert len(tok) == n and tok[0] == 17 and par[0] == -1
    for g in range(gamma + 1):
        assert int((dep == g).sum()) == k ** g
    ref_par, ref_dep = W.full_tree(k, gamma)
    assert np.array_equal(par, ref_par) and np.array_equal(dep, ref_dep)
    for p in range(n):
        kids = np.nonzero(par == p)[0]
        if dep[p] < gamma:
            assert len(kids) == k
            top = sorted(range(V), key=lambda v: (-z[dep[p], v], v))[:k]
            assert tok[kids].tolist() == top
        else:
            assert len(kids) == 0


def _ancestors(par, j):
    out = {j}
    while par[j] >= 0:
        j = int(par[j])
        out.add(j)
    return out


@pytest.mark.parametrize("k,gamma", [(2, 3), (3, 2)])
def test_ss_block_visibility(k, gamma):
    par, _ = W.full_tree(k, gamma)
    n = len(par)
    R = n * (1 + gamma) + 5                      # trailing padding rows
    vp = oracle.ss_block_vparent(par, gamma, R)
    vis, valid, _ = oracle.mask_build(vp[None])
    vis, valid = vis[0], valid[0]
    assert valid[: n * (1 + gamma)].all() and not valid[n * (1 + gamma):].any()
    for j in range(n):
        want = _ancestors(par, j)
        assert set(np.nonzero(vis[j])[0]) == want
        for s in range(1, gamma + 1):
            r = n + j * gamma + (s - 1)
            streams = {n + j * gamma + (t - 1) for t in range(1, s + 1)}
            assert set(np.nonzero(vis[r])[0]) == want | streams
    ref, _ = W.tree_block_rows("ss", par, gamma)
    assert np.array_equal(vp[: len(ref)], ref)


def test_prune_hand_worked():
    # root 0 -> 1 (token 5), 2 (token 6); 1 -> 3 (token 7), 4 (token 8); 2 -> 5 (token 7)
    tok = np.array([9, 5, 6, 7, 8, 7])
    par = np.array([-1, 0, 0, 1, 1, 2])
    V = 10
    big = np.full((6, V), -30.0)
    # root row: token 5 -> p ~ 0.5, token 6 -> p ~ 0.02 (pruned at 0.05)
    big[0, 5], big[0, 6], big[0, 0] = 0.0, np.log(0.04), 0.0
    # node 1 row: token 7 -> ~0.7, token 8 -> ~0.0 (pruned)
    big[1, 7], big[1, 2] = np.log(0.7), np.log(0.3)
    big[2, 7] = 0.0                                  # node 2 pruned anyway
    t2, p2, km = oracle.prune_tree(tok, par, big, 0.05)
    assert km.tolist() == [0, 1, -1, 2, -1, -1]
    assert t2.tolist() == [9, 5, 7] and p2.tolist() == [-1, 0, 1]


@pytest.mark.parametrize("seed", [0, 1])
def test_prune_closure_and_limits(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    k, gamma, V = 3, 3, 60
    tok, par, _ = oracle.draft_tree(rng.standard_normal((gamma, V)), k, 1)
    n = len(tok)
    early = rng.standard_normal((n, V)) * 2.0
    t2, p2, km = oracle.prune_tree(tok, par, early, 0.02)
    for c in range(1, n):
        if km[c] >= 0:
            assert km[par[c]] >= 0
            assert p2[km[c]] == km[par[c]]
            assert t2[km[c]] == tok[c]
            prob = oracle.softmax_t(early[par[c]])[tok[c]]
            assert prob >= 0.02
        elif km[par[c]] >= 0:
            assert oracle.softmax_t(early[par[c]])[tok[c]] < 0.02
    assert (km >= 0).sum() == len(t2)
    assert (oracle.prune_tree(tok, par, early, 0.0)[2] >= 0).all()
    assert (oracle.prune_tree(tok, par, early, 1.5)[2] >= 0).sum() == 1


@pytest.mark.parametrize("seed", [0, 1])
def test_planted_draft_workload(seed):
    """The generator plants top-k winners (with a tie) and every pruning
    decision with a margin; the oracle must recover them."""
    d = W.make_draft(seed, B=3, V=2000)
    for b in range(d.B):
        for j in range(d.gamma):
            assert oracle.topk_tokens(d.stream_logits[b, j], d.k).tolist() == \
                d.expect_top[b, j].tolist()
        tok, par, _ = oracle.draft_tree(d.stream_logits[b], d.k, d.root_token[b])
        _, _, km = oracle.prune_tree(tok, par, d.early_logits[b], d.threshold)
        assert np.array_equal(km >= 0, d.expect_keep[b])
