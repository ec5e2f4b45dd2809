"""Pins of the soft-matching oracle ("Speculative Streaming", verification
step with soft matching: accept a drafted token with probability
min(1, p_target / p_draft), the rejection sampling of Leviathan et al.;
one correction token sampled at the rejection point).

* Leviathan et al.'s theorem: one drafted token x ~ q, accepted with
  probability min(1, p(x)/q(x)), else replaced by a draw from the
  normalised residual max(0, p - q) -- the output token is distributed
  exactly as p.  Integrated over fine grids of the two uniforms, the oracle
  must reproduce p.
* Hand-worked trees (sibling order, certain acceptance, residual draw).
* Temperature: the distributions are scipy's softmax of z / T.
* Greedy limit: T -> 0 with uniform drafts over the children reduces the
  walk to hard matching (the greedy tree walk) and the residual draw to
  the target's argmax.
"""

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from self_speculative_verification_gb300 import workloads as W


def _grid(M):
    return (np.arange(M) + 0.5) / M


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_single_draft_output_is_target_distribution(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    V = 6
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    M = 4000
    grid = _grid(M)
    # residual draw distribution over the u grid
    res = np.zeros(V)
    for u in grid:
        res[oracle.residual_sample(p, q, u)] += 1.0 / M
    out = np.zeros(V)
    parent = np.array([-1, 0])
    for x in range(V):
        toks = np.array([0, x])
        acc = 0.0
        for u in grid:
            path = oracle.accept_soft_tree(toks, parent, 2, lambda c: p, lambda c: q,
                                           np.array([0.0, u]))
            acc += (len(path) == 2) / M
        out[x] += q[x] * acc
        out += q[x] * (1.0 - acc) * res
    np.testing.assert_allclose(out, p, atol=3.0 / M)
    # the residual alone is max(0, p - q) normalised
    r = np.maximum(0.0, p - q)
    np.testing.assert_allclose(res, r / r.sum(), atol=2.0 / M)


def test_hand_worked_tree():
    # root 0: children 1 (token 2) and 2 (token 3); node 1: child 3 (token 1)
    parent = np.array([-1, 0, 0, 1])
    toks = np.array([0, 2, 3, 1])
    p = {0: np.array([0.1, 0.2, 0.3, 0.4]), 1: np.array([0.5, 0.1, 0.2, 0.2]),
         2: np.array([0.25, 0.25, 0.25, 0.25]), 3: np.array([0.7, 0.1, 0.1, 0.1])}
    q = {0: np.array([0.25, 0.25, 0.25, 0.25]), 1: np.array([0.1, 0.6, 0.2, 0.1]),
         2: None, 3: None}
    # node 1: p/q = 1.2 -> accepted whatever u; node 3: p/q = 1/6 < u = 0.5
    u = np.array([0.0, 0.99, 0.0, 0.5])
    path = oracle.accept_soft_tree(toks, parent, 4, p.get, q.get, u)
    assert path == [0, 1]
    # residual at node 1: max(0, p - q) = [.4, 0, 0, .1]; u * 0.5 = 0.45 -> 3
    assert oracle.residual_sample(p[1], q[1], 0.9) == 3
    assert oracle.residual_sample(p[1], q[1], 0.5) == 0          # 0.25 < 0.4
    assert oracle.residual_sample(p[1], q[1], 0.79) == 0         # 0.395 < 0.4
    assert oracle.residual_sample(p[1], q[1], 0.81) == 3         # 0.405 > 0.4
    # node 3 accepted when u < 1/6
    u2 = u.copy()
    u2[3] = 0.1
    assert oracle.accept_soft_tree(toks, parent, 4, p.get, q.get, u2) == [0, 1, 3]
    # sibling order: node 1 rejected (p/q = 0.3/0.5 < u), node 2 tried next
    q0 = np.array([0.1, 0.1, 0.5, 0.3])
    u3 = np.array([0.0, 0.7, 0.9, 0.0])
    # node 2: token 3, p/q = 0.4/0.3 > 1 -> accepted
    path = oracle.accept_soft_tree(toks, parent, 4, p.get, lambda c: q0 if c == 0 else q[c], u3)
    assert path == [0, 2]
    # node 2 has no drafted children: the bonus token is drawn from p(2)
    assert oracle.residual_sample(p[2], None, 0.6) == 2
    # nothing accepted: stop at the root
    u4 = np.array([0.0, 0.7, 0.0, 0.0])
    q_hi = np.array([0.1, 0.1, 0.5, 0.9])      # node 2: 0.4/0.9 < 0.5
    u4[2] = 0.5
    assert oracle.accept_soft_tree(toks, parent, 4, p.get, lambda c: q_hi, u4) == [0]


def test_residual_without_mass_falls_back_to_p():
    p = np.array([0.2, 0.3, 0.5])
    assert oracle.residual_sample(p, p.copy(), 0.1) == 0
    assert oracle.residual_sample(p, p.copy(), 0.6) == 2


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_temperature_softmax(T):
    rng = np.random.Generator(np.random.PCG64(5))
    z = rng.standard_normal(50) * 3
    np.testing.assert_allclose(oracle.softmax_t(z, T), softmax(z / T), rtol=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_greedy_limit_is_hard_matching(seed):
    """T -> 0, drafts uniform over each node's children: soft == greedy walk."""
    rng = np.random.Generator(np.random.PCG64(seed))
    T, V = 12, 40
    par, _ = W.random_tree(rng, T, 4, 3)
    toks = np.array([0] + [int(t) for t in rng.integers(0, V, T - 1)])
    # distinct sibling tokens
    for c in range(1, T):
        sib = [int(toks[s]) for s in range(1, c) if par[s] == par[c]]
        while int(toks[c]) in sib:
            toks[c] = (int(toks[c]) + 1) % V
    # target rows: argmax planted on a child's token half the time
    z = rng.standard_normal((T, V))
    for c in range(T):
        kids = [k for k in range(T) if par[k] == c]
        if kids and rng.random() < 0.7:
            z[c, toks[kids[int(rng.integers(len(kids)))]]] += 6.0
        else:
            z[c, int(rng.integers(V))] += 6.0
    q = np.zeros((T, V))
    for c in range(T):
        kids = [k for k in range(T) if par[k] == c]
        for k in kids:
            q[c, toks[k]] = 1.0 / len(kids)
    u = rng.uniform(0.05, 0.95, T)
    tiny = 1e-3
    path = oracle.accept_soft_tree(toks, par, T, lambda c: oracle.softmax_t(z[c], tiny),
                                   lambda c: q[c] if q[c].any() else None, u)
    g_path, g_next = oracle.accept_greedy_tree(toks, par, T, [int(np.argmax(z[c])) for c in range(T)])
    assert path == g_path
    c = path[-1]
    nxt = oracle.residual_sample(oracle.softmax_t(z[c], tiny), q[c] if q[c].any() else None, 0.5)
    assert nxt == g_next


@pytest.mark.parametrize("seed", [0, 1])
def test_planted_soft_walk(seed):
    """The generator plants each soft decision with a wide margin; the
    oracle's walk must follow the planted path exactly."""
    wl = W.make_workload("ss_soft", seed, B=6, V=3000)
    acc, paths, nxt, last = oracle.accept_soft(
        wl.logits, wl.draft_logits, wl.tokens, wl.tree_parent, None, wl.child_draft_row,
        wl.n_nodes, wl.u_accept, wl.u_sample, wl.temperature)
    assert acc.tolist() == wl.expect_acc_len.tolist()
    for b in range(wl.B):
        assert paths[b] == wl.expect_path[b, : acc[b]].tolist()
        assert last[b] == paths[b][-1]
        # the correction token has residual mass at the last node
        c = paths[b][-1]
        p = oracle.softmax_t(wl.logits[b, c], wl.temperature)
        dr = int(wl.child_draft_row[b, c])
        r = p if dr < 0 else np.maximum(0, p - oracle.softmax_t(wl.draft_logits[b, dr]))
        assert r[nxt[b]] > 0
