"""Pins of the oracle's mask construction against what the pages fix.

* the LA diagram ("Lookahead Attention", sec. 2.1) read as printed,
* the LA block formula's invariants (sec. 3.1),
* closed-form tree sizes and ancestor counts ("Speculative Streaming",
  tree draft construction and the batching formula (1+gamma)(1+sum k^g)),
* ConFu's 2T-row verify layout and soft-prompt visibility (key design 1).
"""

import numpy as np
import pytest

import oracle
from self_speculative_verification_gb300 import workloads as W


def _closure_by_matrix_powers(parent):
    """Ancestor-or-self relation via boolean powers of the parent matrix.

    A different formulation from the oracle's parent-chain walk:
    reach = I + A + A^2 + ... with A[i][p] = 1 iff p is i's parent.
    """
    n = len(parent)
    A = np.zeros((n, n), dtype=np.int64)
    for i, p in enumerate(parent):
        if p >= 0:
            A[i, p] = 1
    reach = np.eye(n, dtype=np.int64)
    P = np.eye(n, dtype=np.int64)
    for _ in range(n):
        P = (P @ A > 0).astype(np.int64)
        reach = ((reach + P) > 0).astype(np.int64)
    return reach.astype(bool)


def test_la_golden_diagram(golden_matrix):
    printed = np.array(golden_matrix("la_mask_7x7.txt"), dtype=bool)
    assert printed.shape == (7, 7)
    n, k = 4, 3
    query_major = printed.T            # the page prints rows = keys
    m = oracle.la_prefill_mask(n, k)
    # every block except the garbled top-left one matches as printed
    assert np.array_equal(m[:n, n:], query_major[:n, n:])
    assert np.array_equal(m[n:, :n], query_major[n:, :n])
    assert np.array_equal(m[n:, n:], query_major[n:, n:])
    # top-left is the standard causal mask named in sec. 3.1
    assert np.array_equal(m[:n, :n], np.tril(np.ones((n, n), dtype=bool)))
    # the printed identity is contained in it (the diagonal survives)
    assert np.all(m[:n, :n][query_major[:n, :n]])


def test_la_prefill_invariants():
    for n, k in [(1, 1), (4, 3), (9, 8), (16, 2)]:
        m = oracle.la_prefill_mask(n, k)
        assert not m[:n, n:].any()          # originals never see lookahead
        assert m[n:, :n].all()              # lookahead sees every original
        assert np.array_equal(m[n:, n:], np.eye(k, dtype=bool))


def test_la_verify_rows_equal_prefill_lookahead_rows():
    """Block rows with vparent=-1 are exactly the lookahead rows of M_LA."""
    for k in (1, 2, 4, 8):
        vis, valid, soft = oracle.mask_build(np.full((1, k), -1))
        assert valid.all() and not soft.any()
        full = oracle.la_prefill_mask(5, k)
        assert np.array_equal(vis[0], full[5:, 5:])


def test_padding_rows():
    vp = np.array([[-1, -1, -2, -2]])
    vis, valid, soft = oracle.mask_build(vp, np.array([[1, 0, 1, 0]]))
    assert valid.tolist() == [[True, True, False, False]]
    assert not vis[0, 2:].any() and not vis[0, :, 2:].any()
    assert soft.tolist() == [[True, False, False, False]]


def test_chain_is_lower_triangular():
    for R in (1, 2, 7, 33, 70):
        vp = np.arange(-1, R - 1)[None, :]
        vis, valid, _ = oracle.mask_build(vp)
        assert np.array_equal(vis[0], np.tril(np.ones((R, R), dtype=bool)))


@pytest.mark.parametrize("k,gamma,size", [(2, 3, 15), (3, 3, 40), (1, 4, 5),
                                          (4, 2, 21)])
def test_full_tree_sizes_and_ancestors(k, gamma, size):
    parent, depth = W.full_tree(k, gamma)
    assert len(parent) == size == 1 + sum(k ** g for g in range(1, gamma + 1))
    vis, valid, _ = oracle.mask_build(np.where(parent < 0, -1, parent)[None])
    # a node at depth g sees exactly g ancestors and itself
    assert np.array_equal(vis[0].sum(axis=1), depth + 1)
    assert vis[0].sum() == sum(k ** g * (g + 1) for g in range(gamma + 1))
    assert np.array_equal(vis[0], _closure_by_matrix_powers(parent))


@pytest.mark.parametrize("k,gamma", [(2, 3), (3, 3), (1, 4)])
def test_stream_batch_rows(k, gamma):
    parent, _ = W.full_tree(k, gamma)
    vp, soft = W.tree_block_rows("ss", parent, gamma)
    T = len(parent)
    assert len(vp) == (1 + gamma) * (1 + sum(k ** g for g in range(1, gamma + 1)))
    vis, valid, sees = oracle.mask_build(vp[None], soft[None])
    anc = _closure_by_matrix_powers(parent)
    assert valid.all() and not sees.any()
    for j in range(T):
        node_cols = set(np.nonzero(anc[j])[0])
        for s in range(1, gamma + 1):
            r = T + j * gamma + (s - 1)
            streams = {T + j * gamma + (t - 1) for t in range(1, s + 1)}
            assert set(np.nonzero(vis[0, r])[0]) == node_cols | streams


def test_confu_rows_and_soft_prompt():
    rng = np.random.Generator(np.random.PCG64(3))
    for T in (1, 5, 30, 60):
        parent, _ = W.random_tree(rng, T, 8, 4)
        vp, soft = W.tree_block_rows("confu", parent)
        assert len(vp) == 2 * T
        vis, valid, sees = oracle.mask_build(vp[None], soft[None])
        anc = _closure_by_matrix_powers(parent)
        # nodes see ancestors + self, never contemplate columns nor soft
        assert np.array_equal(vis[0, :T, :T], anc)
        assert not vis[0, :T, T:].any()
        assert not sees[0, :T].any()
        # contemplate j sees node j's ancestors, node j, itself, the soft prompt
        for j in range(T):
            expect = set(np.nonzero(anc[j])[0]) | {T + j}
            assert set(np.nonzero(vis[0, T + j])[0]) == expect
        assert sees[0, T:].all()


def test_random_trees_match_matrix_closure():
    rng = np.random.Generator(np.random.PCG64(11))
    for _ in range(20):
        T = int(rng.integers(1, 70))
        parent, depth = W.random_tree(rng, T, 8, 4)
        vis, _, _ = oracle.mask_build(np.where(parent < 0, -1, parent)[None])
        assert np.array_equal(vis[0], _closure_by_matrix_powers(parent))
        assert np.array_equal(vis[0].sum(1), depth + 1)


@pytest.mark.parametrize("vp", [[[-1, 1]], [[0]], [[-1, -3]], [[-2, 0]], [[-1, 5, -1]]])
def test_bad_parents_rejected(vp):
    with pytest.raises(ValueError):
        oracle.mask_build(np.array(vp))
