"""Pins of the oracle's vocab reduce, acceptance and KV commit.

* vocab reduce against ``numpy.argmax`` and ``scipy.special.logsumexp``;
* acceptance against the generator's planted outcomes (the generator plants
  argmax tokens / proposal probabilities and records the path it intends,
  without any of the oracle's code) and hand-worked cases: LA threshold
  longest prefix ("Lookahead Attention", sec. 2.4) and the SS greedy walk
  with beta accepted + 1 correction token ("Speculative Streaming",
  verification step);
* commit: only the new slots change, byte for byte (LA sec. 3.2: the other
  speculative K/V is discarded), and a hand-worked paged allocation.
"""

import math

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from self_speculative_verification_gb300 import workloads as W


def test_vocab_reduce_against_library():
    rng = np.random.Generator(np.random.PCG64(0))
    z = rng.standard_normal((6, 1000)) * 3
    z[2, 17] = z[2, 900] = z[2].max() + 1.0      # tie: lowest index wins
    prop = rng.integers(0, 1000, size=6)
    am, lse, zp = oracle.vocab_reduce(z, prop)
    assert am.tolist() == np.argmax(z, axis=1).tolist()
    assert am[2] == 17
    np.testing.assert_allclose(lse, logsumexp(z, axis=1), rtol=1e-14)
    np.testing.assert_array_equal(zp, z[np.arange(6), prop])


def test_threshold_hand_worked():
    # probabilities of the proposals: 0.5, 0.31, 0.29 -> L = 2 at tau = 0.3
    probs = [0.5, 0.31, 0.29, 0.9]
    zprop = [math.log(p) for p in probs]
    lse = [0.0] * 4
    assert oracle.accept_threshold_chain(zprop, lse, 4, 0.3) == 2
    assert oracle.accept_threshold_chain(zprop, lse, 1, 0.3) == 1
    assert oracle.accept_threshold_chain(zprop, lse, 0, 0.3) == 0
    assert oracle.accept_threshold_chain([math.log(0.3)], [0.0], 1, 0.3) == 1


def test_greedy_walk_hand_worked():
    #        0(t=5)
    #       /      \
    #   1(t=7)    2(t=9)
    #    |    \
    #  3(t=1) 4(t=2)
    parent = [-1, 0, 0, 1, 1]
    tokens = [5, 7, 9, 1, 2]
    # target greedy tokens per node: root->9, node2->4 (no child) => path 0,2
    path, nxt = oracle.accept_greedy_tree(tokens, parent, 5, [9, 0, 4, 0, 0])
    assert path == [0, 2] and nxt == 4
    # root->7, node1->2, node4->8 => path 0,1,4, correction 8, beta = 2
    path, nxt = oracle.accept_greedy_tree(tokens, parent, 5, [7, 2, 0, 0, 8])
    assert path == [0, 1, 4] and nxt == 8
    assert len(path) - 1 + 1 == 3     # tokens advanced = beta + 1
    # the wanted token sits on a non-child (node 2): the walk stops at node 1
    path, nxt = oracle.accept_greedy_tree(tokens, parent, 5, [7, 9, 0, 0, 0])
    assert path == [0, 1] and nxt == 9
    # nothing matches: only the root, correction = greedy token at the root
    path, nxt = oracle.accept_greedy_tree(tokens, parent, 5, [3, 0, 0, 0, 0])
    assert path == [0] and nxt == 3
    # duplicate sibling tokens: lowest node index wins
    path, _ = oracle.accept_greedy_tree([5, 7, 7], [-1, 0, 0], 3, [7, 1, 1])
    assert path == [0, 1]


@pytest.mark.parametrize("name,kw", [
    ("tiny_la", {}),
    ("la7b", dict(B=6, seq=("uniform", 10, 20), V=4000)),
    ("confu", dict(B=4, seq=("uniform", 10, 20), V=3000)),
    ("ss", dict(B=6, seq=("uniform", 10, 20), V=3000)),
    ("long_paged", dict(B=6, seq=("uniform", 10, 20), V=4000)),
])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_planted_acceptance(name, kw, seed):
    wl = W.make_workload(name, seed, **kw)
    B = wl.B
    logits = wl.logits.reshape(B * wl.Rj, wl.V)
    prop = wl.tokens.reshape(-1) if wl.mode == "la" else None
    am, lse, zp = oracle.vocab_reduce(logits, prop)
    am, lse, zp = (a.reshape(B, wl.Rj) for a in (am, lse, zp))
    mode = oracle.MODE_THRESH_CHAIN if wl.mode == "la" else oracle.MODE_GREEDY_TREE
    acc, paths, nxt, last = oracle.accept(mode, wl.tau, wl.tokens,
                                          wl.tree_parent, wl.n_nodes, am, lse, zp)
    assert acc.tolist() == wl.expect_acc_len.tolist()
    for b in range(B):
        assert paths[b] == [int(x) for x in wl.expect_path[b, : acc[b]]]
    if wl.mode == "la":
        # planted probabilities stay well away from tau after rounding
        p = np.exp(zp - lse)
        for b in range(B):
            for i in range(int(wl.n_nodes[b])):
                assert p[b, i] > wl.tau + 0.05 or p[b, i] < wl.tau - 0.05
    else:
        # the greedy margin survives storage rounding (no ties)
        z = wl.logits.astype(np.float64)
        top2 = np.sort(z, axis=2)[:, :, -2:]
        assert (top2[:, :, 1] - top2[:, :, 0]).min() >= W.GREEDY_MARGIN - 0.125


def _rand_block(rng, B, Hkv, R, d):
    return rng.standard_normal((B, Hkv, R, d)), rng.standard_normal((B, Hkv, R, d))


def test_commit_contiguous_only_new_slots_change():
    rng = np.random.Generator(np.random.PCG64(1))
    B, Hkv, Smax, R, d = 3, 2, 12, 4, 5
    K = rng.standard_normal((B, Hkv, Smax, d))
    V = rng.standard_normal((B, Hkv, Smax, d))
    seq = np.array([3, 8, 0])
    kb, vb = _rand_block(rng, B, Hkv, R, d)
    paths = [[0, 2, 3], [], [1]]
    K2, V2, seq2 = oracle.kv_commit_contiguous(K, V, seq, kb, vb, paths)
    assert seq2.tolist() == [6, 8, 1]
    changed = np.zeros((B, Smax), dtype=bool)
    changed[0, 3:6] = True
    changed[2, 0] = True
    diff = (K2 != K).any(axis=(1, 3)) | (V2 != V).any(axis=(1, 3))
    assert np.array_equal(diff, changed)
    assert np.array_equal(K2[0, :, 3:6], kb[0][:, [0, 2, 3]])
    assert np.array_equal(V2[2, :, 0], vb[2, :, 1])
    with pytest.raises(OverflowError):
        oracle.kv_commit_contiguous(K, V, np.array([10, 0, 0]), kb, vb,
                                    [[0, 1, 2], [], []])


def test_commit_paged_hand_worked():
    """page_size 4; S = [5, 8]; accept 3 and 2 rows; free list [9, 7, 3].

    Request 0 fills slots 1..3 of its second page (no new page).  Request 1
    is page aligned: position 8 opens a fresh page, the first free one (9),
    position 9 goes to slot 1 of page 9.  free_head ends at 1.
    """
    rng = np.random.Generator(np.random.PCG64(2))
    P, Hkv, ps, d = 10, 1, 4, 2
    Kp = rng.standard_normal((P, Hkv, 1, ps, d))      # one block of d elements
    Vp = rng.standard_normal((P, Hkv, 1, ps, d))
    pt = np.array([[4, 0, -1], [6, 1, -1]])
    kb, vb = _rand_block(rng, 2, Hkv, 3, d)
    out = oracle.kv_commit_paged(Kp, Vp, pt, [5, 8], np.array([9, 7, 3]), 0,
                                 kb, vb, [[0, 1, 2], [2, 0]], ps)
    K2, V2, pt2, seq2, head = out
    assert seq2.tolist() == [8, 10] and head == 1
    assert pt2.tolist() == [[4, 0, -1], [6, 1, 9]]
    assert np.array_equal(K2[0, 0, 0, 1:4], kb[0, 0, [0, 1, 2]])
    assert np.array_equal(K2[9, 0, 0, 0:2], kb[1, 0, [2, 0]])
    assert np.array_equal(V2[9, 0, 0, 0:2], vb[1, 0, [2, 0]])
    touched = np.zeros((P, ps), dtype=bool)
    touched[0, 1:4] = True
    touched[9, 0:2] = True
    diff = (K2 != Kp).any(axis=(1, 2, 4)) | (V2 != Vp).any(axis=(1, 2, 4))
    assert np.array_equal(diff, touched)


def test_commit_paged_exhaustion():
    Kp = np.zeros((3, 1, 1, 2, 1))
    kb = np.zeros((1, 1, 3, 1))
    with pytest.raises(OverflowError):
        oracle.kv_commit_paged(Kp, Kp, np.array([[0, -1, -1]]), [2],
                               np.array([], dtype=np.int64), 0, kb, kb,
                               [[0]], 2)


def test_commit_empty_paths_change_nothing():
    wl = W.make_workload("long_paged", 3, B=4, seq=("uniform", 30, 60), V=100)
    Kp, Vp = wl.paged_cache(fill=0.0)
    paths = [[] for _ in range(wl.B)]
    K2, V2, pt2, seq2, head = oracle.kv_commit_paged(
        Kp, Vp, wl.page_table, wl.seq_len, wl.free_pages, 0, wl.kb, wl.vb,
        paths, wl.page_size)
    assert np.array_equal(K2, Kp) and np.array_equal(V2, Vp)
    assert np.array_equal(pt2, wl.page_table) and head == 0
