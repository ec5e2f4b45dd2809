"""The oracle's pins are sensitive: plausible mistakes planted in the oracle
(on the CPU, by monkeypatching) make at least one pin fail."""

import math
import types

import numpy as np
import pytest

import oracle
import oracle.specverify_oracle as so
import test_oracle_accept_commit as tac
import test_oracle_attention as tat
import test_oracle_mask as tm


def _expect_pin_failure(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_wrong_softmax_scale_is_caught(monkeypatch):
    fake = types.SimpleNamespace(sqrt=lambda x: x, log=math.log, exp=math.exp,
                                 inf=math.inf)
    monkeypatch.setattr(so, "math", fake)       # scale becomes 1/d
    _expect_pin_failure(tat.test_chain_equals_causal_attention)
    _expect_pin_failure(tat.test_single_visible_key)


def test_dropped_self_visibility_is_caught(monkeypatch):
    real = so.mask_build

    def no_self(vparent, soft_flags=None):
        vis, valid, sees = real(vparent, soft_flags)
        vis = vis.copy()
        for b in range(vis.shape[0]):
            np.fill_diagonal(vis[b], False)
        return vis, valid, sees

    monkeypatch.setattr(oracle, "mask_build", no_self)
    _expect_pin_failure(tm.test_la_verify_rows_equal_prefill_lookahead_rows)
    _expect_pin_failure(tm.test_chain_is_lower_triangular)


def test_parent_only_visibility_is_caught(monkeypatch):
    """SS Eq. 4 read literally (immediate parent only) fails the pins."""
    def parent_only(vparent, soft_flags=None):
        vparent = np.asarray(vparent)
        B, R = vparent.shape
        vis = np.zeros((B, R, R), dtype=bool)
        valid = vparent != so.VP_PAD
        for b in range(B):
            for r in range(R):
                if valid[b, r]:
                    vis[b, r, r] = True
                    if vparent[b, r] >= 0:
                        vis[b, r, vparent[b, r]] = True
        sees = np.zeros((B, R), dtype=bool) if soft_flags is None else \
            (np.asarray(soft_flags) != 0) & valid
        return vis, valid, sees

    monkeypatch.setattr(oracle, "mask_build", parent_only)
    _expect_pin_failure(tm.test_full_tree_sizes_and_ancestors, 2, 3, 15)
    _expect_pin_failure(tat.test_chain_equals_causal_attention)


def test_strict_threshold_is_caught(monkeypatch):
    def strict(zprop, lse, n, tau):
        L = 0
        while L < n and math.exp(zprop[L] - lse[L]) > tau + 1e-12:
            L += 1
        return L
    monkeypatch.setattr(oracle, "accept_threshold_chain", strict)
    _expect_pin_failure(tac.test_threshold_hand_worked)


def test_walk_without_root_check_is_caught(monkeypatch):
    """A walk that matches any node's token (not only the children of the
    current node) fails the hand-worked tree pin."""
    def sloppy(tokens, tree_parent, n_nodes, argmax_of_node):
        cur, path = 0, [0]
        while True:
            want = int(argmax_of_node[cur])
            nxt = next((c for c in range(1, n_nodes)
                        if int(tokens[c]) == want and c not in path), None)
            if nxt is None:
                return path, want
            cur = nxt
            path.append(cur)
    monkeypatch.setattr(oracle, "accept_greedy_tree", sloppy)
    _expect_pin_failure(tac.test_greedy_walk_hand_worked)


# ---------------------------------------------------------------- soft matching

import test_oracle_soft as tos


def test_inverted_acceptance_ratio_is_caught(monkeypatch):
    def inverted(tokens, tree_parent, n_nodes, p_of, q_of, u_accept):
        swapped = lambda c: q_of(c)
        return so.accept_soft_tree(tokens, tree_parent, n_nodes, swapped,
                                   lambda c: p_of(c), u_accept)

    monkeypatch.setattr(oracle, "accept_soft_tree", inverted)
    _expect_pin_failure(tos.test_single_draft_output_is_target_distribution, 0)
    _expect_pin_failure(tos.test_hand_worked_tree)


def test_residual_without_draft_subtraction_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "residual_sample",
                        lambda p, q, u: so.residual_sample(p, None, u))
    _expect_pin_failure(tos.test_single_draft_output_is_target_distribution, 1)


def test_residual_sign_flip_is_caught(monkeypatch):
    def flipped(p, q, u):
        if q is None:
            return so.residual_sample(p, None, u)
        return so.residual_sample(q, p, u)

    monkeypatch.setattr(oracle, "residual_sample", flipped)
    _expect_pin_failure(tos.test_single_draft_output_is_target_distribution, 2)
    _expect_pin_failure(tos.test_hand_worked_tree)


# ------------------------------------------------------------ draft trees

import test_oracle_draft as tod


def test_prune_without_parent_closure_is_caught(monkeypatch):
    def no_closure(tokens, parent, early_logits, threshold):
        n = len(tokens)
        keep = np.full(n, -1, dtype=np.int64)
        nt, npar = [], []
        for c in range(n):
            ok = c == 0 or so.softmax_t(early_logits[int(parent[c])])[int(tokens[c])] >= threshold
            if ok:
                keep[c] = len(nt)
                nt.append(int(tokens[c]))
                npar.append(-1 if c == 0 else int(keep[int(parent[c])]))
        return np.array(nt), np.array(npar), keep

    monkeypatch.setattr(oracle, "prune_tree", no_closure)
    _expect_pin_failure(tod.test_prune_hand_worked)


def test_topk_ties_to_higher_id_is_caught(monkeypatch):
    def high_ties(z, k):
        z = np.asarray(z, dtype=np.float64)
        order = np.lexsort((-np.arange(len(z)), -z))
        return order[:k]

    monkeypatch.setattr(oracle, "topk_tokens", high_ties)
    _expect_pin_failure(tod.test_topk_brute_force, 0, 3)


# ------------------------------------------------------ stream value rotation

import test_oracle_stream_ops as tso


def test_rotation_sign_flip_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "rotate_stream_values",
                        lambda vb, n, g, eps: so.rotate_stream_values(vb, n, g, -eps))
    _expect_pin_failure(tso.test_rotation_is_complex_multiplication)


def test_rotation_by_node_index_is_caught(monkeypatch):
    """Rotating by eps * (node index) instead of eps * (stream index)."""
    def by_node(vb, n_nodes, gamma, eps):
        out = np.array(vb, dtype=np.float64, copy=True)
        for b in range(out.shape[0]):
            T = int(n_nodes[b])
            for j in range(T):
                for s in range(1, gamma + 1):
                    r = T + j * gamma + (s - 1)
                    c, sn = math.cos(eps * (j + 1)), math.sin(eps * (j + 1))
                    re, im = out[b, :, j, 0::2], out[b, :, j, 1::2]
                    out[b, :, r, 0::2] = re * c - im * sn
                    out[b, :, r, 1::2] = re * sn + im * c
        return out

    monkeypatch.setattr(oracle, "rotate_stream_values", by_node)
    _expect_pin_failure(tso.test_rotation_is_complex_multiplication)
