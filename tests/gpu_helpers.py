"""Shared helpers of the GPU parity tests: run the oracle on a workload and
compare the CUDA path's outputs with it.

Tolerances (GPU vs float64 oracle):
* bf16 attention outputs: max |O_gpu - O_ref| <= 1e-2 and
  ||O_gpu - O_ref|| / ||O_ref|| <= 1e-2; LSE relative error <= 1e-3.
* fp32 attention: max abs <= 2e-5, LSE relative <= 1e-5.
* vocab reduce: argmax exact; LSE relative <= 1e-5; proposal logit exact.
* mask, acceptance (lengths, paths, next tokens, last nodes) and the
  committed cache: bit-exact.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from self_speculative_verification_gb300 import workloads as W
from self_speculative_verification_gb300.device import DeviceStep

TOL = {
    "bf16": dict(o_abs=1e-2, o_rel_norm=1e-2, lse_rel=1e-3),
    "f32": dict(o_abs=2e-5, o_rel_norm=1e-5, lse_rel=1e-5),
}


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def unpack_vis(vis: np.ndarray, R: int) -> np.ndarray:
    """[B][R][W] int32 words -> [B][R][R] bool (bit c of word c//32)."""
    u = vis.astype(np.int64) & 0xFFFFFFFF
    B = u.shape[0]
    out = np.zeros((B, R, R), dtype=bool)
    for c in range(R):
        out[:, :, c] = (u[:, :, c // 32] >> (c % 32)) & 1
    return out


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_mask(ds: DeviceStep):
    wl = ds.wl
    vis, valid, sees = oracle.mask_build(wl.vparent, wl.soft_flags)
    got = unpack_vis(ds.vis.cpu().numpy(), wl.R)
    assert np.array_equal(got, vis)
    fl = ds.row_flags.cpu().numpy()
    assert np.array_equal((fl & 1) != 0, valid)
    assert np.array_equal((fl & 2) != 0, sees)
    return vis, valid, sees


def block_values(wl):
    """The block V the attention sees: the generator's, with the stream rows
    rotated when the workload has stream values by rotation (SS Eq. 7)."""
    if wl.rotation_eps is None:
        return wl.vb
    rot = oracle.rotate_stream_values(wl.vb, wl.n_nodes, wl.gamma, wl.rotation_eps)
    return W.round_bf16(rot.astype(np.float32)) if wl.dtype == "bf16" else rot


def oracle_attention(wl, vis, valid, sees, requests=None, heads=None):
    pk, pv = [], []
    for b in range(wl.B):
        if requests is None or b in requests:
            k, v = wl.prefix_kv(b)
        else:
            k = v = np.zeros((wl.Hkv, 0, wl.d), dtype=np.float32)
        pk.append(k)
        pv.append(v)
    return oracle.verify_attention(wl.q, pk, pv, wl.kb, block_values(wl), vis, valid, sees,
                                   soft_k=wl.soft_k, soft_v=wl.soft_v,
                                   requests=requests, heads=heads)


def check_attention(ds: DeviceStep, O_ref, L_ref, requests=None, heads=None):
    wl = ds.wl
    tol = TOL[wl.dtype]
    O = f64(ds.o)
    L = ds.lse.cpu().numpy().astype(np.float64)
    bs = list(range(wl.B)) if requests is None else list(requests)
    hs = list(range(wl.Hq)) if heads is None else list(heads)
    Og = O[bs][:, :, hs]
    Or = O_ref[bs][:, :, hs]
    Lg = L[bs][:, hs]
    Lr = L_ref[bs][:, hs]
    assert np.isfinite(Og).all()
    err = np.abs(Og - Or)
    assert err.max() <= tol["o_abs"], f"max abs err {err.max()}"
    nrm = np.linalg.norm(Or)
    if nrm > 0:
        assert np.linalg.norm(Og - Or) / nrm <= tol["o_rel_norm"], \
            f"relative norm err {np.linalg.norm(Og - Or) / nrm}"
    fin = np.isfinite(Lr)
    assert np.array_equal(np.isfinite(Lg), fin)
    assert np.all(Lg[~fin] == -np.inf)
    rel = np.abs(Lg[fin] - Lr[fin]) / np.maximum(np.abs(Lr[fin]), 1e-30)
    if rel.size:
        assert rel.max() <= tol["lse_rel"], f"LSE rel err {rel.max()}"
    return err.max(), (rel.max() if rel.size else 0.0)


def oracle_accept(wl):
    logits = wl.logits.reshape(wl.B * wl.Rj, wl.V)
    prop = wl.tokens.reshape(-1) if wl.mode == "la" else None
    am, lse, zp = oracle.vocab_reduce(logits, prop)
    am, lse, zp = (a.reshape(wl.B, wl.Rj) for a in (am, lse, zp))
    mode = oracle.MODE_THRESH_CHAIN if wl.mode == "la" else oracle.MODE_GREEDY_TREE
    acc, paths, nxt, last = oracle.accept(mode, wl.tau, wl.tokens, wl.tree_parent,
                                          wl.n_nodes, am, lse, zp)
    return am, lse, zp, acc, paths, nxt, last


# A sampled correction token is unique only away from the boundaries of the
# residual CDF.  The kernel sums fp32 masses in at most ~25 sequential
# rounding steps (8 per lane, a 32-lane tree, a few tiles per lane, a
# 32-lane scan) and its probabilities carry ~1e-6 relative error, so its
# cumulative sums stay within 1e-5 of the total of the float64 ones; a draw
# that differs from the oracle's must lie within that band of the boundary.
CDF_TOL = 1e-5


def residual_mass(wl, b, c):
    p = oracle.softmax_t(wl.logits[b, c], wl.temperature)
    dr = int(wl.child_draft_row[b, c])
    if dr < 0:
        return p
    r = np.maximum(0.0, p - oracle.softmax_t(wl.draft_logits[b, dr], wl.temperature))
    return r if r.sum() > 0 else p


def check_soft_draw(wl, b, c, got, want):
    """``got`` is the oracle's draw ``want``, or a neighbour across a CDF
    boundary the fp32 sums cannot resolve."""
    if got == want:
        return
    r = residual_mass(wl, b, c)
    cum = np.cumsum(r)
    target = float(wl.u_sample[b]) * cum[-1]
    tol = CDF_TOL * cum[-1]
    lo = cum[got - 1] if got > 0 else 0.0
    assert r[got] > 0, f"request {b}: drawn token {got} has no residual mass"
    assert lo - tol <= target <= cum[got] + tol, \
        f"request {b}: drawn {got}, oracle {want}, target {target} outside [{lo}, {cum[got]}]"


def check_accept_soft(ds: DeviceStep):
    wl = ds.wl
    acc, paths, nxt, last = oracle.accept_soft(
        wl.logits, wl.draft_logits, wl.tokens, wl.tree_parent, None, wl.child_draft_row,
        wl.n_nodes, wl.u_accept, wl.u_sample, wl.temperature)
    acc_g = ds.acc_len.cpu().numpy()
    path_g = ds.path.cpu().numpy()
    assert acc_g.tolist() == acc.tolist()
    assert acc_g.tolist() == wl.expect_acc_len.tolist()
    for b in range(wl.B):
        assert path_g[b, : acc_g[b]].tolist() == paths[b]
        assert np.all(path_g[b, acc_g[b]:] == -1)
    assert ds.last_node.cpu().numpy().tolist() == last.tolist()
    lse_ref = np.array([[np.log(np.exp(wl.logits[b, j].astype(np.float64) / wl.temperature
                                        - (wl.logits[b, j].max() / wl.temperature)).sum())
                         + wl.logits[b, j].max() / wl.temperature for j in range(wl.Rj)]
                        for b in range(wl.B)])
    lg = ds.lse_v.cpu().numpy().astype(np.float64)
    assert (np.abs(lg - lse_ref) / np.abs(lse_ref)).max() <= 1e-5
    nxt_g = ds.next_token.cpu().numpy()
    for b in range(wl.B):
        check_soft_draw(wl, b, int(last[b]), int(nxt_g[b]), int(nxt[b]))
    return acc, paths


def check_accept(ds: DeviceStep):
    wl = ds.wl
    if wl.soft:
        return check_accept_soft(ds)
    am, lse, zp, acc, paths, nxt, last = oracle_accept(wl)
    assert np.array_equal(ds.argmax.cpu().numpy(), am)
    lg = ds.lse_v.cpu().numpy().astype(np.float64)
    assert (np.abs(lg - lse) / np.abs(lse)).max() <= 1e-5
    if wl.mode == "la":
        assert np.array_equal(ds.zprop.cpu().numpy().astype(np.float64), zp)
    acc_g = ds.acc_len.cpu().numpy()
    path_g = ds.path.cpu().numpy()
    assert acc_g.tolist() == acc.tolist()
    assert acc_g.tolist() == wl.expect_acc_len.tolist()
    for b in range(wl.B):
        assert path_g[b, : acc_g[b]].tolist() == paths[b]
        assert np.all(path_g[b, acc_g[b]:] == -1)
    assert ds.next_token.cpu().numpy().tolist() == nxt.tolist()
    assert ds.last_node.cpu().numpy().tolist() == last.tolist()
    return acc, paths


def cache_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy()
    return t.view(torch.int32).cpu().numpy()


def block_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Storage bits of a generator block array (float32 holding dtype values)."""
    if dtype == "bf16":
        return (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16).view(np.int16)
    return x.astype(np.float32).view(np.int32)


def check_commit(ds: DeviceStep, before_k, before_v, paths):
    """The cache after the step equals the oracle's commit (kv_commit_contiguous
    / kv_commit_paged) applied to the cache's bits before it and the block's
    bits; page table, seq_len and free_head equal the oracle's."""
    wl = ds.wl
    after_k = cache_bits(ds.k_cache)
    after_v = cache_bits(ds.v_cache)
    kb_bits = block_bits(wl.kb, wl.dtype)
    vb_bits = block_bits(wl.vb, wl.dtype)
    if wl.paged:
        exp_k, exp_v, pt, seq2, head = oracle.kv_commit_paged(
            before_k, before_v, wl.page_table, wl.seq_len, wl.free_pages, 0,
            kb_bits, vb_bits, paths, wl.page_size)
        assert np.array_equal(ds.page_table.cpu().numpy(), pt)
        assert int(ds.free_head.item()) == head
    else:
        exp_k, exp_v, seq2 = oracle.kv_commit_contiguous(before_k, before_v, wl.seq_len,
                                                         kb_bits, vb_bits, paths)
    assert np.array_equal(after_k, exp_k)
    assert np.array_equal(after_v, exp_v)
    assert ds.seq_len.cpu().numpy().tolist() == seq2.tolist()


def commit_expected_on_device(ds: DeviceStep, k0, v0, paths):
    """Expected cache after the commit of a full-size workload, without a
    host copy of the cache: the oracle's commit is applied to index arrays
    (one entry per cache slot, holding 1 + b * R + row of the block row the
    slot receives, 0 for untouched slots), which gives every slot's source;
    the device snapshot k0 / v0 then receives those rows.  Returns (k, v,
    page_table, seq_len, free_head) as the oracle computes them."""
    wl = ds.wl
    R = wl.R
    src = (1 + np.arange(wl.B)[:, None] * R + np.arange(R)[None, :]).astype(np.int64)
    blk = src[:, None, :, None]                      # [B][1][R][1]
    ek, ev = k0.clone(), v0.clone()
    if wl.paged:
        n_pages = ds.k_cache.shape[0]
        idx = np.zeros((n_pages, 1, 1, wl.page_size, 1), dtype=np.int64)
        idx, _, pt, seq2, head = oracle.kv_commit_paged(
            idx, idx, wl.page_table, wl.seq_len, wl.free_pages, 0, blk, blk, paths,
            wl.page_size)
        pages, slots = np.nonzero(idx[:, 0, 0, :, 0])
        nb = wl.d // 64
        for p, t in zip(pages.tolist(), slots.tolist()):
            b, row = divmod(int(idx[p, 0, 0, t, 0]) - 1, R)
            ek[p, :, :, t] = ds.kb[b, :, row].view(wl.Hkv, nb, 64)
            ev[p, :, :, t] = ds.vb[b, :, row].view(wl.Hkv, nb, 64)
        return ek, ev, pt, seq2, head
    idx = np.zeros((wl.B, 1, ds.k_cache.shape[2], 1), dtype=np.int64)
    idx, _, seq2 = oracle.kv_commit_contiguous(idx, idx, wl.seq_len, blk, blk, paths)
    reqs, poss = np.nonzero(idx[:, 0, :, 0])
    for bb, t in zip(reqs.tolist(), poss.tolist()):
        b, row = divmod(int(idx[bb, 0, t, 0]) - 1, R)
        ek[bb, :, t] = ds.kb[b, :, row]
        ev[bb, :, t] = ds.vb[b, :, row]
    return ek, ev, None, seq2, None


def run_and_check(wl, split_tokens=0, requests=None, heads=None):
    """Full parity check of one step on a (small) workload."""
    ds = DeviceStep(wl, split_tokens=split_tokens)
    before_k = cache_bits(ds.k_cache)
    before_v = cache_bits(ds.v_cache)
    ds.run()
    torch.cuda.synchronize()
    from self_speculative_verification_gb300 import binding
    assert binding.spec_get_status() == 0
    vis, valid, sees = check_mask(ds)
    O_ref, L_ref = oracle_attention(wl, vis, valid, sees, requests, heads)
    errs = check_attention(ds, O_ref, L_ref, requests, heads)
    acc, paths = check_accept(ds)
    check_commit(ds, before_k, before_v, paths)
    if ds.future is not None:
        # ConFu hand-off: bit-identical to the contemplate row of the last node
        want = oracle.future_gather(ds.o.cpu().float().numpy(), ds.last_node.cpu().numpy(),
                                    wl.N)
        assert np.array_equal(ds.future.cpu().float().numpy(), want)
    return ds, errs
