"""Device buffers for one verification step, and the step itself.

``DeviceStep`` places a ``workloads.Workload`` in torch device memory
(plumbing only: allocation, host-to-device copies, dtype storage) and runs
the step as the four C-ABI calls in order:

    spec_mask_build -> spec_verify_attn -> spec_accept -> kv_commit

Every arithmetic step runs in libspecverify's kernels.
"""

from __future__ import annotations

import concurrent.futures as cf
import math

import numpy as np
import torch

from . import binding as bn
from .workloads import Workload


def torch_dtype(name: str):
    return torch.bfloat16 if name == "bf16" else torch.float32


def to_dev(x: np.ndarray, device, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x)).to(device)
    return t if dtype is None else t.to(dtype)


def _fill_contiguous(wl: Workload, K, V, dt, threads=8, fill=math.nan):
    K.fill_(fill)
    V.fill_(fill)

    def one(b):
        k, v = wl.prefix_kv(b)
        return b, k, v

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for b, k, v in ex.map(one, range(wl.B)):
            S = k.shape[1]
            K[b, :, :S] = to_dev(k, K.device, dt)
            V[b, :, :S] = to_dev(v, V.device, dt)


def _fill_paged(wl: Workload, K, V, dt, threads=8, fill=math.nan):
    K.fill_(fill)
    V.fill_(fill)
    ps = wl.page_size

    def one(b):
        k, v = wl.prefix_kv(b)
        return b, k, v

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for b, k, v in ex.map(one, range(wl.B)):
            S = k.shape[1]
            npg = (S + ps - 1) // ps
            if npg == 0:
                continue
            pages = torch.from_numpy(wl.page_table[b, :npg].astype(np.int64)).to(K.device)
            for src, dst in ((k, K), (v, V)):
                t = to_dev(src, K.device, dt)                     # [Hkv][S][d]
                pad = torch.full((wl.Hkv, npg * ps, wl.d), fill, dtype=dt, device=K.device)
                pad[:, :S] = t
                # -> [page][Hkv][d / 64][page_size][64]
                blk = pad.view(wl.Hkv, npg, ps, wl.d // 64, 64).permute(1, 0, 3, 2, 4)
                dst.index_copy_(0, pages, blk.contiguous())


class DeviceStep:
    """All device buffers of one verification step for a workload."""

    def __init__(self, wl: Workload, device="cuda", split_tokens: int = 0,
                 threads: int = 8, fill=math.nan):
        self.wl = wl
        self.device = torch.device(device)
        dev = self.device
        dt = torch_dtype(wl.dtype)
        ldt = torch_dtype(wl.logit_dtype)
        self.dt = dt
        i32 = torch.int32
        B, R, Hq, Hkv, d = wl.B, wl.R, wl.Hq, wl.Hkv, wl.d
        W = (R + 31) // 32

        # per-step inputs
        self.q = to_dev(wl.q, dev, dt)
        self.kb = to_dev(wl.kb, dev, dt)
        self.vb = to_dev(wl.vb, dev, dt)
        self.soft_k = to_dev(wl.soft_k, dev, dt) if wl.n_soft else None
        self.soft_v = to_dev(wl.soft_v, dev, dt) if wl.n_soft else None
        self.vparent = to_dev(wl.vparent.astype(np.int32), dev)
        self.soft_flags = to_dev(wl.soft_flags.astype(np.uint8), dev)
        self.logits = to_dev(wl.logits, dev, ldt)
        self.tokens = to_dev(wl.tokens.astype(np.int32), dev)
        self.tree_parent = to_dev(wl.tree_parent.astype(np.int32), dev)
        self.n_nodes = to_dev(wl.n_nodes.astype(np.int32), dev)

        # committed cache (state)
        self.seq_len = to_dev(wl.seq_len.astype(np.int32), dev)
        self.seq_len0 = self.seq_len.clone()
        if wl.paged:
            shape = (wl.n_pages, Hkv, d // 64, wl.page_size, 64)
            self.k_cache = torch.empty(shape, dtype=dt, device=dev)
            self.v_cache = torch.empty(shape, dtype=dt, device=dev)
            _fill_paged(wl, self.k_cache, self.v_cache, dt, threads, fill)
            self.page_table = to_dev(wl.page_table.astype(np.int32), dev)
            self.page_table0 = self.page_table.clone()
            self.free_pages = to_dev(wl.free_pages.astype(np.int32), dev)
            self.free_head = torch.zeros(1, dtype=i32, device=dev)
            self.free_head0 = self.free_head.clone()
            self.cache = bn.kv_desc_paged(self.k_cache, self.v_cache, self.page_table)
        else:
            shape = (B, Hkv, wl.max_seq, d)
            self.k_cache = torch.empty(shape, dtype=dt, device=dev)
            self.v_cache = torch.empty(shape, dtype=dt, device=dev)
            _fill_contiguous(wl, self.k_cache, self.v_cache, dt, threads, fill)
            self.page_table = None
            self.free_pages = None
            self.free_head = None
            self.cache = bn.kv_desc_contiguous(self.k_cache, self.v_cache)

        # outputs
        self.vis = torch.zeros((B, R, W), dtype=i32, device=dev)
        self.row_flags = torch.zeros((B, R), dtype=torch.uint8, device=dev)
        self.o = torch.zeros((B, R, Hq, d), dtype=dt, device=dev)
        self.lse = torch.zeros((B, Hq, R), dtype=torch.float32, device=dev)
        self.argmax = torch.zeros((B, wl.Rj), dtype=i32, device=dev)
        self.lse_v = torch.zeros((B, wl.Rj), dtype=torch.float32, device=dev)
        self.zprop = torch.zeros((B, wl.Rj), dtype=torch.float32, device=dev)
        self.acc_len = torch.zeros(B, dtype=i32, device=dev)
        self.path = torch.zeros((B, wl.path_cap), dtype=i32, device=dev)
        self.next_token = torch.zeros(B, dtype=i32, device=dev)
        self.last_node = torch.zeros(B, dtype=i32, device=dev)

        self.attn = bn.attn_desc(B, R, Hq, Hkv, d, bn.spec_dtype(self.q), wl.n_soft, 0.0,
                                 split_tokens)
        ws = bn.spec_verify_attn_workspace_size(self.attn, self.cache)
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        mode = bn.SPEC_ACCEPT_THRESH_CHAIN if wl.mode == "la" else bn.SPEC_ACCEPT_GREEDY_TREE
        self.accept = bn.accept_desc(mode, wl.tau, B, wl.Rj, wl.V, bn.spec_dtype(self.logits),
                                     wl.N, wl.path_cap)
        # soft matching: draft distributions, uniforms, per-row LSE scratch
        self.draft_logits = self.child_draft_row = self.u_accept = self.u_sample = None
        self.lse_d = None
        if wl.soft:
            Rd = wl.draft_logits.shape[1]
            self.draft_logits = to_dev(wl.draft_logits, dev, ldt)
            self.child_draft_row = to_dev(wl.child_draft_row.astype(np.int32), dev)
            self.u_accept = to_dev(wl.u_accept.astype(np.float32), dev)
            self.u_sample = to_dev(wl.u_sample.astype(np.float32), dev)
            self.lse_d = torch.zeros((B, max(Rd, 1)), dtype=torch.float32, device=dev)
            self.soft = bn.soft_desc(B, wl.Rj, Rd, wl.V, bn.spec_dtype(self.logits), wl.N,
                                     wl.path_cap, wl.temperature)
        # stream values by rotation (SS): the block's stream V rows are
        # rewritten from their node rows before the attention
        self.rotate = None
        if wl.rotation_eps is not None:
            self.rotate = bn.RotateDesc(B, R, Hkv, d, bn.spec_dtype(self.vb), wl.gamma,
                                        wl.rotation_eps)
        # ConFu: the contemplate output of the last accepted node (row T + j)
        self.future = None
        if wl.layout == "confu":
            self.future = torch.zeros((B, Hq, d), dtype=dt, device=dev)
        # kernel launches of one run() (see libspecverify's sources): mask 1,
        # attention 2, accept 2 (soft: 3), commit 2, rotation 1, gather 1
        self.launches_per_step = (7 + (1 if wl.soft else 0) + (1 if self.rotate else 0) +
                                  (1 if self.future is not None else 0))

    # the four calls ---------------------------------------------------------
    def mask_build(self, stream=None):
        bn.spec_mask_build(self.vparent, self.soft_flags, self.vis, self.row_flags, stream)

    def verify_attn(self, stream=None):
        bn.spec_verify_attn(self.attn, self.q, self.cache, self.kb, self.vb, self.soft_k,
                            self.soft_v, self.seq_len, self.vis, self.row_flags, self.o,
                            self.lse, self.workspace, stream)

    def accept_step(self, stream=None):
        if self.wl.soft:
            bn.spec_accept_soft(self.soft, self.logits, self.draft_logits, self.tokens,
                                self.tree_parent, None, self.child_draft_row, self.n_nodes,
                                self.u_accept, self.u_sample, self.lse_v, self.lse_d,
                                self.acc_len, self.path, self.next_token, self.last_node,
                                stream)
            return
        tree = self.wl.mode != "la"
        bn.spec_accept(self.accept, self.logits, self.tokens,
                       self.tree_parent if tree else None, None, self.n_nodes,
                       self.argmax, self.lse_v, self.zprop, self.acc_len, self.path,
                       self.next_token, self.last_node, stream)

    def commit(self, stream=None):
        bn.kv_commit(self.cache, self.kb, self.vb, self.path, self.acc_len, self.seq_len,
                     self.free_pages, self.free_head, stream)

    def rotate_values(self, stream=None):
        if self.rotate is not None:
            bn.spec_stream_rotate_values(self.rotate, self.n_nodes, self.vb, stream)

    def gather_future(self, stream=None):
        if self.future is not None:
            bn.spec_future_gather(self.o, self.last_node, self.wl.N, self.future, stream)

    def run(self, stream=None):
        """One whole verification step (mask, attention, accept, commit; the
        stream-value rotation first and the ConFu future gather after the
        acceptance where the workload has them)."""
        self.rotate_values(stream)
        self.mask_build(stream)
        self.verify_attn(stream)
        self.accept_step(stream)
        self.gather_future(stream)
        self.commit(stream)

    def reset_state(self, page_table: bool = False):
        """Restore seq_len / free_head so the same step can run again: the
        re-run takes the same free pages and writes the same slots with the
        same bytes.  ``page_table=True`` also restores the table entries the
        commit added (they are rewritten identically either way)."""
        self.seq_len.copy_(self.seq_len0)
        if self.free_head is not None:
            self.free_head.copy_(self.free_head0)
            if page_table:
                self.page_table.copy_(self.page_table0)

    # kernel launches of one run() with threshold / greedy acceptance
    LAUNCHES_PER_STEP = 7   # mask 1, attention 2, accept 2, commit 2
