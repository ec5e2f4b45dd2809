"""Python binding of the libspecverify C ABI (argument marshalling only).

Every function here has the name of the C entry point it calls, checks the
tensors it is handed (CUDA device, dtype, contiguity, shape), passes raw
device pointers plus the current torch CUDA stream, and raises
``SpecError`` on any non-zero return code.  No arithmetic of the
verification step happens in Python: if the shared library is missing,
``load_library`` raises and nothing runs.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_size_t, c_void_p

import torch

from . import _build

# return codes / enums (include/specverify.h)
SPEC_OK = 0
SPEC_ERR_INVALID_ARG = 1
SPEC_ERR_UNSUPPORTED = 2
SPEC_ERR_CAPACITY = 4
SPEC_ERR_CUDA = 5
SPEC_ERR_DEVICE = 6
SPEC_F32 = 0
SPEC_BF16 = 1
SPEC_KV_CONTIGUOUS = 0
SPEC_KV_PAGED = 1
SPEC_ACCEPT_THRESH_CHAIN = 0
SPEC_ACCEPT_GREEDY_TREE = 1
SPEC_ROW_VALID = 1
SPEC_ROW_SEES_SOFT = 2
SPEC_DEV_BAD_TREE = 0x01
SPEC_DEV_BAD_PAGE = 0x02
SPEC_DEV_SEQ_OVERFLOW = 0x04
SPEC_DEV_CAPACITY = 0x08
SPEC_DEV_BAD_INDEX = 0x10
SPEC_DEV_TIMEOUT = 0x20

EXPORTS = ("spec_version", "spec_status_string", "spec_mask_build",
           "spec_verify_attn_workspace_size", "spec_verify_attn",
           "spec_verify_attn_noalloc", "spec_vocab_reduce", "spec_accept", "kv_commit",
           "spec_get_status", "spec_la_prefill_attn", "spec_accept_soft", "spec_draft_tree",
           "spec_prune_tree", "spec_stream_rotate_values", "spec_future_gather",
           "spec_set_wait_limit")
SPEC_NOALLOC_SCRATCH_BYTES = 64 << 20


class SpecError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed: {msg} (code {code})")
        self.code = code


class KvDesc(ctypes.Structure):
    _fields_ = [("kind", c_int), ("dtype", c_int), ("n_kv_heads", c_int),
                ("head_dim", c_int), ("k", c_void_p), ("v", c_void_p),
                ("batch", c_int), ("max_seq", c_int), ("n_pages", c_int),
                ("page_size", c_int), ("max_pages_per_seq", c_int),
                ("page_table", c_void_p)]


class AttnDesc(ctypes.Structure):
    _fields_ = [("batch", c_int), ("n_rows", c_int), ("n_q_heads", c_int),
                ("n_kv_heads", c_int), ("head_dim", c_int), ("dtype", c_int),
                ("n_soft", c_int), ("scale", c_float), ("split_tokens", c_int)]


class AcceptDesc(ctypes.Structure):
    _fields_ = [("mode", c_int), ("tau", c_float), ("batch", c_int),
                ("n_judge_rows", c_int), ("vocab", c_int), ("logit_dtype", c_int),
                ("max_nodes", c_int), ("path_cap", c_int)]


class SoftDesc(ctypes.Structure):
    _fields_ = [("batch", c_int), ("n_judge_rows", c_int), ("n_draft_rows", c_int),
                ("vocab", c_int), ("logit_dtype", c_int), ("max_nodes", c_int),
                ("path_cap", c_int), ("temperature", c_float)]


class DraftDesc(ctypes.Structure):
    _fields_ = [("batch", c_int), ("n_stream_rows", c_int), ("gamma", c_int), ("k", c_int),
                ("vocab", c_int), ("logit_dtype", c_int), ("max_nodes", c_int),
                ("vparent_rows", c_int)]


class PruneDesc(ctypes.Structure):
    _fields_ = [("batch", c_int), ("max_nodes", c_int), ("vocab", c_int),
                ("logit_dtype", c_int), ("threshold", c_float), ("gamma", c_int),
                ("vparent_rows", c_int)]


class RotateDesc(ctypes.Structure):
    _fields_ = [("batch", c_int), ("n_rows", c_int), ("n_kv_heads", c_int),
                ("head_dim", c_int), ("dtype", c_int), ("gamma", c_int), ("eps", c_float)]


class PrefillDesc(ctypes.Structure):
    _fields_ = [("batch", c_int), ("n_orig", c_int), ("n_look", c_int),
                ("n_q_heads", c_int), ("n_kv_heads", c_int), ("head_dim", c_int),
                ("dtype", c_int), ("scale", c_float)]


_lib = None


def library_path() -> str:
    return os.environ.get("SPECVERIFY_LIB", _build.LIB)


def load_library():
    """Load libspecverify.so (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libspecverify is not built ({path} missing); "
                           "run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    vp = c_void_p
    sig = {
        "spec_version": ([], c_int),
        "spec_status_string": ([c_int], ctypes.c_char_p),
        "spec_mask_build": ([vp, vp, c_int, c_int, vp, vp, vp], c_int),
        "spec_verify_attn_workspace_size": ([POINTER(AttnDesc), POINTER(KvDesc),
                                             POINTER(c_size_t)], c_int),
        "spec_verify_attn": ([POINTER(AttnDesc), vp, POINTER(KvDesc), vp, vp, vp, vp,
                              vp, vp, vp, vp, vp, vp, c_size_t, vp], c_int),
        "spec_verify_attn_noalloc": ([POINTER(AttnDesc), vp, POINTER(KvDesc), vp, vp, vp, vp,
                                      vp, vp, vp, vp, vp, vp], c_int),
        "spec_vocab_reduce": ([vp, c_int, c_int, c_int, vp, vp, vp, vp, vp], c_int),
        "spec_accept": ([POINTER(AcceptDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                         vp, vp, vp], c_int),
        "kv_commit": ([POINTER(KvDesc), c_int, c_int, vp, vp, c_int, vp, vp, vp, vp,
                       c_int, vp, vp], c_int),
        "spec_get_status": ([vp, POINTER(ctypes.c_int32)], c_int),
        "spec_set_wait_limit": ([ctypes.c_longlong], ctypes.c_longlong),
        "spec_la_prefill_attn": ([POINTER(PrefillDesc), vp, vp, vp, vp, vp, vp], c_int),
        "spec_accept_soft": ([POINTER(SoftDesc)] + [vp] * 16, c_int),
        "spec_draft_tree": ([POINTER(DraftDesc)] + [vp] * 8, c_int),
        "spec_prune_tree": ([POINTER(PruneDesc)] + [vp] * 10, c_int),
        "spec_stream_rotate_values": ([POINTER(RotateDesc), vp, vp, vp], c_int),
        "spec_future_gather": ([c_int, c_int, c_int, c_int, vp, vp, c_int, vp, vp], c_int),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _check(fn, code):
    if code != SPEC_OK:
        msg = load_library().spec_status_string(code).decode()
        raise SpecError(fn, code, msg)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return c_void_p(t.data_ptr())


def spec_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


# ----------------------------------------------------------------- descriptors

def kv_desc_contiguous(k: torch.Tensor, v: torch.Tensor) -> KvDesc:
    """k, v: [B][Hkv][max_seq][d]."""
    if k.shape != v.shape or k.dim() != 4:
        raise ValueError("k and v must be [B][Hkv][max_seq][d]")
    _ptr(k, name="k"), _ptr(v, k.dtype, "v")
    B, Hkv, S, d = k.shape
    return KvDesc(SPEC_KV_CONTIGUOUS, spec_dtype(k), Hkv, d, k.data_ptr(), v.data_ptr(),
                  B, S, 0, 0, 0, None)


def kv_desc_paged(k: torch.Tensor, v: torch.Tensor, page_table: torch.Tensor) -> KvDesc:
    """k, v: [n_pages][Hkv][d / 64][page_size][64]; page_table int32 [B][max_pages]."""
    if k.shape != v.shape or k.dim() != 5 or k.shape[4] != 64:
        raise ValueError("k and v must be [n_pages][Hkv][d / 64][page_size][64]")
    _ptr(k, name="k"), _ptr(v, k.dtype, "v")
    _ptr(page_table, torch.int32, "page_table")
    P, Hkv, nblk, ps, _ = k.shape
    d = nblk * 64
    B, maxp = page_table.shape
    return KvDesc(SPEC_KV_PAGED, spec_dtype(k), Hkv, d, k.data_ptr(), v.data_ptr(),
                  B, 0, P, ps, maxp, page_table.data_ptr())


def attn_desc(batch, n_rows, n_q_heads, n_kv_heads, head_dim, dtype, n_soft=0,
              scale=0.0, split_tokens=0) -> AttnDesc:
    return AttnDesc(batch, n_rows, n_q_heads, n_kv_heads, head_dim, dtype, n_soft,
                    scale, split_tokens)


def accept_desc(mode, tau, batch, n_judge_rows, vocab, logit_dtype, max_nodes,
                path_cap) -> AcceptDesc:
    return AcceptDesc(mode, tau, batch, n_judge_rows, vocab, logit_dtype, max_nodes,
                      path_cap)


# ------------------------------------------------------------------- entry points

def prefill_desc(batch, n_orig, n_look, n_q_heads, n_kv_heads, head_dim, dtype=SPEC_BF16,
                 scale=0.0) -> PrefillDesc:
    return PrefillDesc(batch, n_orig, n_look, n_q_heads, n_kv_heads, head_dim, dtype, scale)


def soft_desc(batch, n_judge_rows, n_draft_rows, vocab, logit_dtype, max_nodes, path_cap,
              temperature=1.0) -> SoftDesc:
    return SoftDesc(batch, n_judge_rows, n_draft_rows, vocab, logit_dtype, max_nodes, path_cap,
                    temperature)


def spec_version() -> int:
    return load_library().spec_version()


def spec_mask_build(vparent, soft_flags, vis, row_flags, stream=None):
    lib = load_library()
    B, R = vparent.shape
    W = (R + 31) // 32
    if tuple(vis.shape) != (B, R, W) or tuple(row_flags.shape) != (B, R):
        raise ValueError("vis must be [B][R][ceil(R/32)], row_flags [B][R]")
    _check("spec_mask_build", lib.spec_mask_build(
        _ptr(vparent, torch.int32, "vparent"), _ptr(soft_flags, torch.uint8, "soft_flags"),
        B, R, _ptr(vis, torch.int32, "vis"), _ptr(row_flags, torch.uint8, "row_flags"),
        _stream(stream)))


def spec_verify_attn_workspace_size(attn: AttnDesc, cache: KvDesc) -> int:
    lib = load_library()
    n = c_size_t(0)
    _check("spec_verify_attn_workspace_size",
           lib.spec_verify_attn_workspace_size(ctypes.byref(attn), ctypes.byref(cache),
                                               ctypes.byref(n)))
    return n.value


def spec_verify_attn(attn: AttnDesc, q, cache: KvDesc, kb, vb, soft_k, soft_v, seq_len,
                     vis, row_flags, o, lse, workspace, stream=None):
    lib = load_library()
    dt = q.dtype
    for name, t in (("kb", kb), ("vb", vb), ("o", o)):
        _ptr(t, dt, name)
    _check("spec_verify_attn", lib.spec_verify_attn(
        ctypes.byref(attn), _ptr(q, name="q"), ctypes.byref(cache), _ptr(kb), _ptr(vb),
        _ptr(soft_k, dt, "soft_k"), _ptr(soft_v, dt, "soft_v"),
        _ptr(seq_len, torch.int32, "seq_len"), _ptr(vis, torch.int32, "vis"),
        _ptr(row_flags, torch.uint8, "row_flags"), _ptr(o), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, name="workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def spec_verify_attn_noalloc(attn: AttnDesc, q, cache: KvDesc, kb, vb, soft_k, soft_v,
                             seq_len, vis, row_flags, o, lse, stream=None):
    """spec_verify_attn without a workspace: for callers that cannot
    allocate device memory; the library's own fixed scratch array is used
    (shared by all calls on a device, so overlapping calls must not run)."""
    lib = load_library()
    dt = q.dtype
    for name, t in (("kb", kb), ("vb", vb), ("o", o)):
        _ptr(t, dt, name)
    _check("spec_verify_attn_noalloc", lib.spec_verify_attn_noalloc(
        ctypes.byref(attn), _ptr(q, name="q"), ctypes.byref(cache), _ptr(kb), _ptr(vb),
        _ptr(soft_k, dt, "soft_k"), _ptr(soft_v, dt, "soft_v"),
        _ptr(seq_len, torch.int32, "seq_len"), _ptr(vis, torch.int32, "vis"),
        _ptr(row_flags, torch.uint8, "row_flags"), _ptr(o), _ptr(lse, torch.float32, "lse"),
        _stream(stream)))


def spec_vocab_reduce(logits, proposal, argmax, lse, zprop, stream=None):
    lib = load_library()
    n, V = logits.shape
    _check("spec_vocab_reduce", lib.spec_vocab_reduce(
        _ptr(logits, name="logits"), spec_dtype(logits), n, V,
        _ptr(proposal, torch.int32, "proposal"), _ptr(argmax, torch.int32, "argmax"),
        _ptr(lse, torch.float32, "lse"), _ptr(zprop, torch.float32, "zprop"),
        _stream(stream)))


def spec_accept(desc: AcceptDesc, logits, tokens, tree_parent, row_of, n_nodes, argmax, lse,
                zprop, acc_len, path, next_token, last_node, stream=None):
    lib = load_library()
    i32 = torch.int32
    _check("spec_accept", lib.spec_accept(
        ctypes.byref(desc), _ptr(logits, name="logits"), _ptr(tokens, i32, "tokens"),
        _ptr(tree_parent, i32, "tree_parent"), _ptr(row_of, i32, "row_of"),
        _ptr(n_nodes, i32, "n_nodes"), _ptr(argmax, i32, "argmax"),
        _ptr(lse, torch.float32, "lse"), _ptr(zprop, torch.float32, "zprop"),
        _ptr(acc_len, i32, "acc_len"), _ptr(path, i32, "path"),
        _ptr(next_token, i32, "next_token"), _ptr(last_node, i32, "last_node"),
        _stream(stream)))


def kv_commit(cache: KvDesc, kb, vb, path, acc_len, seq_len, free_pages=None, free_head=None,
              stream=None):
    lib = load_library()
    B, Hkv, R, d = kb.shape
    i32 = torch.int32
    n_free = 0 if free_pages is None else free_pages.numel()
    _check("kv_commit", lib.kv_commit(
        ctypes.byref(cache), B, R, _ptr(kb, name="kb"), _ptr(vb, kb.dtype, "vb"),
        path.shape[1], _ptr(path, i32, "path"), _ptr(acc_len, i32, "acc_len"),
        _ptr(seq_len, i32, "seq_len"), _ptr(free_pages, i32, "free_pages"), n_free,
        _ptr(free_head, i32, "free_head"), _stream(stream)))


def spec_get_status(stream=None) -> int:
    """Synchronise, read and clear the device status word (SPEC_DEV_* bits)."""
    lib = load_library()
    out = ctypes.c_int32(0)
    code = lib.spec_get_status(_stream(stream), ctypes.byref(out))
    if code not in (SPEC_OK, SPEC_ERR_DEVICE):
        _check("spec_get_status", code)
    return out.value


def spec_set_wait_limit(cycles: int) -> int:
    """Limit (SM cycles) of the kernels' pipeline waits from now on; a
    negative value restores the default.  Returns the previous limit."""
    return load_library().spec_set_wait_limit(int(cycles))


def spec_la_prefill_attn(desc: PrefillDesc, q, k, v, o, lse, stream=None):
    """Prefill-form Lookahead Attention: q, o [B][n+k][Hq][d]; k, v
    [B][n+k][Hkv][d] (bf16); lse [B][Hq][n+k] fp32."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _ptr(t, torch.bfloat16, name)
    _check("spec_la_prefill_attn", lib.spec_la_prefill_attn(
        ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
        _ptr(lse, torch.float32, "lse"), _stream(stream)))


def spec_accept_soft(desc: SoftDesc, logits, draft_logits, tokens, tree_parent, row_of,
                     child_draft_row, n_nodes, u_accept, u_sample, lse_t, lse_d, acc_len, path,
                     next_token, last_node, stream=None):
    """Soft-matching acceptance (ratio test down the tree, residual draw)."""
    lib = load_library()
    i32, f32 = torch.int32, torch.float32
    _check("spec_accept_soft", lib.spec_accept_soft(
        ctypes.byref(desc), _ptr(logits, name="logits"),
        _ptr(draft_logits, logits.dtype, "draft_logits"), _ptr(tokens, i32, "tokens"),
        _ptr(tree_parent, i32, "tree_parent"), _ptr(row_of, i32, "row_of"),
        _ptr(child_draft_row, i32, "child_draft_row"), _ptr(n_nodes, i32, "n_nodes"),
        _ptr(u_accept, f32, "u_accept"), _ptr(u_sample, f32, "u_sample"),
        _ptr(lse_t, f32, "lse_t"), _ptr(lse_d, f32, "lse_d"), _ptr(acc_len, i32, "acc_len"),
        _ptr(path, i32, "path"), _ptr(next_token, i32, "next_token"),
        _ptr(last_node, i32, "last_node"), _stream(stream)))


def spec_draft_tree(desc: DraftDesc, stream_logits, stream_row, root_token, tokens, tree_parent,
                    n_nodes, vparent=None, stream=None):
    """Top-k per stream -> complete k-ary draft tree (+ the block's vparent)."""
    lib = load_library()
    i32 = torch.int32
    _check("spec_draft_tree", lib.spec_draft_tree(
        ctypes.byref(desc), _ptr(stream_logits, name="stream_logits"),
        _ptr(stream_row, i32, "stream_row"), _ptr(root_token, i32, "root_token"),
        _ptr(tokens, i32, "tokens"), _ptr(tree_parent, i32, "tree_parent"),
        _ptr(n_nodes, i32, "n_nodes"), _ptr(vparent, i32, "vparent"), _stream(stream)))


def spec_prune_tree(desc: PruneDesc, tokens, tree_parent, n_nodes, early_logits, keep_map,
                    tokens_out, parent_out, n_out, vparent=None, stream=None):
    """Drop subtrees whose edge probability under the early-exit logits is
    below the threshold; compact the survivors."""
    lib = load_library()
    i32 = torch.int32
    _check("spec_prune_tree", lib.spec_prune_tree(
        ctypes.byref(desc), _ptr(tokens, i32, "tokens"), _ptr(tree_parent, i32, "tree_parent"),
        _ptr(n_nodes, i32, "n_nodes"), _ptr(early_logits, name="early_logits"),
        _ptr(keep_map, i32, "keep_map"), _ptr(tokens_out, i32, "tokens_out"),
        _ptr(parent_out, i32, "parent_out"), _ptr(n_out, i32, "n_out"),
        _ptr(vparent, i32, "vparent"), _stream(stream)))


def spec_stream_rotate_values(desc: RotateDesc, n_nodes, vb, stream=None):
    """Stream rows of the block values := their node's values rotated by
    e^{i eps s} (in place)."""
    lib = load_library()
    _check("spec_stream_rotate_values", lib.spec_stream_rotate_values(
        ctypes.byref(desc), _ptr(n_nodes, torch.int32, "n_nodes"), _ptr(vb, name="vb"),
        _stream(stream)))


def spec_future_gather(o, last_node, row_offset, out, stream=None):
    """out[b] = o[b][row_offset + last_node[b]] (o: [B][R][...])."""
    lib = load_library()
    B, R = o.shape[0], o.shape[1]
    row = o[0, 0].numel()
    _ptr(out, o.dtype, "out")
    _check("spec_future_gather", lib.spec_future_gather(
        B, R, row, spec_dtype(o), _ptr(o, name="o"), _ptr(last_node, torch.int32, "last_node"),
        row_offset, _ptr(out), _stream(stream)))
