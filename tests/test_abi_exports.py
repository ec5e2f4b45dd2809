"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point include/specverify.h declares, and its structs have the layout
the Python binding assumes (checked with a C program compiled by gcc)."""

import ctypes
import os
import re
import shutil
import subprocess

import pytest

from self_speculative_verification_gb300 import _build, binding

HEADER = os.path.join(_build.INCLUDE, "specverify.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:spec_status_t|int|char|long long)\s*\*?\s*(\w+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("spec_mask_build", "spec_verify_attn", "spec_verify_attn_workspace_size",
              "spec_vocab_reduce", "spec_accept", "kv_commit", "spec_get_status",
              "spec_version", "spec_status_string", "spec_la_prefill_attn",
              "spec_accept_soft", "spec_draft_tree", "spec_prune_tree",
              "spec_stream_rotate_values", "spec_future_gather"):
        assert n in names
    assert set(names) == set(binding.EXPORTS) | set(n for n in names if n not in binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", _build.LIB], capture_output=True,
                             text=True).stdout
        for n in declared_functions():
            assert re.search(rf"\bT {n}$", out, flags=re.M), n


def test_version_and_strings_without_gpu(lib):
    lib.spec_version.restype = ctypes.c_int
    assert lib.spec_version() == 100
    lib.spec_status_string.restype = ctypes.c_char_p
    lib.spec_status_string.argtypes = [ctypes.c_int]
    assert lib.spec_status_string(0) == b"ok"
    assert b"device" in lib.spec_status_string(6)


def test_host_side_argument_errors_need_no_gpu():
    """Host-checkable errors return before any CUDA call."""
    binding.load_library()
    a = binding.attn_desc(2, 300, 4, 2, 64, binding.SPEC_F32)       # too many rows
    c = binding.KvDesc(binding.SPEC_KV_CONTIGUOUS, binding.SPEC_F32, 2, 64, None, None,
                       2, 16, 0, 0, 0, None)
    with pytest.raises(binding.SpecError) as e:
        binding.spec_verify_attn_workspace_size(a, c)
    assert e.value.code == 2
    a = binding.attn_desc(2, 4, 4, 3, 64, binding.SPEC_F32)         # Hq % Hkv != 0
    with pytest.raises(binding.SpecError) as e:
        binding.spec_verify_attn_workspace_size(a, c)
    assert e.value.code == 1
    a = binding.attn_desc(2, 4, 4, 2, 96, binding.SPEC_F32)         # head_dim 96
    with pytest.raises(binding.SpecError) as e:
        binding.spec_verify_attn_workspace_size(a, c)
    assert e.value.code == 2
    a = binding.attn_desc(2, 4, 4, 2, 64, binding.SPEC_F32)
    assert binding.spec_verify_attn_workspace_size(a, c) > 0


def test_struct_layout_matches_c():
    gcc = shutil.which("gcc") or shutil.which("cc")
    if not gcc:
        pytest.skip("no C compiler")
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "specverify.h"
#define F(T, m) printf("%s.%s %zu\n", #T, #m, offsetof(T, m))
int main(void) {
  printf("spec_kv_desc %zu\n", sizeof(spec_kv_desc));
  printf("spec_attn_desc %zu\n", sizeof(spec_attn_desc));
  printf("spec_accept_desc %zu\n", sizeof(spec_accept_desc));
  printf("spec_prefill_desc %zu\n", sizeof(spec_prefill_desc));
  printf("spec_soft_desc %zu\n", sizeof(spec_soft_desc));
  printf("spec_draft_desc %zu\n", sizeof(spec_draft_desc));
  printf("spec_prune_desc %zu\n", sizeof(spec_prune_desc));
  printf("spec_rotate_desc %zu\n", sizeof(spec_rotate_desc));
  F(spec_kv_desc, k); F(spec_kv_desc, batch); F(spec_kv_desc, page_table);
  F(spec_attn_desc, scale); F(spec_attn_desc, split_tokens);
  F(spec_accept_desc, tau); F(spec_accept_desc, path_cap);
  F(spec_prefill_desc, n_look); F(spec_prefill_desc, dtype); F(spec_prefill_desc, scale);
  F(spec_soft_desc, n_draft_rows); F(spec_soft_desc, path_cap); F(spec_soft_desc, temperature);
  F(spec_draft_desc, k); F(spec_draft_desc, vparent_rows);
  F(spec_prune_desc, threshold); F(spec_prune_desc, vparent_rows);
  F(spec_rotate_desc, gamma); F(spec_rotate_desc, eps);
  return 0;
}
'''
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write(src)
        subprocess.run([gcc, "-I", _build.INCLUDE, c, "-o", exe], check=True)
        out = dict(line.rsplit(" ", 1) for line in
                   subprocess.run([exe], capture_output=True, text=True).stdout.split("\n") if line)
    assert int(out["spec_kv_desc"]) == ctypes.sizeof(binding.KvDesc)
    assert int(out["spec_attn_desc"]) == ctypes.sizeof(binding.AttnDesc)
    assert int(out["spec_accept_desc"]) == ctypes.sizeof(binding.AcceptDesc)
    assert int(out["spec_prefill_desc"]) == ctypes.sizeof(binding.PrefillDesc)
    assert int(out["spec_soft_desc"]) == ctypes.sizeof(binding.SoftDesc)
    assert int(out["spec_draft_desc"]) == ctypes.sizeof(binding.DraftDesc)
    assert int(out["spec_prune_desc"]) == ctypes.sizeof(binding.PruneDesc)
    assert int(out["spec_rotate_desc"]) == ctypes.sizeof(binding.RotateDesc)
    for struct, cls in (("spec_kv_desc", binding.KvDesc), ("spec_attn_desc", binding.AttnDesc),
                        ("spec_accept_desc", binding.AcceptDesc),
                        ("spec_prefill_desc", binding.PrefillDesc),
                        ("spec_soft_desc", binding.SoftDesc),
                        ("spec_draft_desc", binding.DraftDesc),
                        ("spec_prune_desc", binding.PruneDesc),
                        ("spec_rotate_desc", binding.RotateDesc)):
        for key, val in out.items():
            if key.startswith(struct + "."):
                field = key.split(".")[1]
                assert getattr(cls, field).offset == int(val), key


def test_wait_limit_setter_round_trips_without_gpu():
    """spec_set_wait_limit only stores the limit later launches carry."""
    lib = binding.load_library()
    prev = binding.spec_set_wait_limit(12345)
    try:
        assert binding.spec_set_wait_limit(0) == 12345
        assert binding.spec_set_wait_limit(-1) == 0
        assert binding.spec_set_wait_limit(-1) == 2000000000   # the default restored
    finally:
        binding.spec_set_wait_limit(prev)
    assert lib is binding.load_library()


def test_host_side_errors_of_the_other_entry_points_need_no_gpu():
    """Descriptor and pointer checks of the draft, pruning, prefill, rotation,
    gather, vocabulary and mask entry points return before any CUDA call
    (the pointers below are never dereferenced on the host)."""
    lib = binding.load_library()
    BF, F32 = binding.SPEC_BF16, binding.SPEC_F32
    P = ctypes.c_void_p(0x1000)          # a 16-byte aligned address
    Pm = ctypes.c_void_p(0x1008)         # not 16-byte aligned
    N = None

    def draft(desc, ptrs=True, vp=None):
        args = [P] * 6 if ptrs else [N] * 6
        return lib.spec_draft_tree(ctypes.byref(desc) if desc is not None else None,
                                   args[0], None, args[1], args[2], args[3], args[4], vp, None)

    D = binding.DraftDesc
    assert draft(None) == 1
    assert draft(D(2, 3, 3, 9, 100, BF, 1000, 0)) == 2              # k above 8
    assert draft(D(2, 3, 3, 4, 100, 7, 1000, 0)) == 2               # logit dtype
    assert draft(D(2, 3, 3, 4, 100, BF, 84, 0)) == 4                # 85-node tree, 84 slots
    assert draft(D(2, 3, 3, 4, 100, BF, 85, 339), vp=P) == 4        # block rows 340 > 339
    assert draft(D(0, 3, 3, 4, 100, BF, 85, 0), ptrs=False) == 0    # empty batch
    assert draft(D(2, 3, 3, 4, 100, BF, 85, 0), ptrs=False) == 1    # NULL buffers

    def prune(desc, ptrs=True, vp=None):
        args = [P] * 8 if ptrs else [N] * 8
        return lib.spec_prune_tree(ctypes.byref(desc) if desc is not None else None,
                                   *args, vp, None)

    R = binding.PruneDesc
    assert prune(None) == 1
    assert prune(R(2, 85, 100, BF, float("nan"), 3, 340)) == 1      # NaN threshold
    assert prune(R(2, 1025, 100, BF, 0.1, 3, 4100)) == 2            # more than 1024 nodes
    assert prune(R(2, 85, 100, 7, 0.1, 3, 340)) == 2                # logit dtype
    assert prune(R(2, 85, 100, BF, 0.1, 3, 339), vp=P) == 4         # block rows too few
    assert prune(R(0, 85, 100, BF, 0.1, 3, 340), ptrs=False) == 0
    assert prune(R(2, 85, 100, BF, 0.1, 3, 340), ptrs=False) == 1

    def prefill(desc, q=P, k=P, v=P, o=P, lse=P):
        return lib.spec_la_prefill_attn(ctypes.byref(desc) if desc is not None else None,
                                        q, k, v, o, lse, None)

    F = binding.PrefillDesc
    assert prefill(None) == 1
    assert prefill(F(1, 0, 4, 8, 8, 128, BF, 0.0)) == 1             # no original positions
    assert prefill(F(1, 64, 4, 8, 3, 128, BF, 0.0)) == 1            # Hq % Hkv != 0
    assert prefill(F(1, 64, 4, 8, 8, 64, BF, 0.0)) == 2             # head_dim 64
    assert prefill(F(1, 64, 4, 8, 8, 128, F32, 0.0)) == 2           # fp32
    assert prefill(F(0, 64, 4, 8, 8, 128, BF, 0.0), N, N, N, N, N) == 0
    assert prefill(F(1, 64, 4, 8, 8, 128, BF, 0.0), N, N, N, N, N) == 1
    assert prefill(F(1, 64, 4, 8, 8, 128, BF, 0.0), q=Pm) == 1      # q off 16 bytes

    Rt = binding.RotateDesc
    rot = lambda d, nn=P, vb=P: lib.spec_stream_rotate_values(ctypes.byref(d), nn, vb, None)
    assert lib.spec_stream_rotate_values(None, P, P, None) == 1
    assert rot(Rt(2, 16, 4, 12, BF, 3, 0.01)) == 2                  # head_dim not a multiple of 8
    assert rot(Rt(2, 16, 4, 128, BF, 3, float("nan"))) == 1         # NaN angle
    assert rot(Rt(2, 16, 4, 128, BF, 3, 0.01), vb=Pm) == 1          # block off 16 bytes
    assert rot(Rt(0, 16, 4, 128, BF, 3, 0.01), N, N) == 0

    g = lib.spec_future_gather
    assert g(2, 8, 100, BF, P, P, 0, P, None) == 2                  # 200-byte rows
    assert g(2, 8, 12, BF, P, P, 0, P, None) == 2                   # 24-byte rows
    assert g(2, 8, 128, 7, P, P, 0, P, None) == 2                   # dtype
    assert g(2, 8, 128, BF, P, P, -1, P, None) == 1                 # negative offset
    assert g(0, 8, 128, BF, N, N, 0, N, None) == 0
    assert g(2, 8, 128, BF, Pm, P, 0, P, None) == 1                 # O off 16 bytes

    v = lib.spec_vocab_reduce
    assert v(P, BF, 4, 0, N, P, P, N, None) == 1                    # empty vocabulary
    assert v(P, 7, 4, 100, N, P, P, N, None) == 2                   # dtype
    assert v(P, BF, 4, 100, P, P, P, N, None) == 1                  # proposal without zprop
    assert v(N, BF, 0, 100, N, N, N, N, None) == 0

    m = lib.spec_mask_build
    assert m(P, N, 2, 0, P, P, None) == 1                           # no rows
    assert m(P, N, 2, 257, P, P, None) == 2                         # above SPEC_MAX_ROWS
    assert m(N, N, 0, 8, N, N, None) == 0
    assert m(N, N, 2, 8, P, P, None) == 1                           # NULL parents


def test_host_side_errors_of_acceptance_and_commit_need_no_gpu():
    """The same for spec_accept, spec_accept_soft and kv_commit."""
    lib = binding.load_library()
    BF = binding.SPEC_BF16
    CH, TR = binding.SPEC_ACCEPT_THRESH_CHAIN, binding.SPEC_ACCEPT_GREEDY_TREE
    P = ctypes.c_void_p(0x1000)
    N = None

    def acc(d, logits=P, tokens=P, parent=P, row_of=N, zprop=P):
        return lib.spec_accept(ctypes.byref(d) if d is not None else None, logits, tokens,
                               parent, row_of, P, P, P, zprop, P, P, P, P, None)

    A = binding.AcceptDesc
    assert acc(None) == 1
    assert acc(A(5, 0.3, 2, 8, 100, BF, 8, 8)) == 1                 # unknown mode
    assert acc(A(CH, 0.3, 2, 0, 100, BF, 8, 8)) == 1                # no judged rows
    assert acc(A(CH, 0.0, 2, 8, 100, BF, 8, 8)) == 1                # tau not in (0, 1]
    assert acc(A(CH, 0.3, 2, 8, 100, BF, 8, 8), row_of=P) == 1      # chains take no row map
    assert acc(A(CH, 0.3, 2, 8, 100, BF, 6, 8)) == 1                # proposals != judged rows
    assert acc(A(TR, 0.0, 2, 8, 100, BF, 300, 8)) == 2              # tree above 256 nodes
    assert acc(A(TR, 0.0, 2, 8, 100, BF, 8, 8), parent=N) == 1      # tree without parents
    assert acc(A(TR, 0.0, 2, 8, 0, BF, 8, 8)) == 1                  # empty vocabulary
    assert acc(A(TR, 0.0, 2, 8, 100, 7, 8, 8)) == 2                 # logit dtype
    assert acc(A(TR, 0.0, 0, 8, 100, BF, 8, 8), logits=N, tokens=N, parent=N) == 0

    def soft(d, draft=P):
        return lib.spec_accept_soft(ctypes.byref(d) if d is not None else None, P, draft, P, P,
                                    N, P, P, P, P, P, P, P, P, P, P, None)

    S = binding.SoftDesc
    assert soft(None) == 1
    assert soft(S(2, 8, 4, 100, BF, 8, 8, 0.0)) == 1                # temperature 0
    assert soft(S(2, 8, 4, 100, BF, 8, 8, float("inf"))) == 1       # infinite temperature
    assert soft(S(2, 8, 4, 100, 7, 8, 8, 1.0)) == 2                 # logit dtype
    assert soft(S(2, 8, 4, (1 << 20) + 1, BF, 8, 8, 1.0)) == 2      # vocabulary above 2^20
    assert soft(S(2, 8, 4, 100, BF, 300, 8, 1.0)) == 2              # tree above 256 nodes
    assert soft(S(2, 8, 4, 100, BF, 8, 8, 1.0), draft=N) == 1       # draft rows without logits
    assert soft(S(0, 8, 4, 100, BF, 8, 8, 1.0), draft=N) == 0

    K = binding.KvDesc
    com = lambda c, batch=2: lib.kv_commit(ctypes.byref(c) if c is not None else None, batch, 8,
                                           P, P, 8, P, P, P, N, 0, N, None)
    kv = lambda dt=BF, d=128, kind=binding.SPEC_KV_CONTIGUOUS, B=2: K(kind, dt, 4, d, P, P, B, 64,
                                                                     0, 0, 0, N)
    assert com(None) == 1
    assert com(kv(dt=7)) == 2                                       # dtype
    assert com(kv(d=12)) == 2                                       # 24-byte rows
    assert com(kv(d=96, kind=binding.SPEC_KV_PAGED)) == 2           # paged head_dim not 64k
    assert com(kv(B=1)) == 1                                        # cache holds fewer requests
    assert com(kv(), batch=0) == 0
