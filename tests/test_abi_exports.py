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
