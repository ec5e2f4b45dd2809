"""spec_verify_attn_noalloc: the attention entry point for callers that
cannot allocate device memory (an engine that reserved all GPU memory for its
own KV-cache pool, a plugin hook that may not allocate while it runs).  It
must give the same results as spec_verify_attn with a caller workspace, on
consecutive calls that reuse the library's one scratch array.

Both entry points run the same plan and kernels on the same inputs, so their
outputs must agree bit for bit; before the compared calls another no-alloc
call of a different shape leaves other data in the scratch, so a kernel that
read a stale partial would show.

This file is collected last so that a run stopping at the first failure has
already run every other test."""

import pytest
import torch

import gpu_helpers as gh
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300 import workloads as W
from self_speculative_verification_gb300.device import DeviceStep

pytestmark = pytest.mark.gpu

CASES = [
    ("long_paged", dict(B=3, seq=("uniform", 300, 1100), V=4000)),
    ("confu", dict(B=2, seq=("uniform", 150, 600), V=5000)),
    ("ss", dict(B=3, seq=("uniform", 200, 700), V=3000)),
    ("tiny_la", {}),
]

# a shape unlike every case above, run through the no-alloc entry point first
FILLER = ("confu", dict(B=3, seq=("uniform", 700, 1500), V=3000))


def noalloc(ds):
    bn.spec_verify_attn_noalloc(ds.attn, ds.q, ds.cache, ds.kb, ds.vb, ds.soft_k, ds.soft_v,
                                ds.seq_len, ds.vis, ds.row_flags, ds.o, ds.lse)


@pytest.mark.parametrize("name,kw", CASES)
def test_noalloc_matches_workspace_entry_point(name, kw):
    gh.require_gpu()
    filler = DeviceStep(W.make_workload(FILLER[0], 13, **FILLER[1]))
    filler.mask_build()
    noalloc(filler)                        # other data in the scratch
    wl = W.make_workload(name, 11, **kw)
    ds = DeviceStep(wl)
    ds.mask_build()
    ds.verify_attn()                       # reference: caller workspace
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    o_ref, lse_ref = ds.o.clone(), ds.lse.clone()
    vis, valid, sees = gh.check_mask(ds)
    O_or, L_or = gh.oracle_attention(wl, vis, valid, sees)
    for call in range(2):                  # two calls in a row share the scratch
        ds.o.fill_(float("nan"))
        ds.lse.fill_(float("nan"))
        noalloc(ds)
        torch.cuda.synchronize()
        assert bn.spec_get_status() == 0
        assert torch.equal(ds.o, o_ref), f"call {call}: O differs from the workspace entry point"
        assert torch.equal(ds.lse, lse_ref), f"call {call}: LSE differs"
        gh.check_attention(ds, O_or, L_or)  # and against the oracle


def test_noalloc_rejects_shapes_beyond_its_scratch():
    gh.require_gpu()
    wl = W.make_workload("ss", 12, B=2, seq=("uniform", 30, 60), V=500)
    ds = DeviceStep(wl)
    big = bn.attn_desc(4000, 64, 32, 32, 128, bn.SPEC_BF16)
    k = torch.empty((4000, 32, 1, 128), dtype=torch.bfloat16, device="cuda")
    cache = bn.kv_desc_contiguous(k, k)
    assert bn.spec_verify_attn_workspace_size(big, cache) > bn.SPEC_NOALLOC_SCRATCH_BYTES
    with pytest.raises(bn.SpecError) as e:
        bn.spec_verify_attn_noalloc(big, ds.q, cache, ds.kb, ds.vb, None, None, ds.seq_len,
                                    ds.vis, ds.row_flags, ds.o, ds.lse)
    assert e.value.code == bn.SPEC_ERR_CAPACITY
