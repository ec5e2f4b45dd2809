"""Bounded pipeline waits.  With the wait limit set to 0 cycles, any wait of
the tensor-core kernels (or of the vocabulary reduction's row stream) whose
condition is not met at its first test gives up at once: the kernel must
report SPEC_DEV_TIMEOUT, stop, drain its own copies and tensor-core
operations, free its tensor memory and return, so the context stays usable.  The workloads are sized so that every CTA has more
tiles than its stage ring holds (a producer waiting for a stage to be
released cannot find it free at the first test).  After each case the
default limit is restored and a full step on the same process must match the
oracle."""

import numpy as np
import pytest
import torch

import gpu_helpers as gh
import oracle
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300 import workloads as W
from self_speculative_verification_gb300.device import DeviceStep
from self_speculative_verification_gb300.workloads import round_bf16

pytestmark = pytest.mark.gpu

# (workload, generator arguments): the mma.sync kernel (32 packed rows per KV
# head, paged cache) and the tcgen05 kernel (64 and 480 packed rows)
CASES = [
    ("long_paged", dict(B=8, seq=("uniform", 4000, 6000), V=2000)),
    ("ss", dict(B=4, seq=("uniform", 2000, 4000), V=2000)),
    ("confu", dict(B=4, seq=("uniform", 2000, 4000), V=2000)),
]

SMALL = {
    "long_paged": dict(B=3, seq=("uniform", 300, 900), V=3000),
    "ss": dict(B=2, seq=("uniform", 100, 400), V=3000),
    "confu": dict(B=2, seq=("uniform", 150, 500), V=3000),
}


@pytest.mark.parametrize("name,kw", CASES)
def test_verify_wait_runs_out_and_context_recovers(name, kw):
    gh.require_gpu()
    wl = W.make_workload(name, 5, **kw)
    ds = DeviceStep(wl)
    ds.mask_build()
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    bn.spec_set_wait_limit(0)
    try:
        ds.verify_attn()
        torch.cuda.synchronize()
    finally:
        bn.spec_set_wait_limit(-1)
    status = bn.spec_get_status()
    assert status & bn.SPEC_DEV_TIMEOUT, f"status {status:#x}"
    # the same process, default limit: a whole step matches the oracle
    gh.run_and_check(W.make_workload(name, 6, **SMALL[name]))


def test_prefill_wait_runs_out_and_context_recovers():
    gh.require_gpu()
    from test_gpu_la_prefill import check, run_gpu
    wl = W.make_prefill(seed=41, B=2, n=2048, k=8, Hq=8, Hkv=8)
    dev = torch.device("cuda", 0)
    q, k, v = (torch.from_numpy(a).to(dev, torch.bfloat16) for a in (wl.q, wl.kk, wl.v))
    o = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.Hq, wl.L), dtype=torch.float32, device=dev)
    desc = bn.prefill_desc(wl.B, wl.n, wl.k, wl.Hq, wl.Hkv, wl.d)
    bn.spec_set_wait_limit(0)
    try:
        bn.spec_la_prefill_attn(desc, q, k, v, o, lse)
        torch.cuda.synchronize()
    finally:
        bn.spec_set_wait_limit(-1)
    status = bn.spec_get_status()
    assert status & bn.SPEC_DEV_TIMEOUT, f"status {status:#x}"
    # the default limit again: the same call matches the oracle on sampled
    # (request, head) slices
    O, LSE = run_gpu(wl)
    check(wl, O, LSE, pairs=[(0, 0), (1, 5)])


def test_vocab_stream_wait_runs_out_and_context_recovers():
    """bf16 rows on 16-byte boundaries take the bulk row stream, whose chunk
    waits are bounded by the same limit: at 0 the first chunk, tested right
    after its copy was issued, has not landed."""
    gh.require_gpu()
    rows, V = 64, 128256
    rng = np.random.Generator(np.random.PCG64(77))
    z = round_bf16((rng.standard_normal((rows, V), dtype=np.float32) * 3).astype(np.float32))
    prop = rng.integers(0, V, size=rows).astype(np.int32)
    dev = torch.device("cuda", 0)
    dz = torch.from_numpy(z).to(dev, torch.bfloat16)
    dp = torch.from_numpy(prop).to(dev)
    am = torch.empty(rows, dtype=torch.int32, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    zp = torch.empty(rows, dtype=torch.float32, device=dev)
    assert bn.spec_get_status() == 0
    bn.spec_set_wait_limit(0)
    try:
        bn.spec_vocab_reduce(dz, dp, am, lse, zp)
        torch.cuda.synchronize()
    finally:
        bn.spec_set_wait_limit(-1)
    status = bn.spec_get_status()
    assert status & bn.SPEC_DEV_TIMEOUT, f"status {status:#x}"
    # the default limit again: the same call matches the oracle
    bn.spec_vocab_reduce(dz, dp, am, lse, zp)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    am_o, lse_o, zp_o = oracle.vocab_reduce(z, prop)
    assert am.cpu().numpy().tolist() == am_o.tolist()
    rel = np.abs(lse.cpu().numpy().astype(np.float64) - lse_o) / np.abs(lse_o)
    assert rel.max() <= 1e-5
    assert np.array_equal(zp.cpu().numpy().astype(np.float64), zp_o)
