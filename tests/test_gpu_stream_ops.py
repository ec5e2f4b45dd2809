"""GPU parity of the stream value rotation ("Speculative Streaming" Eq. 7)
and of the ConFu future-token gather against the oracle."""

import math

import numpy as np
import pytest
import torch

import gpu_helpers as gh
import oracle
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def _gpu():
    gh.require_gpu()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("eps", [0.3, 1e-3])
def test_rotation_kernel(dtype, eps):
    rng = np.random.Generator(np.random.PCG64(11))
    B, H, R, d, gamma = 4, 3, 70, 128, 3
    n = np.array([16, 5, 1, 17], dtype=np.int32)            # 17 * 4 = 68 <= 70
    vb = rng.standard_normal((B, H, R, d)).astype(np.float32) / 8
    if dtype == "bf16":
        vb = W.round_bf16(vb)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    v = torch.from_numpy(vb).to(DEV, tdt)
    desc = bn.RotateDesc(B, R, H, d, bn.SPEC_BF16 if dtype == "bf16" else bn.SPEC_F32, gamma,
                         eps)
    bn.spec_stream_rotate_values(desc, torch.from_numpy(n).to(DEV), v)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    got = v.float().cpu().numpy().astype(np.float64)
    want = oracle.rotate_stream_values(vb, n, gamma, eps)
    # bf16: the kernel rounds an fp32 result once (half an ulp, 2^-9 relative)
    rel = 2.0 ** -8 if dtype == "bf16" else 2e-6
    assert np.all(np.abs(got - want) <= rel * np.abs(want) + 1e-7)
    for b in range(B):
        T = n[b]
        keep = list(range(T)) + list(range(T * (1 + gamma), R))
        assert np.array_equal(got[b][:, keep], vb[b][:, keep].astype(np.float64))


@pytest.mark.parametrize("eps", [None, 0.25])
def test_ss_rotation_step_parity(eps):
    """The whole SS step with stream values by rotation: the page's eps
    bound, and a large angle so the rotation shows in the outputs."""
    wl = W.make_workload("ss_rot", 2, B=3, seq=("uniform", 100, 500), V=5000)
    if eps is not None:
        wl.rotation_eps = eps
    gh.run_and_check(wl)


def test_rotation_bad_request_is_skipped():
    B, H, R, d = 2, 1, 10, 8
    v = torch.ones((B, H, R, d), dtype=torch.float32, device=DEV)
    n = torch.tensor([2, 3], dtype=torch.int32, device=DEV)       # 3 * 4 = 12 > 10
    bn.spec_stream_rotate_values(bn.RotateDesc(B, R, H, d, bn.SPEC_F32, 3, 0.5), n, v)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == bn.SPEC_DEV_BAD_INDEX
    assert torch.all(v[1] == 1.0)


def test_future_gather_and_bad_rows():
    rng = np.random.Generator(np.random.PCG64(12))
    o = torch.from_numpy(rng.standard_normal((3, 20, 4, 8)).astype(np.float32)).to(DEV,
                                                                                     torch.bfloat16)
    out = torch.full((3, 4, 8), 7.0, dtype=torch.bfloat16, device=DEV)
    last = torch.tensor([0, 9, 3], dtype=torch.int32, device=DEV)
    bn.spec_future_gather(o, last, 10, out)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    want = oracle.future_gather(o.float().cpu().numpy(), last.cpu().numpy(), 10)
    assert np.array_equal(out.float().cpu().numpy(), want)
    bad = torch.tensor([0, 10, -1], dtype=torch.int32, device=DEV)
    bn.spec_future_gather(o, bad, 10, out)
    torch.cuda.synchronize()
    assert bn.spec_get_status() == bn.SPEC_DEV_BAD_INDEX
    assert torch.all(out[1] == 0) and torch.all(out[2] == 0)
    assert np.array_equal(out[0].float().cpu().numpy(), o[0, 10].float().cpu().numpy())
