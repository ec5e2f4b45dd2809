"""spec_vocab_reduce against the oracle's row reduction: exact argmax
(lowest index on exact ties), LSE to 1e-5 relative, the proposal's logit
bit-exact; row lengths that break 16-byte alignment take the scalar path;
large and small row counts exercise 1..8 CTAs per row, and aligned bf16
rows the bulk-copy stream (full chunks, a ragged last chunk, one vector per
row, the full ConFu and SS row counts)."""

import numpy as np
import pytest
import torch

import gpu_helpers as gh
import oracle
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300.workloads import round_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,V", [(3, 7), (5, 1001), (17, 1000), (8, 32000), (480, 8191),
                                    (64, 128256), (2, 50272), (480, 128256), (512, 50272),
                                    (1000, 8), (300, 4104)])
def test_vocab_reduce_matches_oracle(dtype, rows, V):
    gh.require_gpu()
    rng = np.random.Generator(np.random.PCG64(rows * 7 + V))
    z = (rng.standard_normal((rows, V), dtype=np.float32) * 3).astype(np.float32)
    if dtype == "bf16":
        z = round_bf16(z)
    # exact ties at the maximum in some rows: the lowest index must win
    for r in range(0, rows, 3):
        a, b = sorted(rng.choice(V, size=2, replace=False)) if V > 1 else (0, 0)
        z[r, a] = z[r, b] = z[r].max() + 1.0
    if dtype == "bf16":
        # the tied maxima too must be bf16 values (past 16 the spacing is 1/8)
        z = round_bf16(z)
    prop = rng.integers(0, V, size=rows).astype(np.int32)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dz = torch.from_numpy(z).cuda().to(tdt)
    dp = torch.from_numpy(prop).cuda()
    am = torch.empty(rows, dtype=torch.int32, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    zp = torch.empty(rows, dtype=torch.float32, device="cuda")
    bn.spec_vocab_reduce(dz, dp, am, lse, zp)
    torch.cuda.synchronize()
    am_o, lse_o, zp_o = oracle.vocab_reduce(z, prop)
    assert am.cpu().numpy().tolist() == am_o.tolist()
    rel = np.abs(lse.cpu().numpy().astype(np.float64) - lse_o) / np.abs(lse_o)
    assert rel.max() <= 1e-5
    assert np.array_equal(zp.cpu().numpy().astype(np.float64), zp_o)


def test_vocab_reduce_unaligned_rows_bf16():
    """bf16 logits whose first row starts 2 bytes past a 16-byte boundary
    take the plain-load kernel; the results are the same reduction."""
    gh.require_gpu()
    rows, V = 40, 50272
    rng = np.random.Generator(np.random.PCG64(99))
    z = round_bf16((rng.standard_normal((rows, V), dtype=np.float32) * 3).astype(np.float32))
    prop = rng.integers(0, V, size=rows).astype(np.int32)
    flat = torch.empty(rows * V + 8, dtype=torch.bfloat16, device="cuda")
    dz = flat[1:1 + rows * V].view(rows, V)
    dz.copy_(torch.from_numpy(z).cuda().to(torch.bfloat16))
    assert dz.data_ptr() % 16 == 2
    dp = torch.from_numpy(prop).cuda()
    am = torch.empty(rows, dtype=torch.int32, device="cuda")
    lse = torch.empty(rows, dtype=torch.float32, device="cuda")
    zp = torch.empty(rows, dtype=torch.float32, device="cuda")
    bn.spec_vocab_reduce(dz, dp, am, lse, zp)
    torch.cuda.synchronize()
    am_o, lse_o, zp_o = oracle.vocab_reduce(z, prop)
    assert am.cpu().numpy().tolist() == am_o.tolist()
    rel = np.abs(lse.cpu().numpy().astype(np.float64) - lse_o) / np.abs(lse_o)
    assert rel.max() <= 1e-5
    assert np.array_equal(zp.cpu().numpy().astype(np.float64), zp_o)
