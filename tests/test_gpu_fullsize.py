"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (library-chosen splits): the mask, the vocab reduce, the
acceptance and the commit in full, the attention on sampled (request, head)
pairs that the oracle computes one by one."""

import numpy as np
import pytest
import torch

import gpu_helpers as gh
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300 import workloads as W
from self_speculative_verification_gb300.device import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["la7b", "confu", "ss", "long_paged"])
def test_full_size_sampled(name):
    gh.require_gpu()
    wl = W.make_workload(name, 0)
    ds = DeviceStep(wl, threads=16)
    k0, v0 = ds.k_cache.clone(), ds.v_cache.clone()
    ds.run()
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    vis, valid, sees = gh.check_mask(ds)
    reqs = sorted({0, wl.B // 2, wl.B - 1})
    heads = sorted({0, wl.Hq // 2 + 1, wl.Hq - 1})
    O_ref, L_ref = gh.oracle_attention(wl, vis, valid, sees, requests=reqs, heads=heads)
    gh.check_attention(ds, O_ref, L_ref, requests=reqs, heads=heads)
    acc, paths = gh.check_accept(ds)
    # commit: the oracle's commit gives every slot's source row; the whole
    # cache is then compared bit for bit on the device
    ek, ev, pt, seq2, head = gh.commit_expected_on_device(ds, k0, v0, paths)
    if wl.paged:
        assert np.array_equal(ds.page_table.cpu().numpy(), pt)
        assert int(ds.free_head.item()) == head
    assert torch.equal(ds.k_cache.view(torch.int16), ek.view(torch.int16))
    assert torch.equal(ds.v_cache.view(torch.int16), ev.view(torch.int16))
    assert ds.seq_len.cpu().numpy().tolist() == seq2.tolist()
