"""Error handling on the GPU, with no fault: host-checkable errors return a
code before any launch; device-detected errors (bad parent pointers, page
ids, lengths, full caches, short paths) set status bits that
spec_get_status reads and clears, and the kernels skip the offending work."""

import numpy as np
import pytest
import torch

import gpu_helpers as gh
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300 import workloads as W
from self_speculative_verification_gb300.device import DeviceStep

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    gh.require_gpu()
    bn.spec_get_status()          # start from a clear status word


def small(name="long_paged", **kw):
    base = dict(B=3, seq=("uniform", 100, 300), V=1000)
    base.update(kw)
    return DeviceStep(W.make_workload(name, 31, **base))


def test_status_is_read_and_cleared():
    ds = small()
    ds.run()
    assert bn.spec_get_status() == 0
    ds.vparent[0, 1] = 5                       # parent after the row itself
    ds.mask_build()
    assert bn.spec_get_status() == bn.SPEC_DEV_BAD_TREE
    assert bn.spec_get_status() == 0           # cleared by the read


def test_bad_parent_rows_are_masked_out():
    ds = small("confu", B=2)
    ds.vparent[1, 3] = 3                       # self-parent
    ds.vparent[1, 70] = 119                    # forward parent (contemplate row)
    ds.mask_build()
    assert bn.spec_get_status() & bn.SPEC_DEV_BAD_TREE
    fl = ds.row_flags.cpu().numpy()
    assert fl[1, 3] == 0 and fl[1, 70] == 0
    assert np.all(ds.vis[1, 3].cpu().numpy() == 0)
    # rows whose chains do not pass through a bad row are untouched
    assert fl[0].min() >= 1


def test_seq_len_over_capacity_is_clamped_and_flagged():
    ds = small()
    ds.mask_build()
    ds.seq_len[1] = 10 ** 8
    ds.verify_attn()
    assert bn.spec_get_status() & bn.SPEC_DEV_SEQ_OVERFLOW


def test_bad_page_id_is_flagged():
    ds = small()
    ds.mask_build()
    ds.page_table[2, 1] = ds.wl.n_pages + 7
    ds.verify_attn()
    assert bn.spec_get_status() & bn.SPEC_DEV_BAD_PAGE


def test_commit_with_exhausted_free_list_writes_nothing():
    wl = W.make_workload("long_paged", 32, B=4, seq=(16, 32, 48, 64), V=1000)
    ds = DeviceStep(wl)                      # every request page aligned: needs a new page
    ds.free_head.fill_(int(wl.free_pages.size) - 1)    # one free page left
    k0 = ds.k_cache.clone()
    seq0 = ds.seq_len.clone()
    ds.mask_build()
    ds.verify_attn()
    ds.accept_step()
    assert int((ds.acc_len > 0).sum()) >= 2
    ds.commit()
    assert bn.spec_get_status() & bn.SPEC_DEV_CAPACITY
    assert torch.equal(ds.k_cache.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(ds.seq_len, seq0)
    assert int(ds.free_head.item()) == int(wl.free_pages.size) - 1


def test_commit_over_contiguous_capacity_skips_that_request():
    wl = W.make_workload("la7b", 33, B=3, seq=(50, 60, 70), V=1000, k_choices=(8,))
    ds = DeviceStep(wl)
    ds.mask_build()
    ds.verify_attn()
    ds.accept_step()
    acc = ds.acc_len.cpu().numpy()
    ds.seq_len[1] = wl.max_seq - 1             # request 1 has room for one row only
    acc[1] = max(acc[1], 2)
    ds.acc_len.copy_(torch.from_numpy(acc).to(ds.acc_len.device))
    ds.path[1, :2] = torch.tensor([0, 1], dtype=torch.int32)
    seq_before = ds.seq_len.cpu().numpy().copy()
    ds.commit()
    assert bn.spec_get_status() & bn.SPEC_DEV_CAPACITY
    seq_after = ds.seq_len.cpu().numpy()
    assert seq_after[1] == seq_before[1]                      # skipped
    assert seq_after[0] == seq_before[0] + acc[0]             # others committed
    assert seq_after[2] == seq_before[2] + acc[2]


def test_short_path_capacity_is_flagged():
    wl = W.make_workload("confu", 34, B=2, seq=("uniform", 50, 90), V=1000)
    ds = DeviceStep(wl)
    assert wl.expect_acc_len.max() > 1
    ds.accept.path_cap = 1
    ds.path = torch.zeros((wl.B, 1), dtype=torch.int32, device=ds.device)
    ds.accept_step()
    assert bn.spec_get_status() & bn.SPEC_DEV_BAD_INDEX
    assert ds.acc_len.max().item() == 1


def test_n_nodes_out_of_range_is_flagged():
    ds = small("la7b")
    ds.n_nodes[0] = 99
    ds.accept_step()
    assert bn.spec_get_status() & bn.SPEC_DEV_BAD_INDEX


def test_host_errors_launch_nothing():
    ds = small()
    with pytest.raises(bn.SpecError) as e:                    # workspace too small
        bn.spec_verify_attn(ds.attn, ds.q, ds.cache, ds.kb, ds.vb, None, None, ds.seq_len,
                            ds.vis, ds.row_flags, ds.o, ds.lse, ds.workspace[:256])
    assert e.value.code == 4
    with pytest.raises(bn.SpecError) as e:                    # misaligned workspace
        bn.spec_verify_attn(ds.attn, ds.q, ds.cache, ds.kb, ds.vb, None, None, ds.seq_len,
                            ds.vis, ds.row_flags, ds.o, ds.lse, ds.workspace[16:])
    assert e.value.code == 1
    lib = bn.load_library()
    assert lib.spec_mask_build(None, None, 2, 8, None, None, None) == 1
    assert lib.spec_mask_build(None, None, 2, 300, None, None, None) == 2
    d = bn.accept_desc(bn.SPEC_ACCEPT_THRESH_CHAIN, 1.5, 2, 8, 100, bn.SPEC_BF16, 8, 8)
    assert lib.spec_accept(d, None, *([None] * 12)) == 1
    assert bn.spec_get_status() == 0                          # nothing ran
