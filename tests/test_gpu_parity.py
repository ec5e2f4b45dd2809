"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle
on identical seeded inputs.  Sizes here let the oracle finish in seconds
while still spanning several tiles, several splits and ragged tails."""

import numpy as np
import pytest
import torch

import gpu_helpers as gh
from self_speculative_verification_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    gh.require_gpu()


SMALL = {
    "tiny_la": {},
    "la7b": dict(B=3, seq=("uniform", 100, 700), V=4000),
    "confu": dict(B=2, seq=("uniform", 150, 600), V=5000),
    "ss": dict(B=3, seq=("uniform", 100, 500), V=5000),
    "long_paged": dict(B=3, seq=("uniform", 300, 1100), V=4000),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("seed", [0, 1])
def test_step_parity_small(name, seed):
    wl = W.make_workload(name, seed, **SMALL[name])
    gh.run_and_check(wl)


@pytest.mark.parametrize("name", ["la7b", "confu", "ss", "long_paged"])
def test_step_parity_many_splits(name):
    """Force 64-token splits so the combine merges many partials."""
    wl = W.make_workload(name, 5, **SMALL[name])
    gh.run_and_check(wl, split_tokens=64)


@pytest.mark.parametrize("name", ["la7b", "confu", "ss", "long_paged"])
def test_step_parity_sharp_softmax(name):
    """Queries scaled up 16x so the softmax is far from uniform."""
    wl = W.make_workload(name, 7, q_scale=16.0, **SMALL[name])
    gh.run_and_check(wl)


@pytest.mark.parametrize("name,seq", [
    ("la7b", (0, 1, 63, 64)),
    ("long_paged", (0, 16, 17, 64)),
    ("confu", (0, 65)),
    ("ss", (1, 128)),
])
def test_edge_prefix_lengths(name, seq):
    """Empty prefixes, one token, page- and tile-aligned lengths."""
    kw = dict(SMALL[name])
    kw["B"] = len(seq)
    kw["seq"] = seq
    wl = W.make_workload(name, 3, **kw)
    gh.run_and_check(wl)


def test_single_row_blocks():
    wl = W.make_workload("la7b", 4, B=4, seq=("uniform", 50, 300), V=3000, k_choices=(1,))
    gh.run_and_check(wl)


def test_small_tree_sizes():
    for T in (1, 2, 7):
        wl = W.make_workload("confu", 8 + T, B=2, seq=("uniform", 30, 90), V=2000, T=T)
        gh.run_and_check(wl)
        wl = W.make_workload("ss", 8 + T, B=2, seq=("uniform", 30, 90), V=2000, T=T)
        gh.run_and_check(wl)


def test_repeat_step_is_deterministic():
    """Running the same step twice (state restored) gives identical bits."""
    wl = W.make_workload("long_paged", 2, **SMALL["long_paged"])
    ds, _ = gh.run_and_check(wl)
    o1, l1 = ds.o.clone(), ds.lse.clone()
    k1 = ds.k_cache.clone()
    ds.reset_state(page_table=True)
    ds.run()
    torch.cuda.synchronize()
    assert torch.equal(ds.o.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(ds.lse, l1)
    assert torch.equal(k1.view(torch.int16), ds.k_cache.view(torch.int16))
