"""GPU parity for the kernel variants the five workloads do not reach:
head_dim 64 on the tensor-core path (16-, 32- and 64-row tiles), 32- and
64-token pages, and fp32 inputs (CUDA-core path) on tree, soft-prompt and
paged workloads."""

import pytest

import gpu_helpers as gh
from self_speculative_verification_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    gh.require_gpu()


@pytest.mark.parametrize("name,kw", [
    ("la7b", dict(B=3, seq=("uniform", 100, 700), V=3000, d=64)),
    ("long_paged", dict(B=3, seq=("uniform", 200, 900), V=3000, d=64)),
    ("ss", dict(B=2, seq=("uniform", 100, 400), V=3000, d=64)),
    ("confu", dict(B=2, seq=("uniform", 100, 400), V=3000, d=64)),
])
def test_head_dim_64_bf16(name, kw):
    gh.run_and_check(W.make_workload(name, 21, **kw))


@pytest.mark.parametrize("page_size", [32, 64])
@pytest.mark.parametrize("d", [64, 128])
def test_page_sizes(page_size, d):
    wl = W.make_workload("long_paged", 22, B=3, seq=("uniform", 150, 700), V=3000,
                         page_size=page_size, d=d)
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)


@pytest.mark.parametrize("name", ["ss", "confu", "long_paged", "la7b"])
def test_fp32_cuda_core_path(name):
    wl = W.make_workload(name, 23, B=2, seq=("uniform", 60, 300), V=2000, dtype="f32")
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)


def test_gqa_many_row_blocks():
    """ConFu rows (120 x G=4 = 480 packed rows) over several row blocks,
    with sharpened scores."""
    wl = W.make_workload("confu", 24, B=3, seq=("uniform", 500, 1300), V=2000,
                         q_scale=8.0)
    gh.run_and_check(wl)


@pytest.mark.parametrize("name", ["ss", "confu"])
@pytest.mark.parametrize("page_size", [16, 32, 64])
def test_many_rows_on_paged_cache(name, page_size):
    """>= 64 packed rows per KV head (the tcgen05 kernel) on paged caches:
    one MMA per page block for S, V fetched per page block for PV."""
    wl = W.make_workload(name, 25, B=2, seq=("uniform", 150, 700), V=2000, paged=True,
                         page_size=page_size)
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)


@pytest.mark.parametrize("paged", [False, True])
def test_split_row_layout_gqa(paged):
    """64 packed rows with G = 4 (a ConFu tree of 8 nodes: 16 rows x 4
    heads): the tcgen05 kernel's heads mode with two KV heads' rows in one
    query block (query boxes of 16 rows x 4 heads, the second head's rows in
    TMEM lanes 64..127)."""
    wl = W.make_workload("confu", 26, B=3, T=8, seq=("uniform", 150, 900), V=2000,
                         paged=paged)
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)


def test_partial_row_block():
    """96 packed rows (a ConFu tree of 12 nodes, G = 4): one tcgen05 row
    block, its last 32 lanes empty."""
    wl = W.make_workload("confu", 27, B=3, T=12, seq=("uniform", 150, 900), V=2000)
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)


@pytest.mark.parametrize("T", [20, 40])
def test_row_block_pairs(T):
    """The tcgen05 kernel's rows mode: 160 packed rows (two row blocks, one
    unit) and 320 (three row blocks: a unit of two, then a unit whose second
    tile is absent), on ConFu trees of 20 and 40 nodes (G = 4)."""
    wl = W.make_workload("confu", 28, B=3, T=T, seq=("uniform", 150, 900), V=2000)
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)


@pytest.mark.parametrize("name,kw", [
    ("ss", dict(Hq=5, Hkv=5)),              # 64 packed rows, heads share a query block
    ("confu", dict(T=12, Hq=12, Hkv=3)),    # 96 packed rows, a block per head
])
def test_odd_kv_heads(name, kw):
    """The tcgen05 kernel's heads mode with an odd number of KV heads: the
    last unit holds one head."""
    wl = W.make_workload(name, 29, B=3, seq=("uniform", 150, 700), V=2000, **kw)
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)


@pytest.mark.parametrize("page_size", [16, 32, 64])
def test_eight_row_blocks_on_paged_cache(page_size):
    """Blocks of 8 packed rows (the LLaMA-7B Lookahead shape) run transposed
    (the rows as the MMA's N): paged prefix tiles of every page size, ragged
    tails, and 64-token splits so that most segments are merged from
    several CTAs' partials."""
    wl = W.make_workload("la7b", 30, B=3, seq=("uniform", 150, 900), V=3000, paged=True,
                         page_size=page_size)
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)


@pytest.mark.parametrize("paged", [False, True])
def test_eight_row_blocks_gqa(paged):
    """Transposed 8-row blocks with GQA: 4 lookahead rows x 2 query heads
    per KV head, bf16, head_dim 128, contiguous and paged caches."""
    wl = W.make_workload("tiny_la", 31, dtype="bf16", d=128, B=3, seq=("uniform", 100, 500),
                         V=3000, paged=paged)
    gh.run_and_check(wl)
    gh.run_and_check(wl, split_tokens=64)
