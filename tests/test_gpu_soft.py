"""GPU parity of soft-matching acceptance ("Speculative Streaming",
verification step with soft matching) against the float64 oracle.

Acceptance lengths and paths are planted with wide margins around each
uniform and must match bit for bit; the residual draw of the correction
token must equal the oracle's or sit on a CDF boundary that fp32 sums
cannot resolve (gpu_helpers.check_soft_draw)."""

import numpy as np
import pytest
import torch

import gpu_helpers as gh
import oracle
from self_speculative_verification_gb300 import binding as bn
from self_speculative_verification_gb300 import workloads as W
from self_speculative_verification_gb300.device import DeviceStep

pytestmark = pytest.mark.gpu

SMALL = dict(B=4, seq=("uniform", 100, 500), V=5000)


@pytest.fixture(autouse=True)
def _gpu():
    gh.require_gpu()


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_soft_step_parity_small(seed):
    wl = W.make_workload("ss_soft", seed, **SMALL)
    gh.run_and_check(wl)


def test_soft_f32_logits():
    wl = W.make_workload("ss_soft", 4, dtype="f32", **SMALL)
    gh.run_and_check(wl)


def test_soft_full_size_accept():
    """The full ss_soft workload (32 requests, vocab 50272)."""
    wl = W.make_workload("ss_soft", 0)
    ds = DeviceStep(wl)
    ds.run()
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    gh.check_accept_soft(ds)


@pytest.mark.parametrize("T", [0.7, 1.5])
def test_soft_temperature(T):
    """Other temperatures: decisions are no longer planted, so compare with
    the oracle only (a decision within fp32 error of its uniform is a
    ~1e-6 event per test)."""
    wl = W.make_workload("ss_soft", 9, **SMALL)
    wl.temperature = T
    ds = DeviceStep(wl)
    ds.accept_step()
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0
    acc, paths, nxt, last = oracle.accept_soft(
        wl.logits, wl.draft_logits, wl.tokens, wl.tree_parent, None, wl.child_draft_row,
        wl.n_nodes, wl.u_accept, wl.u_sample, T)
    assert ds.acc_len.cpu().numpy().tolist() == acc.tolist()
    pg = ds.path.cpu().numpy()
    for b in range(wl.B):
        assert pg[b, : acc[b]].tolist() == paths[b]
        gh.check_soft_draw(wl, b, int(last[b]), int(ds.next_token[b].item()), int(nxt[b]))


def _tensors(logits, draft, tokens, parent, cdr, n_nodes, ua, us):
    dev = torch.device("cuda", 0)
    i32, f32 = torch.int32, torch.float32
    t = lambda a, dt: torch.tensor(np.asarray(a), dtype=dt, device=dev)
    B = len(n_nodes)
    N = tokens.shape[1]
    out = dict(logits=t(logits, f32), draft=t(draft, f32) if draft is not None else None,
               tokens=t(tokens, i32), parent=t(parent, i32),
               cdr=t(cdr, i32) if cdr is not None else None, n=t(n_nodes, i32),
               ua=t(ua, f32), us=t(us, f32),
               lse_t=torch.zeros(B, logits.shape[1], dtype=f32, device=dev),
               lse_d=torch.zeros(B, max(1, 0 if draft is None else draft.shape[1]),
                                 dtype=f32, device=dev),
               acc=torch.zeros(B, dtype=i32, device=dev),
               path=torch.zeros(B, N, dtype=i32, device=dev),
               nxt=torch.zeros(B, dtype=i32, device=dev),
               last=torch.zeros(B, dtype=i32, device=dev))
    return out


def _run(x, V, Rd, T=1.0):
    B, Rj = x["logits"].shape[0], x["logits"].shape[1]
    d = bn.soft_desc(B, Rj, Rd, V, bn.SPEC_F32, x["tokens"].shape[1], x["tokens"].shape[1], T)
    bn.spec_accept_soft(d, x["logits"], x["draft"], x["tokens"], x["parent"], None, x["cdr"],
                        x["n"], x["ua"], x["us"], x["lse_t"], x["lse_d"], x["acc"], x["path"],
                        x["nxt"], x["last"])
    torch.cuda.synchronize()
    assert bn.spec_get_status() == 0


@pytest.mark.parametrize("u", [0.05, 0.5, 0.95])
def test_residual_without_mass_draws_from_target(u):
    """A lone root whose draft row equals its target row: max(0, p - q) has
    no mass and the correction token is drawn from p."""
    rng = np.random.Generator(np.random.PCG64(1))
    V = 3000
    z = rng.standard_normal((1, 1, V)).astype(np.float32)
    x = _tensors(z, z.copy(), np.zeros((1, 1)), np.full((1, 1), -1), np.zeros((1, 1)), [1],
                 np.zeros((1, 1)), [u])
    _run(x, V, 1)
    assert x["acc"].item() == 1 and x["last"].item() == 0
    p = oracle.softmax_t(z[0, 0])
    want = oracle.residual_sample(p, None, u)
    got = int(x["nxt"].item())
    if got != want:
        cum = np.cumsum(p)
        assert cum[got - 1] - 1e-5 <= u <= cum[got] + 1e-5


def test_no_draft_rows_accepts_down_first_children():
    """n_draft_rows = 0: q = 0 for every child, so the first child of each
    node is taken (p > 0) and the bonus token is drawn from p."""
    rng = np.random.Generator(np.random.PCG64(2))
    V, N = 2000, 7
    parent = np.array([[-1, 0, 0, 1, 1, 3, 2]])
    tokens = np.array([[0, 5, 6, 7, 8, 9, 10]])
    z = rng.standard_normal((1, N, V)).astype(np.float32)
    x = _tensors(z, None, tokens, parent, None, [N], rng.random((1, N)), [0.3])
    _run(x, V, 0)
    assert x["acc"].item() == 4
    assert x["path"][0, :4].tolist() == [0, 1, 3, 5]
    assert x["last"].item() == 5
    want = oracle.residual_sample(oracle.softmax_t(z[0, 5]), None, 0.3)
    got = int(x["nxt"].item())
    if got != want:
        cum = np.cumsum(oracle.softmax_t(z[0, 5]))
        assert cum[got - 1] - 1e-5 <= 0.3 <= cum[got] + 1e-5


def test_soft_rejects_bad_arguments():
    x = _tensors(np.zeros((1, 1, 16), np.float32), None, np.zeros((1, 1)), np.full((1, 1), -1),
                 None, [1], np.zeros((1, 1)), [0.5])
    bad = [
        bn.soft_desc(1, 1, 0, 16, bn.SPEC_F32, 1, 1, 0.0),      # temperature 0
        bn.soft_desc(1, 1, 0, 16, bn.SPEC_F32, 1, 1, -1.0),
        bn.soft_desc(1, 0, 0, 16, bn.SPEC_F32, 1, 1, 1.0),      # no judge rows
        bn.soft_desc(1, 1, 1, 16, bn.SPEC_F32, 1, 1, 1.0),      # draft rows but no draft
    ]
    for d in bad:
        with pytest.raises(bn.SpecError) as e:
            bn.spec_accept_soft(d, x["logits"], x["draft"], x["tokens"], x["parent"], None,
                                x["cdr"], x["n"], x["ua"], x["us"], x["lse_t"], x["lse_d"],
                                x["acc"], x["path"], x["nxt"], x["last"])
        assert e.value.code == bn.SPEC_ERR_INVALID_ARG
    d = bn.soft_desc(1, 1, 0, 16, 7, 1, 1, 1.0)
    with pytest.raises(bn.SpecError) as e:
        bn.spec_accept_soft(d, x["logits"], x["draft"], x["tokens"], x["parent"], None, x["cdr"],
                            x["n"], x["ua"], x["us"], x["lse_t"], x["lse_d"], x["acc"],
                            x["path"], x["nxt"], x["last"])
    assert e.value.code == bn.SPEC_ERR_UNSUPPORTED
