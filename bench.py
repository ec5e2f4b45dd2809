#!/usr/bin/env python
"""Benchmark of the self-speculative verification step on GB300.

One step = the whole hot path on one batch: spec_mask_build ->
spec_verify_attn -> spec_accept (vocab reduce + acceptance) -> kv_commit,
through the libspecverify C ABI, plus the restore of seq_len / free_head
(two 4-byte-per-request device copies) so every step does the same work.

Default workload: the long-context paged verify (64 requests, 32 q heads /
8 KV heads, head_dim 128, bf16, 16-token pages, prefix ~ U[16384, 32768],
8 lookahead rows, threshold acceptance over vocab 32000).

Prints ONE JSON line (rank 0).  Metric: verified speculative tokens per
second (candidate tokens judged per step / step time).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed the same way

``--config la_prefill`` times the prefill form of Lookahead Attention
(spec_la_prefill_attn: 4 requests x (4096 + 8) positions, 32 heads, head_dim
128, bf16) instead; its metric is prefill positions per second and its
roofline is the tensor-core one.  ``--config ss_draft`` times the next
draft (spec_draft_tree + spec_prune_tree: 32 requests, 3 streams, top-4,
vocab 50272); its metric is draft-tree nodes per second.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified spec tokens/s (attn+accept+commit)"
UNIT = "tokens/s"
L2_BYTES = 126 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", default="long_paged")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-workers", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch (small cases for profiling)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def workload_label(wl):
    seq = f"S~U[{int(wl.seq_len.min())},{int(wl.seq_len.max())}]"
    return (f"{wl.name}: B={wl.B} R={wl.R} Hq/Hkv={wl.Hq}/{wl.Hkv} d={wl.d} {wl.dtype} "
            f"{'paged(16-token pages)' if wl.paged else 'contiguous'} KV, {seq}, "
            f"n_soft={wl.n_soft}, V={wl.V}, "
            f"{'threshold' if wl.mode == 'la' else 'soft matching' if wl.soft else 'greedy tree'}")


def attn_algorithmic_bytes(wl):
    """Bytes spec_verify_attn must move (nothing dense over masked columns)."""
    e = 2 if wl.dtype == "bf16" else 4
    W = (wl.R + 31) // 32
    S = wl.seq_len.astype("int64")
    prefix = int(S.sum()) * wl.Hkv * wl.d * 2 * e
    block = wl.B * wl.R * wl.Hkv * wl.d * 2 * e
    soft = wl.n_soft * wl.Hkv * wl.d * 2 * e
    qo = wl.B * wl.R * wl.Hq * wl.d * e * 2
    lse = wl.B * wl.Hq * wl.R * 4
    ints = wl.B * 4 + wl.B * wl.R * (W * 4 + 1)
    if wl.paged:
        ints += int(((S + wl.page_size - 1) // wl.page_size).sum()) * 4
    return prefix + block + soft + qo + lse + ints


def step_algorithmic_bytes(wl, accepted_rows):
    e = 2 if wl.dtype == "bf16" else 4
    le = 2 if wl.logit_dtype == "bf16" else 4
    logits = wl.B * wl.Rj * wl.V * le
    if wl.soft:
        # draft rows once, plus the stop rows' second read for the residual draw
        logits += wl.draft_logits.shape[0] * wl.draft_logits.shape[1] * wl.V * le
    accept_io = wl.B * wl.N * 4 * 3 + wl.B * wl.Rj * 12 + wl.B * (wl.path_cap + 3) * 4
    commit = accepted_rows * wl.Hkv * wl.d * 2 * e * 2
    mask = wl.B * wl.R * (4 + 1 + 1 + 4 * ((wl.R + 31) // 32))
    return attn_algorithmic_bytes(wl) + logits + accept_io + commit + mask


VERIFY_SOURCES = ("attn", "verify_attn", "ptx_")
PREFILL_SOURCES = ("la_prefill", "ptx_")


def kernel_sources_sha(prefixes=VERIFY_SOURCES):
    """Hash of the CUDA sources (file names starting with ``prefixes``) that
    a recorded traffic figure was taken from."""
    from self_speculative_verification_gb300 import _build
    h = hashlib.sha256()
    for f in sorted(os.listdir(_build.CSRC)):
        if f.startswith(prefixes):
            with open(os.path.join(_build.CSRC, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(config, prefixes=VERIFY_SOURCES):
    """DRAM bytes per call of the workload's dominant kernel from the
    committed ncu summary, or None if its sources changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(config)
        if rec and rec.get("source_sha") == kernel_sources_sha(prefixes):
            return rec.get("dram_bytes_per_call")
    except Exception:
        pass
    return None


def max_over_ranks(x: float, device="cpu") -> float:
    """Largest value of x over the ranks of the default process group (x
    itself without one).  The bench takes the slowest rank's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step: int, steps: int, world: int, total_ms: float) -> float:
    """Whole-job verified tokens per second: every rank runs its own replica
    (weak scaling), all ranks' tokens over the slowest rank's time."""
    return tokens_per_step * steps * world / (total_ms / 1e3)


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        load = [r for r in rows if r["power"] > 0.3 * max(x["power"] for x in rows)] or rows
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in load):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
                "samples": len(load)}


# --------------------------------------------------------------- CPU oracle

def _oracle_worker(conn, config, seed, requests):
    """Runs in a spawned process: the oracle on a sample of requests."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import numpy as np
    import oracle
    from self_speculative_verification_gb300 import workloads as W
    wl = W.make_workload(config, seed)
    kv = {b: wl.prefix_kv(b) for b in requests}
    empty = np.zeros((wl.Hkv, 0, wl.d), dtype=np.float32)
    pk = [kv[b][0] if b in kv else empty for b in range(wl.B)]
    pv = [kv[b][1] if b in kv else empty for b in range(wl.B)]
    conn.send(("ready", sum(int(wl.n_nodes[b]) for b in requests)))
    mode = oracle.MODE_THRESH_CHAIN if wl.mode == "la" else oracle.MODE_GREEDY_TREE
    while True:
        msg = conn.recv()
        if msg == "stop":
            break
        t0 = time.perf_counter()
        for b in requests:
            vp = wl.vparent[b:b + 1]
            vis, valid, sees = oracle.mask_build(vp, wl.soft_flags[b:b + 1])
            O, L = oracle.verify_attention(
                wl.q[b:b + 1], [pk[b]], [pv[b]], wl.kb[b:b + 1], wl.vb[b:b + 1], vis, valid,
                sees, soft_k=wl.soft_k, soft_v=wl.soft_v)
            if wl.soft:
                acc, paths, nxt, last = oracle.accept_soft(
                    wl.logits[b:b + 1], wl.draft_logits[b:b + 1], wl.tokens[b:b + 1],
                    wl.tree_parent[b:b + 1], None, wl.child_draft_row[b:b + 1],
                    wl.n_nodes[b:b + 1], wl.u_accept[b:b + 1], wl.u_sample[b:b + 1],
                    wl.temperature)
            else:
                prop = wl.tokens[b] if wl.mode == "la" else None
                am, lse, zp = oracle.vocab_reduce(wl.logits[b], prop)
                acc, paths, nxt, last = oracle.accept(
                    mode, wl.tau, wl.tokens[b:b + 1], wl.tree_parent[b:b + 1],
                    wl.n_nodes[b:b + 1], am[None], lse[None], zp[None])
            # commit the accepted rows into the request's own logical cache
            K = np.concatenate([pk[b], np.zeros((wl.Hkv, wl.R, wl.d), np.float32)], axis=1)
            oracle.kv_commit_contiguous(K[None], K[None], [int(wl.seq_len[b])],
                                        wl.kb[b:b + 1], wl.vb[b:b + 1], paths)
        conn.send(("done", time.perf_counter() - t0))
    conn.close()


class OracleWorkers:
    """A spawned pool of oracle processes, one request sample each."""

    def __init__(self, config, seed, n_workers, B):
        ctx = mp.get_context("spawn")
        n = max(1, min(n_workers, B))
        self.conns, self.procs = [], []
        self.tokens = 0
        self.requests = list(range(n))
        for i in range(n):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(b, config, seed, [i]), daemon=True)
            p.start()
            self.conns.append(a)
            self.procs.append(p)
        for c in self.conns:
            tag, tok = c.recv()
            self.tokens += tok
        self.n = n

    def step(self):
        t0 = time.perf_counter()
        for c in self.conns:
            c.send("go")
        times = [c.recv()[1] for c in self.conns]
        return time.perf_counter() - t0, max(times)

    def close(self):
        for c in self.conns:
            try:
                c.send("stop")
            except Exception:
                pass
        for p in self.procs:
            p.join(timeout=10)


def run_reference(args):
    """--impl reference: the CPU oracle as it stands, timed on host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from self_speculative_verification_gb300 import workloads as W
    cfg = W.CONFIGS[args.config]
    cores = args.cpu_workers or host_cores()
    workers = OracleWorkers(args.config, args.seed, cores, cfg["B"])
    try:
        for _ in range(args.warmup):
            workers.step()
        walls = [workers.step()[0] for _ in range(args.steps)]
    finally:
        workers.close()
    wl = W.make_workload(args.config, args.seed)
    t = sum(walls)
    value = workers.tokens * len(walls) / t
    sample = (f"requests 0..{workers.n - 1} of {args.config} (all heads, their logits rows), "
              f"one per spawned process; each step re-runs the sample")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t / len(walls), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_label(wl), "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": workers.n, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(args, wl):
    cores = args.cpu_workers or host_cores()
    workers = OracleWorkers(args.config, args.seed, cores, wl.B)
    try:
        workers.step()                       # warm
        walls = [workers.step()[0] for _ in range(2)]
    finally:
        workers.close()
    value = workers.tokens * len(walls) / sum(walls)
    return {"value": value, "unit": UNIT, "cores": workers.n, "kind": "oracle",
            "sample": f"requests 0..{workers.n - 1} of the workload (all heads, logits rows, "
                      f"acceptance, commit), one per spawned process, best-effort float64 numpy"}


# ------------------------------------------------------------------- GPU arm

def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    # CPU baseline processes start (spawn) before the first GPU call
    cpu = None
    from self_speculative_verification_gb300 import workloads as W
    from self_speculative_verification_gb300 import binding as bn
    from self_speculative_verification_gb300.device import DeviceStep

    wl = W.make_workload(args.config, args.seed + rank, B=args.batch or None)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, wl)

    bn.load_library()
    ds = DeviceStep(wl, device=dev, threads=16)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)

    attn_bytes = attn_algorithmic_bytes(wl)
    footprint = attn_bytes + wl.B * wl.Rj * wl.V * 2
    flush = footprint < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None

    # the step's calls in order (rotation / gather only where the workload
    # has them); events bracket each call on the launching stream
    stages = [(n, f) for n, f in (("stream_rotate", ds.rotate_values if ds.rotate else None),
                                  ("mask_build", ds.mask_build),
                                  ("verify_attn", ds.verify_attn),
                                  ("accept", ds.accept_step),
                                  ("future_gather",
                                   ds.gather_future if ds.future is not None else None),
                                  ("kv_commit", ds.commit)) if f is not None]
    n_st = len(stages)
    i_attn = [n for n, _ in stages].index("verify_attn")

    def step(ev=None):
        ds.reset_state()
        for i, (_, f) in enumerate(stages):
            if ev is not None:
                ev[i].record(stream)
            f()
        if ev is not None:
            ev[n_st].record(stream)

    for _ in range(args.warmup):
        step()
        if flush:
            flush_buf.random_()
    torch.cuda.synchronize(dev)
    assert bn.spec_get_status() == 0, "device status set during warm-up"

    # The timed steps carry no events between their calls (an event between
    # two kernels would stop the next one from being scheduled while the
    # previous drains); with the L2 flushed between steps each step is timed
    # by its own pair of events, the flush outside them.  The per-call
    # breakdown comes from a separate pass of the same steps with events
    # between the calls.
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    region = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        region[0].record(stream)
        for i in range(args.steps):
            step_ev[i][0].record(stream)
            step()
            step_ev[i][1].record(stream)
            if flush:
                flush_buf.random_()
        region[1].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    status = bn.spec_get_status()
    step_ms = np.array([a.elapsed_time(b) for a, b in step_ev])
    region_ms = region[0].elapsed_time(region[1])
    total_ms = float(step_ms.sum()) if flush else region_ms
    total_ms = max_over_ranks(total_ms, dev)

    # per-call breakdown (not part of the timed region)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_st + 1)]
           for _ in range(args.steps)]
    for i in range(args.steps):
        step(evs[i])
        if flush:
            flush_buf.random_()
    torch.cuda.synchronize(dev)
    status |= bn.spec_get_status()
    per = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(n_st)]
                    for i in range(args.steps)])          # ms per stage

    tokens = wl.verified_tokens()
    value = job_throughput(tokens, args.steps, world, total_ms)
    attn_ms = float(per[:, i_attn].mean())
    hbm, hbm_kind = peaks()
    achieved = attn_bytes / (attn_ms / 1e3) / 1e9
    accepted_rows = int(ds.acc_len.sum().item())

    # e2e: host (pinned) inputs -> device, the four calls, results -> host
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(ds, args.e2e_steps, stream)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    ms_step = total_ms / args.steps
    accepted_tps = accepted_rows * args.steps * world / (total_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype, "data": "synthetic",
        "config": {
            "workload": workload_label(wl),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": ("flushed between steps (2x L2 buffer written)" if flush else
                   f"inputs larger than L2 ({attn_bytes / 1e9:.2f} GB per step vs 126 MB L2)"),
            "seed": args.seed,
            "verified_tokens_per_step": tokens,
            "accepted_rows_per_step": accepted_rows,
            "per_call_ms": {n: float(per[:, i].mean()) for i, (n, _) in enumerate(stages)},
            "step_ms_spread": {"min": float(step_ms.min()), "median": float(np.median(step_ms)),
                               "max": float(step_ms.max())},
            "step_includes": "seq_len/free_head restore (2 small device copies)",
            "step_algorithmic_bytes": step_algorithmic_bytes(wl, accepted_rows),
        },
        "roofline": {
            "kernel": "spec_verify_attn (split kernel + combine kernel)",
            "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "peak_kind": f"{hbm_kind} HBM copy bandwidth",
            "algorithmic_bytes_per_call": attn_bytes,
            "traffic": recorded_traffic(args.config),
        },
        "accepted_tokens_per_s": accepted_tps,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": ds.launches_per_step * args.steps,
        "device_status": status,
    }
    line["clocks"] = clk.summary()
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(ds, steps, stream):
    """The same step through the C ABI with host buffers: every step's inputs
    are copied in from pinned host memory and its results (the acceptance
    outputs) copied out and read by the host.  Two device input sets: while
    step i computes on one, a copy stream uploads step i + 1's inputs into
    the other (independent batches, as a server overlaps them); the host
    waits for step i - 1's results during step i."""
    import torch
    names = [n for n in ("q", "kb", "vb", "soft_k", "soft_v", "vparent", "soft_flags",
                         "logits", "tokens", "tree_parent", "n_nodes", "draft_logits",
                         "child_draft_row", "u_accept", "u_sample")
             if getattr(ds, n, None) is not None]
    # the step's results: acceptance, and the attention outputs O and LSE
    outputs = [ds.acc_len, ds.path, ds.next_token, ds.last_node, ds.o, ds.lse]
    if ds.future is not None:
        outputs.append(ds.future)
    h_in = [getattr(ds, n).cpu().pin_memory() for n in names]
    sets = [{n: getattr(ds, n) for n in names},
            {n: torch.empty_like(getattr(ds, n)) for n in names}]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outputs]
             for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = sum(t.numel() * t.element_size() for t in outputs)
    copy_stream = torch.cuda.Stream(device=stream.device)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # set j's inputs landed
    ev_free = [torch.cuda.Event() for _ in range(2)]   # the step computing on set j is done
    ev_out = [torch.cuda.Event() for _ in range(2)]    # its results are on the host
    for j in range(2):
        ev_free[j].record(stream)

    def upload(j):
        copy_stream.wait_event(ev_free[j])
        with torch.cuda.stream(copy_stream):
            for n, h in zip(names, h_in):
                sets[j][n].copy_(h, non_blocking=True)
        ev_in[j].record(copy_stream)

    def run(n_steps):
        upload(0)
        for i in range(n_steps):
            j = i & 1
            if i + 1 < n_steps:
                upload(1 - j)                   # the next step's inputs
            stream.wait_event(ev_in[j])
            for n in names:
                setattr(ds, n, sets[j][n])
            ds.reset_state()
            ds.run()
            ev_free[j].record(stream)
            for h, d in zip(h_out[j], outputs):
                h.copy_(d, non_blocking=True)
            ev_out[j].record(stream)
            if i > 0:
                ev_out[1 - j].synchronize()     # the host reads step i - 1's results
        ev_out[(n_steps - 1) & 1].synchronize()
        copy_stream.synchronize()

    run(3)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    dt = time.perf_counter() - t0
    for n in names:
        setattr(ds, n, sets[0][n])
    tokens = ds.wl.verified_tokens()
    return {"value": tokens * steps / dt, "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": 1e3 * dt / steps,
            "timing": "host wall clock over the steps; each step's inputs copied in from "
                      "pinned host memory on a copy stream (overlapping the previous step's "
                      "compute) and its results (acceptance outputs, attention O and LSE) "
                      "copied out and waited for by the host"}


# ------------------------------------------------------ prefill-form LA

PREFILL_METRIC = "LA prefill positions/s (full M_LA attention, all heads)"


def prefill_flops(wl):
    """Algorithmic FLOPs of one call: 4 d per visible (query, key) pair per
    head (QK^T and PV), nothing over masked pairs.  Original i sees i + 1
    keys; each lookahead position sees the n originals and itself."""
    pairs = wl.n * (wl.n + 1) // 2 + wl.k * (wl.n + 1)
    return 4 * wl.d * pairs * wl.B * wl.Hq


def prefill_label(wl):
    return (f"la_prefill: B={wl.B} n={wl.n} k={wl.k} (L={wl.L}) Hq/Hkv={wl.Hq}/{wl.Hkv} "
            f"d={wl.d} bf16, full M_LA mask")


def _prefill_oracle_worker(conn, cfg, seed, pairs):
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import oracle
    from self_speculative_verification_gb300 import workloads as W
    wl = W.make_prefill(seed, **cfg)
    G = wl.Hq // wl.Hkv
    conn.send("ready")
    while True:
        if conn.recv() == "stop":
            break
        t0 = time.perf_counter()
        for b, h in pairs:
            oracle.la_prefill_attention(wl.q[b, :, h], wl.kk[b, :, h // G], wl.v[b, :, h // G],
                                        wl.n)
        conn.send(time.perf_counter() - t0)
    conn.close()


def prefill_oracle(cfg, seed, cores, warm, steps):
    """The oracle on one (request, head) slice per spawned process; returns
    (positions/s equivalent over all heads, processes, wall seconds per step)."""
    ctx = mp.get_context("spawn")
    n = max(1, min(cores, cfg["B"] * cfg["Hq"]))
    pairs = [(i % cfg["B"], i // cfg["B"]) for i in range(n)]
    conns, procs = [], []
    for i in range(n):
        a, b = ctx.Pipe()
        p = ctx.Process(target=_prefill_oracle_worker, args=(b, cfg, seed, [pairs[i]]),
                        daemon=True)
        p.start()
        conns.append(a)
        procs.append(p)
    for c in conns:
        c.recv()
    walls = []
    try:
        for i in range(warm + steps):
            t0 = time.perf_counter()
            for c in conns:
                c.send("go")
            for c in conns:
                c.recv()
            if i >= warm:
                walls.append(time.perf_counter() - t0)
    finally:
        for c in conns:
            try:
                c.send("stop")
            except Exception:
                pass
        for p in procs:
            p.join(timeout=10)
    L = cfg["n"] + cfg["k"]
    wall = sum(walls) / len(walls)
    # n slices of L positions each = n / Hq of a full-head pass over L positions
    return n * L / cfg["Hq"] / wall, n, wall


def run_prefill_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from self_speculative_verification_gb300 import workloads as W
    cfg = dict(W.PREFILL_CONFIGS[args.config])
    cores = args.cpu_workers or host_cores()
    value, n, wall = prefill_oracle(cfg, args.seed, cores, min(args.warmup, 1),
                                    max(1, min(args.steps, 3)))
    wl = W.make_prefill(args.seed, B=1, n=1, k=0, Hq=1, Hkv=1)   # label only
    sample = (f"{n} (request, head) slices of {args.config}, one per spawned process, "
              f"float64 numpy; each step re-runs the sample")
    line = {
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "positions/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wall, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"la_prefill: B={cfg['B']} n={cfg['n']} k={cfg['k']} "
                               f"Hq/Hkv={cfg['Hq']}/{cfg['Hkv']} d={cfg['d']}",
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": n, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    del wl
    print(json.dumps(line), flush=True)


def run_prefill_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from self_speculative_verification_gb300 import workloads as W
    from self_speculative_verification_gb300 import binding as bn

    cfg = dict(W.PREFILL_CONFIGS[args.config])
    if args.batch:
        cfg["B"] = args.batch
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n, wall = prefill_oracle(cfg, args.seed, args.cpu_workers or host_cores(), 0, 1)
        cpu = {"value": v, "unit": "positions/s", "cores": n, "kind": "oracle",
               "sample": f"{n} (request, head) slices of the workload, one per spawned "
                         f"process, float64 numpy, scaled to all heads"}
    wl = W.make_prefill(args.seed + rank, **cfg)
    bn.load_library()
    q = torch.from_numpy(wl.q).to(dev, torch.bfloat16)
    k = torch.from_numpy(wl.kk).to(dev, torch.bfloat16)
    v = torch.from_numpy(wl.v).to(dev, torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.Hq, wl.L), dtype=torch.float32, device=dev)
    desc = bn.prefill_desc(wl.B, wl.n, wl.k, wl.Hq, wl.Hkv, wl.d)
    stream = torch.cuda.current_stream(dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    flush = in_bytes < 2 * L2_BYTES
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if flush else None

    for _ in range(args.warmup):
        bn.spec_la_prefill_attn(desc, q, k, v, o, lse, stream)
        if flush:
            flush_buf.random_()
    torch.cuda.synchronize(dev)
    assert bn.spec_get_status() == 0, "device status set during warm-up"
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for e0, e1 in evs:
            e0.record(stream)
            bn.spec_la_prefill_attn(desc, q, k, v, o, lse, stream)
            e1.record(stream)
            if flush:
                flush_buf.random_()
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    status = bn.spec_get_status()
    times = np.array([a.elapsed_time(b) for a, b in evs])
    total_ms = max_over_ranks(float(times.sum()), dev)
    positions = wl.B * wl.L
    value = positions * args.steps * world / (total_ms / 1e3)
    flops = prefill_flops(wl)
    call_ms = float(times.mean())
    achieved = flops / (call_ms / 1e3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        peak, peak_kind = 1900.0, "fallback"

    # e2e: pinned host q/k/v in, o/lse out, every call
    h_in = [t.cpu().pin_memory() for t in (q, k, v)]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (o, lse)]
    e2e = None
    if args.e2e_steps > 0:
        def one():
            for d, h in zip((q, k, v), h_in):
                d.copy_(h, non_blocking=True)
            bn.spec_la_prefill_attn(desc, q, k, v, o, lse, stream)
            for h, d in zip(h_out, (o, lse)):
                h.copy_(d, non_blocking=True)
            stream.synchronize()
        for _ in range(2):
            one()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            one()
        dt = time.perf_counter() - t0
        e2e = {"value": positions * args.e2e_steps / dt, "unit": "positions/s",
               "h2d_bytes_per_step": in_bytes,
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in (o, lse)),
               "ms_per_step": 1e3 * dt / args.e2e_steps}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "positions/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": prefill_label(wl), "seed": args.seed,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": ("flushed between calls" if flush else
                          f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB vs 126 MB)")},
        "roofline": {"kernel": "la_prefill_kernel", "bound": "tensor", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} dense bf16 (burst)",
                     "algorithmic_flops_per_call": flops,
                     "traffic": recorded_traffic(args.config, PREFILL_SOURCES)},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "device_status": status,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------- draft trees

DRAFT_METRIC = "SS draft-tree nodes/s (top-k tree construction + pruning)"


def draft_algorithmic_bytes(dw):
    """Stream rows and the inner nodes' early-exit rows are read once; the
    tree arrays (tokens, parents, keep map, block parent pointers) are
    written."""
    e = 2 if dw.dtype == "bf16" else 4
    inner = dw.N - dw.k ** dw.gamma
    logits = dw.B * (dw.gamma + inner) * dw.V * e
    arrays = dw.B * dw.N * 4 * (2 + 2 + 1 + 2 * (1 + dw.gamma))
    return logits + arrays


def _draft_oracle_worker(conn, cfg, seed, requests):
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import oracle
    from self_speculative_verification_gb300 import workloads as W
    dw = W.make_draft(seed, **cfg)
    conn.send("ready")
    while conn.recv() != "stop":
        t0 = time.perf_counter()
        for b in requests:
            tok, par, _ = oracle.draft_tree(dw.stream_logits[b], dw.k, dw.root_token[b])
            t2, p2, km = oracle.prune_tree(tok, par, dw.early_logits[b], dw.threshold)
            oracle.ss_block_vparent(p2, dw.gamma, dw.N * (1 + dw.gamma))
        conn.send(time.perf_counter() - t0)
    conn.close()


def draft_oracle(cfg, seed, cores, warm, steps):
    ctx = mp.get_context("spawn")
    n = max(1, min(cores, cfg["B"]))
    conns, procs = [], []
    for i in range(n):
        a, b = ctx.Pipe()
        p = ctx.Process(target=_draft_oracle_worker, args=(b, cfg, seed, [i]), daemon=True)
        p.start()
        conns.append(a)
        procs.append(p)
    for c in conns:
        c.recv()
    walls = []
    try:
        for i in range(warm + steps):
            t0 = time.perf_counter()
            for c in conns:
                c.send("go")
            for c in conns:
                c.recv()
            if i >= warm:
                walls.append(time.perf_counter() - t0)
    finally:
        for c in conns:
            try:
                c.send("stop")
            except Exception:
                pass
        for p in procs:
            p.join(timeout=10)
    N = 1 + sum(cfg["k"] ** g for g in range(1, cfg["gamma"] + 1))
    wall = sum(walls) / len(walls)
    return n * N / wall, n, wall


def run_draft_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from self_speculative_verification_gb300 import workloads as W
    cfg = dict(W.DRAFT_CONFIGS[args.config])
    value, n, wall = draft_oracle(cfg, args.seed, args.cpu_workers or host_cores(),
                                  min(args.warmup, 1), max(1, min(args.steps, 3)))
    sample = (f"requests 0..{n - 1} of {args.config}, one per spawned process, float64 "
              f"numpy; each step re-runs the sample")
    line = {
        "impl": "reference", "metric": DRAFT_METRIC, "value": value, "unit": "nodes/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wall, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.config}: {cfg}", "sample": sample},
        "cpu_baseline": {"value": value, "unit": "nodes/s", "cores": n, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "nodes/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_draft_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from self_speculative_verification_gb300 import workloads as W
    from self_speculative_verification_gb300 import binding as bn

    cfg = dict(W.DRAFT_CONFIGS[args.config])
    if args.batch:
        cfg["B"] = args.batch
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, n, wall = draft_oracle(cfg, args.seed, args.cpu_workers or host_cores(), 0, 1)
        cpu = {"value": v, "unit": "nodes/s", "cores": n, "kind": "oracle",
               "sample": f"requests 0..{n - 1} of the workload, one per spawned process, "
                         f"float64 numpy"}
    dw = W.make_draft(args.seed + rank, **cfg)
    bn.load_library()
    B, N, g = dw.B, dw.N, dw.gamma
    R = N * (1 + g)
    ldt = torch.bfloat16 if dw.dtype == "bf16" else torch.float32
    i32 = torch.int32
    stream_l = torch.from_numpy(dw.stream_logits).to(dev, ldt)
    early = torch.from_numpy(dw.early_logits).to(dev, ldt)
    root = torch.from_numpy(dw.root_token).to(dev)
    tok, par, t2, p2, keep = (torch.zeros((B, N), dtype=i32, device=dev) for _ in range(5))
    nn, n2 = torch.zeros(B, dtype=i32, device=dev), torch.zeros(B, dtype=i32, device=dev)
    vp_full, vp = (torch.zeros((B, R), dtype=i32, device=dev) for _ in range(2))
    spec_dt = bn.SPEC_BF16 if dw.dtype == "bf16" else bn.SPEC_F32
    ddesc = bn.DraftDesc(B, g, g, dw.k, dw.V, spec_dt, N, R)
    pdesc = bn.PruneDesc(B, N, dw.V, spec_dt, dw.threshold, g, R)
    stream = torch.cuda.current_stream(dev)
    in_bytes = draft_algorithmic_bytes(dw)
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    def step():
        bn.spec_draft_tree(ddesc, stream_l, None, root, tok, par, nn, vp_full, stream)
        bn.spec_prune_tree(pdesc, tok, par, nn, early, keep, t2, p2, n2, vp, stream)

    for _ in range(args.warmup):
        step()
        flush_buf.random_()
    torch.cuda.synchronize(dev)
    assert bn.spec_get_status() == 0, "device status set during warm-up"
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for e0, e1 in evs:
            e0.record(stream)
            step()
            e1.record(stream)
            flush_buf.random_()
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    status = bn.spec_get_status()
    times = np.array([a.elapsed_time(b) for a, b in evs])
    total_ms = max_over_ranks(float(times.sum()), dev)
    value = B * N * args.steps * world / (total_ms / 1e3)
    step_ms = float(times.mean())
    hbm, hbm_kind = peaks()
    achieved = in_bytes / (step_ms / 1e3) / 1e9

    e2e = None
    if args.e2e_steps > 0:
        h_in = [t.cpu().pin_memory() for t in (stream_l, early, root)]
        outs = (t2, p2, n2, vp)
        h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]

        def one():
            for d, h in zip((stream_l, early, root), h_in):
                d.copy_(h, non_blocking=True)
            step()
            for h, d in zip(h_out, outs):
                h.copy_(d, non_blocking=True)
            stream.synchronize()
        for _ in range(2):
            one()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            one()
        dt = time.perf_counter() - t0
        e2e = {"value": B * N * args.e2e_steps / dt, "unit": "nodes/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in h_in),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in h_out),
               "ms_per_step": 1e3 * dt / args.e2e_steps}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": DRAFT_METRIC, "value": value, "unit": "nodes/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dw.dtype,
        "data": "synthetic",
        "config": {"workload": f"{args.config}: B={B} gamma={g} k={dw.k} V={dw.V} {dw.dtype} "
                               f"threshold={dw.threshold} ({N} nodes per full tree)",
                   "seed": args.seed, "l2": "flushed between steps (2x L2 buffer written)",
                   "survivors_per_step": int(n2.sum().item()),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"kernel": "draft_tree_kernel + prune_edge_kernel + prune_compact_kernel",
                     "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "peak_kind": f"{hbm_kind} HBM copy bandwidth",
                     "algorithmic_bytes_per_call": in_bytes, "traffic": None},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 3 * args.steps,
        "device_status": status,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    from self_speculative_verification_gb300 import workloads as W
    if args.config in W.DRAFT_CONFIGS:
        if args.impl == "reference":
            run_draft_reference(args)
        else:
            run_draft_gpu(args)
        return
    if args.config in W.PREFILL_CONFIGS:
        if args.impl == "reference":
            run_prefill_reference(args)
        else:
            run_prefill_gpu(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
