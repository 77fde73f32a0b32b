#!/usr/bin/env python
"""Verify rounds/s and logit HBM GB/s of libspecverify on one GB300 (or N replicas).

Workload (one "step" = one verify round of the whole hot path over one batch):
batched serving verify, B=32 sequences, gamma=4 drafts, V=262,144 vocabulary,
bf16 target and draft logits (fp32 math), per-sequence T ~ U[0.5, 1.2],
rejection-sampling mode.  Inputs are synthetic (seeded, see workloads/), made
on the GPU before timing; a pool of rounds larger than L2 is cycled so every
step streams its logits from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the reference implementation of
this build) on the host cores on a bounded sample of the same workload.
Multi-GPU runs are independent replicas (the verify step has no exchange).
"""
from __future__ import annotations

import argparse
import contextlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify rounds/s and logit HBM GB/s (fraction of 8 TB/s) at B×(γ+1)×262K vocab"
WORKLOAD = ("batched serving verify: B=32, gamma=4, V=262144, bf16 target+draft logits, "
            "per-sequence T~U[0.5,1.2], rejection sampling")
NOMINAL_HBM_GBS = 8000.0
B, GAMMA, V = 32, 4, 262144
POOL = 4  # rounds in the pool: 4 x 151 MB > L2 (126 MB)


def counted_bytes(B, gamma, V, esize, n_sampling):
    """Bytes of p and q the verify must read: every target row, plus the draft
    rows of sampling sequences."""
    return B * (gamma + 1) * V * esize + n_sampling * gamma * V * esize


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend)


def dist_barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(ws, x, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_id: str | None, period_ms: int = 50):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
               f"-lms={period_ms}"]
        if gpu_id:
            cmd.append(f"--id={gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self):
        self.t_mark = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, skip_first=0):
        rows = []
        for ln in self.lines[skip_first:]:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def time_loop(fn, n, stream):
    """Seconds for n eager calls fn(0..n-1), CUDA events on ``stream``."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


GRAPH_CHUNK = 100


class GraphLoop:
    """fn(i) for i in 0..n-1 captured into CUDA graphs of up to GRAPH_CHUNK
    steps each, so the host launch rate does not limit the measurement.
    Replayed on ``stream``; timed with CUDA events on that stream."""

    def __init__(self, fn, n, stream):
        import torch
        self.graphs = []
        self.stream = stream
        done = 0
        with torch.cuda.stream(stream):
            while done < n:
                k = min(GRAPH_CHUNK, n - done)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(done, done + k):
                        fn(i)
                self.graphs.append(g)
                done += k

    def run(self):
        import torch
        with torch.cuda.stream(self.stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for g in self.graphs:
                g.replay()
            e1.record(self.stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / 1e3


def run_ours(args):
    import torch

    import speculative_decoding_verification_54_gb300 as sv
    import workloads as wl
    from speculative_decoding_verification_54_gb300 import _build

    ws_n, rank, local = dist_setup()
    dist_init(ws_n, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    sv.load()
    stream = torch.cuda.Stream(device=dev)

    pool = [wl.torch_round("batched", r + 1000 * rank, dev) for r in range(POOL)]
    esize = 2
    n_samp = [int((p["temperature"] > 0).sum().item()) for p in pool]
    bytes_round = [counted_bytes(B, GAMMA, V, esize, n) for n in n_samp]
    bytes_mean = sum(bytes_round) / len(bytes_round)
    wsp = sv.make_workspace(B, GAMMA, V, device=dev)
    out = torch.empty((B, GAMMA + 1), dtype=torch.int32, device=dev)
    num = torch.empty((B,), dtype=torch.int32, device=dev)

    def step(i):
        p = pool[i % POOL]
        sv.spec_verify_sample(p["target"], p["draft"], p["draft_tokens"], p["temperature"],
                              p["u_accept"], p["u_resample"], out, num, wsp)

    def reduce_step(i):
        p = pool[i % POOL]
        sv.spec_verify_sample_reduce_only(p["target"], p["draft"], p["draft_tokens"], p["temperature"],
                                          p["u_accept"], p["u_resample"], out, num, wsp)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step(0)  # first call outside capture (per-device set-up)
    torch.cuda.synchronize()
    timed = GraphLoop(step, args.steps, stream)
    warm = GraphLoop(step, args.warmup, stream)
    warm.run()
    timed.run()  # the timed graphs' first replay (upload) stays out of the timed region
    torch.cuda.synchronize()
    assert sv.spec_verify_status(wsp, stream) == sv.SPEC_OK

    gpu_id = None
    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_id.startswith("GPU-"):
            gpu_id = "GPU-" + gpu_id
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    time.sleep(1.0)
    n_before = 0
    dist_barrier(ws_n)
    torch.cuda.synchronize()
    elapsed = timed.run()
    torch.cuda.synchronize()
    dist_barrier(ws_n)
    clocks.stop()
    st = sv.spec_verify_status(wsp, stream)
    if st != sv.SPEC_OK:
        raise SystemExit(f"device status after timed loop: {sv.error_string(st)}")
    elapsed_max = dist_max(ws_n, elapsed, dev)

    value = ws_n * args.steps / elapsed_max
    gbs = value * bytes_mean / 1e9

    # dominant kernel: the row reducer, launched alone with CUDA events on the same stream
    nred = max(50, min(args.steps, 5000))
    red_loop = GraphLoop(reduce_step, nred, stream)
    red_loop.run()
    red_s = red_loop.run() / nred
    del red_loop
    peak, peak_kind = load_peaks()
    achieved = bytes_mean / red_s / 1e9
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "rowstats_traffic.json")
    if os.path.exists(tr_path):
        with open(tr_path) as f:
            tr = json.load(f)
        if tr.get("kernel_source_sha") == _source_sha():
            traffic = tr.get("dram_bytes_per_launch")

    e2e = None if args.no_e2e else e2e_leg(sv, pool, out, num, wsp, dev, stream, args, ws_n)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "rounds/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_max / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "gamma": GAMMA, "V": V, "logits_dtype": "bf16",
                   "global_batch": B * ws_n, "parallelism": f"replicas x{ws_n}",
                   "l2": f"inputs larger than L2: pool of {POOL} rounds x {bytes_mean / 1e6:.1f} MB cycled"},
        "logit_gbs": round(gbs, 1), "frac_of_8tbs": round(gbs / ws_n / NOMINAL_HBM_GBS, 4),
        "frac_of_measured_hbm": round(gbs / ws_n / peak, 4),
        "roofline": {"bound": "hbm",
                     "kernel": "rowstats_kernel<bf16, %s loads>" % os.environ.get("SPECV_ROW_LOADS", "ldg"), "achieved": round(achieved, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": traffic, "bytes_per_launch": bytes_mean,
                     "avg_launch_us": round(red_s * 1e6, 3),
                     "timing": f"CUDA events over {nred} back-to-back reduce-only launches on the bench stream",
                     # the whole call (row reducer + tail) against the stated target: bytes of p and q
                     # read per round over the round time, as a fraction of 8 TB/s
                     "whole_call": {"achieved": round(gbs / ws_n, 1), "unit": "GB/s",
                                    "frac_of_8tbs": round(gbs / ws_n / NOMINAL_HBM_GBS, 4),
                                    "frac_of_measured": round(gbs / ws_n / peak, 4),
                                    "target_frac_of_8tbs": 0.70,
                                    "target_met": bool(gbs / ws_n / NOMINAL_HBM_GBS >= 0.70)}},
        "e2e": e2e,
        "gpu_launches": 2 * args.steps,
        "launch": f"CUDA graphs of up to {GRAPH_CHUNK} steps (2 kernels per step: row reducer, tail), "
                  "replayed on one stream",
        "clocks": clocks.summary(n_before),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"], result["parity"] = cpu_baseline(sv, pool, dev, stream, budget_s=args.cpu_seconds)
    if rank == 0 and not args.no_extra:
        result["other_workloads"] = other_workloads(sv, dev, stream, args)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def e2e_leg(sv, pool, out, num, wsp, dev, stream, args, ws_n):
    """End to end through the C ABI with host buffers: every step copies the
    round's inputs from pinned host memory, calls spec_verify_sample and reads
    the emitted tokens back.  The copies run on a second stream into one of
    two device input sets, so the copy of round i+1 overlaps the verify of
    round i (a serving loop's double buffering); the host link, not the
    verify, bounds the rate."""
    import torch
    hpool = []
    for p in pool[:2]:
        hpool.append({k: (v.to("cpu").pin_memory() if torch.is_tensor(v) else v) for k, v in p.items()})
    dsets = [{k: torch.empty_like(v, device=dev) for k, v in pool[0].items() if torch.is_tensor(v)}
             for _ in range(2)]
    outs = [(torch.empty_like(out), torch.empty_like(num)) for _ in range(2)]
    hout = [torch.empty(tuple(out.shape), dtype=torch.int32).pin_memory() for _ in range(2)]
    hnum = [torch.empty(tuple(num.shape), dtype=torch.int32).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for k, v in hpool[0].items() if torch.is_tensor(v))
    d2h = hout[0].numel() * 4 + hnum[0].numel() * 4
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    for e in free:
        e.record(stream)

    def e2e_step(i):
        j = i % 2
        hp, dp = hpool[i % 2], dsets[j]
        copy_stream.wait_event(free[j])      # the verify that last read set j is done
        with torch.cuda.stream(copy_stream):
            for k, t in dp.items():
                t.copy_(hp[k], non_blocking=True)
            copied[j].record(copy_stream)
        stream.wait_event(copied[j])
        o, n = outs[j]
        sv.spec_verify_sample(dp["target"], dp["draft"], dp["draft_tokens"], dp["temperature"],
                              dp["u_accept"], dp["u_resample"], o, n, wsp, stream=stream)
        free[j].record(stream)
        hout[j].copy_(o, non_blocking=True)
        hnum[j].copy_(n, non_blocking=True)

    torch.cuda.synchronize()  # inputs built on the default stream are complete
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    torch.cuda.synchronize()
    ne2e = max(10, min(args.steps, 400))
    dist_barrier(ws_n)
    with torch.cuda.stream(stream):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)           # no copy of the timed steps starts before e0
        for i in range(ne2e):
            e2e_step(i)
        e1.record(stream)                    # after the last device->host read
        e1.synchronize()
        el = e0.elapsed_time(e1) / 1e3
    el = dist_max(ws_n, el, dev)
    return {"value": round(ws_n * ne2e / el, 2), "unit": "rounds/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": ne2e,
            "how": ("eager calls; per step 6 pinned-host->device copies on a copy stream into one of two "
                    "device input sets, the C-ABI call, 2 device->host copies; round i+1's copy overlaps "
                    "round i's verify")}


def _source_sha():
    import hashlib
    h = hashlib.sha256()
    for f in ("rowstats.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "speculative_decoding_verification_54_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _round_to_host(p):
    import numpy as np
    import torch

    def logits(t):
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).cpu().numpy().view(np.uint16)
        return t.cpu().numpy()

    return dict(target=logits(p["target"]), draft=logits(p["draft"]),
                draft_tokens=p["draft_tokens"].cpu().numpy(), temperature=p["temperature"].cpu().numpy(),
                u_accept=p["u_accept"].cpu().numpy(), u_resample=p["u_resample"].cpu().numpy())


def _oracle_one_thread(h, budget_s):
    """Sequences of one host round verified one after another by the oracle
    until ``budget_s`` seconds have passed: (sequences, seconds)."""
    import oracle
    Bq = h["draft_tokens"].shape[0]
    n, t0 = 0, time.perf_counter()
    while True:
        b = n % Bq
        oracle.verify_sample_seq(h["target"][b], h["draft"][b], h["draft_tokens"][b], h["temperature"][b],
                                 h["u_accept"][b], h["u_resample"][b])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s and n >= 2:
            return n, el


_ORACLE_WORKER = None


def _oracle_worker_init(shm_names, shapes, dtypes, small):
    """Pool initializer: one thread per worker, the round's logits attached
    from the parent's shared memory (nothing is copied)."""
    global _ORACLE_WORKER
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    from multiprocessing import shared_memory

    import numpy as np
    shms = [shared_memory.SharedMemory(name=n) for n in shm_names]
    arrs = [np.ndarray(shape, dtype=np.dtype(dt), buffer=m.buf) for m, shape, dt in zip(shms, shapes, dtypes)]
    _ORACLE_WORKER = (shms, arrs, small)


def _oracle_worker_seq(b):
    import oracle
    _, (tgt, dft), sm = _ORACLE_WORKER
    oracle.verify_sample_seq(tgt[b], dft[b], sm["draft_tokens"][b], sm["temperature"][b], sm["u_accept"][b],
                             sm["u_resample"][b])
    return b


@contextlib.contextmanager
def _oracle_pool(h, cores):
    """A pool of ``cores`` spawned worker processes, each with the host round
    h (logits bf16 as uint16, or fp32) attached from shared memory; warmed
    with one task per worker.  Tasks are sequence indices
    (_oracle_worker_seq)."""
    import multiprocessing as mp
    from multiprocessing import shared_memory

    import numpy as np
    Bq = h["draft_tokens"].shape[0]
    shms, shapes, dtypes = [], [], []
    try:
        for key in ("target", "draft"):
            a = np.ascontiguousarray(h[key])
            m = shared_memory.SharedMemory(create=True, size=a.nbytes)
            np.ndarray(a.shape, dtype=a.dtype, buffer=m.buf)[...] = a
            shms.append(m)
            shapes.append(a.shape)
            dtypes.append(a.dtype.str)
        small = {k: np.asarray(h[k]) for k in ("draft_tokens", "temperature", "u_accept", "u_resample")}
        ctx = mp.get_context("spawn")  # never fork a process that has a CUDA context
        with ctx.Pool(cores, initializer=_oracle_worker_init,
                      initargs=([m.name for m in shms], shapes, dtypes, small)) as pool:
            pool.map(_oracle_worker_seq, [i % Bq for i in range(cores)], chunksize=1)
            yield pool
    finally:
        for m in shms:
            m.close()
            m.unlink()


def _oracle_rw_init(shm_names, shapes, dtypes):
    """Pool initializer for the parity leg: one thread per worker; the round's
    logits are attached from shared memory that the parent rewrites between
    rounds (after every task of the previous round has returned)."""
    global _ORACLE_WORKER
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    from multiprocessing import shared_memory

    import numpy as np
    shms = [shared_memory.SharedMemory(name=n) for n in shm_names]
    arrs = [np.ndarray(shape, dtype=np.dtype(dt), buffer=m.buf) for m, shape, dt in zip(shms, shapes, dtypes)]
    _ORACLE_WORKER = (shms, arrs, None)


def _oracle_rw_verify(task):
    """The oracle's verification of sequence b of the attached round."""
    import oracle
    b, toks, T, ua, ur = task
    _, (tgt, dft), _ = _ORACLE_WORKER
    return b, oracle.verify_sample_seq(tgt[b], dft[b], toks, T, ua, ur)


def _oracle_rw_alpha(task):
    """Acceptance rates alpha_j = sum_x min(p_j(x), q_j(x)) of sequence b's
    draft positions (empty for a greedy sequence)."""
    import numpy as np

    import oracle
    b, T = task
    if not T > 0:
        return b, []
    _, (tgt, dft), _ = _ORACLE_WORKER

    def wide(x):
        return oracle.bf16_bits_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)
    out = []
    for j in range(dft.shape[1]):
        pj = oracle.row_probs(wide(tgt[b, j]), T)
        qj = oracle.row_probs(wide(dft[b, j]), T)
        out.append(float(np.minimum(pj, qj).sum()))
    return b, out


@contextlib.contextmanager
def _oracle_rw_pool(h, cores):
    """``cores`` spawned workers with shared-memory arrays shaped like host
    round h's logits; yields (pool, [target, draft] arrays to fill)."""
    import multiprocessing as mp
    from multiprocessing import shared_memory

    import numpy as np
    shms, shapes, dtypes, arrs = [], [], [], []
    try:
        for key in ("target", "draft"):
            a = np.ascontiguousarray(h[key])
            m = shared_memory.SharedMemory(create=True, size=a.nbytes)
            shms.append(m)
            shapes.append(a.shape)
            dtypes.append(a.dtype.str)
            arrs.append(np.ndarray(a.shape, dtype=a.dtype, buffer=m.buf))
        ctx = mp.get_context("spawn")  # never fork a process that has a CUDA context
        with ctx.Pool(cores, initializer=_oracle_rw_init,
                      initargs=([m.name for m in shms], shapes, dtypes)) as pool:
            yield pool, arrs
    finally:
        for m in shms:
            m.close()
            m.unlink()


def cpu_baseline(sv, pool_rounds, dev, stream, budget_s=40.0, max_rounds=100):
    """The fp64 oracle, as it stands, on the host cores, and the parity of the
    GPU path against it on the bench workload.

    One thread: sequences of the first round one after another for a few
    seconds.  All cores: a pool of spawned processes verifies every sequence
    of up to ``max_rounds`` distinct rounds (the timed pool's rounds first,
    then more of the same recipe) within about ``budget_s`` seconds; the
    baseline value is rounds over the pool's verification time.  Each of those
    rounds also goes through spec_verify_sample once (with the debug outputs)
    and its tokens are compared with the oracle's: exact, excused (a uniform
    within 1e-6 of the boundary it was compared with) or unexcused; p(d) and
    q(d) against the oracle's; and the realised acceptance rate alpha (mean of
    sum_x min(p_j, q_j) over the draft positions) with the mean tokens per
    round against (1 - alpha^(gamma+1)) / (1 - alpha)."""
    import numpy as np
    import torch

    import oracle
    import workloads as wl
    h0 = _round_to_host(pool_rounds[0])
    Bq, g = h0["draft_tokens"].shape
    n1, el1 = _oracle_one_thread(h0, min(4.0, budget_s))
    single = {"value": round(n1 / Bq / el1, 4), "cores": 1,
              "sample": f"{n1} sequences of one B={Bq} round ({n1 / Bq:.2f} rounds) in {el1:.1f} s, numpy fp64"}
    cores = os.cpu_count() or 1
    out = torch.empty((Bq, g + 1), dtype=torch.int32, device=dev)
    num = torch.empty((Bq,), dtype=torch.int32, device=dev)
    dbg = torch.empty((Bq, g + 1, 4), dtype=torch.float32, device=dev)
    ws = sv.make_workspace(Bq, g, h0["target"].shape[2], device=dev)
    exact = excused = unexcused = 0
    max_perr = 0.0
    alphas, counts, worst = [], [], []
    t_oracle, rounds = 0.0, 0
    t_start = time.perf_counter()
    with _oracle_rw_pool(h0, cores) as (opool, arrs):
        while rounds < max_rounds and (rounds < 2 or time.perf_counter() - t_start < budget_s):
            p = pool_rounds[rounds] if rounds < len(pool_rounds) else wl.torch_round("batched", 9000 + rounds, dev)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                sv.spec_verify_sample(p["target"], p["draft"], p["draft_tokens"], p["temperature"], p["u_accept"],
                                      p["u_resample"], out, num, ws, out_debug=dbg)
            st = sv.spec_verify_status(ws, stream)
            if st != sv.SPEC_OK:
                raise SystemExit(f"device status in the parity leg: {sv.error_string(st)}")
            tok_h, num_h, dbg_h = out.cpu().numpy(), num.cpu().numpy(), dbg.cpu().numpy()
            h = _round_to_host(p)
            arrs[0][...] = h["target"]
            arrs[1][...] = h["draft"]
            tasks = [(b, h["draft_tokens"][b], float(h["temperature"][b]), h["u_accept"][b],
                      float(h["u_resample"][b])) for b in range(Bq)]
            t0 = time.perf_counter()
            res = dict(opool.map(_oracle_rw_verify, tasks, chunksize=1))
            t_oracle += time.perf_counter() - t0
            for b, a in opool.map(_oracle_rw_alpha, [(b, float(h["temperature"][b])) for b in range(Bq)], chunksize=1):
                alphas += a
            for b in range(Bq):
                r = res[b]
                counts.append(int(num_h[b]) + 1)
                if int(num_h[b]) == r.n and [int(x) for x in tok_h[b]] == r.tokens:
                    exact += 1
                elif r.margin < 1e-6:
                    excused += 1
                else:
                    unexcused += 1
                    worst.append({"round": rounds, "b": b, "oracle": r.tokens, "gpu": [int(x) for x in tok_h[b]],
                                  "margin": r.margin})
                if r.path != "greedy":
                    for j in range(g):
                        max_perr = max(max_perr, abs(float(dbg_h[b, j, 0]) - r.p_tok[j]),
                                       abs(float(dbg_h[b, j, 1]) - r.q_tok[j]))
            rounds += 1
            if rounds > len(pool_rounds):
                del p
    del ws
    alpha = float(np.mean(alphas)) if alphas else float("nan")
    closed = float(oracle.expected_tokens_per_round(alpha, g)) if alphas else float("nan")
    parity = {"rounds": rounds, "sequences": rounds * Bq, "exact": exact, "excused": excused,
              "unexcused": unexcused, "window": 1e-6, "max_prob_err": max_perr, "prob_atol": 1e-5,
              "alpha_realised": round(alpha, 5), "tokens_per_round": round(float(np.mean(counts)), 4),
              "tokens_per_round_closed_form": round(closed, 4), "unexcused_cases": worst[:5],
              "how": ("every sequence of the timed pool's rounds and further rounds of the same recipe: "
                      "spec_verify_sample (one call per round, debug outputs on) against the fp64 oracle "
                      "run in the cpu_baseline leg's worker pool; alpha = mean over sampled draft positions "
                      "of sum_x min(p_j, q_j); closed form (1 - alpha^(gamma+1)) / (1 - alpha) at that "
                      "mean alpha")}
    base = {"value": round(rounds / t_oracle, 4), "unit": "rounds/s", "cores": cores, "kind": "oracle",
            "sample": (f"{rounds * Bq} sequences of {rounds} distinct B={Bq} rounds in {t_oracle:.1f} s of pool "
                       f"time, numpy fp64, {cores} spawned worker processes, one sequence per task"),
            "single_thread": single}
    return base, parity


def other_workloads(sv, dev, stream, args):
    """Rounds/s of the other configurations (same timing method, fewer steps)."""
    import torch

    import workloads as wl
    res = {}
    for name, steps, pool_n in (("single", 2000, 16), ("longdraft", 200, 2)):
        c = wl.CONFIGS[name]
        pool = [wl.torch_round(name, r, dev) for r in range(pool_n)]
        b, g, v = c["B"], c["gamma"], c["V"]
        esize = 2 if c["dtype"] == "bf16" else 4
        nb = sum(counted_bytes(b, g, v, esize, int((p["temperature"] > 0).sum().item())) for p in pool) / pool_n
        w = sv.make_workspace(b, g, v, device=dev)
        o = torch.empty((b, g + 1), dtype=torch.int32, device=dev)
        n = torch.empty((b,), dtype=torch.int32, device=dev)

        def st(i, pool=pool, w=w, o=o, n=n):
            p = pool[i % len(pool)]
            sv.spec_verify_sample(p["target"], p["draft"], p["draft_tokens"], p["temperature"],
                                  p["u_accept"], p["u_resample"], o, n, w)
        torch.cuda.synchronize()  # inputs built on the default stream are complete
        with torch.cuda.stream(stream):
            st(0)
        torch.cuda.synchronize()
        loop = GraphLoop(st, steps, stream)
        loop.run()
        el = loop.run()
        del loop
        assert sv.spec_verify_status(w, stream) == sv.SPEC_OK
        rps = steps / el
        res[name] = {"rounds_per_s": round(rps, 1), "us_per_round": round(el / steps * 1e6, 2),
                     "logit_gbs": round(rps * nb / 1e9, 1), "frac_of_8tbs": round(rps * nb / 1e9 / NOMINAL_HBM_GBS, 4),
                     "B": b, "gamma": g, "V": v, "logits_dtype": c["dtype"], "steps": steps}
        del pool
        torch.cuda.empty_cache()
    res["topkp"] = topkp_workload(sv, dev, stream)
    res["multi"] = multi_workload(sv, dev, stream)
    res["lmhead"] = lmhead_workload(sv, dev, stream)
    res["centroid"] = centroid_workload(sv, dev, stream)
    return res


def topkp_workload(sv, dev, stream, steps=1000, top_k=64, top_p=0.95):
    """The batched workload with top-k / top-p truncation of p and q
    (top_k=64, top_p=0.95): rounds/s and the logit GB/s the call streams."""
    import torch

    import workloads as wl
    B, g, v = 32, 4, 262144
    pool = [wl.torch_round("batched", r, dev) for r in range(POOL)]
    w = sv.make_topkp_workspace(B, g, v, device=dev)
    o = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    nn = torch.empty((B,), dtype=torch.int32, device=dev)

    def st(i):
        p = pool[i % len(pool)]
        sv.spec_verify_sample_topkp(p["target"], p["draft"], p["draft_tokens"], p["temperature"],
                                    p["u_accept"], p["u_resample"], top_k, top_p, o, nn, w)

    torch.cuda.synchronize()  # inputs built on the default stream are complete
    with torch.cuda.stream(stream):
        st(0)
    torch.cuda.synchronize()
    loop = GraphLoop(st, steps, stream)
    loop.run()
    el = loop.run()
    del loop
    assert sv.spec_verify_status(w, stream) == sv.SPEC_OK
    nb = sum(counted_bytes(B, g, v, 2, int((p["temperature"] > 0).sum().item())) for p in pool) / len(pool)
    rps = steps / el
    res = {"rounds_per_s": round(rps, 1), "us_per_round": round(el / steps * 1e6, 2),
           "logit_gbs": round(rps * nb / 1e9, 1), "frac_of_8tbs": round(rps * nb / 1e9 / NOMINAL_HBM_GBS, 4),
           "B": B, "gamma": g, "V": v, "logits_dtype": "bf16", "top_k": top_k, "top_p": top_p, "steps": steps}
    del pool
    torch.cuda.empty_cache()
    return res


def multi_workload(sv, dev, stream, steps=1000):
    """Several draft candidates per sequence: B=8 sequences x 4 candidates,
    gamma=4, V=262144, bf16, greedy (candidates of a sequence share row 0).
    Rounds/s and the logit GB/s the call streams."""
    import torch

    import workloads as wl
    B, n, g, v = 8, 4, 4, 262144
    pool = []
    for r in range(3):  # 3 x 83.9 MB > L2
        p = wl.torch_round("batched", r, dev, B=B * n, temperature=0.0)
        t = p["target"].view(B, n, g + 1, v).clone()
        t[:, 1:, 0, :] = t[:, :1, 0, :]
        pool.append(dict(target=t.contiguous(), draft_tokens=p["draft_tokens"].view(B, n, g).contiguous()))
        del p
    w = sv.make_workspace(B * n, g, v, device=dev)
    o = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    nn = torch.empty((B,), dtype=torch.int32, device=dev)
    ch = torch.empty((B,), dtype=torch.int32, device=dev)

    def st(i):
        p = pool[i % len(pool)]
        sv.spec_verify_greedy_multi(p["target"], p["draft_tokens"], o, nn, w, out_choice=ch)

    torch.cuda.synchronize()  # inputs built on the default stream are complete
    with torch.cuda.stream(stream):
        st(0)
    torch.cuda.synchronize()
    loop = GraphLoop(st, steps, stream)
    loop.run()
    el = loop.run()
    del loop
    assert sv.spec_verify_status(w, stream) == sv.SPEC_OK
    nb = B * n * (g + 1) * v * 2
    rps = steps / el
    res = {"rounds_per_s": round(rps, 1), "us_per_round": round(el / steps * 1e6, 2),
           "logit_gbs": round(rps * nb / 1e9, 1), "frac_of_8tbs": round(rps * nb / 1e9 / NOMINAL_HBM_GBS, 4),
           "B": B, "n_cand": n, "gamma": g, "V": v, "logits_dtype": "bf16", "mode": "greedy", "steps": steps}
    del pool
    torch.cuda.empty_cache()
    return res


def load_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    return 1900.0, "fallback 1.9 PFLOP/s"


def lmhead_workload(sv, dev, stream, steps=200):
    """Fused lm_head + verify: B=64, gamma=4, V=262144, H=1536 (hidden ~ N(0,1),
    W ~ N(0, 0.02^2), T=1).  Whole-chain rounds/s, and the lm_head GEMM kernel
    alone against the tensor and HBM rooflines."""
    import torch

    import workloads as wl
    c = wl.CONFIGS["lmhead"]
    b, g, v, h = c["B"], c["gamma"], c["V"], c["H"]
    pool = [wl.torch_lmhead_round(0, dev)]
    pool.append(wl.torch_lmhead_round(1, dev, W=pool[0]["W"]))
    w = sv.make_workspace(b, g, v, h, device=dev)
    o = torch.empty((b, g + 1), dtype=torch.int32, device=dev)
    n = torch.empty((b,), dtype=torch.int32, device=dev)

    def st(i, fn=sv.spec_verify_lmhead_sample):
        p = pool[i % len(pool)]
        fn(p["hidden"], p["W"], p["draft"], p["draft_tokens"], p["temperature"], p["u_accept"],
           p["u_resample"], o, n, w)

    def gemm(i):
        st(i, sv.spec_verify_lmhead_gemm_only)

    torch.cuda.synchronize()  # inputs built on the default stream are complete
    with torch.cuda.stream(stream):
        st(0)
    torch.cuda.synchronize()
    assert sv.spec_verify_status(w, stream) == sv.SPEC_OK
    loop = GraphLoop(st, steps, stream)
    loop.run()
    el = loop.run()
    del loop
    assert sv.spec_verify_status(w, stream) == sv.SPEC_OK
    gl = GraphLoop(gemm, steps, stream)
    gl.run()
    gs = gl.run() / steps
    del gl
    R = b * (g + 1)
    flops = 2.0 * R * v * h
    w_bytes = v * h * 2
    store_bytes = b * g * v * 4  # fp32 rows j < gamma (all sequences sample at T=1)
    part_bytes = R * (v // 128) * 16
    peak_t, tk = load_tensor_peak()
    peak_b, bk = load_peaks()
    t_floor = max(flops / (peak_t * 1e12), w_bytes / (peak_b * 1e9))
    res = {"rounds_per_s": round(steps / el, 1), "us_per_round": round(el / steps * 1e6, 2),
           "B": b, "gamma": g, "V": v, "H": h, "steps": steps,
           "gemm_kernel": {"kernel": "lmhead_kernel (tcgen05, M=128 vocabulary x N=hidden-row chunks, K=64 stages); "
                                     "timed without the draft rows its row warps stream in a whole round",
                           "avg_launch_us": round(gs * 1e6, 2),
                           "achieved_tflops": round(flops / gs / 1e12, 1), "peak_tflops": peak_t,
                           "tensor_frac": round(flops / gs / 1e12 / peak_t, 4), "tensor_peak_source": tk,
                           "algorithmic_bytes": w_bytes + R * h * 2 + store_bytes + part_bytes,
                           "hbm_gbs": round((w_bytes + R * h * 2 + store_bytes + part_bytes) / gs / 1e9, 1),
                           "hbm_peak_gbs": peak_b, "hbm_peak_source": bk,
                           "roofline_floor_us": round(t_floor * 1e6, 2),
                           "frac_of_roofline": round(t_floor / gs, 4),
                           "roofline": "max(GEMM FLOPs at the bf16 tensor peak, W bytes at HBM bandwidth)"}}
    del pool
    torch.cuda.empty_cache()
    return res


def centroid_workload(sv, dev, stream, steps=500):
    """The centroid-masked draft head (V=262,144, H=1,536, 2,048 clusters, top
    32) for R=4 draft rows (one sequence, gamma=4) and R=128 (32 sequences),
    and the batched workload verified against sparse draft rows of 4,096
    candidates (random tokens, logits = the target's + N(0, 0.3^2))."""
    import torch

    import workloads as wl
    c = wl.CENTROID
    m = wl.torch_centroid_model(dev)
    V, H, Nc, K = m["V"], m["H"], m["n_clusters"], c["top_k"]
    peak, _ = load_peaks()
    res = {"V": V, "H": H, "n_clusters": Nc, "top_k": K}
    g = torch.Generator(device=dev)
    g.manual_seed(2024)
    for R in (4, 128):
        hids = [torch.randn(R, H, generator=g, device=dev).to(torch.bfloat16) for _ in range(4)]
        ot = torch.empty((R, 8192), dtype=torch.int32, device=dev)
        ol = torch.empty((R, 8192), dtype=torch.float32, device=dev)
        oc = torch.empty((R,), dtype=torch.int32, device=dev)
        ws = sv.make_centroid_head_workspace(R, Nc, K, device=dev)

        def st(i, hids=hids, ot=ot, ol=ol, oc=oc, ws=ws):
            sv.spec_centroid_head(hids[i % 4], m["centroids"], m["W_ord"], m["cluster_off"], m["ord2tok"], K,
                                  ot, ol, oc, ws)
        torch.cuda.synchronize()  # inputs built on the default stream are complete
        with torch.cuda.stream(stream):
            st(0)
        torch.cuda.synchronize()
        cand = float(oc.float().mean().item())
        loop = GraphLoop(st, steps, stream)
        loop.run()
        el = loop.run()
        del loop
        assert sv.spec_verify_status(ws, stream) == sv.SPEC_OK
        nbytes = Nc * H * 2 + R * H * 2 + R * cand * (H * 2 + 16)  # centroids, hidden, gathered rows, outputs
        us = el / steps * 1e6
        res[f"head_R{R}"] = {"us_per_call": round(us, 2), "candidates_per_row": round(cand, 1),
                             "bytes_per_call": int(nbytes), "gbs": round(nbytes / us / 1e3, 1),
                             "frac_of_measured_hbm": round(nbytes / us / 1e3 / peak, 4), "steps": steps}
    del m
    torch.cuda.empty_cache()
    # sparse verification of the batched workload
    B, gam, v = 32, 4, 262144
    pool = [wl.torch_round("batched", r, dev) for r in range(POOL)]
    rounds = []
    for p in pool:
        rows = B * gam
        keys = torch.rand(rows, v, generator=g, device=dev)
        tok = torch.sort(torch.topk(keys, 4096, dim=1).indices, dim=1).values.to(torch.int32)
        del keys
        tgt = p["target"][:, :gam, :].reshape(rows, v).float()
        lg = (torch.gather(tgt, 1, tok.long()) + 0.3 * torch.randn(rows, 4096, generator=g, device=dev)).contiguous()
        del tgt
        cnt = torch.full((rows,), 4096, dtype=torch.int32, device=dev)
        T = p["temperature"].repeat_interleave(gam)[:, None]
        u = torch.rand(rows, 4096, generator=g, device=dev).clamp_(min=1e-20)
        pick = torch.argmax(lg / T - torch.log(-torch.log(u)), dim=1)
        dtok = torch.gather(tok, 1, pick[:, None]).view(B, gam).contiguous()
        rounds.append(dict(tok=tok, lg=lg, cnt=cnt, d=dtok))
    wsv = sv.make_sparse_workspace(B, gam, v, device=dev)
    o = torch.empty((B, gam + 1), dtype=torch.int32, device=dev)
    n = torch.empty((B,), dtype=torch.int32, device=dev)

    def sp(i):
        p, q = pool[i % len(pool)], rounds[i % len(pool)]
        sv.spec_verify_sample_sparse(p["target"], q["tok"], q["lg"], q["cnt"], q["d"], p["temperature"],
                                     p["u_accept"], p["u_resample"], o, n, wsv)
    torch.cuda.synchronize()  # inputs built on the default stream are complete
    with torch.cuda.stream(stream):
        sp(0)
    torch.cuda.synchronize()
    loop = GraphLoop(sp, 1000, stream)
    loop.run()
    el = loop.run()
    del loop
    assert sv.spec_verify_status(wsv, stream) == sv.SPEC_OK
    nb = B * (gam + 1) * v * 2 + B * gam * 4096 * 8
    rps = 1000 / el
    res["sparse_verify"] = {"rounds_per_s": round(rps, 1), "us_per_round": round(el / 1000 * 1e6, 2),
                            "bytes_per_round": nb, "gbs": round(rps * nb / 1e9, 1),
                            "frac_of_measured_hbm": round(rps * nb / 1e9 / peak, 4), "B": B, "gamma": gam, "V": v,
                            "candidates_per_row": 4096, "logits_dtype": "bf16", "steps": 1000}
    del pool, rounds
    torch.cuda.empty_cache()
    return res


def run_only_centroid(args):
    import torch

    import speculative_decoding_verification_54_gb300 as sv
    from speculative_decoding_verification_54_gb300 import _build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    sv.load()
    stream = torch.cuda.Stream(device=dev)
    res = centroid_workload(sv, dev, stream, steps=max(3, min(args.steps, 1000)))
    print(json.dumps({"workload": "centroid", **res}), flush=True)


def run_only_topkp(args):
    import torch

    import speculative_decoding_verification_54_gb300 as sv
    from speculative_decoding_verification_54_gb300 import _build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    sv.load()
    stream = torch.cuda.Stream(device=dev)
    res = topkp_workload(sv, dev, stream, steps=max(3, min(args.steps, 2000)))
    print(json.dumps({"workload": "topkp", **res}), flush=True)


def run_only_multi(args):
    import torch

    import speculative_decoding_verification_54_gb300 as sv
    from speculative_decoding_verification_54_gb300 import _build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    sv.load()
    stream = torch.cuda.Stream(device=dev)
    res = multi_workload(sv, dev, stream, steps=max(3, min(args.steps, 1000)))
    print(json.dumps({"workload": "multi", **res}), flush=True)


def run_only_lmhead(args):
    import torch

    import speculative_decoding_verification_54_gb300 as sv
    from speculative_decoding_verification_54_gb300 import _build
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _build.build()
    sv.load()
    stream = torch.cuda.Stream(device=dev)
    res = lmhead_workload(sv, dev, stream, steps=max(3, min(args.steps, 1000)))
    print(json.dumps({"workload": "lmhead", **res}), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    ws_n, rank, _ = dist_setup()
    if rank != 0:
        return
    import numpy as np

    import workloads as wl
    inp = wl.make_round("batched", 0)
    cores = os.cpu_count() or 1
    # every step verifies `cores` sequences at once, one per spawned worker
    # process; the run is bounded to about two minutes: whole sequences when
    # that fits, else the first V' logits of each row (V' >= 4096)
    est_seq_s = 0.08
    total = args.steps + args.warmup
    frac = min(1.0, 120.0 / max(1, total) / est_seq_s)
    Vs = V if frac >= 1.0 else max(4096, int(V * frac) // 8 * 8)
    h = dict(target=np.ascontiguousarray(inp.target[:, :, :Vs]), draft=np.ascontiguousarray(inp.draft[:, :, :Vs]),
             draft_tokens=np.minimum(inp.draft_tokens, Vs - 1), temperature=inp.temperature,
             u_accept=inp.u_accept, u_resample=inp.u_resample)
    with _oracle_pool(h, cores) as pool:
        t0 = None
        for i in range(total):
            if i == args.warmup:
                t0 = time.perf_counter()
            pool.map(_oracle_worker_seq, [(i * cores + c) % B for c in range(cores)], chunksize=1)
        el = time.perf_counter() - t0
    rounds = args.steps * cores * (Vs / V) / B
    value = rounds / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "rounds/s",
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "gamma": GAMMA, "V": V, "logits_dtype": "bf16"},
        "cpu_baseline": {"value": round(value, 4), "unit": "rounds/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step verifies {cores} sequences of a B={B} round at once, one per "
                                   f"spawned worker process"
                                   + ("" if Vs == V else f", over their first {Vs} vocabulary entries")
                                   + "; value scaled to whole rounds"},
        "e2e": {"value": round(value, 4), "unit": "rounds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=40.0,
                    help="wall-time budget of the oracle baseline and parity leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end host-buffer leg")
    ap.add_argument("--row-loads", choices=("ldg", "tma"), default=None,
                    help="row-reducer load path (default: the library's default, direct loads)")
    ap.add_argument("--only", choices=("lmhead", "topkp", "centroid", "multi"), default=None,
                    help="run one extra workload alone and print its figures (diagnostics, profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        args.steps = 100 if args.steps is None else args.steps
        args.warmup = 3 if args.warmup is None else args.warmup
        run_reference(args)
    else:
        if args.row_loads:
            os.environ["SPECV_ROW_LOADS"] = args.row_loads
        args.steps = 20000 if args.steps is None else args.steps
        args.warmup = 20 if args.warmup is None else max(3, args.warmup)
        if args.only == "lmhead":
            run_only_lmhead(args)
        elif args.only == "topkp":
            run_only_topkp(args)
        elif args.only == "centroid":
            run_only_centroid(args)
        elif args.only == "multi":
            run_only_multi(args)
        else:
            run_ours(args)


if __name__ == "__main__":
    main()
