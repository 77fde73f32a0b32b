"""The multi-GPU path of bench.py on the CPU: replicas only (each rank verifies
its own batch; no collective on the data path).  The plumbing around the
timed region -- the barrier, the max of the elapsed time over ranks and the
whole-job value -- is exercised with world size 2 over gloo, and the
reference arm's rank rule (rank 0 alone runs and prints) through the
environment torchrun sets.  The CPU baseline's pool of spawned oracle
workers is run on a small round."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, ws, port, elapsed, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    n, r, local = bench.dist_setup()
    assert (n, r, local) == (ws, rank, rank)
    bench.dist_init(n, "gloo")
    bench.dist_barrier(n)
    el = bench.dist_max(n, elapsed[rank], "cpu")
    steps = 100
    value = n * steps / el  # the whole-job rounds/s the bench reports
    q.put((rank, el, value))
    bench.dist_barrier(n)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    elapsed = [0.25, 0.40]
    procs = [ctx.Process(target=_replica, args=(r, 2, port, elapsed, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, el, value in got:
        assert el == 0.40                      # every rank sees the slowest rank's time
        assert abs(value - 2 * 100 / 0.40) < 1e-9  # units of all ranks over that time


def test_world_size_one_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(1, 0.5, "cpu") == 0.5
    bench.dist_barrier(1)  # no-op


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "0"], capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)


def test_reference_arm_runs_on_rank_zero_only():
    r1 = _run_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _run_reference({"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"})
    assert r0.returncode == 0
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_oracle_pool_on_all_cores_runs_every_task():
    """The all-cores oracle leg of the bench's cpu_baseline and parity block:
    spawned workers attach the round's logits (fp32 here, bf16 in the bench)
    from shared memory the parent fills, verify one sequence per task and
    report its acceptance rates; every task completes, the results equal the
    oracle's own, and the shared blocks are released."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl
    inp = wl.make_round("tiny", 0)
    h = dict(target=inp.target, draft=inp.draft, draft_tokens=inp.draft_tokens, temperature=inp.temperature,
             u_accept=inp.u_accept, u_resample=inp.u_resample)
    import oracle
    with bench._oracle_rw_pool(h, 2) as (pool, arrs):
        arrs[0][...] = h["target"]
        arrs[1][...] = h["draft"]
        tasks = [(b, h["draft_tokens"][b], float(h["temperature"][b]), h["u_accept"][b],
                  float(h["u_resample"][b])) for b in range(inp.B)]
        got = dict(pool.map(bench._oracle_rw_verify, tasks, chunksize=1))
        alphas = dict(pool.map(bench._oracle_rw_alpha, [(b, float(h["temperature"][b])) for b in range(inp.B)]))
    ref = oracle.verify_sample(inp.target, inp.draft, inp.draft_tokens, inp.temperature, inp.u_accept,
                               inp.u_resample)
    assert [got[b].tokens for b in range(inp.B)] == [r.tokens for r in ref]
    assert all(len(alphas[b]) == inp.gamma and all(0.0 < a <= 1.0 for a in alphas[b]) for b in range(inp.B))
