"""Host logic of bench.py: the multi-rank harness (barrier, max over ranks,
whole-job value) under two gloo processes on CPU, and the reference arm's
JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    bench.barrier()
    elapsed = 1.0 + rank          # rank 1 is the slow one
    mx = bench.max_over_ranks(elapsed)
    val = bench.job_value(1e9, 10, w, mx)
    agree = (bench.all_ranks(True), bench.all_ranks(rank == 0))   # one rank says no
    bench.barrier()
    dist.destroy_process_group()
    q.put((r, w, lr, mx, val, agree))


def test_two_rank_harness_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[:3] for x in res] == [(0, 2, 0), (1, 2, 1)]
    for _, _, _, mx, val, agree in res:
        assert mx == 2.0                     # the slowest rank's time
        assert val == pytest.approx(1e9 * 10 * 2 / 2.0 / 1e9)
        assert agree == (True, False)        # every rank sees the same decision


def _dying_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import time
    import bench
    bench.init_dist("gloo", timeout_s=5.0)
    if rank == 1:
        os._exit(3)                  # leaves between steps, nothing of its own in flight
    t0 = time.monotonic()
    try:
        bench.barrier()
        q.put(("no error", time.monotonic() - t0))
    except Exception as e:           # noqa: BLE001 - any error is the detection
        q.put((type(e).__name__, time.monotonic() - t0))
    q.close()
    q.join_thread()
    os._exit(0)


def test_rank_that_leaves_ends_the_next_barrier_with_an_error():
    """A rank that exits between steps: the other rank's next barrier raises
    within the process-group timeout instead of waiting for it forever."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dying_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    what, waited = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
    assert what != "no error"
    assert waited < 60
    assert procs[0].exitcode == 0 and procs[1].exitcode == 3


def test_job_value_single():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_value(2e9, 5, 1, 1.0) == pytest.approx(10.0)
    assert bench.max_over_ranks(3.5) == 3.5      # no process group: identity
    assert bench.all_ranks(False) is False and bench.all_ranks(True) is True
    assert bench.host_available_bytes() > 0


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         cwd=ROOT, timeout=300)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s"
    assert line["higher_is_better"] is True and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         cwd=ROOT, env=env, timeout=300)
    assert out.returncode == 0 and out.stdout.strip() == ""


@pytest.mark.parametrize("K", [2, 4, 8])
def test_ring_busbw_matches_the_ring_simulation_traffic(K):
    """The bus bandwidth figure times the launch time equals the bf16 bytes one
    rank sends in the oracle's ring simulation of the same collective."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from oracle import ring
    N, t = 4 * K, 0.5
    x = [np.zeros(N, np.uint16) for _ in range(K)]
    sent = {"rs_fp32_m2": ring.reduce_scatter(x, K)[1].sent[0],
            "allgather": ring.allgather([np.zeros(N // K, np.uint16)] * K, K)[1].sent[0],
            "allreduce": ring.allreduce(x, K)[1].sent[0]}
    for name, elems in sent.items():
        assert bench.ring_busbw(name, K, N, t) * t * 1e9 == pytest.approx(2 * elems)
    assert bench.ring_busbw("flatten", K, N, t) is None


class _HostOnlyWorkload:
    """Stand-in for the bench workload with small host tensors: enough for the
    end-to-end leg's host-memory decision, which runs before any device work."""

    def __init__(self):
        import torch
        self.dev = torch.device("cpu")
        self._in = [torch.zeros(1024, dtype=torch.bfloat16)]
        self._out = [torch.zeros(256, dtype=torch.float32)]

    def inputs(self):
        return self._in

    def outputs(self):
        return self._out


def test_e2e_is_skipped_when_host_memory_cannot_hold_it(monkeypatch):
    """Too little available host memory, or a pinned allocation that fails,
    makes the end-to-end leg report itself skipped instead of failing."""
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args([])
    monkeypatch.setattr(bench, "host_available_bytes", lambda: 0)
    e2e = bench.run_e2e(_HostOnlyWorkload(), args, 1)
    assert e2e["value"] is None and "pinned host memory" in e2e["skipped"]
    import torch
    if not torch.cuda.is_available():
        # plenty of memory, but no CUDA to pin it with: the allocation fails
        monkeypatch.setattr(bench, "host_available_bytes", lambda: 1 << 62)
        e2e = bench.run_e2e(_HostOnlyWorkload(), args, 1)
        assert e2e["value"] is None
