"""The multi-GPU path is replicas only: N processes run N independent copies
of the verify pass, and the job's throughput is the bytes all ranks streamed
over the slowest rank's time.  These tests run the host side of that path
on CPU: two gloo ranks on 127.0.0.1, and bench.py's reference arm under
torchrun with two processes (rank 0 reports, rank 1 exits cleanly)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from verify_gemm_gb300 import replicas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_ranks_from_env():
    assert replicas.from_env({}) == replicas.Ranks(1, 0, 0)
    r = replicas.from_env({"WORLD_SIZE": "4", "RANK": "3", "LOCAL_RANK": "1"})
    assert (r.world, r.rank, r.local) == (4, 3, 1)


def test_job_throughput_counts_every_rank_over_the_slowest():
    one = replicas.Ranks(world=1)
    assert replicas.job_gbps(16_335_300_100, 10, 43.0, one) == pytest.approx(3798.9, rel=1e-4)
    two = replicas.Ranks(world=2)
    # two ranks, same per-rank bytes, the job takes the slower rank's time
    assert replicas.job_gbps(1_000_000_000, 5, 2_000.0, two) == pytest.approx(5.0)
    # single process: no process group is needed for the helpers
    assert replicas.max_over_ranks(1.5, one) == 1.5
    replicas.barrier(one)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    ranks = replicas.from_env()
    replicas.init(ranks, "gloo")
    replicas.barrier(ranks)
    local_ms = 100.0 + 50.0 * rank                 # rank 1 is the slow one
    slowest = replicas.max_over_ranks(local_ms, ranks)
    out.put((rank, slowest, replicas.job_gbps(2_000_000_000, 4, slowest, ranks)))
    replicas.barrier(ranks)
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for _, slowest, gbps in results:
        assert slowest == 150.0
        assert gbps == pytest.approx(2e9 * 4 * 2 / 0.150 / 1e9)


def test_bench_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout               # rank 0 alone reports
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    # the line reports what it timed: one sample round per step, on the same
    # config (and exact byte count) as the GPU arm; the full-pass time is a
    # separate, labelled extrapolation
    assert line["config"]["bytes_per_pass"] == 16_335_300_100
    assert line["ms_per_step"] * line["steps"] < 600_000
    assert line["extrapolated_full_pass_ms"] > line["ms_per_step"]
    assert line["cpu_baseline"]["single_thread"]["cores"] == 1


@pytest.mark.parametrize("extra", [["--workload", "fused"], ["--workload", "head", "--fmt", "int4g"]])
def test_bench_reference_arm_without_an_oracle_timing(extra):
    """Workloads the oracle does not time (the fused stack, a configuration
    repacked in another format) make the reference arm print one line that
    says so and exit 0."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--steps", "1", "--warmup", "0", *extra]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unavailable"]
