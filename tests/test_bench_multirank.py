"""The benchmark's multi-rank logic on CPU: gloo, world size 2.

Each rank is an independent replica (weak scaling, no data-path collective);
the timed region ends with a barrier and the step time is the max over ranks.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    m = bench.max_over_ranks(local_ms, world)
    dist.barrier()
    q.put((rank, m, bench.whole_job_tflops(1e12, m, world)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]
    # 2 replicas x 1e12 FLOPs in 15 ms each -> whole-job TFLOP/s
    assert abs(res[0][2] - 2 * 1e12 / 15e-3 / 1e12) < 1e-9


def test_single_rank_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.whole_job_tflops(2e12, 1.0, 1) - 2000.0) < 1e-9


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_runs_oracle_on_cpu():
    import json
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1", "--ref-rows", "8"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["unit"] == "TFLOP/s"


def test_varlen_mix_covers_the_tokens_within_the_table_limits():
    """The bench's packed-sequence line regroups each workload's B*S tokens; the mix
    must cover them exactly with positive lengths and fit the library's table
    (1024 sequences, 4096 tiles of 128 rows)."""
    import bench
    import dit_inputs as di
    for w in di.WORKLOADS.values():
        T = w.B * w.S
        lens = bench.varlen_mix(T)
        assert sum(lens) == T and min(lens) >= 1, w.name
        assert len(lens) <= 1024 and sum((n + 127) // 128 for n in lens) <= 4096, w.name
        assert lens == bench.varlen_mix(T)   # seeded: the same mix every run
    assert bench.varlen_mix(4608) == [1697, 746, 1877, 288]


def test_step_percentiles():
    """p10/p50/p90 of the timed steps (linear interpolation), also for one step."""
    import bench
    assert bench.step_percentiles([2.5]) == {"p10": 2.5, "p50": 2.5, "p90": 2.5}
    got = bench.step_percentiles([float(x) for x in range(10, 0, -1)])   # order does not matter
    assert abs(got["p10"] - 1.9) < 1e-12 and abs(got["p50"] - 5.5) < 1e-12 and abs(got["p90"] - 9.1) < 1e-12
