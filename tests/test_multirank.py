"""The bench's multi-rank path on CPU (gloo, world size 2): every rank decodes its own batch
(replicas, weak scaling, no data-path collective); only the timing is reduced (max over
ranks) and rank 0 alone reports. Also the reference arm (the CPU oracle) end to end."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, out_q):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        got = bench.max_over_ranks(ms)
        seeds = [bench.input_seed(rank, k) for k in range(3)]
        value = bench.whole_job_beams_per_s(1024, world, got)
        out_q.put((rank, got, seeds, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_is_max_over_ranks_and_inputs_differ():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + (os.getpid() % 200)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, seeds0, v0), (r1, ms1, seeds1, v1) = res
    assert ms0 == ms1 == 15.0                       # every rank reports the slowest rank's time
    assert not set(seeds0) & set(seeds1)            # each rank decodes its own batch
    assert v0 == v1 == pytest.approx(2 * 1024 / 15e-3)  # whole-job beams/s


def test_single_process_max_is_identity():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_prints_one_line():
    env = dict(os.environ)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "tiny_r1_bw4_h2x1_d64_L256_t3", "--steps", "3", "--warmup", "1"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "beams/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
           "tiny_r1_bw4_h2x1_d64_L256_t3", "--steps", "2", "--warmup", "1"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == ""
