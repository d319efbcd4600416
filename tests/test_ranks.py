"""bench.py's multi-replica bookkeeping on CPU (gloo, world size 2).

The decode path shards by sequence with no exchange between GPUs, so N GPUs
run N independent replicas; what needs checking without GPUs is the host
side: every rank agrees on the slowest rank's time, the whole-job throughput
counts all replicas, and the reference arm prints one line from rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _torchrun(args, timeout):
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    env = dict(os.environ, OMP_NUM_THREADS="2", PYTHONPATH=ROOT)
    return subprocess.run(cmd, capture_output=True, text=True, timeout=timeout, cwd=ROOT, env=env)


def test_max_over_ranks_without_a_group():
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5


def test_job_throughput_counts_every_replica():
    one = bench.job_tokens_per_s(16, 1, 50.0)
    assert abs(one - 16 / 50e-6) < 1e-6 * one
    assert abs(bench.job_tokens_per_s(16, 4, 50.0) - 4 * one) < 1e-6 * one


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent("""
        import json, os, sys
        import torch.distributed as dist
        import bench
        dist.init_process_group("gloo")
        rank, world = dist.get_rank(), dist.get_world_size()
        mine = [41.0, 57.5][rank]
        slowest = bench.max_over_ranks(mine, dist, "cpu")
        tokens = bench.job_tokens_per_s(16, world, slowest)
        dist.destroy_process_group()
        with open(os.path.join(sys.argv[1], f"rank{rank}.json"), "w") as f:
            json.dump({"rank": rank, "mine": mine, "slowest": slowest, "tokens": tokens}, f)
    """))
    r = _torchrun([str(script), str(tmp_path)], timeout=180)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    assert sorted(d["rank"] for d in lines) == [0, 1]
    for d in lines:
        assert d["slowest"] == 57.5
        assert abs(d["tokens"] - 32 / 57.5e-6) < 1e-3


def test_reference_arm_prints_one_line_from_rank_zero():
    r = _torchrun([os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
                   "--warmup", "0"], timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
