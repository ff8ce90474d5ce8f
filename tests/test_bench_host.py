"""Host-side logic of bench.py: replica aggregation over ranks (gloo, two
processes on CPU) and the JSON contract of the reference (oracle) arm."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(10.0 + 5.0 * rank)
    v = bench.replica_throughput(1_000_000_000, world, t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, t, v))


def test_max_over_ranks_and_replica_value_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == 15.0                    # the slowest rank's time
        assert abs(v - 2 * 1e9 / 15e-3 / 1e9) < 1e-6


def test_single_process_aggregation_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.replica_throughput(2_000_000_000, 1, 1.0) == pytest.approx(2000.0)


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "1", "--steps", "3", "--warmup", "3",
                          "--ref-sample-s", "0.01"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "GB/s" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["config"]["workload"].startswith("tiny_decode")


def test_l2_flush_only_where_the_working_set_fits_in_cache():
    # the tiny decode workload (0.14 MB of K/V) is flushed before every step;
    # the others stream far more than twice the L2 and are not
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    for i, flush in ((1, True), (2, False), (3, False), (4, False), (5, False)):
        w = W.config(i)
        args = argparse.Namespace(gpus=1, partition=0, graph=False, fused=True, concurrent=False)
        l2 = bench._l2_plan(w, args)
        assert l2 > 0 and args.flush is flush, i
        assert ("flushed" in args.l2_note) is flush
        c = bench._config(w, args)
        assert c["workload"] == w.name and c["l2"] == args.l2_note
        assert c["step_calls"] == "pkv_paged_attention_append"
    args.concurrent = True
    assert "beside pkv_paged_prefill" in bench._config(W.config(5), args)["step_calls"]
