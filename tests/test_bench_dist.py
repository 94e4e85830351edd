"""The benchmark's multi-rank host logic (world size 2, gloo, CPU): the step time is the
max over ranks, every rank draws its own episode batch of the same shape, and only rank 0
runs the reference arm."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch.distributed as dist
    import bench
    from dag_packed_paged_gb300 import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.5 + 2.0 * rank)
        ep = W.tiny()
        ep.seed = bench.rank_seed(ep.seed, rank)
        q = W.make_tensors(ep).q
        out.put((rank, t, int(q[:4].astype("int64").sum()), ep.n_rows))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, s0, n0), (r1, t1, s1, n1) = res
    assert t0 == t1 == 3.5                      # max over ranks
    assert n0 == n1 and s0 != s1                # same shape, different draws


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench
    from dag_packed_paged_gb300 import workloads as W

    class A:
        steps, warmup = 1, 0

    bench.run_reference(A(), W.tiny(), world=2, rank=1)
    assert capsys.readouterr().out == ""


def test_reference_arm_line_has_the_contract_keys(capsys):
    import json

    import bench
    from dag_packed_paged_gb300 import workloads as W

    class A:
        steps, warmup, workload = 1, 0, "tiny_tree"

    bench.run_reference(A(), W.tiny(), world=1, rank=0)
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    line = json.loads(out[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"] and line["e2e"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["name"] == "tiny_tree"
