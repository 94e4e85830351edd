"""Benchmark: tree/DAG-packed attention forward + backward on GB300.

One step = one pass of the whole hot path over one synthetic episode batch: the forward
(O, lse) and the backward (delta, dQ, dK/dV, reduction), through the C ABI, with the plan
built once (it is reused by every layer with the same topology; planning time is reported
separately and included in the end-to-end figure).  Default workload: the mount-heavy DAG
(4 independent DAGs of 65,536 rows; a 4,096-row producer span mounted by 32 readers each;
GQA 16/4, head_dim 128, page 64; bf16 inputs ~ N(0,1)/sqrt(128)).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own episode batch of the same shape on its own GPU
(weak scaling, no data-path collective); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from dag_packed_paged_gb300 import workloads as W  # noqa: E402

METRIC = "tree-packed attention fwd & fwd+bwd useful TFLOP/s, % of GB300 BF16 peak"
WORKLOADS = {
    "tiny_tree": 0, "balanced_tree": 1, "commander_worker_dag": 2, "irregular_tree": 3,
    "mount_heavy": 4,
}
DESCRIPTION = {
    0: "tiny tree: 256-row root, 3 x 128-row branches, 1 mount; GQA 4/1, D=64, page 16",
    1: "balanced rollout tree: 4096-row root, fan-out 4 at depth 1 and 2, 2048-row edges; GQA 16/4, D=128, page 64",
    2: "commander-worker DAG: 8192-row root, 8 workers of U[8192,32768] rows, 12 mounts of 1-4 pages; GQA 16/4, D=128, page 64",
    3: "irregular rollout tree: 64 trajectories, lognormal(7,1) edges, unaligned forks, expanded/compact 5.53; GQA 32/8, D=128, page 64",
    4: "mount-heavy: 4 DAGs x 65,536 rows, 4096-row producer span mounted by 32 readers each; GQA 16/4, D=128, page 64",
}
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
NOMINAL_BF16_TFLOPS = 2250.0   # GB300 dense bf16 tensor-core peak, nominal (the measured peaks are the denominators)
KERNEL_SOURCES = {"dkdv": ("bwd.cu",), "dq": ("bwd.cu",), "fwd": ("fwd_pair.cu", "fwd_store.cuh")}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel] + ("ptx.cuh",):
        h.update(open(os.path.join(ROOT, "dag_packed_paged_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    source of that kernel (the summary records the source hash); otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
            if parts[2] == kernel_hash(kernel):
                return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_uuid=None, path=None):
        self.proc = None
        self.path = path or os.path.join(tempfile.gettempdir(), f"treeattn_clocks_{os.getpid()}.csv")
        self.uuid = dev_uuid

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200"]
            if self.uuid:
                cmd.insert(1, f"--id={self.uuid}")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        load = [r for r in rows if r[2] > 200.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank number over all ranks (the step time of a weak-scaling job)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(seed: int, rank: int) -> int:
    """Every rank runs its own episode batch of the same shape."""
    return seed + rank


def rank_episode(make, world: int, rank: int):
    """The rank's share of a global batch of `world` episodes (seeds 0 .. world-1) of one shape:
    the batch's independent DAGs (no row of one is visible to another, so no collective is
    needed in the attention) are placed on the ranks by the replica assignment of HARTS Section
    3.2 on their compact rows, and the rank's DAGs are packed into one strip, in batch order.
    Weak scaling: each rank gets one episode's worth of DAGs.  With one rank the strip is the
    episode itself.  Returns the rank's episode, the placement summary and the indices (in the
    global batch) of the rank's DAGs."""
    import dag_packed_paged_gb300 as ta
    units = []
    for s in range(world):
        ep = make()
        ep.seed = s
        units += W.split_dags(ep)
    work = np.array([u.n_rows for u in units], dtype=np.int64)
    pl = ta.tree_attn_place_units(work, world)
    mine = [u for u, r in zip(units, pl["replica_of"]) if r == rank]
    loads = np.bincount(pl["replica_of"], weights=work, minlength=world)
    ep = W.concat_episodes(mine, name=units[0].name.split("/dag")[0], seed=rank_seed(0, rank))
    info = {"dags": len(units), "dags_per_rank": np.bincount(pl["replica_of"], minlength=world).tolist(),
            "max_rank_rows": int(pl["max_replica_work"]), "imbalance": float(loads.max() / loads.mean()),
            "placement": "independent DAGs of the global batch on ranks by the replica assignment of "
                         "HARTS Section 3.2 (compact rows); no collective in the attention"}
    return ep, info, [i for i, r in enumerate(pl["replica_of"]) if r == rank]


def bf16_dev(bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def cpu_baseline(ep, t, target_s=15.0, seed=0):
    """The fp64 CPU oracle, as it stands, on a bounded sample of query rows of the same
    workload: forward, dQ and the rows' dK/dV contributions.  Useful FLOPs are counted with
    the same convention as the GPU (14 * D * Hq * visible pairs of the sampled rows)."""
    import oracle
    from oracle import dag
    rng = np.random.default_rng(seed)
    N = ep.n_rows

    def run(rows):
        iv = dag.visible_intervals(ep.branches, ep.mounts, rows)
        t0 = time.perf_counter()
        f = oracle.forward(ep.branches, ep.mounts, t.q, t.k, t.v, ep.softmax_scale, intervals=iv)
        b = oracle.backward(ep.branches, ep.mounts, t.q, t.k, t.v, t.do, ep.softmax_scale, f)
        dt = time.perf_counter() - t0
        pairs = int((iv[3] - iv[2]).sum())
        return dt, pairs, b.threads

    # size the sample from a probe, then correct once: the probe's fixed costs make a
    # straight extrapolation undershoot
    n = 32
    dt, pairs, _ = run(rng.choice(N, n, replace=False))
    for _ in range(2):
        n = int(min(4096, max(16, n * target_s / max(dt, 1e-3))))
        dt, pairs, threads = run(rng.choice(N, n, replace=False))
        if dt >= 0.6 * target_s or n >= 4096:
            break
    flops = 14.0 * ep.head_dim * ep.num_q_heads * pairs
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "seconds": round(dt, 2),
            "sample": f"{n} seeded random query rows of the same workload ({pairs} visible pairs): fp64 forward, "
                      f"dQ and their dK/dV contributions, on {threads} host threads"}


def run_reference(args, ep, world, rank):
    """The reference arm: the CPU oracle, timed as it stands on bounded samples."""
    if rank != 0:
        return
    t = W.make_tensors(ep)
    import oracle
    from oracle import dag
    rng = np.random.default_rng(123)
    oracle.build()
    rows_per_step = 48
    total_pairs, total_s, threads = 0, 0.0, 0
    for step in range(args.warmup + args.steps):
        rows = rng.choice(ep.n_rows, rows_per_step, replace=False)
        iv = dag.visible_intervals(ep.branches, ep.mounts, rows)
        t0 = time.perf_counter()
        f = oracle.forward(ep.branches, ep.mounts, t.q, t.k, t.v, ep.softmax_scale, intervals=iv)
        b = oracle.backward(ep.branches, ep.mounts, t.q, t.k, t.v, t.do, ep.softmax_scale, f)
        dt = time.perf_counter() - t0
        threads = b.threads
        if step >= args.warmup:
            total_s += dt
            total_pairs += int((iv[3] - iv[2]).sum())
    flops = 14.0 * ep.head_dim * ep.num_q_heads * total_pairs
    value = flops / total_s / 1e12
    sample = f"{rows_per_step} seeded random query rows per step: fp64 forward, dQ and their dK/dV contributions"
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(ep, args), "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(ep, args, stats=None):
    desc = DESCRIPTION[WORKLOADS[args.workload]]
    if getattr(args, "scale", 1) != 1:
        desc = f"{desc} -- every length divided by {args.scale} (profiling case)"
    cfg = {"workload": desc, "name": args.workload, "rows": ep.n_rows,
           "branches": int(len(ep.branches)), "mounts": int(len(ep.mounts)),
           "heads_q": ep.num_q_heads, "heads_kv": ep.num_kv_heads, "head_dim": ep.head_dim,
           "page_size": ep.page_size, "seed": ep.seed}
    in_bytes = ep.n_rows * (2 * ep.num_q_heads + 2 * ep.num_kv_heads) * ep.head_dim * 2
    cfg["l2"] = (f"inputs ({in_bytes / 1e9:.2f} GB of Q, K, V, dO) larger than the 129 MB L2; no flush between steps"
                 if in_bytes > 129e6 else f"inputs ({in_bytes / 1e6:.1f} MB) fit in L2: not a timing workload")
    if stats:
        cfg["pairs"] = int(stats["pairs"])
        cfg["fwd_useful_tflop"] = stats["fwd_flops"] / 1e12
        cfg["fwdbwd_useful_tflop"] = (stats["fwd_flops"] + stats["bwd_flops"]) / 1e12
    return cfg


def run_rope(args, ep):
    """RoPE of Q and the K pool at the plan's positions, timed alone (HBM-bound): one JSON line
    with the algorithmic bytes (every Q and K element read and written once) per second."""
    import torch
    import dag_packed_paged_gb300 as ta
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    t = W.make_tensors(ep)
    pool = W.make_pool(ep, t)
    N, Hq, Hkv, D = ep.n_rows, ep.num_q_heads, ep.num_kv_heads, ep.head_dim
    plan = ta.tree_attn_plan(ep.branches, ep.mounts, pool.page_table, num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=D, page_size=ep.page_size, num_pages=pool.k_pool.shape[0])
    q = bf16_dev(t.q, dev)
    k_pool = bf16_dev(pool.k_pool, dev)
    for _ in range(args.warmup):
        ta.tree_attn_rope(plan, q, k_pool, 1e4)
    stream = torch.cuda.current_stream(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for _ in range(args.steps):
        ta.tree_attn_rope(plan, q, k_pool, 1e4)       # inputs (Q + K > L2) stream from HBM each call
    ev[1].record(stream)
    torch.cuda.synchronize()
    ta.tree_attn_check(plan)
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    nbytes = 2 * N * (Hq + Hkv) * D * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, kind = load_peaks()
    print(json.dumps({
        "metric": "rope_hbm_throughput", "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "rows": N, "heads": [Hq, Hkv], "head_dim": D},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None, "peak_kind": f"HBM copy ({kind})",
                     "algorithmic": f"{nbytes / 1e9:.3f} GB per launch (Q and K read and written once)"},
        "gpu_launches": args.steps}))


def run_logprob(args, ep, vocab=151_936):
    """Compact-to-semantic log-probabilities (forward + backward) over the episode's compact rows
    with a 151,936-token vocabulary; HBM-bound: the logits are read once forward, read once and
    the logit gradient written once backward."""
    import torch
    import dag_packed_paged_gb300 as ta
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    C = ep.n_rows
    pr, pt, _ = W.semantic_positions(ep, vocab, seed=ep.seed)
    gen = torch.Generator(device=dev)
    gen.manual_seed(ep.seed + 17)
    z = (torch.randn((C, vocab), generator=gen, device=dev) * 3.0).to(torch.bfloat16)
    g = torch.randn(len(pr), generator=gen, device=dev)
    pos_row = torch.from_numpy(pr).to(dev)
    pos_tgt = torch.from_numpy(pt).to(dev)
    ptr_h, pos_h = ta.tree_attn_logprob_index(pr, pt, C, vocab)
    row_ptr, row_pos = torch.from_numpy(ptr_h).to(dev), torch.from_numpy(pos_h).to(dev)
    lse = torch.empty(C, dtype=torch.float32, device=dev)
    lp = torch.empty(len(pr), dtype=torch.float32, device=dev)
    dz = torch.empty_like(z)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        ta.tree_attn_logprob_fwd(z, pos_row, pos_tgt, lse, lp)

    def bwd():
        ta.tree_attn_logprob_bwd(z, lse, row_ptr, row_pos, pos_tgt, g, dz)

    for _ in range(args.warmup):
        fwd()
        bwd()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    torch.cuda.synchronize()
    fwd_ms = bwd_ms = 0.0
    for _ in range(args.steps):                   # logits (13.7 GB at the default) >> L2
        ev[0].record(stream)
        fwd()
        ev[1].record(stream)
        bwd()
        ev[2].record(stream)
        torch.cuda.synchronize()
        fwd_ms += ev[0].elapsed_time(ev[1])
        bwd_ms += ev[1].elapsed_time(ev[2])
    fwd_ms /= args.steps
    bwd_ms /= args.steps
    fwd_bytes, bwd_bytes = C * vocab * 2, 2 * C * vocab * 2
    gbs = (fwd_bytes + bwd_bytes) / ((fwd_ms + bwd_ms) * 1e-3) / 1e9
    peaks, kind = load_peaks()
    print(json.dumps({
        "metric": "logprob_hbm_throughput", "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": fwd_ms + bwd_ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "compact_rows": C, "semantic_positions": int(len(pr)), "vocab": vocab},
        "kernel_ms": {"fwd": fwd_ms, "bwd": bwd_ms},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"], "traffic": None, "peak_kind": f"HBM copy ({kind})",
                     "algorithmic": f"{fwd_bytes / 1e9:.2f} GB forward + {bwd_bytes / 1e9:.2f} GB backward"},
        "gpu_launches": 3 * args.steps}))


def time_workload(name, args, dev, peaks):
    """Device-resident forward + backward of another workload, timed like the headline (plan
    reused, inputs resident, CUDA events on the launching stream, per-kernel trace events):
    its useful TFLOP/s, fractions of the peak and kernel times, for the JSON line."""
    import torch
    import dag_packed_paged_gb300 as ta
    ep = W.config(WORKLOADS[name])
    t = W.make_tensors(ep)
    pool = W.make_pool(ep, t)
    N, Hq, Hkv, D = ep.n_rows, ep.num_q_heads, ep.num_kv_heads, ep.head_dim
    plan = ta.tree_attn_plan(ep.branches, ep.mounts, pool.page_table, num_q_heads=Hq, num_kv_heads=Hkv,
                             head_dim=D, page_size=ep.page_size, num_pages=pool.k_pool.shape[0])
    st = ta.tree_attn_plan_stats(plan)
    q, k_pool, v_pool, d_o = (bf16_dev(x, dev) for x in (t.q, pool.k_pool, pool.v_pool, t.do))
    del t, pool
    o = torch.empty((N, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, N), dtype=torch.float32, device=dev)
    dq = torch.empty((N, Hq, D), dtype=torch.float32, device=dev)
    dk_pool = torch.zeros(k_pool.shape, dtype=torch.float32, device=dev)
    dv_pool = torch.zeros(v_pool.shape, dtype=torch.float32, device=dev)
    ws = torch.empty(max(ta.tree_attn_bwd_workspace_size(plan), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ta.tree_attn_fwd(plan, q, k_pool, v_pool, o, lse)
        ta.tree_attn_bwd(plan, q, k_pool, v_pool, o, lse, d_o, dq, dk_pool, dv_pool, ws)

    for _ in range(args.warmup):
        step()
    ta.tree_attn_check(plan)
    K = args.steps
    trace = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(K)]
    for evs in trace:
        for e in evs:
            e.record(stream)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with ClockSampler(None, None) as clocks:
        time.sleep(0.2)
        ev0.record(stream)
        for k in range(K):
            ta.tree_attn_set_trace_events(plan, trace[k])
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    ta.tree_attn_set_trace_events(plan, None)
    ta.tree_attn_check(plan)
    ms = ev0.elapsed_time(ev1) / K

    def avg(a, b):
        return sum(trace[k][a].elapsed_time(trace[k][b]) for k in range(K)) / K

    kern_ms = {"fwd": avg(0, 1), "delta": avg(2, 3), "dq": avg(3, 4), "dkdv": avg(4, 5), "reduce": avg(5, 6)}
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    fwd_tflops = st["fwd_flops"] / kern_ms["fwd"] / 1e9
    fb_tflops = (st["fwd_flops"] + st["bwd_flops"]) / ms / 1e9
    out = {"workload": DESCRIPTION[WORKLOADS[name]], "rows": N, "pairs": int(st["pairs"]), "steps": K,
           "warmup": args.warmup, "ms_per_step": ms, "fwd_tflops": fwd_tflops, "fwdbwd_tflops": fb_tflops,
           "fwd_frac_of_peak": fwd_tflops / burst, "fwdbwd_frac_of_peak": fb_tflops / burst,
           "fwd_frac_of_nominal": fwd_tflops / NOMINAL_BF16_TFLOPS,
           "fwdbwd_frac_of_nominal": fb_tflops / NOMINAL_BF16_TFLOPS,
           "kernel_ms": {k: round(v, 4) for k, v in kern_ms.items()}, "clocks": clocks.summary(),
           "gpu_launches": K * (1 + (1 if st["n_fwd_split"] > 0 else 0) + 3 + (1 if st["n_partial_slots"] > 0 else 0))}
    del plan
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="mount_heavy", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--clock-log", default=None, help="keep the raw nvidia-smi clock samples in this CSV file")
    ap.add_argument("--scale", type=int, default=1,
                    help="divide every length of the workload by this factor (a small case of the same shape, for "
                         "profiler captures; not a benchmark line)")
    ap.add_argument("--also", default="commander_worker_dag,irregular_tree",
                    help="comma-separated workloads also timed (device-resident fwd + bwd) at N = 1 and "
                         "reported under other_workloads; empty for none")
    ap.add_argument("--op", default="attention", choices=["attention", "rope", "logprob"],
                    help="attention: the forward + backward step (the headline); rope: the RoPE kernel alone; "
                         "logprob: compact log-probabilities forward + backward (vocabulary 151,936)")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference", "at least 3 warm-up steps"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    ep = W.config(WORKLOADS[args.workload])
    placement = None

    if args.impl == "reference":
        run_reference(args, ep, world, rank)
        return
    if args.op == "rope":
        run_rope(args, ep)
        return
    if args.op == "logprob":
        run_logprob(args, ep)
        return

    import torch
    import torch.distributed as dist
    import dag_packed_paged_gb300 as ta

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    make = (lambda: W.config(WORKLOADS[args.workload])) if args.scale == 1 else \
        (lambda: W.scaled(WORKLOADS[args.workload], args.scale))
    ep, placement, _ = rank_episode(make, world, rank)
    t = W.make_tensors(ep)
    pool = W.make_pool(ep, t)
    N, Hq, Hkv, D = ep.n_rows, ep.num_q_heads, ep.num_kv_heads, ep.head_dim

    def plan_now():
        return ta.tree_attn_plan(ep.branches, ep.mounts, pool.page_table, num_q_heads=Hq, num_kv_heads=Hkv,
                                 head_dim=D, page_size=ep.page_size, num_pages=pool.k_pool.shape[0])

    plan_times = []
    for _ in range(3):
        t0 = time.perf_counter()
        plan = plan_now()
        plan_times.append(1000 * (time.perf_counter() - t0))
    st = ta.tree_attn_plan_stats(plan)
    q = bf16_dev(t.q, dev)
    k_pool = bf16_dev(pool.k_pool, dev)
    v_pool = bf16_dev(pool.v_pool, dev)
    d_o = bf16_dev(t.do, dev)
    o = torch.empty((N, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, N), dtype=torch.float32, device=dev)
    dq = torch.empty((N, Hq, D), dtype=torch.float32, device=dev)
    dk_pool = torch.zeros(pool.k_pool.shape, dtype=torch.float32, device=dev)
    dv_pool = torch.zeros(pool.v_pool.shape, dtype=torch.float32, device=dev)
    ws = torch.empty(max(ta.tree_attn_bwd_workspace_size(plan), 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ta.tree_attn_fwd(plan, q, k_pool, v_pool, o, lse)
        ta.tree_attn_bwd(plan, q, k_pool, v_pool, o, lse, d_o, dq, dk_pool, dv_pool, ws)

    cold = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for w in range(args.warmup):
        if w == 0:
            cold[0].record(stream)
        step()
        if w == 0:
            cold[1].record(stream)
    ta.tree_attn_check(plan)

    # ---------------------------------------------------------------- timed region
    K = args.steps
    trace = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(K)]
    for evs in trace:                          # torch creates the CUDA event on first record
        for e in evs:
            e.record(stream)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(uuid if rank == 0 else None, args.clock_log) as clocks:
        time.sleep(0.3)
        ev0.record(stream)
        for k in range(K):
            ta.tree_attn_set_trace_events(plan, trace[k])
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        time.sleep(0.2)
    ta.tree_attn_set_trace_events(plan, None)
    if world > 1:
        dist.barrier()
    ta.tree_attn_check(plan)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / K, dev)

    def avg(a, b):
        return sum(trace[k][a].elapsed_time(trace[k][b]) for k in range(K)) / K

    n_reduce = st["n_partial_slots"] > 0
    n_fwd_split = st["n_fwd_split"] > 0
    kern_ms = {"fwd": avg(0, 1), "delta": avg(2, 3), "dq": avg(3, 4), "dkdv": avg(4, 5), "reduce": avg(5, 6)}
    # per-step times (first kernel's start to last kernel's end) and the first warm-up step,
    # the one that ran with cold caches and TLBs
    step_times = sorted(trace[k][0].elapsed_time(trace[k][6]) for k in range(K))
    step_ms = {"median": round(statistics.median(step_times), 4), "min": round(step_times[0], 4),
               "max": round(step_times[-1], 4), "cold": round(cold[0].elapsed_time(cold[1]), 4) if args.warmup else None}
    flops_fwd, flops_bwd = st["fwd_flops"], st["bwd_flops"]
    base = ep.head_dim * ep.num_q_heads * st["pairs"]
    algo = {"fwd": 4 * base, "dq": 6 * base, "dkdv": 8 * base}
    dominant = max(("fwd", "dq", "dkdv"), key=lambda k: kern_ms[k])
    peaks, peak_kind = load_peaks()
    sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    burst = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    achieved = algo[dominant] / kern_ms[dominant] / 1e9
    # the committed DRAM bytes are for the full-size workload: a --scale run reports none
    traffic = recorded_traffic(dominant, args.workload) if args.scale == 1 else None
    value = (flops_fwd + flops_bwd) * world / ms / 1e9
    fwd_tflops = flops_fwd / kern_ms["fwd"] / 1e9

    # ---------------------------------------------------------------- end to end, host buffers
    # Every step plans its episode on the host, copies its inputs from pinned host memory and
    # reads every output back.  Steps are pipelined the way a training loop feeds a GPU: four
    # sets of device buffers rotate, the copies run on their own streams, and plans are built
    # and freed in stream order (TA_PLAN_STREAM_ORDERED), each one step ahead of its use.  Step
    # i's input copy overlaps the attention of the steps before it (dO last: only the backward
    # needs it); O and lse are read back while the backward runs, dQ while the dK/dV
    # kernel runs (the plan's trace event after the dQ kernel), dK/dV at the end.  With four
    # buffer sets each copy has three steps of compute to finish in: a host<->device copy can
    # run several times slower than its usual rate while other processes load the host's
    # memory, which with two sets would leave the GPU idle.  The
    # timed region starts before the first step's copy and planning and ends after the last
    # step's outputs are on the host.
    e2e = None
    if not args.no_e2e:
        NB = 4
        h_in = [torch.from_numpy(a.view(np.int16)).pin_memory() for a in (t.q, pool.k_pool, pool.v_pool, t.do)]
        d_in = [[q, k_pool, v_pool, d_o]] + [[torch.empty_like(x) for x in (q, k_pool, v_pool, d_o)]
                                             for _ in range(NB - 1)]
        d_out = [[o, lse, dq, dk_pool, dv_pool]] + [[torch.empty_like(x) for x in (o, lse, dq, dk_pool, dv_pool)]
                                                    for _ in range(NB - 1)]
        h_out = [[torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in d_out[0]] for _ in range(NB)]
        h2d = sum(h.numel() * h.element_size() for h in h_in)
        d2h = sum(h.numel() * h.element_size() for h in h_out[0])
        comp_s, h2d_s, d2h_s = (torch.cuda.Stream(dev) for _ in range(3))
        in_fwd = [torch.cuda.Event() for _ in range(NB)]
        in_ready = [torch.cuda.Event() for _ in range(NB)]
        fwd_done = [torch.cuda.Event() for _ in range(NB)]
        dq_done = [torch.cuda.Event() for _ in range(NB)]
        comp_done = [torch.cuda.Event() for _ in range(NB)]
        out_read = [torch.cuda.Event() for _ in range(NB)]
        for b in range(NB):                     # mark every buffer set free
            comp_done[b].record(comp_s)
            out_read[b].record(d2h_s)
            dq_done[b].record(comp_s)           # creates the event the library records
        e2e_steps = max(20, K)

        def plan_async():
            return ta.tree_attn_plan(ep.branches, ep.mounts, pool.page_table, num_q_heads=Hq,
                                     num_kv_heads=ep.num_kv_heads, head_dim=D, page_size=ep.page_size,
                                     num_pages=pool.k_pool.shape[0], flags=ta.TA_PLAN_STREAM_ORDERED,
                                     stream=comp_s)

        def e2e_step(i, p2, last):
            """Step i on buffer set i mod NB with its plan p2, built during step i-1 (None for the
            first step, which plans while its inputs are copied).  Returns (p2, step i+1's plan):
            the next plan is built once step i's kernels and copies are queued, so that its
            upload has a whole step to finish in (a copy engine busy with the large input
            copies can hold a small upload back for tens of ms); None after the last step."""
            b = i % NB
            h2d_s.wait_event(comp_done[b])                    # step i-NB has finished reading set b
            with torch.cuda.stream(h2d_s):
                for dv_, hv in zip(d_in[b][:3], h_in[:3]):   # q, k_pool, v_pool
                    dv_.view(torch.int16).copy_(hv, non_blocking=True)
                in_fwd[b].record(h2d_s)
                d_in[b][3].view(torch.int16).copy_(h_in[3], non_blocking=True)
            in_ready[b].record(h2d_s)
            if p2 is None:
                p2 = plan_async()
            ta.tree_attn_set_trace_events(p2, [None, None, None, None, dq_done[b], None, None])
            comp_s.wait_event(in_fwd[b])
            comp_s.wait_event(out_read[b])                    # step i-NB's outputs are on the host
            qq, kk, vv, dd = d_in[b]
            oo, ll, gq, gk, gv = d_out[b]
            ta.tree_attn_fwd(p2, qq, kk, vv, oo, ll, stream=comp_s)
            fwd_done[b].record(comp_s)
            comp_s.wait_event(in_ready[b])
            ta.tree_attn_bwd(p2, qq, kk, vv, oo, ll, dd, gq, gk, gv, ws, stream=comp_s)
            comp_done[b].record(comp_s)
            for ready, idx in ((fwd_done[b], (0, 1)), (dq_done[b], (2,)), (comp_done[b], (3, 4))):
                d2h_s.wait_event(ready)                       # O, lse | dQ | dK, dV
                with torch.cuda.stream(d2h_s):
                    for k_ in idx:
                        h_out[b][k_].copy_(d_out[b][k_], non_blocking=True)
            out_read[b].record(d2h_s)
            return p2, (None if last else plan_async())      # host planner; upload ordered on comp_s

        warm, nxt = [], None                                  # untimed: one use of each buffer set
        for i in range(NB):
            cur, nxt = e2e_step(i, nxt, i + 1 == NB)
            warm.append(cur)
        torch.cuda.synchronize(dev)
        ta.tree_attn_check(warm[-1], comp_s)
        del warm
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp_s)
        h2d_s.wait_event(e0)
        d2h_s.wait_event(e0)
        plans, nxt = [], None
        for i in range(e2e_steps):
            cur, nxt = e2e_step(i, nxt, i + 1 == e2e_steps)
            plans.append(cur)
            if len(plans) > NB:
                plans.pop(0)                                  # freed in comp_s order, after its use
        comp_s.wait_stream(d2h_s)
        comp_s.wait_stream(h2d_s)
        e1.record(comp_s)
        torch.cuda.synchronize(dev)
        ta.tree_attn_check(plans[-1], comp_s)
        del plans
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
        e2e = {"value": (flops_fwd + flops_bwd) * world / e2e_ms / 1e9, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms,
               "steps": e2e_steps, "includes": "per step: plan + H2D of q/k_pool/v_pool/dO from pinned host + fwd "
                                               "+ bwd + D2H of o/lse/dq/dk_pool/dv_pool; steps pipelined over four "
                                               "buffer sets and three streams; pipeline fill and drain inside the "
                                               "timed region"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": dict(workload_config(ep, args, st), sharding=placement),
        "fwd_tflops": fwd_tflops,
        "fwd_frac_of_peak": fwd_tflops / burst, "fwdbwd_frac_of_peak": value / world / burst,
        "fwd_frac_of_nominal": fwd_tflops / NOMINAL_BF16_TFLOPS,
        "fwdbwd_frac_of_nominal": value / world / NOMINAL_BF16_TFLOPS,
        "peak_tflops": {"burst": burst, "sustained": sustained, "kind": peak_kind},
        "kernel_ms": {k: round(v, 4) for k, v in kern_ms.items()},
        "step_ms": step_ms,
        "plan_ms": statistics.median(plan_times),
        "roofline": {"kernel": dominant, "bound": "tensor", "achieved": achieved, "peak": sustained,
                     "unit": "TFLOP/s", "frac": achieved / sustained, "traffic": traffic,
                     "peak_kind": f"bf16 dense, sustained ({peak_kind})",
                     "algorithmic": f"{algo[dominant] / 1e12:.3f} TFLOP per launch ({2 * {'fwd': 2, 'dq': 3, 'dkdv': 4}[dominant]}*D*Hq*pairs)"},
        "gpu_launches": K * (1 + (1 if n_fwd_split else 0) + 3 + (1 if n_reduce else 0)),
        "e2e": e2e,
    }
    # achieved DRAM rate of each attention kernel (the forward's is the paged K/V gather): the
    # bytes per launch of the committed ncu capture, when it matches the current source, over the
    # kernel's time measured above
    dram = {}
    for k in ("fwd", "dq", "dkdv"):
        b = recorded_traffic(k, args.workload) if args.scale == 1 else None
        if b is not None:
            gbs = b / kern_ms[k] / 1e6
            dram[k] = {"bytes_per_launch": b, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"]}
    if dram:
        line["dram"] = dict(dram, peak_gbs=peaks["hbm_gbs"], peak_kind=f"HBM copy ({peak_kind})")
    if rank == 0:
        line["clocks"] = clocks.summary()
        others = [w for w in args.also.split(",") if w and w != args.workload] if world == 1 else []
        if others:
            line["other_workloads"] = {w: time_workload(w, args, dev, peaks) for w in others}
        if world == 1 and not args.no_cpu_baseline:
            try:
                line["cpu_baseline"] = cpu_baseline(ep, t)
            except Exception as ex:  # report, do not hide, a failed baseline
                line["cpu_baseline"] = {"error": str(ex)}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
