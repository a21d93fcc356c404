"""Benchmark: sparse-FFN decode tokens/s at batch 1 and achieved HBM GB/s
against the roofline, on the OPT-6.7B-shaped FFN layer (d_model 4096, d_ff
16384, predictor rank 256, fp16 weights, fp32 accumulation, 512 decode tokens,
hot-first neuron order from a 1000-token profile pass).

A step is one 512-token decode: every token runs the whole hot path (predictor
h = V x, scores + threshold, fused row gather + ReLU + down projection).  Token
t uses layer replica t mod R: R copies of the layer at distinct addresses, so
that the per-token working set (~37 MB) is not re-read from the 126 MB L2 by
the next token (reuse distance R x 37 MB >= 2 x L2).  The 512 tokens of a step
are one CUDA graph.

Arms: `--impl sffn` (default, the CUDA library through its C ABI) and
`--impl reference` (the CPU oracle on the host cores, a bounded sample per step).
Under torchrun every rank decodes its own tokens on its own GPU (replicas only,
weak scaling): there is no data exchange between ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

if "--cpu-worker" in sys.argv:  # single-threaded BLAS for the timed oracle, before numpy loads
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "c2"
METRIC = "sparse-FFN decode tokens/s at batch 1 and achieved HBM GB/s vs roofline"
L2_BYTES = 126 * 2 ** 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="sffn", choices=["sffn", "reference"])
    p.add_argument("--replicas", type=int, default=8)
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-worker", default=None)
    return p.parse_args()


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.dev)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self):
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip().lower() == "active"})
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": float(np.median(loaded)) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return None


# ---------------------------------------------------------------- the oracle on host cores

def cpu_worker(path, seconds):
    """Runs in a subprocess with single-threaded BLAS: the oracle, as it
    stands, on the stored layer, one token after another until `seconds`."""
    import oracle
    z = np.load(path)
    ol = oracle.OracleLayer(w_up=z["w_up"], w_downT=z["w_downT"], b=z["b"], U=z["U"], V=z["V"], fmt="f16")
    X = z["X"]
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.sparse_ffn(ol, X[done % len(X)], 0.0)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds and done >= 4:
            break
    print(json.dumps({"tokens": done, "seconds": el}))


def run_cpu_baseline(lw, X, seconds):
    from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    try:
        np.savez(path, w_up=st(lw.w_up), w_downT=st(lw.w_downT), b=lw.b.cpu().numpy(), U=st(lw.U), V=st(lw.V),
                 X=st(X[:64, 0]))
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", path, "--cpu-seconds",
                              str(seconds)], capture_output=True, text=True, timeout=seconds * 4 + 120)
        r = json.loads(out.stdout.strip().splitlines()[-1])
    finally:
        os.unlink(path)
    return {"value": r["tokens"] / r["seconds"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{r['tokens']} decode tokens of the same layer (predictor, threshold, compaction, "
                      f"masked FFN in fp64), one thread, {r['seconds']:.1f} s"}


# ---------------------------------------------------------------- the CUDA arm

def bench_sffn(args):
    import torch
    from activation_sparse_decode_gb300 import sffn, workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.get_workload(WORKLOAD)
    T = wl.steps

    # layer, hot-first order from the 1000-token profile pass, replicas
    lw = W.make_layer(wl, seed=0, layer=0, device=dev)
    prof_layer = sffn.Layer.from_weights(lw, tau=wl.tau, max_batch=8)
    ws8 = sffn.new_workspace(sffn.sffn_workspace_size(prof_layer, 8), dev)
    perm, counts = sffn.hot_first_order(prof_layer, W.make_profile_tokens(wl, device=dev), ws8)
    hot_rows = sffn.hot_row_count(counts, wl.profile_tokens)
    expected_active = float(counts.sum().item()) / wl.profile_tokens
    prof_layer.close()
    lw = sffn.permute_layer_weights(lw, torch.from_numpy(perm).to(dev))
    R = max(1, args.replicas)
    reps = [lw] + [W.LayerWeights(w_up=lw.w_up.clone(), w_gate=None, w_downT=lw.w_downT.clone(), b=lw.b.clone(),
                                  U=lw.U.clone(), V=lw.V.clone(), p=lw.p, dtype=lw.dtype, act=lw.act)
                   for _ in range(R - 1)]
    layers = [sffn.Layer.from_weights(r, tau=wl.tau, max_batch=1, hot_rows=hot_rows, expected_active=expected_active)
              for r in reps]
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layers[0], 1), dev)

    X = W.make_tokens(wl, T, batch=1, seed=rank, device=dev)  # [T][1][d] fp16
    Y = torch.empty(T, 1, wl.d_model, dtype=torch.float32, device=dev)
    n_act = torch.empty(T, 1, dtype=torch.int32, device=dev)
    idx_scratch = torch.empty(1, wl.d_ff, dtype=torch.int32, device=dev)

    # active counts of every token (for the algorithmic bytes), outside any timing
    for t in range(T):
        sffn.sffn_forward(layers[t % R], X[t], Y[t], ws, idx_scratch, n_act[t])
    torch.cuda.synchronize()
    n_tok = n_act[:, 0].double().cpu().numpy()

    stream = torch.cuda.Stream(device=dev)

    def step_body():
        for t in range(T):
            sffn.sffn_forward(layers[t % R], X[t], Y[t], ws)

    with torch.cuda.stream(stream):
        step_body()  # eager warm-up of every kernel variant
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_body()
    launches_per_step = T  # one single-launch layer kernel per token

    # ---- device-timed steps (inputs resident in HBM); every replay and event on `stream`
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    clocks = clk.summary()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world)
    ms_per_step = ms_max / args.steps
    value = T * args.steps * world / (ms_max / 1e3)

    # ---- the dominant kernel: the timed graph holds nothing but the layer
    # kernel, one launch per token, so its average launch duration is the
    # device-timed region over the launches in it (inter-launch gaps included,
    # an upper bound).  Events around single launches inside a graph would
    # add their own cost to each launch.
    k_avg_ms = ms / (args.steps * T)
    esz = 2
    gathered = n_tok * wl.d_model * esz * 2  # rows of W_up and W_down^T
    pred_bytes = (wl.rank * wl.d_model + wl.d_ff * wl.rank) * esz + 2 * wl.d_ff * 4  # V, U, both biases
    algo = gathered + pred_bytes + wl.d_model * esz + wl.d_model * 4  # + x read + y written
    achieved_gbs = float(algo.mean()) / (k_avg_ms / 1e3) / 1e9
    gathered_gbs = float(gathered.mean()) / (k_avg_ms / 1e3) / 1e9
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "k_layer_traffic.json")
    if os.path.exists(tpath):
        tj = json.load(open(tpath))
        if tj.get("kernel_source_hash") == kernel_source_hash():
            traffic = tj.get("bytes_per_launch")


    # ---- end to end: pinned host tokens in, host outputs back, every step
    Xh = X.cpu().pin_memory()
    Yh = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(2):
            X.copy_(Xh, non_blocking=True)
            graph.replay()
            Yh.copy_(Y, non_blocking=True)
    torch.cuda.synchronize()
    e_steps = max(3, args.steps // 4)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e_steps):
            X.copy_(Xh, non_blocking=True)
            graph.replay()
            Yh.copy_(Y, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = T * e_steps * world / (e_ms / 1e3)

    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded Zipf/low-rank construction; random weights, no checkpoint)",
        "config": {
            "workload": wl.name,
            "d_model": wl.d_model, "d_ff": wl.d_ff, "rank": wl.rank, "batch": 1, "tokens_per_step": T,
            "act": "relu", "weights": "fp16, fp32 accumulation", "hot_first": True,
            "l2": f"inputs larger than L2: {R} rotating layer replicas "
                  f"({R * (lw.w_up.numel() * 4 + (lw.U.numel() + lw.V.numel()) * 2) / 2**30:.2f} GiB), "
                  f"reuse distance ~{R * 37} MB per token vs {L2_BYTES // 2**20} MB L2",
            "mean_active": round(float(n_tok.mean()), 1),
            "hot_rows": hot_rows,
            "us_per_layer": round(ms_per_step * 1e3 / T, 3),
            "layer_kernel_us_per_launch": round(k_avg_ms * 1e3, 3),
            "kernel_timing": "device-timed graph of single-kernel tokens / launches",
            "predictor_bytes_per_token": int(pred_bytes),
            "gathered_bytes_per_token": round(float(gathered.mean())),
            "gathered_gbs_over_launch": round(gathered_gbs, 1),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "roofline": {
            "kernel": "k_layer (predictor, threshold, row gather, ReLU, down projection: one launch per token)",
            "bound": "hbm",
            "achieved": round(achieved_gbs, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved_gbs / peak, 4),
            "peak_source": "measured" if peaks else "fallback",
            "traffic": traffic,
            "algorithmic_bytes_per_launch": round(float(algo.mean())),
        },
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(Xh.numel() * Xh.element_size()),
                "d2h_bytes_per_step": int(Yh.numel() * Yh.element_size()),
                "wall_s": round(wall, 3)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = run_cpu_baseline(lw, X, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "activation_sparse_decode_gb300", "csrc")
    for name in ("layer_impl.cuh", "common.cuh", "kernels.cuh"):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------- the reference arm (the oracle)

def bench_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    import oracle
    from activation_sparse_decode_gb300 import workloads as W
    from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
    wl = W.get_workload(WORKLOAD)
    lw = W.make_layer(wl, seed=0, layer=0, device="cpu")
    ol = oracle.OracleLayer(w_up=st(lw.w_up), w_downT=st(lw.w_downT), b=lw.b.numpy(), U=st(lw.U), V=st(lw.V),
                            fmt="f16")
    X = st(W.make_tokens(wl, 64, device="cpu"))[:, 0]
    per_step = 4
    for s in range(args.warmup):
        for i in range(per_step):
            oracle.sparse_ffn(ol, X[(s * per_step + i) % 64], 0.0)
    t0 = time.perf_counter()
    for s in range(args.steps):
        for i in range(per_step):
            oracle.sparse_ffn(ol, X[(s * per_step + i) % 64], 0.0)
    el = time.perf_counter() - t0
    v = per_step * args.steps / el
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Zipf/low-rank construction)",
        "config": {"workload": wl.name, "batch": 1, "tokens_per_step": per_step,
                   "note": "CPU oracle, rows in generated order (the hot-first order changes no work)"},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} decode tokens per step, numpy fp64 on the host cores"},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    if args.cpu_worker:
        cpu_worker(args.cpu_worker, args.cpu_seconds)
        return
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_sffn(args)


if __name__ == "__main__":
    main()
