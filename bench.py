"""Benchmark: sparse-FFN decode tokens/s and achieved HBM GB/s against the
roofline.

Default (the headline): the OPT-6.7B-shaped FFN layer at batch 1 (d_model 4096,
d_ff 16384, predictor rank 256, fp16 weights, fp32 accumulation, 512 decode
tokens, hot-first neuron order from a 1000-token profile pass).  A step is one
512-token decode: every token runs the whole hot path (predictor h = V x,
scores + threshold, fused row gather + ReLU + down projection).  Token t uses
layer replica t mod R: R copies of the layer at distinct addresses, so that
the per-token working set (~37 MB) is not re-read from the 126 MB L2 by the
next token (reuse distance R x 37 MB >= 2 x L2).  The 512 tokens of a step are
one CUDA graph.

`--workload c1|c2|c3|c4|c5 --batch B` measures the other workloads the same
way (single layers with rotating replicas; the 40- and 48-layer stacks through
sffn_forward_stack, one graph per step of all decode steps).  Batches of 8-32
tokens run the tensor-core union path; its kernel is timed on its own with
events around each launch.  Single layers also report the no-skip dense FFN
(the library's dense path and two cuBLAS GEMVs) for contrast.

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
DEFAULT_STEPS = {"c1": 300, "c2": 300, "c3": 100, "c4": 10, "c5": 3}
METRIC = "sparse-FFN decode tokens/s at batch 1 and achieved HBM GB/s vs roofline"
L2_BYTES = 126 * 2 ** 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="sffn", choices=["sffn", "reference"])
    p.add_argument("--workload", default=WORKLOAD, choices=["c1", "c2", "c3", "c4", "c5"])
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--row-gather", action="store_true", help="batches: CUDA-core row gather, not the union path")
    p.add_argument("--no-dense", action="store_true", help="skip the dense contrast")
    p.add_argument("--replicas", type=int, default=8)
    p.add_argument("--hot-frac", type=float, default=0.99,
                   help="hot rows: profile frequency at which rows are fetched before the predictor decides")
    p.add_argument("--warm-frac", type=float, default=0.0,
                   help="warm rows (pulled into L2 during the predictor): profile frequency, 0 = none")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-worker", default=None)
    a = p.parse_args()
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.workload]
    return a


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
    ol = oracle.OracleLayer(w_up=z["w_up"], w_downT=z["w_downT"], b=z["b"], U=z["U"], V=z["V"],
                            fmt=str(z["fmt"]), act=str(z["act"]),
                            w_gate=z["w_gate"] if "w_gate" in z.files else None)
    X = z["X"]
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.sparse_ffn(ol, X[done % len(X)], 0.0)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds and done >= 4:
            break
    print(json.dumps({"tokens": done, "seconds": el}))


def run_cpu_baseline(lw, X, seconds, n_layers=1):
    """The oracle on one layer, one token at a time (it has no batched form:
    each token's masked FFN is computed on its own).  For a stack the rate of
    one layer is divided by the number of layers."""
    from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    try:
        arrays = dict(w_up=st(lw.w_up), w_downT=st(lw.w_downT), b=lw.b.cpu().numpy(), U=st(lw.U), V=st(lw.V),
                      X=st(X.reshape(-1, X.shape[-1])[:64]), fmt=np.array(lw.dtype), act=np.array(lw.act))
        if lw.w_gate is not None:
            arrays["w_gate"] = st(lw.w_gate)
        np.savez(path, **arrays)
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", path, "--cpu-seconds",
                              str(seconds)], capture_output=True, text=True, timeout=seconds * 4 + 300)
        r = json.loads(out.stdout.strip().splitlines()[-1])
    finally:
        os.unlink(path)
    what = "decode tokens of the same layer" if n_layers == 1 else \
        f"decode tokens of layer 0 of the {n_layers}-layer stack (rate divided by {n_layers})"
    return {"value": r["tokens"] / r["seconds"] / n_layers, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{r['tokens']} {what} (predictor, threshold, compaction, masked FFN in fp64), "
                      f"one thread, {r['seconds']:.1f} s"}


# ---------------------------------------------------------------- the CUDA arm

ESIZE = {"f32": 4, "f16": 2, "bf16": 2}


def build_layer(sffn, W, wl, layer, dev, hot_frac=0.99, warm_frac=0.0):
    """One layer of the workload; hot-first reordered when the workload asks."""
    import torch
    lw = W.make_layer(wl, seed=0, layer=layer, device=dev)
    hot, ea, warm = 0, 0.0, 0
    if wl.reorder:
        prof = sffn.Layer.from_weights(lw, tau=wl.tau, max_batch=8)
        ws8 = sffn.new_workspace(sffn.sffn_workspace_size(prof, 8), dev)
        perm, counts = sffn.hot_first_order(prof, W.make_profile_tokens(wl, layer=layer, device=dev), ws8)
        hot = sffn.hot_row_count(counts, wl.profile_tokens, hot_frac)
        ea = float(counts.sum().item()) / wl.profile_tokens
        row_bytes = (3 if wl.act == "reglu" else 2) * wl.d_model * ESIZE[wl.dtype]
        warm = sffn.warm_row_count(counts, wl.profile_tokens, row_bytes, warm_frac) if warm_frac > 0 else 0
        prof.close()
        lw = sffn.permute_layer_weights(lw, torch.from_numpy(perm).to(dev))
    return lw, hot, ea, warm


def clone_layer(W, lw):
    return W.LayerWeights(w_up=lw.w_up.clone(), w_gate=None if lw.w_gate is None else lw.w_gate.clone(),
                          w_downT=lw.w_downT.clone(), b=lw.b.clone(), U=lw.U.clone(), V=lw.V.clone(), p=lw.p,
                          dtype=lw.dtype, act=lw.act)


def union_sizes(idx, n):
    """|union of the tokens' active sets| for each step: idx [T][B][f], n [T][B]."""
    out = []
    for t in range(idx.shape[0]):
        sel = [idx[t, b, :n[t, b]] for b in range(idx.shape[1])]
        out.append(np.unique(np.concatenate(sel)).size if sel else 0)
    return np.asarray(out, np.float64)


def bench_sffn(args):
    import torch
    from activation_sparse_decode_gb300 import sffn, workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.get_workload(args.workload)
    B = args.batch
    if B < 1 or B > 32:
        raise SystemExit("--batch must be in [1, 32]")
    T = wl.steps
    L = wl.n_layers
    stack = L > 1
    esz = ESIZE[wl.dtype]
    nm = 2 if wl.act == "reglu" else 1
    d, f, r = wl.d_model, wl.d_ff, wl.rank
    W_words = (f + 31) // 32
    # the layers' weights are written and synchronised before the first call
    # and never written after: batch-1 calls may stage them before the
    # previous kernel on the stream has finished
    flags = (sffn.SFFN_FLAG_ROW_GATHER if args.row_gather else 0) | sffn.SFFN_FLAG_STATIC_WEIGHTS
    union_path = B >= 3 and wl.dtype != "f32" and d % 128 == 0 and not args.row_gather

    # ---- layers: single layers as R rotating replicas, stacks as their L layers
    if stack:
        lws, hots, eas, warms = [], [], [], []
        for l in range(L):
            lw, hot, ea, warm = build_layer(sffn, W, wl, l, dev, args.hot_frac, args.warm_frac)
            lws.append(lw)
            hots.append(hot)
            eas.append(ea)
            warms.append(warm)
        layers = [sffn.Layer.from_weights(lw, tau=wl.tau, max_batch=B, flags=flags, hot_rows=h, expected_active=e,
                                          warm_rows=wr)
                  for lw, h, e, wr in zip(lws, hots, eas, warms)]
        R = 1
        hot_rows = hots[0]
    else:
        lw, hot_rows, ea, warm = build_layer(sffn, W, wl, 0, dev, args.hot_frac, args.warm_frac)
        R = max(1, args.replicas)
        lws = [lw] + [clone_layer(W, lw) for _ in range(R - 1)]
        layers = [sffn.Layer.from_weights(x, tau=wl.tau, max_batch=B, flags=flags, hot_rows=hot_rows,
                                          expected_active=ea, warm_rows=warm) for x in lws]
    torch.cuda.synchronize()
    lw = lws[0]

    X = W.make_tokens(wl, T, batch=B, seed=rank, device=dev)  # [T][B][d]
    if stack:
        ws = sffn.new_workspace(sffn.sffn_stack_workspace_size(layers, B), dev)
        x0 = X[0].contiguous()
        x_out = torch.empty(T, B, d, dtype=x0.dtype, device=dev)
        Y = x_out
    else:
        ws = sffn.new_workspace(sffn.sffn_workspace_size(layers[0], B), dev)
        Y = torch.empty(T, B, d, dtype=torch.float32, device=dev)
    wsl = sffn.new_workspace(sffn.sffn_workspace_size(layers[0], B), dev)  # per-layer calls outside the timing

    # ---- active counts (and unions) for the algorithmic bytes, outside any timing
    idx = torch.empty(B, f, dtype=torch.int32, device=dev)
    nact = torch.empty(B, dtype=torch.int32, device=dev)
    n_list, u_list = [], []
    if stack:
        Tp = min(T, 4)
        trace = torch.empty(Tp, L, B, d, dtype=X.dtype, device=dev)
        xo = torch.empty(Tp, B, d, dtype=X.dtype, device=dev)
        sffn.sffn_forward_stack(layers, x0, Tp, xo, ws, x_trace=trace)
        for t in range(Tp):
            I_t, N_t = [], []
            for l in range(L):
                sffn.sffn_predict(layers[l], trace[t, l], idx, nact, wsl)
                I_t.append(idx.cpu().numpy())
                N_t.append(nact.cpu().numpy())
            n_list.append(np.stack(N_t))                                   # [L][B]
            u_list.append(union_sizes(np.stack(I_t), np.stack(N_t)))       # [L]
        n_tok = np.concatenate([x.reshape(-1) for x in n_list])
        n_union = np.concatenate(u_list)
    else:
        Iall, Nall = [], []
        for t in range(T):
            sffn.sffn_predict(layers[t % R], X[t], idx, nact, wsl)
            Iall.append(idx.cpu().numpy())
            Nall.append(nact.cpu().numpy())
        Iall, Nall = np.stack(Iall), np.stack(Nall)
        n_tok = Nall.reshape(-1).astype(np.float64)
        n_union = union_sizes(Iall, Nall)
    del wsl

    stream = torch.cuda.Stream(device=dev)

    def step_body():
        if stack:
            sffn.sffn_forward_stack(layers, x0, T, x_out, ws)
        else:
            for t in range(T):
                sffn.sffn_forward(layers[t % R], X[t], Y[t], ws)

    with torch.cuda.stream(stream):
        step_body()  # eager warm-up of every kernel variant
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_body()

    # launches of this library's kernels per layer call (the memset of y on the
    # union path is a driver node, not counted)
    groups = (B + 7) // 8
    if B == 1 and not (flags & sffn.SFFN_FLAG_MULTI_KERNEL):
        per_layer = 1 + (1 if stack else 0)  # stacks: the LayerNorm is folded into the next layer's kernel
        launches_per_step = T * L + (1 if stack else 0)
    elif union_path:  # hidden layer, scores (one launch each for the whole batch), union kernel
        per_layer = 3 + (1 if stack else 0)
        launches_per_step = T * L * per_layer
    else:
        per_layer = 2 * groups + (B + 3) // 4 + (1 if stack else 0)
        launches_per_step = T * L * per_layer

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
    value = T * B * args.steps * world / (ms_max / 1e3)
    us_per_layer = ms_per_step * 1e3 / (T * L)

    # ---- algorithmic bytes per layer call
    pred_bytes = (r * d + f * r) * esz + f * 4  # V, U, predictor bias
    io_bytes = B * d * esz + B * d * 4         # tokens in, outputs out
    if union_path:
        gathered = n_union * d * esz * (nm + 1)
        kernel_bytes = gathered + n_union * 4 + B * W_words * 4 + io_bytes  # + gated bias, mask words
    else:
        per_call = n_tok.reshape(-1, B).sum(1) if B > 1 else n_tok
        gathered = per_call * d * esz * (nm + 1)
        kernel_bytes = gathered + pred_bytes + f * 4 + io_bytes  # the single-launch kernel reads both biases
    layer_bytes = float(np.mean(gathered)) + pred_bytes + f * 4 + io_bytes

    # ---- the dominant kernel's average launch duration
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    if union_path:
        kname = "k_union (union gather-GEMM on tcgen05: up/gate, ReLU/ReGLU, down projection)"
        k_ms = time_union_kernel(sffn, layers, X if not stack else None, stack, R, T, L, B, dev, x0 if stack else None)
        ktiming = "events around each union launch, eager (other kernels of the call outside the events)"
    elif B == 1 and not stack:
        kname = "k_layer (predictor, threshold, row gather, ReLU/ReGLU, down projection: one launch per token)"
        k_ms = ms / (args.steps * T)
        ktiming = "device-timed graph of single-kernel tokens / launches"
    elif B == 1:
        kname = "k_layer (one launch per layer and token, LayerNorm of the previous layer folded in)"
        k_ms = ms / (args.steps * (T * L + 1))
        ktiming = "device-timed graph / launches (the final LayerNorm launch included)"
    else:
        kname = "whole layer call (predictor kernels + row-gather passes)"
        k_ms = ms / (args.steps * T * L)
        ktiming = "device-timed graph / layer calls"
    achieved = float(np.mean(kernel_bytes)) / (k_ms / 1e3) / 1e9
    traffic = recorded_traffic(args.workload, B, union_path)

    # ---- end to end: pinned host tokens in, host outputs back, every step
    Xin = x0 if stack else X
    Xh = Xin.cpu().pin_memory()
    Yh = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(2):
            Xin.copy_(Xh, non_blocking=True)
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
            Xin.copy_(Xh, non_blocking=True)
            graph.replay()
            Yh.copy_(Y, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier(world)
    e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = T * B * e_steps * world / (e_ms / 1e3)

    dense = None
    if not stack and not args.no_dense:
        dense = dense_contrast(sffn, torch, lws, layers, X, R, B, dev)

    layer_mb = (lw.w_up.numel() * (nm + 1) + lw.U.numel() + lw.V.numel()) * esz / 2 ** 20
    if stack:
        l2 = f"inputs larger than L2: {L} layers, {layer_mb * L / 1024:.1f} GiB resident"
    else:
        l2 = (f"inputs larger than L2: {R} rotating layer replicas ({layer_mb * R / 1024:.2f} GiB), reuse distance "
              f"~{R * layer_bytes / 2**20:.0f} MB per layer call vs {L2_BYTES // 2**20} MB L2")
    name = "ReGLU" if nm == 2 else "ReLU"
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
        "dtype": wl.dtype,
        "data": "synthetic (seeded Zipf/low-rank construction; random weights, no checkpoint)",
        "config": {
            "workload": wl.name,
            "d_model": d, "d_ff": f, "rank": r, "layers": L, "batch": B, "decode_steps_per_step": T,
            "act": wl.act, "weights": f"{wl.dtype}, fp32 accumulation", "hot_first": bool(wl.reorder),
            "path": ("tensor-core union" if union_path else "single-launch layer kernel" if B == 1
                     else "CUDA-core row gather"),
            "l2": l2,
            "mean_active": round(float(np.mean(n_tok)), 1),
            "mean_union": round(float(np.mean(n_union)), 1) if B > 1 else None,
            "hot_rows": hot_rows,
            "warm_rows": layers[0].desc.warm_rows,
            "us_per_layer": round(us_per_layer, 3),
            "dominant_kernel_us_per_launch": round(k_ms * 1e3, 3),
            "kernel_timing": ktiming,
            "predictor_bytes_per_layer": int(pred_bytes),
            "gathered_bytes_per_layer": round(float(np.mean(gathered))),
            "gathered_gbs_over_kernel": round(float(np.mean(gathered)) / (k_ms / 1e3) / 1e9, 1),
            "layer_gbs": round(layer_bytes / (us_per_layer / 1e6) / 1e9, 1),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "roofline": {
            "kernel": kname,
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": "measured" if peaks else "fallback",
            "traffic": traffic,
            "algorithmic_bytes_per_launch": round(float(np.mean(kernel_bytes))),
        },
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(Xh.numel() * Xh.element_size()),
                "d2h_bytes_per_step": int(Yh.numel() * Yh.element_size()),
                "wall_s": round(wall, 3)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if dense is not None:
        out["dense_contrast"] = dense
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = run_cpu_baseline(lw, X, args.cpu_seconds, L)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def time_union_kernel(sffn, layers, X, stack, R, T, L, B, dev, x0):
    """Average duration of the union kernel: events bracket each union launch
    (sffn_set_profile_events), one call at a time, layers rotating so that the
    rows are not in L2 from the previous call."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layers[0], B), dev)
    y = torch.empty(B, layers[0].d_model, dtype=torch.float32, device=dev)
    calls = [(layers[l], x0) for l in range(L)] if stack else [(layers[t % R], X[t]) for t in range(min(T, 64))]
    for lay, x in calls[:4]:
        sffn.sffn_forward(lay, x, y, ws)
    torch.cuda.synchronize()
    tot, n = 0.0, 0
    e0.record()  # torch creates the CUDA events on first use
    e1.record()
    torch.cuda.synchronize()
    sffn.sffn_set_profile_events(e0, e1)
    try:
        for lay, x in calls:
            sffn.sffn_forward(lay, x, y, ws)
            e1.synchronize()
            tot += e0.elapsed_time(e1)
            n += 1
    finally:
        sffn.sffn_set_profile_events(None, None)
    return tot / n


def dense_contrast(sffn, torch, lws, layers, X, R, B, dev):
    """No-skip FFN for contrast: the library's dense path, and two cuBLAS GEMMs
    (torch.nn.functional.linear) with the activation in between."""
    import torch.nn.functional as F
    T = min(X.shape[0], 32)
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layers[0], B), dev)
    y = torch.empty(B, layers[0].d_model, dtype=torch.float32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def lib():
        for t in range(T):
            sffn.sffn_dense_forward(layers[t % R], X[t], y, ws)

    def cublas():
        for t in range(T):
            w = lws[t % R]
            up = F.linear(X[t], w.w_up)
            if w.w_gate is not None:
                a = torch.relu(F.linear(X[t], w.w_gate) + w.b.to(up.dtype)) * up
            else:
                a = torch.relu(up + w.b.to(up.dtype))
            F.linear(a, w.w_downT.t())

    res = {}
    for name, fn in (("sffn_dense_forward", lib), ("cublas_two_gemv", cublas)):
        fn()
        torch.cuda.synchronize()
        e0.record()
        for _ in range(3):
            fn()
        e1.record()
        e1.synchronize()
        res[name] = round(3 * T * B / (e0.elapsed_time(e1) / 1e3), 1)
    res["unit"] = "tokens/s"
    return res


def recorded_traffic(workload, batch, union_path):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary, when the kernel sources still match the ones it was taken on."""
    if union_path:
        path, key, files = "k_union_traffic.json", f"{workload}_b{batch}", ("union_impl.cuh", "common.cuh",
                                                                           "kernels.cuh", "tcgen05.cuh")
    elif workload == "c2" and batch == 1:
        path, key, files = "k_layer_traffic.json", None, ("layer_impl.cuh", "common.cuh", "kernels.cuh")
    else:
        return None
    tpath = os.path.join(ROOT, "profiles", path)
    if not os.path.exists(tpath):
        return None
    tj = json.load(open(tpath))
    if key is not None:
        tj = tj.get(key, {})
    if tj.get("kernel_source_hash") != kernel_source_hash(files):
        return None
    return tj.get("bytes_per_launch")


def kernel_source_hash(files=("layer_impl.cuh", "common.cuh", "kernels.cuh")):
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "activation_sparse_decode_gb300", "csrc")
    for name in files:
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------- the reference arm (the oracle)

def bench_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from activation_sparse_decode_gb300 import workloads as W
    from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
    wl = W.get_workload(args.workload)
    lw = W.make_layer(wl, seed=0, layer=0, device="cpu")
    ol = oracle.OracleLayer(w_up=st(lw.w_up), w_downT=st(lw.w_downT), b=lw.b.numpy(), U=st(lw.U), V=st(lw.V),
                            fmt=wl.dtype, act=wl.act, w_gate=None if lw.w_gate is None else st(lw.w_gate))
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
    L = wl.n_layers
    v = per_step * args.steps / el / L
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    what = "one layer" if L == 1 else f"layer 0 of {L}, rate divided by {L}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Zipf/low-rank construction)",
        "config": {"workload": wl.name, "batch": 1, "tokens_per_step": per_step,
                   "note": f"CPU oracle, {what}, rows in generated order (the hot-first order changes no work); "
                           "tokens one at a time (the oracle has no batched form)"},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} decode tokens per step, numpy fp64 on the host cores, {what}"},
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
