"""Benchmark: sparse-FFN decode tokens/s and achieved HBM GB/s against the
roofline, on the five synthetic FFN decode workloads.

Headline (the default line's `value`): the 48-layer OPT-175B-shaped FFN stack
(d_model 12288, d_ff 49152, predictor rank 1024, fp16 weights, fp32
accumulation, hot-first neuron order from a 1000-token profile pass, ~114 GiB
resident) at batch 1.  A step is one 64-token greedy-shaped decode through all
48 layers (sffn_forward_stack: per layer the whole hot path -- predictor
h = V x, scores + threshold, row gather + ReLU + down projection -- and the
residual + LayerNorm folded into the next layer's kernel), captured as one CUDA
graph.  The timed region replays K steps with the weights resident in HBM.

Sub-records (`workloads`, skipped with --no-suite): the ReLU d1024 fp32 layer,
the OPT-6.7B-shaped ReLU layer, the Llama-7B-shaped ReGLU layer at batches
1/4/8/32, the 40-layer OPT-13B-shaped stack, and the 48-layer stack at batch
8.  Each gives tokens/s, us per layer call (mean, p10, p90 over the timed
steps), the dominant kernel's time per launch and its gathered-byte and
total-byte fractions of the measured HBM peak, the active / union counts, the
predictor's band count and its recall and precision against the exact ReLU
mask, and for single layers the no-skip dense FFN (the library's dense path
and two cuBLAS GEMMs, both captured in graphs over the same rotating replicas).
Single layers use R rotating replicas (R x the per-token bytes >= 2 x L2), so
no token finds its rows in L2.

`--workload c1..c5 --batch B` puts one workload in the headline instead.
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

if "--cpu-worker" in sys.argv and "--cpu-threads" in sys.argv:  # BLAS threads, before numpy loads
    _n = sys.argv[sys.argv.index("--cpu-threads") + 1]
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = _n

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "c5"
DEFAULT_STEPS = {"c1": 300, "c2": 300, "c3": 100, "c4": 10, "c5": 20}
SUITE_STEPS = {"c1": 40, "c2": 40, "c3": 20, "c4": 4, "c5": 3}  # sub-record steps (timed), each after >= 3 warm-up steps
# (workload, batch, variant): the stacks also at batch 1 with look-ahead masks,
# the ReGLU layer also on the bundled row layout, the batches also through the
# dense fallback (every row, two GEMMs)
SUITE = [("c1", 1, ""), ("c2", 1, ""), ("c3", 1, ""), ("c3", 4, ""), ("c3", 8, ""), ("c3", 16, ""), ("c3", 32, ""),
         ("c3", 1, "bundled"), ("c3", 8, "bundled"), ("c3", 32, "bundled"), ("c3", 4, "dense"), ("c3", 8, "dense"),
         ("c3", 16, "dense"), ("c3", 32, "dense"), ("c4", 1, ""), ("c4", 1, "lookahead"),
         ("c5", 8, ""), ("c5", 8, "dense"), ("c5", 1, "lookahead")]
METRIC = "sparse-FFN decode tokens/s at batch 1 and achieved HBM GB/s vs roofline"
L2_BYTES = 126 * 2 ** 20
ESIZE = {"f32": 4, "f16": 2, "bf16": 2}
BAND = 1e-4


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="sffn", choices=["sffn", "reference"])
    p.add_argument("--workload", default=WORKLOAD, choices=["c1", "c2", "c3", "c4", "c5"])
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--no-suite", action="store_true", help="headline only, no sub-records")
    p.add_argument("--lookahead", action="store_true",
                   help="stacks at batch 1: look-ahead masks (each layer's mask predicted from the previous input)")
    p.add_argument("--bundled", action="store_true", help="bundled row layout ([gate | up | down] per neuron)")
    p.add_argument("--row-gather", action="store_true", help="batches: CUDA-core row gather, not the union path")
    p.add_argument("--no-dense", action="store_true", help="skip the dense contrast")
    p.add_argument("--no-stats", action="store_true", help="skip band / recall / precision statistics")
    p.add_argument("--replicas", type=int, default=8)
    p.add_argument("--layers", type=int, default=None,
                   help="stacks: run only the first N layers (a smaller case of the same kernels, for profiling)")
    p.add_argument("--hot-frac", type=float, default=0.99,
                   help="hot rows: profile frequency at which rows are fetched before the predictor decides")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-worker", default=None)
    p.add_argument("--cpu-threads", default=None)
    a = p.parse_args()
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.workload]
    if a.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
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


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return None


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


# ---------------------------------------------------------------- the oracle on host cores

def cpu_worker(path, seconds):
    """Runs in a subprocess (BLAS thread count set before numpy loads): the
    oracle, as it stands, on the stored layer, one token after another until
    `seconds` have passed."""
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
        if el >= seconds and done >= 2:
            break
    print(json.dumps({"tokens": done, "seconds": el}))


def run_cpu_baseline(lw, X, seconds, n_layers=1):
    """The oracle on one layer, one token at a time (it has no batched form:
    each token's masked FFN is computed on its own), with one BLAS thread and
    with every host core.  For a stack the rate of one layer is divided by the
    number of layers."""
    from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    cores = host_cores()
    res = {}
    try:
        arrays = dict(w_up=st(lw.w_up), w_downT=st(lw.w_downT), b=lw.b.cpu().numpy(), U=st(lw.U), V=st(lw.V),
                      X=st(X.reshape(-1, X.shape[-1])[:16]), fmt=np.array(lw.dtype), act=np.array(lw.act))
        if lw.w_gate is not None:
            arrays["w_gate"] = st(lw.w_gate)
        np.savez(path, **arrays)
        del arrays
        for threads in (1, cores):
            out = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", path, "--cpu-seconds",
                                  str(seconds), "--cpu-threads", str(threads)],
                                 capture_output=True, text=True, timeout=seconds * 6 + 300)
            res[threads] = json.loads(out.stdout.strip().splitlines()[-1])
    finally:
        os.unlink(path)
    what = "decode tokens of the same layer" if n_layers == 1 else \
        f"decode tokens of layer 0 of the {n_layers}-layer stack (rate divided by {n_layers})"
    rate = {k: v["tokens"] / v["seconds"] / n_layers for k, v in res.items()}
    r = res[cores]
    return {"value": rate[cores], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "single_thread_value": rate[1], "cpu_model": cpu_model(),
            "sample": f"{r['tokens']} {what} (predictor, threshold, compaction, masked FFN in fp64, numpy), "
                      f"BLAS on {cores} threads, {r['seconds']:.1f} s; one thread: {res[1]['tokens']} tokens in "
                      f"{res[1]['seconds']:.1f} s"}


# ---------------------------------------------------------------- workload construction

def build_layer(sffn, W, wl, layer, dev, hot_frac=0.99):
    """One layer of the workload; hot-first reordered when the workload asks."""
    import torch
    lw = W.make_layer(wl, seed=0, layer=layer, device=dev)
    hot, ea = 0, 0.0
    if wl.reorder:
        prof = sffn.Layer.from_weights(lw, tau=wl.tau, max_batch=8)
        ws8 = sffn.new_workspace(sffn.sffn_workspace_size(prof, 8), dev)
        perm, counts = sffn.hot_first_order(prof, W.make_profile_tokens(wl, layer=layer, device=dev), ws8)
        hot = sffn.hot_row_count(counts, wl.profile_tokens, hot_frac)
        ea = float(counts.sum().item()) / wl.profile_tokens
        prof.close()
        lw = sffn.permute_layer_weights(lw, torch.from_numpy(perm).to(dev))
    return lw, hot, ea


def clone_layer(W, lw):
    return W.LayerWeights(w_up=lw.w_up.clone(), w_gate=None if lw.w_gate is None else lw.w_gate.clone(),
                          w_downT=lw.w_downT.clone(), b=lw.b.clone(), U=lw.U.clone(), V=lw.V.clone(), p=lw.p,
                          dtype=lw.dtype, act=lw.act)


class Model:
    """The layers of one workload on the device: a stack's L layers, or R
    rotating replicas of a single layer."""

    def __init__(self, sffn, W, wl, dev, max_batch, replicas, hot_frac, flags):
        import torch
        self.wl = wl
        self.stack = wl.n_layers > 1
        if self.stack:
            built = [build_layer(sffn, W, wl, l, dev, hot_frac) for l in range(wl.n_layers)]
            self.lws = [b[0] for b in built]
            self.hots = [b[1] for b in built]
            self.eas = [b[2] for b in built]
        else:
            lw, hot, ea = build_layer(sffn, W, wl, 0, dev, hot_frac)
            self.lws = [lw] + [clone_layer(W, lw) for _ in range(max(1, replicas) - 1)]
            self.hots = [hot] * len(self.lws)
            self.eas = [ea] * len(self.lws)
        self.layers = [sffn.Layer.from_weights(x, tau=wl.tau, max_batch=max_batch, flags=flags, hot_rows=h,
                                               expected_active=e)
                       for x, h, e in zip(self.lws, self.hots, self.eas)]
        self._args = (sffn, max_batch, flags)
        self.bundled = None
        self.dense = None
        self.balanced = None
        torch.cuda.synchronize()

    def dense_layers(self):
        """The same weights with the dense fallback for every batch of 2 or more."""
        if self.dense is None:
            sffn, max_batch, flags = self._args
            self.dense = [sffn.Layer.from_weights(x, tau=self.wl.tau, max_batch=max_batch, flags=flags, hot_rows=h,
                                                  expected_active=e, dense_min_batch=2)
                          for x, h, e in zip(self.lws, self.hots, self.eas)]
        return self.dense

    def balanced_layers(self):
        """The same weights with the batch-1 kernel's global row balancing."""
        if self.balanced is None:
            sffn, max_batch, flags = self._args
            self.balanced = [sffn.Layer.from_weights(x, tau=self.wl.tau, max_batch=max_batch,
                                                     flags=flags | sffn.SFFN_FLAG_BALANCE, hot_rows=h, expected_active=e)
                             for x, h, e in zip(self.lws, self.hots, self.eas)]
        return self.balanced

    def bundled_layers(self):
        """The same layers on the bundled row layout (copies of the rows)."""
        if self.bundled is None:
            sffn, max_batch, flags = self._args
            self.bundled = [sffn.Layer.from_weights(x, tau=self.wl.tau, max_batch=max_batch, flags=flags, hot_rows=h,
                                                    expected_active=e, bundled=True)
                            for x, h, e in zip(self.lws, self.hots, self.eas)]
        return self.bundled

    def close(self):
        for l in self.layers + (self.bundled or []) + (self.dense or []) + (self.balanced or []):
            l.close()
        self.layers, self.lws, self.bundled, self.dense, self.balanced = [], [], None, None, None


# ---------------------------------------------------------------- statistics outside the timing

def union_sizes(idx, n):
    """|union of the tokens' active sets| per call: idx [C][B][f], n [C][B]."""
    out = []
    for c in range(idx.shape[0]):
        sel = [idx[c, b, :n[c, b]] for b in range(idx.shape[1])]
        out.append(np.unique(np.concatenate(sel)).size if sel else 0)
    return np.asarray(out, np.float64)


def predictor_stats(sffn, torch, layer, lw, x, ws, tau):
    """For one call's tokens x [B][d]: active counts, union size, band count
    (fp32 scores within 1e-4 of tau), and recall / precision of the predicted
    mask against the exact ReLU mask {W_gated[i] . x + b_i > 0} (fp32 GEMM)."""
    B, f = x.shape[0], layer.d_ff
    s = torch.empty(B, f, dtype=torch.float32, device=x.device)
    sffn.sffn_predict_scores(layer, x, s, ws)
    pred = s > tau
    wg = lw.w_gate if lw.w_gate is not None else lw.w_up
    xf = x.float()
    exact = torch.cat([(xf @ wg[i:i + 4096].float().t() + lw.b[i:i + 4096]) > 0 for i in range(0, f, 4096)], 1)
    tp = (pred & exact).sum(1).double()
    return {"n": pred.sum(1).double().cpu().numpy(), "union": float(pred.any(0).sum().item()),
            "band": (s - tau).abs().le(BAND).sum(1).double().cpu().numpy(),
            "tp": tp.cpu().numpy(), "n_exact": exact.sum(1).double().cpu().numpy(), "mask": pred}


def collect_stats(sffn, torch, model, calls, B, dev):
    """calls: list of (layer index, x [B][d]).  Aggregates predictor_stats."""
    ws = sffn.new_workspace(sffn.sffn_workspace_size(model.layers[0], B), dev)
    n, band, tp, ne, un, per_layer_union, jacc = [], [], [], [], [], {}, []
    for li, x in calls:
        r = predictor_stats(sffn, torch, model.layers[li], model.lws[li], x, ws, model.wl.tau)
        n.append(r["n"]); band.append(r["band"]); tp.append(r["tp"]); ne.append(r["n_exact"]); un.append(r["union"])
        per_layer_union.setdefault(li, []).append(r["union"])
        if B > 1:  # mean pairwise Jaccard similarity of the tokens' predicted sets
            m = r["mask"].float()
            inter = m @ m.t()
            cnt = m.sum(1)
            uni = cnt[:, None] + cnt[None, :] - inter
            iu = torch.triu_indices(B, B, 1, device=m.device)
            jacc.append(float((inter[iu[0], iu[1]] / uni[iu[0], iu[1]].clamp_min(1)).mean().item()))
    n, band, tp, ne = (np.concatenate(v) for v in (n, band, tp, ne))
    out = {"mean_active": round(float(n.mean()), 1), "band_per_token": round(float(band.mean()), 3),
           "recall_vs_exact": round(float(tp.sum() / max(ne.sum(), 1)), 4),
           "precision_vs_exact": round(float(tp.sum() / max(n.sum(), 1)), 4),
           "stats_tokens": int(n.size)}
    if B > 1:
        out["mean_union"] = round(float(np.mean(un)), 1)
        out["mean_pairwise_jaccard"] = round(float(np.mean(jacc)), 4)
    return out, np.asarray(un), per_layer_union, n


# ---------------------------------------------------------------- one measurement

def measure(sffn, W, torch, model, B, steps, warmup, dev, world, args, stats=True, dense=True, want_e2e=False,
            variant=""):
    """Times `steps` graph replays of one decode step of `model` at batch B.
    Returns (record, extras) where extras carries what the headline line needs."""
    wl = model.wl
    T, L = wl.steps, wl.n_layers
    stack = model.stack
    R = len(model.layers) if not stack else 1
    d, f, r = wl.d_model, wl.d_ff, wl.rank
    esz = ESIZE[wl.dtype]
    nm = 2 if wl.act == "reglu" else 1
    layers = (model.bundled_layers() if variant == "bundled" else model.dense_layers() if variant == "dense"
              else model.balanced_layers() if variant == "balanced" else model.layers)
    dense_path = variant == "dense" and B >= 2
    union_path = B >= 3 and wl.dtype != "f32" and d % 128 == 0 and not args.row_gather and not dense_path
    rank, _, _ = dist_env()
    lookahead = variant == "lookahead" and stack and B == 1
    opts = sffn.SFFN_STACK_LOOKAHEAD if lookahead else 0

    X = W.make_tokens(wl, T, batch=B, seed=rank, device=dev)  # [T][B][d]
    if stack:
        ws = sffn.new_workspace(sffn.sffn_stack_workspace_size(layers, B), dev)
        x0 = X[0].contiguous()
        Y = torch.empty(T, B, d, dtype=x0.dtype, device=dev)
    else:
        ws = sffn.new_workspace(sffn.sffn_workspace_size(layers[0], B), dev)
        Y = torch.empty(T, B, d, dtype=torch.float32, device=dev)

    # ---- active counts, unions and predictor statistics, outside any timing
    la_rec = {}
    if stack:
        Tp = min(T, 2)
        trace = torch.empty(Tp, L, B, d, dtype=X.dtype, device=dev)
        xo = torch.empty(Tp, B, d, dtype=X.dtype, device=dev)
        Wd = (f + 31) // 32
        mtr = torch.zeros(Tp, L, B, Wd, dtype=torch.int32, device=dev)
        sffn.sffn_forward_stack(layers, x0, Tp, xo, ws, x_trace=trace, mask_trace=mtr, options=opts)
        calls = [(l, trace[t, l]) for t in range(Tp) for l in range(L)]
        if lookahead and stats:
            la_rec = lookahead_stats(sffn, torch, model, trace, mtr, dev)
    else:
        calls = [(t % R, X[t]) for t in range(min(T, 64))]
    st_rec, unions, per_layer_union, n_tok = collect_stats(sffn, torch, model, calls if stats else calls[:4], B, dev)
    if not stats:
        st_rec = {k: v for k, v in st_rec.items() if k in ("mean_active", "mean_union")}
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)

    def step_body():
        if stack:
            sffn.sffn_forward_stack(layers, x0, T, Y, ws, options=opts)
        else:
            for t in range(T):
                sffn.sffn_forward(layers[t % R], X[t], Y[t], ws)

    with torch.cuda.stream(stream):
        step_body()  # eager warm-up of every kernel variant
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step_body()

    # launches of this library's kernels per step (the memset of y on the union
    # path is a driver node, not counted)
    groups = (B + 7) // 8
    if B == 1:
        # stacks: LayerNorm folded into the next layer's kernel, one closing
        # LayerNorm launch; look-ahead: one predictor-only launch first
        launches_per_step = T * L + (1 if stack else 0) + (1 if lookahead else 0)
    elif union_path:  # hidden layer, scores (one launch each for the whole batch), union kernel
        launches_per_step = T * L * (3 + (1 if stack else 0))
    elif dense_path:  # hidden layer, scores, activation, combine (the two GEMMs are library kernels)
        launches_per_step = T * L * (4 + (1 if stack else 0))
    else:
        launches_per_step = T * L * (2 * groups + (B + 3) // 4 + (1 if stack else 0))

    # ---- device-timed steps; every replay and event on `stream`
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for i in range(steps):
                graph.replay()
                evs[i + 1].record(stream)
        torch.cuda.synchronize()
        barrier(world)
    clocks = clk.summary()
    step_ms = np.array([evs[i].elapsed_time(evs[i + 1]) for i in range(steps)])
    ms = evs[0].elapsed_time(evs[-1])
    ms_max = max_over_ranks(ms, world)
    ms_per_step = ms_max / steps
    value = T * B * steps * world / (ms_max / 1e3)
    us_layer_steps = step_ms * 1e3 / (T * L)

    # ---- algorithmic bytes per layer call
    pred_bytes = (r * d + f * r) * esz + f * 4  # V, U, predictor bias
    io_bytes = B * d * esz + B * d * 4         # tokens in, outputs out
    W_words = (f + 31) // 32
    if dense_path:
        gathered = float(f) * d * esz * (nm + 1)  # every row
        kernel_bytes = gathered + B * W_words * 4 + io_bytes
    elif union_path:
        gathered = float(np.mean(unions)) * d * esz * (nm + 1)
        kernel_bytes = gathered + float(np.mean(unions)) * 4 + B * W_words * 4 + io_bytes  # + gated bias, masks
    else:
        gathered = float(np.mean(n_tok)) * B * d * esz * (nm + 1)
        kernel_bytes = gathered + pred_bytes + f * 4 + io_bytes  # the batch-1 kernel reads both biases
    layer_bytes = gathered + pred_bytes + f * 4 + io_bytes

    # ---- the dominant kernel's launch durations
    peaks = measured_peaks()
    peak = peaks["hbm_gbs"] if peaks else 6800.0
    if B == 1:
        kname = ("k_layer (predictor, threshold, row gather, ReLU/ReGLU, down projection; one launch per layer "
                 "and token" + (", LayerNorm of the previous layer folded in)" if stack else ")"))
        k_us = ms / (steps * launches_per_step) * 1e3
        k_p10, k_p90 = (float(np.percentile(us_layer_steps, q)) for q in (10, 90))
        ktiming = ("device-timed graph / launches (per-step p10/p90)" +
                   (", the final LayerNorm launch included" if stack else ""))
    elif dense_path:
        kname = "dense fallback (two cuBLASLt GEMMs, masked activation and combine kernels)"
        k_us = ms / (steps * T * L) * 1e3
        k_p10, k_p90 = (float(np.percentile(us_layer_steps, q)) for q in (10, 90))
        ktiming = "device-timed graph / layer calls (predictor included)"
    elif union_path:
        kname = "k_union (union gather-GEMM on tcgen05: up/gate, ReLU/ReGLU, down projection)"
        k_us, k_p10, k_p90 = time_dominant_kernel(sffn, torch, step_body, stream, T * L)
        ktiming = "event pairs around every launch as nodes of the step's graph (one replay)"
    else:
        kname = "whole layer call (predictor kernels + row-gather passes)"
        k_us = ms / (steps * T * L) * 1e3
        k_p10, k_p90 = (float(np.percentile(us_layer_steps, q)) for q in (10, 90))
        ktiming = "device-timed graph / layer calls"
    k_s = k_us / 1e6
    us_per_layer = ms_per_step * 1e3 / (T * L)
    rec = {
        "workload": wl.name, "batch": B, "layers": L, "decode_steps_per_step": T, "variant": variant or "exact",
        "path": ("dense fallback" if dense_path else "tensor-core union" if union_path
                 else "single-launch layer kernel" if B == 1 else "CUDA-core row gather"),
        "tokens_per_s": round(value, 1),
        "us_per_layer": round(us_per_layer, 3),
        "us_per_layer_p10": round(float(np.percentile(us_layer_steps, 10)), 3),
        "us_per_layer_p90": round(float(np.percentile(us_layer_steps, 90)), 3),
        "steps": steps, "warmup": warmup,
        "dominant_kernel": kname.split(" (")[0],
        "kernel_us_per_launch": round(k_us, 3),
        "kernel_us_p10": round(k_p10, 3), "kernel_us_p90": round(k_p90, 3),
        "kernel_timing": ktiming,
        "gathered_bytes_per_layer": round(gathered),
        "kernel_bytes_per_launch": round(kernel_bytes),
        "layer_bytes_per_call": round(layer_bytes),
        "gathered_frac": round(gathered / k_s / 1e9 / peak, 4),
        "kernel_frac": round(kernel_bytes / k_s / 1e9 / peak, 4),
        "total_frac": round(layer_bytes / (us_per_layer / 1e6) / 1e9 / peak, 4),
        "peak_gbs": peak,
    }
    rec.update(st_rec)
    rec.update(la_rec)
    if stack and B > 1:
        if all(per_layer_union.get(l) for l in range(L)):  # filled by the statistics pass
            rec["union_per_layer"] = [round(float(np.mean(per_layer_union[l])), 1) for l in range(L)]
        p = [np.asarray(lw.p) for lw in model.lws]
        rec["union_if_independent"] = round(float(np.mean([np.sum(1 - (1 - q) ** B) for q in p])), 1)
    if dense and not stack:
        rec["dense_contrast"] = dense_contrast(sffn, torch, model, X, B, dev, stream, peak, value)
    extras = {"graph": graph, "stream": stream, "X": X, "Y": Y, "x0": x0 if stack else None, "clocks": clocks,
              "ms_per_step": ms_per_step, "value": value, "launches_per_step": launches_per_step,
              "kname": kname, "kernel_bytes": kernel_bytes, "k_us": k_us, "peak": peak, "peaks": peaks,
              "union_path": union_path}
    if want_e2e:
        extras["e2e"] = e2e_timing(torch, graph, stream, x0 if stack else X, Y, steps, world, T * B)
    return rec, extras


def lookahead_stats(sffn, torch, model, trace, mtr, dev):
    """Look-ahead masks (mtr, what each call of a traced run used) against the
    masks the exact predictor and the exact ReLU pattern give on the same
    call's input (trace): recall and precision over every call of the run."""
    f = model.wl.d_ff
    ws = sffn.new_workspace(sffn.sffn_workspace_size(model.layers[0], 1), dev)
    bits = torch.arange(32, device=dev, dtype=torch.int32)
    tp_p = n_p = n_la = tp_e = n_e = 0.0
    Tp, L = trace.shape[0], trace.shape[1]
    for t in range(Tp):
        for l in range(L):
            x = trace[t, l]
            r = predictor_stats(sffn, torch, model.layers[l], model.lws[l], x, ws, model.wl.tau)
            la = ((mtr[t, l, 0][:, None] >> bits) & 1).reshape(-1)[:f].bool()
            pred = r["mask"][0]
            lw = model.lws[l]
            wg = lw.w_gate if lw.w_gate is not None else lw.w_up
            xf = x.float()
            exact = torch.cat([(xf @ wg[i:i + 4096].float().t() + lw.b[i:i + 4096]) > 0
                               for i in range(0, f, 4096)], 1)[0]
            tp_p += float((la & pred).sum()); n_p += float(pred.sum()); n_la += float(la.sum())
            tp_e += float((la & exact).sum()); n_e += float(exact.sum())
    return {"la_recall_vs_predictor": round(tp_p / max(n_p, 1), 4),
            "la_precision_vs_predictor": round(tp_p / max(n_la, 1), 4),
            "la_recall_vs_exact": round(tp_e / max(n_e, 1), 4),
            "la_precision_vs_exact": round(tp_e / max(n_la, 1), 4),
            "la_mean_active": round(n_la / (Tp * L), 1)}


def time_dominant_kernel(sffn, torch, step_body, stream, n_launches):
    """Per-launch durations of the dominant kernel inside the step's graph: a
    copy of the step is captured with an event pair around every such launch
    (graph nodes), replayed once after a warm-up replay, and every pair read."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_launches)]
    stops = [torch.cuda.Event(enable_timing=True) for _ in range(n_launches)]
    for e in starts + stops:  # create the CUDA events before their handles are passed on
        e.record(stream)
    torch.cuda.synchronize()
    sffn.sffn_set_profile_events(starts, stops)
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, stream=stream):
            step_body()
    finally:
        sffn.sffn_set_profile_events()
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    us = np.array([a.elapsed_time(b) * 1e3 for a, b in zip(starts, stops)])
    del g
    return float(us.mean()), float(np.percentile(us, 10)), float(np.percentile(us, 90))


def e2e_timing(torch, graph, stream, Xin, Y, steps, world, tokens_per_step):
    """The same step through the public API with the tokens copied in from
    pinned host memory and the outputs copied back, inside the timed region."""
    Xh = Xin.cpu().pin_memory()
    Yh = torch.empty(Y.shape, dtype=Y.dtype).pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(3):
            Xin.copy_(Xh, non_blocking=True)
            graph.replay()
            Yh.copy_(Y, non_blocking=True)
    torch.cuda.synchronize()
    e_steps = max(3, steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
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
    return {"value": round(tokens_per_step * e_steps * world / (e_ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(Xh.numel() * Xh.element_size()),
            "d2h_bytes_per_step": int(Yh.numel() * Yh.element_size()), "wall_s": round(wall, 3)}


def dense_contrast(sffn, torch, model, X, B, dev, stream, peak, sparse_value):
    """The no-skip FFN over the same rotating replicas, each arm captured in a
    CUDA graph of the same tokens: the library's dense path, and two cuBLAS
    GEMMs (torch.nn.functional.linear) with the activation in between.  The
    fraction is of the dense bytes (every row of every FFN matrix)."""
    import torch.nn.functional as F
    R = len(model.layers)
    T = min(X.shape[0], 2 * R)
    ws = sffn.new_workspace(sffn.sffn_workspace_size(model.layers[0], B), dev)
    y = torch.empty(B, model.layers[0].d_model, dtype=torch.float32, device=dev)
    wl = model.wl
    nm = 2 if wl.act == "reglu" else 1
    dense_bytes = (nm + 1) * wl.d_ff * wl.d_model * ESIZE[wl.dtype]

    def lib():
        for t in range(T):
            sffn.sffn_dense_forward(model.layers[t % R], X[t], y, ws)

    def cublas():
        for t in range(T):
            w = model.lws[t % R]
            up = F.linear(X[t], w.w_up)
            if w.w_gate is not None:
                a = torch.relu(F.linear(X[t], w.w_gate) + w.b.to(up.dtype)) * up
            else:
                a = torch.relu(up + w.b.to(up.dtype))
            F.linear(a, w.w_downT.t())

    res = {}
    for name, fn in (("sffn_dense_forward", lib), ("cublas_two_gemm", cublas)):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            e0.record(stream)
            for _ in range(5):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        s = e0.elapsed_time(e1) / 1e3
        res[name] = {"tokens_per_s": round(5 * T * B / s, 1),
                     "frac": round(dense_bytes * 5 * T / s / 1e9 / peak, 4)}
        del g
    best = max(v["tokens_per_s"] for v in res.values())
    res["unit"] = "tokens/s"
    res["sparse_over_best_dense"] = round(sparse_value / best, 2)
    return res


# ---------------------------------------------------------------- the CUDA arm

def recorded_traffic(workload, batch, union_path):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary, when the kernel sources still match the ones it was taken on."""
    if union_path:
        path, files = "k_union_traffic.json", ("union_impl.cuh", "common.cuh", "kernels.cuh", "tcgen05.cuh")
    elif batch == 1:
        path, files = "k_layer_traffic.json", ("layer_impl.cuh", "common.cuh", "kernels.cuh")
    else:
        return None
    tpath = os.path.join(ROOT, "profiles", path)
    if not os.path.exists(tpath):
        return None
    tj = json.load(open(tpath)).get(f"{workload}_b{batch}", {})
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


def bench_sffn(args):
    import torch
    from activation_sparse_decode_gb300 import sffn, workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B = args.batch
    if B < 1 or B > 32:
        raise SystemExit("--batch must be in [1, 32]")
    # the layers' weights are written and synchronised before the first call
    # and never written after: batch-1 calls may stage them before the
    # previous kernel on the stream has finished
    flags = (sffn.SFFN_FLAG_ROW_GATHER if args.row_gather else 0) | sffn.SFFN_FLAG_STATIC_WEIGHTS
    head = args.workload

    # ---- sub-records first (each workload built, measured and freed), then the headline
    sub = []
    if not args.no_suite:
        names = [n for i, (n, _, _) in enumerate(SUITE) if n != head and n not in [m for m, _, _ in SUITE[:i]]]
        for name in names:  # the headline's workload is measured with its own layers below
            runs = [(b, v) for n, b, v in SUITE if n == name]
            m = Model(sffn, W, W.get_workload(name), dev, max(b for b, _ in runs), args.replicas, args.hot_frac,
                      flags)
            for b, v in runs:
                rec, _ = measure(sffn, W, torch, m, b, SUITE_STEPS[name], 3, dev, world, args,
                                 stats=not args.no_stats and v not in ("bundled", "balanced"),
                                 dense=not args.no_dense and not v,
                                 variant=v)
                sub.append(rec)
            m.close()
            del m
            torch.cuda.synchronize()
            torch.cuda.empty_cache()

    wl = W.get_workload(head)
    if args.layers is not None and wl.n_layers > 1:
        wl = wl.with_(n_layers=max(2, min(args.layers, wl.n_layers)))
    max_b = max([B] + [b for n, b, _ in SUITE if n == head and not args.no_suite])
    model = Model(sffn, W, wl, dev, max_b, args.replicas, args.hot_frac, flags)
    head_variant = "lookahead" if args.lookahead else "bundled" if args.bundled else ""
    rec, ex = measure(sffn, W, torch, model, B, args.steps, args.warmup, dev, world, args,
                      stats=not args.no_stats, dense=not args.no_dense, want_e2e=True, variant=head_variant)
    if not args.no_suite:
        for n, b, v in SUITE:
            if n == head and (b, v) != (B, head_variant):
                r2, _ = measure(sffn, W, torch, model, b, SUITE_STEPS[n], 3, dev, world, args,
                                stats=not args.no_stats, dense=not args.no_dense and not v, variant=v)
                sub.append(r2)
    lw0 = model.lws[0]

    achieved = ex["kernel_bytes"] / (ex["k_us"] / 1e6) / 1e9
    peak = ex["peak"]
    nm = 2 if wl.act == "reglu" else 1
    esz = ESIZE[wl.dtype]
    layer_mb = (lw0.w_up.numel() * (nm + 1) + lw0.U.numel() + lw0.V.numel()) * esz / 2 ** 20
    if model.stack:
        l2 = f"inputs larger than L2: {wl.n_layers} layers, {layer_mb * wl.n_layers / 1024:.1f} GiB resident"
    else:
        R = len(model.layers)
        l2 = (f"inputs larger than L2: {R} rotating layer replicas ({layer_mb * R / 1024:.2f} GiB), reuse distance "
              f"~{R * rec['layer_bytes_per_call'] / 2**20:.0f} MB per layer call vs {L2_BYTES // 2**20} MB L2")
    config = {"workload": wl.name, "d_model": wl.d_model, "d_ff": wl.d_ff, "rank": wl.rank, "layers": wl.n_layers,
              "batch": B, "act": wl.act, "weights": f"{wl.dtype}, fp32 accumulation", "hot_first": bool(wl.reorder),
              "l2": l2, "hot_rows": model.hots[0], "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}
    config.update({k: v for k, v in rec.items() if k not in ("workload", "batch", "layers")})
    out = {
        "metric": METRIC,
        "value": round(ex["value"], 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ex["ms_per_step"], 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded Zipf/low-rank construction; random weights, no checkpoint)",
        "config": config,
        "roofline": {
            "kernel": ex["kname"],
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "peak_source": "measured" if ex["peaks"] else "fallback",
            "traffic": recorded_traffic(head, B, ex["union_path"]),
            "algorithmic_bytes_per_launch": round(ex["kernel_bytes"]),
        },
        "e2e": ex["e2e"],
        "gpu_launches": ex["launches_per_step"] * args.steps,
        "clocks": ex["clocks"],
    }
    if sub:
        out["workloads"] = sub
    model.close()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        lw_cpu = W.make_layer(wl, seed=0, layer=0, device=dev)
        out["cpu_baseline"] = run_cpu_baseline(lw_cpu, ex["X"], args.cpu_seconds, wl.n_layers)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


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
    del lw
    X = st(W.make_tokens(wl, 16, batch=args.batch, device="cpu")).reshape(-1, wl.d_model)
    per_step = 1 if wl.d_model * wl.d_ff > 10 ** 8 else 4  # a bounded sample: ~1 s of oracle work per step
    for s in range(args.warmup):
        for i in range(per_step):
            oracle.sparse_ffn(ol, X[(s * per_step + i) % len(X)], 0.0)
    t0 = time.perf_counter()
    for s in range(args.steps):
        for i in range(per_step):
            oracle.sparse_ffn(ol, X[(s * per_step + i) % len(X)], 0.0)
    el = time.perf_counter() - t0
    L = wl.n_layers
    v = per_step * args.steps / el / L
    cores = host_cores()
    what = "one layer" if L == 1 else f"layer 0 of {L}, rate divided by {L}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded Zipf/low-rank construction)",
        "config": {"workload": wl.name, "batch": args.batch, "tokens_per_step": per_step,
                   "note": f"CPU oracle, {what}, rows in generated order (the hot-first order changes no work); "
                           "tokens one at a time (the oracle has no batched form)"},
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{per_step} decode token(s) per step, numpy fp64 on the host cores, {what}"},
        "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
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
