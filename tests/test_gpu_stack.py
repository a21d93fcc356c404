"""GPU parity of the layer stacks: 40-layer OPT-13B-shaped and 48-layer
OPT-175B-shaped FFN decode with residual + LayerNorm between layers.

Mask flips inside the band compound over many layers and steps, so parity is
checked teacher-forced per layer: for sampled (step, layer) pairs the oracle
takes the GPU's own layer input x_l, and its mask, output and next input
round(LN(x_l + y_l)) are compared with the GPU's."""

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_gb300 import workloads as W
from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
from gpu_helpers import TOL, check_next_input, check_token, hot_first, lazy_oracle_layer, mask_from_list

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sffn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from activation_sparse_decode_gb300 import build
    build.build()
    from activation_sparse_decode_gb300 import sffn as mod
    return mod


def build_stack(sffn, wl, n_layers, max_batch):
    lws, layers = [], []
    for l in range(n_layers):
        lw = W.make_layer(wl, layer=l, device=DEV)
        hot, ea = 0, 0.0
        if wl.reorder:
            lw, _, counts = hot_first(sffn, lw, wl, layer_idx=l)
            hot = sffn.hot_row_count(counts, wl.profile_tokens)
            ea = float(counts.sum().item()) / wl.profile_tokens
        lws.append(lw)
        layers.append(sffn.Layer.from_weights(lw, tau=wl.tau, max_batch=max_batch, hot_rows=hot, expected_active=ea))
    torch.cuda.synchronize()
    return lws, layers


def run_stack(sffn, layers, x0, n_steps):
    B, d = x0.shape
    L = len(layers)
    ws = sffn.new_workspace(sffn.sffn_stack_workspace_size(layers, B), DEV)
    x_out = torch.empty(n_steps, B, d, dtype=x0.dtype, device=DEV)
    trace = torch.empty(n_steps, L, B, d, dtype=x0.dtype, device=DEV)
    sffn.sffn_forward_stack(layers, x0, n_steps, x_out, ws, x_trace=trace)
    torch.cuda.synchronize()
    assert sffn.sffn_read_device_status(ws) == 0
    return x_out, trace


def teacher_forced(sffn, wl, lws, layers, x_out, trace, pairs, tokens):
    B = trace.shape[2]
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layers[0], B), DEV)
    for t, l in pairs:
        ol = lazy_oracle_layer(lws[l], wl.tau)
        x_l = trace[t, l].contiguous()
        idx = torch.empty(B, wl.d_ff, dtype=torch.int32, device=DEV)
        n = torch.empty(B, dtype=torch.int32, device=DEV)
        y = torch.empty(B, wl.d_model, dtype=torch.float32, device=DEV)
        sffn.sffn_forward(layers[l], x_l, y, ws, idx, n)
        nxt = trace[t, l + 1] if l + 1 < len(layers) else x_out[t]
        xh, yh, ih, nh, nh_next = st(x_l), y.cpu().numpy(), idx.cpu().numpy(), n.cpu().numpy(), st(nxt)
        for b in tokens:
            m = mask_from_list(ih[b], nh[b], wl.d_ff)
            check_token(ol, xh[b], m, yh[b], TOL[wl.dtype], wl.tau)
            want = oracle.residual_layernorm(xh[b], oracle.masked_ffn(ol, xh[b], m), wl.dtype)
            check_next_input(nh_next[b], want, wl.dtype)


@pytest.mark.parametrize("flags", [0, 1, 2], ids=["fused", "multi", "fused-balanced"])
def test_small_stack_both_paths(sffn, flags):
    wl = W.tiny_workload(d_model=512, d_ff=2048, rank=64, dtype="bf16", name="small-stack").with_(n_layers=3)
    lws = [W.make_layer(wl, layer=l, device=DEV) for l in range(3)]
    layers = [sffn.Layer.from_weights(lw, max_batch=1, flags=flags) for lw in lws]
    x0 = W.make_tokens(wl, 1, device=DEV)[0]
    x_out, trace = run_stack(sffn, layers, x0, 4)
    assert torch.equal(trace[0, 0], x0)
    for t in range(1, 4):
        assert torch.equal(trace[t, 0], x_out[t - 1])
    pairs = [(t, l) for t in range(4) for l in range(3)]
    teacher_forced(sffn, wl, lws, layers, x_out, trace, pairs, [0])


def test_opt13b_stack40_fp16(sffn):
    wl = W.get_workload("c4")
    lws, layers = build_stack(sffn, wl, wl.n_layers, 1)
    x0 = W.make_tokens(wl, 1, device=DEV)[0]
    x_out, trace = run_stack(sffn, layers, x0, wl.steps)
    assert torch.equal(trace[0, 0], x0)
    assert torch.equal(trace[1, 0], x_out[0])
    rng = np.random.Generator(np.random.PCG64(4))
    pairs = [(0, 0), (0, wl.n_layers - 1), (wl.steps - 1, wl.n_layers - 1)] + \
        [(int(rng.integers(wl.steps)), int(rng.integers(wl.n_layers))) for _ in range(3)]
    teacher_forced(sffn, wl, lws, layers, x_out, trace, pairs, [0])
    xs = x_out.float()
    assert torch.isfinite(xs).all()
    assert abs(xs.var(-1).mean().item() - 1.0) < 0.01


@pytest.mark.parametrize("batch", [1, 8])
def test_opt175b_stack48_fp16(sffn, batch):
    wl = W.get_workload("c5")
    steps = 2
    if not hasattr(test_opt175b_stack48_fp16, "_stack"):
        test_opt175b_stack48_fp16._stack = build_stack(sffn, wl, wl.n_layers, 8)
    lws, layers = test_opt175b_stack48_fp16._stack
    x0 = W.make_tokens(wl, 1, batch=batch, device=DEV)[0]
    x_out, trace = run_stack(sffn, layers, x0, steps)
    pairs = [(0, 0), (1, wl.n_layers - 1), (1, 17)]
    teacher_forced(sffn, wl, lws, layers, x_out, trace, pairs, [0] if batch == 1 else [0, batch - 1])
    if batch == 8:
        del test_opt175b_stack48_fp16._stack
        torch.cuda.empty_cache()
