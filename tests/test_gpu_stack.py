"""GPU parity of the layer stacks: 40-layer OPT-13B-shaped and 48-layer
OPT-175B-shaped FFN decode with residual + LayerNorm between layers.

Mask flips inside the band compound over many layers and steps, so parity is
checked teacher-forced per layer, on what the stack run itself recorded (its
layer inputs, mask words and outputs, traced by sffn_forward_stack):
* sampled (step, layer) calls against the oracle: the run's mask outside the
  band, its y over that mask (rel-L2 and element by element) and the next
  input it formed, round(LN(x_l + y_l)), from that y;
* every layer call of the checked steps against a rerun of the same call on
  the same input: identical mask words, y equal up to the order of float
  atomic adds -- a race inside the run would show as a difference here."""

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_gb300 import workloads as W
from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
from gpu_helpers import (BAND, TOL, check_elementwise, check_next_input, check_token, hot_first, lazy_oracle_layer,
                         mask_from_list, rel_l2)

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
    """One traced stack run: per (step, layer) the input, the mask words and
    the output that this run itself used."""
    B, d = x0.shape
    L = len(layers)
    Wmax = max((l.d_ff + 31) // 32 for l in layers)
    ws = sffn.new_workspace(sffn.sffn_stack_workspace_size(layers, B), DEV)
    x_out = torch.empty(n_steps, B, d, dtype=x0.dtype, device=DEV)
    trace = torch.empty(n_steps, L, B, d, dtype=x0.dtype, device=DEV)
    masks = torch.empty(n_steps, L, B, Wmax, dtype=torch.int32, device=DEV)
    ys = torch.empty(n_steps, L, B, d, dtype=torch.float32, device=DEV)
    sffn.sffn_forward_stack(layers, x0, n_steps, x_out, ws, x_trace=trace, mask_trace=masks, y_trace=ys)
    torch.cuda.synchronize()
    assert sffn.sffn_read_device_status(ws) == 0
    return x_out, trace, masks, ys


def words_to_mask(words, f):
    """Mask words (int32 view of uint32) -> bool [f]: bit i%32 of word i/32."""
    w = np.asarray(words).astype(np.int64) & 0xFFFFFFFF
    bits = (w[:, None] >> np.arange(32)) & 1
    return bits.reshape(-1)[:f].astype(bool)


# Two runs of the same layer call differ only in the order of their float
# atomic adds: |y1 - y2| <= ATOMIC_EPS * (|y| + rms(y)) element by element
# (about 150 block partials per element: at most ~1e-4 of rms(y) in the worst
# order, ~1e-6 typically; one neuron's term is >= ~0.009 rms(y)).
ATOMIC_EPS = 2.0 ** -12
REPEAT_RUNS = 20


def same_call(y1, y2):
    y1, y2 = np.asarray(y1, np.float64), np.asarray(y2, np.float64)
    scale = np.abs(y2) + np.sqrt(np.mean(y2 * y2))
    return bool(np.all(np.abs(y1 - y2) <= ATOMIC_EPS * scale))


def recompute_all(sffn, layers, trace, masks, ys, wl):
    """Every (step, layer) call of the stack run re-run alone on its own
    recorded input: the mask words must be identical (the predictor is
    deterministic) and the output equal up to the order of atomic adds."""
    n_steps, L, B, d = trace.shape
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layers[0], B), DEV)
    idx = torch.empty(B, wl.d_ff, dtype=torch.int32, device=DEV)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    y = torch.empty(B, d, dtype=torch.float32, device=DEV)
    bad = []
    for t in range(n_steps):
        for l in range(L):
            sffn.sffn_forward(layers[l], trace[t, l].contiguous(), y, ws, idx, n)
            ih, nh, yh = idx.cpu().numpy(), n.cpu().numpy(), y.cpu().numpy()
            mw = masks[t, l].cpu().numpy()
            ys_h = ys[t, l].cpu().numpy()
            for b in range(B):
                m_run = words_to_mask(mw[b], wl.d_ff)
                m_re = mask_from_list(ih[b], nh[b], wl.d_ff)
                if not np.array_equal(m_run, m_re):
                    bad.append((t, l, b, "mask", np.flatnonzero(m_run != m_re)[:8].tolist()))
                elif not same_call(ys_h[b], yh[b]):
                    j = int(np.argmax(np.abs(ys_h[b] - yh[b])))
                    bad.append((t, l, b, "y", j, float(ys_h[b][j]), float(yh[b][j])))
    assert sffn.sffn_read_device_status(ws) == 0
    assert not bad, f"{len(bad)} layer calls of the stack run differ from a rerun: {bad[:4]}"


def teacher_forced(sffn, wl, lws, layers, x_out, trace, masks, ys, pairs, tokens):
    """Sampled (step, layer) calls against the oracle, from the stack run's own
    records: the mask it used (outside the band), its y over that mask (rel-L2
    and element-wise), and the next input it formed, round(LN(x_l + y_l)) from
    its own y (one format ulp on under 1% of the elements)."""
    for t, l in pairs:
        ol = lazy_oracle_layer(lws[l], wl.tau)
        xh = st(trace[t, l])
        nxt = trace[t, l + 1] if l + 1 < len(layers) else x_out[t]
        nh_next = st(nxt)
        mw = masks[t, l].cpu().numpy()
        yh = ys[t, l].cpu().numpy()
        for b in tokens:
            m = words_to_mask(mw[b], wl.d_ff)
            check_token(ol, xh[b], m, yh[b], TOL[wl.dtype], wl.tau)
            want = oracle.residual_layernorm(xh[b], yh[b].astype(np.float64), wl.dtype)
            check_next_input(nh_next[b], want, wl.dtype, max_frac=0.01)


def run_stack_lookahead(sffn, layers, x0, n_steps):
    B, d = x0.shape
    L = len(layers)
    Wmax = max((l.d_ff + 31) // 32 for l in layers)
    ws = sffn.new_workspace(sffn.sffn_stack_workspace_size(layers, B), DEV)
    x_out = torch.empty(n_steps, B, d, dtype=x0.dtype, device=DEV)
    trace = torch.empty(n_steps, L, B, d, dtype=x0.dtype, device=DEV)
    masks = torch.empty(n_steps, L, B, Wmax, dtype=torch.int32, device=DEV)
    ys = torch.empty(n_steps, L, B, d, dtype=torch.float32, device=DEV)
    sffn.sffn_forward_stack(layers, x0, n_steps, x_out, ws, x_trace=trace, mask_trace=masks, y_trace=ys,
                            options=sffn.SFFN_STACK_LOOKAHEAD)
    torch.cuda.synchronize()
    assert sffn.sffn_read_device_status(ws) == 0
    return x_out, trace, masks, ys


def lookahead_checks(sffn, wl, lws, layers, x_out, trace, masks, ys, pairs):
    """Look-ahead calls against the oracle's definition, teacher-forced on the
    run's own records: call (t, l) must use the neurons its layer's predictor
    scores above tau on the input of the call before it (the previous layer's
    input; for layer 0 the last layer's input of the previous step; for the
    first call its own), outside the band; its y over that mask and the next
    input it formed are checked as for the exact predictor."""
    L = len(layers)
    n = 0
    for t, l in pairs:
        ol = lazy_oracle_layer(lws[l], wl.tau)
        if t == 0 and l == 0:
            x_prev = trace[0, 0]
        else:
            x_prev = trace[t, l - 1] if l > 0 else trace[t - 1, L - 1]
        xp, xh = st(x_prev)[0], st(trace[t, l])[0]
        m = words_to_mask(masks[t, l].cpu().numpy()[0], wl.d_ff)
        s_prev = oracle.predictor_scores(ol, xp)
        mo = oracle.predicted_mask(s_prev, wl.tau)
        bad = (mo != m) & ~(np.abs(s_prev - wl.tau) <= BAND)
        assert not bad.any(), f"call ({t}, {l}): {bad.sum()} neurons outside the band differ from the look-ahead mask"
        yh = ys[t, l].cpu().numpy()[0]
        ref = oracle.masked_ffn(ol, xh, m)
        assert rel_l2(yh, ref) <= TOL[wl.dtype]
        check_elementwise(yh, ref, wl.dtype)
        nxt = trace[t, l + 1] if l + 1 < L else x_out[t]
        want = oracle.residual_layernorm(xh, yh.astype(np.float64), wl.dtype)
        check_next_input(st(nxt)[0], want, wl.dtype, max_frac=0.01)
        n += 1
    return n


@pytest.mark.parametrize("flags", [0, 1, 2], ids=["fused", "multi", "fused-balanced"])
def test_small_stack_both_paths(sffn, flags):
    wl = W.tiny_workload(d_model=512, d_ff=2048, rank=64, dtype="bf16", name="small-stack").with_(n_layers=3)
    lws = [W.make_layer(wl, layer=l, device=DEV) for l in range(3)]
    layers = [sffn.Layer.from_weights(lw, max_batch=1, flags=flags) for lw in lws]
    x0 = W.make_tokens(wl, 1, device=DEV)[0]
    x_out, trace, masks, ys = run_stack(sffn, layers, x0, 4)
    assert torch.equal(trace[0, 0], x0)
    for t in range(1, 4):
        assert torch.equal(trace[t, 0], x_out[t - 1])
    pairs = [(t, l) for t in range(4) for l in range(3)]
    teacher_forced(sffn, wl, lws, layers, x_out, trace, masks, ys, pairs, [0])
    recompute_all(sffn, layers, trace, masks, ys, wl)


def test_opt13b_stack40_fp16(sffn):
    wl = W.get_workload("c4")
    lws, layers = build_stack(sffn, wl, wl.n_layers, 1)
    x0 = W.make_tokens(wl, 1, device=DEV)[0]
    x_out, trace, masks, ys = run_stack(sffn, layers, x0, wl.steps)
    assert torch.equal(trace[0, 0], x0)
    assert torch.equal(trace[1, 0], x_out[0])
    rng = np.random.Generator(np.random.PCG64(4))
    pairs = [(0, 0), (0, wl.n_layers - 1), (wl.steps - 1, wl.n_layers - 1)] + \
        [(int(rng.integers(wl.steps)), int(rng.integers(wl.n_layers))) for _ in range(3)]
    teacher_forced(sffn, wl, lws, layers, x_out, trace, masks, ys, pairs, [0])
    # every layer of the first two steps, against a rerun of the same call
    recompute_all(sffn, layers, trace[:2], masks[:2], ys[:2], wl)
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
    x_out, trace, masks, ys = run_stack(sffn, layers, x0, steps)
    pairs = [(0, 0), (1, wl.n_layers - 1), (1, 17)]
    teacher_forced(sffn, wl, lws, layers, x_out, trace, masks, ys, pairs, [0] if batch == 1 else [0, batch - 1])
    recompute_all(sffn, layers, trace, masks, ys, wl)
    # the same two-step decode again and again: every run must record the same
    # layer inputs and masks and outputs equal up to the order of atomic adds
    # (an input that differs is followed through the LayerNorm rounding, so
    # only the first layer where a run departs is reported)
    for rep in range(REPEAT_RUNS):
        xo2, tr2, mk2, ys2 = run_stack(sffn, layers, x0, steps)
        for t in range(steps):
            for l in range(wl.n_layers):
                if not torch.equal(tr2[t, l], trace[t, l]):
                    # legitimate: the previous layer's atomic order moved a
                    # LayerNorm output across a rounding boundary; from here on
                    # the runs decode different inputs
                    break
                same_m = torch.equal(mk2[t, l], masks[t, l])
                same_y = all(same_call(ys2[t, l, b].cpu().numpy(), ys[t, l, b].cpu().numpy()) for b in range(batch))
                assert same_m and same_y, (f"run {rep + 1}, step {t}, layer {l}: same input, but "
                                           f"mask {'same' if same_m else 'differs'}, y {'same' if same_y else 'differs'}")
            else:
                continue
            break
    if batch == 8:
        del test_opt175b_stack48_fp16._stack
        torch.cuda.empty_cache()


@pytest.mark.parametrize("shape", [(512, 2048, 64, "bf16", "relu", 0), (1024, 4096, 64, "f16", "reglu", 8),
                                   (12288, 2048, 128, "f16", "relu", 8)],
                         ids=["bf16-relu", "f16-reglu-static", "f16-wide-pairs"])
def test_lookahead_small_stack(sffn, shape):
    """Look-ahead masks on a 3-layer stack over 4 steps: every call against
    the oracle's look-ahead definition (teacher-forced), on two blocks per SM,
    with weights staged before the dependency wait, and on pairs of blocks."""
    d, f, r, dt, act, flags = shape
    wl = W.tiny_workload(d_model=d, d_ff=f, rank=r, dtype=dt, act=act, mean_p=0.1, name=f"la-{shape}").with_(n_layers=3)
    lws = [W.make_layer(wl, layer=l, device=DEV) for l in range(3)]
    layers = [sffn.Layer.from_weights(lw, flags=flags) for lw in lws]
    x0 = W.make_tokens(wl, 1, device=DEV)[0]
    x_out, trace, masks, ys = run_stack_lookahead(sffn, layers, x0, 4)
    assert torch.equal(trace[0, 0], x0)
    for t in range(1, 4):
        assert torch.equal(trace[t, 0], x_out[t - 1])
    assert lookahead_checks(sffn, wl, lws, layers, x_out, trace, masks, ys,
                            [(t, l) for t in range(4) for l in range(3)]) == 12
    # the first call has no earlier input: its mask is the exact predictor's
    idx = torch.empty(1, f, dtype=torch.int32, device=DEV)
    nn = torch.empty(1, dtype=torch.int32, device=DEV)
    sffn.sffn_predict(layers[0], x0, idx, nn, sffn.new_workspace(sffn.sffn_workspace_size(layers[0], 1), DEV))
    m0 = mask_from_list(idx[0].cpu().numpy(), int(nn.item()), f)
    assert np.array_equal(words_to_mask(masks[0, 0].cpu().numpy()[0], f), m0)


def test_lookahead_rejects_what_it_does_not_serve(sffn):
    wl = W.tiny_workload(d_model=512, d_ff=2048, rank=64, dtype="bf16", name="la-reject").with_(n_layers=2)
    lws = [W.make_layer(wl, layer=l, device=DEV) for l in range(2)]
    x_out = torch.empty(1, 2, 512, dtype=torch.bfloat16, device=DEV)
    for layers, B in (([sffn.Layer.from_weights(lw, max_batch=2) for lw in lws], 2),
                      ([sffn.Layer.from_weights(lws[0]), sffn.Layer.from_weights(lws[1], flags=1)], 1)):
        ws = sffn.new_workspace(sffn.sffn_stack_workspace_size(layers, B), DEV)
        x0 = W.make_tokens(wl, 1, batch=B, device=DEV)[0]
        with pytest.raises(sffn.SffnError) as e:
            sffn.sffn_forward_stack(layers, x0, 1, x_out[:, :B], ws, options=sffn.SFFN_STACK_LOOKAHEAD)
        assert e.value.status == 2


def test_opt13b_stack40_lookahead(sffn):
    """The 40-layer OPT-13B-shaped stack with look-ahead masks: sampled calls
    against the oracle's definition, and a second run that records the same
    inputs and masks until the order of atomic adds first moves a LayerNorm
    rounding."""
    wl = W.get_workload("c4")
    lws, layers = build_stack(sffn, wl, wl.n_layers, 1)
    x0 = W.make_tokens(wl, 1, device=DEV)[0]
    steps = 4
    x_out, trace, masks, ys = run_stack_lookahead(sffn, layers, x0, steps)
    pairs = [(0, 0), (0, 1), (0, wl.n_layers - 1), (1, 0), (steps - 1, 17), (steps - 1, wl.n_layers - 1)]
    lookahead_checks(sffn, wl, lws, layers, x_out, trace, masks, ys, pairs)
    xo2, tr2, mk2, ys2 = run_stack_lookahead(sffn, layers, x0, steps)
    for t in range(steps):
        for l in range(wl.n_layers):
            if not torch.equal(tr2[t, l], trace[t, l]):
                return
            assert torch.equal(mk2[t, l], masks[t, l]), (t, l)
