"""Pins that tie the CPU oracle to facts fixed outside itself.

Each check takes the oracle module as an argument so the same checks can be run
against deliberately broken copies (see test_oracle.py): every planted mistake
must make at least one check fail.  Sources of truth used here:

* the worked example of the sparsity page (blogs.novita.ai, section 單層計算優化),
  stored under tests/golden/ with its citation;
* invariants the pages state: rows whose ReLU output is zero contribute nothing
  (sparsity page, opening section on ReLU sparsity), a pass restricted to the
  recorded subset reproduces the full pass (same page, DejaVu "上下文稀疏性存在的驗證"),
  prefill uses every neuron as one cluster (PowerInfer-2 page, 4.1.1);
* closed forms and special cases that reduce to library routines (torch's MLP
  layers and layer_norm in fp64, torch's bf16/fp16 rounding);
* brute force over every mask of a tiny layer;
* the statistics the workload construction guarantees (activation rate, union
  size of a batch: the batch-size effect of the sparsity page, "吞吐量影響").
"""

import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def random_layer(o, f=40, d=12, r=5, act="relu", seed=0, fmt="f32"):
    g = _rng(seed)
    mk = lambda *s: g.standard_normal(s).astype(np.float32)
    layer = o.OracleLayer(w_up=mk(f, d), w_downT=mk(f, d), b=(0.5 * g.standard_normal(f)).astype(np.float32),
                          U=mk(f, r), V=mk(r, d), fmt="f32", act=act,
                          w_gate=mk(f, d) if act == "reglu" else None)
    if fmt != "f32":
        conv = lambda a: None if a is None else o.round_to(a.astype(np.float64), fmt)
        layer.w_up, layer.w_downT, layer.U, layer.V = map(conv, (layer.w_up, layer.w_downT, layer.U, layer.V))
        layer.w_gate = conv(layer.w_gate)
        layer.fmt = fmt
    return layer


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def _torch_mlp(layer, x, o):
    """The FFN as two torch Linear layers in fp64 (library reference)."""
    F = torch.nn.functional
    t = lambda a: torch.from_numpy(o.decode(a, layer.fmt))
    xt = t(x)
    b = torch.from_numpy(layer.b.astype(np.float64))
    if layer.act == "relu":
        a = F.relu(F.linear(xt, t(layer.w_up), b))
    else:
        a = F.relu(F.linear(xt, t(layer.w_gate), b)) * F.linear(xt, t(layer.w_up))
    return F.linear(a, t(layer.w_downT).T).numpy()


# ---------------------------------------------------------------- FFN formula

def check_dense_matches_library_mlp(o):
    for act in ("relu", "reglu"):
        for fmt in ("f32", "f16", "bf16"):
            layer = random_layer(o, act=act, seed=1, fmt=fmt)
            x = o.round_to(_rng(2).standard_normal(layer.d_model), fmt)
            assert _rel(o.dense_ffn(layer, x), _torch_mlp(layer, x, o)) < 1e-12, (act, fmt)


def check_all_true_mask_is_dense(o):
    for act in ("relu", "reglu"):
        layer = random_layer(o, act=act, seed=3)
        x = _rng(4).standard_normal(layer.d_model).astype(np.float32)
        y = o.masked_ffn(layer, x, np.ones(layer.d_ff, bool))
        assert _rel(y, o.dense_ffn(layer, x)) < 1e-13


def check_exact_mask_is_dense(o):
    for act in ("relu", "reglu"):
        layer = random_layer(o, act=act, seed=5)
        for s in range(4):
            x = _rng(10 + s).standard_normal(layer.d_model).astype(np.float32)
            m = o.exact_mask(layer, x)
            assert 0 < m.sum() < layer.d_ff
            assert _rel(o.masked_ffn(layer, x, m), o.dense_ffn(layer, x)) < 1e-13
            # the exact pattern is the ReLU > 0 set of the library MLP's hidden layer
            w = layer.w_up if act == "relu" else layer.w_gate
            pre = torch.nn.functional.linear(torch.from_numpy(o.decode(x, "f32")),
                                             torch.from_numpy(o.decode(w, "f32")),
                                             torch.from_numpy(layer.b.astype(np.float64)))
            assert np.array_equal(m, (pre > 0).numpy())


def check_disjoint_masks_add(o):
    layer = random_layer(o, seed=6, act="reglu")
    g = _rng(7)
    x = g.standard_normal(layer.d_model).astype(np.float32)
    m1 = g.random(layer.d_ff) < 0.3
    m2 = (~m1) & (g.random(layer.d_ff) < 0.5)
    y12 = o.masked_ffn(layer, x, m1 | m2)
    assert _rel(y12, o.masked_ffn(layer, x, m1) + o.masked_ffn(layer, x, m2)) < 1e-13
    assert np.all(o.masked_ffn(layer, x, np.zeros(layer.d_ff, bool)) == 0.0)


def _worked_layer(o):
    ex = json.load(open(os.path.join(GOLDEN, "powerinfer_worked_example.json")))
    c = ex["construction"]
    f, d = c["d_ff"], c["d_model"]
    w_up = np.zeros((f, d), np.float32)
    w_up[:, 0] = c["w_up_col0"]
    w_downT = np.array([[1, i, i * i, 0] for i in range(f)], np.float32)
    layer = o.OracleLayer(w_up=w_up, w_downT=w_downT, b=np.array(c["b"], np.float32),
                          U=np.zeros((f, 1), np.float32), V=np.zeros((1, d), np.float32), fmt="f32")
    return ex, layer, np.array(c["x"], np.float32)


def check_worked_example(o):
    ex, layer, x = _worked_layer(o)
    e, page = ex["expected"], ex["from_the_page"]
    r = o.sparse_ffn(layer, x, 0.0)
    assert r.idx[0].tolist() == e["idx"] == page["predicted"]
    assert np.array_equal(r.y, np.array(e["y"], np.float64))
    part = lambda ids: o.masked_ffn(layer, x, np.isin(np.arange(layer.d_ff), ids))
    assert np.array_equal(part(page["gpu_part"]), e["y_gpu_part"])
    assert np.array_equal(part(page["cpu_part"]), e["y_cpu_part"])
    assert np.array_equal(part(page["gpu_part"]) + part(page["cpu_part"]), e["y"])
    assert np.array_equal(o.dense_ffn(layer, x), e["y_dense"])
    assert not o.exact_mask(layer, x)[page["hot_but_inactive"]].any()
    perm = np.array(e["hot_first_perm"])
    assert perm[:3].tolist() == page["hot"]
    rp = o.sparse_ffn(o.permute_layer(layer, perm), x, 0.0)
    assert rp.idx[0].tolist() == e["idx_after_perm"]
    assert sorted(perm[rp.idx[0]].tolist()) == page["predicted"]
    assert np.array_equal(rp.y, r.y)


def check_brute_force_tiny(o):
    """Every one of the 2**f masks of an f = 8 layer against scalar loops."""
    for act in ("relu", "reglu"):
        layer = random_layer(o, f=8, d=3, r=2, act=act, seed=8)
        x = _rng(9).standard_normal(3).astype(np.float32)
        W = [[float(v) for v in row] for row in layer.w_up]
        G = None if layer.w_gate is None else [[float(v) for v in row] for row in layer.w_gate]
        D = [[float(v) for v in row] for row in layer.w_downT]
        bb = [float(v) for v in layer.b]
        xx = [float(v) for v in x]
        for bits in range(1 << 8):
            mask = np.array([(bits >> i) & 1 for i in range(8)], bool)
            want = [0.0, 0.0, 0.0]
            for i in range(8):
                if not mask[i]:
                    continue
                up = sum(W[i][k] * xx[k] for k in range(3))
                if act == "relu":
                    a = max(0.0, up + bb[i])
                else:
                    a = max(0.0, sum(G[i][k] * xx[k] for k in range(3)) + bb[i]) * up
                for j in range(3):
                    want[j] += a * D[i][j]
            got = o.masked_ffn(layer, x, mask)
            assert np.allclose(got, want, rtol=1e-12, atol=1e-12), (act, bits)


# ---------------------------------------------------------------- predictor

def check_predictor_associativity(o):
    for fmt in ("f32", "f16", "bf16"):
        layer = random_layer(o, seed=11, fmt=fmt)
        x = o.round_to(_rng(12).standard_normal(layer.d_model), fmt)
        UV = o.decode(layer.U, fmt) @ o.decode(layer.V, fmt)
        want = UV @ o.decode(x, fmt) + layer.b.astype(np.float64)
        assert _rel(o.predictor_scores(layer, x), want) < 1e-12


def check_predictor_zero_factor(o):
    layer = random_layer(o, seed=13)
    layer.U = np.zeros_like(layer.U)
    x = _rng(14).standard_normal(layer.d_model).astype(np.float32)
    s = o.predictor_scores(layer, x)
    assert np.array_equal(s, layer.b.astype(np.float64))
    assert np.array_equal(o.predicted_mask(s, 0.0), layer.b > 0)


def check_threshold_strict(o):
    s = np.array([-1.0, 0.0, 1e-300, 0.25, 0.25, 2.0])
    assert o.predicted_mask(s, 0.0).tolist() == [False, False, True, True, True, True]
    assert o.predicted_mask(s, 0.25).tolist() == [False, False, False, False, False, True]
    assert o.band_neurons(s, 0.25).tolist() == [3, 4]
    assert o.band_neurons(np.array([0.0, 1e-4, -1e-4, 2e-4]), 0.0).tolist() == [0, 1, 2]


def check_compaction(o):
    g = _rng(15)
    for f in (1, 31, 32, 33, 1000):
        m = g.random(f) < 0.3
        idx = o.active_indices(m)
        assert idx.dtype == np.int32
        assert idx.tolist() == [i for i in range(f) if m[i]]
        assert idx.size == int(m.sum())
        assert np.all(np.diff(idx) > 0)
    assert o.active_indices(np.zeros(9, bool)).size == 0
    assert o.active_indices(np.ones(9, bool)).tolist() == list(range(9))


def check_reglu_saturated_gate(o):
    """W_gate = 0 and a large constant bias c: ReLU(gate) = c, so the ReGLU FFN
    is the linear map c W_down^T^T W_up x."""
    layer = random_layer(o, act="reglu", seed=16)
    layer.w_gate = np.zeros_like(layer.w_gate)
    layer.b = np.full(layer.d_ff, 3.0, np.float32)
    x = _rng(17).standard_normal(layer.d_model).astype(np.float32)
    want = 3.0 * (o.decode(layer.w_downT, "f32").T @ (o.decode(layer.w_up, "f32") @ o.decode(x, "f32")))
    assert _rel(o.dense_ffn(layer, x), want) < 1e-12
    assert _rel(o.masked_ffn(layer, x, np.ones(layer.d_ff, bool)), want) < 1e-12


def check_reglu_square(o):
    """W_gate = W_up and b = 0: a = ReLU(g) * g = ReLU(g)**2."""
    layer = random_layer(o, act="reglu", seed=18)
    layer.w_gate = layer.w_up.copy()
    layer.b = np.zeros(layer.d_ff, np.float32)
    x = _rng(19).standard_normal(layer.d_model).astype(np.float32)
    g = o.decode(layer.w_up, "f32") @ o.decode(x, "f32")
    idx = np.arange(layer.d_ff)
    assert _rel(o.neuron_activations(layer, x, idx), np.maximum(g, 0) ** 2) < 1e-13


def check_batch_is_per_token(o):
    layer = random_layer(o, seed=20, act="reglu")
    X = _rng(21).standard_normal((5, layer.d_model)).astype(np.float32)
    rb = o.sparse_ffn(layer, X, 0.0)
    for t in range(5):
        r1 = o.sparse_ffn(layer, X[t], 0.0)
        assert np.array_equal(rb.mask[t], r1.mask)
        assert rb.idx[t].tolist() == r1.idx[0].tolist()
        assert _rel(rb.y[t], r1.y) < 1e-14


def check_union(o):
    g = _rng(22)
    M = g.random((6, 50)) < 0.2
    u = o.union_mask(M)
    assert u.tolist() == [bool(M[:, i].any()) for i in range(50)]
    assert np.all(u[np.flatnonzero(M[3])])


# ---------------------------------------------------------------- statistics

def _generated(o, name="c1", layer=0):
    from activation_sparse_decode_gb300 import workloads as W
    import conftest
    wl = W.get_workload(name)
    lw = W.make_layer(wl, seed=0, layer=layer)
    return wl, lw, conftest.oracle_layer_from(lw, wl.tau)


def check_activation_rate(o):
    """The construction makes P(neuron i active) = p_i for x ~ N(0, I); the
    exact pattern over 64 tokens must match sum(p) within 5 sigma, and the
    predictor (which misses only the 0.1 N term) must track it closely."""
    from activation_sparse_decode_gb300 import workloads as W
    wl, lw, layer = _generated(o)
    X = W.to_numpy_stored(W.make_tokens(wl, 64)[:, 0])
    p = lw.p
    exact = np.stack([o.exact_mask(layer, x) for x in X])
    pred = np.stack([o.predicted_mask(o.predictor_scores(layer, x), 0.0) for x in X])
    mean, sd = 64 * p.sum(), np.sqrt(64 * (p * (1 - p)).sum())
    assert abs(exact.sum() - mean) < 5 * sd, (exact.sum(), mean, sd)
    assert abs(pred.mean() - wl.mean_p) < 0.01
    recall = (pred & exact).sum() / exact.sum()
    assert recall > 0.9
    hot = p > 0.99
    assert exact[:, hot].mean() > 0.97


def check_union_size(o):
    """Batch union (the batch-size effect): E|union_B| = sum_i 1 - (1 - p_i)**B."""
    from activation_sparse_decode_gb300 import workloads as W
    wl, lw, layer = _generated(o)
    X = W.to_numpy_stored(W.make_tokens(wl, 64, seed=3)[:, 0])
    exact = np.stack([o.exact_mask(layer, x) for x in X])
    for B in (2, 4, 8):
        sizes = [o.union_mask(exact[i:i + B]).sum() for i in range(0, 64, B)]
        q = 1 - (1 - lw.p) ** B
        mean, sd = q.sum(), np.sqrt((q * (1 - q)).sum() / len(sizes))
        assert abs(np.mean(sizes) - mean) < 5 * sd, (B, np.mean(sizes), mean, sd)


# ---------------------------------------------------------------- LayerNorm / stack

def check_layernorm(o):
    eps = 1e-5
    assert np.all(o.layernorm(np.full(16, 3.5), eps=eps) == 0.0)
    u, v = 2.0, -1.0
    z = np.array([u, v] * 8)
    half = (u - v) / 2
    want = np.array([half, -half] * 8) / np.sqrt(half ** 2 + eps)
    assert _rel(o.layernorm(z, eps=eps), want) < 1e-14
    g = _rng(23)
    V = g.standard_normal((3, 40)) * 3 + 1
    gam, bet = g.standard_normal(40), g.standard_normal(40)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(V), (40,), torch.from_numpy(gam),
                                         torch.from_numpy(bet), eps).numpy()
    assert _rel(o.layernorm(V, gam, bet, eps), ref) < 1e-13
    out = o.layernorm(V, eps=eps)
    assert np.allclose(out.mean(-1), 0, atol=1e-13)
    assert np.allclose(out.var(-1), V.var(-1) / (V.var(-1) + eps), rtol=1e-12)


def check_formats(o):
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x4049, 0x7F7F], np.uint16)
    vals = o.decode(bits, "bf16")
    assert vals[:4].tolist() == [1.0, -2.0, 0.0, -0.0]
    assert vals[4] == 3.140625
    assert o.round_to(np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)]), "bf16").tolist() == \
        [0x3F80, 0x3F82, 0xBF80]
    g = _rng(24)
    v32 = (g.standard_normal(4096) * np.exp(g.uniform(-8, 8, 4096))).astype(np.float32)
    tb = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.round_to(v32.astype(np.float64), "bf16"), tb)
    th = torch.from_numpy(v32).to(torch.float16).numpy()
    assert np.array_equal(o.round_to(v32.astype(np.float64), "f16").view(np.uint16), th.view(np.uint16))
    assert np.array_equal(o.decode(tb, "bf16"),
                          torch.from_numpy(tb.view(np.int16)).view(torch.bfloat16).double().numpy())


def check_stack(o):
    """Layers whose predictor rejects every neuron add nothing, so each layer
    maps x to round(LN(x)); a 2-step decode feeds the last output back."""
    g = _rng(25)
    layers = []
    for s in range(3):
        lay = random_layer(o, f=24, d=16, seed=30 + s, fmt="bf16")
        lay.tau = 1e30
        layers.append(lay)
    x0 = o.round_to(g.standard_normal(16) * 2 + 1, "bf16")
    tr = o.stack_decode(layers, x0, 2)
    assert len(tr) == 2 and all(len(t) == 4 for t in tr)
    want = o.round_to(o.layernorm(o.decode(x0, "bf16")), "bf16")
    assert np.array_equal(tr[0][1], want)
    assert np.array_equal(tr[1][0], tr[0][3])
    # with neurons active, layer l's output is round(LN(x_l + sparse_ffn(x_l)))
    for lay in layers:
        lay.tau = 0.0
    tr = o.stack_decode(layers, x0, 1)
    for l, lay in enumerate(layers):
        y = o.sparse_ffn(lay, tr[0][l]).y
        assert np.any(y != 0)
        want = o.round_to(o.layernorm(o.decode(tr[0][l], "bf16") + y), "bf16")
        assert np.array_equal(tr[0][l + 1], want)


def _lookahead_layers(o):
    """Two one-neuron fp32 layers on d = 4 built so that the look-ahead masks
    differ from the exact ones (derivation in check_lookahead_worked).
    Layer A: predictor s = x0 - x3, gate a = ReLU(x0), W_down^T row (-4, 4, 0, 0).
    Layer B: predictor s = x0, gate a = ReLU(x1), W_down^T row (1, 0, 0, 0)."""
    row = lambda *v: np.asarray([v], np.float32)  # one row: [1][n]
    A = o.OracleLayer(w_up=row(1, 0, 0, 0), w_downT=row(-4, 4, 0, 0), b=np.zeros(1, np.float32), U=row(1),
                      V=row(1, 0, 0, -1), fmt="f32")
    Bl = o.OracleLayer(w_up=row(0, 1, 0, 0), w_downT=row(1, 0, 0, 0), b=np.zeros(1, np.float32), U=row(1),
                       V=row(1, 0, 0, 0), fmt="f32")
    return [A, Bl], np.asarray([1, -1, 1, -1], np.float32)


def check_lookahead_worked(o):
    """Hand-derived two-step decode (eps = 1e-5, fp32 stored values):
    step 0, call 0 (A): no earlier input, scores x0 = (1,-1,1,-1): s = 2 > 0,
      a = 1, y = (-4,4,0,0); x0 + y = (-3,3,1,-1) has mean 0, variance 5, so
      x1 = (-3,3,1,-1) / sqrt(5 + eps).
    step 0, call 1 (B): scores the earlier input x0: s = 1 > 0, active (its
      own input would give s = x1[0] < 0, inactive); a = ReLU(x1[1]) = 3/q,
      q = sqrt(5 + eps); x1 + y = (0,3,1,-1)/q has mean 0.75/q and centred
      values (-0.75,2.25,0.25,-1.75)/q of variance 2.1875/q^2, so
      x2 = (-0.75,2.25,0.25,-1.75) / sqrt(2.1875 + eps q^2).
    step 1, call 2 (A): scores x1: s = (-3 + 1)/q < 0, inactive (its own input
      x2 would give s = (-0.75 + 1.75)/... > 0), so y = 0 and x3 = LN(x2).
    step 1, call 3 (B): scores x2: s = x2[0] < 0, inactive, x4 = LN(x3)."""
    layers, x0 = _lookahead_layers(o)
    tr, ms = o.lookahead_stack_decode(layers, x0, 2)
    assert [[bool(m[0]) for m in step] for step in ms] == [[True, True], [False, False]]
    eps = 1e-5
    q = np.sqrt(5 + eps)
    x1 = np.array([-3, 3, 1, -1]) / q
    x2 = np.array([-0.75, 2.25, 0.25, -1.75]) / np.sqrt(2.1875 + eps * q * q)
    assert _rel(tr[0][1], x1) < 1e-6
    assert _rel(tr[0][2], x2) < 1e-6
    assert np.array_equal(tr[1][0], tr[0][2])  # the next step starts from the last output
    x3 = (x2 - x2.mean()) / np.sqrt(x2.var() + eps)
    assert _rel(tr[1][1], x3) < 1e-6
    # the exact stack keeps call 1 inactive: it reaches x2 = LN(x1) instead
    ex = o.stack_decode(layers, x0, 1)
    assert _rel(ex[0][2], x1 / np.sqrt(1 + eps)) < 1e-6


def check_lookahead_fixed_input(o):
    """Where every layer call sees the same input the look-ahead masks are the
    exact ones: layers that add nothing (W_down = 0) on a two-point fp16 token
    +-1, which round(LN(.)) maps to itself (1 / sqrt(1 + 1e-5) rounds to 1),
    so the look-ahead decode must equal stack_decode."""
    layers = []
    for s in range(3):
        lay = random_layer(o, f=24, d=16, seed=60 + s, fmt="f16")
        lay.w_downT = np.zeros_like(lay.w_downT)
        layers.append(lay)
    x0 = o.round_to(np.array([1.0, -1.0] * 8), "f16")
    tr, ms = o.lookahead_stack_decode(layers, x0, 2)
    ex = o.stack_decode(layers, x0, 2)
    for t in range(2):
        for l in range(4):
            assert np.array_equal(tr[t][l], x0) and np.array_equal(ex[t][l], x0)
        for l, lay in enumerate(layers):
            assert np.array_equal(ms[t][l], o.predicted_mask(o.predictor_scores(lay, x0), 0.0))
            assert ms[t][l].any() and not ms[t][l].all()


def check_bundle_layout(o):
    """The bundled layout written out by hand for a 2-neuron ReGLU layer with
    d_model 2 (rows [gate | up | down], the page's order Gate, Up, Down) and a
    ReLU layer ([up | down]); unbundling restores the matrices and the masked
    FFN of the unbundled layer equals the original's bit for bit."""
    g = np.array([[1, 2], [3, 4]], np.float32)
    u = np.array([[5, 6], [7, 8]], np.float32)
    dn = np.array([[9, 10], [11, 12]], np.float32)
    lay = o.OracleLayer(w_up=u, w_downT=dn, b=np.zeros(2, np.float32), U=np.ones((2, 1), np.float32),
                        V=np.ones((1, 2), np.float32), fmt="f32", act="reglu", w_gate=g)
    bnd = o.bundle_rows(lay)
    assert bnd.tolist() == [[1, 2, 5, 6, 9, 10], [3, 4, 7, 8, 11, 12]]
    lay_r = o.OracleLayer(w_up=u, w_downT=dn, b=np.zeros(2, np.float32), U=np.ones((2, 1), np.float32),
                          V=np.ones((1, 2), np.float32), fmt="f32")
    assert o.bundle_rows(lay_r).tolist() == [[5, 6, 9, 10], [7, 8, 11, 12]]
    for act in ("relu", "reglu"):
        ref = random_layer(o, f=20, d=8, seed=70, act=act, fmt="bf16")
        ub = o.unbundle_layer(o.bundle_rows(ref), ref.b, ref.U, ref.V, "bf16", act)
        assert np.array_equal(ub.w_up, ref.w_up) and np.array_equal(ub.w_downT, ref.w_downT)
        assert act == "relu" or np.array_equal(ub.w_gate, ref.w_gate)
        x = o.round_to(_rng(71).standard_normal(8), "bf16")
        m = _rng(72).random(20) < 0.5
        assert np.array_equal(o.masked_ffn(ub, x, m), o.masked_ffn(ref, x, m))


def check_profile_and_perm(o):
    layer = random_layer(o, f=30, seed=40)
    layer.U = np.zeros_like(layer.U)
    X = _rng(41).standard_normal((7, layer.d_model)).astype(np.float32)
    c = o.profile_counts(layer, X, 0.0)
    assert np.array_equal(c, 7 * (layer.b > 0))
    counts = np.array([3, 9, 3, 0, 9, 1, 3])
    assert o.hot_first_perm(counts).tolist() == [1, 4, 0, 2, 6, 5, 3]
    layer = random_layer(o, f=30, seed=42, act="reglu")
    c = o.profile_counts(layer, X, 0.0)
    perm = o.hot_first_perm(c)
    assert sorted(perm.tolist()) == list(range(30))
    assert np.all(np.diff(c[perm]) <= 0)
    pl = o.permute_layer(layer, perm)
    for x in X:
        r, rp = o.sparse_ffn(layer, x, 0.0), o.sparse_ffn(pl, x, 0.0)
        assert sorted(perm[rp.idx[0]].tolist()) == r.idx[0].tolist()
        assert _rel(rp.y, r.y) < 1e-13


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
