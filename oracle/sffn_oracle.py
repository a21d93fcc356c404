"""CPU oracle for predictor-gated activation-sparse FFN decode (fp64, numpy).

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline / reference arm may import or call this module.  The
product path (the CUDA library and its Python binding) never does, and this
module imports nothing from it.

What it computes, step by step, in the pages' order:

1. Predictor.  PowerInfer runs an online predictor per layer that scores every
   FFN neuron from the layer input and only the neurons it predicts active are
   computed (PowerInfer page on unite.ai, "Predictores de espacialidad
   adaptativa"; sparsity page on blogs.novita.ai, section "在線推理" / adaptive
   sparse predictor).  The predictor here is the low-rank linear scorer
   s = U (V x) + b, active iff s > tau (strictly).
2. Compaction.  The predicted-active neurons form an ascending index list; this
   plays the role of PowerInfer's neuron table, which maps each computed neuron
   to its row of the original matrix (PowerInfer page, "Colocacion y gestion de
   neuronas").
3. Neuron-aware row gather.  Only the rows of W_up (and W_gate for ReGLU) of the
   listed neurons are read: a_i = max(0, W_up[i].x + b_i), or for ReGLU
   a_i = max(0, W_gate[i].x + b_i) * (W_up[i].x) (PowerInfer page, "Operador
   consciente de neuronas": operators work on individual row/column vectors).
4. Down projection.  y = sum over listed i, ascending, of a_i * W_down^T[i, :].
   Skipped rows contribute nothing because their ReLU output is zero
   (sparsity page, the opening section on ReLU activation sparsity: the
   products of those rows are zero).
5. Dense FFN (the no-skip definition): the same with every neuron listed.
6. Stack: x_{l+1} = round_dtype(LayerNorm(x_l + y_l)), gamma = 1, beta = 0,
   eps = 1e-5, biased variance; the next decode step starts from the last x.
   Look-ahead variant: an asynchronous predictor forecasts a layer's MLP
   sparsity before that layer's input exists (sparsity page, section
   "如何充分利用結構化稀疏性進行加速", the DejaVu design): each layer call's
   mask comes from its own predictor applied to the input of the call
   before it, so prediction can overlap the previous layer's work.
8. Bundled rows: neuron i's rows of Gate, Up and Down stored side by side
   (PowerInfer-2 page, section 4.4: the i-th neurons of the three matrices
   co-activate, so they are bundled); a layout, results unchanged.
7. Offline profile: per-neuron count of predicted activations over profile
   tokens, sorted descending with ties broken by ascending index (hot-first
   order; PowerInfer page, "Fase fuera de linea": the profiler records neuron
   activations and hot neurons are those activated most often).

Inputs are the exact stored bits the GPU path uses (float32 / float16 arrays;
bfloat16 as uint16 bit patterns) and are decoded to fp64 here.
All arithmetic is fp64.  Every function is pinned by the not-gpu tests
(closed forms, invariants, brute force, the worked example of the sparsity
page's "單層計算優化" section).
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

FORMATS = ("f32", "f16", "bf16")


# --------------------------------------------------------------------------
# stored-format decode / rounding
# --------------------------------------------------------------------------

def decode(a: np.ndarray, fmt: str) -> np.ndarray:
    """Stored values -> float64.  bf16 arrives as uint16 bit patterns: a
    bfloat16 is the upper half of an IEEE binary32, so widen by a 16-bit shift."""
    a = np.asarray(a)
    if fmt == "bf16":
        bits = a.astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if fmt in ("f32", "f16"):
        return a.astype(np.float64)
    raise ValueError(f"unknown format {fmt!r}")


def round_to(v: np.ndarray, fmt: str) -> np.ndarray:
    """float64 -> stored format, round to nearest, ties to even.

    bf16 keeps 8 significant bits: write v = m * 2**e with 0.5 <= |m| < 1,
    round m * 2**8 to the nearest integer (ties to even) and scale back.  The
    values rounded here (LayerNorm outputs) are normal and far from overflow."""
    v = np.asarray(v, dtype=np.float64)
    if fmt == "f32":
        return v.astype(np.float32)
    if fmt == "f16":
        return v.astype(np.float16)
    if fmt == "bf16":
        m, e = np.frexp(v)
        r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
        bits = r.astype(np.float32).view(np.uint32) >> np.uint32(16)
        return bits.astype(np.uint16)
    raise ValueError(f"unknown format {fmt!r}")


# --------------------------------------------------------------------------
# the layer as the oracle sees it
# --------------------------------------------------------------------------

@dataclasses.dataclass
class OracleLayer:
    """Stored tensors of one FFN layer; rows are neurons.

    w_up, w_gate, w_downT : [d_ff][d_model]   (w_gate only for ReGLU)
    b                     : [d_ff] float32     (predictor bias == gated bias)
    U                     : [d_ff][rank],  V : [rank][d_model]
    """

    w_up: np.ndarray
    w_downT: np.ndarray
    b: np.ndarray
    U: np.ndarray
    V: np.ndarray
    fmt: str
    act: str = "relu"
    w_gate: Optional[np.ndarray] = None
    tau: float = 0.0

    @property
    def d_ff(self) -> int:
        return self.w_up.shape[0]

    @property
    def d_model(self) -> int:
        return self.w_up.shape[1]


# --------------------------------------------------------------------------
# steps 1-2: predictor, mask, compaction
# --------------------------------------------------------------------------

def predictor_scores(layer: OracleLayer, x: np.ndarray) -> np.ndarray:
    """s = U (V x) + b for one token x [d] (or a batch [B][d] -> [B][d_ff])."""
    xs = decode(x, layer.fmt)
    U = decode(layer.U, layer.fmt)
    V = decode(layer.V, layer.fmt)
    b = layer.b.astype(np.float64)
    if xs.ndim == 1:
        h = V @ xs
        return U @ h + b
    return np.stack([U @ (V @ xb) + b for xb in xs])


def predicted_mask(scores: np.ndarray, tau: float) -> np.ndarray:
    """Active iff the score is strictly above the threshold."""
    return np.asarray(scores) > tau


def active_indices(mask: np.ndarray) -> np.ndarray:
    """Ascending list of the neurons whose mask bit is set (int32)."""
    return np.flatnonzero(np.asarray(mask, dtype=bool)).astype(np.int32)


def band_neurons(scores: np.ndarray, tau: float, width: float = 1e-4) -> np.ndarray:
    """Neurons whose score is within `width` of tau: their predicted bit may
    legitimately differ between two correct implementations."""
    return np.flatnonzero(np.abs(np.asarray(scores) - tau) <= width).astype(np.int32)


def union_mask(masks: np.ndarray) -> np.ndarray:
    """Rows a batch must read: neurons active for at least one token."""
    return np.asarray(masks, dtype=bool).any(axis=0)


# --------------------------------------------------------------------------
# steps 3-5: gathered activations, masked FFN, dense FFN
# --------------------------------------------------------------------------

def neuron_activations(layer: OracleLayer, x: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """a_k for the listed neurons idx[k] of one token x [d]."""
    xs = decode(x, layer.fmt)
    idx = np.asarray(idx, dtype=np.int64)
    b = layer.b.astype(np.float64)[idx]
    up = decode(layer.w_up[idx], layer.fmt) @ xs
    if layer.act == "relu":
        return np.maximum(0.0, up + b)
    if layer.act == "reglu":
        gate = decode(layer.w_gate[idx], layer.fmt) @ xs
        return np.maximum(0.0, gate + b) * up
    raise ValueError(f"unknown activation {layer.act!r}")


def masked_ffn(layer: OracleLayer, x: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """y = sum over the masked-in neurons i (ascending) of a_i * W_down^T[i, :].
    One token x [d], or a batch [B][d] with per-token masks [B][d_ff]."""
    x = np.asarray(x)
    if x.ndim == 2:
        return np.stack([masked_ffn(layer, xb, mb) for xb, mb in zip(x, np.asarray(mask))])
    idx = active_indices(mask)
    if idx.size == 0:
        return np.zeros(layer.d_model)
    a = neuron_activations(layer, x, idx)
    return a @ decode(layer.w_downT[idx], layer.fmt)


def dense_ffn(layer: OracleLayer, x: np.ndarray) -> np.ndarray:
    """The no-skip FFN: W_down^T^T act(W x + b), every neuron computed."""
    x = np.asarray(x)
    if x.ndim == 2:
        return np.stack([dense_ffn(layer, xb) for xb in x])
    xs = decode(x, layer.fmt)
    b = layer.b.astype(np.float64)
    up = decode(layer.w_up, layer.fmt) @ xs
    if layer.act == "relu":
        a = np.maximum(0.0, up + b)
    else:
        a = np.maximum(0.0, decode(layer.w_gate, layer.fmt) @ xs + b) * up
    return decode(layer.w_downT, layer.fmt).T @ a


def exact_mask(layer: OracleLayer, x: np.ndarray) -> np.ndarray:
    """The true activation pattern: neurons whose gated pre-activation is > 0."""
    xs = decode(x, layer.fmt)
    w = layer.w_up if layer.act == "relu" else layer.w_gate
    return decode(w, layer.fmt) @ xs + layer.b.astype(np.float64) > 0.0


@dataclasses.dataclass
class SparseResult:
    y: np.ndarray        # [d] or [B][d] fp64
    scores: np.ndarray   # [d_ff] or [B][d_ff]
    mask: np.ndarray     # bool, same shape as scores
    idx: List[np.ndarray]  # per token ascending index lists


def sparse_ffn(layer: OracleLayer, x: np.ndarray, tau: Optional[float] = None) -> SparseResult:
    """The whole decode-time path for one token or a batch: predict, threshold,
    compact, gather, accumulate."""
    tau = layer.tau if tau is None else tau
    s = predictor_scores(layer, x)
    m = predicted_mask(s, tau)
    y = masked_ffn(layer, x, m)
    idx = [active_indices(mb) for mb in np.atleast_2d(m)]
    return SparseResult(y=y, scores=s, mask=m, idx=idx)


# --------------------------------------------------------------------------
# step 6: residual + LayerNorm between stacked layers
# --------------------------------------------------------------------------

def layernorm(v: np.ndarray, gamma=None, beta=None, eps: float = 1e-5) -> np.ndarray:
    """(v - mean) / sqrt(biased variance + eps) * gamma + beta over the last axis."""
    v = np.asarray(v, dtype=np.float64)
    mu = v.mean(axis=-1, keepdims=True)
    var = ((v - mu) ** 2).mean(axis=-1, keepdims=True)
    out = (v - mu) / np.sqrt(var + eps)
    if gamma is not None:
        out = out * np.asarray(gamma, dtype=np.float64)
    if beta is not None:
        out = out + np.asarray(beta, dtype=np.float64)
    return out


def residual_layernorm(x: np.ndarray, y: np.ndarray, fmt: str, gamma=None, beta=None,
                       eps: float = 1e-5) -> np.ndarray:
    """Next layer input in stored format: round(LN(x + y))."""
    return round_to(layernorm(decode(x, fmt) + np.asarray(y, dtype=np.float64), gamma, beta, eps), fmt)


def stack_decode(layers: Sequence[OracleLayer], x0: np.ndarray, n_steps: int,
                 gamma=None, beta=None, eps: float = 1e-5):
    """Greedy-shaped decode through a stack: each step runs every layer
    (sparse FFN, then residual + LayerNorm) and the next step starts from the
    last layer's output.  Returns the per-step, per-layer inputs
    [n_steps][n_layers + 1][...] in stored format."""
    fmt = layers[0].fmt
    x = np.asarray(x0)
    trace = []
    for _ in range(n_steps):
        xs = [x]
        for layer in layers:
            y = sparse_ffn(layer, x).y
            x = residual_layernorm(x, y, fmt, gamma, beta, eps)
            xs.append(x)
        trace.append(xs)
    return trace


def lookahead_stack_decode(layers: Sequence[OracleLayer], x0: np.ndarray, n_steps: int,
                           gamma=None, beta=None, eps: float = 1e-5):
    """The stack decode with look-ahead masks.  Layer calls are numbered across
    steps (layer l of step t is call t * n_layers + l).  Call k > 0 keeps the
    neurons its own predictor (U, V, b, tau of that layer) scores above tau
    on the input of call k - 1; call 0 has no earlier input and scores its
    own.  The FFN itself, the residual and the LayerNorm are as in
    stack_decode.  Returns (inputs [n_steps][n_layers + 1][...], masks
    [n_steps][n_layers][...]) in stored format / bool."""
    fmt = layers[0].fmt
    x = np.asarray(x0)
    prev = x  # input of the call before the current one
    trace, masks = [], []
    for _ in range(n_steps):
        xs, ms = [x], []
        for layer in layers:
            m = predicted_mask(predictor_scores(layer, prev), layer.tau)
            y = masked_ffn(layer, x, m)
            prev = x
            x = residual_layernorm(x, y, fmt, gamma, beta, eps)
            xs.append(x)
            ms.append(m)
        trace.append(xs)
        masks.append(ms)
    return trace, masks


# --------------------------------------------------------------------------
# step 7: offline profile and hot-first order
# --------------------------------------------------------------------------

def profile_counts(layer: OracleLayer, X: np.ndarray, tau: Optional[float] = None) -> np.ndarray:
    """How many profile tokens each neuron was predicted active for."""
    tau = layer.tau if tau is None else tau
    counts = np.zeros(layer.d_ff, dtype=np.int64)
    for x in np.asarray(X):
        counts += predicted_mask(predictor_scores(layer, x), tau)
    return counts


def hot_first_perm(counts: np.ndarray) -> np.ndarray:
    """perm[new] = old: neurons by descending count, ties by ascending index."""
    counts = np.asarray(counts)
    order = sorted(range(counts.size), key=lambda i: (-int(counts[i]), i))
    return np.asarray(order, dtype=np.int32)


# --------------------------------------------------------------------------
# bundled row layout
# --------------------------------------------------------------------------

def bundle_rows(layer: OracleLayer) -> np.ndarray:
    """Neuron i's rows side by side in one matrix, in the order the
    PowerInfer-2 page names the matrices whose i-th neurons co-activate
    (section 4.4, "Neuron-Cluster-Level Pipeline": Gate, Up and Down):
    [W_gate[i] | W_up[i] | W_down^T[i]] for ReGLU, [W_up[i] | W_down^T[i]]
    for ReLU.  A storage layout: it changes no result."""
    parts = ([layer.w_gate] if layer.act == "reglu" else []) + [layer.w_up, layer.w_downT]
    return np.concatenate([np.asarray(p) for p in parts], axis=1)


def unbundle_layer(bundle: np.ndarray, b, U, V, fmt: str, act: str = "relu", tau: float = 0.0) -> OracleLayer:
    """The layer whose bundled rows are `bundle` (inverse of bundle_rows)."""
    bundle = np.asarray(bundle)
    k = 3 if act == "reglu" else 2
    d = bundle.shape[1] // k
    cols = [bundle[:, j * d:(j + 1) * d] for j in range(k)]
    gate = cols[0] if act == "reglu" else None
    return OracleLayer(w_up=cols[-2], w_downT=cols[-1], b=b, U=U, V=V, fmt=fmt, act=act, w_gate=gate, tau=tau)


def permute_layer(layer: OracleLayer, perm: np.ndarray) -> OracleLayer:
    """Rows of W_up, W_gate, W_down^T, U and b moved together: new row j = old perm[j]."""
    p = np.asarray(perm, dtype=np.int64)
    return dataclasses.replace(
        layer, w_up=layer.w_up[p], w_downT=layer.w_downT[p], b=layer.b[p], U=layer.U[p],
        w_gate=None if layer.w_gate is None else layer.w_gate[p])
