"""GPU parity of the batched union-of-active-rows path (tensor cores): batches
of 8 to 32 tokens against the CPU oracle, token by token, on ragged shapes,
degenerate masks and several neuron tiles per block; and against the
CUDA-core row gather on the same inputs."""

import numpy as np
import pytest
import torch

import oracle
from activation_sparse_decode_gb300 import workloads as W
from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
from gpu_helpers import TOL, check_elementwise, check_token, mask_from_list, oracle_layer, rel_l2, run_tokens, same_lists

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


UNION = [  # (d_model, d_ff, rank, dtype, act, batch, mean activity)
    (128, 1000, 16, "f16", "relu", 8, 0.2),
    (256, 777, 16, "bf16", "reglu", 9, 0.15),
    (1024, 4097, 64, "bf16", "reglu", 17, 0.1),
    (384, 100, 8, "f16", "reglu", 32, 0.3),      # fewer union members than blocks
    (2048, 6000, 128, "f16", "relu", 32, 0.12),
    (12288, 500, 256, "f16", "relu", 8, 0.2),    # wide rows, 96 GEMM1 jobs per tile
    (1024, 20000, 64, "bf16", "relu", 24, 0.4),  # about 0.99 of the neurons in the union
]


@pytest.mark.parametrize("shape", UNION, ids=lambda s: "d%d_f%d_r%d_%s_%s_b%d_p%g" % s)
def test_union_ragged(sffn, shape):
    d, f, r, dt, act, batch, p = shape
    wl = W.tiny_workload(d_model=d, d_ff=f, rank=r, dtype=dt, act=act, mean_p=p, name=f"union{shape}")
    lw = W.make_layer(wl, device=DEV)
    ol = oracle_layer(lw)
    layer = sffn.Layer.from_weights(lw, max_batch=batch)
    gather = sffn.Layer.from_weights(lw, max_batch=batch, flags=sffn.SFFN_FLAG_ROW_GATHER)
    X = W.make_tokens(wl, 2, batch=batch, device=DEV)
    Y, I, N = run_tokens(sffn, layer, X)
    Yg, Ig, Ng = run_tokens(sffn, gather, X)
    assert same_lists(I, N, Ig, Ng)
    Xh = st(X)
    for s in range(2):
        for b in range(batch):
            m = mask_from_list(I[s, b], N[s, b], f)
            _, _, r = check_token(ol, Xh[s, b], m, Y[s, b], TOL[dt])
            # The activations enter the second product as a 16-bit high part
            # plus a 16-bit remainder, so both paths stay at fp32 accuracy
            # (sqrt(d) * 2^-24 for the sums, 2^-17 for the bf16 split), far
            # inside the 1e-3 bar.
            assert r < 1e-4
            ref = oracle.masked_ffn(ol, Xh[s, b], m)
            assert rel_l2(Yg[s, b], ref) < 1e-4
            check_elementwise(Yg[s, b], ref, dt)


# Wide predictor ranks on the batch path (the OPT-175B shape's rank is 1024):
# ragged 16-row groups of the hidden layer's clusters, every token-column
# width, and the ReGLU form.
WIDE_RANK = [  # (d_model, d_ff, rank, dtype, act, batch, mean activity)
    (4096, 3000, 1024, "f16", "relu", 8, 0.15),
    (1536, 2500, 1088, "bf16", "reglu", 20, 0.12),  # 17 row tiles, three jobs per block
    (2048, 1500, 1024, "bf16", "relu", 32, 0.2),
]


@pytest.mark.parametrize("shape", WIDE_RANK, ids=lambda s: "d%d_f%d_r%d_%s_%s_b%d_p%g" % s)
def test_union_wide_rank_predictor(sffn, shape):
    """Masks and outputs against the oracle token by token (masks outside the
    band), and the same lists from a second run of the same inputs (the
    hidden layer's cluster reduction runs in a fixed order)."""
    d, f, r, dt, act, batch, p = shape
    wl = W.tiny_workload(d_model=d, d_ff=f, rank=r, dtype=dt, act=act, mean_p=p, name=f"widerank{shape}")
    lw = W.make_layer(wl, device=DEV)
    ol = oracle_layer(lw)
    layer = sffn.Layer.from_weights(lw, max_batch=batch)
    X = W.make_tokens(wl, 2, batch=batch, device=DEV)
    Y, I, N = run_tokens(sffn, layer, X)
    Y2, I2, N2 = run_tokens(sffn, layer, X)
    assert same_lists(I, N, I2, N2)
    assert np.array_equal(N, N2)
    Xh = st(X)
    for s in range(2):
        for b in range(batch):
            m = mask_from_list(I[s, b], N[s, b], f)
            check_token(ol, Xh[s, b], m, Y[s, b], TOL[dt])


@pytest.mark.parametrize("batch", [8, 32])
@pytest.mark.parametrize("tau,expect", [(1e30, "none"), (-1e30, "all")])
def test_union_degenerate_masks(sffn, tau, expect, batch):
    """Empty union (every block idle, y stays zero) and the full union: 40000
    neurons over 152 blocks is three tiles of up to 128 neurons per block."""
    wl = W.tiny_workload(d_model=256, d_ff=40000, rank=16, dtype="bf16", act="reglu", name="union-degenerate")
    lw = W.make_layer(wl, device=DEV)
    ol = oracle_layer(lw, tau)
    layer = sffn.Layer.from_weights(lw, tau=tau, max_batch=batch)
    X = W.make_tokens(wl, 1, batch=batch, device=DEV)
    Y, I, N = run_tokens(sffn, layer, X)
    if expect == "none":
        assert (N == 0).all()
        assert (Y == 0).all()
    else:
        assert (N == wl.d_ff).all()
        Xh = st(X)
        for b in range(batch):
            ref = oracle.dense_ffn(ol, Xh[0, b])
            assert rel_l2(Y[0, b], ref) < TOL["bf16"]
            check_elementwise(Y[0, b], ref, "bf16")


def test_union_tokens_keep_their_own_neurons(sffn):
    """Tokens with disjoint predicted sets share a batch: each token's output
    must use its own neurons only.  Half the tokens are the negatives of the
    others; with a zero bias the linear scorer gives them complementary masks,
    so the union is (almost) every neuron while each token keeps about half."""
    wl = W.tiny_workload(d_model=512, d_ff=3000, rank=32, dtype="f16", act="relu", name="union-split")
    lw = W.make_layer(wl, device=DEV)
    lw.b = torch.zeros_like(lw.b)
    ol = oracle_layer(lw)
    layer = sffn.Layer.from_weights(lw, max_batch=16)
    X = W.make_tokens(wl, 1, batch=8, device=DEV)[0]
    X = torch.cat([X, -X], 0).unsqueeze(0).contiguous()
    Y, I, N = run_tokens(sffn, layer, X)
    assert (N[0, :8] + N[0, 8:] <= wl.d_ff).all() and (N[0] > 0).all()
    Xh = st(X)
    for b in range(16):
        check_token(ol, Xh[0, b], mask_from_list(I[0, b], N[0, b], wl.d_ff), Y[0, b], TOL["f16"])


DENSE = [  # (d_model, d_ff, rank, dtype, act, batch, mean activity)
    (1024, 4097, 64, "bf16", "reglu", 17, 0.1),
    (2048, 6000, 128, "f16", "relu", 32, 0.12),
    (512, 3000, 32, "f16", "relu", 2, 0.3),
    (12288, 500, 256, "f16", "relu", 8, 0.2),
    (4096, 11008, 256, "bf16", "reglu", 32, 0.12),
]


@pytest.mark.parametrize("shape", DENSE, ids=lambda s: "d%d_f%d_r%d_%s_%s_b%d_p%g" % s)
def test_dense_fallback(sffn, shape):
    """The dense fallback (every row, two tensor-core GEMMs, the tokens' masks
    between them) against the oracle's masked FFN token by token, and against
    the union path on the same inputs: the masks are the same predictor's,
    and each token still keeps only its own neurons."""
    d, f, r, dt, act, batch, p = shape
    wl = W.tiny_workload(d_model=d, d_ff=f, rank=r, dtype=dt, act=act, mean_p=p, name=f"dense{shape}")
    lw = W.make_layer(wl, device=DEV)
    ol = oracle_layer(lw)
    dense = sffn.Layer.from_weights(lw, max_batch=batch, dense_min_batch=2)
    union = sffn.Layer.from_weights(lw, max_batch=batch)
    X = W.make_tokens(wl, 2, batch=batch, device=DEV)
    Y, I, N = run_tokens(sffn, dense, X)
    Yu, Iu, Nu = run_tokens(sffn, union, X)
    assert same_lists(I, N, Iu, Nu)
    Xh = st(X)
    for s in range(2):
        for b in range(batch):
            m = mask_from_list(I[s, b], N[s, b], f)
            check_token(ol, Xh[s, b], m, Y[s, b], TOL[dt])
            check_elementwise(Y[s, b], Yu[s, b], dt, "dense fallback vs union path")


def test_dense_fallback_bounds(sffn):
    wl = W.tiny_workload(d_model=256, d_ff=512, rank=16, dtype="f32", name="dense-bad")
    lw = W.make_layer(wl, device=DEV)
    with pytest.raises(sffn.SffnError) as e:
        sffn.Layer.from_weights(lw, max_batch=4, dense_min_batch=2)
    assert e.value.status == 2
    wl = W.tiny_workload(d_model=256, d_ff=512, rank=16, dtype="f16", name="dense-bad16")
    lw = W.make_layer(wl, device=DEV)
    with pytest.raises(sffn.SffnError) as e:
        sffn.Layer.from_weights(lw, max_batch=4, dense_min_batch=33)
    assert e.value.status == 1
