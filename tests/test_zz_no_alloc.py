"""The no-allocation entry point (collected last on purpose).

sffn_forward_noalloc serves callers that cannot allocate device memory -- a
runtime that owns all device memory in a fixed pool, or a host program whose
memory belongs to another framework's allocator -- by keeping the kernel's
scratch in a fixed array inside the library.  Its output must match the
workspace-based sffn_forward on the same layer and token, on two calls in a row
(the second call reuses the array the first one left behind), and the oracle.
Cases: two blocks per SM (the ReLU d1024 fp32 and OPT-6.7B-shaped layers), one
block per SM in pairs of blocks that share their rows (48 KB rows), and a layer
created with SFFN_FLAG_STATIC_WEIGHTS."""

import numpy as np
import pytest
import torch

from activation_sparse_decode_gb300 import workloads as W
from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
from gpu_helpers import TOL, check_elementwise, check_token, mask_from_list, oracle_layer, rel_l2

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


CASES = {
    "c1": (lambda: W.get_workload("c1"), 0, None),
    "c2": (lambda: W.get_workload("c2"), 0, None),
    "pairs": (lambda: W.tiny_workload(d_model=12288, d_ff=4096, rank=64, dtype="f16", mean_p=0.1,
                                      name="noalloc-pairs"), 0, 2),
    "static": (lambda: W.get_workload("c3"), 8, None),
}


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_workspace_forward(sffn, case):
    make_wl, flags, cluster = CASES[case]
    wl = make_wl()
    lw = W.make_layer(wl, device=DEV)
    layer = sffn.Layer.from_weights(lw, tau=wl.tau, flags=flags)
    if cluster is not None:
        assert sffn.sffn_get_layer_info(layer)["cluster"] == cluster
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layer, 1), DEV)
    X = W.make_tokens(wl, 2, device=DEV)
    ol = oracle_layer(lw, wl.tau)
    for t in range(2):  # two calls in a row
        y_ref = torch.empty(1, wl.d_model, dtype=torch.float32, device=DEV)
        idx = torch.empty(1, wl.d_ff, dtype=torch.int32, device=DEV)
        n = torch.empty(1, dtype=torch.int32, device=DEV)
        y = torch.full((1, wl.d_model), float("nan"), dtype=torch.float32, device=DEV)
        sffn.sffn_forward(layer, X[t], y_ref, ws, idx, n)
        sffn.sffn_forward_noalloc(layer, X[t], y)
        torch.cuda.synchronize()
        assert sffn.sffn_noalloc_read_status() == 0
        a, b = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(a).all()
        assert rel_l2(a, b) <= TOL[wl.dtype], (t, rel_l2(a, b))
        check_elementwise(a[0], b[0], wl.dtype, "noalloc vs workspace")
        # the same mask (the predictor is deterministic), so the oracle's
        # masked FFN over the workspace call's list checks both outputs
        m = mask_from_list(idx[0].cpu().numpy(), int(n.item()), wl.d_ff)
        check_token(ol, st(X[t])[0], m, a[0], TOL[wl.dtype], wl.tau)
    assert sffn.sffn_read_device_status(ws) == 0


def test_noalloc_rejects_layers_without_the_single_launch_kernel(sffn):
    wl = W.tiny_workload(d_model=256, d_ff=512, rank=16, dtype="f16", name="noalloc-multi")
    lw = W.make_layer(wl, device=DEV)
    layer = sffn.Layer.from_weights(lw, flags=sffn.SFFN_FLAG_MULTI_KERNEL)
    y = torch.empty(1, wl.d_model, dtype=torch.float32, device=DEV)
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_forward_noalloc(layer, W.make_tokens(wl, 1, device=DEV)[0], y)
    assert e.value.status == 2
