"""The no-allocation entry point (collected last on purpose).

sffn_forward_noalloc serves callers that cannot allocate device memory -- a
runtime that owns all device memory in a fixed pool, or a host program whose
memory belongs to another framework's allocator -- by keeping the kernel's
scratch in a fixed array inside the library.  Its output must match the
workspace-based sffn_forward on the same layer and token, on two calls in a row
(the second call reuses the array the first one left behind)."""

import numpy as np
import pytest
import torch

from activation_sparse_decode_gb300 import workloads as W
from gpu_helpers import TOL, rel_l2

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


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_noalloc_matches_workspace_forward(sffn, name):
    wl = W.get_workload(name)
    lw = W.make_layer(wl, device=DEV)
    layer = sffn.Layer.from_weights(lw, tau=wl.tau)
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layer, 1), DEV)
    X = W.make_tokens(wl, 2, device=DEV)
    for t in range(2):  # two calls in a row
        y_ref = torch.empty(1, wl.d_model, dtype=torch.float32, device=DEV)
        y = torch.full((1, wl.d_model), float("nan"), dtype=torch.float32, device=DEV)
        sffn.sffn_forward(layer, X[t], y_ref, ws)
        sffn.sffn_forward_noalloc(layer, X[t], y)
        torch.cuda.synchronize()
        a, b = y.cpu().numpy(), y_ref.cpu().numpy()
        assert np.isfinite(a).all()
        assert rel_l2(a, b) <= TOL[wl.dtype], (t, rel_l2(a, b))


def test_noalloc_rejects_layers_without_the_single_launch_kernel(sffn):
    wl = W.tiny_workload(d_model=256, d_ff=512, rank=16, dtype="f16", name="noalloc-multi")
    lw = W.make_layer(wl, device=DEV)
    layer = sffn.Layer.from_weights(lw, flags=sffn.SFFN_FLAG_MULTI_KERNEL)
    y = torch.empty(1, wl.d_model, dtype=torch.float32, device=DEV)
    with pytest.raises(sffn.SffnError) as e:
        sffn.sffn_forward_noalloc(layer, W.make_tokens(wl, 1, device=DEV)[0], y)
    assert e.value.status == 2
