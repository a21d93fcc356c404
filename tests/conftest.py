import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of wall time")


def oracle_layer_from(lw, tau=0.0):
    """Stored tensors of a generated layer, as numpy arrays for the oracle."""
    import oracle
    from activation_sparse_decode_gb300.workloads import to_numpy_stored as st
    return oracle.OracleLayer(
        w_up=st(lw.w_up), w_downT=st(lw.w_downT), b=lw.b.detach().cpu().numpy().astype(np.float32),
        U=st(lw.U), V=st(lw.V), fmt=lw.dtype, act=lw.act,
        w_gate=None if lw.w_gate is None else st(lw.w_gate), tau=tau)


@pytest.fixture(scope="session")
def have_gpu():
    import torch
    return torch.cuda.is_available()
