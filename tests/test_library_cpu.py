"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, validates arguments before touching a device, and its
host-side hot-first sort matches the oracle."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sffn.h")


@pytest.fixture(scope="module")
def lib():
    from activation_sparse_decode_gb300 import build
    build.build()
    from activation_sparse_decode_gb300 import sffn
    return sffn


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sffn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("sffn_create_layer", "sffn_predict", "sffn_forward", "sffn_forward_stack"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in sffn.h but not exported"
    assert sorted(lib.EXPORTED) == declared_functions()


def test_version_and_status_strings(lib):
    assert lib.sffn_version() >= 1
    assert lib.sffn_status_string(0) == "ok"
    assert "timed out" in lib.sffn_status_string(5)


def test_hot_first_perm_matches_oracle(lib):
    g = np.random.Generator(np.random.PCG64(0))
    for f in (1, 7, 100, 4096):
        counts = g.integers(0, 20, size=f).astype(np.int32)
        assert np.array_equal(lib.sffn_hot_first_perm(counts), oracle.hot_first_perm(counts))
    counts = np.array([3, 9, 3, 0, 9, 1, 3], np.int32)
    assert lib.sffn_hot_first_perm(counts).tolist() == [1, 4, 0, 2, 6, 5, 3]


def _desc(lib, **kw):
    base = dict(d_model=64, d_ff=128, rank=16, max_batch=1, dtype=1, act=0, w_up=256, w_gate=None,
                w_downT=512, b=768, pred_U=1024, pred_V=1280, pred_b=1536, tau=0.0)
    base.update(kw)
    return lib.sffn_layer_desc(**base)


@pytest.mark.parametrize("bad", [
    dict(d_model=0), dict(d_ff=-1), dict(rank=0), dict(max_batch=0), dict(max_batch=33), dict(dtype=7),
    dict(act=3), dict(d_model=60), dict(rank=12), dict(w_up=None), dict(w_up=258), dict(pred_b=None),
    dict(act=1), dict(w_gate=2048)])
def test_create_layer_rejects_bad_descriptors_without_a_device(lib, bad):
    d = _desc(lib, **bad)
    h = ctypes.c_void_p()
    st = lib._c["create"](ctypes.byref(d), ctypes.byref(h))
    assert st == 1, (bad, st, lib._c["last_error"]().decode())
    assert h.value is None


def test_null_arguments(lib):
    assert lib._c["create"](None, None) == 1
    assert lib._c["ws_size"](None, 1) == 0
    assert lib._c["hot_first"](None, 4, None) == 1
    assert lib._c["permute"](None, None, None, 1, 16, None) == 1
    assert lib._c["wait_limit"](0) == 1
