"""Python binding of libsffn (ctypes).  Argument marshalling only: every step
of the sparse FFN runs in the library's CUDA kernels.  Tensors are torch CUDA
tensors used as plain device memory; streams are torch streams.

Importing this module loads libsffn.so and raises if it is missing: there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsffn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with activation_sparse_decode_gb300.build.build() "
                      "(nvcc, sm_103a); the sparse FFN has no non-CUDA implementation")
_lib = ctypes.CDLL(LIB_PATH)

SFFN_OK = 0
STATUS_NAMES = {0: "SFFN_OK", 1: "SFFN_ERR_INVALID_ARG", 2: "SFFN_ERR_UNSUPPORTED", 3: "SFFN_ERR_CUDA",
                4: "SFFN_ERR_CAPACITY", 5: "SFFN_ERR_TIMEOUT", 6: "SFFN_ERR_WORKSPACE"}
DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
ACT_CODES = {"relu": 0, "reglu": 1}

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t


class sffn_layer_info(ctypes.Structure):
    _fields_ = [("fused", _i32), ("grid", _i32), ("blocks_per_sm", _i32), ("cluster", _i32),
                ("ring_stages", _i32), ("hot_stages", _i32)]


class sffn_layer_desc(ctypes.Structure):
    _fields_ = [("d_model", _i32), ("d_ff", _i32), ("rank", _i32), ("max_batch", _i32),
                ("dtype", _i32), ("act", _i32),
                ("w_up", _vp), ("w_gate", _vp), ("w_downT", _vp), ("b", _vp),
                ("pred_U", _vp), ("pred_V", _vp), ("pred_b", _vp), ("tau", ctypes.c_float), ("flags", _i32),
                ("hot_rows", _i32), ("expected_active", ctypes.c_float), ("warm_rows", _i32),
                ("dense_min_batch", _i32)]

SFFN_FLAG_MULTI_KERNEL = 1
SFFN_FLAG_BALANCE = 2
SFFN_FLAG_ROW_GATHER = 4
SFFN_FLAG_STATIC_WEIGHTS = 8
SFFN_FLAG_BUNDLED = 16


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_c = {
    "create": _sig("sffn_create_layer", _i32, ctypes.POINTER(sffn_layer_desc), ctypes.POINTER(_vp)),
    "destroy": _sig("sffn_destroy_layer", _i32, _vp),
    "ws_size": _sig("sffn_workspace_size", _sz, _vp, _i32),
    "layer_info": _sig("sffn_get_layer_info", _i32, _vp, ctypes.POINTER(sffn_layer_info)),
    "ws_init": _sig("sffn_workspace_init", _i32, _vp, _sz, _vp),
    "predict": _sig("sffn_predict", _i32, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp),
    "scores": _sig("sffn_predict_scores", _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp),
    "forward": _sig("sffn_forward", _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _sz, _vp),
    "dense": _sig("sffn_dense_forward", _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp),
    "ln": _sig("sffn_residual_layernorm", _i32, _vp, _vp, _i32, _i32, _i32, _vp, _vp, ctypes.c_float, _vp, _vp),
    "stack": _sig("sffn_forward_stack", _i32, ctypes.POINTER(_vp), _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp,
                  _vp, _vp, ctypes.c_float, _i32, _vp, _sz, _vp),
    "stack_ws": _sig("sffn_stack_workspace_size", _sz, ctypes.POINTER(_vp), _i32, _i32),
    "profile": _sig("sffn_profile_counts", _i32, _vp, _vp, _i32, _vp, _vp, _sz, _vp),
    "hot_first": _sig("sffn_hot_first_perm", _i32, ctypes.POINTER(_i32), _i32, ctypes.POINTER(_i32)),
    "permute": _sig("sffn_permute_rows", _i32, _vp, _vp, _vp, _i32, _i64, _vp),
    "status": _sig("sffn_read_device_status", _i32, _vp, ctypes.POINTER(_i32), _vp),
    "bundle": _sig("sffn_bundle_rows", _i32, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp),
    "debug_wait": _sig("sffn_debug_wait_timeout", _i32, _vp, _sz, _i64, _vp),
    "debug_occupy": _sig("sffn_debug_occupy", _i32, _i64, _i32, _i32, _vp),
    "wait_limit": _sig("sffn_set_wait_limit_ns", _i32, _i64),
    "prof_events": _sig("sffn_set_profile_events", _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _i32),
    "noalloc": _sig("sffn_forward_noalloc", _i32, _vp, _vp, _vp, _vp),
    "noalloc_status": _sig("sffn_noalloc_read_status", _i32, ctypes.POINTER(_i32), _vp),
    "status_string": _sig("sffn_status_string", ctypes.c_char_p, _i32),
    "last_error": _sig("sffn_last_error", ctypes.c_char_p),
    "version": _sig("sffn_version", _i32),
}

EXPORTED = ["sffn_create_layer", "sffn_destroy_layer", "sffn_workspace_size", "sffn_get_layer_info",
            "sffn_workspace_init",
            "sffn_predict", "sffn_predict_scores", "sffn_forward", "sffn_dense_forward",
            "sffn_residual_layernorm", "sffn_forward_stack", "sffn_stack_workspace_size",
            "sffn_profile_counts", "sffn_hot_first_perm", "sffn_permute_rows", "sffn_bundle_rows",
            "sffn_read_device_status",
            "sffn_debug_wait_timeout", "sffn_debug_occupy", "sffn_set_wait_limit_ns", "sffn_set_profile_events", "sffn_forward_noalloc", "sffn_noalloc_read_status",
            "sffn_status_string", "sffn_last_error", "sffn_version"]


class SffnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _check(st: int):
    if st != SFFN_OK:
        raise SffnError(st, _c["last_error"]().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Layer:
    """A layer handle plus references to the tensors it borrows."""

    def __init__(self, w_up, w_downT, b, U, V, pred_b=None, w_gate=None, tau: float = 0.0, max_batch: int = 1,
                 flags: int = 0, hot_rows: int = 0, expected_active: float = 0.0, warm_rows: int = 0,
                 act: Optional[str] = None, dense_min_batch: int = 0):
        """Bundled layers (flags with SFFN_FLAG_BUNDLED) pass the bundle as
        w_up, w_downT = w_gate = None and the activation in `act`."""
        self.tensors = [w_up, w_downT, b, U, V, pred_b, w_gate]
        self.act = act if act is not None else ("reglu" if w_gate is not None else "relu")
        self.dtype = w_up.dtype
        nrows = (3 if self.act == "reglu" else 2) if flags & SFFN_FLAG_BUNDLED else 1
        desc = sffn_layer_desc(
            d_model=w_up.shape[1] // nrows, d_ff=w_up.shape[0], rank=U.shape[1], max_batch=max_batch,
            dtype=DTYPE_CODES[w_up.dtype], act=ACT_CODES[self.act],
            w_up=_ptr(w_up), w_gate=_ptr(w_gate), w_downT=_ptr(w_downT), b=_ptr(b),
            pred_U=_ptr(U), pred_V=_ptr(V), pred_b=_ptr(pred_b if pred_b is not None else b), tau=tau,
            flags=flags, hot_rows=hot_rows, expected_active=expected_active, warm_rows=warm_rows,
            dense_min_batch=dense_min_batch)
        self.desc = desc
        h = ctypes.c_void_p()
        _check(_c["create"](ctypes.byref(desc), ctypes.byref(h)))
        self.handle = h
        self.d_model, self.d_ff, self.rank, self.max_batch = desc.d_model, desc.d_ff, desc.rank, max_batch

    @classmethod
    def from_weights(cls, lw, tau: float = 0.0, max_batch: int = 1, flags: int = 0, hot_rows: int = 0,
                     expected_active: float = 0.0, warm_rows: int = 0, bundled: bool = False,
                     dense_min_batch: int = 0) -> "Layer":
        """From a workloads.LayerWeights already on the GPU.  bundled: the
        rows are first copied into the bundled layout (sffn_bundle_rows) and
        the layer reads that copy."""
        if bundled:
            bnd = bundle_rows(lw.w_up, lw.w_gate, lw.w_downT)
            return cls(bnd, None, lw.b, lw.U, lw.V, pred_b=lw.b, tau=tau, max_batch=max_batch,
                       flags=flags | SFFN_FLAG_BUNDLED, hot_rows=hot_rows, expected_active=expected_active,
                       warm_rows=warm_rows, act=lw.act, dense_min_batch=dense_min_batch)
        return cls(lw.w_up, lw.w_downT, lw.b, lw.U, lw.V, pred_b=lw.b, w_gate=lw.w_gate, tau=tau,
                   max_batch=max_batch, flags=flags, hot_rows=hot_rows, expected_active=expected_active,
                   warm_rows=warm_rows, dense_min_batch=dense_min_batch)

    def close(self):
        if getattr(self, "handle", None):
            _c["destroy"](self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- C-ABI mirrors

def sffn_version() -> int:
    return _c["version"]()


def sffn_create_layer(**kw) -> Layer:
    return Layer(**kw)


def sffn_destroy_layer(layer: Layer):
    layer.close()


def sffn_get_layer_info(layer: Layer) -> dict:
    """How the layer's batch-1 calls run: fused kernel, grid, blocks per SM,
    cluster size, ring stages, hot stages."""
    info = sffn_layer_info()
    _check(_c["layer_info"](layer.handle, ctypes.byref(info)))
    return {k: getattr(info, k) for k, _ in sffn_layer_info._fields_}


def sffn_workspace_size(layer: Layer, batch: int) -> int:
    return int(_c["ws_size"](layer.handle, batch))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace (torch allocations are 512-byte aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def sffn_workspace_init(ws: torch.Tensor, stream=None):
    _check(_c["ws_init"](_ptr(ws), ws.numel(), _stream(stream)))


def sffn_predict(layer: Layer, x: torch.Tensor, idx: torch.Tensor, n_active: torch.Tensor, ws: torch.Tensor,
                 stream=None):
    _check(_c["predict"](layer.handle, _ptr(x), x.shape[0], _ptr(idx), _ptr(n_active), _ptr(ws), ws.numel(),
                         _stream(stream)))


def sffn_predict_scores(layer: Layer, x: torch.Tensor, scores: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(_c["scores"](layer.handle, _ptr(x), x.shape[0], _ptr(scores), _ptr(ws), ws.numel(), _stream(stream)))


def sffn_forward(layer: Layer, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor, idx=None, n_active=None,
                 stream=None):
    _check(_c["forward"](layer.handle, _ptr(x), x.shape[0], _ptr(y), _ptr(idx), _ptr(n_active), _ptr(ws),
                         ws.numel(), _stream(stream)))


def sffn_forward_noalloc(layer: Layer, x: torch.Tensor, y: torch.Tensor, stream=None):
    """Batch-1 forward whose scratch is the library's own fixed array (no
    workspace, no device allocation); see sffn.h for who needs it."""
    _check(_c["noalloc"](layer.handle, _ptr(x), _ptr(y), _stream(stream)))


def sffn_noalloc_read_status(stream=None) -> int:
    """First device-side error of sffn_forward_noalloc calls on the current
    device since the last read (0 if none); reading clears it."""
    st = ctypes.c_int32(0)
    _check(_c["noalloc_status"](ctypes.byref(st), _stream(stream)))
    return st.value


def sffn_dense_forward(layer: Layer, x: torch.Tensor, y: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(_c["dense"](layer.handle, _ptr(x), x.shape[0], _ptr(y), _ptr(ws), ws.numel(), _stream(stream)))


def sffn_residual_layernorm(x: torch.Tensor, y: torch.Tensor, out: torch.Tensor, gamma=None, beta=None,
                            eps: float = 1e-5, stream=None):
    _check(_c["ln"](_ptr(x), _ptr(y), x.shape[0], x.shape[1], DTYPE_CODES[x.dtype], _ptr(gamma), _ptr(beta),
                    eps, _ptr(out), _stream(stream)))


def _handles(layers: Sequence[Layer]):
    arr = (ctypes.c_void_p * len(layers))(*[l.handle.value for l in layers])
    return arr


def sffn_stack_workspace_size(layers: Sequence[Layer], batch: int) -> int:
    return int(_c["stack_ws"](_handles(layers), len(layers), batch))


SFFN_STACK_LOOKAHEAD = 1


def sffn_forward_stack(layers: Sequence[Layer], x0: torch.Tensor, n_steps: int, x_out: torch.Tensor,
                       ws: torch.Tensor, x_trace=None, gamma=None, beta=None, eps: float = 1e-5, stream=None,
                       mask_trace=None, y_trace=None, options: int = 0):
    _check(_c["stack"](_handles(layers), len(layers), _ptr(x0), x0.shape[0], n_steps, _ptr(x_out),
                       _ptr(x_trace), _ptr(mask_trace), _ptr(y_trace), _ptr(gamma), _ptr(beta), eps, options,
                       _ptr(ws), ws.numel(), _stream(stream)))


def sffn_profile_counts(layer: Layer, X: torch.Tensor, counts: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(_c["profile"](layer.handle, _ptr(X), X.shape[0], _ptr(counts), _ptr(ws), ws.numel(), _stream(stream)))


def sffn_hot_first_perm(counts) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(counts, dtype=np.int32))
    perm = np.empty_like(c)
    _check(_c["hot_first"](c.ctypes.data_as(ctypes.POINTER(_i32)), c.size,
                           perm.ctypes.data_as(ctypes.POINTER(_i32))))
    return perm


def sffn_permute_rows(src: torch.Tensor, dst: torch.Tensor, perm: torch.Tensor, stream=None):
    row_bytes = src[0].numel() * src.element_size()
    _check(_c["permute"](_ptr(src), _ptr(dst), _ptr(perm), src.shape[0], row_bytes, _stream(stream)))


def sffn_bundle_rows(w_up: torch.Tensor, w_gate: Optional[torch.Tensor], w_downT: torch.Tensor,
                     bundle: torch.Tensor, stream=None):
    f, d = w_up.shape
    _check(_c["bundle"](_ptr(w_up), _ptr(w_gate), _ptr(w_downT), f, d, DTYPE_CODES[w_up.dtype], _ptr(bundle),
                        _stream(stream)))


def bundle_rows(w_up: torch.Tensor, w_gate: Optional[torch.Tensor], w_downT: torch.Tensor, stream=None):
    """A new [d_ff][(2 or 3) d_model] tensor holding each neuron's rows side by side."""
    f, d = w_up.shape
    nrows = 3 if w_gate is not None else 2
    out = torch.empty(f, nrows * d, dtype=w_up.dtype, device=w_up.device)
    sffn_bundle_rows(w_up, w_gate, w_downT, out, stream)
    return out


def sffn_read_device_status(ws: torch.Tensor, stream=None) -> int:
    st = ctypes.c_int32(0)
    _check(_c["status"](_ptr(ws), ctypes.byref(st), _stream(stream)))
    return st.value


def sffn_debug_wait_timeout(ws: torch.Tensor, timeout_ns: int, stream=None):
    _check(_c["debug_wait"](_ptr(ws), ws.numel(), int(timeout_ns), _stream(stream)))


def sffn_debug_occupy(ns: int, blocks: int, smem_bytes: int, stream=None):
    _check(_c["debug_occupy"](int(ns), int(blocks), int(smem_bytes), _stream(stream)))


def sffn_set_wait_limit_ns(ns: int):
    _check(_c["wait_limit"](int(ns)))


def sffn_set_profile_events(starts: Sequence[torch.cuda.Event] = (), stops: Sequence[torch.cuda.Event] = ()):
    """Bracket the next len(starts) dominant-kernel launches with these
    (timing-enabled, already created) event pairs, one pair per launch; no
    arguments turns it off."""
    n = len(starts)
    assert len(stops) == n
    a = (ctypes.c_void_p * max(n, 1))(*[e.cuda_event for e in starts])
    b = (ctypes.c_void_p * max(n, 1))(*[e.cuda_event for e in stops])
    _check(_c["prof_events"](a, b, n))


def sffn_status_string(st: int) -> str:
    return _c["status_string"](st).decode()


# ---------------------------------------------------------------- conveniences

def permute_layer_weights(lw, perm_dev: torch.Tensor):
    """Hot-first reorder of a LayerWeights on the GPU: rows of W_up, W_gate,
    W_down^T, U and b gathered by the library's permute kernel."""
    import dataclasses

    def pk(t):
        if t is None:
            return None
        src = t if t.dim() == 2 else t.view(-1, 1)
        out = torch.empty_like(src)
        sffn_permute_rows(src, out, perm_dev)
        return out.view_as(t)
    return dataclasses.replace(lw, w_up=pk(lw.w_up), w_gate=pk(lw.w_gate), w_downT=pk(lw.w_downT), b=pk(lw.b),
                               U=pk(lw.U), p=lw.p[perm_dev.cpu().numpy()])


def hot_first_order(layer: Layer, X: torch.Tensor, ws: torch.Tensor) -> np.ndarray:
    """Offline profile pass on the GPU, then the host-side hot-first sort."""
    counts = torch.empty(layer.d_ff, dtype=torch.int32, device=X.device)
    sffn_profile_counts(layer, X, counts, ws)
    return sffn_hot_first_perm(counts.cpu().numpy()), counts


def warm_row_count(counts, n_tokens: int, row_bytes: int, frac: float = 0.2, budget_bytes: int = 32 << 20) -> int:
    """Leading rows of a hot-first order predicted active for at least `frac`
    of the profile tokens, capped so that their rows fit in `budget_bytes`
    (the L2 the batch-1 kernel may fill speculatively)."""
    c = np.asarray(counts.cpu() if hasattr(counts, "cpu") else counts)
    return int(min((c >= frac * n_tokens).sum(), budget_bytes // max(1, row_bytes)))


def hot_row_count(counts, n_tokens: int, frac: float = 0.99) -> int:
    """Neurons predicted active for at least `frac` of the profile tokens: under
    the hot-first order they are the first rows."""
    c = np.asarray(counts.cpu() if hasattr(counts, "cpu") else counts)
    return int((c >= frac * n_tokens).sum())
