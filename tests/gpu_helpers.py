"""Shared pieces of the GPU parity tests: building layers on the device,
handing their stored bits to the oracle, and the comparison rules.

Comparison rules (readings of the problem statement):
* active-index lists must match the oracle's bit for bit, except for neurons
  whose oracle score lies within 1e-4 of tau (the band), which are counted;
* the output is compared with the oracle's masked FFN over the GPU's own mask,
  so a band neuron decided differently does not count as an output error;
* relative L2 error <= 1e-5 for fp32 weights, <= 1e-3 for fp16/bf16 weights.
"""

import numpy as np
import torch

import oracle
from activation_sparse_decode_gb300 import workloads as W
from activation_sparse_decode_gb300.workloads import to_numpy_stored as st

BAND = 1e-4
TOL = {"f32": 1e-5, "f16": 1e-3, "bf16": 1e-3}


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / nb if nb > 0 else np.linalg.norm(a)


def oracle_layer(lw, tau=0.0):
    return oracle.OracleLayer(
        w_up=st(lw.w_up), w_downT=st(lw.w_downT), b=lw.b.detach().cpu().numpy().astype(np.float32),
        U=st(lw.U), V=st(lw.V), fmt=lw.dtype, act=lw.act,
        w_gate=None if lw.w_gate is None else st(lw.w_gate), tau=tau)


def hot_first(sffn, lw, wl, layer_idx=0, device="cuda"):
    """Offline profile on the GPU (1000 seeded tokens), hot-first perm, rows
    permuted on the GPU.  Returns the permuted weights and the perm."""
    layer = sffn.Layer.from_weights(lw, tau=wl.tau, max_batch=8)
    X = W.make_profile_tokens(wl, layer=layer_idx, device=device)
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layer, 8), device)
    perm, counts = sffn.hot_first_order(layer, X, ws)
    layer.close()
    perm_dev = torch.from_numpy(perm).to(device)
    return sffn.permute_layer_weights(lw, perm_dev), perm, counts[torch.from_numpy(perm).to(device).long()]


def mask_from_list(idx_row, n, f):
    m = np.zeros(f, bool)
    sel = np.asarray(idx_row[:n])
    assert np.all(np.diff(sel) > 0), "active list not strictly ascending"
    assert sel.size == 0 or (sel[0] >= 0 and sel[-1] < f)
    m[sel] = True
    return m


def check_token(ol, x_stored, gpu_mask, y_gpu, tol, tau=0.0):
    """One token: mask parity outside the band, output parity over the GPU mask.
    Returns (band size, band neurons decided differently, rel-L2)."""
    s = oracle.predictor_scores(ol, x_stored)
    mo = oracle.predicted_mask(s, tau)
    band = np.abs(s - tau) <= BAND
    bad = (mo != gpu_mask) & ~band
    assert not bad.any(), f"{bad.sum()} neurons outside the band differ, e.g. {np.flatnonzero(bad)[:8]}"
    ref = oracle.masked_ffn(ol, x_stored, gpu_mask)
    r = rel_l2(y_gpu, ref)
    assert r <= tol, f"rel-L2 {r:.3e} > {tol:g}"
    return int(band.sum()), int(((mo != gpu_mask) & band).sum()), r


class DeviceRows:
    """Row access to a device matrix for the oracle: only the rows the oracle
    asks for are copied back (stored bits, no arithmetic)."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        ii = torch.as_tensor(np.asarray(idx, dtype=np.int64), device=self.t.device)
        return st(self.t.index_select(0, ii))


def lazy_oracle_layer(lw, tau=0.0):
    """Like oracle_layer, but the big matrices stay on the device."""
    return oracle.OracleLayer(
        w_up=DeviceRows(lw.w_up), w_downT=DeviceRows(lw.w_downT),
        b=lw.b.detach().cpu().numpy().astype(np.float32), U=st(lw.U), V=st(lw.V), fmt=lw.dtype, act=lw.act,
        w_gate=None if lw.w_gate is None else DeviceRows(lw.w_gate), tau=tau)


def check_next_input(x_next_gpu, x_next_oracle, fmt):
    """Stored next-layer inputs: equal up to one rounding step of the format on
    a small fraction of elements (fp32 vs fp64 LayerNorm before rounding)."""
    g, o = oracle.decode(x_next_gpu, fmt), oracle.decode(x_next_oracle, fmt)
    ulp = {"f32": 2.0 ** -23, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}[fmt]
    err = np.abs(g - o) / np.maximum(np.abs(o), 2.0 ** -6)
    assert err.max() <= 1.01 * ulp + 1e-5, err.max()
    assert (g != o).mean() < 0.05


def run_tokens(sffn, layer, X, want_idx=True, device="cuda"):
    """Decode the tokens X [T][B][d] one step at a time (batch B per step);
    returns outputs, active lists and counts as numpy arrays."""
    T, B, d = X.shape
    f = layer.d_ff
    ws = sffn.new_workspace(sffn.sffn_workspace_size(layer, B), device)
    Y = torch.empty(T, B, d, dtype=torch.float32, device=device)
    I = torch.empty(T, B, f, dtype=torch.int32, device=device) if want_idx else None
    N = torch.empty(T, B, dtype=torch.int32, device=device) if want_idx else None
    for t in range(T):
        sffn.sffn_forward(layer, X[t], Y[t], ws, None if I is None else I[t], None if N is None else N[t])
    torch.cuda.synchronize()
    assert sffn.sffn_read_device_status(ws) == 0
    return Y.cpu().numpy(), None if I is None else I.cpu().numpy(), None if N is None else N.cpu().numpy()
