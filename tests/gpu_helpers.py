"""Shared pieces of the GPU parity tests: building layers on the device,
handing their stored bits to the oracle, and the comparison rules.

Comparison rules (readings of the problem statement):
* active-index lists must match the oracle's bit for bit, except for neurons
  whose oracle score lies within 1e-4 of tau (the band), which are counted;
* the output is compared with the oracle's masked FFN over the GPU's own mask,
  so a band neuron decided differently does not count as an output error;
* relative L2 error <= 1e-5 for fp32 weights, <= 1e-3 for fp16/bf16 weights;
* and element by element (ELEM_EPS below): the L2 bar alone cannot see one
  wrong element, e.g. one neuron's contribution added twice or dropped.
"""

import numpy as np
import torch

import oracle
from activation_sparse_decode_gb300 import workloads as W
from activation_sparse_decode_gb300.workloads import to_numpy_stored as st

BAND = 1e-4
TOL = {"f32": 1e-5, "f16": 1e-3, "bf16": 1e-3}

# Element-wise bound: |y_gpu[j] - y_oracle[j]| <= ELEM_EPS * (|y_oracle[j]| + rms(y_oracle)).
# Derivation.  The GPU sums in fp32 (unit roundoff u = 2^-24), in tree orders:
# each output element is a sum of n neuron terms a_i W[i, j] (n = active
# neurons, 400-13000 here) whose a_i are themselves fp32 dot products over
# d_model; for random-sign terms the rounding error grows like u * sqrt(terms)
# times the partial sums, about 1e-6 of rms(y) for the widest layer.  The
# batch tensor-core path feeds a_i to the second product as a 16-bit high part
# plus a 16-bit remainder (relative error <= 2^-17 per term for bf16), and the
# tensor cores' fp32 accumulation may truncate (2u per step); together about
# 1e-4 of rms(y) at most.  ELEM_EPS is 2^-10 ~ 1e-3 (2^-16 for fp32 weights,
# which never take the 16-bit split): ten times that estimate, while one
# neuron's term a_i W[i, j] is about rms(y) / sqrt(n) >= 0.009 rms(y) for every
# workload here, so a single misplaced term on one element still fails.
ELEM_EPS = {"f32": 2.0 ** -16, "f16": 2.0 ** -10, "bf16": 2.0 ** -10}


def elementwise_ratio(y_gpu, y_ref, fmt):
    """max over j of |y_gpu[j] - y_ref[j]| / (ELEM_EPS * (|y_ref[j]| + rms(y_ref))); <= 1 passes."""
    g, r = np.asarray(y_gpu, np.float64), np.asarray(y_ref, np.float64)
    scale = np.abs(r) + np.sqrt(np.mean(r * r))
    err = np.abs(g - r)
    if not np.any(scale > 0):
        return 0.0 if not np.any(err > 0) else np.inf
    return float(np.max(err / (ELEM_EPS[fmt] * scale)))


def check_elementwise(y_gpu, y_ref, fmt, what="y"):
    ratio = elementwise_ratio(y_gpu, y_ref, fmt)
    if ratio > 1.0:
        g, r = np.asarray(y_gpu, np.float64), np.asarray(y_ref, np.float64)
        j = int(np.argmax(np.abs(g - r) / (np.abs(r) + np.sqrt(np.mean(r * r)) + 1e-300)))
        raise AssertionError(f"{what}: element {j} off by {abs(g[j] - r[j]):.3e} (gpu {g[j]:.6e}, oracle {r[j]:.6e}); "
                             f"{ratio:.2f} x the element-wise bound")
    return ratio


def ulp_distance(a, b, fmt):
    """Number of representable values of the stored format between a and b
    (stored bits: float32 / float16 arrays, bf16 as uint16 patterns)."""
    def ordered(v):
        if fmt == "f32":
            i = np.asarray(v, np.float32).view(np.int32).astype(np.int64)
            return np.where(i < 0, -(i & 0x7FFFFFFF), i)
        bits = (np.asarray(v, np.float16).view(np.uint16) if fmt == "f16" else np.asarray(v, np.uint16)).astype(np.int64)
        return np.where(bits & 0x8000, -(bits & 0x7FFF), bits)
    return np.abs(ordered(a) - ordered(b))


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


def same_lists(I1, N1, I2, N2):
    """Two runs' active lists agree: equal counts, and equal first N entries
    of every list (entries past a list's count are not written)."""
    if not np.array_equal(N1, N2):
        return False
    I1, I2, N1 = np.asarray(I1), np.asarray(I2), np.asarray(N1)
    for ix in np.ndindex(N1.shape):
        n = int(N1[ix])
        if not np.array_equal(I1[ix][:n], I2[ix][:n]):
            return False
    return True


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
    check_elementwise(y_gpu, ref, ol.fmt)
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


def check_next_input(x_next_gpu, x_next_oracle, fmt, max_frac=0.05):
    """Stored next-layer inputs: equal up to one rounding step of the format
    (ulp distance <= 1) on a small fraction of elements.  Where the oracle's
    value was formed from the GPU's own y, only fp32 against fp64 LayerNorm
    arithmetic separates the two (a few 2^-24 relative before rounding to a
    2^-11 or 2^-8 half-step), so callers pass a smaller fraction then."""
    dist = ulp_distance(x_next_gpu, x_next_oracle, fmt)
    assert dist.max() <= 1, f"next input: element {int(np.argmax(dist))} is {int(dist.max())} ulps off"
    assert (dist > 0).mean() < max_frac, (dist > 0).mean()


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
