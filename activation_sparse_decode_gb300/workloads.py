"""Seeded synthetic workloads for predictor-gated activation-sparse FFN decode.

This module only *draws inputs*: FFN weights, the low-rank predictor factors, the
bias vector and decode tokens, in the stored precision both the CUDA path and the
CPU oracle consume.  It holds none of the method's arithmetic (no predictor
scores, masks, activations or FFN outputs are computed here), so it can serve
the kernels and the oracle alike without coupling them.

Construction (the workload statement of the five FFN shapes; the pages give the
activity levels and the power-law skew only in prose):

* Activation probabilities.  Neuron i gets a Zipf rank k_i from a seeded random
  permutation of 1..d_ff; p_i = min(p_max, c * k_i**-s) with p_max = 0.999 and
  c found by bisection so that mean(p) equals the target activity.  The pages
  report ~10% of neurons active per decode token and a power-law split into a
  small always-hot set and an input-dependent cold set (PowerInfer page, the
  introduction and "Arquitectura y Metodologia"; PowerInfer-2 page, section 3.1).
* Low-rank structure.  U ~ N(0, 1/r) [d_ff][r], V ~ N(0, 1/d) [r][d],
  N ~ N(0, 1/d) [d_ff][d]; the gated matrix (W_up for ReLU, W_gate for ReGLU) is
  round_dtype(U V + 0.1 N).  The predictor stores round_dtype(U), round_dtype(V).
* Bias.  b_i = sigma_i * Phi^-1(p_i) with sigma_i the L2 norm of the stored gated
  row, so that P(W[i] x + b_i > 0) = p_i exactly for x ~ N(0, I).  The same b is
  the predictor bias and the bias of the gated pre-activation.
* W_down^T ~ N(0, 1/d_ff) [d_ff][d]; ReGLU's W_up ~ N(0, 1/d) [d_ff][d].
* Tokens x ~ N(0, I), drawn in fp32 and rounded to the layer dtype.

Every tensor comes from its own counter-derived sub-stream keyed by
(workload, seed, layer, tensor name), so a layer can be regenerated alone.
"""

from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional

import numpy as np
import torch

P_MAX = 0.999

# dtype names used across the C-ABI, the oracle and these fixtures.
TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One FFN decode workload: shapes, precision, activity statistics, steps."""

    name: str
    d_model: int
    d_ff: int
    rank: int
    dtype: str            # "f32" | "f16" | "bf16"
    act: str              # "relu" | "reglu"
    mean_p: float         # target mean activation probability (per layer)
    zipf_s: float         # Zipf exponent of the neuron frequencies
    n_layers: int = 1
    batches: tuple = (1,)
    steps: int = 64       # decode steps (tokens per batch slot)
    reorder: bool = False  # hot-first neuron reordering from a profile pass
    mean_p_range: Optional[tuple] = None  # stacks: per-layer mean ~ U(lo, hi)
    tau: float = 0.0
    profile_tokens: int = 1000

    def layer_mean_p(self, layer: int, seed: int = 0) -> float:
        if self.mean_p_range is None:
            return self.mean_p
        lo, hi = self.mean_p_range
        rng = np.random.Generator(np.random.PCG64(_substream_seed(self.name, seed, layer, "mean_p")))
        return float(rng.uniform(lo, hi))

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five FFN decode workloads.  Readings where the statement is silent: seed 0
# everywhere, tau = 0, the ReGLU layer uses predictor rank 256 (as the
# OPT-6.7B shape at the same d_model), the 40-layer stack uses Zipf s = 1.1.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("opt_relu_d1024_f4096_fp32", 1024, 4096, 128, "f32", "relu", 0.10, 1.1,
                 steps=64),
        Workload("opt6.7b_relu_d4096_f16384_fp16", 4096, 16384, 256, "f16", "relu", 0.10, 1.1,
                 steps=512, reorder=True),
        Workload("llama7b_reglu_d4096_f11008_bf16", 4096, 11008, 256, "bf16", "reglu", 0.12, 1.0,
                 batches=(1, 4, 8, 32), steps=256),
        Workload("opt13b_stack40_d5120_f20480_fp16", 5120, 20480, 384, "f16", "relu", 0.095, 1.1,
                 n_layers=40, steps=128, reorder=True, mean_p_range=(0.04, 0.15)),
        Workload("opt175b_stack48_d12288_f49152_fp16", 12288, 49152, 1024, "f16", "relu", 0.07, 1.2,
                 n_layers=48, batches=(1, 8), steps=64, reorder=True),
    ]
}

# Short aliases in the order the workloads are listed above.
ALIASES = dict(zip(["c1", "c2", "c3", "c4", "c5"], WORKLOADS))


def get_workload(name: str) -> Workload:
    return WORKLOADS[ALIASES.get(name, name)]


def _substream_seed(*key) -> int:
    digest = hashlib.sha256(repr(key).encode()).digest()
    return int.from_bytes(digest[:8], "little") & ((1 << 63) - 1)


def _torch_gen(device, *key) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_substream_seed(*key))
    return g


def zipf_probabilities(d_ff: int, s: float, mean_p: float, seed_key: tuple,
                       p_max: float = P_MAX) -> np.ndarray:
    """p_i = min(p_max, c * rank_i**-s) over a seeded random rank permutation,
    with c bisected so that mean(p) == mean_p to ~1e-13."""
    rng = np.random.Generator(np.random.PCG64(_substream_seed(*seed_key, "zipf_ranks")))
    ranks = rng.permutation(d_ff).astype(np.float64) + 1.0
    base = ranks ** (-s)
    lo, hi = 0.0, p_max / base.min()
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if np.minimum(p_max, mid * base).mean() < mean_p:
            lo = mid
        else:
            hi = mid
    return np.minimum(p_max, 0.5 * (lo + hi) * base)


def _inverse_normal_cdf(p: np.ndarray) -> np.ndarray:
    from scipy.special import ndtri  # library inverse of the standard normal CDF
    return ndtri(p)


@dataclasses.dataclass
class LayerWeights:
    """Stored tensors of one layer (all on one device).  Rows are neurons."""

    w_up: torch.Tensor             # [d_ff][d_model] dtype
    w_gate: Optional[torch.Tensor]  # [d_ff][d_model] dtype (ReGLU) or None
    w_downT: torch.Tensor          # [d_ff][d_model] dtype
    b: torch.Tensor                # [d_ff] fp32 (predictor bias == gated bias)
    U: torch.Tensor                # [d_ff][rank] dtype
    V: torch.Tensor                # [rank][d_model] dtype
    p: np.ndarray                  # [d_ff] fp64 target activation probabilities
    dtype: str
    act: str

    @property
    def d_ff(self) -> int:
        return self.w_up.shape[0]

    @property
    def d_model(self) -> int:
        return self.w_up.shape[1]

    @property
    def rank(self) -> int:
        return self.U.shape[1]

    def to(self, device) -> "LayerWeights":
        mv = lambda t: None if t is None else t.to(device)
        return dataclasses.replace(self, w_up=mv(self.w_up), w_gate=mv(self.w_gate),
                                   w_downT=mv(self.w_downT), b=mv(self.b), U=mv(self.U), V=mv(self.V))

    def permuted(self, perm: torch.Tensor) -> "LayerWeights":
        """Rows reordered: new row j is old row perm[j] (host-side helper for tests)."""
        pi = perm.to(self.w_up.device).long()
        pk = lambda t: None if t is None else t.index_select(0, pi).contiguous()
        return dataclasses.replace(self, w_up=pk(self.w_up), w_gate=pk(self.w_gate),
                                   w_downT=pk(self.w_downT), b=pk(self.b), U=pk(self.U),
                                   p=self.p[perm.cpu().numpy()])


def _randn(shape, std, device, *key) -> torch.Tensor:
    g = _torch_gen(device, *key)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).mul_(std)


def _row_norms_f64(w: torch.Tensor, chunk: int = 2048) -> np.ndarray:
    out = []
    for i in range(0, w.shape[0], chunk):
        out.append(w[i:i + chunk].double().pow(2).sum(1).sqrt().cpu())
    return torch.cat(out).numpy()


def make_layer(wl: Workload, seed: int = 0, layer: int = 0, device="cpu") -> LayerWeights:
    """Draw one layer of workload `wl` in stored precision on `device`."""
    f, d, r = wl.d_ff, wl.d_model, wl.rank
    dt = TORCH_DTYPES[wl.dtype]
    key = (wl.name, seed, layer)
    p = zipf_probabilities(f, wl.zipf_s, wl.layer_mean_p(layer, seed), key)

    U32 = _randn((f, r), r ** -0.5, device, *key, "U")
    V32 = _randn((r, d), d ** -0.5, device, *key, "V")
    gated = _randn((f, d), 0.1 * d ** -0.5, device, *key, "N")
    gated.addmm_(U32, V32)  # U V + 0.1 N, fp32
    gated = gated.to(dt)
    U, V = U32.to(dt), V32.to(dt)
    del U32, V32

    sigma = _row_norms_f64(gated)
    b = torch.from_numpy(sigma * _inverse_normal_cdf(p)).to(torch.float32).to(device)

    w_downT = _randn((f, d), f ** -0.5, device, *key, "W_downT").to(dt)
    if wl.act == "reglu":
        w_gate = gated
        w_up = _randn((f, d), d ** -0.5, device, *key, "W_up").to(dt)
    else:
        w_gate = None
        w_up = gated
    return LayerWeights(w_up=w_up, w_gate=w_gate, w_downT=w_downT, b=b, U=U, V=V, p=p,
                        dtype=wl.dtype, act=wl.act)


def make_tokens(wl: Workload, n_tokens: int, batch: int = 1, seed: int = 0,
                stream: str = "decode", device="cpu") -> torch.Tensor:
    """x ~ N(0, I), [n_tokens][batch][d_model] in the workload dtype."""
    x = _randn((n_tokens, batch, wl.d_model), 1.0, device, wl.name, seed, stream, batch, "x")
    return x.to(TORCH_DTYPES[wl.dtype])


def make_profile_tokens(wl: Workload, n_tokens: Optional[int] = None, seed: int = 1,
                        layer: int = 0, device="cpu") -> torch.Tensor:
    """The offline profile pass's inputs: i.i.d. N(0, I) tokens (seed 1), [n][d]."""
    n = wl.profile_tokens if n_tokens is None else n_tokens
    x = _randn((n, wl.d_model), 1.0, device, wl.name, seed, "profile", layer)
    return x.to(TORCH_DTYPES[wl.dtype])


def tiny_workload(d_model=24, d_ff=96, rank=8, dtype="f32", act="relu", mean_p=0.2,
                  zipf_s=1.1, name="tiny") -> Workload:
    """A small layer for unit tests (same construction, small shapes)."""
    return Workload(name, d_model, d_ff, rank, dtype, act, mean_p, zipf_s)


def to_numpy_stored(t: torch.Tensor) -> np.ndarray:
    """Stored bits as numpy: f32 -> float32, f16 -> float16, bf16 -> uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
