"""The oracle against its pins, and planted mistakes against the same pins.

Each mutant is a fresh copy of the oracle module with one plausible mistake
planted on the CPU; at least one pin must catch it.
"""

import importlib.util
import os
import sys

import numpy as np
import pytest

import oracle
import oracle_pins as pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "sffn_oracle.py")


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(oracle)


def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_mutant", ORACLE_SRC)
    mod = importlib.util.module_from_spec(spec)
    sys.modules["oracle_mutant"] = mod  # dataclasses resolve annotations through sys.modules
    try:
        spec.loader.exec_module(mod)
    finally:
        del sys.modules["oracle_mutant"]
    return mod


def _mutant_no_bias(o):
    orig = o.neuron_activations
    def f(layer, x, idx):
        saved = layer.b
        layer.b = np.zeros_like(saved)
        try:
            return orig(layer, x, idx)
        finally:
            layer.b = saved
    o.neuron_activations = f


def _mutant_gate_up_swapped(o):
    orig = o.neuron_activations
    def f(layer, x, idx):
        if layer.act != "reglu":
            return orig(layer, x, idx)
        swapped = o.OracleLayer(**{**layer.__dict__, "w_up": layer.w_gate, "w_gate": layer.w_up})
        return orig(swapped, x, idx)
    o.neuron_activations = f


def _mutant_threshold_ge(o):
    o.predicted_mask = lambda s, tau: np.asarray(s) >= tau


def _mutant_bias_sign(o):
    orig = o.predictor_scores
    def f(layer, x):
        return orig(layer, x) - 2 * layer.b.astype(np.float64)
    o.predictor_scores = f


def _mutant_down_uses_up_rows(o):
    def masked(layer, x, mask):
        x = np.asarray(x)
        if x.ndim == 2:
            return np.stack([masked(layer, xb, mb) for xb, mb in zip(x, mask)])
        idx = o.active_indices(mask)
        if idx.size == 0:
            return np.zeros(layer.d_model)
        return o.neuron_activations(layer, x, idx) @ o.decode(layer.w_up[idx], layer.fmt)
    o.masked_ffn = masked


def _mutant_mask_ignored(o):
    orig = o.masked_ffn
    o.masked_ffn = lambda layer, x, mask: orig(layer, x, np.ones_like(np.asarray(mask, bool)))


def _mutant_descending_idx(o):
    o.active_indices = lambda m: np.flatnonzero(np.asarray(m, bool))[::-1].astype(np.int32)


def _mutant_unbiased_variance(o):
    def ln(v, gamma=None, beta=None, eps=1e-5):
        v = np.asarray(v, np.float64)
        mu = v.mean(-1, keepdims=True)
        out = (v - mu) / np.sqrt(v.var(-1, ddof=1, keepdims=True) + eps)
        return out if gamma is None else out * gamma + (0 if beta is None else beta)
    o.layernorm = ln


def _mutant_no_residual(o):
    o.residual_layernorm = lambda x, y, fmt, gamma=None, beta=None, eps=1e-5: \
        o.round_to(o.layernorm(np.asarray(y, np.float64), gamma, beta, eps), fmt)


def _mutant_ties_descending(o):
    o.hot_first_perm = lambda c: np.asarray(sorted(range(len(c)), key=lambda i: (-int(c[i]), -i)), np.int32)


def _mutant_bf16_truncate(o):
    orig = o.round_to
    def r(v, fmt):
        if fmt != "bf16":
            return orig(v, fmt)
        return (np.asarray(v, np.float64).astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    o.round_to = r


def _mutant_lookahead_own_input(o):
    def la(layers, x0, n_steps, gamma=None, beta=None, eps=1e-5):
        tr = o.stack_decode(layers, x0, n_steps, gamma, beta, eps)
        ms = [[o.predicted_mask(o.predictor_scores(lay, tr[t][l]), lay.tau) for l, lay in enumerate(layers)]
              for t in range(n_steps)]
        return tr, ms
    o.lookahead_stack_decode = la


def _mutant_lookahead_restarts_each_step(o):
    orig = o.lookahead_stack_decode
    def la(layers, x0, n_steps, gamma=None, beta=None, eps=1e-5):
        tr, ms = [], []
        x = x0
        for _ in range(n_steps):
            t1, m1 = orig(layers, x, 1, gamma, beta, eps)
            tr += t1
            ms += m1
            x = t1[0][-1]
        return tr, ms
    o.lookahead_stack_decode = la


def _mutant_bundle_up_first(o):
    def bundle(layer):
        parts = [layer.w_up] + ([layer.w_gate] if layer.act == "reglu" else []) + [layer.w_downT]
        return np.concatenate([np.asarray(p) for p in parts], axis=1)
    o.bundle_rows = bundle


MUTANTS = [_mutant_no_bias, _mutant_gate_up_swapped, _mutant_threshold_ge, _mutant_bias_sign,
           _mutant_down_uses_up_rows, _mutant_mask_ignored, _mutant_descending_idx,
           _mutant_unbiased_variance, _mutant_no_residual, _mutant_ties_descending,
           _mutant_bf16_truncate, _mutant_lookahead_own_input, _mutant_lookahead_restarts_each_step,
           _mutant_bundle_up_first]


@pytest.mark.parametrize("plant", MUTANTS, ids=lambda m: m.__name__[len("_mutant_"):])
def test_planted_mistake_is_caught(plant):
    mod = _fresh_oracle()
    plant(mod)
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(mod)
        except (AssertionError, ValueError, IndexError, TypeError):
            caught.append(check.__name__)
    assert caught, f"no pin caught {plant.__name__}"
