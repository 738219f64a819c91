"""The pins of the feature-map and layer oracles catch plausible mistakes.

Each case plants one mistake in a copy of an oracle function (on the CPU, in
this process only), runs the pin tests of that oracle against it and requires
at least one of them to fail: a dropped term, a wrong scale, a transposed
operand, a lost mask, a misplaced eps, a swapped projection.
"""
import numpy as np
import pytest

from oracle import feature_maps as fm
from oracle import layer

import test_oracle_features as pins_fm
import test_oracle_layer as pins_layer


def _prf_no_half_norm(x, W, shift=0.0):
    x, W = np.asarray(x, float), np.asarray(W, float)
    return np.exp(x @ W.T - shift) / np.sqrt(W.shape[0])


def _prf_wrong_scale(x, W, shift=0.0):
    x, W = np.asarray(x, float), np.asarray(W, float)
    return np.exp(x @ W.T - 0.5 * (x * x).sum(-1, keepdims=True) - shift) / W.shape[0]


def _prf_shift_added(x, W, shift=0.0):
    x, W = np.asarray(x, float), np.asarray(W, float)
    return np.exp(x @ W.T - 0.5 * (x * x).sum(-1, keepdims=True) + shift) / np.sqrt(W.shape[0])


def _attn_no_mask(fq, fk, v, causal, eps=1e-6):
    fq, fk, v = (np.asarray(a, float) for a in (fq, fk, v))
    w = fq @ np.swapaxes(fk, -1, -2)
    return (w @ v) / (w.sum(axis=-1, keepdims=True) + eps)


def _attn_exclusive(fq, fk, v, causal, eps=1e-6):
    fq, fk, v = (np.asarray(a, float) for a in (fq, fk, v))
    w = fq @ np.swapaxes(fk, -1, -2)
    if causal:
        w = np.tril(w, k=-1)
    with np.errstate(invalid="ignore", divide="ignore"):   # row 0 has no weight at all
        return (w @ v) / (w.sum(axis=-1, keepdims=True) + eps)


def _attn_eps_in_numerator(fq, fk, v, causal, eps=1e-6):
    fq, fk, v = (np.asarray(a, float) for a in (fq, fk, v))
    w = fq @ np.swapaxes(fk, -1, -2)
    if causal:
        w = np.tril(w)
    return (w @ v + eps) / w.sum(axis=-1, keepdims=True)


FEATURE_PINS = [
    pins_fm.test_elu_features_match_the_c_oracle,
    pins_fm.test_quadratic_and_recurrent_forms_agree,
    pins_fm.test_decode_steps_reproduce_the_causal_rows,
    pins_fm.test_two_tokens_by_hand,
    pins_fm.test_random_features_estimate_the_exponential_kernel,
    pins_fm.test_random_features_closed_forms,
    pins_fm.test_random_features_approach_softmax_attention,
]


def _some_pin_fails(pins):
    failed = 0
    for pin in pins:
        args = {"causal": [True, False]} if "causal" in pin.__code__.co_varnames[:pin.__code__.co_argcount] else None
        try:
            if args:
                for c in args["causal"]:
                    pin(c)
            else:
                pin()
        except AssertionError:
            failed += 1
    return failed > 0


@pytest.mark.parametrize("name,mutant", [
    ("positive_random_features", _prf_no_half_norm),
    ("positive_random_features", _prf_wrong_scale),
    ("positive_random_features", _prf_shift_added),
    ("attention_from_features", _attn_no_mask),
    ("attention_from_features", _attn_exclusive),
    ("attention_from_features", _attn_eps_in_numerator),
])
def test_feature_map_pins_catch_a_planted_mistake(monkeypatch, name, mutant):
    monkeypatch.setattr(fm, name, mutant)
    assert _some_pin_fails(FEATURE_PINS), f"no pin caught the planted mistake in {name}"


def _layer_swapped_kv(x, Wqkv, Wo, S, z, H, eps=1e-6):
    import oracle
    x, Wqkv, Wo = (np.asarray(a, float) for a in (x, Wqkv, Wo))
    B, dm = x.shape
    D = dm // H
    qkv = x @ Wqkv
    q = qkv[:, 0:dm].reshape(B, H, D)
    v = qkv[:, dm:2 * dm].reshape(B, H, D)        # k and v exchanged
    k = qkv[:, 2 * dm:3 * dm].reshape(B, H, D)
    return oracle.decode_step(q, k, v, S, z, eps).reshape(B, dm) @ Wo


def _layer_wo_transposed(x, Wqkv, Wo, S, z, H, eps=1e-6):
    import oracle
    x, Wqkv, Wo = (np.asarray(a, float) for a in (x, Wqkv, Wo))
    B, dm = x.shape
    D = dm // H
    qkv = x @ Wqkv
    q, k, v = (qkv[:, i * dm:(i + 1) * dm].reshape(B, H, D) for i in range(3))
    return oracle.decode_step(q, k, v, S, z, eps).reshape(B, dm) @ Wo.T


def _layer_heads_interleaved(x, Wqkv, Wo, S, z, H, eps=1e-6):
    import oracle
    x, Wqkv, Wo = (np.asarray(a, float) for a in (x, Wqkv, Wo))
    B, dm = x.shape
    D = dm // H
    qkv = x @ Wqkv
    # head h taken as the strided columns h, h + H, ... instead of h D .. h D + D - 1
    q, k, v = (qkv[:, i * dm:(i + 1) * dm].reshape(B, D, H).transpose(0, 2, 1) for i in range(3))
    o = oracle.decode_step(np.ascontiguousarray(q), np.ascontiguousarray(k),
                           np.ascontiguousarray(v), S, z, eps)
    return o.reshape(B, dm) @ Wo


LAYER_PINS = [
    pins_layer.test_identity_projections_reduce_to_the_decode_step,
    pins_layer.test_steps_equal_causal_attention_on_the_projected_sequence,
    pins_layer.test_output_is_linear_in_Wo,
]


@pytest.mark.parametrize("mutant", [_layer_swapped_kv, _layer_wo_transposed,
                                    _layer_heads_interleaved])
def test_layer_pins_catch_a_planted_mistake(monkeypatch, mutant):
    monkeypatch.setattr(layer, "layer_decode_step", mutant)
    assert _some_pin_fails(LAYER_PINS), f"no pin caught {mutant.__name__}"
