"""Pins of the float64 gradient oracle (oracle/backward.py), CPU only.

The oracle is PyTorch autograd over the forward definitions. It is pinned to
things other than itself: its forward against the C oracle (which the worked
example pins), its gradients against central finite differences of the
forward, the quadratic and recurrent forms' gradients against each other, and
the one-token closed form.
"""
import numpy as np
import pytest

import oracle
from oracle import backward as bwd


def _rand(rng, *shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("causal", [True, False])
def test_identity_map_matches_the_feature_oracle(causal):
    # The identity-map forward on features equals the numpy feature-map oracle,
    # itself pinned against the C oracle on elu + 1 features.
    from oracle import feature_maps as fm
    rng = np.random.default_rng(5)
    fq, fk, v = rng.random((2, 23, 4)), rng.random((2, 23, 4)), _rand(rng, 2, 23, 3)
    np.testing.assert_allclose(bwd.forward(fq, fk, v, causal, phi="identity"),
                               fm.attention_from_features(fq, fk, v, causal), rtol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_forward_matches_c_oracle(causal):
    rng = np.random.default_rng(0)
    q, k, v = _rand(rng, 2, 37, 5), _rand(rng, 2, 37, 5), _rand(rng, 2, 37, 3)
    ref = oracle.recurrent(q, k, v, causal)
    np.testing.assert_allclose(bwd.forward(q, k, v, causal, form="quadratic"), ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(bwd.forward(q, k, v, causal, form="recurrent"), ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal,phi", [(True, "elu1"), (False, "elu1"), (True, "identity"),
                                        (False, "identity")])
def test_gradients_match_central_differences(causal, phi):
    rng = np.random.default_rng(1)
    N, D, M = 6, 3, 2
    q, k, v, g = _rand(rng, N, D), _rand(rng, N, D), _rand(rng, N, M), _rand(rng, N, M)
    if phi == "identity":       # non-negative features keep the denominators away from 0
        q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
    dq, dk, dv = bwd.grads(q, k, v, g, causal, phi=phi)
    loss = lambda q_, k_, v_: float((bwd.forward(q_, k_, v_, causal, phi=phi) * g).sum())
    h = 1e-6
    for name, x, dx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [xp if n == name else a for n, a in (("q", q), ("k", k), ("v", v))]
            args_m = [xm if n == name else a for n, a in (("q", q), ("k", k), ("v", v))]
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(dx, fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_quadratic_and_recurrent_gradients_agree():
    rng = np.random.default_rng(2)
    q, k, v, g = _rand(rng, 2, 40, 4), _rand(rng, 2, 40, 4), _rand(rng, 2, 40, 3), _rand(rng, 2, 40, 3)
    a = bwd.grads(q, k, v, g, True, form="quadratic")
    b = bwd.grads(q, k, v, g, True, form="recurrent")
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-12)


def test_one_token_closed_form():
    # N = 1: o = v * w / (w + eps) with w = phi(q).phi(k), so dL/dv = g * w / (w + eps).
    rng = np.random.default_rng(3)
    q, k, v, g = _rand(rng, 1, 4), _rand(rng, 1, 4), _rand(rng, 1, 2), _rand(rng, 1, 2)
    eps = 0.25
    w = float((oracle.phi(q) @ oracle.phi(k).T)[0, 0])
    _, _, dv = bwd.grads(q, k, v, g, True, eps=eps)
    np.testing.assert_allclose(dv, g * w / (w + eps), rtol=1e-13)


def test_future_tokens_do_not_affect_earlier_gradients_of_v():
    # Causality: o_i depends on v_j only for j <= i, so a loss on row 0 alone
    # gives dv = 0 for every later token.
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 7, 3), _rand(rng, 7, 3), _rand(rng, 7, 2)
    g = np.zeros((7, 2))
    g[0] = rng.standard_normal(2)
    dq, dk, dv = bwd.grads(q, k, v, g, True)
    assert np.all(dv[1:] == 0) and np.all(dk[1:] == 0) and np.all(dq[1:] == 0)
