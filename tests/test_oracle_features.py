"""Pins of the feature-map oracle (oracle/feature_maps.py), CPU only.

Each form is tied to something other than itself: attention on given features
against the C oracle fed with elu+1 features (the C oracle is pinned by the
pages' worked example), the quadratic and recurrent forms against each other,
decode steps against the recurrence, a two-token case worked by hand, and the
positive random features against the Gaussian identity E[phi(x).phi(y)] =
exp(x.y), by Monte Carlo with a tolerance from the sample's own spread, and
against softmax attention on a small case.
"""
import numpy as np
import pytest

import oracle
from oracle import feature_maps as fm


@pytest.mark.parametrize("causal", [True, False])
def test_elu_features_match_the_c_oracle(causal):
    rng = np.random.default_rng(11)
    q, k = rng.standard_normal((2, 3, 37, 8)), rng.standard_normal((2, 3, 37, 8))
    v = rng.standard_normal((2, 3, 37, 5))
    ref = oracle.quadratic(q, k, v, causal)
    got = fm.attention_from_features(oracle.phi(q), oracle.phi(k), v, causal)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_quadratic_and_recurrent_forms_agree(causal):
    rng = np.random.default_rng(12)
    # Non-negative features of a width (r = 6) unlike the value width (M = 3).
    fq, fk = rng.random((2, 29, 6)), rng.random((2, 29, 6))
    v = rng.standard_normal((2, 29, 3))
    o, S, z = fm.recurrent_from_features(fq, fk, v, causal, return_state=True)
    np.testing.assert_allclose(o, fm.attention_from_features(fq, fk, v, causal), rtol=1e-12)
    np.testing.assert_allclose(S, np.swapaxes(fk, -1, -2) @ v, rtol=1e-12)
    np.testing.assert_allclose(z, fk.sum(axis=-2), rtol=1e-12)


def test_decode_steps_reproduce_the_causal_rows():
    rng = np.random.default_rng(13)
    fq, fk, v = rng.random((4, 19, 5)), rng.random((4, 19, 5)), rng.standard_normal((4, 19, 7))
    S, z = np.zeros((4, 5, 7)), np.zeros((4, 5))
    rows = []
    for i in range(19):
        o, S, z = fm.decode_from_features(fq[:, i], fk[:, i], v[:, i], S, z)
        rows.append(o)
    np.testing.assert_allclose(np.stack(rows, axis=1),
                               fm.attention_from_features(fq, fk, v, True), rtol=1e-12, atol=1e-14)


def test_two_tokens_by_hand():
    # r = 1: fq = (1, 2), fk = (3, 1), v = (1, 2), eps = 0.
    # Causal: o_0 = 1*3*1 / (1*3) = 1; o_1 = (2*3*1 + 2*1*2) / (2*3 + 2*1) = 10/8.
    # Non-causal: o_0 = (3*1 + 1*2) / (3 + 1) = 5/4; o_1 = (6 + 4) / (6 + 2) = 5/4.
    fq, fk, v = np.array([[1.0], [2.0]]), np.array([[3.0], [1.0]]), np.array([[1.0], [2.0]])
    np.testing.assert_allclose(fm.attention_from_features(fq, fk, v, True, eps=0.0)[:, 0],
                               [1.0, 1.25], rtol=1e-15)
    np.testing.assert_allclose(fm.attention_from_features(fq, fk, v, False, eps=0.0)[:, 0],
                               [1.25, 1.25], rtol=1e-15)


def test_random_features_estimate_the_exponential_kernel():
    rng = np.random.default_rng(14)
    D, r = 6, 200_000
    x, y = 0.3 * rng.standard_normal(D), 0.3 * rng.standard_normal(D)
    W = rng.standard_normal((r, D))
    fx, fy = fm.positive_random_features(x, W), fm.positive_random_features(y, W)
    terms = r * fx * fy                     # per-feature samples of exp(w.x - |x|^2/2) exp(w.y - |y|^2/2)
    est, se = terms.mean(), terms.std() / np.sqrt(r)
    assert abs(est - np.exp(x @ y)) <= 5 * se, (est, np.exp(x @ y), se)
    assert (fx > 0).all()


def test_random_features_closed_forms():
    rng = np.random.default_rng(15)
    x = rng.standard_normal((3, 4))
    # All-zero projections: every feature is exp(-|x|^2 / 2) / sqrt(r).
    f0 = fm.positive_random_features(x, np.zeros((9, 4)))
    np.testing.assert_allclose(f0, np.exp(-0.5 * (x * x).sum(-1))[:, None] / 3.0 * np.ones((1, 9)),
                               rtol=1e-14)
    # A shift scales every feature by exp(-shift).
    W = rng.standard_normal((5, 4))
    np.testing.assert_allclose(fm.positive_random_features(x, W, shift=1.5),
                               np.exp(-1.5) * fm.positive_random_features(x, W), rtol=1e-14)


def test_random_features_approach_softmax_attention():
    rng = np.random.default_rng(16)
    N, D, r = 8, 4, 400_000
    q, k = 0.4 * rng.standard_normal((N, D)), 0.4 * rng.standard_normal((N, D))
    v = rng.standard_normal((N, 3))
    W = rng.standard_normal((r, D))
    got = fm.attention_from_features(fm.positive_random_features(q, W),
                                     fm.positive_random_features(k, W), v, False, eps=0.0)
    s = np.exp(q @ k.T)
    ref = (s @ v) / s.sum(-1, keepdims=True)
    assert np.abs(got - ref).max() <= 0.02 * np.abs(ref).max()
