"""Pins the float64 oracle to things other than itself.

* The hand-traced n = 4, d = 2 example ("Why Replace Attention? The Softmax
  Bottleneck and the Path to Linear Time", sections 5.5, 6.5 and 7.3), stored
  in tests/golden/worked_example_n4_d2.json with its citations.
* Exact rational results computed with Python fractions on integer inputs
  (where phi(x) = x + 1 is exact), by brute force over all pairs.
* Closed forms of phi (exp values at powers of two, the product rule of exp).
* Invariants: constant phi gives a running mean of V; o_1 = v_1 under the
  causal mask ("Tracing the recurrence", step i = 1); outputs are convex
  combinations of the visible values (section 5.4, non-negative weights);
  S_n = S (end of section 7.3); permuting the (k, v) pairs leaves the
  non-causal output unchanged; linearity and shift-equivariance in V.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example_n4_d2.json")


@pytest.fixture(scope="module")
def ex():
    with open(GOLDEN) as f:
        return json.load(f)


def _frac_vec(o):
    return [Fraction(n, o["den"]) for n in o["num"]]


# ---------------------------------------------------------------- phi


def test_phi_worked_example(ex):
    np.testing.assert_array_equal(oracle.phi(ex["Q"]), np.array(ex["phi_Q"], float))
    np.testing.assert_array_equal(oracle.phi(ex["K"]), np.array(ex["phi_K"], float))


def test_phi_closed_forms():
    # Positive branch: x + 1, exact for these binary fractions.
    x = np.array([0.5, 1.0, 3.0, 1e-300, 2.0 ** 40])
    np.testing.assert_array_equal(oracle.phi(x), x + 1.0)
    # phi(0) = 1 from either branch (elu(0) = 0).
    assert oracle.phi([0.0])[0] == 1.0
    assert oracle.phi([-0.0])[0] == 1.0
    # Negative branch is exp(x), not exp(x) - 1 or 1 - exp(-x): exact halvings.
    ln2 = math.log(2.0)
    for n in range(1, 8):
        assert abs(oracle.phi([-n * ln2])[0] - 2.0 ** (-n)) <= 4e-16 * 2.0 ** (-n) * n
    # Product rule exp(a)exp(b) = exp(a+b) on the negative branch.
    a, b = -0.375, -1.25
    pa, pb, pab = oracle.phi([a, b, a + b])
    assert abs(pa * pb - pab) <= 1e-15
    # Strictly positive, continuous at 0, monotone.
    xs = np.linspace(-30, 30, 10001)
    ys = oracle.phi(xs)
    assert np.all(ys > 0) and np.all(np.diff(ys) > 0)
    assert abs(oracle.phi([-1e-12])[0] - 1.0) < 2e-12


# ------------------------------------------------------ worked example


@pytest.mark.parametrize("form", ["quadratic", "recurrent"])
def test_worked_example_noncausal(ex, form):
    Q, K, V = (np.array(ex[n], float) for n in "QKV")
    fn = getattr(oracle, form)
    o = fn(Q, K, V, causal=False, eps=0.0)
    # Printed o_1 = (20, 11) / 20 = (1.00, 0.55).
    np.testing.assert_allclose(o[0], [float(x) for x in _frac_vec(ex["noncausal"]["o1"])],
                               rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[0], ex["noncausal"]["o1"]["printed"], rtol=0, atol=5e-3)
    # Rows 2..4 are not printed; they follow exactly from the printed S and z
    # and the printed phi(Q): o_i = phi(q_i)^T S / phi(q_i)^T z.
    S = [[Fraction(x) for x in r] for r in ex["noncausal"]["S"]]
    z = [Fraction(x) for x in ex["noncausal"]["z"]]
    for i, fq in enumerate(ex["phi_Q"]):
        den = sum(Fraction(fq[c]) * z[c] for c in range(2))
        num = [sum(Fraction(fq[c]) * S[c][m] for c in range(2)) for m in range(2)]
        np.testing.assert_allclose(o[i], [float(n / den) for n in num], rtol=1e-15, atol=0)


def test_worked_example_state(ex):
    Q, K, V = (np.array(ex[n], float) for n in "QKV")
    _, S, z = oracle.recurrent(Q, K, V, causal=False, eps=0.0, return_state=True)
    np.testing.assert_array_equal(S, np.array(ex["noncausal"]["S"], float))
    np.testing.assert_array_equal(z, np.array(ex["noncausal"]["z"], float))
    # Each prefix of the sequence reproduces the printed S_i, z_i.
    for step in ex["causal"]:
        i = step["i"]
        _, Si, zi = oracle.recurrent(Q[:i], K[:i], V[:i], causal=True, eps=0.0,
                                     return_state=True)
        np.testing.assert_array_equal(Si, np.array(step["S"], float))
        np.testing.assert_array_equal(zi, np.array(step["z"], float))
    # S_4 equals the non-causal S (the trace's closing remark).
    np.testing.assert_array_equal(np.array(ex["causal"][-1]["S"]), np.array(ex["noncausal"]["S"]))


def test_worked_example_similarity_row1(ex):
    # Row 1 of the printed similarity matrix, normalised, gives the printed weights;
    # checked through the oracle: o_1 with V = identity-like probes picks the weights.
    Q, K = (np.array(ex[n], float) for n in "QK")
    probe = np.eye(4)  # v_j = e_j, so o_1 = normalised similarity row 1
    o = oracle.quadratic(Q, K, probe, causal=False, eps=0.0)
    sim = np.array(ex["similarity"], float)
    np.testing.assert_allclose(o, sim / sim.sum(1, keepdims=True), rtol=1e-15, atol=0)
    np.testing.assert_allclose(o[0], ex["noncausal"]["row1_weights_printed"], atol=1e-15)
    oc = oracle.quadratic(Q, K, probe, causal=True, eps=0.0)
    masked = np.tril(sim)
    np.testing.assert_allclose(oc, masked / masked.sum(1, keepdims=True), rtol=1e-15, atol=0)


@pytest.mark.parametrize("form", ["quadratic", "recurrent", "decode"])
def test_worked_example_causal_trace(ex, form):
    Q, K, V = (np.array(ex[n], float) for n in "QKV")
    if form == "decode":
        S = np.zeros((2, 2))
        z = np.zeros(2)
        o = np.stack([oracle.decode_step(Q[i], K[i], V[i], S, z, eps=0.0) for i in range(4)])
        np.testing.assert_array_equal(S, np.array(ex["causal"][-1]["S"], float))
        np.testing.assert_array_equal(z, np.array(ex["causal"][-1]["z"], float))
    else:
        o = getattr(oracle, form)(Q, K, V, causal=True, eps=0.0)
    for step in ex["causal"]:
        i = step["i"] - 1
        np.testing.assert_allclose(o[i], [float(x) for x in _frac_vec(step["o"])],
                                   rtol=1e-15, atol=0)
        np.testing.assert_allclose(o[i], step["o"]["printed"], rtol=0, atol=5e-4)


def test_worked_example_eps_shift(ex):
    # eps = 1e-6 is added once to the scalar denominator: o = num / (den + eps).
    Q, K, V = (np.array(ex[n], float) for n in "QKV")
    o = oracle.recurrent(Q, K, V, causal=True, eps=1e-6)
    for step in ex["causal"]:
        i = step["i"] - 1
        num, den = step["o"]["num"], step["o"]["den"]
        np.testing.assert_allclose(o[i], [n / (den + 1e-6) for n in num], rtol=1e-15, atol=0)


# ----------------------------------------------------- brute force (exact)


def _exact(q, k, v, causal):
    """All pairs in exact rationals; integer inputs >= 0 make phi(x) = x + 1 exact."""
    n = len(q)
    out = []
    for i in range(n):
        fq = [Fraction(int(x) + 1) for x in q[i]]
        num = [Fraction(0)] * len(v[0])
        den = Fraction(0)
        for j in range(i + 1 if causal else n):
            fk = [Fraction(int(x) + 1) for x in k[j]]
            w = sum(a * b for a, b in zip(fq, fk))
            den += w
            num = [a + w * int(b) for a, b in zip(num, v[j])]
        out.append([a / den for a in num])
    return out


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [True, False])
def test_brute_force_exact(seed, causal):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 9))
    d = int(rng.integers(1, 5))
    m = int(rng.integers(1, 5))
    q = rng.integers(0, 5, (n, d))
    k = rng.integers(0, 5, (n, d))
    v = rng.integers(-6, 7, (n, m))
    ref = np.array([[float(x) for x in r] for r in _exact(q.tolist(), k.tolist(), v.tolist(),
                                                          causal)])
    for fn in (oracle.quadratic, oracle.recurrent):
        o = fn(q, k, v, causal=causal, eps=0.0)
        np.testing.assert_allclose(o, ref, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------- invariants


def _rand(seed, BH=3, N=97, D=8, M=5, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((BH, N, D)) * scale, rng.standard_normal((BH, N, D)) * scale,
            rng.standard_normal((BH, N, M)))


@pytest.mark.parametrize("causal", [True, False])
def test_quadratic_equals_recurrent(causal):
    q, k, v = _rand(1)
    a = oracle.quadratic(q, k, v, causal, eps=1e-6)
    b = oracle.recurrent(q, k, v, causal, eps=1e-6)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_causal_last_row_is_noncausal():
    q, k, v = _rand(2)
    c = oracle.recurrent(q, k, v, True)
    nc = oracle.quadratic(q, k, v, False)
    np.testing.assert_allclose(c[:, -1], nc[:, -1], rtol=1e-12, atol=1e-13)
    # Every non-causal row reads the same final state: row i of the non-causal
    # output equals the causal output of a sequence whose last query is q_i.
    for i in (0, 40, 96):
        q2 = q.copy()
        q2[:, -1] = q[:, i]
        np.testing.assert_allclose(oracle.recurrent(q2, k, v, True)[:, -1], nc[:, i],
                                   rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("form", ["quadratic", "recurrent"])
def test_constant_phi_running_mean(form):
    rng = np.random.default_rng(3)
    N, D, M = 50, 6, 4
    v = rng.standard_normal((N, M))
    zeros = np.zeros((N, D))  # phi(0) = 1 everywhere: all weights equal
    fn = getattr(oracle, form)
    oc = fn(zeros, zeros, v, causal=True, eps=0.0)
    running = np.cumsum(v, axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(oc, running, rtol=1e-13, atol=1e-14)
    onc = fn(zeros, zeros, v, causal=False, eps=0.0)
    np.testing.assert_allclose(onc, np.broadcast_to(v.mean(0), (N, M)), rtol=1e-13, atol=1e-14)
    # With eps the denominator is i * D + eps.
    oe = fn(zeros, zeros, v, causal=True, eps=1e-3)
    i = np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(oe, np.cumsum(v, 0) * D / (i * D + 1e-3), rtol=1e-13)


def test_first_row_is_v1_and_convex_hull():
    q, k, v = _rand(4, scale=2.0)
    o = oracle.recurrent(q, k, v, True, eps=0.0)
    np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=1e-14)
    lo = np.minimum.accumulate(v, axis=1)
    hi = np.maximum.accumulate(v, axis=1)
    assert np.all(o >= lo - 1e-12) and np.all(o <= hi + 1e-12)


def test_noncausal_permutation_invariance():
    q, k, v = _rand(5)
    perm = np.random.default_rng(0).permutation(q.shape[1])
    a = oracle.recurrent(q, k, v, False)
    b = oracle.recurrent(q, k[:, perm], v[:, perm], False)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    # Permuting queries permutes output rows.
    c = oracle.quadratic(q[:, perm], k, v, False)
    np.testing.assert_allclose(c, a[:, perm], rtol=1e-12, atol=1e-13)


def test_linear_and_shift_in_v():
    q, k, v = _rand(6)
    o = oracle.recurrent(q, k, v, True, eps=0.0)
    np.testing.assert_allclose(oracle.recurrent(q, k, 3.0 * v, True, eps=0.0), 3.0 * o,
                               rtol=1e-12, atol=1e-13)
    # Weights sum to one (eps = 0): adding c to every value shifts every output by c.
    np.testing.assert_allclose(oracle.recurrent(q, k, v + 2.5, True, eps=0.0), o + 2.5,
                               rtol=1e-12, atol=1e-12)


def test_rows_match_full():
    q, k, v = _rand(7, BH=4, N=70)
    for causal in (True, False):
        full = oracle.quadratic(q, k, v, causal)
        heads = [0, 1, 3, 3, 2]
        idx = [0, 69, 5, 33, 64]
        np.testing.assert_allclose(oracle.rows(q, k, v, causal, heads, idx),
                                   full[heads, idx], rtol=1e-13, atol=1e-14)


def test_decode_matches_causal():
    q, k, v = _rand(8, BH=5, N=20)
    S = np.zeros((5, 8, 5))
    z = np.zeros((5, 8))
    o = np.stack([oracle.decode_step(q[:, i], k[:, i], v[:, i], S, z) for i in range(20)], 1)
    oc, Sc, zc = oracle.recurrent(q, k, v, True, return_state=True)
    np.testing.assert_allclose(o, oc, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S, Sc, rtol=1e-13)
    np.testing.assert_allclose(z, zc, rtol=1e-13)


def test_denominator_underflow_uses_eps():
    # A very negative query gives phi(q) = exp(q) -> 0 in double: den -> 0 and the
    # output is num / eps, i.e. 0 when num underflows too.
    q, k, v = _rand(9, BH=1, N=10)
    q[0, 3] = -1000.0
    o = oracle.recurrent(q, k, v, True, eps=1e-6)
    assert np.all(o[0, 3] == 0.0)
    assert np.all(np.isfinite(o))


def test_threads_do_not_change_results():
    q, k, v = _rand(10, BH=7, N=33)
    a = oracle.recurrent(q, k, v, True, nthreads=1)
    b = oracle.recurrent(q, k, v, True, nthreads=4)
    np.testing.assert_array_equal(a, b)
