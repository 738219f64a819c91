"""Edge cases of the method on the bf16 paths (the tensor-core kernels take
bf16 causal at Dk = Dv = 64 and bf16 non-causal at Dk = Dv = 128), against the
float64 oracle at the bf16 gate.

phi(x) = elu(x) + 1 is e^x on the negative half ("Why Replace Attention?",
section 5.3), so inputs drawn in the negative range exercise the exponential
branch where a reduced-precision exponent loses the most: q and k centred at
-6, individual features between -30 and -8, whole query rows at -30 (the
denominator falls to the size of eps; "Transformers Are RNNs: Linear
Attention", "Where It Breaks"), rows at -200 (phi underflows to zero), and
Q = K = 0 (constant phi: every output is the running mean of v, the weighted
average reading of "Why Replace Attention?", section 5.4).

Error measure as in the other parity tests: per output row
max_d |gpu - oracle| / max_d |oracle|, gate 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_qkv, to_f64

pytestmark = pytest.mark.gpu

TOL = 2e-2
# (operation, D): the tensor-core shapes first, then the other bf16 widths.
PATHS = [("causal", 64), ("noncausal", 128), ("causal", 128), ("noncausal", 64)]


@pytest.fixture(scope="module")
def la():
    import linear_attention_elu_gb300 as m
    return m


def rowwise_rel(got, ref):
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-300)
    return num / den


def run(la, op, q, k, v, eps=1e-6):
    dev = torch.device("cuda")
    fn = la.la_causal_fwd if op == "causal" else la.la_noncausal_fwd
    o = fn(q.to(dev), k.to(dev), v.to(dev), eps=eps)
    torch.cuda.synchronize()
    return to_f64(o)


def ref(op, q, k, v, eps=1e-6):
    return oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), causal=(op == "causal"), eps=eps)


def inputs(case, D, N=1000, seed=0):
    """bf16 q, k, v for one edge case (float32 draws of make_qkv, then shaped)."""
    q, k, v = make_qkv(1, 2, N, D, "f32", seed=seed)
    g = torch.Generator().manual_seed(seed + 101)
    if case == "shifted":                 # q, k ~ N(-6, 1)
        q, k = q - 6.0, k - 6.0
    elif case == "deep_features":         # a quarter of the features in [-30, -8)
        for t in (q, k):
            pick = torch.rand(t.shape, generator=g) < 0.25
            t[pick] = -8.0 - 22.0 * torch.rand(int(pick.sum()), generator=g)
    elif case == "rows_at_minus30":       # whole query rows at -30: den ~ eps
        q[:, :, ::97] = -30.0
    elif case == "constant_phi":          # phi(q) = phi(k) = 1
        q.zero_()
        k.zero_()
    return q.bfloat16(), k.bfloat16(), v.bfloat16()


@pytest.mark.parametrize("op,D", PATHS)
@pytest.mark.parametrize("case", ["shifted", "deep_features", "rows_at_minus30", "constant_phi"])
def test_negative_range_and_constant_phi(la, op, D, case):
    q, k, v = inputs(case, D, seed=D + len(case))
    got = run(la, op, q, k, v)
    r = ref(op, q, k, v)
    err = rowwise_rel(got, r)
    assert np.all(np.isfinite(got))
    assert err.max() <= TOL, (case, float(err.max()), np.unravel_index(err.argmax(), err.shape))


@pytest.mark.parametrize("op,D", PATHS)
def test_rows_at_minus30_reach_eps_regime(la, op, D):
    # The oracle's denominators on those rows are far below eps, so eps decides
    # the outputs: a kernel that dropped or misplaced eps fails this.
    q, k, v = inputs("rows_at_minus30", D, seed=7)
    got = run(la, op, q, k, v)
    r_eps = ref(op, q, k, v)
    r_big = ref(op, q, k, v, eps=1e-3)
    rows = slice(None, None, 97)
    assert rowwise_rel(got[:, :, rows], r_eps[:, :, rows]).max() <= TOL
    assert rowwise_rel(r_big[:, :, rows], r_eps[:, :, rows]).min() > 0.5


@pytest.mark.parametrize("op,D", PATHS)
def test_constant_phi_is_running_mean(la, op, D):
    q, k, v = inputs("constant_phi", D, seed=3)
    got = run(la, op, q, k, v, eps=0.0)
    vf = to_f64(v)
    if op == "causal":
        mean = np.cumsum(vf, axis=2) / np.arange(1, vf.shape[2] + 1)[:, None]
    else:
        mean = np.broadcast_to(vf.mean(axis=2, keepdims=True), vf.shape)
    assert rowwise_rel(got, mean).max() <= TOL


@pytest.mark.parametrize("op,D", PATHS)
def test_phi_underflow_rows(la, op, D):
    # exp(-200) is 0 in every GPU precision but ~1e-87 in float64: both rows are
    # zero to within 1e-70, and the other rows are unaffected.
    q, k, v = inputs("none", D, N=300, seed=5)
    q = q.float()
    q[0, 1, 7] = -200.0
    q = q.bfloat16()
    got = run(la, op, q, k, v)
    r = ref(op, q, k, v)
    assert np.abs(got[0, 1, 7]).max() <= 1e-70 and np.abs(r[0, 1, 7]).max() <= 1e-70
    keep = np.ones(300, bool)
    keep[7] = False
    assert rowwise_rel(got[0, 1, keep], r[0, 1, keep]).max() <= TOL
    assert rowwise_rel(got[0, 0], r[0, 0]).max() <= TOL
