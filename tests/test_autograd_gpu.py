"""linear_attention_elu_gb300.autograd: the forward and backward entry points as
one differentiable function. Its gradients equal the backward entry point's
bit for bit (it only marshals arguments) and match the float64 gradient
oracle under the backward's gates."""
import numpy as np
import pytest
import torch

from oracle import backward as bwd
from workloads import make_qkv, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    import linear_attention_elu_gb300 as m
    return m


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dt,tol", [("f32", 1e-4), ("bf16", 2e-2)])
def test_autograd_matches_entry_points_and_oracle(la, causal, dt, tol):
    from linear_attention_elu_gb300.autograd import linear_attention
    q, k, v = make_qkv(2, 2, 200, 64, dt, seed=51)
    g = make_qkv(2, 2, 200, 64, dt, seed=52)[2]
    dev = torch.device("cuda")
    qd, kd, vd = (t.to(dev).requires_grad_(True) for t in (q, k, v))
    o = linear_attention(qd, kd, vd, causal=causal)
    o.backward(g.to(dev))
    fn = la.la_causal_bwd if causal else la.la_noncausal_bwd
    dq, dk, dv = fn(q.to(dev), k.to(dev), v.to(dev), g.to(dev))
    torch.cuda.synchronize()
    for got, want in ((qd.grad, dq), (kd.grad, dk), (vd.grad, dv)):
        assert torch.equal(got, want)
    refs = bwd.grads(to_f64(q), to_f64(k), to_f64(v), to_f64(g), causal)
    for got, ref in zip((qd.grad, kd.grad, vd.grad), refs):
        num = np.abs(to_f64(got) - ref).max(axis=(-1, -2))
        den = np.maximum(np.abs(ref).max(axis=(-1, -2)), 1e-30)
        assert float((num / den).max()) <= tol
