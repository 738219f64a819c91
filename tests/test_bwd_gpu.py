"""la_causal_bwd against the float64 gradient oracle (oracle/backward.py).

Gate, per gradient tensor and head: max |gpu - oracle| / max |oracle| over the
head's [N, D] gradient, with 1e-4 for float32 inputs and 2e-2 for bfloat16
inputs (fp32 arithmetic either way; bf16 inputs give bf16 gradients). Unlike
the forward's outputs, single gradient rows can vanish by cancellation: the
first token's dphi(q_0) is phi(k_0) (g_0 . (v_0 - o_0)) / den_0 with o_0 = v_0
up to eps, so a row-wise relative measure would divide rounding noise by
nearly zero. The oracle sees the exact values the GPU sees, upcast to float64.
"""
import numpy as np
import pytest
import torch

from oracle import backward as bwd
from workloads import make_qkv, to_f64

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module")
def la():
    import linear_attention_elu_gb300 as m
    return m


def headwise_rel(got, ref):
    num = np.abs(got - ref).max(axis=(-1, -2))
    den = np.maximum(np.abs(ref).max(axis=(-1, -2)), 1e-30)
    return float((num / den).max())


@pytest.mark.parametrize("B,H,N,D,M,dt", [
    (1, 1, 5, 3, 2, "f32"),          # shorter than a chunk, odd widths
    (2, 2, 200, 64, 64, "f32"),      # several chunks, ragged tail
    (1, 3, 130, 32, 48, "f32"),      # Dk != Dv
    (2, 2, 333, 64, 64, "bf16"),     # bf16 inputs and gradients
])
def test_gradients_match_oracle(la, B, H, N, D, M, dt):
    q, k, v = make_qkv(B, H, N, D, dt, seed=N + D, Dv=M)
    g = make_qkv(B, H, N, M, dt, seed=N + D + 1)[2]
    dev = torch.device("cuda")
    dq, dk, dv = la.la_causal_bwd(q.to(dev), k.to(dev), v.to(dev), g.to(dev))
    torch.cuda.synchronize()
    rq, rk, rv = bwd.grads(to_f64(q), to_f64(k), to_f64(v), to_f64(g), True)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        err = headwise_rel(to_f64(got), ref)
        assert err <= TOL[dt], (name, err)


def test_zero_upstream_gradient_gives_zero(la):
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 150, 64, "f32", seed=3))
    dq, dk, dv = la.la_causal_bwd(q, k, v, torch.zeros_like(v))
    torch.cuda.synchronize()
    assert float(dq.abs().max()) == 0 and float(dk.abs().max()) == 0 and float(dv.abs().max()) == 0


def test_loss_on_first_row_only_touches_first_token(la):
    # Causality: a loss on row 0 alone reaches token 0 only.
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 100, 64, "f32", seed=4))
    g = torch.zeros_like(v)
    g[0, 0, 0] = torch.randn(64, device="cuda")
    dq, dk, dv = la.la_causal_bwd(q, k, v, g)
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert float(t[0, 0, 1:].abs().max()) == 0 and float(t[0, 0, 0].abs().max()) > 0


def test_wide_heads_are_refused(la):
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 64, 128, "bf16", seed=5))
    with pytest.raises(la.LinAttnError) as e:
        la.la_causal_bwd(q, k, v, torch.zeros_like(v))
    assert e.value.status == 2  # LA_ERR_UNSUPPORTED
