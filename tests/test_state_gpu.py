"""la_causal_fwd_state: a causal forward that continues from a given state.

A sequence cut in two, the second part started from the first part's final
state (S_out, z_out), must give the rows and the final state of the whole
sequence: the recurrence carries nothing but (S, z) forward ("Transformers Are
RNNs: Linear Attention", "Turn Causal Attention into a Recurrence"). The
reference is the float64 oracle run once over the whole sequence, so the
initial-state handling is checked against the definition, not against itself.
Cases cover both GPU paths and the places where the tensor-core kernel injects
the initial state: a range that starts a head (its seed), a step-1 sum whose
run starts a head (what later ranges add up), and a head that starts inside a
range (the state role's reset).
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_qkv, to_f64

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module")
def la():
    import linear_attention_elu_gb300 as m
    return m


def rowwise_rel(got, ref):
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return float((num / den).max())


@pytest.mark.parametrize("B,H,N,n1,D,dt", [
    (2, 3, 1500, 700, 64, "bf16"),     # tensor cores; ragged halves
    (4, 64, 200, 100, 64, "bf16"),     # one chunk per head: many heads start inside a range
    (1, 2, 5000, 2500, 64, "bf16"),    # heads spread over many ranges: the look-back adds S0
    (2, 2, 333, 100, 64, "f32"),       # fp32 SIMT path
    (1, 3, 260, 130, 32, "f32"),       # fp32 SIMT path, D = 32
])
def test_second_half_from_first_half_state(la, B, H, N, n1, D, dt):
    q, k, v = make_qkv(B, H, N, D, dt, seed=N + 10 * H + B)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    S1 = torch.empty(B, H, D, D, device=dev)
    z1 = torch.empty(B, H, D, device=dev)
    la.la_causal_fwd(qd[:, :, :n1].contiguous(), kd[:, :, :n1].contiguous(),
                     vd[:, :, :n1].contiguous(), S_out=S1, z_out=z1)
    S2 = torch.full((B, H, D, D), float("nan"), device=dev)
    z2 = torch.full((B, H, D), float("nan"), device=dev)
    o2 = la.la_causal_fwd_state(qd[:, :, n1:].contiguous(), kd[:, :, n1:].contiguous(),
                                vd[:, :, n1:].contiguous(), S1, z1, S_out=S2, z_out=z2)
    torch.cuda.synchronize()
    ref, Sr, zr = oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), True, return_state=True)
    assert rowwise_rel(to_f64(o2), ref[:, :, n1:]) <= TOL[dt]
    if dt == "f32":
        np.testing.assert_allclose(to_f64(S2), Sr, rtol=1e-4, atol=1e-3)
        np.testing.assert_allclose(to_f64(z2), zr, rtol=1e-5, atol=1e-4)
    else:
        rel = np.abs(to_f64(S2) - Sr).max(axis=(-1, -2)) / np.abs(Sr).max(axis=(-1, -2))
        assert rel.max() <= 1e-2, rel.max()
        np.testing.assert_allclose(to_f64(z2), zr, rtol=5e-3)


@pytest.mark.parametrize("D,dt", [(64, "bf16"), (64, "f32")])
def test_zero_initial_state_equals_plain_forward(la, D, dt):
    B, H, N = 2, 4, 777
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, dt, seed=9))
    S0 = torch.zeros(B, H, D, D, device="cuda")
    z0 = torch.zeros(B, H, D, device="cuda")
    S_a, S_b = torch.empty_like(S0), torch.empty_like(S0)
    z_a, z_b = torch.empty_like(z0), torch.empty_like(z0)
    ws = la.workspace(la.LA_OP_CAUSAL, B, H, N, D, D, q.dtype, q.device)
    o_a = la.la_causal_fwd(q, k, v, S_out=S_a, z_out=z_a, ws=ws)
    o_b = la.la_causal_fwd_state(q, k, v, S0, z0, S_out=S_b, z_out=z_b, ws=ws)
    torch.cuda.synchronize()
    # Adding exact zeros changes no bit; the two calls run the same partition.
    assert torch.equal(o_a, o_b) and torch.equal(S_a, S_b) and torch.equal(z_a, z_b)


def test_empty_sequence_passes_the_state_through(la):
    B, H, D = 1, 3, 64
    q = torch.empty(B, H, 0, D, device="cuda", dtype=torch.bfloat16)
    S0 = torch.randn(B, H, D, D, device="cuda")
    z0 = torch.rand(B, H, D, device="cuda")
    S = torch.full_like(S0, float("nan"))
    z = torch.full_like(z0, float("nan"))
    la.la_causal_fwd_state(q, q, q, S0, z0, S_out=S, z_out=z)
    torch.cuda.synchronize()
    assert torch.equal(S, S0) and torch.equal(z, z0)


def test_rejects_half_a_state_and_overlap(la):
    B, H, N, D = 1, 2, 128, 64
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "bf16", seed=4))
    S0 = torch.zeros(B, H, D, D, device="cuda")
    z0 = torch.zeros(B, H, D, device="cuda")
    with pytest.raises(la.LinAttnError) as e:
        la._check(la._lib.la_causal_fwd_state(
            la._ptr(q), la._ptr(k), la._ptr(v), la._ptr(torch.empty_like(v)), B, H, N, D, D,
            la.LA_BF16, 1e-6, la._ptr(S0), None, None, None, None, 0, None), "state")
    assert e.value.status == 1
    with pytest.raises(la.LinAttnError) as e:
        la.la_causal_fwd_state(q, k, v, S0, z0, S_out=S0)     # in place: refused
    assert e.value.status == 1
