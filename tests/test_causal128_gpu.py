"""The bf16 causal path at Dk = Dv = 128 (run sums, seed scan, output pass).

Checked against the float64 oracle: continuation from a given state (the seed
scan adds the initial state where a range starts its head, the state warps
reset to it where a head starts inside a range), the identity feature map,
sampled rows of a large shape with many ranges per head, and the bounded-wait
failure path. The ragged and multi-head partitions and the final states are
covered with the 64-wide kernel in test_parity_gpu.py.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import feature_maps as fm
from workloads import make_features, make_qkv, to_f64

pytestmark = pytest.mark.gpu

D = 128
TOL = 2e-2
MAX_SPIN_WORD, HOLD_WORD = 4, 5   # uint32 index of max_spin and hold_item in the header


@pytest.fixture(scope="module")
def la():
    import linear_attention_elu_gb300 as m
    return m


def rowwise_rel(got, ref):
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return float((num / den).max())


def state_rel(S, Sr):
    # S sums bf16-rounded phi(k) v products in fp32: compare per head in max norm.
    return float((np.abs(S - Sr).max(axis=(-1, -2)) / np.abs(Sr).max(axis=(-1, -2))).max())


@pytest.mark.parametrize("B,H,N,n1", [
    (2, 3, 1500, 700),     # ragged halves
    (4, 64, 200, 100),     # one chunk per head: many heads start inside a range
    (1, 2, 5000, 2500),    # heads over many ranges: the seed scan carries S0
])
def test_second_half_from_first_half_state(la, B, H, N, n1):
    q, k, v = make_qkv(B, H, N, D, "bf16", seed=N + 10 * H + B + 128)
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
    assert rowwise_rel(to_f64(o2), ref[:, :, n1:]) <= TOL
    assert state_rel(to_f64(S2), Sr) <= 1e-2
    np.testing.assert_allclose(to_f64(z2), zr, rtol=5e-3)


def test_zero_initial_state_equals_plain_forward(la):
    B, H, N = 2, 4, 777
    q, k, v = (t.cuda() for t in make_qkv(B, H, N, D, "bf16", seed=9))
    S0 = torch.zeros(B, H, D, D, device="cuda")
    z0 = torch.zeros(B, H, D, device="cuda")
    o_a = la.la_causal_fwd(q, k, v)
    o_b = la.la_causal_fwd_state(q, k, v, S0, z0)
    torch.cuda.synchronize()
    # Same kernels, same partition, zero added: the same bits.
    assert torch.equal(o_a, o_b)


def test_identity_feature_map(la):
    B, H, N = 2, 3, 700
    fq, fk, v = make_features(B, H, N, D, "bf16", seed=77)
    dev = torch.device("cuda")
    S = torch.empty(B, H, D, D, device=dev)
    z = torch.empty(B, H, D, device=dev)
    o = la.la_causal_fwd(fq.to(dev), fk.to(dev), v.to(dev), S_out=S, z_out=z,
                         phi=la.LA_PHI_IDENTITY)
    torch.cuda.synchronize()
    ref, Sr, zr = fm.recurrent_from_features(to_f64(fq), to_f64(fk), to_f64(v), True,
                                             return_state=True)
    assert rowwise_rel(to_f64(o), ref) <= TOL
    assert state_rel(to_f64(S), Sr) <= 1e-2
    np.testing.assert_allclose(to_f64(z), zr, rtol=5e-3)


def test_large_shape_rows_sampled_against_quadratic(la):
    # The bidirectional workload's shape run causally: 8192 chunks over the
    # grid, about 54 per range, each head spread over several ranges.
    B, H, N = 16, 8, 8192
    q, k, v = make_qkv(B, H, N, D, "bf16", seed=5)
    dev = torch.device("cuda")
    o = la.la_causal_fwd(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    got = to_f64(o.cpu()).reshape(B * H, N, D)
    rng = np.random.default_rng(5)
    heads = rng.integers(0, B * H, 16)
    idx = np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 12)])
    qf, kf, vf = (to_f64(t).reshape(B * H, N, D) for t in (q, k, v))
    r = oracle.rows(qf, kf, vf, True, heads, idx)
    assert rowwise_rel(got[heads, idx], r) <= TOL


def test_withheld_load_times_out_and_context_survives(la):
    dev = torch.device("cuda")
    q, k, v = make_qkv(2, 2, 1000, D, "bf16", seed=3)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ws = la.workspace(la.LA_OP_CAUSAL, 2, 2, 1000, D, D, torch.bfloat16, dev)
    hdr = ws[:256].view(torch.int32)
    hdr[MAX_SPIN_WORD] = 2000  # 2 ms
    hdr[HOLD_WORD] = 1
    la.la_causal_fwd(qd, kd, vd, ws=ws)
    assert la.la_query_status(ws) == la.LA_ERR_TIMEOUT
    la.la_workspace_init(ws)
    o = la.la_causal_fwd(qd, kd, vd, ws=ws)
    assert la.la_query_status(ws) == 0
    ref = oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), True)
    assert rowwise_rel(to_f64(o), ref) <= TOL
