"""Other feature maps through the same kernels: LA_PHI_IDENTITY on every path,
and la_positive_random_features, against the float64 feature-map oracle
(oracle/feature_maps.py) and the float64 gradient oracle (oracle/backward.py).

Gates as elsewhere: row-wise relative error 1e-4 for float32 inputs, 2e-2 for
bfloat16 (features rounded to bf16 once); gradients head-wise relative.
Inputs are seeded non-negative features (uniform on [0, 1)) of widths that
differ from the value width where the path allows it (r != Dv).
"""
import numpy as np
import pytest
import torch

from oracle import backward as bwd
from oracle import feature_maps as fm
from workloads import make_features, make_qkv, to_f64

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


def headwise_rel(got, ref):
    num = np.abs(got - ref).max(axis=(-1, -2))
    den = np.maximum(np.abs(ref).max(axis=(-1, -2)), 1e-30)
    return float((num / den).max())


@pytest.mark.parametrize("B,H,N,C,M,dt", [
    (2, 3, 700, 64, 64, "bf16"),    # tensor-core causal path
    (1, 2, 200, 48, 32, "f32"),     # fp32 SIMT, r != Dv, ragged tail
    (2, 2, 333, 100, 64, "bf16"),   # SIMT general path (r > 64)
])
def test_causal_identity_map(la, B, H, N, C, M, dt):
    fq, fk, v = make_features(B, H, N, C, dt, seed=N + C, Dv=M)
    dev = torch.device("cuda")
    S = torch.empty(B, H, C, M, device=dev)
    z = torch.empty(B, H, C, device=dev)
    o = la.la_causal_fwd(fq.to(dev), fk.to(dev), v.to(dev), S_out=S, z_out=z,
                         phi=la.LA_PHI_IDENTITY)
    torch.cuda.synchronize()
    ref, Sr, zr = fm.recurrent_from_features(to_f64(fq), to_f64(fk), to_f64(v), True,
                                             return_state=True)
    assert rowwise_rel(to_f64(o), ref) <= TOL[dt]
    rel = np.abs(to_f64(S) - Sr).max(axis=(-1, -2)) / np.abs(Sr).max(axis=(-1, -2))
    assert rel.max() <= (1e-5 if dt == "f32" else 1e-2)
    np.testing.assert_allclose(to_f64(z), zr, rtol=1e-5 if dt == "f32" else 5e-3)


@pytest.mark.parametrize("B,H,N,C,M,dt", [
    (2, 2, 1000, 128, 128, "bf16"),  # tensor-core non-causal path, D = 128
    (2, 2, 1000, 64, 64, "bf16"),    # tensor-core non-causal path, D = 64
    (1, 3, 300, 64, 48, "f32"),      # fp32 SIMT tiled
    (1, 2, 150, 96, 64, "bf16"),     # SIMT general path
])
def test_noncausal_identity_map(la, B, H, N, C, M, dt):
    fq, fk, v = make_features(B, H, N, C, dt, seed=N + C + 1, Dv=M)
    dev = torch.device("cuda")
    o = la.la_noncausal_fwd(fq.to(dev), fk.to(dev), v.to(dev), phi=la.LA_PHI_IDENTITY)
    torch.cuda.synchronize()
    ref = fm.attention_from_features(to_f64(fq), to_f64(fk), to_f64(v), False)
    assert rowwise_rel(to_f64(o), ref) <= TOL[dt]


def test_causal_identity_map_continues_from_a_state(la):
    B, H, N, n1, C = 2, 2, 900, 400, 64
    fq, fk, v = make_features(B, H, N, C, "bf16", seed=21)
    dev = torch.device("cuda")
    q, k, vv = fq.to(dev), fk.to(dev), v.to(dev)
    S1 = torch.empty(B, H, C, C, device=dev)
    z1 = torch.empty(B, H, C, device=dev)
    la.la_causal_fwd(q[:, :, :n1].contiguous(), k[:, :, :n1].contiguous(),
                     vv[:, :, :n1].contiguous(), S_out=S1, z_out=z1, phi=la.LA_PHI_IDENTITY)
    o2 = la.la_causal_fwd_state(q[:, :, n1:].contiguous(), k[:, :, n1:].contiguous(),
                                vv[:, :, n1:].contiguous(), S1, z1, phi=la.LA_PHI_IDENTITY)
    torch.cuda.synchronize()
    ref = fm.attention_from_features(to_f64(fq), to_f64(fk), to_f64(v), True)
    assert rowwise_rel(to_f64(o2), ref[:, :, n1:]) <= TOL["bf16"]


@pytest.mark.parametrize("B,H,C,M,dt", [(16, 8, 64, 64, "bf16"), (3, 5, 48, 40, "f32")])
def test_decode_identity_map(la, B, H, C, M, dt):
    steps = 12
    fq, fk, v = make_features(B, H, steps, C, dt, seed=C + M, Dv=M)
    dev = torch.device("cuda")
    S = torch.zeros(B, H, C, M, device=dev)
    z = torch.zeros(B, H, C, device=dev)
    outs = []
    for t in range(steps):
        outs.append(la.la_decode_step(fq[:, :, t].contiguous().to(dev), fk[:, :, t].contiguous().to(dev),
                                      v[:, :, t].contiguous().to(dev), S, z,
                                      phi=la.LA_PHI_IDENTITY))
    torch.cuda.synchronize()
    got = np.stack([to_f64(o) for o in outs], axis=2)
    ref = fm.attention_from_features(to_f64(fq), to_f64(fk), to_f64(v), True)
    assert rowwise_rel(got, ref) <= TOL[dt]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_backward_identity_map(la, causal, dt):
    B, H, N, C = 2, 2, 200, 64
    fq, fk, v = make_features(B, H, N, C, dt, seed=31 + causal)
    g = make_qkv(B, H, N, C, dt, seed=33)[2]
    dev = torch.device("cuda")
    fn = la.la_causal_bwd if causal else la.la_noncausal_bwd
    dq, dk, dv = fn(fq.to(dev), fk.to(dev), v.to(dev), g.to(dev), phi=la.LA_PHI_IDENTITY)
    torch.cuda.synchronize()
    rq, rk, rv = bwd.grads(to_f64(fq), to_f64(fk), to_f64(v), to_f64(g), causal, phi="identity")
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert headwise_rel(to_f64(got), ref) <= TOL[dt], name


@pytest.mark.parametrize("rows,D,R,dt", [
    (1000, 64, 64, "bf16"),         # tensor-core path, ragged last tile
    (100_000, 64, 64, "bf16"),      # tensor-core path, several tiles per CTA
    (5, 64, 64, "bf16"),            # tensor-core path, one partial tile
    (1000, 64, 64, "f32"),
    (777, 64, 96, "bf16"),          # R not a multiple of 64
    (130, 128, 64, "f32"),          # the wide-row tile
    (5, 3, 7, "f32"),               # odd widths, one partial block
])
def test_positive_random_features(la, rows, D, R, dt):
    x = make_qkv(1, 1, rows, D, dt, seed=rows + D)[0][0, 0] * 0.5
    W = make_qkv(1, 1, R, D, dt, seed=R + 7)[1][0, 0]
    got = la.la_positive_random_features(x.cuda(), W.cuda(), shift=0.25)
    torch.cuda.synchronize()
    ref = fm.positive_random_features(to_f64(x), to_f64(W), shift=0.25)
    rel = np.abs(to_f64(got) - ref) / ref
    assert rel.max() <= (2e-5 if dt == "f32" else 8e-3), rel.max()


def test_random_features_then_attention(la):
    # The chain a caller runs: features from (x, W), then the identity-map causal
    # forward on the tensor-core path; the oracle computes its own features.
    B, H, N, D, R = 2, 2, 500, 64, 64
    q, k, v = make_qkv(B, H, N, D, "bf16", seed=41)
    q, k = q * 0.4, k * 0.4
    W = make_qkv(1, 1, R, D, "bf16", seed=42)[0][0, 0]
    dev = torch.device("cuda")
    fq = la.la_positive_random_features(q.to(dev), W.to(dev))
    fk = la.la_positive_random_features(k.to(dev), W.to(dev))
    o = la.la_causal_fwd(fq, fk, v.to(dev), phi=la.LA_PHI_IDENTITY)
    torch.cuda.synchronize()
    Wf = to_f64(W)
    ref = fm.attention_from_features(fm.positive_random_features(to_f64(q), Wf),
                                     fm.positive_random_features(to_f64(k), Wf), to_f64(v), True)
    assert rowwise_rel(to_f64(o), ref) <= TOL["bf16"]


def test_bad_feature_map_is_refused(la):
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 64, 64, "bf16", seed=5))
    with pytest.raises(la.LinAttnError) as e:
        la.la_causal_fwd(q, k, v, phi=7)
    assert e.value.status == 1
