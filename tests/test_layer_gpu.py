"""la_layer_decode_step against the float64 layer oracle (oracle/layer.py).

The projections run in the input dtype with fp32 accumulation and round q, k,
v and the heads' outputs to that dtype once each; the oracle keeps float64
throughout. Gates: row-wise relative error 1e-4 for float32, 2e-2 for bfloat16
(the attention gates); the state S per head in norm, 1e-5 / 1e-2.
"""
import numpy as np
import pytest
import torch

from oracle import layer
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


def weights(dm, dt, seed):
    # Synthetic projections scaled by 1/sqrt(d_model) (random weights only).
    Wqkv = make_qkv(1, 1, dm, 3 * dm, "f32", seed=seed)[0][0, 0] * dm ** -0.5
    Wo = make_qkv(1, 1, dm, dm, "f32", seed=seed + 1)[1][0, 0] * dm ** -0.5
    cast = torch.bfloat16 if dt == "bf16" else torch.float32
    return Wqkv.to(cast), Wo.to(cast)


@pytest.mark.parametrize("B,H,D,dt,steps", [
    (512, 8, 64, "bf16", 4),     # the blog's layer shape, batch of 512 sequences
    (7, 3, 32, "f32", 5),        # odd batch, generic decode kernel
    (16, 2, 48, "bf16", 3),      # tensor-core products with K and N tails (d_model 96)
    (300, 4, 40, "bf16", 2),     # three row tiles, the last partial (d_model 160)
    (5, 3, 5, "bf16", 3),        # d_model 15: rows not 16-byte multiples, fp32-FMA products
])
def test_layer_steps_match_oracle(la, B, H, D, dt, steps):
    dm = H * D
    Wqkv, Wo = weights(dm, dt, seed=B + D)
    xs = make_qkv(1, steps, B, dm, dt, seed=B * 3 + D)[2][0]          # [steps, B, dm]
    dev = torch.device("cuda")
    S = torch.zeros(B, H, D, D, device=dev)
    z = torch.zeros(B, H, D, device=dev)
    Sr, zr = np.zeros((B, H, D, D)), np.zeros((B, H, D))
    ws = la.workspace(la.LA_OP_LAYER_DECODE, B, H, 1, D, D, xs.dtype, dev)
    Wq_d, Wo_d = Wqkv.to(dev), Wo.to(dev)
    for t in range(steps):
        y = la.la_layer_decode_step(xs[t].to(dev), Wq_d, Wo_d, S, z, H, ws=ws)
        torch.cuda.synchronize()
        ref = layer.layer_decode_step(to_f64(xs[t]), to_f64(Wqkv), to_f64(Wo), Sr, zr, H)
        assert rowwise_rel(to_f64(y), ref) <= TOL[dt], t
    rel = np.abs(to_f64(S) - Sr).max(axis=(-1, -2)) / np.abs(Sr).max(axis=(-1, -2))
    assert rel.max() <= (1e-5 if dt == "f32" else 1e-2)


def test_layer_with_16_byte_aligned_buffers(la):
    # x and y 16 bytes past a 256-byte boundary: the entry point promises 16-byte
    # alignment, so the projections must not assume more.
    B, H, D = 64, 8, 64
    dm = H * D
    Wqkv, Wo = weights(dm, "bf16", seed=3)
    x = make_qkv(1, 1, B, dm, "bf16", seed=4)[2][0, 0]
    dev = torch.device("cuda")
    xbuf = torch.zeros(B * dm + 8, dtype=torch.bfloat16, device=dev)
    ybuf = torch.zeros(B * dm + 8, dtype=torch.bfloat16, device=dev)
    xs = xbuf[8:].view(B, dm)
    ys = ybuf[8:].view(B, dm)
    xs.copy_(x.to(dev))
    assert xs.data_ptr() % 256 == 16 and ys.data_ptr() % 256 == 16
    S = torch.zeros(B, H, D, D, device=dev)
    z = torch.zeros(B, H, D, device=dev)
    la.la_layer_decode_step(xs, Wqkv.to(dev), Wo.to(dev), S, z, H, y=ys)
    torch.cuda.synchronize()
    Sr, zr = np.zeros((B, H, D, D)), np.zeros((B, H, D))
    ref = layer.layer_decode_step(to_f64(x), to_f64(Wqkv), to_f64(Wo), Sr, zr, H)
    assert rowwise_rel(to_f64(ys), ref) <= TOL["bf16"]


def test_layer_rejects_mismatched_heads(la):
    with pytest.raises(ValueError):
        la.la_layer_decode_step(torch.zeros(2, 100, device="cuda", dtype=torch.bfloat16),
                                torch.zeros(100, 300, device="cuda", dtype=torch.bfloat16),
                                torch.zeros(100, 100, device="cuda", dtype=torch.bfloat16),
                                torch.zeros(2, 3, 33, 33, device="cuda"),
                                torch.zeros(2, 3, 33, device="cuda"), 3)
