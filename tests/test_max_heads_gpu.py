"""The largest head count the library accepts, B*H = 65535 (heads map to a grid
dimension on the fp32 paths), on every forward path, the decode step and the
backward, with a short sequence so that the inputs stay small. Heads are
independent, so sampled heads (the first, the middle, the last) are compared
with the oracle run on those heads alone; the gates are the parity gates.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as bwd
from workloads import make_qkv, to_f64

pytestmark = pytest.mark.gpu

B, H = 5, 13107                 # B * H = 65535
HEADS = [0, 1, 32767, 65533, 65534]
TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module")
def la():
    import linear_attention_elu_gb300 as m
    return m


def rowwise_rel(got, ref):
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return float((num / den).max())


def sampled(t):
    return to_f64(t.reshape((-1,) + tuple(t.shape[2:]))[HEADS])


@pytest.mark.parametrize("causal,dt,N,D", [
    (True, "bf16", 3, 64),    # tensor-core causal: ~431 one-chunk heads per CTA range
    (True, "bf16", 3, 128),   # 128-wide causal: ~431 runs per range (4.3 GB of run sums)
    (True, "f32", 3, 64),     # fp32 path: grid.y = 65535
    (False, "bf16", 3, 64),   # non-causal at D = 64: tensor-core pair, one-chunk heads
    (False, "f32", 3, 64),    # non-causal fp32 path
])
def test_forward_at_maximum_head_count(la, causal, dt, N, D):
    q, k, v = make_qkv(B, H, N, D, dt, seed=N)
    dev = torch.device("cuda")
    fn = la.la_causal_fwd if causal else la.la_noncausal_fwd
    o = fn(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    ref = oracle.recurrent(sampled(q), sampled(k), sampled(v), causal)
    assert rowwise_rel(sampled(o.cpu()), ref) <= TOL[dt]


def test_decode_at_maximum_head_count(la):
    dev = torch.device("cuda")
    S = torch.zeros(B, H, 64, 64, device=dev)
    z = torch.zeros(B, H, 64, device=dev)
    Sr, zr = np.zeros((len(HEADS), 64, 64)), np.zeros((len(HEADS), 64))
    for step in range(2):
        q, k, v = make_qkv(B, H, 1, 64, "bf16", seed=100 + step)
        q, k, v = (t[:, :, 0].contiguous() for t in (q, k, v))
        o = la.la_decode_step(q.to(dev), k.to(dev), v.to(dev), S, z)
        torch.cuda.synchronize()
        ref = oracle.decode_step(sampled(q), sampled(k), sampled(v), Sr, zr)
        assert rowwise_rel(sampled(o.cpu()), ref) <= TOL["bf16"]


def test_backward_at_maximum_head_count(la):
    N = 3
    q, k, v = make_qkv(B, H, N, 64, "f32", seed=7)
    g = make_qkv(B, H, N, 64, "f32", seed=8)[2]
    dev = torch.device("cuda")
    dq, dk, dv = la.la_causal_bwd(q.to(dev), k.to(dev), v.to(dev), g.to(dev))
    torch.cuda.synchronize()
    refs = bwd.grads(sampled(q), sampled(k), sampled(v), sampled(g), True)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        num = np.abs(sampled(got.cpu()) - ref).max(axis=(-1, -2))
        den = np.maximum(np.abs(ref).max(axis=(-1, -2)), 1e-30)
        assert float((num / den).max()) <= TOL["f32"], name


def test_one_head_more_is_refused(la):
    q = torch.empty(1, 65536, 1, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(la.LinAttnError) as e:
        la.la_causal_fwd(q, q, q)
    assert e.value.status == 2  # LA_ERR_UNSUPPORTED
