"""la_causal_fwd_host: host q, k, v in, host o out, transfers overlapped.

The heads go through the device in groups (a quarter of the heads each, the
last quarter split into all but four heads and four); each group is an
ordinary causal forward on its heads, so the output is checked against the
float64 oracle with the gates of the device entry (row-wise relative error,
1e-4 for float32 inputs, 2e-2 for bfloat16), and the final state against the
oracle's S_N, z_N. For the fp32 SIMT path, which treats every head on its own,
the grouping cannot change a single bit: there the host entry must equal the
device entry exactly.
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


@pytest.mark.parametrize("B,H,N,D,dt,pinned", [
    (2, 5, 700, 64, "bf16", True),     # tensor-core path; groups of 4, 4, 2 heads; ragged N
    (1, 1, 129, 64, "bf16", True),     # a single head, one group
    (3, 3, 300, 32, "f32", True),      # fp32 SIMT path; groups of 4, 4, 1 heads
    (1, 6, 256, 64, "bf16", False),    # pageable host memory: correct, not overlapped
    (4, 8, 300, 64, "bf16", True),     # groups of 8, 8, 8, 4, 4: the last group is split
])
def test_host_entry_matches_oracle(la, B, H, N, D, dt, pinned):
    q, k, v = make_qkv(B, H, N, D, dt, seed=B * 1000 + H * 10 + N)
    if pinned:
        q, k, v = (t.pin_memory() for t in (q, k, v))
    dev = torch.device("cuda")
    S = torch.full((B, H, D, D), float("nan"), device=dev)
    z = torch.full((B, H, D), float("nan"), device=dev)
    o = la.la_causal_fwd_host(q, k, v, S_out=S, z_out=z)
    torch.cuda.synchronize()
    assert not o.is_cuda and o.shape == v.shape and o.dtype == v.dtype
    ref, Sr, zr = oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), True, return_state=True)
    assert rowwise_rel(to_f64(o), ref) <= TOL[dt]
    if dt == "f32":
        np.testing.assert_allclose(to_f64(S), Sr, rtol=1e-4, atol=1e-3)
        np.testing.assert_allclose(to_f64(z), zr, rtol=1e-5, atol=1e-4)
    else:
        # S accumulates bf16-rounded phi(k) v products in fp32: compare per head in norm.
        rel = np.abs(to_f64(S) - Sr).max(axis=(-1, -2)) / np.abs(Sr).max(axis=(-1, -2))
        assert rel.max() <= 1e-2, rel.max()
        np.testing.assert_allclose(to_f64(z), zr, rtol=5e-3)


@pytest.mark.parametrize("B,H", [(2, 7), (4, 8)])   # groups 4, 4, 4, 2 and 8, 8, 8, 4, 4
def test_host_entry_equals_device_entry_fp32(la, B, H):
    N, D = 333, 64
    q, k, v = (t.pin_memory() for t in make_qkv(B, H, N, D, "f32", seed=77))
    o_host = la.la_causal_fwd_host(q, k, v)
    dev = torch.device("cuda")
    o_dev = la.la_causal_fwd(q.to(dev), k.to(dev), v.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(o_host, o_dev.cpu())


def test_host_entry_on_a_stream_orders_with_prior_work(la):
    # Inputs filled by work queued on the same stream just before the call: the
    # call must start after it (the copy-in stream waits on the caller's stream).
    B, H, N, D = 2, 4, 512, 64
    q, k, v = (t.pin_memory() for t in make_qkv(B, H, N, D, "bf16", seed=5))
    q2 = torch.empty_like(q).pin_memory()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        src = q.to("cuda", non_blocking=True)
        torch.cuda._sleep(2_000_000)                  # keep the stream busy before the copy out
        q2.copy_(src, non_blocking=True)
        o = la.la_causal_fwd_host(q2, k, v, stream=s)
    s.synchronize()
    ref = oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), True)
    assert rowwise_rel(to_f64(o), ref) <= TOL["bf16"]


def test_host_entry_empty_sequence_zeroes_state(la):
    B, H, D = 1, 3, 64
    q = torch.empty(B, H, 0, D, dtype=torch.bfloat16)
    S = torch.full((B, H, D, D), 7.0, device="cuda")
    z = torch.full((B, H, D), 7.0, device="cuda")
    la.la_causal_fwd_host(q, q, q, S_out=S, z_out=z)
    torch.cuda.synchronize()
    assert float(S.abs().max()) == 0.0 and float(z.abs().max()) == 0.0


def test_host_entry_rejects_small_staging(la):
    B, H, N, D = 1, 2, 128, 64
    q, k, v = make_qkv(B, H, N, D, "bf16", seed=3)
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(la.LinAttnError) as e:
        la.la_causal_fwd_host(q, k, v, staging=small)
    assert e.value.status == 3  # LA_ERR_WORKSPACE
