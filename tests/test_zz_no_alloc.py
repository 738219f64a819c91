"""The causal entry point for callers that cannot allocate device memory.

la_causal_fwd_noalloc takes no workspace: its scratch is a fixed array inside
the library, shared by every call on a device. These tests call it through the
C ABI and check it against la_causal_fwd (which uses a caller-provided
workspace) and against the float64 oracle, on two calls in a row, so that the
second call also shows that left-over contents of the shared array do not leak
into a new result. They also run the fp32 path at the array's exact capacity,
alternate fp32 and bf16 calls (the fp32 path leaves per-chunk fp32 states
where the bf16 path reads tagged words), make a bounded wait run out through
the header's test hook and read the status back, and check that host memory
is refused before any launch, and take the 128-wide bf16 path up to the
largest shape whose last-run sums and seeds fit the array.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from workloads import make_qkv, to_f64

LA_F32, LA_BF16 = 0, 1
LA_ERR_INVALID_ARG, LA_ERR_WORKSPACE, LA_ERR_TIMEOUT = 1, 3, 5
TOL = {"f32": 1e-4, "bf16": 2e-2}


def _lib():
    import linear_attention_elu_gb300 as la
    so = ctypes.CDLL(la.library_path())
    f = so.la_causal_fwd_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P]
    f.restype = I
    so.la_noalloc_query_status.argtypes = [P]
    so.la_noalloc_query_status.restype = I
    so.la_noalloc_set_wait_limit.argtypes = [ctypes.c_uint, I, P]
    so.la_noalloc_set_wait_limit.restype = I
    return la, so


def _rowwise_rel(got, ref):
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return float((num / den).max())


def _call(so, q, k, v, o, S, z, dtype):
    B, H, N, D = q.shape
    return so.la_causal_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    B, H, N, D, D, LA_BF16 if dtype == "bf16" else LA_F32, 1e-6,
                                    S.data_ptr() if S is not None else None,
                                    z.data_ptr() if z is not None else None,
                                    torch.cuda.current_stream().cuda_stream)


def _check_against_oracle(la, so, B, H, N, dtype, seed, with_workspace_entry=True, D=64):
    dev = torch.device("cuda")
    q, k, v = make_qkv(B, H, N, D, dtype, seed=seed)
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o = torch.full_like(vd, float("nan"))
    S = torch.full((B, H, D, D), float("nan"), device=dev)
    z = torch.full((B, H, D), float("nan"), device=dev)
    rc = _call(so, qd, kd, vd, o, S, z, dtype)
    assert rc == 0, la.la_status_string(rc)
    assert so.la_noalloc_query_status(torch.cuda.current_stream().cuda_stream) == 0
    ref, S_ref, z_ref = oracle.recurrent(to_f64(q), to_f64(k), to_f64(v), True, return_state=True)
    assert _rowwise_rel(to_f64(o), ref) <= TOL[dtype]
    if dtype == "bf16":
        # The bf16 path adds bf16-rounded phi(k) v products into its fp32 state:
        # compare each head's S in max norm, as for the workspace entry point.
        Sg = to_f64(S)
        rel = np.abs(Sg - S_ref).max(axis=(-1, -2)) / np.abs(S_ref).max(axis=(-1, -2))
        assert rel.max() <= 1e-2, rel.max()
        np.testing.assert_allclose(to_f64(z), z_ref, rtol=5e-3)
    else:
        np.testing.assert_allclose(to_f64(S), S_ref, rtol=1e-4, atol=1e-3)
        np.testing.assert_allclose(to_f64(z), z_ref, rtol=1e-5, atol=1e-4)
    if with_workspace_entry:
        S_w = torch.empty_like(S)
        z_w = torch.empty_like(z)
        o_w = la.la_causal_fwd(qd, kd, vd, S_out=S_w, z_out=z_w)
        torch.cuda.synchronize()
        assert _rowwise_rel(to_f64(o), to_f64(o_w)) <= TOL[dtype]
        np.testing.assert_allclose(to_f64(S), to_f64(S_w), rtol=1e-5, atol=1e-4)
        np.testing.assert_allclose(to_f64(z), to_f64(z_w), rtol=1e-6, atol=1e-4)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,dtype", [(8, 8, 3072, "bf16"), (2, 3, 1000, "bf16"),
                                         (1, 2, 300, "f32")])
def test_noalloc_matches_workspace_entry_point_and_oracle(B, H, N, dtype):
    la, so = _lib()
    for seed in (31, 32):
        _check_against_oracle(la, so, B, H, N, dtype, seed)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N", [(1, 2, 1000), (1, 1, 127 * 128)])
def test_noalloc_bf16_d128(B, H, N):
    # The 128-wide tensor-core path keeps one last-run sum and one seed per CTA
    # (2 x 66,048 bytes): (1, 2, 1000) is 16 chunks; (1, 1, 127 x 128) is 127
    # chunks on 127 CTAs, the most the array holds (128 is refused below).
    la, so = _lib()
    _check_against_oracle(la, so, B, H, N, "bf16", seed=60 + H, D=128)


@pytest.mark.gpu
def test_noalloc_fp32_at_capacity():
    # B*H*ceil(N/64) = 16 * 63 = 1008 chunk states: exactly what the array holds.
    la, so = _lib()
    _check_against_oracle(la, so, 1, 16, 63 * 64, "f32", seed=40, with_workspace_entry=False)


@pytest.mark.gpu
def test_noalloc_alternating_paths():
    # fp32 calls write per-chunk fp32 states into the array; the bf16 call after
    # each must still find no stale word that passes for one of its tags.
    la, so = _lib()
    for i, dtype in enumerate(("f32", "bf16", "f32", "bf16", "bf16", "f32", "bf16")):
        _check_against_oracle(la, so, 2, 4, 700 + 64 * i, dtype, seed=50 + i,
                              with_workspace_entry=False)


@pytest.mark.gpu
def test_noalloc_wait_timeout_is_reported_and_cleared():
    la, so = _lib()
    st = torch.cuda.current_stream().cuda_stream
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(2, 2, 1000, 64, "bf16", seed=60))
    o = torch.empty_like(v)
    try:
        assert so.la_noalloc_set_wait_limit(2000, 1, st) == 0   # 2 ms, loads withheld
        assert _call(so, q, k, v, o, None, None, "bf16") == 0   # the launch itself succeeds
        assert so.la_noalloc_query_status(st) == LA_ERR_TIMEOUT
        assert so.la_noalloc_query_status(st) == 0              # cleared by the query
    finally:
        assert so.la_noalloc_set_wait_limit(0, 0, st) == 0      # default limit, hook off
    _check_against_oracle(la, so, 2, 2, 1000, "bf16", seed=61)


@pytest.mark.gpu
def test_noalloc_refuses_host_memory():
    _, so = _lib()
    dev = torch.device("cuda")
    q, k, v = make_qkv(1, 1, 128, 64, "bf16", seed=70)
    qd = q.to(dev)
    o = torch.empty_like(qd)
    pinned = k.pin_memory()
    for host in (k, pinned):
        rc = so.la_causal_fwd_noalloc(qd.data_ptr(), host.data_ptr(), qd.data_ptr(), o.data_ptr(),
                                      1, 1, 128, 64, 64, LA_BF16, 1e-6, None, None,
                                      torch.cuda.current_stream().cuda_stream)
        assert rc == LA_ERR_INVALID_ARG


def test_noalloc_rejects_shapes_beyond_its_capacity():
    # Paths that keep one state per chunk need more scratch than the fixed array
    # holds at these shapes: the call must refuse before touching any pointer
    # (these are never dereferenced). 1009 fp32 chunk states at D = 64 is one more
    # than the array holds.
    _, so = _lib()
    fake = 1 << 20
    f = so.la_causal_fwd_noalloc
    assert f(fake, fake, fake, fake, 64, 1000, 128, 32, 32, LA_BF16, 1e-6, None, None, None) \
        == LA_ERR_WORKSPACE
    assert f(fake, fake, fake, fake, 8, 8, 65536, 64, 64, LA_F32, 1e-6, None, None, None) \
        == LA_ERR_WORKSPACE
    assert f(fake, fake, fake, fake, 1, 1, 1009 * 64, 64, 64, LA_F32, 1e-6, None, None, None) \
        == LA_ERR_WORKSPACE
    # 128 chunks at Dk = Dv = 128: neither the tensor-core path (128 CTAs x two
    # 66,048-byte states) nor the fp32 path (256 chunk states) fits.
    assert f(fake, fake, fake, fake, 1, 1, 128 * 128, 128, 128, LA_BF16, 1e-6, None, None, None) \
        == LA_ERR_WORKSPACE
