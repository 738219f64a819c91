"""The causal entry point for callers that cannot allocate device memory.

la_causal_fwd_noalloc takes no workspace: its scratch is a fixed array inside
the library. These tests call it through the C ABI and compare it with
la_causal_fwd (which uses a caller-provided workspace) on two calls in a row,
so that the second call also shows that left-over contents of the shared
array do not leak into a new result. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import make_qkv, to_f64

LA_F32, LA_BF16, LA_ERR_WORKSPACE = 0, 1, 3
TOL = {"f32": 1e-4, "bf16": 2e-2}


def _fn():
    import linear_attention_elu_gb300 as la
    so = ctypes.CDLL(la.library_path())
    f = so.la_causal_fwd_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P]
    f.restype = I
    return la, f


def _rowwise_rel(got, ref):
    num = np.abs(got - ref).max(axis=-1)
    den = np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    return float((num / den).max())


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,N,dtype", [(8, 8, 3072, "bf16"), (1, 2, 300, "f32")])
def test_noalloc_matches_workspace_entry_point(B, H, N, dtype):
    la, f = _fn()
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    for call, seed in enumerate((31, 32)):
        q, k, v = (t.to(dev) for t in make_qkv(B, H, N, 64, dtype, seed=seed))
        S_ref = torch.empty(B, H, 64, 64, device=dev)
        z_ref = torch.empty(B, H, 64, device=dev)
        o_ref = la.la_causal_fwd(q, k, v, S_out=S_ref, z_out=z_ref)
        o = torch.full_like(v, float("nan"))
        S = torch.full_like(S_ref, float("nan"))
        z = torch.full_like(z_ref, float("nan"))
        rc = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, N, 64, 64,
               LA_BF16 if dtype == "bf16" else LA_F32, 1e-6, S.data_ptr(), z.data_ptr(),
               stream.cuda_stream)
        assert rc == 0, f"call {call}: {la.la_status_string(rc)}"
        torch.cuda.synchronize()
        assert _rowwise_rel(to_f64(o), to_f64(o_ref)) <= TOL[dtype], f"call {call}"
        np.testing.assert_allclose(to_f64(S), to_f64(S_ref), rtol=1e-5, atol=1e-4)
        np.testing.assert_allclose(to_f64(z), to_f64(z_ref), rtol=1e-6, atol=1e-4)


def test_noalloc_rejects_shapes_beyond_its_capacity():
    # Paths that keep one state per chunk need more scratch than the fixed array
    # holds at these shapes: the call must refuse before touching any pointer
    # (these are never dereferenced).
    _, f = _fn()
    fake = 1 << 20
    rc = f(fake, fake, fake, fake, 64, 1000, 128, 32, 32, LA_BF16, 1e-6, None, None, None)
    assert rc == LA_ERR_WORKSPACE
    rc = f(fake, fake, fake, fake, 8, 8, 65536, 64, 64, LA_F32, 1e-6, None, None, None)
    assert rc == LA_ERR_WORKSPACE
