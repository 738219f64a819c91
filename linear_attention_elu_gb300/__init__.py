"""Python binding of liblinattn.so (kernelized linear attention, phi = elu + 1).

Argument marshalling only: every function here checks shapes and dtypes,
passes raw device pointers and the current CUDA stream to the C ABI declared
in include/linattn.h, and raises on a non-OK status. All arithmetic runs in
the library's CUDA kernels; there is no other code path. PyTorch supplies
device memory and streams.

Importing the package loads the library and fails loudly if it has not been
built (``python linear_attention_elu_gb300/build.py``).
"""
import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "LA_F32", "LA_BF16", "LA_OP_NONCAUSAL", "LA_OP_CAUSAL", "LA_OP_DECODE", "LinAttnError",
    "la_status_string", "la_version", "la_workspace_size", "la_launch_count", "la_workspace_init",
    "la_noncausal_fwd", "la_causal_fwd", "la_decode_step", "la_query_status", "workspace",
    "la_host_staging_size", "host_staging", "la_causal_fwd_host", "la_causal_fwd_state",
    "la_causal_bwd", "LA_OP_CAUSAL_BWD", "la_noncausal_bwd", "LA_OP_NONCAUSAL_BWD",
    "LA_PHI_ELU1", "LA_PHI_IDENTITY", "la_positive_random_features", "LA_OP_LAYER_DECODE",
    "la_layer_decode_step", "la_causal_fwd_noalloc", "la_noalloc_query_status",
    "la_noalloc_set_wait_limit", "library_path",
]

LA_F32, LA_BF16 = 0, 1
LA_OP_NONCAUSAL, LA_OP_CAUSAL, LA_OP_DECODE, LA_OP_CAUSAL_BWD, LA_OP_NONCAUSAL_BWD = 0, 1, 2, 3, 4
LA_OP_LAYER_DECODE = 5
LA_PHI_ELU1, LA_PHI_IDENTITY = 0, 1
LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_WORKSPACE, LA_ERR_CUDA, LA_ERR_TIMEOUT = 0, 1, 2, 3, 4, 5

_DTYPES = {torch.float32: LA_F32, torch.bfloat16: LA_BF16}


class LinAttnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {la_status_string(status)}")


def library_path():
    return _build.LIB


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"liblinattn.so is not built ({path}); run `python linear_attention_elu_gb300/build.py`"
            " or __graft_entry__.build(). There is no fallback implementation.")
    lib = ctypes.CDLL(path)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.la_status_string.argtypes = [I]
    lib.la_status_string.restype = ctypes.c_char_p
    lib.la_version.argtypes = []
    lib.la_version.restype = ctypes.c_uint32
    lib.la_workspace_size.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(Z)]
    lib.la_workspace_size.restype = I
    lib.la_launch_count.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(I)]
    lib.la_launch_count.restype = I
    lib.la_workspace_init.argtypes = [P, Z, P]
    lib.la_workspace_init.restype = I
    lib.la_noncausal_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, Z, P]
    lib.la_noncausal_fwd.restype = I
    lib.la_causal_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P, Z, P]
    lib.la_causal_fwd.restype = I
    lib.la_causal_bwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, Z, P]
    lib.la_causal_bwd.restype = I
    lib.la_noncausal_bwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, Z, P]
    lib.la_noncausal_bwd.restype = I
    lib.la_causal_fwd_state.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P, P, P, Z, P]
    lib.la_causal_fwd_state.restype = I
    lib.la_host_staging_size.argtypes = [I, I, I, I, I, I, ctypes.POINTER(Z)]
    lib.la_host_staging_size.restype = I
    lib.la_causal_fwd_host.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P, Z, P, Z, P]
    lib.la_causal_fwd_host.restype = I
    lib.la_decode_step.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P]
    lib.la_decode_step.restype = I
    L = ctypes.c_int64
    lib.la_noncausal_fwd_phi.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, P, Z, P]
    lib.la_noncausal_fwd_phi.restype = I
    lib.la_causal_fwd_phi.argtypes = [P, P, P, P, I, I, I, I, I, I, I, F, P, P, P, P, P, Z, P]
    lib.la_causal_fwd_phi.restype = I
    lib.la_decode_step_phi.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, P]
    lib.la_decode_step_phi.restype = I
    lib.la_causal_bwd_phi.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, Z, P]
    lib.la_causal_bwd_phi.restype = I
    lib.la_noncausal_bwd_phi.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, Z, P]
    lib.la_noncausal_bwd_phi.restype = I
    lib.la_positive_random_features.argtypes = [P, P, P, L, I, I, I, F, P]
    lib.la_positive_random_features.restype = I
    lib.la_causal_fwd_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P]
    lib.la_causal_fwd_noalloc.restype = I
    lib.la_noalloc_query_status.argtypes = [P]
    lib.la_noalloc_query_status.restype = I
    lib.la_noalloc_set_wait_limit.argtypes = [ctypes.c_uint, I, P]
    lib.la_noalloc_set_wait_limit.restype = I
    lib.la_layer_decode_step.argtypes = [P, P, P, P, P, P, I, I, I, I, F, P, Z, P]
    lib.la_layer_decode_step.restype = I
    lib.la_query_status.argtypes = [P, P]
    lib.la_query_status.restype = I
    return lib


_lib = _load()


def _check(status, where):
    if status != LA_OK:
        raise LinAttnError(status, where)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _dt(t):
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")
    return _DTYPES[t.dtype]


def _need_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous ([B, H, N, D], D innermost)")


def la_status_string(status):
    return _lib.la_status_string(int(status)).decode()


def la_version():
    return int(_lib.la_version())


def la_workspace_size(op, B, H, N, Dk, Dv, dtype):
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    n = ctypes.c_size_t(0)
    _check(_lib.la_workspace_size(int(op), B, H, N, Dk, Dv, dt, ctypes.byref(n)),
           "la_workspace_size")
    return int(n.value)


def la_launch_count(op, B, H, N, Dk, Dv, dtype):
    """Kernel launches one call of `op` makes at this shape (host-only query)."""
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    n = ctypes.c_int(0)
    _check(_lib.la_launch_count(int(op), B, H, N, Dk, Dv, dt, ctypes.byref(n)), "la_launch_count")
    return int(n.value)


def la_workspace_init(ws, stream=None):
    _need_cuda(ws)
    _check(_lib.la_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "la_workspace_init")
    return ws


def workspace(op, B, H, N, Dk, Dv, dtype, device=None, stream=None):
    """Allocates (through PyTorch) and initialises a workspace for `op` at this shape."""
    n = la_workspace_size(op, B, H, N, Dk, Dv, dtype)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")
    return la_workspace_init(ws, stream)


def _shape4(q, k, v):
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError(f"expected q, k [B,H,N,Dk] and v [B,H,N,Dv]; got {tuple(q.shape)}, "
                         f"{tuple(k.shape)}, {tuple(v.shape)}")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    B, H, N, Dk = q.shape
    return B, H, N, Dk, v.shape[3]


def la_noncausal_fwd(q, k, v, o=None, eps=1e-6, ws=None, stream=None, phi=LA_PHI_ELU1):
    """o_i = phi(q_i)^T S / (phi(q_i)^T z + eps), S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j).

    `phi`: LA_PHI_ELU1 (elu + 1) or LA_PHI_IDENTITY (q, k are features already)."""
    B, H, N, Dk, Dv = _shape4(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    _need_cuda(q, k, v, o, ws)
    if ws is None:
        ws = workspace(LA_OP_NONCAUSAL, B, H, N, Dk, Dv, q.dtype, q.device, stream)
    if phi == LA_PHI_ELU1:
        _check(_lib.la_noncausal_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, Dk, Dv, _dt(q),
                                     float(eps), _ptr(ws), ws.numel(), _stream(stream)),
               "la_noncausal_fwd")
    else:
        _check(_lib.la_noncausal_fwd_phi(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, Dk, Dv,
                                         _dt(q), int(phi), float(eps), _ptr(ws), ws.numel(),
                                         _stream(stream)),
               "la_noncausal_fwd_phi")
    return o


def la_causal_fwd(q, k, v, o=None, eps=1e-6, S_out=None, z_out=None, ws=None, stream=None,
                  phi=LA_PHI_ELU1):
    """Causal o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + eps); optional final state out (fp32)."""
    if phi != LA_PHI_ELU1:
        return _causal_phi(q, k, v, None, None, o, eps, S_out, z_out, ws, stream, phi)
    B, H, N, Dk, Dv = _shape4(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    _need_cuda(q, k, v, o, ws, S_out, z_out)
    for t, shp in ((S_out, (B, H, Dk, Dv)), (z_out, (B, H, Dk))):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != shp):
            raise ValueError(f"state outputs must be float32 with shape {shp}")
    if ws is None:
        ws = workspace(LA_OP_CAUSAL, B, H, N, Dk, Dv, q.dtype, q.device, stream)
    _check(_lib.la_causal_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, Dk, Dv, _dt(q),
                              float(eps), _ptr(S_out), _ptr(z_out), _ptr(ws), ws.numel(),
                              _stream(stream)),
           "la_causal_fwd")
    return o


def _causal_phi(q, k, v, S0, z0, o, eps, S_out, z_out, ws, stream, phi):
    B, H, N, Dk, Dv = _shape4(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    _need_cuda(q, k, v, o, ws, S0, z0, S_out, z_out)
    for t, shp in ((S0, (B, H, Dk, Dv)), (z0, (B, H, Dk)), (S_out, (B, H, Dk, Dv)),
                   (z_out, (B, H, Dk))):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != shp):
            raise ValueError(f"states must be float32 with shape {shp}")
    if ws is None:
        ws = workspace(LA_OP_CAUSAL, B, H, N, Dk, Dv, q.dtype, q.device, stream)
    _check(_lib.la_causal_fwd_phi(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, Dk, Dv, _dt(q),
                                  int(phi), float(eps), _ptr(S0), _ptr(z0), _ptr(S_out),
                                  _ptr(z_out), _ptr(ws), ws.numel(), _stream(stream)),
           "la_causal_fwd_phi")
    return o


def la_causal_fwd_noalloc(q, k, v, o=None, eps=1e-6, S_out=None, z_out=None, stream=None):
    """la_causal_fwd without a workspace (scratch is a fixed array inside the library).

    The library uses the array of the current device, so the call runs with
    q's device current."""
    B, H, N, Dk, Dv = _shape4(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    _need_cuda(q, k, v, o, S_out, z_out)
    for t, shp in ((S_out, (B, H, Dk, Dv)), (z_out, (B, H, Dk))):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != shp):
            raise ValueError(f"state outputs must be float32 with shape {shp}")
    with torch.cuda.device(q.device):
        _check(_lib.la_causal_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, Dk, Dv,
                                          _dt(q), float(eps), _ptr(S_out), _ptr(z_out),
                                          _stream(stream)),
               "la_causal_fwd_noalloc")
    return o


def la_noalloc_query_status(device=None, stream=None):
    """Reads and clears the device-side status of the no-allocation calls on `device`."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return _lib.la_noalloc_query_status(_stream(stream))


def la_noalloc_set_wait_limit(max_spin_us=0, hold_loads=False, device=None, stream=None):
    """Wait limit (microseconds, 0 = default) and load-withholding test hook of the
    no-allocation calls on `device`."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _check(_lib.la_noalloc_set_wait_limit(int(max_spin_us), 1 if hold_loads else 0,
                                              _stream(stream)),
               "la_noalloc_set_wait_limit")


def la_causal_fwd_state(q, k, v, S0, z0, o=None, eps=1e-6, S_out=None, z_out=None, ws=None,
                        stream=None, phi=LA_PHI_ELU1):
    """Causal forward continuing from the state (S0 [B,H,Dk,Dv], z0 [B,H,Dk], float32)."""
    if phi != LA_PHI_ELU1:
        return _causal_phi(q, k, v, S0, z0, o, eps, S_out, z_out, ws, stream, phi)
    B, H, N, Dk, Dv = _shape4(q, k, v)
    if o is None:
        o = torch.empty_like(v)
    _need_cuda(q, k, v, o, ws, S0, z0, S_out, z_out)
    for t, shp in ((S0, (B, H, Dk, Dv)), (z0, (B, H, Dk)), (S_out, (B, H, Dk, Dv)),
                   (z_out, (B, H, Dk))):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != shp):
            raise ValueError(f"states must be float32 with shape {shp}")
    if ws is None:
        ws = workspace(LA_OP_CAUSAL, B, H, N, Dk, Dv, q.dtype, q.device, stream)
    _check(_lib.la_causal_fwd_state(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, Dk, Dv, _dt(q),
                                    float(eps), _ptr(S0), _ptr(z0), _ptr(S_out), _ptr(z_out),
                                    _ptr(ws), ws.numel(), _stream(stream)),
           "la_causal_fwd_state")
    return o


def _bwd(fn, op, q, k, v, dout, dq, dk, dv, eps, ws, stream, phi=LA_PHI_ELU1):
    B, H, N, Dk, Dv = _shape4(q, k, v)
    if dout.shape != v.shape or dout.dtype != v.dtype:
        raise ValueError("dout must be shaped and typed like v")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need_cuda(q, k, v, dout, dq, dk, dv, ws)
    if ws is None:
        ws = workspace(op, B, H, N, Dk, Dv, q.dtype, q.device, stream)
    if phi == LA_PHI_ELU1:
        _check(getattr(_lib, fn)(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, H, N, Dk, Dv, _dt(q), float(eps), _ptr(ws),
                                 ws.numel(), _stream(stream)),
               fn)
    else:
        _check(getattr(_lib, fn + "_phi")(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq),
                                          _ptr(dk), _ptr(dv), B, H, N, Dk, Dv, _dt(q), int(phi),
                                          float(eps), _ptr(ws), ws.numel(), _stream(stream)),
               fn + "_phi")
    return dq, dk, dv


def la_causal_bwd(q, k, v, dout, dq=None, dk=None, dv=None, eps=1e-6, ws=None, stream=None,
                  phi=LA_PHI_ELU1):
    """Gradients (dq, dk, dv) of sum(o * dout) for the causal forward o of (q, k, v)."""
    return _bwd("la_causal_bwd", LA_OP_CAUSAL_BWD, q, k, v, dout, dq, dk, dv, eps, ws, stream,
                phi)


def la_noncausal_bwd(q, k, v, dout, dq=None, dk=None, dv=None, eps=1e-6, ws=None, stream=None,
                     phi=LA_PHI_ELU1):
    """Gradients (dq, dk, dv) of sum(o * dout) for the non-causal forward o of (q, k, v)."""
    return _bwd("la_noncausal_bwd", LA_OP_NONCAUSAL_BWD, q, k, v, dout, dq, dk, dv, eps, ws,
                stream, phi)


def la_host_staging_size(B, H, N, Dk, Dv, dtype):
    """Device staging bytes la_causal_fwd_host needs at this shape."""
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    n = ctypes.c_size_t(0)
    _check(_lib.la_host_staging_size(B, H, N, Dk, Dv, dt, ctypes.byref(n)), "la_host_staging_size")
    return int(n.value)


def host_staging(B, H, N, Dk, Dv, dtype, device=None):
    """Allocates (through PyTorch) the device staging buffer of la_causal_fwd_host."""
    n = la_host_staging_size(B, H, N, Dk, Dv, dtype)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def la_causal_fwd_host(q, k, v, o=None, eps=1e-6, S_out=None, z_out=None, staging=None, ws=None,
                       device=None, stream=None):
    """Causal forward on host (CPU) tensors, transfers overlapped with compute; returns o on the
    host. q, k, v should be pinned (tensor.pin_memory()); S_out, z_out are CUDA tensors."""
    B, H, N, Dk, Dv = _shape4(q, k, v)
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous host tensors")
    if o is None:
        o = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    if o.is_cuda or not o.is_contiguous() or o.shape != v.shape or o.dtype != v.dtype:
        raise ValueError("o must be a contiguous host tensor shaped and typed like v")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    _need_cuda(S_out, z_out, staging, ws)
    for t, shp in ((S_out, (B, H, Dk, Dv)), (z_out, (B, H, Dk))):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != shp):
            raise ValueError(f"state outputs must be float32 with shape {shp}")
    if staging is None:
        staging = host_staging(B, H, N, Dk, Dv, q.dtype, dev)
    if ws is None:
        ws = workspace(LA_OP_CAUSAL, B, H, N, Dk, Dv, q.dtype, dev, stream)
    _check(_lib.la_causal_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, N, Dk, Dv, _dt(q),
                                   float(eps), _ptr(S_out), _ptr(z_out), _ptr(staging),
                                   staging.numel(), _ptr(ws), ws.numel(), _stream(stream)),
           "la_causal_fwd_host")
    return o


def la_decode_step(q, k, v, S, z, o=None, eps=1e-6, stream=None, phi=LA_PHI_ELU1):
    """One recurrent step on (S, z) in place; q, k [B,H,Dk], v [B,H,Dv]; returns o [B,H,Dv]."""
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[:2] != q.shape[:2]:
        raise ValueError("expected q, k [B,H,Dk] and v [B,H,Dv]")
    B, H, Dk = q.shape
    Dv = v.shape[2]
    if S.dtype != torch.float32 or z.dtype != torch.float32 or tuple(S.shape) != (B, H, Dk, Dv) \
            or tuple(z.shape) != (B, H, Dk):
        raise ValueError("S must be float32 [B,H,Dk,Dv] and z float32 [B,H,Dk]")
    if o is None:
        o = torch.empty_like(v)
    _need_cuda(q, k, v, o, S, z)
    if phi == LA_PHI_ELU1:
        _check(_lib.la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(S), _ptr(z), B, H, Dk,
                                   Dv, _dt(q), float(eps), _stream(stream)),
               "la_decode_step")
    else:
        _check(_lib.la_decode_step_phi(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(S), _ptr(z), B, H,
                                       Dk, Dv, _dt(q), int(phi), float(eps), _stream(stream)),
               "la_decode_step_phi")
    return o


def la_positive_random_features(x, W, out=None, shift=0.0, stream=None):
    """exp(W x - |x|^2 / 2 - shift) / sqrt(R) over the last axis of x [..., D]; W [R, D].

    Returns out [..., R] in x's dtype: features for the LA_PHI_IDENTITY entries."""
    if W.dim() != 2 or x.shape[-1] != W.shape[1] or W.dtype != x.dtype:
        raise ValueError("expected x [..., D] and W [R, D] of one dtype")
    R, D = W.shape
    rows = x.numel() // D if D else 0
    if out is None:
        out = torch.empty(tuple(x.shape[:-1]) + (R,), dtype=x.dtype, device=x.device)
    _need_cuda(x, W, out)
    _check(_lib.la_positive_random_features(_ptr(x), _ptr(W), _ptr(out), rows, D, R, _dt(x),
                                            float(shift), _stream(stream)),
           "la_positive_random_features")
    return out


def la_layer_decode_step(x, Wqkv, Wo, S, z, H, y=None, eps=1e-6, ws=None, stream=None):
    """One decode step of a linear-attention layer: x [B, d_model] -> y [B, d_model].

    Wqkv [d_model, 3 H D] (q | k | v, head-major within each), Wo [H D, d_model];
    S [B, H, D, D] and z [B, H, D] (float32) are updated in place."""
    if x.dim() != 2 or Wqkv.dim() != 2 or Wo.dim() != 2:
        raise ValueError("expected x [B, d_model], Wqkv [d_model, 3 H D], Wo [H D, d_model]")
    B, dm = x.shape
    D = dm // H if H else 0
    if H * D != dm or tuple(Wqkv.shape) != (dm, 3 * dm) or tuple(Wo.shape) != (dm, dm):
        raise ValueError("d_model must equal H D, Wqkv be [d_model, 3 d_model], Wo [d_model, d_model]")
    if Wqkv.dtype != x.dtype or Wo.dtype != x.dtype:
        raise TypeError("x, Wqkv and Wo must share one dtype")
    if S.dtype != torch.float32 or z.dtype != torch.float32 or tuple(S.shape) != (B, H, D, D) \
            or tuple(z.shape) != (B, H, D):
        raise ValueError("S must be float32 [B,H,D,D] and z float32 [B,H,D]")
    if y is None:
        y = torch.empty_like(x)
    _need_cuda(x, Wqkv, Wo, y, S, z, ws)
    if ws is None:
        ws = workspace(LA_OP_LAYER_DECODE, B, H, 1, D, D, x.dtype, x.device, stream)
    _check(_lib.la_layer_decode_step(_ptr(x), _ptr(Wqkv), _ptr(Wo), _ptr(y), _ptr(S), _ptr(z), B,
                                     H, D, _dt(x), float(eps), _ptr(ws), ws.numel(),
                                     _stream(stream)),
           "la_layer_decode_step")
    return y


def la_query_status(ws, stream=None):
    """Synchronises the stream and returns (and clears) the workspace status code."""
    return int(_lib.la_query_status(_ptr(ws), _stream(stream)))
