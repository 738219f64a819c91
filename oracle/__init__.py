"""Float64 CPU oracle for elu+1 linear attention — TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package. It shares no code with the CUDA library: it is a separate C
file (linattn_oracle.c) compiled by the host C compiler and loaded here with
ctypes. Inputs are numpy arrays; they are converted to contiguous float64.

Forms (each written out as its definition, see linattn_oracle.c):
  * ``quadratic`` — w_ij = phi(q_i).phi(k_j), masked to j <= i when causal,
    row-normalised, times V ("Why Replace Attention? The Softmax Bottleneck
    and the Path to Linear Time", sections 5.7, 6.5 and 7.1).
  * ``recurrent`` — S_i = S_{i-1} + phi(k_i) v_i^T, z_i = z_{i-1} + phi(k_i),
    o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + eps) (same blog, section 7.2);
    non-causal rows read the final S, z (section 6.2).
  * ``decode_step`` — one iteration of that recurrence on caller state.
  * ``rows`` — selected output rows by the quadratic definition.

Pins: tests/test_oracle.py checks every function against the pages' worked
example (tests/golden/), closed forms and invariants.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        lp = ctypes.POINTER(ctypes.c_long)
        L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
        lib.ora_phi.argtypes = [D]
        lib.ora_phi.restype = D
        lib.ora_phi_array.argtypes = [dp, dp, L]
        lib.ora_phi_array.restype = None
        lib.ora_quadratic.argtypes = [dp, dp, dp, dp, L, L, I, I, I, D, I]
        lib.ora_quadratic.restype = I
        lib.ora_recurrent.argtypes = [dp, dp, dp, dp, dp, dp, L, L, I, I, I, D, I]
        lib.ora_recurrent.restype = I
        lib.ora_decode_step.argtypes = [dp, dp, dp, dp, dp, dp, L, I, I, D]
        lib.ora_decode_step.restype = I
        lib.ora_rows.argtypes = [dp, dp, dp, L, L, I, I, I, D, lp, lp, L, dp]
        lib.ora_rows.restype = I
        _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads():
    return max(1, os.cpu_count() or 1)


def _heads(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim < 2 or q.shape != k.shape or v.shape[:-1] != q.shape[:-1]:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    lead = q.shape[:-2]
    N, D = q.shape[-2:]
    M = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    return q, k, v, lead, BH, N, D, M


def phi(x):
    """elu(x) + 1 element-wise, in float64."""
    x = _f64(x)
    y = np.empty_like(x)
    _load().ora_phi_array(_ptr(x), _ptr(y), x.size)
    return y


def quadratic(q, k, v, causal, eps=1e-6, nthreads=None):
    """Quadratic (masked, row-normalised) form; q, k: [..., N, D], v: [..., N, M]."""
    q, k, v, lead, BH, N, D, M = _heads(q, k, v)
    o = np.empty(lead + (N, M), dtype=np.float64)
    rc = _load().ora_quadratic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), BH, N, D, M,
                               int(bool(causal)), float(eps), nthreads or default_threads())
    if rc:
        raise RuntimeError(f"ora_quadratic failed ({rc})")
    return o


def recurrent(q, k, v, causal, eps=1e-6, nthreads=None, return_state=False):
    """Recurrent form; returns o (and the final S [..., D, M], z [..., D])."""
    q, k, v, lead, BH, N, D, M = _heads(q, k, v)
    o = np.empty(lead + (N, M), dtype=np.float64)
    S = np.empty(lead + (D, M), dtype=np.float64)
    z = np.empty(lead + (D,), dtype=np.float64)
    rc = _load().ora_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(S), _ptr(z),
                               BH, N, D, M, int(bool(causal)), float(eps),
                               nthreads or default_threads())
    if rc:
        raise RuntimeError(f"ora_recurrent failed ({rc})")
    return (o, S, z) if return_state else o


def decode_step(q, k, v, S, z, eps=1e-6):
    """One recurrent step on (S, z), updated in place (float64 arrays).

    q, k: [..., D]; v: [..., M]; S: [..., D, M]; z: [..., D]. Returns o [..., M].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if S.dtype != np.float64 or z.dtype != np.float64 or not S.flags.c_contiguous \
            or not z.flags.c_contiguous:
        raise ValueError("S and z must be contiguous float64 arrays (updated in place)")
    D, M = q.shape[-1], v.shape[-1]
    lead = q.shape[:-1]
    BH = int(np.prod(lead)) if lead else 1
    if S.shape != lead + (D, M) or z.shape != lead + (D,) or k.shape != q.shape:
        raise ValueError("shape mismatch")
    o = np.empty(lead + (M,), dtype=np.float64)
    rc = _load().ora_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(S), _ptr(z),
                                 BH, D, M, float(eps))
    if rc:
        raise RuntimeError(f"ora_decode_step failed ({rc})")
    return o


def rows(q, k, v, causal, heads, idx, eps=1e-6):
    """Output rows (heads[r], idx[r]) by the quadratic definition; q: [BH, N, D]."""
    q, k, v, lead, BH, N, D, M = _heads(q, k, v)
    h = np.ascontiguousarray(np.asarray(heads, dtype=np.int64)).astype(np.dtype("long"))
    i = np.ascontiguousarray(np.asarray(idx, dtype=np.int64)).astype(np.dtype("long"))
    if h.shape != i.shape:
        raise ValueError("heads and idx must have the same length")
    out = np.empty((h.size, M), dtype=np.float64)
    lp = ctypes.POINTER(ctypes.c_long)
    rc = _load().ora_rows(_ptr(q), _ptr(k), _ptr(v), BH, N, D, M, int(bool(causal)),
                          float(eps), h.ctypes.data_as(lp), i.ctypes.data_as(lp), h.size,
                          _ptr(out))
    if rc:
        raise RuntimeError(f"ora_rows failed ({rc})")
    return out
