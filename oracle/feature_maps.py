"""Float64 forms for other feature maps — TEST INFRASTRUCTURE ONLY.

Only tests/ may import this module. It shares no code with the CUDA library.

The method leaves phi free: any map of a query or key into a feature space of
its own width r (which need not equal the head width) turns the similarity into
the dot product phi(q).phi(k) ("Why Replace Attention? The Softmax Bottleneck
and the Path to Linear Time", section 4.5; the Core ML "Linear Attention" page,
"The kernel decomposition", naming elu(x) + 1 and random features as examples).
Two pieces follow from that:

  * ``attention_from_features`` / ``recurrent_from_features`` — the attention
    on features the caller has already computed: w_ij = fq_i . fk_j over j <= i
    (causal) or all j, o_i = sum_j w_ij v_j / (sum_j w_ij + eps), in the
    quadratic form and as the explicit recurrence S_i = S_{i-1} + fk_i v_i^T,
    z_i = z_{i-1} + fk_i (same blog, sections 6 and 7).
  * ``positive_random_features`` — phi(x)_r = exp(w_r . x - |x|^2 / 2 - shift)
    / sqrt(r) for the rows w_r of a matrix W whose entries the caller draws
    from N(0, 1). The research-hub "Linear Attention" page ("Key math / How it
    works") says Performers use positive random features for an unbiased
    estimate of the softmax kernel; it prints no formula. This is the plainest
    map with that property: for w ~ N(0, I), E[exp(w.(x + y))] = exp(|x + y|^2 / 2)
    (the Gaussian moment generating function), so
    E[exp(w.x - |x|^2/2) exp(w.y - |y|^2/2)] = exp(x.y). `shift` is a constant
    the caller may subtract in the exponent against overflow; it scales every
    feature of the call by exp(-shift), which cancels in o when one shift is
    used for all keys of a head (or per query row).

Pins: tests/test_oracle_features.py.
"""
import numpy as np


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def attention_from_features(fq, fk, v, causal, eps=1e-6):
    """o [..., N, M] from features fq, fk [..., N, r] and values v [..., N, M]."""
    fq, fk, v = _f64(fq), _f64(fk), _f64(v)
    w = fq @ np.swapaxes(fk, -1, -2)
    if causal:
        w = np.tril(w)
    return (w @ v) / (w.sum(axis=-1, keepdims=True) + eps)


def recurrent_from_features(fq, fk, v, causal, eps=1e-6, return_state=False):
    """The recurrence on features, one token at a time (small inputs only)."""
    fq, fk, v = _f64(fq), _f64(fk), _f64(v)
    N = fq.shape[-2]
    S = np.zeros(fq.shape[:-2] + (fq.shape[-1], v.shape[-1]))
    z = np.zeros(fq.shape[:-2] + (fq.shape[-1],))
    rows = []
    for i in range(N):
        S = S + fk[..., i, :, None] * v[..., i, None, :]
        z = z + fk[..., i, :]
        if causal:
            num = np.einsum("...r,...rm->...m", fq[..., i, :], S)
            den = np.einsum("...r,...r->...", fq[..., i, :], z)[..., None] + eps
            rows.append(num / den)
    if causal:
        o = np.stack(rows, axis=-2)
    else:
        o = np.einsum("...nr,...rm->...nm", fq, S) / (
            np.einsum("...nr,...r->...n", fq, z)[..., None] + eps)
    return (o, S, z) if return_state else o


def decode_from_features(fq, fk, v, S, z, eps=1e-6):
    """One step of the recurrence on features; returns (o, S', z') without mutation."""
    fq, fk, v, S, z = _f64(fq), _f64(fk), _f64(v), _f64(S), _f64(z)
    S = S + fk[..., :, None] * v[..., None, :]
    z = z + fk
    o = np.einsum("...r,...rm->...m", fq, S) / (np.einsum("...r,...r->...", fq, z)[..., None] + eps)
    return o, S, z


def positive_random_features(x, W, shift=0.0):
    """phi(x) [..., r] = exp(W x - |x|^2 / 2 - shift) / sqrt(r) for x [..., D], W [r, D]."""
    x, W = _f64(x), _f64(W)
    r = W.shape[0]
    proj = x @ W.T
    half_sq = 0.5 * np.sum(x * x, axis=-1, keepdims=True)
    return np.exp(proj - half_sq - float(shift)) / np.sqrt(r)
