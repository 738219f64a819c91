"""Float64 gradients of the forward pass — TEST INFRASTRUCTURE ONLY.

Only tests/ may import this module. It shares no code with the CUDA library.

The gradient of a scalar loss L through o with respect to q, k and v, computed
by PyTorch's reverse-mode autograd in float64 on the CPU over the plain
definitions of the forward:

  * quadratic form: w_ij = phi(q_i).phi(k_j) for j <= i (causal) or all j,
    o_i = sum_j w_ij v_j / (sum_j w_ij + eps)
    ("Why Replace Attention? The Softmax Bottleneck and the Path to Linear
    Time", sections 5.7 and 7.1; phi(x) = elu(x) + 1, section 5.3);
  * recurrent form: S_i = S_{i-1} + phi(k_i) v_i^T, z_i = z_{i-1} + phi(k_i),
    o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + eps) (same blog, section 7.2),
    written as an explicit loop (small inputs only).

The pages print no backward formulas; they note only that gradients taken as
forward and reverse cumulative sums keep causal training linear in N without
storing every S_i ("Transformers Are RNNs: Linear Attention", "Turn Causal
Attention into a Recurrence"). The reference here is therefore the derivative
of the definition itself; tests/test_oracle_bwd.py pins it with central finite
differences and with the agreement of the two forms.
"""
import numpy as np
import torch


def _phi(x, phi="elu1"):
    # elu(x) + 1: x + 1 for x > 0, e^x for x <= 0 (the exp branch is evaluated
    # on min(x, 0) so that its unused values never overflow). "identity": the
    # inputs are already features (the method leaves phi free, "Why Replace
    # Attention?", section 4.5).
    if phi == "identity":
        return x
    return torch.where(x > 0, x + 1.0, torch.exp(torch.clamp(x, max=0.0)))


def _t(a):
    return torch.tensor(np.asarray(a, dtype=np.float64), dtype=torch.float64)


def forward_quadratic(q, k, v, causal, eps=1e-6, phi="elu1"):
    fq, fk = _phi(q, phi), _phi(k, phi)
    w = fq @ fk.transpose(-1, -2)
    if causal:
        w = torch.tril(w)
    return (w @ v) / (w.sum(-1, keepdim=True) + eps)


def forward_recurrent(q, k, v, causal, eps=1e-6, phi="elu1"):
    fq, fk = _phi(q, phi), _phi(k, phi)
    N = q.shape[-2]
    S = torch.zeros(q.shape[:-2] + (q.shape[-1], v.shape[-1]), dtype=q.dtype)
    z = torch.zeros(q.shape[:-2] + (q.shape[-1],), dtype=q.dtype)
    rows = []
    for i in range(N):
        S = S + fk[..., i, :, None] * v[..., i, None, :]
        z = z + fk[..., i, :]
        if causal:
            rows.append((fq[..., i, None, :] @ S)[..., 0, :] / ((fq[..., i, :] * z).sum(-1, keepdim=True) + eps))
    if not causal:
        num = fq @ S
        den = (fq * z[..., None, :]).sum(-1, keepdim=True) + eps
        return num / den
    return torch.stack(rows, dim=-2)


def grads(q, k, v, dout, causal=True, eps=1e-6, form="quadratic", phi="elu1"):
    """dL/dq, dL/dk, dL/dv for L = sum(o * dout); inputs [..., N, D] / [..., N, M].

    Returns float64 numpy arrays. `form` selects the forward definition the
    derivative is taken of ("quadratic" or "recurrent"); `phi` the feature map
    ("elu1" or "identity")."""
    qt, kt, vt = (_t(a).requires_grad_(True) for a in (q, k, v))
    g = _t(dout)
    fwd = forward_quadratic if form == "quadratic" else forward_recurrent
    o = fwd(qt, kt, vt, causal, eps, phi)
    (o * g).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def forward(q, k, v, causal=True, eps=1e-6, form="quadratic", phi="elu1"):
    """The forward of the chosen form, as a float64 numpy array."""
    fwd = forward_quadratic if form == "quadratic" else forward_recurrent
    with torch.no_grad():
        return fwd(_t(q), _t(k), _t(v), causal, eps, phi).numpy()
