"""The decode step over the whole decode configuration: 512 sequences x 8 heads,
Dk = Dv = 64, 3072 consecutive bf16 tokens per head, fp32 state updated in
place ("Transformers Are RNNs: Linear Attention", "Turn Causal Attention into
a Recurrence": S and z are running sums, updated then read at every step).

Tokens are drawn on the device from a seeded generator (one draw of q, k, v
per step); the outputs and tokens of sampled heads are copied out at every
step and compared with the float64 oracle's causal recurrence over the same
3072 tokens (decode x N = causal), so rounding drift accumulated over all
steps is checked at the 2e-2 bf16 gate, and the final fp32 state against the
oracle's state.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import WORKLOADS, to_f64

pytestmark = pytest.mark.gpu


def test_decode_config_all_steps_sampled_heads():
    import linear_attention_elu_gb300 as la
    w = WORKLOADS["decode"]
    dev = torch.device("cuda")
    B, H, D, T = w.B, w.H, w.D, w.N
    rng = np.random.default_rng(5)
    flat = rng.choice(B * H, size=16, replace=False)
    bi = torch.tensor(flat // H, device=dev)
    hi = torch.tensor(flat % H, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(2024)
    S = torch.zeros(B, H, D, D, device=dev)
    z = torch.zeros(B, H, D, device=dev)
    o = torch.empty(B, H, D, device=dev, dtype=torch.bfloat16)
    toks = torch.empty(3, T, 16, D, device=dev, dtype=torch.bfloat16)
    outs = torch.empty(T, 16, D, device=dev, dtype=torch.bfloat16)
    for t in range(T):
        q, k, v = (torch.randn(B, H, D, device=dev, generator=gen).bfloat16() for _ in range(3))
        la.la_decode_step(q, k, v, S, z, o=o)
        for j, x in enumerate((q, k, v)):
            toks[j, t] = x[bi, hi]
        outs[t] = o[bi, hi]
    torch.cuda.synchronize()
    qs, ks, vs = (to_f64(toks[j]).transpose(1, 0, 2) for j in range(3))   # [16, T, D]
    ref, S_ref, z_ref = oracle.recurrent(qs, ks, vs, True, return_state=True)
    got = to_f64(outs).transpose(1, 0, 2)
    err = np.abs(got - ref).max(-1) / np.abs(ref).max(-1)
    assert err.max() <= 2e-2, (err.max(), np.unravel_index(err.argmax(), err.shape))
    Sg = to_f64(S[bi, hi])
    zg = to_f64(z[bi, hi])
    rel_S = np.abs(Sg - S_ref).max(axis=(-1, -2)) / np.abs(S_ref).max(axis=(-1, -2))
    assert rel_S.max() <= 1e-4, rel_S.max()
    np.testing.assert_allclose(zg, z_ref, rtol=1e-5)
