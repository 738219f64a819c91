"""Float64 linear-attention layer decode step — TEST INFRASTRUCTURE ONLY.

Only tests/ may import this module. It shares no code with the CUDA library.

One generation step of a linear-attention layer for B sequences: the token's
hidden vector x [d_model] is projected to queries, keys and values of H heads
of width D (d_model = H D), each head takes one step of the recurrence on its
state, and the heads' outputs are projected back ("Why Replace Attention? The
Softmax Bottleneck and the Path to Linear Time", section 7.2, steps 1-4:
compute phi(k_i) and v_i from the token's hidden state, update S and z, read
with phi(q_i); "Transformers Are RNNs: Linear Attention", the generation loop
that carries only (S, z) from token to token):

    [q | k | v] = x Wqkv            (Wqkv [d_model, 3 H D]; head h of q is
                                     columns h D .. h D + D - 1, likewise k, v)
    o_h = decode step of head h     (the C oracle's decode_step)
    y = [o_1 | ... | o_H] Wo        (Wo [H D, d_model])

The projections are plain matrix products; the attention step is the C
oracle's, which the pages' worked example pins. Pins: tests/test_oracle_layer.py.
"""
import numpy as np

import oracle


def layer_decode_step(x, Wqkv, Wo, S, z, H, eps=1e-6):
    """Returns y [B, d_model]; S [B, H, D, D] and z [B, H, D] (float64) are updated in place."""
    x, Wqkv, Wo = (np.ascontiguousarray(np.asarray(a, dtype=np.float64)) for a in (x, Wqkv, Wo))
    B, dm = x.shape
    D = dm // H
    qkv = x @ Wqkv
    q = qkv[:, 0:H * D].reshape(B, H, D)
    k = qkv[:, H * D:2 * H * D].reshape(B, H, D)
    v = qkv[:, 2 * H * D:3 * H * D].reshape(B, H, D)
    o = oracle.decode_step(q, k, v, S, z, eps)
    return o.reshape(B, H * D) @ Wo
