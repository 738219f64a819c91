"""Pins of the layer decode-step oracle (oracle/layer.py), CPU only.

It is tied to the C oracle, which the pages' worked example pins: with identity
projections the layer step is the bare decode step; a run of steps equals the
causal recurrence over the projected sequence followed by the output
projection; and the output is linear in Wo.
"""
import numpy as np

import oracle
from oracle import layer


def test_identity_projections_reduce_to_the_decode_step():
    rng = np.random.default_rng(1)
    B, H, D = 3, 2, 4
    dm = H * D
    x = rng.standard_normal((B, dm))
    Wqkv = np.concatenate([np.eye(dm)] * 3, axis=1)       # q = k = v = x
    S, z = np.zeros((B, H, D, D)), np.zeros((B, H, D))
    S2, z2 = S.copy(), z.copy()
    y = layer.layer_decode_step(x, Wqkv, np.eye(dm), S, z, H)
    ref = oracle.decode_step(x.reshape(B, H, D), x.reshape(B, H, D), x.reshape(B, H, D), S2, z2)
    np.testing.assert_allclose(y, ref.reshape(B, dm), rtol=1e-14)
    np.testing.assert_allclose(S, S2, rtol=1e-14)
    np.testing.assert_allclose(z, z2, rtol=1e-14)


def test_steps_equal_causal_attention_on_the_projected_sequence():
    rng = np.random.default_rng(2)
    B, H, D, T = 2, 3, 4, 9
    dm = H * D
    xs = rng.standard_normal((T, B, dm))
    Wqkv, Wo = rng.standard_normal((dm, 3 * dm)) / 4, rng.standard_normal((dm, dm)) / 4
    S, z = np.zeros((B, H, D, D)), np.zeros((B, H, D))
    ys = np.stack([layer.layer_decode_step(xs[t], Wqkv, Wo, S, z, H) for t in range(T)], axis=1)
    qkv = xs.transpose(1, 0, 2) @ Wqkv                          # [B, T, 3 dm]
    heads = lambda a: a.reshape(B, T, H, D).transpose(0, 2, 1, 3)
    q, k, v = heads(qkv[..., :dm]), heads(qkv[..., dm:2 * dm]), heads(qkv[..., 2 * dm:])
    o, Sr, zr = oracle.recurrent(q, k, v, True, return_state=True)
    ref = o.transpose(0, 2, 1, 3).reshape(B, T, dm) @ Wo
    np.testing.assert_allclose(ys, ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(S, Sr, rtol=1e-12)
    np.testing.assert_allclose(z, zr, rtol=1e-12)


def test_output_is_linear_in_Wo():
    rng = np.random.default_rng(3)
    B, H, D = 2, 2, 3
    dm = H * D
    x = rng.standard_normal((B, dm))
    Wqkv = rng.standard_normal((dm, 3 * dm))
    A, C = rng.standard_normal((dm, dm)), rng.standard_normal((dm, dm))
    outs = []
    for Wo in (A, C, 2 * A - C):
        S, z = np.zeros((B, H, D, D)), np.zeros((B, H, D))
        outs.append(layer.layer_decode_step(x, Wqkv, Wo, S, z, H))
    np.testing.assert_allclose(outs[2], 2 * outs[0] - outs[1], rtol=1e-12, atol=1e-12)
