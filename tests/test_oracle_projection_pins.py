"""Pins for the oracle's QKV projection (CPU only): the product against a
brute-force triple loop, the rotated copy against the pinned RoPE of the
projected heads, and positions restarting at every sequence."""
import math

import numpy as np
import pytest

import oracle


def test_projection_brute_force():
    rng = np.random.default_rng(1)
    B, T, Cm, NH, NKV, hd = 2, 3, 5, 2, 1, 4
    N = (NH + 2 * NKV) * hd
    x, w = rng.normal(size=(B * T, Cm)), rng.normal(size=(N, Cm))
    qkv, rot = oracle.qkv_projection(x, w, T, NH, NKV, 0.0)
    for m in range(B * T):
        for n in range(N):
            assert abs(qkv[m, n] - math.fsum(x[m, k] * w[n, k] for k in range(Cm))) <= 1e-12
    assert np.array_equal(rot, qkv[:, :(NH + NKV) * hd])          # no RoPE: the plain Q | K columns


@pytest.mark.parametrize("interleaved", [False, True])
def test_projection_rotation_per_sequence(interleaved):
    rng = np.random.default_rng(2)
    B, T, Cm, NH, NKV, hd = 3, 7, 16, 4, 2, 8
    N = (NH + 2 * NKV) * hd
    x, w = rng.normal(size=(B * T, Cm)), rng.normal(size=(N, Cm))
    qkv, rot = oracle.qkv_projection(x, w, T, NH, NKV, 1e4, rope_interleaved=interleaved)
    Q, K, _ = oracle.split_qkv(qkv.reshape(B, T, N), NH * hd, NH, NKV)
    f = oracle.rope_rotate_interleaved if interleaved else oracle.rope_rotate
    want = np.concatenate([f(Q, 1e4), f(K, 1e4)], axis=2).reshape(B * T, -1)
    np.testing.assert_allclose(rot, want, rtol=1e-13, atol=1e-13)
    # position 0 of every sequence is unrotated
    for b in range(B):
        np.testing.assert_allclose(rot[b * T], qkv[b * T, :(NH + NKV) * hd], rtol=1e-14, atol=1e-14)
