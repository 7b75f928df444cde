"""Pins for the oracle's single-query (decode) attention (CPU only).

The decode oracle is tied to the full causal forward (itself pinned in
test_oracle_pins.py): the last position of a sequence sees every key, so the
forward's last row is exactly one decode step over a cache holding that
sequence's rotated keys and values.  Closed forms and the ragged-length rule
pin the rest.
"""
import math

import numpy as np
import pytest

import oracle


def rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).normal(0, std, size=shape)


@pytest.mark.parametrize("NH,NKV,theta", [(4, 4, 0.0), (8, 2, 1e6), (6, 1, 1e4)])
def test_decode_equals_forward_last_row(NH, NKV, theta):
    B, T, hd = 2, 37, 8
    C = NH * hd
    qkv = rand((B, T, (NH + 2 * NKV) * hd), seed=NH + NKV)
    out, lse = oracle.attention_forward(qkv, C, NH, NKV, theta)
    Q, K, V = oracle.split_qkv(qkv, C, NH, NKV)
    if theta > 0:
        Q, K = oracle.rope_rotate(Q, theta), oracle.rope_rotate(K, theta)
    d_out, d_lse = oracle.attention_decode(Q[:, T - 1], K, V, [T] * B)
    for h in range(NH):
        np.testing.assert_allclose(d_out[:, h], out[:, T - 1, h * hd:(h + 1) * hd], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(d_lse, lse[:, :, T - 1], rtol=1e-12, atol=1e-13)


def test_decode_shorter_length_equals_forward_at_that_row():
    """len = t + 1 reproduces forward row t (the cache rows past len are ignored)."""
    B, T, NH, NKV, hd = 1, 20, 4, 2, 8
    C = NH * hd
    qkv = rand((B, T, (NH + 2 * NKV) * hd), seed=3)
    out, lse = oracle.attention_forward(qkv, C, NH, NKV, 1e6)
    Q, K, V = oracle.split_qkv(qkv, C, NH, NKV)
    Q, K = oracle.rope_rotate(Q, 1e6), oracle.rope_rotate(K, 1e6)
    for t in (0, 5, 19):
        d_out, d_lse = oracle.attention_decode(Q[:, t], K, V, [t + 1])
        for h in range(NH):
            np.testing.assert_allclose(d_out[0, h], out[0, t, h * hd:(h + 1) * hd], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(d_lse[0], lse[0, :, t], rtol=1e-12, atol=1e-13)


def test_decode_single_key_returns_v():
    B, L, NH, NKV, hd = 3, 5, 4, 2, 16
    q, k, v = rand((B, NH, hd), 1), rand((B, L, NKV, hd), 2), rand((B, L, NKV, hd), 3)
    out, lse = oracle.attention_decode(q, k, v, [1, 1, 1])
    for b in range(B):
        for h in range(NH):
            assert np.array_equal(out[b, h], v[b, 0, h // 2])
            ref = math.fsum(q[b, h] * k[b, 0, h // 2]) / math.sqrt(hd)
            assert abs(lse[b, h] - ref) <= 1e-13


def test_decode_zero_query_gives_mean_of_visible_values():
    B, L, NH, NKV, hd = 2, 9, 2, 1, 4
    k, v = rand((B, L, NKV, hd), 4), rand((B, L, NKV, hd), 5)
    lens = [9, 4]
    out, lse = oracle.attention_decode(np.zeros((B, NH, hd)), k, v, lens)
    for b, n in enumerate(lens):
        for h in range(NH):
            np.testing.assert_allclose(out[b, h], v[b, :n, 0].mean(axis=0), rtol=1e-13, atol=1e-14)
            assert abs(lse[b, h] - math.log(n)) <= 1e-13


def test_decode_ignores_rows_past_the_length():
    B, L, NH, NKV, hd = 2, 12, 4, 4, 8
    q, k, v = rand((B, NH, hd), 6), rand((B, L, NKV, hd), 7), rand((B, L, NKV, hd), 8)
    lens = [5, 12]
    out, lse = oracle.attention_decode(q, k, v, lens)
    k2, v2 = k.copy(), v.copy()
    k2[0, 5:] = 1e3
    v2[0, 5:] = -7.0
    out2, lse2 = oracle.attention_decode(q, k2, v2, lens)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
