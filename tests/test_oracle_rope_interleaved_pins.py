"""Pins for the oracle's interleaved (GPT-J) RoPE and the attention it feeds
(CPU only): a hand-worked rotation, the permutation that maps it onto the
NEOX form, the rotation properties, and the attention built on it against the
NEOX attention of permuted inputs."""
import math

import numpy as np
import pytest

import oracle


def test_interleaved_rotation_worked_example():
    """hd = 4, theta = 1e4, position 1: pair 0 turns by 1 rad, pair 1 by
    1e4^(-1/2) = 0.01 rad (worked by hand from rope_kernel's formula)."""
    x = np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 1, 4)
    x = np.concatenate([np.zeros_like(x), x], axis=0)          # positions 0 and 1
    y = oracle.rope_rotate_interleaved(x, 1e4)
    c0, s0, c1, s1 = math.cos(1.0), math.sin(1.0), math.cos(0.01), math.sin(0.01)
    want = [1 * c0 - 2 * s0, 1 * s0 + 2 * c0, 3 * c1 - 4 * s1, 3 * s1 + 4 * c1]
    np.testing.assert_allclose(y[1, 0], want, rtol=1e-15, atol=1e-15)
    assert np.array_equal(y[0], x[0])                           # identity at t = 0


def perm(hd):
    """Column order that puts interleaved pair (2i, 2i+1) at NEOX slots (i, i + hd/2)."""
    return np.concatenate([np.arange(0, hd, 2), np.arange(1, hd, 2)])


@pytest.mark.parametrize("hd,theta", [(8, 1e4), (16, 1e6), (64, 1e4)])
def test_interleaved_is_neox_under_the_pair_permutation(hd, theta):
    x = np.random.default_rng(hd).normal(size=(9, 3, hd))
    p = perm(hd)
    y = oracle.rope_rotate_interleaved(x, theta)
    z = oracle.rope_rotate(x[..., p], theta)
    np.testing.assert_allclose(y[..., p], z, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("hd", [4, 32])
def test_interleaved_rotation_properties(hd):
    rng = np.random.default_rng(3)
    x, g = rng.normal(size=(12, 2, hd)), rng.normal(size=(12, 2, hd))
    y = oracle.rope_rotate_interleaved(x, 1e4)
    # norm of every pair preserved
    np.testing.assert_allclose(y[..., 0::2] ** 2 + y[..., 1::2] ** 2, x[..., 0::2] ** 2 + x[..., 1::2] ** 2,
                               rtol=1e-12)
    # the transpose is the adjoint (and the inverse)
    lhs = np.sum(y * g)
    rhs = np.sum(x * oracle.rope_rotate_interleaved_transpose(g, 1e4))
    assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(lhs))
    np.testing.assert_allclose(oracle.rope_rotate_interleaved_transpose(y, 1e4), x, rtol=1e-12, atol=1e-12)
    # relative position: <R_m q, R_n k> depends on n - m only
    q, k = rng.normal(size=hd), rng.normal(size=hd)
    def dot(m, n):
        a = np.zeros((max(m, n) + 1, 1, hd)); a[m, 0] = q
        b = np.zeros((max(m, n) + 1, 1, hd)); b[n, 0] = k
        return np.dot(oracle.rope_rotate_interleaved(a, 1e4)[m, 0], oracle.rope_rotate_interleaved(b, 1e4)[n, 0])
    assert abs(dot(2, 7) - dot(5, 10)) <= 1e-12


def test_attention_with_interleaved_rope_matches_neox_on_permuted_inputs():
    """Scores depend on q.k only, so permuting every Q and K head by the pair
    permutation turns interleaved-RoPE attention into NEOX-RoPE attention with
    the same out and lse; dQ and dK come back permuted, dV unchanged."""
    B, T, NH, NKV, hd = 2, 23, 4, 2, 8
    C = NH * hd
    rng = np.random.default_rng(7)
    qkv = rng.normal(size=(B, T, (NH + 2 * NKV) * hd))
    dout = rng.normal(size=(B, T, C))
    p = perm(hd)
    cols = np.arange(qkv.shape[2])
    for h in range(NH + NKV):                              # Q heads, then K heads
        cols[h * hd:(h + 1) * hd] = h * hd + p
    qkv_p = qkv[..., cols]
    dq_i, aux_i = oracle.attention_backward(qkv, dout, C, NH, NKV, 1e4, return_aux=True, rope_interleaved=True)
    dq_n, aux_n = oracle.attention_backward(qkv_p, dout, C, NH, NKV, 1e4, return_aux=True)
    np.testing.assert_allclose(aux_i["out"], aux_n["out"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(aux_i["lse"], aux_n["lse"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dq_i[..., cols], dq_n, rtol=1e-10, atol=1e-11)
    out_i, lse_i = oracle.attention_forward(qkv, C, NH, NKV, 1e4, rope_interleaved=True)
    np.testing.assert_allclose(out_i, aux_i["out"], rtol=1e-12, atol=1e-13)
