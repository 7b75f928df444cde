"""Pins for the double-precision oracle (CPU only).

Each test ties the oracle to something other than itself: a closed form, a
worked example derived by hand, an invariant of the method, an independent
library routine (PyTorch's causal scaled-dot-product attention and autograd
in float64), high-precision brute force, or central finite differences.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.attention import rope_rot_matrix
from causal_attention_gqa_gb300.workloads import WORKLOADS, make_inputs, shape_workload

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rand_qkv(B, T, C, NH, NKV, seed=0, std=1.0):
    hd = C // NH
    rng = np.random.default_rng(seed)
    return rng.normal(0, std, size=(B, T, (NH + 2 * NKV) * hd))


# ---------------------------------------------------------------- layout
def test_packed_layout_columns():
    B, T, C, NH, NKV = 1, 3, 8, 4, 2
    hd = C // NH
    width = (NH + 2 * NKV) * hd
    qkv = np.tile(np.arange(width, dtype=np.float64), (B, T, 1))
    Q, K, V = oracle.split_qkv(qkv, C, NH, NKV)
    for h in range(NH):
        assert np.array_equal(Q[0, 0, h], h * hd + np.arange(hd))
    for kh in range(NKV):
        assert np.array_equal(K[0, 0, kh], C + kh * hd + np.arange(hd))
        assert np.array_equal(V[0, 0, kh], C + NKV * hd + kh * hd + np.arange(hd))


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("NH,NKV,theta", [(4, 4, 0.0), (4, 2, 1e6), (8, 1, 1e4)])
def test_single_position_returns_v(NH, NKV, theta):
    """T = 1: the only probability is exactly 1, so out = V bit for bit, and
    lse = q.k / sqrt(hd) (RoPE is the identity at position 0)."""
    B, T, hd = 3, 1, 8
    C = NH * hd
    qkv = rand_qkv(B, T, C, NH, NKV, seed=1)
    out, lse = oracle.attention_forward(qkv, C, NH, NKV, theta)
    Q, K, V = oracle.split_qkv(qkv, C, NH, NKV)
    grp = NH // NKV
    for b in range(B):
        for h in range(NH):
            assert np.array_equal(out[b, 0, h * hd:(h + 1) * hd], V[b, 0, h // grp])
            ref = math.fsum(Q[b, 0, h] * K[b, 0, h // grp]) / math.sqrt(hd)
            assert abs(lse[b, h, 0] - ref) <= 1e-14 * max(1.0, abs(ref))


@pytest.mark.parametrize("theta", [0.0, 1e6])
def test_zero_queries_give_causal_prefix_means(theta):
    """Q = 0: every allowed score is 0, so out_t = mean(V_0..V_t) and
    lse_t = ln(t + 1), with or without RoPE."""
    B, T, C, NH, NKV = 2, 23, 16, 4, 2
    hd = C // NH
    qkv = rand_qkv(B, T, C, NH, NKV, seed=2)
    qkv[:, :, :C] = 0.0
    out, lse = oracle.attention_forward(qkv, C, NH, NKV, theta)
    _, _, V = oracle.split_qkv(qkv, C, NH, NKV)
    counts = np.arange(1, T + 1, dtype=np.float64)
    for b in range(B):
        for h in range(NH):
            prefix = np.cumsum(V[b, :, h // (NH // NKV)], axis=0) / counts[:, None]
            np.testing.assert_allclose(out[b, :, h * hd:(h + 1) * hd], prefix,
                                       rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse[b, h], np.log(counts), rtol=1e-14, atol=1e-14)


def test_worked_example_two_positions():
    """A two-token, one-head example derived by hand.

    q0=(1,0) k0=(1,0) v0=(1,2); q1=(0,2) k1=(0,1) v1=(3,-1); hd=2 so the
    scale is 1/sqrt(2).  Row 0 sees only key 0: out0 = v0, lse0 = 1/sqrt(2).
    Row 1: s10 = 0, s11 = 2/sqrt(2) = sqrt(2), so
    out1 = (v0 + e^sqrt2 v1) / (1 + e^sqrt2), lse1 = ln(1 + e^sqrt2).
    """
    qkv = np.array([[[1.0, 0.0, 1.0, 0.0, 1.0, 2.0],
                     [0.0, 2.0, 0.0, 1.0, 3.0, -1.0]]])
    out, lse = oracle.attention_forward(qkv, C=2, NH=1, NKV=1)
    e = math.exp(math.sqrt(2.0))
    np.testing.assert_allclose(out[0, 0], [1.0, 2.0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[0, 1], [(1 + 3 * e) / (1 + e), (2 - e) / (1 + e)],
                               rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0, 0], 1 / math.sqrt(2.0), rtol=1e-15)
    np.testing.assert_allclose(lse[0, 0, 1], math.log(1 + e), rtol=1e-15)


def test_lse_matches_high_precision_bruteforce():
    """lse against log(sum(exp(s))) evaluated with 50-digit mpmath (no max
    subtraction), plus the bounds max_s <= lse_t <= max_s + ln(t+1)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    B, T, C, NH, NKV = 1, 9, 8, 2, 1
    hd = C // NH
    qkv = rand_qkv(B, T, C, NH, NKV, seed=3, std=2.0)
    _, lse = oracle.attention_forward(qkv, C, NH, NKV)
    Q, K, _ = oracle.split_qkv(qkv, C, NH, NKV)
    for h in range(NH):
        for t in range(T):
            scores = [mpmath.fsum(mpmath.mpf(a) * mpmath.mpf(c) for a, c in zip(Q[0, t, h], K[0, s, 0]))
                      / mpmath.sqrt(hd) for s in range(t + 1)]
            ref = mpmath.log(mpmath.fsum(mpmath.exp(x) for x in scores))
            assert abs(lse[0, h, t] - float(ref)) <= 1e-14 * max(1.0, abs(float(ref)))
            mx = float(max(scores))
            assert mx - 1e-12 <= lse[0, h, t] <= mx + math.log(t + 1) + 1e-12


# ---------------------------------------------------------------- invariants
def test_causality_perturbation():
    """Changing every value at position t' leaves all rows t < t' bit-identical."""
    B, T, C, NH, NKV = 2, 20, 16, 4, 2
    qkv = rand_qkv(B, T, C, NH, NKV, seed=4)
    out, lse = oracle.attention_forward(qkv, C, NH, NKV, 1e6)
    tp = 11
    qkv2 = qkv.copy()
    qkv2[:, tp, :] += np.random.default_rng(5).normal(size=qkv.shape[2])
    out2, lse2 = oracle.attention_forward(qkv2, C, NH, NKV, 1e6)
    assert np.array_equal(out[:, :tp], out2[:, :tp])
    assert np.array_equal(lse[:, :, :tp], lse2[:, :, :tp])
    assert not np.allclose(out[:, tp], out2[:, tp])


@pytest.mark.parametrize("grp", [2, 4])
def test_gqa_equals_replicated_mha(grp):
    """GQA with grp query heads per KV head equals MHA on K/V replicated per
    query head; the GQA dK/dV are the MHA dK/dV summed over each group."""
    B, T, NKV, hd = 2, 13, 2, 4
    NH = NKV * grp
    C = NH * hd
    rng = np.random.default_rng(6)
    qkv = rand_qkv(B, T, C, NH, NKV, seed=7)
    dout = rng.normal(size=(B, T, C))
    Q, K, V = oracle.split_qkv(qkv, C, NH, NKV)
    Km = np.repeat(K, grp, axis=2)
    Vm = np.repeat(V, grp, axis=2)
    qkv_m = oracle.attention.pack_qkv(Q, Km, Vm)
    for theta in (0.0, 1e6):
        o_g, l_g = oracle.attention_forward(qkv, C, NH, NKV, theta)
        o_m, l_m = oracle.attention_forward(qkv_m, C, NH, NH, theta)
        np.testing.assert_allclose(o_g, o_m, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(l_g, l_m, rtol=1e-14, atol=1e-14)
        d_g = oracle.attention_backward(qkv, dout, C, NH, NKV, theta)
        d_m = oracle.attention_backward(qkv_m, dout, C, NH, NH, theta)
        dq_g, dk_g, dv_g = oracle.split_qkv(d_g, C, NH, NKV)
        dq_m, dk_m, dv_m = oracle.split_qkv(d_m, C, NH, NH)
        np.testing.assert_allclose(dq_g, dq_m, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(dk_g, dk_m.reshape(B, T, NKV, grp, hd).sum(3), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dv_g, dv_m.reshape(B, T, NKV, grp, hd).sum(3), rtol=1e-12, atol=1e-13)


def test_backward_sum_invariants():
    """Without RoPE: sum_s dK_s = 0 for every KV head (each row of dS sums to
    0), and sum_s dV_s = sum over t and over the group's heads of dO_t (each
    row of P sums to 1)."""
    B, T, C, NH, NKV = 2, 31, 32, 8, 2
    hd, grp = C // NH, NH // NKV
    qkv = rand_qkv(B, T, C, NH, NKV, seed=8)
    dout = np.random.default_rng(9).normal(size=(B, T, C))
    dqkv = oracle.attention_backward(qkv, dout, C, NH, NKV)
    _, dK, dV = oracle.split_qkv(dqkv, C, NH, NKV)
    scale = np.abs(dK).max()
    np.testing.assert_allclose(dK.sum(axis=1), 0.0, atol=1e-13 * scale * T)
    dO = dout.reshape(B, T, NKV, grp, hd).sum(axis=3).sum(axis=1)
    np.testing.assert_allclose(dV.sum(axis=1), dO, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- RoPE
def test_rope_identity_at_position_zero():
    x = np.random.default_rng(10).normal(size=(1, 1, 3, 16))
    assert np.array_equal(oracle.rope_rotate(x, 1e6), x)


def test_rope_closed_form_values():
    """hd = 2: pair (x0, x1) at position t turns by angle t (frequency
    theta^0 = 1).  hd = 4, theta = 1e6: the second pair (x1, x3) turns by
    t * 1e6^(-1/2) = t / 1000."""
    t = 3
    x = np.zeros((t + 1, 1, 2))
    x[t, 0] = [0.7, -1.3]
    y = oracle.rope_rotate(x, 1e6)[t, 0]
    c, s = math.cos(t), math.sin(t)
    np.testing.assert_allclose(y, [0.7 * c + 1.3 * s, -1.3 * c + 0.7 * s], rtol=1e-15)
    t = 1234
    x = np.zeros((t + 1, 1, 4))
    x[t, 0] = [0.5, 2.0, -1.0, 0.25]
    y = oracle.rope_rotate(x, 1e6)[t, 0]
    a0, a1 = float(t), t / 1000.0
    expect = [0.5 * math.cos(a0) + 1.0 * math.sin(a0),
              2.0 * math.cos(a1) - 0.25 * math.sin(a1),
              -1.0 * math.cos(a0) + 0.5 * math.sin(a0),
              0.25 * math.cos(a1) + 2.0 * math.sin(a1)]
    np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-15)


def test_rope_rot_matrix_is_rotate_half():
    x = np.arange(1.0, 9.0)
    assert np.array_equal(x @ rope_rot_matrix(8), [-5, -6, -7, -8, 1, 2, 3, 4])


def test_rope_preserves_pair_norms_and_is_orthogonal():
    rng = np.random.default_rng(11)
    T, H, hd = 50, 3, 16
    x = rng.normal(size=(T, H, hd))
    y = oracle.rope_rotate(x, 1e4)
    half = hd // 2
    np.testing.assert_allclose(x[..., :half] ** 2 + x[..., half:] ** 2,
                               y[..., :half] ** 2 + y[..., half:] ** 2, rtol=1e-13)
    np.testing.assert_allclose(oracle.rope_rotate_transpose(y, 1e4), x, rtol=1e-13, atol=1e-13)
    g = rng.normal(size=x.shape)
    lhs = np.sum(y * g)
    rhs = np.sum(x * oracle.rope_rotate_transpose(g, 1e4))
    assert abs(lhs - rhs) <= 1e-12 * abs(lhs)


def test_rope_relative_position_property():
    """<R_m q, R_n k> depends only on n - m."""
    rng = np.random.default_rng(12)
    hd = 8
    q, k = rng.normal(size=hd), rng.normal(size=hd)
    T = 40
    xs = np.zeros((T, 1, hd))
    ys = np.zeros((T, 1, hd))
    xs[:, 0] = q
    ys[:, 0] = k
    Rq = oracle.rope_rotate(xs, 1e6)[:, 0]
    Rk = oracle.rope_rotate(ys, 1e6)[:, 0]
    for m, n, s in [(3, 7, 10), (0, 5, 20), (12, 2, 25)]:
        assert abs(Rq[m] @ Rk[n] - Rq[m + s] @ Rk[n + s]) < 1e-12


# ---------------------------------------------------------------- library routine
@pytest.mark.parametrize("B,T,C,NH,NKV", [(2, 37, 32, 4, 2), (1, 19, 24, 3, 3), (1, 8, 32, 8, 1)])
def test_against_torch_sdpa_float64(B, T, C, NH, NKV):
    """No RoPE: the oracle's out and dqkv equal PyTorch's causal
    scaled_dot_product_attention and its autograd, both in float64."""
    torch = pytest.importorskip("torch")
    hd, grp = C // NH, NH // NKV
    qkv = rand_qkv(B, T, C, NH, NKV, seed=13)
    dout = np.random.default_rng(14).normal(size=(B, T, C))
    Q, K, V = (torch.tensor(a, requires_grad=True) for a in oracle.split_qkv(qkv, C, NH, NKV))
    q = Q.permute(0, 2, 1, 3)
    k = K.permute(0, 2, 1, 3).repeat_interleave(grp, dim=1)
    v = V.permute(0, 2, 1, 3).repeat_interleave(grp, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    o = o.permute(0, 2, 1, 3).reshape(B, T, C)
    (o * torch.tensor(dout)).sum().backward()
    out, _ = oracle.attention_forward(qkv, C, NH, NKV)
    np.testing.assert_allclose(out, o.detach().numpy(), rtol=1e-12, atol=1e-13)
    dqkv = oracle.attention_backward(qkv, dout, C, NH, NKV)
    dq, dk, dv = oracle.split_qkv(dqkv, C, NH, NKV)
    np.testing.assert_allclose(dq, Q.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, K.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, V.grad.numpy(), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- finite differences
def _fd_check(qkv, dout, C, NH, NKV, theta, entries, tol):
    dqkv = oracle.attention_backward(qkv, dout, C, NH, NKV, theta)
    fd = np.zeros(len(entries))
    for n, idx in enumerate(entries):
        x0 = qkv[idx]
        h = 1e-5 * max(1.0, abs(x0))
        qkv[idx] = x0 + h
        lp = np.sum(dout * oracle.attention_forward(qkv, C, NH, NKV, theta)[0])
        qkv[idx] = x0 - h
        lm = np.sum(dout * oracle.attention_forward(qkv, C, NH, NKV, theta)[0])
        qkv[idx] = x0
        fd[n] = (lp - lm) / (2 * h)
    an = np.array([dqkv[idx] for idx in entries])
    err = np.abs(fd - an).max() / np.abs(an).max()
    assert err < tol, err


def test_finite_differences_microgpt_tiny_every_entry():
    """Central differences of L = sum(dout * out) against every one of the
    768 qkv entries of the microgpt-shaped workload."""
    w = WORKLOADS["microgpt_tiny"]
    qkv, dout = (a.astype(np.float64) for a in make_inputs(w))
    entries = [tuple(i) for i in np.ndindex(*qkv.shape)]
    assert len(entries) == 768
    _fd_check(qkv, dout, w.C, w.NH, w.NKV, w.rope_theta, entries, 1e-7)


def test_finite_differences_qwen2_rope_sampled():
    """Same on the single-head RoPE workload, 256 seeded entries."""
    w = WORKLOADS["qwen2_single_head"]
    qkv, dout = (a.astype(np.float64) for a in make_inputs(w))
    rng = np.random.default_rng(15)
    flat = rng.choice(qkv.size, size=256, replace=False)
    entries = [np.unravel_index(f, qkv.shape) for f in flat]
    _fd_check(qkv, dout, w.C, w.NH, w.NKV, w.rope_theta, entries, 1e-7)


def test_finite_differences_gqa_rope_sampled():
    """GQA (grp 2) with RoPE and a ragged length, 200 seeded entries."""
    w = shape_workload(2, 21, 32, 4, 2, rope_theta=1e6, seed=16)
    qkv, dout = (a.astype(np.float64) for a in make_inputs(w))
    rng = np.random.default_rng(17)
    flat = rng.choice(qkv.size, size=200, replace=False)
    entries = [np.unravel_index(f, qkv.shape) for f in flat]
    _fd_check(qkv, dout, w.C, w.NH, w.NKV, w.rope_theta, entries, 1e-7)


# ---------------------------------------------------------------- sampled mode
def test_sampled_mode_equals_full_oracle():
    B, T, C, NH, NKV = 2, 70, 32, 4, 2
    hd, grp = C // NH, NH // NKV
    qkv = rand_qkv(B, T, C, NH, NKV, seed=18)
    dout = np.random.default_rng(19).normal(size=(B, T, C))
    theta = 1e6
    dqkv, aux = oracle.attention_backward(qkv, dout, C, NH, NKV, theta, return_aux=True)
    dq, dk, dv = oracle.split_qkv(dqkv, C, NH, NKV)
    qr = np.array([0, 5, 33, 69])
    kr = np.array([0, 1, 40, 69])
    groups = [(0, 1), (1, 0)]
    s = oracle.attention_sampled(qkv, dout, C, NH, NKV, theta, qr, groups, kr, row_block=16)
    np.testing.assert_allclose(s["out_rows"], aux["out"][:, qr], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s["lse_rows"], aux["lse"][:, :, qr], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s["dq_rows"], dq[:, qr], rtol=1e-11, atol=1e-13)
    for (b, kh) in groups:
        np.testing.assert_allclose(s["dk_rows"][(b, kh)], dk[b, kr, kh], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(s["dv_rows"][(b, kh)], dv[b, kr, kh], rtol=1e-11, atol=1e-13)


def test_key_shift_and_value_scale_invariances():
    """Without RoPE, adding one vector c to every key adds q.c/sqrt(hd) to all
    scores of a query row: the softmax (so out) is unchanged and lse shifts by
    q.c/sqrt(hd).  Scaling V by a scales out by a and leaves lse alone."""
    rng = np.random.default_rng(17)
    B, T, NH, NKV, hd = 2, 9, 4, 2, 8
    C = NH * hd
    qkv = rng.normal(size=(B, T, (NH + 2 * NKV) * hd))
    out, lse = oracle.attention_forward(qkv, C, NH, NKV, 0.0)
    c = rng.normal(size=hd)
    shifted = qkv.copy()
    for kh in range(NKV):
        shifted[:, :, C + kh * hd:C + (kh + 1) * hd] += c
    out_s, lse_s = oracle.attention_forward(shifted, C, NH, NKV, 0.0)
    np.testing.assert_allclose(out_s, out, rtol=0, atol=1e-12)
    Q, _, _ = oracle.split_qkv(qkv, C, NH, NKV)
    want = lse + np.einsum("bthd,d->bht", Q, c) / np.sqrt(hd)
    np.testing.assert_allclose(lse_s, want, rtol=0, atol=1e-12)
    scaled = qkv.copy()
    scaled[:, :, C + NKV * hd:] *= -2.5
    out_v, lse_v = oracle.attention_forward(scaled, C, NH, NKV, 0.0)
    np.testing.assert_allclose(out_v, -2.5 * out, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(lse_v, lse)
