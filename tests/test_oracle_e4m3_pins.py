"""Pins of the e4m3 quantization oracle (oracle/e4m3.py) to things other
than itself: the E4M3 format's bit-level definition (every code, every
midpoint), PyTorch's float8_e4m3fn conversion as an independent library
routine, the saturation rule, the per-tile error bound, inputs whose
quantization is exact (the result must then equal the float64 attention
oracle), and for the rounding of the softmax weights: blocks worked by hand
(including the lazy renewal of the row maximum), score gaps that make every
weight exactly representable (the result must then equal exact softmax
attention), the log-sum-exp's independence of the rounding and of the
renewal decisions, and the reporting of weights next to a midpoint."""
import numpy as np
import pytest

import oracle
from oracle.e4m3 import (attention_forward_e4m3, e4m3_round, quantize_e4m3, quantize_rows_e4m3,
                         weighted_row_e4m3)


def decode_e4m3(code: int) -> float:
    """Value of an 8-bit E4M3 code from its fields (NaN for e=15, m=7)."""
    s, e, m = code >> 7, (code >> 3) & 0xF, code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    mag = 2.0 ** (e - 7) * (1.0 + m / 8.0) if e else 2.0 ** -6 * (m / 8.0)
    return -mag if s else mag


POSITIVE = [(c, decode_e4m3(c)) for c in range(0x00, 0x7F)]    # 0 .. 448, code order = value order


def test_every_code_is_a_fixed_point():
    vals = np.array([decode_e4m3(c) for c in range(256) if not np.isnan(decode_e4m3(c))])
    assert vals.size == 254
    np.testing.assert_array_equal(e4m3_round(vals), vals)
    assert max(vals) == 448.0 and min(v for v in vals if v > 0) == 2.0 ** -9


def test_midpoints_round_to_even_code():
    for (c0, v0), (c1, v1) in zip(POSITIVE[:-1], POSITIVE[1:]):
        assert v1 > v0
        want = v0 if c0 % 2 == 0 else v1
        mid = 0.5 * (v0 + v1)
        assert e4m3_round(mid) == want, (c0, v0, v1)
        assert e4m3_round(-mid) == -want
        # just off the midpoint: nearest wins
        assert e4m3_round(mid - (v1 - v0) * 1e-3) == v0
        assert e4m3_round(mid + (v1 - v0) * 1e-3) == v1


def test_saturates_finite_values_beyond_448():
    np.testing.assert_array_equal(e4m3_round([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, -1e6]),
                                  [448.0, 448.0, 448.0, 448.0, 448.0, 448.0, -448.0])


def test_matches_torch_float8_e4m3fn_inside_the_range():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.Generator(np.random.PCG64(4242))
    mag = 2.0 ** rng.uniform(-12.0, np.log2(448.0), size=200_000)
    x = (mag * rng.choice([-1.0, 1.0], size=mag.size)).astype(np.float32)
    mids = np.array([0.5 * (a[1] + b[1]) for a, b in zip(POSITIVE[:-1], POSITIVE[1:])], dtype=np.float32)
    x = np.concatenate([x, mids, -mids, [0.0]]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(e4m3_round(x), want)


def test_block_scale_maps_the_maximum_to_448():
    rng = np.random.Generator(np.random.PCG64(7))
    for amp in (1e-3, 1.0, 37.5, 1e4):
        x = (amp * rng.standard_normal((128, 64))).astype(np.float32)
        codes, d = quantize_e4m3(x)
        assert np.abs(codes).max() == 448.0
        assert d == float(np.float32(np.abs(x).max()) / np.float32(448.0))
    codes, d = quantize_e4m3(np.zeros((128, 8), np.float32))
    assert d == 1.0 and not codes.any()


def test_per_tile_error_bound_with_wildly_different_tiles():
    """Rows 0..127 near 1e-3, rows 128..255 near 1e3: each tile keeps its own
    scale, so every element is within half an e4m3 step of its tile grid:
    |x - xq| <= 2^-4 |x| + 2^-10 a/448 (+ float32 rounding)."""
    rng = np.random.Generator(np.random.PCG64(11))
    x = rng.standard_normal((1, 300, 2, 32))
    x[:, :128] *= 1e-3
    x[:, 128:256] *= 1e3
    xq = quantize_rows_e4m3(x, 128)
    x32 = x.astype(np.float32).astype(np.float64)
    for h in range(2):
        for t0 in (0, 128, 256):
            blk = x32[0, t0:t0 + 128, h]
            a = np.abs(blk).max()
            err = np.abs(blk - xq[0, t0:t0 + 128, h])
            bound = 2.0 ** -4 * np.abs(blk) + 2.0 ** -10 * a / 448.0
            assert (err <= bound * (1 + 1e-6) + 1e-30).all(), (h, t0)
    # one scale per (b, h) over all rows when rows_per_tile is None
    xv = quantize_rows_e4m3(x, None)
    assert np.abs(xv[0, :128] - x32[0, :128]).max() > 1e-3 > np.abs(xq[0, :128] - x32[0, :128]).max()


def _exact_qkv(B, T, NH, NKV, hd, seed):
    """qkv whose e4m3 quantization is exact: every value is an e4m3 value
    times a power of two fixed per 128-row tile of a Q/K head (per kv head
    for V), and each such block holds +-448 times its power of two."""
    rng = np.random.Generator(np.random.PCG64(seed))
    grid = np.array([v for _, v in POSITIVE])
    heads = NH + 2 * NKV
    x = rng.choice(grid, size=(B, T, heads, hd)) * rng.choice([-1.0, 1.0], size=(B, T, heads, hd))
    for b in range(B):
        for h in range(heads):
            if h < NH + NKV:
                for t0 in range(0, T, 128):
                    k = int(rng.integers(-14, -6))
                    x[b, t0:t0 + 128, h] *= 2.0 ** k
                    x[b, t0, h, 0] = 448.0 * 2.0 ** k
            else:
                k = int(rng.integers(-12, -8))
                x[b, :, h] *= 2.0 ** k
                x[b, 0, h, 0] = -448.0 * 2.0 ** k
    return x.reshape(B, T, heads * hd)


@pytest.mark.parametrize("B,T,NH,NKV,hd", [(1, 300, 4, 2, 16), (2, 130, 2, 1, 32)])
def test_exactly_representable_inputs_give_the_float64_attention(B, T, NH, NKV, hd):
    qkv = _exact_qkv(B, T, NH, NKV, hd, seed=B * 1000 + T)
    C = NH * hd
    out, lse, vd = attention_forward_e4m3(qkv, C, NH, NKV, 0.0, round_weights=False)
    ref_out, ref_lse = oracle.attention_forward(qkv, C, NH, NKV, 0.0)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12 * np.abs(ref_out).max())
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    _, _, V = oracle.split_qkv(qkv, C, NH, NKV)
    np.testing.assert_array_equal(vd, V)


def test_rotation_precedes_quantization():
    """With RoPE the codes come from the rotated rows: quantizing the oracle's
    rotated Q/K by hand and running exact attention gives the same result."""
    rng = np.random.Generator(np.random.PCG64(5))
    B, T, NH, NKV, hd = 1, 200, 2, 1, 32
    qkv = rng.standard_normal((B, T, (NH + 2 * NKV) * hd))
    out, lse, _ = attention_forward_e4m3(qkv, NH * hd, NH, NKV, 1e4, round_weights=False)
    Q, K, V = oracle.split_qkv(qkv, NH * hd, NH, NKV)
    Qd = quantize_rows_e4m3(oracle.rope_rotate(Q, 1e4), 128)
    Kd = quantize_rows_e4m3(oracle.rope_rotate(K, 1e4), 128)
    Vd = quantize_rows_e4m3(V, None)
    qkv_d = np.concatenate([Qd.reshape(B, T, -1), Kd.reshape(B, T, -1), Vd.reshape(B, T, -1)], axis=2)
    ref_out, ref_lse = oracle.attention_forward(qkv_d, NH * hd, NH, NKV, 0.0)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ weights
def test_weight_rounding_worked_by_hand():
    """One block, scores (log2 units) 0, -1/2, -1, -9/4 and unit V rows.
    m = 0; 112 * 2^s = 112, 79.196, 56, 23.546.  In e4m3: 112 = 1.75 * 2^6
    exactly; 79.196 lies in [64, 128) where codes are 8 apart -> 80; 56 in
    [32, 64), 4 apart, exact; 23.546 in [16, 32), 2 apart -> 24.  l sums the
    unrounded weights: 270.742; the log-sum-exp (log2) is
    m + log2 l - log2 112 = log2(1 + 2^-1/2 + 2^-1 + 2^-9/4)."""
    s2 = np.array([0.0, -0.5, -1.0, -2.25])
    r = weighted_row_e4m3(s2, np.eye(4))
    np.testing.assert_array_equal(r["o"], [112.0, 80.0, 56.0, 24.0])
    assert abs(r["l"] - (112.0 + 79.19595949289332 + 56.0 + 23.545099627104007)) < 1e-9
    assert r["m"] == 0.0 and r["taken"] == [True]
    lse2 = r["m"] + np.log2(r["l"]) - np.log2(112.0)
    assert abs(lse2 - np.log2(1 + 2 ** -0.5 + 0.5 + 2 ** -2.25)) < 1e-12


def test_row_maximum_is_renewed_only_past_the_threshold():
    """Blocks of two keys, scores [0, -1 | 1.5, 0.5 | 2.5, 0]:
    block 0 sets m = 0 (weights 112, 56); block 1's maximum 1.5 is not more
    than 2 above m, so m stays and its weights are 112 * 2^1.5 = 316.78 -> 320
    ([256, 512), 32 apart) and 112 * 2^0.5 = 158.39 -> 160 ([128, 256), 16
    apart); block 2's maximum 2.5 exceeds m + 2: m becomes 2.5, the partial
    sums shrink by 2^-2.5, and its weights are 112 and 112 * 2^-2.5 = 19.80
    -> 20."""
    s2 = np.array([0.0, -1.0, 1.5, 0.5, 2.5, 0.0])
    r = weighted_row_e4m3(s2, np.eye(6), block=2)
    assert r["taken"] == [True, False, True] and r["m"] == 2.5
    c = 2.0 ** -2.5
    np.testing.assert_allclose(r["o"], [112 * c, 56 * c, 320 * c, 160 * c, 112.0, 20.0], rtol=1e-15)
    l_want = c * (112 + 56 + 112 * 2 ** 1.5 + 112 * 2 ** 0.5) + 112 + 112 * 2 ** -2.5
    assert abs(r["l"] - l_want) < 1e-12 * l_want
    assert np.abs(r["o"]).max() <= 448.0


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_integer_score_gaps_give_exact_softmax(seed):
    """With s - m an integer in [-13, 2], 112 * 2^(s - m) = 7 * 2^(4 + s - m)
    is an e4m3 value (3 mantissa bits suffice for 7; 2^-9 is the smallest
    subnormal step), so nothing is rounded and the walk must reproduce exact
    softmax weights, including across renewals (the scores climb by more
    than 2 in some blocks)."""
    rng = np.random.Generator(np.random.PCG64(100 + seed))
    n, hd = 700, 24
    base = np.repeat(np.arange(0, 3 * ((n + 127) // 128), 3), 128)[:n].astype(float)   # block k tops out at 3k
    s2 = base - rng.integers(0, 11, size=n)
    v = rng.choice(np.array([x for _, x in POSITIVE[1:]]), size=(n, hd)) * rng.choice([-1.0, 1.0], size=(n, hd))
    r = weighted_row_e4m3(s2, v)
    assert r["taken"].count(True) > 1
    w = 2.0 ** (s2 - s2.max())
    want = (w / w.sum()) @ v
    np.testing.assert_allclose(r["o"] / r["l"], want, rtol=0, atol=1e-12 * np.abs(v).max())


def test_log_sum_exp_does_not_depend_on_rounding_or_renewals():
    """l sums unrounded weights, so lse = m + log2 l - log2 112 is the exact
    log-sum-exp of the scores whatever renewal decisions the walk takes; the
    weighted sum itself does depend on them (the weights are rounded at
    different scales)."""
    rng = np.random.Generator(np.random.PCG64(77))
    s2 = rng.normal(0.0, 3.0, size=900)
    v = rng.standard_normal((900, 8))
    want = np.log2(np.sum(2.0 ** (s2 - s2.max()))) + s2.max()
    base = weighted_row_e4m3(s2, v)
    outs = []
    for k in range(1, 8):
        r = weighted_row_e4m3(s2, v, decisions={k: not base["taken"][k]})
        assert abs(r["m"] + np.log2(r["l"]) - np.log2(112.0) - want) < 1e-12
        outs.append(r["o"] / r["l"])
    assert max(np.abs(o - base["o"] / base["l"]).max() for o in outs) > 0


def test_rounded_weights_stay_within_the_e4m3_step_of_exact_attention():
    """Every weight above 2^-6 is rounded with relative error <= 2^-4; below
    that the absolute error is <= 2^-10; l >= 112 (the maximum key
    contributes 112 * 2^0 at least... once m is that key's score), so
    |o/l - exact| <= (2^-4 + n 2^-10 / 112) max|v|."""
    rng = np.random.Generator(np.random.PCG64(9))
    for n in (1, 5, 130, 1000):
        s2 = rng.normal(0.0, 4.0, size=n)
        v = rng.standard_normal((n, 16))
        r = weighted_row_e4m3(s2, v)
        w = 2.0 ** (s2 - s2.max())
        want = (w / w.sum()) @ v
        assert np.abs(r["o"] / r["l"] - want).max() <= (2.0 ** -4 + n * 2.0 ** -10 / 112) * np.abs(v).max()


def test_weights_next_to_a_midpoint_are_reported():
    """84 is the midpoint of the e4m3 neighbours 80 and 88 (ties go to the
    even code, 80): a score whose weight is 84 must be reported as open by
    one code step (8), a weight of exactly 80 (a code) must not."""
    v = np.eye(2)
    s_mid = np.log2(84.0 / 112.0)
    r = weighted_row_e4m3(np.array([0.0, s_mid]), v, ds2=np.full(2, 1e-6))
    assert r["o"][1] == 80.0
    np.testing.assert_allclose(r["o_bound"], [0.0, 8.0])
    r = weighted_row_e4m3(np.array([0.0, np.log2(80.0 / 112.0)]), v, ds2=np.full(2, 1e-6))
    np.testing.assert_array_equal(r["o_bound"], [0.0, 0.0])
    # a block maximum within reach of m + 2 is an open decision
    r = weighted_row_e4m3(np.array([0.0, -1.0, 2.0 + 1e-9, 0.0]), np.eye(4), ds2=np.full(4, 1e-6), block=2)
    assert r["open_blocks"] == [1]


@pytest.mark.parametrize("B,T,NH,NKV,hd,theta", [(1, 300, 4, 2, 16, 0.0), (2, 130, 2, 1, 32, 1e4)])
def test_rounded_forward_keeps_the_exact_lse_and_the_quantized_operands(B, T, NH, NKV, hd, theta):
    """The weight rounding changes out by at most the e4m3 step bound and the
    log-sum-exp not at all (up to float64 rounding): the rounded forward and
    exact attention on the same quantized operands share every lse."""
    rng = np.random.Generator(np.random.PCG64(B + T))
    qkv = rng.standard_normal((B, T, (NH + 2 * NKV) * hd))
    C = NH * hd
    out, lse, vd = attention_forward_e4m3(qkv, C, NH, NKV, theta)
    out_x, lse_x, vd_x = attention_forward_e4m3(qkv, C, NH, NKV, theta, round_weights=False)
    np.testing.assert_array_equal(vd, vd_x)
    np.testing.assert_allclose(lse, lse_x, rtol=0, atol=1e-11)
    d = np.abs(out - out_x).max() / np.abs(vd).max()
    assert 0 < d <= 2.0 ** -4 + T * 2.0 ** -10 / 112
