"""Pins of the e4m3 quantization oracle (oracle/e4m3.py) to things other
than itself: the E4M3 format's bit-level definition (every code, every
midpoint), PyTorch's float8_e4m3fn conversion as an independent library
routine, the saturation rule, the per-tile error bound, and inputs whose
quantization is exact (the result must then equal the float64 attention
oracle)."""
import numpy as np
import pytest

import oracle
from oracle.e4m3 import attention_forward_e4m3, e4m3_round, quantize_e4m3, quantize_rows_e4m3


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
    out, lse, vd = attention_forward_e4m3(qkv, C, NH, NKV, 0.0)
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
    out, lse, _ = attention_forward_e4m3(qkv, NH * hd, NH, NKV, 1e4)
    Q, K, V = oracle.split_qkv(qkv, NH * hd, NH, NKV)
    Qd = quantize_rows_e4m3(oracle.rope_rotate(Q, 1e4), 128)
    Kd = quantize_rows_e4m3(oracle.rope_rotate(K, 1e4), 128)
    Vd = quantize_rows_e4m3(V, None)
    qkv_d = np.concatenate([Qd.reshape(B, T, -1), Kd.reshape(B, T, -1), Vd.reshape(B, T, -1)], axis=2)
    ref_out, ref_lse = oracle.attention_forward(qkv_d, NH * hd, NH, NKV, 0.0)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
