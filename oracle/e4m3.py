"""Plain restatement of the e4m3 (FP8) forward's quantization, for tests.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``; never by the product path.

The FP8 forward is not a method of the attention pages; it is this library's
own reduced-precision variant of their forward (scores, causal softmax, PV).
What it computes, step by step:

  1. Q and K are rotated (RoPE, as in the attention oracle) and the rotated
     values are taken in float32, the precision in which the kernels decide
     every 8-bit code.
  2. Every 128-row tile of every Q and K head gets its own scale: with
     a = max |x| over the tile, the codes are e4m3(x * (448 / a)), both the
     quotient and the product rounded to float32, and the tile dequantizes
     with d = float32(a / 448).  A tile of zeros has a = 0 and scale 1.
  3. V keeps one scale per (batch row, kv head), formed the same way from the
     maximum over all rows.
  4. Attention runs exactly (float64) on the dequantized operands code * d.

The kernel also rounds the softmax weights P to e4m3 (as 448 p) before the
PV product; that rounding is not modelled here -- the parity tests bound it.

e4m3 is the OCP 8-bit floating-point format E4M3 (1 sign bit, 4 exponent bits
with bias 7, 3 mantissa bits; no infinities; largest finite 448 = 1.75 * 2^8;
subnormals below 2^-6 with spacing 2^-9).  Conversion rounds to nearest, ties
to even, and saturates finite values beyond 448 to +-448.
"""
from __future__ import annotations

import numpy as np

from .attention import _dims, _head_probs, _rotated_qk, split_qkv

E4M3_MAX = 448.0
_E4M3_MIN_EXP = -6          # exponent of the smallest normal binade
_E4M3_MANT_BITS = 3


def e4m3_round(x) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at +-448.

    Inside binade [2^e, 2^(e+1)) the representable values are spaced
    2^(e-3); below 2^-6 the subnormals keep the spacing of that binade,
    2^-9.  Dividing by the spacing (a power of two, exact) puts the grid on
    the integers, where np.round rounds half to even.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, E = np.frexp(a)                      # a = f * 2^E with f in [0.5, 1)
    e = np.maximum(E - 1, _E4M3_MIN_EXP)    # binade exponent, floored at the normals'
    spacing = np.ldexp(1.0, e - _E4M3_MANT_BITS)
    q = np.round(a / spacing) * spacing
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, x)


def quantize_e4m3(x32: np.ndarray):
    """Codes and dequantization factor of one block of float32 values.

    Returns (codes as float64, d) with codes = e4m3(x * float32(448 / a)) and
    d = float32(a / 448); a = max |x| (scale 1, d = 1 for a block of zeros).
    """
    x32 = np.asarray(x32, dtype=np.float32)
    a = np.float32(np.abs(x32).max()) if x32.size else np.float32(0.0)
    if a > 0:
        scale = np.float32(E4M3_MAX) / a
        d = a / np.float32(E4M3_MAX)
    else:
        scale = np.float32(1.0)
        d = np.float32(1.0)
    codes = e4m3_round((x32 * scale).astype(np.float32))
    return codes, float(d)


def quantize_rows_e4m3(x: np.ndarray, rows_per_tile: int | None) -> np.ndarray:
    """Dequantized e4m3 copy of x [B, T, H, hd]: one scale per (b, h) and
    block of ``rows_per_tile`` rows (all T rows when None)."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    B, T, H, _ = x32.shape
    step = T if rows_per_tile is None else rows_per_tile
    out = np.zeros(x32.shape, dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for t0 in range(0, T, step):
                codes, d = quantize_e4m3(x32[b, t0:t0 + step, h])
                out[b, t0:t0 + step, h] = codes * d
    return out


def attention_forward_e4m3(qkv, C: int, NH: int, NKV: int, rope_theta: float = 0.0,
                           rope_interleaved: bool = False, tile: int = 128):
    """out [B,T,C] and lse [B,NH,T] of exact attention on the e4m3-quantized
    operands: rotated Q and K with one scale per ``tile`` rows of a head, V
    with one scale per (batch row, kv head)."""
    hd, grp, _ = _dims(C, NH, NKV)
    Q, K, V = split_qkv(qkv, C, NH, NKV)
    Qr, Kr = _rotated_qk(Q, K, rope_theta, rope_interleaved)
    Qd = quantize_rows_e4m3(Qr, tile)
    Kd = quantize_rows_e4m3(Kr, tile)
    Vd = quantize_rows_e4m3(V, None)
    B, T = Q.shape[:2]
    scale = 1.0 / np.sqrt(hd)
    out = np.zeros((B, T, C))
    lse = np.zeros((B, NH, T))
    for b in range(B):
        for h in range(NH):
            kh = h // grp
            P, lse[b, h] = _head_probs(Qd[b, :, h], Kd[b, :, kh], scale)
            out[b, :, h * hd:(h + 1) * hd] = P @ Vd[b, :, kh]
    return out, lse, Vd
