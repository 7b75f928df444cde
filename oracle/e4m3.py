"""Plain restatement of the e4m3 (FP8) forward, for tests.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``; never by the product path.

The FP8 forward is not a method of the attention pages; it is this library's
own reduced-precision variant of their forward ("nanoeuler -- CUDA kernels",
attention_forward_kernel: scores, causal softmax, PV).  What it computes,
step by step:

  1. Q and K are rotated (RoPE, as in the attention oracle) and the rotated
     values are taken in float32, the precision in which the kernels decide
     every 8-bit code.
  2. Every 128-row tile of every Q and K head gets its own scale: with
     a = max |x| over the tile, the codes are e4m3(x * (448 / a)), both the
     quotient and the product rounded to float32, and the tile dequantizes
     with d = float32(a / 448).  A tile of zeros has a = 0 and scale 1.
  3. V keeps one scale per (batch row, kv head), formed the same way from the
     maximum over all rows.
  4. Scores of the dequantized operands, s = q . k / sqrt(hd), are taken in
     log2 units (times log2 e).  Each query row walks its visible keys in
     blocks of 128 (the kernel's key tiles, in order).  A running maximum m
     starts at the first block's maximum and is renewed -- the partial sums
     rescaled by 2^(m_old - m_new) -- only when a block's maximum exceeds it
     by more than 2; so every weight 2^(s - m) is at most 4.  The weight used
     in the PV product is rounded to e4m3 as P8 = e4m3(112 * 2^(s - m))
     (112 * 4 = 448, the largest finite code); the normaliser l sums the
     unrounded 112 * 2^(s - m).
  5. out = (sum_j P8_j V8_j) * d_v / l with V8 the V codes, and
     lse = (m + log2 l - log2 112) ln 2, the natural-log log-sum-exp.

Where the kernel takes a decision in float32 that this float64 restatement
can only locate up to the float32 rounding of its inputs -- a weight or an
operand that lies within that rounding of an e4m3 midpoint, a block maximum
within it of the renewal threshold -- ``weighted_row_e4m3`` reports the
decision as open (both outcomes are correct results of the method), and the
parity tests accept either outcome.

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
P_SCALE = 112.0             # weights are stored as e4m3(112 * 2^(s - m)); 112 * 4 = 448
RESCALE_THRESHOLD = 2.0     # log2 units: m is renewed only when exceeded by more than this
KEY_BLOCK = 128             # keys per block of the row walk (the kernel's key tile)
LOG2E = 1.4426950408889634


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


def weighted_row_e4m3(s2, vcodes, ds2=None, decisions=None, block: int = KEY_BLOCK,
                      threshold: float = RESCALE_THRESHOLD, pscale: float = P_SCALE):
    """Step 4 for one query row: the e4m3-weighted sum of its V codes.

    s2      : float64 scores of the row's visible keys (key 0 first), log2 units.
    vcodes  : [n, hd] e4m3 codes of those keys' V rows.
    ds2     : optional per-key bound on how far a float32 evaluation of s2
              may lie from this one (log2 units); when given, the row also
              reports what float32 may decide either way (a weight's exponent
              s - m moves by its own key's reach plus that of m).
    decisions : optional {block index: bool} that replaces the renewal decision
              of those blocks (to follow the other outcome of an open
              decision); the other blocks decide as usual.

    Returns a dict: o [hd] = sum P8_j vcodes_j (rescaled to the final m),
    l = sum of the unrounded weights, m (log2 units), taken = the renewal
    decision of every block, o_abs [hd] = sum P8_j |vcodes_j| (the scale of
    the accumulation's rounding); with ds2 also o_bound [hd] (how far o may
    move when weights near an e4m3 midpoint round the other way), l_bound
    (how far l may move), open_blocks = blocks whose maximum lies within
    reach of the renewal threshold.
    """
    s2 = np.asarray(s2, dtype=np.float64)
    v = np.asarray(vcodes, dtype=np.float64)
    n, hd = v.shape
    o = np.zeros(hd)
    o_abs = np.zeros(hd)
    l = 0.0
    m = -np.inf
    taken, open_blocks = [], []
    o_bound = np.zeros(hd)
    l_bound = 0.0
    for k, j0 in enumerate(range(0, n, block)):
        sb = s2[j0:j0 + block]
        mb = sb.max()
        renew = bool(mb > m + threshold)
        if ds2 is not None and k > 0:
            # float32 forms the block maximum and the comparison with its own
            # rounding: a maximum this close to m + threshold may go either way
            reach = ds2[j0:j0 + block].max() + ds2[:j0].max()
            if abs(mb - (m + threshold)) <= reach:
                open_blocks.append(k)
        if decisions is not None and k > 0 and k in decisions:
            renew = bool(decisions[k])
        taken.append(renew)
        if renew:
            c = 2.0 ** (m - mb) if np.isfinite(m) else 0.0
            o *= c
            o_abs *= c
            l *= c
            o_bound *= c
            l_bound *= c
            m = mb
        p = pscale * 2.0 ** (sb - m)
        p8 = e4m3_round(p)
        l += p.sum()
        o += p8 @ v[j0:j0 + block]
        o_abs += p8 @ np.abs(v[j0:j0 + block])
        if ds2 is not None:
            # s - m moves by the reach of s and by that of m (the score of a
            # key seen so far)
            db = ds2[j0:j0 + block] + ds2[:j0 + sb.size].max()
            lo = e4m3_round(p * 2.0 ** (-db))
            hi = e4m3_round(p * 2.0 ** db)
            dev = np.maximum(hi - p8, p8 - lo)          # > 0 only next to a midpoint
            o_bound += dev @ np.abs(v[j0:j0 + block])
            l_bound += (p * (2.0 ** db - 1.0)).sum()
    res = {"o": o, "l": l, "m": m, "taken": taken, "o_abs": o_abs}
    if ds2 is not None:
        res.update({"o_bound": o_bound, "l_bound": l_bound, "open_blocks": open_blocks})
    return res


def _qk_codes(x64: np.ndarray, tile: int):
    """Codes and per-tile dequantization factors of a rotated Q or K [B,T,H,hd]
    (float64 values, taken in float32): codes [B,T,H,hd], d [B,H,n_tiles]."""
    x32 = x64.astype(np.float32)
    B, T, H, hd = x32.shape
    n_t = (T + tile - 1) // tile
    codes = np.zeros(x32.shape)
    d = np.ones((B, H, n_t))
    for b in range(B):
        for h in range(H):
            for i, t0 in enumerate(range(0, T, tile)):
                c, dd = quantize_e4m3(x32[b, t0:t0 + tile, h])
                codes[b, t0:t0 + tile, h] = c
                d[b, h, i] = dd
    return codes, d


def _code_reach(x64: np.ndarray, pair_norm: np.ndarray, rel_angle: float, tile: int):
    """How far a dequantized rotated Q/K element may lie from the oracle's
    when the rotation is computed with an angle error of up to `rel_angle`
    radians (absolute error rel_angle * |pair| per element, on top of float32
    rounding): the codes of the perturbed inputs under the perturbed tile
    maximum, taken in float32 like every code.  Returns u [B,T,H,hd] >= 0."""
    x32 = x64.astype(np.float32).astype(np.float64)
    B, T, H, hd = x32.shape
    u = np.zeros(x32.shape)
    if rel_angle == 0.0:
        # no rotation: both sides quantize the very same float32 values with
        # the same float32 arithmetic, so every code agrees
        return u
    ex = rel_angle * pair_norm + np.abs(x32) * 2.0 ** -23
    for b in range(B):
        for h in range(H):
            for t0 in range(0, T, tile):
                xs = x32[b, t0:t0 + tile, h]
                es = ex[b, t0:t0 + tile, h]
                a = np.abs(xs).max()
                if a == 0.0 and es.max() == 0.0:
                    continue
                c, d = quantize_e4m3(xs.astype(np.float32))
                val = c * d
                ea = es[np.unravel_index(np.argmax(np.abs(xs)), xs.shape)] + es.max()
                worst = np.zeros_like(xs)
                for sa in (-1.0, 1.0):
                    a2 = max(a + sa * ea, 1e-300)
                    scale = E4M3_MAX / a2
                    d2 = a2 / E4M3_MAX
                    for sx in (-1.0, 1.0):
                        y = (xs + sx * es) * scale * (1.0 + sx * 2.0 ** -22)
                        worst = np.maximum(worst, np.abs(e4m3_round(y) * d2 - val))
                u[b, t0:t0 + tile, h] = worst
    return u


def _pair_norms(x: np.ndarray, interleaved: bool) -> np.ndarray:
    """|(x_i, x_partner)| for every element of [..., hd]: the rotation moves
    each element by at most its pair's norm times the angle error."""
    hd = x.shape[-1]
    if interleaved:
        n = np.sqrt(x[..., 0::2] ** 2 + x[..., 1::2] ** 2)
        return np.repeat(n, 2, axis=-1)
    half = hd // 2
    n = np.sqrt(x[..., :half] ** 2 + x[..., half:] ** 2)
    return np.concatenate([n, n], axis=-1)


def attention_forward_e4m3(qkv, C: int, NH: int, NKV: int, rope_theta: float = 0.0,
                           rope_interleaved: bool = False, tile: int = 128, round_weights: bool = True,
                           rows=None, angle_error: float | None = None, mma_rel: float = 2.0 ** -23):
    """out [B,T,C], lse [B,NH,T] and the dequantized V of the e4m3 forward.

    round_weights=True follows steps 1-5 (the weights rounded to e4m3 as
    P8 = e4m3(112 * 2^(s - m)) with the lazily renewed row maximum);
    round_weights=False is exact softmax attention on the dequantized
    operands (steps 1-3 only).

    rows: optional query positions to evaluate (others stay zero).
    angle_error: when given (radians; 0 without RoPE), also returns a dict of
    per-row reach for the parity bars: for every evaluated (b, h, t) the
    bound on how far float32 evaluation may move o and l (see
    weighted_row_e4m3), the open renewal decisions, and the results of
    the other outcome of each open decision.
    mma_rel: relative rounding of one tensor-core accumulation step (a K=32
    slice added to the float32 accumulator), applied to the sum of the
    magnitudes it adds, for the score reach and the "o_acc" bound.
    """
    hd, grp, _ = _dims(C, NH, NKV)
    Q, K, V = split_qkv(qkv, C, NH, NKV)
    Qr, Kr = _rotated_qk(Q, K, rope_theta, rope_interleaved)
    B, T = Q.shape[:2]
    scale = 1.0 / np.sqrt(hd)
    out = np.zeros((B, T, C))
    lse = np.zeros((B, NH, T))
    if not round_weights:
        Qd = quantize_rows_e4m3(Qr, tile)
        Kd = quantize_rows_e4m3(Kr, tile)
        Vd = quantize_rows_e4m3(V, None)
        for b in range(B):
            for h in range(NH):
                kh = h // grp
                P, lse[b, h] = _head_probs(Qd[b, :, h], Kd[b, :, kh], scale)
                out[b, :, h * hd:(h + 1) * hd] = P @ Vd[b, :, kh]
        return out, lse, Vd
    qc, qdq = _qk_codes(Qr, tile)
    kc, kdq = _qk_codes(Kr, tile)
    tix = np.arange(T) // tile
    Qd = qc * qdq.transpose(0, 2, 1)[:, tix][..., None]          # [B,T,NH,hd]
    Kd = kc * kdq.transpose(0, 2, 1)[:, tix][..., None]          # [B,T,NKV,hd]
    vc = np.zeros(V.shape)
    dv = np.ones((B, NKV))
    for b in range(B):
        for kh in range(NKV):
            vc[b, :, kh], dv[b, kh] = quantize_e4m3(V[b, :, kh].astype(np.float32))
    Vd = vc * dv[:, None, :, None]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    reach = None
    if angle_error is not None:
        uq = _code_reach(Qr, _pair_norms(Qr, rope_interleaved), angle_error, tile)
        uk = _code_reach(Kr, _pair_norms(Kr, rope_interleaved), angle_error, tile)
        reach = {"o_bound": np.zeros((B, T, C)), "o_acc": np.zeros((B, T, C)), "l_rel": np.zeros((B, NH, T)), "s_reach": np.zeros((B, NH, T)),
                 "open": {}}
    for b in range(B):
        for h in range(NH):
            kh = h // grp
            for t in rows:
                s2 = (Kd[b, :t + 1, kh] @ Qd[b, t, h]) * scale * LOG2E
                ds2 = None
                if reach is not None:
                    # float32 scores, maxima and exponents: a few ulps of the
                    # magnitudes involved; the operands' own reach from the
                    # rotation (zero without RoPE).
                    mag = np.abs(s2).max()
                    sabs = (np.abs(Kd[b, :t + 1, kh]) @ np.abs(Qd[b, t, h])) * scale * LOG2E
                    ds2 = 8.0 * 2.0 ** -24 * (np.abs(s2) + mag + 8.0) + 2.0 ** -21 + mma_rel * (hd // 32) * sabs
                    ds2 = ds2 + mma_rel * (hd // 32) * sabs.max()
                    ds2 = ds2 + scale * LOG2E * (np.abs(Kd[b, :t + 1, kh]) @ uq[b, t, h]
                                                 + uk[b, :t + 1, kh] @ (np.abs(Qd[b, t, h]) + uq[b, t, h]))
                r = weighted_row_e4m3(s2, vc[b, :t + 1, kh], ds2)
                out[b, t, h * hd:(h + 1) * hd] = r["o"] * dv[b, kh] / r["l"]
                lse[b, h, t] = (r["m"] + np.log2(r["l"]) - np.log2(P_SCALE)) * np.log(2.0)
                if reach is not None:
                    reach["o_bound"][b, t, h * hd:(h + 1) * hd] = r["o_bound"] * dv[b, kh] / r["l"]
                    n_acc = (t + 1 + 31) // 32
                    reach["o_acc"][b, t, h * hd:(h + 1) * hd] = mma_rel * n_acc * r["o_abs"] * dv[b, kh] / r["l"]
                    reach["l_rel"][b, h, t] = r["l_bound"] / r["l"]
                    reach["s_reach"][b, h, t] = ds2.max()
                    if r["open_blocks"]:
                        alts = []
                        for k in r["open_blocks"][:3]:
                            ra = weighted_row_e4m3(s2, vc[b, :t + 1, kh], ds2, decisions={k: not r["taken"][k]})
                            alts.append((ra["o"] * dv[b, kh] / ra["l"], ra["o_bound"] * dv[b, kh] / ra["l"],
                                         ra["l_bound"] / ra["l"]))
                        reach["open"][(b, h, int(t))] = alts
    if reach is not None:
        return out, lse, Vd, reach
    return out, lse, Vd
