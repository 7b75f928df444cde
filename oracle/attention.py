"""Plain double-precision restatement of causal MHA/GQA self-attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.

What the method computes (for every batch row b, query head h, position t,
with hd = C/NH, grp = NH/NKV and kv head kh = floor(h / grp)):

  1. RoPE (optional, NEOX form): q = R_t Q[b,t,h], k_s = R_s K[b,s,kh]; V is
     not rotated.  ("nx_f32_qwen2_train_gate.nx source": build_rope builds the
     COS/SIN tables with inverse frequency exp(-2i ln(theta)/D) and the ROT
     matrix; rope_node forms x*COS + (x ROT)*SIN; the Qwen2 block applies it to
     Q and K only.)
  2. Scores s_ts = q . k_s / sqrt(hd) for s <= t, a causal mask for s > t.
     ("nanoeuler -- CUDA kernels", "Causal multi-head attention with GQA":
     scale 1/sqrt(hs), kv head h/(NH/NKV), packed Q | K | V column blocks with
     row width C + 2*NKV*hs.)
  3. Row softmax P_ts = exp(s_ts - m_t) / l_t, and the log-sum-exp
     lse_t = m_t + ln(l_t) of the scaled scores.  (Same page: the forward
     kernel declaration writes `lse` next to `out`; its buffer has B*NH*T
     floats per layer.)
  4. out_t = sum_s P_ts V_s, written at columns h*hd .. (h+1)*hd of out[b,t].
  5. Backward for an upstream gradient dO = dout[b,t,h]:
       dP_ts = dO_t . V_s,   D_t = sum_s P_ts dP_ts = dO_t . O_t
       ("CUDA C microgpt": attention_backward_kernel's weighted_sum),
       dS_ts = P_ts (dP_ts - D_t)  (the softmax Jacobian written out in
       "nanoeuler"'s attention_backward_kernel and in the quoted GPT-2
       attention_backward),
       dq_t = scale sum_s dS_ts k_s,  dk_s = scale sum_t dS_ts q_t,
       dv_s = sum_t P_ts dO_t, with dk and dv summed over the grp query heads
       that share kv head kh ("nanoeuler": atomicAdd into the shared dk/dv).
  6. With RoPE the gradients are carried back through the rotation:
     dQ = R_t^T dq, dK = R_s^T dk ("nanoeuler" runs rope_kernel with
     inverse=1 on dqkv after the attention backward).

Everything is float64 NumPy; the only library primitive used as a step is the
matrix product.  There is no tiling, no online softmax and no fusion: the
full T x T score matrix of a head is formed, masked and normalised as written
above.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Packed QKV layout ("nanoeuler -- CUDA kernels", causal GQA attention section)
# --------------------------------------------------------------------------
def _dims(C: int, NH: int, NKV: int):
    if C % NH or NH % NKV:
        raise ValueError("C must be a multiple of NH and NH of NKV")
    hd = C // NH
    return hd, NH // NKV, (NH + 2 * NKV) * hd


def split_qkv(qkv: np.ndarray, C: int, NH: int, NKV: int):
    """Split packed qkv [B, T, C + 2*NKV*hd] into float64 Q, K, V.

    Q[b,t,h] = qkv[b,t,h*hd:(h+1)*hd], K[b,t,kh] starts at column C + kh*hd,
    V[b,t,kh] at column C + NKV*hd + kh*hd.
    Returns Q [B,T,NH,hd], K [B,T,NKV,hd], V [B,T,NKV,hd].
    """
    hd, _, width = _dims(C, NH, NKV)
    x = np.asarray(qkv, dtype=np.float64)
    B, T, W = x.shape
    if W != width:
        raise ValueError(f"qkv row width {W} != (NH + 2*NKV)*hd = {width}")
    Q = x[:, :, :C].reshape(B, T, NH, hd)
    K = x[:, :, C:C + NKV * hd].reshape(B, T, NKV, hd)
    V = x[:, :, C + NKV * hd:].reshape(B, T, NKV, hd)
    return Q.copy(), K.copy(), V.copy()


def pack_qkv(dQ, dK, dV) -> np.ndarray:
    """Inverse of split_qkv: [B,T,NH,hd], [B,T,NKV,hd] x2 -> [B,T,width]."""
    B, T = dQ.shape[:2]
    return np.concatenate(
        [dQ.reshape(B, T, -1), dK.reshape(B, T, -1), dV.reshape(B, T, -1)], axis=2)


# --------------------------------------------------------------------------
# NEOX RoPE ("nx_f32_qwen2_train_gate.nx source": build_rope, rope_node)
# --------------------------------------------------------------------------
def rope_cos_sin(positions, hd: int, theta: float):
    """Full-width COS/SIN tables [len(positions), hd] for the given positions.

    For pair index i < hd/2 the inverse frequency is exp(-2 i ln(theta) / hd)
    (= theta^(-2i/hd)) and the angle at position t is t * inv_freq_i; columns
    i and i + hd/2 carry the same value, as in build_rope.
    """
    if hd % 2:
        raise ValueError("RoPE needs an even head size")
    half = hd // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = np.exp(-2.0 * i * np.log(float(theta)) / hd)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos = np.concatenate([np.cos(ang), np.cos(ang)], axis=1)
    sin = np.concatenate([np.sin(ang), np.sin(ang)], axis=1)
    return cos, sin


def rope_rot_matrix(hd: int) -> np.ndarray:
    """The rotate-half matrix ROT of build_rope: (x ROT)_k = -x_{k+hd/2} for
    k < hd/2 and x_{k-hd/2} for k >= hd/2."""
    half = hd // 2
    rot = np.zeros((hd, hd), dtype=np.float64)
    for k in range(half):
        rot[k + half, k] = -1.0
    for k in range(half, hd):
        rot[k - half, k] = 1.0
    return rot


def rope_rotate(x: np.ndarray, theta: float, positions=None) -> np.ndarray:
    """y = x*COS + (x ROT)*SIN over the last axis (rope_node).

    ``x`` has shape [..., T, H, hd] (axis -3 is the position) unless
    ``positions`` is given, in which case axis -3 indexes those positions.
    """
    x = np.asarray(x, dtype=np.float64)
    T, hd = x.shape[-3], x.shape[-1]
    pos = np.arange(T) if positions is None else np.asarray(positions)
    cos, sin = rope_cos_sin(pos, hd, theta)
    rot = rope_rot_matrix(hd)
    cos = cos[:, None, :]
    sin = sin[:, None, :]
    return x * cos + (x @ rot) * sin


def rope_rotate_transpose(g: np.ndarray, theta: float, positions=None) -> np.ndarray:
    """Adjoint of rope_rotate: with y = x M, M = diag(COS) + ROT diag(SIN),
    the gradient is g M^T = g*COS + (g*SIN) ROT^T."""
    g = np.asarray(g, dtype=np.float64)
    T, hd = g.shape[-3], g.shape[-1]
    pos = np.arange(T) if positions is None else np.asarray(positions)
    cos, sin = rope_cos_sin(pos, hd, theta)
    rot = rope_rot_matrix(hd)
    cos = cos[:, None, :]
    sin = sin[:, None, :]
    return g * cos + (g * sin) @ rot.T


def rope_rotate_interleaved(x: np.ndarray, theta: float, positions=None) -> np.ndarray:
    """The interleaved (GPT-J) form of "nanoeuler -- CUDA kernels",
    rope_kernel: pair (2i, 2i+1) of each head turns by angle t * freq_i with
    freq_i = theta^(-2i/hd):
        y[2i]   = x[2i] cos - x[2i+1] sin,
        y[2i+1] = x[2i] sin + x[2i+1] cos.
    Axis -3 is the position (or indexes ``positions``), the last axis hd."""
    x = np.asarray(x, dtype=np.float64)
    T, hd = x.shape[-3], x.shape[-1]
    pos = np.arange(T) if positions is None else np.asarray(positions)
    i = np.arange(hd // 2, dtype=np.float64)
    freq = float(theta) ** (-2.0 * i / hd)
    ang = pos.astype(np.float64)[:, None] * freq[None, :]          # [T, hd/2]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * cos - x1 * sin
    y[..., 1::2] = x0 * sin + x1 * cos
    return y


def rope_rotate_interleaved_transpose(g: np.ndarray, theta: float, positions=None) -> np.ndarray:
    """Inverse (transposed) interleaved rotation, rope_kernel's inverse=1:
        y[2i] = g[2i] cos + g[2i+1] sin,  y[2i+1] = -g[2i] sin + g[2i+1] cos."""
    g = np.asarray(g, dtype=np.float64)
    T, hd = g.shape[-3], g.shape[-1]
    pos = np.arange(T) if positions is None else np.asarray(positions)
    i = np.arange(hd // 2, dtype=np.float64)
    freq = float(theta) ** (-2.0 * i / hd)
    ang = pos.astype(np.float64)[:, None] * freq[None, :]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    g0, g1 = g[..., 0::2], g[..., 1::2]
    y = np.empty_like(g)
    y[..., 0::2] = g0 * cos + g1 * sin
    y[..., 1::2] = -g0 * sin + g1 * cos
    return y


def _rope_fns(interleaved: bool):
    if interleaved:
        return rope_rotate_interleaved, rope_rotate_interleaved_transpose
    return rope_rotate, rope_rotate_transpose


def _rotated_qk(Q, K, rope_theta, interleaved=False):
    if rope_theta and rope_theta > 0:
        rot, _ = _rope_fns(interleaved)
        return rot(Q, rope_theta), rot(K, rope_theta)
    return Q, K


# --------------------------------------------------------------------------
# Softmax attention of one head, written out in full
# --------------------------------------------------------------------------
def _head_probs(q, k, scale, rows=None):
    """Causal softmax of the scaled scores of one head.

    q [R, hd] are the query rows at positions ``rows`` (all T positions when
    None), k [T, hd] all keys.  Returns (P [R, T], lse [R]).
    """
    T = k.shape[0]
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    S = scale * (q @ k.T)
    allowed = np.arange(T)[None, :] <= rows[:, None]          # key s <= query t
    S = np.where(allowed, S, -np.inf)
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])                                 # masked -> 0
    l = E.sum(axis=1)
    return E / l[:, None], m + np.log(l)


def attention_forward(qkv, C: int, NH: int, NKV: int, rope_theta: float = 0.0, rope_interleaved: bool = False):
    """out [B,T,C] and lse [B,NH,T] (natural log of the scaled scores), float64.
    rope_interleaved selects the interleaved (GPT-J) pairing instead of NEOX."""
    hd, grp, _ = _dims(C, NH, NKV)
    Q, K, V = split_qkv(qkv, C, NH, NKV)
    Qr, Kr = _rotated_qk(Q, K, rope_theta, rope_interleaved)
    B, T = Q.shape[:2]
    scale = 1.0 / np.sqrt(hd)
    out = np.zeros((B, T, C))
    lse = np.zeros((B, NH, T))
    for b in range(B):
        for h in range(NH):
            kh = h // grp
            P, lse[b, h] = _head_probs(Qr[b, :, h], Kr[b, :, kh], scale)
            out[b, :, h * hd:(h + 1) * hd] = P @ V[b, :, kh]
    return out, lse


def attention_backward(qkv, dout, C: int, NH: int, NKV: int, rope_theta: float = 0.0,
                       return_aux: bool = False, rope_interleaved: bool = False):
    """Gradient of L = sum(dout * out) with respect to the packed qkv, float64.

    Returns dqkv [B, T, (NH + 2*NKV)*hd]; with ``return_aux`` also a dict with
    out, lse and D (= rowsum(dO * O), [B,NH,T]).
    """
    hd, grp, _ = _dims(C, NH, NKV)
    Q, K, V = split_qkv(qkv, C, NH, NKV)
    Qr, Kr = _rotated_qk(Q, K, rope_theta, rope_interleaved)
    dO_all = np.asarray(dout, dtype=np.float64)
    B, T = Q.shape[:2]
    scale = 1.0 / np.sqrt(hd)
    dq = np.zeros_like(Q)
    dk = np.zeros_like(K)
    dv = np.zeros_like(V)
    out = np.zeros((B, T, C))
    lse = np.zeros((B, NH, T))
    Dsum = np.zeros((B, NH, T))
    for b in range(B):
        for h in range(NH):
            kh = h // grp
            q, k, v = Qr[b, :, h], Kr[b, :, kh], V[b, :, kh]
            P, lse[b, h] = _head_probs(q, k, scale)
            O = P @ v
            out[b, :, h * hd:(h + 1) * hd] = O
            dO = dO_all[b, :, h * hd:(h + 1) * hd]
            dP = dO @ v.T
            D = np.sum(dO * O, axis=1)
            Dsum[b, h] = D
            dS = P * (dP - D[:, None])
            dq[b, :, h] = scale * (dS @ k)
            dk[b, :, kh] += scale * (dS.T @ q)
            dv[b, :, kh] += P.T @ dO
    if rope_theta and rope_theta > 0 and rope_interleaved:
        dq = rope_rotate_interleaved_transpose(dq, rope_theta)
        dk = rope_rotate_interleaved_transpose(dk, rope_theta)
    elif rope_theta and rope_theta > 0:
        dq = rope_rotate_transpose(dq, rope_theta)
        dk = rope_rotate_transpose(dk, rope_theta)
    dqkv = pack_qkv(dq, dk, dv)
    if return_aux:
        return dqkv, {"out": out, "lse": lse, "D": Dsum}
    return dqkv


def attention_sampled(qkv, dout, C: int, NH: int, NKV: int, rope_theta: float,
                      q_rows, kv_groups, k_rows, row_block: int = 1024):
    """Sampled oracle for sequences too long to form every T x T matrix at once.

    * For every (b, h): out, lse and dQ at the query positions ``q_rows``
      (each needs only its own score row).
    * For each (b, kh) in ``kv_groups``: dK and dV at the key positions
      ``k_rows``; those sum over every query t >= s of every head in the
      group, so all rows of those heads are formed, ``row_block`` rows at a
      time.

    Returns a dict: out_rows [B,R,C], lse_rows [B,NH,R], dq_rows [B,R,NH,hd]
    (pre-rotation gradient, i.e. w.r.t. the packed qkv), and dk_rows /
    dv_rows {(b, kh): [Rk, hd]}.
    """
    hd, grp, _ = _dims(C, NH, NKV)
    Q, K, V = split_qkv(qkv, C, NH, NKV)
    Qr, Kr = _rotated_qk(Q, K, rope_theta)
    dO_all = np.asarray(dout, dtype=np.float64)
    B, T = Q.shape[:2]
    scale = 1.0 / np.sqrt(hd)
    q_rows = np.asarray(q_rows)
    k_rows = np.asarray(k_rows)
    R = len(q_rows)
    out_rows = np.zeros((B, R, C))
    lse_rows = np.zeros((B, NH, R))
    dq_rows = np.zeros((B, R, NH, hd))
    for b in range(B):
        for h in range(NH):
            kh = h // grp
            q, k, v = Qr[b, q_rows, h], Kr[b, :, kh], V[b, :, kh]
            P, lse_rows[b, h] = _head_probs(q, k, scale, rows=q_rows)
            O = P @ v
            out_rows[b, :, h * hd:(h + 1) * hd] = O
            dO = dO_all[b, q_rows, h * hd:(h + 1) * hd]
            dS = P * ((dO @ v.T) - np.sum(dO * O, axis=1)[:, None])
            dq_rows[b, :, h] = scale * (dS @ k)
    if rope_theta and rope_theta > 0:
        dq_rows = rope_rotate_transpose(dq_rows, rope_theta, positions=q_rows)

    dk_rows, dv_rows = {}, {}
    for (b, kh) in kv_groups:
        k, v = Kr[b, :, kh], V[b, :, kh]
        dk_acc = np.zeros((len(k_rows), hd))
        dv_acc = np.zeros((len(k_rows), hd))
        for h in range(kh * grp, (kh + 1) * grp):
            for t0 in range(0, T, row_block):
                rows = np.arange(t0, min(T, t0 + row_block))
                q = Qr[b, rows, h]
                P, _ = _head_probs(q, k, scale, rows=rows)
                O = P @ v
                dO = dO_all[b, rows, h * hd:(h + 1) * hd]
                dS = P * ((dO @ v.T) - np.sum(dO * O, axis=1)[:, None])
                dk_acc += scale * (dS[:, k_rows].T @ q)
                dv_acc += P[:, k_rows].T @ dO
        if rope_theta and rope_theta > 0:
            dk_acc = rope_rotate_transpose(dk_acc[:, None, :], rope_theta,
                                           positions=k_rows)[:, 0, :]
        dk_rows[(b, kh)] = dk_acc
        dv_rows[(b, kh)] = dv_acc
    return {"out_rows": out_rows, "lse_rows": lse_rows, "dq_rows": dq_rows,
            "dk_rows": dk_rows, "dv_rows": dv_rows}


# --------------------------------------------------------------------------
# Single-query (decode) attention over a KV cache
# --------------------------------------------------------------------------
def attention_decode(q, k_cache, v_cache, seq_lens):
    """One new query per batch row against the cached keys and values.

    The per-position form of the forward ("CUDA C microgpt",
    attention_forward_kernel: one query at position pos_id against the keys
    0 .. pos_id), with the grouped heads of "nanoeuler -- CUDA kernels"
    (query head h reads kv head h / (NH/NKV)).

    q [B, NH, hd]: the new token's queries, already rotated at its position
    when RoPE is in use.  k_cache, v_cache [B, Lmax, NKV, hd]: keys (already
    rotated at their positions) and values of positions 0 .. Lmax-1.
    seq_lens [B], 1 <= len <= Lmax: the query attends to cache rows
    0 .. len-1 (its own key and value included).

    Returns out [B, NH, hd] and lse [B, NH] (natural log of the sum of the
    exponentials of the scaled scores), float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    B, NH, hd = q.shape
    NKV = k_cache.shape[2]
    grp = NH // NKV
    scale = 1.0 / np.sqrt(hd)
    out = np.zeros((B, NH, hd))
    lse = np.zeros((B, NH))
    for b in range(B):
        n = int(seq_lens[b])
        for h in range(NH):
            kh = h // grp
            s = scale * (k_cache[b, :n, kh] @ q[b, h])     # scores of the n visible keys
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            out[b, h] = (e / l) @ v_cache[b, :n, kh]
            lse[b, h] = m + np.log(l)
    return out, lse


# --------------------------------------------------------------------------
# QKV projection feeding the attention (for the fused projection epilogue)
# --------------------------------------------------------------------------
def qkv_projection(x, w, T: int, NH: int, NKV: int, rope_theta: float = 0.0, rope_interleaved: bool = False):
    """The packed QKV projection of the trainers on the pages ("nanoeuler --
    CUDA kernels": qkv = x W_qkv, row width C + 2 NKV hs, followed by the RoPE
    passes over the Q and K column blocks).

    x [M, Cm] (M = B*T rows, row m at position m % T), w [N, Cm] with
    N = (NH + 2*NKV)*hd (output column n of the packed Q | K | V layout reads
    row n of w).  Returns (qkv [M, N], qk_rot [M, (NH+NKV)*hd]): the
    unrotated projection, and its Q and K heads rotated at their positions
    (columns in the natural order of each head), float64.
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    M = x.shape[0]
    N = w.shape[0]
    hd = N // (NH + 2 * NKV)
    qkv = x @ w.T
    qk = qkv[:, :(NH + NKV) * hd].reshape(M // T, T, NH + NKV, hd)
    if rope_theta and rope_theta > 0:
        rot, _ = _rope_fns(rope_interleaved)
        qk = rot(qk, rope_theta)
    return qkv, qk.reshape(M, (NH + NKV) * hd)
