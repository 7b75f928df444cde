"""Seeded synthetic workloads for causal MHA/GQA attention.

This module only *generates inputs*: shapes, value distributions and seeds.
It holds none of the attention arithmetic, so both the CUDA path and the
double-precision oracle can draw the very same inputs from it.

The five workloads mirror the attention shapes of the trainers on the source
pages:

* ``microgpt_tiny``      -- "CUDA C microgpt" (microgpt.cu): N_EMBD 16, 4 heads
                            of size 4, block 16.
* ``qwen2_single_head``  -- "nx_f32_qwen2_train_gate.nx source": one head of
                            size 16, NEOX RoPE with base 1e6, up to 64 positions.
* ``gpt2_124m_mha``      -- the GPT-2 trainer quoted on "@possumtech/rummy
                            2.1.0 -> 2.2.0" (C=768, 12 heads, packed 3C qkv).
* ``gqa_block``          -- a GQA block (16 query heads sharing 4 KV heads,
                            head size 128, NEOX RoPE 1e6), the grouped layout of
                            "nanoeuler -- CUDA kernels" at a realistic size.
* ``long_context_gqa``   -- the same block at T=8192 with 32/8 heads.

Values are drawn from a NumPy PCG64 generator (stable across machines) as
float32 normals; bf16 workloads round those float32 values once to bf16
(round-to-nearest-even), and the oracle consumes the rounded values.
Distribution "N(0, s)" means standard deviation ``s``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    C: int
    NH: int
    NKV: int
    rope_theta: float      # <= 0 disables RoPE
    dtypes: tuple          # element types the workload runs in ("f32", "bf16")
    qkv_std: float
    dout_std: float
    seed: int

    @property
    def hd(self) -> int:
        return self.C // self.NH

    @property
    def qkv_width(self) -> int:
        return (self.NH + 2 * self.NKV) * self.hd

    @property
    def causal_pairs(self) -> int:
        return self.T * (self.T + 1) // 2

    def flops_fwd(self) -> float:
        """Algorithmic causal forward FLOPs: QK^T and PV over the causal pairs."""
        return 4.0 * self.B * self.NH * self.hd * self.causal_pairs

    def flops_bwd(self) -> float:
        """Algorithmic backward FLOPs: five GEMM-equivalents (S, dP, dV, dK, dQ)."""
        return 2.5 * self.flops_fwd()

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("microgpt_tiny", 1, 16, 16, 4, 4, 0.0, ("f32",), 1.0, 1.0, 1001),
        Workload("qwen2_single_head", 4, 64, 16, 1, 1, 1e6, ("f32",), 1.0, 1.0, 1002),
        Workload("gpt2_124m_mha", 8, 1024, 768, 12, 12, 0.0, ("f32", "bf16"), 0.5, 1e-2, 1003),
        Workload("gqa_block", 4, 2048, 2048, 16, 4, 1e6, ("bf16",), 1.0, 1e-2, 1004),
        Workload("long_context_gqa", 1, 8192, 4096, 32, 8, 1e6, ("bf16",), 1.0, 1e-2, 1005),
    ]
}

WORKLOAD_ORDER = list(WORKLOADS)


def shape_workload(B, T, C, NH, NKV, rope_theta=0.0, qkv_std=1.0, dout_std=1.0,
                   seed=7, name: Optional[str] = None) -> Workload:
    """An ad-hoc workload (parity sweeps over odd shapes)."""
    return Workload(name or f"B{B}_T{T}_C{C}_NH{NH}_NKV{NKV}", B, T, C, NH, NKV,
                    float(rope_theta), ("f32", "bf16"), qkv_std, dout_std, seed)


def rank_shard(w: Workload, rank: int, world: int) -> Workload:
    """Rank ``rank``'s share of a data-parallel job over ``world`` ranks: the
    batch rows rank*B .. rank*B + B - 1 of a global batch of world*B rows.

    Batch rows are independent problems (no term of the method couples two of
    them), so each rank draws its own rows from its own seed -- the workload's
    seed plus 7919 * rank, shard 0 being the workload itself -- and the global
    batch is the concatenation of the shards in rank order.
    """
    if not 0 <= rank < world:
        raise ValueError("rank must lie in [0, world)")
    return w if rank == 0 else w.replace(seed=w.seed + 7919 * rank)


def make_inputs(w: Workload, dtype: str = "f32"):
    """Return (qkv, dout) as float32 NumPy arrays, already rounded to ``dtype``.

    qkv has shape [B, T, (NH + 2*NKV)*hd] (Q | K | V column blocks per row),
    dout has shape [B, T, C].  For ``dtype == "bf16"`` the float32 draw is
    rounded to bf16 and widened back, so the values are exactly what a bf16
    tensor holds.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed))
    qkv = rng.standard_normal((w.B, w.T, w.qkv_width), dtype=np.float32)
    qkv *= np.float32(w.qkv_std)
    dout = rng.standard_normal((w.B, w.T, w.C), dtype=np.float32)
    dout *= np.float32(w.dout_std)
    if dtype == "bf16":
        qkv = round_to_bf16(qkv)
        dout = round_to_bf16(dout)
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype!r}")
    return qkv, dout


def make_decode_inputs(B, NH, NKV, hd, max_len, dtype="bf16", seed=11, std=1.0):
    """Seeded single-query (decode) inputs: q [B,NH,hd], k_cache and v_cache
    [B,max_len,NKV,hd], float32 arrays already rounded to ``dtype``; N(0, std)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal((B, NH, hd), dtype=np.float32) * np.float32(std)
    k = rng.standard_normal((B, max_len, NKV, hd), dtype=np.float32) * np.float32(std)
    v = rng.standard_normal((B, max_len, NKV, hd), dtype=np.float32) * np.float32(std)
    if dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype!r}")
    return q, k, v


def make_proj_inputs(M, Cm, N, seed=13):
    """Seeded QKV-projection inputs, bf16-rounded float32 arrays: x [M, Cm]
    ~ N(0, 1) and w [N, Cm] ~ N(0, 1/Cm) (so the projection is ~ N(0, 1))."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((M, Cm), dtype=np.float32)
    w = rng.standard_normal((N, Cm), dtype=np.float32) * np.float32(1.0 / np.sqrt(Cm))
    return round_to_bf16(x), round_to_bf16(w)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def sample_rows(T: int, count: int, seed: int) -> np.ndarray:
    """Seeded, sorted, distinct row indices in [0, T); always includes 0 and T-1."""
    rng = np.random.Generator(np.random.PCG64(seed))
    picks = rng.choice(T, size=min(count, T), replace=False)
    return np.unique(np.concatenate([picks, [0, T - 1]])).astype(np.int64)
