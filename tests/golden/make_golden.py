"""Writes the stored expected values under tests/golden/ from the oracle alone.

Run from the repository root:  python tests/golden/make_golden.py

The inputs come from the seeded generator (causal_attention_gqa_gb300.workloads,
which holds no attention arithmetic); every expected value comes from
oracle.attention_backward in float64.  Nothing here runs or reads the CUDA
library.  A change to the oracle's arithmetic that moves these values is made
on purpose: regenerate the fixture in the same commit and name there the
passage of the pages that justifies the change.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from causal_attention_gqa_gb300.workloads import make_inputs, shape_workload  # noqa: E402

# Small GQA case with NEOX RoPE: two batch rows, five positions, two query heads
# sharing one kv head of size 4 (two rotation pairs per head).
CASE = dict(B=2, T=5, C=8, NH=2, NKV=1, rope_theta=1e4, qkv_std=1.0, dout_std=1.0, seed=2024)
PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_gqa_rope_B2_T5.txt")


def arrays():
    w = shape_workload(**CASE)
    qkv, dout = make_inputs(w, "f32")
    dqkv, aux = oracle.attention_backward(qkv.astype(np.float64), dout.astype(np.float64), w.C, w.NH, w.NKV,
                                          w.rope_theta, return_aux=True)
    return w, {"qkv": qkv.astype(np.float64), "dout": dout.astype(np.float64), "out": aux["out"],
               "lse": aux["lse"], "dqkv": dqkv}


def main():
    w, arr = arrays()
    with open(PATH, "w") as f:
        f.write("# Oracle fixture: causal GQA attention with NEOX RoPE, float64 (oracle.attention_backward).\n")
        f.write("# Written by tests/golden/make_golden.py; inputs from the seeded generator, rounded to float32.\n")
        f.write("# case " + " ".join(f"{k}={v}" for k, v in CASE.items()) + "\n")
        f.write("# layout: qkv [B,T,(NH+2NKV)*hd], dout/out [B,T,C], lse [B,NH,T], dqkv [B,T,(NH+2NKV)*hd]\n")
        for name in ("qkv", "dout", "out", "lse", "dqkv"):
            a = arr[name]
            f.write(f"{name} {' '.join(str(n) for n in a.shape)}\n")
            f.write(" ".join(repr(float(x)) for x in a.ravel()) + "\n")


def load():
    """The stored arrays, by name, and the case they were written for."""
    out = {}
    with open(PATH) as f:
        lines = [ln.rstrip("\n") for ln in f if not ln.startswith("#")]
    for head, body in zip(lines[0::2], lines[1::2]):
        name, *shape = head.split()
        out[name] = np.array([float(x) for x in body.split()], dtype=np.float64).reshape([int(s) for s in shape])
    return out


if __name__ == "__main__":
    main()
