"""Shared helpers for the GPU parity tests: run the CUDA library through its
C ABI on seeded inputs and measure the normalised error against the oracle."""
import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_err(x, ref) -> float:
    """max |x - ref| / max |ref| (the normalised error metric of the parity bars)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = np.abs(ref).max()
    return float(np.abs(x - ref).max() / (denom if denom > 0 else 1.0))


def to_device(a, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device="cuda", dtype=torch.bfloat16 if dtype == "bf16" else torch.float32)


def to_numpy(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_gpu(lib, w, qkv_np, dout_np, dtype, backward=True, fwd_ws=False):
    """Forward (and backward) through the C ABI; returns numpy float64 arrays.
    fwd_ws: run the forward through attn_fwd_ws (pre-rotated Q/K) instead of
    attn_fwd, and the backward through attn_bwd_rot on the forward's rotated
    copy instead of attn_bwd."""
    import torch
    qkv = to_device(qkv_np, dtype)
    dout = to_device(dout_np, dtype)
    if fwd_ws:
        # The benchmark's configuration: attn_fwd_ws, then attn_bwd_rot reusing
        # the forward's rotated Q/K.
        out, lse, fws = lib.forward_ws(qkv, w.NH, w.NKV, w.rope_theta)
    else:
        out, lse = lib.forward(qkv, w.NH, w.NKV, w.rope_theta)
        fws = None
    res = {"out": out, "lse": lse}
    if backward:
        res["dqkv"] = lib.backward(qkv, out, dout, lse, w.NH, w.NKV, w.rope_theta, qk_rot=fws)
    torch.cuda.synchronize()
    return {k: to_numpy(v) for k, v in res.items()}
