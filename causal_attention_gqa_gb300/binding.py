"""Python binding of the C ABI in ``include/attn_gb300.h`` (ctypes).

Argument marshalling only: every step of the attention runs in the CUDA
library.  PyTorch supplies device memory and streams.  If the shared library
has not been built this module raises on first use; there is no fallback.

The entry points keep the C names and argument order:

    attn_fwd(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype, stream=None)
    attn_fwd_workspace_bytes(B, T, C, NH, NKV, dtype)
    attn_fwd_ws(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype,
                workspace, workspace_bytes, stream=None)
    attn_bwd_workspace_bytes(B, T, C, NH, NKV, dtype)
    attn_bwd(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype,
             workspace, workspace_bytes, stream=None)
    attn_bwd_rot(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype,
                 qk_rot, workspace, workspace_bytes, stream=None)

Tensor arguments may be torch tensors (their data pointers are passed) or
raw integer addresses.  ``stream`` defaults to PyTorch's current stream.
A non-zero status raises AttnError.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

DTYPE_F32 = 0
DTYPE_TF32 = 1
DTYPE_BF16 = 2
FLAG_ROPE_INTERLEAVED = 0x100   # OR-ed into dtype: GPT-J (interleaved) RoPE pairing

_STATUS_NAMES = {
    0: "ATTN_OK", -1: "ATTN_ERR_NULL_POINTER", -2: "ATTN_ERR_BAD_SHAPE", -3: "ATTN_ERR_UNSUPPORTED",
    -4: "ATTN_ERR_MISALIGNED", -5: "ATTN_ERR_WORKSPACE", -6: "ATTN_ERR_CUDA",
    -7: "ATTN_ERR_DEVICE_TIMEOUT", -8: "ATTN_ERR_BAD_ARGUMENT",
}


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, status)} ({attn_strerror(status)})")


_lib = None


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"CUDA attention library not found at {LIB_PATH}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.attn_fwd.restype = i
    lib.attn_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.attn_fwd_workspace_bytes.restype = sz
    lib.attn_fwd_ws.argtypes = [vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
    lib.attn_fwd_ws.restype = i
    lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.attn_bwd_workspace_bytes.restype = sz
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd_rot.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, sz, vp]
    lib.attn_bwd_rot.restype = i
    lib.attn_strerror.argtypes = [i]
    lib.attn_strerror.restype = ctypes.c_char_p
    lib.attn_device_status.argtypes = [ctypes.POINTER(i), i]
    lib.attn_device_status.restype = i
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_longlong, ctypes.POINTER(i)]
    lib.attn_selftest_wait_timeout.restype = i
    lib.attn_abi_version.argtypes = []
    lib.attn_abi_version.restype = i
    lib.attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.attn_qkv_proj.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.attn_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i, i, i]
    lib.attn_fwd_fp8_workspace_bytes.restype = sz
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
    lib.attn_fwd_fp8.restype = i
    lib.attn_qkv_proj.restype = i
    lib.attn_fwd_rot.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.attn_fwd_rot.restype = i
    lib.attn_decode_workspace_bytes.restype = sz
    lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, sz, vp]
    lib.attn_decode.restype = i
    lib.attn_bwd_noalloc.restype = i
    lib.attn_profile_start.argtypes = []
    lib.attn_profile_start.restype = i
    lib.attn_profile_stop.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i), i]
    lib.attn_profile_stop.restype = i
    lib.attn_kernel_name.argtypes = [i]
    lib.attn_kernel_name.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise ValueError("tensor arguments must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != 0:
        raise AttnError(status, where)


def attn_strerror(status: int) -> str:
    return load().attn_strerror(int(status)).decode()


def attn_abi_version() -> int:
    return load().attn_abi_version()


def attn_fwd(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype, stream=None) -> None:
    st = load().attn_fwd(_ptr(out), _ptr(lse), _ptr(qkv), B, T, C, NH, NKV, float(rope_theta), int(dtype),
                         _stream(stream))
    _check(st, "attn_fwd")


def attn_fwd_workspace_bytes(B, T, C, NH, NKV, dtype) -> int:
    return int(load().attn_fwd_workspace_bytes(B, T, C, NH, NKV, int(dtype)))


def attn_fwd_ws(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype, workspace, workspace_bytes, stream=None) -> None:
    st = load().attn_fwd_ws(_ptr(out), _ptr(lse), _ptr(qkv), B, T, C, NH, NKV, float(rope_theta), int(dtype),
                            _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "attn_fwd_ws")


def attn_bwd_workspace_bytes(B, T, C, NH, NKV, dtype) -> int:
    return int(load().attn_bwd_workspace_bytes(B, T, C, NH, NKV, int(dtype)))


def attn_bwd(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype, workspace, workspace_bytes,
             stream=None) -> None:
    st = load().attn_bwd(_ptr(dqkv), _ptr(qkv), _ptr(out), _ptr(dout), _ptr(lse), B, T, C, NH, NKV,
                         float(rope_theta), int(dtype), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "attn_bwd")


def attn_bwd_rot(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype, qk_rot, workspace, workspace_bytes,
                 stream=None) -> None:
    """attn_bwd reading the RoPE-rotated Q/K from the forward's attn_fwd_ws workspace `qk_rot`."""
    st = load().attn_bwd_rot(_ptr(dqkv), _ptr(qkv), _ptr(out), _ptr(dout), _ptr(lse), B, T, C, NH, NKV,
                             float(rope_theta), int(dtype), _ptr(qk_rot), _ptr(workspace), int(workspace_bytes),
                             _stream(stream))
    _check(st, "attn_bwd_rot")


def attn_fwd_fp8_workspace_bytes(B, T, C, NH, NKV, dtype) -> int:
    return int(load().attn_fwd_fp8_workspace_bytes(B, T, C, NH, NKV, int(dtype)))


def attn_fwd_fp8(out, lse, qkv, B, T, C, NH, NKV, rope_theta, dtype, workspace, workspace_bytes, stream=None) -> None:
    st = load().attn_fwd_fp8(_ptr(out), _ptr(lse), _ptr(qkv), B, T, C, NH, NKV, float(rope_theta), int(dtype),
                             _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "attn_fwd_fp8")


def forward_fp8(qkv, NH: int, NKV: int, rope_theta: float = 0.0, rope_interleaved: bool = False, stream=None):
    """(out, lse) of the e4m3 forward (attn_fwd_fp8) on a bf16 qkv."""
    import torch
    B, T, W = qkv.shape
    hd = W // (NH + 2 * NKV)
    C = NH * hd
    code = DTYPE_BF16 | (FLAG_ROPE_INTERLEAVED if rope_interleaved else 0)
    nbytes = attn_fwd_fp8_workspace_bytes(B, T, C, NH, NKV, code)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=qkv.device)
    out = torch.empty((B, T, C), dtype=qkv.dtype, device=qkv.device)
    lse = torch.empty((B, NH, T), dtype=torch.float32, device=qkv.device)
    attn_fwd_fp8(out, lse, qkv, B, T, C, NH, NKV, rope_theta, code, ws, ws.numel(), stream)
    return out, lse


def attn_qkv_proj(qkv, qk_rot, x, w, B, T, Cm, NH, NKV, hd, rope_theta, flags=0, stream=None) -> None:
    st = load().attn_qkv_proj(_ptr(qkv), _ptr(qk_rot), _ptr(x), _ptr(w), B, T, Cm, NH, NKV, hd, float(rope_theta),
                              int(flags), _stream(stream))
    _check(st, "attn_qkv_proj")


def attn_fwd_rot(out, lse, qkv, qk_rot, B, T, C, NH, NKV, rope_theta, dtype, stream=None) -> None:
    st = load().attn_fwd_rot(_ptr(out), _ptr(lse), _ptr(qkv), _ptr(qk_rot), B, T, C, NH, NKV, float(rope_theta),
                             int(dtype), _stream(stream))
    _check(st, "attn_fwd_rot")


def qkv_proj(x, w, T: int, NH: int, NKV: int, rope_theta: float = 0.0, rope_interleaved: bool = False,
             stream=None):
    """(qkv, qk_rot) = the QKV projection of x [B*T, Cm] by w [(NH+2NKV)*hd, Cm]
    (bf16) and the rotated Q/K copy (None when rope_theta <= 0)."""
    import torch
    M, Cm = x.shape
    N = w.shape[0]
    hd = N // (NH + 2 * NKV)
    qkv = torch.empty((M // T, T, N), dtype=torch.bfloat16, device=x.device)
    rot = None
    if rope_theta > 0:
        rot = torch.empty(((M * (NH + NKV) * hd * 2 + 255) // 256 * 256,), dtype=torch.uint8, device=x.device)
    attn_qkv_proj(qkv, rot, x, w, M // T, T, Cm, NH, NKV, hd, rope_theta,
                  FLAG_ROPE_INTERLEAVED if rope_interleaved else 0, stream)
    return qkv, rot


def attn_decode_workspace_bytes(B, NH, NKV, hd, max_len, dtype) -> int:
    return int(load().attn_decode_workspace_bytes(B, NH, NKV, hd, max_len, int(dtype)))


def attn_decode(out, lse, q, k_cache, v_cache, seq_lens, B, NH, NKV, hd, max_len, dtype, workspace,
                workspace_bytes, stream=None) -> None:
    st = load().attn_decode(_ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), B, NH,
                            NKV, hd, max_len, int(dtype), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check(st, "attn_decode")


def decode(q, k_cache, v_cache, seq_lens, dtype=None, stream=None, workspace=None):
    """Single-query attention over a KV cache: q [B,NH,hd], k_cache/v_cache
    [B,max_len,NKV,hd], seq_lens int32 [B] on the device.  Returns (out, lse)."""
    import torch
    B, NH, hd = q.shape
    max_len, NKV = k_cache.shape[1], k_cache.shape[2]
    code = dtype_code(q) if dtype is None else dtype
    if workspace is None:
        nbytes = attn_decode_workspace_bytes(B, NH, NKV, hd, max_len, code)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q)
    lse = torch.empty((B, NH), dtype=torch.float32, device=q.device)
    attn_decode(out, lse, q, k_cache, v_cache, seq_lens, B, NH, NKV, hd, max_len, code, workspace,
                workspace.numel(), stream)
    return out, lse


def attn_bwd_noalloc(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, dtype, stream=None) -> None:
    """attn_bwd without a workspace argument, for callers that cannot allocate
    device memory; uses the library's built-in scratch buffer (see the header
    for its size limit and the rule that overlapping calls race)."""
    st = load().attn_bwd_noalloc(_ptr(dqkv), _ptr(qkv), _ptr(out), _ptr(dout), _ptr(lse), B, T, C, NH, NKV,
                                 float(rope_theta), int(dtype), _stream(stream))
    _check(st, "attn_bwd_noalloc")


def attn_device_status(reset: bool = False) -> int:
    v = ctypes.c_int(0)
    _check(load().attn_device_status(ctypes.byref(v), 1 if reset else 0), "attn_device_status")
    return v.value


def attn_selftest_wait_timeout(limit_ns: int) -> int:
    v = ctypes.c_int(0)
    _check(load().attn_selftest_wait_timeout(int(limit_ns), ctypes.byref(v)), "attn_selftest_wait_timeout")
    return v.value


N_KERNEL_IDS = 17


def attn_profile_start() -> None:
    _check(load().attn_profile_start(), "attn_profile_start")


def attn_profile_stop() -> dict:
    """{kernel name: (launches, total ms)} for kernels launched since start."""
    ms = (ctypes.c_double * N_KERNEL_IDS)()
    n = (ctypes.c_int * N_KERNEL_IDS)()
    _check(load().attn_profile_stop(ms, n, N_KERNEL_IDS), "attn_profile_stop")
    return {load().attn_kernel_name(k).decode(): (n[k], ms[k]) for k in range(N_KERNEL_IDS) if n[k]}


# ---------------------------------------------------------------------------
# Convenience wrappers: allocate outputs with PyTorch, then call the C ABI.
# ---------------------------------------------------------------------------
def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported tensor dtype {t.dtype}")


def forward(qkv, NH: int, NKV: int, rope_theta: float = 0.0, dtype=None, stream=None, workspace=None,
            rope_interleaved: bool = False):
    """out, lse = attention forward of packed qkv [B, T, (NH+2*NKV)*hd].

    With ``workspace`` (a uint8 tensor, or True to allocate one of
    attn_fwd_workspace_bytes) the call goes through attn_fwd_ws, else attn_fwd."""
    import torch
    B, T, W = qkv.shape
    hd = W // (NH + 2 * NKV)
    C = NH * hd
    code = (dtype_code(qkv) if dtype is None else dtype) | (FLAG_ROPE_INTERLEAVED if rope_interleaved else 0)
    out = torch.empty((B, T, C), dtype=qkv.dtype, device=qkv.device)
    lse = torch.empty((B, NH, T), dtype=torch.float32, device=qkv.device)
    if workspace is None:
        attn_fwd(out, lse, qkv, B, T, C, NH, NKV, rope_theta, code, stream)
    else:
        if workspace is True:
            nbytes = attn_fwd_workspace_bytes(B, T, C, NH, NKV, code)
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=qkv.device)
        attn_fwd_ws(out, lse, qkv, B, T, C, NH, NKV, rope_theta, code, workspace, workspace.numel(), stream)
    return out, lse


def forward_ws(qkv, NH: int, NKV: int, rope_theta: float = 0.0, dtype=None, stream=None,
               rope_interleaved: bool = False):
    """(out, lse, workspace) through attn_fwd_ws; the workspace holds the
    rotated Q/K that backward(..., qk_rot=workspace) can reuse."""
    import torch
    B, T, W = qkv.shape
    hd = W // (NH + 2 * NKV)
    code = (dtype_code(qkv) if dtype is None else dtype) | (FLAG_ROPE_INTERLEAVED if rope_interleaved else 0)
    nbytes = attn_fwd_workspace_bytes(B, T, NH * hd, NH, NKV, code)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=qkv.device)
    out, lse = forward(qkv, NH, NKV, rope_theta, code, stream, workspace=ws)
    return out, lse, ws


def backward(qkv, out, dout, lse, NH: int, NKV: int, rope_theta: float = 0.0, dtype=None, stream=None,
             workspace=None, qk_rot=None, rope_interleaved: bool = False):
    """dqkv = attention backward; allocates the workspace unless one is given.
    With ``qk_rot`` (the workspace of the attn_fwd_ws call that made out/lse)
    the call goes through attn_bwd_rot, else attn_bwd."""
    import torch
    B, T, W = qkv.shape
    C = out.shape[2]
    code = (dtype_code(qkv) if dtype is None else dtype) | (FLAG_ROPE_INTERLEAVED if rope_interleaved else 0)
    nbytes = attn_bwd_workspace_bytes(B, T, C, NH, NKV, code)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=qkv.device)
    dqkv = torch.empty_like(qkv)
    if qk_rot is None:
        attn_bwd(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, code, workspace, workspace.numel(), stream)
    else:
        attn_bwd_rot(dqkv, qkv, out, dout, lse, B, T, C, NH, NKV, rope_theta, code, qk_rot, workspace,
                     workspace.numel(), stream)
    return dqkv
