"""CPU checks of the C ABI: the library builds, loads, exports every symbol
declared in include/*.h, and rejects invalid arguments before any CUDA work
(no compute call is made here)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cdll():
    from causal_attention_gqa_gb300 import build, binding
    build.build()
    return binding.load()


def declared_symbols():
    names = set()
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        names.update(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_symbols()
    for required in ("attn_fwd", "attn_fwd_ws", "attn_fwd_workspace_bytes", "attn_bwd", "attn_bwd_workspace_bytes",
                     "attn_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(cdll):
    for name in declared_symbols():
        assert hasattr(cdll, name), name
        assert isinstance(getattr(cdll, name), ctypes._CFuncPtr)


def test_strerror_and_version(cdll):
    from causal_attention_gqa_gb300 import binding
    assert binding.attn_abi_version() == 1
    for code in range(-8, 1):
        assert binding.attn_strerror(code) != "unknown status"
    assert binding.attn_strerror(-99) == "unknown status"


def test_workspace_size(cdll):
    from causal_attention_gqa_gb300 import binding
    B, T, C, NH, NKV = 4, 2048, 2048, 16, 4
    # bf16: (lse, D) float tables per (b, h) over T rounded up to 128, then
    # the rotated Q/K copy, the dQ kernel's work-item counter and the RoPE
    # (cos, sin) table [hd/2][T]; each part rounded up to 256 bytes.
    def up(n):
        return (n + 255) // 256 * 256
    row_bytes = B * NH * T * 8
    rot_bytes = B * T * (NH + NKV) * (C // NH) * 2
    cnt_bytes = 256
    cs_bytes = T * (C // NH) * 4
    assert binding.attn_bwd_workspace_bytes(B, T, C, NH, NKV, binding.DTYPE_BF16) == \
        row_bytes + rot_bytes + cnt_bytes + cs_bytes
    ragged = binding.attn_bwd_workspace_bytes(1, 100, 256, 2, 1, binding.DTYPE_BF16)
    assert ragged == 2 * 128 * 8 + up(100 * 3 * 128 * 2) + 256 + up(100 * 128 * 4)
    assert binding.attn_bwd_workspace_bytes(1, 16, 16, 4, 4, binding.DTYPE_F32) == 256
    assert binding.attn_bwd_workspace_bytes(1, 16, 16, 3, 4, binding.DTYPE_F32) == 0


@pytest.mark.parametrize("args,code", [
    ((1, 16, 16, 3, 3, 0.0, 0), -2),     # C % NH
    ((1, 16, 16, 4, 3, 0.0, 0), -2),     # NH % NKV
    ((0, 16, 16, 4, 4, 0.0, 0), -2),     # B < 1
    ((1, 0, 16, 4, 4, 0.0, 0), -2),      # T < 1
    ((1, 16, 12, 4, 4, 1e4, 0), -2),     # odd head size with RoPE
    ((1, 16, 1024, 4, 4, 0.0, 0), -3),   # hd 256 unsupported
    ((1, 16, 128, 4, 4, 0.0, 2), -3),    # bf16 needs hd 64 or 128 (hd 32 here)
    ((1, 16, 1024, 4, 4, 0.0, 1), -3),   # TF32 (float32 kernels): hd 256 unsupported
    ((1, 16, 512, 4, 4, 0.0, 1), -1),    # TF32 accepted: fails only on the null pointers
    ((1, 16, 512, 4, 4, 0.0, 7), -8),    # unknown dtype
    ((1, 16, 512, 4, 4, 0.0, 2 | 0x200), -8),   # unknown flag bit
    ((1, 16, 512, 4, 4, 1e4, 2 | 0x100), -1),   # interleaved RoPE flag accepted (null pointers)
    ((1, 16, 512, 4, 4, float("nan"), 2), -8),
])
def test_forward_rejects_invalid_shapes(cdll, args, code):
    assert cdll.attn_fwd(None, None, None, *args, None) == code


def test_forward_rejects_null_pointers(cdll):
    assert cdll.attn_fwd(None, None, None, 1, 16, 16, 4, 4, 0.0, 0, None) == -1


def test_backward_rejects_missing_workspace(cdll):
    p = 1 << 20   # never dereferenced: validation fails first
    assert cdll.attn_bwd(p, p, p, p, p, 1, 16, 16, 4, 4, 0.0, 0, None, 0, None) == -5
    assert cdll.attn_bwd(p, p, p, p, p, 1, 16, 16, 4, 4, 0.0, 0, p, 8, None) == -5
    assert cdll.attn_bwd(p, p, p, p, p, 1, 16, 16, 4, 4, 0.0, 0, p + 16, 4096, None) == -4


def test_forward_workspace_size_and_validation(cdll):
    from causal_attention_gqa_gb300 import binding
    B, T, C, NH, NKV = 4, 2048, 2048, 16, 4
    # bf16: the rotated Q/K copy [B, T, (NH+NKV)*hd], rounded up to 256 bytes.
    assert binding.attn_fwd_workspace_bytes(B, T, C, NH, NKV, binding.DTYPE_BF16) == B * T * (NH + NKV) * 128 * 2
    assert binding.attn_fwd_workspace_bytes(1, 100, 256, 2, 1, binding.DTYPE_BF16) == (100 * 3 * 128 * 2 + 255) // 256 * 256
    assert binding.attn_fwd_workspace_bytes(1, 99, 256, 2, 1, binding.DTYPE_BF16) == (99 * 3 * 128 * 2 + 255) // 256 * 256
    assert binding.attn_fwd_workspace_bytes(1, 16, 16, 4, 4, binding.DTYPE_F32) == 0
    assert binding.attn_fwd_workspace_bytes(1, 16, 16, 3, 4, binding.DTYPE_BF16) == 0
    p = 1 << 20   # never dereferenced: validation fails first
    args = (1, 128, 512, 4, 1, 1e6, binding.DTYPE_BF16)
    assert cdll.attn_fwd_ws(p, p, p, *args, None, 0, None) == -5
    assert cdll.attn_fwd_ws(p, p, p, *args, p, 64, None) == -5
    assert cdll.attn_fwd_ws(p, p, p, 1, 16, 16, 3, 3, 0.0, 0, None, 0, None) == -2
    assert cdll.attn_fwd_ws(None, None, None, 1, 16, 16, 4, 4, 0.0, 0, None, 0, None) == -1


def test_backward_rot_validation(cdll):
    p = 1 << 20   # never dereferenced: validation fails first
    args = (1, 128, 512, 4, 1, 1e6, 2)
    assert cdll.attn_bwd_rot(p, p, p, p, p, *args, p, None, 0, None) == -5
    assert cdll.attn_bwd_rot(p, p, p, p, p, *args, p + 16, p, 1 << 24, None) == -4
    assert cdll.attn_bwd_rot(None, p, p, p, p, *args, p, p, 1 << 24, None) == -1


def _a256(n):
    return (n + 255) // 256 * 256


def test_fp8_forward_workspace_size_and_validation(cdll):
    from causal_attention_gqa_gb300 import binding
    bf16 = binding.DTYPE_BF16

    def expected(B, T, NH, NKV, hd):
        # e4m3 Q/K copy, e4m3 V^T over T rounded up to 128, Q/K tile scales,
        # V head scales, V tile maxima; each part rounded up to 256 bytes.
        n_qt = (T + 127) // 128
        heads = NH + NKV
        return (_a256(B * T * heads * hd) + _a256(B * NKV * hd * n_qt * 128) + _a256(B * heads * n_qt * 4)
                + _a256(B * NKV * 4) + _a256(B * NKV * n_qt * 4))

    assert binding.attn_fwd_fp8_workspace_bytes(4, 2048, 2048, 16, 4, bf16) == expected(4, 2048, 16, 4, 128)
    assert binding.attn_fwd_fp8_workspace_bytes(1, 300, 256, 2, 1, bf16) == expected(1, 300, 2, 1, 128) == 165120
    # unsupported: head size 64, odd group, float32 dtype -> no workspace
    assert binding.attn_fwd_fp8_workspace_bytes(1, 128, 256, 4, 2, bf16) == 0
    assert binding.attn_fwd_fp8_workspace_bytes(1, 128, 384, 3, 1, bf16) == 0
    assert binding.attn_fwd_fp8_workspace_bytes(1, 128, 512, 4, 2, binding.DTYPE_F32) == 0
    p = 1 << 20   # never dereferenced: validation fails first
    need = expected(1, 128, 4, 2, 128)
    args = (1, 128, 512, 4, 2, 1e6, bf16)
    assert cdll.attn_fwd_fp8(p, p, p, 1, 128, 256, 4, 2, 1e6, bf16, p, need, None) == -3     # hd 64
    assert cdll.attn_fwd_fp8(p, p, p, 1, 128, 384, 3, 1, 1e6, bf16, p, need, None) == -3     # odd group
    assert cdll.attn_fwd_fp8(p, p, p, 1, 128, 512, 4, 2, 1e6, binding.DTYPE_F32, p, need, None) == -3
    assert cdll.attn_fwd_fp8(p, p, p, 1, 128, 512, 4, 3, 1e6, bf16, p, need, None) == -2     # NH % NKV
    assert cdll.attn_fwd_fp8(None, p, p, *args, p, need, None) == -1
    assert cdll.attn_fwd_fp8(p + 2, p, p, *args, p, need, None) == -4                       # out not 16-byte aligned
    assert cdll.attn_fwd_fp8(p, p, p, *args, None, need, None) == -5
    assert cdll.attn_fwd_fp8(p, p, p, *args, p, need - 1, None) == -5
    assert cdll.attn_fwd_fp8(p, p, p, *args, p + 16, need, None) == -4                      # workspace not 256-aligned
    assert cdll.attn_fwd_fp8(p, p, p, 1, 128, 512, 4, 2, 1e6, bf16 | 0x200, p, need, None) == -8


def test_decode_validation(cdll):
    from causal_attention_gqa_gb300 import binding
    bf16 = binding.DTYPE_BF16
    nb = binding.attn_decode_workspace_bytes(4, 8, 2, 128, 1000, bf16)
    assert nb > 0 and nb % 256 == 0
    assert binding.attn_decode_workspace_bytes(4, 8, 3, 128, 1000, bf16) == 0     # NH % NKV
    assert binding.attn_decode_workspace_bytes(4, 8, 2, 96, 1000, bf16) == 0      # head size 96
    assert binding.attn_decode_workspace_bytes(4, 8, 2, 128, 0, bf16) == 0        # empty cache
    assert binding.attn_decode_workspace_bytes(4, 8, 2, 128, 1000, 7) == 0        # unknown dtype
    p = 1 << 20
    shape = (4, 8, 2, 128, 1000)
    assert cdll.attn_decode(p, p, p, p, p, p, 4, 8, 3, 128, 1000, bf16, p, nb, None) == -2
    assert cdll.attn_decode(p, p, p, p, p, p, 4, 8, 2, 96, 1000, bf16, p, nb, None) == -3
    assert cdll.attn_decode(p, p, p, p, p, p, *shape, 7, p, nb, None) == -8
    assert cdll.attn_decode(p, p, p, p, p, None, *shape, bf16, p, nb, None) == -1           # seq_lens
    assert cdll.attn_decode(p, p, p, p, p, p, *shape, bf16, None, nb, None) == -5
    assert cdll.attn_decode(p, p, p, p, p, p, *shape, bf16, p, nb - 256, None) == -5
    assert cdll.attn_decode(p, p, p + 8, p, p, p, *shape, bf16, p, nb, None) == -4          # q
    assert cdll.attn_decode(p, p + 2, p, p, p, p, *shape, bf16, p, nb, None) == -4          # lse


def test_qkv_projection_validation(cdll):
    p = 1 << 20
    ok = (2, 64, 512, 4, 2, 128, 1e6)
    assert cdll.attn_qkv_proj(p, p, p, p, 0, 64, 512, 4, 2, 128, 1e6, 0, None) == -2        # B < 1
    assert cdll.attn_qkv_proj(p, p, p, p, 2, 64, 512, 4, 3, 128, 1e6, 0, None) == -2        # NH % NKV
    assert cdll.attn_qkv_proj(p, p, p, p, 2, 64, 516, 4, 2, 128, 1e6, 0, None) == -2        # Cm % 8
    assert cdll.attn_qkv_proj(p, p, p, p, 2, 64, 512, 4, 2, 96, 1e6, 0, None) == -3         # head size 96
    assert cdll.attn_qkv_proj(p, p, p, p, *ok, 0x200, None) == -8                          # unknown flag
    assert cdll.attn_qkv_proj(p, p, p, p, 2, 64, 512, 4, 2, 128, float("inf"), 0, None) == -8
    assert cdll.attn_qkv_proj(None, p, p, p, *ok, 0, None) == -1
    assert cdll.attn_qkv_proj(p, p, p, p + 4, *ok, 0, None) == -4                          # w
    assert cdll.attn_qkv_proj(p, p + 4, p, p, *ok, 0x100, None) == -4                      # rotated copy


def test_forward_rot_validation(cdll):
    p = 1 << 20
    assert cdll.attn_fwd_rot(p, p, p, None, 1, 128, 512, 4, 1, 1e6, 2, None) == -1         # bf16 RoPE needs the copy
    assert cdll.attn_fwd_rot(p, p, p, p, 1, 128, 512, 4, 3, 1e6, 2, None) == -2
    assert cdll.attn_fwd_rot(p, p, p, p, 1, 128, 512, 4, 1, 1e6, 7, None) == -8
