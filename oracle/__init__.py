"""Double-precision CPU oracle for causal MHA/GQA attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it, to check and to time the CUDA library against a
plain, slow, obviously correct restatement of the method.
"""
from .attention import (  # noqa: F401
    split_qkv,
    rope_cos_sin,
    rope_rotate,
    rope_rotate_transpose,
    rope_rotate_interleaved,
    rope_rotate_interleaved_transpose,
    attention_forward,
    attention_backward,
    attention_sampled,
    attention_decode,
    qkv_projection,
)
from .e4m3 import e4m3_round, attention_forward_e4m3  # noqa: F401,E402
