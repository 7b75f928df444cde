"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle/`` to a temporary directory, plants one mistake in
the copy (a flipped sign, a wrong index, a dropped term, a transposed
operand), and runs the pin suite against the copy in a subprocess.  The pin
suite must fail for every planted mistake.  Nothing here touches the CUDA
path.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = {
    "rope_rotates_backwards": ("rot[k + half, k] = -1.0", "rot[k + half, k] = 1.0"),
    "rope_adjoint_not_transposed": ("(g * sin) @ rot.T", "(g * sin) @ rot"),
    "rope_frequency_exponent": ("-2.0 * i * np.log(float(theta)) / hd",
                                "-1.0 * i * np.log(float(theta)) / hd"),
    "gqa_head_mapping_modulo": ("kh = h // grp\n            P, lse[b, h]",
                                "kh = h % (NH // grp)\n            P, lse[b, h]"),
    "mask_excludes_diagonal": ("np.arange(T)[None, :] <= rows[:, None]",
                               "np.arange(T)[None, :] < rows[:, None]"),
    "mask_anticausal": ("np.arange(T)[None, :] <= rows[:, None]",
                        "np.arange(T)[None, :] >= rows[:, None]"),
    "missing_score_scale": ("S = scale * (q @ k.T)", "S = (q @ k.T)"),
    "lse_base2": ("return E / l[:, None], m + np.log(l)", "return E / l[:, None], m + np.log2(l)"),
    "dS_drops_D": ("dS = P * (dP - D[:, None])", "dS = P * dP"),
    "dk_transposed_operand": ("dk[b, :, kh] += scale * (dS.T @ q)", "dk[b, :, kh] += scale * (dS @ q)"),
    "dq_missing_scale": ("dq[b, :, h] = scale * (dS @ k)", "dq[b, :, h] = (dS @ k)"),
    "dv_not_summed_over_group": ("dv[b, :, kh] += P.T @ dO", "dv[b, :, kh] = P.T @ dO"),
    "v_column_offset": ("V = x[:, :, C + NKV * hd:]", "V = x[:, :, C:C + NKV * hd]"),
    "dk_not_unrotated": ("        dk = rope_rotate_transpose(dk, rope_theta)\n", ""),
    # single-query (decode) attention, pinned by test_oracle_decode_pins.py
    "decode_gqa_head_mapping_modulo": ("            kh = h // grp\n            s = scale",
                                       "            kh = h % NKV\n            s = scale"),
    "decode_length_off_by_one": ("n = int(seq_lens[b])", "n = int(seq_lens[b]) - 1"),
    "decode_missing_score_scale": ("s = scale * (k_cache[b, :n, kh] @ q[b, h])", "s = (k_cache[b, :n, kh] @ q[b, h])"),
    "decode_lse_drops_max": ("lse[b, h] = m + np.log(l)", "lse[b, h] = np.log(l)"),
    "decode_reads_past_length": ("(e / l) @ v_cache[b, :n, kh]", "(e / l) @ v_cache[b, -n:, kh]"),
    # interleaved (GPT-J) RoPE, pinned by test_oracle_rope_interleaved_pins.py
    "gptj_rotation_sign": ("    y[..., 0::2] = x0 * cos - x1 * sin\n", "    y[..., 0::2] = x0 * cos + x1 * sin\n"),
    "gptj_frequency_exponent": ("    freq = float(theta) ** (-2.0 * i / hd)\n    ang = pos.astype(np.float64)[:, None] * freq[None, :]          # [T, hd/2]",
                                "    freq = float(theta) ** (-1.0 * i / hd)\n    ang = pos.astype(np.float64)[:, None] * freq[None, :]          # [T, hd/2]"),
    "gptj_pairs_swapped": ("    x0, x1 = x[..., 0::2], x[..., 1::2]", "    x1, x0 = x[..., 0::2], x[..., 1::2]"),
    "gptj_adjoint_sign": ("    y[..., 1::2] = -g0 * sin + g1 * cos", "    y[..., 1::2] = g0 * sin + g1 * cos"),
    # QKV projection, pinned by test_oracle_projection_pins.py
    "proj_rotates_v_too": ("    qk = qkv[:, :(NH + NKV) * hd].reshape(M // T, T, NH + NKV, hd)",
                           "    qk = qkv.reshape(M // T, T, NH + 2 * NKV, hd)"),
    "proj_positions_run_across_sequences": ("    qk = qkv[:, :(NH + NKV) * hd].reshape(M // T, T, NH + NKV, hd)",
                                            "    qk = qkv[:, :(NH + NKV) * hd].reshape(1, M, NH + NKV, hd)"),
    "proj_ignores_interleaved_flag": ("        rot, _ = _rope_fns(rope_interleaved)\n        qk = rot(qk, rope_theta)",
                                      "        rot, _ = _rope_fns(False)\n        qk = rot(qk, rope_theta)"),
    # e4m3 quantization (oracle/e4m3.py), pinned by test_oracle_e4m3_pins.py
    "e4m3_ties_away_from_zero": ("q = np.round(a / spacing) * spacing", "q = np.floor(a / spacing + 0.5) * spacing"),
    "e4m3_no_subnormal_floor": ("e = np.maximum(E - 1, _E4M3_MIN_EXP)", "e = E - 1"),
    "e4m3_two_mantissa_bits": ("_E4M3_MANT_BITS = 3", "_E4M3_MANT_BITS = 2"),
    "e4m3_no_saturation": ("    q = np.minimum(q, E4M3_MAX)\n", ""),
    "e4m3_scale_per_head": ("Qd = quantize_rows_e4m3(Qr, tile)", "Qd = quantize_rows_e4m3(Qr, None)"),
    "e4m3_v_scale_per_tile": ("Vd = quantize_rows_e4m3(V, None)", "Vd = quantize_rows_e4m3(V, tile)"),
    "e4m3_gqa_head_mapping_modulo": ("kh = h // grp\n                P, lse[b, h]",
                                     "kh = h % NKV\n                P, lse[b, h]"),
    "e4m3_dequant_uses_scale": ("out[b, t0:t0 + step, h] = codes * d", "out[b, t0:t0 + step, h] = codes / d"),
    # rounding of the softmax weights in the e4m3 forward (oracle/e4m3.py)
    "e4m3_weight_scale_448": ("P_SCALE = 112.0 ", "P_SCALE = 448.0 "),
    "e4m3_renewal_threshold_zero": ("RESCALE_THRESHOLD = 2.0 ", "RESCALE_THRESHOLD = 0.0 "),
    "e4m3_renew_every_block": ("renew = bool(mb > m + threshold)", "renew = True"),
    "e4m3_weights_unrounded": ("p8 = e4m3_round(p)", "p8 = p"),
    "e4m3_l_sums_rounded_weights": ("l += p.sum()", "l += p8.sum()"),
    "e4m3_no_rescale_on_renewal": ("            o *= c\n            o_abs *= c", "            o_abs *= c"),
    "e4m3_rounded_path_head_mapping": ("            kh = h // grp\n            for t in rows:",
                                       "            kh = h % NKV\n            for t in rows:"),
    "e4m3_midpoint_not_reported": ("dev = np.maximum(hi - p8, p8 - lo)", "dev = np.zeros_like(p8)"),
}
MUTATED_FILE = {name: "e4m3.py" for name in MUTATIONS if name.startswith("e4m3_")}
PIN_FILE = {name: "test_oracle_decode_pins.py" for name in MUTATIONS if name.startswith("decode_")}
PIN_FILE.update({name: "test_oracle_rope_interleaved_pins.py" for name in MUTATIONS if name.startswith("gptj_")})
PIN_FILE.update({name: "test_oracle_e4m3_pins.py" for name in MUTATIONS if name.startswith("e4m3_")})
PIN_FILE.update({name: "test_oracle_projection_pins.py" for name in MUTATIONS if name.startswith("proj_")})


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src_dir = os.path.join(ROOT, "oracle")
    dst_dir = tmp_path / "oracle"
    shutil.copytree(src_dir, dst_dir, ignore=shutil.ignore_patterns("__pycache__"))
    path = dst_dir / MUTATED_FILE.get(name, "attention.py")
    text = path.read_text()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path.write_text(text.replace(old, new))
    mark = tmp_path / "imported.mark"
    init = dst_dir / "__init__.py"
    init.write_text(init.read_text() + "\nopen(%r, 'w').write('mutant')\n" % str(mark))
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([str(tmp_path), ROOT, env.get("PYTHONPATH", "")])
    res = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         "--rootdir", str(tmp_path), os.path.join(ROOT, "tests", PIN_FILE.get(name, "test_oracle_pins.py"))],
        cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    assert mark.exists(), "the pin suite did not import the mutant oracle"
    assert res.returncode != 0, f"pins did not catch mutation {name}:\n{res.stdout[-2000:]}"
