"""The oracle's pins catch plausible mistakes.

Each mutant below is the oracle source with one deliberate slip (a flipped
sign, a dropped term, a wrong index, a transposed layout). The mutant is
compiled into a temporary directory -- the oracle itself is untouched -- and
at least one pin of tests/test_oracle_pins.py must fail against it.
"""
import inspect
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kvinj_oracle.c")

MUTANTS = [
    ("rope_sin_sign", "y[i] = a * c - b * s;", "y[i] = a * c + b * s;"),
    ("rope_dropped_term", "y[i + half] = b * c + a * s;", "y[i + half] = b * c;"),
    ("rope_pairing_adjacent", "double a = x[i], b = x[i + half];",
     "double a = x[i], b = x[(i + 1) % (2 * half)];"),
    ("rope_freq_exponent", "pow(theta, -(2.0 * (double)i) / (double)D)",
     "pow(theta, -((double)i) / (double)D)"),
    ("round_truncates", "double n = nearbyint(a / q);", "double n = floor(a / q);"),
    ("slot_offset", "slot_out[i] = (int64_t)blk * B + p % B;",
     "slot_out[i] = (int64_t)blk * B + p / B;"),
    ("cache_layout_transposed", "return (((layer * num_blocks + blk) * Hkv + h) * B + off) * D;",
     "return (((layer * num_blocks + blk) * B + off) * Hkv + h) * D;"),
    ("attention_no_scale", "s[j] = scale * acc;", "s[j] = acc;"),
    ("softmax_unnormalised", "double w = exp(s[j] - m) / z;", "double w = exp(s[j] - m);"),
    ("gqa_interleaved", "int r = (int)(rq / Hq), qh = (int)(rq % Hq), h = qh / G;",
     "int r = (int)(rq / Hq), qh = (int)(rq % Hq), h = qh % Hkv;"),
    ("inject_v_from_k", "const uint16_t *vp = kp + kv_half;", "const uint16_t *vp = kp;"),
    ("inject_position_dropped", "int64_t pos = (int64_t)start_pos[j] + t;",
     "int64_t pos = (int64_t)start_pos[j];"),
    ("decode_block_index", "int32_t blk = block_tables[(int64_t)r * max_blocks + j / B];",
     "int32_t blk = block_tables[(int64_t)r * max_blocks + j % B];"),
    ("decode_query_not_rotated", "if (rotate_q) orc_rope(q0, D, q_pos, theta, q);",
     "if (0) orc_rope(q0, D, q_pos, theta, q);"),
    ("copy_blocks_first_layer_only", "for (int l = l0; l < l1; ++l)\n      for (int h = 0; h < Hkv; ++h)\n        for (int t = 0; t < B; ++t) {",
     "for (int l = l0; l < l0 + 1; ++l)\n      for (int h = 0; h < Hkv; ++h)\n        for (int t = 0; t < B; ++t) {"),
    ("window_off_by_one", "int64_t j0 = (window > 0 && ctx > window) ? ctx - window : 0",
     "int64_t j0 = (window > 0 && ctx > window) ? ctx - window + 1 : 0"),
    ("prefill_excludes_itself", "    int64_t ctx = (int64_t)pos[i] + 1;\n    if (r < 0",
     "    int64_t ctx = (int64_t)pos[i];\n    if (r < 0"),
    ("prefill_first_request_table", "    int r = seq[i];\n", "    int r = 0;\n"),
    ("i8_scale_128", "float s = (float)(amax / 127.0);", "float s = (float)(amax / 128.0);"),
    ("i8_round_floor", "double v = s > 0.0f ? nearbyint(dec16(in[r * D + d], f) / (double)s) : 0.0;",
     "double v = s > 0.0f ? floor(dec16(in[r * D + d], f) / (double)s) : 0.0;"),
    ("i8_value_takes_key_scale", "V[j * D + d] = (double)vq[e + d] * (double)vs[e / D];",
     "V[j * D + d] = (double)vq[e + d] * (double)ks[e / D];"),
    ("copy_blocks_k_only", "            v_cache[to + d] = v_cache[from + d];\n", ""),
]


def _pin_functions():
    return [(n, f) for n, f in inspect.getmembers(pins, inspect.isfunction)
            if n.startswith("test_")]


def _run_pins(golden_dir):
    failed = []
    for name, fn in _pin_functions():
        kwargs = {"golden_dir": golden_dir} if "golden_dir" in inspect.signature(fn).parameters else {}
        try:
            fn(**kwargs)
        except Exception:  # noqa: BLE001 - any failure counts as caught
            failed.append(name)
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, golden_dir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(path), "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    with oracle.use_library(str(lib)):
        failed = _run_pins(golden_dir)
    assert failed, f"mutant {name} passed every pin"


def test_unmutated_source_passes_every_pin(tmp_path, golden_dir):
    lib = tmp_path / "libsame.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", SRC, "-o", str(lib), "-lm"],
                   check=True, capture_output=True)
    with oracle.use_library(str(lib)):
        assert _run_pins(golden_dir) == []
