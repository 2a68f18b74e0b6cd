"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a swapped nibble or byte, a wrong index, sign or rounding rule), builds
the copy, and runs the pin suite against it in a child process: the suite must
fail. Everything here runs on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qm_oracle.c")

MUTANTS = {
    "mxfp4_nibble_swap": ("return (i % 2 == 0) ? (b & 0xF) : (b >> 4);",
                          "return (i % 2 == 0) ? (b >> 4) : (b & 0xF);"),
    "mxfp4_blocks_half_swap": ("return (t < 16) ? (b & 0xF) : (b >> 4);",
                               "return (t < 16) ? (b >> 4) : (b & 0xF);"),
    "mxfp4_blocks_byte_index": ("uint8_t b = block[1 + (t % 16)];", "uint8_t b = block[1 + (t / 2)];"),
    "mxfp4_blocks_scale_byte": ("or_e8m0_to_f64(blk[0])", "or_e8m0_to_f64(blk[16])"),
    "quantize_half_even": ("q[j] = isfinite(p) ? (int8_t)roundf(p) : 0;",
                           "q[j] = isfinite(p) ? (int8_t)rintf(p) : 0;"),
    "quantize_amax_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "quantize_inf_scale_sign": ("h = has_nan ? 0x7E00 : 0x7C00;", "h = has_nan ? 0x7E00 : 0xFC00;"),
    "affine_bias_dropped": ("v[i] = fmaf((float)c, s, b);", "v[i] = fmaf((float)c, s, 0.0f * b);"),
    "affine_bit_order": ("c |= bit << t;", "c |= bit << (bits - 1 - t);"),
    "affine_group_index": ("r * ng + i / gs, sdt);\n            float b",
                           "r * ng + (i / gs + 1) % ng, sdt);\n            float b"),
    "e8m0_bias": ("return ldexp(1.0, s - 127);", "return ldexp(1.0, s - 128);"),
    "e2m1_table": ("{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0}"),
    "e2m1_negzero": ("return (code & 8) ? -m : m;", "return (code & 8) ? 0.0 - m : m;"),
    "q8_0_d_byte_order": ("block[0] | (block[1] << 8)", "block[1] | (block[0] << 8)"),
    "q8_0_unsigned_quant": ("return (int)(int8_t)block[2 + t];", "return (int)block[2 + t];"),
    "f16_subnormal": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)f, -25);"),
    "bf16_tie_rule": ("r = (lo & 1) ? hi : lo;", "r = lo;"),
    "f16_round_tie": ("n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;", "n = fl + 1.0;"),
    "product_sign": ("acc += xd[m * k + i] * (double)v[i];", "acc -= xd[m * k + i] * (double)v[i];"),
    "product_transposed_x": ("acc += xd[m * k + i] * (double)v[i];",
                             "acc += xd[m * k + (k - 1 - i)] * (double)v[i];"),
    "take_nonzero_fill": ("memset(dp, 0, (size_t)inner_bytes);", "memset(dp, 1, (size_t)inner_bytes);"),
    "route_unstable": ("for (int64_t p = 0; p < P; ++p)\n            if (or_id(ids, ids64, p) == e) {",
                       "for (int64_t p = P - 1; p >= 0; --p)\n            if (or_id(ids, ids64, p) == e) {"),
    "experts_out_of_range_uses_expert0": ("if (id < 0 || id >= E) {\n                for",
                                          "if (id < 0 || id >= E) id = 0;\n            if (0) {\n                for"),
    "experts_broadcast_row": ("return (x_rows == T) ? p / topk : p;", "return (x_rows == T) ? p % T : p;"),
    "q4_k_nibble_halves": ("int q = (r < 32) ? (byte & 0x0F) : (byte >> 4);",
                           "int q = (r < 32) ? (byte >> 4) : (byte & 0x0F);"),
    "q4_k_high_bits_source": ("*sc = (b[8 + (j - 4)] & 0x0F) | ((b[j - 4] >> 6) << 4);",
                              "*sc = (b[8 + (j - 4)] & 0x0F) | ((b[j] >> 6) << 4);"),
    "q4_k_scale_min_swap": ("*sc = b[j] & 0x3F;\n        *m = b[4 + j] & 0x3F;",
                            "*m = b[j] & 0x3F;\n        *sc = b[4 + j] & 0x3F;"),
    "q4_k_min_sign": ("return (float)(d * sc * q - dmin * m);", "return (float)(d * sc * q + dmin * m);"),
    "q6_k_offset": ("return (float)(d * sc * (q - 32));", "return (float)(d * sc * (q - 31));"),
    "q6_k_high_bits": ("int hi = (qh[32 * h + l] >> (2 * t)) & 3;", "int hi = (qh[32 * h + l] >> t) & 3;"),
    "q6_k_scale_index": ("int sc = scales[8 * h + 2 * t + l / 16];", "int sc = scales[8 * h + 2 * t];"),
    "q6_k_ql_half": ("uint8_t lo_byte = ql[64 * h + l + 32 * (t % 2)];",
                     "uint8_t lo_byte = ql[64 * h + l + 32 * (t / 2)];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(lib),
                    str(path), "-lm"], check=True)
    env = dict(os.environ, QM_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake {name} passed every pin:\n{r.stdout[-2000:]}"
