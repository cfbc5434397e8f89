"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of oracle/bq_oracle.c (on the CPU, in a
temporary folder), builds it, and runs tests/test_oracle_pins.py against the
broken copy; the pin suite has to fail. The real oracle is never modified.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "bq_oracle.c")

# (name, exact text in bq_oracle.c, replacement)
MUTANTS = [
    ("scale_divisor_8", "float d = amax / (float)qmax;", "float d = amax / (float)(qmax + 1);"),
    ("divide_by_unrounded_scale", "oracle_round_half_even(x[j] / ds)", "oracle_round_half_even(x[j] / d)"),
    ("round_half_away", "return nearbyintf(v);", "return roundf(v);"),
    ("amax_without_abs", "float a = fabsf(x[j]);", "float a = x[j];"),
    ("interleaved_nibbles", "((unsigned)(q[j + QK / 2] + 8) << 4)", "((unsigned)(q[j ^ 1] + 8) << 4)"),
    ("decode_missing_offset", "q[j] = (int)(blk[2 + j] & 0x0Fu) - 8;", "q[j] = (int)(blk[2 + j] & 0x0Fu);"),
    ("fp16_truncates", "if (rem > half || (rem == half && (q & 1u)))", "if (0)"),
    ("fp16_ties_up", "if (rem > half || (rem == half && (q & 1u)))", "if (rem >= half)"),
    ("scale_big_endian", "out[0] = (uint8_t)(d16 & 0xFFu);", "out[0] = (uint8_t)(d16 >> 8); out[1] = (uint8_t)(d16 & 0xFFu); if (0)"),
    ("dot_uses_weight_scale_twice", "(double)block_scale(wb) * (double)block_scale(xb)", "(double)block_scale(wb) * (double)block_scale(wb)"),
    ("dot_drops_last_block", "for (int64_t b = 0; b < nb; b++) {\n        const uint8_t *wb", "for (int64_t b = 0; b + 1 < nb; b++) {\n        const uint8_t *wb"),
    ("gemm_output_transposed", "Y + n * M + m, mag ? mag + n * M + m : NULL", "Y + m * N + n, mag ? mag + m * N + n : NULL"),
    ("kv_bias_added", "v = v - bias[h * head_dim + b * QK + j];", "v = v + bias[h * head_dim + b * QK + j];"),
    ("kv_bias_ignores_head", "v = v - bias[h * head_dim + b * QK + j];", "v = v - bias[b * QK + j];"),
    ("q8_clamp_narrow", "const int qmin = (type == ORACLE_TYPE_Q4_0) ? -8 : -127;", "const int qmin = (type == ORACLE_TYPE_Q4_0) ? -8 : -126;"),
    ("attn_kv_head_modulo", "int64_t kvh = h / group;", "int64_t kvh = h % n_kv_heads;"),
    ("attn_no_scale", "s[t] = (double)scale * acc;", "s[t] = acc;"),
    ("attn_weights_unnormalized", "double w = s[t] / l;", "double w = s[t];"),
    ("attn_v_decoded_as_k", "oracle_dequantize_rows(v_type, V +", "oracle_dequantize_rows(k_type, V +"),
    ("attn_k_scale_twice", "(double)block_scale(kt + b * bk) * (double)block_scale(qh + b * bq)",
     "(double)block_scale(kt + b * bk) * (double)block_scale(kt + b * bk)"),
    ("legacy_min_not_added", "v = v + mn; /* R18: then the minimum, a second fp32 operation */", "(void)mn;"),
    ("legacy_qh_reversed", "qh |= (uint32_t)((u[j] >> 4) & 1) << j;", "qh |= (uint32_t)((u[j] >> 4) & 1) << (31 - j);"),
    ("legacy_q5_0_divisor_16", "float d = amax / 15.0f; /* R17 */", "float d = amax / 16.0f; /* R17 */"),
    ("legacy_min_term_dropped", "acc += mterm;", "(void)mterm;"),
    ("legacy_5bit_range_15", "const int umax = (1 << legacy_bits(type)) - 1;", "const int umax = 15;"),
    ("legacy_unrounded_min", "float ds = oracle_f16_to_f32(d16), ms = oracle_f16_to_f32(m16);",
     "float ds = oracle_f16_to_f32(d16), ms = mn;"),
    ("q4k_min_added", "dst[i] = S[i / 32] * (float)u[i] - M[i / 32];", "dst[i] = S[i / 32] * (float)u[i] + M[i / 32];"),
    ("q4k_scale_stream_shifted", "int bit = 6 * k, v;", "int bit = 6 * k + 1, v;"),
    ("q6k_offset_31", "dst[i] = (d * (float)(int8_t)blk[192 + i / 16]) * (float)(u[i] - 32);",
     "dst[i] = (d * (float)(int8_t)blk[192 + i / 16]) * (float)(u[i] - 31);"),
    ("q6k_high_bits_order", "int hi = (blk[128 + (i & 63)] >> (2 * (i >> 6))) & 3;",
     "int hi = (blk[128 + (i >> 2)] >> (2 * (i & 3))) & 3;"),
    ("q4k_superscale_64", "smax / 63.0f", "smax / 64.0f"),
    ("q4k_supermin_64", "mmax / 63.0f", "mmax / 64.0f"),
    ("q4k_min_unclamped", "m[j] = lo < 0.0f ? -lo : 0.0f;", "m[j] = -lo;"),
    ("q4k_range_16", "s[j] = (hi + m[j]) / 15.0f;", "s[j] = (hi + m[j]) / 16.0f;"),
    ("q4k_code_clamp_14", "clampi((int)oracle_round_half_even((x[32 * j + i] + M) / S), 0, 15)",
     "clampi((int)oracle_round_half_even((x[32 * j + i] + M) / S), 0, 14)"),
    ("q4k_codes_from_unrounded_factors", "float S = d * (float)sc[j], M = dm * (float)mn[j];", "float S = s[j], M = m[j];"),
    ("q6k_sub_32", "s[k] = amax / 31.0f;", "s[k] = amax / 32.0f;"),
    ("q6k_super_128", "uint16_t d16 = oracle_f32_to_f16(smax / 127.0f);",
     "uint16_t d16 = oracle_f32_to_f16(smax / 128.0f);"),
    ("q6k_clamp_31", "clampi((int)oracle_round_half_even(x[16 * k + i] / S), -32, 31)) + 32",
     "clampi((int)oracle_round_half_even(x[16 * k + i] / S), -31, 31)) + 32"),
    ("q6k_codes_from_unrounded_factor", "float S = d * (float)sc;", "float S = s[k];"),
    ("kquant_gemv_min_term_dropped", "double t1 = dx * (double)S[j] * (double)su, t2 = -dx * (double)M[j] * (double)sx;",
     "double t1 = dx * (double)S[j] * (double)su, t2 = 0.0 * (double)M[j] * (double)sx;"),
    ("kquant_row_stride", "int64_t nb = K / QK, row_bytes = K / bv * bw;\n    uint8_t *xq = (uint8_t *)malloc((size_t)(nb * oracle_block_bytes(ORACLE_TYPE_Q8_0)) + 1);",
     "int64_t nb = K / QK, row_bytes = nb * bw;\n    uint8_t *xq = (uint8_t *)malloc((size_t)(nb * oracle_block_bytes(ORACLE_TYPE_Q8_0)) + 1);"),
    ("hadamard_scaled_by_1_64", "v[j] = v[j] * 0.125f;", "v[j] = v[j] * 0.015625f;"),
    ("hadamard_no_minus", "v[j + h] = a - b;", "v[j + h] = a + b;"),
    ("hadamard_32_point", "for (int h = 1; h < 64; h *= 2)", "for (int h = 1; h < 32; h *= 2)"),
    ("hadamard_bias_basis_unchecked", "if (bias && bias_basis != basis)", "if (0)"),
    ("hadamard_bias_measured_plain", "if (basis == ORACLE_BASIS_HADAMARD64) /* [ROT] measured in the cache's basis */",
     "if (0)"),
    ("hadamard_q_not_rotated", "oracle_hadamard64(qr, n_heads * head_dim);", "(void)0;"),
    ("hadamard_kv_write_not_rotated", "if (basis == ORACLE_BASIS_HADAMARD64) /* R14: rotate first, then center */\n                oracle_hadamard64(row, head_dim);",
     "if (0) oracle_hadamard64(row, head_dim);"),
]


def _build_mutant(tmp, name, old, new):
    src = open(SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    src = src.replace(old, new)
    d = os.path.join(tmp, name)
    os.makedirs(d, exist_ok=True)
    with open(os.path.join(d, "bq_oracle.c"), "w", encoding="utf-8") as f:
        f.write(src)
    with open(os.path.join(ROOT, "oracle", "bq_oracle.h"), encoding="utf-8") as f:
        hdr = f.read()
    with open(os.path.join(d, "bq_oracle.h"), "w", encoding="utf-8") as f:
        f.write(hdr)
    lib = os.path.join(d, "libmut.so")
    subprocess.run(["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
                    "-shared", "-o", lib, os.path.join(d, "bq_oracle.c"), "-lm"], check=True)
    return lib


def _pins_fail(lib):
    env = dict(os.environ, BQ_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode != 0, r.stdout[-400:]


def test_pins_catch_every_mutant(tmp_path):
    libs = {name: _build_mutant(str(tmp_path), name, old, new) for name, old, new in MUTANTS}
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        res = dict(zip(libs, ex.map(_pins_fail, libs.values())))
    survived = [n for n, (failed, _) in res.items() if not failed]
    assert not survived, f"pins did not catch: {survived}"


def test_unmutated_copy_passes(tmp_path):
    """Control: the same harness on an unmodified copy passes."""
    lib = _build_mutant(str(tmp_path), "control", "#define QK 32", "#define QK 32")
    failed, out = _pins_fail(lib)
    assert not failed, out
