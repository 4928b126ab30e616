"""Planted mistakes: each case copies the oracle's C source, plants one plausible
mistake (a wrong rounding, a dropped term, a swapped index, a wrong sign or
offset), compiles the copy on the CPU and runs the pin suite against it.  Every
planted mistake must make at least one pin fail; a survivor means the pins do
not constrain that part of the oracle."""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kvq_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in the oracle, replacement): each text occurs exactly once
MUTANTS = [
    ("round_half_up", "float r = nearbyintf(q);", "float r = floorf(q + 0.5f);"),
    ("scale_not_rounded_to_fp16", "float s = kvq_oracle_f16_to_f32(s16);", "float s = (amax > 0.0f) ? s32 : 1.0f;"),
    ("divide_by_8", "float s32 = amax / 7.0f;", "float s32 = amax / 8.0f;"),
    ("zero_rule_before_rounding", "if ((s16 & 0x7fffu) == 0) s16 = 0x3c00u;", "if (amax == 0.0f) s16 = 0x3c00u;"),
    ("clamp_to_minus_8", "if (r < -7.0f) r = -7.0f;", "if (r < -8.0f) r = -8.0f;"),
    ("nibbles_swapped", "codes_row[j] = (uint8_t)(lo | (hi << 4));", "codes_row[j] = (uint8_t)(hi | (lo << 4));"),
    ("offset_7", "unsigned lo = (unsigned)(c[2 * j] + 8);", "unsigned lo = (unsigned)(c[2 * j] + 7);"),
    ("dequant_wrong_group", "float s = kvq_oracle_f16_to_f32(get_u16(scales_row + (size_t)(i / G) * 2u));",
     "float s = kvq_oracle_f16_to_f32(get_u16(scales_row + (size_t)((i / G) ^ 1) % (size_t)(d / G) * 2u));"),
    ("gqa_modulo_map", "int h = hq / n_rep;", "int h = hq % Hkv;"),
    ("no_max_subtraction", "double p = exp(z - zmax);", "double p = exp(z);"),
    ("softmax_scale_dropped_in_pass2", "        z *= softmax_scale;\n                double p",
     "        double p"),
    ("page_slot_swapped", "uint8_t *blk = block_ptr(&L, pool, page, h);\n                quantize_row",
     "uint8_t *blk = block_ptr(&L, pool, page, (h + 1) % Hkv);\n                quantize_row"),
    ("v_scales_overlap_k_scales", "return blk + (size_t)L->P * (size_t)L->d + (size_t)L->P * (size_t)(L->d / L->Gk) * 2u +",
     "return blk + (size_t)L->P * (size_t)L->d + (size_t)(L->d / L->Gk) * 2u +"),
    ("f16_ties_away", "if (rem > half || (rem == half && (q & 1))) q += 1;", "if (rem >= half) q += 1;"),
    ("f16_subnormal_off_by_one", "int s = -(e + 1);", "int s = -e;"),
    ("window_start_off_by_one", "if (t >= len - window) return 1;", "if (t > len - window) return 1;"),
    ("window_sinks_inclusive", "return sinks > 0 && t < sinks;", "return sinks > 0 && t <= sinks;"),
    ("window_sinks_ignored", "return sinks > 0 && t < sinks;", "return 0;"),
    ("window_gqa_modulo_map", "int kv = hq / n_rep;", "int kv = hq % Hkv;"),
    ("window_no_max_subtraction", "double w = exp(z - zmax);", "double w = exp(z);"),
    ("fp16_k_v_swapped", "uint8_t *kr = fp16_row(pool16, Hkv, d, P, page, h, 0, slot);",
     "uint8_t *kr = fp16_row(pool16, Hkv, d, P, page, h, 1, slot);"),
    ("fp16_block_stride_2pd", "size_t blk = ((size_t)page * (size_t)Hkv + (size_t)h) * ((size_t)4 * (size_t)P * (size_t)d);",
     "size_t blk = ((size_t)page * (size_t)Hkv + (size_t)h) * ((size_t)2 * (size_t)P * (size_t)d);"),
    ("fp16_gqa_modulo", "int kvh = hq / rep;", "int kvh = hq % Hkv;"),
    ("fp16_dequant_truncated", "put_u16(kr + 2 * i, kvq_oracle_f32_to_f16(rk[i]));",
     "put_u16(kr + 2 * i, (uint16_t)(kvq_oracle_f32_to_f16(rk[i]) & 0xfffeu));"),
    ("fp16_attention_scale_dropped", "        z *= softmax_scale;\n                double wz",
     "        double wz"),
    ("mixed_split_off_by_one", "                    if (t < split) {", "                    if (t <= split) {"),
    ("mixed_fp16_part_from_int4_table",
     "int page = block_table16[(size_t)b * (size_t)max_blocks16 + (size_t)(t / P)];",
     "int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];"),
    ("int8_divide_by_128", "float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    # (the INT8 clamp at -128 cannot bind: with scale = amax / 127 every |x / scale| <= 127,
    # so moving it to -127 changes nothing and is not planted)
    ("int8_ties_away", "float r = nearbyintf(kvq_oracle_f16_to_f32(x[i]) / s);",
     "float r = roundf(kvq_oracle_f16_to_f32(x[i]) / s);"),
    ("int8_k_scale_for_v", "float sv = get_f32(blk + (size_t)2 * (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot));\n            size_t off",
     "float sv = get_f32(blk + (size_t)2 * (size_t)P * (size_t)d + (size_t)4 * (size_t)slot);\n            size_t off"),
    ("int8_attention_gqa_modulo", "int kh = hq / per;", "int kh = hq % Hkv;"),
    ("last_token_dropped", "for (int t = 0; t < len; ++t) {\n                int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];\n                uint8_t *blk",
     "for (int t = 0; t < len - 1; ++t) {\n                int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(t / P)];\n                uint8_t *blk"),
    # the rotated 4-bit codec
    ("wht_f32_butterfly_sign", "float a = y[i], b = y[i + h];\n                y[i] = a + b;\n                y[i + h] = a - b;",
     "float a = y[i], b = y[i + h];\n                y[i] = a + b;\n                y[i + h] = b - a;"),
    ("wht_f64_butterfly_sign", "double a = y[i], b = y[i + h];\n                y[i] = a + b;\n                y[i + h] = a - b;",
     "double a = y[i], b = y[i + h];\n                y[i] = a + b;\n                y[i + h] = b - a;"),
    ("wht_stage_skipped", "    for (int h = 1; h < d; h <<= 1)\n        for (int i = 0; i < d; ++i)\n            if ((i & h) == 0) {\n                float a",
     "    for (int h = 2; h < d; h <<= 1)\n        for (int i = 0; i < d; ++i)\n            if ((i & h) == 0) {\n                float a"),
    ("wht4_sigma_rms_of_x", "float sigma = sqrtf(s[0]);", "float sigma = sqrtf(s[0] / 128.0f);"),
    ("wht4_threshold_strict", "for (int j = 0; j < 15; ++j) code += u >= T[j];", "for (int j = 0; j < 15; ++j) code += u > T[j];"),
    ("wht4_nibbles_swapped", "codes[i / 2] |= (uint8_t)(code << (4 * (i & 1)));", "codes[i / 2] |= (uint8_t)(code << (4 * (1 - (i & 1))));"),
    ("wht4_no_division_by_d", "    wht_f64(out, d);\n    for (int i = 0; i < d; ++i) out[i] /= d;", "    wht_f64(out, d);"),
    ("lloyd_threshold_not_midpoint", "for (int j = 1; j < n; ++j) tb[j] = 0.5 * (lv[j - 1] + lv[j]);",
     "for (int j = 1; j < n; ++j) tb[j] = 0.6 * lv[j - 1] + 0.4 * lv[j];"),
    ("lloyd_centroid_sign", "double nl = (std_normal_pdf(tb[j]) - std_normal_pdf(tb[j + 1])) / mass;",
     "double nl = (std_normal_pdf(tb[j + 1]) - std_normal_pdf(tb[j])) / mass;"),
    ("wht4_attention_v_from_k", "wht4_dequant_row_f64(blk + ((size_t)P + (size_t)slot) * (size_t)(d / 2),\n                                         get_f32(blk + (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot)), d, rv);",
     "wht4_dequant_row_f64(blk + (size_t)slot * (size_t)(d / 2),\n                                         get_f32(blk + (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot)), d, rv);"),
    ("wht4_attention_gqa_modulo", "int kvh = hq / grp;", "int kvh = hq % Hkv;"),
    ("wht4_sigma_slot_of_k_for_v", "put_f32(blk + (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot), sv);",
     "put_f32(blk + (size_t)P * (size_t)d + (size_t)4 * ((size_t)P + (size_t)slot), sk);"),
    ("attention_not_normalized", "o[i] += p * (double)rv[i];\n            }\n            for (int i = 0; i < d; ++i) o[i] /= l;",
     "o[i] += p * (double)rv[i];\n            }"),
    ("group_amax_signed",
     "float a = fabsf(kvq_oracle_f16_to_f32(x[i]));\n        if (a > amax) amax = a;\n    }\n    float s32",
     "float a = kvq_oracle_f16_to_f32(x[i]);\n        if (a > amax) amax = a;\n    }\n    float s32"),
    ("int8_amax_signed",
     "float a = fabsf(kvq_oracle_f16_to_f32(x[i]));\n        if (a > amax) amax = a;\n    }\n    float s = amax / 127.0f;",
     "float a = kvq_oracle_f16_to_f32(x[i]);\n        if (a > amax) amax = a;\n    }\n    float s = amax / 127.0f;"),
    ("int8_scale_floor_dropped", "    if (s < 1e-8f) s = 1e-8f;\n", ""),
    ("dequant_fp16_v_from_k", "((uint16_t *)out_v)[off + i] = kvq_oracle_f32_to_f16(rv[i]);",
     "((uint16_t *)out_v)[off + i] = kvq_oracle_f32_to_f16(rk[i]);"),
    ("dequant_fp32_v_from_k", "((float *)out_v)[off + i] = rv[i];", "((float *)out_v)[off + i] = rk[i];"),
    ("window_zero_hides_all", "if (window <= 0) return 1;", "if (window <= 0) return 0;"),
    ("mixed_split_from_start", "int split = len - residual > 0 ? len - residual : 0;",
     "int split = residual < len ? residual : len;"),
    ("f16_overflow_saturates", "if (e > 15) return (uint16_t)(sign | 0x7c00u);",
     "if (e > 15) return (uint16_t)(sign | 0x7bffu);"),
    ("f16_mantissa_carry_dropped", "if (m16 == 2048) { m16 = 1024; e += 1; }", "if (m16 == 2048) { m16 = 2047; }"),
    ("f16_to_f64_subnormal_exponent", "v = ldexp((double)fr, -24);", "v = ldexp((double)fr, -25);"),
    ("f16_nan_to_inf", "(ax > 0x7f800000u ? 0x0200u : 0u)", "0u"),
    ("append_token_offset_dropped",
     "            long pos = (long)start_pos[b] + t;\n            if (pos < 0 || pos / P >= max_blocks) return ORACLE_ERANGE;\n            int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];\n            if (page < 0 || page >= num_pages) return ORACLE_ERANGE;\n            int slot = (int)(pos % P);\n            for (int h = 0; h < Hkv; ++h) {\n                size_t off = (((size_t)b * (size_t)n_new",
     "            long pos = (long)start_pos[b];\n            if (pos < 0 || pos / P >= max_blocks) return ORACLE_ERANGE;\n            int page = block_table[(size_t)b * (size_t)max_blocks + (size_t)(pos / P)];\n            if (page < 0 || page >= num_pages) return ORACLE_ERANGE;\n            int slot = (int)(pos % P);\n            for (int h = 0; h < Hkv; ++h) {\n                size_t off = (((size_t)b * (size_t)n_new"),
    ("dequant_start_ignored",
     "    float rk[256], rv[256];\n    for (int t = 0; t < n; ++t) {\n        long pos = (long)start + t;",
     "    float rk[256], rv[256];\n    for (int t = 0; t < n; ++t) {\n        long pos = (long)t;"),
    ("lloyd_single_iteration", "        if (moved <= 1e-15) break;", "        if (moved <= 1e-15 || it >= 1) break;"),
    ("lloyd_loose_tolerance", "        if (moved <= 1e-15) break;", "        if (moved <= 1e-6) break;"),
    ("int8_v_scale_for_k", "rk[i] = (float)(int8_t)blk[(size_t)slot * (size_t)d + (size_t)i] * sk;",
     "rk[i] = (float)(int8_t)blk[(size_t)slot * (size_t)d + (size_t)i] * sv;"),
    ("lloyd_not_symmetrized", "        lv[j] = -a;\n        lv[n - 1 - j] = a;", "        (void)a;"),
]


def _run_mutant(name, old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: anchor occurs {src.count(old)} times"
    mdir = os.path.join(tmp, name)
    os.makedirs(mdir, exist_ok=True)
    msrc = os.path.join(mdir, "kvq_oracle.c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(mdir, "libkvq_oracle.so")
    sys.path.insert(0, ROOT)
    from oracle import build as obuild
    obuild.build(msrc, lib, force=True)
    env = dict(os.environ, KVQ_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_planted_mistake_is_caught(tmp_path):
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = list(ex.map(lambda m: _run_mutant(*m, str(tmp_path)), MUTANTS))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, f"planted mistakes the pins missed: {survivors}"
    # and the unmodified oracle passes the same suite (rc 0) -- run in-process elsewhere
    assert all(rc == 1 for _, rc, _ in results), [(n, rc, out) for n, rc, out in results if rc != 1]
