"""Every plausible mistake planted in a copy of the C oracle must trip a pin.

The planted mistakes live only in temporary copies compiled here on the CPU;
the oracle source itself is untouched.
"""
import os
import subprocess

import pytest

import oracle as O
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(O.__file__), "pa_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("offset_shift", "*offset = (int32_t)(i % B);", "*offset = (int32_t)((i + 1) % B);"),
    ("block_index", "int64_t block_idx = i / B;", "int64_t block_idx = (i + 1) / B;"),
    ("gqa_head_map", "int hkv = h / G; /* consecutive", "int hkv = h % p->Hkv; /* consecutive"),
    ("garbled_key_term", "(d / x) * B * x + slot * x + d % x", "(d / x) * B + slot * x + d % x"),
    ("value_prior_transposed", "head * kv_head_stride + d * B + slot;", "head * kv_head_stride + slot * D + d;"),
    ("normaliser_unshifted", "den += exp(scores[i] - mx);", "den += exp(scores[i]);"),
    ("no_max_subtraction", "double mx = -INFINITY;\n    for (int64_t i = 0; i < L; ++i) mx = scores[i] > mx ? scores[i] : mx;",
     "double mx = 0.0;"),
    ("dropped_scale", "scores[i - t0] = p->scale * dot;", "scores[i - t0] = dot;"),
    ("q_transposed", "((int64_t)s * p->Hq + h) * p->D + d", "((int64_t)h * p->N + s) * p->D + d"),
    ("f16_exponent", "ldexp((double)(1024 + m), e - 25)", "ldexp((double)(1024 + m), e - 24)"),
    ("f16_subnormal", "ldexp((double)m, -24)", "ldexp((double)m, -25)"),
    ("bf16_shift", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("merge_weight_dropped", "den += exp(m[part] - mstar) * l[part];", "den += l[part];"),
    ("slot_decode_swapped", "int64_t block = slot / B, off = slot % B;", "int64_t block = slot % B, off = slot / B;"),
    ("copy_direction", "int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];",
     "int32_t dst = pairs[2 * i], src = pairs[2 * i + 1];"),
    ("padding_written", "if (slot < 0) continue;", "if (slot < 0) slot = -slot;"),
    ("alibi_sign", "p->alibi[h] * (double)(i - (p->seq_lens[s] - 1))", "p->alibi[h] * (double)((p->seq_lens[s] - 1) - i)"),
    ("prefill_causal_offset", "const int32_t len = (int32_t)(pos + 1);", "const int32_t len = (int32_t)(pos + 2);"),
    ("prefill_query_origin", "const int64_t pos = seq_lens[s] - n + (t - query_start[s]);",
     "const int64_t pos = seq_lens[s] - n + t;"),
    ("alibi_kv_head_slope", "p->alibi[h] * (double)(i", "p->alibi[h / (p->Hq / p->Hkv)] * (double)(i"),
    ("e4m3_bias", "ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 9)"),
    ("e4m3_subnormal", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -8);"),
    ("e4m3_round_down", "nearbyint(a / ldexp(1.0, e - 3))", "floor(a / ldexp(1.0, e - 3))"),
    ("e4m3_no_saturation", "if (v > 448.0) return sign | 0x7E;", "if (v > 480.0) return sign | 0x7E;"),
    ("fp8_value_layout", "if (layout == PAO_LAYOUT_FP8) return pao_value_offset_fp8(",
     "if (layout == PAO_LAYOUT_FP8) return pao_value_offset_prior("),
    ("fp8_value_tile", "(slot / 16) * D * 16 + d * 16 + slot % 16", "(slot / 16) * D * 16 + d * 16 + slot % 8"),
    ("fp8_v_scale_dropped", "return p->v_scale * pao_load(", "return pao_load("),
    ("fp8_k_scale_dropped", "double kd = p->k_scale *", "double kd = 1.0 *"),
    ("fp8_append_value_offset", "v_cache[pao_value_offset_fp8(blk, h, off, d, Hkv, B, D)]",
     "v_cache[pao_offset_ours(blk, h, off, d, Hkv, B, D)]"),
    ("fp8_append_slot_swapped", "const int64_t blk = sl / B, off = sl % B;", "const int64_t blk = sl % B, off = sl / B;"),
    ("fp8_append_padding_written", "if (sl < 0) continue; /* padding token */", "if (sl < 0) sl = -sl;"),
    ("fp8_append_scale_multiplied", "const float rk = xk / k_scale, rv = xv / v_scale;",
     "const float rk = xk * k_scale, rv = xv / v_scale;"),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: anchor text must occur exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(path), "-o", str(lib), "-lm"],
                   check=True)
    return str(lib)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    path = _build_mutant(tmp_path, name, old, new)
    caught = None
    with O.use_library(path):
        for pin in ALL_PINS:
            try:
                pin()
            except (AssertionError, O.OracleError) as e:  # the pin noticed
                caught = pin.__name__
                break
    assert caught is not None, f"planted mistake {name} passed every pin"
