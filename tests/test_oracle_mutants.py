"""Plant plausible mistakes in copies of the oracle (on the CPU only) and
check that the pin suite catches every one of them."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "csa_oracle.c")
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_visibility.py", "tests/test_oracle_indexer.py",
        "tests/test_oracle_topk.py", "tests/test_oracle_attention.py", "tests/test_oracle_epilogue.py"]

MUTANTS = {
    "relu_dropped": ("acc += (double)w[h] * (dot > 0.0 ? dot : 0.0);", "acc += (double)w[h] * dot;"),
    "query_scale_dropped": ("* (double)q_scale[h];", ";"),
    "key_scale_dropped": ("(oracle_e4m3_value(k8[(size_t)c * Di + d]) * (double)k_scale[c]);",
                          "(oracle_e4m3_value(k8[(size_t)c * Di + d]));"),
    "visible_off_by_one": ("nv = p / m;", "nv = (p + 1) / m;"),
    "window_excludes_own_token": ("for (j = swa_first(p, W); j <= p; ++j)", "for (j = swa_first(p, W); j < p; ++j)"),
    "window_one_too_long": ("int j0 = p - W + 1;", "int j0 = p - W;"),
    "ring_slot_mod_window": ("(j % R)", "(j % W)"),
    "sink_dropped_from_denominator": ("den = exp((double)sink[h] - M);", "den = 0.0;"),
    "sink_not_in_running_max": ("double M = (double)sink[h], den;", "double M = -INFINITY, den;"),
    "softmax_scale_dropped": ("z[j] = scale * dot;", "z[j] = dot;"),
    "lse_missing_max": ("lse[h] = M + log(den);", "lse[h] = log(den);"),
    "scale_block_wrong_size": ("f32_at(scales + 4 * (d / SB))", "f32_at(scales + 4 * (d / (2 * SB)))"),
    "rope_reversed": ("oracle_bf16_value(u16_at(rope + 2 * r))", "oracle_bf16_value(u16_at(rope + 2 * (Dr - 1 - r)))"),
    "e4m3_bias_8": ("ldexp(1.0 + (double)mant / 8.0, expo - 7)", "ldexp(1.0 + (double)mant / 8.0, expo - 8)"),
    "e4m3_subnormal_hidden_one": ("ldexp((double)mant / 8.0, -6)", "ldexp(1.0 + (double)mant / 8.0, -6)"),
    "bf16_low_half": ("uint32_t u = (uint32_t)bits << 16;", "uint32_t u = (uint32_t)bits << 15;"),
    "topk_ties_to_higher_index": ("return (x->index > y->index) - (x->index < y->index);",
                                  "return (x->index < y->index) - (x->index > y->index);"),
    "topk_smallest_first": ("if (x->score > y->score)\n        return -1;", "if (x->score < y->score)\n        return -1;"),
    "page_index_wrong": ("int page = c / page_records;", "int page = c % page_records;"),
    "seq_stride_ignored": ("rec = (int64_t)b * seq_stride + c;", "rec = (int64_t)b + c;"),
    "selected_list_truncated": ("for (i = 0; i < cnt; ++i) {\n        const uint8_t *rec", "for (i = 1; i < cnt; ++i) {\n        const uint8_t *rec"),
    "e2m1_bias_0": ("ldexp(1.0 + (double)mant / 2.0, expo - 1)", "ldexp(1.0 + (double)mant / 2.0, expo)"),
    "e2m1_ties_to_odd": ("(c & 1) == 0 && (best & 1) == 1", "(c & 1) == 1 && (best & 1) == 0"),
    "e2m1_scale_amax_over_4": ("s = amax > 0.0 ? amax / 6.0 : 1.0;", "s = amax > 0.0 ? amax / 4.0 : 1.0;"),
    "inverse_rope_turns_forward": ("double c = cos(a), s = sin(a);", "double c = cos(a), s = -sin(a);"),
    "rope_frequency_exponent": ("pow(theta, -2.0 * (double)i / (double)Dr)", "pow(theta, -(double)i / (double)Dr)"),
    "value_uses_query_not_latent": ("acc += exp(z[j] - M) * x[(size_t)j * D + d];", "acc += exp(z[j] - M) * qd[d];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(lib), str(mut), "-lm"],
                   check=True)
    env = dict(os.environ, CSA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
