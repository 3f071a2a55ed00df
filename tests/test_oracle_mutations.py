"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, and runs the pin suite against that build
in a subprocess: the suite has to fail.  The committed oracle is untouched."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "aircache_oracle.c")

MUTATIONS = {
    "elite reads the wrong query row": ("scaled_dot(q, n_t - 1, h,", "scaled_dot(q, n_t - 2, h,"),
    "elite averages logits, not softmax rows": ("P[j] += exp(logit[j] - m) / z;", "P[j] += logit[j];"),
    "elite threshold exclusive": ("if (P[j] >= alpha * mx)", "if (P[j] > alpha * mx)"),
    "head map h mod h_kv": ("const int kvh = h / g;\n        double m = -INFINITY;",
                            "const int kvh = h % h_kv;\n        double m = -INFINITY;"),
    "scale by D instead of sqrt(D)": ("return s / sqrt((double)d);", "return s / (double)d;"),
    "softmax drops the elite text keys": ("for (int c = 0; c < n_keys; ++c) z +=",
                                          "for (int c = 0; c < n_v; ++c) z +="),
    "elite text key index not mapped": ("text_row(n_p, n_v, elite[e2]), kvh, d);", "text_row(n_p, n_v, e2), kvh, d);"),
    "score query row not mapped": ("const int64_t q_tok = elite[e];", "const int64_t q_tok = e;"),
    "I_v not averaged over heads": ("const double norm = (double)h_q * (double)n_tk;",
                                    "const double norm = (double)n_tk;"),
    "population sigma": ("sqrt(ss / (n_v - 1))", "sqrt(ss / n_v)"),
    "skewness prefactor dropped": ("s_k = (double)n_v / ((double)(n_v - 1) * (double)(n_v - 2)) * cube;",
                                   "s_k = cube;"),
    "budget skips the min shift": ("mean_u += s_k[l] - min_sk + 1e-6;", "mean_u += s_k[l] + 1e-6;"),
    "budget uses banker's rounding": ("floor(rl * (double)n_v + 0.5)", "nearbyint(rl * (double)n_v)"),
    "budget drops the 1/2": ("const double rl = 0.5 * (st_n[l] + sk_n[l]) * r;", "const double rl = (st_n[l] + sk_n[l]) * r;"),
    "ties go to the higher index": ("return (x->i > y->i) - (x->i < y->i);", "return (x->i < y->i) - (x->i > y->i);"),
    "selection left in score order": ("    qsort(idx, (size_t)keep, sizeof(int32_t), ascending_int);\n", ""),
    "text rows shifted by one": ("? vis_row(n_p, idx[j]) : text_row(n_p, n_v, j - keep);",
                                 "? vis_row(n_p, idx[j]) : text_row(n_p, n_v, j - keep) - (j > keep);"),
    "per-head I_v normalised over all heads": ("const double norm_h = (double)g * (double)n_tk;",
                                               "const double norm_h = (double)h_q * (double)n_tk;"),
    "per-head I_v all into head 0": ("iv_heads[(int64_t)kvh * n_v + c] +=", "iv_heads[(int64_t)0 * n_v + c] +="),
    "per-head compaction reads head 0's set": ("vis_row(n_p, idx_heads[(int64_t)h * n_v + j])",
                                               "vis_row(n_p, idx_heads[j])"),
    "visual window scores the text keys too": ("for (int c = 0; c < n_v; ++c) z += exp(logit[c] - m);\n            for (int c = 0; c < n_v; ++c) iv[c] +=",
                                               "for (int c = 0; c < n_v; ++c) z += exp(logit[c] - m);\n            z += 1.0;\n            for (int c = 0; c < n_v; ++c) iv[c] +="),
    "visual window reads the first visual tokens": ("for (int e = 0; e < w; ++e) positions[e] = n_v - w + e;",
                                                    "for (int e = 0; e < w; ++e) positions[e] = e;"),
    "visual rows ignore the prefix": ("return (int64_t)n_p + i;", "return (int64_t)i;"),
    "text rows ignore the prefix": ("return j < n_p ? (int64_t)j : (int64_t)n_v + j;", "return (int64_t)n_v + j;"),
    "decode head map h mod h_kv": ("const int kv_head = h / group;", "const int kv_head = h % h_kv;"),
    "decode weights not normalised": ("acc += w[j] / total * elem(v, j, kv_head, i);",
                                      "acc += w[j] * elem(v, j, kv_head, i);"),
    "decode reads keys as values": ("acc += w[j] / total * elem(v, j, kv_head, i);",
                                    "acc += w[j] / total * elem(k, j, kv_head, i);"),
    "decode drops the last row": ("for (int64_t j = 0; j < n_rows; ++j) acc +=",
                                  "for (int64_t j = 0; j + 1 < n_rows; ++j) acc +="),
    "decode logits unscaled": ("w[j] = scaled_dot(q, 0, h, k, j, kv_head, d);",
                               "w[j] = scaled_dot(q, 0, h, k, j, kv_head, d) * sqrt((double)d);"),
    "quantization rounds half to even": ("float r = roundf(t);", "float r = rintf(t);"),
    "quantization truncates": ("float r = roundf(t);", "float r = truncf(t);"),
    "quantization range 128": ("const float s = big / 127.0f;", "const float s = big / 128.0f;"),
    "one head's scale for every head": ("const float a = fabsf((float)elem(src, j, h, i));",
                                        "const float a = fabsf((float)elem(src, j, 0, i));"),
}
PIN_FILES = ["test_oracle_pins.py", "test_oracle_variants.py", "test_oracle_decode.py", "test_oracle_quant.py",
             "test_oracle_prefix.py", "test_oracle_heads.py", "test_oracle_visual_window.py"]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation anchor not unique/found: {name}"
    mutated = tmp_path / "aircache_oracle.c"
    mutated.write_text(src.replace(before, after))
    (tmp_path / "aircache_oracle.h").write_text(open(os.path.join(ROOT, "oracle", "aircache_oracle.h")).read())
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           "-o", str(so), str(mutated), "-lm"])
    env = dict(os.environ, AIRCACHE_ORACLE_LIB=str(so))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          *[os.path.join(ROOT, "tests", f) for f in PIN_FILES]],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"pins did not catch: {name}\n{res.stdout[-2000:]}"
