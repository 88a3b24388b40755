"""Plant plausible mistakes in a copy of the oracle's C source and check that
the pins in test_oracle_pins.py catch every one of them (CPU only)."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "mla_oracle.c")

MUTANTS = {
    "scale dropped": ("s[j] = dot(q, kbase + r * Dqk, Dqk) * scale;",
                      "s[j] = dot(q, kbase + r * Dqk, Dqk);"),
    "mask off by one": ("int64_t n = P + i + 1;", "int64_t n = P + i + (i > 0);"),
    "min for max": ("if (s[j] > m) m = s[j];", "if (s[j] < m) m = s[j];"),
    "gate sign": ("out[d] = g ? z[d] * sigmoid(g[d]) : z[d];",
                  "out[d] = g ? z[d] * sigmoid(-g[d]) : z[d];"),
    "output transposed": ("int64_t o = (((int64_t)b * Tq + i) * H + h) * Dv;",
                          "int64_t o = (((int64_t)b * H + h) * Tq + i) * Dv;"),
    "unnormalised denominator": ("denom += exp(s[j] - m);", "denom += exp(s[j]);"),
    "relu dropped": ("(zh > 0.0 ? zh : 0.0)", "zh"),
    "tie-break reversed": ("return (x->pos > y->pos) - (x->pos < y->pos);",
                           "return (x->pos < y->pos) - (x->pos > y->pos);"),
    "lowest scores kept": ("if (x->score > y->score) return -1;",
                           "if (x->score < y->score) return -2;"),
    "decode drops last key": ("attend(qb, kb, vb, NULL, T, Dqk, Dv, scale, z, NULL)",
                              "attend(qb, kb, vb, NULL, T > 1 ? T - 1 : T, Dqk, Dv, scale, z, NULL)"),
    "decode query index transposed": ("const double* qb = q + ((int64_t)b * H + h) * Dqk;\n"
                                      "            err |= attend(qb, kb, vb, NULL, T,",
                                      "const double* qb = q + ((int64_t)h * B + b) * Dqk;\n"
                                      "            err |= attend(qb, kb, vb, NULL, T,"),
    "sparse skips position 0": ("if (s >= 0) pos[n++] = s;", "if (s > 0) pos[n++] = s;"),
    "sparse reads padding as position 0": ("if (s >= 0) pos[n++] = s;",
                                           "pos[n++] = s < 0 ? 0 : s;"),
    "index weights of the first sequence": ("acc += w[(int64_t)b * NH + h] *",
                                            "acc += w[h] *"),
    "index query of the first sequence": ("dot(iq + ((int64_t)b * NH + h) * Di, ks, Di)",
                                          "dot(iq + (int64_t)h * Di, ks, Di)"),
    "index scores without the sequence offset": ("scores[cu[b] + s] = acc;",
                                                 "scores[s] = acc;"),
    "top-k left in rank order": ("qsort(row, (size_t)kk, sizeof(int32_t), by_value);", ""),
    "prefill keys of head 0": ("const double* kb = k + ((int64_t)b * H + h) * Tk * Dqk;",
                               "const double* kb = k + ((int64_t)b * H) * Tk * Dqk;"),
    "probabilities not normalised": ("double pj = exp(s[j] - m) / denom;",
                                     "double pj = exp(s[j] - m);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.build(force=True, out=str(tmp_path / "libmutant.so"), src=str(mutant_src))
    env = dict(os.environ, MLA_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"planted mistake '{name}' passed every pin"
