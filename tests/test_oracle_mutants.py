"""The pins catch plausible mistakes: each mutant below plants one in a copy
of the oracle's C source (on the CPU only), builds it, and runs the pin suite
against it; every mutant must make at least one pin fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qsa_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("no_relu", "float r = acc > 0.0f ? acc : 0.0f;", "float r = acc;"),
    ("relu_after_head_sum", "float r = acc > 0.0f ? acc : 0.0f;\n        s = s + r;",
     "s = s + acc;"),
    ("pool_drops_a_key", "acc = acc + k4[3 * d + j];", ""),
    ("pool_wrong_row", "acc = acc + k4[2 * d + j];", "acc = acc + k4[1 * d + j];"),
    ("dot_ignores_head", "fmaf(q[(int64_t)h * d + j], p[j], acc)", "fmaf(q[j], p[j], acc)"),
    ("ties_prefer_later", "return (x->g > y->g) - (x->g < y->g);",
     "return (x->g < y->g) - (x->g > y->g);"),
    ("rank_order_emission", "qsort(chosen, (size_t)k, sizeof(int32_t), qsao_cmp_pos);", ""),
    ("no_tail", "for (int32_t t = QSAO_GROUP * G; t < T; ++t) ids[n++] = t;  /* raw tail */", ""),
    ("tail_first_group_dropped", "for (int32_t r = 0; r < k; ++r)\n        for (int32_t u",
     "for (int32_t r = (k > 0 && G > budget); r < k; ++r)\n        for (int32_t u"),
    ("denominator_not_rescaled", "l = l * alpha + p;", "l = l + p;"),
    ("acc_not_rescaled", "acc[j] = acc[j] * alpha + p * v[j];", "acc[j] = acc[j] + p * v[j];"),
    ("wrong_kv_head", "int32_t kvh = h / group;", "int32_t kvh = h % n_kv;"),
    ("scale_dropped", "float x = scale * dot;", "float x = dot;"),
    ("slot_map_skipped", "int32_t s = slot_map[ids[i]];", "int32_t s = ids[i];"),
]


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, orig, bad):
    import oracle
    src = open(SRC).read()
    assert src.count(orig) == 1, name
    mut_src = tmp_path / f"{name}.c"
    mut_src.write_text(src.replace(orig, bad))
    so = oracle.build(force=True, out=str(tmp_path / f"lib_{name}.so"), src=str(mut_src))
    env = dict(os.environ, QSA_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout or "error" in r.stdout.lower()
