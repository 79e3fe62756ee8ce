"""The oracle's pins catch plausible mistakes: each mutant below is oracle.c
with one planted mistake (a dropped term, a wrong sign, index or bound, a
different reading of the pages), compiled on the CPU; the oracle pins
(test_oracle.py, test_oracle_properties.py) run against it in a separate
process and must fail. CPU only."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = [
    ("bf16 rounding ties away from zero",
     "double n = nearbyint(a / q);", "double n = floor(a / q + 0.5);"),
    ("bf16 rounding truncates", "double n = nearbyint(a / q);", "double n = trunc(a / q);"),
    ("gate weights read transposed",
     "oracle_bf16_to_double(W[(int64_t)e * H + h]);", "oracle_bf16_to_double(W[(int64_t)h * E + e]);"),
    ("bias dropped", "acc += (double)bias[e];", "acc += 0.0;"),
    ("ties go to the highest id",
     "return (a->id < b->id) ? -1 : (a->id > b->id);", "return (a->id > b->id) ? -1 : (a->id < b->id);"),
    ("softmax not renormalised over the top-k",
     "int nden = renormalize ? k : E;", "int nden = E;"),
    ("renormalised even when renormalize = 0",
     "int nden = renormalize ? k : E;", "int nden = k;"),
    ("sigmoid sign flipped", "(1.0 / (1.0 + exp(-s)))", "(1.0 / (1.0 + exp(s)))"),
    ("shared scale dropped",
     "return (float)((double)scale * (1.0 / (1.0 + exp(-s))));",
     "return (float)(1.0 / (1.0 + exp(-s)));"),
    ("shared logit rounded to bf16 before the sigmoid without the flag",
     "double sr = shared_bf16 ? oracle_bf16_to_double(oracle_bf16_from_double(s)) : s;",
     "double sr = oracle_bf16_to_double(oracle_bf16_from_double(s));"),
    ("shared_bf16 flag ignored",
     "double sr = shared_bf16 ? oracle_bf16_to_double(oracle_bf16_from_double(s)) : s;",
     "double sr = s;"),
    ("top-k on the unrounded logits", "oracle_select(E, k, renormalize, zh, ids",
     "oracle_select(E, k, renormalize, z, ids"),
    ("tier boundary inclusive",
     "< (int64_t)128 * num_experts) ? 64 : 128;", "<= (int64_t)128 * num_experts) ? 64 : 128;"),
    ("capacity one row too large",
     "return numel + (int64_t)num_experts * (A - 1);", "return numel + (int64_t)num_experts * A;"),
    ("full blocks padded again",
     "off[e + 1] = off[e] + (cnt[e] + A - 1) / A * A;", "off[e + 1] = off[e] + (cnt[e] + A) / A * A;"),
    ("untouched experts get a block",
     "off[e + 1] = off[e] + (cnt[e] + A - 1) / A * A;",
     "off[e + 1] = off[e] + (cnt[e] + A - 1) / A * A + (cnt[e] == 0 ? A : 0);"),
    ("padding sentinel 0", "sorted[p] = (int32_t)numel;", "sorted[p] = 0;"),
    ("EPLB replica chosen by slot instead of token",
     "int p = map[(int64_t)e * max_replicas + (int)(t % count[e])];",
     "int p = map[(int64_t)e * max_replicas + (int)(i % count[e])];"),
    ("EPLB remap skipped", "phys[i] = p;", "phys[i] = e;"),
    ("e4m3 truncates", "double m = nearbyint(a / step);", "double m = trunc(a / step);"),
    ("e4m3 overflow to NaN instead of saturating",
     "if (a >= 448.0) return (uint8_t)(sign | 0x7E);", "if (a >= 464.0) return (uint8_t)(sign | 0x7F);"),
    ("block scale over 240 instead of 448",
     "float scale = (float)(amax / 448.0);", "float scale = (float)(amax / 240.0);"),
    ("codes from the unscaled values",
     "float v = (float)(oracle_bf16_to_double(xb[i]) * (double)inv);",
     "float v = (float)(oracle_bf16_to_double(xb[i]));"),
    ("expert GEMM reads the slot's expert from the wrong slot",
     "const uint16_t *we = W + (int64_t)ids[i] * N * H;",
     "const uint16_t *we = W + (int64_t)ids[i / width * width] * N * H;"),
    ("expert GEMM weights read transposed",
     "oracle_bf16_to_double(we[(int64_t)n * H + h]);", "oracle_bf16_to_double(we[(int64_t)h * N + n]);"),
    ("descending order inside an expert",
     "for (int64_t i = 0; i < numel; ++i) sorted[cur[ids[i]]++] = (int32_t)i;",
     "for (int64_t i = numel - 1; i >= 0; --i) sorted[cur[ids[i]]++] = (int32_t)i;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not found: {old}"
    mut = tmp_path / "oracle_mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
                           "-ffp-contract=off", "-o", str(lib), str(mut), "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py"),
                        os.path.join(ROOT, "tests", "test_oracle_properties.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    # exit code 1: the pins ran and at least one failed (2+ would mean they
    # could not run at all)
    assert r.returncode == 1, f"{name}: pins did not fail (exit {r.returncode})\n{r.stdout[-2000:]}"
