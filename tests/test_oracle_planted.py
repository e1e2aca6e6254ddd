"""Planted faults in the oracle must turn its pin suite red.

The six fault classes are the ones "Qwen3.5 batched prefill has no f32
dequant for IQ2_XXS, IQ3_S, IQ3_XXS, Q2_K" (§Acceptance) plants in its
kernels: signs, high bits, scale selector, d, row stride and tail guard;
a seventh plants a Q5_K high-bit-plane index slip.
Each is planted in a copy of the oracle source on the CPU, compiled, and the
pin tests are run against that copy (QPO_LIB); they must fail.  The restored
oracle passing is the rest of the suite.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qpo.c")

PLANTS = {
    "signs": ("const float q = (float)(int8_t)b[2 + v];", "const float q = (float)(uint8_t)b[2 + v];"),
    "high_bits": ("*sc = (scales[s + 4] & 0x0f) | ((scales[s - 4] >> 6) << 4);",
                  "*sc = (scales[s + 4] & 0x0f) | ((scales[s - 4] >> 6) << 5);"),
    "scale_selector": ("const int sc = scales[s] & 0x0f;", "const int sc = scales[s ^ 1] & 0x0f;"),
    "d": ("const float dl = d * (float)sc;\n    const float ml = dmin * (float)m;\n    const float dq = dl * (float)q;\n    return dq - ml;\n}\n\n/* Q2_K",
          "const float dl = dmin * (float)sc;\n    const float ml = dmin * (float)m;\n    const float dq = dl * (float)q;\n    return dq - ml;\n}\n\n/* Q2_K"),
    "row_stride": ("const int64_t nb = (cols + qk - 1) / qk;\n    const uint8_t *base = (const uint8_t *)blocks;\n#pragma omp parallel for schedule(static)\n    for (int64_t r = 0; r < rows; ++r) {\n        for (int64_t c = 0; c < cols; ++c) {\n            const uint8_t *blk = base + (r * nb + c / qk) * bb;\n            out[r * cols + c] = qpo_decode_value",
                   "const int64_t nb = cols / qk;\n    const uint8_t *base = (const uint8_t *)blocks;\n#pragma omp parallel for schedule(static)\n    for (int64_t r = 0; r < rows; ++r) {\n        for (int64_t c = 0; c < cols; ++c) {\n            const uint8_t *blk = base + (r * nb + c / qk) * bb;\n            out[r * cols + c] = qpo_decode_value"),
    # writes the padding values of a partial last block (into the next row,
    # and for the last row into the wrapper's NaN guard band)
    # the fifth bit of a Q5_K value taken from the neighbouring sub-block's bit
    "q5_k_high_bit": ("const int q = lo | (((qh[l] >> s) & 1) << 4);",
                      "const int q = lo | (((qh[l] >> (s ^ 1)) & 1) << 4);"),
    "tail_guard": ("for (int64_t c = 0; c < cols; ++c) {\n            const uint8_t *blk = base + (r * nb + c / qk) * bb;\n            out[r * cols + c] = qpo_decode_value(type, blk, (int)(c % qk));",
                   "for (int64_t c = 0; c < nb * qk; ++c) {\n            const uint8_t *blk = base + (r * nb + c / qk) * bb;\n            out[r * cols + c] = qpo_decode_value(type, blk, (int)(c % qk));"),
}


@pytest.mark.parametrize("name", sorted(PLANTS))
def test_planted_fault_is_caught(name, tmp_path):
    src = open(SRC).read()
    old, new = PLANTS[name]
    assert src.count(old) >= 1, "plant site for %s not found" % name
    mutated = src.replace(old, new, 1)
    c = tmp_path / "qpo.c"
    c.write_text(mutated)
    (tmp_path / "qpo.h").write_text(open(os.path.join(ROOT, "oracle", "qpo.h")).read())
    so = tmp_path / "libqpo_planted.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", "-fopenmp", "-o", str(so), str(c), "-lm"])
    env = dict(os.environ, QPO_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "planted fault %s passed the pin suite:\n%s" % (name, r.stdout[-2000:])
