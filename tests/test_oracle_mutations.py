"""Mutation check of the oracle pins (CPU only).

Each case plants one plausible mistake in a private copy of the oracle's C source,
compiles it, and runs the pin suite against it in a subprocess: the pins must fail.
This shows the pins constrain the oracle rather than restate it.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "bf16 double rounding through fp32": ("double a = fabs(v);", "double a = (double)(float)fabs(v);"),
    "bf16 ties away from zero": ("ldexp(rint(n), qexp)", "ldexp(round(n), qexp)"),
    "dot product drops the last term": ("for (int k = 0; k < K; ++k)", "for (int k = 0; k + 1 < K; ++k)"),
    "residual subtracted": ("s += oracle_bf16_to_double(R[(int64_t)b * N + n]);",
                            "s -= oracle_bf16_to_double(R[(int64_t)b * N + n]);"),
    "ties to the higher index": ("if (best < 0 || v > bestv)", "if (best < 0 || v >= bestv)"),
    "weights not renormalised over top-k": ("exp(l[idx[(int64_t)b * topk + j]] - m) / zs;",
                                            "exp(l[idx[(int64_t)b * topk + j]] - m) / z;"),
    "gate and up swapped": ("double g = dot_bf16(x, Wgu + (int64_t)i * H, H);",
                            "double g = dot_bf16(x, Wgu + (int64_t)(I + i) * H, H);"),
    "silu sign": ("return t / (1.0 + exp(-t));", "return t / (1.0 + exp(t));"),
    "shared expert dropped": ("acc += s[(int64_t)b * H + h];", "acc += 0.0 * s[(int64_t)b * H + h];"),
    "latent taken from router rows": ("oracle_bf16_from_double(z[(int64_t)b * N + E + i])",
                                      "oracle_bf16_from_double(z[(int64_t)b * N + i])"),
    "route map pairs unsorted within expert": ("pairs[at] = p;", "pairs[offsets[e + 1] - 1 - (at - offsets[e])] = p;"),
    "combine weight index transposed": ("acc += w[(int64_t)b * topk + j]", "acc += w[(int64_t)j * topk + (b % topk)]"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    str(mutated), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch: {name}\n{r.stdout[-2000:]}"
