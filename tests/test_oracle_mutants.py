"""Planted mistakes in a copy of the oracle must each fail some oracle pin.

Every mutant below is a plausible slip (a dropped term, a wrong sign, index or
layout, a transposed operand).  The copy is compiled on the CPU into a temp
directory and the pin suite (tests/test_oracle.py) is run against it in a
subprocess; the suite must fail.  The real oracle source is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

# (name, text in pkv_oracle.c, replacement)
MUTANTS = [
    ("kv-head-mapping", "int32_t g = h / G;\n    const uint16_t *qh",
     "int32_t g = h % Hkv;\n    const uint16_t *qh"),
    ("dropped-scale", "s[t - t0] = scale * dot;", "s[t - t0] = dot;"),
    ("slot-index", "int64_t slot = t % P;", "int64_t slot = (t + 1) % P;"),
    ("page-index", "bt[(int64_t)i * bt_stride + t / P]", "bt[(int64_t)i * bt_stride + t % P]"),
    ("hnd-layout", "return ((page * P + slot) * Hkv + g) * (int64_t)d;",
     "return ((page * Hkv + g) * P + slot) * (int64_t)d;"),
    ("no-normalise", "            out[c] /= L;\n        lse[r] = M + log(L);",
     "            out[c] /= 1.0;\n        lse[r] = M + log(L);"),
    ("lse-drops-max", "lse[r] = M + log(L);", "lse[r] = log(L);"),
    ("unshifted-exp", "double w = exp(s[t] - M);", "double w = exp(s[t]);"),
    ("merge-drops-rescale", "L += l[slot] * w;", "L += l[slot];"),
    ("merge-acc-unscaled", "out[c] += acc[slot * d + c] * w;", "out[c] += acc[slot * d + c];"),
    ("partial-wrong-max", "double w = exp(s[t - t0] - mj);", "double w = exp(s[t - t0]);"),
    ("plan-state-base", "rec[3] = (int32_t)((o + j) * Hq + (int64_t)g * G);",
     "rec[3] = (int32_t)((o + j) * Hq + (int64_t)g);"),
    ("plan-floor", "int64_t n = (N + C - 1) / C;\n        if (offsets)",
     "int64_t n = N / C;\n        if (offsets)"),
    ("half-exponent-bias", "v = ldexp((double)(1024 + f), e - 25);",
     "v = ldexp((double)(1024 + f), e - 24);"),
    ("half-subnormal", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    ("neutral-state", "                m[slot] = -INFINITY;\n                l[slot] = 0.0;",
     "                m[slot] = 0.0;\n                l[slot] = 0.0;"),
    ("exact-bucket-count", "out->attn_launches = 2 * distinct;", "out->attn_launches = 2 * B;"),
    ("rect-empty-flag", "empty[T] = ((int64_t)j * C >= seq_lens[i]) ? 1 : 0;",
     "empty[T] = ((int64_t)j * C > seq_lens[i]) ? 1 : 0;"),
    ("rect-writes-only-nonempty", "out->states_written = (int64_t)B * S_b * Hq;",
     "out->states_written = sum_n * Hq;"),
    ("state-bytes-drop-ml", "int64_t state_bytes = (int64_t)(d + 2) * 4;",
     "int64_t state_bytes = (int64_t)d * 4;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(name, old, new, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique/found"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", str(mutant), "-o",
                    str(lib), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, PKV_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
