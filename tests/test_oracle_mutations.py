"""The pins of the C oracle catch plausible mistakes in it.

Each case below copies oracle/attn_oracle.c with one planted mistake, builds the copy into a
temporary library and runs tests/test_oracle_pins.py against it (through the oracle package's
ORACLE_LIB_OVERRIDE hook): at least one pin must fail.  An unchanged copy built the same way
must pass them all, so a failure comes from the mistake and not from the build route.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "attn_oracle.c")

# (id, text in attn_oracle.c, replacement, occurrences replaced)
MUTATIONS = [
    # causal mask on the wrong side of the diagonal
    ("mask_side", "if (causal && j > i + off)", "if (causal && j < i + off)", 1),
    # grouped-query heads interleaved instead of contiguous
    ("gqa_modulo", "const int64_t hk = h / group;", "const int64_t hk = h % Hkv;", 2),
    # the scale left out of the scores
    ("scale_dropped", "s[j] = scale * acc;", "s[j] = acc;", 2),
    # the row maximum left out of L = m + ln l
    ("lse_without_m", "*lse = m + log(l);", "*lse = log(l);", 2),
    # the probabilities not normalised
    ("p_unnormalised", "p[j] = exp(s[j] - m) / l;", "p[j] = exp(s[j] - m);", 2),
    # the online recurrence forgets to rescale the running sum
    ("alpha_dropped_from_l", "l = alpha * l + bsum;", "l = l + bsum;", 1),
    # the merge weighs the first state by its exponential alone
    ("l1_dropped_from_merge", "exp(m1 - mm) * l1;", "exp(m1 - mm);", 1),
    # key rows read in reverse order
    ("k_rows_reversed", "const double *kr = kd + plane + j * d;",
     "const double *kr = kd + plane + (Nkv - 1 - j) * d;", 1),
    # the window one key too wide
    ("window_off_by_one", "i + off - j > window", "i + off - j > window + 1", 1),
    # fp16 exponent bias off by one
    ("f16_bias", "ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)", 1),
]


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    lib = tmp_path / f"lib{name}.so"
    src.write_text(text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(src), "-o",
                    str(lib), "-lm"], check=True)
    return str(lib)


def _run_pins(lib):
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=lib, OMP_NUM_THREADS="4")
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           "-m", "not gpu", os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unchanged_copy_passes_the_pins(tmp_path):
    with open(SRC) as f:
        text = f.read()
    r = _run_pins(_build(tmp_path, "unchanged", text))
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name,old,new,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new, count):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) == count, f"{name}: expected {count} occurrence(s) of {old!r}"
    r = _run_pins(_build(tmp_path, name, text.replace(old, new)))
    # exit code 1: a test failed (not a collection or usage error)
    assert r.returncode == 1, f"{name}: the pins passed or did not run\n" + r.stdout[-2000:]
    assert "failed" in r.stdout, r.stdout[-2000:]
