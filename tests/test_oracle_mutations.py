"""Plant plausible mistakes in copies of the oracle's C source and check that
the pins catch every one (CPU only).  The oracle under test is never edited;
each mutant is compiled to a temporary library and run in a process of its
own."""
import json
import os
import subprocess
import sys

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")
PINS = os.path.join(os.path.dirname(os.path.abspath(__file__)), "pins.py")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text to replace, replacement, which occurrence (0-based))
MUTANTS = [
    ("scale dropped", "x[t - t0] = scale * dot;", "x[t - t0] = dot;", 0),
    ("gqa map modulo", "int g = h / (H / Hkv);", "int g = h % Hkv;", 0),
    ("offset shifted", "*off = (int32_t)(t % B);", "*off = (int32_t)((t + 1) % B);", 0),
    ("logical block used as physical", "*phys = table_row[t / B];", "*phys = (int32_t)(t / B);", 0),
    ("no normalisation", "o[i] = l > 0.0 ? o[i] / l : 0.0;", "o[i] = l > 0.0 ? o[i] : 0.0;", 0),
    ("value read from key cache", "const uint16_t *v = value_cache +", "const uint16_t *v = key_cache +", 0),
    ("last token dropped from PV", "for (int64_t t = t0; t < t1; t++) {", "for (int64_t t = t0; t + 1 < t1; t++) {", 1),
    ("half exponent bias", "e - 15 - 10", "e - 14 - 10", 0),
    ("half subnormal scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)", 0),
    ("bfloat16 shift", "(uint32_t)b << 16", "(uint32_t)b << 15", 0),
    ("cache write offset", "int64_t blk = s / B, off = s % B;", "int64_t blk = s / B, off = (s + 1) % B;", 0),
    ("negative slot not skipped", "if (s < 0)\n            continue;", "if (s < -1)\n            continue;", 0),
    ("copy direction swapped",
     "cache[(int64_t)dst * block_elems + i] = cache[(int64_t)src * block_elems + i];",
     "cache[(int64_t)src * block_elems + i] = cache[(int64_t)dst * block_elems + i];", 0),
    ("merge ignores partition weight", "L += l[p] * w;", "L += l[p];", 0),
    ("partition end off by one", "int64_t t1 = t0 + P < ctx ? t0 + P : ctx;",
     "int64_t t1 = t0 + P < ctx ? t0 + P - 1 : ctx;", 0),
    ("prefill own token not attended", "0, p + 1, B, Hkv,", "0, p, B, Hkv,", 0),
    ("prefill prefix ignored", "int64_t p = context_lens[s] - n + (tok - query_start[s]);",
     "int64_t p = tok - query_start[s];", 0),
    ("prefill sequence search off by one", "while (query_start[s + 1] <= tok)", "while (query_start[s + 1] < tok)", 0),
    ("prefill gqa map modulo", "h / (H / Hkv), d, scale, is_bf16, &m, &l, o, x);",
     "h % Hkv, d, scale, is_bf16, &m, &l, o, x);", 0),
    ("prefill no normalisation", "o[i] = l > 0.0 ? o[i] / l : 0.0;", "o[i] = l > 0.0 ? o[i] : 0.0;", 1),
    ("copy between pools reversed", "dst_pool[(int64_t)dst * block_elems + i] = src_pool[(int64_t)src * block_elems + i];",
     "dst_pool[(int64_t)src * block_elems + i] = src_pool[(int64_t)dst * block_elems + i];", 0),
    ("copy between pools skips the last pair", "for (int p = 0; p < n; p++) {\n        int32_t src = pairs[2 * p], dst",
     "for (int p = 0; p + 1 < n; p++) {\n        int32_t src = pairs[2 * p], dst", 0),
    ("max not tracked", "if (x[t - t0] > m)\n            m = x[t - t0];", "if (x[t - t0] > m)\n            m = 0.0;", 0),
]


def _replace_nth(text, old, new, n):
    idx = -1
    for _ in range(n + 1):
        idx = text.index(old, idx + 1)
    return text[:idx] + new + text[idx + len(old):]


@pytest.mark.parametrize("name,old,new,nth", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, nth):
    src = open(SRC).read()
    mutated = _replace_nth(src, old, new, nth)
    assert mutated != src
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(so), str(c), "-lm"], check=True)
    # each mutant runs in a process of its own: a planted mistake may write
    # out of bounds or crash, and must not corrupt this process
    r = subprocess.run([sys.executable, PINS, str(so)], capture_output=True, text=True, timeout=300,
                       cwd=ROOT, env={**os.environ, "PYTHONPATH": os.pathsep.join([ROOT, os.path.dirname(PINS)])})
    caught = r.returncode != 0 or bool(json.loads(r.stdout.strip().splitlines()[-1]))
    assert caught, f"no pin caught the planted mistake: {name}"


def test_unmutated_oracle_passes_in_a_subprocess():
    r = subprocess.run([sys.executable, PINS, str(oracle.build())], capture_output=True, text=True,
                       timeout=300, cwd=ROOT,
                       env={**os.environ, "PYTHONPATH": os.pathsep.join([ROOT, os.path.dirname(PINS)])})
    assert r.returncode == 0, r.stderr
    assert json.loads(r.stdout.strip().splitlines()[-1]) == []
