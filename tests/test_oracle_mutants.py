"""The oracle's pins catch planted mistakes (CPU only).

Each mutant below is a copy of oracle/spl_oracle.c with one plausible mistake: a wrong tie
rule, a wrong divisor, a swapped sub-field, a double rounding, a missing check, and so on.
Each is compiled with the oracle's own flags and the two pin suites (test_oracle_pins.py and
test_oracle_codec_pins.py) are run against it in a child process (the oracle package loads the
library named by SPL_ORACLE_LIB).  Every mutant must fail at least one pin, and the unmutated
source, built the same way, must pass them all.  Only the C file is mutated, on the CPU.
(Mutants that cannot change any output are left out: reversing the order of a pairwise sum
over a power-of-two count adds the same pairs, and the decoder's guard on pads past n only
skips accumulator slots that are never written out.)
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "spl_oracle.c")
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py"),
        os.path.join(ROOT, "tests", "test_oracle_codec_pins.py")]

# (name, text in spl_oracle.c, replacement); each text occurs exactly once
MUTANTS = [
    ("tie to the higher index",
     "return (a->idx > b->idx) - (a->idx < b->idx);",
     "return (a->idx < b->idx) - (a->idx > b->idx);"),
    ("NaN ranked last",
     "if (a->is_nan != b->is_nan) return a->is_nan ? -1 : 1;",
     "if (a->is_nan != b->is_nan) return a->is_nan ? 1 : -1;"),
    ("smallest magnitudes kept",
     "return a->mag > b->mag ? -1 : 1;",
     "return a->mag < b->mag ? -1 : 1;"),
    ("indices left in rank order",
     "qsort(out_idx, (size_t)k, sizeof(int), orc_cmp_int);",
     ";"),
    ("scale divisor 2",
     "float orc_scale(float m) { return m / 1.5f; }",
     "float orc_scale(float m) { return m / 2.0f; }"),
    ("midpoint to the larger level",
     "int mag = fabsf(v) > s;",
     "int mag = fabsf(v) >= s;"),
    ("-0.0 coded negative",
     "int sign = v < 0.0f;",
     "int sign = signbit(v) ? 1 : 0;"),
    ("upper level 2s",
     "float q = (code & 1) ? 1.5f * s : 0.5f * s;",
     "float q = (code & 1) ? 2.0f * s : 0.5f * s;"),
    ("code bits swapped in the field",
     "uint32_t field = (uint32_t)(code[r] & 3u) | (((uint32_t)idx[r] & idx_mask) << ORC_VALUE_BITS);",
     "uint32_t field = (uint32_t)(((code[r] & 1u) << 1) | ((code[r] >> 1) & 1u)) | (((uint32_t)idx[r] & idx_mask) << ORC_VALUE_BITS);"),
    ("bits written most significant first",
     "if ((field >> b) & 1u) out[bit >> 3] |= (uint8_t)(1u << (bit & 7));",
     "if ((field >> b) & 1u) out[bit >> 3] |= (uint8_t)(0x80u >> (bit & 7));"),
    ("index mask one bit short",
     "const uint32_t idx_mask = (1u << cd->idx_bits) - 1u;",
     "const uint32_t idx_mask = (1u << (cd->idx_bits - 1)) - 1u;"),
    ("index width one bit wide",
     "while ((1 << b) < L) ++b;",
     "while ((1 << b) <= L) ++b;"),
    ("record four bytes long",
     "cd->record_bytes = (k * cd->field_bits + 7) / 8;",
     "cd->record_bytes = (k * cd->field_bits + 7) / 8 + 4;"),
    ("accumulate with two roundings",
     "a[j] = fmaf(beta, ef[i], d);",
     "a[j] = beta * ef[i] + d;"),
    ("beta ignored",
     "a[j] = fmaf(beta, ef[i], d);",
     "a[j] = ef[i] + d;"),
    ("non-finite values not flagged",
     "if (!isfinite(a[j])) flags |= ORC_FLAG_NONFINITE;",
     ";"),
    ("scale from the lowest chosen index",
     "s = orc_scale(fabsf(a[top]));",
     "s = orc_scale(fabsf(a[sel[0]]));"),
    ("residual with the wrong sign",
     "a[sel[r]] = v - orc_level(code[r], s); /* residual at a transmitted position */",
     "a[sel[r]] = v + orc_level(code[r], s);"),
    ("no residual (error buffer keeps the sent value)",
     "a[sel[r]] = v - orc_level(code[r], s); /* residual at a transmitted position */",
     "a[sel[r]] = v;"),
    ("pairwise split after the middle",
     "h = n / 2;",
     "h = (n + 1) / 2;"),
    ("mean-abs summed left to right",
     "s = orc_pairwise_sum(mags, k) / (float)k;",
     "{ float t = 0.0f; for (r = 0; r < k; ++r) t += mags[r]; s = t / (float)k; }"),
    ("mean-abs divided by k - 1",
     "s = orc_pairwise_sum(mags, k) / (float)k;",
     "s = orc_pairwise_sum(mags, k) / (float)(k - 1);"),
    ("mean-abs over a rotated index order",
     "for (r = 0; r < k; ++r) mags[r] = fabsf(a[sel[r]]);",
     "for (r = 0; r < k; ++r) mags[(r + 1) % k] = fabsf(a[sel[r]]);"),
    ("negative scales accepted",
     "if (isnan(s) || isinf(s) || s < 0.0f) return 0;",
     "if (isnan(s) || isinf(s)) return 0;"),
    ("duplicate indices accepted",
     "if (!(idx[r - 1] < idx[r])) return 0;",
     "if (!(idx[r - 1] <= idx[r])) return 0;"),
    ("validity checked over the first 64 entries only",
     "for (r = 1; r < k; ++r)\n        if (!(idx[r - 1] < idx[r])) return 0;",
     "for (r = 1; r < k && r < 64; ++r)\n        if (!(idx[r - 1] < idx[r])) return 0;"),
    ("mean divided by P + 1",
     "mean_out[i] = acc[j] / (float)P;",
     "mean_out[i] = acc[j] / (float)(P + 1);"),
    ("outer step with the wrong sign",
     "if (theta) theta[i] = fmaf(-lr, mean_out[i], theta[i]);",
     "if (theta) theta[i] = fmaf(lr, mean_out[i], theta[i]);"),
    ("tail pads not zero",
     "                a[j] = 0.0f;",
     "                a[j] = 1.0e-30f;"),
    ("statistics count sign bits as big",
     "big[p] += code[r] & 1u;",
     "big[p] += (code[r] >> 1) & 1u;"),
    ("statistics keep the smallest scale",
     "if (s > max_scale[p]) max_scale[p] = s;",
     "if (s < max_scale[p] || max_scale[p] == 0.0f) max_scale[p] = s;"),
]


def _compile(src_text: str, out: str):
    c = out[:-3] + ".c"
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *oracle._CFLAGS, "-o", out, c, "-lm"], check=True)


def _run_pins(lib: str) -> subprocess.CompletedProcess:
    env = dict(os.environ, SPL_ORACLE_LIB=lib)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           "-m", "not gpu", *PINS], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=300)


def test_every_mutant_fails_a_pin(tmp_path):
    text = open(SRC).read()
    jobs = [("unmutated", text)]
    for name, old, new in MUTANTS:
        assert text.count(old) == 1, f"mutant '{name}': its text no longer occurs once"
        jobs.append((name, text.replace(old, new)))
    libs = []
    for i, (name, src) in enumerate(jobs):
        libs.append((name, str(tmp_path / f"mutant{i}.so")))
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(lambda j: _compile(j[0][1], j[1][1]), zip(jobs, libs)))
        results = list(ex.map(lambda l: (l[0], _run_pins(l[1])), libs))
    base = results[0][1]
    assert base.returncode == 0, "the unmutated oracle fails its pins:\n" + base.stdout[-2000:]
    survivors = [name for name, r in results[1:] if r.returncode == 0]
    assert not survivors, f"mutants no pin catches: {survivors}"
    for name, r in results[1:]:
        assert r.returncode == 1, f"mutant '{name}': pins did not run cleanly:\n{r.stdout[-1500:]}"
