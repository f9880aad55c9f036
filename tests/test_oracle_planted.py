"""Planted mistakes: the oracle's pins must catch each of them.

Each case copies ``oracle/tq_oracle.c``, plants one plausible mistake by an
exact text substitution (the kind a restatement of the method could make: a
transposed operand, a wrong constant, a dropped term, an off-by-one), compiles
the copy under ``oracle/_build/planted/`` and runs the oracle's pin tests
against it in a child process (``TQO_LIBRARY`` points the binding at the
copy). The pins pass on the unmodified source (the control case) and must fail
on every mutant: a mutant that survives means the oracle has a step that no
pin ties to the method.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "tq_oracle.c")
OUT = os.path.join(ROOT, "oracle", "_build", "planted")
PINS = ["tests/test_oracle_codec.py", "tests/test_oracle_encode.py", "tests/test_oracle_decode.py"]

# name, original text, planted text, occurrences replaced (all of them, so
# the mistake is made consistently wherever the formula appears)
MUTANTS = [
    # SplitMix64: a wrong increment (the published outputs)
    ("splitmix_increment", "(i + 1) * 0x9E3779B97F4A7C15ULL", "(i + 1) * 0x9E3779B97F4A7C13ULL", 1),
    # rotation: R = Q without the sign fix of the QR factorisation
    ("qr_sign_fix_dropped", "Rout[i * D + j] = Q[i * D + j] * d[j];", "Rout[i * D + j] = Q[i * D + j];", 1),
    # Lloyd-Max: density exponent (D - 1)/2 instead of (D - 3)/2
    ("density_exponent", "0.5 * (double)(D - 3)", "0.5 * (double)(D - 1)", 2),
    # Lloyd-Max: centroid = minus the cell's mean
    ("centroid_moment_sign", "double mom = Ge[j + 1] - Ge[j];", "double mom = Ge[j] - Ge[j + 1];", 1),
    # Lloyd-Max: thresholds at the left centroid instead of the midpoint
    ("threshold_not_midpoint", "m[j] = 0.5 * (c[j] + c[j + 1]);", "m[j] = c[j];", 1),
    # Lloyd-Max: iterations stopped at a step of 1e-3
    ("lloyd_stops_early", "if (delta <= 1e-17) break;", "if (delta <= 1e-3) break;", 1),
    # Lloyd-Max: the cell-mass recurrence loses its factor 2
    ("mass_recurrence", "I = (t * p + 2.0 * a * I) / (2.0 * a + 1.0);", "I = (t * p + a * I) / (2.0 * a + 1.0);", 1),
    # packing: codes that straddle two words lose their high bits
    ("pack_straddle_dropped", "if ((p & 31) + b > 32) words[(p >> 5) + 1] |= (uint32_t)(v >> 32);", "", 1),
    # binary16: truncation instead of round to nearest even
    ("fp16_truncates", "if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;", "", 1),
    # encode: the norm misses the last coordinate
    ("norm_drops_last_coordinate", "for (int k = 0; k < D; ++k) n2 = fmaf(x[k], x[k], n2);",
     "for (int k = 0; k < D - 1; ++k) n2 = fmaf(x[k], x[k], n2);", 1),
    # encode: y = R^T x instead of R x
    ("rotation_transposed_in_encode", "t = fmaf(R[(size_t)i * D + k], x[k], t);",
     "t = fmaf(R[(size_t)k * D + i], x[k], t);", 1),
    # prod: residual y + c instead of y - c
    ("residual_sign", "r[i] = y[i] - c[codes[i]];", "r[i] = y[i] + c[codes[i]];", 1),
    # prod: sign bit set for negative projections
    ("qjl_sign_flipped", "if (z >= 0.0f) sw[j >> 5]", "if (z < 0.0f) sw[j >> 5]", 1),
    # prod: QJL constant sqrt(2/pi)/D instead of sqrt(pi/2)/D, everywhere
    ("qjl_constant", "sqrt(M_PI / 2.0) / (double)D", "sqrt(2.0 / M_PI) / (double)D", 3),
    # group: the fp16 minimum taken from the group maximum
    ("group_min_from_max", "mh = tqo_f32_to_f16(lo);", "mh = tqo_f32_to_f16(hi);", 1),
    # dequantisers: the vector norm dropped
    ("dequant_norm_dropped", "out[v * D + d] = (double)norm[v] * s;", "out[v * D + d] = s;", 2),
    # attention: the score scale applied twice
    ("score_scale_squared", "s[t] = a * scale;", "s[t] = a * scale * scale;", 1),
    # rotated decode: the key norm dropped from the score
    ("key_norm_dropped_in_decode", "double s = scale * (double)knorm[t] * a;", "double s = scale * a;", 2),
    # attention: the causal window one token short, everywhere
    ("causal_off_by_one", "const int64_t nv = N - Lq + l + 1;", "const int64_t nv = N - Lq + l;", 2),
    # rotated decode: q'' = S^T q' instead of S q'
    ("qjl_matrix_transposed_in_decode", "s += (double)kS[(size_t)j * D + i] * q1[i];",
     "s += (double)kS[(size_t)i * D + j] * q1[i];", 2),
    # rotated decode: the residual norm dropped from the QJL term
    ("residual_norm_dropped_in_decode", "a += kappa * (double)krn[t] * z;", "a += kappa * z;", 2),
    # rotated decode: the output rotated by R_v instead of back by R_v^T
    ("value_rotation_not_inverted", "s += acc[i] * (double)vR[(size_t)i * D + d];",
     "s += acc[i] * (double)vR[(size_t)d * D + i];", 1),
    # fractional widths: the keys take the upper width
    ("fractional_split_swapped", "fractional ? (int)floor(b)", "fractional ? (int)ceil(b)", 1),
    # group: codes rounded down instead of to nearest
    ("group_rounds_down", "float r = rintf((xv[gi * g + k] - mf) / sf);",
     "float r = floorf((xv[gi * g + k] - mf) / sf);", 1),
    # group: the minimum dropped when dequantising
    ("group_dequant_min_dropped", "out[v * D + d] = (double)codes[d] * s + m0;",
     "out[v * D + d] = (double)codes[d] * s;", 1),
    # rotated decode: the group minimum dropped from the value sum
    ("group_decode_min_dropped", "acc[d] += p * ((double)codes[d] * sc + m0);",
     "acc[d] += p * ((double)codes[d] * sc);", 2),
    # sharded decode: a shard's causal window one token short
    ("shard_causal_end_off_by_one", "int64_t nv = E - Lq + l + 1; /* visible local keys t < nv */",
     "int64_t nv = E - Lq + l; /* visible local keys t < nv */", 1),
    # shard merge: parts weighted by e^(M - m_p) instead of e^(m_p - M)
    ("merge_weight_inverted", "const double w = exp(mp - M);", "const double w = exp(M - mp);", 1),
    # shard merge: the parts' sums added without their weights
    ("merge_sum_unweighted", "L += w * l[(size_t)p * rows + r];", "L += l[(size_t)p * rows + r];", 1),
    # pool writer: the block table ignored
    ("block_table_ignored",
     "int64_t p = table ? table[(int64_t)seq * max_blocks + lb] : (int64_t)seq * max_blocks + lb;",
     "int64_t p = (int64_t)seq * max_blocks + lb;", 1),
]


_WORKERS = 4
_THREADS = max(1, (os.cpu_count() or 8) // _WORKERS)


def _build(name, old, new, count):
    with open(SRC) as f:
        text = f.read()
    if old is not None:
        assert text.count(old) == count, f"{name}: expected {count} occurrence(s) of the planted site"
        text = text.replace(old, new)
    os.makedirs(OUT, exist_ok=True)
    src = os.path.join(OUT, f"{name}.c")
    with open(src, "w") as f:
        f.write(text)
    return oracle.compile_source(src, os.path.join(OUT, f"{name}.so"))


def _run_pins(so):
    # four children at a time, two OpenMP threads each: spinning OpenMP
    # teams oversubscribing the cores slow every child down many times
    env = dict(os.environ, TQO_LIBRARY=so, OMP_NUM_THREADS=str(_THREADS),
               PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    failed = [ln for ln in r.stdout.splitlines() if ln.startswith("FAILED")]
    return r.returncode, failed, r.stdout[-2000:]


@pytest.fixture(scope="module")
def outcomes():
    oracle.build()
    cases = [("control", None, None, 0)] + MUTANTS
    libs = {c[0]: _build(*c) for c in cases}
    with ThreadPoolExecutor(max_workers=_WORKERS) as ex:
        res = dict(zip(libs, ex.map(_run_pins, libs.values())))
    return res


def test_pins_pass_on_the_unmodified_source(outcomes):
    rc, failed, tail = outcomes["control"]
    assert rc == 0, tail


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(outcomes, name):
    rc, failed, tail = outcomes[name]
    # exit status 1: the pins ran and at least one failed (not a crash or a
    # collection error)
    assert rc == 1 and failed, f"{name} survived the pins (exit {rc}):\n{tail}"
