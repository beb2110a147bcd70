"""The oracle's pins catch plausible mistakes.

Each case copies oracle/tdp_oracle.c to a temporary directory, plants one
mistake in the copy (a dropped term, an off-by-one, a swapped index or operand,
a wrong divisor), compiles it, and runs the fast subset of the pin suite
(tests/test_oracle_pins.py) against that build in a separate process.  At least
one pin must fail (or the broken build must crash) for every mistake.  The real
oracle source is never modified.
"""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "tdp_oracle.c")
FAST_PINS = "not temporal and not medium and not large"

# (name, text in tdp_oracle.c, replacement)
MUTANTS = [
    ("ramp_rise_off_by_one", "return (x - lo[i]) + 1;", "return (x - lo[i]);"),
    ("ramp_fall_off_by_one", "return o - (x - lo[i + 1]);", "return o - (x - lo[i + 1]) + 1;"),
    ("ramp_denominator", "*den = o + 1;", "*den = o + 2;"),
    ("box_halves_swapped", "lo[i] = (i > 0) ? c0 - a : c0;", "lo[i] = (i > 0) ? c0 - b : c0;"),
    ("box_right_edge", "hi[i] = (i < n - 1) ? c1 + b : c1;", "hi[i] = (i < n - 1) ? c1 + a : c1;"),
    ("cores_rounding", "int32_t c1 = (int32_t)(((int64_t)(i + 1) * L) / n);",
     "int32_t c1 = (int32_t)(((int64_t)(i + 1) * L + n - 1) / n);"),
    ("offsets_exclusive", "off[t] = acc;\n        acc += tt;", "acc += tt;\n        off[t] = acc;"),
    ("mask_uses_h_for_w", "* ramp(p, 2, iW, w);", "* ramp(p, 2, iW, h);"),
    ("split_h_w_swapped", "int64_t g = ((int64_t)f * p->H + h) * p->W + w;\n                        const char *src",
     "int64_t g = ((int64_t)f * p->W + h) * p->H + w;\n                        const char *src"),
    ("split_batch_stride", "+ (int64_t)b * Tt + j) * (int64_t)row;", "+ (int64_t)j * p->B + b) * (int64_t)row;"),
    ("bounds_min_of_end", "if (q[2 * j] < lo) lo = q[2 * j];", "if (q[2 * j + 1] < lo) lo = q[2 * j + 1];"),
    ("normalise_start_only", "for (int64_t j = 0; j < 2 * Tt; ++j) q[j] = wrap_sub(q[j], m);",
     "for (int64_t j = 0; j < 2 * Tt; j += 2) q[j] = wrap_sub(q[j], m);"),
    ("filter_no_negative_time", "int kept = inside || negative_time;", "int kept = inside;"),
    ("filter_closed_intervals", "if (!(a < z)) inside = 0;", "if (!(a <= z)) inside = 0;"),
    ("filter_negative_end", "int negative_time = K[(((int64_t)b * 3 + 0) * N + k) * 2 + 0] < 0;",
     "int negative_time = K[(((int64_t)b * 3 + 0) * N + k) * 2 + 1] < 0;"),
    ("filter_shift_by_max", "normalize ? wrap_sub(v, mn[tb * 3 + d]) : v;", "normalize ? wrap_sub(v, mx[tb * 3 + d]) : v;"),
    ("filter_pad_zero", "for (int32_t k = cnt; k < N; ++k) idx[tb * N + k] = -1;",
     "for (int32_t k = cnt; k < N; ++k) idx[tb * N + k] = 0;"),
    ("blend_overwrites", "Z[((int64_t)b * T + g) * p->C + c] += m * load_elem(Yout, p->esize, src + c);",
     "Z[((int64_t)b * T + g) * p->C + c] = m * load_elem(Yout, p->esize, src + c);"),
    ("blend_mask_dropped_f", "return (ramp(p, 0, iF, f) * ramp(p, 1, iH, h)) * ramp(p, 2, iW, w);",
     "return ramp(p, 1, iH, h) * ramp(p, 2, iW, w);"),
    ("bf16_decode_shift", "uint32_t bits = (uint32_t)((const uint16_t *)Y)[i] << 16;",
     "uint32_t bits = (uint32_t)((const uint16_t *)Y)[i] << 15;"),
    ("cond_divides_by_tiles", "for (int32_t c = 0; c < p->C; ++c) o[c] /= (double)n_keep;",
     "for (int32_t c = 0; c < p->C; ++c) o[c] /= (double)nt;"),
    ("cond_skips_first_tile", "for (int t = 0; t < nt; ++t) {\n                int64_t tb = (int64_t)t * p->B + b;\n                if (!keep",
     "for (int t = 1; t < nt; ++t) {\n                int64_t tb = (int64_t)t * p->B + b;\n                if (!keep"),
    ("cond_divides_by_stored_rows", "if (pos < 0 || pos >= ncap) continue;",
     "if (pos < 0 || pos >= ncap) { n_keep -= 1; continue; }"),
    ("mean_off_by_one", "out[i] = acc / (double)nt;", "out[i] = acc / (double)(nt + 1);"),
    ("slot_off_by_one", "slot[tb * N + k] = kept ? cnt : -1;", "slot[tb * N + k] = kept ? cnt + 1 : -1;"),
]


def _run_pins(lib_path):
    env = dict(os.environ, TDP_ORACLE_LIB=lib_path, PYTHONDONTWRITEBYTECODE="1")
    return subprocess.Popen(
        [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
         "-p", "no:cacheprovider", "-k", FAST_PINS],
        cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)


@pytest.fixture(scope="module")
def mutant_results():
    """Build every mutant and run the pins against all of them in parallel."""
    src = open(SRC).read()
    results = {}
    with tempfile.TemporaryDirectory() as tmp:
        procs = {}
        for name, old, new in MUTANTS:
            assert src.count(old) == 1, f"mutant {name}: text to replace not found exactly once"
            path = os.path.join(tmp, f"{name}.c")
            with open(path, "w") as fh:
                fh.write(src.replace(old, new))
            lib = oracle.compile_source(path, os.path.join(tmp, f"lib{name}.so"))
            procs[name] = _run_pins(lib)
        for name, p in procs.items():
            out, _ = p.communicate(timeout=600)
            results[name] = (p.returncode, out)
    return results


def test_pins_pass_on_the_real_oracle():
    lib = oracle.build()
    p = _run_pins(lib)
    out, _ = p.communicate(timeout=600)
    assert p.returncode == 0, out[-2000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_mutant(mutant_results, name):
    rc, out = mutant_results[name]
    assert rc != 0, f"no pin failed for the planted mistake {name}:\n{out[-1500:]}"
