"""Strength of the oracle pins (CPU): each case plants one plausible mistake in
a copy of oracle/oracle.c -- a dropped or inverted ReLU, a wrong weight index or
sign, a wrong scale exponent or block, misaligned operands, a wrong E2M1 value, a
reversed tie, zero-sign or NaN rule, an off-by-one short-row boundary, a page
table that is ignored, a query row that is ignored, an fp32-exactness flag that
never fires or counts 53 significant bits -- builds it, and runs
tests/test_oracle_pins.py against it.  Every mutant must fail at least one pin;
the unmodified copy must pass them all."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_C = os.path.join(ROOT, "oracle", "oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

MUTANTS = [
    ("relu dropped", "double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    ("relu keeps the negative part", "double relu = dot > 0.0 ? dot : 0.0;",
     "double relu = dot < 0.0 ? dot : 0.0;"),
    ("weight of the next head", "acc += w[h] * relu;", "acc += w[(h + 1) % NH] * relu;"),
    ("weight sign", "acc += w[h] * relu;", "acc -= w[h] * relu;"),
    ("scale exponent off by one", "ex[k] = (a->e[k] - 127) + (b->e[k] - 127) - 2;",
     "ex[k] = (a->e[k] - 127) + (b->e[k] - 127) - 1;"),
    ("scale blocks reversed", "out->e[b] = (int)scales[b];", "out->e[b] = (int)scales[NSF - 1 - b];"),
    # swapping the nibble order of both operands alike leaves every dot product
    # unchanged (a common permutation of both vectors), so the method cannot show
    # it; pairing misaligned elements of the two operands is the visible form
    ("operands misaligned within a byte",
     "acc += (int)a->v[32 * k + i] * (int)b->v[32 * k + i];",
     "acc += (int)a->v[32 * k + i] * (int)b->v[32 * k + (i ^ 1)];"),
    ("E2M1 code 5 read as 2.5", "{0, 1, 2, 3, 4, 6, 8, 12,", "{0, 1, 2, 3, 4, 5, 8, 12,"),
    ("ties to the higher index", "return a->idx < b->idx;", "return a->idx > b->idx;"),
    ("-0 above +0", "if (sa != sb) return sb;", "if (sa != sb) return sa;"),
    ("NaN above numbers", "if (na != nb) return nb;", "if (na != nb) return na;"),
    ("short rows only below topk", "if (len <= topk) {", "if (len < topk) {"),
    ("page table ignored", "*phys_row = (int64_t)page * NPAGE + (s % NPAGE);",
     "*phys_row = (int64_t)p * NPAGE + (s % NPAGE);"),
    ("fp32 exactness flag never set",
     "if (bits > 24 || m < -149 || m + bits > 128) *f32_exact = 0;",
     "if (0) *f32_exact = 0;"),
    ("fp32 significand taken as 53 bits",
     "if (bits > 24 || m < -149 || m + bits > 128) *f32_exact = 0;",
     "if (bits > 53 || m < -149 || m + bits > 128) *f32_exact = 0;"),
    ("query row ignored",
     "decode_row(q_fp4 + ((int64_t)row * NH + h) * NDB, q_scale + ((int64_t)row * NH + h) * NSF, &qr[h]);\n"
     "    w[h]",
     "decode_row(q_fp4 + ((int64_t)0 * NH + h) * NDB, q_scale + ((int64_t)0 * NH + h) * NSF, &qr[h]);\n"
     "    w[h]"),
]


def _build(tmp, text, name):
    src = tmp / f"{name}.c"
    src.write_text(text)
    lib = tmp / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=gnu11", str(src), "-o",
                    str(lib), "-lm"], check=True, capture_output=True)
    return str(lib)


def _pins_pass(lib):
    env = dict(os.environ, IDXTOPK_ORACLE_LIB=lib, OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        PINS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode == 0, r.stdout[-2000:]


@pytest.fixture(scope="module")
def tmp(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    return tmp_path_factory.mktemp("mutants")


def test_unmodified_copy_passes(tmp):
    ok, out = _pins_pass(_build(tmp, open(ORACLE_C).read(), "unmodified"))
    assert ok, out


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_the_mutant(tmp, name, old, new):
    text = open(ORACLE_C).read()
    assert text.count(old) == 1, name
    ok, out = _pins_pass(_build(tmp, text.replace(old, new), "m" + str(abs(hash(name)))))
    assert not ok, f"no pin fails with the planted mistake: {name}\n{out}"
