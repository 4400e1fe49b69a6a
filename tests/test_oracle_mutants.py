"""Plants plausible mistakes in private copies of the oracle source and checks
that the pin suite catches every one of them (CPU only, the oracle is never
modified in place)."""
import pytest

import oracle
import oracle_pins

MUTANTS = [
    ("phase sign", "const double ph = ORACLE_TWO_PI * f_demod * tau;",
     "const double ph = -ORACLE_TWO_PI * f_demod * tau;"),
    ("phase drops t0 the wrong way", "const double ph = ORACLE_TWO_PI * f_demod * tau;",
     "const double ph = ORACLE_TWO_PI * f_demod * (tau - t0);"),
    ("interp weights swapped", "const double vr = (1.0 - a) * s0r + a * s1r;",
     "const double vr = a * s0r + (1.0 - a) * s1r;"),
    ("fraction from the wrong side", "const double a = f - k0f;",
     "const double a = k0f + 1.0 - f;"),
    ("wrong neighbour sample", "k0 + 1, &s1r, &s1i", "k0 - 1, &s1r, &s1i"),
    ("transmit weight dropped", "const double cr = wt * (vr * pr - vi * pim);",
     "const double cr = (vr * pr - vi * pim);"),
    ("imaginary part sign", "out[ncomp * o + 1] += ci;", "out[ncomp * o + 1] -= ci;"),
    ("aperture boundary exclusive", "(lhs <= rhs)", "(lhs < rhs)"),
    ("aperture uses F# not 2F#", "(2.0 * fnum) * (2.0 * fnum)", "fnum * fnum"),
    ("aperture ignores depth sign", "inside = (ez > 0.0) && (lhs <= rhs);",
     "inside = (lhs <= rhs);"),
    ("receive delay units", "tau_t + dist / c", "tau_t + dist * c"),
    ("t0 sign", "(tau - t0) * fs", "(tau + t0) * fs"),
    ("record axes q, m swapped", "const int64_t i = (((int64_t)b * Q + q) * M + m) * K + k;\n    if (rf_type & 1)",
     "const int64_t i = (((int64_t)b * M + m) * Q + q) * K + k;\n    if (rf_type & 1)"),
    ("permute reads q, m swapped", "const int64_t i = (((int64_t)b * Q + q) * M + m) * K + k;\n                    const int64_t o",
     "const int64_t i = (((int64_t)b * M + m) * Q + q) * K + k;\n                    const int64_t o"),
    ("last sample dropped", "if (k < 0 || k > (int64_t)K - 1) {",
     "if (k < 0 || k > (int64_t)K - 2) {"),
    ("pair dropped below the record", "if (k0f < -1.0 || k0f > (double)K - 1.0) continue;",
     "if (k0f < 0.0 || k0f > (double)K - 1.0) continue;"),
    ("tau_tx transposed", "tau_tx[(int64_t)q * N + n]", "tau_tx[(int64_t)n * Q + q]"),
    ("w_tx transposed", "w_tx[(int64_t)q * N + n]", "w_tx[(int64_t)n * Q + q]"),
    ("receiver x/y swapped", "px - rx_xyz[3 * m + 0]", "px - rx_xyz[3 * m + 1]"),
    ("slack signed", "slack[o] += sqrt(cr * cr + ci * ci);", "slack[o] += cr;"),
    ("permute q/m order", "(((int64_t)k * Q + q) * M + m) * B + b",
     "(((int64_t)k * M + m) * Q + q) * B + b"),
    ("double records read as float", "const int is_double = rf_type >> 1;", "const int is_double = 0;"),
    ("grid y index", "const int64_t iy = (n / nx) % ny;", "const int64_t iy = (n / ny) % nx;"),
]


def _run_pins(orc):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError) as exc:   # a caught mistake
            failed.append((pin.__name__, type(exc).__name__))
    return failed


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = oracle.SOURCE.read_text()
    assert src.count(old) == 1, f"mutation target not unique: {old!r}"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.compile_source(mutant, tmp_path / "libmutant.so")
    failed = _run_pins(oracle.Oracle(lib))
    assert failed, f"no pin catches the planted mistake: {name}"
