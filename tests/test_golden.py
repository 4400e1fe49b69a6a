"""The oracle against the hand-worked examples of tests/golden/ (closed forms
of the delay-and-sum definition: record edges, the F-number aperture, the IQ
demodulation phase and its sign)."""
import numpy as np
import pytest

import golden_cases
import oracle as oracle_mod


@pytest.mark.parametrize("ex", golden_cases.examples(), ids=lambda e: e["name"])
def test_oracle_matches_worked_example(oracle, ex):
    rf, tau, w, rx = golden_cases.inputs(ex)
    y = oracle.beamform(rf, tau, w, rx.astype(np.float64), oracle_mod.Grid(*ex["grid"]),
                        c=ex["c"], fs=ex["fs"], t0=ex["t0"], fnum=ex["fnum"], f_demod=ex["f_demod"])
    ref = golden_cases.expected(ex)
    assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max()


def test_records_follow_their_formulas():
    real, iq = golden_cases.examples()
    rf, _, _, _ = golden_cases.inputs(real)
    assert rf.dtype == np.float32 and rf.shape == (8, 2, 3, 8)
    assert rf[0, 0, 0, 0] == 1 and rf[1, 1, 2, 7] == 2 * (1 + 7 + 20 + 100)
    rf, _, _, _ = golden_cases.inputs(iq)
    assert rf.dtype == np.complex64 and rf[2, 0, 1, 3] == 3 * (14 + 6j)
