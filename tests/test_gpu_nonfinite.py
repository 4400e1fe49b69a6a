"""Non-finite samples in the record, every kernel against the oracle.

The sum multiplies the two samples of a pair by their weights, so a NaN sample
makes every output whose pair holds it NaN, and a +inf sample makes it +inf
(weights here are positive), element by element as in the oracle.  A sample
outside the record counts as zero and is never read, so a NaN next to the
record's edge stays out of a pair that hangs over that edge.

The window kernel departs by design: its coefficient rows hold zeros for
voxels of a quad that do not use a row, so a non-finite sample reaches every
voxel of the quad whose window holds it.  Its test checks that departure as
documented: no finite oracle value is lost, and every finite window value
matches the oracle."""
import numpy as np
import pytest

from parity import TOL, gpu_beamform, kernel_serves, oracle_beamform
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

EXACT = ["bl", "bi", "brick", "pair"]


def _index(prob, n, q, m):
    """float64 fractional sample index of (voxel n, transmit q, receiver m)."""
    p = synth.grid_points(prob.grid, [n])[0]
    d = np.linalg.norm(p - prob.rx[m].astype(np.float64))
    return (float(prob.tau_tx[q, n]) + d / prob.c - prob.t0) * prob.fs


def _inside(prob, n, m):
    p = synth.grid_points(prob.grid, [n])[0]
    e = p - prob.rx[m].astype(np.float64)
    return e[2] > 0 and (2 * prob.fnum) ** 2 * (e[0] ** 2 + e[1] ** 2) <= e[2] ** 2


def _plant(prob, picks, value):
    """Puts `value` at the sample k0 (or k0 + 1) a chosen (b, n, q, m) reads."""
    for b, n, q, m, second in picks:
        assert _inside(prob, n, m)
        k = int(np.floor(_index(prob, n, q, m))) + (1 if second else 0)
        assert 2 <= k <= prob.K - 3
        prob.rf[b, q, m, k] = value


def _compare(y, ref, slack):
    """Same NaN / +inf / -inf pattern, finite values within the parity bar."""
    y = np.asarray(y, dtype=np.complex128)
    for part in (np.real, np.imag):
        yp, rp = part(y), part(ref)
        assert np.array_equal(np.isnan(yp), np.isnan(rp))
        assert np.array_equal(np.isposinf(yp), np.isposinf(rp))
        assert np.array_equal(np.isneginf(yp), np.isneginf(rp))
    fin = np.isfinite(ref)
    peak = float(np.abs(ref[fin]).max())
    err = np.maximum(np.abs(y[fin] - ref[fin]) - slack[fin], 0.0)
    assert float(err.max()) <= TOL * peak


def _problem(kind):
    if kind == "real":
        prob = synth.make_problem("full", n_el=8, nx=19, ny=13, nz=5)
        n0 = 19 * 13 * 3 + 19 * 6 + 9
        _plant(prob, [(3, n0, 2, 27, False), (3, n0 + 40, 5, 36, True)], np.float32(np.nan))
        _plant(prob, [(11, n0 - 30, 7, 18, False)], np.float32(np.inf))
    else:
        prob = synth.make_problem("iq", n_el=8, nx=11, ny=9, nz=4)
        n0 = 11 * 9 * 2 + 11 * 4 + 5
        _plant(prob, [(5, n0, 1, 27, False)], np.complex64(complex(np.nan, 0.0)))
        _plant(prob, [(40, n0 + 12, 6, 36, True)], np.complex64(complex(0.0, np.nan)))
    return prob


@pytest.fixture(scope="module", params=["real", "iq"])
def planted(request, oracle):
    prob = _problem(request.param)
    ref, slack = oracle_beamform(oracle, prob)
    assert (~np.isfinite(ref)).sum() >= 2        # the planted samples reach some outputs
    assert np.isfinite(ref).mean() > 0.99
    return prob, ref, slack


@pytest.mark.parametrize("kernel", EXACT)
def test_nonfinite_samples_match_oracle(planted, kernel):
    prob, ref, slack = planted
    if not kernel_serves(kernel, prob):
        pytest.skip(f"the {kernel} kernel does not serve this record")
    y, used = gpu_beamform(prob, kernel)
    assert used == kernel
    _compare(y, ref, slack)


def test_window_kernel_nonfinite_departure(oracle):
    prob = _problem("real")
    ref, slack = oracle_beamform(oracle, prob)
    y, used = gpu_beamform(prob, "window")
    assert used == "window"
    y = np.asarray(y, dtype=np.float64)
    bad_ref, bad_y = ~np.isfinite(ref), ~np.isfinite(y)
    assert np.all(bad_y[bad_ref])                # every oracle non-finite output stays so
    planted_frames = {3, 11}
    extra = np.argwhere(bad_y & ~bad_ref)
    assert all(int(b) in planted_frames for b, _ in extra)   # spread only within those frames
    fin = ~bad_y
    peak = float(np.abs(ref[np.isfinite(ref)]).max())
    err = np.maximum(np.abs(y[fin] - ref[fin]) - slack[fin], 0.0)
    assert float(err.max()) <= TOL * peak


@pytest.mark.parametrize("edge", ["start", "end"])
@pytest.mark.parametrize("kernel", EXACT)
def test_nan_beside_record_edge_stays_out(oracle, kernel, edge):
    """A pair straddling an end of the record keeps only its in-record sample:
    a NaN at the sample beyond that one (k = 1 at the start, k = K - 2 at the
    end) must not reach the output through a zero weight."""
    base = synth.make_problem("tiny", B=16)
    n, q, m = 16 * 16 * 8 + 16 * 8 + 8, 1, 27
    f = _index(base, n, q, m)
    # t0 shifted so that this term's index lands at -0.5 (pair k0 = -1) or K - 0.5
    target = -0.5 if edge == "start" else base.K - 0.5
    t0 = float(np.float32(base.t0 + (f - target) / base.fs))
    prob = synth.make_problem("tiny", B=16, t0=t0)
    f = _index(prob, n, q, m)
    assert (-1 < f < 0) if edge == "start" else (prob.K - 1 < f < prob.K)
    k_nan = 1 if edge == "start" else prob.K - 2
    prob.rf[:, q, m, k_nan] = np.nan
    ref, slack = oracle_beamform(oracle, prob)
    y, used = gpu_beamform(prob, kernel)
    assert used == kernel
    assert np.all(np.isfinite(ref[:, n]))        # the oracle skips the out-of-record sample
    _compare(y, ref, slack)
