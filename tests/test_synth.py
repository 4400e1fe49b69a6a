"""The seeded workload generator: sizes, determinism and its stated conventions."""
import math

import numpy as np
import pytest

from volumetric_ultrasound_delay_gb300 import synth


@pytest.mark.parametrize("name,acc", [
    ("tiny", 6_291_456), ("mid", 2_264_924_160), ("full", 77_309_411_328),
    ("iq", 154_618_822_656), ("large", 858_993_459_200)])
def test_workload_sizes(name, acc):
    assert synth.WORKLOADS[name].accumulations == acc


def test_tiny_problem_shapes_and_determinism():
    p1 = synth.make_problem("tiny")
    p2 = synth.make_problem("tiny")
    assert p1.rf.shape == (8, 3, 64, 512) and p1.rf.dtype == np.float32
    assert p1.tau_tx.shape == (3, 4096) and p1.w_tx.shape == (3, 4096)
    assert np.array_equal(p1.rf, p2.rf) and np.array_equal(p1.tau_tx, p2.tau_tx)
    nx, ny, nz, x0, y0, z0, dx, dy, dz = p1.grid
    assert (nx, ny, nz) == (16, 16, 16)
    assert math.isclose(x0, -2.4e-3, rel_tol=1e-6) and math.isclose(x0 + 15 * dx, 2.4e-3, rel_tol=1e-6)
    assert math.isclose(z0, 5e-3, rel_tol=1e-6) and math.isclose(z0 + 15 * dz, 20e-3, rel_tol=1e-6)
    # noise is unit variance; three unit echoes barely move it
    assert 0.9 < float(p1.rf.std()) < 1.1


def test_iq_problem_is_circular():
    p = synth.make_problem("iq", nx=4, ny=4, nz=4, B=2, K=256, n_el=4, n_scat=0)
    assert p.rf.dtype == np.complex64 and p.rf.shape == (2, 9, 16, 256)
    assert abs(float(p.rf.real.var()) - 0.5) < 0.05 and abs(float(p.rf.imag.var()) - 0.5) < 0.05


def test_plane_wave_and_diverging_wave_delays():
    wl = synth.workload("tiny")
    pts = np.array([[0.0, 0.0, 10e-3], [1e-3, 0.0, 10e-3]])
    tau = synth.transmit_delays(wl, pts)
    # broadside plane wave: tau = z / c; steered +10 deg: (x sin + z cos) / c
    assert math.isclose(tau[1, 0], 10e-3 / 1540.0)
    th = math.radians(10.0)
    assert math.isclose(tau[2, 1], (1e-3 * math.sin(th) + 10e-3 * math.cos(th)) / 1540.0)
    dw = synth.workload("full")
    # diverging wave: zero at the array centre, |x - v| - |v| elsewhere
    t = synth.transmit_delays(dw, np.array([[0.0, 0.0, 0.0], [0.0, 0.0, 5e-3]]))
    assert np.allclose(t[:, 0], 0.0, atol=1e-15)
    assert math.isclose(t[4, 1], 5e-3 / 1540.0)          # source straight behind: (15 - 10) mm


def test_array_layout():
    rx = synth.array_positions(4)
    assert rx.shape == (16, 3)
    assert np.allclose(rx[0], [-0.45e-3, -0.45e-3, 0.0])
    assert np.allclose(rx[1], [-0.15e-3, -0.45e-3, 0.0])     # x varies fastest
    assert np.allclose(rx[4], [-0.45e-3, -0.15e-3, 0.0])


def test_echo_lands_at_its_delay():
    wl = synth.workload("tiny", n_scat=0)
    rx = synth.array_positions(wl.n_el)
    p = np.array([[0.0, 0.0, 10e-3]])
    rec = synth.echo_record(wl, rx, p)
    tau = synth.transmit_delays(wl, p)[1, 0] + np.linalg.norm(p[0] - rx[0]) / wl.c
    k = int(np.argmax(np.abs(rec[1, 0])))
    assert abs(k - tau * wl.fs) <= 1.0


def test_sample_voxels_seeded():
    a = synth.sample_voxels(1000, 10, 5)
    assert np.array_equal(a, synth.sample_voxels(1000, 10, 5))
    assert len(set(a.tolist())) == 10 and np.all(np.diff(a) > 0)
