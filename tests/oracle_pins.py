"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each ``pin_*`` takes an :class:`oracle.Oracle` and raises ``AssertionError``
when the oracle disagrees with:

* closed forms worked out by hand below (impulse records, constant IQ records,
  exact Pythagorean geometry with dyadic delays, so every expected value is an
  exact binary fraction);
* an independent pure-Python statement of the formula (``brute_force.py``);
* exact rational counts of the receivers inside the F-number aperture;
* invariants of the method: linearity in the record, shift of the record
  against t0, a point scatterer focusing at its own voxel;
* the library routine ``numpy.transpose`` (permute) and hand-computed grid
  positions.

The same list runs against mutated copies of the oracle in
``test_oracle_mutants.py``: every planted mistake must fail at least one pin.
"""
from __future__ import annotations

import cmath
import math
from fractions import Fraction

import numpy as np

from brute_force import das_bruteforce
from oracle import Grid
from volumetric_ultrasound_delay_gb300 import synth

# --------------------------------------------------------------------------
# exact Pythagorean geometry: one voxel at (0, 0, 10), receivers at integer
# distances from it (units with c = fs = 1, so a delay in seconds is a sample)
VOX = Grid(1, 1, 1, 0.0, 0.0, 10.0, 1.0, 1.0, 1.0)
RX_PYTH = np.array([
    [1.0, 2.0, 8.0],     # d = 3   (1, 2, 2)
    [2.0, 3.0, 4.0],     # d = 7   (2, 3, 6)
    [1.0, 4.0, 2.0],     # d = 9   (1, 4, 8)
    [4.0, 4.0, 3.0],     # d = 9   (4, 4, 7)
    [0.0, 6.0, 2.0],     # d = 10  (0, 6, 8)
    [2.0, 6.0, 1.0],     # d = 11  (2, 6, 9)
    [0.0, 0.0, 19.0],    # d = 9, above the voxel (dz < 0)
    [3.0, 4.0, -2.0],    # d = 13  (3, 4, 12)
])
TAU_Q = np.array([[0.0], [0.25], [0.5]], dtype=np.float32)   # Q = 3, dyadic
W_Q = np.array([[1.0], [2.0], [3.0]], dtype=np.float32)


def _impulse(B, K, kstar):
    rf = np.zeros((B, 3, RX_PYTH.shape[0], K), dtype=np.float32)
    for b in range(B):
        rf[b, :, :, kstar] = b + 1
    return rf


def pin_impulse_interior(orc):
    """Impulse at k*=10: hat weights of f = d + tau_q, worked out by hand.

    d = 9 (three receivers, aperture off): f = 9, 9.25, 9.5 -> 0, .25, .5;
    weighted by w = 1, 2, 3 -> 2.0 each -> 6.0.  d = 10: f = 10, 10.25, 10.5 ->
    1, .75, .5 -> 1 + 1.5 + 1.5 = 4.0.  d = 11: f >= 11 -> 0.  Total 10 (b+1).
    """
    B = 2
    y = orc.beamform(_impulse(B, 16, 10), TAU_Q, W_Q, RX_PYTH, VOX, c=1.0, fs=1.0,
                     t0=0.0, fnum=0.0)
    expect = np.array([[10.0], [20.0]])
    assert np.allclose(y, expect, rtol=0, atol=1e-12), (y, expect)


def pin_impulse_upper_edge(orc):
    """Impulse at the last sample k* = K-1 = 9: a sample past the record counts
    as zero on its own, so f in (9, 10) keeps (1 - a) s[9].

    d = 9: f = 9, 9.25, 9.5 -> 1, .75, .5 -> 1 + 1.5 + 1.5 = 4 per receiver,
    three receivers -> 12.  d = 10 starts at k0 = 10 > K-1 -> 0.  Total 12 (b+1).
    """
    B = 2
    y = orc.beamform(_impulse(B, 10, 9), TAU_Q, W_Q, RX_PYTH, VOX, c=1.0, fs=1.0,
                     t0=0.0, fnum=0.0)
    expect = np.array([[12.0], [24.0]])
    assert np.allclose(y, expect, rtol=0, atol=1e-12), (y, expect)


def pin_impulse_lower_edge(orc):
    """Impulse at k* = 0 with t0 = 3.75 s (c = fs = 1): only d = 3 reaches it,
    at f = -0.75, -0.5, -0.25, i.e. k0 = -1 with a = .25, .5, .75 -> a s[0];
    weighted 1, 2, 3 -> 0.25 + 1 + 2.25 = 3.5 (b+1)."""
    B = 2
    y = orc.beamform(_impulse(B, 16, 0), TAU_Q, W_Q, RX_PYTH, VOX, c=1.0, fs=1.0,
                     t0=3.75, fnum=0.0)
    expect = np.array([[3.5], [7.0]])
    assert np.allclose(y, expect, rtol=0, atol=1e-12), (y, expect)


def pin_iq_constant_record(orc):
    """Constant IQ record s = 0.5 - 0.25i, one receiver at d = 9, tau_tx = 0.25,
    t0 = 2, w = 3, f_demod = 1/16: y = 3 s exp(+i 2 pi f_demod (0.25 + 9)); the
    phase uses the two-way delay, not the delay minus t0."""
    rf = np.full((1, 1, 1, 16), 0.5 - 0.25j, dtype=np.complex64)
    y = orc.beamform(rf, np.array([[0.25]], np.float32), np.array([[3.0]], np.float32),
                     RX_PYTH[2:3], VOX, c=1.0, fs=1.0, t0=2.0, fnum=0.0, f_demod=1.0 / 16)
    expect = 3.0 * (0.5 - 0.25j) * cmath.exp(2j * math.pi * (9.25 / 16))
    assert abs(y[0, 0] - expect) < 1e-12, (y, expect)


# --------------------------------------------------------------------------
# all-ones record: y = Q * (number of receivers inside the aperture), counted
# with exact rational arithmetic on dyadic coordinates (so float64 is exact)
def _aperture_count(vox, rx, fnum):
    two_f = Fraction(2) * Fraction(fnum)
    count, ties = 0, 0
    for r in rx:
        ex, ey, ez = (Fraction(float(vox[i])) - Fraction(float(r[i])) for i in range(3))
        if ez <= 0:
            continue
        lhs = two_f * two_f * (ex * ex + ey * ey)
        if lhs <= ez * ez:
            count += 1
            ties += lhs == ez * ez
    return count, ties


def _dyadic_scene():
    grid = Grid(5, 4, 3, -1.0, -0.75, 0.5, 0.5, 0.5, 1.0)
    ii, jj = np.meshgrid(np.arange(6), np.arange(5), indexing="xy")
    rx = np.stack([ii.ravel() * 0.25 - 0.75, jj.ravel() * 0.375 - 0.75,
                   np.zeros(ii.size)], axis=1)
    rx = np.vstack([rx, [[0.0, 0.0, 2.0], [0.5, -0.5, 1.25]]])  # two receivers above some voxels
    return grid, rx


def pin_all_ones_aperture_count(orc):
    """s = 1, w_tx = 1, every f inside the record: y[b,n] = Q * count(n),
    where count uses (2 F#) rho <= dz, boundary included, dz > 0 only."""
    grid, rx = _dyadic_scene()
    Q, B, K, fnum = 2, 2, 64, 1.5
    rf = np.ones((B, Q, rx.shape[0], K), np.float32)
    tau = np.ones((Q, grid.n), np.float32)
    w = np.ones((Q, grid.n), np.float32)
    y = orc.beamform(rf, tau, w, rx, grid, c=1.0, fs=1.0, fnum=fnum)
    vox = [(grid.x0 + (n % grid.nx) * grid.dx, grid.y0 + (n // grid.nx % grid.ny) * grid.dy,
            grid.z0 + (n // (grid.nx * grid.ny)) * grid.dz) for n in range(grid.n)]
    total_ties = 0
    for n in range(grid.n):
        cnt, ties = _aperture_count(vox[n], rx, fnum)
        total_ties += ties
        for b in range(B):
            assert abs(y[b, n] - Q * cnt) < 1e-9, (n, b, y[b, n], Q * cnt)
    assert total_ties > 0  # the inclusive boundary is really exercised


def pin_aperture_tie_slack(orc):
    """A receiver exactly on the aperture boundary is counted, and its
    |contribution| is reported as slack; a strictly inside one is not."""
    vox = Grid(1, 1, 1, 0.0, 0.0, 3.0, 1.0, 1.0, 1.0)
    rx = np.array([[0.0, 0.0, 0.0],      # rho = 0: strictly inside
                   [1.0, 0.0, 0.0]])     # rho = 1, dz = 3, F# = 1.5: exactly on it
    rf = -np.ones((1, 1, 2, 16), np.float32)
    y, slack = orc.beamform(rf, np.zeros((1, 1), np.float32), np.full((1, 1), 2.0, np.float32),
                            rx, vox, c=1.0, fs=1.0, fnum=1.5, want_slack=True)
    assert abs(y[0, 0] - (-4.0)) < 1e-12, y
    assert abs(slack[0, 0] - 2.0) < 1e-12, slack


# --------------------------------------------------------------------------
# against the independent pure-Python statement of the formula
def _small_random_case(seed, complex_data):
    rng = np.random.default_rng(seed)
    grid = Grid(2, 2, 2, -0.2e-3, 0.1e-3, 1.0e-3, 0.35e-3, 0.3e-3, 0.6e-3)
    rx = np.column_stack([rng.uniform(-0.5e-3, 0.5e-3, 4), rng.uniform(-0.4e-3, 0.6e-3, 4),
                          np.array([0.0, 0.0, 0.0, 1.5e-3])])
    B, Q, M, K = 3, 2, 4, 40
    fs, c = 20e6, 1540.0
    tau = (rng.uniform(-30.0, 20.0, (Q, grid.n)) / fs).astype(np.float32)
    w = rng.uniform(0.5, 1.5, (Q, grid.n)).astype(np.float32)
    if complex_data:
        rf = (rng.standard_normal((B, Q, M, K)) + 1j * rng.standard_normal((B, Q, M, K))
              ).astype(np.complex64)
    else:
        rf = rng.standard_normal((B, Q, M, K)).astype(np.float32)
    return grid, rx, rf, tau, w, c, fs


def _grid_xyz(grid):
    n = np.arange(grid.n)
    return np.stack([grid.x0 + (n % grid.nx) * grid.dx,
                     grid.y0 + (n // grid.nx % grid.ny) * grid.dy,
                     grid.z0 + (n // (grid.nx * grid.ny)) * grid.dz], axis=1)


def pin_bruteforce_real(orc):
    grid, rx, rf, tau, w, c, fs = _small_random_case(11, False)
    kw = dict(c=c, fs=fs, t0=2.5 / fs, fnum=1.0)
    y = orc.beamform(rf, tau, w, rx, grid, **kw)
    ref = das_bruteforce(rf, tau, w, rx, _grid_xyz(grid), **kw)
    assert np.abs(ref).max() > 1.0
    assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max(), np.abs(y - ref).max()


def pin_bruteforce_complex(orc):
    grid, rx, rf, tau, w, c, fs = _small_random_case(12, True)
    kw = dict(c=c, fs=fs, t0=-1.5 / fs, fnum=1.0, f_demod=5e6)
    y = orc.beamform(rf, tau, w, rx, grid, **kw)
    ref = das_bruteforce(rf, tau, w, rx, _grid_xyz(grid), **kw)
    assert np.abs(ref).max() > 1.0
    assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max(), np.abs(y - ref).max()


def pin_bruteforce_float64_records(orc):
    """float64 and complex128 records are read at full precision: values that
    float32 cannot hold (1 + 1e-12 style) must survive into y."""
    for seed, complex_data in ((17, False), (18, True)):
        grid, rx, rf32, tau, w, c, fs = _small_random_case(seed, complex_data)
        rng = np.random.default_rng(seed + 100)
        rf = rf32.astype(np.complex128 if complex_data else np.float64)
        rf = rf + rng.standard_normal(rf.shape) * 1e-9          # below float32 resolution
        kw = dict(c=c, fs=fs, t0=0.5 / fs, fnum=1.0, f_demod=5e6 if complex_data else 0.0)
        y = orc.beamform(rf, tau, w, rx, grid, **kw)
        ref = das_bruteforce(rf, tau, w, rx, _grid_xyz(grid), **kw)
        assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max(), np.abs(y - ref).max()
        y32 = orc.beamform(rf32, tau, w, rx, grid, **kw)
        assert np.abs(y - y32).max() > 1e-12 * np.abs(ref).max()   # the perturbation is seen


# --------------------------------------------------------------------------
# invariants
def pin_linearity(orc):
    """y(2 s1 - 3 s2) = 2 y(s1) - 3 y(s2); the records hold small integers so the
    combination is exact in float32."""
    grid, rx, _, tau, w, c, fs = _small_random_case(13, False)
    rng = np.random.default_rng(14)
    s1 = rng.integers(-8, 9, (2, 2, 4, 40)).astype(np.float32)
    s2 = rng.integers(-8, 9, (2, 2, 4, 40)).astype(np.float32)
    kw = dict(c=c, fs=fs, fnum=1.0)
    y12 = orc.beamform(2 * s1 - 3 * s2, tau, w, rx, grid, **kw)
    y1 = orc.beamform(s1, tau, w, rx, grid, **kw)
    y2 = orc.beamform(s2, tau, w, rx, grid, **kw)
    assert np.abs(y12 - (2 * y1 - 3 * y2)).max() <= 1e-12 * max(1.0, np.abs(y12).max())


def pin_shift_invariance(orc):
    """A record that starts j samples earlier holds the same data j samples
    later (zero filled in front) and has its t0 moved j / fs earlier: y is
    unchanged (t0 is the time of sample 0, in seconds, subtracted from tau)."""
    rng = np.random.default_rng(15)
    grid = Grid(3, 2, 2, -0.3e-3, -0.2e-3, 3.0e-3, 0.3e-3, 0.4e-3, 0.5e-3)
    rx = np.column_stack([rng.uniform(-1e-3, 1e-3, 6), rng.uniform(-1e-3, 1e-3, 6), np.zeros(6)])
    B, Q, M, K, j = 2, 2, 6, 256, 5
    fs, c, t0 = 20e6, 1540.0, 1.0 / 20e6
    tau = (rng.uniform(10.0, 40.0, (Q, grid.n)) / fs).astype(np.float32)
    w = rng.uniform(0.5, 1.0, (Q, grid.n)).astype(np.float32)
    rf = rng.standard_normal((B, Q, M, K)).astype(np.float32)
    shifted = np.zeros_like(rf)
    shifted[..., j:] = rf[..., :-j]
    y = orc.beamform(rf, tau, w, rx, grid, c=c, fs=fs, t0=t0, fnum=1.0)
    ys = orc.beamform(shifted, tau, w, rx, grid, c=c, fs=fs, t0=t0 - j / fs, fnum=1.0)
    assert np.abs(y).max() > 1.0
    assert np.abs(y - ys).max() <= 1e-9 * np.abs(y).max(), np.abs(y - ys).max()


def _scatter_scene(iq):
    """Noise-free echo of one scatterer placed exactly on the central voxel."""
    wl = synth.workload("iq" if iq else "tiny", n_el=8, nx=9, ny=9, nz=9,
                        z_range=(8e-3, 16e-3), half_width=2.4e-3, K=256 if iq else 512,
                        B=2, n_scat=0)
    grid = synth.grid_params(wl)
    g = Grid(*grid)
    n_s = 4 + 9 * (4 + 9 * 4)                       # the central voxel
    pos = synth.grid_points(grid, [n_s])
    rx = synth.array_positions(wl.n_el).astype(np.float32).astype(np.float64)
    rec = synth.echo_record(wl, rx, pos)
    rf = np.broadcast_to(rec[None], (2,) + rec.shape).astype(np.complex64 if iq else np.float32)
    tau = synth.transmit_delays(wl, synth.grid_points(grid)).astype(np.float32)
    w = np.ones_like(tau)
    return wl, g, rx, rf, tau, w, n_s


def pin_point_scatterer_real(orc):
    wl, g, rx, rf, tau, w, n_s = _scatter_scene(False)
    y = orc.beamform(rf, tau, w, rx, g, c=wl.c, fs=wl.fs, fnum=wl.fnum)
    for b in range(2):
        assert int(np.argmax(np.abs(y[b]))) == n_s
        # all 64 receivers are inside the aperture at 12 mm; linear interpolation
        # of a 5 MHz pulse at 4 samples per period keeps at least cos(pi/4)
        assert 0.7 * wl.Q * 64 <= y[b, n_s] <= wl.Q * 64 + 1e-9


def pin_point_scatterer_iq(orc):
    wl, g, rx, rf, tau, w, n_s = _scatter_scene(True)
    y = orc.beamform(rf, tau, w, rx, g, c=wl.c, fs=wl.fs, fnum=wl.fnum, f_demod=wl.f_demod)
    for b in range(2):
        assert int(np.argmax(np.abs(y[b]))) == n_s
        # phase-aligned sum of the Gaussian envelope (sigma = 4 samples at 10 MHz)
        assert 0.95 * wl.Q * 64 <= abs(y[b, n_s]) <= wl.Q * 64 + 1e-9


# --------------------------------------------------------------------------
# layout helpers
def pin_permute_matches_numpy(orc):
    rng = np.random.default_rng(16)
    for dt in (np.float32, np.complex64, np.float16):
        B, Q, M, K = 3, 2, 5, 7
        if dt == np.complex64:
            rf = (rng.standard_normal((B, Q, M, K)) + 1j * rng.standard_normal((B, Q, M, K))).astype(dt)
        else:
            rf = rng.standard_normal((B, Q, M, K)).astype(dt)
        out = orc.permute(rf, "kqmb")
        assert out.tobytes() == np.ascontiguousarray(rf.transpose(3, 1, 2, 0)).tobytes()
        out = orc.permute(rf, "qmkb")
        assert out.tobytes() == np.ascontiguousarray(rf.transpose(1, 2, 3, 0)).tobytes()


def pin_voxel_positions(orc):
    g = Grid(3, 4, 5, -1.0, 2.0, 0.5, 0.25, 0.5, 2.0)
    xyz = orc.voxel_positions(g, [0, 2, 3, 11, 12, 59])
    expect = np.array([[-1.0, 2.0, 0.5],       # n = 0
                       [-0.5, 2.0, 0.5],       # ix = 2
                       [-1.0, 2.5, 0.5],       # iy = 1
                       [-0.5, 3.5, 0.5],       # ix = 2, iy = 3
                       [-1.0, 2.0, 2.5],       # iz = 1
                       [-0.5, 3.5, 8.5]])      # last voxel
    assert np.array_equal(xyz, expect), xyz


def pin_hand_worked_examples(orc):
    """The two delay-and-sum sums of tests/golden/ (record edges, the aperture,
    the IQ phase and its sign), worked out by hand in the fixture."""
    import golden_cases
    for ex in golden_cases.examples():
        rf, tau, w, rx = golden_cases.inputs(ex)
        y = orc.beamform(rf, tau, w, rx.astype(np.float64), Grid(*ex["grid"]), c=ex["c"],
                         fs=ex["fs"], t0=ex["t0"], fnum=ex["fnum"], f_demod=ex["f_demod"])
        ref = golden_cases.expected(ex)
        assert np.abs(y - ref).max() <= 1e-12 * np.abs(ref).max(), ex["name"]


ALL_PINS = [
    pin_hand_worked_examples,
    pin_impulse_interior, pin_impulse_upper_edge, pin_impulse_lower_edge,
    pin_iq_constant_record, pin_all_ones_aperture_count, pin_aperture_tie_slack,
    pin_bruteforce_real, pin_bruteforce_complex, pin_bruteforce_float64_records,
    pin_linearity, pin_shift_invariance,
    pin_point_scatterer_real, pin_point_scatterer_iq, pin_permute_matches_numpy,
    pin_voxel_positions,
]
