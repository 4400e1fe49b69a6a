"""The oracle against the independent pure-Python statement of the sum
(tests/brute_force.py) on many seeded random small problems: grids of 1 to 3
voxels per axis, receivers on both sides of the voxels (behind the array the
aperture is closed), records of 2 to 24 samples with delays running off both
ends, t0 on either side of zero, the aperture on and off, real and IQ records.
Each case is small enough for the brute force (hat-function interpolation
over every sample, fsum) to run in milliseconds."""
import numpy as np
import pytest

from brute_force import das_bruteforce
from oracle import Grid

CASES = 48


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    nx, ny, nz = (int(v) for v in rng.integers(1, 4, 3))
    grid = Grid(nx, ny, nz, *rng.uniform(-0.5e-3, 0.5e-3, 2), rng.uniform(1e-3, 3e-3),
                *rng.uniform(0.05e-3, 0.4e-3, 3))
    B, Q, M, K = int(rng.integers(1, 4)), int(rng.integers(1, 4)), int(rng.integers(1, 7)), int(rng.integers(2, 25))
    rx = np.column_stack([rng.uniform(-1e-3, 1e-3, M), rng.uniform(-1e-3, 1e-3, M),
                          rng.choice([0.0, 0.0, 0.0, 5e-3], M)])          # some receivers below the voxels
    c, fs = 1540.0, float(rng.choice([10e6, 20e6, 40e6]))
    t0 = float(rng.uniform(-2.0, 2.0)) / fs
    fnum = float(rng.choice([0.0, 0.0, 0.5, 1.0, 1.5]))
    # delays that put f anywhere in [-3, K + 3] for a typical voxel-receiver distance
    d_typ = np.sqrt(1e-6 + grid.z0 ** 2) / c
    tau = (rng.uniform(-3.0, K + 3.0, (Q, grid.n)) / fs - d_typ + t0).astype(np.float32)
    w = rng.uniform(-1.0, 2.0, (Q, grid.n)).astype(np.float32)
    complex_data = bool(rng.integers(0, 2))
    if complex_data:
        rf = (rng.standard_normal((B, Q, M, K)) + 1j * rng.standard_normal((B, Q, M, K))).astype(np.complex64)
        f_demod = float(rng.uniform(1e6, 8e6))
    else:
        rf = rng.standard_normal((B, Q, M, K)).astype(np.float32)
        f_demod = 0.0
    return grid, rx, rf, tau, w, dict(c=c, fs=fs, t0=t0, fnum=fnum, f_demod=f_demod)


def _xyz(grid):
    n = np.arange(grid.n)
    return np.stack([grid.x0 + (n % grid.nx) * grid.dx,
                     grid.y0 + (n // grid.nx % grid.ny) * grid.dy,
                     grid.z0 + (n // (grid.nx * grid.ny)) * grid.dz], axis=1)


@pytest.mark.parametrize("seed", range(CASES))
def test_oracle_matches_brute_force_on_random_problems(oracle, seed):
    grid, rx, rf, tau, w, kw = _case(seed)
    y = oracle.beamform(rf, tau, w, rx, grid, **kw)
    ref = das_bruteforce(rf, tau, w, rx, _xyz(grid), **kw)
    scale = max(1.0, float(np.abs(ref).max()))
    assert np.abs(y - ref).max() <= 1e-12 * scale, (seed, float(np.abs(y - ref).max()))


def test_random_problems_reach_every_branch(oracle):
    """The seeded cases together cover what they are meant to: non-zero output,
    pairs off both record ends, closed apertures, complex records."""
    lo = hi = closed = cplx = nonzero = 0
    for seed in range(CASES):
        grid, rx, rf, tau, w, kw = _case(seed)
        xyz = _xyz(grid)
        cplx += np.iscomplexobj(rf)
        d = np.linalg.norm(xyz[None, :, :] - rx[:, None, :], axis=2)        # M x N
        f = ((tau.astype(np.float64)[:, None, :] + d[None] / kw["c"]) - kw["t0"]) * kw["fs"]
        lo += int((f < 0).any())
        hi += int((f > rf.shape[-1] - 1).any())
        closed += int((xyz[None, :, 2] - rx[:, None, 2] <= 0).any() or kw["fnum"] > 0)
        y = oracle.beamform(rf, tau, w, rx, grid, **kw)
        nonzero += int(np.abs(y).max() > 0)
    assert min(lo, hi, closed, cplx) >= 5 and nonzero >= CASES * 3 // 4, (lo, hi, closed, cplx, nonzero)
