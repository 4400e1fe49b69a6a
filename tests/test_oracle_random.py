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
from random_cases import grid_xyz as _xyz
from random_cases import make_case as _case

CASES = 48


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
