"""Seeded random small delay-and-sum problems for the randomized tests: a
regular grid, receivers on both sides of the voxels (behind the array the
aperture is closed), delays that run off both ends of the record, t0 of either
sign, the aperture on or off, real or IQ records.  Inputs only: no part of the
sum is computed here."""
from __future__ import annotations

import numpy as np

from oracle import Grid


def make_case(seed, frames=(1, 2, 3), max_k=24, max_m=6, max_q=3, max_side=3):
    """(grid, rx, rf, tau_tx, w_tx, kwargs of the sum) for one seed."""
    rng = np.random.default_rng(1000 + seed)
    nx, ny, nz = (int(v) for v in rng.integers(1, max_side + 1, 3))
    grid = Grid(nx, ny, nz, *rng.uniform(-0.5e-3, 0.5e-3, 2), rng.uniform(1e-3, 3e-3),
                *rng.uniform(0.05e-3, 0.4e-3, 3))
    B = int(rng.choice(frames))
    Q, M, K = int(rng.integers(1, max_q + 1)), int(rng.integers(1, max_m + 1)), int(rng.integers(2, max_k + 1))
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
    return grid, rx.astype(np.float32), rf, tau, w, dict(c=c, fs=fs, t0=t0, fnum=fnum, f_demod=f_demod)


def grid_xyz(grid):
    n = np.arange(grid.n)
    return np.stack([grid.x0 + (n % grid.nx) * grid.dx,
                     grid.y0 + (n // grid.nx % grid.ny) * grid.dy,
                     grid.z0 + (n // (grid.nx * grid.ny)) * grid.dz], axis=1)
