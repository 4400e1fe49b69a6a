"""Seeded synthetic workloads for volumetric delay-and-sum.

This module only makes inputs: the matrix-array geometry, the voxel grid, the
per-voxel transmit delays and weights, and RF (or IQ) records that hold
Gaussian noise plus point-scatterer echoes.  It holds none of the beamforming
arithmetic (no receive delays of voxels, no interpolation, no summation) and
imports neither the CUDA library nor the oracle, so both sides can be fed the
same seeded arrays.

Workloads (all with c = 1540 m/s, t0 = 0, F# = 1.5, 0.3 mm pitch):

=======  ==========  ==============================  ==========================  ====  ====
name     array (M)   transmits (Q)                   record                      grid   B
=======  ==========  ==============================  ==========================  ====  ====
tiny     8x8 (64)    3 plane waves, x-z, -10/0/10 deg  K=512  f32  20 MHz          16^3    8
mid      16x16 (256) 5 plane waves, x-z, -12..12 deg   K=1024 f32  20 MHz          48^3   16
full     32x32 (1024) 9 diverging waves (3x3 sources)  K=2048 f32  20 MHz          64^3   32
iq       32x32 (1024) as full                           K=1024 c64 10 MHz, fd 5 MHz 64^3   64
large    32x32 (1024) 25 plane waves, 5x5 (tx, ty)      K=1536 f32  20 MHz         128^3   16
=======  ==========  ==============================  ==========================  ====  ====

Conventions chosen where the workload text leaves them open:
  * receiver m = iy * n_el + ix sits at ((ix - (n_el-1)/2) p, (iy - (n_el-1)/2) p, 0);
  * voxel grid: x, y in [-W, W] with W = n_el * p, z over the stated range, all
    axes sampled with both end points; voxel n = ix + nx * (iy + ny * iz);
  * plane wave with direction u = (sin tx, sin ty, sqrt(1 - sin^2 tx - sin^2 ty)):
    tau_tx = u . x / c (time zero when the front crosses the array centre);
  * diverging wave from virtual source v = (i 3.2 mm, j 3.2 mm, -10 mm),
    i, j in {-1, 0, 1}: tau_tx = (|x - v| - |v|) / c;
  * pulse: exp(-t^2 / (2 sigma^2)) cos(2 pi 5 MHz t), sigma = 2 cycles = 0.4 us,
    truncated at |t| <= 6 sigma; IQ echoes are the envelope times
    exp(-i 2 pi fd tau); amplitude 1 per channel, no spreading loss;
  * scatterers uniform in the grid's bounding box, shared by all frames;
    noise N(0, 1) per real sample (variance 1/2 per component for IQ),
    independent per frame;
  * draw order from ``numpy.random.default_rng(seed)``: scatterer positions,
    then w_tx (only when uniform in [0.5, 1]), then the noise.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

C_SOUND = 1540.0
PITCH = 0.3e-3
F0 = 5.0e6
SIGMA_T = 2.0 / F0          # two cycles of the 5 MHz centre frequency
TRUNC = 6.0                 # pulse support, in sigmas
FNUM = 1.5


@dataclass(frozen=True)
class Workload:
    name: str
    n_el: int                       # elements per side of the square array
    transmit: str                   # "pw" (plane waves) or "dw" (diverging waves)
    angles_x_deg: tuple = ()
    angles_y_deg: tuple = ()
    K: int = 512
    fs: float = 20e6
    iq: bool = False
    f_demod: float = 0.0
    nx: int = 16
    ny: int = 16
    nz: int = 16
    z_range: tuple = (5e-3, 20e-3)
    half_width: float | None = None  # default n_el * pitch
    B: int = 8
    n_scat: int = 3
    w_tx: str = "ones"              # "ones" or "uniform" ([0.5, 1])
    seed: int = 1
    c: float = C_SOUND
    t0: float = 0.0
    fnum: float = FNUM
    noise: bool = True
    echoes: bool = True
    extra: dict = field(default_factory=dict, compare=False)

    @property
    def M(self) -> int:
        return self.n_el * self.n_el

    @property
    def Q(self) -> int:
        if self.transmit == "dw":
            return 9
        if self.angles_y_deg:
            return len(self.angles_x_deg) * len(self.angles_y_deg)
        return len(self.angles_x_deg)

    @property
    def N(self) -> int:
        return self.nx * self.ny * self.nz

    @property
    def accumulations(self) -> int:
        return self.B * self.N * self.Q * self.M


_LIN12 = tuple(np.linspace(-12.0, 12.0, 5).tolist())

WORKLOADS = {
    "tiny": Workload("tiny", 8, "pw", angles_x_deg=(-10.0, 0.0, 10.0), K=512, fs=20e6,
                     nx=16, ny=16, nz=16, z_range=(5e-3, 20e-3), B=8, n_scat=3,
                     w_tx="ones", seed=1),
    "mid": Workload("mid", 16, "pw", angles_x_deg=_LIN12, K=1024, fs=20e6,
                    nx=48, ny=48, nz=48, z_range=(5e-3, 35e-3), B=16, n_scat=20,
                    w_tx="uniform", seed=2),
    "full": Workload("full", 32, "dw", K=2048, fs=20e6, nx=64, ny=64, nz=64,
                     z_range=(5e-3, 50e-3), B=32, n_scat=50, w_tx="ones", seed=3),
    "iq": Workload("iq", 32, "dw", K=1024, fs=10e6, iq=True, f_demod=5e6, nx=64, ny=64,
                   nz=64, z_range=(5e-3, 50e-3), B=64, n_scat=50, w_tx="ones", seed=4),
    "large": Workload("large", 32, "pw", angles_x_deg=_LIN12, angles_y_deg=_LIN12, K=1536,
                      fs=20e6, nx=128, ny=128, nz=128, z_range=(5e-3, 60e-3), B=16,
                      n_scat=200, w_tx="uniform", seed=5),
}


def workload(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (e.g. a smaller grid)."""
    return replace(WORKLOADS[name], **overrides)


@dataclass
class Problem:
    """Arrays of one synthetic workload, in the library's input layouts."""
    wl: Workload
    rx: np.ndarray          # M x 3 float32, metres
    grid: tuple             # (nx, ny, nz, x0, y0, z0, dx, dy, dz), spacings as float32 values
    tau_tx: np.ndarray      # Q x N float32, seconds
    w_tx: np.ndarray        # Q x N float32
    rf: np.ndarray          # B x Q x M x K float32 or complex64
    scatterers: np.ndarray  # S x 3 float64

    @property
    def B(self):
        return self.rf.shape[0]

    @property
    def Q(self):
        return self.rf.shape[1]

    @property
    def M(self):
        return self.rf.shape[2]

    @property
    def K(self):
        return self.rf.shape[3]

    @property
    def N(self):
        return self.tau_tx.shape[1]

    @property
    def c(self):
        return float(np.float32(self.wl.c))

    @property
    def fs(self):
        return float(np.float32(self.wl.fs))

    @property
    def t0(self):
        return float(np.float32(self.wl.t0))

    @property
    def fnum(self):
        return float(np.float32(self.wl.fnum))

    @property
    def f_demod(self):
        return float(np.float32(self.wl.f_demod))


def array_positions(n_el: int, pitch: float = PITCH) -> np.ndarray:
    """Square matrix array centred at the origin in the z = 0 plane (M x 3, float64)."""
    off = (np.arange(n_el, dtype=np.float64) - (n_el - 1) / 2.0) * pitch
    ix, iy = np.meshgrid(off, off, indexing="xy")      # ix varies fastest along a row
    return np.stack([ix.ravel(), iy.ravel(), np.zeros(n_el * n_el)], axis=1)


def grid_params(wl: Workload) -> tuple:
    """(nx, ny, nz, x0, y0, z0, dx, dy, dz) with float32-representable values."""
    W = wl.half_width if wl.half_width is not None else wl.n_el * PITCH
    z0, z1 = wl.z_range

    def axis(lo, hi, n):
        d = (hi - lo) / (n - 1) if n > 1 else 0.0
        return float(np.float32(lo)), float(np.float32(d))

    x0, dx = axis(-W, W, wl.nx)
    y0, dy = axis(-W, W, wl.ny)
    zz0, dz = axis(z0, z1, wl.nz)
    return (wl.nx, wl.ny, wl.nz, x0, y0, zz0, dx, dy, dz)


def grid_points(grid: tuple, idx=None) -> np.ndarray:
    """float64 positions of the listed voxels (default all), N x 3."""
    nx, ny, nz, x0, y0, z0, dx, dy, dz = grid
    n = np.arange(nx * ny * nz, dtype=np.int64) if idx is None else np.asarray(idx, np.int64)
    ix = n % nx
    iy = (n // nx) % ny
    iz = n // (nx * ny)
    return np.stack([x0 + ix * dx, y0 + iy * dy, z0 + iz * dz], axis=1)


def transmit_directions(wl: Workload) -> np.ndarray:
    """Unit propagation vectors of the plane waves (Q x 3)."""
    if wl.angles_y_deg:
        tx, ty = np.meshgrid(np.deg2rad(wl.angles_x_deg), np.deg2rad(wl.angles_y_deg),
                             indexing="xy")
        sx, sy = np.sin(tx.ravel()), np.sin(ty.ravel())
    else:
        sx = np.sin(np.deg2rad(np.asarray(wl.angles_x_deg, dtype=np.float64)))
        sy = np.zeros_like(sx)
    sz = np.sqrt(1.0 - sx * sx - sy * sy)
    return np.stack([sx, sy, sz], axis=1)


def virtual_sources() -> np.ndarray:
    """3 x 3 diverging-wave sources 10 mm behind the array (Q=9 x 3)."""
    s = 3.2e-3
    ii, jj = np.meshgrid([-1.0, 0.0, 1.0], [-1.0, 0.0, 1.0], indexing="xy")
    return np.stack([ii.ravel() * s, jj.ravel() * s, np.full(9, -10e-3)], axis=1)


def transmit_delays(wl: Workload, pts: np.ndarray) -> np.ndarray:
    """Transmit arrival time at each point for each transmit, Q x P float64 (s)."""
    if wl.transmit == "dw":
        v = virtual_sources()
        out = np.empty((9, pts.shape[0]), dtype=np.float64)
        for q in range(9):
            out[q] = (np.linalg.norm(pts - v[q], axis=1) - np.linalg.norm(v[q])) / wl.c
        return out
    u = transmit_directions(wl)
    return (u @ pts.T) / wl.c


def pulse(t: np.ndarray) -> np.ndarray:
    """Gaussian-windowed 5 MHz pulse, zero beyond 6 sigma."""
    g = np.exp(-0.5 * (t / SIGMA_T) ** 2) * np.cos(2.0 * math.pi * F0 * t)
    return np.where(np.abs(t) <= TRUNC * SIGMA_T, g, 0.0)


def envelope(t: np.ndarray) -> np.ndarray:
    """Complex-baseband envelope of :func:`pulse` (Gaussian), zero beyond 6 sigma."""
    g = np.exp(-0.5 * (t / SIGMA_T) ** 2)
    return np.where(np.abs(t) <= TRUNC * SIGMA_T, g, 0.0)


def echo_record(wl: Workload, rx: np.ndarray, scat: np.ndarray, K: int | None = None,
                amplitude: float = 1.0) -> np.ndarray:
    """Noise-free echoes of the point scatterers, Q x M x K (float64 or complex128).

    Forward model: the echo of scatterer s on transmit q and receiver m arrives
    at tau_tx(q, x_s) + |x_s - r_m| / c and has the pulse (or, for IQ, its
    envelope times exp(-i 2 pi fd tau)) as its shape.
    """
    K = wl.K if K is None else K
    Q, M = wl.Q, rx.shape[0]
    rec = np.zeros((Q, M, K), dtype=np.complex128 if wl.iq else np.float64)
    half = int(math.ceil(TRUNC * SIGMA_T * wl.fs)) + 1
    offs = np.arange(-half, half + 1, dtype=np.int64)
    qq, mm = np.meshgrid(np.arange(Q), np.arange(M), indexing="ij")
    for s in range(scat.shape[0]):
        p = scat[s:s + 1]
        tau = transmit_delays(wl, p)[:, 0][:, None] + np.linalg.norm(p - rx, axis=1)[None, :] / wl.c
        kc = np.rint((tau - wl.t0) * wl.fs).astype(np.int64)          # Q x M
        kk = kc[..., None] + offs                                      # Q x M x W
        ok = (kk >= 0) & (kk < K)
        t = wl.t0 + kk / wl.fs - tau[..., None]
        if wl.iq:
            val = envelope(t) * np.exp(-2j * math.pi * wl.f_demod * tau)[..., None]
        else:
            val = pulse(t)
        val = amplitude * val
        qi = np.broadcast_to(qq[..., None], kk.shape)[ok]
        mi = np.broadcast_to(mm[..., None], kk.shape)[ok]
        rec[qi, mi, kk[ok]] += val[ok]        # indices are unique within one scatterer
    return rec


def make_problem(wl: Workload | str, **overrides) -> Problem:
    """Builds every input array of a workload from its seed."""
    if isinstance(wl, str):
        wl = workload(wl, **overrides)
    elif overrides:
        wl = replace(wl, **overrides)
    rng = np.random.default_rng(wl.seed)
    rx64 = array_positions(wl.n_el)
    grid = grid_params(wl)
    pts = grid_points(grid)
    nx, ny, nz, x0, y0, z0, dx, dy, dz = grid
    lo = np.array([x0, y0, z0])
    hi = np.array([x0 + (nx - 1) * dx, y0 + (ny - 1) * dy, z0 + (nz - 1) * dz])
    scat = lo + (hi - lo) * rng.random((wl.n_scat, 3))
    Q, M, K, B, N = wl.Q, wl.M, wl.K, wl.B, wl.N
    tau_tx = transmit_delays(wl, pts).astype(np.float32)
    if wl.w_tx == "uniform":
        w_tx = rng.uniform(0.5, 1.0, size=(Q, N)).astype(np.float32)
    else:
        w_tx = np.ones((Q, N), dtype=np.float32)
    rx = rx64.astype(np.float32)
    if wl.iq:
        parts = np.zeros((B, Q, M, K, 2), dtype=np.float32)
        if wl.noise:
            rng.standard_normal(out=parts, dtype=np.float32)
            parts *= np.float32(math.sqrt(0.5))
        rf = parts.view(np.complex64)[..., 0]
    else:
        rf = np.zeros((B, Q, M, K), dtype=np.float32)
        if wl.noise:
            rng.standard_normal(out=rf, dtype=np.float32)
    if wl.echoes and wl.n_scat > 0:
        # the echoes travel to the float32 receiver positions the library is given
        rec = echo_record(wl, rx.astype(np.float64), scat)
        rf += rec.astype(rf.dtype)[None]
    return Problem(wl=wl, rx=rx, grid=grid, tau_tx=tau_tx, w_tx=w_tx, rf=rf, scatterers=scat)


def sample_voxels(N: int, count: int, seed: int) -> np.ndarray:
    """Sorted seeded sample of distinct voxel indices (``default_rng(seed)``)."""
    count = min(count, N)
    return np.sort(np.random.default_rng(seed).choice(N, count, replace=False)).astype(np.int64)
