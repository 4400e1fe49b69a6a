"""TEST INFRASTRUCTURE ONLY: ctypes front end to the float64 CPU oracle.

The oracle (``das_oracle.c`` beside this file) is the plain, slow definition of
volumetric delay-and-sum that the CUDA library is checked against.  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product library never does, and it shares no code
with it.

Functions:
  * :func:`build` compiles ``das_oracle.c`` with gcc (OpenMP when available).
  * :class:`Oracle` wraps one compiled copy; ``load()`` returns the default one.
    ``Oracle(path)`` loads another build of the same source (the mutation
    tests use this to plant mistakes in a private copy).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "das_oracle.c"
BUILD_DIR = HERE / "_build"
LIBRARY = BUILD_DIR / "liboracle.so"

_I64P = ctypes.POINTER(ctypes.c_int64)
_F32P = ctypes.POINTER(ctypes.c_float)
_F64P = ctypes.POINTER(ctypes.c_double)


def compile_source(src: Path, out: Path) -> Path:
    """Compiles one oracle source file to a shared library with gcc."""
    out.parent.mkdir(parents=True, exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", str(src), "-o", str(out)]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # no OpenMP runtime: the oracle is still correct, just single threaded
        subprocess.run(base + ["-lm"], check=True, capture_output=True, text=True)
    return out


def build(force: bool = False) -> Path:
    """Builds ``_build/liboracle.so`` unless it is newer than the source."""
    if force or not LIBRARY.exists() or LIBRARY.stat().st_mtime < SOURCE.stat().st_mtime:
        tmp = LIBRARY.with_suffix(f".{os.getpid()}.tmp.so")
        compile_source(SOURCE, tmp)
        os.replace(tmp, LIBRARY)
    return LIBRARY


@dataclass(frozen=True)
class Grid:
    """Regular voxel grid: n = ix + nx*(iy + ny*iz), x = x0 + ix*dx, etc. (metres)."""
    nx: int
    ny: int
    nz: int
    x0: float
    y0: float
    z0: float
    dx: float
    dy: float
    dz: float

    @property
    def n(self) -> int:
        return self.nx * self.ny * self.nz


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


class Oracle:
    """One loaded copy of the compiled oracle."""

    def __init__(self, path: str | os.PathLike | None = None):
        if path is None:
            path = build()
        self.path = str(path)
        lib = ctypes.CDLL(self.path)
        lib.das_oracle_voxel_positions.restype = ctypes.c_int
        lib.das_oracle_voxel_positions.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_double, ctypes.c_double,
            ctypes.c_double, ctypes.c_double, ctypes.c_double,
            _I64P, ctypes.c_int64, _F64P]
        lib.das_oracle_beamform.restype = ctypes.c_int
        lib.das_oracle_beamform.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int, _F32P, _F32P, _F64P,
            _F64P, _I64P, ctypes.c_int64,
            ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double,
            ctypes.c_double, ctypes.c_double, _F64P, ctypes.c_void_p, ctypes.c_int]
        lib.das_oracle_permute.restype = ctypes.c_int
        lib.das_oracle_permute.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        self._lib = lib

    # ------------------------------------------------------------------ grid
    def voxel_positions(self, grid: Grid, idx) -> np.ndarray:
        """float64 positions (n_eval x 3) of the listed voxels of ``grid``."""
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        xyz = np.empty((idx.size, 3), dtype=np.float64)
        rc = self._lib.das_oracle_voxel_positions(
            grid.nx, grid.ny, grid.nz, float(grid.x0), float(grid.y0), float(grid.z0),
            float(grid.dx), float(grid.dy), float(grid.dz), _ptr(idx, _I64P), idx.size,
            _ptr(xyz, _F64P))
        if rc != 0:
            raise ValueError("das_oracle_voxel_positions: invalid arguments")
        return xyz

    # ------------------------------------------------------------- beamform
    def beamform(self, rf, tau_tx, w_tx, rx_xyz, grid: Grid | None = None, *,
                 vox_xyz=None, idx=None, c: float, fs: float, t0: float = 0.0,
                 fnum: float = 0.0, f_demod: float = 0.0, tie_rel: float = 1e-5,
                 want_slack: bool = False, nthreads: int = 0):
        """Evaluates y[b, n] for the voxels ``idx`` (default: all of ``grid``).

        ``rf`` is B x Q x M x K float32, complex64, float64 or complex128;
        ``tau_tx``/``w_tx`` are
        Q x N float32; ``rx_xyz`` is M x 3.  Voxel positions come from ``grid``
        (the regular-grid definition) unless ``vox_xyz`` (n_eval x 3) is given.
        Returns ``y`` (B x n_eval, float64 or complex128) and, with
        ``want_slack``, the per-output aperture-tie slack (B x n_eval).
        """
        rf = np.ascontiguousarray(rf)
        types = {np.dtype(np.float32): 0, np.dtype(np.complex64): 1,
                 np.dtype(np.float64): 2, np.dtype(np.complex128): 3}
        if rf.dtype not in types:
            raise TypeError("rf must be float32, complex64, float64 or complex128")
        rf_type = types[rf.dtype]
        is_complex = rf_type & 1
        B, Q, M, K = rf.shape
        tau_tx = np.ascontiguousarray(tau_tx, dtype=np.float32)
        w_tx = np.ascontiguousarray(w_tx, dtype=np.float32)
        if tau_tx.ndim != 2 or tau_tx.shape[0] != Q or w_tx.shape != tau_tx.shape:
            raise ValueError("tau_tx / w_tx must both be Q x N")
        N = tau_tx.shape[1]
        rx = np.ascontiguousarray(rx_xyz, dtype=np.float64).reshape(M, 3)
        if idx is None:
            idx = np.arange(N, dtype=np.int64)
        idx = np.ascontiguousarray(idx, dtype=np.int64)
        if vox_xyz is None:
            if grid is None:
                raise ValueError("need grid or vox_xyz")
            vox_xyz = self.voxel_positions(grid, idx)
        vox_xyz = np.ascontiguousarray(vox_xyz, dtype=np.float64).reshape(idx.size, 3)
        n_eval = idx.size
        out = np.zeros((B, n_eval, 2 if is_complex else 1), dtype=np.float64)
        slack = np.zeros((B, n_eval), dtype=np.float64) if want_slack else None
        rc = self._lib.das_oracle_beamform(
            B, Q, M, K, N, rf.ctypes.data_as(ctypes.c_void_p), rf_type,
            _ptr(tau_tx, _F32P), _ptr(w_tx, _F32P), _ptr(rx, _F64P),
            _ptr(vox_xyz, _F64P), _ptr(idx, _I64P), n_eval,
            float(c), float(fs), float(t0), float(fnum), float(f_demod), float(tie_rel),
            _ptr(out, _F64P),
            slack.ctypes.data_as(ctypes.c_void_p) if slack is not None else None,
            int(nthreads))
        if rc != 0:
            raise ValueError("das_oracle_beamform: invalid arguments")
        y = out[..., 0] + 1j * out[..., 1] if is_complex else out[..., 0]
        return (y, slack) if want_slack else y

    # -------------------------------------------------------------- permute
    def permute(self, rf, layout: str = "kqmb") -> np.ndarray:
        """B x Q x M x K -> K x Q x M x B (``kqmb``) or Q x M x K x B (``qmkb``)."""
        rf = np.ascontiguousarray(rf)
        B, Q, M, K = rf.shape
        lay = {"kqmb": 0, "qmkb": 1}[layout]
        shape = (K, Q, M, B) if lay == 0 else (Q, M, K, B)
        out = np.empty(shape, dtype=rf.dtype)
        rc = self._lib.das_oracle_permute(
            rf.ctypes.data_as(ctypes.c_void_p), out.ctypes.data_as(ctypes.c_void_p),
            rf.dtype.itemsize, B, Q, M, K, lay)
        if rc != 0:
            raise ValueError("das_oracle_permute: invalid arguments")
        return out


_DEFAULT: Oracle | None = None


def load() -> Oracle:
    """The oracle built from ``das_oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
