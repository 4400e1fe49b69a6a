"""A second, independent float64 statement of delay-and-sum, in pure Python.

Used only to pin the C oracle on tiny inputs.  It is written from the formula,
not from the oracle, and deliberately uses different formulations:

* linear interpolation as a sum over every sample of the record weighted by
  the hat function max(0, 1 - |f - k|) (the oracle uses floor / fraction);
* the F-number aperture as a ratio test rho / dz <= 1 / (2 F#) (the oracle
  compares squares);
* the demodulation phase through ``cmath.exp``;
* exact summation with ``math.fsum`` per output.

Samples outside the record simply never appear in the hat sum, which is the
"count as zero" rule.
"""
from __future__ import annotations

import cmath
import math

import numpy as np


def in_aperture(dx: float, dy: float, dz: float, fnum: float) -> bool:
    if fnum <= 0.0:
        return True
    if dz <= 0.0:
        return False
    return math.hypot(dx, dy) / dz <= 1.0 / (2.0 * fnum)


def das_bruteforce(rf, tau_tx, w_tx, rx, vox, c, fs, t0=0.0, fnum=0.0, f_demod=0.0):
    """y[b, e] for voxel positions ``vox`` (E x 3); tau_tx / w_tx are Q x E here."""
    rf = np.asarray(rf)
    B, Q, M, K = rf.shape
    is_complex = np.iscomplexobj(rf)
    E = len(vox)
    y = np.zeros((B, E), dtype=np.complex128 if is_complex else np.float64)
    for e in range(E):
        px, py, pz = (float(v) for v in vox[e])
        terms = [[] for _ in range(B)]
        terms_im = [[] for _ in range(B)]
        for q in range(Q):
            for m in range(M):
                dx, dy, dz = px - float(rx[m][0]), py - float(rx[m][1]), pz - float(rx[m][2])
                if not in_aperture(dx, dy, dz, fnum):
                    continue
                tau = float(tau_tx[q][e]) + math.sqrt(dx * dx + dy * dy + dz * dz) / c
                f = (tau - t0) * fs
                rot = cmath.exp(2j * math.pi * f_demod * tau) if is_complex else 1.0
                wt = float(w_tx[q][e])
                for k in range(K):
                    h = 1.0 - abs(f - k)
                    if h <= 0.0:
                        continue
                    for b in range(B):
                        v = complex(rf[b, q, m, k]) if is_complex else float(rf[b, q, m, k])
                        t = wt * h * v * rot
                        if is_complex:
                            terms[b].append(t.real)
                            terms_im[b].append(t.imag)
                        else:
                            terms[b].append(t)
        for b in range(B):
            if is_complex:
                y[b, e] = complex(math.fsum(terms[b]), math.fsum(terms_im[b]))
            else:
                y[b, e] = math.fsum(terms[b])
    return y
