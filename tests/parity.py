"""Helpers shared by the GPU parity tests: run a problem through the C ABI and
through the oracle, and measure the difference against the oracle's peak."""
from __future__ import annotations

import numpy as np

import oracle as oracle_mod

TOL = 1e-4   # max |y_gpu - y_oracle| (less the aperture-tie slack) / max |y_oracle|


DTYPE_NAMES = {np.dtype(np.float32): "f32", np.dtype(np.complex64): "c64",
               np.dtype(np.float64): "f64", np.dtype(np.complex128): "c128"}


def kernel_serves(kernel, prob) -> bool:
    """Whether a kernel with a restricted scope serves a problem's record: the
    window kernel takes float32 records of 8, 16 or 32 frames, the pair kernel
    float32 records of 16, 32 or 64 frames (the others serve, or reject, more
    general shapes themselves)."""
    if kernel == "window":
        return prob.rf.dtype == np.float32 and prob.B in (8, 16, 32)
    if kernel == "pair":
        return prob.rf.dtype == np.float32 and prob.B in (16, 32, 64)
    return True


def plan_for(prob, kernel="auto"):
    from volumetric_ultrasound_delay_gb300 import das
    dtype = DTYPE_NAMES[prob.rf.dtype]
    return das.Plan(prob.grid, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, dtype,
                    prob.B, prob.Q, prob.M, prob.K, kernel=kernel, f_demod=prob.f_demod)


def device_inputs(prob):
    import torch
    return (torch.from_numpy(np.ascontiguousarray(prob.rf)).cuda(),
            torch.from_numpy(prob.tau_tx).cuda(), torch.from_numpy(prob.w_tx).cuda())


def gpu_beamform(prob, kernel="auto", inputs=None):
    import torch
    plan = plan_for(prob, kernel)
    rf, tau, w = inputs if inputs is not None else device_inputs(prob)
    y = plan.beamform(rf, tau, w)
    torch.cuda.synchronize()
    used = plan.kernel
    plan.close()
    return y.cpu().numpy(), used


def oracle_beamform(orc, prob, idx=None):
    return orc.beamform(prob.rf, prob.tau_tx, prob.w_tx, prob.rx.astype(np.float64),
                        oracle_mod.Grid(*prob.grid), idx=idx, c=prob.c, fs=prob.fs, t0=prob.t0,
                        fnum=prob.fnum, f_demod=prob.f_demod, want_slack=True)


def error_ratio(y_gpu, y_ref, slack=None):
    err = np.abs(np.asarray(y_gpu, dtype=np.complex128) - y_ref)
    if slack is not None:
        err = np.maximum(err - slack, 0.0)
    peak = float(np.abs(y_ref).max())
    return float(err.max()) / peak if peak > 0 else float(err.max())
