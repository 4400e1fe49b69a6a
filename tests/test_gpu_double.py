"""float64 / complex128 plans (BL kernel in double precision, the pages' ALG1
data types).  The record carries a perturbation below float32 resolution, so
only a double-precision path reproduces the oracle to 1e-9 of the peak."""
import copy

import numpy as np
import pytest

from parity import device_inputs, error_ratio, gpu_beamform, oracle_beamform, plan_for
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

TOL64 = 1e-9


def as_double(prob, seed=0):
    p = copy.copy(prob)
    rng = np.random.default_rng(seed)
    if prob.rf.dtype == np.complex64:
        p.rf = prob.rf.astype(np.complex128) + 1e-9 * (rng.standard_normal(prob.rf.shape)
                                                       + 1j * rng.standard_normal(prob.rf.shape))
    else:
        p.rf = prob.rf.astype(np.float64) + 1e-9 * rng.standard_normal(prob.rf.shape)
    return p


CASES = {
    "tiny": dict(base="tiny"),
    "full_s": dict(base="full", n_el=8, nx=11, ny=9, nz=4),
    "iq_s": dict(base="iq", n_el=8, nx=11, ny=9, nz=4, B=5),
    "B1": dict(base="tiny", B=1, nx=8, ny=8, nz=4),
    "iq_B1": dict(base="iq", n_el=8, nx=7, ny=5, nz=3, B=1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_double_plan_matches_oracle(oracle, name):
    kw = dict(CASES[name])
    prob = as_double(synth.make_problem(kw.pop("base"), **kw))
    y, used = gpu_beamform(prob)
    assert used == "bl" and y.dtype in (np.float64, np.complex128)
    ref, slack = oracle_beamform(oracle, prob)
    assert error_ratio(y, ref, slack) <= TOL64


def test_double_voxel_list(oracle):
    from volumetric_ultrasound_delay_gb300 import das
    prob = as_double(synth.make_problem("full", n_el=8, nx=9, ny=7, nz=3))
    idx = np.random.default_rng(3).choice(prob.N, 100, replace=False)
    pts = synth.grid_points(prob.grid, idx).astype(np.float32)
    tau, w = np.ascontiguousarray(prob.tau_tx[:, idx]), np.ascontiguousarray(prob.w_tx[:, idx])
    plan = das.Plan(None, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, "f64", prob.B, prob.Q,
                    prob.M, prob.K, points=pts)
    y = plan.beamform(torch.from_numpy(prob.rf).cuda(), torch.from_numpy(tau).cuda(),
                      torch.from_numpy(w).cuda()).cpu().numpy()
    plan.close()
    ref, slack = oracle.beamform(prob.rf, tau, w, prob.rx.astype(np.float64),
                                 vox_xyz=pts.astype(np.float64), idx=np.arange(len(idx)), c=prob.c,
                                 fs=prob.fs, fnum=prob.fnum, want_slack=True)
    assert error_ratio(y, ref, slack) <= TOL64


def test_double_host_path_and_rejections(oracle):
    from volumetric_ultrasound_delay_gb300 import das
    prob = as_double(synth.make_problem("tiny", nx=8, ny=8, nz=4))
    plan = plan_for(prob)
    out = np.empty((prob.B, prob.N), dtype=np.float64)
    plan.beamform_host(np.ascontiguousarray(prob.rf), prob.tau_tx, prob.w_tx, out)
    ref, slack = oracle_beamform(oracle, prob)
    assert error_ratio(out, ref, slack) <= TOL64
    for kernel in ("bi", "brick", "window"):
        plan.kernel = kernel
        with pytest.raises(das.DasError) as exc:
            plan.beamform(*device_inputs(prob))
        assert exc.value.status == das.DAS_ERR_UNSUPPORTED
    plan.close()
