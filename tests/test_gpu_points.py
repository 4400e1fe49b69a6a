"""Plans over an explicit voxel list (das_plan_create_points): every kernel
against the oracle evaluated at the same positions, and against a grid plan at
the voxels the list was drawn from."""
import numpy as np
import pytest

from parity import TOL, error_ratio
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

KERNELS = ["bl", "bi", "brick", "window", "pair"]


def run_points(prob, pts, tau, w, kernel):
    from volumetric_ultrasound_delay_gb300 import das
    dtype = "c64" if prob.rf.dtype == np.complex64 else "f32"
    plan = das.Plan(None, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, dtype, prob.B, prob.Q,
                    prob.M, prob.K, kernel=kernel, f_demod=prob.f_demod, points=pts)
    assert plan.N == len(pts) and plan.kernel == kernel
    y = plan.beamform(torch.from_numpy(np.ascontiguousarray(prob.rf)).cuda(),
                      torch.from_numpy(np.ascontiguousarray(tau)).cuda(),
                      torch.from_numpy(np.ascontiguousarray(w)).cuda())
    torch.cuda.synchronize()
    plan.close()
    return y.cpu().numpy()


def oracle_points(oracle, prob, pts, tau, w):
    return oracle.beamform(prob.rf, tau, w, prob.rx.astype(np.float64),
                           vox_xyz=pts.astype(np.float64), idx=np.arange(len(pts)), c=prob.c,
                           fs=prob.fs, t0=prob.t0, fnum=prob.fnum, f_demod=prob.f_demod,
                           want_slack=True)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("base", ["full", "iq"])
def test_sampled_grid_voxels_as_a_list(oracle, base, kernel):
    if kernel in ("window", "pair") and base == "iq":
        pytest.skip("the window and pair kernels serve float32 records only")
    prob = synth.make_problem(base, n_el=8, nx=19, ny=13, nz=5)
    rng = np.random.default_rng(21)
    idx = rng.choice(prob.N, 333, replace=False)            # shuffled: no spatial order
    pts = synth.grid_points(prob.grid, idx).astype(np.float32)
    tau, w = prob.tau_tx[:, idx], prob.w_tx[:, idx]
    y = run_points(prob, pts, tau, w, kernel)
    ref, slack = oracle_points(oracle, prob, pts, tau, w)
    assert error_ratio(y, ref, slack) <= TOL
    # the same voxels through a grid plan
    from parity import gpu_beamform
    y_grid, _ = gpu_beamform(prob, kernel)
    assert np.abs(y - y_grid[:, idx]).max() <= TOL * np.abs(y_grid).max()


@pytest.mark.parametrize("kernel", KERNELS)
def test_list_order_does_not_change_the_result(kernel):
    """The plan keeps a list in its own compact order; permuting the caller's
    list permutes y and nothing else: bit for bit where each voxel's sum runs
    in the same order wherever it lands (BL, BI, brick), to float32 rounding
    for the window kernel (its passes run over the receivers active for the
    warp's voxels, so the order of the terms depends on the neighbours)."""
    prob = synth.make_problem("full", n_el=8, nx=19, ny=13, nz=5)
    rng = np.random.default_rng(24)
    idx = rng.choice(prob.N, 400, replace=False)
    perm = rng.permutation(len(idx))
    runs = []
    for sel in (idx, idx[perm]):
        pts = synth.grid_points(prob.grid, sel).astype(np.float32)
        runs.append(run_points(prob, pts, prob.tau_tx[:, sel], prob.w_tx[:, sel], kernel))
    if kernel == "window":
        assert np.abs(runs[0][:, perm] - runs[1]).max() <= 1e-5 * np.abs(runs[1]).max()
    else:
        assert np.array_equal(runs[0][:, perm], runs[1])


@pytest.mark.parametrize("kernel", KERNELS)
def test_degenerate_lists(oracle, kernel):
    """Lists the ordering cannot spread out: one point, repeated points, a
    flat sheet (one depth), a line."""
    prob = synth.make_problem("mid", n_el=8, nx=4, ny=4, nz=4, B=16)
    wl = prob.wl
    rng = np.random.default_rng(25)
    sheet = np.column_stack([rng.uniform(-2e-3, 2e-3, 70), rng.uniform(-2e-3, 2e-3, 70),
                             np.full(70, 12e-3)])
    line = np.column_stack([np.zeros(37), np.zeros(37), np.linspace(5e-3, 25e-3, 37)])
    cases = {"one": np.array([[0.0, 0.0, 10e-3]]), "repeated": np.tile([[1e-3, -1e-3, 15e-3]], (33, 1)),
             "sheet": sheet, "line": line}
    for name, pts in cases.items():
        pts = pts.astype(np.float32)
        tau = synth.transmit_delays(wl, pts.astype(np.float64)).astype(np.float32)
        w = rng.uniform(0.5, 1.0, (wl.Q, len(pts))).astype(np.float32)
        y = run_points(prob, pts, tau, w, kernel)
        ref, slack = oracle_points(oracle, prob, pts, tau, w)
        assert error_ratio(y, ref, slack) <= TOL, (name, kernel)


def test_list_through_the_grid_struct_matches_points_plan():
    """das_plan_create with grid.xyz set builds the same plan as
    das_plan_create_points: identical output, bit for bit."""
    from volumetric_ultrasound_delay_gb300 import das
    prob = synth.make_problem("full", n_el=8, nx=19, ny=13, nz=5)
    rng = np.random.default_rng(23)
    idx = rng.choice(prob.N, 240, replace=False)
    pts = synth.grid_points(prob.grid, idx).astype(np.float32)
    tau, w = prob.tau_tx[:, idx], prob.w_tx[:, idx]
    ys = []
    for grid in (None, (4, 6, 10, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0)):
        plan = das.Plan(grid, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, "f32", prob.B, prob.Q,
                        prob.M, prob.K, points=pts)
        assert plan.N == len(pts)
        y = plan.beamform(torch.from_numpy(np.ascontiguousarray(prob.rf)).cuda(),
                          torch.from_numpy(np.ascontiguousarray(tau)).cuda(),
                          torch.from_numpy(np.ascontiguousarray(w)).cuda())
        torch.cuda.synchronize()
        ys.append(y.cpu().numpy())
        plan.close()
    assert np.array_equal(ys[0], ys[1])


@pytest.mark.parametrize("kernel", KERNELS)
def test_random_point_cloud(oracle, kernel):
    prob = synth.make_problem("mid", n_el=8, nx=4, ny=4, nz=4, B=16)
    rng = np.random.default_rng(22)
    n = 517                                                  # not a multiple of any brick
    pts = np.column_stack([rng.uniform(-3e-3, 3e-3, n), rng.uniform(-3e-3, 3e-3, n),
                           rng.uniform(4e-3, 30e-3, n)]).astype(np.float32)
    wl = prob.wl
    tau = synth.transmit_delays(wl, pts.astype(np.float64)).astype(np.float32)
    w = rng.uniform(0.5, 1.0, (wl.Q, n)).astype(np.float32)
    y = run_points(prob, pts, tau, w, kernel)
    ref, slack = oracle_points(oracle, prob, pts, tau, w)
    assert error_ratio(y, ref, slack) <= TOL
