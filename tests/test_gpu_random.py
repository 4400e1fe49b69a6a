"""Every kernel through the C ABI against the float64 oracle on seeded random
small problems (random geometry with receivers on both sides of the voxels,
delays off both record ends, t0 of either sign, aperture on or off, real and IQ
records, 1 to 64 frames), element by element under the parity bar."""
import numpy as np
import pytest

from parity import TOL, error_ratio
from random_cases import make_case

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

CASES = 24
KERNELS = ["auto", "bl", "bi", "brick", "window", "pair"]


def _case(seed):
    return make_case(seed, frames=(1, 2, 4, 8, 16, 32, 64), max_k=64, max_m=40, max_q=4, max_side=6)


@pytest.mark.parametrize("seed", range(CASES))
def test_kernels_match_oracle_on_random_problem(oracle, seed):
    from volumetric_ultrasound_delay_gb300 import das
    grid, rx, rf, tau, w, kw = _case(seed)
    ref, slack = oracle.beamform(rf, tau, w, rx.astype(np.float64), grid, want_slack=True, **kw)
    B, Q, M, K = rf.shape
    dtype = "c64" if np.iscomplexobj(rf) else "f32"
    inputs = [torch.from_numpy(a).cuda() for a in (rf, tau, w)]
    served = []
    for kernel in KERNELS:
        plan = das.Plan((grid.nx, grid.ny, grid.nz, grid.x0, grid.y0, grid.z0, grid.dx, grid.dy, grid.dz),
                        rx, kw["c"], kw["fs"], kw["t0"], kw["fnum"], dtype, B, Q, M, K, kernel=kernel,
                        f_demod=kw["f_demod"])
        try:
            y = plan.beamform(*inputs)
        except das.DasError as exc:
            assert exc.status == das.DAS_ERR_UNSUPPORTED and kernel in ("bi", "brick", "window", "pair"), \
                (seed, kernel, exc)
            plan.close()
            continue
        torch.cuda.synchronize()
        plan.close()
        served.append(kernel)
        err = error_ratio(y.cpu().numpy(), ref, slack)
        assert err <= TOL, (seed, kernel, B, dtype, err)
    assert {"auto", "bl"} <= set(served)


def test_random_problems_exercise_every_kernel():
    """Across the seeds each kernel serves several problems (so the random
    cases reach BI, brick and window, not only the baseline)."""
    from volumetric_ultrasound_delay_gb300 import das
    counts = dict.fromkeys(KERNELS[2:], 0)
    for seed in range(CASES):
        grid, rx, rf, tau, w, kw = _case(seed)
        B, Q, M, K = rf.shape
        dtype = "c64" if np.iscomplexobj(rf) else "f32"
        inputs = [torch.from_numpy(a).cuda() for a in (rf, tau, w)]
        for kernel in counts:
            plan = das.Plan((grid.nx, grid.ny, grid.nz, grid.x0, grid.y0, grid.z0, grid.dx, grid.dy,
                             grid.dz), rx, kw["c"], kw["fs"], kw["t0"], kw["fnum"], dtype, B, Q, M, K,
                            kernel=kernel, f_demod=kw["f_demod"])
            try:
                plan.beamform(*inputs)
                counts[kernel] += 1
            except das.DasError:
                pass
            plan.close()
    assert min(counts.values()) >= 3, counts
