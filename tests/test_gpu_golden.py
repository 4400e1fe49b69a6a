"""Every kernel through the C ABI against the hand-worked examples of
tests/golden/ (closed forms of the delay-and-sum definition; every
intermediate value there is exact in float32, and the records are integers
that half precision holds exactly too)."""
import numpy as np
import pytest

import golden_cases

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

TOL = 1e-6   # relative to the peak; the sums are exact in float32 up to summation order

CASES = [(ex["name"], kernel, storage)
         for ex in golden_cases.examples()
         for kernel, storage in [("auto", "native"), ("bl", "native"), ("bi", "native"),
                                 ("brick", "native"), ("window", "native"), ("brick", "f16")]
         if not (kernel == "window" and ex["dtype"] == "c64")]


def _plan(ex, kernel, storage):
    from volumetric_ultrasound_delay_gb300 import das
    _, _, _, rx = golden_cases.inputs(ex)
    return das.Plan(tuple(ex["grid"]), rx, ex["c"], ex["fs"], ex["t0"], ex["fnum"], ex["dtype"],
                    ex["B"], ex["Q"], ex["M"], ex["K"], kernel=kernel, f_demod=ex["f_demod"],
                    storage=storage)


@pytest.mark.parametrize("name,kernel,storage", CASES)
def test_kernel_matches_worked_example(name, kernel, storage):
    ex = {e["name"]: e for e in golden_cases.examples()}[name]
    rf, tau, w, _ = golden_cases.inputs(ex)
    plan = _plan(ex, kernel, storage)
    y = plan.beamform(torch.from_numpy(rf).cuda(), torch.from_numpy(tau).cuda(),
                      torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    plan.close()
    ref = golden_cases.expected(ex)
    err = np.abs(y.cpu().numpy().astype(np.complex128) - ref).max()
    assert err <= TOL * np.abs(ref).max(), (name, kernel, storage, err)


@pytest.mark.parametrize("ex", golden_cases.examples(), ids=lambda e: e["name"])
def test_host_entry_point_matches_worked_example(ex):
    rf, tau, w, _ = golden_cases.inputs(ex)
    plan = _plan(ex, "auto", "native")
    out = torch.empty((ex["B"], 2), dtype=torch.complex64 if ex["dtype"] == "c64" else torch.float32)
    plan.beamform_host(torch.from_numpy(rf), torch.from_numpy(tau), torch.from_numpy(w), out)
    plan.close()
    ref = golden_cases.expected(ex)
    assert np.abs(out.numpy().astype(np.complex128) - ref).max() <= TOL * np.abs(ref).max()
