"""das_beamform_noalloc, the entry point for callers that cannot allocate
device memory (for example a scanner's real-time loop, where cudaMalloc could
stall acquisition, or a framework that owns all device memory): it keeps its
scratch in a static 64 MiB array inside libdas.  Its output must match the
plan-based entry point running the same kernel, on two calls in a row whose
sizes differ (the second call must not see the first call's leftovers).

This file is named so pytest collects it last."""
import numpy as np
import pytest

from parity import TOL, error_ratio, gpu_beamform
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _run_noalloc(prob):
    from volumetric_ultrasound_delay_gb300 import das
    rf = torch.from_numpy(np.ascontiguousarray(prob.rf)).cuda()
    tau = torch.from_numpy(prob.tau_tx).cuda()
    w = torch.from_numpy(prob.w_tx).cuda()
    rx = torch.from_numpy(np.ascontiguousarray(prob.rx)).cuda()
    out = torch.empty((prob.B, prob.N), dtype=rf.dtype, device="cuda")
    das.beamform_noalloc(prob.grid, rx, prob.c, prob.fs, prob.t0, prob.fnum, prob.f_demod,
                         rf, tau, w, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_noalloc_matches_plan_on_two_calls_in_a_row():
    first = synth.make_problem("iq", n_el=8, nx=11, ny=9, nz=4, B=16, K=256)   # 19 MB scratch
    second = synth.make_problem("tiny")                                        # 3.2 MB scratch
    for prob in (first, second):
        y = _run_noalloc(prob)
        ref, used = gpu_beamform(prob, "brick")
        assert used == "brick"
        assert np.all(np.isfinite(y))
        assert error_ratio(y, ref) <= TOL


def test_noalloc_rejects_requests_beyond_its_scratch():
    from volumetric_ultrasound_delay_gb300 import das
    prob = synth.make_problem("tiny", K=4096, B=32)    # 32*3*64*4099*4 bytes > 64 MiB
    with pytest.raises(das.DasError) as exc:
        _run_noalloc(prob)
    assert exc.value.status == das.DAS_ERR_INVALID_ARG
    assert "scratch" in str(exc.value)
