"""das_beamform_noalloc, the entry point for callers that cannot allocate
device memory (for example a scanner's real-time loop, where cudaMalloc could
stall acquisition, or a framework that owns all device memory): it keeps its
scratch in a static 64 MiB array inside libdas.  Its output must match the
float64 oracle and the plan-based entry point running the same kernel, on two
calls in a row whose sizes differ (the second call must not see the first
call's leftovers), and on a request that fills the array almost to the byte.

This file is named so pytest collects it last."""
import numpy as np
import pytest

from parity import TOL, error_ratio, gpu_beamform, oracle_beamform
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

SCRATCH = 64 << 20


def _scratch_bytes(prob):
    elem = 8 if np.iscomplexobj(prob.rf) else 4
    return -(-16 * prob.M // 256) * 256 + prob.B * prob.Q * prob.M * (prob.K + 3) * elem


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


def _check(oracle, prob):
    y = _run_noalloc(prob)
    assert np.all(np.isfinite(y))
    ref, slack = oracle_beamform(oracle, prob)
    assert error_ratio(y, ref, slack) <= TOL
    plan_y, used = gpu_beamform(prob, "brick")
    assert used == "brick"
    assert error_ratio(y, plan_y) <= TOL


def test_noalloc_matches_oracle_and_plan_on_two_calls_in_a_row(oracle):
    first = synth.make_problem("iq", n_el=8, nx=11, ny=9, nz=4, B=16, K=256)   # 19 MB scratch
    second = synth.make_problem("tiny")                                        # 3.2 MB scratch
    for prob in (first, second):
        _check(oracle, prob)


def test_noalloc_request_that_nearly_fills_the_scratch(oracle):
    # 32 frames, 1 transmit, 64 receivers, 8188 samples: 1 KiB of receivers plus
    # 67,100,672 bytes of padded record, 7 KiB short of the 64 MiB array
    prob = synth.make_problem("tiny", K=8188, B=32, angles_x_deg=(0.0,), n_scat=2)
    assert SCRATCH - 8192 < _scratch_bytes(prob) <= SCRATCH
    _check(oracle, prob)


def test_noalloc_rejects_requests_beyond_its_scratch():
    from volumetric_ultrasound_delay_gb300 import das
    # two samples more than the case above: 9,216 bytes over the array
    prob = synth.make_problem("tiny", K=8190, B=32, angles_x_deg=(0.0,), n_scat=2)
    assert _scratch_bytes(prob) > SCRATCH
    with pytest.raises(das.DasError) as exc:
        _run_noalloc(prob)
    assert exc.value.status == das.DAS_ERR_INVALID_ARG
    assert "scratch" in str(exc.value)
