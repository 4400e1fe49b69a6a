"""Plan lifecycle on the GPU: das_plan_destroy waits for no stream.

A plan's device memory is freed in stream order after the plan's own last
queued work, so destroying a plan neither blocks on another plan's stream nor
cuts short the plan's own queued work."""
import numpy as np
import pytest

from parity import TOL, error_ratio, oracle_beamform, plan_for
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)


def _busy_plan():
    """A plan over the 32 x 32-array geometry (8 depth slices) with a random
    record on the device: about 2 ms of kernels per call."""
    prob = synth.make_problem("full", nx=64, ny=64, nz=8, noise=False, echoes=False)
    plan = plan_for(prob)
    g = torch.Generator(device="cuda").manual_seed(5)
    rf = torch.randn((prob.B, prob.Q, prob.M, prob.K), device="cuda", generator=g)
    tau = torch.from_numpy(prob.tau_tx).cuda()
    w = torch.from_numpy(prob.w_tx).cuda()
    out = torch.empty((prob.B, prob.N), device="cuda")
    plan.beamform(rf, tau, w, out)          # allocates the scratch, loads the kernels
    torch.cuda.synchronize()
    return plan, (rf, tau, w, out)


def test_destroy_does_not_wait_for_another_plans_stream():
    busy, args = _busy_plan()
    prob = synth.make_problem("tiny")
    idle = plan_for(prob)
    y = idle.beamform(*[torch.from_numpy(np.ascontiguousarray(a)).cuda()
                        for a in (prob.rf, prob.tau_tx, prob.w_tx)])
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    for _ in range(40):
        busy.beamform(*args, stream=s)
    idle.close()
    still_running = not s.query()
    torch.cuda.synchronize()
    busy.close()
    assert still_running, "das_plan_destroy waited for another plan's stream"
    assert y.shape == (prob.B, prob.N)


def test_destroy_with_own_work_queued_completes_that_work(oracle):
    busy, args = _busy_plan()
    prob = synth.make_problem("tiny")
    inputs = [torch.from_numpy(np.ascontiguousarray(a)).cuda()
              for a in (prob.rf, prob.tau_tx, prob.w_tx)]
    s = torch.cuda.Stream()
    for _ in range(20):
        busy.beamform(*args, stream=s)     # keeps the stream busy for ~40 ms
    victim = plan_for(prob)
    y = victim.beamform(*inputs, stream=s)  # queued behind the busy plan's calls
    victim.close()                          # returns at once; memory freed after the call
    queued = not s.query()
    # a new plan on another stream may now be handed the memory the pool got back
    other = plan_for(prob)
    s2 = torch.cuda.Stream()
    y2 = other.beamform(*inputs, stream=s2)
    torch.cuda.synchronize()
    other.close()
    busy.close()
    assert queued
    ref, slack = oracle_beamform(oracle, prob)
    assert error_ratio(y.cpu().numpy(), ref, slack) <= TOL
    assert error_ratio(y2.cpu().numpy(), ref, slack) <= TOL
