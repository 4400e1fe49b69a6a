"""das_beamform_host_volumes: a stream of volumes from host memory.

Volume v + 1's record is copied while volume v's kernels run, so the call must
give, for every volume, exactly what das_beamform_host gives for that volume
alone (the same transmit groups, the same launches): compared bit for bit, for
the kernels that sum transmit ranges (brick, window, pair) and for those that
take the record whole (BI, BL), and against the oracle for one volume.
"""
import numpy as np
import pytest

from parity import TOL, error_ratio, kernel_serves, oracle_beamform, plan_for
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

V = 3


@pytest.fixture(scope="module")
def problems():
    return {"real": synth.make_problem("full", n_el=8, nx=13, ny=11, nz=6),
            "iq": synth.make_problem("iq", n_el=8, nx=11, ny=9, nz=4)}


def _records(prob):
    """V different records of the problem's shape (scaled and sign-flipped copies)."""
    return np.stack([prob.rf * np.float32(v + 1) * np.float32(-1 if v % 2 else 1) for v in range(V)])


def _one_by_one(prob, kernel, recs, groups):
    from volumetric_ultrasound_delay_gb300 import das
    plan = plan_for(prob, kernel)
    plan.set_option(das.OPT_HOST_GROUPS, groups)
    outs = []
    for r in recs:
        out = np.empty((prob.B, prob.N), dtype=prob.rf.dtype)
        plan.beamform_host(np.ascontiguousarray(r), prob.tau_tx, prob.w_tx, out)
        outs.append(out)
    plan.close()
    return np.stack(outs)


def _stream(prob, kernel, recs, groups):
    from volumetric_ultrasound_delay_gb300 import das
    plan = plan_for(prob, kernel)
    plan.set_option(das.OPT_HOST_GROUPS, groups)
    rf = torch.from_numpy(np.ascontiguousarray(recs)).pin_memory()
    out = torch.empty((len(recs), prob.B, prob.N),
                      dtype=torch.complex64 if prob.rf.dtype == np.complex64 else torch.float32).pin_memory()
    plan.beamform_host_volumes(rf, prob.tau_tx, prob.w_tx, out)
    plan.close()
    return out.numpy()


@pytest.mark.parametrize("groups", [0, 1, 3])
@pytest.mark.parametrize("kernel", ["auto", "window", "pair", "bi", "bl"])
@pytest.mark.parametrize("name", ["real", "iq"])
def test_stream_equals_volume_by_volume(problems, name, kernel, groups):
    prob = problems[name]
    if not kernel_serves(kernel, prob):
        pytest.skip(f"the {kernel} kernel does not serve this record")
    recs = _records(prob)
    assert np.array_equal(_stream(prob, kernel, recs, groups), _one_by_one(prob, kernel, recs, groups))


@pytest.mark.parametrize("name", ["real", "iq"])
def test_stream_matches_oracle(oracle, problems, name):
    import copy
    prob = problems[name]
    recs = _records(prob)
    y = _stream(prob, "auto", recs, 0)
    last = copy.copy(prob)
    last.rf = np.ascontiguousarray(recs[-1])
    ref, slack = oracle_beamform(oracle, last)
    assert error_ratio(y[-1], ref, slack) <= TOL


def test_single_volume_equals_host_call(problems):
    prob = problems["real"]
    recs = _records(prob)[:1]
    assert np.array_equal(_stream(prob, "auto", recs, 0), _one_by_one(prob, "auto", recs, 0))


def test_stream_rejects_mismatched_buffers(problems):
    prob = problems["real"]
    plan = plan_for(prob)
    recs = _records(prob)
    with pytest.raises(ValueError):
        plan.beamform_host_volumes(recs, prob.tau_tx, prob.w_tx, np.empty((V - 1, prob.B, prob.N), np.float32))
    with pytest.raises(ValueError):
        plan.beamform_host_volumes(recs.reshape(-1)[:-1].copy(), prob.tau_tx, prob.w_tx,
                                   np.empty((V, prob.B, prob.N), np.float32))
    plan.close()
