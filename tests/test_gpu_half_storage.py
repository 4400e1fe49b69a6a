"""Half-precision storage of the permuted record (DAS_STORAGE_F16).

The permute rounds every float32 sample (complex: each component) to float16,
and the brick and BI kernels convert back to float32 before interpolating.  So
a kernel computes DAS of the half-rounded record exactly as well as it computes
DAS of a float32 record: the oracle, fed that same rounded record, is held to
the usual 1e-4-of-peak bar.  The rounding itself is checked bit for bit
against numpy's float16 conversion (round to nearest even).
"""
import zlib

import numpy as np
import pytest

from parity import TOL, device_inputs, error_ratio, oracle_beamform, plan_for
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)


def half_rounded(prob):
    """The problem with its record replaced by the float16-rounded record."""
    import copy
    rounded = copy.copy(prob)
    if prob.rf.dtype == np.complex64:
        parts = prob.rf.view(np.float32).astype(np.float16).astype(np.float32)
        rounded.rf = parts.view(np.complex64)
    else:
        rounded.rf = prob.rf.astype(np.float16).astype(np.float32)
    return rounded


def run_half(prob, host=False, groups=0, kernel="auto"):
    from volumetric_ultrasound_delay_gb300 import das
    plan = plan_for(prob, kernel)
    plan.set_option(das.OPT_STORAGE, das.STORAGE_F16)
    assert plan.kernel == ("brick" if kernel == "auto" else kernel)
    if host:
        plan.set_option(das.OPT_HOST_GROUPS, groups)
        out = np.empty((prob.B, prob.N), dtype=prob.rf.dtype)
        plan.beamform_host(np.ascontiguousarray(prob.rf), prob.tau_tx, prob.w_tx, out)
        plan.close()
        return out
    y = plan.beamform(*device_inputs(prob))
    torch.cuda.synchronize()
    plan.close()
    return y.cpu().numpy()


@pytest.mark.parametrize("shape", [(32, 3, 5, 64), (16, 2, 3, 37), (8, 1, 4, 100), (64, 2, 2, 33)])
@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_half_permute_rounds_like_numpy(shape, dtype):
    from volumetric_ultrasound_delay_gb300 import das
    rng = np.random.default_rng(zlib.crc32(repr((shape, dtype)).encode()))
    B, Q, M, K = shape
    x = (rng.standard_normal(shape) * 3).astype(np.float32)
    if dtype == "c64":
        x = (x + 1j * (rng.standard_normal(shape) * 3)).astype(np.complex64)
    comps = 2 if dtype == "c64" else 1
    dst = torch.full((Q * M * (K + 3) * B * comps,), 7.5, dtype=torch.float16, device="cuda")
    das.permute(torch.from_numpy(x).cuda(), dst, 2, storage="f16")
    torch.cuda.synchronize()
    got = dst.cpu().numpy().reshape(Q, M, K + 3, B * comps)
    want = np.ascontiguousarray(x.transpose(1, 2, 3, 0))
    want = (want.view(np.float32) if dtype == "c64" else want).astype(np.float16).reshape(Q, M, K, B * comps)
    assert got[:, :, 1:K + 1].tobytes() == want.tobytes()
    assert np.all(got[:, :, 0] == 7.5) and np.all(got[:, :, K + 1:] == 7.5)


SMALL = {
    "tiny": dict(base="tiny"),
    "mid_s": dict(base="mid", n_el=8, nx=17, ny=9, nz=6),
    "full_s": dict(base="full", n_el=8, nx=19, ny=13, nz=5),
    "iq_s": dict(base="iq", n_el=8, nx=11, ny=9, nz=4),
    "large_s": dict(base="large", n_el=8, nx=13, ny=11, nz=3),
    "iq_B16": dict(base="iq", n_el=8, nx=9, ny=7, nz=3, B=16),
    "f32_B64": dict(base="full", n_el=8, nx=9, ny=7, nz=3, B=64, K=1024),
}


@pytest.mark.parametrize("kernel", ["auto", "bi"])
@pytest.mark.parametrize("name", list(SMALL))
def test_half_storage_matches_oracle_on_rounded_record(oracle, name, kernel):
    kw = dict(SMALL[name])
    prob = synth.make_problem(kw.pop("base"), **kw)
    if kernel == "bi" and name == "tiny":
        pytest.skip("8 half frames fill one 16-byte chunk: BI needs two per voxel")
    y = run_half(prob, kernel=kernel)
    ref, slack = oracle_beamform(oracle, half_rounded(prob))
    assert error_ratio(y, ref, slack) <= TOL
    # and it stays close to DAS of the float32 record (half rounding ~5e-4 per sample)
    ref32, slack32 = oracle_beamform(oracle, prob)
    assert error_ratio(y, ref32, slack32) <= 1e-3


def test_half_storage_host_path_streams(oracle):
    prob = synth.make_problem("full", n_el=8, nx=19, ny=13, nz=5)
    ref, slack = oracle_beamform(oracle, half_rounded(prob))
    for groups in (1, 3):
        y = run_half(prob, host=True, groups=groups)
        assert error_ratio(y, ref, slack) <= TOL


@pytest.mark.parametrize("kernel", ["auto", "bi"])
def test_half_storage_full_size_sampled(oracle, kernel):
    prob = synth.make_problem("full")
    idx = synth.sample_voxels(prob.N, 512, seed=prob.wl.seed)
    y = run_half(prob, kernel=kernel)
    ref, slack = oracle_beamform(oracle, half_rounded(prob), idx=idx)
    assert error_ratio(y[:, idx], ref, slack) <= TOL


def test_half_storage_rejections():
    from volumetric_ultrasound_delay_gb300 import das
    prob = synth.make_problem("tiny", B=4)           # 8-byte half rows
    plan = plan_for(prob)
    plan.set_option(das.OPT_STORAGE, das.STORAGE_F16)
    with pytest.raises(das.DasError) as exc:
        plan.beamform(*device_inputs(prob))
    assert exc.value.status == das.DAS_ERR_UNSUPPORTED
    for kernel in ("bi", "bl", "window", "pair"):
        plan.set_option(das.OPT_KERNEL, das.KERNELS[kernel])
        with pytest.raises(das.DasError) as exc:
            plan.beamform(*device_inputs(prob))
        assert exc.value.status == das.DAS_ERR_UNSUPPORTED
    plan.close()
