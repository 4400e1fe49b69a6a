"""Records that arrive in half precision (DAS_F16, DAS_C32H).

A half record holds exactly the values FP16 storage holds, so a plan of one of
these dtypes does the arithmetic of a float32 / complex64 plan with half
storage, on a record of half the size: the permute copies the half samples bit
for bit into the padded layout and the brick or BI kernel converts them to
float32 before interpolating.  Checked here: the oracle on the same values at
the usual bar, bit-identity with the float plan with half storage, the host
entry point, the permute, and the kernels that do not read half rows.
"""
import zlib

import numpy as np
import pytest

import oracle as oracle_mod
from parity import TOL, error_ratio
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

CASES = {
    "real": dict(base="full", n_el=8, nx=13, ny=11, nz=6),
    "iq": dict(base="iq", n_el=8, nx=11, ny=9, nz=4),
    "mid16": dict(base="mid", n_el=8, nx=12, ny=10, nz=5),
}


def _problem(name):
    args = dict(CASES[name])
    return synth.make_problem(args.pop("base"), **args)


def _half_record(prob):
    """(float16 view of the record as B x Q x M x K [x 2], the same values as float32 / complex64)"""
    if prob.rf.dtype == np.complex64:
        h = prob.rf.view(np.float32).astype(np.float16).reshape(prob.rf.shape + (2,))
        return h, h.astype(np.float32).reshape(-1).view(np.complex64).reshape(prob.rf.shape)
    h = prob.rf.astype(np.float16)
    return h, h.astype(np.float32)


def _plan(prob, dtype, kernel="auto", storage="native"):
    from volumetric_ultrasound_delay_gb300 import das
    return das.Plan(prob.grid, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, dtype, prob.B, prob.Q,
                    prob.M, prob.K, kernel=kernel, f_demod=prob.f_demod, storage=storage)


def _device_half(h):
    t = torch.from_numpy(np.ascontiguousarray(h)).cuda()
    return torch.view_as_complex(t) if h.ndim == 5 else t


def _run(plan, rf, prob):
    tau = torch.from_numpy(prob.tau_tx).cuda()
    w = torch.from_numpy(prob.w_tx).cuda()
    y = plan.beamform(rf, tau, w)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.fixture(scope="module")
def cases(oracle):
    out = {}
    for name in CASES:
        prob = _problem(name)
        h, same = _half_record(prob)
        ref, slack = oracle.beamform(same, prob.tau_tx, prob.w_tx, prob.rx.astype(np.float64),
                                     oracle_mod.Grid(*prob.grid), c=prob.c, fs=prob.fs, t0=prob.t0,
                                     fnum=prob.fnum, f_demod=prob.f_demod, want_slack=True)
        out[name] = (prob, h, same, ref, slack)
    return out


@pytest.mark.parametrize("kernel", ["auto", "brick", "bi"])
@pytest.mark.parametrize("name", list(CASES))
def test_half_record_matches_oracle(cases, name, kernel):
    prob, h, _, ref, slack = cases[name]
    dtype = "c32h" if prob.rf.dtype == np.complex64 else "f16"
    plan = _plan(prob, dtype, kernel)
    assert plan.kernel == ("brick" if kernel == "auto" else kernel)
    y = _run(plan, _device_half(h), prob)
    plan.close()
    assert y.dtype == (np.complex64 if dtype == "c32h" else np.float32)
    assert error_ratio(y, ref, slack) <= TOL, (name, kernel)


@pytest.mark.parametrize("kernel", ["brick", "bi"])
@pytest.mark.parametrize("name", list(CASES))
def test_half_record_equals_float_record_with_half_storage(cases, name, kernel):
    """The same half values in the rows, the same kernel, the same launches:
    the two plans agree bit for bit."""
    prob, h, same, _, _ = cases[name]
    dtype = "c32h" if prob.rf.dtype == np.complex64 else "f16"
    ph = _plan(prob, dtype, kernel)
    pf = _plan(prob, "c64" if dtype == "c32h" else "f32", kernel, storage="f16")
    assert ph.launches == pf.launches
    y_h = _run(ph, _device_half(h), prob)
    y_f = _run(pf, torch.from_numpy(np.ascontiguousarray(same)).cuda(), prob)
    ph.close()
    pf.close()
    assert np.array_equal(y_h, y_f), (name, kernel)


@pytest.mark.parametrize("groups", [1, 0, 3])
@pytest.mark.parametrize("name", ["real", "iq"])
def test_half_record_host_entry_point(cases, name, groups):
    """das_beamform_host copies half the bytes of the float record and gives the
    device entry point's output bit for bit (the same transmit groups)."""
    from volumetric_ultrasound_delay_gb300 import das
    prob, h, _, _, _ = cases[name]
    dtype = "c32h" if prob.rf.dtype == np.complex64 else "f16"
    plan = _plan(prob, dtype)
    plan.set_option(das.OPT_HOST_GROUPS, groups)
    host = torch.from_numpy(np.ascontiguousarray(h))
    if h.ndim == 5:
        host = torch.view_as_complex(host)
    out = torch.empty((prob.B, prob.N), dtype=torch.complex64 if dtype == "c32h" else torch.float32)
    plan.beamform_host(host.pin_memory(), prob.tau_tx, prob.w_tx, out)
    dev = _plan(prob, dtype)
    dev.set_option(das.OPT_TX_GROUPS, groups if groups > 0 else min(prob.Q, 5))
    y = _run(dev, _device_half(h), prob)
    plan.close()
    dev.close()
    assert np.array_equal(out.numpy(), y), (name, groups)


@pytest.mark.parametrize("layout", [0, 1, 2, 3])
@pytest.mark.parametrize("complex_", [False, True])
def test_half_record_permute_bit_exact(layout, complex_):
    from volumetric_ultrasound_delay_gb300 import das
    shape = (16, 3, 5, 37)
    rng = np.random.default_rng(zlib.crc32(repr((layout, complex_)).encode()))
    B, Q, M, K = shape
    x = (rng.standard_normal(shape + ((2,) if complex_ else ())) * 3).astype(np.float16)
    pad = {2: 3, 3: 2}.get(layout, 0)
    rf = _device_half(x)
    n_out = B * Q * M * (K + pad)
    out = torch.full((n_out * (2 if complex_ else 1),), 7.0, dtype=torch.float16, device="cuda")
    out_t = torch.view_as_complex(out.view(n_out, 2)) if complex_ else out
    das.permute(rf, out_t, layout=layout)
    torch.cuda.synchronize()
    got = out.cpu().numpy().reshape(n_out, -1)
    src = x.reshape(B, Q, M, K, -1)
    if layout == 0:
        want = src.transpose(3, 1, 2, 0, 4)
    elif layout == 1:
        want = src.transpose(1, 2, 3, 0, 4)
    elif layout == 2:
        want = np.full((Q, M, K + 3, B, src.shape[-1]), 7.0, np.float16)
        want[:, :, 1:K + 1] = src.transpose(1, 2, 3, 0, 4)
    else:
        want = np.full((K + 2, Q, M, B, src.shape[-1]), 7.0, np.float16)
        want[1:K + 1] = src.transpose(3, 1, 2, 0, 4)
    assert np.array_equal(got.view(np.uint16), np.ascontiguousarray(want).reshape(n_out, -1).view(np.uint16))


@pytest.mark.parametrize("kernel", ["bl", "window", "pair"])
def test_half_record_rejected_by_float_kernels(cases, kernel):
    from volumetric_ultrasound_delay_gb300 import das
    prob, h, _, _, _ = cases["real"]
    plan = _plan(prob, "f16", kernel)
    with pytest.raises(das.DasError) as exc:
        _run(plan, _device_half(h), prob)
    assert exc.value.status == das.DAS_ERR_UNSUPPORTED
    plan.close()
