"""GPU parity: every kernel through the C ABI against the float64 oracle.

Bars: the permute is bit-exact; beamformed output satisfies
max(|y_gpu - y_oracle| - slack) <= 1e-4 * max|y_oracle| (slack: aperture-tie
pairs the oracle flags, usually none).  Small cases are compared element by
element on every voxel; the full-size workloads run in the bench's launch
configuration and are compared on seeded voxel samples.
"""
import zlib

import numpy as np
import pytest

from parity import TOL, device_inputs, error_ratio, gpu_beamform, kernel_serves, oracle_beamform, plan_for
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

KERNELS = ["bl", "bi", "brick", "window", "pair"]
RESTRICTED = ("bi", "brick", "window", "pair")     # may reject a record shape

# Workloads shrunk (8x8 array, small ragged grids) so the oracle finishes in a
# second or two; B, Q, K, dtype and transmit geometry are those of each workload.
SMALL = {
    "tiny": dict(),
    "mid_s": dict(base="mid", n_el=8, nx=17, ny=9, nz=6),
    "full_s": dict(base="full", n_el=8, nx=19, ny=13, nz=5),
    "iq_s": dict(base="iq", n_el=8, nx=11, ny=9, nz=4),
    "large_s": dict(base="large", n_el=8, nx=13, ny=11, nz=3),
}


def small_problem(name):
    kw = dict(SMALL[name])
    base = kw.pop("base", name)
    return synth.make_problem(base, **kw)


@pytest.fixture(scope="module")
def small_problems():
    return {k: small_problem(k) for k in SMALL}


# ------------------------------------------------------------------ permute
@pytest.mark.parametrize("shape", [(32, 9, 16, 2048), (16, 3, 7, 100), (3, 2, 5, 37),
                                   (1, 1, 1, 1), (5, 1, 3, 64), (40, 2, 3, 33)])
@pytest.mark.parametrize("dtype", ["f32", "c64"])
@pytest.mark.parametrize("layout", [0, 1, 2, 3])
def test_permute_bit_exact(oracle, shape, dtype, layout):
    from volumetric_ultrasound_delay_gb300 import das
    rng = np.random.default_rng(zlib.crc32(repr((shape, dtype, layout)).encode()))
    if dtype == "c64":
        x = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    else:
        x = rng.standard_normal(shape).astype(np.float32)
    src = torch.from_numpy(x).cuda()
    B, Q, M, K = shape
    if layout == 2:
        # padded slabs: data rows 1..K of each (q, m) slab, pad rows left as they were
        dst = torch.full((Q * M * (K + 3) * B,), 7.5, dtype=src.dtype, device="cuda")
        das.permute(src, dst, layout)
        torch.cuda.synchronize()
        got = dst.cpu().numpy().reshape(Q, M, K + 3, B)
        want = oracle.permute(x, "qmkb")
        assert got[:, :, 1:K + 1].tobytes() == want.tobytes()
        pads = np.concatenate([got[:, :, :1], got[:, :, K + 1:]], axis=2)
        assert np.all(pads == np.asarray(7.5, dtype=x.dtype))
        return
    if layout == 3:
        # padded planes: data planes 1..K, planes 0 and K + 1 left as they were
        dst = torch.full(((K + 2) * Q * M * B,), 7.5, dtype=src.dtype, device="cuda")
        das.permute(src, dst, layout)
        torch.cuda.synchronize()
        got = dst.cpu().numpy().reshape(K + 2, Q, M, B)
        assert got[1:K + 1].tobytes() == oracle.permute(x, "kqmb").tobytes()
        assert np.all(got[0] == np.asarray(7.5, dtype=x.dtype))
        assert np.all(got[K + 1] == np.asarray(7.5, dtype=x.dtype))
        return
    dst = torch.empty_like(src).reshape(-1)
    das.permute(src, dst, layout)
    torch.cuda.synchronize()
    want = oracle.permute(x, "kqmb" if layout == 0 else "qmkb")
    assert dst.cpu().numpy().tobytes() == want.tobytes()


@pytest.mark.parametrize("dtype", ["f32", "c64"])
def test_batch_inner_permute_entry_point(oracle, dtype):
    """das_permute_bqmk_to_kqmb: the pages' K x Q x M x B layout, bit for bit."""
    from volumetric_ultrasound_delay_gb300 import das
    rng = np.random.default_rng(31)
    shape = (24, 3, 7, 130)
    if dtype == "c64":
        x = (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)
    else:
        x = rng.standard_normal(shape).astype(np.float32)
    src = torch.from_numpy(x).cuda()
    dst = torch.empty_like(src).reshape(-1)
    das.permute_bqmk_to_kqmb(src, dst)
    torch.cuda.synchronize()
    assert dst.cpu().numpy().tobytes() == oracle.permute(x, "kqmb").tobytes()


# ------------------------------------------------- small workloads, all voxels
@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", list(SMALL))
def test_small_workload_all_voxels(oracle, small_problems, name, kernel):
    from volumetric_ultrasound_delay_gb300 import das
    prob = small_problems[name]
    if not kernel_serves(kernel, prob):
        with pytest.raises(das.DasError) as exc:
            gpu_beamform(prob, kernel)
        assert exc.value.status == das.DAS_ERR_UNSUPPORTED
        return
    y, used = gpu_beamform(prob, kernel)
    assert used == kernel
    ref, slack = oracle_beamform(oracle, prob)
    ratio = error_ratio(y, ref, slack)
    assert ratio <= TOL, (name, kernel, ratio)


@pytest.mark.parametrize("name,auto", [("full_s", "brick"), ("large_s", "brick"),
                                       ("iq_s", "brick")])
def test_auto_choice_and_kernels_agree(small_problems, name, auto):
    prob = small_problems[name]
    kernels = [k for k in KERNELS if kernel_serves(k, prob)]
    outs = {k: gpu_beamform(prob, k)[0] for k in kernels}
    y_auto, used = gpu_beamform(prob, "auto")
    assert used == auto
    assert np.array_equal(y_auto, outs[auto])
    peak = np.abs(outs["bl"]).max()
    for k in kernels:
        assert np.abs(outs[k] - outs["bl"]).max() <= TOL * peak, k


# ------------------------------------------------------------- edge cases
def _custom(**kw):
    base = dict(n_el=4, nx=5, ny=3, nz=2, B=8, K=64, n_scat=2, z_range=(2e-3, 4e-3))
    base.update(kw)
    return synth.make_problem(synth.workload("tiny", **base))


EDGE = {
    "B1": dict(B=1),
    "B3": dict(B=3),
    "B8": dict(B=8),
    "B4": dict(B=4),
    "K2": dict(K=2),
    "K3": dict(K=3),
    "M1": dict(n_el=1),
    "Q1": dict(angles_x_deg=(5.0,)),
    "N1": dict(nx=1, ny=1, nz=1),
    "past_record": dict(K=20),                       # most delays beyond the record
    "no_aperture": dict(fnum=0.0),
    "t0_shift": dict(t0=1.5e-6),
    "iq_B2": dict(iq=True, fs=10e6, f_demod=5e6, B=2, K=128),
    "iq_B6": dict(iq=True, fs=10e6, f_demod=5e6, B=6, K=128),
    "iq_B16": dict(iq=True, fs=10e6, f_demod=5e6, B=16, K=128),
    "iq_B32": dict(iq=True, fs=10e6, f_demod=5e6, B=32, K=128),
    "f32_B64": dict(B=64, K=96),
    "f32_B128": dict(B=128, K=64),
    "B16": dict(B=16),
    "B32": dict(B=32, K=96),
    # neighbouring voxels many samples apart: windows too wide, two rows per voxel
    "coarse_grid": dict(B=32, half_width=15e-3, K=1024, fnum=0.0),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_cases(oracle, name):
    prob = _custom(**EDGE[name])
    ref, slack = oracle_beamform(oracle, prob)
    from volumetric_ultrasound_delay_gb300 import das
    for kernel in ["auto"] + KERNELS:
        try:
            y, _ = gpu_beamform(prob, kernel)
        except das.DasError as exc:
            assert exc.status == das.DAS_ERR_UNSUPPORTED and kernel in RESTRICTED, (name, kernel)
            assert kernel not in ("window", "pair") or not kernel_serves(kernel, prob), (name, kernel)
            continue
        assert error_ratio(y, ref, slack) <= TOL, (name, kernel, error_ratio(y, ref, slack))


def test_nan_delay_contributes_nothing(oracle):
    prob = _custom(B=8)
    prob.tau_tx[1, 3] = np.nan
    prob.tau_tx[0, 5] = np.inf
    ref, slack = oracle_beamform(oracle, prob)
    for kernel in [k for k in KERNELS if kernel_serves(k, prob)]:
        y, _ = gpu_beamform(prob, kernel)
        assert np.all(np.isfinite(y)), kernel
        assert error_ratio(y, ref, slack) <= TOL, kernel


def test_all_outside_aperture_is_zero():
    # voxels above the array (dz < 0): no receiver is inside any aperture
    prob = _custom(z_range=(-4e-3, -2e-3), B=16)
    for kernel in KERNELS:
        y, _ = gpu_beamform(prob, kernel)
        assert not np.any(y), kernel


def test_unsupported_requests_are_rejected():
    from volumetric_ultrasound_delay_gb300 import das
    prob = _custom(B=3)
    for kernel in RESTRICTED:
        with pytest.raises(das.DasError) as exc:
            gpu_beamform(prob, kernel)
        assert exc.value.status == das.DAS_ERR_UNSUPPORTED
    plan = plan_for(prob)
    with pytest.raises(das.DasError):
        plan.set_option(das.OPT_DEMOD_HZ, 5e6)   # real plan cannot demodulate
    for opt in (das.OPT_RX_GROUPS, das.OPT_TX_GROUPS):
        for bad in (-1, 65, 1.5):
            with pytest.raises(das.DasError) as exc:
                plan.set_option(opt, bad)
            assert exc.value.status == das.DAS_ERR_INVALID_ARG
    plan.close()


def test_bi_transmit_table_limit(oracle):
    """BI keeps its CTA's transmit table in shared memory: with more transmits
    than fit it rejects the plan, and AUTO serves it with the brick kernel;
    AUTO and the per-voxel baseline match the oracle."""
    import oracle as oracle_mod
    from volumetric_ultrasound_delay_gb300 import das
    B, Q, M, K = 8, 1000, 1, 8
    rng = np.random.default_rng(11)
    grid = (2, 2, 1, -1e-3, -1e-3, 10e-3, 2e-3, 2e-3, 1e-3)
    rx = np.zeros((M, 3), np.float32)
    rf = torch.from_numpy(rng.standard_normal((B, Q, M, K)).astype(np.float32)).cuda()
    # every voxel is 10.0995 mm from the receiver: delays that land inside the
    # 8-sample record, f = (tau + d / c) * fs in [1, 6]
    d = np.sqrt(1e-6 + 1e-6 + 100e-6)
    tau_np = (-d / 1540.0 + rng.uniform(1.0, 6.0, (Q, 4)) / 20e6).astype(np.float32)
    tau = torch.from_numpy(tau_np).cuda()
    w = torch.from_numpy(rng.uniform(0.5, 1.0, (Q, 4)).astype(np.float32)).cuda()
    ys = {}
    for kernel in ("bi", "auto", "bl"):
        plan = das.Plan(grid, rx, 1540.0, 20e6, 0.0, 0.0, "f32", B, Q, M, K, kernel=kernel)
        if kernel == "bi":
            with pytest.raises(das.DasError) as exc:
                plan.beamform(rf, tau, w)
            assert exc.value.status == das.DAS_ERR_UNSUPPORTED
        else:
            if kernel == "auto":
                assert plan.kernel == "brick"
            ys[kernel] = plan.beamform(rf, tau, w).cpu().numpy()
        plan.close()
    ref, slack = oracle.beamform(rf.cpu().numpy(), tau.cpu().numpy(), w.cpu().numpy(),
                                 rx.astype(np.float64), oracle_mod.Grid(*grid), c=1540.0, fs=20e6,
                                 t0=0.0, fnum=0.0, want_slack=True)
    assert np.abs(ref).max() > 0
    for kernel, y in ys.items():
        assert error_ratio(y, ref, slack) <= TOL, (kernel, error_ratio(y, ref, slack))


def test_bi_chunk_index_limit():
    """BI indexes rows in 32 bits of 16-byte chunks: a record of 2^34 chunks
    (B = 64, M = 2^20, K = 1024) is rejected before anything is read, and AUTO
    picks the brick kernel for it."""
    from volumetric_ultrasound_delay_gb300 import das
    B, Q, M, K = 64, 1, 1 << 20, 1024
    rx = np.zeros((M, 3), np.float32)
    plan = das.Plan((2, 2, 1, 0.0, 0.0, 0.01, 1e-3, 1e-3, 1e-3), rx, 1540.0, 20e6, 0.0, 1.5, "f32",
                    B, Q, M, K)
    assert plan.kernel == "brick"
    plan.kernel = "bi"
    dummy = torch.empty(1024, dtype=torch.float32, device="cuda")
    st = das.lib().das_beamform(plan._h, dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                                dummy.data_ptr() + 2048, None)
    assert st == das.DAS_ERR_UNSUPPORTED
    assert b"2^32" in das.lib().das_last_error_string()
    plan.close()


def test_misaligned_and_wrong_sizes_rejected():
    from volumetric_ultrasound_delay_gb300 import das
    prob = _custom(B=8)
    plan = plan_for(prob)
    rf, tau, w = device_inputs(prob)
    out = torch.empty((prob.B, prob.N), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        plan.beamform(rf[:, :, :, :-1].contiguous(), tau, w, out)
    flat = torch.empty(rf.numel() + 1, dtype=torch.float32, device="cuda")
    mis = flat[1:]
    mis.copy_(rf.reshape(-1))
    h = das.lib().das_beamform(plan._h, mis.data_ptr(), tau.data_ptr(), w.data_ptr(),
                               out.data_ptr(), None)
    assert h == das.DAS_ERR_INVALID_ARG
    plan.close()


@pytest.mark.parametrize("groups", [1, 0, 4, 9])
@pytest.mark.parametrize("name,kernel", [("full_s", "auto"), ("iq_s", "auto"), ("large_s", "auto"),
                                         ("full_s", "window"), ("large_s", "window"),
                                         ("full_s", "pair"), ("large_s", "pair")])
def test_host_entry_point_matches_device(oracle, small_problems, name, kernel, groups):
    """Host buffers in, host buffer out: copying everything first (groups=1)
    reproduces the device entry point bit for bit; streaming the record in
    transmit groups (0 = automatic, 4 = uneven groups of 2-3 transmits, 9 = one
    per transmit) only changes the float32 summation order."""
    from volumetric_ultrasound_delay_gb300 import das
    prob = small_problems[name]
    y_dev, _ = gpu_beamform(prob, kernel)
    plan = plan_for(prob, kernel)
    plan.set_option(das.OPT_HOST_GROUPS, groups)
    out = torch.empty((prob.B, prob.N), dtype=torch.complex64 if prob.wl.iq else torch.float32).pin_memory()
    rf = torch.from_numpy(np.ascontiguousarray(prob.rf)).pin_memory()
    tau = torch.from_numpy(prob.tau_tx).pin_memory()
    w = torch.from_numpy(prob.w_tx).pin_memory()
    for _ in range(2):                       # a second call reuses the staging buffers
        plan.beamform_host(rf, tau, w, out)
    plan.close()
    y = out.numpy()
    if groups == 1:
        assert np.array_equal(y, y_dev)
    ref, slack = oracle_beamform(oracle, prob)
    assert error_ratio(y, ref, slack) <= TOL
    assert np.abs(y - y_dev).max() <= 1e-5 * np.abs(y_dev).max()


def test_host_entry_point_from_two_threads(small_problems):
    """Two plans, each driven by its own host thread through the host entry
    point on its own stream (what bench.py times as e2e.two_threads): every
    call of either thread gives the single-threaded result."""
    import threading
    from volumetric_ultrasound_delay_gb300 import das
    prob = small_problems["full_s"]
    y_dev, _ = gpu_beamform(prob, "auto")
    rf = torch.from_numpy(np.ascontiguousarray(prob.rf)).pin_memory()
    tau = torch.from_numpy(prob.tau_tx).pin_memory()
    w = torch.from_numpy(prob.w_tx).pin_memory()
    plans = [plan_for(prob), plan_for(prob)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results, errors = [[], []], []

    def drive(i):
        try:
            out = torch.empty((prob.B, prob.N), dtype=torch.float32).pin_memory()
            for _ in range(4):
                plans[i].beamform_host(rf, tau, w, out, stream=streams[i])
                results[i].append(out.numpy().copy())
        except Exception as exc:
            errors.append(exc)

    threads = [threading.Thread(target=drive, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    for p in plans:
        p.close()
    assert not errors, errors
    for ys in results:
        assert len(ys) == 4
        for y in ys:
            assert np.abs(y - y_dev).max() <= 1e-5 * np.abs(y_dev).max()


def test_two_plans_pipeline_volumes_on_two_streams(small_problems):
    """Successive volumes alternate between two plans on two streams (the
    permute of one volume can run beside the DAS kernel of the previous one);
    every output equals the serial result, bit for bit."""
    from volumetric_ultrasound_delay_gb300 import das
    prob = small_problems["full_s"]
    rng = np.random.default_rng(41)
    rfs = [torch.from_numpy((prob.rf * rng.uniform(0.5, 2.0)).astype(np.float32)).cuda()
           for _ in range(6)]
    tau = torch.from_numpy(prob.tau_tx).cuda()
    w = torch.from_numpy(prob.w_tx).cuda()
    serial_plan = plan_for(prob)
    serial = [serial_plan.beamform(rf, tau, w).clone() for rf in rfs]
    serial_plan.close()
    plans = [plan_for(prob), plan_for(prob)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty_like(serial[0]) for _ in rfs]
    torch.cuda.synchronize()
    for i, rf in enumerate(rfs):
        plans[i % 2].beamform(rf, tau, w, outs[i], stream=streams[i % 2])
    torch.cuda.synchronize()
    for p in plans:
        p.close()
    for a, b in zip(outs, serial):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["full_s", "iq_s", "large_s"])
def test_launch_groups_match_oracle(oracle, small_problems, name):
    """DAS_OPT_RX_GROUPS and DAS_OPT_TX_GROUPS split the brick launch over
    blocks of 32 receivers and ranges of transmits, each launch adding its
    terms to y: every split (one launch per block or transmit, a few,
    automatic) matches the oracle and the single launch up to the float32
    summation order, and the plan reports the launches it makes."""
    from volumetric_ultrasound_delay_gb300 import das
    prob = small_problems[name]
    ref, slack = oracle_beamform(oracle, prob)
    inputs = device_inputs(prob)
    splits = [(1, 1), (2, 1), (64, 1), (1, 2), (1, prob.Q), (2, 3), (0, 0)]
    ys = {}
    for rx, tx in splits:
        plan = plan_for(prob, "brick")
        plan.set_option(das.OPT_RX_GROUPS, rx)
        plan.set_option(das.OPT_TX_GROUPS, tx)
        assert plan.get_option(das.OPT_TX_GROUPS) == tx
        if rx > 0 and tx > 0:
            assert plan.launches == 1 + min(rx, (prob.M + 31) // 32) * min(tx, prob.Q)
        ys[rx, tx] = plan.beamform(*inputs).cpu().numpy()
        plan.close()
        assert error_ratio(ys[rx, tx], ref, slack) <= TOL, (name, rx, tx)
    peak = np.abs(ys[1, 1]).max()
    for key in splits[1:]:
        assert np.abs(ys[key] - ys[1, 1]).max() <= 1e-5 * peak, (name, key)


@pytest.mark.parametrize("kernel", ["brick", "bi", "bl"])
def test_weights_scaled_by_a_power_of_two(small_problems, kernel):
    """Scaling every transmit weight by 2^90 scales every product of the sum by
    the same power of two, so y scales bit for bit: the brick kernel's weight
    arithmetic (the weight scaled again by 2^(23 - fraction bits) inside) stays
    exact far from float32's range limits."""
    prob = small_problems["full_s"]
    rf, tau, w = device_inputs(prob)
    y1, _ = gpu_beamform(prob, kernel, inputs=(rf, tau, w))
    y2, _ = gpu_beamform(prob, kernel, inputs=(rf, tau, w * 2.0 ** 90))
    assert np.array_equal(y2, (y1.astype(np.float64) * 2.0 ** 90).astype(np.float32))


def test_timing_option_reports_both_kernels(small_problems):
    from volumetric_ultrasound_delay_gb300 import das
    prob = small_problems["full_s"]
    plan = plan_for(prob)
    plan.set_option(das.OPT_TIMING, 1)
    plan.beamform(*device_inputs(prob))
    perm_ms, das_ms = plan.last_times()
    assert perm_ms > 0 and das_ms > 0
    plan.close()


def test_repeated_calls_are_deterministic(small_problems):
    prob = small_problems["iq_s"]
    inputs = device_inputs(prob)
    a, _ = gpu_beamform(prob, inputs=inputs)
    b, _ = gpu_beamform(prob, inputs=inputs)
    assert np.array_equal(a, b)


# --------------------------------------- full-size workloads, sampled voxels
FULL = [("mid", 1024), ("full", 1024), ("iq", 512), ("large", 4096)]


@pytest.mark.parametrize("name,samples", FULL)
def test_full_size_sampled(oracle, name, samples):
    prob = synth.make_problem(name)
    inputs = device_inputs(prob)
    idx = synth.sample_voxels(prob.N, samples, seed=prob.wl.seed)
    ref, slack = oracle_beamform(oracle, prob, idx=idx)
    kernels = ["auto", "bi", "brick"] + (["window", "pair"] if name != "iq" else []) + \
        (["bl"] if name in ("mid", "full") else [])
    for kernel in kernels:
        y, used = gpu_beamform(prob, kernel, inputs=inputs)
        ratio = error_ratio(y[:, idx], ref, slack)
        assert ratio <= TOL, (name, used, ratio)
        # every output is finite and the volume is not empty
        assert np.all(np.isfinite(y)) and np.abs(y).max() > 0
    del inputs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,storage,launches", [
    ("full", "native", 3), ("full", "f16", 2), ("iq", "native", 4), ("iq", "f16", 3),
    ("large", "native", 2), ("mid", "native", 2), ("tiny", "native", 2)])
def test_automatic_transmit_groups(name, storage, launches):
    """The automatic transmit split of the brick kernel on the five workloads:
    one launch where the permuted record holds less than one byte per 64
    accumulations (large) or fits 16 times the L2 (mid, tiny, half storage on
    the full volume), else enough launches for a share of at most 16 times the
    L2 (full: 2, IQ: 3, IQ half2: 2).  The plan reports the permute plus those
    launches; no record is needed to ask."""
    from volumetric_ultrasound_delay_gb300 import das, synth
    wl = synth.workload(name)
    grid = synth.grid_params(wl)
    rx = synth.array_positions(wl.n_el).astype(np.float32)
    props = torch.cuda.get_device_properties(0)
    if not 101e6 <= props.L2_cache_size < 151e6:
        pytest.skip("the counts above hold for an L2 of 101 to 151 MB")
    plan = das.Plan(grid, rx, wl.c, wl.fs, wl.t0, wl.fnum, "c64" if wl.iq else "f32", wl.B, wl.Q, wl.M,
                    wl.K, kernel="brick", f_demod=wl.f_demod, storage=storage)
    assert plan.launches == launches
    plan.set_option(das.OPT_TX_GROUPS, 1)
    assert plan.launches == 2
    plan.close()
