"""Long records (K = 16384 and 65536 samples): every kernel against the oracle.

The voxels sit 5-20 mm or 5-50 mm from the 8 x 8 array at 20 MHz, so the
delays use the first few thousand samples of a long record.  That is where
the record length, not the delay, sets how finely the brick kernel's packed
32-bit entries can hold the interpolation fraction: the kernel packs entries
only while at least 14 fraction bits remain (K <= 8189) and takes float
entries for longer records, so the fraction is never coarser than float32
(packed, K = 65536 would leave 10 bits, a step of 1e-3 samples: on these
20 MHz echoes, whose slope reaches 1.6 per sample, a rounding error of that
size per term comes close to the parity bar).  Records are noise-free
point-scatterer echoes
(scatterers at voxel positions), a few frames, and small grids, so the oracle
stays fast (16 frames, one transmit)."""
import numpy as np
import pytest

from parity import TOL, error_ratio, gpu_beamform, oracle_beamform
from volumetric_ultrasound_delay_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU containers skip these
    pytest.skip("needs a CUDA device", allow_module_level=True)

KERNELS = ["bl", "bi", "brick", "window", "pair"]

CASES = {
    "K16384_shallow": dict(base="tiny", K=16384, fs=20e6, z_range=(5e-3, 20e-3)),
    "K65536_shallow": dict(base="tiny", K=65536, fs=20e6, z_range=(5e-3, 20e-3)),
    "K65536_50mm": dict(base="tiny", K=65536, fs=20e6, z_range=(5e-3, 50e-3)),
}


def long_problem(name):
    kw = dict(CASES[name])
    base = kw.pop("base")
    wl = synth.workload(base, nx=6, ny=6, nz=12, B=16, angles_x_deg=(0.0,), noise=False, n_scat=0,
                        **kw)
    prob = synth.make_problem(wl)
    pts = synth.grid_points(prob.grid)
    picks = np.linspace(0, prob.N - 1, 6).astype(int)[1:-1]
    prob.rf += synth.echo_record(wl, prob.rx.astype(np.float64), pts[picks]).astype(np.float32)[None]
    return prob


@pytest.fixture(scope="module")
def long_problems(oracle):
    out = {}
    for name in CASES:
        prob = long_problem(name)
        out[name] = (prob, *oracle_beamform(oracle, prob))
    return out


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", list(CASES))
def test_long_record(long_problems, name, kernel):
    prob, ref, slack = long_problems[name]
    assert float(np.abs(ref).max()) > 10.0          # the echoes focus on their voxels
    y, used = gpu_beamform(prob, kernel)
    assert used == kernel
    ratio = error_ratio(y, ref, slack)
    assert ratio <= TOL, (name, kernel, ratio)
