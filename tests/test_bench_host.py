"""Host-side pieces of bench.py that need no GPU: the in-aperture pair count
behind frac_in_aperture, and the rule that a stored DRAM-traffic figure is
reported only while the kernel source it was taken on is unchanged."""
import json
import os
import sys
import types

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from volumetric_ultrasound_delay_gb300 import synth  # noqa: E402


def _count_directly(prob):
    """The F-number test voxel by voxel and receiver by receiver."""
    nx, ny, nz, x0, y0, z0, dx, dy, dz = prob.grid
    rx = prob.rx.astype(np.float64)
    total = 0
    for iz in range(nz):
        for iy in range(ny):
            for ix in range(nx):
                x, y, z = x0 + ix * dx, y0 + iy * dy, z0 + iz * dz
                ez = z - rx[:, 2]
                rho2 = (x - rx[:, 0]) ** 2 + (y - rx[:, 1]) ** 2
                total += int(np.count_nonzero((ez > 0) & ((2 * prob.fnum) ** 2 * rho2 <= ez * ez)))
    return total


def test_aperture_pairs_match_a_direct_count():
    prob = synth.make_problem("tiny", nx=7, ny=5, nz=4)
    assert bench.aperture_pairs(prob) == _count_directly(prob)
    assert 0 < bench.aperture_pairs(prob) < prob.N * prob.M


def test_aperture_pairs_without_aperture_count_every_pair():
    prob = synth.make_problem("tiny", nx=3, ny=3, nz=2)
    off = types.SimpleNamespace(grid=prob.grid, rx=prob.rx, fnum=0.0)
    assert bench.aperture_pairs(off) == prob.N * prob.M


def test_traffic_is_reported_only_for_the_measured_source(tmp_path, monkeypatch):
    rec = {"brick/full": {"source_sha": bench.source_sha("brick"), "dram_bytes_per_launch": 123},
           "window/full": {"source_sha": "0000000000000000", "dram_bytes_per_launch": 456}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.measured_traffic("brick", "full") == 123
    assert bench.measured_traffic("window", "full") is None          # kernel changed since
    assert bench.measured_traffic("brick", "mid") is None            # never measured
    assert bench.measured_traffic("brick", "full", "f16") is None


def test_committed_traffic_record_names_its_commands():
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)
    for key, r in rec.items():
        total = r.get("dram_bytes_per_call", r.get("dram_bytes_per_launch"))
        assert total == r["dram_read"] + r["dram_write"], key
        assert r["command"].startswith("ncu ") and "--clock-control none" in r["command"], key
        if "dram_bytes_per_call" in r:
            # one capture of all the DAS launches of one call: -c equals the launch count
            assert f"-c {r['launches_per_call']} " in r["command"], key


def test_traffic_per_call_sums_the_launches(tmp_path, monkeypatch):
    rec = {"brick/full": {"source_sha": bench.source_sha("brick"), "dram_bytes_per_call": 300,
                          "launches_per_call": 2, "dram_read": 280, "dram_write": 20}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.measured_traffic("brick", "full") == 300
