#!/usr/bin/env python3
"""Benchmark of volumetric delay-and-sum on GB300: DAS accumulations/s.

One step = one das_beamform call over the whole workload (RF permute + DAS
kernel), inputs resident in HBM.  Default workload: the 32 x 32 matrix-array
volume (M = 1024 receivers, Q = 9 diverging waves, K = 2048 float32 samples,
64^3 voxels, B = 32 frames) -- 7.73e10 accumulations per step.  Its 2.4 GB RF
record is far larger than the 129 MB L2, so no explicit L2 flush is needed;
workloads whose record is smaller than twice the L2 (the small ones) get a
write of twice the L2 size between timed steps, and each step is then timed
by its own pair of events.

Prints ONE JSON line (rank 0).  Besides the device-timed value it reports:
  roofline      the DAS kernel against the FP32 issue roofline (alu bound):
                5 issue slots (2 loads + 3 FMA) per accumulation, B*N*Q*M
                accumulations per launch; frac_in_aperture counts only the
                accumulations inside the F-number aperture (the rest are zero);
                diagnostics: the L1-return ceiling and the FMA floor over the
                in-aperture accumulations;
  cpu_baseline  the float64 oracle on the host cores, on a bounded voxel sample;
  e2e           the same metric through das_beamform_host with pinned host
                buffers (host->device and device->host copies inside the timing);
                two_threads: a stream of volumes on two plans, one host thread each;
  clocks        SM clocks and throttle reasons sampled during the timed region;
  pipeline      volumes alternating between two plans on two streams (the
                permute of one overlaps the DAS kernel of the other), per volume;
  relative      every kernel (and half-precision storage where a kernel takes
                it) on the same workload, DAS-kernel time by CUDA events, with
                the two ratios the pages report: BI over BL and BI-FP16 over BI.

``--impl reference`` times the oracle itself (the reference arm: a plain CPU
program) on bounded samples of the same workload.  Under torchrun with N > 1
GPUs every rank runs an independent replica (weak scaling, no collective on the
data path); the timing takes the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DAS accumulations/s (B·N·Q·M/time) at 1 GB300; fraction of roofline"
UNIT = "accumulations/s"
ISSUE_SLOTS_PER_ACC = 5        # ~2 loads + 3 FMA per accumulation at FP32 issue peak
FP32_LANES_PER_SM = 128
L2_FALLBACK = 129 * 2**20       # GB300 L2 bytes, if the device properties do not say
L1_BYTES_PER_CLK = 128          # L1 return to registers per SM and clock (one 128-byte wavefront)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="full", choices=["tiny", "mid", "full", "iq", "large"])
    ap.add_argument("--kernel", default="auto", choices=["auto", "bl", "bi", "brick", "window", "pair"])
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-volumes", type=int, default=3,
                    help="e2e.stream: volumes per das_beamform_host_volumes call (0 = skip)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--pipeline", type=int, default=20, metavar="V",
                    help="also time V volumes alternating between two plans on two streams "
                         "(the permute of one volume can overlap the DAS kernel of the other); "
                         "0 = off; skipped for records that fit in L2")
    ap.add_argument("--n-el", type=int, default=None, help="override: array elements per side")
    ap.add_argument("--grid", type=int, nargs=3, default=None, metavar=("NX", "NY", "NZ"),
                    help="override: voxel grid (for small profiling cases)")
    ap.add_argument("--storage", default="native", choices=["native", "f16"],
                    help="element type of the permuted record copy (f16: half precision)")
    ap.add_argument("--record", default="native", choices=["native", "f16"],
                    help="element type of the record the caller passes: native (float32 / "
                         "complex64) or f16 (the synthetic record rounded to float16 / half2: "
                         "DAS_F16 / DAS_C32H plans, half the bytes to copy and permute)")
    ap.add_argument("--host-groups", type=int, default=None,
                    help="e2e: transmit groups the host entry point streams the record in "
                         "(default: the library's automatic choice)")
    ap.add_argument("--tx-groups", type=int, default=None,
                    help="brick kernel: launches the transmits are split into (default: the "
                         "library's automatic choice)")
    ap.add_argument("--relative-steps", type=int, default=3,
                    help="timed calls per kernel of the relative table (0 = no table)")
    return ap.parse_args()


def make_workload(args):
    from volumetric_ultrasound_delay_gb300 import synth
    kw = {}
    if args.n_el:
        kw["n_el"] = args.n_el
    if args.grid:
        kw["nx"], kw["ny"], kw["nz"] = args.grid
    return synth.make_problem(args.workload, **kw)


def describe(wl) -> str:
    tx = {"dw": f"{wl.Q} diverging waves", "pw": f"{wl.Q} plane waves"}[wl.transmit]
    dt = "c64 IQ" if wl.iq else "f32 RF"
    return (f"{wl.name}: {wl.n_el}x{wl.n_el} array (M={wl.M}), {tx}, K={wl.K} {dt} at "
            f"{wl.fs / 1e6:g} MHz, {wl.nx}x{wl.ny}x{wl.nz} voxels (N={wl.N}), B={wl.B}, F#={wl.fnum}")


def aperture_pairs(prob) -> int:
    """Number of (voxel, receiver) pairs inside the F-number aperture (all
    pairs when F# <= 0 switches the aperture off)."""
    nx, ny, nz, x0, y0, z0, dx, dy, dz = prob.grid
    if prob.fnum <= 0:
        return nx * ny * nz * len(prob.rx)
    xs = x0 + np.arange(nx) * dx
    ys = y0 + np.arange(ny) * dy
    rx = prob.rx.astype(np.float64)
    two_f2 = (2.0 * prob.fnum) ** 2
    ddx = (xs[:, None] - rx[None, :, 0]) ** 2          # nx x M
    ddy = (ys[:, None] - rx[None, :, 1]) ** 2          # ny x M
    total = 0
    for iz in range(nz):
        ez = z0 + iz * dz - rx[:, 2]                    # M
        lim = np.where(ez > 0, ez * ez / two_f2, -1.0)  # rho^2 limit per receiver
        for m0 in range(0, rx.shape[0], 256):
            sl = slice(m0, m0 + 256)
            inside = (ddx[:, None, sl] + ddy[None, :, sl]) <= lim[None, None, sl]
            total += int(inside.sum())
    return total


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(float(r[2]) for r in rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()),
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------ CPU oracle
def time_oracle(prob, target_s: float, seed: int):
    """Oracle accumulations/s on a seeded voxel sample sized to ~target_s."""
    import oracle
    orc = oracle.load()
    cores = os.cpu_count() or 1
    per_voxel = prob.B * prob.Q * prob.M
    g = oracle.Grid(*prob.grid)
    kw = dict(c=prob.c, fs=prob.fs, t0=prob.t0, fnum=prob.fnum, f_demod=prob.f_demod,
              nthreads=cores)
    probe = synth_sample(prob.N, min(prob.N, 4 * cores), seed)
    t = time.perf_counter()
    orc.beamform(prob.rf, prob.tau_tx, prob.w_tx, prob.rx.astype(np.float64), g, idx=probe, **kw)
    rate = len(probe) / max(time.perf_counter() - t, 1e-6)
    count = int(min(prob.N, max(len(probe), rate * target_s)))
    idx = synth_sample(prob.N, count, seed + 1)
    t = time.perf_counter()
    orc.beamform(prob.rf, prob.tau_tx, prob.w_tx, prob.rx.astype(np.float64), g, idx=idx, **kw)
    dt = time.perf_counter() - t
    return {"value": count * per_voxel / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{count} seeded voxels of {prob.N} (all B, Q, M); {dt:.1f} s",
            "seconds": dt}


def synth_sample(N, count, seed):
    from volumetric_ultrasound_delay_gb300 import synth
    return synth.sample_voxels(N, count, seed)


# --------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def source_sha(kernel: str) -> str:
    name = {"brick": "das_brick.cu", "window": "das_window.cu", "bi": "das_bi.cu", "bl": "das_bl.cu",
            "pair": "das_pair.cu"}[kernel]
    h = hashlib.sha256()
    # the kernel and the host code that splits its launches
    for f in (name, "das_device.cuh", "das_internal.cuh", "das_api.cu"):
        with open(os.path.join(ROOT, "volumetric_ultrasound_delay_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str, storage: str = "native"):
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    key = f"{kernel}/{workload}" + ("" if storage == "native" else f"/{storage}")
    r = rec.get(key)
    if not r or r.get("source_sha") != source_sha(kernel):
        return None   # never measured, or the kernel changed since the counters were taken
    # DRAM bytes of the DAS kernel's launches in one call (one launch, or the
    # transmit / receiver groups of the brick kernel together)
    return r.get("dram_bytes_per_call", r.get("dram_bytes_per_launch"))


def relative_table(args, prob, rf, tau, w, out, stream, dev):
    """DAS-kernel milliseconds of every kernel that serves the workload, float32
    and half-precision storage, by the CUDA events the library records on the
    launching stream (mean of the timed calls after two warm-up calls), and the
    pages' two relative measurements: batch-inner over the per-voxel baseline,
    and half-precision storage over float32 on the batch-inner kernel (ffdas
    paper, Results, Fig. 2A-C; ffdas docs, ALG2 and "Mixed-precision storage")."""
    import torch
    from volumetric_ultrasound_delay_gb300 import das
    dtype = "c64" if prob.wl.iq else "f32"
    A = prob.B * prob.N * prob.Q * prob.M
    rows = {}
    for kernel, storage in [("bl", "native"), ("bi", "native"), ("bi", "f16"), ("brick", "native"),
                            ("brick", "f16"), ("window", "native"), ("pair", "native")]:
        try:
            plan = das.Plan(prob.grid, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, dtype, prob.B,
                            prob.Q, prob.M, prob.K, kernel=kernel, f_demod=prob.f_demod,
                            storage=storage)
        except das.DasError:
            continue
        plan.set_option(das.OPT_TIMING, 1)
        try:
            for _ in range(2):
                plan.beamform(rf, tau, w, out, stream=stream)
            ms = []
            for _ in range(args.relative_steps):
                plan.beamform(rf, tau, w, out, stream=stream)
                ms.append(plan.last_times()[1])
        except das.DasError:
            plan.close()
            continue
        torch.cuda.synchronize(dev)
        plan.close()
        das_ms = statistics.mean(ms)
        rows[f"{kernel}/{storage}"] = {"das_ms": das_ms, "value": A / (das_ms / 1e3)}
    ratios = {}
    if "bi/native" in rows and "bl/native" in rows:
        ratios["bi_over_bl"] = rows["bl/native"]["das_ms"] / rows["bi/native"]["das_ms"]
    if "bi/f16" in rows and "bi/native" in rows:
        ratios["bi_f16_over_bi"] = rows["bi/native"]["das_ms"] / rows["bi/f16"]["das_ms"]
    if "brick/f16" in rows and "brick/native" in rows:
        ratios["brick_f16_over_brick"] = rows["brick/native"]["das_ms"] / rows["brick/f16"]["das_ms"]
    return {"kernels": rows, "ratios": ratios, "unit": UNIT,
            "note": "DAS kernel only (permute excluded), mean of timed calls; ratios are speed-ups; "
                    "the pages quote BI about 1.4x BL and FP16 storage about 1.2x, hardware unstated"}


# ------------------------------------------------------------- arms
def run_reference(args, world, rank):
    if rank != 0:
        return
    from volumetric_ultrasound_delay_gb300 import synth
    import oracle
    oracle.build()
    prob = make_workload(args)
    cores = os.cpu_count() or 1
    per_step = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    # size one step's voxel sample from a probe run
    cal = time_oracle(prob, per_step, seed=100)
    count = min(prob.N, max(1, int(cal["value"] * per_step / (prob.B * prob.Q * prob.M))))
    import oracle as om
    orc = om.load()
    g = om.Grid(*prob.grid)
    kw = dict(c=prob.c, fs=prob.fs, t0=prob.t0, fnum=prob.fnum, f_demod=prob.f_demod, nthreads=cores)
    rx64 = prob.rx.astype(np.float64)
    times = []
    for s in range(args.warmup + args.steps):
        idx = synth.sample_voxels(prob.N, count, 1000 + s)
        t = time.perf_counter()
        orc.beamform(prob.rf, prob.tau_tx, prob.w_tx, rx64, g, idx=idx, **kw)
        if s >= args.warmup:
            times.append(time.perf_counter() - t)
    acc = count * prob.B * prob.Q * prob.M
    value = acc * len(times) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded numpy: noise + point-scatterer echoes)",
        "config": {"workload": describe(prob.wl), "sample_per_step": f"{count} seeded voxels"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{count} seeded voxels of {prob.N} per step (all B, Q, M)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch
    from volumetric_ultrasound_delay_gb300 import das, synth
    from volumetric_ultrasound_delay_gb300 import build as libbuild
    libbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    prob = make_workload(args)
    half_rec = args.record == "f16"
    dtype = ("c32h" if half_rec else "c64") if prob.wl.iq else ("f16" if half_rec else "f32")
    A = prob.B * prob.N * prob.Q * prob.M
    rf_src = torch.from_numpy(prob.rf)
    if half_rec:
        rf_src = rf_src.to(torch.complex32 if prob.wl.iq else torch.float16)
    rf = rf_src.to(dev)
    rec_bytes = rf.numel() * rf.element_size()
    tau = torch.from_numpy(prob.tau_tx).to(dev)
    w = torch.from_numpy(prob.w_tx).to(dev)
    out = torch.empty((prob.B, prob.N), dtype=torch.complex64 if prob.wl.iq else torch.float32,
                      device=dev)
    plan = das.Plan(prob.grid, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, dtype, prob.B,
                    prob.Q, prob.M, prob.K, kernel=args.kernel, f_demod=prob.f_demod,
                    storage=args.storage)
    if args.tx_groups is not None:
        plan.set_option(das.OPT_TX_GROUPS, args.tx_groups)
    kernel = plan.kernel
    launches_per_call = plan.launches          # permute + DAS launches of one call
    plan.set_option(das.OPT_TIMING, 1)
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(3, args.warmup)):
        plan.beamform(rf, tau, w, out, stream=stream)
    torch.cuda.synchronize(dev)

    # a record smaller than twice the L2 could stay cached from one step to the
    # next: then a write of twice the L2 size runs between the timed steps
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_FALLBACK)
    flush = rec_bytes < 2 * l2_bytes
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    das_ms, perm_ms, step_ms = [], [], []
    ev0.record(stream)
    for i in range(args.steps):
        if flush:
            flush_buf.fill_(i & 0xff)
            ev0.record(stream)
        plan.beamform(rf, tau, w, out, stream=stream)
        if flush:
            ev1.record(stream)
            ev1.synchronize()
            step_ms.append(ev0.elapsed_time(ev1))
        p_ms, d_ms = plan.last_times()      # events recorded by the library on `stream`
        perm_ms.append(p_ms)
        das_ms.append(d_ms)
    if not flush:
        ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(world, sum(step_ms) if flush else ev0.elapsed_time(ev1))
    ms_per_step = elapsed_ms / args.steps
    l2_note = (f"L2 flushed between steps (write of {2 * l2_bytes / 1e6:.0f} MB; "
               f"{rec_bytes / 1e6:.0f} MB RF record), steps timed one by one" if flush else
               f"inputs larger than L2 ({rec_bytes / 1e9:.2f} GB RF record), no flush")
    value = world * A / (ms_per_step / 1e3)

    # ---------------- e2e through the host entry point (pinned buffers)
    e2e = None
    if not args.no_e2e:
        rf_h = rf_src.pin_memory()
        tau_h = torch.from_numpy(prob.tau_tx).pin_memory()
        w_h = torch.from_numpy(prob.w_tx).pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        if args.host_groups is not None:
            plan.set_option(das.OPT_HOST_GROUPS, args.host_groups)
        plan.beamform_host(rf_h, tau_h, w_h, out_h, stream=stream)      # warm-up, allocates
        barrier(world)
        # median of the steps: the host link is shared with other jobs and an
        # occasional step can take several times longer
        e2e_t = []
        for _ in range(args.e2e_steps):
            t = time.perf_counter()
            plan.beamform_host(rf_h, tau_h, w_h, out_h, stream=stream)
            e2e_t.append(time.perf_counter() - t)
        e2e_s = max_over_ranks(world, statistics.median(e2e_t))
        e2e = {"value": world * A / e2e_s, "unit": UNIT,
               "h2d_bytes_per_step": int(rf_h.numel() * rf_h.element_size() + 2 * tau_h.numel() * 4),
               "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size()),
               "ms_per_step": 1e3 * e2e_s, "statistic": f"median of {args.e2e_steps} steps",
               "steps_ms": [round(1e3 * x, 3) for x in e2e_t]}
        ref = out.cpu()
        if float((out_h - ref).abs().max()) > 1e-5 * float(ref.abs().max()):
            raise RuntimeError("host entry point disagrees with the device entry point")
        if args.e2e_volumes > 0:
            # a stream of volumes through one call: each volume's record copied
            # and its y read back inside the timed region
            nv = args.e2e_volumes
            rf_v = torch.empty((nv,) + tuple(rf_src.shape), dtype=rf_src.dtype).pin_memory()
            rf_v.copy_(rf_src.unsqueeze(0).expand_as(rf_v))
            out_v = torch.empty((nv,) + tuple(out.shape), dtype=out.dtype).pin_memory()
            plan.beamform_host_volumes(rf_v, tau_h, w_h, out_v, stream=stream)      # warm-up
            barrier(world)
            t = time.perf_counter()
            plan.beamform_host_volumes(rf_v, tau_h, w_h, out_v, stream=stream)
            vol_s = max_over_ranks(world, time.perf_counter() - t)
            if float((out_v[-1] - ref).abs().max()) > 1e-5 * float(ref.abs().max()):
                raise RuntimeError("volume stream disagrees with the device entry point")
            e2e["stream"] = {"volumes": nv, "ms_per_volume": 1e3 * vol_s / nv,
                             "value": world * A * nv / vol_s, "unit": UNIT,
                             "h2d_bytes_per_volume": e2e["h2d_bytes_per_step"] - int(2 * tau_h.numel() * 4),
                             "note": "das_beamform_host_volumes: one call, one plan; each volume's record "
                                     "copied and its y read back inside the timed region"}
            del rf_v, out_v
        if args.pipeline > 0 and not flush:
            # a stream of volumes: two plans, each driven by its own host thread
            # through the same host entry point, so one volume's upload overlaps
            # the other's kernels; every volume still includes its copies
            plan_b = das.Plan(prob.grid, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, dtype, prob.B,
                              prob.Q, prob.M, prob.K, kernel=args.kernel, f_demod=prob.f_demod,
                              storage=args.storage)
            out_b = torch.empty(out.shape, dtype=out.dtype).pin_memory()
            if args.host_groups is not None:
                plan_b.set_option(das.OPT_HOST_GROUPS, args.host_groups)
            s_a, s_b = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
            plan_b.beamform_host(rf_h, tau_h, w_h, out_b, stream=s_b)       # warm-up, allocates
            errors = []

            def drive(p, o, s):
                try:
                    for _ in range(args.e2e_steps):
                        p.beamform_host(rf_h, tau_h, w_h, o, stream=s)
                except Exception as exc:        # reported after the join
                    errors.append(exc)

            threads = [threading.Thread(target=drive, args=(plan, out_h, s_a)),
                       threading.Thread(target=drive, args=(plan_b, out_b, s_b))]
            barrier(world)
            t = time.perf_counter()
            for th in threads:
                th.start()
            for th in threads:
                th.join()
            both_s = max_over_ranks(world, time.perf_counter() - t)
            if errors:
                raise errors[0]
            if float((out_b - ref).abs().max()) > 1e-5 * float(ref.abs().max()):
                raise RuntimeError("pipelined host entry point disagrees with the device entry point")
            vols = 2 * args.e2e_steps
            e2e["two_threads"] = {"volumes": vols, "ms_per_volume": 1e3 * both_s / vols,
                                  "value": world * A * vols / both_s, "unit": UNIT,
                                  "note": "two plans, one host thread each, das_beamform_host; "
                                          "copies of every volume inside the timed region"}
            plan_b.close()

    # ---------------- every kernel on the same workload (the pages' relative figures)
    relative = None
    if args.relative_steps > 0 and rank == 0 and not half_rec:
        plan.set_option(das.OPT_TIMING, 0)
        relative = relative_table(args, prob, rf, tau, w, out, stream, dev)
        plan.set_option(das.OPT_TIMING, 1)

    # ---------------- two plans on two streams, volumes alternating (optional)
    pipeline = None
    if args.pipeline > 0 and not flush:
        plan2 = das.Plan(prob.grid, prob.rx, prob.c, prob.fs, prob.t0, prob.fnum, dtype, prob.B,
                         prob.Q, prob.M, prob.K, kernel=args.kernel, f_demod=prob.f_demod,
                         storage=args.storage)
        if args.tx_groups is not None:
            plan2.set_option(das.OPT_TX_GROUPS, args.tx_groups)
        streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
        outs = [out, torch.empty_like(out)]
        plans = [plan, plan2]
        plan.set_option(das.OPT_TIMING, 0)
        for i in range(4):                               # warm-up of both plans
            plans[i % 2].beamform(rf, tau, w, outs[i % 2], stream=streams[i % 2])
        torch.cuda.synchronize(dev)
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        joined = torch.cuda.Event()
        start.record(streams[0])
        streams[1].wait_event(start)
        for i in range(args.pipeline):
            plans[i % 2].beamform(rf, tau, w, outs[i % 2], stream=streams[i % 2])
        joined.record(streams[1])
        streams[0].wait_event(joined)
        stop.record(streams[0])
        torch.cuda.synchronize(dev)
        p_ms = max_over_ranks(world, start.elapsed_time(stop)) / args.pipeline
        pipeline = {"volumes": args.pipeline, "ms_per_volume": p_ms, "value": world * A / (p_ms / 1e3),
                    "unit": UNIT, "plans": 2, "streams": 2,
                    "vs_one_stream": ms_per_step / p_ms}
        plan2.close()
        plan.set_option(das.OPT_TIMING, 1)

    # ---------------- roofline of the dominant kernel (the DAS kernel)
    pairs = aperture_pairs(prob)
    a_eff = prob.B * prob.Q * pairs
    props = torch.cuda.get_device_properties(dev)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        sm_max = float(peaks["sm_max_mhz"])
        peak_src = "MEASURED_PEAKS.json sm_max_mhz"
    except (OSError, ValueError, KeyError):
        sm_max = 2070.0
        peak_src = "nominal max SM clock"
    peak = props.multi_processor_count * FP32_LANES_PER_SM * sm_max * 1e6 / 1e12   # T issue/s
    das_mean = statistics.mean(das_ms)
    # algorithmic work: 2 sample loads + 3 FMA = 5 FP32 issue slots for each of
    # the B*N*Q*M accumulations of one launch
    achieved = ISSUE_SLOTS_PER_ACC * A / (das_mean / 1e3) / 1e12
    achieved_in = ISSUE_SLOTS_PER_ACC * a_eff / (das_mean / 1e3) / 1e12
    # the captures were taken with the library's own launch split
    traffic = (measured_traffic(kernel, args.workload, args.storage)
               if args.tx_groups is None and args.record == "native" else None)
    roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Tinst/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": f"das_{kernel}_kernel", "kernel_ms": das_mean,
                "das_launches_per_call": launches_per_call - (0 if kernel == "bl" else 1),
                "work": f"{ISSUE_SLOTS_PER_ACC} FP32 issue slots x {A:.4g} accumulations "
                        f"(B*N*Q*M) per call (all DAS launches of the call; CUDA events "
                        f"around them on the launching stream)",
                # the terms outside the F-number aperture are zero and skipped;
                # counting only the rest gives the stricter figure
                "frac_in_aperture": achieved_in / peak,
                "in_aperture_fraction": pairs / (prob.N * prob.M),
                "peak_source": f"{props.multi_processor_count} SMs x {FP32_LANES_PER_SM} lanes x "
                               f"{sm_max:g} MHz ({peak_src})"}
    # the two ceilings beside the issue roofline, over the in-aperture
    # accumulations the kernels actually do: the L1 return of the samples
    # (two rows of the frame's element per accumulation, at 128 B/clk/SM; the
    # one that binds in practice) and the FMA floor (2 FMA per real
    # accumulation with the weights folded, 8 per complex one, at 128/clk/SM)
    sample_bytes = (2 if args.storage == "f16" else 4) * (2 if prob.wl.iq else 1)
    sm_cycles = props.multi_processor_count * sm_max * 1e6            # SM clocks per second
    l1_floor_ms = 1e3 * a_eff * 2 * sample_bytes / (sm_cycles * L1_BYTES_PER_CLK)
    fma_per_acc = 8 if prob.wl.iq else 2
    fma_floor_ms = 1e3 * a_eff * fma_per_acc / (sm_cycles * FP32_LANES_PER_SM)
    roofline["diagnostics"] = {
        "l1_return": {"bytes_per_accumulation": 2 * sample_bytes, "floor_ms": l1_floor_ms,
                      "frac": l1_floor_ms / das_mean,
                      "basis": f"{a_eff:.4g} in-aperture accumulations x {2 * sample_bytes} B at "
                               f"{L1_BYTES_PER_CLK} B/clk/SM"},
        "fma": {"fma_per_accumulation": fma_per_acc, "floor_ms": fma_floor_ms,
                "frac": fma_floor_ms / das_mean,
                "basis": f"{a_eff:.4g} in-aperture accumulations x {fma_per_acc} FMA at "
                         f"{FP32_LANES_PER_SM}/clk/SM"},
    }

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(prob, args.cpu_seconds, seed=7)
        cpu.pop("seconds", None)

    launches = args.steps * launches_per_call
    plan.close()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "c64" if prob.wl.iq else "f32",
        "data": "synthetic (seeded numpy: N(0,1) noise + point-scatterer echoes)",
        "config": {"workload": describe(prob.wl), "kernel": kernel, "storage": args.storage,
                   "launches_per_step": launches_per_call, "record": args.record,
                   "accumulations_per_step": A,
                   "in_aperture_fraction": pairs / (prob.N * prob.M),
                   "l2": l2_note,
                   "replicas": world},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": launches,
        "kernel_ms": {"permute": statistics.mean(perm_ms), "das": das_mean},
    }
    if pipeline is not None:
        line["pipeline"] = pipeline
    if relative is not None:
        line["relative"] = relative
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
