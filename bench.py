"""Benchmark of the depth-decoder frame on one GB300 (or N replicas).

A step is one frame: the whole hot path (input projection, 5 layers x 16
positions, 15 heads, 15 draws, 16 embedding steps; 432 phases) over one batch
of rows. The headline workload is the full-shape frame at 64 rows with the
sampled settings (temperature 0.9, top-k 50, top-p 0.8, seed = row), frames
chained on the device (each frame's first code is the previous frame's last
code, offsets carried, a fresh talker hidden state per frame). Weights are
synthetic (bf16 N(0, 0.02)) with the 1.7B CodePredictor's shapes.

Printed: one JSON line (rank 0). `value` is frames/s of cp_frame with inputs
resident; `e2e` the same through the C ABI with the step's inputs copied from
pinned host memory and its codes/offsets copied back inside the timed region;
`roofline` the frame kernel's weight-stream bandwidth against the measured HBM
copy peak (`traffic`: the DRAM bytes per launch of the committed ncu capture,
kept only while the kernel source it was taken from is unchanged); `split` the
per-phase graph (cp_frame_split); `sweep` the row sweep 1/16/32/59/64 (mixed
per-row samplers, 200 chained frames per point) of both; `sweep128` frames of
65/96/128 rows on a 128-row handle; `clocks` NVML samples of the timed region;
`cpu_baseline` the oracle on the host cores (and on one core).

By default the line also carries (`--quick` skips them): `trace_breakdown` and
`trace_breakdown_128`, the per-task timestamp breakdowns of one traced frame
at 64 and 128 rows (wait, handoff, input landing, weights, MMA, exchange,
epilogue, signal; trace_report.py) and `tensor_pipe_by_kind`; `cuts`, the same
frame as one kernel per depth position, per layer and as attention-phase plus
MLP-phase kernels, beside cp_frame and cp_frame_split, with the last two
predicted from the first by the event-graph simulation (simulate.py); `wide`,
the 2x-wide shape (hidden 2048, 16 kv heads, FFN 6144).

`--impl reference` times the CPU oracle instead (bounded samples per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

ROWS = 64
WORKLOAD = ("full-shape depth-decoder frame (5 layers, hidden 1024, 16/8 heads x 128, FFN 3072, "
            "16 positions, vocab 2048, input 2048->1024), 64 rows, sampled (T 0.9, top-k 50, top-p 0.8)")
METRIC = "frames/s"


# the files the frame kernel is compiled from (the traffic record names their hash)
KERNEL_SOURCES = ("cp_kernel.cu", "cp_ptx.cuh", "cp_internal.h")


def _traffic():
    """DRAM bytes per frame-kernel launch from the committed ncu capture, or
    None when the kernel source has changed since it was taken."""
    import hashlib
    try:
        csrc = os.path.join(ROOT, "persistent_megakernel_streaming_gb300", "csrc")
        src = b"".join(open(os.path.join(csrc, f), "rb").read() for f in KERNEL_SOURCES)
        rec = dict(l.split(":", 1) for l in open(os.path.join(ROOT, "profiles", "frame_kernel_traffic.txt"))
                   if ":" in l and not l.startswith("#"))
        if rec.get("kernel_source_sha256", "").strip() != hashlib.sha256(src).hexdigest():
            return None
        return int(rec["dram_bytes_per_launch"].strip())
    except Exception:
        return None


def _peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


class Clocks:
    """nvidia-smi clock samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


class NvmlClocks:
    """SM clock and throttle reasons read through NVML every `period_s`
    during the timed region (a short region holds a single 200 ms
    nvidia-smi sample; this one holds dozens). Reading only: nothing is set."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, uuid, index, period_s=0.01):
        self.uuid, self.index, self.period = uuid, index, period_s
        self.samples, self.mask, self.max_mhz = [], 0, None

    def _open(self):
        import ctypes
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit")
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = L.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok and L.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) != 0:
            raise RuntimeError("nvml handle")
        return L, h

    def _run(self):
        import ctypes
        try:
            L, h = self._open()
        except Exception:
            return
        mhz, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = mx.value
        get_r = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(L, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self.stop:
            if L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if get_r(h, ctypes.byref(rs)) == 0:
                self.mask |= rs.value
            time.sleep(self.period)
        L.nvmlShutdown()

    def __enter__(self):
        import threading
        self.stop = False
        self.th = threading.Thread(target=self._run, daemon=True)
        self.th.start()
        return self

    def __exit__(self, *a):
        self.stop = True
        self.th.join(timeout=5)

    def summary(self):
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples),
                "reasons": sorted(n for b, n in self.REASONS.items() if self.mask & b)}


def cpu_model():
    """The host CPU's model name (lscpu; /proc/cpuinfo as a fallback)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for l in out.splitlines():
            if l.lower().startswith("model name"):
                return l.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for l in open("/proc/cpuinfo"):
            if l.lower().startswith("model name"):
                return l.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def time_oracle_one_core(rows, budget_s):
    """The oracle on one host core: a child process with every BLAS pool
    limited to one thread before numpy loads. Returns (64-row frame
    equivalents per second, frames, seconds) or None."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1", NUMEXPR_NUM_THREADS="1")
    code = ("import json,sys; sys.path.insert(0, %r); import bench, synth; s = synth.shape('full'); "
            "print(json.dumps(bench.time_oracle(s, synth.weights(s, 0), %d, %f)))" % (ROOT, rows, budget_s))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=budget_s * 6 + 120)
        return tuple(json.loads(r.stdout.strip().splitlines()[-1]))
    except Exception:
        return None


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return n
    except Exception:
        pass
    return os.cpu_count()


def time_oracle(s, w, rows, budget_s):
    """Run the oracle frame on `rows` rows until about budget_s seconds pass.
    Returns (64-row frame equivalents per second, frames run, seconds)."""
    import oracle
    import synth
    from oracle.frame import Weights
    W = Weights(w)
    samp = synth.sampler("fixed", rows, 0)
    t0 = time.perf_counter()
    n = 0
    while True:
        h = synth.talker_hidden(s, rows, 0, frame=n)
        c0 = synth.first_codes(s, rows, 0)
        oracle.run_frame(s, W, h, c0, samp, "fp64")
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 50:
            return (n * rows / ROWS) / el, n, el


def _clocks(smi, nvml, ms):
    """The clock record of the timed region: NVML's 10 ms samples when there
    are any (nvidia-smi's 200 ms ones otherwise, and always beside them), plus
    time x median SM clock, which compares runs taken at different clocks."""
    best = nvml if nvml.get("samples") else smi
    out = dict(best)
    out["source"] = "nvml_10ms" if best is nvml else "nvidia-smi_200ms"
    out["reasons"] = sorted(set(smi.get("reasons", [])) | set(nvml.get("reasons", [])))
    out["nvidia_smi"] = smi
    if out.get("sm_mhz"):
        out["us_x_mhz_per_frame"] = ms * 1e3 * out["sm_mhz"]
    return out


def _traced(cp, s, w, local, args, run, R, keep):
    """The per-task trace of one frame (third of three) on a traced handle."""
    import torch
    from persistent_megakernel_streaming_gb300 import torch_io
    ft = cp.Frame(s, torch_io.weights_to_torch(w), device=local, cluster=args.cluster, trace=True)
    keep.append(ft)
    run(ft.frame, R, 3, 0)
    tr = torch.zeros((ft.info.tasks, 16), dtype=torch.int64, device="cuda")
    ft.trace(tr)
    torch.cuda.synchronize()
    return tr.cpu().numpy()


def max_over_ranks(ms, dist):
    """The slowest rank's time: the job ends with it (`dist` None: one process)."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores: each step one oracle frame
    over a row sample sized so the whole run stays within a few minutes."""
    if rank != 0:
        return
    import oracle  # noqa: F401
    import synth
    s = synth.shape("full")
    w = synth.weights(s, 0)
    from oracle.frame import Weights
    W = Weights(w)
    # calibrate one row-frame, then size the per-step sample
    rows = 1
    t = time.perf_counter()
    import oracle as orc
    orc.run_frame(s, W, synth.talker_hidden(s, 1, 0), synth.first_codes(s, 1, 0), synth.sampler("fixed", 1, 0))
    per_row = time.perf_counter() - t
    budget = 150.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(ROWS, budget / max(per_row, 1e-3))))
    samp = synth.sampler("fixed", rows, 0)
    for i in range(args.warmup):
        orc.run_frame(s, W, synth.talker_hidden(s, rows, 0, i), synth.first_codes(s, rows, 0), samp)
    t0 = time.perf_counter()
    for i in range(args.steps):
        orc.run_frame(s, W, synth.talker_hidden(s, rows, 0, 100 + i), synth.first_codes(s, rows, 0), samp)
    el = time.perf_counter() - t0
    value = (args.steps * rows / ROWS) / el
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "rows": ROWS, "rows_timed_per_step": rows,
                       "row_sample": f"each step times {rows} of the 64 rows (the oracle's rows are "
                                     f"independent) and scales to 64-row frames"},
            "cpu_baseline": {"value": value, "unit": "frames/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"each step one float64 oracle frame over {rows} of the 64 rows; "
                                       f"value scaled to 64-row frames"},
            "e2e": {"value": value, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle timing")
    ap.add_argument("--no-sweep", action="store_true", help="skip the row sweep")
    ap.add_argument("--cluster", type=int, default=0)
    ap.add_argument("--profile", action="store_true",
                    help="only warm-up plus `steps` chained cp_frame calls (for ncu captures)")
    ap.add_argument("--profile-split", action="store_true",
                    help="with --profile: run cp_frame_split instead")
    ap.add_argument("--quick", action="store_true",
                    help="skip the per-task traces, the cut compositions and the 2x-wide shape "
                         "(by default they run)")
    ap.add_argument("--trace", action="store_true", help="add the per-task timestamp breakdown")
    ap.add_argument("--trace128", action="store_true",
                    help="add the per-task breakdown of a 128-row frame (a 128-row handle)")
    ap.add_argument("--cuts", action="store_true", help="time per-layer and attention/MLP kernel cuts")
    ap.add_argument("--wide", action="store_true", help="time the 2x-wide shape")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if not args.quick:  # the default run carries every measurement
        args.trace = args.trace128 = args.cuts = args.wide = True

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
        if dist:
            dist.barrier()
        return

    import torch
    import synth
    from persistent_megakernel_streaming_gb300 import build, cp, torch_io
    build.build()
    torch.cuda.set_device(local)
    s = synth.shape("full")
    w = synth.weights(s, 0)
    fr = cp.Frame(s, torch_io.weights_to_torch(w), device=local, cluster=args.cluster)
    P, R = s["positions"], ROWS
    stream = torch.cuda.Stream()
    nfr = args.steps + args.warmup
    hs = torch.from_numpy(np.stack([synth.talker_hidden(s, R, 0, frame=f) for f in range(nfr)])).cuda()
    c0 = torch.from_numpy(synth.first_codes(s, R, 0)).cuda()
    samp_np = synth.sampler("fixed", R, 0)
    samp = torch_io.sampler_to_torch(samp_np)
    codes = torch.zeros((nfr + 1, R, P - 1), dtype=torch.int32, device="cuda")
    firsts = torch.zeros((nfr + 1, R), dtype=torch.int32, device="cuda")  # contiguous first codes

    def run(fn, rows, n, first, sampler=None):
        """n chained frames starting at step `first` (each frame's first code
        is the previous frame's last code, offsets carried); returns device ms
        per frame."""
        sp = samp if sampler is None else sampler
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            cc = c0[:rows]
            ev0.record(stream)
            for i in range(n):
                f = (first + i) % nfr
                fn(hs[f, :rows], cc, {k: v[:rows] for k, v in sp.items()}, rows, codes[f + 1, :rows],
                   None, stream)
                firsts[f + 1, :rows].copy_(codes[f + 1, :rows, -1])
                cc = firsts[f + 1, :rows]
            ev1.record(stream)
        ev1.synchronize()
        return ev0.elapsed_time(ev1) / n

    if args.profile:
        fn = fr.frame_split if args.profile_split else fr.frame
        run(fn, R, args.warmup, 0)
        run(fn, R, args.steps, args.warmup)
        torch.cuda.synchronize()
        st = fr.status()
        fr.close()
        if st != 0:
            raise RuntimeError(f"frame status {cp.STATUS.get(st, st)}")
        return

    # warm-up (both paths; the split graph is built on its first call)
    run(fr.frame, R, args.warmup, 0)
    run(fr.frame_split, R, args.warmup, 0)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    props = torch.cuda.get_device_properties(local)
    uuid = getattr(props, "uuid", None)
    uuid = f"GPU-{uuid}" if uuid is not None and not str(uuid).startswith("GPU-") else (str(uuid) if uuid else None)
    with Clocks(uuid or local) as clk, NvmlClocks(uuid, local) as nclk:
        ms = run(fr.frame, R, args.steps, args.warmup)
    torch.cuda.synchronize()
    ms = max_over_ranks(ms, dist)
    st = fr.status()
    if st != 0:
        raise RuntimeError(f"frame status {cp.STATUS.get(st, st)}")
    ms_split = run(fr.frame_split, R, args.steps, args.warmup)

    # end to end through the C ABI: host inputs in, codes and offsets out, every step
    pin_h = torch.from_numpy(synth.talker_hidden(s, R, 0, frame=999)).pin_memory()
    pin_c0 = torch.from_numpy(synth.first_codes(s, R, 0)).pin_memory()
    pin_s = {k: v.cpu().pin_memory() for k, v in samp.items()}
    out_codes = torch.empty((R, P - 1), dtype=torch.int32).pin_memory()
    out_off = torch.empty((R,), dtype=torch.int64).pin_memory()
    d_h = torch.empty_like(hs[0])
    d_c0 = torch.empty_like(c0)
    d_s = {k: torch.empty_like(v) for k, v in samp.items()}
    d_codes = torch.empty((R, P - 1), dtype=torch.int32, device="cuda")
    h2d = pin_h.numel() * 4 + pin_c0.numel() * 4 + sum(v.numel() * v.element_size() for v in pin_s.values())
    d2h = out_codes.numel() * 4 + out_off.numel() * 8

    def e2e_step():
        with torch.cuda.stream(stream):
            d_h.copy_(pin_h, non_blocking=True)
            d_c0.copy_(pin_c0, non_blocking=True)
            for k in d_s:
                d_s[k].copy_(pin_s[k], non_blocking=True)
            fr.frame(d_h, d_c0, d_s, R, d_codes, None, stream)
            out_codes.copy_(d_codes, non_blocking=True)
            out_off.copy_(d_s["offset"], non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    stream.synchronize()
    n_e2e = max(3, args.steps // 2)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
        stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / n_e2e

    sweep = None
    if not args.no_sweep:
        # the row sweep: mixed per-row samplers (temperature U[0, 1.2], top-k from
        # {0, 20, 50, 200}, top-p U[0.5, 1], seeds from SplitMix64), 200 chained
        # frames per point, each frame's first code the previous frame's last
        samp_mixed = torch_io.sampler_to_torch(synth.sampler("mixed", R, 0))
        sweep = {"rows": [], "frame_us": [], "split_us": [], "frames_per_point": 200, "sampler": "mixed"}
        for rows in (1, 16, 32, 59, 64):
            sweep["rows"].append(rows)
            sweep["frame_us"].append(round(run(fr.frame, rows, 200, args.warmup, samp_mixed) * 1e3, 2))
            sweep["split_us"].append(round(run(fr.frame_split, rows, 200, args.warmup, samp_mixed) * 1e3, 2))

    sweep128 = None
    if not args.no_sweep:
        # frames of more than 64 rows: a handle built for 128 (M = 128 projections)
        s128 = synth.shape("full_r128")
        f128 = cp.Frame(s128, torch_io.weights_to_torch(w), device=local, cluster=args.cluster)
        hs128 = torch.from_numpy(np.stack([synth.talker_hidden(s, 128, 0, frame=f) for f in range(2)])).cuda()
        c128 = torch.from_numpy(synth.first_codes(s, 128, 0)).cuda()
        samp128 = torch_io.sampler_to_torch(synth.sampler("fixed", 128, 0))
        codes128 = torch.zeros((128, P - 1), dtype=torch.int32, device="cuda")
        sweep128 = {"rows": [], "frame_us": [], "split_us": []}
        nsw = max(5, args.steps // 4)
        for rows in (65, 96, 128):
            us = []
            for fn in (f128.frame, f128.frame_split):
                with torch.cuda.stream(stream):
                    for i in range(args.warmup):
                        fn(hs128[i % 2, :rows], c128[:rows], {k: v[:rows] for k, v in samp128.items()}, rows,
                           codes128[:rows], None, stream)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for i in range(nsw):
                        fn(hs128[i % 2, :rows], c128[:rows], {k: v[:rows] for k, v in samp128.items()}, rows,
                           codes128[:rows], None, stream)
                    e1.record(stream)
                e1.synchronize()
                us.append(round(e0.elapsed_time(e1) / nsw * 1e3, 2))
            sweep128["rows"].append(rows)
            sweep128["frame_us"].append(us[0])
            sweep128["split_us"].append(us[1])
        st128 = f128.status()
        f128.close()
        if st128 != 0:
            raise RuntimeError(f"128-row frame status {cp.STATUS.get(st128, st128)}")
        sweep128["note"] = "a 128-row handle (M = 128 projection tiles); first codes not chained"

    if rank != 0:
        if dist:
            dist.barrier()
        return

    peaks = _peaks()
    hbm = peaks.get("hbm_gbs")
    alg_bytes = fr.info.weight_bytes
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    value = world * 1e3 / ms
    cpu = None
    if not args.no_cpu and world == 1:  # the oracle baseline: rank 0 of a one-process run
        try:
            v, n, el = time_oracle(s, w, ROWS, 12.0)
            cpu = {"value": v, "unit": "frames/s", "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"{n} float64 oracle frame(s) of the same 64-row workload in {el:.1f} s",
                   "cpu_model": cpu_model(), "nproc": os.cpu_count()}
            one = time_oracle_one_core(8, 10.0)
            if one:
                cpu["one_core"] = {"value": one[0], "unit": "frames/s", "cores": 1,
                                   "sample": f"{one[1]} float64 oracle frame(s) over 8 of the 64 rows in "
                                             f"{one[2]:.1f} s, scaled to 64-row frames (BLAS limited to one "
                                             f"thread)"}
        except Exception as e:  # the oracle is a reported baseline, not the product
            cpu = {"value": None, "unit": "frames/s", "cores": cpu_cores(), "kind": "oracle",
                   "sample": f"failed: {e}"}
    line = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows": ROWS, "frames_chained_on_device": True,
                   "l2": "inputs larger than L2: 2.58 GB of weights streamed per frame",
                   "grid": fr.info.grid, "cluster": fr.info.cluster, "parallelism": f"replicas{world}"},
        "us_per_frame": ms * 1e3,
        "row_frames_per_s": value * ROWS,
        "split": {"us_per_frame": ms_split * 1e3, "frames_per_s": 1e3 / ms_split,
                  "speedup_of_cp_frame": ms_split / ms},
        "sweep": sweep,
        "sweep128": sweep128,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": (achieved / hbm) if hbm else None, "traffic": _traffic(),
                     "peak_source": "measured" if hbm else "fallback",
                     "algorithmic_bytes_per_launch": alg_bytes},
        "e2e": {"value": world / e2e_s, "unit": "frames/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": args.steps * 1,
        "clocks": _clocks(clk.summary(), nclk.summary(), ms),
        "cpu_baseline": cpu,
    }
    extra_handles = []
    trace = None
    if args.trace:
        from persistent_megakernel_streaming_gb300 import trace_report
        trace = _traced(cp, s, w, local, args, run, R, extra_handles)
        b = trace_report.breakdown(trace)
        print(trace_report.format_table(b), file=sys.stderr, flush=True)
        line["trace_breakdown"] = b
        line["trace_breakdown"]["mma_stage_split"] = trace_report.mma_stage_split(trace)
        # tensor pipe per projection kind: 2 x weights x rows per phase over the kind's phase spans
        H, F, Hq, Hkv, D, V, T = (s["hidden"], s["ffn"], s["q_heads"], s["kv_heads"], s["head_dim"],
                                  s["vocab"], s["talker_hidden"])
        wts = {"inproj": H * T, "qkv": (Hq + 2 * Hkv) * D * H, "o": H * Hq * D, "gate_up": 2 * F * H,
               "down": H * F, "head": V * H}
        peak_tf = _peaks().get("bf16_tflops") or 1900.0
        line["tensor_pipe_by_kind"] = trace_report.tensor_utilisation(
            trace, {k: 2.0 * v * R for k, v in wts.items()}, peak_tf)
    if args.trace128:
        from persistent_megakernel_streaming_gb300 import trace_report
        s128 = synth.shape("full_r128")
        ft = cp.Frame(s128, torch_io.weights_to_torch(w), device=local, cluster=args.cluster, trace=True)
        extra_handles.append(ft)
        h128 = torch.from_numpy(synth.talker_hidden(s, 128, 0)).cuda()
        c128 = torch.from_numpy(synth.first_codes(s, 128, 0)).cuda()
        samp128 = torch_io.sampler_to_torch(synth.sampler("fixed", 128, 0))
        codes128 = torch.zeros((128, P - 1), dtype=torch.int32, device="cuda")
        for _ in range(3):  # the third frame is the one traced
            ft.frame(h128, c128, samp128, 128, codes128)
        tr = torch.zeros((ft.info.tasks, 16), dtype=torch.int64, device="cuda")
        ft.trace(tr)
        torch.cuda.synchronize()
        if ft.status() != 0:
            raise RuntimeError(f"128-row traced frame status {cp.STATUS.get(ft.status(), ft.status())}")
        b128 = trace_report.breakdown(tr.cpu().numpy())
        print(trace_report.format_table(b128), file=sys.stderr, flush=True)
        line["trace_breakdown_128"] = b128
    if args.cuts:
        # the cut compositions (one launch per layer; attention-phase and
        # MLP-phase launches), each measured and predicted beforehand by the
        # event-graph simulation (simulate.py) from the traced single launch's
        # phase spans and one measured single-cut composition
        from persistent_megakernel_streaming_gb300 import simulate, trace_report
        L, nl = s["layers"], 5
        def first_phase(pos, l):  # input projection, first embedding, then 5 per layer (+ head, draw)
            return 2 + (0 if pos == 0 else nl * L + (pos - 1) * (nl * L + 2)) + nl * l
        per_layer = [first_phase(p_, l) for p_ in range(P) for l in range(L)]
        attn_mlp = sorted(per_layer + [c + 3 for c in per_layer])
        # calibration: one launch per depth position (15 cuts), so the noise of
        # two frame timings is divided by 15 in the per-launch cost
        per_position = [first_phase(p_, 0) for p_ in range(1, P)]
        if trace is None:
            trace = _traced(cp, s, w, local, args, run, R, extra_handles)
        spans = trace_report.phase_spans(trace)
        res = {"frame_us": ms * 1e3, "split_us": ms_split * 1e3}
        for name, cuts in (("per_position", per_position), ("per_layer", per_layer),
                           ("attention_and_mlp", attn_mlp)):
            fc = cp.Frame(s, torch_io.weights_to_torch(w), device=local, cluster=args.cluster, cuts=cuts)
            extra_handles.append(fc)
            run(fc.frame, R, args.warmup, 0)
            res[name + "_us"] = run(fc.frame, R, max(5, args.steps // 2), args.warmup) * 1e3
            res[name + "_launches"] = len(cuts) + 1
        d, scaled = simulate.calibrate_dispatch(spans, per_position, res["per_position_us"], res["frame_us"])
        res["simulate"] = {"dispatch_us_per_launch": d, "calibrated_on": "per_position"}
        for name, cuts in (("per_layer", per_layer), ("attention_and_mlp", attn_mlp)):
            pred = simulate.predict_frame_us(scaled, cuts, d, grid=fr.info.grid)
            res["simulate"][name] = {"predicted_us": pred, "measured_us": res[name + "_us"],
                                     "error_pct": 100.0 * (pred - res[name + "_us"]) / res[name + "_us"]}
        line["cuts"] = res
    if args.wide:
        sw = synth.shape("wide")
        ww = synth.weights(sw, 0)
        fw = cp.Frame(sw, torch_io.weights_to_torch(ww), device=local, cluster=args.cluster)
        extra_handles.append(fw)
        hw = torch.from_numpy(synth.talker_hidden(sw, R, 0)).cuda()
        cw = torch.from_numpy(synth.first_codes(sw, R, 0)).cuda()
        codes_w = torch.zeros((R, sw["positions"] - 1), dtype=torch.int32, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fw.frame(hw, cw, samp, R, codes_w, None, stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            nw = max(5, args.steps // 2)
            e0.record(stream)
            for _ in range(nw):
                fw.frame(hw, cw, samp, R, codes_w, None, stream)
            e1.record(stream)
        e1.synchronize()
        wms = e0.elapsed_time(e1) / nw
        line["wide"] = {"us_per_frame": wms * 1e3, "weight_bytes": fw.info.weight_bytes,
                        "achieved_GBps": fw.info.weight_bytes / (wms * 1e-3) / 1e9, "status": fw.status()}
    print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
    for h_ in extra_handles:
        h_.close()
    fr.close()


if __name__ == "__main__":
    main()
