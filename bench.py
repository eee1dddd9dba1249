#!/usr/bin/env python3
"""Benchmark: one step = fwd + bwd_data + bwd_weight + bwd_bias of the AlexNet-style
2-group convolution (x [128,96,27,27] bf16, w [256,48,5,5], groups 2, pad 2,
stride 1; fp32 outputs), through the C ABI of libgconv: one gconv_step_ex call, which
builds each blocked copy once for all three passes and takes the bias gradient from the
weight gradient's MMAs.  Per-pass times come from events the step records at its pass
boundaries (gconv_debug_set_step_events).

Prints ONE JSON line (rank 0).  `value` is whole-job TFLOP/s with inputs resident
in HBM (3 x 2*N*C_out*Ho*Wo*(C_in/G)*kH*kW FLOP per step over the device time of
the step, CUDA events on the launch stream, L2 flushed between steps outside the
timed events).  `e2e` is the same metric through the host-buffer entry point
gconv_step_host: every step copies the inputs from pinned host memory and the four
outputs back inside the timed region (the library overlaps those copies with the
passes on its own copy streams).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

`--impl reference` times the fp64 CPU oracle (the only reference this project
has) on a bounded sample of the same workload on the host cores.
Multi-GPU (torchrun): every rank runs an independent replica (the path needs no
exchange); the step time is the max over ranks and value sums all ranks' work.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "grouped-conv fwd+bwd TFLOP/s and % roofline on 1 GB300"
WORKLOAD = "alexnet_g2"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def flop_per_pass(geom):
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    from bwd_gconv_fwd_gb300.workloads import out_hw
    Ho, Wo = out_hw(geom)
    return 2.0 * N * Cout * Ho * Wo * (Cin // G) * kH * kW


def algorithmic_bytes(geom, in_bytes=2):
    """Minimum bytes per pass: read inputs once, write fp32 outputs once."""
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    from bwd_gconv_fwd_gb300.workloads import out_hw
    Ho, Wo = out_hw(geom)
    x, y, w = N * Cin * H * W, N * Cout * Ho * Wo, Cout * (Cin // G) * kH * kW
    return {"fwd": x * in_bytes + w * in_bytes + Cout * in_bytes + y * 4,
            "bwd_data": y * in_bytes + w * in_bytes + x * 4,
            "bwd_weight": x * in_bytes + y * in_bytes + w * 4,
            "bwd_bias": y * in_bytes + Cout * 4,
            "bwd_weight_bias": x * in_bytes + y * in_bytes + w * 4 + Cout * 4}


# The sources of the headline step's kernels and their launch planning (the tensor-core
# convolution family and the headers it includes): recorded ncu traffic stays valid while
# these are unchanged.
STEP_SOURCES = ("bwd_gconv_fwd_gb300/csrc/tc_conv.cu", "bwd_gconv_fwd_gb300/csrc/ptx.cuh",
                "bwd_gconv_fwd_gb300/csrc/internal.h", "bwd_gconv_fwd_gb300/csrc/common.cuh", "include/gconv.h")


def _code_only(text):
    """Source text without comments and with whitespace collapsed (comment edits do not
    change a kernel)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in STEP_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            h.update(os.path.basename(rel).encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(pass_name):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(pass_name)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            self.tmpdir = tempfile.mkdtemp(prefix="gconv_clocks_")
            self.path = os.path.join(self.tmpdir, "clocks.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu_index), "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        shutil.rmtree(self.tmpdir, ignore_errors=True)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        smax = max(r[1] for r in rows)
        loaded = [r for r in rows if r[0] > 0.5 * smax] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows)}


def reduce_max(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------

def cpu_oracle_sample(geom, x, w, b, dy, target_s=12.0, max_images=None):
    """Times the oracle (as it stands) on the first n images of the workload, n chosen
    so the four passes take about target_s seconds.  Returns (TFLOP/s, cores, sample text)."""
    import oracle
    import torch
    N = geom[0]
    f64 = lambda t: None if t is None else t.to(torch.float64).numpy()

    def run(n):
        g = (n,) + tuple(geom[1:])
        xs, dys = f64(x[:n]), f64(dy[:n])
        ws, bs = f64(w), f64(b)
        t0 = time.perf_counter()
        oracle.fwd(g, xs, ws, bs)
        oracle.bwd_data(g, dys, ws)
        oracle.bwd_weight(g, xs, dys)
        oracle.bwd_bias(g, dys)
        return time.perf_counter() - t0, 3 * flop_per_pass(g)

    t1, f1 = run(1)
    n = max(1, min(max_images or N, int(target_s / max(t1, 1e-3))))
    if n > 1:
        t1, f1 = run(n)
    return f1 / t1 / 1e12, oracle.max_threads(), f"first {n} of {N} images, all four passes", t1


def bench_reference(args):
    """The reference arm: the fp64 CPU oracle, timed per step on a bounded sample."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from bwd_gconv_fwd_gb300 import workloads as wl
    wk = wl.WORKLOADS[WORKLOAD]
    x, w, b, dy = wl.make_inputs(wk)
    import oracle
    oracle.build()
    # calibrate the per-step sample so K + W steps end within a few minutes
    _, _, _, t_one = cpu_oracle_sample(wk.geom, x, w, b, dy, target_s=0.0, max_images=1)
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = max(1, min(wk.geom[0], int(budget / max(t_one, 1e-3))))
    f64 = lambda t: t.to(torch.float64).numpy()
    g = (n,) + tuple(wk.geom[1:])
    xs, dys, ws, bs = f64(x[:n]), f64(dy[:n]), f64(w), f64(b)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.fwd(g, xs, ws, bs)
        oracle.bwd_data(g, dys, ws)
        oracle.bwd_weight(g, xs, dys)
        oracle.bwd_bias(g, dys)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    step = statistics.mean(times)
    value = 3 * flop_per_pass(g) / step / 1e12
    sample = f"first {n} of {wk.geom[0]} images per step, fwd+bwd_data+bwd_weight+bwd_bias in fp64"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(wk),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_dict(wk):
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = wk.geom
    return {"workload": f"{wk.name}: x[{N},{Cin},{H},{W}] {wk.dtype}, w[{Cout},{Cin // G},{kH},{kW}], groups {G}, "
                        f"stride {s}, pads {pt}/{pb}/{pl}/{pr}, dilation {d}; fp32 outputs",
            "step": "fwd + bwd_data + (bwd_weight + bwd_bias in one call)", "N": N, "C_in": Cin, "H": H, "W": W,
            "C_out": Cout, "kH": kH, "kW": kW, "groups": G, "stride": s, "pads": [pt, pb, pl, pr],
            "dilation": d, "l2": "flushed between steps by a 256 MiB write outside the timed events",
            "parallelism": "replicas"}


def bench_gpu(args):
    import torch
    import bwd_gconv_fwd_gb300 as gc
    from bwd_gconv_fwd_gb300 import binding as B
    from bwd_gconv_fwd_gb300 import workloads as wl

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from bwd_gconv_fwd_gb300 import build
    build.build()

    wk = wl.WORKLOADS[WORKLOAD]
    geom = wk.geom
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    Ho, Wo = wl.out_hw(geom)
    x, w, b, dy = wl.make_inputs(wk)
    xd, wd, bd, dyd = (t.to(dev) for t in (x, w, b, dy))
    y = torch.empty((N, Cout, Ho, Wo), device=dev)
    dx = torch.empty((N, Cin, H, W), device=dev)
    dw = torch.empty(tuple(w.shape), device=dev)
    db = torch.empty((Cout,), device=dev)
    dt = B.GCONV_BF16
    ws_bytes = max(gc.gconv_workspace_size(geom, dt, p) for p in range(4))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    wsp, wsb = ws.data_ptr(), ws.numel()

    # one step = one gconv_step_ex call: y, dx, dw and db (the bias gradient from the weight
    # gradient's own MMAs); the library shares the blocked copies between the passes where it can
    step_ws = gc.gconv_step_workspace_size(geom, dt)
    sws = torch.empty(max(step_ws, 16), dtype=torch.uint8, device=dev)

    def step():
        B.gconv_step_ex_ptr(geom, dt, B.GCONV_F32, xd.data_ptr(), wd.data_ptr(), bd.data_ptr(), dyd.data_ptr(),
                            y.data_ptr(), dx.data_ptr(), dw.data_ptr(), db.data_ptr(), sws.data_ptr(), sws.numel(), sp)

    names = ["fwd", "bwd_data", "bwd_weight_bias"]
    plans = {nm: gc.gconv_plan(geom, dt, p) for p, nm in enumerate(names)}
    shared, launches_per_step = gc.gconv_step_plan(geom, dt)
    pass_launches = {nm: plans[nm][1] for nm in names}
    if shared:
        # the weight gradient reads the other passes' blocked copies
        pass_launches["bwd_weight_bias"] = launches_per_step - pass_launches["fwd"] - pass_launches["bwd_data"]

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert gc.gconv_check_device_error(stream) == B.GCONV_OK

    # the step records these at its pass boundaries (each event recorded once first, so that
    # its handle exists)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    for row in ev:
        for e in row:
            e.record(stream)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    try:
        with ClockSampler(local) as clk:
            wall0 = time.perf_counter()
            for k in range(args.steps):
                flush.zero_()
                B.gconv_debug_set_step_events(ev[k])
                step()
            torch.cuda.synchronize()
            wall = time.perf_counter() - wall0
    finally:
        B.gconv_debug_set_step_events(None)
    if world > 1:
        torch.distributed.barrier()
    assert gc.gconv_check_device_error(stream) == B.GCONV_OK
    # the step's results are the separate passes' results, bit for bit
    ref = {k: torch.empty_like(t) for k, t in (("y", y), ("dx", dx), ("dw", dw), ("db", db))}
    B.gconv_fwd_ptr(geom, dt, xd.data_ptr(), wd.data_ptr(), bd.data_ptr(), ref["y"].data_ptr(), wsp, wsb, sp)
    B.gconv_bwd_data_ptr(geom, dt, dyd.data_ptr(), wd.data_ptr(), ref["dx"].data_ptr(), wsp, wsb, sp)
    B.gconv_bwd_weight_ex_ptr(geom, dt, xd.data_ptr(), dyd.data_ptr(), ref["dw"].data_ptr(), ref["db"].data_ptr(),
                              wsp, wsb, sp)
    torch.cuda.synchronize()
    for k, t in (("y", y), ("dx", dx), ("dw", dw), ("db", db)):
        assert torch.equal(t, ref[k]), f"step {k} differs from the separate passes"
    del ref
    per_pass = {nm: [ev[k][j].elapsed_time(ev[k][j + 1]) for k in range(args.steps)] for j, nm in enumerate(names)}
    step_ms = [ev[k][0].elapsed_time(ev[k][len(names)]) for k in range(args.steps)]
    total_ms = reduce_max(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    fpp = flop_per_pass(geom)
    value = world * 3 * fpp * args.steps / (total_ms * 1e-3) / 1e12

    # ---- end-to-end: pinned host inputs in, four outputs back, every step, through the
    # library's host-buffer entry point (copies on its own streams, overlapped with the passes)
    hx, hw_, hb, hdy = (t.pin_memory() for t in (x, w, b, dy))
    hy, hdx, hdw, hdb = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (y, dx, dw, db))
    h2d = sum(t.numel() * t.element_size() for t in (hx, hw_, hb, hdy))
    d2h = sum(t.numel() * t.element_size() for t in (hy, hdx, hdw, hdb))
    step_bytes = gc.gconv_step_device_bytes(geom, dt, True)
    step_buf = torch.empty(step_bytes, dtype=torch.uint8, device=dev)

    def e2e_step():
        B.gconv_step_host_ptr(geom, dt, hx.data_ptr(), hw_.data_ptr(), hb.data_ptr(), hdy.data_ptr(),
                              hy.data_ptr(), hdx.data_ptr(), hdw.data_ptr(), hdb.data_ptr(),
                              step_buf.data_ptr(), step_bytes, sp)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(3, args.steps // 2)
    if world > 1:
        torch.distributed.barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world)
    e2e_value = world * 3 * fpp * e2e_steps / (e2e_ms * 1e-3) / 1e12
    assert gc.gconv_check_device_error(stream) == B.GCONV_OK
    # the host results are the device passes' results, bit for bit
    for host_t, dev_t in ((hy, y), (hdx, dx), (hdw, dw), (hdb, db)):
        assert torch.equal(host_t, dev_t.cpu()), "host-buffer step disagrees with the device passes"

    launch_bound = time_launch_bound(dev)
    peaks, peak_src = load_peaks()
    configs = None if args.no_configs or world > 1 else bench_configs(dev, peaks, peak_src)

    if world > 1:
        torch.distributed.barrier()
    if rank != 0:
        return 0

    # ---- roofline of the dominant pass ----
    avg = {nm: statistics.mean(v) for nm, v in per_pass.items()}
    dom = max(avg, key=avg.get)
    abytes = algorithmic_bytes(geom)
    hbm = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12
    t_c, t_m = fpp / tc, abytes[dom] / hbm
    if t_c >= t_m:
        bound, ach, peak, unit = "tensor", fpp / (avg[dom] * 1e-3) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    else:
        bound, ach, peak, unit = "hbm", abytes[dom] / (avg[dom] * 1e-3) / 1e9, peaks["hbm_gbs"], "GB/s"
    roof_step_s = sum(max(fpp / tc, abytes[nm] / hbm) for nm in names)
    clocks = clk.summary()

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        v, cores, sample, secs = cpu_oracle_sample(geom, x, w, b, dy, target_s=args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{sample} ({secs:.1f} s, fp64 direct loops, OpenMP)"}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_dict(wk),
        "roofline": {"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
                     "traffic": recorded_traffic(dom), "kernel": f"{dom} ({pass_launches[dom]} launch(es), "
                     f"{gc.PATH_NAMES[plans[dom][0]]})", "peak_source": f"{peak_src} (burst)",
                     "algorithmic": (f"{fpp / 1e9:.2f} GFLOP" if bound == "tensor" else f"{abytes[dom] / 1e6:.1f} MB")
                     + " per launch"},
        "step_roofline_frac": roof_step_s * 1e3 / ms_per_step,
        "step": {"call": "gconv_step_ex", "shared_copies": shared, "launches": launches_per_step},
        "passes": {nm: {"us": avg[nm] * 1e3, "path": gc.PATH_NAMES[plans[nm][0]], "launches": pass_launches[nm],
                        "tflops": fpp / (avg[nm] * 1e-3) / 1e12,
                        "gbs": abytes[nm] / (avg[nm] * 1e-3) / 1e9} for nm in names},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms / e2e_steps},
        "gpu_launches": launches_per_step * args.steps,
        "launch_bound": launch_bound,
        "configs": configs,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def time_launch_bound(dev, reps=200):
    """The launch-bound case (tiny_g5: fp32, groups 5, x [2,100,28,28]): one step of the
    four passes as separate API calls, and the same step captured once in a CUDA graph and
    replayed; microseconds per step for each (inputs resident, L2 warm)."""
    import torch
    import bwd_gconv_fwd_gb300 as gc
    from bwd_gconv_fwd_gb300 import binding as B
    from bwd_gconv_fwd_gb300 import workloads as wl

    wk = wl.WORKLOADS["tiny_g5"]
    geom = wk.geom
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    Ho, Wo = wl.out_hw(geom)
    x, w, b, dy = (t.to(dev) for t in wl.make_inputs(wk))
    y = torch.empty((N, Cout, Ho, Wo), device=dev)
    dx = torch.empty((N, Cin, H, W), device=dev)
    dw = torch.empty(tuple(w.shape), device=dev)
    db = torch.empty((Cout,), device=dev)
    dt = B.GCONV_F32
    wsb = max(16, max(gc.gconv_workspace_size(geom, dt, p) for p in range(4)))
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(dev)
    sp = st.cuda_stream

    def step():
        B.gconv_fwd_ptr(geom, dt, x.data_ptr(), w.data_ptr(), b.data_ptr(), y.data_ptr(), ws.data_ptr(), wsb, sp)
        B.gconv_bwd_data_ptr(geom, dt, dy.data_ptr(), w.data_ptr(), dx.data_ptr(), ws.data_ptr(), wsb, sp)
        B.gconv_bwd_weight_ptr(geom, dt, x.data_ptr(), dy.data_ptr(), dw.data_ptr(), ws.data_ptr(), wsb, sp)
        B.gconv_bwd_bias_ptr(geom, dt, dy.data_ptr(), db.data_ptr(), ws.data_ptr(), wsb, sp)

    for _ in range(5):
        step()
    st.synchronize()
    ref = [t.clone() for t in (y, dx, dw, db)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        step()
    e1.record(st)
    e1.synchronize()
    us_calls = e0.elapsed_time(e1) * 1e3 / reps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        step()
    for _ in range(5):
        graph.replay()
    torch.cuda.synchronize()
    e0.record(st)
    with torch.cuda.stream(st):
        for _ in range(reps):
            graph.replay()
    e1.record(st)
    e1.synchronize()
    us_graph = e0.elapsed_time(e1) * 1e3 / reps
    assert all(torch.equal(a, c) for a, c in zip(ref, (y, dx, dw, db))), "graph replay disagrees with the calls"
    assert gc.gconv_check_device_error(st) == B.GCONV_OK
    return {"workload": "tiny_g5: x[2,100,28,28] fp32, w[15,20,3,3], groups 5", "us_per_step_calls": us_calls,
            "us_per_step_graph": us_graph, "launches_per_step": sum(gc.gconv_plan(geom, dt, p)[1] for p in range(4))}


FP32_FMA_PER_SM_CLK = 128          # FP32 FMA lanes per SM per clock (4 SMSPs x 32)


def fp32_peak_tflops(peaks):
    """FP32 FMA peak of the CUDA-core kernels: SMs x 128 FMA lanes x 2 FLOP x max SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * FP32_FMA_PER_SM_CLK * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12


def time_workload(wk, dev, reps, warmup, flush, peaks, only=None):
    """Per-pass timing of one workload: CUDA events on the current stream around each call, L2
    flushed before every call, median of `reps` after `warmup`.  Returns the passes' records,
    and the one-call step (gconv_step_ex: y, dx, dw and db) as "step".  `only`: names of the
    calls to time (default all)."""
    import torch
    import bwd_gconv_fwd_gb300 as gc
    from bwd_gconv_fwd_gb300 import binding as B
    from bwd_gconv_fwd_gb300 import workloads as wl
    geom = wk.geom
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    Ho, Wo = wl.out_hw(geom)
    st = torch.cuda.current_stream(dev)
    sp = st.cuda_stream
    dt = B.GCONV_BF16 if wk.dtype == "bf16" else B.GCONV_F32
    x, w, b, dy = (t.to(dev) for t in wl.make_inputs(wk))
    y = torch.empty((N, Cout, Ho, Wo), device=dev)
    dx = torch.empty((N, Cin, H, W), device=dev)
    dw = torch.empty(tuple(w.shape), device=dev)
    db = torch.empty((Cout,), device=dev)
    wsb = max(16, max(gc.gconv_workspace_size(geom, dt, p) for p in range(4)))
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    swsb = max(16, gc.gconv_step_workspace_size(geom, dt))
    sws = torch.empty(swsb, dtype=torch.uint8, device=dev)
    calls = {
        "fwd": lambda: B.gconv_fwd_ptr(geom, dt, x.data_ptr(), w.data_ptr(), b.data_ptr(), y.data_ptr(), ws.data_ptr(), wsb, sp),
        "bwd_data": lambda: B.gconv_bwd_data_ptr(geom, dt, dy.data_ptr(), w.data_ptr(), dx.data_ptr(), ws.data_ptr(), wsb, sp),
        "bwd_weight": lambda: B.gconv_bwd_weight_ptr(geom, dt, x.data_ptr(), dy.data_ptr(), dw.data_ptr(), ws.data_ptr(), wsb, sp),
        "bwd_bias": lambda: B.gconv_bwd_bias_ptr(geom, dt, dy.data_ptr(), db.data_ptr(), ws.data_ptr(), wsb, sp),
        "bwd_weight_bias": lambda: B.gconv_bwd_weight_ex_ptr(geom, dt, x.data_ptr(), dy.data_ptr(), dw.data_ptr(),
                                                             db.data_ptr(), ws.data_ptr(), wsb, sp),
        "step": lambda: B.gconv_step_ex_ptr(geom, dt, B.GCONV_F32, x.data_ptr(), w.data_ptr(), b.data_ptr(),
                                            dy.data_ptr(), y.data_ptr(), dx.data_ptr(), dw.data_ptr(), db.data_ptr(),
                                            sws.data_ptr(), swsb, sp),
    }
    if only:
        calls = {k: v for k, v in calls.items() if k in only}
    pass_code = {"fwd": 0, "bwd_data": 1, "bwd_weight": 2, "bwd_bias": 3, "bwd_weight_bias": 2}
    in_bytes = 2 if wk.dtype == "bf16" else 4
    fpp = flop_per_pass(geom)
    abytes = algorithmic_bytes(geom, in_bytes)
    hbm = peaks["hbm_gbs"] * 1e9
    out = {}
    step_rec = None
    for nm, f in calls.items():
        times = []
        for k in range(warmup + reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            f()
            e1.record(st)
            e1.synchronize()
            if k >= warmup:
                times.append(e0.elapsed_time(e1) * 1e-3)
        t = statistics.median(times)
        if nm == "step":
            shared, launches = gc.gconv_step_plan(geom, dt)
            step_rec = {"us": t * 1e6, "shared_copies": shared, "launches": launches,
                        "tflops": 3 * fpp / t / 1e12}
            continue
        path, launches = gc.gconv_plan(geom, dt, pass_code[nm])
        pname = gc.PATH_NAMES[path]
        t_mem = abytes[nm] / hbm
        if nm == "bwd_bias":
            t_cmp, unit_peak = 0.0, None
        elif pname.startswith("tc_"):
            t_cmp, unit_peak = fpp / (peaks["bf16_tflops"] * 1e12), "bf16 tensor (measured burst)"
        else:
            t_cmp, unit_peak = fpp / (fp32_peak_tflops(peaks) * 1e12), "fp32 FMA (derived)"
        out[nm] = {"us": t * 1e6, "path": pname, "launches": launches,
                   "tflops": (fpp / t / 1e12) if nm != "bwd_bias" else None,
                   "gbs": abytes[nm] / t / 1e9, "hbm_frac": abytes[nm] / t / hbm,
                   "bound": "hbm" if t_mem >= t_cmp else ("tensor" if unit_peak.startswith("bf16") else "fp32"),
                   "roofline_us": max(t_mem, t_cmp) * 1e6, "roofline_frac": max(t_mem, t_cmp) / t}
    assert gc.gconv_check_device_error(st) == B.GCONV_OK
    rec = {"passes": out, "gflop_per_pass": fpp / 1e9}
    step = ("fwd", "bwd_data", "bwd_weight_bias")      # the step's passes (weight and bias gradients in one)
    if all(k in out for k in step):
        roof_us = sum(out[k]["roofline_us"] for k in step)
        rec["passes_sum_us"] = sum(out[k]["us"] for k in step)
        if step_rec:
            step_rec["roofline_frac"] = roof_us / step_rec["us"]
    if step_rec:
        rec["step"] = step_rec
    return rec


# The other configurations of the metric, each timed pass by pass (c1 also as a graph, in
# `launch_bound`); the headline line times the AlexNet-style layer.
CONFIGS = [("c1", "tiny_g5"), ("c3", "fc_mode"), ("c3_ones", "fc_mode_ones_x"), ("c4", "dense3x3"),
           ("c4b", "dense3x3_s2_asym"), ("c5", "resnext_g32"), ("c5b", "depthwise")]


def bench_configs(dev, peaks, peak_src, reps=10, warmup=3):
    import torch
    from bwd_gconv_fwd_gb300 import workloads as wl
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    out = {}
    for key, name in CONFIGS:
        wk = wl.WORKLOADS[name]
        rec = time_workload(wk, dev, reps, warmup, flush, peaks)
        rec["workload"] = config_dict(wk)["workload"]
        out[key] = rec
        torch.cuda.empty_cache()
    out["_timing"] = (f"per pass: median of {reps} calls after {warmup} warm-up calls, CUDA events on the "
                      f"launch stream, L2 flushed by a 256 MiB write before every call; roofline per pass = "
                      f"max(algorithmic bytes / HBM, FLOP / peak of the unit the path uses); peaks {peak_src}")
    return out


def bench_sweep(args):
    """--sweep: per-pass timing of the model-zoo layer sweep (ResNeXt-50 32x4d grouped 3x3,
    MobileNet-v2 depthwise 3x3) at batch 32; one JSON line per layer.  CUDA events on one
    stream, L2 flushed before each pass, median of --steps repetitions after --warmup."""
    import torch
    from bwd_gconv_fwd_gb300 import workloads as wl
    from bwd_gconv_fwd_gb300 import build
    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    layers = dict(wl.model_zoo(32))
    layers.update(wl.pointwise_zoo(32))
    only = set(args.passes.split(",")) if args.passes else None
    for name, wk in layers.items():
        rec = time_workload(wk, dev, args.steps, args.warmup, flush, peaks, only)
        print(json.dumps({"sweep": name, "geom": list(wk.geom), "gflop_per_pass": rec["gflop_per_pass"],
                          "passes": rec["passes"], "step": rec.get("step"), "peak_source": peak_src}), flush=True)
    return 0


def bench_one_workload(args):
    """--workload NAME: per-pass timing of one named workload (the command the kernel profiles
    run under ncu); one JSON line.  --warmup may be 0 here, so that each pass launches once."""
    import torch
    from bwd_gconv_fwd_gb300 import workloads as wl
    from bwd_gconv_fwd_gb300 import build
    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks, peak_src = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    zoo = dict(wl.model_zoo(32))
    zoo.update(wl.pointwise_zoo(32))
    wk = wl.WORKLOADS[args.workload] if args.workload in wl.WORKLOADS else zoo[args.workload]
    only = set(args.passes.split(",")) if args.passes else None
    rec = time_workload(wk, dev, args.steps, args.warmup, flush, peaks, only)
    rec["workload"] = config_dict(wk)["workload"]
    rec["peak_source"] = peak_src
    print(json.dumps(rec), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gconv", choices=["gconv", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config pass timings")
    ap.add_argument("--sweep", action="store_true", help="time the model-zoo layer sweep instead")
    ap.add_argument("--workload", default=None, help="time the passes of one named workload only")
    ap.add_argument("--passes", default=None,
                    help="with --workload: comma list of calls to time (fwd, bwd_data, bwd_weight, bwd_bias, "
                         "bwd_weight_bias, step)")
    args = ap.parse_args()
    if args.workload:
        return bench_one_workload(args)
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps, whatever is asked
    if args.impl == "reference":
        return bench_reference(args)
    if args.sweep:
        return bench_sweep(args)
    return bench_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
