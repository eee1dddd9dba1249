"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.

Tolerances (per output tensor): max |gpu - oracle| <= 1e-2 * RMS(oracle) for
bf16 inputs with fp32 accumulation, <= 1e-4 * RMS(oracle) for fp32 inputs on
the CUDA-core path.  Shapes, untouched-pixel zeros and the all-ones
fully-connected script are checked bit-exactly.  Small geometries are compared
element by element over whole tensors; the full-size workloads, in the launch
configuration the benchmark uses, on sampled elements the oracle computes one by
one (RMS taken over the same sample).
"""
import numpy as np
import pytest
import torch

import bwd_gconv_fwd_gb300 as gc
from bwd_gconv_fwd_gb300 import binding as B
from bwd_gconv_fwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "f32": 1e-4}


@pytest.fixture(scope="module")
def dev(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_gconv_fwd_gb300 import build
    build.build()
    gc.binding.gconv_debug_force_path(B.PATH_NONE)
    return torch.device("cuda:0")


def _kw(geom):
    N, Cin, H, W, Cout, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, G = wl.per_axis(geom)
    return dict(stride=(sh, sw), padding=(pt, pb, pl, pr), dilation=(dh, dw), groups=G)


# Guard regions around every output: 4 KiB of a NaN bit pattern no kernel computes, checked
# untouched after the call (a substitute for a memory checker, which this pool does not run).
GUARD = 1024
CANARY = 0x7FC0DEAD


def guarded(shape, dev):
    """An fp32 output of `shape` (NaN-filled, so unwritten elements show) inside a buffer whose
    GUARD elements before and after hold CANARY; returns (output view, buffer)."""
    n = 1
    for v in shape:
        n *= int(v)
    buf = torch.full((GUARD + n + GUARD,), float("nan"), device=dev)
    buf.view(torch.int32)[:GUARD] = CANARY
    buf.view(torch.int32)[GUARD + n:] = CANARY
    return buf[GUARD:GUARD + n].view(shape), buf


def check_guards(name, buf):
    words = buf.view(torch.int32)
    n = buf.numel() - 2 * GUARD
    assert bool((words[:GUARD] == CANARY).all()), f"{name}: write before the output"
    assert bool((words[GUARD + n:] == CANARY).all()), f"{name}: write past the output"


def run_gpu(geom, x, w, b, dy, dev, passes=("y", "dx", "dw", "db"), fused_bias=False):
    """All four passes on the GPU; returns fp32 CPU tensors.  Every output sits between guard
    regions that must come back untouched.  fused_bias: db from the weight-gradient call."""
    N, Cin, H, W, Cout, kH, kW = wl.per_axis(geom)[:7]
    Ho, Wo = wl.out_hw(geom)
    kw = _kw(geom)
    xd, wd, dyd = x.to(dev), w.to(dev), dy.to(dev)
    bd = None if b is None else b.to(dev)
    out, bufs = {}, {}
    if "y" in passes:
        y, bufs["y"] = guarded((N, Cout, Ho, Wo), dev)
        gc.gconv_fwd(xd, wd, bd, y, **kw)
        out["y"] = y
    if "dx" in passes:
        dx, bufs["dx"] = guarded((N, Cin, H, W), dev)
        gc.gconv_bwd_data(dyd, wd, dx, **kw)
        out["dx"] = dx
    if "db" in passes:
        db, bufs["db"] = guarded((Cout,), dev)
        if not fused_bias:
            gc.gconv_bwd_bias(dyd, db, geom=geom)
        out["db"] = db
    if "dw" in passes:
        dw, bufs["dw"] = guarded(tuple(w.shape), dev)
        gc.gconv_bwd_weight(xd, dyd, dw, db=out["db"] if fused_bias else None, **kw)
        out["dw"] = dw
    torch.cuda.synchronize()
    assert gc.gconv_check_device_error() == B.GCONV_OK
    for k, bf in bufs.items():
        check_guards(f"{geom} {k}", bf)
    return {k: v.cpu() for k, v in out.items()}


def assert_paths(geom, dtype, expect):
    """The pass families the planner picks, as the test expects them (fwd, bwd_data,
    bwd_weight, bwd_bias path codes)."""
    dt = B.GCONV_BF16 if dtype == "bf16" else B.GCONV_F32
    got = tuple(gc.gconv_plan(geom, dt, p)[0] for p in range(4))
    assert got == tuple(expect), (geom, [B.PATH_NAMES[v] for v in got], [B.PATH_NAMES[v] for v in expect])


def f64(t):
    return None if t is None else t.to(torch.float64).numpy()


def check(name, got, ref, tol):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    assert err <= tol * rms + 1e-30, f"{name}: max err {err:.3e} > {tol:g} * rms {rms:.3e}"
    return err / rms if rms else 0.0


def full_compare(geom, dtype, x, w, b, dy, dev, oracle_mod, label=""):
    got = run_gpu(geom, x, w, b, dy, dev)
    tol = TOL[dtype]
    check(f"{label} y", got["y"].numpy(), oracle_mod.fwd(geom, f64(x), f64(w), f64(b)), tol)
    check(f"{label} dx", got["dx"].numpy(), oracle_mod.bwd_data(geom, f64(dy), f64(w)), tol)
    check(f"{label} dw", got["dw"].numpy(), oracle_mod.bwd_weight(geom, f64(x), f64(dy)), tol)
    check(f"{label} db", got["db"].numpy(), oracle_mod.bwd_bias(geom, f64(dy)), tol)
    return got


SMALL = [
    # (N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G)
    (2, 32, 14, 13, 64, 3, 3, 1, 1, 0, 2, 1, 1, 2),
    (3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2),       # AlexNet-like, ragged
    (2, 64, 17, 15, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1),
    (2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1),         # stride 2, asymmetric pads
    (2, 16, 9, 9, 16, 3, 3, 1, 2, 2, 2, 2, 2, 1),           # dilation 2
    (1, 40, 7, 23, 24, 2, 4, 1, 0, 3, 1, 0, 1, 1),          # odd channel counts
    (2, 128, 6, 6, 96, 6, 6, 1, 0, 0, 0, 0, 1, 1),          # input == kernel (FC mode)
    (2, 32, 12, 12, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8),         # 4 channels per group
    (2, 16, 10, 10, 16, 3, 3, 1, 1, 1, 1, 1, 1, 16),        # depthwise
    (1, 8, 9, 7, 12, 1, 1, 1, 0, 0, 0, 0, 1, 1),            # 1x1
    (1, 16, 8, 8, 16, 2, 2, 3, 0, 0, 0, 0, 1, 1),           # stride > kernel
    (2, 256, 9, 9, 256, 3, 3, 1, 1, 1, 1, 1, 1, 1),         # several channel tiles
    (1, 96, 13, 40, 160, 3, 3, 1, 1, 1, 1, 1, 1, 2),        # wide rows, Cout/G = 80
]


@pytest.mark.parametrize("geom", SMALL)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_small_geometries_full(dev, oracle_mod, geom, dtype):
    wk = wl.Workload("small", geom, dtype, w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 7 + (dtype == "f32"))
    full_compare(geom, dtype, x, w, b, dy, dev, oracle_mod, label=str(geom))


def test_random_sweep(dev, oracle_mod):
    rng = np.random.default_rng(1234)
    for i in range(40):
        geom = wl.random_geometry(rng, max_n=3, max_c=40, max_hw=15, max_k=4)
        dtype = "bf16" if i % 3 else "f32"
        wk = wl.Workload("sweep", geom, dtype, w=("normal", 0.3))
        x, w, b, dy = wl.make_inputs(wk, seed=5000 + i)
        full_compare(geom, dtype, x, w, b, dy, dev, oracle_mod, label=f"sweep{i} {geom}")


def test_random_sweep_tensor_core(dev, oracle_mod):
    """Random bf16 geometries that the planner sends to the tensor-core correlation and
    weight-gradient kernels on all three contraction passes (at least 16 channels a group on
    each side, kernels up to 5 x 5, stride and dilation up to 2, asymmetric pads), compared
    over whole tensors; most of the generated cases must reach that family."""
    rng = np.random.default_rng(4321)
    ran = 0
    for i in range(32):
        G = int(rng.choice([1, 1, 2, 3]))
        cgi, cgo = int(rng.integers(16, 65)), int(rng.integers(16, 97))
        kH, kW = int(rng.integers(1, 6)), int(rng.integers(1, 6))
        s, d = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        pads = [int(v) for v in rng.integers(0, 3, size=4)]
        geom = (int(rng.integers(1, 4)), cgi * G, int(rng.integers(6, 17)), int(rng.integers(6, 17)), cgo * G,
                kH, kW, s, *pads, d, G)
        ho, wo = wl.out_hw(geom)
        if ho < 1 or wo < 1:
            continue
        if any(gc.gconv_plan(geom, B.GCONV_BF16, p)[0] != B.PATH_TC_IGEMM for p in range(3)):
            continue
        wk = wl.Workload("tcsweep", geom, "bf16", w=("normal", 0.2))
        x, w, b, dy = wl.make_inputs(wk, seed=7000 + i)
        full_compare(geom, "bf16", x, w, b, dy, dev, oracle_mod, label=f"tcsweep{i} {geom}")
        ran += 1
    assert ran >= 20, ran


def test_tiny_g5_full(dev, oracle_mod):
    """The NNlib.jl groups=5 example at its own size, fp32, whole tensors at 1e-4."""
    wk = wl.WORKLOADS["tiny_g5"]
    x, w, b, dy = wl.make_inputs(wk)
    full_compare(wk.geom, wk.dtype, x, w, b, dy, dev, oracle_mod, label="tiny_g5")


def _sampled(wk, dev, oracle_mod, n_out=6000, n_w=1500, seed=77):
    x, w, b, dy = wl.make_inputs(wk)
    geom = wk.geom
    got = run_gpu(geom, x, w, b, dy, dev)
    rng = np.random.default_rng(seed)
    tol = TOL[wk.dtype]
    X, Wt, Bt, DY = f64(x), f64(w), f64(b), f64(dy)
    iy = rng.choice(got["y"].numel(), min(n_out, got["y"].numel()), replace=False)
    check(f"{wk.name} y", got["y"].numpy().ravel()[iy], oracle_mod.fwd_points(geom, X, Wt, Bt, iy), tol)
    ix = rng.choice(got["dx"].numel(), min(n_out, got["dx"].numel()), replace=False)
    check(f"{wk.name} dx", got["dx"].numpy().ravel()[ix], oracle_mod.bwd_data_points(geom, DY, Wt, ix), tol)
    iw = rng.choice(got["dw"].numel(), min(n_w, got["dw"].numel()), replace=False)
    check(f"{wk.name} dw", got["dw"].numpy().ravel()[iw], oracle_mod.bwd_weight_points(geom, X, DY, iw), tol)
    check(f"{wk.name} db", got["db"].numpy(), oracle_mod.bwd_bias(geom, DY), tol)
    return got


TC, FC, CC, RD, PW = B.PATH_TC_IGEMM, B.PATH_TC_FC, B.PATH_DIRECT, B.PATH_REDUCE, B.PATH_TC_GEMM
WORKLOAD_PATHS = {
    "alexnet_g2": (TC, TC, TC, RD), "fc_mode": (FC, FC, FC, RD), "fc_mode_ones_x": (FC, FC, FC, RD),
    "dense3x3": (TC, TC, TC, RD), "dense3x3_s2_asym": (TC, TC, TC, RD),
    "resnext_g32": (CC, CC, CC, RD), "depthwise": (CC, CC, CC, RD),
}


@pytest.mark.parametrize("name", ["alexnet_g2", "fc_mode", "fc_mode_ones_x", "dense3x3",
                                  "dense3x3_s2_asym", "resnext_g32", "depthwise"])
def test_workload_sampled(dev, oracle_mod, name):
    """The full-size workloads in the benchmark's launch configuration, on the family the
    benchmark times (asserted), against the oracle on sampled outputs."""
    assert_paths(wl.WORKLOADS[name].geom, wl.WORKLOADS[name].dtype, WORKLOAD_PATHS[name])
    got = _sampled(wl.WORKLOADS[name], dev, oracle_mod)
    if name == "fc_mode_ones_x":
        # x = 1: every image gives the same y row; gradOutput = 1: every dx row is the same
        y = got["y"].reshape(1600, 4096)
        assert torch.equal(y, y[:1].expand_as(y))
        dx = got["dx"].reshape(1600, -1)
        assert torch.equal(dx, dx[:1].expand_as(dx))


def test_fc_all_ones_script_exact(dev):
    """The all-ones script of cudnn.torch issue #118 at its size: every value is an
    exactly representable integer, so the GPU must match bit for bit."""
    wk = wl.WORKLOADS["fc_mode_all_ones"]
    assert_paths(wk.geom, wk.dtype, (FC, FC, FC, RD))
    x, w, b, dy = wl.make_inputs(wk)
    got = run_gpu(wk.geom, x, w, b, dy, dev)
    assert torch.all(got["y"] == 256 * 6 * 6 + 1)
    assert torch.all(got["dx"] == 4096)
    assert torch.all(got["dw"] == 1600)
    assert torch.all(got["db"] == 1600)


def test_untouched_pixels_exact_zero(dev):
    geom = (2, 16, 11, 11, 16, 2, 2, 3, 0, 0, 0, 0, 1, 1)
    wk = wl.Workload("gap", geom, "bf16")
    x, w, b, dy = wl.make_inputs(wk, seed=3)
    dx = run_gpu(geom, x, w, b, dy, dev, passes=("dx",))["dx"]
    assert torch.all(dx[:, :, 2::3, :] == 0) and torch.all(dx[:, :, :, 2::3] == 0)


def test_results_are_bitwise_reproducible(dev):
    wk = wl.Workload("rep", (4, 64, 20, 20, 64, 3, 3, 1, 1, 1, 1, 1, 1, 2), "bf16")
    x, w, b, dy = wl.make_inputs(wk, seed=8)
    a = run_gpu(wk.geom, x, w, b, dy, dev)
    c = run_gpu(wk.geom, x, w, b, dy, dev)
    for k in a:
        assert torch.equal(a[k], c[k]), k


def test_outputs_overwritten_not_accumulated(dev, oracle_mod):
    geom = (2, 32, 10, 10, 32, 3, 3, 1, 1, 1, 1, 1, 1, 1)
    wk = wl.Workload("ovw", geom, "bf16")
    x, w, b, dy = wl.make_inputs(wk, seed=9)
    xd, wd, dyd = x.to(dev), w.to(dev), dy.to(dev)
    dw = torch.full(tuple(w.shape), 1e6, device=dev)
    gc.gconv_bwd_weight(xd, dyd, dw, **_kw(geom))
    torch.cuda.synchronize()
    check("dw", dw.cpu().numpy(), oracle_mod.bwd_weight(geom, f64(x), f64(dy)), 1e-2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_empty_batch(dev, dtype):
    """N = 0: nothing to compute for y and dx; dw and db are sums over no terms and come
    back as exact zeros (through every weight-gradient entry point)."""
    geom = (0, 32, 6, 6, 32, 3, 3, 1, 1, 1, 1, 1, 1, 1)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = torch.empty((0, 32, 6, 6), dtype=tdt, device=dev)
    dy = torch.empty((0, 32, 6, 6), dtype=tdt, device=dev)
    w = torch.randn((32, 32, 3, 3), device=dev).to(tdt)
    y = torch.empty((0, 32, 6, 6), device=dev)
    dx = torch.empty((0, 32, 6, 6), device=dev)
    gc.gconv_fwd(x, w, None, y, padding=1)
    gc.gconv_bwd_data(dy, w, dx, padding=1)
    dw = torch.full((32, 32, 3, 3), float("nan"), device=dev)
    gc.gconv_bwd_weight(x, dy, dw, padding=1)
    dw2 = torch.full((32, 32, 3, 3), float("nan"), device=dev)
    gc.binding.gconv_bwd_weight_noalloc(x, dy, dw2, padding=1)
    db = torch.full((32,), float("nan"), device=dev)
    gc.gconv_bwd_bias(dy, db, geom=geom)
    torch.cuda.synchronize()
    assert gc.gconv_check_device_error() == B.GCONV_OK
    for t in (dw, dw2, db):
        assert bool((t == 0).all())


def test_forced_direct_agrees_with_default(dev):
    """The CUDA-core family and whatever the planner picks agree on the same inputs."""
    geom = (3, 64, 15, 14, 128, 3, 3, 1, 1, 1, 1, 1, 1, 2)
    wk = wl.Workload("cross", geom, "bf16", w=("normal", 0.1))
    x, w, b, dy = wl.make_inputs(wk, seed=21)
    auto = run_gpu(geom, x, w, b, dy, dev)
    try:
        gc.binding.gconv_debug_force_path(B.PATH_DIRECT)
        direct = run_gpu(geom, x, w, b, dy, dev)
    finally:
        gc.binding.gconv_debug_force_path(B.PATH_NONE)
    for k in auto:
        r = direct[k].double().numpy()
        check(f"cross {k}", auto[k].numpy(), r, 1e-2)


@pytest.mark.parametrize("geom,dtype,with_bias", [
    ((3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2), "bf16", True),     # tensor-core passes
    ((2, 32, 12, 12, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8), "f32", False),      # CUDA-core passes, no bias
    ((2, 128, 6, 6, 96, 6, 6, 1, 0, 0, 0, 0, 1, 1), "bf16", True),       # FC mode
    ((35, 32, 10, 9, 64, 3, 3, 1, 1, 1, 1, 1, 1, 2), "bf16", True),      # forward in eight batch chunks, ragged
    ((32, 16, 8, 8, 16, 3, 3, 1, 1, 1, 1, 1, 1, 4), "f32", True),        # chunks on the CUDA-core path
    ((36, 3, 7, 7, 8, 3, 3, 1, 0, 0, 0, 0, 1, 1), "bf16", True),         # 294-byte images: chunks would misalign
])
def test_step_host_matches_device_passes(dev, oracle_mod, geom, dtype, with_bias):
    """gconv_step_host on pinned host tensors gives bit for bit what the device passes give
    (the weight gradient with its bias gradient in one call), and meets the oracle
    tolerance; run twice in a row on one stream."""
    wk = wl.Workload("host", geom, dtype)
    x, w, b, dy = wl.make_inputs(wk, seed=31)
    if not with_bias:
        b = None
    ref = run_gpu(geom, x, w, b, dy, dev, fused_bias=True)
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    Ho, Wo = wl.out_hw(geom)
    hx, hw_, hdy = (t.contiguous().pin_memory() for t in (x, w, dy))
    hb = None if b is None else b.contiguous().pin_memory()
    dt = B.GCONV_BF16 if dtype == "bf16" else B.GCONV_F32
    nbytes = gc.gconv_step_device_bytes(geom, dt, with_bias)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream()
    for rep in range(2):
        outs = {"y": torch.full((N, Cout, Ho, Wo), float("nan")).pin_memory(),
                "dx": torch.full((N, Cin, H, W), float("nan")).pin_memory(),
                "dw": torch.full(tuple(w.shape), float("nan")).pin_memory(),
                "db": torch.full((Cout,), float("nan")).pin_memory()}
        gc.gconv_step_host(hx, hw_, hb, hdy, outs["y"], outs["dx"], outs["dw"], outs["db"], buf,
                           stream=stream, **_kw(geom))
        stream.synchronize()
        assert gc.gconv_check_device_error(stream) == B.GCONV_OK
        for k in ref:
            assert torch.equal(outs[k], ref[k]), (rep, k)
    check("host y", outs["y"].numpy(), oracle_mod.fwd(geom, f64(x), f64(w), f64(b)), TOL[dtype])
    check("host db", outs["db"].numpy(), oracle_mod.bwd_bias(geom, f64(dy)), TOL[dtype])


@pytest.mark.parametrize("geom", [
    (2, 256, 14, 14, 256, 3, 3, 2, 1, 1, 1, 1, 1, 1),   # stride 2, two 128-channel tiles in every output phase
    (1, 128, 15, 15, 128, 5, 5, 2, 2, 2, 2, 2, 1, 1),   # stride 2, 5x5: output phases with 9, 6, 6 and 4 taps
])
def test_stride2_tensor_core_wide_full(dev, oracle_mod, geom):
    """Stride-2 layers on the tensor-core kernels (one launch a pass for every phase) over
    whole tensors against the oracle."""
    assert_paths(geom, "bf16", (B.PATH_TC_IGEMM, B.PATH_TC_IGEMM, B.PATH_TC_IGEMM, B.PATH_REDUCE))
    wk = wl.Workload("s2wide", geom, "bf16")
    x, w, b, dy = wl.make_inputs(wk, seed=808)
    full_compare(geom, "bf16", x, w, b, dy, dev, oracle_mod, label="s2 wide")


STEP_EX = [
    # (geometry, dtype, bias, db, output dtype)
    ((3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2), "bf16", True, True, "f32"),     # shared copies, db fused
    ((3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2), "bf16", True, True, "bf16"),    # y and dx as bf16
    ((2, 64, 17, 15, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1), "bf16", True, True, "f32"),      # shared, no spare slot: db apart
    ((2, 16, 9, 9, 16, 3, 3, 1, 2, 2, 2, 2, 2, 1), "bf16", False, False, "f32"),      # shared, dilation 2, no db
    ((2, 96, 10, 12, 64, 3, 3, 1, 0, 2, 2, 0, 1, 1), "bf16", True, True, "f32"),      # shared, one-sided pads
    ((2, 32, 11, 13, 32, 3, 3, 1, 1, 1, 1, 2, 2, 1, 2, 1), "bf16", False, True, "f32"),  # shared, per-axis dilation
    ((2, 32, 14, 13, 64, 3, 3, 1, 1, 0, 2, 1, 1, 2), "bf16", True, True, "f32"),      # passes in turn (widths differ)
    ((2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1), "bf16", True, True, "f32"),      # stride 2: passes in turn
    ((2, 64, 12, 12, 64, 3, 3, 1, 1, 1, 1, 1, 1, 8), "bf16", True, True, "f32"),      # merged groups, shared copies
    ((2, 48, 10, 10, 48, 3, 3, 1, 1, 1, 1, 1, 1, 6), "bf16", True, True, "f32"),      # merged by 6: db fused
    ((2, 48, 10, 10, 48, 3, 3, 1, 1, 1, 1, 1, 1, 6), "bf16", True, True, "bf16"),     # the same, bf16 y and dx
    ((2, 32, 12, 12, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8), "f32", True, True, "f32"),       # CUDA-core passes
    ((0, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2), "bf16", True, True, "f32"),     # empty batch
]


@pytest.mark.parametrize("geom,dtype,with_bias,with_db,out", STEP_EX)
def test_step_ex_matches_device_passes(dev, oracle_mod, geom, dtype, with_bias, with_db, out):
    """gconv_step_ex (y, dx, dw and db from one call, blocked copies shared where the
    tensor-core route allows) gives bit for bit what the separate passes give, twice in a
    row on one workspace, and meets the oracle tolerance."""
    wk = wl.Workload("step", geom, dtype)
    x, w, b, dy = wl.make_inputs(wk, seed=43)
    if not with_bias:
        b = None
    N, Cin, H, W, Cout = wl.per_axis(geom)[:5]
    Ho, Wo = wl.out_hw(geom)
    kw = _kw(geom)
    odt = torch.bfloat16 if out == "bf16" else torch.float32
    xd, wd, dyd = x.to(dev), w.to(dev), dy.to(dev)
    bd = None if b is None else b.to(dev)
    # the separate passes
    ry = torch.empty((N, Cout, Ho, Wo), dtype=odt, device=dev)
    rdx = torch.empty((N, Cin, H, W), dtype=odt, device=dev)
    rdw = torch.empty(tuple(w.shape), device=dev)
    rdb = torch.empty((Cout,), device=dev) if with_db else None
    gc.gconv_fwd(xd, wd, bd, ry, **kw)
    gc.gconv_bwd_data(dyd, wd, rdx, **kw)
    gc.gconv_bwd_weight(xd, dyd, rdw, db=rdb, **kw)
    ws = torch.empty(max(1, gc.gconv_step_workspace_size(B.per_axis(geom), B.GCONV_BF16 if dtype == "bf16"
                                                         else B.GCONV_F32)), dtype=torch.uint8, device=dev)
    for rep in range(2):
        bufs = {}
        if out == "f32":
            y, bufs["y"] = guarded((N, Cout, Ho, Wo), dev)
            dx, bufs["dx"] = guarded((N, Cin, H, W), dev)
        else:
            y = torch.full((N, Cout, Ho, Wo), float("nan"), dtype=odt, device=dev)
            dx = torch.full((N, Cin, H, W), float("nan"), dtype=odt, device=dev)
        dw, bufs["dw"] = guarded(tuple(w.shape), dev)
        db = None
        if with_db:
            db, bufs["db"] = guarded((Cout,), dev)
        gc.gconv_step(xd, wd, bd, dyd, y, dx, dw, db, workspace=ws, **kw)
        torch.cuda.synchronize()
        assert gc.gconv_check_device_error() == B.GCONV_OK
        for k, bf in bufs.items():
            check_guards(f"step {geom} {k}", bf)
        assert torch.equal(y, ry), rep
        assert torch.equal(dx, rdx), rep
        assert torch.equal(dw, rdw), rep
        if with_db:
            assert torch.equal(db, rdb), rep
    tol = TOL[dtype] if out == "f32" else 2e-2
    check("step y", y.float().cpu().numpy(), oracle_mod.fwd(geom, f64(x), f64(w), f64(b)), tol)
    check("step dx", dx.float().cpu().numpy(), oracle_mod.bwd_data(geom, f64(dy), f64(w)), tol)
    check("step dw", dw.cpu().numpy(), oracle_mod.bwd_weight(geom, f64(x), f64(dy)), TOL[dtype])
    if with_db:
        check("step db", db.cpu().numpy(), oracle_mod.bwd_bias(geom, f64(dy)), TOL[dtype])


def test_step_ex_full_size_alexnet_matches_passes(dev):
    """The benchmark's layer at full size: gconv_step_ex on the shared copies equals the
    separate passes bit for bit (the passes meet the oracle in the sampled workload test)."""
    wk = wl.WORKLOADS["alexnet_g2"]
    x, w, b, dy = (t.to(dev) for t in wl.make_inputs(wk, seed=5))
    geom = wk.geom
    N, Cin, H, W, Cout = geom[:5]
    Ho, Wo = wl.out_hw(geom)
    kw = _kw(geom)
    ry, y = (torch.empty((N, Cout, Ho, Wo), device=dev) for _ in range(2))
    rdx, dx = (torch.empty((N, Cin, H, W), device=dev) for _ in range(2))
    rdw, dw = (torch.empty(tuple(w.shape), device=dev) for _ in range(2))
    rdb, db = (torch.empty((Cout,), device=dev) for _ in range(2))
    gc.gconv_fwd(x, w, b, ry, **kw)
    gc.gconv_bwd_data(dy, w, rdx, **kw)
    gc.gconv_bwd_weight(x, dy, rdw, db=rdb, **kw)
    gc.gconv_step(x, w, b, dy, y, dx, dw, db, **kw)
    torch.cuda.synchronize()
    assert gc.gconv_check_device_error() == B.GCONV_OK
    for a, r in ((y, ry), (dx, rdx), (dw, rdw), (db, rdb)):
        assert torch.equal(a, r)


@pytest.mark.parametrize("name", list(wl.model_zoo(2)))
def test_model_zoo_layers_full(dev, oracle_mod, name):
    """The grouped 3x3 layers of ResNeXt-50 (32x4d) and the depthwise 3x3 layers of
    MobileNet-v2 (stride 1 and 2), batch 2, all four passes against the oracle."""
    wk = wl.model_zoo(2)[name]
    x, w, b, dy = wl.make_inputs(wk, seed=41)
    full_compare(wk.geom, "bf16", x, w, b, dy, dev, oracle_mod, label=name)


# Tensor-core edge cases, whole tensors against the oracle, each on the family asserted:
# stride-2 phases that no tap reaches (their dx must be exactly 0), the largest kernels,
# stride with dilation, asymmetric pads at stride 2 on both sides, and the channel counts at
# the edges of the tensor-core thresholds.
TC_EDGES = [
    # geometry, expected (fwd, bwd_data, bwd_weight, bias) families, untouched dx (step, row phase, col phase)
    ((2, 16, 11, 11, 16, 1, 1, 2, 0, 0, 0, 0, 1, 1), (TC, TC, TC, RD), (2, 1, 1)),   # 1x1 stride 2: odd rows, odd cols
    ((2, 32, 12, 13, 32, 2, 2, 2, 0, 0, 0, 0, 1, 1), (TC, TC, TC, RD), None),     # 2x2 stride 2: last column untouched
    ((2, 16, 13, 12, 32, 1, 1, 2, 1, 0, 0, 1, 1, 1), (TC, TC, TC, RD), (2, 0, 1)),   # 1x1 stride 2, pads shift the phase
    ((2, 32, 15, 14, 32, 7, 7, 1, 3, 3, 3, 3, 1, 1), (TC, TC, TC, RD), None),     # 7x7, 49 taps
    ((2, 16, 20, 19, 32, 7, 7, 2, 3, 3, 3, 3, 1, 1), (TC, TC, TC, RD), None),     # 7x7 stride 2
    ((2, 32, 17, 16, 32, 3, 3, 2, 2, 2, 2, 2, 2, 1), (TC, TC, TC, RD), None),     # stride 2 with dilation 2
    ((2, 32, 15, 16, 32, 3, 3, 2, 0, 2, 1, 0, 1, 1), (TC, TC, TC, RD), None),     # stride 2, pads 0/2/1/0
    ((2, 64, 16, 15, 64, 4, 4, 2, 2, 1, 0, 3, 1, 2), (TC, TC, TC, RD), None),     # stride 2, pads 2/1/0/3, groups 2
    ((2, 16, 12, 12, 16, 3, 3, 2, 1, 1, 1, 1, 1, 1), (TC, TC, TC, RD), None),     # 16 channels, stride 2
    ((2, 32, 10, 11, 32, 3, 3, 1, 1, 1, 1, 1, 1, 2), (TC, TC, TC, RD), None),     # 16 channels per group
    ((2, 32, 9, 9, 32, 1, 1, 1, 0, 0, 0, 0, 1, 1), (TC, TC, TC, RD), None),       # 1x1 stride 1
]


def _edge_paths():
    return [(g, p, z) for g, p, z in TC_EDGES]


@pytest.mark.parametrize("geom,paths,untouched", _edge_paths())
def test_tensor_core_edges_full(dev, oracle_mod, geom, paths, untouched):
    assert_paths(geom, "bf16", paths)
    wk = wl.Workload("edge", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 13)
    got = full_compare(geom, "bf16", x, w, b, dy, dev, oracle_mod, label=f"edge {geom}")
    ref_dx = oracle_mod.bwd_data(geom, f64(dy), f64(w))
    zero = ref_dx == 0.0
    # every pixel the oracle leaves at exactly zero (no tap reaches it) is exactly zero here too
    assert np.array_equal(got["dx"].numpy()[zero], np.zeros(int(zero.sum()), np.float32)), geom
    if untouched is not None:
        step, rp, cp = untouched
        assert bool((got["dx"][:, :, rp::step, :] == 0).all()) and bool((got["dx"][:, :, :, cp::step] == 0).all())
        assert int(zero.sum()) > 0


# The thresholds of the tensor-core families: a group with 8 input and 16 output channels
# (forward and weight gradient on the kernels directly, backward-data on two merged groups),
# and the mirror.
THRESHOLDS = [
    ((2, 16, 10, 10, 32, 3, 3, 1, 1, 1, 1, 1, 1, 2), (TC, TC, TC, RD)),
    ((2, 32, 10, 10, 16, 3, 3, 1, 1, 1, 1, 1, 1, 2), (TC, TC, TC, RD)),
]


@pytest.mark.parametrize("geom,paths", THRESHOLDS)
def test_tensor_core_thresholds_full(dev, oracle_mod, geom, paths):
    assert_paths(geom, "bf16", paths)
    wk = wl.Workload("threshold", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 17)
    full_compare(geom, "bf16", x, w, b, dy, dev, oracle_mod, label=f"threshold {geom}")


# Groups too thin for the tensor-core kernels that the thin-plane kernels do not take (8
# channels a side, mixed 8/4 and 8/16, 1x1, stride 2, 5x5): consecutive groups merged into
# one with block-diagonal weights, whole tensors against the oracle.
MERGED = [
    (2, 64, 13, 12, 64, 3, 3, 1, 1, 1, 1, 1, 1, 8),          # 8 a side: all 8 groups as one
    (2, 64, 14, 13, 64, 3, 3, 2, 1, 1, 1, 1, 1, 8),          # stride 2
    (2, 48, 11, 11, 24, 3, 3, 1, 1, 1, 1, 1, 1, 6),          # 8 in, 4 out: 6 groups as one
    (2, 24, 9, 10, 48, 5, 5, 1, 2, 2, 2, 2, 1, 3),           # 8 in, 16 out: backward-data merged
    (2, 64, 9, 9, 64, 1, 1, 1, 0, 0, 0, 0, 1, 8),            # 1x1
    (3, 128, 10, 11, 128, 3, 3, 1, 0, 2, 1, 1, 1, 16),       # 2 merged groups, asymmetric pads
]


@pytest.mark.parametrize("geom", MERGED)
def test_merged_groups_full(dev, oracle_mod, geom):
    assert_paths(geom, "bf16", (TC, TC, TC, RD))
    wk = wl.Workload("merged", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 23)
    full_compare(geom, "bf16", x, w, b, dy, dev, oracle_mod, label=f"merged {geom}")


def test_merged_groups_forced_on_thin_layer(dev, oracle_mod):
    """A 4-channel-group layer the thin-plane kernels normally serve, forced onto the
    tensor-core family: 8 groups merged into one of 32 channels."""
    geom = (2, 32, 12, 12, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8)
    assert_paths(geom, "bf16", (CC, CC, CC, RD))
    B.gconv_debug_force_path(B.PATH_TC_IGEMM)
    try:
        assert tuple(gc.gconv_plan(geom, B.GCONV_BF16, p)[0] for p in range(3)) == (TC, TC, TC)
        wk = wl.Workload("merged_forced", geom, "bf16", w=("normal", 0.2))
        x, w, b, dy = wl.make_inputs(wk, seed=97)
        got = run_gpu(geom, x, w, b, dy, dev, passes=("y", "dx", "dw"))
    finally:
        B.gconv_debug_force_path(B.PATH_NONE)
    tol = TOL["bf16"]
    check("forced merged y", got["y"].numpy(), oracle_mod.fwd(geom, f64(x), f64(w), f64(b)), tol)
    check("forced merged dx", got["dx"].numpy(), oracle_mod.bwd_data(geom, f64(dy), f64(w)), tol)
    check("forced merged dw", got["dw"].numpy(), oracle_mod.bwd_weight(geom, f64(x), f64(dy)), tol)


# Per-axis stride and dilation (the 16-integer geometry of the *_ex entry points): whole
# tensors against the oracle, on the families the planner picks (asserted).
PER_AXIS = [
    # (N, C_in, H, W, C_out, kH, kW, s_h, s_w, pt, pb, pl, pr, d_h, d_w, G), dtype, families
    ((2, 32, 13, 12, 32, 3, 3, 2, 1, 1, 1, 1, 1, 1, 1, 1), "bf16", (TC, TC, TC, RD)),
    ((2, 32, 12, 15, 64, 3, 3, 1, 2, 1, 0, 1, 1, 1, 2, 1), "bf16", (TC, TC, TC, RD)),
    ((2, 32, 11, 13, 32, 3, 3, 1, 1, 2, 2, 1, 1, 1, 2, 1), "bf16", (TC, TC, TC, RD)),
    ((2, 32, 12, 9, 64, 3, 5, 1, 1, 1, 1, 2, 2, 2, 1, 2), "bf16", (TC, TC, TC, RD)),
    ((2, 16, 14, 10, 16, 5, 3, 2, 1, 2, 2, 1, 1, 1, 2, 1), "bf16", (TC, TC, TC, RD)),
    ((2, 12, 13, 12, 12, 3, 3, 2, 1, 1, 1, 1, 1, 1, 1, 3), "bf16", (CC, CC, CC, RD)),
    ((2, 8, 11, 14, 8, 3, 2, 1, 3, 0, 2, 1, 0, 2, 1, 8), "bf16", (CC, CC, CC, RD)),
    ((2, 12, 13, 12, 12, 3, 3, 2, 1, 1, 1, 1, 1, 1, 1, 3), "f32", (CC, CC, CC, RD)),
    ((1, 6, 9, 17, 9, 2, 3, 3, 2, 1, 0, 2, 1, 2, 3, 3), "f32", (CC, CC, CC, RD)),
]


@pytest.mark.parametrize("geom,dtype,paths", PER_AXIS)
def test_per_axis_geometries_full(dev, oracle_mod, geom, dtype, paths):
    assert_paths(geom, dtype, paths)
    wk = wl.Workload("axes", geom, dtype, w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 19)
    full_compare(geom, dtype, x, w, b, dy, dev, oracle_mod, label=f"axes {geom}")


def test_per_axis_random_sweep(dev, oracle_mod):
    rng = np.random.default_rng(4321)
    for i in range(30):
        geom = wl.random_geometry(rng, max_n=3, max_c=40, max_hw=15, max_k=4, axes=True)
        dtype = "bf16" if i % 3 else "f32"
        wk = wl.Workload("axes_sweep", geom, dtype, w=("normal", 0.3))
        x, w, b, dy = wl.make_inputs(wk, seed=7000 + i)
        full_compare(geom, dtype, x, w, b, dy, dev, oracle_mod, label=f"axes sweep{i} {geom}")


@pytest.mark.parametrize("geom", [
    (3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2),       # tensor cores: bias column from the MMAs
    (2, 64, 17, 15, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1),         # tensor cores, 64 channels: separate reduction
    (2, 96, 13, 40, 160, 3, 3, 1, 1, 1, 1, 1, 1, 2),        # tensor cores, 48 of 64 channels, 80 outputs
    (2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1),         # stride-2 tensor cores: separate reduction
    (2, 32, 12, 12, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8),         # CUDA-core weight gradient
    (2, 128, 6, 6, 96, 6, 6, 1, 0, 0, 0, 0, 1, 1),          # 1x1 output
    (2, 64, 13, 12, 64, 3, 3, 1, 1, 1, 1, 1, 1, 8),         # merged groups, 64 channels: separate reduction
    (2, 48, 11, 11, 24, 3, 3, 1, 1, 1, 1, 1, 1, 6),         # merged groups, 48 channels: bias column
])
def test_weight_gradient_with_bias_gradient(dev, oracle_mod, geom):
    """gconv_bwd_weight_ex with db: dw and db from one call.  dw equals the separate entry
    point bit for bit; db (summed by the weight-gradient kernels themselves where the
    family fuses it, so in another order) is within tolerance of the oracle."""
    wk = wl.Workload("wdb", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=55)
    sep = run_gpu(geom, x, w, b, dy, dev, passes=("dw", "db"))
    xd, dyd = x.to(dev), dy.to(dev)
    dw, bw = guarded(tuple(w.shape), dev)
    db, bb = guarded((geom[4],), dev)
    gc.gconv_bwd_weight(xd, dyd, dw, db=db, **_kw(geom))
    torch.cuda.synchronize()
    assert gc.gconv_check_device_error() == B.GCONV_OK
    check_guards("fused dw", bw)
    check_guards("fused db", bb)
    assert torch.equal(dw.cpu(), sep["dw"])
    check("fused db", db.cpu().numpy(), oracle_mod.bwd_bias(geom, f64(dy)), TOL["bf16"])


@pytest.mark.parametrize("geom", [
    (3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2),        # AlexNet-like, ragged, bias column
    (2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1),         # stride 2: stride-phase planes, asymmetric pads
    (2, 16, 9, 9, 16, 3, 3, 1, 2, 2, 2, 2, 2, 1),           # dilation 2
    (2, 32, 15, 14, 32, 7, 7, 1, 3, 3, 3, 3, 1, 1),         # 7 x 7: 49 taps in several job groups
    (2, 64, 13, 12, 64, 3, 3, 1, 1, 1, 1, 1, 1, 8),         # merged groups
    (2, 256, 9, 9, 256, 3, 3, 1, 1, 1, 1, 1, 1, 1),         # several channel tiles
])
def test_weight_gradient_cp_async_staging(dev, oracle_mod, geom):
    """The tensor-core weight gradient's cp.async staging (the form it takes when a tensor
    map cannot be encoded) gives the same dw and db as its TMA staging, bit for bit: both
    put the same rows in the same shared-memory layout for the same MMAs."""
    assert gc.gconv_plan(geom, B.GCONV_BF16, B.PASS_BWD_WEIGHT)[0] == B.PATH_TC_IGEMM
    wk = wl.Workload("cpasync", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=61)
    xd, dyd = x.to(dev), dy.to(dev)
    got = {}
    for tma in (True, False):
        B.gconv_debug_set_wgrad_tma(tma)
        try:
            dw, bw = guarded(tuple(w.shape), dev)
            db, bb = guarded((geom[4],), dev)
            gc.gconv_bwd_weight(xd, dyd, dw, db=db, **_kw(geom))
            torch.cuda.synchronize()
            assert gc.gconv_check_device_error() == B.GCONV_OK
        finally:
            B.gconv_debug_set_wgrad_tma(True)
        check_guards(f"dw tma={tma}", bw)
        check_guards(f"db tma={tma}", bb)
        got[tma] = (dw.cpu(), db.cpu())
    check("cp.async dw", got[False][0].numpy(), oracle_mod.bwd_weight(geom, f64(x), f64(dy)), TOL["bf16"])
    check("cp.async db", got[False][1].numpy(), oracle_mod.bwd_bias(geom, f64(dy)), TOL["bf16"])
    assert torch.equal(got[False][0], got[True][0])
    assert torch.equal(got[False][1], got[True][1])


# bf16 outputs (y, dx through the *_ex entry points): the stored value is the fp32 result
# rounded once to nearest even, so it must equal the fp32 output rounded by torch, bit for
# bit; against the oracle the bound adds that rounding, half a bf16 ulp (2^-8 relative).
BF16_OUT = [
    ((3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2), (TC, TC)),    # stride-1 correlation, paired taps
    ((2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1), (TC, TC)),     # stride-2 correlation, phases
    ((2, 128, 6, 6, 96, 6, 6, 1, 0, 0, 0, 0, 1, 1), (FC, FC)),      # 1x1 output, two images
    ((64, 64, 4, 4, 128, 4, 4, 1, 0, 0, 0, 0, 1, 1), (FC, FC)),     # FC GEMM
    ((2, 32, 12, 12, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8), (CC, CC)),     # thin 3x3
    ((2, 64, 13, 12, 64, 3, 3, 1, 1, 1, 1, 1, 1, 8), (TC, TC)),     # merged groups
    ((2, 12, 13, 12, 12, 3, 3, 2, 1, 1, 1, 1, 1, 1, 1, 3), (CC, CC)),   # CUDA-core tiles, per-axis stride
    ((1, 8, 9, 7, 12, 1, 1, 1, 0, 0, 0, 0, 1, 1), (CC, CC)),        # 1x1, 8 channels
]


@pytest.mark.parametrize("geom,paths", BF16_OUT)
def test_bf16_outputs(dev, oracle_mod, geom, paths):
    got = tuple(gc.gconv_plan(geom, B.GCONV_BF16, p)[0] for p in range(2))
    assert got == paths, (geom, got)
    N, Cin, H, W, Cout = wl.per_axis(geom)[:5]
    Ho, Wo = wl.out_hw(geom)
    wk = wl.Workload("bf16out", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 23)
    xd, wd, bd, dyd = (t.to(dev) for t in (x, w, b, dy))
    kw = _kw(geom)
    y32 = torch.empty((N, Cout, Ho, Wo), device=dev)
    dx32 = torch.empty((N, Cin, H, W), device=dev)
    y16 = torch.full((N, Cout, Ho, Wo), float("nan"), device=dev, dtype=torch.bfloat16)
    dx16 = torch.full((N, Cin, H, W), float("nan"), device=dev, dtype=torch.bfloat16)
    gc.gconv_fwd(xd, wd, bd, y32, **kw)
    gc.gconv_bwd_data(dyd, wd, dx32, **kw)
    gc.gconv_fwd(xd, wd, bd, y16, **kw)
    gc.gconv_bwd_data(dyd, wd, dx16, **kw)
    torch.cuda.synchronize()
    assert gc.gconv_check_device_error() == B.GCONV_OK
    assert torch.equal(y16, y32.to(torch.bfloat16)), geom
    assert torch.equal(dx16, dx32.to(torch.bfloat16)), geom
    for name, got16, ref in (("y", y16, oracle_mod.fwd(geom, f64(x), f64(w), f64(b))),
                             ("dx", dx16, oracle_mod.bwd_data(geom, f64(dy), f64(w)))):
        g = got16.cpu().double().numpy()
        rms = float(np.sqrt(np.mean(ref * ref)))
        bound = 1e-2 * rms + 2.0 ** -8 * np.abs(ref)
        assert np.all(np.abs(g - ref) <= bound), (name, geom, float(np.max(np.abs(g - ref) - bound)))


# The thin-plane kernels (3x3, one, two or four channels per group on both sides, stride 1 or
# 2): widths that select 1, 2 and 4 outputs per thread, pads 0..2, strips of rows, both
# input dtypes, and the weight gradient with its bias gradient from the same call.
THIN_PLANE = [
    (2, 16, 10, 10, 16, 3, 3, 1, 1, 1, 1, 1, 1, 16),        # depthwise, 1 output per thread
    (2, 8, 21, 20, 8, 3, 3, 1, 0, 2, 2, 0, 1, 8),           # depthwise, pads 0/2/2/0, 2 per thread
    (2, 8, 9, 60, 8, 3, 3, 1, 2, 1, 1, 2, 1, 2),            # 4 channels per group, 4 per thread
    (3, 12, 17, 33, 12, 3, 3, 2, 1, 1, 1, 1, 1, 6),         # 2 channels per group, stride 2
    (2, 32, 23, 50, 32, 3, 3, 2, 0, 1, 0, 1, 1, 8),         # 4 per group, stride 2, asymmetric pads
    (1, 6, 7, 7, 6, 3, 3, 2, 1, 1, 1, 1, 1, 6),             # depthwise stride 2, tiny plane
    (4, 64, 7, 7, 64, 3, 3, 1, 1, 1, 1, 1, 1, 64),          # small planes, many groups
    # rows of 16-byte multiples, stride 1: the register-tile forms (4 columns per thread)
    (2, 16, 12, 16, 16, 3, 3, 1, 1, 1, 1, 1, 1, 16),        # depthwise, 16 columns
    (2, 16, 12, 16, 16, 3, 3, 1, 1, 1, 1, 0, 1, 16),        # 15 produced columns: ragged last chunk
    (1, 2, 6, 200, 2, 3, 3, 1, 1, 1, 1, 1, 1, 2),           # depthwise, 200 columns
    (1, 4, 5, 256, 4, 3, 3, 1, 1, 1, 1, 1, 1, 2),           # 2 per group, 256 columns
    (2, 8, 13, 40, 8, 3, 3, 1, 0, 2, 2, 0, 1, 8),           # depthwise, pads 0/2/2/0
    (2, 16, 11, 64, 16, 3, 3, 1, 2, 0, 0, 2, 1, 4),         # 4 per group, 64 columns, pads 2/0/0/2
    (3, 12, 9, 72, 12, 3, 3, 1, 1, 1, 1, 1, 1, 6),          # 2 per group, 72 columns (4 per lane)
    (2, 32, 35, 120, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8),        # 4 per group, 120 columns, strips
    (1, 4, 8, 128, 4, 3, 3, 1, 1, 1, 0, 0, 1, 4),           # depthwise, 128 columns, pads 1/1/0/0
]


@pytest.mark.parametrize("geom", THIN_PLANE)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_thin_plane_kernels_full(dev, oracle_mod, geom, dtype):
    assert_paths(geom, dtype, (CC, CC, CC, RD))
    wk = wl.Workload("thin", geom, dtype, w=("normal", 0.3))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 29 + (dtype == "f32"))
    got = full_compare(geom, dtype, x, w, b, dy, dev, oracle_mod, label=f"thin {geom}")
    # the bias gradient computed with the weight gradient: identical to the separate pass
    xd, dyd = x.to(dev), dy.to(dev)
    dw, bw = guarded(tuple(w.shape), dev)
    db, bb = guarded((geom[4],), dev)
    gc.gconv_bwd_weight(xd, dyd, dw, db=db, **_kw(geom))
    torch.cuda.synchronize()
    assert gc.gconv_check_device_error() == B.GCONV_OK
    check_guards("thin fused dw", bw)
    check_guards("thin fused db", bb)
    assert torch.equal(dw.cpu(), got["dw"])
    check("thin fused db", db.cpu().numpy(), oracle_mod.bwd_bias(geom, f64(dy)), TOL[dtype])



# 1x1 layers at stride 1 without padding: forward and backward-data as a batched per-image GEMM
# (the case the cudnn.torch issue #118 thread sets apart from the fully-connected one), the
# weight gradient on the implicit-GEMM family; fp32 and bf16 outputs.
POINTWISE = [
    (2, 64, 8, 8, 32, 1, 1, 1, 0, 0, 0, 0, 1, 1),           # one M tile, K = 64
    (3, 48, 12, 12, 24, 1, 1, 1, 0, 0, 0, 0, 1, 1),         # K and M not multiples of the tiles
    (2, 64, 8, 16, 128, 1, 1, 1, 0, 0, 0, 0, 1, 2),         # grouped: 32 -> 64 per group
    (2, 256, 14, 12, 272, 1, 1, 1, 0, 0, 0, 0, 1, 1),       # several M and K tiles, ragged N tile
]


@pytest.mark.parametrize("geom", POINTWISE)
def test_pointwise_gemm_full(dev, oracle_mod, geom):
    assert_paths(geom, "bf16", (PW, PW, TC, RD))
    wk = wl.Workload("pw", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 31)
    got = full_compare(geom, "bf16", x, w, b, dy, dev, oracle_mod, label=f"pointwise {geom}")
    N, Cin, H, W, Cout = geom[:5]
    xd, wd, bd, dyd = (t.to(dev) for t in (x, w, b, dy))
    y16 = torch.empty((N, Cout, H, W), device=dev, dtype=torch.bfloat16)
    dx16 = torch.empty((N, Cin, H, W), device=dev, dtype=torch.bfloat16)
    gc.gconv_fwd(xd, wd, bd, y16, **_kw(geom))
    gc.gconv_bwd_data(dyd, wd, dx16, **_kw(geom))
    torch.cuda.synchronize()
    assert gc.gconv_check_device_error() == B.GCONV_OK
    assert torch.equal(y16.cpu(), got["y"].to(torch.bfloat16))
    assert torch.equal(dx16.cpu(), got["dx"].to(torch.bfloat16))


@pytest.mark.parametrize("name", list(wl.pointwise_zoo(2)))
def test_pointwise_zoo_layers_full(dev, oracle_mod, name):
    """The 1x1 layers of ResNet-50 bottlenecks (and a grouped 1x1), batch 2, all four passes."""
    wk = wl.pointwise_zoo(2)[name]
    x, w, b, dy = wl.make_inputs(wk, seed=43)
    H, W = wk.geom[2], wk.geom[3]
    # rows of H*W elements must be 16-byte multiples for the GEMM's tensor maps
    assert gc.gconv_plan(wk.geom, B.GCONV_BF16, B.PASS_FWD)[0] == (PW if (H * W) % 8 == 0 else TC)
    full_compare(wk.geom, "bf16", x, w, b, dy, dev, oracle_mod, label=name)



# Input size == kernel size with groups: a block-diagonal GEMM on the fully-connected path
# (G matrix products over the same tensors, read in place), plus shapes whose row counts and
# channel counts do not fill the GEMM tiles.
FC_SHAPES = [
    (4, 64, 5, 5, 96, 5, 5, 1, 0, 0, 0, 0, 1, 4),           # 4 groups, K = 400 per group, 24 outputs
    (3, 96, 4, 4, 64, 4, 4, 1, 0, 0, 0, 0, 1, 2),           # 2 groups, K = 768, 32 outputs
    (70, 48, 3, 3, 40, 3, 3, 1, 0, 0, 0, 0, 1, 1),          # K = 432, 40 outputs, 70 images
    (5, 32, 1, 1, 24, 1, 1, 1, 0, 0, 0, 0, 1, 1),           # 1x1 input: a plain matrix product
]


@pytest.mark.parametrize("geom", FC_SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fully_connected_gemm_full(dev, oracle_mod, geom, out):
    assert_paths(geom, "bf16", (FC, FC, FC, RD))
    wk = wl.Workload("fc", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=sum(geom) * 37)
    got = full_compare(geom, "bf16", x, w, b, dy, dev, oracle_mod, label=f"fc {geom}")
    if out == "bf16":
        N, Cin, H, W, Cout = geom[:5]
        xd, wd, bd, dyd = (t.to(dev) for t in (x, w, b, dy))
        y16 = torch.empty((N, Cout, 1, 1), device=dev, dtype=torch.bfloat16)
        dx16 = torch.empty((N, Cin, H, W), device=dev, dtype=torch.bfloat16)
        gc.gconv_fwd(xd, wd, bd, y16, **_kw(geom))
        gc.gconv_bwd_data(dyd, wd, dx16, **_kw(geom))
        torch.cuda.synchronize()
        assert torch.equal(y16.cpu(), got["y"].to(torch.bfloat16))
        assert torch.equal(dx16.cpu(), got["dx"].to(torch.bfloat16))


@pytest.mark.parametrize("geom", [
    (3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2),    # shared copies, side stream, dependent launches
    (2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1),     # stride 2: passes in turn, phases in one launch
])
def test_step_ex_in_a_cuda_graph(dev, geom):
    """gconv_step_ex captured into a CUDA graph (its side-stream fork and join and its
    programmatic dependent launches are captured with it) and replayed twice gives the
    eager call's results bit for bit."""
    wk = wl.Workload("graph", geom, "bf16")
    x, w, b, dy = (t.to(dev) for t in wl.make_inputs(wk, seed=515))
    N, Cin, H, W, Cout = wl.per_axis(geom)[:5]
    Ho, Wo = wl.out_hw(geom)
    kw = _kw(geom)
    ws = torch.empty(max(1, gc.gconv_step_workspace_size(B.per_axis(geom), B.GCONV_BF16)), dtype=torch.uint8,
                     device=dev)
    outs = lambda: (torch.empty((N, Cout, Ho, Wo), device=dev), torch.empty((N, Cin, H, W), device=dev),
                    torch.empty(tuple(w.shape), device=dev), torch.empty((Cout,), device=dev))
    ref = outs()
    gc.gconv_step(x, w, b, dy, *ref, workspace=ws, **kw)
    torch.cuda.synchronize()
    got = outs()
    for t in got:
        t.fill_(float("nan"))
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        gc.gconv_step(x, w, b, dy, *got, workspace=ws, **kw)
    for _ in range(2):
        for t in got:
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert gc.gconv_check_device_error() == B.GCONV_OK
        for a, r in zip(got, ref):
            assert torch.equal(a, r)
