"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, and its host-side validation, shape arithmetic, planning and workspace
sizing behave as include/gconv.h states.  No call here reaches a kernel launch.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import bwd_gconv_fwd_gb300 as gc
from bwd_gconv_fwd_gb300 import binding as B
from bwd_gconv_fwd_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from bwd_gconv_fwd_gb300 import build
    build.build()
    return B.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "gconv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gconv_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    declared = _declared()
    assert len(declared) >= 10
    for name in declared:
        assert hasattr(L, name), name
    assert set(declared) == set(B.EXPORTED)


def test_out_shape_matches_floor_formula(L, oracle_mod):
    rng = np.random.default_rng(5)
    for _ in range(200):
        geom = wl.random_geometry(rng, max_hw=40, max_k=7, max_s=4, max_d=3, max_pad=4)
        assert gc.gconv_out_shape(geom) == oracle_mod.out_shape(geom)


BAD = [
    (1, 6, 5, 5, 4, 3, 3, 1, 0, 0, 0, 0, 1, 4),      # C_in % G
    (1, 4, 5, 5, 6, 3, 3, 1, 0, 0, 0, 0, 1, 4),      # C_out % G
    (1, 4, 2, 5, 4, 3, 3, 1, 0, 0, 0, 0, 1, 1),      # no output row
    (1, 4, 5, 5, 4, 3, 3, 0, 0, 0, 0, 0, 1, 1),      # stride 0
    (1, 4, 5, 5, 4, 3, 3, 1, 0, -1, 0, 0, 1, 1),     # negative pad
    (1, 4, 5, 5, 4, 3, 3, 1, 0, 0, 0, 0, 0, 1),      # dilation 0
    (-1, 4, 5, 5, 4, 3, 3, 1, 0, 0, 0, 0, 1, 1),     # negative N
    (1, 0, 5, 5, 4, 3, 3, 1, 0, 0, 0, 0, 1, 1),      # no channels
    (70000, 4096, 100, 100, 4, 3, 3, 1, 0, 0, 0, 0, 1, 1),  # x beyond 2^31 elements
]


@pytest.mark.parametrize("geom", BAD)
def test_invalid_geometry_rejected(L, geom):
    ho, wo = ctypes.c_int(), ctypes.c_int()
    assert L.gconv_out_shape(*geom, ctypes.byref(ho), ctypes.byref(wo)) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_workspace_size(*geom, B.GCONV_BF16, B.PASS_FWD) == ctypes.c_size_t(-1).value
    fake = ctypes.c_void_p(1 << 20)
    for call in (lambda: L.gconv_fwd(*geom, 1, fake, fake, None, fake, None, 0, None),
                 lambda: L.gconv_bwd_data(*geom, 1, fake, fake, fake, None, 0, None),
                 lambda: L.gconv_bwd_weight(*geom, 1, fake, fake, fake, None, 0, None),
                 lambda: L.gconv_bwd_bias(*geom, 1, fake, fake, None, 0, None)):
        assert call() == B.GCONV_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_rejected(L):
    geom = (2, 8, 6, 6, 8, 3, 3, 1, 1, 1, 1, 1, 1, 1)
    ok = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 2)
    assert L.gconv_fwd(*geom, 1, None, ok, None, ok, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_fwd(*geom, 1, ok, None, None, ok, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_fwd(*geom, 1, ok, ok, None, None, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_fwd(*geom, 1, mis, ok, None, ok, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_fwd(*geom, 1, ok, ok, mis, ok, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_bwd_data(*geom, 1, ok, ok, None, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_bwd_weight(*geom, 1, ok, None, ok, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_bwd_bias(*geom, 1, None, ok, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_fwd(*geom, 7, ok, ok, None, ok, None, 0, None) == B.GCONV_ERR_INVALID_ARG  # dtype


def test_empty_batch_is_a_noop(L):
    geom = (0, 8, 6, 6, 8, 3, 3, 1, 1, 1, 1, 1, 1, 1)
    for p in range(4):
        path, launches = gc.gconv_plan(geom, B.GCONV_BF16, p)
        assert path == B.PATH_NONE and launches == 0
        assert gc.gconv_workspace_size(geom, B.GCONV_BF16, p) == 0
    # nothing is read or written by the forward and backward-data passes: null pointers are fine
    assert L.gconv_fwd(*geom, 1, None, None, None, None, None, 0, None) == B.GCONV_OK
    assert L.gconv_bwd_data(*geom, 1, None, None, None, None, 0, None) == B.GCONV_OK
    # dw and db are sums over no terms and are written as zeros: they must be given
    assert L.gconv_bwd_weight(*geom, 1, None, None, None, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_bwd_bias(*geom, 1, None, None, None, 0, None) == B.GCONV_ERR_INVALID_ARG
    assert L.gconv_bwd_weight_noalloc(*geom, 1, None, None, None, None) == B.GCONV_ERR_INVALID_ARG


def test_workspace_too_small_rejected_before_launch(L):
    for name, wk in wl.WORKLOADS.items():
        geom = wk.geom
        dt = B.GCONV_BF16 if wk.dtype == "bf16" else B.GCONV_F32
        need = gc.gconv_workspace_size(geom, dt, B.PASS_BWD_WEIGHT)
        if need == 0:
            continue
        ok = ctypes.c_void_p(1 << 20)
        st = L.gconv_bwd_weight(*geom, dt, ok, ok, ok, ok, need - 16, None)
        assert st == B.GCONV_ERR_WORKSPACE, name
        st = L.gconv_bwd_weight(*geom, dt, ok, ok, ok, None, 0, None)
        assert st == B.GCONV_ERR_WORKSPACE, name


def test_plans_are_consistent(L):
    for name, wk in wl.WORKLOADS.items():
        dt = B.GCONV_BF16 if wk.dtype == "bf16" else B.GCONV_F32
        for p in range(4):
            path, launches = gc.gconv_plan(wk.geom, dt, p)
            assert path in (B.PATH_DIRECT, B.PATH_TC_IGEMM, B.PATH_TC_FC, B.PATH_REDUCE, B.PATH_TC_GEMM), (name, p)
            assert 1 <= launches <= 9
            if p == B.PASS_BWD_BIAS:
                assert path == B.PATH_REDUCE
            if dt == B.GCONV_F32:
                assert path in (B.PATH_DIRECT, B.PATH_REDUCE)


def test_forcing_a_family(L):
    geom = wl.WORKLOADS["tiny_g5"].geom
    try:
        gc.binding.gconv_debug_force_path(B.PATH_TC_IGEMM)
        with pytest.raises(gc.GconvError) as e:
            gc.gconv_plan(geom, B.GCONV_F32, B.PASS_FWD)   # no tensor-core path for fp32
        assert e.value.status == B.GCONV_ERR_UNSUPPORTED
        gc.binding.gconv_debug_force_path(B.PATH_DIRECT)
        assert gc.gconv_plan(wl.WORKLOADS["alexnet_g2"].geom, B.GCONV_BF16, B.PASS_FWD)[0] == B.PATH_DIRECT
    finally:
        gc.binding.gconv_debug_force_path(B.PATH_NONE)


def test_status_strings(L):
    for s in range(6):
        assert B.status_string(s).startswith("GCONV_")
    assert "unknown" in B.status_string(99)


def test_python_geometry_helper():
    assert gc.geometry((2, 6, 9, 9), (4, 3, 3, 3), 2, (1, 0, 2, 1), 1, 2) == (2, 6, 9, 9, 4, 3, 3, 2, 1, 0, 2, 1, 1, 2)
    assert gc.geometry((2, 6, 9, 9), (4, 6, 3, 3), padding=1) == (2, 6, 9, 9, 4, 3, 3, 1, 1, 1, 1, 1, 1, 1)
    with pytest.raises(gc.GconvError):
        gc.geometry((2, 6, 9, 9), (4, 4, 3, 3), groups=2)


def test_step_host_sizing_and_argument_checks(L):
    """gconv_step_host: its device-buffer size covers inputs, outputs and the largest
    workspace; bad arguments are rejected before anything is enqueued (no GPU needed)."""
    for name, wk in wl.WORKLOADS.items():
        geom = wk.geom
        N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
        Ho, Wo = wl.out_hw(geom)
        dt = B.GCONV_BF16 if wk.dtype == "bf16" else B.GCONV_F32
        es = 2 if dt == B.GCONV_BF16 else 4
        ws = max(gc.gconv_workspace_size(geom, dt, p) for p in range(4))
        tensors = (N * Cin * H * W * (es + 4) + Cout * (Cin // G) * kH * kW * (es + 4)
                   + N * Cout * Ho * Wo * (es + 4) + Cout * 4)
        with_b = gc.gconv_step_device_bytes(geom, dt, True)
        without_b = gc.gconv_step_device_bytes(geom, dt, False)
        assert with_b >= tensors + ws + Cout * es, name
        assert without_b >= tensors + ws and without_b <= with_b, name
        ok = ctypes.c_void_p(1 << 20)
        full = (ok, ok, ok, ok, ok, ok, ok, ok)
        # buffer too small / missing
        assert L.gconv_step_host(*geom, dt, *full, ok, with_b - 16, None) == B.GCONV_ERR_WORKSPACE, name
        assert L.gconv_step_host(*geom, dt, *full, None, 0, None) == B.GCONV_ERR_WORKSPACE, name
        # a NULL host pointer (other than bias) or a misaligned device buffer
        for i in (0, 1, 3, 4, 5, 6, 7):
            args = list(full)
            args[i] = None
            assert L.gconv_step_host(*geom, dt, *args, ok, with_b, None) == B.GCONV_ERR_INVALID_ARG, (name, i)
        mis = ctypes.c_void_p((1 << 20) + 8)
        assert L.gconv_step_host(*geom, dt, *full, mis, with_b, None) == B.GCONV_ERR_INVALID_ARG, name
        assert L.gconv_step_host(*geom, 9, *full, ok, with_b, None) == B.GCONV_ERR_INVALID_ARG, name
    # empty batch: dw and db still come back (as zeros) through the device buffer, so it is required
    geom = (0, 8, 6, 6, 8, 3, 3, 1, 1, 1, 1, 1, 1, 1)
    ok = ctypes.c_void_p(1 << 20)
    assert L.gconv_step_host(*geom, 1, ok, ok, None, ok, ok, ok, ok, ok, None, 0, None) == B.GCONV_ERR_WORKSPACE
    assert gc.gconv_step_device_bytes(geom, B.GCONV_BF16, False) >= 8 * 8 * 9 * 4 + 8 * 4
    # invalid geometry
    assert gc.binding.lib().gconv_step_device_bytes(1, 8, 6, 6, 8, 9, 9, 1, 0, 0, 0, 0, 1, 1, 1, 1) == ctypes.c_size_t(-1).value


def test_model_zoo_layers_have_plans(L):
    """Every layer of the model-zoo sweep (ResNeXt-50 grouped, MobileNet-v2 depthwise, stride 1
    and 2) is served by some kernel family for every pass, with a bounded workspace, and the
    host-step buffer covers it (host-only)."""
    for N in (2, 32):
        for name, wk in wl.model_zoo(N).items():
            geom = wk.geom
            for p in range(4):
                path, launches = gc.gconv_plan(geom, B.GCONV_BF16, p)
                assert path in (B.PATH_DIRECT, B.PATH_TC_IGEMM, B.PATH_TC_FC, B.PATH_REDUCE, B.PATH_TC_GEMM), (name, p)
                assert 1 <= launches <= 9, (name, p)
                ws = gc.gconv_workspace_size(geom, B.GCONV_BF16, p)
                assert 0 <= ws < (1 << 32), (name, p)
            assert gc.gconv_step_device_bytes(geom, B.GCONV_BF16, True) > 0, name


def test_step_ex_sizing_and_argument_checks(L):
    """gconv_step_ex: its workspace covers each pass's (or the shared route's), and a bad
    argument is rejected before anything is enqueued (no GPU needed)."""
    for name, wk in wl.WORKLOADS.items():
        geom = B.per_axis(wk.geom)
        dt = B.GCONV_BF16 if wk.dtype == "bf16" else B.GCONV_F32
        need = gc.gconv_step_workspace_size(geom, dt)
        assert 0 <= need < (1 << 34), name
        rec = B.geometry_record(geom)
        ok = ctypes.c_void_p(1 << 20)
        mis = ctypes.c_void_p((1 << 20) + 8)
        step = lambda *a: L.gconv_step_ex(ctypes.byref(rec), *a)
        full = [ok, ok, None, ok, ok, ok, ok, None]   # x w bias dy y dx dw db
        if need:
            assert step(dt, B.GCONV_F32, *full, ok, need - 16, None) == B.GCONV_ERR_WORKSPACE, name
            assert step(dt, B.GCONV_F32, *full, None, 0, None) == B.GCONV_ERR_WORKSPACE, name
            assert step(dt, B.GCONV_F32, *full, mis, need, None) == B.GCONV_ERR_INVALID_ARG, name
        for i in (0, 1, 3, 4, 5, 6):
            args = list(full)
            args[i] = None
            assert step(dt, B.GCONV_F32, *args, ok, need, None) == B.GCONV_ERR_INVALID_ARG, (name, i)
            args[i] = mis
            assert step(dt, B.GCONV_F32, *args, ok, need, None) == B.GCONV_ERR_INVALID_ARG, (name, i)
        assert step(dt, 7, *full, ok, need, None) == B.GCONV_ERR_INVALID_ARG, name
        assert step(9, B.GCONV_F32, *full, ok, need, None) == B.GCONV_ERR_INVALID_ARG, name
    with pytest.raises(gc.GconvError):
        gc.gconv_step_workspace_size((1, 8, 6, 6, 8, 9, 9, 1, 0, 0, 0, 0, 1, 1), B.GCONV_BF16)


def test_step_plan_routes(L):
    """gconv_step_plan_ex: which layers share the blocked copies between the passes (bf16,
    every pass on the tensor-core kernels unmerged at stride 1, output as wide as the input),
    and the step's launch count; every other layer runs its passes in turn (host-only)."""
    bf, f32 = B.GCONV_BF16, B.GCONV_F32
    assert gc.gconv_step_plan(wl.WORKLOADS["alexnet_g2"].geom, bf) == (True, 6)
    assert gc.gconv_step_plan(wl.WORKLOADS["dense3x3"].geom, bf) == (True, 6)
    assert gc.gconv_step_plan(wl.WORKLOADS["dense3x3"].geom, f32)[0] is False
    for name in ("dense3x3_s2_asym", "resnext_g32", "depthwise", "fc_mode", "tiny_g5"):
        geom = wl.WORKLOADS[name].geom
        dt = bf if wl.WORKLOADS[name].dtype == "bf16" else f32
        shared, launches = gc.gconv_step_plan(geom, dt)
        assert not shared, name
        assert launches == sum(gc.gconv_plan(geom, dt, p)[1] for p in range(3)), name
    # an output narrower than the input: the backward-data copy has another pitch
    assert gc.gconv_step_plan((2, 32, 14, 13, 64, 3, 3, 1, 1, 0, 2, 1, 1, 2), bf)[0] is False
    assert gc.gconv_step_plan((2, 64, 17, 15, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1), bf) == (True, 6)
    # groups of 8 channels run merged (block-diagonal weights): the step shares the merged
    # geometry's copies, with the weight widening and the diagonal extraction around it
    assert gc.gconv_step_plan((2, 64, 12, 12, 64, 3, 3, 1, 1, 1, 1, 1, 1, 8), bf) == (True, 8)
    assert gc.gconv_step_plan(wl.model_zoo(2)["resnext_s1_256x28"].geom, bf) == (True, 8)
    # a forced family turns sharing off
    B.gconv_debug_force_path(B.PATH_TC_IGEMM)
    try:
        assert gc.gconv_step_plan(wl.WORKLOADS["alexnet_g2"].geom, bf)[0] is False
    finally:
        B.gconv_debug_force_path(B.PATH_NONE)
    with pytest.raises(gc.GconvError):
        gc.gconv_step_plan((1, 8, 6, 6, 8, 3, 3, 1, 0, 0, 0, 0, 1, 1), 5)
