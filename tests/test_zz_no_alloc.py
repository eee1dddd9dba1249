"""The weight gradient that allocates nothing (gconv_bwd_weight_noalloc).

Some callers cannot allocate device memory: a plug-in inside a host application
that owns every device allocation through its own pool or memory budget, or a
caller on a latency-critical path where a cudaMalloc could synchronise the
device.  For them the library offers one entry point whose split-K scratch is a
fixed 128 MiB array held by the library itself.  These tests call it through the
C ABI and check it against the regular gconv_bwd_weight (which takes a
caller-provided workspace), on two calls in a row, since every call shares and
reuses the same scratch array.  Both entry points run the same deterministic
kernels (fixed-order reductions), so their results must agree bit for bit; the
small case is also checked against the fp64 oracle.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import bwd_gconv_fwd_gb300 as gc
from bwd_gconv_fwd_gb300 import binding as B
from bwd_gconv_fwd_gb300 import workloads as wl

TOL = {"bf16": 1e-2, "f32": 1e-4}

CASES = [
    ("alexnet_g2", wl.WORKLOADS["alexnet_g2"].geom, "bf16"),                  # tcgen05 path, ~106 MiB scratch
    ("dense3x3_s2_asym", wl.WORKLOADS["dense3x3_s2_asym"].geom, "bf16"),      # stride 2: phase planes
    ("f32_split", (16, 16, 20, 20, 16, 3, 3, 1, 1, 1, 1, 1, 1, 1), "f32"),     # fp32 inputs, split-K
]


def _max_err_over_rms(got, ref):
    ref = ref.double()
    rms = float(ref.pow(2).mean().sqrt())
    return float((got.double() - ref).abs().max()) / rms


@pytest.mark.gpu
@pytest.mark.parametrize("name,geom,dtype", CASES)
def test_noalloc_matches_workspace_entry_point(oracle_mod, name, geom, dtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_gconv_fwd_gb300 import build
    build.build()
    L = B.lib()
    dt = B.GCONV_BF16 if dtype == "bf16" else B.GCONV_F32
    need = gc.gconv_workspace_size(geom, dt, B.PASS_BWD_WEIGHT)
    assert 0 < need <= L.gconv_noalloc_scratch_bytes(), (name, need)
    dev = torch.device("cuda:0")
    wk = wl.Workload(name, geom, dtype)
    x, w, b, dy = wl.make_inputs(wk, seed=777)
    xd, dyd = x.to(dev), dy.to(dev)
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    kw = dict(stride=s, padding=(pt, pb, pl, pr), dilation=d, groups=G)
    ref = torch.empty(tuple(w.shape), device=dev)
    gc.gconv_bwd_weight(xd, dyd, ref, **kw)        # regular entry point, caller workspace
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):                            # two calls in a row share the scratch
        out = torch.full(tuple(w.shape), float("nan"), device=dev)
        st = L.gconv_bwd_weight_noalloc(*geom, dt, ctypes.c_void_p(xd.data_ptr()), ctypes.c_void_p(dyd.data_ptr()),
                                        ctypes.c_void_p(out.data_ptr()), stream)
        assert st == B.GCONV_OK, B.status_string(st)
        torch.cuda.synchronize()
        assert gc.gconv_check_device_error() == B.GCONV_OK
        assert torch.isfinite(out).all(), (name, call)
        assert torch.equal(out, ref), (name, call, _max_err_over_rms(out, ref))
    if name == "f32_split":
        f = lambda t: t.to(torch.float64).numpy()
        expect = torch.from_numpy(oracle_mod.bwd_weight(geom, f(x), f(dy)))
        assert _max_err_over_rms(out.cpu(), expect) <= TOL[dtype]


def test_noalloc_rejects_scratch_beyond_its_fixed_size():
    """A geometry whose split-K scratch exceeds the fixed array is refused before any launch."""
    from bwd_gconv_fwd_gb300 import build
    build.build()
    L = B.lib()
    cap = L.gconv_noalloc_scratch_bytes()
    assert cap == 128 << 20
    geom = (64, 4096, 32, 32, 64, 5, 5, 1, 2, 2, 2, 2, 1, 1)   # dw 25 MiB x 10 splits
    need = gc.gconv_workspace_size(geom, B.GCONV_F32, B.PASS_BWD_WEIGHT)
    assert need > cap
    fake = ctypes.c_void_p(1 << 20)
    st = L.gconv_bwd_weight_noalloc(*geom, B.GCONV_F32, fake, fake, fake, None)
    assert st == B.GCONV_ERR_WORKSPACE
    assert "workspace" in B.status_string(st)
