"""The bounded-wait path of the tensor-core kernels, driven without hanging anything.

Every wait of a tensor-core kernel on an mbarrier (staged tiles, weight blocks, free
buffers, finished accumulators) gives up after a time limit, records GCONV_ERR_TIMEOUT in
the library's device error word, and unwinds: the kernel waits (with its own one-second
bound) for the copies and MMAs it already issued, frees its tensor memory and returns.
Setting the limit to 0 makes the first unsuccessful poll give up, so every family below
takes that path on its first tile.  The test then checks that the error is reported once,
that the next calls with the default limit run clean, and that their results match the
oracle: a timed-out kernel leaves the device usable.
"""
import numpy as np
import pytest
import torch

import bwd_gconv_fwd_gb300 as gc
from bwd_gconv_fwd_gb300 import binding as B
from bwd_gconv_fwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [
    # name, geometry, pass, family the planner must pick
    ("stride-1 correlation (forward)", (2, 32, 14, 13, 64, 3, 3, 1, 1, 0, 2, 1, 1, 2), B.PASS_FWD, B.PATH_TC_IGEMM),
    ("stride-1 correlation (backward-data)", (3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2), B.PASS_BWD_DATA,
     B.PATH_TC_IGEMM),
    ("stride-2 correlation (forward)", (2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1), B.PASS_FWD, B.PATH_TC_IGEMM),
    ("stride-2 correlation (backward-data, every output phase in one launch)",
     (2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1), B.PASS_BWD_DATA, B.PATH_TC_IGEMM),
    ("weight gradient", (2, 32, 14, 13, 64, 3, 3, 1, 1, 0, 2, 1, 1, 2), B.PASS_BWD_WEIGHT, B.PATH_TC_IGEMM),
    ("stride-2 weight gradient", (2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1), B.PASS_BWD_WEIGHT,
     B.PATH_TC_IGEMM),
    ("fully-connected GEMM", (64, 64, 4, 4, 128, 4, 4, 1, 0, 0, 0, 0, 1, 1), B.PASS_FWD, B.PATH_TC_FC),
]


def _run(geom, pass_, x, w, b, dy, dev):
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    Ho, Wo = wl.out_hw(geom)
    kw = dict(stride=s, padding=(pt, pb, pl, pr), dilation=d, groups=G)
    xd, wd, bd, dyd = (t.to(dev) for t in (x, w, b, dy))
    if pass_ == B.PASS_FWD:
        out = torch.zeros((N, Cout, Ho, Wo), device=dev)
        gc.gconv_fwd(xd, wd, bd, out, **kw)
    elif pass_ == B.PASS_BWD_DATA:
        out = torch.zeros((N, Cin, H, W), device=dev)
        gc.gconv_bwd_data(dyd, wd, out, **kw)
    else:
        out = torch.zeros(tuple(w.shape), device=dev)
        gc.gconv_bwd_weight(xd, dyd, out, **kw)
    return out


def _oracle(oracle_mod, geom, pass_, x, w, b, dy):
    f = lambda t: t.to(torch.float64).numpy()
    if pass_ == B.PASS_FWD:
        return oracle_mod.fwd(geom, f(x), f(w), f(b))
    if pass_ == B.PASS_BWD_DATA:
        return oracle_mod.bwd_data(geom, f(dy), f(w))
    return oracle_mod.bwd_weight(geom, f(x), f(dy))


@pytest.mark.parametrize("name,geom,pass_,family", CASES)
def test_wait_timeout_is_reported_and_recovered(oracle_mod, name, geom, pass_, family):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_gconv_fwd_gb300 import build
    build.build()
    dev = torch.device("cuda:0")
    assert gc.gconv_plan(geom, B.GCONV_BF16, pass_)[0] == family, name
    wk = wl.Workload("timeout", geom, "bf16", w=("normal", 0.2))
    x, w, b, dy = wl.make_inputs(wk, seed=606)
    stream = torch.cuda.current_stream()
    assert gc.gconv_check_device_error(stream) == B.GCONV_OK      # nothing pending from earlier tests
    try:
        B.gconv_debug_set_wait_limit(0)
        _run(geom, pass_, x, w, b, dy, dev)
        status = gc.gconv_check_device_error(stream)
    finally:
        B.gconv_debug_set_wait_limit(-1)
    assert status == B.GCONV_ERR_TIMEOUT, (name, B.status_string(status))
    # the error word was read and cleared; the device is usable and the next call is right
    assert gc.gconv_check_device_error(stream) == B.GCONV_OK
    out = _run(geom, pass_, x, w, b, dy, dev)
    assert gc.gconv_check_device_error(stream) == B.GCONV_OK
    ref = _oracle(oracle_mod, geom, pass_, x, w, b, dy)
    got = out.cpu().double().numpy()
    rms = float(np.sqrt(np.mean(ref * ref)))
    assert float(np.abs(got - ref).max()) <= 1e-2 * rms, name
