"""CPU replays of the tensor-core launches' host planning and index arithmetic.

The programs under tests/replay/ include the library source, rebuild the launch
parameters the library would use for a geometry, and walk every tile's reads and writes
on the host, checking them against the buffers' extents (bounds are checked by reading
the index arithmetic, not by running a possibly faulting kernel).  They need nvcc (to
compile the included CUDA source) but no GPU.
"""
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

from bwd_gconv_fwd_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))


def _nvcc():
    return shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)


@pytest.fixture(scope="module")
def replay_bins(tmp_path_factory):
    nvcc = _nvcc()
    if not nvcc:
        pytest.skip("nvcc not available")
    out = tmp_path_factory.mktemp("replay")
    names = ("corr2_plan_replay", "wgrad_plan_replay", "wgrad_phase_replay", "thin3_plan_replay", "thin_tile_replay",
             "step_plan_replay")

    def build(name):
        exe = str(out / name)
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O1", "-std=c++17", "-o", exe,
               os.path.join(HERE, "replay", name + ".cu"), "-lcuda"]
        return name, exe, subprocess.run(cmd, capture_output=True, text=True)

    bins = {}
    with ThreadPoolExecutor(max_workers=len(names)) as pool:
        for name, exe, r in pool.map(build, names):
            assert r.returncode == 0, r.stderr[-2000:]
            bins[name] = exe
    return bins


def _run(exe, geom, *extra):
    r = subprocess.run([exe, *map(str, geom), *map(str, extra)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "errors: 0" in r.stdout, (geom, r.stdout[-2000:])


STRIDE1 = [
    (3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2),       # AlexNet-like, ragged
    (2, 32, 14, 13, 64, 3, 3, 1, 1, 0, 2, 1, 1, 2),
    (2, 64, 17, 15, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1),
    (2, 16, 9, 9, 16, 3, 3, 1, 2, 2, 2, 2, 2, 1),           # dilation 2
    (2, 256, 9, 9, 256, 3, 3, 1, 1, 1, 1, 1, 1, 1),         # several channel tiles
    (1, 96, 13, 40, 160, 3, 3, 1, 1, 1, 1, 1, 1, 2),        # wide rows, 80 produced channels
    (1, 40, 7, 23, 24, 2, 4, 1, 0, 3, 1, 0, 1, 1),          # odd channel counts, 2 x 4 kernel
    (2, 64, 20, 20, 64, 7, 7, 1, 3, 3, 3, 3, 1, 1),         # 49 taps
    # per-axis dilation (16 integers: ..., s_h, s_w, pads, d_h, d_w, G)
    (2, 32, 11, 13, 32, 3, 3, 1, 1, 2, 2, 1, 1, 1, 2, 1),
    (2, 32, 12, 9, 64, 3, 5, 1, 1, 1, 1, 2, 2, 2, 1, 2),
    # merged groups: the geometry the kernels see when consecutive thin groups run as one
    # (8 groups of 8 channels as one of 64; 6 groups of 8/4 as one of 48/24; 16 groups as 2)
    (2, 64, 13, 12, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1),
    (2, 48, 11, 11, 24, 3, 3, 1, 1, 1, 1, 1, 1, 1),
    (2, 24, 9, 10, 48, 5, 5, 1, 2, 2, 2, 2, 1, 1),
    (3, 128, 10, 11, 128, 3, 3, 1, 0, 2, 1, 1, 1, 2),
    (2, 256, 28, 28, 256, 3, 3, 1, 1, 1, 1, 1, 1, 4),      # ResNeXt 256x28, 8 channels a group, merged
    (2, 512, 14, 14, 512, 3, 3, 1, 1, 1, 1, 1, 1, 8),      # ResNeXt 512x14, 16 a group, merged by 4
    (2, 1024, 7, 7, 1024, 3, 3, 1, 1, 1, 1, 1, 1, 16),     # ResNeXt 1024x7, 32 a group, merged by 2
]


@pytest.mark.parametrize("geom", STRIDE1 + [wk.geom for wk in wl.WORKLOADS.values() if wk.geom[7] == 1]
                         + [wk.geom for wk in wl.model_zoo(2).values() if wk.geom[7] == 1])
def test_correlation_plan_replay(replay_bins, geom):
    _run(replay_bins["corr2_plan_replay"], geom)


@pytest.mark.parametrize("geom", STRIDE1 + [wk.geom for wk in wl.WORKLOADS.values() if wk.geom[7] == 1]
                         + [wk.geom for wk in wl.model_zoo(2).values() if wk.geom[7] == 1])
def test_weight_gradient_plan_replay(replay_bins, geom):
    _run(replay_bins["wgrad_plan_replay"], geom)


STRIDE2 = [
    (2, 64, 19, 16, 64, 3, 3, 2, 0, 1, 0, 1, 1, 1),         # asymmetric pads
    (2, 32, 15, 15, 64, 5, 5, 2, 2, 2, 2, 2, 1, 2),
    (1, 48, 13, 17, 32, 3, 3, 2, 1, 1, 1, 1, 1, 1),
    (2, 16, 12, 12, 32, 3, 3, 2, 2, 2, 2, 2, 2, 1),         # dilation 2
    (2, 256, 14, 14, 256, 3, 3, 2, 1, 1, 1, 1, 1, 1),       # two 128-channel tiles in every phase
    (1, 128, 15, 15, 128, 5, 5, 2, 2, 2, 2, 2, 1, 1),       # 5x5: the phases have 9, 6, 6 and 4 taps
    # per-axis strides: one stride-2 axis and one stride-1 axis (two phase planes)
    (2, 32, 13, 12, 32, 3, 3, 2, 1, 1, 1, 1, 1, 1, 1, 1),
    (2, 32, 12, 15, 64, 3, 3, 1, 2, 1, 0, 1, 1, 1, 2, 1),
    # merged groups (see above)
    (2, 64, 14, 13, 64, 3, 3, 2, 1, 1, 1, 1, 1, 1),
    (2, 256, 56, 56, 256, 3, 3, 2, 1, 1, 1, 1, 1, 4),      # ResNeXt 256x56 stride 2, merged
    (2, 512, 28, 28, 512, 3, 3, 2, 1, 1, 1, 1, 1, 8),      # ResNeXt 512x28 stride 2, merged by 4
    (2, 1024, 14, 14, 1024, 3, 3, 2, 1, 1, 1, 1, 1, 16),   # ResNeXt 1024x14 stride 2, merged by 2
]


@pytest.mark.parametrize("geom", STRIDE2 + [wk.geom for wk in wl.WORKLOADS.values() if wk.geom[7] == 2]
                         + [wk.geom for wk in wl.model_zoo(2).values() if wk.geom[7] == 2])
def test_stride2_correlation_plan_replay(replay_bins, geom):
    """The stride-2 forward on the correlation kernel: stride-phase planes as staged chunks."""
    _run(replay_bins["corr2_plan_replay"], geom)


@pytest.mark.parametrize("geom", STRIDE2 + [wk.geom for wk in wl.WORKLOADS.values() if wk.geom[7] == 2]
                         + [wk.geom for wk in wl.model_zoo(2).values() if wk.geom[7] == 2])
def test_stride2_weight_gradient_plan_replay(replay_bins, geom):
    _run(replay_bins["wgrad_phase_replay"], geom)


THIN3 = [
    (2, 16, 10, 10, 16, 3, 3, 1, 1, 1, 1, 1, 1, 16),        # depthwise
    (2, 32, 12, 12, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8),         # 4 channels per group
    (3, 12, 13, 9, 12, 3, 3, 1, 1, 0, 2, 1, 1, 3),          # asymmetric pads, ragged
    (1, 6, 5, 30, 6, 3, 3, 1, 2, 2, 0, 0, 1, 3),            # pads 2, wide rows
    (4, 64, 7, 7, 64, 3, 3, 1, 1, 1, 1, 1, 1, 64),          # small planes, several groups per block
]


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("geom", THIN3 + [wk.geom for wk in wl.WORKLOADS.values() if wk.geom[5:8] == (3, 3, 1)]
                         + [wk.geom for wk in wl.model_zoo(32).values() if wk.geom[7] == 1])
def test_thin_3x3_plan_replay(replay_bins, geom, dtype):
    _run(replay_bins["thin3_plan_replay"], geom, dtype)


# The register-tile thin-group kernels (stride 1, 1, 2 or 4 channels a group, rows of
# 16-byte multiples): the parity tests' layers, the workloads and the model-zoo layers.
THIN_TILE = [
    (2, 16, 12, 16, 16, 3, 3, 1, 1, 1, 1, 1, 1, 16),
    (2, 16, 12, 16, 16, 3, 3, 1, 1, 1, 1, 0, 1, 16),
    (2, 8, 13, 40, 8, 3, 3, 1, 0, 2, 2, 0, 1, 8),
    (2, 16, 11, 64, 16, 3, 3, 1, 2, 0, 0, 2, 1, 4),
    (3, 12, 9, 72, 12, 3, 3, 1, 1, 1, 1, 1, 1, 6),
    (2, 32, 35, 120, 32, 3, 3, 1, 1, 1, 1, 1, 1, 8),
    (1, 4, 8, 128, 4, 3, 3, 1, 1, 1, 0, 0, 1, 4),
    (1, 2, 6, 200, 2, 3, 3, 1, 1, 1, 1, 1, 1, 2),
    (1, 4, 5, 256, 4, 3, 3, 1, 1, 1, 1, 1, 1, 2),
]


@pytest.mark.parametrize("dtype", [0, 1])
@pytest.mark.parametrize("geom", THIN_TILE + [wk.geom for wk in wl.model_zoo(2).values() if wk.geom[7] == 1])
def test_thin_tile_plan_replay(replay_bins, geom, dtype):
    _run(replay_bins["thin_tile_replay"], geom, dtype)


@pytest.mark.parametrize("name", [n for n, wk in wl.WORKLOADS.items() if wk.geom[5:8] == (3, 3, 1)])
def test_thin_tile_plan_replay_workloads(replay_bins, name):
    """The full-size workloads in their storage dtype (their plans depend on the batch)."""
    wk = wl.WORKLOADS[name]
    _run(replay_bins["thin_tile_replay"], wk.geom, 0 if wk.dtype == "bf16" else 1)


# The training step's shared blocked copies: (geometry, whether the step shares them).  The
# step shares when every pass runs on the tensor-core kernels at stride 1 and the output is
# as wide as the input (the backward-data copy of gradOutput then has the weight gradient's
# pitch).
STEP = [
    ((128, 96, 27, 27, 256, 5, 5, 1, 2, 2, 2, 2, 1, 2), 1),      # AlexNet-style 2-group layer
    ((3, 48, 11, 11, 128, 5, 5, 1, 2, 2, 2, 2, 1, 2), 1),
    ((2, 64, 17, 15, 64, 3, 3, 1, 1, 1, 1, 1, 1, 1), 1),
    ((2, 16, 9, 9, 16, 3, 3, 1, 2, 2, 2, 2, 2, 1), 1),           # dilation 2
    ((2, 256, 9, 9, 256, 3, 3, 1, 1, 1, 1, 1, 1, 1), 1),         # several channel chunks
    ((2, 64, 20, 20, 64, 7, 7, 1, 3, 3, 3, 3, 1, 1), 1),
    ((2, 32, 11, 13, 32, 3, 3, 1, 1, 1, 1, 2, 2, 1, 2, 1), 1),    # per-axis dilation
    ((2, 32, 11, 13, 32, 3, 3, 1, 1, 2, 2, 1, 1, 1, 2, 1), 0),    # per-axis dilation, output 2 columns narrower
    ((2, 96, 10, 12, 64, 3, 3, 1, 0, 2, 2, 0, 1, 1), 1),         # one-sided pads
    ((1, 40, 7, 23, 24, 2, 4, 1, 0, 3, 1, 0, 1, 1), 0),          # output narrower than the input
    ((2, 32, 14, 13, 64, 3, 3, 1, 1, 0, 2, 1, 1, 2), 0),         # output wider than the input
    ((2, 64, 16, 16, 64, 3, 3, 2, 1, 1, 1, 1, 1, 1), 0),         # stride 2
]


@pytest.mark.parametrize("geom,shared", STEP)
def test_step_shared_copy_replay(replay_bins, geom, shared):
    _run(replay_bins["step_plan_replay"], geom, shared)
