"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself: brute force on tiny
inputs, library routines (torch conv2d in float64 with autograd, scipy
correlate2d, numpy matmul), the adjoint identities, finite differences, closed
forms of the all-ones fully-connected-mode script, and the shapes and printed
values of the pages' worked examples (tests/golden/).
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from bwd_gconv_fwd_gb300 import workloads as wlm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(rng, shape):
    return rng.standard_normal(shape)


def _inputs(rng, geom):
    sh = wlm.tensor_shapes(geom)
    return (_rand(rng, sh["x"]), _rand(rng, sh["w"]), _rand(rng, sh["b"]), _rand(rng, sh["dy"]))


def _torch_ref(geom, x, w, b, dy):
    """torch conv2d in float64 (asymmetric pads via F.pad, per-axis stride and dilation as
    tuples), gradients by autograd."""
    N, Cin, H, W, Cout, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, G = wlm.per_axis(geom)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    y = F.conv2d(F.pad(xt, (pl, pr, pt, pb)), wt, bt, stride=(sh, sw), dilation=(dh, dw), groups=G)
    y.backward(torch.tensor(dy, dtype=torch.float64))
    return y.detach().numpy(), xt.grad.numpy(), wt.grad.numpy(), bt.grad.numpy()


def _brute_operators(geom):
    """Every (output, input, weight) connection, by plain enumeration of
    (n, o, oh, ow, c, kh, kw).  The test assembles two dense operators from it:
      A_w[y_idx, x_idx] (built from w):  y = A_w x + b,  dx = A_w^T dy
      B_x[y_idx, w_idx] (built from x):  y = B_x w + b,  dw = B_x^T dy
    so the backward passes are checked as matrix transposes, not index inversions.
    """
    N, Cin, H, W, Cout, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, G = wlm.per_axis(geom)
    Ho, Wo = wlm.out_hw(geom)
    Cgi, Cgo = Cin // G, Cout // G
    conns = []  # (y_idx, x_idx, w_idx)
    for n, o, oh, ow in itertools.product(range(N), range(Cout), range(Ho), range(Wo)):
        g = o // Cgo
        yi = ((n * Cout + o) * Ho + oh) * Wo + ow
        for c, kh, kw in itertools.product(range(Cgi), range(kH), range(kW)):
            ih, iw = oh * sh - pt + kh * dh, ow * sw - pl + kw * dw
            if 0 <= ih < H and 0 <= iw < W:
                xi = ((n * Cin + g * Cgi + c) * H + ih) * W + iw
                wi = ((o * Cgi + c) * kH + kh) * kW + kw
                conns.append((yi, xi, wi))
    return conns, (N * Cout * Ho * Wo, N * Cin * H * W, Cout * Cgi * kH * kW)


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    scale = max(1.0, float(np.abs(b).max(initial=0.0)))
    return float(np.abs(a - b).max(initial=0.0)) / scale


TINY_GEOMS = [
    (1, 1, 1, 1, 1, 1, 1, 1, 0, 0, 0, 0, 1, 1),
    (2, 4, 5, 6, 6, 3, 2, 1, 1, 0, 2, 1, 1, 2),
    (1, 6, 7, 7, 3, 3, 3, 2, 0, 1, 0, 1, 1, 3),
    (2, 2, 6, 5, 4, 2, 3, 3, 2, 2, 1, 0, 2, 1),
    (1, 3, 7, 4, 6, 3, 1, 1, 2, 1, 0, 0, 2, 3),
    (1, 4, 3, 3, 4, 3, 3, 1, 1, 1, 1, 1, 1, 4),   # depthwise, pad 1
    (2, 2, 4, 4, 2, 4, 4, 1, 0, 0, 0, 0, 1, 1),   # input == kernel
    (1, 2, 5, 5, 2, 2, 2, 3, 0, 0, 0, 0, 1, 1),   # stride > kernel: untouched pixels
    # per-axis stride and dilation (N, C_in, H, W, C_out, kH, kW, s_h, s_w, pads, d_h, d_w, G)
    (1, 2, 7, 6, 4, 3, 2, 2, 1, 1, 0, 0, 1, 1, 2, 2),
    (2, 3, 5, 8, 3, 2, 3, 1, 3, 0, 1, 2, 0, 2, 1, 3),
    (1, 4, 9, 5, 2, 3, 3, 3, 2, 2, 1, 1, 0, 1, 2, 2),
    (1, 2, 6, 7, 2, 1, 2, 2, 1, 0, 0, 0, 0, 1, 3, 1),
]


@pytest.mark.parametrize("geom", TINY_GEOMS)
def test_brute_force_operators(oracle_mod, geom):
    """O1: all four outputs equal the enumerated dense operators (and their transposes)."""
    rng = np.random.default_rng(7)
    x, w, b, dy = _inputs(rng, geom)
    conns, (ny, nx, nw) = _brute_operators(geom)
    xf, wf, dyf = x.ravel(), w.ravel(), dy.ravel()
    A = np.zeros((ny, nx))
    B = np.zeros((ny, nw))
    for yi, xi, wi in conns:
        A[yi, xi] += wf[wi]
        B[yi, wi] += xf[xi]
    Ho, Wo = wlm.out_hw(geom)
    bias_full = np.broadcast_to(b[None, :, None, None], wlm.tensor_shapes(geom)["dy"]).ravel()
    y_bf = A @ xf + bias_full
    assert _rel(oracle_mod.fwd(geom, x, w, b).ravel(), y_bf) <= 1e-12
    assert _rel(B @ wf + bias_full, y_bf) <= 1e-12
    assert _rel(oracle_mod.bwd_data(geom, dy, w).ravel(), A.T @ dyf) <= 1e-12
    assert _rel(oracle_mod.bwd_weight(geom, x, dy).ravel(), B.T @ dyf) <= 1e-12
    db = dy.reshape(geom[0], geom[4], -1).sum(axis=(0, 2))
    assert _rel(oracle_mod.bwd_bias(geom, dy), db) <= 1e-12


def test_random_geometries_vs_torch_float64(oracle_mod):
    """Library pin: torch conv2d in float64 + autograd, over a seeded sweep."""
    rng = np.random.default_rng(2024)
    for _ in range(40):
        geom = wlm.random_geometry(rng)
        x, w, b, dy = _inputs(rng, geom)
        y_t, dx_t, dw_t, db_t = _torch_ref(geom, x, w, b, dy)
        assert _rel(oracle_mod.fwd(geom, x, w, b), y_t) <= 1e-12, geom
        assert _rel(oracle_mod.bwd_data(geom, dy, w), dx_t) <= 1e-12, geom
        assert _rel(oracle_mod.bwd_weight(geom, x, dy), dw_t) <= 1e-12, geom
        assert _rel(oracle_mod.bwd_bias(geom, dy), db_t) <= 1e-12, geom


def test_per_axis_geometries_vs_torch_float64(oracle_mod):
    """Library pin for per-axis stride and dilation (the cudnn constructor's dW, dH): torch
    conv2d with stride=(s_h, s_w), dilation=(d_h, d_w) in float64 + autograd."""
    rng = np.random.default_rng(2025)
    for _ in range(40):
        geom = wlm.random_geometry(rng, axes=True)
        x, w, b, dy = _inputs(rng, geom)
        y_t, dx_t, dw_t, db_t = _torch_ref(geom, x, w, b, dy)
        assert _rel(oracle_mod.fwd(geom, x, w, b), y_t) <= 1e-12, geom
        assert _rel(oracle_mod.bwd_data(geom, dy, w), dx_t) <= 1e-12, geom
        assert _rel(oracle_mod.bwd_weight(geom, x, dy), dw_t) <= 1e-12, geom
        assert _rel(oracle_mod.bwd_bias(geom, dy), db_t) <= 1e-12, geom


def test_square_geometry_has_one_reading(oracle_mod):
    """A 14-integer geometry and its 16-integer form (equal strides and dilations) are the
    same request: identical results."""
    rng = np.random.default_rng(11)
    for _ in range(10):
        g14 = wlm.random_geometry(rng)
        g16 = wlm.per_axis(g14)
        x, w, b, dy = _inputs(rng, g14)
        assert np.array_equal(oracle_mod.fwd(g14, x, w, b), oracle_mod.fwd(g16, x, w, b))
        assert np.array_equal(oracle_mod.bwd_data(g14, dy, w), oracle_mod.bwd_data(g16, dy, w))
        assert np.array_equal(oracle_mod.bwd_weight(g14, x, dy), oracle_mod.bwd_weight(g16, x, dy))


def _scipy_ungrouped(geom, x, w):
    """O2: an independently written ungrouped conv via scipy correlate2d on the padded
    image, the kernel dilated with zeros, output subsampled by the stride."""
    from scipy.signal import correlate2d
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    assert G == 1
    xp = np.pad(x, ((0, 0), (0, 0), (pt, pb), (pl, pr)))
    kd = np.zeros((Cout, Cin, d * (kH - 1) + 1, d * (kW - 1) + 1))
    kd[:, :, ::d, ::d] = w
    Ho, Wo = wlm.out_hw(geom)
    y = np.zeros((N, Cout, Ho, Wo))
    for n in range(N):
        for o in range(Cout):
            acc = sum(correlate2d(xp[n, c], kd[o, c], mode="valid") for c in range(Cin))
            y[n, o] = acc[::s, ::s][:Ho, :Wo]
    return y


@pytest.mark.parametrize("geom", [
    (2, 3, 9, 8, 4, 3, 3, 1, 1, 1, 1, 1, 1, 1),
    (1, 2, 10, 11, 3, 3, 2, 2, 0, 1, 2, 0, 1, 1),
    (1, 2, 12, 9, 2, 3, 3, 1, 2, 2, 2, 2, 2, 1),
    (2, 3, 6, 6, 5, 6, 6, 1, 0, 0, 0, 0, 1, 1),
])
def test_ungrouped_matches_scipy(oracle_mod, geom):
    rng = np.random.default_rng(11)
    x, w, b, dy = _inputs(rng, geom)
    assert _rel(oracle_mod.fwd(geom, x, w, None), _scipy_ungrouped(geom, x, w)) <= 1e-12


@pytest.mark.parametrize("geom", [
    (2, 12, 7, 6, 8, 3, 3, 1, 1, 1, 1, 1, 1, 4),
    (1, 6, 8, 8, 9, 3, 2, 2, 0, 1, 1, 0, 2, 3),
])
def test_grouped_is_concat_of_narrowed_groups(oracle_mod, geom):
    """O3: a grouped conv equals G ungrouped convs on narrowed channel slices, with
    the weight and bias sliced the same way (the narrow-per-group scheme)."""
    rng = np.random.default_rng(3)
    x, w, b, dy = _inputs(rng, geom)
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = geom
    Cgi, Cgo = Cin // G, Cout // G
    y, dx, dw = oracle_mod.fwd(geom, x, w, b), oracle_mod.bwd_data(geom, dy, w), oracle_mod.bwd_weight(geom, x, dy)
    g1 = (N, Cgi, H, W, Cgo, kH, kW, s, pt, pb, pl, pr, d, 1)
    for g in range(G):
        ci, co = slice(g * Cgi, (g + 1) * Cgi), slice(g * Cgo, (g + 1) * Cgo)
        assert _rel(y[:, co], oracle_mod.fwd(g1, x[:, ci], w[co], b[co])) == 0.0
        assert _rel(dx[:, ci], oracle_mod.bwd_data(g1, dy[:, co], w[co])) == 0.0
        assert _rel(dw[co], oracle_mod.bwd_weight(g1, x[:, ci], dy[:, co])) == 0.0


def test_fc_mode_is_matmul(oracle_mod):
    """O4: input size == kernel size, no pad, dilation 1: y = X W^T + b, dX = dY W, dW = dY^T X."""
    geom = (5, 4, 3, 3, 7, 3, 3, 1, 0, 0, 0, 0, 1, 1)
    rng = np.random.default_rng(5)
    x, w, b, dy = _inputs(rng, geom)
    X, Wm, dY = x.reshape(5, -1), w.reshape(7, -1), dy.reshape(5, 7)
    assert _rel(oracle_mod.fwd(geom, x, w, b).reshape(5, 7), X @ Wm.T + b) <= 1e-13
    assert _rel(oracle_mod.bwd_data(geom, dy, w).reshape(5, -1), dY @ Wm) <= 1e-13
    assert _rel(oracle_mod.bwd_weight(geom, x, dy).reshape(7, -1), dY.T @ X) <= 1e-13


def test_linear_1x1_worked_example(oracle_mod):
    """The page's double-precision 1x1-conv-vs-Linear check: 16x128x1x1 input,
    Linear(128, 32); the printed max abs difference is 8.9e-16, i.e. rounding only."""
    gold = _load_golden("linear_1x1.json")
    n, cin = gold["input_shape"][0], gold["linear_in"]
    cout = gold["linear_out"]
    geom = (n, cin, 1, 1, cout, 1, 1, 1, 0, 0, 0, 0, 1, 1)
    rng = np.random.default_rng(128)
    x = rng.standard_normal((n, cin, 1, 1))
    w = rng.uniform(-1 / np.sqrt(cin), 1 / np.sqrt(cin), (cout, cin))
    b = rng.uniform(-1 / np.sqrt(cin), 1 / np.sqrt(cin), cout)
    lin = x.reshape(n, cin) @ w.T + b
    conv = oracle_mod.fwd(geom, x, w.reshape(cout, cin, 1, 1), b).reshape(n, cout)
    diff = float(np.abs(lin - conv).max())
    # same order as the printed 8.88e-16: a few ulps of values of size ~1
    assert diff <= 16 * gold["printed_max_abs_diff"]


@pytest.mark.parametrize("geom", TINY_GEOMS[1:] + [(2, 8, 9, 7, 6, 3, 3, 2, 1, 0, 2, 1, 2, 2)])
def test_adjoint_identities(oracle_mod, geom):
    """O5: <conv(x,w), r> = <x, bwd_data(r,w)> = <w, bwd_weight(x,r)> (bias off)."""
    rng = np.random.default_rng(17)
    x, w, b, r = _inputs(rng, geom)
    lhs = float(np.sum(oracle_mod.fwd(geom, x, w, None) * r))
    rd = float(np.sum(x * oracle_mod.bwd_data(geom, r, w)))
    rw = float(np.sum(w * oracle_mod.bwd_weight(geom, x, r)))
    scale = max(1.0, abs(lhs))
    assert abs(lhs - rd) / scale <= 1e-12
    assert abs(lhs - rw) / scale <= 1e-12


def test_finite_differences(oracle_mod):
    """O6: central differences of L = <conv(x,w)+b, r> at sampled entries of x, w, b."""
    geom = (2, 6, 7, 6, 4, 3, 2, 2, 1, 0, 0, 1, 1, 2)
    rng = np.random.default_rng(23)
    x, w, b, r = _inputs(rng, geom)
    h = 1e-6

    def L(xx, ww, bb):
        return float(np.sum(oracle_mod.fwd(geom, xx, ww, bb) * r))

    gx, gw, gb = oracle_mod.bwd_data(geom, r, w), oracle_mod.bwd_weight(geom, x, r), oracle_mod.bwd_bias(geom, r)
    for arr, grad, which in ((x, gx, 0), (w, gw, 1), (b, gb, 2)):
        flat = arr.ravel()
        for i in rng.choice(flat.size, size=min(12, flat.size), replace=False):
            plus, minus = flat.copy(), flat.copy()
            plus[i] += h
            minus[i] -= h
            args_p, args_m = [x, w, b], [x, w, b]
            args_p[which] = plus.reshape(arr.shape)
            args_m[which] = minus.reshape(arr.shape)
            fd = (L(*args_p) - L(*args_m)) / (2 * h)
            assert abs(fd - grad.ravel()[i]) <= 1e-6 * max(1.0, abs(fd)), (which, i)


def test_bias_gradient_is_sum_over_n_h_w(oracle_mod):
    """O7: gradBias = np.sum(dy, dims=(0,2,3)) (the broadcast-reduce description)."""
    geom = (3, 4, 5, 5, 6, 3, 3, 1, 1, 1, 1, 1, 1, 2)
    rng = np.random.default_rng(29)
    dy = rng.standard_normal(wlm.tensor_shapes(geom)["dy"])
    assert _rel(oracle_mod.bwd_bias(geom, dy), dy.sum(axis=(0, 2, 3))) <= 1e-13


def test_fc_all_ones_closed_form_small(oracle_mod):
    """O8 on a scaled-down copy: with x = w = b = dy = 1 and input == kernel,
    y = C_in*kH*kW + 1, dx = C_out, dw = N, db = N, exactly."""
    geom = (7, 5, 3, 4, 6, 3, 4, 1, 0, 0, 0, 0, 1, 1)
    sh = wlm.tensor_shapes(geom)
    x, w, b, dy = (np.ones(sh[k]) for k in ("x", "w", "b", "dy"))
    assert np.all(oracle_mod.fwd(geom, x, w, b) == 5 * 3 * 4 + 1)
    assert np.all(oracle_mod.bwd_data(geom, dy, w) == 6)
    assert np.all(oracle_mod.bwd_weight(geom, x, dy) == 7)
    assert np.all(oracle_mod.bwd_bias(geom, dy) == 7)


@pytest.mark.slow
def test_fc_all_ones_page_script(oracle_mod):
    """O8 at the script's own size (1600x256x6x6 -> 4096), sampled: every value
    is an exact integer, consistent with the printed 0.000000 differences."""
    gold = _load_golden("fc_all_ones.json")
    geom = tuple(gold["geom"])
    N, Cin, H, W, Cout, kH, kW = geom[:7]
    sh = wlm.tensor_shapes(geom)
    x = np.ones(sh["x"])
    w = np.ones(sh["w"])
    b = np.ones(sh["b"])
    dy = np.ones(sh["dy"])
    rng = np.random.default_rng(31)
    iy = rng.choice(N * Cout, 200, replace=False)
    ix = rng.choice(N * Cin * H * W, 200, replace=False)
    iw = rng.choice(Cout * Cin * kH * kW, 50, replace=False)
    assert np.all(oracle_mod.fwd_points(geom, x, w, b, iy) == Cin * kH * kW + 1)
    assert np.all(oracle_mod.bwd_data_points(geom, dy, w, ix) == Cout)
    assert np.all(oracle_mod.bwd_weight_points(geom, x, dy, iw) == N)
    assert Cin * kH * kW + 1 == 9217 and Cout == 4096 and N == 1600
    assert all(v == 0.0 for v in gold["printed_sum_abs_diff"].values())


def test_depthwise_is_per_channel_correlation(oracle_mod):
    """O10: G = C_in = C_out equals a per-channel 2D correlation written as its own loop."""
    geom = (2, 5, 6, 7, 5, 3, 3, 1, 1, 1, 1, 1, 1, 5)
    rng = np.random.default_rng(37)
    x, w, b, dy = _inputs(rng, geom)
    xp = np.pad(x, ((0, 0), (0, 0), (1, 1), (1, 1)))
    ref = np.zeros((2, 5, 6, 7))
    for n in range(2):
        for c in range(5):
            for i in range(6):
                for j in range(7):
                    ref[n, c, i, j] = np.sum(xp[n, c, i:i + 3, j:j + 3] * w[c, 0])
    assert _rel(oracle_mod.fwd(geom, x, w, None), ref) <= 1e-13


def test_groups_planes_worked_example(oracle_mod):
    """32 planes in and out with 4 groups of 8: the weight holds G x 8 x 8 filter
    planes (the page's factors; their product is 256, the page prints 128), against
    32 x 32 = 1024 ungrouped; each output plane depends only on its group's 8 inputs."""
    gold = _load_golden("groups_planes.json")
    Cin, Cout, G = gold["C_in"], gold["C_out"], gold["groups"]
    geom = (1, Cin, 5, 5, Cout, 3, 3, 1, 1, 1, 1, 1, 1, G)
    sh = wlm.tensor_shapes(geom)
    f = gold["printed_factors"]
    assert (G, Cin // G, Cout // G) == tuple(f)
    assert sh["w"][0] * sh["w"][1] == f[0] * f[1] * f[2] == 256
    sh1 = wlm.tensor_shapes(geom[:-1] + (1,))
    assert sh1["w"][0] * sh1["w"][1] == gold["filter_planes_ungrouped"]
    rng = np.random.default_rng(41)
    x, w, b, dy = _inputs(rng, geom)
    y0 = oracle_mod.fwd(geom, x, w, b)
    x2 = x.copy()
    x2[:, 8:16] += 1.0  # perturb group 1 only
    y1 = oracle_mod.fwd(geom, x2, w, b)
    changed = np.abs(y1 - y0).reshape(Cout, -1).max(axis=1) > 0
    assert list(np.nonzero(changed)[0]) == list(range(8, 16))


def test_shapes_of_the_workloads(oracle_mod):
    """O11: output shapes of every workload, and the NNlib example's WHCN shapes."""
    expect = {
        "tiny_g5": (2, 15, 26, 26), "alexnet_g2": (128, 256, 27, 27),
        "fc_mode": (1600, 4096, 1, 1), "dense3x3": (32, 64, 56, 56),
        "dense3x3_s2_asym": (32, 64, 28, 28), "resnext_g32": (64, 128, 56, 56),
        "depthwise": (64, 256, 56, 56),
    }
    for name, shp in expect.items():
        geom = wlm.WORKLOADS[name].geom
        assert oracle_mod.shapes(geom)["y"] == shp, name
    gold = _load_golden("nnlib_groups5.json")
    W_, H_, C_, N_ = gold["x_whcn"]
    kw, kh, cgi, cout = gold["w_whio"]
    geom = (N_, C_, H_, W_, cout, kh, kw, 1, 0, 0, 0, 0, 1, gold["groups"])
    assert geom == wlm.WORKLOADS["tiny_g5"].geom
    assert oracle_mod.shapes(geom)["w"] == (cout, cgi, kh, kw)


@pytest.mark.parametrize("bad", [
    (1, 6, 5, 5, 4, 3, 3, 1, 0, 0, 0, 0, 1, 4),     # C_in not divisible by G
    (1, 4, 5, 5, 6, 3, 3, 1, 0, 0, 0, 0, 1, 4),     # C_out not divisible by G
    (1, 4, 2, 5, 4, 3, 3, 1, 0, 0, 0, 0, 1, 1),     # no output row
    (1, 4, 5, 5, 4, 3, 3, 0, 0, 0, 0, 0, 1, 1),     # stride 0
    (1, 4, 5, 5, 4, 3, 3, 1, -1, 0, 0, 0, 1, 1),    # negative pad
    (1, 4, 5, 5, 4, 3, 3, 1, 0, 0, 0, 0, 0, 1),     # dilation 0
])
def test_oracle_rejects_bad_geometry(oracle_mod, bad):
    with pytest.raises(ValueError):
        oracle_mod.out_shape(bad)


def test_untouched_pixels_are_exact_zero(oracle_mod):
    """With stride 3 and a 2x2 kernel, every third input row/column receives no tap."""
    geom = (1, 2, 6, 6, 3, 2, 2, 3, 0, 0, 0, 0, 1, 1)
    rng = np.random.default_rng(43)
    x, w, b, dy = _inputs(rng, geom)
    dx = oracle_mod.bwd_data(geom, dy, w)
    assert np.all(dx[:, :, 2::3, :] == 0.0) and np.all(dx[:, :, :, 2::3] == 0.0)
    assert np.all(dx[:, :, 0:2, 0:2] != 0.0)


def test_points_match_full(oracle_mod):
    geom = (2, 6, 9, 8, 4, 3, 3, 2, 1, 0, 1, 2, 1, 2)
    rng = np.random.default_rng(47)
    x, w, b, dy = _inputs(rng, geom)
    y, dx, dw = oracle_mod.fwd(geom, x, w, b), oracle_mod.bwd_data(geom, dy, w), oracle_mod.bwd_weight(geom, x, dy)
    for full, fn, args in ((y, oracle_mod.fwd_points, (x, w, b)), (dx, oracle_mod.bwd_data_points, (dy, w)),
                           (dw, oracle_mod.bwd_weight_points, (x, dy))):
        idx = rng.choice(full.size, 30, replace=False)
        assert np.array_equal(fn(geom, *args, idx), full.ravel()[idx])


def test_thread_count_does_not_change_results(oracle_mod):
    geom = (2, 8, 10, 9, 6, 3, 3, 1, 1, 1, 1, 1, 1, 2)
    rng = np.random.default_rng(53)
    x, w, b, dy = _inputs(rng, geom)
    assert np.array_equal(oracle_mod.bwd_weight(geom, x, dy, threads=1), oracle_mod.bwd_weight(geom, x, dy, threads=4))
    assert np.array_equal(oracle_mod.fwd(geom, x, w, b, threads=1), oracle_mod.fwd(geom, x, w, b, threads=3))


def test_model_zoo_layers_vs_torch_float64(oracle_mod):
    """Library pin on the full-size channel counts of the model-zoo sweep (ResNeXt-50
    grouped and MobileNet-v2 depthwise 3x3 layers, stride 1 and 2) at batch 1: the oracle
    against torch conv2d in float64 + autograd."""
    rng = np.random.default_rng(77)
    for name, wk in wlm.model_zoo(1).items():
        geom = wk.geom
        x, w, b, dy = _inputs(rng, geom)
        y_t, dx_t, dw_t, db_t = _torch_ref(geom, x, w, b, dy)
        assert _rel(oracle_mod.fwd(geom, x, w, b), y_t) <= 1e-12, name
        assert _rel(oracle_mod.bwd_data(geom, dy, w), dx_t) <= 1e-12, name
        assert _rel(oracle_mod.bwd_weight(geom, x, dy), dw_t) <= 1e-12, name
        assert _rel(oracle_mod.bwd_bias(geom, dy), db_t) <= 1e-12, name
