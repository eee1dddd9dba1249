"""ctypes binding of libgconv.so (include/gconv.h): argument marshalling only.

Every function here forwards to the C entry point of the same name; all
arithmetic runs in the library's CUDA kernels.  There is no CPU fallback: if
libgconv.so is missing the first call raises.  PyTorch only supplies device
memory (tensors, workspaces) and the CUDA stream.

Geometry is the ABI's 14-tuple ``(N, C_in, H, W, C_out, kH, kW, stride, pad_top,
pad_bottom, pad_left, pad_right, dilation, groups)``, or the 16-tuple of the per-axis
entry points ``(N, C_in, H, W, C_out, kH, kW, stride_h, stride_w, pad_top, pad_bottom,
pad_left, pad_right, dilation_h, dilation_w, groups)`` (the ``gconv_geometry`` record);
the tensor-level wrappers derive it from the tensor shapes plus ``stride`` (an int or
(s_h, s_w)), ``padding`` (an int, (p_h, p_w) or (top, bottom, left, right)),
``dilation`` (an int or (d_h, d_w)) and ``groups``.  They call the 14-integer entry
points when the request fits them (equal strides and dilations, fp32 outputs, no fused
bias gradient) and the per-axis ``*_ex`` entry points otherwise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgconv.so")

GCONV_OK, GCONV_ERR_INVALID_ARG, GCONV_ERR_UNSUPPORTED, GCONV_ERR_WORKSPACE, GCONV_ERR_CUDA, \
    GCONV_ERR_TIMEOUT = range(6)
GCONV_F32, GCONV_BF16 = 0, 1
PASS_FWD, PASS_BWD_DATA, PASS_BWD_WEIGHT, PASS_BWD_BIAS = range(4)
PATH_NONE, PATH_DIRECT, PATH_TC_IGEMM, PATH_TC_FC, PATH_REDUCE, PATH_TC_GEMM = range(6)
PATH_NAMES = {PATH_NONE: "none", PATH_DIRECT: "direct", PATH_TC_IGEMM: "tc_igemm",
              PATH_TC_FC: "tc_fc", PATH_REDUCE: "reduce", PATH_TC_GEMM: "tc_gemm1x1"}

EXPORTED = ("gconv_out_shape", "gconv_workspace_size", "gconv_plan", "gconv_fwd", "gconv_bwd_data",
            "gconv_bwd_weight", "gconv_bwd_bias", "gconv_check_device_error", "gconv_status_string",
            "gconv_debug_force_path", "gconv_debug_set_wait_limit", "gconv_debug_set_trace", "gconv_bwd_weight_noalloc",
            "gconv_noalloc_scratch_bytes", "gconv_step_host", "gconv_step_device_bytes",
            "gconv_out_shape_ex", "gconv_workspace_size_ex", "gconv_plan_ex", "gconv_fwd_ex", "gconv_bwd_data_ex",
            "gconv_bwd_weight_ex", "gconv_bwd_bias_ex", "gconv_step_workspace_size_ex", "gconv_step_plan_ex", "gconv_step_ex",
            "gconv_debug_set_step_events", "gconv_debug_set_wgrad_tma")


class Geometry(ctypes.Structure):
    """The gconv_geometry record of include/gconv.h."""
    _fields_ = [(n, ctypes.c_int) for n in ("N", "C_in", "H", "W", "C_out", "kH", "kW", "stride_h", "stride_w",
                                             "pad_top", "pad_bottom", "pad_left", "pad_right", "dilation_h",
                                             "dilation_w", "groups")]


def per_axis(geom):
    """16-integer form of a 14- or 16-integer geometry."""
    g = tuple(int(v) for v in geom)
    if len(g) == 16:
        return g
    if len(g) != 14:
        raise ValueError("geometry must have 14 or 16 integers")
    N, Cin, H, W, Cout, kH, kW, s, pt, pb, pl, pr, d, G = g
    return (N, Cin, H, W, Cout, kH, kW, s, s, pt, pb, pl, pr, d, d, G)


def square(geom):
    """The 14-integer form when strides and dilations agree across axes, else None."""
    g = per_axis(geom)
    N, Cin, H, W, Cout, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, G = g
    if sh != sw or dh != dw:
        return None
    return (N, Cin, H, W, Cout, kH, kW, sh, pt, pb, pl, pr, dh, G)


def geometry_record(geom):
    return Geometry(*per_axis(geom))

_lib = None


class GconvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def lib():
    """Load libgconv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run bwd_gconv_fwd_gb300.build.build() "
                           "(or __graft_entry__.build()) -- there is no fallback path")
    L = ctypes.CDLL(LIB_PATH)
    i, vp, sz = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    geo = [i] * 14
    L.gconv_out_shape.argtypes = geo + [ctypes.POINTER(i), ctypes.POINTER(i)]
    L.gconv_out_shape.restype = i
    L.gconv_workspace_size.argtypes = geo + [i, i]
    L.gconv_workspace_size.restype = sz
    L.gconv_plan.argtypes = geo + [i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
    L.gconv_plan.restype = i
    L.gconv_fwd.argtypes = geo + [i, vp, vp, vp, vp, vp, sz, vp]
    L.gconv_fwd.restype = i
    L.gconv_bwd_data.argtypes = geo + [i, vp, vp, vp, vp, sz, vp]
    L.gconv_bwd_data.restype = i
    L.gconv_bwd_weight.argtypes = geo + [i, vp, vp, vp, vp, sz, vp]
    L.gconv_bwd_weight.restype = i
    L.gconv_bwd_bias.argtypes = geo + [i, vp, vp, vp, sz, vp]
    L.gconv_bwd_bias.restype = i
    L.gconv_bwd_weight_noalloc.argtypes = geo + [i, vp, vp, vp, vp]
    L.gconv_bwd_weight_noalloc.restype = i
    L.gconv_noalloc_scratch_bytes.argtypes = []
    L.gconv_noalloc_scratch_bytes.restype = sz
    L.gconv_step_host.argtypes = geo + [i, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.gconv_step_host.restype = i
    L.gconv_step_device_bytes.argtypes = geo + [i, i]
    L.gconv_step_device_bytes.restype = sz
    L.gconv_check_device_error.argtypes = [vp]
    L.gconv_check_device_error.restype = i
    L.gconv_status_string.argtypes = [i]
    L.gconv_status_string.restype = ctypes.c_char_p
    L.gconv_debug_force_path.argtypes = [i]
    L.gconv_debug_force_path.restype = None
    L.gconv_debug_set_wait_limit.argtypes = [ctypes.c_longlong]
    L.gconv_debug_set_wait_limit.restype = None
    L.gconv_debug_set_wgrad_tma.argtypes = [i]
    L.gconv_debug_set_wgrad_tma.restype = None
    L.gconv_debug_set_trace.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    L.gconv_debug_set_trace.restype = None
    gp = ctypes.POINTER(Geometry)
    L.gconv_out_shape_ex.argtypes = [gp, ctypes.POINTER(i), ctypes.POINTER(i)]
    L.gconv_out_shape_ex.restype = i
    L.gconv_workspace_size_ex.argtypes = [gp, i, i]
    L.gconv_workspace_size_ex.restype = sz
    L.gconv_plan_ex.argtypes = [gp, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
    L.gconv_plan_ex.restype = i
    L.gconv_fwd_ex.argtypes = [gp, i, i, vp, vp, vp, vp, vp, sz, vp]
    L.gconv_fwd_ex.restype = i
    L.gconv_bwd_data_ex.argtypes = [gp, i, i, vp, vp, vp, vp, sz, vp]
    L.gconv_bwd_data_ex.restype = i
    L.gconv_bwd_weight_ex.argtypes = [gp, i, vp, vp, vp, vp, vp, sz, vp]
    L.gconv_bwd_weight_ex.restype = i
    L.gconv_bwd_bias_ex.argtypes = [gp, i, vp, vp, vp, sz, vp]
    L.gconv_bwd_bias_ex.restype = i
    L.gconv_step_workspace_size_ex.argtypes = [gp, i]
    L.gconv_step_workspace_size_ex.restype = sz
    L.gconv_step_ex.argtypes = [gp, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.gconv_step_ex.restype = i
    L.gconv_step_plan_ex.argtypes = [gp, i, ctypes.POINTER(i), ctypes.POINTER(i)]
    L.gconv_step_plan_ex.restype = i
    L.gconv_debug_set_step_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i]
    L.gconv_debug_set_step_events.restype = None
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().gconv_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != GCONV_OK:
        raise GconvError(status, what)


# ---- host-only queries ---------------------------------------------------------

def gconv_out_shape(geom):
    ho, wo = ctypes.c_int(), ctypes.c_int()
    if len(geom) == 16:
        rec = geometry_record(geom)
        _check(lib().gconv_out_shape_ex(ctypes.byref(rec), ctypes.byref(ho), ctypes.byref(wo)), "gconv_out_shape_ex")
    else:
        _check(lib().gconv_out_shape(*map(int, geom), ctypes.byref(ho), ctypes.byref(wo)), "gconv_out_shape")
    return ho.value, wo.value


def gconv_workspace_size(geom, dtype: int, pass_: int) -> int:
    if len(geom) == 16:
        rec = geometry_record(geom)
        n = lib().gconv_workspace_size_ex(ctypes.byref(rec), int(dtype), int(pass_))
    else:
        n = lib().gconv_workspace_size(*map(int, geom), int(dtype), int(pass_))
    if n == ctypes.c_size_t(-1).value:
        raise GconvError(GCONV_ERR_INVALID_ARG, "gconv_workspace_size")
    return int(n)


def gconv_plan(geom, dtype: int, pass_: int):
    """(path, launches) the library would use for this call."""
    path, launches = ctypes.c_int(), ctypes.c_int()
    if len(geom) == 16:
        rec = geometry_record(geom)
        _check(lib().gconv_plan_ex(ctypes.byref(rec), int(dtype), int(pass_), ctypes.byref(path),
                                   ctypes.byref(launches)), "gconv_plan_ex")
    else:
        _check(lib().gconv_plan(*map(int, geom), int(dtype), int(pass_), ctypes.byref(path),
                                ctypes.byref(launches)), "gconv_plan")
    return path.value, launches.value


def gconv_step_workspace_size(geom, dtype: int) -> int:
    """Workspace bytes gconv_step_ex needs for this geometry (14 or 16 integers)."""
    rec = geometry_record(per_axis(geom))
    n = lib().gconv_step_workspace_size_ex(ctypes.byref(rec), int(dtype))
    if n == ctypes.c_size_t(-1).value:
        raise GconvError(GCONV_ERR_INVALID_ARG, "gconv_step_workspace_size_ex")
    return int(n)


def gconv_step_plan(geom, dtype: int):
    """(shared, launches) of gconv_step_ex for this geometry: whether the passes share their
    blocked copies, and the step's kernel launches without db."""
    rec = geometry_record(per_axis(geom))
    shared, launches = ctypes.c_int(), ctypes.c_int()
    _check(lib().gconv_step_plan_ex(ctypes.byref(rec), int(dtype), ctypes.byref(shared), ctypes.byref(launches)),
           "gconv_step_plan_ex")
    return bool(shared.value), launches.value


def gconv_debug_force_path(path: int):
    lib().gconv_debug_force_path(int(path))


def gconv_debug_set_wait_limit(limit: int):
    lib().gconv_debug_set_wait_limit(int(limit))


def gconv_debug_set_wgrad_tma(enable: bool):
    """Test hook: False makes the tensor-core weight gradient stage its tiles by cp.async."""
    lib().gconv_debug_set_wgrad_tma(1 if enable else 0)



def gconv_debug_set_trace(device_ptr: int, nbytes: int):
    """Sets (or, with 0, clears) the device buffer the correlation kernel writes phase stamps to."""
    lib().gconv_debug_set_trace(ctypes.c_void_p(device_ptr or None), int(nbytes))


def gconv_debug_set_step_events(events):
    """Sets (a sequence of four torch.cuda.Event, each recorded once so that it exists) or,
    with None, clears the events gconv_step_ex records at its pass boundaries."""
    if not events:
        lib().gconv_debug_set_step_events(None, 0)
        return
    if len(events) != 4:
        raise ValueError("four events: start, after forward, after backward-data, after the weight gradient")
    arr = (ctypes.c_void_p * 4)(*(ctypes.c_void_p(e.cuda_event) for e in events))
    lib().gconv_debug_set_step_events(arr, 4)


def gconv_check_device_error(stream=None) -> int:
    """Synchronise the stream and return the status of the device error word."""
    return int(lib().gconv_check_device_error(_stream_ptr(stream)))


# ---- marshalling helpers -----------------------------------------------------

def _stream_ptr(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return GCONV_BF16
    if t == torch.float32:
        return GCONV_F32
    raise TypeError(f"unsupported input dtype {t}; use bfloat16 or float32")


def _pads(padding):
    if isinstance(padding, int):
        return (padding,) * 4
    p = tuple(int(v) for v in padding)
    if len(p) == 2:
        return (p[0], p[0], p[1], p[1])
    if len(p) != 4:
        raise ValueError("padding is an int, (ph, pw) or (top, bottom, left, right)")
    return p


def _pair(v):
    if isinstance(v, int):
        return int(v), int(v)
    a, b = (int(u) for u in v)
    return a, b


def geometry(x_shape, w_shape, stride=1, padding=0, dilation=1, groups=1):
    """The ABI geometry: a 14-tuple when strides and dilations agree across axes, else the
    16-tuple of the per-axis entry points."""
    N, Cin, H, W = (int(v) for v in x_shape)
    Cout, cgi, kH, kW = (int(v) for v in w_shape)
    if cgi * int(groups) != Cin:
        raise GconvError(GCONV_ERR_INVALID_ARG, f"weight has {cgi} input channels per group, "
                                                f"x has {Cin} channels for {groups} groups")
    pt, pb, pl, pr = _pads(padding)
    sh, sw = _pair(stride)
    dh, dw = _pair(dilation)
    if sh == sw and dh == dw:
        return (N, Cin, H, W, Cout, kH, kW, sh, pt, pb, pl, pr, dh, int(groups))
    return (N, Cin, H, W, Cout, kH, kW, sh, sw, pt, pb, pl, pr, dh, dw, int(groups))


def _dev(t: torch.Tensor, name: str):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _workspace(geom, dt, pass_, workspace, device):
    need = gconv_workspace_size(geom, dt, pass_)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


# ---- the four passes (tensor level) -------------------------------------------

def _out_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return GCONV_F32
    if t.dtype == torch.bfloat16:
        return GCONV_BF16
    raise TypeError(f"unsupported output dtype {t.dtype}; use float32 or bfloat16")


def gconv_fwd(x, w, bias, y, *, stride=1, padding=0, dilation=1, groups=1, workspace=None, stream=None):
    """y <- conv(x, w) + bias (bias may be None).  y: fp32 or bf16 [N, C_out, Ho, Wo]."""
    geom = geometry(x.shape, w.shape, stride, padding, dilation, groups)
    dt, odt = dtype_code(x.dtype), _out_code(y)
    ws, wsb = _workspace(geom, dt, PASS_FWD, workspace, x.device)
    args = (_dev(x, "x"), _dev(w, "w"), _dev(bias, "bias"), _dev(y, "y"), ws, wsb, _stream_ptr(stream))
    if len(geom) == 14 and odt == GCONV_F32:
        _check(lib().gconv_fwd(*geom, dt, *args), "gconv_fwd")
    else:
        rec = geometry_record(geom)
        _check(lib().gconv_fwd_ex(ctypes.byref(rec), dt, odt, *args), "gconv_fwd_ex")
    return y


def gconv_bwd_data(dy, w, dx, *, stride=1, padding=0, dilation=1, groups=1, workspace=None, stream=None):
    """dx <- gradient of <y, dy> w.r.t. x.  dx: fp32 or bf16 [N, C_in, H, W]."""
    geom = geometry(dx.shape, w.shape, stride, padding, dilation, groups)
    dt, odt = dtype_code(dy.dtype), _out_code(dx)
    ws, wsb = _workspace(geom, dt, PASS_BWD_DATA, workspace, dy.device)
    args = (_dev(dy, "dy"), _dev(w, "w"), _dev(dx, "dx"), ws, wsb, _stream_ptr(stream))
    if len(geom) == 14 and odt == GCONV_F32:
        _check(lib().gconv_bwd_data(*geom, dt, *args), "gconv_bwd_data")
    else:
        rec = geometry_record(geom)
        _check(lib().gconv_bwd_data_ex(ctypes.byref(rec), dt, odt, *args), "gconv_bwd_data_ex")
    return dx


def gconv_bwd_weight(x, dy, dw, *, db=None, stride=1, padding=0, dilation=1, groups=1, workspace=None,
                     stream=None):
    """dw <- gradient of <y, dy> w.r.t. w, fp32 [C_out, C_in/G, kH, kW]; with db (fp32
    [C_out]) also the bias gradient of the same dy, in the same call."""
    geom = geometry(x.shape, dw.shape, stride, padding, dilation, groups)
    dt = dtype_code(x.dtype)
    ws, wsb = _workspace(geom, dt, PASS_BWD_WEIGHT, workspace, x.device)
    if len(geom) == 14 and db is None:
        _check(lib().gconv_bwd_weight(*geom, dt, _dev(x, "x"), _dev(dy, "dy"), _dev(dw, "dw"), ws, wsb,
                                      _stream_ptr(stream)), "gconv_bwd_weight")
    else:
        rec = geometry_record(geom)
        _check(lib().gconv_bwd_weight_ex(ctypes.byref(rec), dt, _dev(x, "x"), _dev(dy, "dy"), _dev(dw, "dw"),
                                         _dev(db, "db"), ws, wsb, _stream_ptr(stream)), "gconv_bwd_weight_ex")
    return dw


def gconv_bwd_weight_noalloc(x, dy, dw, *, stride=1, padding=0, dilation=1, groups=1, stream=None):
    """dw <- gradient w.r.t. w, using the library's fixed scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/gconv.h)."""
    geom = geometry(x.shape, dw.shape, stride, padding, dilation, groups)
    dt = dtype_code(x.dtype)
    _check(lib().gconv_bwd_weight_noalloc(*geom, dt, _dev(x, "x"), _dev(dy, "dy"), _dev(dw, "dw"),
                                          _stream_ptr(stream)), "gconv_bwd_weight_noalloc")
    return dw


def gconv_noalloc_scratch_bytes() -> int:
    return int(lib().gconv_noalloc_scratch_bytes())


def gconv_step_device_bytes(geom, dtype: int, with_bias: bool = True) -> int:
    n = lib().gconv_step_device_bytes(*map(int, geom), int(dtype), int(bool(with_bias)))
    if n == ctypes.c_size_t(-1).value:
        raise GconvError(GCONV_ERR_INVALID_ARG, "gconv_step_device_bytes")
    return int(n)


def _host(t, name: str):
    if t is None:
        return None
    if t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host tensor")
    return ctypes.c_void_p(t.data_ptr())


def gconv_step(x, w, bias, dy, y, dx, dw, db=None, *, stride=1, padding=0, dilation=1, groups=1, workspace=None,
               stream=None):
    """One step on device tensors: y <- forward(x, w, bias), dx <- backward-data(dy, w),
    dw <- weight gradient(x, dy) and, with db, the bias gradient; y and dx fp32 or bf16
    (the same dtype), dw and db fp32.  Equal bit for bit to the separate passes."""
    geom = per_axis(geometry(x.shape, w.shape, stride, padding, dilation, groups))
    dt, odt = dtype_code(x.dtype), _out_code(y)
    if _out_code(dx) != odt:
        raise TypeError("y and dx must have the same dtype")
    need = gconv_step_workspace_size(geom, dt)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws = ctypes.c_void_p(workspace.data_ptr()) if need else None
    wsb = workspace.numel() * workspace.element_size() if need else 0
    rec = geometry_record(geom)
    _check(lib().gconv_step_ex(ctypes.byref(rec), dt, odt, _dev(x, "x"), _dev(w, "w"), _dev(bias, "bias"),
                               _dev(dy, "dy"), _dev(y, "y"), _dev(dx, "dx"), _dev(dw, "dw"), _dev(db, "db"), ws, wsb,
                               _stream_ptr(stream)), "gconv_step_ex")
    return y, dx, dw, db


def gconv_step_host(x, w, bias, dy, y, dx, dw, db, device_buffer, *, stride=1, padding=0, dilation=1,
                    groups=1, stream=None):
    """One step on host tensors (pinned for overlap): inputs copied in, the four passes,
    y/dx/dw/db copied back; done when `stream` reaches this point (see include/gconv.h)."""
    geom = geometry(x.shape, w.shape, stride, padding, dilation, groups)
    dt = dtype_code(x.dtype)
    if not device_buffer.is_cuda:
        raise ValueError("device_buffer must be a device tensor")
    _check(lib().gconv_step_host(*geom, dt, _host(x, "x"), _host(w, "w"), _host(bias, "bias"), _host(dy, "dy"),
                                 _host(y, "y"), _host(dx, "dx"), _host(dw, "dw"), _host(db, "db"),
                                 ctypes.c_void_p(device_buffer.data_ptr()),
                                 device_buffer.numel() * device_buffer.element_size(), _stream_ptr(stream)),
           "gconv_step_host")


def gconv_step_host_ptr(geom, dt, x, w, bias, dy, y, dx, dw, db, buf, buf_bytes, stream=0):
    """Pointer-level form of gconv_step_host (host pointers for tensors, a device buffer)."""
    _check(lib().gconv_step_host(*map(int, geom), int(dt), x, w, bias or None, dy, y, dx, dw, db, buf,
                                 int(buf_bytes), stream or None), "gconv_step_host")


def gconv_bwd_bias(dy, db, *, geom=None, workspace=None, stream=None):
    """db <- sum of dy over (N, Ho, Wo).  geom defaults to a 1x1 geometry on dy's shape."""
    if geom is None:
        N, C, Ho, Wo = (int(v) for v in dy.shape)
        geom = (N, C, Ho, Wo, C, 1, 1, 1, 0, 0, 0, 0, 1, 1)
    dt = dtype_code(dy.dtype)
    ws, wsb = _workspace(geom, dt, PASS_BWD_BIAS, workspace, dy.device)
    if len(geom) == 14:
        _check(lib().gconv_bwd_bias(*geom, dt, _dev(dy, "dy"), _dev(db, "db"), ws, wsb, _stream_ptr(stream)),
               "gconv_bwd_bias")
    else:
        rec = geometry_record(geom)
        _check(lib().gconv_bwd_bias_ex(ctypes.byref(rec), dt, _dev(dy, "dy"), _dev(db, "db"), ws, wsb,
                                       _stream_ptr(stream)), "gconv_bwd_bias_ex")
    return db


# ---- raw pointer level (same C signatures), for callers holding pointers ------

def gconv_fwd_ptr(geom, dt, x, w, bias, y, ws=0, ws_bytes=0, stream=0):
    _check(lib().gconv_fwd(*map(int, geom), int(dt), x, w, bias or None, y, ws or None, int(ws_bytes),
                           stream or None), "gconv_fwd")


def gconv_bwd_data_ptr(geom, dt, dy, w, dx, ws=0, ws_bytes=0, stream=0):
    _check(lib().gconv_bwd_data(*map(int, geom), int(dt), dy, w, dx, ws or None, int(ws_bytes),
                                stream or None), "gconv_bwd_data")


def gconv_bwd_weight_ptr(geom, dt, x, dy, dw, ws=0, ws_bytes=0, stream=0):
    _check(lib().gconv_bwd_weight(*map(int, geom), int(dt), x, dy, dw, ws or None, int(ws_bytes),
                                  stream or None), "gconv_bwd_weight")


def gconv_bwd_bias_ptr(geom, dt, dy, db, ws=0, ws_bytes=0, stream=0):
    _check(lib().gconv_bwd_bias(*map(int, geom), int(dt), dy, db, ws or None, int(ws_bytes),
                                stream or None), "gconv_bwd_bias")


# ---- per-axis entry points at pointer level (16-integer geometry) ------------

def gconv_fwd_ex_ptr(geom, dt, out_dt, x, w, bias, y, ws=0, ws_bytes=0, stream=0):
    rec = geometry_record(geom)
    _check(lib().gconv_fwd_ex(ctypes.byref(rec), int(dt), int(out_dt), x, w, bias or None, y, ws or None,
                              int(ws_bytes), stream or None), "gconv_fwd_ex")


def gconv_bwd_data_ex_ptr(geom, dt, out_dt, dy, w, dx, ws=0, ws_bytes=0, stream=0):
    rec = geometry_record(geom)
    _check(lib().gconv_bwd_data_ex(ctypes.byref(rec), int(dt), int(out_dt), dy, w, dx, ws or None, int(ws_bytes),
                                   stream or None), "gconv_bwd_data_ex")


def gconv_step_ex_ptr(geom, dt, out_dt, x, w, bias, dy, y, dx, dw, db=0, ws=0, ws_bytes=0, stream=0):
    """Pointer-level gconv_step_ex: y, dx, dw and (db not 0) db of one layer in one call."""
    rec = geometry_record(per_axis(geom))
    _check(lib().gconv_step_ex(ctypes.byref(rec), int(dt), int(out_dt), x, w, bias or None, dy, y, dx, dw,
                               db or None, ws or None, int(ws_bytes), stream or None), "gconv_step_ex")


def gconv_bwd_weight_ex_ptr(geom, dt, x, dy, dw, db=0, ws=0, ws_bytes=0, stream=0):
    rec = geometry_record(geom)
    _check(lib().gconv_bwd_weight_ex(ctypes.byref(rec), int(dt), x, dy, dw, db or None, ws or None, int(ws_bytes),
                                     stream or None), "gconv_bwd_weight_ex")
