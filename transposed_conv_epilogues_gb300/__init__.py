"""GB300 (sm_103a) 3-D convolution and transposed convolution with fused epilogues.

Python binding of the C ABI in ``include/tc3d.h`` (``libtc3d.so``): argument
marshalling only.  Every step of the computation runs in the library's CUDA
kernels; PyTorch supplies device memory and the current stream.  There is no
CPU or PyTorch fallback: if the library cannot be loaded, every call raises.

Entry points (same names as the C ABI, without the ``tc3d_`` prefix):

* ``conv3d_fwd(x, w, bias, stride, padding, dilation, groups)``
* ``conv3d_fwd_ndhwc(x, w, bias, stride, padding, dilation, groups)`` (x, y channels-last)
* ``conv_transpose3d_fwd(x, w, bias, stride, padding, dilation, output_padding, groups)``
* ``conv_maxpool_lse_relu(x, w, bias, stride, padding, dilation, groups)``
* ``convT_bn_avgpool(x, w, bias, gamma, beta, eps, stride, padding, dilation,
  output_padding, groups)``
* ``convT_bneval_avgpool(x, w, bias, running_mean, running_var, gamma, beta, eps,
  stride, padding, dilation, output_padding, groups)``

Host-only queries: ``out_shape``, ``workspace_bytes``, ``plan_describe``,
``status_string``; device diagnostics: ``last_device_error``,
``set_wait_timeout_ns``, ``selftest_wait_timeout``.
"""
from __future__ import annotations

import ctypes
import json
from pathlib import Path

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libtc3d.so"

OP_CONV3D = 0
OP_CONV_TRANSPOSE3D = 1
OP_CONV_MAXPOOL_LSE_RELU = 2
OP_CONVT_BN_AVGPOOL = 3
OP_CONVT_BNEVAL_AVGPOOL = 4
OP_CONV3D_NDHWC = 5

TC3D_OK = 0
TC3D_ERR_NULL = -1
TC3D_ERR_SHAPE = -2
TC3D_ERR_GROUPS = -3
TC3D_ERR_OUTPUT_PADDING = -4
TC3D_ERR_ALIGN = -5
TC3D_ERR_WORKSPACE = -6
TC3D_ERR_UNSUPPORTED = -7
TC3D_ERR_CUDA = -8
TC3D_ERR_DEVICE_TIMEOUT = -9
TC3D_ERR_DEVICE = -10

EXPORTED = [
    "tc3d_conv3d_fwd", "tc3d_conv_transpose3d_fwd", "tc3d_conv_maxpool_lse_relu",
    "tc3d_convT_bn_avgpool", "tc3d_workspace_bytes", "tc3d_out_shape", "tc3d_plan_describe",
    "tc3d_last_device_error", "tc3d_set_wait_timeout_ns", "tc3d_selftest_wait_timeout",
    "tc3d_status_string", "tc3d_conv_maxpool_lse_relu_noalloc", "tc3d_convT_bneval_avgpool",
    "tc3d_conv3d_fwd_ndhwc",
]

_lib = None
_I3 = ctypes.c_int * 3
_P = ctypes.c_void_p
_I = ctypes.c_int


class Tc3dError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: tc3d status {status} ({status_string(status)})")


def load(path: str | Path | None = None):
    """Load libtc3d.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = Path(path) if path else LIB_PATH
    if not p.exists():
        raise RuntimeError(
            f"tc3d CUDA library not found at {p}; build it with "
            "transposed_conv_epilogues_gb300.build.build()")
    lib = ctypes.CDLL(str(p))
    geom = [_I] * 9 + [_I3, _I3, _I3, _I3, _I]  # N Cin S0 S1 S2 Cout k0 k1 k2 | s p d op | groups
    tail = [_P, ctypes.c_size_t, _P]  # workspace, bytes, stream
    for name in ("tc3d_conv3d_fwd", "tc3d_conv_transpose3d_fwd", "tc3d_conv_maxpool_lse_relu",
                 "tc3d_conv3d_fwd_ndhwc"):
        f = getattr(lib, name)
        f.argtypes = [_P, _P, _P, _P] + geom + tail
        f.restype = _I
    lib.tc3d_conv_maxpool_lse_relu_noalloc.argtypes = [_P, _P, _P, _P] + geom + [_P]
    lib.tc3d_conv_maxpool_lse_relu_noalloc.restype = _I
    lib.tc3d_convT_bn_avgpool.argtypes = [_P, _P, _P, _P, _P, ctypes.c_float, _P] + geom + tail
    lib.tc3d_convT_bn_avgpool.restype = _I
    lib.tc3d_convT_bneval_avgpool.argtypes = ([_P] * 7 + [ctypes.c_float, _P]) + geom + tail
    lib.tc3d_convT_bneval_avgpool.restype = _I
    lib.tc3d_workspace_bytes.argtypes = [_I] + geom + [ctypes.POINTER(ctypes.c_size_t)]
    lib.tc3d_workspace_bytes.restype = _I
    lib.tc3d_out_shape.argtypes = [_I] + geom + [ctypes.POINTER(ctypes.c_int64)]
    lib.tc3d_out_shape.restype = _I
    lib.tc3d_plan_describe.argtypes = [_I] + geom + [ctypes.c_char_p, ctypes.c_size_t]
    lib.tc3d_plan_describe.restype = _I
    lib.tc3d_last_device_error.argtypes = [_P]
    lib.tc3d_last_device_error.restype = _I
    lib.tc3d_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.tc3d_set_wait_timeout_ns.restype = None
    lib.tc3d_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _P]
    lib.tc3d_selftest_wait_timeout.restype = _I
    lib.tc3d_status_string.argtypes = [_I]
    lib.tc3d_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().tc3d_status_string(int(status)).decode()


def _t3(v, default):
    if v is None:
        v = default
    if isinstance(v, int):
        return (int(v),) * 3
    v = tuple(int(t) for t in v)
    if len(v) != 3:
        raise ValueError("expected an int or 3 ints")
    return v


def _geom(x_shape, w_shape, transposed, stride, padding, dilation, output_padding, groups):
    N, Cin, S0, S1, S2 = (int(v) for v in x_shape)
    k0, k1, k2 = (int(v) for v in w_shape[2:])
    Cout = int(w_shape[1]) * int(groups) if transposed else int(w_shape[0])
    return (N, Cin, S0, S1, S2, Cout, k0, k1, k2, _I3(*_t3(stride, 1)), _I3(*_t3(padding, 0)),
            _I3(*_t3(dilation, 1)), _I3(*_t3(output_padding, 0)), int(groups))


def _is_transposed(op):
    return op in (OP_CONV_TRANSPOSE3D, OP_CONVT_BN_AVGPOOL, OP_CONVT_BNEVAL_AVGPOOL)


def out_shape(op, x_shape, w_shape, stride=1, padding=0, dilation=1, output_padding=0, groups=1):
    g = _geom(x_shape, w_shape, _is_transposed(op), stride, padding, dilation, output_padding,
              groups)
    dims = (ctypes.c_int64 * 5)()
    rc = load().tc3d_out_shape(op, *g, dims)
    if rc:
        raise Tc3dError(rc, "out_shape")
    return tuple(int(v) for v in dims)


def workspace_bytes(op, x_shape, w_shape, stride=1, padding=0, dilation=1, output_padding=0,
                    groups=1):
    g = _geom(x_shape, w_shape, _is_transposed(op), stride, padding, dilation, output_padding,
              groups)
    n = ctypes.c_size_t(0)
    rc = load().tc3d_workspace_bytes(op, *g, ctypes.byref(n))
    if rc:
        raise Tc3dError(rc, "workspace_bytes")
    return int(n.value)


def plan_describe(op, x_shape, w_shape, stride=1, padding=0, dilation=1, output_padding=0,
                  groups=1) -> dict:
    g = _geom(x_shape, w_shape, _is_transposed(op), stride, padding, dilation, output_padding,
              groups)
    buf = ctypes.create_string_buffer(1 << 16)
    load().tc3d_plan_describe(op, *g, buf, len(buf))
    return json.loads(buf.value.decode())


# ---------------------------------------------------------------------------
# device entry points (torch tensors for memory and stream only)
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tensor(t, name, device=None):
    torch = _torch()
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError(f"{name} must be a float32 CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (NCDHW)")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _check_weight(op, xs, ws, bias, groups):
    """The C ABI receives only pointers; the tensor shapes are checked here."""
    Cin = int(xs[1])
    if _is_transposed(op):
        ok = int(ws[0]) == Cin
        cout = int(ws[1]) * int(groups)
    else:
        ok = int(ws[1]) * int(groups) == Cin
        cout = int(ws[0])
    if not ok:
        raise ValueError(f"weight shape {tuple(ws)} does not match {Cin} input channels "
                         f"and groups={groups}")
    if bias is not None and bias.numel() != cout:
        raise ValueError(f"bias has {bias.numel()} elements, expected {cout}")


def _stream(stream, device):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if workspace is not None:
        return workspace  # its size is checked by the library (TC3D_ERR_WORKSPACE)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _run(op, x, w, bias, stride, padding, dilation, output_padding, groups, out, workspace,
         stream, extra=None):
    torch = _torch()
    lib = load()
    dev = x.device
    for t, n in ((x, "x"), (w, "w"), (bias, "bias"), (out, "out")):
        _check_tensor(t, n, dev)
    if x.dim() != 5 or w.dim() != 5:
        raise ValueError("x and w must be 5-D (NCDHW / [*, *, k0, k1, k2])")
    # shapes in NCDHW terms (channels-last x is [N, S0, S1, S2, C])
    xs = tuple(x.shape)
    if op == OP_CONV3D_NDHWC:
        xs = (xs[0], xs[4], xs[1], xs[2], xs[3])
    _check_weight(op, xs, w.shape, bias, groups)
    shp = out_shape(op, xs, w.shape, stride, padding, dilation, output_padding, groups)
    if out is None:
        out = torch.empty(shp, dtype=torch.float32, device=dev)
    elif tuple(out.shape) != shp:
        raise ValueError(f"out has shape {tuple(out.shape)}, expected {shp}")
    nbytes = workspace_bytes(op, xs, w.shape, stride, padding, dilation, output_padding, groups)
    ws = _workspace(nbytes, dev, workspace)
    g = _geom(xs, w.shape, _is_transposed(op), stride, padding, dilation, output_padding, groups)
    tail = (ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(ws.numel() * ws.element_size()),
            _stream(stream, dev))
    with torch.cuda.device(dev):
        if op == OP_CONV3D:
            rc = lib.tc3d_conv3d_fwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), *g, *tail)
        elif op == OP_CONV3D_NDHWC:
            rc = lib.tc3d_conv3d_fwd_ndhwc(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), *g, *tail)
        elif op == OP_CONV_TRANSPOSE3D:
            rc = lib.tc3d_conv_transpose3d_fwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), *g, *tail)
        elif op == OP_CONV_MAXPOOL_LSE_RELU:
            rc = lib.tc3d_conv_maxpool_lse_relu(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), *g,
                                                *tail)
        else:
            gamma, beta, eps, rmean, rvar = extra
            for t, n in ((gamma, "gamma"), (beta, "beta"), (rmean, "running_mean"),
                         (rvar, "running_var")):
                _check_tensor(t, n, dev)
                if t is not None and t.numel() != shp[1]:
                    raise ValueError(f"{n} has {t.numel()} elements, expected {shp[1]}")
            if op == OP_CONVT_BN_AVGPOOL:
                rc = lib.tc3d_convT_bn_avgpool(_ptr(x), _ptr(w), _ptr(bias), _ptr(gamma),
                                               _ptr(beta), ctypes.c_float(eps), _ptr(out), *g,
                                               *tail)
            else:
                if rmean is None or rvar is None:
                    raise ValueError("running_mean and running_var are required")
                rc = lib.tc3d_convT_bneval_avgpool(_ptr(x), _ptr(w), _ptr(bias), _ptr(rmean),
                                                   _ptr(rvar), _ptr(gamma), _ptr(beta),
                                                   ctypes.c_float(eps), _ptr(out), *g, *tail)
    if rc:
        raise Tc3dError(rc, ["conv3d_fwd", "conv_transpose3d_fwd", "conv_maxpool_lse_relu",
                             "convT_bn_avgpool", "convT_bneval_avgpool",
                             "conv3d_fwd_ndhwc"][op])
    return out


def conv3d_fwd(x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, out=None,
               workspace=None, stream=None):
    """Conv3d forward; w [Cout, Cin/groups, k0, k1, k2]."""
    return _run(OP_CONV3D, x, w, bias, stride, padding, dilation, 0, groups, out, workspace,
                stream)


def conv3d_fwd_ndhwc(x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, out=None,
                     workspace=None, stream=None):
    """Conv3d forward on channels-last tensors: x [N, S0, S1, S2, Cin] ->
    y [N, O0, O1, O2, Cout]; w [Cout, Cin/groups, k0, k1, k2]."""
    return _run(OP_CONV3D_NDHWC, x, w, bias, stride, padding, dilation, 0, groups, out, workspace,
                stream)


def conv_transpose3d_fwd(x, w, bias=None, stride=1, padding=0, dilation=1, output_padding=0,
                         groups=1, out=None, workspace=None, stream=None):
    """ConvTranspose3d forward; w [Cin, Cout/groups, k0, k1, k2]."""
    return _run(OP_CONV_TRANSPOSE3D, x, w, bias, stride, padding, dilation, output_padding,
                groups, out, workspace, stream)


def conv_maxpool_lse_relu(x, w, bias=None, stride=1, padding=0, dilation=1, groups=1, out=None,
                          workspace=None, stream=None):
    """Conv3d -> MaxPool3d(2,2) -> logsumexp over channels -> ReLU; y [N,1,O/2...]."""
    return _run(OP_CONV_MAXPOOL_LSE_RELU, x, w, bias, stride, padding, dilation, 0, groups, out,
                workspace, stream)


def convT_bn_avgpool(x, w, bias=None, gamma=None, beta=None, eps=1e-5, stride=1, padding=0,
                     dilation=1, output_padding=0, groups=1, out=None, workspace=None,
                     stream=None):
    """ConvTranspose3d -> BatchNorm3d (batch stats) -> AvgPool3d(2) -> AvgPool3d(2)."""
    return _run(OP_CONVT_BN_AVGPOOL, x, w, bias, stride, padding, dilation, output_padding,
                groups, out, workspace, stream, extra=(gamma, beta, float(eps), None, None))


def convT_bneval_avgpool(x, w, bias=None, running_mean=None, running_var=None, gamma=None,
                         beta=None, eps=1e-5, stride=1, padding=0, dilation=1, output_padding=0,
                         groups=1, out=None, workspace=None, stream=None):
    """ConvTranspose3d -> BatchNorm3d (running stats, evaluation mode) -> AvgPool3d(2)
    -> AvgPool3d(2).  running_mean / running_var are read, never updated."""
    return _run(OP_CONVT_BNEVAL_AVGPOOL, x, w, bias, stride, padding, dilation, output_padding,
                groups, out, workspace, stream,
                extra=(gamma, beta, float(eps), running_mean, running_var))


def last_device_error(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load().tc3d_last_device_error(ctypes.c_void_p(s.cuda_stream)))


def set_wait_timeout_ns(ns: int) -> None:
    load().tc3d_set_wait_timeout_ns(int(ns))


def selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load().tc3d_selftest_wait_timeout(int(timeout_ns), ctypes.c_void_p(s.cuda_stream)))
