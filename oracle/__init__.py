"""fp64 CPU oracle for the conv3d / conv_transpose3d hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library: the arithmetic lives in
``oracle.c`` (plain loop nests of the definitions, fp64), and this module only
compiles it with gcc, loads it with ctypes and marshals numpy arrays.

Every function takes and returns NCDHW arrays (spatial axes positional, the
last one contiguous).  Inputs of any float dtype are promoted to float64.

Definitions and their sources (the four POPCORNBENCH transcript pages):

* ``conv3d`` -- gather definition with per-axis stride/padding/dilation and
  groups ("Kimi-K2.6 l1_p59", direct-convolution formula).
* ``conv_transpose3d`` -- receive form, a tap counts iff (z + p - d k) is
  divisible by s and the quotient is in range ("Kimi-K2.6 l1_p77",
  receive-form derivation); ``conv_transpose3d_scatter`` -- the scatter view
  of the same page, an independent second formulation.
* ``maxpool3d_2`` / ``logsumexp_channels`` / ``relu`` -- "Kimi-K2.6 l2_p43".
* ``batchnorm3d_train`` / ``avgpool3d_2`` -- "Kimi-K2.6 l2_p72";
  ``batchnorm3d_eval`` -- the same page's fused kernel, which normalises with
  running statistics (evaluation mode).

Parity pins: every function is pinned by ``tests/test_oracle.py`` (sizes from
the pages, adjoint identity, impulse response, slice-wise 2-D conv, per-voxel
matrix product, gather == scatter, pooling identities, LSE bounds, BN moments,
and a PyTorch-CPU fp64 cross-check when torch is importable).  No function is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_HDR = _HERE / "oracle.h"
_LIB = _HERE / "liboracle.so"
_lib = None

_I64P = ctypes.POINTER(ctypes.c_int64)
_DP = ctypes.POINTER(ctypes.c_double)
_IP = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> Path:
    """Compile oracle.c into liboracle.so (gcc, no FMA contraction)."""
    stale = (not _LIB.exists()) or any(
        p.stat().st_mtime > _LIB.stat().st_mtime for p in (_SRC, _HDR))
    if not (force or stale):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=str(_HERE))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC",
           "-pthread", str(_SRC), "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB)
    except subprocess.CalledProcessError as e:  # pragma: no cover
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{e.stderr}") from e
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(str(build()))
    lib.oracle_conv_out_len.restype = ctypes.c_int64
    lib.oracle_conv_out_len.argtypes = [ctypes.c_int64] + [ctypes.c_int] * 4
    lib.oracle_convT_out_len.restype = ctypes.c_int64
    lib.oracle_convT_out_len.argtypes = [ctypes.c_int64] + [ctypes.c_int] * 5
    lib.oracle_relu.restype = None
    D, I, L, F = _DP, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    I3 = ctypes.c_int * 3
    geom = [I] * 9 + [I3, I3, I3]  # N Cin S0 S1 S2 Cout k0 k1 k2 | stride pad dil
    sig = {
        "oracle_conv3d": [D, D, D, D] + geom + [I, I],
        "oracle_conv3d_at": [D, D, D] + geom + [I, _I64P, L, D, I],
        "oracle_conv_transpose3d": [D, D, D, D] + geom + [I3, I, I],
        "oracle_conv_transpose3d_at": [D, D, D] + geom + [I3, I, _I64P, L, D, I],
        "oracle_conv_transpose3d_scatter": [D, D, D, D] + geom + [I3, I],
        "oracle_maxpool3d_2": [D, D, I, I, I, I, I],
        "oracle_avgpool3d_2": [D, D, I, I, I, I, I],
        "oracle_logsumexp_channels": [D, D, I, I, L],
        "oracle_relu": [D, L],
        "oracle_batchnorm3d_train": [D, D, I, I, L, D, D, F, D, D],
        "oracle_convT_bn_avgpool": [D, D, D, D, D, F, D] + geom + [I3, I, I],
        "oracle_convT_bn_avgpool_at": [D, D, D, D, D, F] + geom + [I3, I, _I64P, L, D, D, D, I],
        "oracle_batchnorm3d_eval": [D, D, I, I, L, D, D, D, D, F],
        "oracle_convT_bneval_avgpool": [D, D, D, D, D, D, D, F, D] + geom + [I3, I, I],
        "oracle_convT_bneval_avgpool_at": [D, D, D, D, D, D, D, F] + geom + [I3, I, _I64P, L, D, I],
        "oracle_conv_maxpool_lse_relu": [D, D, D, D] + geom + [I, I],
        "oracle_conv_maxpool_lse_relu_at": [D, D, D] + geom + [I, _I64P, L, D, I],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        if name != "oracle_relu":
            fn.restype = ctypes.c_int
    _lib = lib
    return lib


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _d(a):
    """fp64 C-contiguous copy/view and its pointer."""
    if a is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a, a.ctypes.data_as(_DP)


def _i3(v):
    v = (int(v),) * 3 if np.isscalar(v) else tuple(int(t) for t in v)
    assert len(v) == 3
    return (ctypes.c_int * 3)(*v)


def conv_out_len(L, k, s, p, d):
    return int(_load().oracle_conv_out_len(L, k, s, p, d))


def convT_out_len(L, k, s, p, d, op=0):
    return int(_load().oracle_convT_out_len(L, k, s, p, d, op))


def conv_out_shape(xshape, wshape, stride=1, padding=0, dilation=1):
    s, p, d = (tuple(_i3(v)) for v in (stride, padding, dilation))
    N, _, S0, S1, S2 = xshape
    Cout = wshape[0]
    return (N, Cout) + tuple(conv_out_len(L, k, s_, p_, d_) for L, k, s_, p_, d_ in
                             zip((S0, S1, S2), wshape[2:], s, p, d))


def convT_out_shape(xshape, wshape, stride=1, padding=0, dilation=1,
                    output_padding=0, groups=1):
    s, p, d, op = (tuple(_i3(v)) for v in (stride, padding, dilation, output_padding))
    N, _, S0, S1, S2 = xshape
    Cout = wshape[1] * groups
    return (N, Cout) + tuple(convT_out_len(L, k, a, b, c, e) for L, k, a, b, c, e in
                             zip((S0, S1, S2), wshape[2:], s, p, d, op))


def _geom(x, w):
    N, Cin, S0, S1, S2 = x.shape
    k0, k1, k2 = w.shape[2:]
    return N, Cin, S0, S1, S2, k0, k1, k2


def _check_w(x, w, groups, transposed):
    ok = w.shape[0] == x.shape[1] if transposed else w.shape[1] * groups == x.shape[1]
    if not ok or w.ndim != 5 or x.ndim != 5:
        raise ValueError(f"weight {w.shape} does not fit input {x.shape} with groups={groups}")


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments")


def conv3d(x, w, b=None, stride=1, padding=0, dilation=1, groups=1, nthreads=None):
    """Conv3d, gather form.  w: [Cout, Cin/G, k0, k1, k2]."""
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, False)
    Cout = w.shape[0]
    shp = conv_out_shape(x.shape, w.shape, stride, padding, dilation)
    if min(shp) <= 0:
        raise ValueError("empty conv output")
    y = np.empty(shp, np.float64)
    _check(_load().oracle_conv3d(xp, wp, bp, y.ctypes.data_as(_DP), N, Cin, S0, S1, S2, Cout,
                                 k0, k1, k2, _i3(stride), _i3(padding), _i3(dilation), groups,
                                 _threads(nthreads)), "conv3d")
    return y


def conv3d_at(x, w, b, idx, stride=1, padding=0, dilation=1, groups=1, nthreads=None):
    """Conv3d at flat NCDHW output indices ``idx``."""
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, False)
    out = np.empty(idx.shape, np.float64)
    _check(_load().oracle_conv3d_at(xp, wp, bp, N, Cin, S0, S1, S2, w.shape[0], k0, k1, k2,
                                    _i3(stride), _i3(padding), _i3(dilation), groups,
                                    idx.ctypes.data_as(_I64P), ctypes.c_int64(idx.size), out.ctypes.data_as(_DP),
                                    _threads(nthreads)), "conv3d_at")
    return out


def conv_transpose3d(x, w, b=None, stride=1, padding=0, dilation=1, output_padding=0,
                     groups=1, nthreads=None):
    """ConvTranspose3d, receive (gather) form.  w: [Cin, Cout/G, k0, k1, k2]."""
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, True)
    shp = convT_out_shape(x.shape, w.shape, stride, padding, dilation, output_padding, groups)
    if min(shp) <= 0:
        raise ValueError("empty convT output")
    y = np.empty(shp, np.float64)
    _check(_load().oracle_conv_transpose3d(xp, wp, bp, y.ctypes.data_as(_DP), N, Cin, S0, S1, S2,
                                           shp[1], k0, k1, k2, _i3(stride), _i3(padding),
                                           _i3(dilation), _i3(output_padding), groups,
                                           _threads(nthreads)), "conv_transpose3d")
    return y


def conv_transpose3d_at(x, w, b, idx, stride=1, padding=0, dilation=1, output_padding=0,
                        groups=1, nthreads=None):
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, True)
    out = np.empty(idx.shape, np.float64)
    _check(_load().oracle_conv_transpose3d_at(
        xp, wp, bp, N, Cin, S0, S1, S2, w.shape[1] * groups, k0, k1, k2, _i3(stride),
        _i3(padding), _i3(dilation), _i3(output_padding), groups, idx.ctypes.data_as(_I64P),
        idx.size, out.ctypes.data_as(_DP), _threads(nthreads)), "conv_transpose3d_at")
    return out


def conv_transpose3d_scatter(x, w, b=None, stride=1, padding=0, dilation=1,
                             output_padding=0, groups=1):
    """ConvTranspose3d, scatter form (single-threaded; small inputs only)."""
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, True)
    shp = convT_out_shape(x.shape, w.shape, stride, padding, dilation, output_padding, groups)
    y = np.empty(shp, np.float64)
    _check(_load().oracle_conv_transpose3d_scatter(
        xp, wp, bp, y.ctypes.data_as(_DP), N, Cin, S0, S1, S2, shp[1], k0, k1, k2, _i3(stride),
        _i3(padding), _i3(dilation), _i3(output_padding), groups), "conv_transpose3d_scatter")
    return y


def _pool(t, fn, name):
    t, tp = _d(t)
    N, C, L0, L1, L2 = t.shape
    out = np.empty((N, C, L0 // 2, L1 // 2, L2 // 2), np.float64)
    _check(fn(tp, out.ctypes.data_as(_DP), N, C, L0, L1, L2), name)
    return out


def maxpool3d_2(t):
    return _pool(t, _load().oracle_maxpool3d_2, "maxpool3d_2")


def avgpool3d_2(t):
    return _pool(t, _load().oracle_avgpool3d_2, "avgpool3d_2")


def logsumexp_channels(t):
    t, tp = _d(t)
    N, C = t.shape[:2]
    L = int(np.prod(t.shape[2:]))
    out = np.empty((N, 1) + t.shape[2:], np.float64)
    _check(_load().oracle_logsumexp_channels(tp, out.ctypes.data_as(_DP), N, C,
                                             ctypes.c_int64(L)), "logsumexp")
    return out


def relu(t):
    t = np.array(t, dtype=np.float64, copy=True, order="C")
    _load().oracle_relu(t.ctypes.data_as(_DP), ctypes.c_int64(t.size))
    return t


def batchnorm3d_train(t, gamma=None, beta=None, eps=1e-5, return_stats=False):
    t, tp = _d(t)
    g, gp = _d(gamma)
    be, bep = _d(beta)
    N, C = t.shape[:2]
    L = int(np.prod(t.shape[2:]))
    out = np.empty_like(t)
    mean = np.empty(C, np.float64)
    var = np.empty(C, np.float64)
    _check(_load().oracle_batchnorm3d_train(tp, out.ctypes.data_as(_DP), N, C, ctypes.c_int64(L),
                                            gp, bep, ctypes.c_double(eps),
                                            mean.ctypes.data_as(_DP), var.ctypes.data_as(_DP)),
           "batchnorm3d_train")
    return (out, mean, var) if return_stats else out


def convT_bn_avgpool(x, w, b=None, gamma=None, beta=None, eps=1e-5, stride=1, padding=0,
                     dilation=1, output_padding=0, groups=1, nthreads=None):
    """ConvTranspose3d -> BatchNorm3d (batch stats) -> AvgPool3d(2) -> AvgPool3d(2)."""
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    g, gp = _d(gamma)
    be, bep = _d(beta)
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, True)
    shp = convT_out_shape(x.shape, w.shape, stride, padding, dilation, output_padding, groups)
    out_shape = shp[:2] + tuple(o // 2 // 2 for o in shp[2:])
    y = np.empty(out_shape, np.float64)
    _check(_load().oracle_convT_bn_avgpool(
        xp, wp, bp, gp, bep, ctypes.c_double(eps), y.ctypes.data_as(_DP), N, Cin, S0, S1, S2,
        shp[1], k0, k1, k2, _i3(stride), _i3(padding), _i3(dilation), _i3(output_padding), groups,
        _threads(nthreads)), "convT_bn_avgpool")
    return y


def convT_bn_avgpool_at(x, w, b, idx, gamma=None, beta=None, eps=1e-5, stride=1, padding=0,
                        dilation=1, output_padding=0, groups=1, nthreads=None,
                        return_stats=False):
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    g, gp = _d(gamma)
    be, bep = _d(beta)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, True)
    Cout = w.shape[1] * groups
    out = np.empty(idx.shape, np.float64)
    mean = np.empty(Cout, np.float64)
    var = np.empty(Cout, np.float64)
    _check(_load().oracle_convT_bn_avgpool_at(
        xp, wp, bp, gp, bep, ctypes.c_double(eps), N, Cin, S0, S1, S2, Cout, k0, k1, k2,
        _i3(stride), _i3(padding), _i3(dilation), _i3(output_padding), groups,
        idx.ctypes.data_as(_I64P), ctypes.c_int64(idx.size), out.ctypes.data_as(_DP), mean.ctypes.data_as(_DP),
        var.ctypes.data_as(_DP), _threads(nthreads)), "convT_bn_avgpool_at")
    return (out, mean, var) if return_stats else out


def batchnorm3d_eval(t, running_mean, running_var, gamma=None, beta=None, eps=1e-5):
    """BatchNorm3d in evaluation mode: (t - running_mean) / sqrt(running_var + eps)
    * gamma + beta per channel ("Kimi-K2.6 l2_p72", its fused kernel's form)."""
    t, tp = _d(t)
    rm, rmp = _d(running_mean)
    rv, rvp = _d(running_var)
    g, gp = _d(gamma)
    be, bep = _d(beta)
    N, C = t.shape[:2]
    L = int(np.prod(t.shape[2:]))
    out = np.empty_like(t)
    _check(_load().oracle_batchnorm3d_eval(tp, out.ctypes.data_as(_DP), N, C, ctypes.c_int64(L),
                                           rmp, rvp, gp, bep, ctypes.c_double(eps)),
           "batchnorm3d_eval")
    return out


def convT_bneval_avgpool(x, w, b, running_mean, running_var, gamma=None, beta=None, eps=1e-5,
                         stride=1, padding=0, dilation=1, output_padding=0, groups=1,
                         nthreads=None):
    """ConvTranspose3d -> BatchNorm3d (running stats) -> AvgPool3d(2) -> AvgPool3d(2)."""
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    rm, rmp = _d(running_mean)
    rv, rvp = _d(running_var)
    g, gp = _d(gamma)
    be, bep = _d(beta)
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, True)
    shp = convT_out_shape(x.shape, w.shape, stride, padding, dilation, output_padding, groups)
    out_shape = shp[:2] + tuple(o // 2 // 2 for o in shp[2:])
    y = np.empty(out_shape, np.float64)
    _check(_load().oracle_convT_bneval_avgpool(
        xp, wp, bp, rmp, rvp, gp, bep, ctypes.c_double(eps), y.ctypes.data_as(_DP), N, Cin, S0,
        S1, S2, shp[1], k0, k1, k2, _i3(stride), _i3(padding), _i3(dilation),
        _i3(output_padding), groups, _threads(nthreads)), "convT_bneval_avgpool")
    return y


def convT_bneval_avgpool_at(x, w, b, running_mean, running_var, idx, gamma=None, beta=None,
                            eps=1e-5, stride=1, padding=0, dilation=1, output_padding=0,
                            groups=1, nthreads=None):
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    rm, rmp = _d(running_mean)
    rv, rvp = _d(running_var)
    g, gp = _d(gamma)
    be, bep = _d(beta)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, True)
    Cout = w.shape[1] * groups
    out = np.empty(idx.shape, np.float64)
    _check(_load().oracle_convT_bneval_avgpool_at(
        xp, wp, bp, rmp, rvp, gp, bep, ctypes.c_double(eps), N, Cin, S0, S1, S2, Cout, k0, k1,
        k2, _i3(stride), _i3(padding), _i3(dilation), _i3(output_padding), groups,
        idx.ctypes.data_as(_I64P), ctypes.c_int64(idx.size), out.ctypes.data_as(_DP),
        _threads(nthreads)), "convT_bneval_avgpool_at")
    return out


def conv_maxpool_lse_relu(x, w, b=None, stride=1, padding=0, dilation=1, groups=1,
                          nthreads=None):
    """Conv3d -> MaxPool3d(2,2) -> logsumexp over channels (keepdim) -> ReLU."""
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, False)
    shp = conv_out_shape(x.shape, w.shape, stride, padding, dilation)
    y = np.empty((N, 1) + tuple(o // 2 for o in shp[2:]), np.float64)
    _check(_load().oracle_conv_maxpool_lse_relu(
        xp, wp, bp, y.ctypes.data_as(_DP), N, Cin, S0, S1, S2, w.shape[0], k0, k1, k2,
        _i3(stride), _i3(padding), _i3(dilation), groups, _threads(nthreads)),
        "conv_maxpool_lse_relu")
    return y


def conv_maxpool_lse_relu_at(x, w, b, idx, stride=1, padding=0, dilation=1, groups=1,
                             nthreads=None):
    x, xp = _d(x)
    w, wp = _d(w)
    b, bp = _d(b)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    N, Cin, S0, S1, S2, k0, k1, k2 = _geom(x, w)
    _check_w(x, w, groups, False)
    out = np.empty(idx.shape, np.float64)
    _check(_load().oracle_conv_maxpool_lse_relu_at(
        xp, wp, bp, N, Cin, S0, S1, S2, w.shape[0], k0, k1, k2, _i3(stride), _i3(padding),
        _i3(dilation), groups, idx.ctypes.data_as(_I64P), ctypes.c_int64(idx.size), out.ctypes.data_as(_DP),
        _threads(nthreads)), "conv_maxpool_lse_relu_at")
    return out
