"""GPU test of tc3d_conv_maxpool_lse_relu_noalloc, the entry point for callers
that cannot allocate device memory (code inside an allocator or pool
callback, hosts that own every device allocation, paths where an allocation
is not allowed).  It takes its scratch from an array compiled into the
library instead of a caller-provided workspace.

The test calls it through the C ABI with raw device pointers and compares
its output with the regular workspace-taking entry point, within the
tolerance the other GPU tests use, on two calls in a row (different problems,
so the second call must fully rewrite the shared scratch).  This file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest

from transposed_conv_epilogues_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ATOL = 1e-4
RTOL = 1e-4


@pytest.fixture(scope="module")
def tc():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from transposed_conv_epilogues_gb300 import build
    build.build()
    import transposed_conv_epilogues_gb300 as t
    t.load()
    return t


def _problem(seed, xs, ws):
    x = inputs.normal(seed, xs)
    bound = 1.0 / np.sqrt(float(np.prod(ws[1:])))
    w = inputs.uniform(seed + 1, ws, -bound, bound)
    b = inputs.uniform(seed + 2, (ws[0],), -bound, bound) - 0.2
    return [torch.from_numpy(a).cuda() for a in (x, w, b)]


def _call_noalloc(tc, x, w, b, y, pad, groups=1):
    I3 = ctypes.c_int * 3
    N, Cin, S0, S1, S2 = x.shape
    Cout, _, k0, k1, k2 = w.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return tc.load().tc3d_conv_maxpool_lse_relu_noalloc(
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(w.data_ptr()),
        ctypes.c_void_p(b.data_ptr()), ctypes.c_void_p(y.data_ptr()), N, Cin, S0, S1, S2, Cout,
        k0, k1, k2, I3(1, 1, 1), I3(pad, pad, pad), I3(1, 1, 1), I3(0, 0, 0), groups, stream)


def test_noalloc_matches_workspace_entry_point_two_calls(tc):
    problems = [((2, 8, 12, 16, 32), (32, 8, 3, 3, 3)),  # call 1
                ((1, 5, 10, 14, 24), (20, 5, 3, 3, 3))]  # call 2: other sizes, same scratch
    for i, (xs, ws) in enumerate(problems):
        x, w, b = _problem(100 + 10 * i, xs, ws)
        ref = tc.conv_maxpool_lse_relu(x, w, b, 1, 1)
        y = torch.full_like(ref, float("nan"))
        rc = _call_noalloc(tc, x, w, b, y, 1)
        assert rc == tc.TC3D_OK, tc.status_string(rc)
        torch.cuda.synchronize()
        g = y.double().cpu().numpy()
        r = ref.double().cpu().numpy()
        assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r)), f"call {i + 1}"
    assert tc.last_device_error() == tc.TC3D_OK


def test_noalloc_rejects_problems_beyond_its_scratch(tc):
    # 64 -> 256 channels, k3: packed weights alone take 3.5 MB > 1 MiB
    x = torch.zeros((1, 64, 4, 4, 8), device="cuda")
    w = torch.zeros((256, 64, 3, 3, 3), device="cuda")
    b = torch.zeros(256, device="cuda")
    y = torch.full((1, 1, 2, 2, 4), 3.0, device="cuda")
    assert _call_noalloc(tc, x, w, b, y, 1) == tc.TC3D_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())


def test_noalloc_grouped_matches_workspace_entry_point(tc):
    """A depthwise problem (groups = Cin = Cout) through the same scratch."""
    x, w, b = _problem(300, (2, 8, 10, 12, 16), (8, 1, 3, 3, 3))
    ref = tc.conv_maxpool_lse_relu(x, w, b, 1, 1, groups=8)
    y = torch.full_like(ref, float("nan"))
    rc = _call_noalloc(tc, x, w, b, y, 1, groups=8)
    assert rc == tc.TC3D_OK, tc.status_string(rc)
    torch.cuda.synchronize()
    g = y.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r))
    assert tc.last_device_error() == tc.TC3D_OK
