"""GPU parity on seeded random shapes: convs, transposed convs, channels-last
convs and the BN-pool op drawn over strides, paddings, dilations, groups and
output paddings, each against the fp64 oracle on every output.

The hand-picked cases of test_gpu_parity.py target the plan's branches one
by one; these draws cover their combinations.  Draws whose output would be
empty (or whose pooled output would be) are redrawn; the library must
accept every drawn problem (no TC3D_ERR_UNSUPPORTED at these sizes).
"""
import numpy as np
import pytest

import oracle as orc
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


def _dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(gpu, ref, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    bad = ~(np.abs(gpu - ref) <= ATOL + RTOL * np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance"


def _conv_len(S, k, s, p, d):
    return (S + 2 * p - d * (k - 1) - 1) // s + 1


def _convT_len(S, k, s, p, d, op):
    return (S - 1) * s - 2 * p + d * (k - 1) + op + 1


def _draw(rng, transposed, pooled=0, dense=False):
    """One problem: (x shape, w shape, stride, pad, dil, output_padding,
    groups), with every output extent >= max(1, pooled).  dense: groups 1
    and more than 16 channel pairs (the engine's channels-last mode takes
    those channels-last convs)."""
    while True:
        G = 1 if dense else int(rng.choice([1, 1, 1, 2, 3]))
        cin = G * int(rng.integers(1, 7))
        cout = G * int(rng.integers(1, 9))
        if dense:
            cin = int(rng.choice([3, 4, 8, 12, 16, 20, 24, 36]))
            cout = int(rng.integers(6, 41))
        N = int(rng.integers(1, 3))
        S = [int(rng.integers(2, 11)) for _ in range(3)]
        k = [int(rng.integers(1, 4)) for _ in range(3)]
        s = [int(rng.integers(1, 4)) for _ in range(3)]
        d = [int(rng.integers(1, 3)) for _ in range(3)]
        p = [int(rng.integers(0, d[a] * (k[a] - 1) + 1)) for a in range(3)]
        op = [int(rng.integers(0, max(s[a], d[a]))) if transposed else 0 for a in range(3)]
        if transposed:
            O = [_convT_len(S[a], k[a], s[a], p[a], d[a], op[a]) for a in range(3)]
            w = (cin, cout // G, *k)
        else:
            O = [_conv_len(S[a], k[a], s[a], p[a], d[a]) for a in range(3)]
            w = (cout, cin // G, *k)
        if min(O) >= max(1, pooled) and int(np.prod(O)) * N * cout <= 400_000:
            return (N, cin, *S), w, tuple(s), tuple(p), tuple(d), tuple(op), G


def _make(seed, xs, ws, cout, bias=True):
    x = inputs.normal(seed, xs)
    bound = 1.0 / np.sqrt(int(np.prod(ws[1:])))
    w = inputs.uniform(seed + 1, ws, -bound, bound)
    b = inputs.uniform(seed + 2, (cout,), -bound, bound) if bias else None
    return x, w, b


@pytest.mark.parametrize("i", range(24))
def test_random_conv3d(tc, i):
    rng = np.random.default_rng(1000 + i)
    xs, ws, s, p, d, _, G = _draw(rng, False)
    x, w, b = _make(5000 + 10 * i, xs, ws, ws[0], bias=bool(i % 3))
    y = tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), s, p, d, G).cpu().numpy()
    _check(y, orc.conv3d(x, w, b, s, p, d, G), f"conv {xs} {ws} s{s} p{p} d{d} G{G}")


@pytest.mark.parametrize("i", range(24))
def test_random_conv_transpose3d(tc, i):
    rng = np.random.default_rng(2000 + i)
    xs, ws, s, p, d, op, G = _draw(rng, True)
    cout = ws[1] * G
    x, w, b = _make(6000 + 10 * i, xs, ws, cout, bias=bool(i % 3))
    y = tc.conv_transpose3d_fwd(_dev(x), _dev(w), _dev(b), s, p, d, op, G).cpu().numpy()
    _check(y, orc.conv_transpose3d(x, w, b, s, p, d, op, G),
           f"convT {xs} {ws} s{s} p{p} d{d} op{op} G{G}")


@pytest.mark.parametrize("i", range(16))
def test_random_conv3d_ndhwc(tc, i):
    rng = np.random.default_rng(3000 + i)
    xs, ws, s, p, d, _, G = _draw(rng, False, dense=i % 4 != 0)
    x, w, b = _make(7000 + 10 * i, xs, ws, ws[0])
    x_cl = np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1))
    y = tc.conv3d_fwd_ndhwc(_dev(x_cl), _dev(w), _dev(b), s, p, d, G).cpu().numpy()
    ref = orc.conv3d(x, w, b, s, p, d, G).transpose(0, 2, 3, 4, 1)
    _check(y, ref, f"ndhwc {xs} {ws} s{s} p{p} d{d} G{G}")


@pytest.mark.parametrize("i", range(12))
def test_random_convT_bn_avgpool(tc, i):
    """Batch statistics; the transposed conv's output extents are at least 4
    so that the 4^3 pool has an output."""
    rng = np.random.default_rng(4000 + i)
    xs, ws, s, p, d, op, G = _draw(rng, True, pooled=4)
    cout = ws[1] * G
    x, w, b = _make(8000 + 10 * i, xs, ws, cout)
    g = inputs.uniform(8100 + i, (cout,), 0.5, 1.5) if i % 2 else None
    be = inputs.uniform(8200 + i, (cout,), -0.5, 0.5) if i % 2 else None
    y = tc.convT_bn_avgpool(_dev(x), _dev(w), _dev(b), _dev(g), _dev(be), 1e-5, s, p, d, op,
                            G).cpu().numpy()
    _check(y, orc.convT_bn_avgpool(x, w, b, g, be, 1e-5, s, p, d, op, G),
           f"bn-pool {xs} {ws} s{s} p{p} d{d} op{op} G{G}")
