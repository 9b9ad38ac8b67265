"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

None of these re-types the oracle's own formula: each check goes through a
different route (sizes printed on the pages, hand-worked tap lists, the
adjoint identity, impulse responses, reshape identities, a per-voxel matrix
product, an independent scatter formulation, pooling identities, logsumexp
bounds, batch-norm moments, and PyTorch's CPU fp64 operators).
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b)))


# --------------------------------------------------------------------------
# sizes printed on the pages
# --------------------------------------------------------------------------
def _read_sizes():
    rows = []
    for line in open(os.path.join(GOLDEN, "sizes.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        rows.append((f[0],) + tuple(int(v) for v in f[1:8]))
    return rows


@pytest.mark.parametrize("row", _read_sizes())
def test_sizes_from_pages(oracle, row):
    op, L, k, s, p, d, opad, expected = row
    if op == "conv":
        assert oracle.conv_out_len(L, k, s, p, d) == expected
    elif op == "convT":
        assert oracle.convT_out_len(L, k, s, p, d, opad) == expected
    else:  # pool2 = conv-size formula with k=2, s=2 (floor mode)
        assert oracle.conv_out_len(L, 2, 2, 0, 1) == expected
        t = np.zeros((1, 1, L, 2, 2))
        assert oracle.maxpool3d_2(t).shape[2] == expected


def test_workload_shapes(oracle):
    from transposed_conv_epilogues_gb300.workloads import WORKLOADS
    expect = {
        1: (2, 8, 14, 14, 4),
        2: (16, 64, 126, 126, 8),
        3: (16, 64, 33, 65, 65),
        4: (64, 16, 63, 63, 63),
        5: (4, 64, 32, 128, 128),
    }
    for wl in WORKLOADS:
        if wl.transposed:
            shp = oracle.convT_out_shape(wl.x_shape, wl.w_shape, wl.stride, wl.padding,
                                         wl.dilation, wl.output_padding, wl.groups)
        else:
            shp = oracle.conv_out_shape(wl.x_shape, wl.w_shape, wl.stride, wl.padding,
                                        wl.dilation)
        assert shp == expect[wl.index]


def test_output_size_brute_force(oracle):
    """Conv length = number of output positions whose first tap index is a
    valid window start; convT length = 1 + the largest scattered index."""
    for L in range(1, 14):
        for k in range(1, 5):
            for s in range(1, 4):
                for d in range(1, 4):
                    for p in range(0, 3):
                        # conv: o valid iff o*s - p >= -p and the last tap lands
                        # inside the padded input of length L + 2p
                        cnt = sum(1 for o in range(0, L + 2 * p + 1)
                                  if o * s + d * (k - 1) <= L + 2 * p - 1)
                        assert oracle.conv_out_len(L, k, s, p, d) == cnt
                        for op in range(0, max(s, d)):
                            top = max(i * s + d * j for i in range(L) for j in range(k))
                            expect = top + 1 - 2 * p + op
                            assert oracle.convT_out_len(L, k, s, p, d, op) == max(0, expect)


# --------------------------------------------------------------------------
# hand-worked tap lists on the pages (via impulse responses of the oracle)
# --------------------------------------------------------------------------
def _read_taps(name):
    rows, total = {}, None
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "total_pairs":
            total = int(f[1])
            continue
        rows[int(f[0])] = set() if f[1] == "none" else {tuple(int(v) for v in t.split(","))
                                                         for t in f[1:]}
    return rows, total


@pytest.mark.parametrize("name,L,s,p,d", [("convT_taps_s2p1d2k3_L16.txt", 16, 2, 1, 2),
                                          ("convT_taps_s2p1d1k3_L32.txt", 32, 2, 1, 1)])
def test_convT_tap_lists_from_pages(oracle, name, L, s, p, d):
    rows, total = _read_taps(name)
    k = 3
    O = oracle.convT_out_len(L, k, s, p, d, 0)
    contrib = {z: set() for z in range(O)}
    for zi in range(L):
        for kd in range(k):
            x = np.zeros((1, 1, L, 1, 1))
            x[0, 0, zi] = 1.0
            w = np.zeros((1, 1, k, 1, 1))
            w[0, 0, kd] = 1.0
            y = oracle.conv_transpose3d(x, w, None, (s, 1, 1), (p, 0, 0), (d, 1, 1))
            for z in np.nonzero(y[0, 0, :, 0, 0])[0]:
                contrib[int(z)].add((zi, kd))
    for z, pairs in rows.items():
        assert contrib[z] == pairs, (z, contrib[z], pairs)
    if total is not None:
        assert sum(len(v) for v in contrib.values()) == total


# --------------------------------------------------------------------------
# adjoint identity <conv(x;W), y> = <x, convT(y;W)>
# --------------------------------------------------------------------------
ADJ_CASES = [
    # (Cin, Cout, S, k, s, p, d, G)
    (3, 4, (7, 6, 5), (3, 3, 3), (1, 1, 1), (1, 1, 1), (1, 1, 1), 1),
    (4, 6, (9, 8, 7), (3, 2, 3), (2, 2, 3), (1, 0, 2), (1, 2, 1), 2),
    (6, 6, (11, 5, 6), (2, 3, 1), (3, 1, 2), (0, 2, 0), (2, 1, 1), 3),
    (2, 3, (8, 8, 8), (3, 3, 3), (2, 2, 2), (1, 1, 1), (2, 2, 2), 1),
    (4, 8, (5, 9, 4), (1, 3, 2), (1, 2, 1), (0, 1, 1), (1, 3, 2), 4),
]


@pytest.mark.parametrize("case", ADJ_CASES)
def test_adjoint_identity(oracle, case):
    Cin, Cout, S, k, s, p, d, G = case
    x = rng.standard_normal((2, Cin) + S)
    W = rng.standard_normal((Cout, Cin // G) + k)
    y = oracle.conv3d(x, W, None, s, p, d, G)
    u = rng.standard_normal(y.shape)
    # the same W memory read as a ConvTranspose3d weight [Cin_T=Cout, Cout_T/G=Cin/G, k]
    op = tuple((S[a] + 2 * p[a] - d[a] * (k[a] - 1) - 1) % s[a] for a in range(3))
    xt = oracle.conv_transpose3d(u, W, None, s, p, d, op, G)
    assert xt.shape == x.shape
    lhs = float(np.sum(y * u))
    rhs = float(np.sum(x * xt))
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs), np.sum(np.abs(y * u)))


# --------------------------------------------------------------------------
# impulse response of the transposed convolution reproduces W
# --------------------------------------------------------------------------
@pytest.mark.parametrize("s,p,d,G", [((2, 2, 2), (1, 1, 1), (2, 2, 2), 1),
                                     ((2, 3, 1), (0, 1, 2), (1, 2, 3), 2),
                                     ((1, 1, 1), (0, 0, 0), (1, 1, 1), 1)])
def test_convT_impulse_response(oracle, s, p, d, G):
    Cin, Cout, S, k = 4, 6, (5, 4, 6), (3, 2, 3)
    W = rng.standard_normal((Cin, Cout // G) + k)
    for (n, ic, i) in [(0, 0, (0, 0, 0)), (1, 3, (2, 1, 4)), (0, 2, (4, 3, 5))]:
        x = np.zeros((2, Cin) + S)
        x[n, ic][i] = 1.0
        y = oracle.conv_transpose3d(x, W, None, s, p, d, 0, G)
        expect = np.zeros_like(y)
        g = ic // (Cin // G)
        cg = Cout // G
        for ocl in range(cg):
            for a in range(k[0]):
                for b in range(k[1]):
                    for c in range(k[2]):
                        z = tuple(i[t] * s[t] - p[t] + d[t] * kk for t, kk in
                                  enumerate((a, b, c)))
                        if all(0 <= z[t] < y.shape[2 + t] for t in range(3)):
                            expect[n, g * cg + ocl][z] = W[ic, ocl, a, b, c]
        np.testing.assert_array_equal(y, expect)


# --------------------------------------------------------------------------
# gather convT == scatter convT (two formulations on the page)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("s", [1, 2, 3, 4])
@pytest.mark.parametrize("d", [1, 2, 3])
def test_convT_gather_equals_scatter(oracle, s, d):
    for p in range(0, 3):
        for k in (1, 2, 3, 4):
            for op in range(0, max(s, d)):
                L = 4
                if oracle.convT_out_len(L, k, s, p, d, op) <= 0:
                    continue
                x = rng.standard_normal((1, 2, L, 3, 2))
                W = rng.standard_normal((2, 3, k, 2, 1))
                b = rng.standard_normal(3)
                kw = dict(stride=(s, 1, 2), padding=(p, 0, 0), dilation=(d, 1, 1),
                          output_padding=(op, 0, 0))
                g = oracle.conv_transpose3d(x, W, b, **kw)
                sc = oracle.conv_transpose3d_scatter(x, W, b, **kw)
                assert _rel(g, sc) <= 1e-12


def test_convT_gather_equals_scatter_groups(oracle):
    x = rng.standard_normal((2, 6, 5, 4, 6))
    W = rng.standard_normal((6, 2, 3, 3, 2))
    b = rng.standard_normal(6)
    kw = dict(stride=(2, 3, 1), padding=(1, 2, 0), dilation=(2, 1, 3), output_padding=(1, 0, 2),
              groups=3)
    assert _rel(oracle.conv_transpose3d(x, W, b, **kw),
                oracle.conv_transpose3d_scatter(x, W, b, **kw)) <= 1e-12


# --------------------------------------------------------------------------
# (k,k,1) conv == per-depth-slice 2-D conv; k=1 conv == per-voxel matmul
# --------------------------------------------------------------------------
def _conv2d_slices(x4, W2, b, s, p, d):
    """Reference 2-D conv of [B,C,H,W] by shifting whole planes (no 3-D loop)."""
    B, C, H, Wd = x4.shape
    Co, _, kh, kw = W2.shape
    xp = np.pad(x4, ((0, 0), (0, 0), (p[0], p[0]), (p[1], p[1])))
    Ho = (H + 2 * p[0] - d[0] * (kh - 1) - 1) // s[0] + 1
    Wo = (Wd + 2 * p[1] - d[1] * (kw - 1) - 1) // s[1] + 1
    out = np.zeros((B, Co, Ho, Wo))
    for a in range(kh):
        for c in range(kw):
            plane = xp[:, :, a * d[0]: a * d[0] + s[0] * (Ho - 1) + 1: s[0],
                       c * d[1]: c * d[1] + s[1] * (Wo - 1) + 1: s[1]]
            out += np.einsum("oc,bchw->bohw", W2[:, :, a, c], plane)
    if b is not None:
        out += b[None, :, None, None]
    return out


@pytest.mark.parametrize("s,p,d", [((1, 1), (0, 0), (1, 1)), ((2, 1), (1, 2), (1, 2))])
def test_kk1_conv_equals_slicewise_2d(oracle, s, p, d):
    N, C, Co, H, Wd, D = 2, 3, 5, 9, 8, 4
    x = rng.standard_normal((N, C, H, Wd, D))
    W = rng.standard_normal((Co, C, 3, 3, 1))
    b = rng.standard_normal(Co)
    y = oracle.conv3d(x, W, b, (s[0], s[1], 1), (p[0], p[1], 0), (d[0], d[1], 1))
    # depth as extra batch: [N,C,H,W,D] -> [N*D,C,H,W]
    x4 = x.transpose(0, 4, 1, 2, 3).reshape(N * D, C, H, Wd)
    y2 = _conv2d_slices(x4, W[..., 0], b, s, p, d)
    y2 = y2.reshape(N, D, Co, y2.shape[2], y2.shape[3]).transpose(0, 2, 3, 4, 1)
    assert y.shape == y2.shape
    assert _rel(y, y2) <= 1e-13


def test_kernel1_axis_takes_padding(oracle):
    """A (3,3,1) kernel with padding 1 on the kernel-1 axis grows it by 2 and
    the padded depth slices hold only the bias (padding applies per axis)."""
    x = rng.standard_normal((1, 2, 5, 5, 3))
    W = rng.standard_normal((3, 2, 3, 3, 1))
    b = rng.standard_normal(3)
    y = oracle.conv3d(x, W, b, 1, (0, 0, 1), 1)
    assert y.shape == (1, 3, 3, 3, 5)
    np.testing.assert_allclose(y[0, :, :, :, 0], np.broadcast_to(b[:, None, None], (3, 3, 3)),
                               rtol=0, atol=0)
    y0 = oracle.conv3d(x, W, b, 1, 0, 1)
    np.testing.assert_allclose(y[..., 1:4], y0, rtol=1e-15, atol=0)


def test_k1_conv_equals_matmul(oracle):
    x = rng.standard_normal((3, 6, 4, 5, 7))
    W = rng.standard_normal((4, 6, 1, 1, 1))
    b = rng.standard_normal(4)
    y = oracle.conv3d(x, W, b)
    ref = np.einsum("oi,nidhw->nodhw", W[:, :, 0, 0, 0], x) + b[None, :, None, None, None]
    assert _rel(y, ref) <= 1e-14
    # grouped k=1: block-diagonal matmul
    Wg = rng.standard_normal((4, 3, 1, 1, 1))
    yg = oracle.conv3d(x, Wg, None, groups=2)
    ref0 = np.einsum("oi,nidhw->nodhw", Wg[:2, :, 0, 0, 0], x[:, :3])
    ref1 = np.einsum("oi,nidhw->nodhw", Wg[2:, :, 0, 0, 0], x[:, 3:])
    assert _rel(yg, np.concatenate([ref0, ref1], axis=1)) <= 1e-14


def test_stride_picks_every_sth_output(oracle):
    """Stride s of a conv equals the stride-1 conv sampled every s-th output."""
    x = rng.standard_normal((1, 2, 11, 9, 10))
    W = rng.standard_normal((3, 2, 3, 2, 3))
    y1 = oracle.conv3d(x, W, None, 1, (1, 0, 2), (1, 2, 1))
    y3 = oracle.conv3d(x, W, None, (2, 3, 2), (1, 0, 2), (1, 2, 1))
    np.testing.assert_array_equal(y3, y1[:, :, ::2, ::3, ::2][:, :, :y3.shape[2], :y3.shape[3],
                                                                :y3.shape[4]])


# --------------------------------------------------------------------------
# pooling, logsumexp, batch norm
# --------------------------------------------------------------------------
@pytest.mark.parametrize("L", list(range(4, 41)))
def test_two_avgpool2_equal_avgpool4(oracle, L):
    t = rng.standard_normal((1, 2, L, 5, 8))
    two = oracle.avgpool3d_2(oracle.avgpool3d_2(t))
    P = L // 4
    crop = t[:, :, :4 * P, :4, :8]
    four = crop.reshape(1, 2, P, 4, 1, 4, 2, 4).mean(axis=(3, 5, 7))
    assert two.shape == four.shape
    assert _rel(two, four) <= 1e-14


def test_maxpool_matches_reshape_max(oracle):
    t = rng.standard_normal((2, 3, 7, 9, 6))
    m = oracle.maxpool3d_2(t)
    ref = t[:, :, :6, :8, :6].reshape(2, 3, 3, 2, 4, 2, 3, 2).max(axis=(3, 5, 7))
    np.testing.assert_array_equal(m, ref)


def test_logsumexp_bounds_and_library(oracle):
    from scipy.special import logsumexp
    for C in (1, 2, 7, 64):
        t = 5 * rng.standard_normal((2, C, 3, 4, 5))
        l = oracle.logsumexp_channels(t)
        mx = t.max(axis=1, keepdims=True)
        assert np.all(l >= mx - 1e-12) and np.all(l <= mx + math.log(C) + 1e-12)
        assert _rel(l, logsumexp(t, axis=1, keepdims=True)) <= 1e-14
        if C == 1:
            np.testing.assert_array_equal(l, t)
    # large magnitudes must not overflow (stable form)
    t = np.full((1, 3, 1, 1, 2), 1000.0)
    np.testing.assert_allclose(oracle.logsumexp_channels(t), 1000.0 + math.log(3), rtol=1e-15)
    # negative LSE survives only until ReLU
    t = np.full((1, 2, 1, 1, 1), -10.0)
    l = oracle.logsumexp_channels(t)
    assert l.item() < 0 and oracle.relu(l).item() == 0.0


def test_batchnorm_moments(oracle):
    t = 3.0 + 2.0 * rng.standard_normal((4, 5, 3, 4, 6))
    g = rng.standard_normal(5)
    be = rng.standard_normal(5)
    eps = 1e-5
    out, mean, var = oracle.batchnorm3d_train(t, None, None, eps, return_stats=True)
    np.testing.assert_allclose(mean, t.mean(axis=(0, 2, 3, 4)), rtol=1e-13)
    np.testing.assert_allclose(var, t.var(axis=(0, 2, 3, 4)), rtol=1e-12)  # biased (ddof=0)
    np.testing.assert_allclose(out.mean(axis=(0, 2, 3, 4)), 0.0, atol=1e-13)
    np.testing.assert_allclose(out.var(axis=(0, 2, 3, 4)), var / (var + eps), rtol=1e-12)
    out2 = oracle.batchnorm3d_train(t, g, be, eps)
    np.testing.assert_allclose(out2, out * g[None, :, None, None, None] +
                               be[None, :, None, None, None], rtol=1e-13, atol=1e-13)


def test_bn_commutes_with_avgpool(oracle):
    """A per-channel affine map commutes with average pooling (l2_p72)."""
    t = rng.standard_normal((2, 3, 8, 8, 8))
    out, mean, var = oracle.batchnorm3d_train(t, None, None, 1e-5, return_stats=True)
    a = oracle.avgpool3d_2(oracle.avgpool3d_2(out))
    p = oracle.avgpool3d_2(oracle.avgpool3d_2(t))
    b = (p - mean[None, :, None, None, None]) / np.sqrt(var + 1e-5)[None, :, None, None, None]
    assert _rel(a, b) <= 1e-13


def test_batchnorm_eval_closed_forms(oracle):
    """Evaluation-mode BN (running statistics, l2_p72's fused kernel):
    identity statistics give the input back exactly, eps = 0 with a perfect
    square variance gives a hand-checkable affine map, and running statistics
    equal to the batch moments reproduce training mode."""
    t = 3.0 + 2.0 * rng.standard_normal((3, 4, 2, 5, 3))
    C = t.shape[1]
    eps = 1e-5
    ident = oracle.batchnorm3d_eval(t, np.zeros(C), np.ones(C), None, None, 0.0)
    np.testing.assert_array_equal(ident, t)
    rm = np.array([2.0, -1.0, 0.5, 0.0])
    rv = np.array([4.0, 0.25, 1.0, 16.0])
    g = np.array([1.5, -2.0, 0.0, 1.0])
    be = np.array([0.0, 1.0, 3.0, -4.0])
    out = oracle.batchnorm3d_eval(t, rm, rv, g, be, 0.0)
    sd = np.array([2.0, 0.5, 1.0, 4.0])
    want = (t - rm[None, :, None, None, None]) / sd[None, :, None, None, None] \
        * g[None, :, None, None, None] + be[None, :, None, None, None]
    np.testing.assert_allclose(out, want, rtol=1e-15, atol=1e-15)
    assert np.all(out[:, 2] == 3.0)  # gamma 0: the channel is beta alone
    tr, mean, var = oracle.batchnorm3d_train(t, g, be, eps, return_stats=True)
    ev = oracle.batchnorm3d_eval(t, mean, var, g, be, eps)
    np.testing.assert_allclose(ev, tr, rtol=1e-13, atol=1e-13)


def test_convT_bneval_avgpool_reductions(oracle):
    """The eval composite reduces to the pinned pieces: identity statistics
    give avgpool(avgpool(convT)), and the batch moments as running
    statistics give the training-mode composite."""
    x = rng.standard_normal((2, 3, 5, 6, 5))
    W = rng.standard_normal((3, 4, 3, 3, 3))
    b = rng.standard_normal(4)
    g = rng.standard_normal(4)
    be = rng.standard_normal(4)
    kt = dict(stride=2, padding=1)
    C = 4
    y = oracle.convT_bneval_avgpool(x, W, b, np.zeros(C), np.ones(C), None, None, 0.0, **kt)
    ref = oracle.avgpool3d_2(oracle.avgpool3d_2(oracle.conv_transpose3d(x, W, b, **kt)))
    assert _rel(y, ref) <= 1e-14
    full = oracle.conv_transpose3d(x, W, b, **kt)
    mean, var = full.mean(axis=(0, 2, 3, 4)), full.var(axis=(0, 2, 3, 4))
    ev = oracle.convT_bneval_avgpool(x, W, b, mean, var, g, be, 1e-5, **kt)
    tr = oracle.convT_bn_avgpool(x, W, b, g, be, 1e-5, **kt)
    assert _rel(ev, tr) <= 1e-12


# --------------------------------------------------------------------------
# sampled evaluators equal the full ones
# --------------------------------------------------------------------------
def test_sampled_equal_full(oracle):
    x = rng.standard_normal((2, 4, 9, 8, 10))
    Wc = rng.standard_normal((6, 2, 3, 3, 2))
    b = rng.standard_normal(6)
    kw = dict(stride=(1, 2, 1), padding=(1, 1, 0), dilation=(1, 1, 2), groups=2)
    y = oracle.conv3d(x, Wc, b, **kw)
    idx = np.arange(0, y.size, 7)
    np.testing.assert_array_equal(oracle.conv3d_at(x, Wc, b, idx, **kw), y.ravel()[idx])
    Wt = rng.standard_normal((4, 3, 3, 2, 3))
    bt = rng.standard_normal(6)
    kt = dict(stride=(2, 1, 2), padding=(1, 0, 1), dilation=(2, 1, 1), output_padding=(1, 0, 1),
              groups=2)
    yt = oracle.conv_transpose3d(x, Wt, bt, **kt)
    idx = np.arange(0, yt.size, 5)
    np.testing.assert_array_equal(oracle.conv_transpose3d_at(x, Wt, bt, idx, **kt),
                                  yt.ravel()[idx])
    m = oracle.conv_maxpool_lse_relu(x, Wc, b, **kw)
    idx = np.arange(m.size)
    np.testing.assert_array_equal(oracle.conv_maxpool_lse_relu_at(x, Wc, b, idx, **kw),
                                  m.ravel())
    xs = rng.standard_normal((2, 4, 5, 6, 4))
    c = oracle.convT_bn_avgpool(xs, Wt, bt, None, None, 1e-5, **kt)
    idx = np.arange(c.size)
    cs, mean, var = oracle.convT_bn_avgpool_at(xs, Wt, bt, idx, None, None, 1e-5,
                                               return_stats=True, **kt)
    assert _rel(cs, c.ravel()) <= 1e-12
    full = oracle.conv_transpose3d(xs, Wt, bt, **kt)
    np.testing.assert_allclose(mean, full.mean(axis=(0, 2, 3, 4)), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(var, full.var(axis=(0, 2, 3, 4)), rtol=1e-12)
    rm = rng.standard_normal(6)
    rv = rng.uniform(0.5, 2.0, 6)
    g = rng.standard_normal(6)
    be = rng.standard_normal(6)
    e = oracle.convT_bneval_avgpool(xs, Wt, bt, rm, rv, g, be, 1e-5, **kt)
    es = oracle.convT_bneval_avgpool_at(xs, Wt, bt, rm, rv, np.arange(e.size), g, be, 1e-5, **kt)
    assert _rel(es, e.ravel()) <= 1e-12


# --------------------------------------------------------------------------
# PyTorch CPU fp64 cross-check (a library routine, test-only)
# --------------------------------------------------------------------------
torch = pytest.importorskip("torch")
F = torch.nn.functional


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a))


TORCH_CASES = [
    ((2, 4, 7, 8, 6), (6, 2, 3, 3, 2), (1, 2, 1), (1, 0, 2), (1, 1, 2), 2),
    ((1, 3, 6, 5, 9), (4, 3, 3, 1, 3), (2, 1, 3), (0, 1, 1), (2, 1, 1), 1),
    ((2, 4, 16, 16, 4), (8, 4, 3, 3, 1), (1, 1, 1), (0, 0, 0), (1, 1, 1), 1),
]


@pytest.mark.parametrize("xs,ws,s,p,d,G", TORCH_CASES)
def test_conv3d_vs_torch(oracle, xs, ws, s, p, d, G):
    x = rng.standard_normal(xs)
    W = rng.standard_normal(ws)
    b = rng.standard_normal(ws[0])
    y = oracle.conv3d(x, W, b, s, p, d, G)
    ref = F.conv3d(_t(x), _t(W), _t(b), s, p, d, G).numpy()
    assert _rel(y, ref) <= 1e-13


CT_CASES = [
    ((2, 4, 5, 6, 4), (4, 3, 3, 3, 3), (2, 2, 2), (1, 1, 1), (2, 2, 2), (0, 1, 1), 1),
    ((1, 6, 4, 5, 3), (6, 2, 3, 2, 3), (2, 3, 1), (1, 0, 2), (1, 2, 3), (1, 2, 0), 3),
    ((2, 3, 6, 6, 6), (3, 4, 3, 3, 3), (2, 2, 2), (1, 1, 1), (1, 1, 1), (0, 0, 0), 1),
]


@pytest.mark.parametrize("xs,ws,s,p,d,op,G", CT_CASES)
def test_conv_transpose3d_vs_torch(oracle, xs, ws, s, p, d, op, G):
    x = rng.standard_normal(xs)
    W = rng.standard_normal(ws)
    b = rng.standard_normal(ws[1] * G)
    y = oracle.conv_transpose3d(x, W, b, s, p, d, op, G)
    ref = F.conv_transpose3d(_t(x), _t(W), _t(b), s, p, op, G, d).numpy()
    assert _rel(y, ref) <= 1e-13


def test_convT_bn_avgpool_vs_torch(oracle):
    x = rng.standard_normal((3, 3, 8, 9, 8))
    W = rng.standard_normal((3, 5, 3, 3, 3))
    b = rng.standard_normal(5)
    g = rng.standard_normal(5)
    be = rng.standard_normal(5)
    y = oracle.convT_bn_avgpool(x, W, b, g, be, 1e-5, stride=2, padding=1)
    t = F.conv_transpose3d(_t(x), _t(W), _t(b), 2, 1)
    t = F.batch_norm(t, None, None, _t(g), _t(be), training=True, eps=1e-5)
    t = F.avg_pool3d(F.avg_pool3d(t, 2), 2)
    assert _rel(y, t.numpy()) <= 1e-12


def test_convT_bneval_avgpool_vs_torch(oracle):
    x = rng.standard_normal((2, 3, 7, 8, 9))
    W = rng.standard_normal((3, 6, 3, 2, 3))
    b = rng.standard_normal(6)
    rm = rng.standard_normal(6)
    rv = rng.uniform(0.2, 3.0, 6)
    g = rng.standard_normal(6)
    be = rng.standard_normal(6)
    kt = dict(stride=(2, 2, 1), padding=(1, 0, 1), output_padding=(1, 0, 0))
    y = oracle.convT_bneval_avgpool(x, W, b, rm, rv, g, be, 1e-5, **kt)
    t = F.conv_transpose3d(_t(x), _t(W), _t(b), (2, 2, 1), (1, 0, 1), (1, 0, 0))
    t = F.batch_norm(t, _t(rm), _t(rv), _t(g), _t(be), training=False, eps=1e-5)
    t = F.avg_pool3d(F.avg_pool3d(t, 2), 2)
    assert _rel(y, t.numpy()) <= 1e-12
    rb = oracle.batchnorm3d_eval(x, rm[:3], rv[:3], g[:3], be[:3], 1e-3)
    tb = F.batch_norm(_t(x), _t(rm[:3]), _t(rv[:3]), _t(g[:3]), _t(be[:3]), training=False,
                      eps=1e-3)
    assert _rel(rb, tb.numpy()) <= 1e-14


def test_conv_maxpool_lse_relu_vs_torch(oracle):
    x = rng.standard_normal((2, 4, 8, 10, 9))
    W = rng.standard_normal((6, 4, 3, 3, 3))
    b = rng.standard_normal(6) - 2.0  # push some LSE values negative
    y = oracle.conv_maxpool_lse_relu(x, W, b, padding=1)
    t = F.conv3d(_t(x), _t(W), _t(b), 1, 1)
    t = torch.relu(torch.logsumexp(F.max_pool3d(t, 2, 2), dim=1, keepdim=True))
    assert _rel(y, t.numpy()) <= 1e-13
