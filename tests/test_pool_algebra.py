"""The algebraic BN-pool path, replayed on the CPU from the library's plan.

The library plans stride-2 transposed convs with few input channels as:
- batch statistics from patch Gram matrices over a few row boxes (the full
  row box and its last planes), combined per parity class by
  inclusion-exclusion; or, with at most 3 channels, in lag form: sums of
  x[c, z] x[c', z + delta] per region of x, each class entry the sum of the
  regions its position range covers;
- the pooled output as a stride-2 conv of x with summed weights, the
  BatchNorm scale and shift folded into that conv's weights and bias.

These tests take the plan's tables from ``plan_describe``, carry the same
algebra out in fp64 numpy, and compare with the oracle's literal composite
(conv_transpose3d -> batch_norm -> two AvgPool3d(2)).  A wrong offset,
tap, box or sign in the plan fails here without a GPU.
"""
import numpy as np
import pytest

import oracle as orc
import transposed_conv_epilogues_gb300 as tc

pytestmark = pytest.mark.usefixtures("lib")

rng = np.random.default_rng(11)


@pytest.fixture(scope="module")
def lib():
    from transposed_conv_epilogues_gb300 import build
    build.build()
    tc.load()


def _gather(x, lo, hi, U):
    """P[row, d] for the rows of box [lo, hi), d = ci * V + (i0 * n1 + i1) * n2 + i2,
    x taken as zero outside its extent."""
    a = x
    for ax in range(3):
        L = x.shape[2 + ax]
        idx = np.arange(lo[ax], hi[ax])[:, None] + np.asarray(U[ax])[None, :]
        ok = (idx >= 0) & (idx < L)
        a = np.take(a, np.clip(idx, 0, L - 1), axis=2 + 2 * ax)
        shape = [1] * a.ndim
        shape[2 + 2 * ax], shape[3 + 2 * ax] = ok.shape
        a = a * ok.reshape(shape)
    # a: (N, C, e0, n0, e1, n1, e2, n2) -> (N, e0, e1, e2, C, n0, n1, n2)
    a = a.transpose(0, 2, 4, 6, 1, 3, 5, 7)
    return a.reshape(-1, int(np.prod(a.shape[4:])))


def _region_sums(f, seg):
    """Sum of f [N, L0, L1, L2] over every region (product of segments)."""
    r = f.sum(axis=0)
    for ax in range(3):
        r = np.add.reduceat(r, seg[ax][:-1], axis=ax)
    return r


def _lag_stats(x, W, pl):
    """Batch mean and variance of the transposed conv from the lag form: sums
    of x[c, z] and of x[c, z] x[c2, z + delta] per region, each class entry
    the sum of the regions its z range covers (the plan's segment ranges)."""
    N, C = x.shape[:2]
    L = x.shape[2:]
    Cout = W.shape[1]
    U, taps, seg, sr = pl["pool_U"], pl["pool_taps"], pl["lag_seg"], pl["lag_srange"]
    nU = [len(u) for u in U]
    xp = np.pad(x, ((0, 0), (0, 0), (1, 1), (1, 1), (1, 1)))

    def shifted(c, dl):
        return xp[:, c, 1 + dl[0]:1 + dl[0] + L[0], 1 + dl[1]:1 + dl[1] + L[1],
                  1 + dl[2]:1 + dl[2] + L[2]]

    first = {c: _region_sums(x[:, c], seg) for c in range(C)}
    prod = {}

    def region_prod(c, c2, dl):
        key = (c, c2, tuple(dl))
        if key not in prod:
            prod[key] = _region_sums(x[:, c] * shifted(c2, dl), seg)
        return prod[key]

    def covered(rs, r, v):
        (a0, b0), (a1, b1), (a2, b2) = (sr[ax][r[ax]][v[ax]] for ax in range(3))
        return rs[a0:b0, a1:b1, a2:b2].sum()

    O = pl["O"]
    count = N * O[0] * O[1] * O[2]
    mean, var = np.zeros(Cout), np.zeros(Cout)
    for co in range(Cout):
        s1 = s2 = 0.0
        for r, _coef in pl["pool_cls"]:
            ent = []  # (channel, offset indices, weight)
            for ci in range(C):
                for k0, u0 in taps[0][r[0]]:
                    for k1, u1 in taps[1][r[1]]:
                        for k2, u2 in taps[2][r[2]]:
                            ent.append((ci, (u0, u1, u2), W[ci, co, k0, k1, k2]))
            for ci, vi, wi in ent:
                s1 += wi * covered(first[ci], r, vi)
                for cj, vj, wj in ent:
                    # the factor earlier in (channel, offsets) order comes first
                    (ca, va), (cb, vb) = sorted([(ci, vi), (cj, vj)])
                    dl = [vb[ax] - va[ax] for ax in range(3)]
                    s2 += wi * wj * covered(region_prod(ca, cb, dl), r, va)
        mean[co] = s1 / count
        var[co] = s2 / count - mean[co] ** 2
    assert all(n <= 2 for n in nU)
    return mean, var


def _replay(x, W, b, gamma, beta, eps, kw, op, rm=None, rv=None):
    s, p, d, outp = kw["stride"], kw["padding"], kw["dilation"], kw["output_padding"]
    pl = tc.plan_describe(op, x.shape, W.shape, s, p, d, outp)
    assert pl["status"] == 0 and pl["pool_ok"] == 1, pl.get("pool_ok")
    N, C = x.shape[:2]
    Cout = W.shape[1]
    U, taps = pl["pool_U"], pl["pool_taps"]
    nU = [len(u) for u in U]
    V = nU[0] * nU[1] * nU[2]
    assert pl["pool_D"] == C * V
    k = W.shape[2:]
    pad = [p] * 3 if np.isscalar(p) else list(p)
    dil = [d] * 3 if np.isscalar(d) else list(d)
    if op == 3 and pl.get("lag"):
        mean, var = _lag_stats(x, W, pl)
        t = orc.conv_transpose3d(x, W, None, s, p, d, outp)
        np.testing.assert_allclose(mean, t.mean(axis=(0, 2, 3, 4)), rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(var, t.var(axis=(0, 2, 3, 4)), rtol=1e-10)
        scale = gamma / np.sqrt(var + eps)
        shift = beta - mean * scale
    elif op == 3:
        Gs, ss = [], []
        for bx in pl["pool_boxes"]:
            P = _gather(x, bx[:3], bx[3:], U)
            Gs.append(P.T @ P)
            ss.append(P.sum(axis=0))
        O = pl["O"]
        count = N * O[0] * O[1] * O[2]
        mean = np.zeros(Cout)
        var = np.zeros(Cout)
        for co in range(Cout):
            s1 = s2 = 0.0
            for r, coef in pl["pool_cls"]:
                ds, ws = [], []
                for ci in range(C):
                    for k0, u0 in taps[0][r[0]]:
                        for k1, u1 in taps[1][r[1]]:
                            for k2, u2 in taps[2][r[2]]:
                                ds.append(ci * V + (u0 * nU[1] + u1) * nU[2] + u2)
                                ws.append(W[ci, co, k0, k1, k2])
                ds, ws = np.array(ds), np.array(ws)
                for cf, G, sv in zip(coef, Gs, ss):
                    if cf:
                        s1 += cf * ws @ sv[ds]
                        s2 += cf * ws @ G[np.ix_(ds, ds)] @ ws
            mean[co] = s1 / count
            var[co] = s2 / count - mean[co] ** 2
        # the statistics themselves, against the literal transposed conv
        t = orc.conv_transpose3d(x, W, None, s, p, d, outp)
        np.testing.assert_allclose(mean, t.mean(axis=(0, 2, 3, 4)), rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(var, t.var(axis=(0, 2, 3, 4)), rtol=1e-10)
        scale = gamma / np.sqrt(var + eps)
        shift = beta - mean * scale
    else:
        scale = gamma / np.sqrt(rv + eps)
        shift = beta + (b - rm) * scale
    # summed weights: W'[e] = sum of W[k] over taps with 2e - p + d k in [0, 3]
    emin, Ke = pl["pool_e_min"], pl["pool_Ke"]
    ind = []
    for ax in range(3):
        m = np.zeros((Ke[ax], k[ax]))
        for e in range(Ke[ax]):
            for kk in range(k[ax]):
                j = 2 * (emin[ax] + e) - pad[ax] + dil[ax] * kk
                m[e, kk] = 0 <= j <= 3
        ind.append(m)
    W2 = np.einsum("ioabc,xa,yb,zc->oixyz", W, *ind) * (scale / 64.0)[:, None, None, None, None]
    y = orc.conv3d(x, W2, shift, stride=2, padding=tuple(-e for e in emin))
    Pp = pl["P"]
    return y[:, :, :Pp[0], :Pp[1], :Pp[2]]


CASES = [
    # x shape, convT weight shape, stride, pad, dil, output_padding
    ((2, 3, 8, 8, 8), (3, 5, 3, 3, 3), 2, 1, 1, 0),              # the workload's form
    ((2, 2, 9, 7, 10), (2, 4, 3, 3, 3), 2, 0, 1, 0),             # pad 0: e_min = -1
    ((1, 4, 5, 6, 7), (4, 3, 3, 3, 3), 2, 1, 1, (1, 0, 1)),      # D = 32, no slab on some axes
    ((2, 1, 9, 8, 7), (1, 4, 2, 3, 5), 2, (0, 1, 2), (1, 1, 3), 1),  # widened pooled-conv pad
    ((3, 2, 6, 5, 9), (2, 3, 2, 4, 3), 2, (0, 1, 1), 1, (1, 0, 0)),
    # one parity class per axis (the fused epilogue cannot run): k 1, and k 2 at dilation 2
    ((2, 3, 8, 7, 9), (3, 4, 1, 1, 1), 2, 0, 1, (1, 0, 1)),
    ((2, 4, 7, 8, 6), (4, 5, 2, 2, 2), 2, 0, 2, 1),
]


# the lag form applies: at most 3 channels, one or two consecutive offsets
# per axis, rows along axis 2 a multiple of 4
LAG_CASES = [
    ((2, 3, 8, 8, 8), (3, 5, 3, 3, 3), 2, 1, 1, 0),
    ((2, 2, 9, 7, 12), (2, 4, 3, 3, 3), 2, 0, 1, 0),              # pad 0: offsets {-1, 0}
    ((1, 3, 5, 6, 36), (3, 3, 3, 3, 3), 2, 1, 1, (1, 0, 1)),      # two column blocks
    ((2, 1, 9, 10, 8), (1, 4, 2, 3, 1), 2, (0, 1, 0), 1, (1, 1, 1)),  # one offset on axis 2
    ((3, 2, 6, 17, 4), (2, 3, 3, 2, 3), 2, (1, 0, 1), 1, 0),      # ragged row block
]


@pytest.mark.parametrize("case", LAG_CASES)
def test_pool_path_lag_replay(case):
    xs, ws, s, p, d, op = case
    pl = tc.plan_describe(3, xs, ws, s, p, d, op)
    assert pl["pool_path"] == 1 and pl["lag"] == 1, (pl.get("pool_path"), pl.get("lag"))
    x = rng.standard_normal(xs)
    W = rng.standard_normal(ws) * 0.3
    b = rng.standard_normal(ws[1]) * 0.2
    g = rng.uniform(0.5, 1.5, ws[1])
    be = rng.uniform(-0.5, 0.5, ws[1])
    kw = dict(stride=s, padding=p, dilation=d, output_padding=op)
    y = _replay(x, W, b, g, be, 1e-5, kw, 3)
    ref = orc.convT_bn_avgpool(x, W, b, g, be, 1e-5, **kw)
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("case", LAG_CASES + [((64, 3, 32, 32, 32), (3, 16, 3, 3, 3), 2, 1, 1, 0)])
def test_lag_work_split(case):
    """Every (sample, plane, row, column) of x is a step of exactly one CTA
    thread; a CTA's planes lie in one segment of axis 0, and the grid stays
    at one CTA per SM where the jobs allow."""
    xs, ws, s, p, d, op = case
    pl = tc.plan_describe(3, xs, ws, s, p, d, op)
    assert pl["lag"] == 1
    N, L = xs[0], xs[2:]
    seg0, nc, cta0 = pl["lag_seg"][0], pl["lag_nc"], pl["lag_cta0"]
    nb1, nb2 = pl["lag_nb"]
    assert nb1 == -(-L[1] // 8) and nb2 == -(-L[2] // 32)
    grid = pl["lag_grid"]
    assert cta0[-1] == grid
    assert grid <= max(152, nb1 * nb2 * (len(seg0) - 1))
    cover = np.zeros((N, L[0], nb1 * 8, nb2 * 32), np.int32)
    for bid in range(grid):
        s0 = max(i for i in range(len(nc)) if cta0[i] <= bid)
        local = bid - cta0[s0]
        job, k = divmod(local, nc[s0])
        b1, b2 = divmod(job, nb2)
        z0a, ln = seg0[s0], seg0[s0 + 1] - seg0[s0]
        items = N * ln
        for it in range(items * k // nc[s0], items * (k + 1) // nc[s0]):
            n, z0 = divmod(it, ln)
            cover[n, z0a + z0, 8 * b1:8 * b1 + 8, 32 * b2:32 * b2 + 32] += 1
    assert (cover[:, :, :L[1], :L[2]] == 1).all()


@pytest.mark.parametrize("case", CASES)
def test_pool_path_batch_stats_replay(case):
    xs, ws, s, p, d, op = case
    x = rng.standard_normal(xs)
    W = rng.standard_normal(ws) * 0.3
    b = rng.standard_normal(ws[1]) * 0.2
    g = rng.uniform(0.5, 1.5, ws[1])
    be = rng.uniform(-0.5, 0.5, ws[1])
    kw = dict(stride=s, padding=p, dilation=d, output_padding=op)
    y = _replay(x, W, b, g, be, 1e-5, kw, 3)
    ref = orc.convT_bn_avgpool(x, W, b, g, be, 1e-5, **kw)
    assert y.shape == ref.shape
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("case", CASES[:3])
def test_pool_path_eval_replay(case):
    xs, ws, s, p, d, op = case
    x = rng.standard_normal(xs)
    W = rng.standard_normal(ws) * 0.3
    b = rng.standard_normal(ws[1]) * 0.2
    rm = rng.standard_normal(ws[1]) * 0.2
    rv = rng.uniform(0.05, 0.5, ws[1])
    g = rng.uniform(0.5, 1.5, ws[1])
    be = rng.uniform(-0.5, 0.5, ws[1])
    kw = dict(stride=s, padding=p, dilation=d, output_padding=op)
    y = _replay(x, W, b, g, be, 1e-5, kw, 4, rm, rv)
    ref = orc.convT_bneval_avgpool(x, W, b, rm, rv, g, be, 1e-5, **kw)
    np.testing.assert_allclose(y, ref, rtol=1e-9, atol=1e-11)


def test_pool_path_selection():
    """Where the algebraic path applies: stride 2 everywhere, groups 1, patch
    of at most 32 entries.  The workload shape has a 24-entry patch
    (3 channels x 2x2x2 offsets), 8 boxes and 8 classes.  It is taken for
    running statistics always, for batch statistics only where the fused
    engine epilogue cannot run."""
    c4 = tc.plan_describe(3, (64, 3, 32, 32, 32), (3, 16, 3, 3, 3), 2, 1)
    assert c4["pool_ok"] == 1 and c4["pool_D"] == 24 and c4["pool_nbox"] == 8
    assert c4["pool_ncls"] == 8 and c4["pool_Ke"] == [3, 3, 3] and c4["pool_e_min"] == [0, 0, 0]
    # batch statistics in lag form: segments {0}, [1, 31), {31} per axis
    assert c4["fused"] == 1 and c4["pool_path"] == 1 and c4["lag"] == 1
    assert c4["lag_seg"] == [[0, 1, 31, 32]] * 3 and c4["lag_grid"] == 152
    # 4 channels: the patch-Gram statistics; the fused epilogue stays faster
    c4b = tc.plan_describe(3, (8, 4, 16, 16, 16), (4, 16, 3, 3, 3), 2, 1)
    assert c4b["pool_ok"] == 1 and c4b["lag"] == 0 and c4b["pool_path"] == 0
    assert tc.plan_describe(4, (64, 3, 32, 32, 32), (3, 16, 3, 3, 3), 2, 1)["pool_path"] == 1
    k1 = tc.plan_describe(3, (2, 3, 8, 7, 9), (3, 4, 1, 1, 1), 2, 0, 1, (1, 0, 1))
    assert k1["fused"] == 0 and k1["pool_path"] == 1
    # 7 channels: 56 patch entries -> the fused engine epilogue
    assert tc.plan_describe(3, (2, 7, 9, 8, 10), (7, 5, 3, 3, 3), 2, 1)["pool_ok"] == 0
    # a stride-1 axis or groups -> not this path
    assert tc.plan_describe(3, (2, 3, 9, 5, 6), (3, 4, 3, 3, 3), (1, 2, 2), 1)["pool_path"] == 0
    assert tc.plan_describe(3, (2, 4, 6, 7, 8), (4, 3, 3, 3, 3), 2, 1, 1, 0,
                            2)["pool_path"] == 0
