"""CPU tests of the C-ABI library: it loads, exports every declared symbol, and
its host-side logic (output shapes, argument validation, the transposed
convolution's parity classes and tap tables) is exact.  No device calls."""
import ctypes
import itertools
import os
import re

import numpy as np
import pytest

import transposed_conv_epilogues_gb300 as tc
from transposed_conv_epilogues_gb300 import build as tcbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    tcbuild.build()
    return tc.load()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "tc3d.h")).read()
    return sorted(set(re.findall(r"\b(tc3d_[A-Za-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_symbols()
    assert set(declared) == set(tc.EXPORTED)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for st in range(-10, 1):
        assert tc.status_string(st) not in ("", "unknown status")
    assert tc.status_string(-99) == "unknown status"


# --------------------------------------------------------------------------
# output shapes agree with the oracle's independent size formulas
# --------------------------------------------------------------------------
def test_out_shapes_vs_oracle(lib, oracle):
    rng = np.random.default_rng(3)
    for _ in range(300):
        S = tuple(int(v) for v in rng.integers(1, 12, 3))
        k = tuple(int(v) for v in rng.integers(1, 5, 3))
        s = tuple(int(v) for v in rng.integers(1, 4, 3))
        p = tuple(int(v) for v in rng.integers(0, 3, 3))
        d = tuple(int(v) for v in rng.integers(1, 4, 3))
        G = int(rng.choice([1, 2]))
        xs, wc, wt = (2, 2 * G) + S, (2 * G, 2) + k, (2 * G, 3) + k
        ref = oracle.conv_out_shape(xs, wc, s, p, d)
        if min(ref) > 0:
            assert tc.out_shape(0, xs, wc, s, p, d, 0, G) == ref
            if min(ref[2:]) >= 2:
                assert tc.out_shape(2, xs, wc, s, p, d, 0, G) == (2, 1) + tuple(
                    o // 2 for o in ref[2:])
        else:
            with pytest.raises(tc.Tc3dError):
                tc.out_shape(0, xs, wc, s, p, d, 0, G)
        op = tuple(int(rng.integers(0, max(a, b))) for a, b in zip(s, d))
        reft = oracle.convT_out_shape(xs, wt, s, p, d, op, G)
        if min(reft) > 0:
            assert tc.out_shape(1, xs, wt, s, p, d, op, G) == reft
            if min(reft[2:]) >= 4:
                assert tc.out_shape(3, xs, wt, s, p, d, op, G) == reft[:2] + tuple(
                    o // 4 for o in reft[2:])


def test_workload_shapes(lib):
    from transposed_conv_epilogues_gb300.workloads import WORKLOADS
    ops = {"conv3d": 0, "conv_transpose3d": 1, "conv_maxpool_lse_relu": 2, "convT_bn_avgpool": 3,
           "convT_bneval_avgpool": 4}
    expect = {1: (2, 8, 14, 14, 4), 2: (16, 64, 126, 126, 8), 3: (16, 64, 33, 65, 65),
              4: (64, 16, 15, 15, 15), 5: (4, 1, 16, 64, 64)}
    for wl in WORKLOADS:
        assert tc.out_shape(ops[wl.op], wl.x_shape, wl.w_shape, wl.stride, wl.padding,
                            wl.dilation, wl.output_padding, wl.groups) == expect[wl.index]


# --------------------------------------------------------------------------
# argument validation happens on the host, before any device work
# --------------------------------------------------------------------------
def _call(lib, fn, ptrs, geom, ws=256):
    dummy = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    return fn(*ptrs, *geom, dummy if ws else None, ctypes.c_size_t(ws), None)


def _geom(N=1, Cin=2, S=(4, 4, 4), Cout=2, k=(3, 3, 3), s=(1, 1, 1), p=(0, 0, 0), d=(1, 1, 1),
          op=(0, 0, 0), G=1):
    I3 = ctypes.c_int * 3
    return (N, Cin, *S, Cout, *k, I3(*s), I3(*p), I3(*d), I3(*op), G)


@pytest.mark.parametrize("name", ["tc3d_conv3d_fwd", "tc3d_conv_transpose3d_fwd",
                                  "tc3d_conv_maxpool_lse_relu"])
def test_argument_errors(lib, name):
    fn = getattr(lib, name)
    P = ctypes.c_void_p
    ok = (P(256), P(512), None, P(1024))
    assert _call(lib, fn, (None, P(512), None, P(1024)), _geom()) == tc.TC3D_ERR_NULL
    assert _call(lib, fn, (P(256), None, None, P(1024)), _geom()) == tc.TC3D_ERR_NULL
    assert _call(lib, fn, (P(256), P(512), None, None), _geom()) == tc.TC3D_ERR_NULL
    assert _call(lib, fn, ok, _geom(N=0)) == tc.TC3D_ERR_SHAPE
    assert _call(lib, fn, ok, _geom(S=(4, -1, 4))) == tc.TC3D_ERR_SHAPE
    assert _call(lib, fn, ok, _geom(s=(1, 0, 1))) == tc.TC3D_ERR_SHAPE
    assert _call(lib, fn, ok, _geom(Cin=3, G=2)) == tc.TC3D_ERR_GROUPS
    assert _call(lib, fn, ok, _geom(Cout=3, G=2, Cin=2)) == tc.TC3D_ERR_GROUPS
    assert _call(lib, fn, ok, _geom(k=(17, 1, 1), S=(20, 4, 4))) == tc.TC3D_ERR_UNSUPPORTED
    assert _call(lib, fn, (P(258), P(512), None, P(1024)), _geom()) == tc.TC3D_ERR_ALIGN
    assert _call(lib, fn, ok, _geom(), ws=0) == tc.TC3D_ERR_WORKSPACE
    if name == "tc3d_conv_transpose3d_fwd":
        assert _call(lib, fn, ok, _geom(s=(2, 2, 2), op=(2, 0, 0))) == tc.TC3D_ERR_OUTPUT_PADDING
        assert _call(lib, fn, ok, _geom(s=(2, 1, 1), d=(3, 1, 1), op=(2, 0, 0))) != \
            tc.TC3D_ERR_OUTPUT_PADDING  # op < max(stride, dilation) is allowed
    else:
        assert _call(lib, fn, ok, _geom(op=(1, 0, 0))) == tc.TC3D_ERR_OUTPUT_PADDING
        assert _call(lib, fn, ok, _geom(S=(2, 4, 4))) == tc.TC3D_ERR_SHAPE  # empty output
    if name == "tc3d_conv_maxpool_lse_relu":
        assert _call(lib, fn, ok, _geom(S=(3, 4, 4))) == tc.TC3D_ERR_SHAPE  # pool of 1 -> 0


def test_convT_bn_avgpool_argument_errors(lib):
    fn = lib.tc3d_convT_bn_avgpool
    P = ctypes.c_void_p
    dummy = P(256)

    def call(geom, eps=1e-5, ws=256, x=P(256)):
        return fn(x, P(512), None, None, None, ctypes.c_float(eps), P(1024), *geom,
                  dummy if ws else None, ctypes.c_size_t(ws), None)

    assert call(_geom(S=(2, 2, 2), s=(2, 2, 2), p=(1, 1, 1))) == tc.TC3D_ERR_SHAPE  # 3 -> 0
    assert call(_geom(), x=None) == tc.TC3D_ERR_NULL
    assert call(_geom(s=(2, 2, 2)), ws=0) == tc.TC3D_ERR_WORKSPACE
    assert call(_geom(s=(2, 2, 2)), eps=-1.0) == tc.TC3D_ERR_SHAPE


def test_convT_bneval_avgpool_argument_errors(lib):
    fn = lib.tc3d_convT_bneval_avgpool
    P = ctypes.c_void_p
    dummy = P(256)

    def call(geom, eps=1e-5, ws=256, x=P(256), rm=P(2048), rv=P(4096)):
        return fn(x, P(512), None, rm, rv, None, None, ctypes.c_float(eps), P(1024), *geom,
                  dummy if ws else None, ctypes.c_size_t(ws), None)

    g2 = _geom(s=(2, 2, 2))
    assert call(_geom(S=(2, 2, 2), s=(2, 2, 2), p=(1, 1, 1))) == tc.TC3D_ERR_SHAPE  # 3 -> 0
    assert call(g2, x=None) == tc.TC3D_ERR_NULL
    assert call(g2, rm=None) == tc.TC3D_ERR_NULL
    assert call(g2, rv=None) == tc.TC3D_ERR_NULL
    assert call(g2, ws=0) == tc.TC3D_ERR_WORKSPACE
    assert call(g2, eps=-1.0) == tc.TC3D_ERR_SHAPE
    big = 1 << 24
    assert call(g2, ws=big, rm=P(2050)) == tc.TC3D_ERR_ALIGN
    # same plan as the batch-statistics op, but no partial-sum region
    a = tc.plan_describe(3, (2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 2, 1)
    b = tc.plan_describe(4, (2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 2, 1)
    assert b["fused"] == a["fused"] == 1 and b["tiles"] == a["tiles"]
    wa = tc.workspace_bytes(3, (2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 2, 1)
    wb = tc.workspace_bytes(4, (2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 2, 1)
    assert wb < wa
    assert tc.out_shape(4, (2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 2, 1) == tc.out_shape(
        3, (2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 2, 1) == (2, 16, 3, 3, 3)


def test_direct_and_ndhwc_plans(lib):
    """Grouped convs with few channels per group take the direct kernel;
    dense channels-last convs the engine's channels-last mode (workspace: the
    packed weights only); grouped ones that are not direct the route through
    two layout transposes (workspace: + NCDHW copies of x and y)."""
    dw = tc.plan_describe(0, (2, 8, 9, 10, 13), (8, 1, 3, 3, 3), 1, 1, 1, 0, 8)
    assert dw["direct"] == 1 and dw["ndhwc"] == 0
    assert tc.plan_describe(0, (2, 8, 7, 9, 8), (12, 4, 3, 3, 3), 1, 1, 1, 0, 2)["direct"] == 0
    assert tc.plan_describe(0, (2, 5, 9, 10, 12), (7, 5, 3, 3, 3), 1, 1)["direct"] == 0
    # 8 taps along x, or stride 3 there: not the direct kernel
    assert tc.plan_describe(0, (2, 8, 9, 10, 13), (8, 1, 3, 3, 8), 1, 1, 1, 0, 8)["direct"] == 0
    assert tc.plan_describe(0, (2, 8, 9, 10, 13), (8, 1, 3, 3, 3), 3, 1, 1, 0, 8)["direct"] == 0
    nd = tc.plan_describe(5, (2, 5, 9, 10, 12), (7, 5, 3, 3, 3), 1, 1)
    assert nd["ndhwc"] == 1 and nd["direct"] == 0 and nd["cl"] == 1 and nd["view"] == 0
    assert tc.out_shape(5, (2, 5, 9, 10, 12), (7, 5, 3, 3, 3), 1, 1) == (2, 9, 10, 12, 7)
    dense = tc.workspace_bytes(5, (2, 5, 9, 10, 12), (7, 5, 3, 3, 3), 1, 1)
    assert dense < 4 * (2 * 5 * 9 * 10 * 12 + 2 * 7 * 9 * 10 * 12)
    # grouped, 8 x 8 channels per group: not direct, not channels-last mode
    g2 = tc.plan_describe(5, (2, 16, 9, 10, 12), (16, 8, 3, 3, 3), 1, 1, 1, 0, 2)
    assert g2["ndhwc"] == 1 and g2["direct"] == 0 and g2["cl"] == 0
    assert tc.workspace_bytes(5, (2, 16, 9, 10, 12), (16, 8, 3, 3, 3), 1, 1, 1, 0, 2) >= \
        tc.workspace_bytes(0, (2, 16, 9, 10, 12), (16, 8, 3, 3, 3), 1, 1, 1, 0, 2) + \
        4 * (2 * 16 * 9 * 10 * 12 + 2 * 16 * 9 * 10 * 12)
    assert tc.workspace_bytes(5, (2, 8, 9, 10, 13), (8, 1, 3, 3, 3), 1, 1, 1, 0, 8) == 256


def test_direct_forms(lib):
    """Which direct kernel a conv takes: 0 the general one, 1 the NCDHW
    shared-memory tiled one, 2 the channels-last register-blocked 3 x 3 one,
    3 the channels-last streaming one (one input channel per group, a
    multiplier dividing 32, k0 <= 3 at stride 1, a 3 x 3 (y, x) plane), 4 the
    NCDHW streaming one (one input channel per group, a 3 x 3 x 3 filter,
    stride 1 along z and y)."""
    def form(op, xs, ws, s, p, d, G):
        pl = tc.plan_describe(op, xs, ws, s, p, d, 0, G)
        assert pl["direct"] == 1
        return pl["direct_form"]
    dw = ((2, 8, 9, 10, 13), (8, 1, 3, 3, 3), 1, 1, 1, 8)
    assert form(0, *dw) == 4 and form(5, *dw) == 3
    assert form(0, (1, 3, 7, 37, 136), (6, 1, 3, 3, 3), (1, 1, 2), (1, 1, 2), 1, 3) == 4
    # NCDHW, k0 = 1 or 2, or a 5-row filter: the tiled kernel
    assert form(0, (1, 3, 7, 35, 133), (6, 1, 1, 3, 3), (1, 1, 2), (0, 1, 1), 1, 3) == 1
    assert form(0, (2, 4, 9, 40, 70), (4, 1, 2, 3, 3), 1, 1, 1, 4) == 1
    assert form(0, (2, 2, 6, 33, 66), (2, 1, 3, 5, 2), 1, (1, 2, 0), (1, 1, 2), 2) == 1
    # k0 = 2 at stride 2 along x: its ring of 3 planes is over the tiled
    # kernel's shared-memory budget -> the general kernel
    assert form(0, (1, 3, 7, 35, 133), (6, 1, 2, 3, 3), (1, 1, 2), (0, 1, 1), 1, 3) == 0
    # stride 2 along x, a channel multiplier of 2, k0 = 2 / 1
    assert form(5, (1, 3, 7, 35, 133), (6, 1, 2, 3, 3), (1, 1, 2), (0, 1, 1), 1, 3) == 3
    assert form(5, (2, 36, 6, 7, 9), (36, 1, 1, 3, 3), 1, (0, 1, 0), 1, 36) == 3
    assert form(5, (1, 6, 11, 5, 6), (96, 1, 3, 3, 3), 1, 1, 1, 6) == 3      # multiplier 16
    # not streaming: two input channels per group, stride 2 along z, k0 = 4,
    # a multiplier of 3 -> the register-blocked 3 x 3 kernel
    assert form(5, (2, 8, 6, 9, 11), (8, 2, 3, 3, 3), 1, 1, 1, 4) == 2
    assert form(5, (1, 6, 9, 8, 10), (6, 1, 3, 3, 3), (2, 1, 1), 1, 1, 6) == 2
    assert form(5, (1, 4, 9, 8, 10), (4, 1, 4, 3, 3), 1, 1, 1, 4) == 2
    assert form(5, (1, 4, 9, 8, 10), (12, 1, 3, 3, 3), 1, 1, 1, 4) == 2
    # a 5-tap x extent or dilation 2 along x -> the general kernel
    assert form(5, (1, 6, 7, 9, 17), (12, 1, 3, 3, 5), (1, 2, 2), (1, 0, 2), 1, 6) == 0
    assert form(5, (2, 4, 8, 6, 11), (4, 2, 2, 3, 3), 1, (0, 1, 2), (1, 1, 2), 2) == 0
    assert form(0, (1, 9, 5, 6, 23), (9, 3, 1, 3, 7), (2, 1, 2), (0, 1, 3), (1, 2, 2), 3) == 0
    assert tc.plan_describe(5, (2, 5, 9, 10, 12), (7, 5, 3, 3, 3), 1, 1)["direct_form"] == -1
    # the NCDHW streaming and tiled grids put (n, channel) in grid z: above
    # 65535 pairs -> the general kernel (persistent, no such limit)
    assert form(0, (1023, 64, 3, 4, 4), (64, 1, 3, 3, 3), 1, 1, 1, 64) == 4
    assert form(0, (1024, 64, 3, 4, 4), (64, 1, 3, 3, 3), 1, 1, 1, 64) == 0


def test_ndhwc_transpose_route_limits(lib):
    """The channels-last route through two layout transposes puts the batch
    in the transpose grid's y dimension: a batch above 65535 is rejected on
    the host.  The engine's channels-last mode has no such limit."""
    with pytest.raises(tc.Tc3dError) as e:
        tc.workspace_bytes(5, (70000, 16, 4, 4, 4), (16, 8, 3, 3, 3), 1, 1, 1, 0, 2)
    assert e.value.status == tc.TC3D_ERR_UNSUPPORTED
    assert tc.plan_describe(5, (70000, 5, 4, 4, 4), (7, 5, 3, 3, 3), 1, 1)["cl"] == 1
    assert tc.workspace_bytes(5, (70000, 5, 4, 4, 4), (7, 5, 3, 3, 3), 1, 1) > 0
    # the direct kernel (few channels per group) has no such limit
    assert tc.workspace_bytes(5, (70000, 8, 4, 4, 4), (8, 1, 3, 3, 3), 1, 1, 1, 0, 8) == 256


def test_ndhwc_argument_errors(lib):
    fn = lib.tc3d_conv3d_fwd_ndhwc
    P = ctypes.c_void_p
    ok = (P(256), P(512), None, P(1024))
    assert _call(lib, fn, (None, P(512), None, P(1024)), _geom()) == tc.TC3D_ERR_NULL
    assert _call(lib, fn, ok, _geom(N=0)) == tc.TC3D_ERR_SHAPE
    assert _call(lib, fn, ok, _geom(Cin=3, G=2)) == tc.TC3D_ERR_GROUPS
    assert _call(lib, fn, ok, _geom(Cin=4, Cout=6, G=2), ws=0) == tc.TC3D_ERR_WORKSPACE


def test_workspace_bytes(lib):
    for op in range(6):
        n = tc.workspace_bytes(op, (2, 4, 9, 9, 9), (4, 4, 3, 3, 3), 2 if op % 2 else 1, 1)
        assert n >= 256 and n % 256 == 0


# --------------------------------------------------------------------------
# parity classes and tap tables of the plan, against brute force and the pages
# --------------------------------------------------------------------------
def _axis_tables(s, p, d, k):
    plan = tc.plan_describe(1, (1, 1, 8, 1, 1), (1, 1, k, 1, 1), (s, 1, 1), (p, 0, 0),
                            (d, 1, 1), 0, 1)
    assert plan["status"] == 0
    return plan, plan["axes"][0]


@pytest.mark.parametrize("s,p,d,k", list(itertools.product(range(1, 5), range(0, 4),
                                                           range(1, 5), range(1, 5))))
def test_parity_tables_brute_force(lib, s, p, d, k):
    plan, ax = _axis_tables(s, p, d, k)
    u = ax["u"]
    # brute force: class r, tap kk contributes iff s | (r + p - d kk); offset (r+p-d kk)/s
    expect = {}
    for r in range(s):
        taps = {}
        for kk in range(k):
            t = r + p - d * kk
            if t % s == 0:
                taps[t // s] = kk
        if taps:
            expect[r] = taps
    assert ax["classes"] == sorted(expect)
    assert sorted(u) == sorted({uu for t in expect.values() for uu in t})
    for ri, r in enumerate(ax["classes"]):
        got = {u[t]: kk for t, kk in enumerate(ax["kidx"][ri]) if kk >= 0}
        assert got == expect[r]
    assert plan["nEmpty"] == s - len(expect)


def _golden_pairs(name):
    rows = {}
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "total_pairs":
            continue
        rows[int(f[0])] = set() if f[1] == "none" else {tuple(int(v) for v in t.split(","))
                                                         for t in f[1:]}
    return rows


@pytest.mark.parametrize("name,L,s,p,d", [("convT_taps_s2p1d2k3_L16.txt", 16, 2, 1, 2),
                                          ("convT_taps_s2p1d1k3_L32.txt", 32, 2, 1, 1)])
def test_parity_tables_match_pages(lib, name, L, s, p, d):
    plan, ax = _axis_tables(s, p, d, 3)
    u = ax["u"]
    for z, pairs in _golden_pairs(name).items():
        m, r = divmod(z, s)
        got = set()
        if r in ax["classes"]:
            ri = ax["classes"].index(r)
            for t, kk in enumerate(ax["kidx"][ri]):
                if kk >= 0 and 0 <= m + u[t] < L:
                    got.add((m + u[t], kk))
        assert got == pairs, (z, got, pairs)


def test_plans_of_workloads(lib):
    """Structural facts of the five workloads' plans."""
    from transposed_conv_epilogues_gb300.workloads import BY_NAME
    ops = {"conv3d": 0, "conv_transpose3d": 1, "conv_maxpool_lse_relu": 2, "convT_bn_avgpool": 3,
           "convT_bneval_avgpool": 4, "conv3d_ndhwc": 5}

    def plan(n):
        wl = BY_NAME[n]
        return tc.plan_describe(ops[wl.op], wl.x_shape, wl.w_shape, wl.stride, wl.padding,
                                wl.dilation, wl.output_padding, wl.groups)

    c3 = plan("convT_s2p1d2")  # only the all-odd class has taps: 1 of 8, 27 taps
    assert c3["nR"] == 1 and c3["nEmpty"] == 7 and c3["M"] == [16, 32, 32]
    assert all(ax["classes"] == [1] and sorted(ax["kidx"][0]) == [0, 1, 2] for ax in c3["axes"])
    # the engine writes the rows of the odd (z, y) pair; the bias fill the others
    assert c3["fill_slab"] == 1 and c3["fill_rows"] == 1
    c4 = plan("convT_bn_avgpool")
    assert c4["fused"] == 1 and c4["nR"] == 8 and c4["M"] == [32, 32, 32]
    assert c4["fill_rows"] == 0
    c5 = plan("conv_maxpool_lse_relu")
    assert c5["Q"] == [2, 2, 8] and c5["n_tile"] == 64
    for n in BY_NAME:
        pl = plan(n)
        assert pl["status"] == 0 and pl["smem_bytes"] <= 227 * 1024
    # grouped / channels-last workloads: depthwise in the direct kernel, the
    # dense channels-last conv through the engine
    assert plan("dwconv_k3")["direct"] == 1 and plan("dwconv_k3_ndhwc")["direct"] == 1
    assert plan("conv_k3_ndhwc")["direct"] == 0 and plan("conv_k3_ndhwc")["ndhwc"] == 1
    k3 = plan("conv_k3_ndhwc")
    assert k3["cl"] == 1 and k3["cin_chunk"] == 16 and k3["cl_cb"] == 20


@pytest.mark.parametrize("s, d, want", [
    ((2, 2, 2), (2, 2, 2), 1),   # one class with taps, stride 2 along x, 4 row pairs
    ((1, 2, 2), (1, 2, 2), 1),   # 2 row pairs (y only)
    ((2, 1, 2), (2, 1, 2), 1),   # 2 row pairs (z only)
    ((1, 1, 2), (1, 1, 2), 0),   # one row pair: the engine writes every row
    ((2, 2, 1), (2, 2, 1), 0),   # stride 1 along x: the general one-class store
    ((2, 2, 2), (1, 1, 1), 0),   # every class has taps
    ((1, 4, 2), (1, 4, 2), 1),   # y stride 4: rows y % 4 != r1 filled in row mode
    ((3, 1, 2), (3, 1, 2), 1),   # z stride 3: whole planes z % 3 != r0
    ((4, 1, 2), (4, 1, 2), 1),   # z stride 4
    ((2, 3, 2), (2, 3, 2), 0),   # 12 classes: above the one-class store's 8
])
def test_fill_rows_plan(lib, s, d, want):
    """Row mode of the bias fill: exactly when the engine stores through the
    one-class stride-2-along-x path with more than one (z, y) class pair."""
    pl = tc.plan_describe(1, (1, 3, 4, 5, 6), (3, 4, 3, 3, 3), s, 1, d)
    assert pl["status"] == 0 and pl["fill_rows"] == want
    if want:
        assert pl["fill_slab"] == 1 and pl["nR"] == 1


@pytest.mark.parametrize("cin", [3, 8, 12, 16, 32, 40])
@pytest.mark.parametrize("xext", [16, 64])
def test_channels_last_chunks(lib, cin, xext):
    """The engine's channels-last mode: a raw box of cl_cb = cin_chunk + 4
    channels per position (cl_cb / 4 odd: 16-byte loads of consecutive
    positions start in distinct bank groups), GEMM-K tap-major in chunks of
    8, 16, 24 or 32 channels, the fewest K-steps over all chunks among those
    whose raw stage fits (at most 96 KB)."""
    pl = tc.plan_describe(5, (2, cin, 6, 8, xext), (16, cin, 3, 3, 3), 1, 1)
    assert pl["status"] == 0 and pl["cl"] == 1 and pl["view"] == 0
    cc = pl["cin_chunk"]
    assert cc in (8, 16, 24, 32) and pl["cl_cb"] == cc + 4 and (pl["cl_cb"] // 4) % 2 == 1
    assert pl["ksteps_chunk"] == (cc // 8) * 27 and pl["n_chunks"] == -(-cin // cc)
    assert pl["smem_bytes"] <= 227 * 1024
    bvol = pl["box"][0] * pl["box"][1] * pl["box"][2]
    assert pl["raw_stage_bytes"] >= bvol * pl["cl_cb"] * 4
    steps = pl["n_chunks"] * pl["ksteps_chunk"]
    for c2 in (8, 16, 24, 32):
        if c2 <= -(-cin // 8) * 8 and bvol * (c2 + 4) * 4 <= 96 * 1024:
            assert steps <= -(-cin // c2) * (c2 // 8) * 27
    # the box has no x slack: channels, not x, are the innermost axis
    assert pl["box"][2] == pl["T"][2] + 2
    # transposed convs keep the NCDHW planning
    assert tc.plan_describe(3, (2, cin, 6, 8, xext), (cin, 16, 3, 3, 3), 2, 1)["cl"] == 0


def test_channels_last_tile_search(lib):
    """A strided channels-last conv whose NCDHW-planned tile (x-long) gives a
    box over the channels-last stage budget gets a tile of its own search:
    the mode still applies, every raw stage fits in 96 KB and the plan's
    shared memory in 227 KB; the tile covers the rows."""
    xs, ws = (1, 32, 5, 6, 40), (64, 32, 3, 3, 3)
    s, p, d = (1, 2, 2), (1, 0, 1), (2, 1, 1)
    ncdhw = tc.plan_describe(0, xs, ws, s, p, d)
    pl = tc.plan_describe(5, xs, ws, s, p, d)
    assert pl["status"] == 0 and pl["cl"] == 1
    assert pl["T"] != ncdhw["T"]
    bvol = pl["box"][0] * pl["box"][1] * pl["box"][2]
    assert bvol * pl["cl_cb"] * 4 <= 96 * 1024 and pl["smem_bytes"] <= 227 * 1024
    for a in range(3):
        st = s[a]
        span = d[a] * (ws[2 + a] - 1)
        assert pl["box"][a] == st * (pl["T"][a] - 1) + span + 1
    assert pl["tiles"] == 1 * np.prod([-(-pl["M"][a] // pl["T"][a]) for a in range(3)])
