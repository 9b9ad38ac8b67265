"""GPU parity tests: the CUDA path (through the C ABI) against the fp64 oracle.

Bar: |gpu - oracle| <= 1e-4 + 1e-4 * |oracle| for every compared element
(3xTF32 products accumulated in fp32; the tolerance is the one the workloads
are specified with), and exact integer shapes.  Small cases compare every
output; the full-size workloads compare sampled outputs that the oracle
evaluates one by one.
"""
import numpy as np
import pytest

import oracle as orc
from transposed_conv_epilogues_gb300 import inputs
from transposed_conv_epilogues_gb300.workloads import BY_NAME

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


def check(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argmax(np.where(bad, err - bound, -np.inf))
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at "
                             f"{np.unravel_index(i, ref.shape)}: gpu {gpu.flat[i]!r} "
                             f"oracle {ref.flat[i]!r}")


def make(xs, ws, cout, bias=True, seed=7, xdist="normal"):
    x = (inputs.normal(seed, xs) if xdist == "normal"
         else inputs.uniform(seed, xs, 0.0, 1.0))
    fan = int(np.prod(ws[1:]))
    bound = 1.0 / np.sqrt(fan)
    w = inputs.uniform(seed + 1, ws, -bound, bound)
    b = inputs.uniform(seed + 2, (cout,), -bound, bound) if bias else None
    return x, w, b


# --------------------------------------------------------------------------
# small cases: every output compared
# --------------------------------------------------------------------------
CONV_CASES = [
    # x shape, w shape, stride, pad, dil, groups, bias
    ((2, 5, 9, 10, 12), (7, 5, 3, 3, 3), 1, 1, 1, 1, True),
    ((2, 4, 11, 9, 13), (6, 2, 3, 2, 3), (2, 1, 2), (1, 0, 2), (1, 2, 1), 2, True),
    ((2, 3, 11, 9, 5), (4, 3, 3, 3, 1), 1, 1, 1, 1, True),         # (k,k,1), pad on k=1 axis
    ((1, 6, 7, 8, 9), (40, 6, 1, 1, 1), 1, 0, 1, 1, False),          # k = 1
    ((1, 4, 6, 6, 8), (200, 4, 3, 1, 3), 1, (1, 0, 1), 1, 1, True),  # 2 column blocks
    ((2, 8, 7, 9, 8), (8, 2, 3, 3, 3), 1, 1, 1, 4, True),            # groups 4 (direct kernel)
    ((2, 8, 7, 9, 8), (12, 4, 3, 3, 3), 1, 1, 1, 2, True),           # groups 2, 4x6 per group: engine
    ((1, 3, 13, 12, 16), (5, 3, 5, 3, 5), (1, 2, 1), 2, 2, 1, True),  # k5 dil 2
    ((3, 17, 6, 5, 20), (9, 17, 2, 3, 2), 1, 0, 1, 1, True),         # Cin 17: 2 chunks
    # view mode: one tap along x, x lines filling 128-row accumulators
    ((2, 8, 7, 9, 8), (5, 8, 3, 3, 1), 1, (1, 1, 0), 1, 1, True),
    ((1, 8, 9, 10, 16), (8, 8, 3, 3, 1), 1, (2, 0, 0), (2, 1, 1), 1, True),
    ((1, 16, 4, 5, 32), (20, 16, 2, 2, 1), 1, 0, 1, 1, False),
    ((2, 8, 6, 20, 4), (4, 8, 1, 3, 1), 1, (0, 1, 0), 1, 1, True),
    ((1, 40, 6, 6, 8), (16, 40, 3, 3, 1), 1, (1, 1, 0), 1, 1, True),  # 5 channel chunks
    ((1, 24, 5, 7, 8), (130, 24, 3, 3, 1), 1, 1, 1, 1, True),         # 2 column blocks: gather path
    # merged (S1*S2) form of (k,k,1) convs: line segments, channels padded to octets
    ((2, 3, 11, 9, 5), (4, 3, 3, 3, 1), 1, (1, 1, 0), 1, 1, True),    # Cin 3, shifted windows
    ((2, 3, 12, 14, 10), (6, 3, 3, 3, 1), 1, 0, 1, 1, True),          # x extent 10
    ((1, 5, 7, 30, 6), (7, 5, 3, 5, 1), 1, (1, 4, 0), (1, 2, 1), 1, True),  # dilation along y
]


@pytest.mark.parametrize("case", CONV_CASES)
def test_conv3d_small(tc, case):
    xs, ws, s, p, d, G, bias = case
    x, w, b = make(xs, ws, ws[0], bias)
    y = tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), s, p, d, G).cpu().numpy()
    check(y, orc.conv3d(x, w, b, s, p, d, G), f"conv3d {case}")


CONVT_CASES = [
    # x shape, w shape, stride, pad, dil, output_padding, groups, bias
    ((2, 6, 5, 7, 8), (6, 10, 3, 3, 3), 2, 1, 2, 0, 1, False),
    ((2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 2, 1, 1, 0, 1, True),
    ((2, 4, 5, 6, 7), (4, 3, 3, 2, 4), (3, 2, 1), (1, 0, 2), (1, 2, 1), (2, 1, 0), 2, True),
    ((1, 5, 6, 7, 8), (5, 6, 3, 3, 3), 1, 1, 1, 0, 1, True),
    ((2, 3, 3, 4, 4), (3, 5, 2, 2, 2), 4, 0, 1, (3, 0, 2), 1, True),  # many empty classes
    ((1, 2, 4, 5, 6), (2, 3, 1, 3, 2), (2, 3, 2), (0, 1, 1), (1, 1, 2), (1, 2, 0), 1, True),
    # one parity class with taps, stride 2 along x: the dense pair-store path
    ((1, 4, 3, 5, 20), (4, 6, 3, 3, 3), 2, 1, 2, (1, 0, 1), 1, True),
    ((2, 3, 4, 6, 9), (3, 5, 3, 3, 3), (1, 2, 2), 1, (1, 2, 2), 0, 1, True),
    ((1, 4, 5, 4, 11), (4, 3, 3, 3, 3), (2, 1, 2), 1, (2, 1, 2), 0, 2, True),
    ((1, 3, 2, 3, 40), (3, 40, 3, 3, 3), 2, 1, 2, 0, 1, True),
    # one parity class with taps, stride 1 along x
    ((1, 3, 4, 5, 6), (3, 4, 3, 3, 3), (2, 2, 1), 1, (2, 2, 1), 0, 1, True),
    # no engine tiles (the only class with taps lies past the output): every
    # output is the bias, written by the stand-alone fill
    ((2, 3, 2, 2, 2), (3, 4, 1, 1, 1), 2, 1, 1, 0, 1, True),
    ((2, 3, 2, 5, 6), (3, 4, 1, 3, 3), 2, (1, 1, 0), 1, 0, 1, True),
    # row mode of the fill with other strides: y stride 4 (rows y % 4 != r1
    # filled a warp per row for long rows, a lane per row for short ones),
    # and y stride 1 with z stride 3 or 4 (whole planes z % s0 != r0)
    ((1, 3, 4, 5, 20), (3, 4, 3, 3, 3), (1, 4, 2), 1, (1, 4, 2), 0, 1, True),
    ((2, 3, 3, 4, 6), (3, 5, 3, 3, 3), (1, 4, 2), 1, (1, 4, 2), (0, 3, 1), 1, True),
    ((1, 2, 3, 4, 18), (2, 4, 3, 3, 3), (3, 1, 2), (1, 0, 1), (3, 1, 2), 0, 1, True),
    ((2, 4, 3, 5, 7), (4, 6, 2, 2, 2), (4, 1, 2), (1, 1, 1), (4, 1, 2), (2, 0, 1), 1, False),
    # the bias fill inside the engine over many slices and planes (units
    # taken from the shared counter by every CTA), with and without bias
    ((3, 8, 9, 10, 12), (8, 24, 3, 3, 3), 2, 1, 2, 0, 1, True),
    ((3, 8, 9, 10, 12), (8, 24, 3, 3, 3), 2, 1, 2, (1, 1, 1), 1, False),
]


@pytest.mark.parametrize("case", CONVT_CASES)
def test_conv_transpose3d_small(tc, case):
    xs, ws, s, p, d, op, G, bias = case
    x, w, b = make(xs, ws, ws[1] * G, bias)
    y = tc.conv_transpose3d_fwd(_dev(x), _dev(w), _dev(b), s, p, d, op, G).cpu().numpy()
    check(y, orc.conv_transpose3d(x, w, b, s, p, d, op, G), f"convT {case}")


LSE_CASES = [
    ((2, 5, 8, 10, 16), (12, 5, 3, 3, 3), 1, 1, 1, 1),
    ((1, 4, 9, 11, 13), (40, 2, 3, 3, 3), 1, 1, 1, 2),     # groups: running LSE across blocks
    ((2, 3, 13, 12, 18), (6, 3, 3, 3, 3), (2, 1, 2), 1, 1, 1),  # stride, odd extents
    ((1, 2, 6, 6, 8), (300, 2, 3, 3, 3), 1, 1, 1, 1),       # Cout 300: two column blocks
    ((1, 4, 7, 9, 10), (8, 4, 3, 3, 1), 1, (1, 1, 0), (1, 2, 1), 1),
]


@pytest.mark.parametrize("case", LSE_CASES)
def test_conv_maxpool_lse_relu_small(tc, case):
    xs, ws, s, p, d, G = case
    x, w, b = make(xs, ws, ws[0], True)
    b = b - 0.3  # push some LSE values below zero so the ReLU matters
    y = tc.conv_maxpool_lse_relu(_dev(x), _dev(w), _dev(b), s, p, d, G).cpu().numpy()
    check(y, orc.conv_maxpool_lse_relu(x, w, b, s, p, d, G), f"pool-lse {case}")


BN_CASES = [
    # x shape, w shape, stride, pad, dil, output_padding, groups, gamma/beta
    ((2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 2, 1, 1, 0, 1, False),        # lag form (the workload's form)
    ((2, 7, 9, 8, 10), (7, 5, 3, 3, 3), 2, 1, 1, (0, 1, 1), 1, True),  # fused, ragged
    ((2, 4, 6, 7, 8), (4, 3, 3, 3, 3), 2, 1, 1, 0, 2, True),          # fused, groups
    ((1, 5, 10, 12, 9), (5, 40, 3, 3, 3), 2, 1, 1, (1, 0, 1), 1, True),  # fused, 3 column blocks
    ((4, 3, 24, 24, 24), (3, 16, 3, 3, 3), 2, 1, 1, 0, 1, False),     # lag form, many pooled items
    ((4, 5, 24, 24, 24), (5, 16, 3, 3, 3), 2, 1, 1, 0, 1, True),     # fused, 5 channels, many tiles
    # the algebraic path (patch Gram or lag-form statistics + summed-weight
    # pooled conv): batch statistics where the fused epilogue cannot run (one
    # parity class per axis); running statistics always (the eval test reuses
    # these)
    ((2, 3, 8, 7, 9), (3, 4, 1, 1, 1), 2, 0, 1, (1, 0, 1), 1, True),  # k 1
    ((2, 4, 7, 8, 6), (4, 5, 2, 2, 2), 2, 0, 2, 1, 1, True),          # k 2, dilation 2
    ((3, 1, 20, 22, 24), (1, 6, 1, 1, 1), 2, 0, 1, 1, 1, False),      # k 1, lag form
    ((2, 2, 9, 7, 10), (2, 4, 3, 3, 3), 2, 0, 1, 0, 1, True),         # pad 0
    ((1, 4, 5, 6, 7), (4, 3, 3, 3, 3), 2, 1, 1, (1, 0, 1), 1, True),  # 32-entry patch
    ((2, 1, 9, 8, 7), (1, 4, 2, 3, 5), 2, (0, 1, 2), (1, 1, 3), 1, 1, True),  # widened pad
    ((3, 2, 6, 5, 9), (2, 3, 2, 4, 3), 2, (0, 1, 1), 1, (1, 0, 0), 1, False),
    ((2, 3, 9, 5, 6), (3, 4, 3, 3, 3), (1, 2, 2), 1, 1, 0, 1, True),  # unfused: stride 1 axis
    ((2, 3, 6, 6, 6), (3, 4, 3, 3, 3), 2, 1, 2, 0, 1, True),          # unfused: dilation 2
    # batch statistics in lag form (at most 3 channels, one or two consecutive
    # offsets per axis, axis-2 rows a multiple of 4 floats) + the pooled conv
    # on CUDA cores; the workload's form is the first BN case above
    ((2, 2, 9, 7, 12), (2, 4, 3, 3, 3), 2, 0, 1, 0, 1, True),         # offsets {-1, 0}
    ((1, 3, 5, 6, 36), (3, 3, 3, 3, 3), 2, 1, 1, (1, 0, 1), 1, True),  # two column blocks
    ((2, 1, 9, 10, 8), (1, 4, 2, 3, 1), 2, (0, 1, 0), 1, (1, 1, 1), 1, True),  # one offset on x
    ((3, 2, 6, 17, 4), (2, 3, 3, 2, 3), 2, (1, 0, 1), 1, 0, 1, False),  # ragged row block
    ((5, 3, 12, 40, 16), (3, 24, 3, 3, 3), 2, 1, 1, 0, 1, True),      # 24 channels, 5 row blocks
]


@pytest.mark.parametrize("case", BN_CASES)
def test_convT_bn_avgpool_small(tc, case):
    xs, ws, s, p, d, op, G, affine = case
    cout = ws[1] * G
    x, w, b = make(xs, ws, cout, True)
    g = inputs.uniform(99, (cout,), 0.5, 1.5) if affine else None
    be = inputs.uniform(98, (cout,), -0.5, 0.5) if affine else None
    y = tc.convT_bn_avgpool(_dev(x), _dev(w), _dev(b), _dev(g), _dev(be), 1e-5, s, p, d, op,
                            G).cpu().numpy()
    check(y, orc.convT_bn_avgpool(x, w, b, g, be, 1e-5, s, p, d, op, G), f"bn-pool {case}")


def _running_stats(cout, seed):
    # running statistics of the scale the BN input has (|t| ~ 0.5): means
    # around 0, variances in [0.05, 0.5] so the normalisation amplifies
    rm = 0.2 * inputs.normal(seed, (cout,))
    rv = inputs.uniform(seed + 1, (cout,), 0.05, 0.5)
    return rm, rv


@pytest.mark.parametrize("case", BN_CASES)
def test_convT_bneval_avgpool_small(tc, case):
    """Evaluation-mode BatchNorm (running statistics): the fused cases store
    final values from the engine, the others pool the workspace output."""
    xs, ws, s, p, d, op, G, affine = case
    cout = ws[1] * G
    x, w, b = make(xs, ws, cout, True, seed=13)
    rm, rv = _running_stats(cout, 77)
    g = inputs.uniform(99, (cout,), 0.5, 1.5) if affine else None
    be = inputs.uniform(98, (cout,), -0.5, 0.5) if affine else None
    y = tc.convT_bneval_avgpool(_dev(x), _dev(w), _dev(b), _dev(rm), _dev(rv), _dev(g), _dev(be),
                                1e-5, s, p, d, op, G).cpu().numpy()
    check(y, orc.convT_bneval_avgpool(x, w, b, rm, rv, g, be, 1e-5, s, p, d, op, G),
          f"bn-eval-pool {case}")


def test_convT_bn_avgpool_gram_path_many_units(tc):
    """Batch statistics from patch Gram matrices at a size with many work
    units per box (a one-class-per-axis transposed conv: k 2, dilation 2,
    a 32-entry patch), every output against the oracle."""
    x, w, b = make((8, 4, 32, 32, 32), (4, 8, 2, 2, 2), 8, True, seed=61)
    assert tc.plan_describe(3, x.shape, w.shape, 2, 0, 2)["pool_path"] == 1
    g = inputs.uniform(62, (8,), 0.5, 1.5)
    be = inputs.uniform(63, (8,), -0.5, 0.5)
    y = tc.convT_bn_avgpool(_dev(x), _dev(w), _dev(b), _dev(g), _dev(be), 1e-5, 2, 0, 2)
    check(y.cpu().numpy(), orc.convT_bn_avgpool(x, w, b, g, be, 1e-5, 2, 0, 2), "gram path")


def test_convT_bneval_matches_train_with_batch_stats(tc):
    """With the batch moments passed as running statistics, evaluation mode
    gives the training-mode result (both against the oracle, and each other)."""
    x, w, b = make((2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 16, True, seed=21)
    full = orc.conv_transpose3d(x, w, b, 2, 1)
    # float32, as the library takes them (rounding moves the result ~1e-7)
    rm = full.mean(axis=(0, 2, 3, 4)).astype(np.float32)
    rv = full.var(axis=(0, 2, 3, 4)).astype(np.float32)
    ev = tc.convT_bneval_avgpool(_dev(x), _dev(w), _dev(b), _dev(rm), _dev(rv), None, None,
                                 1e-5, 2, 1).cpu().numpy()
    tr = tc.convT_bn_avgpool(_dev(x), _dev(w), _dev(b), None, None, 1e-5, 2, 1).cpu().numpy()
    ref = orc.convT_bn_avgpool(x, w, b, None, None, 1e-5, 2, 1)
    check(ev, ref, "eval with batch stats")
    check(tr, ref, "train")


def test_convT_bneval_rejects_missing_stats(tc):
    x, w, b = make((1, 3, 6, 6, 6), (3, 4, 3, 3, 3), 4)
    with pytest.raises(ValueError):
        tc.convT_bneval_avgpool(_dev(x), _dev(w), _dev(b), None, None, stride=2, padding=1)
    rm, rv = _running_stats(4, 5)
    with pytest.raises(ValueError):  # wrong length: checked before the C call
        tc.convT_bneval_avgpool(_dev(x), _dev(w), _dev(b), _dev(rm[:3]), _dev(rv), stride=2,
                                padding=1)


def test_uniform01_inputs(tc):
    """torch.rand-style inputs (all positive) as on the pages."""
    x, w, b = make((2, 6, 9, 8, 12), (8, 6, 3, 3, 3), 8, True, seed=31, xdist="uniform01")
    check(tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), 1, 1).cpu().numpy(),
          orc.conv3d(x, w, b, 1, 1), "conv uniform01")
    xt, wt, bt = make((2, 3, 6, 6, 6), (3, 16, 3, 3, 3), 16, True, seed=41, xdist="uniform01")
    check(tc.convT_bn_avgpool(_dev(xt), _dev(wt), _dev(bt), None, None, 1e-5, 2, 1)
          .cpu().numpy(), orc.convT_bn_avgpool(xt, wt, bt, None, None, 1e-5, 2, 1),
          "bn-pool uniform01")


# --------------------------------------------------------------------------
# grouped / depthwise convs in the direct kernel, and channels-last layout
# --------------------------------------------------------------------------
DIRECT_CASES = [
    # x shape, w shape, stride, pad, dil, groups
    ((2, 8, 9, 10, 13), (8, 1, 3, 3, 3), 1, 1, 1, 8),                  # depthwise k3
    ((1, 6, 7, 9, 17), (12, 1, 3, 3, 5), (1, 2, 2), (1, 0, 2), 1, 6),   # depthwise x2, stride 2 on x
    ((2, 4, 8, 6, 11), (4, 2, 2, 3, 3), 1, (0, 1, 2), (1, 1, 2), 2),    # dilation 2 on x
    ((1, 9, 5, 6, 23), (9, 3, 1, 3, 7), (2, 1, 2), (0, 1, 3), (1, 2, 2), 3),  # 7 taps, s2 d2
    ((3, 4, 4, 5, 6), (8, 1, 3, 1, 2), 1, 1, 1, 4),                    # ragged, k2 = 2
    # the NCDHW streaming form (3 x 3 x 3), 4-byte copies: several y / x
    # tiles and output-plane chunks
    ((2, 4, 9, 40, 70), (4, 1, 3, 3, 3), 1, 1, 1, 4),
    # the shared-memory tiled form (one input channel per group): a 3x3 filter
    # plane unrolled with k0 = 1 and stride 2 along x (a channel multiplier
    # of 2) and with k0 = 2; a 5 x 2 plane at dilation 2 along x
    ((1, 3, 7, 35, 133), (6, 1, 1, 3, 3), (1, 1, 2), (0, 1, 1), 1, 3),
    ((2, 4, 9, 40, 70), (4, 1, 2, 3, 3), 1, 1, 1, 4),
    ((2, 2, 6, 33, 66), (2, 1, 3, 5, 2), 1, (1, 2, 0), (1, 1, 2), 2),
    # the NCDHW streaming form with 16-byte copies (rows a multiple of 4
    # floats), the window starting 2, 0 and 1 columns into its first piece;
    # stride 2 along x with a channel multiplier of 2; several x and y tiles
    ((1, 3, 7, 37, 136), (6, 1, 3, 3, 3), (1, 1, 2), (1, 1, 2), 1, 3),
    ((1, 4, 6, 34, 68), (4, 1, 3, 3, 3), 1, (0, 1, 0), 1, 4),
    ((2, 2, 5, 9, 72), (2, 1, 3, 3, 3), 1, (2, 1, 3), 1, 2),
]


@pytest.mark.parametrize("case", DIRECT_CASES)
def test_direct_grouped_conv(tc, case):
    xs, ws, s, p, d, G = case
    x, w, b = make(xs, ws, ws[0], True, seed=71)
    assert tc.plan_describe(0, xs, ws, s, p, d, 0, G)["direct"] == 1
    y = tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), s, p, d, G).cpu().numpy()
    check(y, orc.conv3d(x, w, b, s, p, d, G), f"direct {case}")


NDHWC_CASES = DIRECT_CASES[:3] + DIRECT_CASES[5:6] + [
    ((1, 3, 7, 35, 133), (6, 1, 2, 3, 3), (1, 1, 2), (0, 1, 1), 1, 3),
    ((2, 3, 11, 9, 5), (4, 3, 3, 3, 1), 1, (1, 1, 0), 1, 1),           # (k,k,1), direct
    # not for the direct kernel: the engine's channels-last mode (5 channels,
    # not a multiple of 4: plain loads of the box instead of TMA)
    ((2, 5, 9, 10, 12), (7, 5, 3, 3, 3), 1, 1, 1, 1),
    # channels-last mode through TMA: a ragged output-channel chunk (24),
    # strides and dilation 2 (4 chunks of 8 channels), channels past Cin
    # zero-filled by the load (12 in a 16-channel chunk), a ragged last chunk
    # (40 = 5 x 8)
    ((2, 16, 7, 9, 20), (24, 16, 3, 3, 3), 1, 1, 1, 1),
    ((2, 32, 5, 9, 14), (64, 32, 3, 3, 3), (2, 1, 2), 1, (1, 2, 1), 1),
    ((2, 12, 6, 5, 9), (20, 12, 2, 3, 1), 1, (0, 1, 0), 1, 1),
    ((1, 40, 4, 7, 12), (8, 40, 3, 1, 3), 1, 1, 1, 1),
    # grouped, 4 x 6 channels per group: through the engine with layout
    # transposes
    ((1, 8, 6, 7, 9), (12, 4, 3, 2, 3), (1, 2, 1), 1, 1, 2),
    # the streaming form: ragged 32-channel blocks with a multiplier of 2,
    # pad 2 along z and stride 2 along x; k0 = 1; a multiplier of 16 and a
    # channel count that is not a multiple of 4 (4-byte copies); several
    # output-plane chunks of 9 planes (9, 9, 7)
    ((1, 40, 5, 9, 18), (80, 1, 3, 3, 3), (1, 1, 2), (2, 1, 1), 1, 40),
    ((2, 36, 6, 7, 9), (36, 1, 1, 3, 3), 1, (0, 1, 0), 1, 36),
    ((1, 6, 11, 5, 6), (96, 1, 3, 3, 3), 1, 1, 1, 6),
    ((2, 6, 8, 21, 19), (6, 1, 3, 3, 3), 1, 1, 1, 6),
    ((2, 64, 25, 40, 64), (64, 1, 3, 3, 3), 1, 1, 1, 64),
    # the register-blocked 3 x 3 kernel: two input channels per group, and
    # stride 2 along z
    ((2, 8, 6, 9, 11), (8, 2, 3, 3, 3), 1, 1, 1, 4),
    ((1, 6, 9, 8, 10), (6, 1, 3, 3, 3), (2, 1, 1), 1, 1, 6),
]


@pytest.mark.parametrize("case", NDHWC_CASES)
def test_conv3d_ndhwc(tc, case):
    xs, ws, s, p, d, G = case
    x, w, b = make(xs, ws, ws[0], True, seed=72)
    x_cl = np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1))
    y = tc.conv3d_fwd_ndhwc(_dev(x_cl), _dev(w), _dev(b), s, p, d, G).cpu().numpy()
    ref = orc.conv3d(x, w, b, s, p, d, G).transpose(0, 2, 3, 4, 1)
    check(y, ref, f"ndhwc {case}")


def test_conv3d_ndhwc_stream_chunks(tc):
    """The streaming form splits the (2, 64, 25, 40, 64) depthwise conv into
    output-plane chunks of 9, 9 and 7 planes on a 152-SM GB300; each chunk
    walks its planes plus a 2-plane halo."""
    xs, ws = (2, 64, 25, 40, 64), (64, 1, 3, 3, 3)
    assert tc.plan_describe(5, xs, ws, 1, 1, 1, 0, 64)["direct_form"] == 3
    x, w, b = make(xs, ws, 64, True, seed=74)
    x_cl = np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1))
    y = tc.conv3d_fwd_ndhwc(_dev(x_cl), _dev(w), _dev(b), 1, 1, 1, 64).cpu().numpy()
    check(y, orc.conv3d(x, w, b, 1, 1, 1, 64).transpose(0, 2, 3, 4, 1), "ndhwc stream chunks")


def test_direct_stream_misaligned(tc):
    """NCDHW x 4 bytes past a 16-byte boundary: the streaming form copies
    with 4-byte pieces."""
    xs, ws = (2, 4, 6, 9, 64), (4, 1, 3, 3, 3)
    x, w, b = make(xs, ws, 4, True, seed=76)
    buf = torch.zeros(x.size + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(x.ravel()).cuda()
    xv = buf[1:].view(xs)
    assert xv.data_ptr() % 16 != 0
    y = tc.conv3d_fwd(xv, _dev(w), _dev(b), 1, 1, 1, 4).cpu().numpy()
    check(y, orc.conv3d(x, w, b, 1, 1, 1, 4), "direct stream misaligned")


def test_conv3d_ndhwc_stream_misaligned(tc):
    """x 4 bytes past a 16-byte boundary: the streaming form copies with
    4-byte pieces."""
    xs, ws = (2, 32, 7, 9, 20), (32, 1, 3, 3, 3)
    x, w, b = make(xs, ws, 32, True, seed=75)
    x_cl = np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1))
    buf = torch.zeros(x_cl.size + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(x_cl.ravel()).cuda()
    xv = buf[1:].view(x_cl.shape)
    assert xv.data_ptr() % 16 != 0
    y = tc.conv3d_fwd_ndhwc(xv, _dev(w), _dev(b), 1, 1, 1, 32).cpu().numpy()
    check(y, orc.conv3d(x, w, b, 1, 1, 1, 32).transpose(0, 2, 3, 4, 1), "ndhwc stream misaligned")


# --------------------------------------------------------------------------
# edge cases
# --------------------------------------------------------------------------
def test_misaligned_input_uses_plain_loads(tc):
    """x starting 4 bytes past a 16-byte boundary cannot be a TMA source; the
    plain-load producer must give the same result (NCDHW, and the
    channels-last mode's own box layout)."""
    x, w, b = make((2, 4, 6, 7, 8), (5, 4, 3, 3, 3), 5)
    buf = torch.zeros(x.size + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(x.ravel()).cuda()
    xv = buf[1:].view(x.shape)
    assert xv.data_ptr() % 16 != 0
    y = tc.conv3d_fwd(xv, _dev(w), _dev(b), 1, 1).cpu().numpy()
    check(y, orc.conv3d(x, w, b, 1, 1), "misaligned x")
    x, w, b = make((2, 16, 6, 7, 9), (24, 16, 3, 3, 3), 24, seed=75)
    x_cl = np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1))
    assert tc.plan_describe(5, x.shape, w.shape, 1, 1)["cl"] == 1
    buf = torch.zeros(x.size + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(x_cl.ravel()).cuda()
    xv = buf[1:].view(x_cl.shape)
    assert xv.data_ptr() % 16 != 0
    y = tc.conv3d_fwd_ndhwc(xv, _dev(w), _dev(b), 1, 1).cpu().numpy()
    check(y, orc.conv3d(x, w, b, 1, 1).transpose(0, 2, 3, 4, 1), "misaligned channels-last x")


def test_guard_bands_untouched(tc):
    x, w, b = make((2, 6, 5, 7, 8), (6, 10, 3, 3, 3), 10)
    shp = tc.out_shape(1, x.shape, w.shape, 2, 1, 2)
    n = int(np.prod(shp))
    G = 4096
    buf = torch.full((n + 2 * G,), 12345.0, dtype=torch.float32, device="cuda")
    out = buf[G:G + n].view(shp)
    tc.conv_transpose3d_fwd(_dev(x), _dev(w), _dev(b), 2, 1, 2, out=out)
    h = buf.cpu().numpy()
    assert np.all(h[:G] == 12345.0) and np.all(h[G + n:] == 12345.0)
    check(out.cpu().numpy(), orc.conv_transpose3d(x, w, b, 2, 1, 2), "guarded convT")


def test_deterministic_repeat(tc):
    x, w, b = make((2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 16)
    a1 = tc.convT_bn_avgpool(_dev(x), _dev(w), _dev(b), None, None, 1e-5, 2, 1)
    a2 = tc.convT_bn_avgpool(_dev(x), _dev(w), _dev(b), None, None, 1e-5, 2, 1)
    assert torch.equal(a1, a2)
    x, w, b = make((2, 5, 8, 10, 16), (12, 5, 3, 3, 3), 12)
    c1 = tc.conv_maxpool_lse_relu(_dev(x), _dev(w), _dev(b), 1, 1)
    c2 = tc.conv_maxpool_lse_relu(_dev(x), _dev(w), _dev(b), 1, 1)
    assert torch.equal(c1, c2)


def test_fill_stream_does_not_couple_callers(tc):
    """A transposed conv with a bias fill enqueues all its work on the
    caller's stream.  Work another caller queued on another stream must not
    hold it up: stream B sleeps (a bounded spin kernel) before its own
    transposed conv; the call on stream A, queued after it, still completes
    while B sleeps."""
    x, w, b = make((2, 6, 5, 7, 8), (6, 10, 3, 3, 3), 10)   # k3 s2 p1 d2: a bias slab
    xd, wd, bd = _dev(x), _dev(w), _dev(b)
    kw = dict(stride=2, padding=1, dilation=2)
    ref = tc.conv_transpose3d_fwd(xd, wd, bd, **kw)
    assert tc.plan_describe(tc.OP_CONV_TRANSPOSE3D, x.shape, w.shape, 2, 1, 2)["fill_slab"] == 1
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    ya, yb = torch.empty_like(ref), torch.empty_like(ref)
    with torch.cuda.stream(sb):
        torch.cuda._sleep(2_000_000_000)  # about a second at 2 GHz
        tc.conv_transpose3d_fwd(xd, wd, bd, **kw, out=yb)
        done_b = torch.cuda.Event()
        done_b.record(sb)
    with torch.cuda.stream(sa):
        tc.conv_transpose3d_fwd(xd, wd, bd, **kw, out=ya)
        done_a = torch.cuda.Event()
        done_a.record(sa)
    done_a.synchronize()
    b_pending = not done_b.query()
    torch.cuda.synchronize()
    assert b_pending, "stream B finished first: the check could not tell"
    assert torch.equal(ya, ref) and torch.equal(yb, ref)


def test_cuda_graph_capture_replays(tc):
    """Every entry point enqueues only stream-ordered work on the caller's
    stream (the transposed conv's bias fill runs inside the engine).  So a
    call can be captured into a CUDA graph and replayed, giving the same bits
    as a direct call."""
    calls = []
    x, w, b = make((2, 8, 7, 9, 8), (5, 8, 3, 3, 1), 5)                 # conv, view mode
    calls.append((tc.OP_CONV3D, (_dev(x), _dev(w), _dev(b)), dict(stride=1, padding=(1, 1, 0))))
    x, w, b = make((2, 6, 5, 7, 8), (6, 10, 3, 3, 3), 10)               # convT with a bias slab
    calls.append((tc.OP_CONV_TRANSPOSE3D, (_dev(x), _dev(w), _dev(b)),
                  dict(stride=2, padding=1, dilation=2)))
    x, w, b = make((2, 5, 8, 10, 16), (12, 5, 3, 3, 3), 12)
    calls.append((tc.OP_CONV_MAXPOOL_LSE_RELU, (_dev(x), _dev(w), _dev(b)), dict(stride=1, padding=1)))
    x, w, b = make((2, 3, 8, 8, 8), (3, 16, 3, 3, 3), 16)
    calls.append((tc.OP_CONVT_BN_AVGPOOL, (_dev(x), _dev(w), _dev(b)), dict(stride=2, padding=1)))
    rm, rv = _running_stats(16, 3)
    calls.append((tc.OP_CONVT_BNEVAL_AVGPOOL, (_dev(x), _dev(w), _dev(b)),
                  dict(running_mean=_dev(rm), running_var=_dev(rv), stride=2, padding=1)))
    fns = {tc.OP_CONV3D: tc.conv3d_fwd, tc.OP_CONV_TRANSPOSE3D: tc.conv_transpose3d_fwd,
           tc.OP_CONV_MAXPOOL_LSE_RELU: tc.conv_maxpool_lse_relu,
           tc.OP_CONVT_BN_AVGPOOL: tc.convT_bn_avgpool,
           tc.OP_CONVT_BNEVAL_AVGPOOL: tc.convT_bneval_avgpool}
    side = torch.cuda.Stream()
    for op, (xd, wd, bd), kw in calls:
        fn = fns[op]
        ref = fn(xd, wd, bd, **kw)  # direct call (also initialises the device state)
        torch.cuda.synchronize()
        geo = {k: v for k, v in kw.items() if k not in ("running_mean", "running_var")}
        ws = torch.empty(max(tc.workspace_bytes(op, tuple(xd.shape), tuple(wd.shape), **geo),
                             256), dtype=torch.uint8, device="cuda")
        y = torch.full_like(ref, float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                fn(xd, wd, bd, **kw, out=y, workspace=ws)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref), op
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref), op
    assert tc.last_device_error() == tc.TC3D_OK


def test_error_leaves_output_untouched(tc):
    x, w, b = make((1, 4, 6, 6, 8), (4, 4, 3, 3, 3), 4)
    y = torch.full(tc.out_shape(0, x.shape, w.shape, 1, 1), 7.0, device="cuda")
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(tc.Tc3dError) as e:
        tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), 1, 1, out=y, workspace=small)
    assert e.value.status == tc.TC3D_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


def test_bounded_wait_reports_timeout(tc):
    """A wait on an mbarrier nobody arrives on gives up after its limit and
    the host sees TC3D_ERR_DEVICE_TIMEOUT; the context stays usable."""
    assert tc.selftest_wait_timeout(20_000_000) == tc.TC3D_ERR_DEVICE_TIMEOUT
    assert tc.last_device_error() == tc.TC3D_OK
    x, w, b = make((1, 3, 5, 6, 8), (4, 3, 3, 3, 3), 4)
    check(tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), 1, 1).cpu().numpy(),
          orc.conv3d(x, w, b, 1, 1), "after timeout")
    assert tc.last_device_error() == tc.TC3D_OK


# --------------------------------------------------------------------------
# the five workloads at full size (sampled outputs)
# --------------------------------------------------------------------------
def _wl(name):
    wl = BY_NAME[name]
    x, w, b = wl.make_inputs()
    return wl, x, w, b


def test_workload_conv331_tiny_full(tc):
    wl, x, w, b = _wl("conv331_tiny")
    y = tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), **wl.kwargs()).cpu().numpy()
    check(y, orc.conv3d(x, w, b, **wl.kwargs()), wl.name)


def test_workload_conv331_sampled(tc):
    wl, x, w, b = _wl("conv331")
    y = tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), **wl.kwargs()).cpu().numpy().ravel()
    idx = inputs.sample_indices(202, y.size, 20000)
    idx = np.concatenate([idx, [0, y.size - 1]])
    check(y[idx], orc.conv3d_at(x, w, b, idx, **wl.kwargs()), wl.name)


def test_workload_convT_s2p1d2_sampled(tc):
    wl, x, w, b = _wl("convT_s2p1d2")
    y = tc.conv_transpose3d_fwd(_dev(x), _dev(w), None, **wl.kwargs()).cpu().numpy()
    assert y.shape == (16, 64, 33, 65, 65)
    # outputs with any even coordinate belong to classes without taps: exactly 0
    odd = np.zeros(y.shape[2:], bool)
    odd[1::2, 1::2, 1::2] = True
    assert np.all(y[:, :, ~odd] == 0.0)
    flat = y.ravel()
    idx = inputs.sample_indices(303, flat.size, 20000)
    idx = np.concatenate([idx, [0, flat.size - 1]])
    check(flat[idx], orc.conv_transpose3d_at(x, w, None, idx, **wl.kwargs()), wl.name)


def test_workload_convT_bn_avgpool_full(tc):
    """The transposed-conv + BN + pool workload at full size, every one of its
    3,456,000 outputs against the oracle (whose statistics pass streams the
    whole transposed conv anyway)."""
    wl, x, w, b = _wl("convT_bn_avgpool")
    y = tc.convT_bn_avgpool(_dev(x), _dev(w), _dev(b), None, None, wl.eps,
                            **wl.kwargs()).cpu().numpy()
    assert y.shape == (64, 16, 15, 15, 15)
    flat = y.ravel()
    idx = np.arange(flat.size, dtype=np.int64)
    ref = orc.convT_bn_avgpool_at(x, w, b, idx, None, None, wl.eps, **wl.kwargs())
    check(flat, ref, wl.name)
    # BatchNorm with gamma 1, beta 0: each channel of the pooled output has
    # mean ~ 0 (pooling averages whole windows of the normalised tensor)
    assert np.all(np.abs(y.mean(axis=(0, 2, 3, 4))) < 0.05)


def test_workload_convT_bn_avgpool_uniform01_affine(tc):
    """The same workload with torch.rand-style inputs (all positive: the
    transposed conv's mean is far from 0, so the statistics difference
    E[t^2] - mean^2 cancels) and a non-trivial gamma / beta, on sampled
    outputs plus two whole (sample, channel) blocks."""
    wl = BY_NAME["convT_bn_avgpool"]
    x, w, b = wl.make_inputs(x_dist="uniform01")
    c = wl.cout
    g = inputs.uniform(4401, (c,), 0.5, 1.5)
    be = inputs.uniform(4402, (c,), -0.5, 0.5)
    y = tc.convT_bn_avgpool(_dev(x), _dev(w), _dev(b), _dev(g), _dev(be), wl.eps,
                            **wl.kwargs()).cpu().numpy()
    flat = y.ravel()
    per_nc = int(np.prod(y.shape[2:]))
    idx = inputs.sample_indices(4403, flat.size, 20000)
    blocks = [np.arange(per_nc, dtype=np.int64) + (n * c + co) * per_nc for n, co in ((0, 0), (63, 15))]
    idx = np.concatenate([idx] + blocks)
    ref = orc.convT_bn_avgpool_at(x, w, b, idx, g, be, wl.eps, **wl.kwargs())
    check(flat[idx], ref, wl.name + " uniform01")


def test_workload_convT_bneval_avgpool_sampled(tc):
    """The transposed-conv + BN + pool workload in evaluation mode."""
    wl, x, w, b = _wl("convT_bn_avgpool")
    rm, rv = _running_stats(16, 505)
    g = inputs.uniform(506, (16,), 0.5, 1.5)
    be = inputs.uniform(507, (16,), -0.5, 0.5)
    y = tc.convT_bneval_avgpool(_dev(x), _dev(w), _dev(b), _dev(rm), _dev(rv), _dev(g), _dev(be),
                                wl.eps, **wl.kwargs()).cpu().numpy()
    assert y.shape == (64, 16, 15, 15, 15)
    flat = y.ravel()
    idx = inputs.sample_indices(505, flat.size, 20000)
    idx = np.concatenate([idx, [0, flat.size - 1]])
    ref = orc.convT_bneval_avgpool_at(x, w, b, rm, rv, idx, g, be, wl.eps, **wl.kwargs())
    check(flat[idx], ref, wl.name + " eval")


@pytest.mark.parametrize("name", ["dwconv_k3", "dwconv_k3_ndhwc", "conv_k3_ndhwc"])
def test_workload_grouped_and_channels_last_sampled(tc, name):
    """The depthwise conv (direct kernel) in both layouts and the dense
    channels-last conv (engine between layout transposes) at full size,
    sampled outputs against the oracle."""
    wl, x, w, b = _wl(name)
    kw = dict(stride=wl.stride, padding=wl.padding, dilation=wl.dilation, groups=wl.groups)
    if wl.op == "conv3d_ndhwc":
        y = tc.conv3d_fwd_ndhwc(_dev(np.ascontiguousarray(x.transpose(0, 2, 3, 4, 1))), _dev(w),
                                _dev(b), **kw).cpu().numpy()
        y = y.transpose(0, 4, 1, 2, 3)  # compare in NCDHW order
    else:
        y = tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), **kw).cpu().numpy()
    flat = np.ascontiguousarray(y).ravel()
    idx = inputs.sample_indices(606 + wl.index, flat.size, 20000)
    idx = np.concatenate([idx, [0, flat.size - 1]])
    check(flat[idx], orc.conv3d_at(x, w, b, idx, **kw), name)


def test_workload_conv_maxpool_lse_relu_sampled(tc):
    wl, x, w, b = _wl("conv_maxpool_lse_relu")
    y = tc.conv_maxpool_lse_relu(_dev(x), _dev(w), _dev(b), **wl.kwargs()).cpu().numpy()
    assert y.shape == (4, 1, 16, 64, 64)
    flat = y.ravel()
    # random points, plus whole blocks: every pooled output of sample 0 in
    # depth planes 0 and 15, and of sample 3 in plane 8 (entire engine tiles,
    # among them the first and the last tiles of the persistent schedule)
    P = y.shape[2:]
    blocks = [np.arange(P[1] * P[2]) + ((n * P[0] + d) * P[1] * P[2]) for n, d in ((0, 0), (0, 15), (3, 8))]
    idx = inputs.sample_indices(505, flat.size, 1500)
    idx = np.concatenate([idx, [0, flat.size - 1]] + blocks).astype(np.int64)
    check(flat[idx], orc.conv_maxpool_lse_relu_at(x, w, b, idx, **wl.kwargs()), wl.name)
    # logsumexp over 64 channels >= their max, so ReLU rarely clips here
    assert np.all(flat >= 0.0)


# --------------------------------------------------------------------------
# second workloads at full size (outputs sampled on the device)
# --------------------------------------------------------------------------
def test_workload_conv331_p1_sampled(tc):
    wl, x, w, b = _wl("conv331_p1")
    y = tc.conv3d_fwd(_dev(x), _dev(w), _dev(b), **wl.kwargs())
    assert tuple(y.shape) == (16, 64, 254, 254, 10)
    n = y.numel()
    idx = np.concatenate([inputs.sample_indices(206, n, 20000), [0, n - 1]]).astype(np.int64)
    got = y.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy()
    check(got, orc.conv3d_at(x, w, b, idx, **wl.kwargs()), wl.name)


def test_workload_convT_s2p1d2_cin128_sampled(tc):
    wl, x, w, b = _wl("convT_s2p1d2_cin128")
    y = tc.conv_transpose3d_fwd(_dev(x), _dev(w), None, **wl.kwargs())
    assert tuple(y.shape) == (16, 64, 33, 65, 65)
    n = y.numel()
    idx = np.concatenate([inputs.sample_indices(207, n, 20000), [0, n - 1]]).astype(np.int64)
    got = y.reshape(-1)[torch.from_numpy(idx).cuda()].cpu().numpy()
    check(got, orc.conv_transpose3d_at(x, w, None, idx, **wl.kwargs()), wl.name)
