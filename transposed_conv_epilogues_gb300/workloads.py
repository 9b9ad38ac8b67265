"""The five benchmark / parity workloads and three second workloads, with
their synthetic input recipes.

Shapes follow the four POPCORNBENCH transcript pages:

* ``conv331_tiny`` / ``conv331``: Conv3d with a (3,3,1) kernel, the depth-1
  case of "Kimi-K2.6 l1_p59" (scaled: Cin 16, Cout 64, 16x128x128x8 input).
* ``convT_s2p1d2``: ConvTranspose3d 32->64, k3 s2 p1 d2 on a [16,32,16,32,32]
  input ("Kimi-K2.6 l1_p77" test case).  The output is [16,64,33,65,65]: the
  page's own output-size formula applied per axis (its 33^3 applies the depth
  length to all three axes).
* ``convT_bn_avgpool``: ConvTranspose3d 3->16, k3 s2 p1 + bias -> BatchNorm3d
  (batch statistics, eps 1e-5, gamma 1, beta 0) -> AvgPool3d(2) twice on a
  [64,3,32,32,32] input ("Kimi-K2.6 l2_p72").
* ``conv_maxpool_lse_relu``: Conv3d 32->64, k3 s1 p1 + bias -> MaxPool3d(2,2)
  -> logsumexp over channels -> ReLU on a [4,32,32,128,128] input
  ("Kimi-K2.6 l2_p43").

Inputs: x ~ N(0,1); weights and bias ~ U(-1/sqrt(fan_in), +1/sqrt(fan_in)).
fan_in is Cin/G * kernel volume for the convolutions and for the
ConvTranspose3d 32->64 workload (32*27, as its recipe states); for the
ConvTranspose3d 3->16 workload, whose recipe gives no bound, it is PyTorch's
default for that layer, weight.size(1) * kvol = 16*27.  Seeds: x 1000*i+1,
w 1000*i+2, bias 1000*i+3 for workload i = 1..5.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import inputs


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    op: str  # "conv3d" | "conv3d_ndhwc" | "conv_transpose3d" | "convT_bn_avgpool"
    #          | "convT_bneval_avgpool" | "conv_maxpool_lse_relu"
    # x_shape / w_shape are NCDHW / PyTorch layouts; a "conv3d_ndhwc" workload
    # feeds x and reads y channels-last
    x_shape: tuple
    w_shape: tuple
    bias: bool
    stride: tuple = (1, 1, 1)
    padding: tuple = (0, 0, 0)
    dilation: tuple = (1, 1, 1)
    output_padding: tuple = (0, 0, 0)
    groups: int = 1
    eps: float = 1e-5
    desc: str = ""
    fan_in: int = 0

    @property
    def transposed(self) -> bool:
        return self.op in ("conv_transpose3d", "convT_bn_avgpool", "convT_bneval_avgpool")

    @property
    def cout(self) -> int:
        return self.w_shape[1] * self.groups if self.transposed else self.w_shape[0]

    def make_inputs(self, x_dist: str = "normal"):
        """(x, w, b) float32 arrays; b is None without bias."""
        i = self.index
        bound = 1.0 / math.sqrt(self.fan_in)
        if x_dist == "normal":
            x = inputs.normal(1000 * i + 1, self.x_shape)
        else:  # "uniform01": torch.rand-style inputs used on the pages
            x = inputs.uniform(1000 * i + 1, self.x_shape, 0.0, 1.0)
        w = inputs.uniform(1000 * i + 2, self.w_shape, -bound, bound)
        b = inputs.uniform(1000 * i + 3, (self.cout,), -bound, bound) if self.bias else None
        return x, w, b

    def make_bn_eval_params(self):
        """(running_mean, running_var, gamma, beta) float32 [Cout] arrays of
        the evaluation-mode BatchNorm: means ~ 0.2 N(0,1), variances
        ~ U(0.05, 0.5) (the scale of the transposed-conv output), gamma
        ~ U(0.5, 1.5), beta ~ U(-0.5, 0.5); seeds 1000*i+4 .. 1000*i+7."""
        i, c = self.index, self.cout
        rm = (0.2 * inputs.normal(1000 * i + 4, (c,))).astype(np.float32)
        rv = inputs.uniform(1000 * i + 5, (c,), 0.05, 0.5)
        g = inputs.uniform(1000 * i + 6, (c,), 0.5, 1.5)
        be = inputs.uniform(1000 * i + 7, (c,), -0.5, 0.5)
        return rm, rv, g, be

    def kwargs(self) -> dict:
        kw = dict(stride=self.stride, padding=self.padding, dilation=self.dilation,
                  groups=self.groups)
        if self.transposed:
            kw["output_padding"] = self.output_padding
        return kw


WORKLOADS = [
    Workload(1, "conv331_tiny", "conv3d", (2, 4, 16, 16, 4), (8, 4, 3, 3, 1), True,
             fan_in=4 * 9, desc="Conv3d (3,3,1) tiny oracle check"),
    Workload(2, "conv331", "conv3d", (16, 16, 128, 128, 8), (64, 16, 3, 3, 1), True,
             fan_in=16 * 9, desc="Conv3d (3,3,1), depth axis acts as extra batch"),
    Workload(3, "convT_s2p1d2", "conv_transpose3d", (16, 32, 16, 32, 32), (32, 64, 3, 3, 3),
             False, stride=(2, 2, 2), padding=(1, 1, 1), dilation=(2, 2, 2),
             fan_in=32 * 27, desc="ConvTranspose3d 32->64 k3 s2 p1 d2"),
    Workload(4, "convT_bn_avgpool", "convT_bn_avgpool", (64, 3, 32, 32, 32), (3, 16, 3, 3, 3),
             True, stride=(2, 2, 2), padding=(1, 1, 1), fan_in=16 * 27,
             desc="ConvTranspose3d 3->16 k3 s2 p1 + BN(batch) + AvgPool3d(2) x2"),
    Workload(5, "conv_maxpool_lse_relu", "conv_maxpool_lse_relu", (4, 32, 32, 128, 128),
             (64, 32, 3, 3, 3), True, padding=(1, 1, 1), fan_in=32 * 27,
             desc="Conv3d 32->64 k3 p1 + MaxPool3d(2) + logsumexp_c + ReLU"),
]

# Second workloads (not part of the default bench step): the (k,k,1) conv at
# the shape "Kimi-K2.6 l1_p59" itself uses (Cin 3, Cout 64, a [16,3,256,256,10]
# input; its 2.6 GB output makes it output-write-bound), and the k3 s2 p1 d2
# transposed conv of "Kimi-K2.6 l1_p77" at a larger input channel count (Cin
# 128), which makes the GEMM K 3456, and the transposed-conv + BN + pool
# pipeline of "Kimi-K2.6 l2_p72" with BatchNorm in evaluation mode (running
# statistics, as that page's first fused kernel reads them) at the same shape.
# Seeds follow the same rule (i = 6, 7, 8).  Then grouped and channels-last
# convs (the direct kernel and the layout route, i = 9, 10, 11): a depthwise
# k3 conv on [8,64,32,64,64] in NCDHW and in NDHWC, and a dense k3 conv
# 32 -> 64 on [4,32,32,64,64] in NDHWC (fan_in: Cin/G * 27).
EXTRA_WORKLOADS = [
    Workload(6, "conv331_p1", "conv3d", (16, 3, 256, 256, 10), (64, 3, 3, 3, 1), True,
             fan_in=3 * 9, desc="Conv3d (3,3,1) 3->64 at the page's original shape"),
    Workload(7, "convT_s2p1d2_cin128", "conv_transpose3d", (16, 128, 16, 32, 32),
             (128, 64, 3, 3, 3), False, stride=(2, 2, 2), padding=(1, 1, 1),
             dilation=(2, 2, 2), fan_in=128 * 27,
             desc="ConvTranspose3d 128->64 k3 s2 p1 d2"),
    Workload(8, "convT_bneval_avgpool", "convT_bneval_avgpool", (64, 3, 32, 32, 32),
             (3, 16, 3, 3, 3), True, stride=(2, 2, 2), padding=(1, 1, 1), fan_in=16 * 27,
             desc="ConvTranspose3d 3->16 k3 s2 p1 + BN(running stats) + AvgPool3d(2) x2"),
    Workload(9, "dwconv_k3", "conv3d", (8, 64, 32, 64, 64), (64, 1, 3, 3, 3), True,
             padding=(1, 1, 1), groups=64, fan_in=27, desc="depthwise Conv3d k3 p1, 64 channels"),
    Workload(10, "dwconv_k3_ndhwc", "conv3d_ndhwc", (8, 64, 32, 64, 64), (64, 1, 3, 3, 3), True,
             padding=(1, 1, 1), groups=64, fan_in=27,
             desc="depthwise Conv3d k3 p1, 64 channels, channels-last"),
    Workload(11, "conv_k3_ndhwc", "conv3d_ndhwc", (4, 32, 32, 64, 64), (64, 32, 3, 3, 3), True,
             padding=(1, 1, 1), fan_in=32 * 27, desc="Conv3d 32->64 k3 p1, channels-last"),
]

BY_NAME = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS}


def _axis_pairs(L, K, s, p, d, O, transposed):
    """Number of (output position, tap) pairs of one axis whose input index is
    in range (and, for a transposed conv, exactly divisible)."""
    n = 0
    for o in range(O):
        for k in range(K):
            if transposed:
                t = o + p - d * k
                if t % s == 0 and 0 <= t // s < L:
                    n += 1
            else:
                if 0 <= o * s - p + d * k < L:
                    n += 1
    return n


def out_spatial(wl: Workload):
    """Output extents of the convolution / transposed convolution (before pooling)."""
    dims = []
    for a in range(3):
        L, K = wl.x_shape[2 + a], wl.w_shape[2 + a]
        s, p, d = wl.stride[a], wl.padding[a], wl.dilation[a]
        if wl.transposed:
            dims.append((L - 1) * s - 2 * p + d * (K - 1) + wl.output_padding[a] + 1)
        else:
            dims.append((L + 2 * p - d * (K - 1) - 1) // s + 1)
    return tuple(dims)


def valid_macs(wl: Workload) -> int:
    """Multiply-adds of the definition's sum, counting only taps whose input
    index is in range (zero taps ignored): the algorithmic work."""
    O = out_spatial(wl)
    prod = 1
    for a in range(3):
        prod *= _axis_pairs(wl.x_shape[2 + a], wl.w_shape[2 + a], wl.stride[a], wl.padding[a],
                            wl.dilation[a], O[a], wl.transposed)
    cin_g = wl.x_shape[1] // wl.groups
    return wl.x_shape[0] * wl.cout * cin_g * prod


def dense_macs(wl: Workload) -> int:
    """Multiply-adds of the dense definition (every tap of every output)."""
    O = out_spatial(wl)
    cin_g = wl.x_shape[1] // wl.groups
    return wl.x_shape[0] * wl.cout * cin_g * int(np.prod(O)) * int(np.prod(wl.w_shape[2:]))


def y_shape(wl: Workload):
    O = out_spatial(wl)
    N = wl.x_shape[0]
    if wl.op == "conv_maxpool_lse_relu":
        return (N, 1) + tuple(o // 2 for o in O)
    if wl.op in ("convT_bn_avgpool", "convT_bneval_avgpool"):
        return (N, wl.cout) + tuple(o // 2 // 2 for o in O)
    if wl.op == "conv3d_ndhwc":
        return (N,) + O + (wl.cout,)
    return (N, wl.cout) + O


def algorithmic_bytes(wl: Workload) -> int:
    """Read x and the weights (and bias, and the BatchNorm running
    statistics and affine parameters) once, write y once; fused intermediates
    count zero."""
    n = int(np.prod(wl.x_shape)) + int(np.prod(wl.w_shape)) + int(np.prod(y_shape(wl)))
    if wl.bias:
        n += wl.cout
    if wl.op == "convT_bneval_avgpool":
        n += 4 * wl.cout
    return 4 * n
