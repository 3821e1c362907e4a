"""Seeded synthetic inputs, shared by the CUDA path's tests/benchmark and the
oracle's tests.  This module draws random numbers and rounds them to the
storage dtype; it holds none of the convolution's arithmetic.

Recipe (the model files the pages benchmark are not available; only the layer
shapes are used):

* ``uniform``: x, W ~ U[-1, 1] rounded to bf16 (round-to-nearest-even),
  bias ~ U[-0.1, 0.1] fp32.
* ``normal``: x ~ N(0, 1) -> bf16; W He-normal (sigma^2 = 2 / fan_in) -> bf16;
  BN gamma ~ U[0.5, 1.5], beta ~ N(0, 0.1), mean ~ N(0, 0.1), var ~ U[0.5, 1.5]; when the
  ResNet-50 layers run as one network, each block's last BN has gamma scaled by
  RESIDUAL_BRANCH_GAMMA (``residual_branch_inputs``).
* ``int``: x ~ U{-128..127}, W ~ U{-127..127} (int8), bias ~ U{-2^16..2^16}
  (int32), per-channel requant multiplier M in [2^30, 2^31) and shift sh with
  M / 2^sh ~ 127 / (4 sigma_acc) * U[0.5, 1.5], sigma_acc = 73.9^2 sqrt(C R S),
  so that the int8 outputs span the range without saturating everywhere.

All draws come from ``torch.Generator().manual_seed(seed)`` on the CPU.  The
logical layout of every tensor is the ONNX one (NCHW / KCRS); callers choose
the storage layout.
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import torch

from .workloads import ConvSpec


def seed_for(config: int, layer_index: int) -> int:
    return 1000 * config + layer_index


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _uniform(g, shape, lo, hi):
    return torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo


def conv_inputs(spec: ConvSpec, seed: int) -> Dict[str, Optional[torch.Tensor]]:
    """x (bf16, NCHW), w (bf16, KCRS), bias (fp32 or None), bn = (gamma, beta, mean, var)."""
    g = _gen(seed)
    Cg = spec.C // spec.group
    xs = (spec.N, spec.C, spec.H, spec.W)
    ws = (spec.K, Cg, spec.R, spec.S)
    if spec.values == "uniform":
        x = _uniform(g, xs, -1.0, 1.0)
        w = _uniform(g, ws, -1.0, 1.0)
    else:
        x = torch.randn(xs, generator=g, dtype=torch.float32)
        w = torch.randn(ws, generator=g, dtype=torch.float32) * math.sqrt(2.0 / (Cg * spec.R * spec.S))
    out = {"x": x.to(torch.bfloat16), "w": w.to(torch.bfloat16), "bias": None, "bn": None}
    if spec.has_bias:
        out["bias"] = _uniform(g, (spec.K,), -0.1, 0.1)
    if spec.has_bn:
        gamma = _uniform(g, (spec.K,), 0.5, 1.5)
        beta = torch.randn(spec.K, generator=g) * 0.1
        mean = torch.randn(spec.K, generator=g) * 0.1
        var = _uniform(g, (spec.K,), 0.5, 1.5)
        out["bn"] = (gamma, beta, mean, var)
    return out


# The BN scale (gamma) of each bottleneck's last conv, relative to conv_inputs', when the layers
# run as one network: with every BN drawn as in conv_inputs the residual stream roughly doubles
# in every block (each block adds a branch of its own size), reaching 10^4 by the last stage, where
# a conv output is a near-cancelling sum of terms up to 10^5 that no fp32 accumulation resolves
# to 1e-3 of its value.  A smaller gamma on the branch (the usual initialisation of a residual
# network keeps it small, or zero) keeps the stream's scale steady.
RESIDUAL_BRANCH_GAMMA = 0.25


def residual_branch_inputs(spec: ConvSpec, seed: int) -> Dict[str, Optional[torch.Tensor]]:
    """conv_inputs with the BN gamma scaled by RESIDUAL_BRANCH_GAMMA (a block's last conv)."""
    out = conv_inputs(spec, seed)
    gamma, beta, mean, var = out["bn"]
    out["bn"] = (gamma * RESIDUAL_BRANCH_GAMMA, beta, mean, var)
    return out


def int8_inputs(spec: ConvSpec, seed: int) -> Dict[str, torch.Tensor]:
    """x int8, w int8 (NCHW / KCRS), bias int32[K], mult int32[K], shift int32[K]."""
    g = _gen(seed)
    Cg = spec.C // spec.group
    x = torch.randint(-128, 128, (spec.N, spec.C, spec.H, spec.W), generator=g, dtype=torch.int8)
    w = torch.randint(-127, 128, (spec.K, Cg, spec.R, spec.S), generator=g, dtype=torch.int8)
    bias = torch.randint(-(1 << 16), (1 << 16) + 1, (spec.K,), generator=g, dtype=torch.int32)
    sigma_acc = 73.9 * 73.9 * math.sqrt(Cg * spec.R * spec.S)
    u = _uniform(g, (spec.K,), 0.5, 1.5).double()
    mult = torch.empty(spec.K, dtype=torch.int32)
    shift = torch.empty(spec.K, dtype=torch.int32)
    for k in range(spec.K):
        scale = 127.0 / (4.0 * sigma_acc) * float(u[k])
        e = math.floor(math.log2(scale))           # scale = f * 2^e, f in [1, 2)
        sh = 30 - e
        m = int(round(scale * 2.0 ** sh))
        if m >= (1 << 31):
            m >>= 1
            sh -= 1
        mult[k] = m
        shift[k] = sh
    return {"x": x, "w": w, "bias": bias, "mult": mult, "shift": shift}


def qlinear_inputs(spec: ConvSpec, seed: int, x_signed: bool = False, w_signed: bool = True,
                   y_signed: bool = False) -> Dict[str, object]:
    """ONNX QLinearConv operands: x (uint8 U{0..255} or int8 U{-128..127}) with a zero point near
    the middle of its range, w (int8 U{-127..127} or uint8 U{0..255}) with small per-channel zero
    points, int32 bias U{-2^15..2^15}, x_scale ~ U[0.01, 0.03], w_scale[k] ~ U[0.002, 0.006], and
    y_scale / y_zero_point chosen so that the outputs span the 8-bit range (y_scale = 4 sigma of
    the real-valued sums / 127)."""
    g = _gen(seed)
    Cg = spec.C // spec.group
    xs = (spec.N, spec.C, spec.H, spec.W)
    ws = (spec.K, Cg, spec.R, spec.S)
    if x_signed:
        x = torch.randint(-128, 128, xs, generator=g, dtype=torch.int8)
        x_zp = int(torch.randint(-30, 31, (1,), generator=g))
    else:
        x = torch.randint(0, 256, xs, generator=g, dtype=torch.int32).to(torch.uint8)
        x_zp = int(torch.randint(98, 159, (1,), generator=g))
    if w_signed:
        w = torch.randint(-127, 128, ws, generator=g, dtype=torch.int8)
        w_zp = torch.randint(-10, 11, (spec.K,), generator=g, dtype=torch.int32)
    else:
        w = torch.randint(0, 256, ws, generator=g, dtype=torch.int32).to(torch.uint8)
        w_zp = torch.randint(118, 139, (spec.K,), generator=g, dtype=torch.int32)
    bias = torch.randint(-(1 << 15), (1 << 15) + 1, (spec.K,), generator=g, dtype=torch.int32)
    x_scale = float(_uniform(g, (1,), 0.01, 0.03))
    w_scale = _uniform(g, (spec.K,), 0.002, 0.006)
    sigma = 74.0 * 74.0 * math.sqrt(Cg * spec.R * spec.S) * x_scale * float(w_scale.mean())
    y_scale = float(4.0 * sigma / 127.0)
    y_zp = int(torch.randint(-20, 21, (1,), generator=g)) if y_signed else int(torch.randint(100, 157, (1,), generator=g))
    return {"x": x, "x_zp": x_zp, "w": w, "w_zp": w_zp, "bias": bias, "x_scale": x_scale, "w_scale": w_scale,
            "y_scale": y_scale, "y_zp": y_zp, "x_signed": x_signed, "y_signed": y_signed}


def block_inputs(N: int, Cin: int, H: int, Ch: int, Cout: int, expand: bool, seed: int) -> Dict[str, object]:
    """A MobileNetV2 block's tensors: x ~ N(0,1) -> bf16, He-normal bf16 weights per conv
    (fan-in Cin, 9 and Ch), and per stage BN = (gamma ~ U[0.5,1.5], beta ~ N(0,0.1),
    mean ~ N(0,0.1), var ~ U[0.5,1.5])."""
    g = _gen(seed)

    def bn(k):
        return (_uniform(g, (k,), 0.5, 1.5), torch.randn(k, generator=g) * 0.1, torch.randn(k, generator=g) * 0.1,
                _uniform(g, (k,), 0.5, 1.5))

    x = torch.randn((N, Cin, H, H), generator=g).to(torch.bfloat16)
    we = (torch.randn((Ch, Cin, 1, 1), generator=g) * math.sqrt(2.0 / Cin)).to(torch.bfloat16) if expand else None
    wd = (torch.randn((Ch, 1, 3, 3), generator=g) * math.sqrt(2.0 / 9)).to(torch.bfloat16)
    wp = (torch.randn((Cout, Ch, 1, 1), generator=g) * math.sqrt(2.0 / Ch)).to(torch.bfloat16)
    return {"x": x, "we": we, "bn_e": bn(Ch) if expand else None, "wd": wd, "bn_d": bn(Ch), "wp": wp,
            "bn_p": bn(Cout)}


def sample_points(spec: ConvSpec, count: int, seed: int) -> torch.Tensor:
    """``count`` output coordinates (n, k, oh, ow), always including the corners
    and edges of the output (where padding matters) and the last channel."""
    ho, wo = spec.out_hw
    g = _gen(seed)
    pts = torch.stack([torch.randint(0, spec.N, (count,), generator=g),
                       torch.randint(0, spec.K, (count,), generator=g),
                       torch.randint(0, ho, (count,), generator=g),
                       torch.randint(0, wo, (count,), generator=g)], dim=1)
    fixed = []
    for n in {0, spec.N - 1}:
        for k in {0, spec.K - 1}:
            for oh in {0, ho - 1}:
                for ow in {0, wo - 1}:
                    fixed.append((n, k, oh, ow))
    return torch.cat([torch.tensor(fixed, dtype=torch.int64), pts.to(torch.int64)], dim=0)
