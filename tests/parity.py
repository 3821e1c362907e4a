"""Helpers shared by the GPU parity tests and the smoke check: run one conv spec through the
C-ABI library and compare with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import synthetic
from convolution_onnx_conv_gb300.workloads import ConvSpec

ATOL = 1e-3
RTOL = 1e-3


def to_device_nhwc(x: torch.Tensor) -> torch.Tensor:
    return x.contiguous(memory_format=torch.channels_last).cuda()


def make_conv(spec: ConvSpec, inp, variant=cf.CONVF_VARIANT_AUTO, act=None):
    act = spec.act if act is None else act
    if spec.dtype == "s8":
        return cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                            stride=spec.stride, pads=spec.pads, dilation=spec.dilation, group=spec.group,
                            act=act, variant=variant, requant_mult=inp["mult"], requant_shift=inp["shift"],
                            out_zero_point=inp.get("zp", 0))
    scale = shift = None
    if inp["bn"] is not None:
        scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5)
    return cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                        scale, shift, stride=spec.stride, pads=spec.pads, dilation=spec.dilation,
                        group=spec.group, act=act, clip=inp.get("clip", (0.0, 6.0)), variant=variant)


def oracle_full(spec: ConvSpec, inp, act=None):
    act = spec.act if act is None else act
    if spec.dtype == "s8":
        acc = oracle.conv2d_s8(inp["x"].numpy(), inp["w"].numpy(), spec.stride, spec.pads, spec.dilation,
                               spec.group)
        return oracle.requant_s8(acc, None, inp["bias"].numpy(), inp["mult"].numpy(), inp["shift"].numpy(),
                                 inp.get("zp", 0), relu=act == cf.CONVF_ACT_RELU)
    bn = None if inp["bn"] is None else tuple(t.numpy() for t in inp["bn"])
    lo, hi = inp.get("clip", (0.0, 6.0))
    return oracle.conv_bn_act(inp["x"].double().numpy(), inp["w"].double().numpy(),
                              None if inp["bias"] is None else inp["bias"].numpy(), bn, act, lo, hi,
                              spec.stride, spec.pads, spec.dilation, spec.group)


def oracle_points(spec: ConvSpec, inp, pts, act=None):
    act = spec.act if act is None else act
    if spec.dtype == "s8":
        acc = oracle.conv2d_s8_points(inp["x"].numpy(), inp["w"].numpy(), spec.stride, spec.pads,
                                      spec.dilation, spec.group, pts)
        return oracle.requant_s8(acc, pts[:, 1], inp["bias"].numpy(), inp["mult"].numpy(),
                                 inp["shift"].numpy(), inp.get("zp", 0), relu=act == cf.CONVF_ACT_RELU)
    bn = None if inp["bn"] is None else tuple(t.numpy() for t in inp["bn"])
    lo, hi = inp.get("clip", (0.0, 6.0))
    return oracle.conv_bn_act_points(inp["x"].double().numpy(), inp["w"].double().numpy(),
                                     None if inp["bias"] is None else inp["bias"].numpy(), bn, act,
                                     spec.stride, spec.pads, spec.dilation, spec.group, pts, lo, hi)


def inputs_for(spec: ConvSpec, seed: int):
    return synthetic.int8_inputs(spec, seed) if spec.dtype == "s8" else synthetic.conv_inputs(spec, seed)


def run_gpu(spec: ConvSpec, inp, variant=cf.CONVF_VARIANT_AUTO, act=None, runs: int = 1):
    conv = make_conv(spec, inp, variant, act)
    x = to_device_nhwc(inp["x"])
    y = None
    for _ in range(runs):
        y = conv(x, y)
    torch.cuda.synchronize()
    status = conv.status()
    used = conv.variant
    desc = conv.describe()
    conv.close()
    return y.cpu().contiguous(), status, used, desc


def compare(y, ref, integer: bool):
    """(ok, worst allowance ratio or mismatch count, flat index of the worst element)."""
    y = np.asarray(y)
    ref = np.asarray(ref)
    if integer:
        bad = np.flatnonzero(y.reshape(-1) != ref.reshape(-1))
        return bad.size == 0, int(bad.size), int(bad[0]) if bad.size else -1
    return oracle.tolerance_ok(y, ref, ATOL, RTOL)


def check_full(spec: ConvSpec, seed: int, variant=cf.CONVF_VARIANT_AUTO, act=None, inp=None):
    inp = inp if inp is not None else inputs_for(spec, seed)
    y, status, used, desc = run_gpu(spec, inp, variant, act)
    ref = oracle_full(spec, inp, act)
    ok, worst, idx = compare(y.numpy(), ref, spec.dtype == "s8")
    return ok, worst, idx, status, used, desc


def check_sampled(spec: ConvSpec, seed: int, count: int = 2000, variant=cf.CONVF_VARIANT_AUTO):
    inp = inputs_for(spec, seed)
    y, status, used, desc = run_gpu(spec, inp, variant)
    pts = synthetic.sample_points(spec, count, seed + 17).numpy()
    ref = oracle_points(spec, inp, pts)
    got = y.numpy()[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    ok, worst, idx = compare(got, ref, spec.dtype == "s8")
    return ok, worst, idx, status, used, desc, y


# ------------------------------------------------------------------ QLinearConv

def make_qconv(spec: ConvSpec, inp, relu=False, variant=cf.CONVF_VARIANT_AUTO, **kw):
    return cf.QLinearConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                          x_scale=inp["x_scale"], x_zero_point=inp["x_zp"], w_scale=inp["w_scale"].numpy(),
                          w_zero_point=inp["w_zp"].numpy(), y_scale=inp["y_scale"], y_zero_point=inp["y_zp"],
                          x_signed=inp["x_signed"], y_signed=inp["y_signed"], relu=relu, stride=spec.stride,
                          pads=spec.pads, dilation=spec.dilation, group=spec.group, variant=variant, **kw)


def oracle_qlinear(spec: ConvSpec, inp, relu=False):
    acc = oracle.qlinear_conv_acc(inp["x"].numpy(), inp["x_zp"], inp["w"].numpy(), inp["w_zp"].numpy(),
                                  inp["bias"].numpy(), spec.stride, spec.pads, spec.dilation, spec.group)
    return oracle.qlinear_requant(acc, inp["x_scale"], inp["w_scale"].numpy(), inp["y_scale"], inp["y_zp"],
                                  np.int8 if inp["y_signed"] else np.uint8, relu=relu)


def check_qlinear(spec: ConvSpec, inp, relu=False, **kw):
    """(mismatch count, flat index of the first mismatch, status, describe) over every output."""
    conv = make_qconv(spec, inp, relu, **kw)
    x = to_device_nhwc(inp["x"])
    y = conv(x)
    torch.cuda.synchronize()
    status, desc = conv.status(), conv.describe()
    conv.close()
    got = y.cpu().contiguous().numpy()
    ref = oracle_qlinear(spec, inp, relu)
    bad = np.flatnonzero(got.reshape(-1) != ref.reshape(-1))
    return int(bad.size), int(bad[0]) if bad.size else -1, status, desc
