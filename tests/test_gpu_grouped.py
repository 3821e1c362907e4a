"""GPU parity of grouped convolutions (1 < group < C) against the CPU oracle, every output.

On the tensor cores, an output-channel tile covers whole groups or lies inside one, its
activation loads read that tile's window of input channels and the weights are packed block
diagonally over the window; shapes that cannot be tiled that way run on the direct CUDA-core
kernel.  bf16 in, fp32 accumulate: |y - ref| <= 1e-3 + 1e-3 |ref|.
"""
import numpy as np
import pytest
import torch

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import synthetic, workloads
from convolution_onnx_conv_gb300.workloads import ConvSpec, ACT_NONE, ACT_RELU, ACT_RELU6

import oracle
from parity import ATOL, RTOL, check_full, inputs_for, to_device_nhwc

pytestmark = pytest.mark.gpu
V = cf


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cf.load_library(build_if_missing=True)


def G(name, N, C, H, W, K, R, S_, group, stride=(1, 1), pads=(0, 0, 0, 0), dil=(1, 1), act=ACT_RELU, bias=False):
    return ConvSpec(name, N, C, H, W, K, R, S_, stride, pads, dil, group, act, bias, True, "bf16", "normal")


CASES = [
    # (spec, expected variant)
    (G("g32_cg4_3x3", 2, 128, 12, 12, 128, 3, 3, 32, pads=(1, 1, 1, 1)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (G("g32_cg8_3x3_s2", 2, 256, 13, 13, 256, 3, 3, 32, (2, 2), (1, 1, 1, 1), bias=True), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (G("g2_cg128_3x3_k256", 1, 256, 9, 11, 256, 3, 3, 2, pads=(1, 1, 1, 1)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (G("g4_cg64_kg96_3x3", 2, 256, 10, 10, 384, 3, 3, 4, pads=(1, 1, 1, 1), act=ACT_RELU6), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (G("g3_cg8_kg4_5x5", 2, 24, 11, 9, 12, 5, 5, 3, pads=(2, 2, 2, 2), act=ACT_NONE), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (G("g8_1x1_cg32", 3, 256, 9, 10, 256, 1, 1, 8), V.CONVF_VARIANT_GEMM_1X1),
    (G("g16_1x1_cg8_kg16", 2, 128, 7, 9, 256, 1, 1, 16, bias=True), V.CONVF_VARIANT_GEMM_1X1),
    (G("g4_dil2_asym", 1, 64, 13, 12, 64, 3, 3, 4, (1, 1), (2, 1, 2, 2), (2, 2)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    # direct kernel: groups of 3, channel multiplier 2 (Cg = 1), C % 8 != 0, depthwise 5x5
    (G("gd_g8_cg3", 2, 24, 10, 10, 24, 3, 3, 8, pads=(1, 1, 1, 1)), V.CONVF_VARIANT_GROUPED_DIRECT),
    (G("gd_mult2_cg1", 2, 32, 9, 9, 64, 3, 3, 32, (2, 2), (1, 1, 1, 1), act=ACT_RELU6), V.CONVF_VARIANT_GROUPED_DIRECT),
    (G("gd_c12_g3", 1, 12, 8, 8, 6, 3, 3, 3, pads=(1, 1, 1, 1), bias=True), V.CONVF_VARIANT_GROUPED_DIRECT),
    (G("gd_g2_kg100", 1, 256, 9, 11, 200, 3, 3, 2, pads=(1, 1, 1, 1)), V.CONVF_VARIANT_GROUPED_DIRECT),
    (G("dw_5x5_c40", 2, 40, 14, 14, 40, 5, 5, 40, pads=(2, 2, 2, 2), act=ACT_RELU6), V.CONVF_VARIANT_DEPTHWISE),
    (G("dw_5x5_s2_c96", 2, 96, 15, 15, 96, 5, 5, 96, (2, 2), (2, 2, 2, 2), act=ACT_RELU6), V.CONVF_VARIANT_DEPTHWISE),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_grouped_every_output(case):
    spec, variant = case
    ok, worst, idx, status, used, desc = check_full(spec, 9300 + CASES.index(case))
    assert status == cf.CONVF_OK, desc
    assert used == variant, desc
    assert ok, f"{spec.name}: worst={worst} at {idx} ({desc})"


@pytest.mark.parametrize("tile_n", [32, 64])
def test_grouped_tile_widths(tile_n):
    """A tile of 32 covers 8 groups of 4 (a 32-channel window padded to 64), 64 covers 16 (a
    64-channel window: 16x the grouped work, the most the tensor-core path takes)."""
    spec = G("g32_tiles", 2, 128, 11, 11, 128, 3, 3, 32, pads=(1, 1, 1, 1))
    inp = inputs_for(spec, 9350)
    c = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], None,
                     *cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5), stride=spec.stride,
                     pads=spec.pads, group=spec.group, act=spec.act, tile_n=tile_n)
    d = c.describe()
    assert f"tile=128x{tile_n} " in d and "group=32" in d, d
    y = c(to_device_nhwc(inp["x"]))
    torch.cuda.synchronize()
    assert c.status() == cf.CONVF_OK
    from parity import compare, oracle_full
    ok, worst, idx = compare(y.cpu().contiguous().numpy(), oracle_full(spec, inp), False)
    c.close()
    assert ok, (worst, idx, d)


@pytest.mark.parametrize("spec", workloads.resnext50_grouped_layers(32), ids=lambda s: s.name)
def test_resnext50_grouped_layers_b32(spec):
    ok, worst, idx, status, used, desc = check_full(spec, synthetic.seed_for(10, workloads.resnext50_grouped_layers(32).index(spec)))
    assert status == cf.CONVF_OK and used == V.CONVF_VARIANT_IMPLICIT_GEMM, desc
    assert ok, f"{spec.name}: worst={worst} at {idx} ({desc})"
    print(f"{spec.name}: worst ratio={worst:.4g} ({desc})")


@pytest.mark.parametrize("out_bf16,residual", [(False, True), (True, False), (True, True)])
def test_direct_grouped_residual_and_bf16(out_bf16, residual):
    spec = G("gd_ext", 2, 24, 9, 10, 24, 3, 3, 8, pads=(1, 1, 1, 1), act=ACT_RELU6)
    inp = inputs_for(spec, 9380)
    conv = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], None,
                        *cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5), pads=spec.pads,
                        group=spec.group, act=spec.act, out_bf16=out_bf16, residual=residual)
    assert conv.variant == V.CONVF_VARIANT_GROUPED_DIRECT
    N, K, Ho, Wo = conv.out_shape
    g = torch.Generator().manual_seed(9381)
    r = torch.randn((N, K, Ho, Wo), generator=g)
    r = r.to(torch.bfloat16) if out_bf16 else r
    ref = oracle.conv_bn_act(inp["x"].double().numpy(), inp["w"].double().numpy(), None,
                             tuple(t.numpy() for t in inp["bn"]), spec.act, 0.0, 6.0, spec.stride, spec.pads,
                             spec.dilation, spec.group, residual=r.double().numpy() if residual else None)
    y = conv(to_device_nhwc(inp["x"]), r=to_device_nhwc(r) if residual else None)
    torch.cuda.synchronize()
    assert conv.status() == cf.CONVF_OK
    got = y.cpu().contiguous().float().numpy().astype(np.float64)
    allow = ATOL + RTOL * np.abs(ref)
    if out_bf16:
        # one bf16 step on top of the fp32 bound (a value near a rounding midpoint may go either way)
        allow = allow + np.abs(ref) * 2.0 ** -7
    assert np.all(np.abs(got - ref) <= allow), float(np.max(np.abs(got - ref) / allow))
    conv.close()
