"""GPU parity of the pre-activation prologue (ResNet-v2: the conv reads act(scale*x + shift) of
its input, zero-padded after the activation, as bf16) against the CPU oracle, every output, on
every kernel variant that reads a bf16 input."""
import numpy as np
import pytest
import torch

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import synthetic, workloads
from convolution_onnx_conv_gb300.workloads import ConvSpec, ACT_NONE, ACT_RELU, ACT_RELU6

import oracle
from parity import ATOL, RTOL, inputs_for, to_device_nhwc

pytestmark = pytest.mark.gpu
V = cf


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cf.load_library(build_if_missing=True)


def P(name, N, C, H, W, K, R, S_, stride=(1, 1), pads=(0, 0, 0, 0), group=1, act=ACT_RELU):
    return ConvSpec(name, N, C, H, W, K, R, S_, stride, pads, (1, 1), group, act, False, True, "bf16", "normal")


CASES = [
    # (spec, pre activation, expected variant)
    (P("pre_1x1_c256", 2, 256, 14, 14, 64, 1, 1), ACT_RELU, V.CONVF_VARIANT_GEMM_1X1),
    (P("pre_3x3_s2_im2col", 2, 128, 15, 15, 128, 3, 3, (2, 2), (1, 1, 1, 1)), ACT_RELU, V.CONVF_VARIANT_IMPLICIT_GEMM),
    (P("pre_3x3_halo_w56", 2, 64, 8, 56, 64, 3, 3, pads=(1, 1, 1, 1)), ACT_RELU, V.CONVF_VARIANT_IMPLICIT_GEMM_HALO),
    (P("pre_stem_c3", 2, 3, 64, 64, 64, 7, 7, (2, 2), (3, 3, 3, 3)), ACT_RELU6, V.CONVF_VARIANT_IMPLICIT_GEMM_WINDOW),
    (P("pre_gather_c5", 1, 5, 19, 21, 24, 3, 3, pads=(1, 1, 1, 1)), ACT_NONE, V.CONVF_VARIANT_IMPLICIT_GEMM_GATHER),
    (P("pre_dw_c96", 2, 96, 15, 15, 96, 3, 3, pads=(1, 1, 1, 1), group=96, act=ACT_RELU6), ACT_RELU6,
     V.CONVF_VARIANT_DEPTHWISE),
    (P("pre_grouped_g32", 2, 128, 10, 10, 128, 3, 3, pads=(1, 1, 1, 1), group=32), ACT_RELU, V.CONVF_VARIANT_IMPLICIT_GEMM),
    (P("pre_grouped_direct", 2, 24, 9, 9, 24, 3, 3, pads=(1, 1, 1, 1), group=8), ACT_RELU, V.CONVF_VARIANT_GROUPED_DIRECT),
]


def _pre_params(C, seed):
    g = torch.Generator().manual_seed(seed)
    gamma = torch.rand(C, generator=g) + 0.5
    beta = torch.randn(C, generator=g) * 0.3       # shifts that move the ReLU threshold
    mean = torch.randn(C, generator=g) * 0.1
    var = torch.rand(C, generator=g) + 0.5
    return cf.conv_bn_scale_shift(gamma.numpy(), beta.numpy(), mean.numpy(), var.numpy(), 1e-5)


def _check(spec, pre_act, seed, variant=None):
    inp = inputs_for(spec, seed)
    ps, pt = _pre_params(spec.C, seed + 1)
    scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5)
    conv = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], None, scale, shift,
                        stride=spec.stride, pads=spec.pads, group=spec.group, act=spec.act, pre_scale=ps,
                        pre_shift=pt, pre_act=pre_act, variant=variant or cf.CONVF_VARIANT_AUTO)
    used = conv.variant
    x = to_device_nhwc(inp["x"])
    for _ in range(2):   # the staging copy is rewritten by every run
        y = conv(x)
    torch.cuda.synchronize()
    assert conv.status() == cf.CONVF_OK
    desc = conv.describe()
    conv.close()
    ref = oracle.conv_bn_act(inp["x"].double().numpy(), inp["w"].double().numpy(), None,
                             tuple(t.numpy() for t in inp["bn"]), spec.act, 0.0, 6.0, spec.stride, spec.pads,
                             spec.dilation, spec.group, pre=(ps.astype(np.float64), pt.astype(np.float64), pre_act))
    ok, worst, idx = oracle.tolerance_ok(y.cpu().contiguous().numpy(), ref, ATOL, RTOL)
    return ok, worst, idx, used, desc


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_preactivation_every_output(case):
    spec, pre_act, variant = case
    ok, worst, idx, used, desc = _check(spec, pre_act, 9500 + CASES.index(case))
    assert used == variant, desc
    assert ok, f"{spec.name}: worst={worst} at {idx} ({desc})"


R50 = {s.name: s for s in workloads.resnet50_layers(32)}


@pytest.mark.parametrize("name", ["r50_15_s1b1_1x1a@b32", "r50_44_s3b0_3x3@b32"])
def test_preactivation_resnet50_b32_layers(name):
    """ResNet-v2 block inputs at full size: the 512 -> 128 1x1 at 28x28 and the strided 3x3."""
    spec = R50[name]
    ok, worst, idx, used, desc = _check(spec, ACT_RELU, 9550 + list(R50).index(name))
    assert ok, f"{spec.name}: worst={worst} at {idx} ({desc})"
    print(f"{name} with prologue: worst ratio={worst:.4g} ({desc})")


def test_preactivation_refusals():
    spec = CASES[0][0]
    inp = inputs_for(spec, 9590)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], pre_scale=np.ones(spec.C),
                     pre_shift=np.zeros(spec.C), pre_act=cf.CONVF_ACT_CLIP)
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "pre_act" in str(e.value)
    bad = np.ones(spec.C, np.float32)
    bad[3] = np.inf
    with pytest.raises(cf.ConvFusedError) as e:
        cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], pre_scale=bad,
                     pre_shift=np.zeros(spec.C), pre_act=cf.CONVF_ACT_RELU)
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "not finite" in str(e.value)
