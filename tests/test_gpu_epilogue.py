"""bf16 output and the residual input of the fused epilogue against the oracle.

y = act(scale * conv(x) + bias' + r): the residual joins after the folded BN and before the
clamp (the oracle's residual stage).  With bf16 output the kernel rounds its fp32 result to
nearest-even bf16, so the bound is the fp32 parity tolerance plus one bf16 unit in the last
place of the reference (a value within the fp32 tolerance of a rounding midpoint may round
either way).  Residuals handed to a bf16 handle are bf16 and the oracle sees exactly those
values.
"""
import numpy as np
import pytest
import torch

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300.workloads import ConvSpec, ACT_NONE, ACT_RELU, ACT_RELU6

from parity import ATOL, RTOL, compare, inputs_for, to_device_nhwc

import oracle

pytestmark = pytest.mark.gpu
V = cf


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cf.load_library(build_if_missing=True)


def S(name, N, C, H, W, K, R, S_, stride=(1, 1), pads=(0, 0, 0, 0), act=ACT_RELU, bias=False, bn=True):
    return ConvSpec(name, N, C, H, W, K, R, S_, stride, pads, act=act, has_bias=bias, has_bn=bn)


def ulp_bf16(v):
    """Unit in the last place of bf16 (8 significant bits) at |v| (normal range)."""
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def check_bf16(y, ref):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    allow = ATOL + RTOL * np.abs(ref) + ulp_bf16(ref)
    ratio = np.abs(y - ref) / allow
    idx = int(np.argmax(ratio))
    return bool(ratio.reshape(-1)[idx] <= 1.0), float(ratio.reshape(-1)[idx]), idx


def build(spec, inp, out_bf16, residual, **kw):
    scale, shift = (cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5) if inp["bn"] is not None
                    else (None, None))
    return cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"], scale, shift,
                        stride=spec.stride, pads=spec.pads, act=spec.act,
                        variant=V.CONVF_VARIANT_GEMM_1X1 if spec.R == 1 else V.CONVF_VARIANT_IMPLICIT_GEMM,
                        out_bf16=out_bf16, residual=residual, **kw)


def residual_for(conv, seed, out_bf16):
    """Seeded residual of y's shape: NCHW CPU tensor (bf16-rounded when y is bf16)."""
    N, K, Ho, Wo = conv.out_shape
    g = torch.Generator().manual_seed(seed)
    r = torch.randn((N, K, Ho, Wo), generator=g)
    return r.to(torch.bfloat16) if out_bf16 else r


def oracle_ref(spec, inp, r):
    bn = None if inp["bn"] is None else tuple(t.numpy() for t in inp["bn"])
    return oracle.conv_bn_act(inp["x"].double().numpy(), inp["w"].double().numpy(),
                              None if inp["bias"] is None else inp["bias"].numpy(), bn, spec.act, 0.0, 6.0,
                              spec.stride, spec.pads, spec.dilation, spec.group,
                              residual=None if r is None else r.double().numpy())


def check(y, ref, out_bf16):
    got = y.cpu().float().contiguous().numpy() if out_bf16 else y.cpu().contiguous().numpy()
    return check_bf16(got, ref) if out_bf16 else compare(got, ref, False)


CASES = [
    # (spec, bf16 output, residual, extra options)
    (S("res_1x1_c256_f32", 2, 256, 14, 15, 128, 1, 1), False, True, {}),
    (S("bf16out_3x3_c64", 2, 64, 12, 12, 96, 3, 3, pads=(1, 1, 1, 1), act=ACT_RELU6, bias=True), True, False, {}),
    (S("res_bf16_3x3_s2_k200", 2, 128, 15, 15, 200, 3, 3, (2, 2), (1, 1, 1, 1)), True, True, {}),
    # K % 8 == 4: bf16 rows are not 16-byte aligned, the 4-channel (8-byte) store path serves them
    (S("res_bf16_k100_8byte_rows", 2, 64, 9, 10, 100, 1, 1), True, True, {}),
    # more than 8 tiles per CTA: the epilogue groups take alternate tiles
    (S("res_bf16_1x1_many_tiles", 4, 128, 56, 57, 256, 1, 1), True, True, {"tile_n": 64}),
    (S("res_f32_stream_k", 2, 256, 14, 14, 256, 3, 3, pads=(1, 1, 1, 1)), False, True, {"stream_k": 2}),
    (S("res_bf16_cta_pair", 2, 128, 12, 12, 128, 3, 3, pads=(1, 1, 1, 1)), True, True, {"cta_pair": 2}),
    (S("bf16out_tile128_k256", 2, 128, 12, 12, 256, 3, 3, pads=(1, 1, 1, 1)), True, False, {"tile_n": 128}),
    # the residual staged in shared memory by TMA: 128-wide tiles, ragged M, two tiles on some
    # CTAs (both residual buffers), K a multiple of 8 but not of 64 (zero-filled box columns)
    (S("res_bf16_staged_tile128", 4, 64, 56, 57, 264, 1, 1), True, True, {"tile_n": 128}),
    (S("res_bf16_staged_3x3_k72", 3, 64, 17, 19, 72, 3, 3, pads=(1, 1, 1, 1)), True, True, {"tile_n": 64}),
]

# handles whose bf16 residual is staged in shared memory (single CTAs, whole 64/128-wide tiles)
STAGED = {"res_bf16_1x1_many_tiles", "res_bf16_staged_tile128", "res_bf16_staged_3x3_k72"}


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0].name)
def test_epilogue_options_every_output(case):
    spec, out_bf16, residual, kw = case
    seed = 8100 + CASES.index(case)
    inp = inputs_for(spec, seed)
    conv = build(spec, inp, out_bf16, residual, **kw)
    d = conv.describe()
    assert f"out={'bf16' if out_bf16 else 'f32'} residual={int(residual)}" in d, d
    assert f"residual_staged={int(spec.name in STAGED)}" in d, d
    r = residual_for(conv, seed + 1, out_bf16) if residual else None
    ref = oracle_ref(spec, inp, r)
    x = to_device_nhwc(inp["x"])
    rd = to_device_nhwc(r) if residual else None
    for _ in range(2):
        y = conv(x, r=rd)
        torch.cuda.synchronize()
        assert conv.status() == cf.CONVF_OK
        assert y.dtype == (torch.bfloat16 if out_bf16 else torch.float32)
        ok, worst, idx = check(y, ref, out_bf16)
        assert ok, (spec.name, worst, idx, d)
    conv.close()


def test_residual_may_be_the_output_buffer():
    """In place: y starts as the residual; every element is read before it is written."""
    spec = S("res_inplace", 2, 64, 10, 11, 128, 3, 3, pads=(1, 1, 1, 1))
    inp = inputs_for(spec, 8190)
    for out_bf16 in (False, True):
        conv = build(spec, inp, out_bf16, True)
        r = residual_for(conv, 8191, out_bf16)
        y = to_device_nhwc(r)
        conv(to_device_nhwc(inp["x"]), y=y, r=y)
        torch.cuda.synchronize()
        assert conv.status() == cf.CONVF_OK
        ok, worst, idx = check(y, oracle_ref(spec, inp, r), out_bf16)
        assert ok, (out_bf16, worst, idx)
        conv.close()


def test_run_entry_points_match_the_handle():
    spec = S("res_refusals", 1, 64, 8, 8, 64, 1, 1)
    inp = inputs_for(spec, 8192)
    x = to_device_nhwc(inp["x"])
    plain = build(spec, inp, False, False)
    y = plain.new_output()
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run_residual(plain.handle, x, y, y)
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "without a residual" in str(e.value)
    res = build(spec, inp, False, True)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run(res.handle, x, y)
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "conv_fused_run_residual" in str(e.value)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run_residual(res.handle, x, 0, y)
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "NULL" in str(e.value)
    big = torch.empty(2 * y.numel() + 64, dtype=torch.float32, device="cuda")
    with pytest.raises(cf.ConvFusedError) as e:   # r starts 16 bytes into y
        cf.conv_fused_run_residual(res.handle, x, big.data_ptr() + 16, big.data_ptr())
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "overlaps y" in str(e.value)
    plain.close()
    res.close()


def E(name, N, C, H, W, K, R, S_, stride=(1, 1), pads=(0, 0, 0, 0), dil=(1, 1), group=1, act=ACT_RELU, bias=False):
    return ConvSpec(name, N, C, H, W, K, R, S_, stride, pads, dil, group, act, bias, True, "bf16", "normal")


EXT_KERNELS = [
    # (spec, forced variant): the halo tiles (stride-1 3x3: the 56x56 ResNet layers), the TMA
    # depthwise (3x3, strides 1 and 2, several images per tile) and the direct depthwise (5x5 dilated)
    (E("halo_w56", 2, 64, 8, 56, 64, 3, 3, pads=(1, 1, 1, 1)), V.CONVF_VARIANT_IMPLICIT_GEMM_HALO),
    (E("halo_c128_k200", 2, 128, 14, 14, 200, 3, 3, pads=(1, 1, 1, 1), bias=True), V.CONVF_VARIANT_IMPLICIT_GEMM_HALO),
    (E("dw_s1_c96", 2, 96, 15, 17, 96, 3, 3, pads=(1, 1, 1, 1), group=96, act=ACT_RELU6),
     V.CONVF_VARIANT_DEPTHWISE),
    (E("dw_s2_c64", 2, 64, 17, 16, 64, 3, 3, (2, 2), (1, 1, 1, 1), group=64, act=ACT_RELU6),
     V.CONVF_VARIANT_DEPTHWISE),
    (E("dw_narrow_c96", 5, 96, 7, 7, 96, 3, 3, pads=(1, 1, 1, 1), group=96), V.CONVF_VARIANT_DEPTHWISE),
    # stride 1 on 16-column tiles (a 48-wide image) and on 32-column pairs with an odd width
    (E("dw_s1_w48_c64", 2, 64, 9, 48, 64, 3, 3, pads=(1, 1, 1, 1), group=64, act=ACT_RELU6),
     V.CONVF_VARIANT_DEPTHWISE),
    (E("dw_s1_w27_c40", 2, 40, 11, 27, 40, 3, 3, pads=(1, 1, 1, 1), group=40), V.CONVF_VARIANT_DEPTHWISE),
    (E("dw_5x5_dil2_c32", 2, 32, 13, 13, 32, 5, 5, (1, 1), (4, 4, 4, 4), (2, 2), group=32, act=ACT_NONE),
     V.CONVF_VARIANT_DEPTHWISE),
]


@pytest.mark.parametrize("mode", [(True, False), (False, True), (True, True)], ids=["bf16", "res", "bf16_res"])
@pytest.mark.parametrize("case", EXT_KERNELS, ids=lambda c: c[0].name)
def test_halo_and_depthwise_extended_epilogue(case, mode):
    spec, variant = case
    out_bf16, residual = mode
    seed = 8300 + EXT_KERNELS.index(case)
    inp = inputs_for(spec, seed)
    scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5)
    conv = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"], scale, shift,
                        stride=spec.stride, pads=spec.pads, dilation=spec.dilation, group=spec.group, act=spec.act,
                        variant=variant, out_bf16=out_bf16, residual=residual)
    assert conv.variant == variant, conv.describe()
    r = residual_for(conv, seed + 1, out_bf16) if residual else None
    ref = oracle_ref(spec, inp, r)
    x = to_device_nhwc(inp["x"])
    for in_place in ((False, True) if residual else (False,)):
        rd = to_device_nhwc(r) if residual else None
        y = rd if in_place else None        # in place: y starts as the residual
        y = conv(x, y, r=rd)
        torch.cuda.synchronize()
        assert conv.status() == cf.CONVF_OK
        assert y.dtype == (torch.bfloat16 if out_bf16 else torch.float32)
        ok, worst, idx = check(y, ref, out_bf16)
        assert ok, (spec.name, mode, in_place, worst, idx)
    conv.close()
