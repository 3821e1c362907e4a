"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element
on the same seeded inputs.  bf16/fp32 paths: |y - ref| <= 1e-3 + 1e-3 |ref|; int8: bit-exact.
Small cases compare every output (several tiles plus a ragged tail); the full-size workloads
(every ResNet-50, MobileNetV2 and int8 layer at the benchmark's batch sizes) compare every output
too, so the exact tile schedules, wave counts and TMA box coordinates the benchmark times are
checked, not spot-checked."""
import numpy as np
import pytest
import torch

import oracle

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import synthetic, workloads
from convolution_onnx_conv_gb300.workloads import ConvSpec, ACT_NONE, ACT_RELU, ACT_RELU6, ACT_CLIP

from parity import check_full, check_sampled, inputs_for, make_conv, oracle_full, run_gpu, to_device_nhwc

pytestmark = pytest.mark.gpu

V = cf


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cf.load_library(build_if_missing=True)


def _assert(res, spec, variant=None):
    ok, worst, idx, status, used, desc = res[:6]
    assert status == cf.CONVF_OK, (spec.name, status, desc)
    if variant is not None:
        assert used == variant, (spec.name, used, desc)
    assert ok, f"{spec.name}: worst={worst} at flat index {idx} ({desc})"


# ------------------------------------------------------------------ the single-conv config

def test_single_conv_bias_relu():
    spec = workloads.single_conv_relu()
    _assert(check_full(spec, synthetic.seed_for(1, 0)), spec)


# ------------------------------------------------------------------ small shapes, all outputs

def S(name, N, C, H, W, K, R, S_, stride=(1, 1), pads=(0, 0, 0, 0), dil=(1, 1), group=1, act=ACT_RELU,
      bias=False, bn=True, values="normal"):
    return ConvSpec(name, N, C, H, W, K, R, S_, stride, pads, dil, group, act, bias, bn, "bf16", values)


SMALL = [
    # 1x1 GEMM mode: ragged M (3 tiles), C not a multiple of 64, K not a multiple of the tile
    (S("g1x1_c72_k96", 2, 72, 13, 13, 96, 1, 1), V.CONVF_VARIANT_GEMM_1X1),
    (S("g1x1_c64_k256", 2, 64, 12, 12, 256, 1, 1, act=ACT_NONE), V.CONVF_VARIANT_GEMM_1X1),
    (S("g1x1_c16_k24", 3, 16, 11, 9, 24, 1, 1, act=ACT_RELU6, bias=True), V.CONVF_VARIANT_GEMM_1X1),
    (S("g1x1_c256_k512", 1, 256, 14, 14, 512, 1, 1), V.CONVF_VARIANT_GEMM_1X1),
    # TMA im2col
    (S("i2c_3x3_s1", 2, 64, 15, 15, 64, 3, 3, pads=(1, 1, 1, 1)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (S("i2c_3x3_s2", 2, 64, 15, 15, 128, 3, 3, (2, 2), (1, 1, 1, 1)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (S("i2c_3x3_c72_ragged", 1, 72, 10, 13, 40, 3, 3, pads=(1, 1, 1, 1), bias=True),
     V.CONVF_VARIANT_IMPLICIT_GEMM),
    (S("i2c_dil2_asym", 2, 16, 12, 11, 32, 3, 3, (1, 1), (2, 1, 0, 2), (2, 2)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (S("i2c_5x3_s2x1", 1, 8, 17, 9, 16, 5, 3, (2, 1), (2, 1, 2, 1)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (S("i2c_7x7_s2_c8", 2, 8, 23, 23, 64, 7, 7, (2, 2), (3, 3, 3, 3)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (S("i2c_1x1_s2", 2, 64, 14, 14, 128, 1, 1, (2, 2)), V.CONVF_VARIANT_IMPLICIT_GEMM),
    (S("i2c_3x3_c256_k256", 1, 256, 9, 9, 256, 3, 3, pads=(1, 1, 1, 1), act=ACT_NONE),
     V.CONVF_VARIANT_IMPLICIT_GEMM),
    # thread-gathered rows (C not a multiple of 8)
    (S("gat_stem_c3", 2, 3, 30, 30, 64, 7, 7, (2, 2), (3, 3, 3, 3)), V.CONVF_VARIANT_IMPLICIT_GEMM_GATHER),
    (S("gat_c5_3x3", 1, 5, 19, 21, 20, 3, 3, pads=(1, 1, 1, 1), bias=True), V.CONVF_VARIANT_IMPLICIT_GEMM_GATHER),
    # gathered rows assembled from input rows staged in shared memory (tiles within one image)
    (S("gat_patch_c3_7x7", 2, 3, 32, 32, 64, 7, 7, (2, 2), (3, 3, 3, 3)), V.CONVF_VARIANT_IMPLICIT_GEMM_GATHER),
    (S("gat_patch_c6_3x3", 3, 6, 16, 16, 32, 3, 3, pads=(1, 1, 1, 1), bias=True),
     V.CONVF_VARIANT_IMPLICIT_GEMM_GATHER),
    # depthwise
    (S("dw_s1_c32", 2, 32, 15, 15, 32, 3, 3, pads=(1, 1, 1, 1), group=32, act=ACT_RELU6), V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_s2_c40", 2, 40, 17, 16, 40, 3, 3, (2, 2), (1, 1, 1, 1), group=40, act=ACT_RELU6),
     V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_5x5_dil2", 1, 16, 13, 13, 16, 5, 5, (1, 1), (4, 4, 4, 4), (2, 2), group=16, act=ACT_NONE, bias=True),
     V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_3x3_s2_asym", 1, 24, 9, 12, 24, 3, 3, (2, 2), (0, 1, 1, 0), group=24), V.CONVF_VARIANT_DEPTHWISE),
    # 3x3 tiles of 7 rows x 16 columns x 32 channels: windows wider than the image and than C,
    # a half-empty last channel slab, ragged row and column blocks, pads larger than the halo
    (S("dw_s1_c8_tiny", 3, 8, 5, 6, 8, 3, 3, pads=(1, 1, 1, 1), group=8, act=ACT_NONE, bias=True),
     V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_s1_c144_ragged", 2, 144, 15, 37, 144, 3, 3, pads=(1, 1, 1, 1), group=144, act=ACT_RELU6),
     V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_s1_pad3_asym", 1, 64, 8, 9, 64, 3, 3, pads=(3, 2, 0, 3), group=64), V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_s2_c96_odd", 2, 96, 23, 31, 96, 3, 3, (2, 2), (1, 1, 1, 1), group=96, act=ACT_RELU6),
     V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_s2_pad0", 1, 32, 16, 16, 32, 3, 3, (2, 2), group=32), V.CONVF_VARIANT_DEPTHWISE),
    # outputs at most 8 columns wide: two images per tile, the last image group half past N
    (S("dw_s1_narrow_odd_n", 5, 96, 7, 7, 96, 3, 3, pads=(1, 1, 1, 1), group=96, act=ACT_RELU6),
     V.CONVF_VARIANT_DEPTHWISE),
    # stride-1 tiles of 32 column lanes: two 16-column images with an odd image count, an odd
    # width (the second column of the last pair falls outside), two column blocks with a
    # one-column tail and a ragged channel slab, tall images with a ragged last row block
    (S("dw_s1_w16_three_images", 3, 48, 16, 16, 48, 3, 3, pads=(1, 1, 1, 1), group=48, act=ACT_RELU6),
     V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_s1_w9_odd", 2, 32, 9, 9, 32, 3, 3, pads=(1, 1, 1, 1), group=32, bias=True), V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_s1_w61_c40", 1, 40, 30, 61, 40, 3, 3, pads=(1, 1, 1, 1), group=40, act=ACT_NONE),
     V.CONVF_VARIANT_DEPTHWISE),
    (S("dw_s2_narrow_odd_n", 3, 64, 13, 15, 64, 3, 3, (2, 2), (1, 1, 1, 1), group=64, bias=True),
     V.CONVF_VARIANT_DEPTHWISE),
]


@pytest.mark.parametrize("spec,variant", SMALL, ids=[s.name for s, _ in SMALL])
def test_small_shapes_full(spec, variant):
    _assert(check_full(spec, 7000 + SMALL.index((spec, variant)), variant), spec, variant)


WINDOW = [
    # one filter row of one output pixel is a contiguous window of E = 16 / 32 / 64 elements
    S("win_stem_c3_7x7_s2", 2, 3, 40, 40, 64, 7, 7, (2, 2), (3, 3, 3, 3)),
    S("win_stem_c3_two_col_blocks", 1, 3, 300, 300, 64, 7, 7, (2, 2), (3, 3, 3, 3), bias=True),
    S("win_c3_3x3_s2_relu6", 2, 3, 64, 64, 32, 3, 3, (2, 2), (1, 1, 1, 1), act=ACT_RELU6),
    S("win_c8_3x3_s1_k40", 2, 8, 40, 40, 40, 3, 3, (1, 1), (1, 1, 1, 1), bias=True),
    S("win_c5_3x7_s2_asym", 2, 5, 33, 45, 24, 3, 7, (2, 2), (1, 3, 0, 2), act=ACT_NONE),
    S("win_c4_5x5_s4_k192", 1, 4, 64, 64, 192, 5, 5, (4, 4), (2, 2, 2, 2)),
    S("win_c1_3x3_s2_nopad", 3, 1, 21, 50, 16, 3, 3, (2, 2)),
]


@pytest.mark.parametrize("spec", WINDOW, ids=lambda s: s.name)
def test_window_variant_full(spec):
    _assert(check_full(spec, 7400 + WINDOW.index(spec), V.CONVF_VARIANT_IMPLICIT_GEMM_WINDOW), spec,
            V.CONVF_VARIANT_IMPLICIT_GEMM_WINDOW)


@pytest.mark.parametrize("spec", [
    S("dw_s1_many_tiles", 16, 192, 56, 56, 192, 3, 3, pads=(1, 1, 1, 1), group=192, act=ACT_RELU6),
    S("dw_s2_many_tiles", 32, 192, 57, 57, 192, 3, 3, (2, 2), (1, 1, 1, 1), group=192, act=ACT_RELU6),
], ids=lambda s: s.name)
def test_depthwise_every_output_with_several_tiles_per_cta(spec):
    """More tiles than resident CTAs, so every CTA cycles its shared-memory stages more than once
    (the stride-2 case about four times); every output is compared."""
    _assert(check_full(spec, 7200, V.CONVF_VARIANT_DEPTHWISE), spec, V.CONVF_VARIANT_DEPTHWISE)


@pytest.mark.parametrize("variant", [V.CONVF_VARIANT_IMPLICIT_GEMM, V.CONVF_VARIANT_IMPLICIT_GEMM_GATHER])
def test_same_shape_through_both_activation_loaders(variant):
    spec = S("both_3x3", 2, 64, 12, 12, 64, 3, 3, pads=(1, 1, 1, 1), bias=True)
    _assert(check_full(spec, 7100, variant), spec, variant)


@pytest.mark.parametrize("cta_pair", [1, 2])
@pytest.mark.parametrize("tile_n", [32, 64, 128, 256])
@pytest.mark.parametrize("shape", ["3x3", "1x1", "1x1s2"])
def test_every_tile_width(tile_n, cta_pair, shape):
    """Every tile width on single CTAs and on CTA pairs (256-row tiles, half the weight tile
    per CTA); M = 578 / 300 / 98 leaves a last pair tile whose second half is partly or
    entirely past the end; K = 200 leaves a ragged last column tile."""
    if shape == "3x3":
        spec = S(f"tiles{tile_n}", 2, 64, 17, 17, 200, 3, 3, pads=(1, 1, 1, 1), bias=True)
    elif shape == "1x1":
        spec = S(f"tiles{tile_n}_1x1", 3, 72, 10, 10, 200, 1, 1, bias=True)
    else:
        spec = S(f"tiles{tile_n}_1x1s2", 2, 64, 14, 14, 200, 1, 1, (2, 2), bias=True)
    inp = inputs_for(spec, 7150)
    from parity import compare
    c = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                     *cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5), stride=spec.stride,
                     pads=spec.pads, act=spec.act, tile_n=tile_n, cta_pair=cta_pair,
                     variant=V.CONVF_VARIANT_GEMM_1X1 if shape == "1x1" else V.CONVF_VARIANT_IMPLICIT_GEMM)
    assert f"tile={256 if cta_pair == 2 else 128}x{tile_n} cta_pair={cta_pair - 1}" in c.describe()
    y = c(to_device_nhwc(inp["x"]))
    torch.cuda.synchronize()
    assert c.status() == cf.CONVF_OK
    ok, worst, idx = compare(y.cpu().contiguous().numpy(), oracle_full(spec, inp), False)
    c.close()
    assert ok, (worst, idx)


HALO = [
    # rows of W + pl + pr positions; one padded-input box per 64-channel block serves every tap
    S("halo_3x3_w56", 2, 64, 8, 56, 64, 3, 3, pads=(1, 1, 1, 1)),
    S("halo_3x3_c128_w28_k200", 2, 128, 28, 28, 200, 3, 3, pads=(1, 1, 1, 1), bias=True),
    S("halo_3x3_c256_w14", 3, 256, 14, 14, 256, 3, 3, pads=(1, 1, 1, 1), act=ACT_RELU6),
    S("halo_5x3_asym_pads", 2, 64, 12, 30, 64, 5, 3, pads=(2, 0, 1, 3), bias=True),
    S("halo_c8_3x3", 2, 8, 17, 20, 32, 3, 3, pads=(1, 1, 1, 1), act=ACT_NONE),
    S("halo_c72_ragged_blocks_k40", 2, 72, 9, 13, 40, 3, 3, pads=(1, 1, 1, 1), bias=True),
    S("halo_short_images", 4, 64, 5, 10, 64, 3, 3, pads=(1, 1, 1, 1)),
    S("halo_nopad_2x2", 2, 64, 9, 11, 64, 2, 2),
]


@pytest.mark.parametrize("spec", HALO, ids=lambda s: s.name)
def test_halo_variant_full(spec):
    _assert(check_full(spec, 7700 + HALO.index(spec), V.CONVF_VARIANT_IMPLICIT_GEMM_HALO), spec,
            V.CONVF_VARIANT_IMPLICIT_GEMM_HALO)


@pytest.mark.parametrize("tile_n", [64, 128, 256])
def test_halo_every_tile_width(tile_n):
    spec = S(f"halo_tiles{tile_n}", 2, 128, 14, 14, 200, 3, 3, pads=(1, 1, 1, 1), bias=True)
    inp = inputs_for(spec, 7750)
    from parity import compare
    c = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                     *cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5), stride=spec.stride,
                     pads=spec.pads, act=spec.act, tile_n=tile_n, variant=V.CONVF_VARIANT_IMPLICIT_GEMM_HALO)
    assert f"tile=128x{tile_n}" in c.describe(), c.describe()
    y = c(to_device_nhwc(inp["x"]))
    torch.cuda.synchronize()
    assert c.status() == cf.CONVF_OK
    ok, worst, idx = compare(y.cpu().contiguous().numpy(), oracle_full(spec, inp), False)
    c.close()
    assert ok, (worst, idx)


SK_CASES = [
    # 8 tiles x 36 reduction blocks over 152 CTAs: every tile split across about 19 CTAs
    S("sk_3x3_c256_many_splits", 2, 256, 14, 14, 256, 3, 3, pads=(1, 1, 1, 1), bias=True),
    # M = 300 (ragged last row tile), 8 blocks per tile
    S("sk_1x1_c512_ragged_m", 1, 512, 15, 20, 64, 1, 1),
    # 100 tiles x 2 blocks over 152 CTAs: CTAs hold a tile's tail and the next tile's head
    S("sk_1x1_tails_and_heads", 4, 128, 56, 57, 64, 1, 1, act=ACT_RELU6),
    # strided im2col, K = 200 (ragged last column tile)
    S("sk_3x3_s2_k200", 2, 128, 15, 15, 200, 3, 3, (2, 2), (1, 1, 1, 1)),
]


@pytest.mark.parametrize("tile_n", [0, 32, 128, 256])
@pytest.mark.parametrize("spec", SK_CASES, ids=lambda s: s.name)
def test_stream_k_every_output(spec, tile_n):
    """Stream-K forced on: split tiles are finished by the CTA holding their first reduction
    block from the other CTAs' fp32 partials.  Three runs on one handle: the flags that gate the
    partials must be back at zero for the next launch."""
    inp = inputs_for(spec, 7600 + SK_CASES.index(spec))
    from parity import compare
    c = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                     *cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5), stride=spec.stride,
                     pads=spec.pads, act=spec.act, tile_n=tile_n, stream_k=2,
                     variant=V.CONVF_VARIANT_GEMM_1X1 if spec.R == 1 else V.CONVF_VARIANT_IMPLICIT_GEMM)
    assert "stream_k=1" in c.describe(), c.describe()
    x = to_device_nhwc(inp["x"])
    ref = oracle_full(spec, inp)
    for _ in range(3):
        y = c(x)
        torch.cuda.synchronize()
        assert c.status() == cf.CONVF_OK
        ok, worst, idx = compare(y.cpu().contiguous().numpy(), ref, False)
        assert ok, (spec.name, worst, idx, c.describe())
    c.close()


def test_stream_k_off_matches_on():
    spec = SK_CASES[0]
    inp = inputs_for(spec, 7650)
    outs = []
    for sk in (1, 2):
        c = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                         *cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5), stride=spec.stride,
                         pads=spec.pads, act=spec.act, stream_k=sk, variant=V.CONVF_VARIANT_IMPLICIT_GEMM)
        assert f"stream_k={sk - 1}" in c.describe()
        outs.append(c(to_device_nhwc(inp["x"])).cpu())
        c.close()
    # the same partial products summed in a different order: equal within the parity tolerance
    from parity import compare
    ok, worst, idx = compare(outs[1].contiguous().numpy(), outs[0].contiguous().numpy().astype(np.float64), False)
    assert ok, (worst, idx)


KPB_CASES = [
    # (spec, tile width, k-blocks per pipeline step to run)
    (S("kpb_1x1_c256_ragged_m", 1, 256, 15, 20, 64, 1, 1), 64, [1, 2, 4]),
    (S("kpb_1x1_c192_three", 2, 192, 9, 9, 136, 1, 1, act=ACT_RELU), 128, [1, 3]),
    # C % 64 != 0: no 3-D activation box, the step's loads split between the producer warps
    (S("kpb_1x1_c96_split_loads", 2, 96, 11, 13, 64, 1, 1), 64, [2]),
    # 400 tiles over at most 152 CTAs: the stage ring wraps across tiles
    (S("kpb_1x1_many_tiles_per_cta", 4, 128, 56, 57, 256, 1, 1, act=ACT_RELU6), 64, [1, 2]),
    (S("kpb_3x3_c64_s2", 2, 64, 15, 15, 96, 3, 3, (2, 2), (1, 1, 1, 1)), 128, [1, 3]),
    (S("kpb_3x3_c128_k200", 2, 128, 12, 12, 200, 3, 3, pads=(1, 1, 1, 1), bias=True), 128, [2, 3]),
    (S("kpb_3x3_c256_four", 1, 256, 10, 10, 64, 3, 3, pads=(1, 1, 1, 1)), 64, [2, 4]),
    (S("kpb_3x3_c128_tile256", 1, 128, 10, 10, 256, 3, 3, pads=(1, 1, 1, 1)), 256, [1, 2]),
]


@pytest.mark.parametrize("case", KPB_CASES, ids=lambda c: c[0].name)
def test_kblocks_per_step_every_output(case):
    """Several k-blocks per pipeline step: one weight box (and one activation box for 1x1 with
    C % 64 == 0) per step, or activation loads shared by the two producer warps."""
    spec, tile_n, kpbs = case
    inp = inputs_for(spec, 7700 + KPB_CASES.index(case))
    from parity import compare
    ref = oracle_full(spec, inp)
    x = to_device_nhwc(inp["x"])
    for kpb in kpbs:
        c = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                         *cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5), stride=spec.stride,
                         pads=spec.pads, act=spec.act, tile_n=tile_n, kblocks_per_step=kpb,
                         variant=V.CONVF_VARIANT_GEMM_1X1 if spec.R == 1 else V.CONVF_VARIANT_IMPLICIT_GEMM)
        assert f"kblocks_per_step={kpb} " in c.describe(), c.describe()
        y = c(x)
        torch.cuda.synchronize()
        assert c.status() == cf.CONVF_OK
        ok, worst, idx = compare(y.cpu().contiguous().numpy(), ref, False)
        assert ok, (spec.name, kpb, worst, idx, c.describe())
        c.close()


PAIR_KPB_CASES = [
    # CTA pairs (256-row tiles, half the weight tile per CTA) with several k-blocks per step
    (S("pkpb_1x1_c256_ragged_m", 1, 256, 15, 21, 200, 1, 1), 64, [2, 4]),
    (S("pkpb_1x1_c256_tile256", 2, 256, 9, 9, 256, 1, 1, act=ACT_RELU), 256, [2]),
    (S("pkpb_1x1_c96_split_loads", 2, 96, 11, 13, 128, 1, 1), 128, [2]),
    (S("pkpb_3x3_c128", 2, 128, 12, 12, 256, 3, 3, pads=(1, 1, 1, 1), bias=True), 256, [2, 3]),
    (S("pkpb_3x3_s2_c128", 2, 128, 15, 15, 128, 3, 3, (2, 2), (1, 1, 1, 1)), 128, [3]),
    (S("pkpb_1x1_many_tiles_per_cta", 4, 128, 56, 57, 256, 1, 1, act=ACT_RELU6), 128, [2]),
]


@pytest.mark.parametrize("case", PAIR_KPB_CASES, ids=lambda c: c[0].name)
def test_cta_pair_kblocks_per_step_every_output(case):
    spec, tile_n, kpbs = case
    inp = inputs_for(spec, 7760 + PAIR_KPB_CASES.index(case))
    from parity import compare
    ref = oracle_full(spec, inp)
    x = to_device_nhwc(inp["x"])
    for kpb in kpbs:
        c = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                         *cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5), stride=spec.stride,
                         pads=spec.pads, act=spec.act, tile_n=tile_n, cta_pair=2, kblocks_per_step=kpb,
                         variant=V.CONVF_VARIANT_GEMM_1X1 if spec.R == 1 else V.CONVF_VARIANT_IMPLICIT_GEMM)
        d = c.describe()
        assert f"kblocks_per_step={kpb} " in d and "cta_pair=1" in d, d
        y = c(x)
        torch.cuda.synchronize()
        assert c.status() == cf.CONVF_OK
        ok, worst, idx = compare(y.cpu().contiguous().numpy(), ref, False)
        assert ok, (spec.name, kpb, worst, idx, d)
        c.close()


def test_kblocks_per_step_must_divide_blocks_and_stages():
    spec = S("kpb_refused", 1, 192, 8, 8, 64, 1, 1)
    inp = inputs_for(spec, 7790)
    for tile_n, kpb in ((64, 3), (128, 4), (64, 2)):   # 8 stages vs 3; 6 stages vs 4; 3 blocks vs 2
        with pytest.raises(cf.ConvFusedError) as e:
            cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], tile_n=tile_n,
                         kblocks_per_step=kpb, variant=V.CONVF_VARIANT_GEMM_1X1)
        assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and "must divide" in str(e.value)


def test_1x1_forced_through_im2col_and_gather():
    spec = S("one_by_one", 2, 64, 10, 10, 64, 1, 1)
    for v in (V.CONVF_VARIANT_GEMM_1X1, V.CONVF_VARIANT_IMPLICIT_GEMM, V.CONVF_VARIANT_IMPLICIT_GEMM_GATHER):
        _assert(check_full(spec, 7200, v), spec, v)


@pytest.mark.parametrize("act", [ACT_NONE, ACT_RELU, ACT_RELU6, ACT_CLIP])
def test_activations(act):
    spec = S("acts", 1, 64, 9, 9, 64, 3, 3, pads=(1, 1, 1, 1), act=act, values="uniform", bias=True, bn=False)
    inp = inputs_for(spec, 7300)
    inp["clip"] = (-0.5, 0.75)
    _assert(check_full(spec, 7300, act=act, inp=inp), spec)
    dw = S("acts_dw", 1, 64, 9, 9, 64, 3, 3, pads=(1, 1, 1, 1), group=64, act=act, values="uniform")
    inp = inputs_for(dw, 7301)
    inp["clip"] = (-0.5, 0.75)
    _assert(check_full(dw, 7301, act=act, inp=inp), dw)


def test_empty_batch_is_a_no_op():
    spec = S("empty", 0, 64, 8, 8, 64, 3, 3, pads=(1, 1, 1, 1))
    inp = inputs_for(S("e1", 1, 64, 8, 8, 64, 3, 3, pads=(1, 1, 1, 1)), 1)
    conv = make_conv(spec, inp)
    x = torch.empty((0, 64, 8, 8), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((0, 64, 8, 8), dtype=torch.float32, device="cuda")
    cf.conv_fused_run(conv.handle, 0, 0)
    cf.conv_fused_run(conv.handle, x.data_ptr(), y.data_ptr())
    torch.cuda.synchronize()
    assert conv.status() == cf.CONVF_OK
    conv.close()


def test_run_refuses_bad_pointers():
    spec = S("ptrs", 1, 64, 8, 8, 64, 3, 3, pads=(1, 1, 1, 1))
    conv = make_conv(spec, inputs_for(spec, 2))
    buf = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run(conv.handle, p + 8, p + 65536)
    assert "aligned" in str(e.value)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run(conv.handle, p, p + 4096)
    assert "overlap" in str(e.value)
    conv.close()
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run(conv.handle or 0, p, p + 65536)


# ------------------------------------------------------------------ int8, bit-exact

INT8_SMALL = [
    ConvSpec("s8_3x3_s1", 2, 64, 12, 12, 64, 3, 3, (1, 1), (1, 1, 1, 1), act=ACT_RELU, has_bias=True,
             has_bn=False, dtype="s8", values="int"),
    ConvSpec("s8_3x3_s2_k80", 2, 128, 13, 13, 80, 3, 3, (2, 2), (1, 1, 1, 1), act=ACT_RELU, has_bias=True,
             has_bn=False, dtype="s8", values="int"),
    ConvSpec("s8_1x1_noact", 3, 64, 9, 11, 144, 1, 1, act=ACT_NONE, has_bias=True, has_bn=False, dtype="s8",
             values="int"),
    ConvSpec("s8_dil2_asym", 1, 64, 11, 10, 32, 3, 3, (1, 1), (2, 0, 1, 2), (2, 2), act=ACT_RELU,
             has_bias=True, has_bn=False, dtype="s8", values="int"),
]


@pytest.mark.parametrize("spec", INT8_SMALL, ids=[s.name for s in INT8_SMALL])
def test_int8_bit_exact(spec):
    _assert(check_full(spec, 7400 + INT8_SMALL.index(spec)), spec, V.CONVF_VARIANT_INT8_TC)


def test_int8_zero_point_and_saturation():
    spec = INT8_SMALL[0]
    inp = inputs_for(spec, 7450)
    inp["zp"] = -5
    inp["mult"] = inp["mult"] * 0 + (1 << 30)   # scale 2^30 / 2^sh: many saturate at both ends
    inp["shift"] = inp["shift"] * 0 + 38
    _assert(check_full(spec, 7450, inp=inp), spec)
    ref = oracle_full(spec, inp)
    assert (ref == 127).any() and (ref == -5).any()


# ------------------------------------------------------------------ full-size workloads (every output)

# A layer whose oracle would take much longer than ~30 s on the host (above this many FLOPs) is
# compared on sampled outputs instead; every workload layer below is under it, so all of them
# are compared element by element in the launch configuration the benchmark times.
FULL_COMPARE_MAX_FLOPS = 400e9


def _full(spec, seed):
    if spec.flops > FULL_COMPARE_MAX_FLOPS:
        res = check_sampled(spec, seed, count=20000)
    else:
        res = check_full(spec, seed)
    _assert(res, spec)
    ok, worst, idx, status, used, desc = res[:6]
    # the worst |y - ref| / allowance (bf16 paths) or mismatch count (int8) over every output
    print(f"{spec.name}: {'mismatches' if spec.dtype == 's8' else 'worst ratio'}={worst:.4g} ({desc})")


@pytest.mark.parametrize("spec", workloads.bottleneck_1x1(32), ids=lambda s: s.name)
def test_bottleneck_1x1_b32(spec):
    _full(spec, synthetic.seed_for(2, workloads.bottleneck_1x1(32).index(spec)))


RESNET = workloads.resnet50_layers(32) + workloads.resnet50_layers(1)


@pytest.mark.parametrize("spec", RESNET, ids=lambda s: s.name)
def test_resnet50_layers(spec):
    _full(spec, synthetic.seed_for(3, RESNET.index(spec)))


MBV2 = workloads.mobilenetv2_layers(64) + workloads.mobilenetv2_layers(1)


@pytest.mark.parametrize("spec", MBV2, ids=lambda s: s.name)
def test_mobilenetv2_layers(spec):
    _full(spec, synthetic.seed_for(4, MBV2.index(spec)))


INT8 = workloads.int8_layers(64)


@pytest.mark.parametrize("spec", INT8, ids=lambda s: s.name)
def test_int8_layers_b64(spec):
    _full(spec, synthetic.seed_for(5, INT8.index(spec)))


# ------------------------------------------------------------------ streams, reuse, failure detection

def test_non_default_stream_after_a_producer():
    """The two-stream race class: x is produced by a kernel on a side stream, and the conv
    runs on that same stream right after it; the result must match the oracle exactly as
    when the input was copied synchronously."""
    spec = S("stream", 2, 64, 20, 20, 128, 3, 3, pads=(1, 1, 1, 1), act=ACT_NONE)
    inp = inputs_for(spec, 7500)
    conv = make_conv(spec, inp)
    ref = oracle_full(spec, inp)
    s = torch.cuda.Stream()
    src = to_device_nhwc(inp["x"])
    with torch.cuda.stream(s):
        x = torch.empty_like(src)
        torch.cuda._sleep(1000000)           # keep the stream busy so a race would show
        x.copy_(src * 1.0)
        y = conv(x)
    s.synchronize()
    from parity import compare
    ok, worst, idx = compare(y.cpu().contiguous().numpy(), ref, False)
    assert ok, worst
    conv.close()


def test_back_to_back_runs_reuse_buffers():
    spec = S("reuse", 2, 64, 14, 14, 64, 3, 3, pads=(1, 1, 1, 1))
    inp = inputs_for(spec, 7600)
    y1, st1, _, _ = run_gpu(spec, inp, runs=1)
    y5, st5, _, _ = run_gpu(spec, inp, runs=5)
    assert st1 == st5 == cf.CONVF_OK
    assert torch.equal(y1, y5)


def test_int8_mma_rate_measurement():
    tops = cf.conv_fused_measure_int8_mma_rate()
    assert 1.0 < tops < 20000.0


def test_injected_device_allocation_failure_leaves_the_library_usable():
    """The allocation-failure hook on the device allocation (a create call's second allocation):
    create returns CONVF_ERR_OOM, frees its handle and takes no device memory; the next creates
    and runs are unaffected and still match the oracle."""
    spec = S("oom_then_ok", 2, 64, 15, 15, 64, 3, 3, pads=(1, 1, 1, 1))
    inp = inputs_for(spec, 4242)
    live = cf.conv_fused_debug_live_handles()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    cf.conv_fused_debug_fail_alloc(2)
    with pytest.raises(cf.ConvFusedError) as e:
        make_conv(spec, inp)
    assert e.value.status == cf.CONVF_ERR_OOM and "cudaMalloc" in str(e.value) and "(injected)" in str(e.value)
    assert cf.conv_fused_debug_live_handles() == live
    assert torch.cuda.mem_get_info()[0] >= free0 - (2 << 20)
    # a countdown of 3: the first create (handle, device block) succeeds, the second fails at
    # its handle allocation; the first handle is unaffected
    cf.conv_fused_debug_fail_alloc(3)
    conv = make_conv(spec, inp)
    with pytest.raises(cf.ConvFusedError) as e:
        make_conv(spec, inp)
    assert e.value.status == cf.CONVF_ERR_OOM and "host allocation failed (injected)" in str(e.value)
    assert cf.conv_fused_debug_live_handles() == live + 1
    y = conv(to_device_nhwc(inp["x"]))
    torch.cuda.synchronize()
    assert conv.status() == cf.CONVF_OK
    conv.close()
    assert cf.conv_fused_debug_live_handles() == live
    ok, worst, idx = oracle.tolerance_ok(y.cpu().contiguous().numpy(), oracle_full(spec, inp))
    assert ok, (worst, idx)
    _assert(check_full(spec, 4243), spec)


def test_watchdog_gives_up_and_reports():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cf.conv_fused_watchdog_selftest(status, 2_000_000)     # ~1 ms: nobody ever arrives
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    # the context is still usable afterwards
    assert float((torch.ones(4, device="cuda") * 2).sum()) == 8.0
