"""GPU parity of the 8-bit convolutions on the tensor cores, bit-exact against the CPU oracle.

Static int8 (fixed-point requantisation) and ONNX QLinearConv (zero points, float32
requantisation) both run on the exact-integer tcgen05 path: 8-bit values minus their zero
points are exact in bf16, every product is an integer of at most 16 bits, and the fp32
accumulator restarts every chunk of reduction blocks small enough that no partial sum exceeds
2^24, so every partial sum is an exactly represented integer; the epilogue adds the chunks in
int32.  The warp-level mma.sync int8 kernel stays as a forced variant and must agree too.
"""
import numpy as np
import pytest
import torch

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import synthetic, workloads
from convolution_onnx_conv_gb300.workloads import ConvSpec, ACT_NONE, ACT_RELU

from parity import check_full, check_qlinear, compare, inputs_for, make_conv, oracle_full, to_device_nhwc

pytestmark = pytest.mark.gpu
V = cf


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cf.load_library(build_if_missing=True)


def S8(name, N, C, H, W, K, R, S_, stride=(1, 1), pads=(0, 0, 0, 0), dil=(1, 1), act=ACT_RELU):
    return ConvSpec(name, N, C, H, W, K, R, S_, stride, pads, dil, 1, act, True, False, "s8", "int")


SMALL = [
    # one chunk (576 terms), two chunks (1152 = 1024 + 128), five chunks (4608), 1x1 matrix mode
    S8("s8tc_3x3_c64", 2, 64, 12, 12, 64, 3, 3, pads=(1, 1, 1, 1)),
    S8("s8tc_3x3_c128_two_chunks", 2, 128, 9, 9, 80, 3, 3, pads=(1, 1, 1, 1)),
    S8("s8tc_3x3_c512_five_chunks", 1, 512, 7, 7, 64, 3, 3, pads=(1, 1, 1, 1), act=ACT_NONE),
    S8("s8tc_1x1_c256", 3, 256, 9, 11, 144, 1, 1, act=ACT_NONE),
    S8("s8tc_1x1_c72_ragged", 2, 72, 7, 9, 48, 1, 1),
    S8("s8tc_3x3_s2_k200", 2, 128, 13, 13, 208, 3, 3, (2, 2), (1, 1, 1, 1)),
    S8("s8tc_dil2_asym_c24", 1, 24, 11, 10, 32, 3, 3, (1, 1), (2, 0, 1, 2), (2, 2)),
    S8("s8tc_5x5_s2_c40", 2, 40, 17, 15, 96, 5, 5, (2, 2), (2, 2, 2, 2)),
    S8("s8tc_many_tiles", 4, 64, 30, 31, 128, 3, 3, pads=(1, 1, 1, 1)),
]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_int8_tcgen05_bit_exact(spec):
    ok, worst, idx, status, used, desc = check_full(spec, 8400 + SMALL.index(spec))
    assert status == cf.CONVF_OK, desc
    assert used == V.CONVF_VARIANT_INT8_TC, desc
    assert ok, f"{spec.name}: {worst} mismatches, first at {idx} ({desc})"


@pytest.mark.parametrize("tile_n,kpb", [(64, 1), (64, 2), (128, 1), (128, 2), (128, 3)])
def test_int8_tile_widths_and_steps(tile_n, kpb):
    """Both tile widths and several reduction blocks per pipeline step (the exact chunk is a whole
    number of steps, so 3 blocks per step give chunks of 15 blocks)."""
    spec = S8("s8tc_knobs", 2, 128, 12, 12, 256, 3, 3, pads=(1, 1, 1, 1))
    inp = inputs_for(spec, 8450)
    conv = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"],
                        stride=spec.stride, pads=spec.pads, act=spec.act, requant_mult=inp["mult"],
                        requant_shift=inp["shift"], tile_n=tile_n, kblocks_per_step=kpb)
    d = conv.describe()
    assert f"tile=128x{tile_n} " in d and f"kblocks_per_step={kpb} " in d, d
    chunk = int(d.split("exact_chunk_kblocks=")[1].split()[0])
    assert chunk % kpb == 0 and chunk * 64 * 128 * 127 <= (1 << 24), d
    y = conv(to_device_nhwc(inp["x"]))
    torch.cuda.synchronize()
    assert conv.status() == cf.CONVF_OK
    ok, worst, idx = compare(y.cpu().contiguous().numpy(), oracle_full(spec, inp), True)
    conv.close()
    assert ok, (worst, idx, d)


@pytest.mark.parametrize("wval", [-127, -128])
def test_int8_exact_at_the_largest_chunk_sums(wval):
    """Every x = -128 and every w = wval: each chunk of 1024 products sums to 1024 * 128 * |wval|,
    16,646,144 or exactly 2^24, the largest magnitude the fp32 accumulator must hold exactly; the
    interior sum over 1152 taps is beyond 2^24 and right only because the chunks are added in
    int32.  The bias cancels the interior sum up to 5 and the requantisation is the identity
    (M = 2^30, sh = 30), so any error in the sum shows in the interior outputs."""
    spec = S8("s8tc_worst", 1, 128, 6, 6, 32, 3, 3, pads=(1, 1, 1, 1), act=ACT_NONE)
    interior = 1152 * 128 * abs(wval)
    inp = {"x": torch.full((1, 128, 6, 6), -128, dtype=torch.int8),
           "w": torch.full((32, 128, 3, 3), wval, dtype=torch.int8),
           "bias": torch.full((32,), -interior + 5, dtype=torch.int32),
           "mult": torch.full((32,), 1 << 30, dtype=torch.int32),
           "shift": torch.full((32,), 30, dtype=torch.int32)}
    ok, worst, idx, status, used, desc = check_full(spec, 0, inp=inp)
    assert status == cf.CONVF_OK and used == V.CONVF_VARIANT_INT8_TC, desc
    assert ok, (worst, idx, desc)
    ref = oracle_full(spec, inp)
    assert (ref[:, :, 1:5, 1:5] == 5).all()


@pytest.mark.parametrize("spec", SMALL[:2] + SMALL[3:4], ids=lambda s: s.name)
def test_int8_mma_sync_variant_still_agrees(spec):
    if spec.C % 64:
        pytest.skip("the mma.sync kernel needs C % 64 == 0")
    ok, worst, idx, status, used, desc = check_full(spec, 8400 + SMALL.index(spec), V.CONVF_VARIANT_INT8)
    assert status == cf.CONVF_OK and used == V.CONVF_VARIANT_INT8, desc
    assert ok, (worst, idx, desc)


# ------------------------------------------------------------------ QLinearConv

def Q(name, N, C, H, W, K, R, S_, stride=(1, 1), pads=(0, 0, 0, 0), dil=(1, 1)):
    return ConvSpec(name, N, C, H, W, K, R, S_, stride, pads, dil, 1, ACT_NONE, True, False, "s8", "int")


QCASES = [
    # (spec, x signed, w signed, y signed, relu)
    (Q("q_3x3_u8_s8_u8", 2, 64, 12, 12, 64, 3, 3, pads=(1, 1, 1, 1)), False, True, False, False),
    (Q("q_3x3_u8_u8_s8_relu", 2, 32, 11, 13, 48, 3, 3, pads=(1, 1, 1, 1)), False, False, True, True),
    (Q("q_3x3_s8_s8_s8_s2", 2, 128, 15, 15, 96, 3, 3, (2, 2), (1, 1, 1, 1)), True, True, True, False),
    (Q("q_1x1_u8_s8_u8", 3, 256, 9, 9, 128, 1, 1), False, True, False, True),
    (Q("q_5x5_u8_u8_u8_asym", 1, 16, 14, 12, 32, 5, 5, (1, 2), (2, 1, 0, 2)), False, False, False, False),
    (Q("q_3x3_c512_u8_u8_chunks", 1, 512, 7, 7, 64, 3, 3, pads=(1, 1, 1, 1)), False, False, False, False),
]


@pytest.mark.parametrize("case", QCASES, ids=lambda c: c[0].name)
def test_qlinear_bit_exact(case):
    spec, xs, ws, ys, relu = case
    inp = synthetic.qlinear_inputs(spec, 8500 + QCASES.index(case), xs, ws, ys)
    bad, first, status, desc = check_qlinear(spec, inp, relu)
    assert status == cf.CONVF_OK and "int8_tcgen05_exact" in desc and "requant=float32" in desc, desc
    assert bad == 0, f"{spec.name}: {bad} mismatches, first at {first} ({desc})"


def test_qlinear_zero_points_matter():
    """The same operands with every zero point set to 0 give other codes (the correction is live)."""
    spec = QCASES[0][0]
    inp = synthetic.qlinear_inputs(spec, 8550, False, True, False)
    bad, _, status, _ = check_qlinear(spec, inp)
    assert status == cf.CONVF_OK and bad == 0
    from parity import oracle_qlinear
    flat = dict(inp, x_zp=0, w_zp=torch.zeros_like(inp["w_zp"]))
    assert not np.array_equal(oracle_qlinear(spec, inp), oracle_qlinear(spec, flat))


QRESNET = [ConvSpec(f"q_{s.name}", s.N, s.C, s.H, s.W, s.K, s.R, s.S, s.stride, s.pads, s.dilation, 1, ACT_NONE,
                    True, False, "s8", "int") for s in workloads.int8_layers(64)]


@pytest.mark.parametrize("spec", QRESNET, ids=lambda s: s.name)
def test_qlinear_resnet_3x3_b64_every_output(spec):
    """The seven ResNet-50 3x3 shapes at batch 64 as QLinearConv: uint8 x with a zero point near
    128, int8 w with per-channel zero points, uint8 y; every output compared."""
    inp = synthetic.qlinear_inputs(spec, 8600 + QRESNET.index(spec), False, True, False)
    bad, first, status, desc = check_qlinear(spec, inp, relu=True)
    assert status == cf.CONVF_OK, desc
    assert bad == 0, f"{spec.name}: {bad} mismatches, first at {first} ({desc})"
    print(f"{spec.name}: 0 mismatches ({desc})")
