"""GPU parity of the fused MobileNetV2 inverted-residual block (expand 1x1 + BN + ReLU6,
depthwise 3x3 + BN + ReLU6, project 1x1 + BN, + x for stride-1 blocks with equal channels, in one
kernel) against the oracle's stage-by-stage float64 composition, every output:
|y - ref| <= 1e-3 + 1e-3 |ref|."""
import numpy as np
import pytest
import torch

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import synthetic, workloads

import oracle
from parity import ATOL, RTOL, to_device_nhwc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cf.load_library(build_if_missing=True)


def run_block(name, N, Cin, H, Ch, Cout, stride, expand, residual, seed, runs=2):
    inp = synthetic.block_inputs(N, Cin, H, Ch, Cout, expand, seed)
    aff = lambda bn: cf.conv_bn_scale_shift(*[t.numpy() for t in bn], 1e-5)
    blk = cf.InvertedResidualBlock(N, Cin, H, H, Ch, Cout, stride, inp["we"], aff(inp["bn_e"]) if expand else None,
                                   inp["wd"], aff(inp["bn_d"]), inp["wp"], aff(inp["bn_p"]), residual=residual)
    assert blk.variant == cf.CONVF_VARIANT_MBV2_BLOCK
    desc = blk.describe()
    x = to_device_nhwc(inp["x"])
    for _ in range(runs):
        y = blk(x)
    torch.cuda.synchronize()
    assert blk.status() == cf.CONVF_OK, desc
    blk.close()
    t = lambda a: None if a is None else (a.double().numpy() if hasattr(a, "double") else a)
    bnn = lambda bn: None if bn is None else tuple(v.numpy() for v in bn)
    ref = oracle.inverted_residual(inp["x"].double().numpy(), t(inp["we"]), bnn(inp["bn_e"]), t(inp["wd"]),
                                   bnn(inp["bn_d"]), t(inp["wp"]), bnn(inp["bn_p"]), stride, residual)
    ok, worst, idx = oracle.tolerance_ok(y.cpu().contiguous().numpy(), ref, ATOL, RTOL)
    return ok, worst, idx, desc


SMALL = [
    # (name, N, Cin, H, Ch, Cout, stride, expand, residual): ragged tiles, both strides, two halo
    # row blocks, several hidden chunks with a ragged last one, the t = 1 block, a split project
    ("mb_s1_res_c24", 2, 24, 19, 144, 24, 1, True, True),
    ("mb_s2_c16_k24", 2, 16, 23, 96, 24, 2, True, False),
    ("mb_s1_t1_c32", 2, 32, 21, 32, 16, 1, False, False),
    ("mb_s1_c64_k96_chunks", 1, 64, 14, 384, 96, 1, True, False),
    ("mb_s2_c96_k160", 2, 96, 14, 576, 160, 2, True, False),
    ("mb_s1_c160_k320_split", 2, 160, 7, 960, 320, 1, True, False),
    ("mb_s1_res_c160", 2, 160, 9, 960, 160, 1, True, True),
    ("mb_s1_tiny", 3, 8, 5, 40, 8, 1, True, True),
    # batch 64: tall tiles (8 and 7 rows, two halo row blocks) with ragged last rows and columns
    ("mb_s1_res_ragged_b64", 64, 24, 19, 144, 24, 1, True, True),
    ("mb_s2_ragged_b64", 64, 16, 23, 96, 24, 2, True, False),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c[0])
def test_fused_block_every_output(case):
    ok, worst, idx, desc = run_block(*case, seed=9700 + SMALL.index(case))
    assert ok, f"{case[0]}: worst={worst} at {idx} ({desc})"


BLOCKS = workloads.mobilenetv2_blocks(64) + workloads.mobilenetv2_blocks(1)


@pytest.mark.parametrize("case", BLOCKS, ids=lambda c: c[0])
def test_mobilenetv2_blocks(case):
    ok, worst, idx, desc = run_block(*case, seed=synthetic.seed_for(11, BLOCKS.index(case)))
    assert ok, f"{case[0]}: worst={worst} at {idx} ({desc})"
    print(f"{case[0]}: worst ratio={worst:.4g} ({desc})")


def test_fused_block_refusals():
    d = cf.BlockDesc()
    d.N, d.H, d.W, d.Cin, d.Ch, d.Cout, d.stride, d.expand, d.residual = 1, 8, 8, 12, 48, 12, 1, 1, 0
    w = np.zeros(48 * 12, np.uint16)
    v = np.ones(48, np.float32)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create_mbv2_block(d, w, v, v, np.zeros(48 * 9, np.uint16), v, v, w, v[:12], v[:12])
    assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and "Cin % 8" in str(e.value)
    d.Cin, d.Cout, d.stride, d.residual = 16, 24, 1, 1
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create_mbv2_block(d, w, v, v, np.zeros(48 * 9, np.uint16), v, v, w, v[:24], v[:24])
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "skip connection" in str(e.value)
