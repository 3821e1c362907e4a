"""The allocation-free entry point (conv_fused_run_noalloc) against the regular handle path.

Callers that cannot allocate device memory (code running during CUDA-graph capture, inside a
device-memory budget owned by a host framework, or on a real-time path) get one entry point
that takes every buffer from them and keeps its only scratch in a fixed device array.  Here it
must give the handle path's result, within the parity tolerance, on two calls in a row (the
second call finds the scratch holding the first call's contents).  This file runs last so a
failure here leaves every other test already run; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import synthetic
from convolution_onnx_conv_gb300.workloads import ConvSpec, ACT_RELU

import oracle
from parity import ATOL, RTOL, make_conv, oracle_full, to_device_nhwc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cf.load_library(build_if_missing=True)


CASES = [
    # an RGB stem (3 channels padded to taps of 4) and an 8-channel 3x3 conv (taps of 8)
    ConvSpec("noalloc_stem", 2, 3, 32, 32, 64, 7, 7, (2, 2), (3, 3, 3, 3), act=ACT_RELU, has_bias=True,
             has_bn=True),
    ConvSpec("noalloc_c8_3x3", 2, 8, 16, 16, 40, 3, 3, (1, 1), (1, 1, 1, 1), act=ACT_RELU, has_bias=True,
             has_bn=True),
]


def _desc(spec):
    return cf.make_desc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride, spec.pads,
                        spec.dilation, spec.group, act=spec.act)


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_noalloc_matches_the_handle_path_on_two_calls(spec):
    inp = synthetic.conv_inputs(spec, 9100 + CASES.index(spec))
    # the handle path with the same kernel (the selector may prefer another one for this shape)
    conv = make_conv(spec, inp, cf.CONVF_VARIANT_IMPLICIT_GEMM_GATHER)
    assert conv.variant == cf.CONVF_VARIANT_IMPLICIT_GEMM_GATHER
    x = to_device_nhwc(inp["x"])
    y_ref = conv(x)
    torch.cuda.synchronize()
    conv.close()
    ref_handle = y_ref.cpu().contiguous().numpy().astype(np.float64)
    ref_oracle = oracle_full(spec, inp)

    # the caller's buffers: prepacked weights and the folded epilogue vectors, on the device
    desc = _desc(spec)
    _, _, ktot = cf.conv_fused_plan(desc)
    wpk = np.zeros((spec.K, ktot), np.uint16)
    cf.conv_fused_pack_weights(desc, cf.CONVF_VARIANT_IMPLICIT_GEMM_GATHER,
                               inp["w"].contiguous().view(torch.int16).numpy().view(np.uint16), wpk)
    scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5)
    bias = (scale.astype(np.float64) * inp["bias"].numpy().astype(np.float64) + shift).astype(np.float32)
    w_dev = torch.from_numpy(wpk.view(np.int16)).cuda()
    sc_dev = torch.from_numpy(scale).cuda()
    bi_dev = torch.from_numpy(bias).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty_like(y_ref)

    for _ in range(2):
        y.fill_(float("nan"))
        cf.conv_fused_run_noalloc(desc, x, w_dev, sc_dev, bi_dev, y, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        got = y.cpu().contiguous().numpy().astype(np.float64)
        # against the handle path (the same kernel's other entry point) ...
        assert np.all(np.abs(got - ref_handle) <= ATOL + RTOL * np.abs(ref_handle))
        # ... and against the CPU oracle (NCHW logical view of the channels-last result)
        ok, worst, idx = oracle.tolerance_ok(got, ref_oracle, ATOL, RTOL)
        assert ok, (spec.name, worst, idx)


def test_noalloc_refuses_what_it_cannot_serve():
    """Refusals happen before any pointer is used: NULL buffers, nothing reaches the GPU."""
    big = ConvSpec("stem_b64", 64, 3, 224, 224, 64, 7, 7, (2, 2), (3, 3, 3, 3))   # 25.7 MB padded input
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run_noalloc(_desc(big), 0, 0, 0, 0, 0)
    assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and "maximum" in str(e.value)
    wide = ConvSpec("wide", 2, 64, 16, 16, 64, 3, 3, (1, 1), (1, 1, 1, 1))
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run_noalloc(_desc(wide), 0, 0, 0, 0, 0)
    assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and "at most 8 input channels" in str(e.value)
    spec = CASES[0]
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_run_noalloc(_desc(spec), 0, 0, 0, 0, 0)
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "NULL" in str(e.value)
    # options the gathered-row kernel cannot honour are refused by name, not ignored
    for kw, word in (({"stream_k": 2}, "stream_k"), ({"kblocks_per_step": 2}, "kblocks_per_step"),
                     ({"out_dtype": cf.CONVF_OUT_BF16}, "bf16 output")):
        d = cf.make_desc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride, spec.pads,
                         spec.dilation, spec.group, act=spec.act, **kw)
        with pytest.raises(cf.ConvFusedError) as e:
            cf.conv_fused_run_noalloc(d, 0, 0, 0, 0, 0)
        assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and word in str(e.value)
