"""Host-side tests of the C-ABI library (no GPU, no kernel launch): the shared library
loads and exports every entry point the header declares; validation and refusal codes;
auto_pad and output shapes; the BN affine; the selector; the weight prepack layout."""
import ctypes
import os
import re

import numpy as np
import pytest

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import _build, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return cf.load_library()


def header_functions():
    src = open(os.path.join(ROOT, "include", "conv_fused.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:convf_status|void|int|const char\*)\s+(\w+)\s*\(", src,
                                 flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(cf.EXPORTED) == names


def desc(**kw):
    base = dict(N=1, C=16, H=8, W=8, K=32, R=3, S=3, stride=(1, 1), pads=(1, 1, 1, 1))
    base.update(kw)
    return cf.make_desc(**base)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(C=0), cf.CONVF_ERR_INVALID_ARG, "C=0"),
    (dict(N=-1), cf.CONVF_ERR_INVALID_ARG, "N=-1"),
    (dict(stride=(0, 1)), cf.CONVF_ERR_INVALID_ARG, "strides"),
    (dict(dilation=(1, 0)), cf.CONVF_ERR_INVALID_ARG, "dilations"),
    (dict(pads=(-1, 0, 0, 0)), cf.CONVF_ERR_INVALID_ARG, "pads[0]"),
    (dict(group=3), cf.CONVF_ERR_INVALID_ARG, "group=3"),
    (dict(R=11, pads=(0, 0, 0, 0)), cf.CONVF_ERR_INVALID_ARG, "does not fit"),
    (dict(auto_pad=7), cf.CONVF_ERR_INVALID_ARG, "auto_pad"),
    (dict(layout=cf.CONVF_NCHW), cf.CONVF_ERR_UNSUPPORTED, "channels-last"),
    (dict(act=9), cf.CONVF_ERR_INVALID_ARG, "act=9"),
    (dict(act=cf.CONVF_ACT_CLIP, clip=(2.0, 1.0)), cf.CONVF_ERR_INVALID_ARG, "clip"),
    (dict(group=2, K=32, cta_pair=2, variant=cf.CONVF_VARIANT_IMPLICIT_GEMM), cf.CONVF_ERR_UNSUPPORTED,
     "single CTAs"),
    (dict(C=12, K=12, group=12, variant=cf.CONVF_VARIANT_DEPTHWISE), cf.CONVF_ERR_UNSUPPORTED, "C % 8"),
    (dict(K=30, variant=cf.CONVF_VARIANT_IMPLICIT_GEMM), cf.CONVF_ERR_UNSUPPORTED, "K % 4"),
    (dict(dtype=cf.CONVF_S8, C=12), cf.CONVF_ERR_UNSUPPORTED, "C % 64"),
    (dict(dtype=cf.CONVF_S8, C=64, act=cf.CONVF_ACT_RELU6), cf.CONVF_ERR_UNSUPPORTED, "int8"),
    (dict(variant=cf.CONVF_VARIANT_GEMM_1X1), cf.CONVF_ERR_UNSUPPORTED, "forced variant"),
    (dict(variant=cf.CONVF_VARIANT_DEPTHWISE), cf.CONVF_ERR_UNSUPPORTED, "group == C == K"),
    (dict(variant=11), cf.CONVF_ERR_INVALID_ARG, "variant=11"),
    (dict(cta_pair=3), cf.CONVF_ERR_INVALID_ARG, "cta_pair=3"),
    (dict(C=3, K=32, cta_pair=2), cf.CONVF_ERR_UNSUPPORTED, "single CTAs"),
    (dict(N=1 << 14, H=1 << 10, W=1 << 10), cf.CONVF_ERR_UNSUPPORTED, "2^31"),
])
def test_refusals_name_the_offender(kw, status, needle):
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_plan(desc(**kw))
    assert e.value.status == status
    assert needle in str(e.value)


def test_create_refuses_before_touching_the_gpu():
    d = desc()
    w = np.zeros((32, 16, 3, 3), np.uint16)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create(d, None)
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create(d, w, bn_scale=np.ones(32, np.float32))
    assert "together" in str(e.value)
    s8 = desc(dtype=cf.CONVF_S8, C=64)
    w8 = np.zeros((32, 64, 3, 3), np.int8)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create(s8, w8)
    assert "requant" in str(e.value)
    bad_shift = np.zeros(32, np.int32)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create(s8, w8, None, None, None, np.ones(32, np.int32), bad_shift)
    assert "requant_shift[0]" in str(e.value)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create(s8, w8, None, None, None, np.ones(32, np.int32), np.ones(32, np.int32), 300)
    assert "out_zero_point" in str(e.value)


def test_handle_checks(lib):
    assert lib.conv_fused_run(None, None, None, None) == cf.CONVF_ERR_INVALID_ARG
    assert lib.conv_fused_status(None) == cf.CONVF_ERR_INVALID_ARG
    assert lib.conv_fused_variant(None) == cf.CONVF_ERR_INVALID_ARG
    junk = (ctypes.c_uint32 * 64)()
    assert lib.conv_fused_run(ctypes.addressof(junk), None, None, None) == cf.CONVF_ERR_INVALID_ARG
    assert "not a convf handle" in cf.conv_fused_last_error()
    lib.conv_fused_destroy(None)   # no-op


@pytest.mark.parametrize("n_in,k,s,d,mode", [(5, 3, 2, 1, "SAME_UPPER"), (4, 3, 2, 1, "SAME_UPPER"),
                                              (4, 3, 2, 1, "SAME_LOWER"), (224, 7, 2, 1, "SAME_LOWER"),
                                              (6, 3, 1, 2, "SAME_UPPER"), (9, 4, 3, 1, "VALID"),
                                              (9, 4, 3, 1, "NOTSET")])
def test_auto_pad_and_output_shape(n_in, k, s, d, mode):
    dsc = cf.make_desc(2, 8, n_in, n_in + 1, 16, k, k, (s, s), (1, 0, 2, 1), (d, d), auto_pad=mode)
    pads = cf.conv_fused_resolve_pads(dsc)
    if mode.startswith("SAME"):
        total_h = max(0, (-(-n_in // s) - 1) * s + (k - 1) * d + 1 - n_in)
        small = total_h // 2
        want_h = (small, total_h - small) if mode == "SAME_UPPER" else (total_h - small, small)
        assert (pads[0], pads[2]) == want_h
    elif mode == "VALID":
        assert pads == (0, 0, 0, 0)
    else:
        assert pads == (1, 0, 2, 1)
    N, K, Ho, Wo = cf.conv_fused_output_shape(dsc)
    assert (N, K) == (2, 16)
    assert Ho == (n_in + pads[0] + pads[2] - d * (k - 1) - 1) // s + 1
    assert Wo == (n_in + 1 + pads[1] + pads[3] - d * (k - 1) - 1) // s + 1


def test_bn_scale_shift_matches_formula():
    rng = np.random.default_rng(0)
    K = 37
    g, b = rng.uniform(0.5, 1.5, K), rng.normal(0, 0.1, K)
    m, v = rng.normal(0, 0.1, K), rng.uniform(0.5, 1.5, K)
    g, b, m, v = (a.astype(np.float32) for a in (g, b, m, v))
    scale, shift = cf.conv_bn_scale_shift(g, b, m, v, 1e-5)
    s64 = g.astype(np.float64) / np.sqrt(v.astype(np.float64) + np.float64(np.float32(1e-5)))
    t64 = b.astype(np.float64) - m.astype(np.float64) * s64
    assert np.array_equal(scale, s64.astype(np.float32))
    assert np.array_equal(shift, t64.astype(np.float32))
    with pytest.raises(cf.ConvFusedError):
        cf.conv_bn_scale_shift(g, b, m, np.full(K, -1.0, np.float32), 1e-5)


def test_tile_choice_and_overrides():
    # 3x3 128->128 at 28x28, batch 32, through TMA im2col: 128-wide single-CTA tiles (the
    # measured best)
    d = cf.make_desc(32, 128, 28, 28, 128, 3, 3, (1, 1), (1, 1, 1, 1), variant=cf.CONVF_VARIANT_IMPLICIT_GEMM)
    v, bn, kt, pair = cf.conv_fused_plan(d, with_pair=True)
    assert (v, bn, kt, pair) == (cf.CONVF_VARIANT_IMPLICIT_GEMM, 128, 1152, 0)
    d.cta_pair = 2
    assert cf.conv_fused_plan(d, with_pair=True)[3] == 1
    d.tile_n = 64
    assert cf.conv_fused_plan(d, with_pair=True)[1] == 64


def test_selector_on_the_workloads():
    names = {}
    for spec in workloads.resnet50_layers(32) + workloads.mobilenetv2_layers(64) + workloads.int8_layers(64):
        d = cf.make_desc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride, spec.pads,
                         spec.dilation, spec.group, cf.CONVF_S8 if spec.dtype == "s8" else cf.CONVF_BF16)
        v, bn, kt = cf.conv_fused_plan(d)
        names[spec.name] = v
        if spec.dtype == "s8":
            # the exact-integer tcgen05 kernel: 3x3 with 64-channel runs per tap, 128- or 64-wide tiles
            assert v == cf.CONVF_VARIANT_INT8_TC and kt == 9 * spec.C and bn in (64, 128)
        elif spec.group > 1:
            assert v == cf.CONVF_VARIANT_DEPTHWISE
        elif spec.C == 3:
            # 3 channels padded to 4; one filter row of one output pixel is a run of S*4
            # elements, padded to a 16/32/64-element window: 7 rows x 32 for the 7x7 stem
            E = 16 if spec.S * 4 <= 16 else 32 if spec.S * 4 <= 32 else 64
            assert v == cf.CONVF_VARIANT_IMPLICIT_GEMM_WINDOW and kt == spec.R * E
            assert bn == -(-spec.K // 32) * 32
        elif spec.R == 1 and spec.stride == (1, 1):
            assert v == cf.CONVF_VARIANT_GEMM_1X1 and kt == -(-spec.C // 64) * 64
        elif spec.stride == (1, 1) and spec.W == 56:
            # stride-1 3x3 on rows of 58 (2 output rows per tile) whose 64 x 576 weights stay
            # resident in shared memory
            assert v == cf.CONVF_VARIANT_IMPLICIT_GEMM_HALO and kt == spec.R * spec.S * (-(-spec.C // 64) * 64)
            assert bn == 64
        else:
            # strided; weights too large to stay resident; or 7x7 images (7 rows of 9: 38% of a
            # tile would be outputs)
            assert v == cf.CONVF_VARIANT_IMPLICIT_GEMM and kt == spec.R * spec.S * (-(-spec.C // 64) * 64)
    assert len(names) == 53 + 50 + 7


@pytest.mark.parametrize("variant,C,R,S,HW,cp", [(cf.CONVF_VARIANT_GEMM_1X1, 72, 1, 1, 9, 128),
                                                 (cf.CONVF_VARIANT_IMPLICIT_GEMM, 72, 3, 3, 9, 128),
                                                 (cf.CONVF_VARIANT_IMPLICIT_GEMM_GATHER, 3, 7, 7, 9, 3),
                                                 (cf.CONVF_VARIANT_IMPLICIT_GEMM_GATHER, 24, 3, 2, 9, 24),
                                                 # 16x16 outputs: tiles stay inside one image, rows
                                                 # staged in smem -> whole taps of 4 / 8 channels
                                                 (cf.CONVF_VARIANT_IMPLICIT_GEMM_GATHER, 3, 3, 3, 16, 4),
                                                 (cf.CONVF_VARIANT_IMPLICIT_GEMM_GATHER, 6, 3, 3, 16, 8)])
def test_weight_prepack_layout(variant, C, R, S, HW, cp):
    K = 20
    pad = (R // 2, S // 2, R // 2, S // 2)
    d = cf.make_desc(1, C, HW, HW, K, R, S, (1, 1), pad, variant=variant)
    _, _, kt = cf.conv_fused_plan(d)
    assert kt == -(-(R * S * cp) // 64) * 64
    rng = np.random.default_rng(1)
    W = rng.integers(1, 1 << 15, (K, C, R, S)).astype(np.uint16)
    out = np.full((K, kt), 7, np.uint16)
    cf.conv_fused_pack_weights(d, variant, W, out)
    want = np.zeros((K, kt), np.uint16)
    for r in range(R):
        for s in range(S):
            want[:, (r * S + s) * cp:(r * S + s) * cp + C] = W[:, :, r, s]
    assert np.array_equal(out, want)
    assert kt % 64 == 0


def test_fast_division_by_invariant_integers():
    """The depthwise kernel decodes tile indices with the round-up multiply-high method of
    Granlund and Montgomery: l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1, and
    q = (umulhi(n, m) + n) >> l for n < 2^31.  Checked against n // d at the edges of the range
    and on random pairs, with the 32-bit wrap of the device arithmetic made explicit."""
    import random
    rng = random.Random(5)
    ds = [1, 2, 3, 5, 7, 12, 30, 64, 1000, 2**16 + 1, 2**30, 2**31 - 1] + [rng.randrange(1, 2**31) for _ in range(200)]
    ns = [0, 1, 2**31 - 1, 2**31 - 2] + [rng.randrange(0, 2**31) for _ in range(200)]
    for d in ds:
        l = 0
        while (1 << l) < d:
            l += 1
        m = ((1 << 32) * ((1 << l) - d)) // d + 1
        assert 0 < m < 2**32 or (d == 1 and m == 1)
        for n in ns + [d - 1, d, d + 1, 2 * d - 1, (2**31 - 1) // d * d]:
            if not 0 <= n < 2**31:
                continue
            hi = (n * m) >> 32
            s = (hi + n) & 0xFFFFFFFF
            assert s == hi + n            # no 32-bit overflow for n < 2^31
            assert s >> l == n // d, (n, d)


@pytest.mark.parametrize("C,R,S,stride,dil,K,W,ok_or_reason", [
    (3, 7, 7, (2, 2), (1, 1), 64, 224, None),                  # the ResNet stem: windows of 32
    (3, 3, 3, (2, 2), (1, 1), 32, 224, None),                  # the MobileNet stem: windows of 16
    (8, 3, 3, (1, 1), (1, 1), 64, 64, None),                   # 8 channels: any stride
    (6, 3, 7, (2, 2), (1, 1), 64, 64, None),                   # 7 taps x 8 = 56 -> windows of 64
    (3, 3, 3, (1, 1), (1, 1), 32, 64, "multiple of 16 bytes"),  # 4 channels need an even stride
    (3, 3, 3, (2, 2), (2, 2), 32, 64, "dilation 1"),
    (3, 11, 11, (4, 4), (1, 1), 64, 224, "R*E <= 256"),        # 11 x 64 windows
    (3, 3, 3, (2, 2), (1, 1), 288, 64, "K <= 256"),
    (16, 3, 3, (2, 2), (1, 1), 32, 64, "C <= 8"),
])
def test_window_variant_rules(C, R, S, stride, dil, K, W, ok_or_reason):
    pad = (R // 2, S // 2, R // 2, S // 2)
    d = cf.make_desc(2, C, W, W, K, R, S, stride, pad, dil, variant=cf.CONVF_VARIANT_IMPLICIT_GEMM_WINDOW)
    if ok_or_reason is None:
        v, bn, kt = cf.conv_fused_plan(d)
        E = 16 if S * (4 if C <= 4 else 8) <= 16 else 32 if S * (4 if C <= 4 else 8) <= 32 else 64
        assert v == cf.CONVF_VARIANT_IMPLICIT_GEMM_WINDOW and kt == R * E and bn == -(-K // 32) * 32
    else:
        with pytest.raises(cf.ConvFusedError) as e:
            cf.conv_fused_plan(d)
        assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and ok_or_reason in str(e.value)


def test_window_variant_is_automatic_only_for_wide_outputs():
    narrow = cf.make_desc(2, 3, 30, 30, 64, 7, 7, (2, 2), (3, 3, 3, 3))     # 15 output columns
    wide = cf.make_desc(2, 3, 64, 64, 64, 7, 7, (2, 2), (3, 3, 3, 3))       # 32 output columns
    assert cf.conv_fused_plan(narrow)[0] == cf.CONVF_VARIANT_IMPLICIT_GEMM_GATHER
    assert cf.conv_fused_plan(wide)[0] == cf.CONVF_VARIANT_IMPLICIT_GEMM_WINDOW


def test_kblocks_per_step_is_validated():
    """kblocks_per_step takes 0 (auto) or 1..4; anything else is refused before any device work."""
    spec = {s.name: s for s in workloads.resnet50_layers(32)}["r50_28_s2b1_1x1a@b32"]
    for k in (0, 1, 2, 4):
        d = cf.make_desc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride, spec.pads,
                         kblocks_per_step=k)
        assert cf.conv_fused_plan(d)[0] == cf.CONVF_VARIANT_GEMM_1X1
    for k in (-1, 5, 8):
        d = cf.make_desc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride, spec.pads,
                         kblocks_per_step=k)
        with pytest.raises(cf.ConvFusedError) as e:
            cf.conv_fused_plan(d)
        assert e.value.status == cf.CONVF_ERR_INVALID_ARG and "kblocks_per_step" in str(e.value)


def test_bf16_output_and_residual_are_validated_and_routed():
    """out_dtype and residual take 0/1; with either, the TMA implicit-GEMM, 1x1, halo, depthwise
    and direct grouped kernels serve the conv and the RGB stem (window / gathered rows) is
    refused."""
    layers = {s.name: s for s in workloads.resnet50_layers(32)}

    def plan(spec, **kw):
        return cf.conv_fused_plan(cf.make_desc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S,
                                               spec.stride, spec.pads, group=spec.group, **kw))[0]

    halo = layers["r50_02_s0b0_3x3@b32"]
    assert plan(halo) == cf.CONVF_VARIANT_IMPLICIT_GEMM_HALO
    # the halo tiles and depthwise keep their layers with bf16 output and the residual
    assert plan(halo, out_dtype=cf.CONVF_OUT_BF16) == cf.CONVF_VARIANT_IMPLICIT_GEMM_HALO
    assert plan(halo, residual=1) == cf.CONVF_VARIANT_IMPLICIT_GEMM_HALO
    dw = next(iter(workloads.depthwise_layers(64)))
    assert plan(dw, out_dtype=1, residual=1) == cf.CONVF_VARIANT_DEPTHWISE
    assert plan(layers["r50_03_s0b0_1x1b@b32"], residual=1, out_dtype=1) == cf.CONVF_VARIANT_GEMM_1X1
    for kw in ({"out_dtype": 1}, {"residual": 1}):
        with pytest.raises(cf.ConvFusedError) as e:
            plan(layers["r50_00_stem7x7@b32"], **kw)
        assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and "kernels only" in str(e.value)
    for kw in ({"out_dtype": 2}, {"out_dtype": -1}, {"residual": 2}):
        with pytest.raises(cf.ConvFusedError) as e:
            plan(halo, **kw)
        assert e.value.status == cf.CONVF_ERR_INVALID_ARG


def test_stream_k_mode_is_validated():
    """stream_k takes 0 (auto: whole tiles), 1 (off) or 2 (on); anything else is refused."""
    spec = {s.name: s for s in workloads.resnet50_layers(32)}["r50_12_s1b0_3x3@b32"]   # strided: im2col
    for sk in (0, 1, 2):
        d = cf.make_desc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride, spec.pads,
                         stream_k=sk)
        assert cf.conv_fused_plan(d)[0] == cf.CONVF_VARIANT_IMPLICIT_GEMM
    for sk in (-1, 3):
        d = cf.make_desc(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, spec.stride, spec.pads,
                         stream_k=sk)
        with pytest.raises(cf.ConvFusedError) as e:
            cf.conv_fused_plan(d)
        assert e.value.status == cf.CONVF_ERR_INVALID_ARG


@pytest.mark.parametrize("W,pads,R,S,ok", [
    (56, (1, 1, 1, 1), 3, 3, None),          # rows of 58: 2 output rows per tile
    (14, (1, 1, 1, 1), 3, 3, None),          # rows of 16: 8 output rows per tile
    (30, (2, 0, 1, 3), 5, 3, None),          # asymmetric pads: rows of 33
    (127, (1, 1, 1, 1), 3, 3, "W + pl + pr <= 128"),
    (20, (1, 1, 1, 1), 1, 1, "more than one tap"),
])
def test_halo_variant_rules(W, pads, R, S, ok):
    d = cf.make_desc(2, 64, 12, W, 64, R, S, (1, 1), pads, variant=cf.CONVF_VARIANT_IMPLICIT_GEMM_HALO)
    if ok is None:
        v, bn, kt = cf.conv_fused_plan(d)
        assert v == cf.CONVF_VARIANT_IMPLICIT_GEMM_HALO and kt == R * S * 64 and bn == 64
    else:
        with pytest.raises(cf.ConvFusedError) as e:
            cf.conv_fused_plan(d)
        assert ok in str(e.value)
    strided = cf.make_desc(2, 64, 12, 20, 64, 3, 3, (2, 2), (1, 1, 1, 1), variant=cf.CONVF_VARIANT_IMPLICIT_GEMM_HALO)
    with pytest.raises(cf.ConvFusedError):
        cf.conv_fused_plan(strided)


def _qdesc(C=64, K=64, R=3, pads=(1, 1, 1, 1), **kw):
    return cf.make_desc(2, C, 8, 8, K, R, R, (1, 1), pads, dtype=cf.CONVF_Q8, **kw)


def _qparams(K, xz=128, wz=0, x_signed=0, w_signed=1, y_signed=0, yz=120, xs=0.02, ws=0.004, ys=0.5):
    q = cf.QParams()
    q.x_signed, q.w_signed, q.y_signed = x_signed, w_signed, y_signed
    q.x_zero_point, q.y_zero_point = xz, yz
    q.x_scale, q.y_scale = xs, ys
    wzs = np.full(K, wz, np.int32)
    wss = np.full(K, ws, np.float32)
    q.w_zero_point, q.w_scale = wzs.ctypes.data, wss.ctypes.data
    q.relu = 0
    return q, (wzs, wss)


def test_qlinear_create_refuses_before_any_cuda_call():
    """Every QLinearConv refusal (zero points outside their types, bad scales, shapes the
    exact-integer kernel cannot serve, the wrong entry point) happens on the host."""
    w = np.zeros((64, 64, 3, 3), np.int8)
    cases = [
        (dict(xz=300), "x_zero_point", cf.CONVF_ERR_INVALID_ARG),
        (dict(xz=-1), "x_zero_point", cf.CONVF_ERR_INVALID_ARG),
        (dict(x_signed=1, xz=128), "x_zero_point", cf.CONVF_ERR_INVALID_ARG),
        (dict(yz=-3), "y_zero_point", cf.CONVF_ERR_INVALID_ARG),
        (dict(y_signed=1, yz=200), "y_zero_point", cf.CONVF_ERR_INVALID_ARG),
        (dict(wz=130), "w_zero_point", cf.CONVF_ERR_INVALID_ARG),
        (dict(xs=0.0), "x_scale", cf.CONVF_ERR_INVALID_ARG),
        (dict(ws=-1.0), "w_scale", cf.CONVF_ERR_INVALID_ARG),
    ]
    for kw, word, status in cases:
        q, keep = _qparams(64, **kw)
        with pytest.raises(cf.ConvFusedError) as e:
            cf.conv_fused_create_qlinear(_qdesc(), w, None, q)
        assert e.value.status == status and word in str(e.value), (kw, str(e.value))
    q, keep = _qparams(64)
    for desc, word in ((_qdesc(C=12, K=64), "C % 8"), (_qdesc(K=40), "K % 16"),
                       (cf.make_desc(2, 64, 8, 8, 64, 3, 3, (1, 1), (1, 1, 1, 1), group=2, dtype=cf.CONVF_Q8),
                        "group")):
        with pytest.raises(cf.ConvFusedError) as e:
            cf.conv_fused_create_qlinear(desc, np.zeros((desc.K, desc.C // desc.group, 3, 3), np.int8), None, q)
        assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and word in str(e.value), str(e.value)
    # the plain create refuses CONVF_Q8 and the QLinearConv create refuses other dtypes
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create(_qdesc(), w)
    assert "conv_fused_create_qlinear" in str(e.value)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create_qlinear(cf.make_desc(2, 64, 8, 8, 64, 3, 3, (1, 1), (1, 1, 1, 1), dtype=cf.CONVF_S8),
                                     w, None, q)
    assert "CONVF_Q8" in str(e.value)


def test_int8_selector_prefers_the_exact_tcgen05_kernel():
    d = cf.make_desc(64, 128, 28, 28, 128, 3, 3, (1, 1), (1, 1, 1, 1), dtype=cf.CONVF_S8)
    assert cf.conv_fused_plan(d)[0] == cf.CONVF_VARIANT_INT8_TC
    d.variant = cf.CONVF_VARIANT_INT8
    assert cf.conv_fused_plan(d)[0] == cf.CONVF_VARIANT_INT8
    # K % 16 != 0: neither kernel serves it
    d = cf.make_desc(2, 64, 8, 8, 40, 3, 3, (1, 1), (1, 1, 1, 1), dtype=cf.CONVF_S8)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_plan(d)
    assert e.value.status == cf.CONVF_ERR_UNSUPPORTED and "K % 16" in str(e.value)


@pytest.mark.parametrize("C,K,group,R,variant,tile,ktot", [
    # ResNeXt-style 32 groups of 4: 32-wide tiles cover 8 groups, a 32-channel window padded to 64
    (128, 128, 32, 3, cf.CONVF_VARIANT_IMPLICIT_GEMM, 32, 9 * 64),
    # 2 groups of 128 -> 128: tiles inside one group, a 128-channel window
    (256, 256, 2, 3, cf.CONVF_VARIANT_IMPLICIT_GEMM, None, 9 * 128),
    # grouped 1x1 (ShuffleNet-like): 8 groups of 32 -> 32
    (256, 256, 8, 1, cf.CONVF_VARIANT_GEMM_1X1, None, None),
    # channel multiplier 2 on 64 channels (Cg = 1): 64x block-diagonal padding -> direct kernel
    (64, 128, 64, 3, cf.CONVF_VARIANT_GROUPED_DIRECT, 0, None),
    # 3 groups of 8 -> 4: one 32-wide tile holds all three, a 24-channel window padded to 64
    (24, 12, 3, 3, cf.CONVF_VARIANT_IMPLICIT_GEMM, 32, 9 * 64),
    # 8 groups of 3 -> 3: no power-of-two tile covers whole groups or fits in one -> direct
    (24, 24, 8, 3, cf.CONVF_VARIANT_GROUPED_DIRECT, 0, None),
])
def test_grouped_selection(C, K, group, R, variant, tile, ktot):
    d = cf.make_desc(8, C, 14, 14, K, R, R, (1, 1), (R // 2,) * 4, group=group)
    v, bn, kt = cf.conv_fused_plan(d)
    assert v == variant, (v, bn, kt)
    if tile is not None:
        assert bn == tile, bn
    if ktot is not None:
        assert kt == ktot, kt
    if variant != cf.CONVF_VARIANT_GROUPED_DIRECT:
        Kg, Cg = K // group, C // group
        assert bn % Kg == 0 or Kg % bn == 0
        assert all(((j * bn) // Kg) * Cg % 8 == 0 for j in range(-(-K // bn)))


def test_injected_host_allocation_failure_cleans_up_before_any_cuda_call():
    """The allocation-failure hook: the handle allocation is a create call's first allocation and
    comes before any CUDA call, so its failure is testable without a GPU.  The call returns
    CONVF_ERR_OOM, says the failure was injected, leaves no handle behind, and the hook disarms."""
    live = cf.conv_fused_debug_live_handles()
    w = np.zeros((32, 16, 3, 3), np.uint16)
    cf.conv_fused_debug_fail_alloc(1)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create(desc(), w)
    assert e.value.status == cf.CONVF_ERR_OOM and str(e.value).endswith("(injected)")
    assert cf.conv_fused_debug_live_handles() == live
    # the same for the other create calls: pre-activation and the fused block
    cf.conv_fused_debug_fail_alloc(1)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create_preact(desc(), w, pre_scale=np.ones(16, np.float32), pre_shift=np.zeros(16, np.float32))
    assert e.value.status == cf.CONVF_ERR_OOM and "(injected)" in str(e.value)
    bd = cf.BlockDesc()
    bd.N, bd.H, bd.W, bd.Cin, bd.Ch, bd.Cout, bd.stride, bd.expand, bd.residual = 1, 8, 8, 16, 96, 16, 1, 1, 1
    ones = np.ones(96, np.float32)
    cf.conv_fused_debug_fail_alloc(1)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_create_mbv2_block(bd, np.zeros((96, 16), np.uint16), ones, ones, np.zeros((96, 9), np.uint16),
                                        ones, ones, np.zeros((16, 96), np.uint16), ones[:16], ones[:16])
    assert e.value.status == cf.CONVF_ERR_OOM and "(injected)" in str(e.value)
    assert cf.conv_fused_debug_live_handles() == live
    # disarmed: the next failure (if any: no GPU here) is not an injected one
    try:
        h = cf.conv_fused_create(desc(), w)
    except cf.ConvFusedError as err:
        assert "(injected)" not in str(err)
    else:
        cf.conv_fused_destroy(h)
    # a countdown past the first allocation does not fire on it; 0 disarms; negatives are refused
    cf.conv_fused_debug_fail_alloc(5)
    cf.conv_fused_debug_fail_alloc(0)
    with pytest.raises(cf.ConvFusedError) as e:
        cf.conv_fused_debug_fail_alloc(-1)
    assert e.value.status == cf.CONVF_ERR_INVALID_ARG
