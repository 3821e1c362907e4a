"""CPU oracle for the fused ONNX Conv path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library and never imports
it; the CUDA library never imports this.

Every function is the plain definition of one stage, kept separate on purpose:

``conv2d`` / ``conv2d_points``
    ONNX Conv (public operator specification: NCHW input X[N][C][H][W], weight
    W[K][C/group][R][S], optional bias B[K], attributes strides, pads in the
    order [x1_begin, x2_begin, x1_end, x2_end], dilations, group, auto_pad).
    The seven loops run in C (``conv_oracle.c``) in double precision.
``batchnorm``
    ONNX BatchNormalization, inference form
    ``(z - mean) / sqrt(var + eps) * gamma + beta``.  The pages fold this into
    the conv weights offline ("tensorforge", section "ResNet fusion":
    W' = scale * W, bias = shift); here it stays a separate stage so that the
    library's fold is checked, not assumed.
``residual_add``
    The skip connection of a residual block, r added element-wise to the conv +
    BN result before the activation, as in the single fused conv, residual,
    bias and ReLU operation the "Kyanite" README lists (section "Cuda
    Executor").  Where it sits relative to BN is not stated there; here it
    follows the folded BN affine (the bottleneck's shortcut joins after the
    block's last BN), a reading.
``round_bf16`` / ``preactivation``
    The pre-activation of a ResNet-v2 block ("tensorforge", section "ResNet
    fusion": the remaining BN -> ReLU pairs): per input channel
    u = act(x * scale + shift) (a BatchNorm folded to its affine, then the
    activation), applied to the conv's input before its zero padding.  The
    conv consumes u as its operand, so u is stored in the operand type:
    rounded to bf16 to nearest-even (a reading; the affine is evaluated in
    float32 first, as the storage of x, scale and shift is float32/bf16).
``inverted_residual``
    A MobileNetV2 block composed from the stages above: expand 1x1 + BN + ReLU6,
    depthwise 3x3 + BN + ReLU6, project 1x1 + BN, and the skip connection for
    stride-1 blocks with equal channel counts (checked against torch).
``activation``
    ReLU = max(u, 0); ReLU6 = min(max(u, 0), 6), the two clamps of the
    residual + batchnorm + relu6 example kernel in the "Kyanite" README
    (section "Cuda Executor"); Clip(lo, hi) generally.
``qlinear_conv_acc`` / ``qlinear_requant``
    ONNX QLinearConv (public operator specification): uint8 or int8 x and w
    with zero points (w's per output channel), integer sums of the corrected
    operands ``sum (x - x_zp)(w - w_zp[k]) + B[k]`` (the quantized input pads
    with its zero point, so padded taps add nothing), then
    ``y = saturate(round_half_even(acc * x_scale * w_scale[k] / y_scale) + y_zp)``.
    The specification fixes no precision for this product; it is taken in the
    GPU kernel's precision (a reading): one per-channel multiplier
    ``m[k] = float32(x_scale * w_scale[k] / y_scale)`` (the quotient formed in
    float64 on the float32 scales, rounded once), then
    ``round_half_even(float32(acc) * m[k])`` with both the int->float conversion
    and the product rounded to nearest-even float32.  The oracle subtracts the zero
    points before multiplying; the expanded form of the same sums is the
    zero-point correction identity the "onnx-vulkan-rs" page gives, in its notes
    on the quantized kernels, for blocks of four products (the tests check one
    against the other).
``conv2d_s8`` / ``requant_s8``
    The static-int8 path ("onnx-vulkan-rs", feature list: static int8
    convolutions on the tensor cores; ConvInteger via im2col): exact integer
    sums, then the fixed-point requantisation
    ``q = (v * M + 2**(sh - 1)) >> sh`` (a reading: the pages fix no rounding
    rule), output zero point, clamp, optional ReLU at the zero point.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(brute force, closed forms, library routines on tiny cases, the BN-fold
invariant, hand-computed requant cases and golden fixtures).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

_LIB = None

ACT_NONE, ACT_RELU, ACT_RELU6, ACT_CLIP = 0, 1, 2, 3


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        i8p = ctypes.POINTER(ctypes.c_int8)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        ints = [ctypes.c_int] * 16
        lib.oracle_conv2d_f64.argtypes = [dp, dp, dp] + ints + [dp]
        lib.oracle_conv2d_f64_points.argtypes = [dp, dp, dp] + ints + [i64p, ctypes.c_int64, dp]
        lib.oracle_conv2d_s8.argtypes = [i8p, i8p] + ints + [i64p]
        lib.oracle_conv2d_s8_points.argtypes = [i8p, i8p] + ints + [i64p, ctypes.c_int64, i64p]
        lib.oracle_requant_s8.argtypes = [i64p, i64p, ctypes.c_int64, i32p, i32p, i32p,
                                          ctypes.c_int32, ctypes.c_int, i8p]
        lib.oracle_conv2d_f32acc.argtypes = [fp, fp, fp] + ints + [fp]
        i16p = ctypes.POINTER(ctypes.c_int16)
        lib.oracle_conv2d_i16.argtypes = [i16p, i16p] + ints + [i64p]
        lib.oracle_conv2d_i16.restype = ctypes.c_int
        lib.oracle_out_extent.argtypes = [ctypes.c_long] * 6
        lib.oracle_out_extent.restype = ctypes.c_long
        lib.oracle_num_threads.restype = ctypes.c_int
        for f in ("oracle_conv2d_f64", "oracle_conv2d_f64_points", "oracle_conv2d_s8",
                  "oracle_conv2d_s8_points", "oracle_requant_s8", "oracle_conv2d_f32acc"):
            getattr(lib, f).restype = ctypes.c_int
        _LIB = lib
    return _LIB


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use (1 when built without OpenMP)."""
    return int(_lib().oracle_num_threads())


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# ----------------------------------------------------------------- attributes

def resolve_pads(H, W, R, S, strides=(1, 1), dilations=(1, 1), pads=(0, 0, 0, 0),
                 auto_pad="NOTSET"):
    """Explicit pads (top, left, bottom, right) per the ONNX Conv auto_pad rule.

    NOTSET keeps ``pads`` (ONNX order h_begin, w_begin, h_end, w_end).  VALID
    means no padding.  SAME_UPPER / SAME_LOWER pad so that the output extent is
    ceil(in / stride); an odd total puts the extra element at the end (UPPER)
    or at the beginning (LOWER).
    """
    if auto_pad in ("NOTSET", None, ""):
        return tuple(int(p) for p in pads)
    if auto_pad == "VALID":
        return (0, 0, 0, 0)
    begins, ends = [], []
    for n_in, k, st, d in ((H, R, strides[0], dilations[0]), (W, S, strides[1], dilations[1])):
        out = -(-n_in // st)
        total = max(0, (out - 1) * st + (k - 1) * d + 1 - n_in)
        small = total // 2
        if auto_pad == "SAME_UPPER":
            begins.append(small)
            ends.append(total - small)
        elif auto_pad == "SAME_LOWER":
            begins.append(total - small)
            ends.append(small)
        else:
            raise ValueError(f"unknown auto_pad {auto_pad!r}")
    return (begins[0], begins[1], ends[0], ends[1])


def out_hw(H, W, R, S, strides, pads, dilations):
    """(Ho, Wo) from the ONNX Conv output-shape rule with explicit pads."""
    lib = _lib()
    pt, pl, pb, pr = pads
    ho = lib.oracle_out_extent(H, R, strides[0], pt, pb, dilations[0])
    wo = lib.oracle_out_extent(W, S, strides[1], pl, pr, dilations[1])
    return int(ho), int(wo)


def _dims(x_shape, w_shape, strides, pads, dilations, group):
    N, C, H, W = (int(v) for v in x_shape)
    K, Cg, R, S = (int(v) for v in w_shape)
    if Cg * group != C:
        raise ValueError(f"weight has C/group={Cg} but input has C={C}, group={group}")
    return [N, C, H, W, K, R, S, int(strides[0]), int(strides[1]), int(pads[0]), int(pads[1]),
            int(pads[2]), int(pads[3]), int(dilations[0]), int(dilations[1]), int(group)]


# ----------------------------------------------------------------- float conv

def conv2d(x, w, bias=None, strides=(1, 1), pads=(0, 0, 0, 0), dilations=(1, 1), group=1):
    """ONNX Conv in double precision: returns z[N][K][Ho][Wo] (float64).

    ``x`` and ``w`` are converted to float64 exactly (bf16/fp32 values are
    representable), so the oracle sees the identical rounded inputs.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    dims = _dims(x.shape, w.shape, strides, pads, dilations, group)
    Ho, Wo = out_hw(dims[2], dims[3], dims[5], dims[6], strides, pads, dilations)
    if Ho < 1 or Wo < 1:
        raise ValueError("empty output")
    z = np.empty((dims[0], dims[4], Ho, Wo), dtype=np.float64)
    rc = _lib().oracle_conv2d_f64(_ptr(x, ctypes.c_double), _ptr(w, ctypes.c_double),
                                  None if b is None else _ptr(b, ctypes.c_double),
                                  *dims, _ptr(z, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_conv2d_f64 rejected its arguments")
    return z


def conv2d_points(x, w, bias, strides, pads, dilations, group, pts):
    """Selected outputs z[n, k, oh, ow] for each row (n, k, oh, ow) of ``pts``."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
    dims = _dims(x.shape, w.shape, strides, pads, dilations, group)
    out = np.empty(pts.shape[0], dtype=np.float64)
    rc = _lib().oracle_conv2d_f64_points(_ptr(x, ctypes.c_double), _ptr(w, ctypes.c_double),
                                         None if b is None else _ptr(b, ctypes.c_double),
                                         *dims, _ptr(pts, ctypes.c_int64), pts.shape[0],
                                         _ptr(out, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle_conv2d_f64_points rejected its arguments")
    return out


def conv2d_f32acc(x, w, bias=None, strides=(1, 1), pads=(0, 0, 0, 0), dilations=(1, 1),
                  group=1):
    """Same loops with a float32 accumulator (tolerance-attainability check only)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    dims = _dims(x.shape, w.shape, strides, pads, dilations, group)
    Ho, Wo = out_hw(dims[2], dims[3], dims[5], dims[6], strides, pads, dilations)
    z = np.empty((dims[0], dims[4], Ho, Wo), dtype=np.float32)
    rc = _lib().oracle_conv2d_f32acc(_ptr(x, ctypes.c_float), _ptr(w, ctypes.c_float),
                                     None if b is None else _ptr(b, ctypes.c_float),
                                     *dims, _ptr(z, ctypes.c_float))
    if rc != 0:
        raise ValueError("oracle_conv2d_f32acc rejected its arguments")
    return z


# ------------------------------------------------------- BN and activation

def batchnorm(z, gamma, beta, mean, var, eps=1e-5, chan=None):
    """ONNX BatchNormalization (inference): (z - mean)/sqrt(var + eps)*gamma + beta.

    ``z`` is NCHW (channel axis 1) unless ``chan`` gives the channel index of
    each element of a flat ``z``.
    """
    z = np.asarray(z, dtype=np.float64)
    g, b, m, v = (np.asarray(a, dtype=np.float64) for a in (gamma, beta, mean, var))
    if chan is not None:
        chan = np.asarray(chan)
        return (z - m[chan]) / np.sqrt(v[chan] + eps) * g[chan] + b[chan]
    shp = (1, -1) + (1,) * (z.ndim - 2)
    return ((z - m.reshape(shp)) / np.sqrt(v.reshape(shp) + eps) * g.reshape(shp)
            + b.reshape(shp))


def residual_add(u, r):
    """u + r element-wise, in float64 (the residual stage; see the module docstring)."""
    return np.asarray(u, dtype=np.float64) + np.asarray(r, dtype=np.float64)


def round_bf16(a):
    """float32 values -> the nearest bf16 values (ties to even), returned as float64.

    A bf16 value is the top 16 bits of a float32: add half of the dropped 16-bit part's range
    (0x7FFF, plus 1 when the kept part is odd, so that ties go to the even neighbour) and drop
    those bits.  Finite inputs only."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    if not np.all(np.isfinite(f)):
        raise ValueError("round_bf16 takes finite values")
    bits = f.view(np.uint32).astype(np.uint64)
    r = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def preactivation(x, scale, shift, act=ACT_RELU, lo=0.0, hi=6.0):
    """u = round_bf16(act(float32(x * scale[c] + shift[c]))) for NCHW x (channel axis 1)."""
    x = np.asarray(x, dtype=np.float64)
    shp = (1, -1) + (1,) * (x.ndim - 2)
    s = np.asarray(scale, dtype=np.float64).reshape(shp)
    t = np.asarray(shift, dtype=np.float64).reshape(shp)
    u = (x * s + t).astype(np.float32).astype(np.float64)
    return round_bf16(activation(u, act, lo, hi))


def activation(u, act=ACT_NONE, lo=0.0, hi=6.0):
    """none: u;  ReLU: max(u, 0);  ReLU6: min(max(u, 0), 6);  Clip: min(max(u, lo), hi)."""
    u = np.asarray(u, dtype=np.float64)
    if act == ACT_NONE:
        return u.copy()
    if act == ACT_RELU:
        return np.maximum(u, 0.0)
    if act == ACT_RELU6:
        return np.minimum(np.maximum(u, 0.0), 6.0)
    if act == ACT_CLIP:
        return np.minimum(np.maximum(u, lo), hi)
    raise ValueError(f"unknown activation {act}")


# ------------------------------------------------------------------ int8 path

def conv2d_s8(x, w, strides=(1, 1), pads=(0, 0, 0, 0), dilations=(1, 1), group=1):
    """Exact integer conv sums acc[N][K][Ho][Wo] (int64), pad value 0."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    dims = _dims(x.shape, w.shape, strides, pads, dilations, group)
    Ho, Wo = out_hw(dims[2], dims[3], dims[5], dims[6], strides, pads, dilations)
    acc = np.empty((dims[0], dims[4], Ho, Wo), dtype=np.int64)
    rc = _lib().oracle_conv2d_s8(_ptr(x, ctypes.c_int8), _ptr(w, ctypes.c_int8), *dims,
                                 _ptr(acc, ctypes.c_int64))
    if rc != 0:
        raise ValueError("oracle_conv2d_s8 rejected its arguments")
    return acc


def conv2d_s8_points(x, w, strides, pads, dilations, group, pts):
    x = np.ascontiguousarray(x, dtype=np.int8)
    w = np.ascontiguousarray(w, dtype=np.int8)
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
    dims = _dims(x.shape, w.shape, strides, pads, dilations, group)
    out = np.empty(pts.shape[0], dtype=np.int64)
    rc = _lib().oracle_conv2d_s8_points(_ptr(x, ctypes.c_int8), _ptr(w, ctypes.c_int8), *dims,
                                        _ptr(pts, ctypes.c_int64), pts.shape[0],
                                        _ptr(out, ctypes.c_int64))
    if rc != 0:
        raise ValueError("oracle_conv2d_s8_points rejected its arguments")
    return out


def requant_s8(acc, chan, bias, mult, shift, zero_point=0, relu=False):
    """Fixed-point requantisation of integer sums to int8 (see module docstring).

    ``acc`` is any int array; ``chan`` gives each element's output channel
    (same shape), or is None for an NCHW ``acc`` (channel axis 1).
    """
    acc = np.asarray(acc, dtype=np.int64)
    shape = acc.shape
    if chan is None:
        K = shape[1]
        chan = np.broadcast_to(np.arange(K, dtype=np.int64).reshape((1, K) + (1,) * (acc.ndim - 2)),
                               shape)
    flat = np.ascontiguousarray(acc.reshape(-1))
    ch = np.ascontiguousarray(np.asarray(chan, dtype=np.int64).reshape(-1))
    b = np.ascontiguousarray(bias, dtype=np.int32)
    m = np.ascontiguousarray(mult, dtype=np.int32)
    s = np.ascontiguousarray(shift, dtype=np.int32)
    out = np.empty(flat.shape[0], dtype=np.int8)
    rc = _lib().oracle_requant_s8(_ptr(flat, ctypes.c_int64), _ptr(ch, ctypes.c_int64),
                                  flat.shape[0], _ptr(b, ctypes.c_int32), _ptr(m, ctypes.c_int32),
                                  _ptr(s, ctypes.c_int32), int(zero_point), int(bool(relu)),
                                  _ptr(out, ctypes.c_int8))
    if rc != 0:
        raise ValueError("oracle_requant_s8 rejected its arguments")
    return out.reshape(shape)


# ------------------------------------------------------------ QLinearConv path

def _per_channel(v, K, dtype):
    v = np.asarray(v, dtype=dtype).reshape(-1)
    if v.size == 1:
        return np.full(K, v[0], dtype=dtype)
    if v.size != K:
        raise ValueError(f"per-channel parameter has {v.size} entries for {K} output channels")
    return v


def qlinear_conv_acc(x, x_zero_point, w, w_zero_point, bias=None, strides=(1, 1), pads=(0, 0, 0, 0),
                     dilations=(1, 1), group=1):
    """Integer sums sum (x - x_zp)(w - w_zp[k]) (+ B[k]) of ONNX QLinearConv, int64 [N][K][Ho][Wo].

    x, w: uint8 or int8 arrays (NCHW, KCRS); x_zero_point a scalar; w_zero_point a scalar or one
    per output channel; bias int32[K] or None.
    """
    x = np.asarray(x)
    w = np.asarray(w)
    for a in (x, w):
        if a.dtype not in (np.uint8, np.int8):
            raise ValueError("QLinearConv operands are uint8 or int8")
    K = w.shape[0]
    # each zero point has its tensor's element type (ONNX QLinearConv type constraints)
    _check_range(x_zero_point, x.dtype, "x_zero_point")
    _check_range(w_zero_point, w.dtype, "w_zero_point")
    xd = np.ascontiguousarray(x.astype(np.int16) - np.int16(int(x_zero_point)))
    wz = _per_channel(w_zero_point, K, np.int16)
    wd = np.ascontiguousarray(w.astype(np.int16) - wz.reshape((K,) + (1,) * (w.ndim - 1)))
    dims = _dims(xd.shape, wd.shape, strides, pads, dilations, group)
    Ho, Wo = out_hw(dims[2], dims[3], dims[5], dims[6], strides, pads, dilations)
    acc = np.empty((dims[0], dims[4], Ho, Wo), dtype=np.int64)
    rc = _lib().oracle_conv2d_i16(_ptr(xd, ctypes.c_int16), _ptr(wd, ctypes.c_int16), *dims,
                                  _ptr(acc, ctypes.c_int64))
    if rc != 0:
        raise ValueError("oracle_conv2d_i16 rejected its arguments")
    if bias is not None:
        acc += np.asarray(bias, dtype=np.int64).reshape(1, K, 1, 1)
    return acc


def _check_range(v, dtype, name):
    info = np.iinfo(dtype)
    a = np.asarray(v, dtype=np.int64).reshape(-1)
    if a.size and (a.min() < info.min or a.max() > info.max):
        raise ValueError(f"{name} must lie in {np.dtype(dtype).name}'s range [{info.min}, {info.max}]")


def qlinear_multiplier(x_scale, w_scale, y_scale, K):
    """Per-channel requantisation multiplier float32(x_scale * w_scale[k] / y_scale), the quotient
    formed in float64 on the float32 scales and rounded once to float32."""
    ws = _per_channel(w_scale, K, np.float32).astype(np.float64)
    return (np.float64(np.float32(x_scale)) * ws / np.float64(np.float32(y_scale))).astype(np.float32)


def qlinear_requant(acc, x_scale, w_scale, y_scale, y_zero_point, y_dtype=np.uint8, relu=False):
    """y = saturate(round_half_even(float32(acc) * m[k]) + y_zp) for NCHW acc (module docstring:
    float32 steps, each rounded to nearest even).  y's type is y_zero_point's type.  ``relu``: a
    Relu fused after the conv, which in the quantized domain keeps the codes whose real value
    (y - y_zp) * y_scale is >= 0, i.e. raises every code below y_zp to y_zp."""
    if np.dtype(y_dtype) not in (np.dtype(np.uint8), np.dtype(np.int8)):
        raise ValueError("QLinearConv's y is uint8 or int8")
    _check_range(y_zero_point, y_dtype, "y_zero_point")
    acc = np.asarray(acc, dtype=np.int64)
    K = acc.shape[1]
    m = qlinear_multiplier(x_scale, w_scale, y_scale, K)
    p = acc.astype(np.float32) * m.reshape(1, K, 1, 1)          # float32 * float32 -> float32
    v = np.rint(p).astype(np.int64) + int(y_zero_point)
    info = np.iinfo(y_dtype)
    y = np.clip(v, info.min, info.max)
    if relu:
        y = np.maximum(y, int(y_zero_point))
    return y.astype(y_dtype)


# ------------------------------------------------------------- whole pipeline

def conv_bn_act(x, w, bias=None, bn=None, act=ACT_NONE, lo=0.0, hi=6.0, strides=(1, 1),
                pads=(0, 0, 0, 0), dilations=(1, 1), group=1, eps=1e-5, residual=None, pre=None):
    """Optional pre-activation of the input (``pre`` = (scale, shift, act): ``preactivation``),
    conv, then BN (if ``bn`` = (gamma, beta, mean, var)), then the residual (if given, NCHW of
    the output's shape), then activation."""
    if pre is not None:
        x = preactivation(x, *pre)
    z = conv2d(x, w, bias, strides, pads, dilations, group)
    if bn is not None:
        z = batchnorm(z, *bn, eps=eps)
    if residual is not None:
        z = residual_add(z, residual)
    return activation(z, act, lo, hi)


def conv_bn_act_points(x, w, bias, bn, act, strides, pads, dilations, group, pts, lo=0.0,
                       hi=6.0, eps=1e-5, residual=None):
    """The same stages evaluated at selected (n, k, oh, ow) points only (``residual``: NCHW)."""
    pts = np.ascontiguousarray(pts, dtype=np.int64).reshape(-1, 4)
    z = conv2d_points(x, w, bias, strides, pads, dilations, group, pts)
    if bn is not None:
        z = batchnorm(z, *bn, eps=eps, chan=pts[:, 1])
    if residual is not None:
        r = np.asarray(residual)
        z = residual_add(z, r[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]])
    return activation(z, act, lo, hi)


def inverted_residual(x, w_expand, bn_expand, w_dw, bn_dw, w_project, bn_project, stride=1, residual=False,
                      eps=1e-5):
    """MobileNetV2 inverted-residual block, stage by stage in float64: 1x1 expand -> BN -> ReLU6
    (skipped when ``w_expand`` is None: the t = 1 block), depthwise 3x3 (pad 1, ``stride``) ->
    BN -> ReLU6, 1x1 project -> BN (linear bottleneck, no activation), then + x when
    ``residual`` (stride 1 and equal in/out channels).  Each ``bn_*`` is (gamma, beta, mean,
    var).  The fused block of the "tensorforge" page's "ResNet fusion" direction (BN -> ReLU
    pairs folded into one kernel), applied to the whole block."""
    h = np.asarray(x, dtype=np.float64)
    if w_expand is not None:
        h = conv_bn_act(h, w_expand, None, bn_expand, ACT_RELU6, eps=eps)
    ch = h.shape[1]
    h = conv_bn_act(h, w_dw, None, bn_dw, ACT_RELU6, strides=(stride, stride), pads=(1, 1, 1, 1), group=ch, eps=eps)
    y = conv_bn_act(h, w_project, None, bn_project, ACT_NONE, eps=eps)
    if residual:
        y = residual_add(y, x)
    return y


def tolerance_ok(y, ref, atol=1e-3, rtol=1e-3):
    """Element-wise |y - ref| <= atol + rtol*|ref|; returns (ok, worst ratio, argmax)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    allow = atol + rtol * np.abs(ref)
    ratio = np.abs(y - ref) / allow
    ratio = np.where(np.isnan(ratio), np.inf, ratio)
    idx = int(np.argmax(ratio)) if ratio.size else 0
    worst = float(ratio.reshape(-1)[idx]) if ratio.size else 0.0
    return bool(worst <= 1.0), worst, idx
