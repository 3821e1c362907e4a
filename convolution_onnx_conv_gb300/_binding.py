"""ctypes binding of ``libconvfused.so`` (argument marshalling only).

The Python names are the C names; every compute step runs in the library's CUDA
kernels.  There is no fallback: if the library is missing this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import _build

# --- enums (mirror include/conv_fused.h)
CONVF_OK, CONVF_ERR_INVALID_ARG, CONVF_ERR_UNSUPPORTED, CONVF_ERR_OOM, CONVF_ERR_CUDA, \
    CONVF_ERR_TIMEOUT, CONVF_ERR_BOUNDS = 0, -1, -2, -3, -4, -5, -6
CONVF_BF16, CONVF_S8, CONVF_Q8 = 0, 1, 2
CONVF_OUT_F32, CONVF_OUT_BF16 = 0, 1
CONVF_NCHW, CONVF_NHWC = 0, 1
CONVF_ACT_NONE, CONVF_ACT_RELU, CONVF_ACT_RELU6, CONVF_ACT_CLIP = 0, 1, 2, 3
CONVF_AUTO_PAD_NOTSET, CONVF_AUTO_PAD_SAME_UPPER, CONVF_AUTO_PAD_SAME_LOWER, \
    CONVF_AUTO_PAD_VALID = 0, 1, 2, 3
CONVF_VARIANT_AUTO, CONVF_VARIANT_IMPLICIT_GEMM, CONVF_VARIANT_GEMM_1X1, CONVF_VARIANT_DEPTHWISE, \
    CONVF_VARIANT_INT8, CONVF_VARIANT_IMPLICIT_GEMM_GATHER, CONVF_VARIANT_IMPLICIT_GEMM_WINDOW, \
    CONVF_VARIANT_IMPLICIT_GEMM_HALO, CONVF_VARIANT_INT8_TC, CONVF_VARIANT_GROUPED_DIRECT, \
    CONVF_VARIANT_MBV2_BLOCK = 0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10
VARIANT_NAMES = {0: "auto", 1: "implicit_gemm_im2col", 2: "gemm_1x1", 3: "depthwise",
                 4: "int8_mma", 5: "implicit_gemm_gather", 6: "implicit_gemm_window", 7: "implicit_gemm_halo",
                 8: "int8_tcgen05_exact", 9: "grouped_direct", 10: "mbv2_block"}
AUTO_PAD = {"NOTSET": 0, "SAME_UPPER": 1, "SAME_LOWER": 2, "VALID": 3}

EXPORTED = ["conv_fused_output_shape", "conv_fused_resolve_pads", "conv_bn_scale_shift",
            "conv_fused_plan", "conv_fused_pack_weights", "conv_fused_create", "conv_fused_run",
            "conv_fused_status", "conv_fused_clear_status", "conv_fused_destroy",
            "conv_fused_variant", "conv_fused_describe", "conv_fused_last_error",
            "conv_fused_watchdog_selftest", "conv_fused_run_noalloc", "conv_fused_measure_int8_mma_rate",
            "conv_fused_run_residual", "conv_fused_create_qlinear", "conv_fused_create_preact",
            "conv_fused_create_mbv2_block", "conv_fused_debug_fail_alloc", "conv_fused_debug_live_handles",
            "conv_fused_chain_create", "conv_fused_chain_create_ex", "conv_fused_chain_run", "conv_fused_chain_status",
            "conv_fused_chain_clear_status", "conv_fused_chain_describe", "conv_fused_chain_destroy"]


class ConvDesc(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("C", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int),
                ("K", ctypes.c_int), ("R", ctypes.c_int), ("S", ctypes.c_int),
                ("stride", ctypes.c_int * 2), ("dilation", ctypes.c_int * 2),
                ("pads", ctypes.c_int * 4), ("auto_pad", ctypes.c_int), ("group", ctypes.c_int),
                ("dtype", ctypes.c_int), ("x_layout", ctypes.c_int), ("y_layout", ctypes.c_int),
                ("act", ctypes.c_int), ("clip_lo", ctypes.c_float), ("clip_hi", ctypes.c_float),
                ("variant", ctypes.c_int), ("tile_n", ctypes.c_int), ("cta_pair", ctypes.c_int),
                ("stream_k", ctypes.c_int), ("kblocks_per_step", ctypes.c_int),
                ("out_dtype", ctypes.c_int), ("residual", ctypes.c_int)]


class BlockDesc(ctypes.Structure):
    """convf_block_desc: one MobileNetV2 inverted-residual block."""
    _fields_ = [("N", ctypes.c_int), ("H", ctypes.c_int), ("W", ctypes.c_int), ("Cin", ctypes.c_int),
                ("Ch", ctypes.c_int), ("Cout", ctypes.c_int), ("stride", ctypes.c_int), ("expand", ctypes.c_int),
                ("residual", ctypes.c_int)]


class ChainStep(ctypes.Structure):
    """convf_chain_step: one conv run of a chain (handle, x, residual or NULL, y)."""
    _fields_ = [("conv", ctypes.c_void_p), ("x", ctypes.c_void_p), ("r", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class QParams(ctypes.Structure):
    """convf_qparams: ONNX QLinearConv scales and zero points (host arrays for w's)."""
    _fields_ = [("x_signed", ctypes.c_int), ("w_signed", ctypes.c_int), ("y_signed", ctypes.c_int),
                ("x_zero_point", ctypes.c_int32), ("w_zero_point", ctypes.c_void_p), ("x_scale", ctypes.c_float),
                ("w_scale", ctypes.c_void_p), ("y_scale", ctypes.c_float), ("y_zero_point", ctypes.c_int32),
                ("relu", ctypes.c_int)]


def make_desc(N, C, H, W, K, R, S, stride=(1, 1), pads=(0, 0, 0, 0), dilation=(1, 1), group=1,
              dtype=CONVF_BF16, act=CONVF_ACT_NONE, clip=(0.0, 6.0), auto_pad="NOTSET",
              variant=CONVF_VARIANT_AUTO, layout=CONVF_NHWC, tile_n=0, cta_pair=0, stream_k=0,
              kblocks_per_step=0, out_dtype=CONVF_OUT_F32, residual=0) -> ConvDesc:
    d = ConvDesc()
    d.N, d.C, d.H, d.W, d.K, d.R, d.S = N, C, H, W, K, R, S
    d.stride[:] = list(stride)
    d.dilation[:] = list(dilation)
    d.pads[:] = list(pads)
    d.auto_pad = AUTO_PAD[auto_pad] if isinstance(auto_pad, str) else int(auto_pad)
    d.group = group
    d.dtype = dtype
    d.x_layout = d.y_layout = layout
    d.act = act
    d.clip_lo, d.clip_hi = float(clip[0]), float(clip[1])
    d.variant = variant
    d.tile_n = tile_n
    d.cta_pair = cta_pair
    d.stream_k = stream_k
    d.kblocks_per_step = kblocks_per_step
    d.out_dtype = out_dtype
    d.residual = residual
    return d


class ConvFusedError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"status {status}: {msg}")
        self.status = status


_LIB = None


def _bounds_build() -> bool:
    return os.environ.get("CONVF_DEBUG_BOUNDS", "") not in ("", "0")


def library_path() -> str:
    """The library this process loads: libconvfused.so, or the bounds-checking build when the
    environment sets CONVF_DEBUG_BOUNDS=1."""
    return _build.LIB_BOUNDS if _bounds_build() else _build.LIB


def load_library(build_if_missing: bool = False):
    """Load the CUDA library (building it first only when asked)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if build_if_missing:
        _build.build(debug_bounds=_bounds_build())
    if not os.path.exists(path):
        raise ImportError(f"{os.path.basename(path)} is not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    dptr = P(ConvDesc)
    vp = ctypes.c_void_p
    lib.conv_fused_output_shape.argtypes = [dptr, P(ctypes.c_int)]
    lib.conv_fused_resolve_pads.argtypes = [dptr, P(ctypes.c_int)]
    lib.conv_bn_scale_shift.argtypes = [ctypes.c_int] + [P(ctypes.c_float)] * 4 + [ctypes.c_float] + \
        [P(ctypes.c_float)] * 2
    lib.conv_fused_plan.argtypes = [dptr, ctypes.c_int, P(ctypes.c_int), P(ctypes.c_int), P(ctypes.c_int),
                                    P(ctypes.c_int)]
    lib.conv_fused_pack_weights.argtypes = [dptr, ctypes.c_int, vp, vp, ctypes.c_size_t]
    lib.conv_fused_create.argtypes = [dptr, vp, vp, vp, vp, vp, vp, ctypes.c_int32, P(vp)]
    lib.conv_fused_create_qlinear.argtypes = [dptr, vp, vp, P(QParams), P(vp)]
    lib.conv_fused_create_preact.argtypes = [dptr, vp, vp, vp, vp, vp, vp, ctypes.c_int, P(vp)]
    lib.conv_fused_create_mbv2_block.argtypes = [P(BlockDesc)] + [vp] * 9 + [P(vp)]
    lib.conv_fused_run.argtypes = [vp, vp, vp, vp]
    lib.conv_fused_run_residual.argtypes = [vp, vp, vp, vp, vp]
    lib.conv_fused_status.argtypes = [vp]
    lib.conv_fused_clear_status.argtypes = [vp]
    lib.conv_fused_destroy.argtypes = [vp]
    lib.conv_fused_destroy.restype = None
    lib.conv_fused_variant.argtypes = [vp]
    lib.conv_fused_describe.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
    lib.conv_fused_last_error.argtypes = []
    lib.conv_fused_last_error.restype = ctypes.c_char_p
    lib.conv_fused_watchdog_selftest.argtypes = [vp, ctypes.c_longlong, vp]
    lib.conv_fused_run_noalloc.argtypes = [dptr, vp, vp, vp, vp, vp, vp, vp]
    lib.conv_fused_measure_int8_mma_rate.argtypes = [vp, P(ctypes.c_double)]
    lib.conv_fused_debug_fail_alloc.argtypes = [ctypes.c_int]
    lib.conv_fused_debug_live_handles.argtypes = []
    lib.conv_fused_chain_create.argtypes = [P(ChainStep), ctypes.c_int, P(vp)]
    lib.conv_fused_chain_create_ex.argtypes = [P(ChainStep), ctypes.c_int, ctypes.c_int, P(vp)]
    lib.conv_fused_chain_run.argtypes = [vp, vp]
    lib.conv_fused_chain_status.argtypes = [vp]
    lib.conv_fused_chain_clear_status.argtypes = [vp]
    lib.conv_fused_chain_describe.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
    lib.conv_fused_chain_destroy.argtypes = [vp]
    lib.conv_fused_chain_destroy.restype = None
    for name in EXPORTED:
        if name not in ("conv_fused_destroy", "conv_fused_last_error", "conv_fused_chain_destroy"):
            getattr(lib, name).restype = ctypes.c_int
    _LIB = lib
    return lib


def _check(status: int):
    if status != CONVF_OK:
        raise ConvFusedError(status, conv_fused_last_error())


def _addr(a) -> Optional[int]:
    """Host address of a numpy array / CPU tensor, device address of a CUDA tensor, or an int."""
    if a is None:
        return None
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    return a.ctypes.data


# --------------------------------------------------------------------------- C entry points

def conv_fused_last_error() -> str:
    return load_library().conv_fused_last_error().decode()


def conv_fused_output_shape(desc: ConvDesc):
    out = (ctypes.c_int * 4)()
    _check(load_library().conv_fused_output_shape(ctypes.byref(desc), out))
    return tuple(out)


def conv_fused_resolve_pads(desc: ConvDesc):
    out = (ctypes.c_int * 4)()
    _check(load_library().conv_fused_resolve_pads(ctypes.byref(desc), out))
    return tuple(out)


def conv_bn_scale_shift(gamma, beta, mean, var, eps: float = 1e-5):
    """Returns (scale, shift) as float32 numpy arrays."""
    import numpy as np
    arrs = [np.ascontiguousarray(np.asarray(a, dtype=np.float32)) for a in (gamma, beta, mean, var)]
    K = arrs[0].shape[0]
    scale = np.empty(K, np.float32)
    shift = np.empty(K, np.float32)
    fp = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
    _check(load_library().conv_bn_scale_shift(K, *[fp(a) for a in arrs], float(eps), fp(scale), fp(shift)))
    return scale, shift


def conv_fused_plan(desc: ConvDesc, num_sms: int = 152, with_pair: bool = False):
    """(variant, tile_n, ktot) or, with with_pair, (variant, tile_n, ktot, cta_pair)."""
    v, bn, kt, pr = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(load_library().conv_fused_plan(ctypes.byref(desc), num_sms, ctypes.byref(v), ctypes.byref(bn),
                                          ctypes.byref(kt), ctypes.byref(pr)))
    return (v.value, bn.value, kt.value, pr.value) if with_pair else (v.value, bn.value, kt.value)


def conv_fused_pack_weights(desc: ConvDesc, variant: int, W_bits, out):
    _check(load_library().conv_fused_pack_weights(ctypes.byref(desc), variant, _addr(W_bits), _addr(out),
                                                  out.size if hasattr(out, "size") and not callable(out.size)
                                                  else out.numel()))


def conv_fused_create(desc: ConvDesc, W, bias=None, bn_scale=None, bn_shift=None, requant_mult=None,
                      requant_shift=None, out_zero_point: int = 0) -> int:
    """Host arrays (numpy or CPU tensors, contiguous) in, handle (int) out."""
    h = ctypes.c_void_p()
    _check(load_library().conv_fused_create(ctypes.byref(desc), _addr(W), _addr(bias), _addr(bn_scale),
                                            _addr(bn_shift), _addr(requant_mult), _addr(requant_shift),
                                            int(out_zero_point), ctypes.byref(h)))
    return h.value


def conv_fused_create_preact(desc: ConvDesc, W, bias=None, bn_scale=None, bn_shift=None, pre_scale=None,
                             pre_shift=None, pre_act: int = CONVF_ACT_RELU) -> int:
    """Handle with a pre-activation prologue: the conv reads clamp(pre_scale*x + pre_shift)."""
    h = ctypes.c_void_p()
    _check(load_library().conv_fused_create_preact(ctypes.byref(desc), _addr(W), _addr(bias), _addr(bn_scale),
                                                   _addr(bn_shift), _addr(pre_scale), _addr(pre_shift),
                                                   int(pre_act), ctypes.byref(h)))
    return h.value


def conv_fused_create_mbv2_block(d: BlockDesc, w_expand, e_scale, e_shift, w_dw, d_scale, d_shift, w_project,
                                 p_scale, p_shift) -> int:
    """Fused MobileNetV2 block handle (host arrays: bf16 bits for weights, float32 affines)."""
    h = ctypes.c_void_p()
    _check(load_library().conv_fused_create_mbv2_block(ctypes.byref(d), _addr(w_expand), _addr(e_scale),
                                                       _addr(e_shift), _addr(w_dw), _addr(d_scale), _addr(d_shift),
                                                       _addr(w_project), _addr(p_scale), _addr(p_shift),
                                                       ctypes.byref(h)))
    return h.value


def conv_fused_create_qlinear(desc: ConvDesc, W, bias, q: QParams) -> int:
    """QLinearConv handle: desc.dtype == CONVF_Q8, W host int8/uint8 [K][C/group][R][S], bias host
    int32[K] or None, q the scales and zero points (its w arrays host pointers)."""
    h = ctypes.c_void_p()
    _check(load_library().conv_fused_create_qlinear(ctypes.byref(desc), _addr(W), _addr(bias), ctypes.byref(q),
                                                    ctypes.byref(h)))
    return h.value


def conv_fused_run(handle: int, x, y, stream=None):
    """x, y: device pointers (ints) or CUDA tensors; stream: cudaStream_t int, torch stream or None."""
    s = stream
    if s is not None and hasattr(s, "cuda_stream"):
        s = s.cuda_stream
    _check(load_library().conv_fused_run(handle, _addr(x), _addr(y), s))


def conv_fused_run_residual(handle: int, x, r, y, stream=None):
    """conv_fused_run for residual handles: y = act(scale * conv(x) + bias' + r)."""
    s = stream
    if s is not None and hasattr(s, "cuda_stream"):
        s = s.cuda_stream
    _check(load_library().conv_fused_run_residual(handle, _addr(x), _addr(r), _addr(y), s))


def conv_fused_status(handle: int) -> int:
    return load_library().conv_fused_status(handle)


def conv_fused_clear_status(handle: int):
    _check(load_library().conv_fused_clear_status(handle))


def conv_fused_destroy(handle: int):
    load_library().conv_fused_destroy(handle)


def conv_fused_variant(handle: int) -> int:
    v = load_library().conv_fused_variant(handle)
    if v < 0:
        _check(v)
    return v


def conv_fused_describe(handle: int) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(load_library().conv_fused_describe(handle, buf, 512))
    return buf.value.decode()


def conv_fused_watchdog_selftest(status_dev, budget_cycles: int, stream=None):
    s = stream.cuda_stream if stream is not None and hasattr(stream, "cuda_stream") else stream
    _check(load_library().conv_fused_watchdog_selftest(_addr(status_dev), int(budget_cycles), s))


def conv_fused_debug_fail_alloc(n: int):
    """Test hook: the n-th allocation the create calls make from now on fails (0 disarms)."""
    _check(load_library().conv_fused_debug_fail_alloc(int(n)))


def conv_fused_debug_live_handles() -> int:
    """Number of handles created and not yet destroyed."""
    return int(load_library().conv_fused_debug_live_handles())


def conv_fused_measure_int8_mma_rate(stream=None) -> float:
    """TOP/s of back-to-back int8 mma.sync on this GPU (register operands)."""
    s = stream.cuda_stream if stream is not None and hasattr(stream, "cuda_stream") else stream
    out = ctypes.c_double()
    _check(load_library().conv_fused_measure_int8_mma_rate(s, ctypes.byref(out)))
    return out.value


def conv_fused_run_noalloc(desc: ConvDesc, x, w_packed, scale, bias, y, status=None, stream=None):
    """Allocation-free run: every argument a device pointer (int) or CUDA tensor."""
    s = stream.cuda_stream if stream is not None and hasattr(stream, "cuda_stream") else stream
    _check(load_library().conv_fused_run_noalloc(ctypes.byref(desc), _addr(x), _addr(w_packed), _addr(scale),
                                                 _addr(bias), _addr(y), _addr(status), s))


def conv_fused_chain_create(steps, cta_pairs: int = 0) -> int:
    """steps: sequence of (handle, x, r or None, y) with device pointers (ints) or CUDA tensors;
    cta_pairs: 0 automatic, 1 single CTAs, 2 CTA pairs (conv_fused_chain_create_ex)."""
    arr = (ChainStep * len(steps))()
    for i, (h, x, r, y) in enumerate(steps):
        arr[i] = ChainStep(h, _addr(x), _addr(r), _addr(y))
    c = ctypes.c_void_p()
    _check(load_library().conv_fused_chain_create_ex(arr, len(steps), cta_pairs, ctypes.byref(c)))
    return c.value


def conv_fused_chain_run(chain: int, stream=None):
    s = stream
    if s is not None and hasattr(s, "cuda_stream"):
        s = s.cuda_stream
    _check(load_library().conv_fused_chain_run(chain, s))


def conv_fused_chain_status(chain: int) -> int:
    return load_library().conv_fused_chain_status(chain)


def conv_fused_chain_clear_status(chain: int):
    _check(load_library().conv_fused_chain_clear_status(chain))


def conv_fused_chain_describe(chain: int) -> str:
    buf = ctypes.create_string_buffer(65536)
    _check(load_library().conv_fused_chain_describe(chain, buf, 65536))
    return buf.value.decode()


def conv_fused_chain_destroy(chain: int):
    load_library().conv_fused_chain_destroy(chain)


# --------------------------------------------------------------------------- torch convenience

class FusedConv:
    """One prepared conv node over torch tensors.

    ``w`` (bf16 KCRS or int8), ``bias`` and the BN affine are CPU tensors; they are copied
    to the device once here.  Calling the object runs the kernel on the current torch stream
    with ``x`` a CUDA tensor in channels-last storage (logical NCHW) and returns y (fp32 or
    int8, channels-last).
    """

    def __init__(self, N, C, H, W, K, R, S, w, bias=None, bn_scale=None, bn_shift=None, stride=(1, 1),
                 pads=(0, 0, 0, 0), dilation=(1, 1), group=1, act=CONVF_ACT_NONE, clip=(0.0, 6.0),
                 auto_pad="NOTSET", variant=CONVF_VARIANT_AUTO, requant_mult=None, requant_shift=None,
                 out_zero_point=0, tile_n=0, cta_pair=0, stream_k=0, kblocks_per_step=0,
                 out_bf16=False, residual=False, pre_scale=None, pre_shift=None, pre_act=None):
        import torch
        s8 = w.dtype == torch.int8
        self.desc = make_desc(N, C, H, W, K, R, S, stride, pads, dilation, group,
                              CONVF_S8 if s8 else CONVF_BF16, act, clip, auto_pad, variant, tile_n=tile_n,
                              cta_pair=cta_pair, stream_k=stream_k, kblocks_per_step=kblocks_per_step,
                              out_dtype=CONVF_OUT_BF16 if out_bf16 else CONVF_OUT_F32, residual=int(bool(residual)))
        self.out_bf16 = bool(out_bf16)
        self.residual = bool(residual)
        wc = w.contiguous().cpu()
        wbits = wc if s8 else wc.view(torch.int16)
        keep = [wbits]

        def host(t, dt):
            if t is None:
                return None
            t = torch.as_tensor(t).to(dt).contiguous().cpu()
            keep.append(t)
            return t

        if pre_act is not None:
            # pre-activation prologue (bf16 convs): the conv reads clamp(pre_scale*x + pre_shift)
            self.handle = conv_fused_create_preact(self.desc, wbits, host(bias, torch.float32),
                                                   host(bn_scale, torch.float32), host(bn_shift, torch.float32),
                                                   host(pre_scale, torch.float32), host(pre_shift, torch.float32),
                                                   pre_act)
        else:
            self.handle = conv_fused_create(self.desc, wbits, host(bias, torch.int32 if s8 else torch.float32),
                                            host(bn_scale, torch.float32), host(bn_shift, torch.float32),
                                            host(requant_mult, torch.int32), host(requant_shift, torch.int32),
                                            out_zero_point)
        self.out_shape = conv_fused_output_shape(self.desc)
        self.s8 = s8

    @property
    def variant(self) -> int:
        return conv_fused_variant(self.handle)

    def describe(self) -> str:
        return conv_fused_describe(self.handle)

    def new_output(self):
        import torch
        N, K, Ho, Wo = self.out_shape
        dt = torch.int8 if self.s8 else (torch.bfloat16 if self.out_bf16 else torch.float32)
        return torch.empty((N, Ho, Wo, K), dtype=dt, device="cuda").permute(0, 3, 1, 2)

    def __call__(self, x, y=None, stream=None, r=None):
        """Runs on the current torch stream; ``r`` is the residual (y's shape, dtype and
        channels-last storage) for handles made with ``residual=True``."""
        import torch
        if not x.is_cuda:
            raise ValueError("x must be a CUDA tensor")
        if not x.is_contiguous(memory_format=torch.channels_last) and x.numel() > 0:
            raise ValueError("x must use channels-last storage")
        if y is None:
            y = self.new_output()
        s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
        if self.residual:
            if r is None:
                raise ValueError("this conv adds a residual: pass r")
            conv_fused_run_residual(self.handle, x.data_ptr(), r.data_ptr(), y.data_ptr(), s)
        else:
            conv_fused_run(self.handle, x.data_ptr(), y.data_ptr(), s)
        return y

    def status(self) -> int:
        return conv_fused_status(self.handle)

    def close(self):
        if self.handle:
            conv_fused_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class QLinearConv(FusedConv):
    """ONNX QLinearConv over torch tensors: ``w`` int8 or uint8 (KCRS, CPU), ``bias`` int32[K] or
    None, per-channel ``w_scale`` / ``w_zero_point`` (or scalars).  Calling it with an 8-bit
    channels-last CUDA tensor x returns the 8-bit y (uint8 or int8 per ``y_signed``)."""

    def __init__(self, N, C, H, W, K, R, S, w, bias=None, x_scale=1.0, x_zero_point=0, w_scale=1.0,
                 w_zero_point=0, y_scale=1.0, y_zero_point=0, x_signed=False, y_signed=False, relu=False,
                 stride=(1, 1), pads=(0, 0, 0, 0), dilation=(1, 1), group=1, auto_pad="NOTSET",
                 variant=CONVF_VARIANT_AUTO, tile_n=0, kblocks_per_step=0):
        import numpy as np
        import torch
        self.desc = make_desc(N, C, H, W, K, R, S, stride, pads, dilation, group, CONVF_Q8, CONVF_ACT_NONE,
                              (0.0, 6.0), auto_pad, variant, tile_n=tile_n, kblocks_per_step=kblocks_per_step)
        self.out_bf16 = False
        self.residual = False
        self.s8 = True
        self.y_signed = bool(y_signed)
        wc = w.contiguous().cpu()
        ws = np.ascontiguousarray(np.broadcast_to(np.asarray(w_scale, dtype=np.float32).reshape(-1), (K,)))
        wz = np.ascontiguousarray(np.broadcast_to(np.asarray(w_zero_point, dtype=np.int32).reshape(-1), (K,)))
        b = None if bias is None else torch.as_tensor(bias).to(torch.int32).contiguous().cpu()
        self._keep = [wc, ws, wz, b]
        q = QParams()
        q.x_signed, q.w_signed, q.y_signed = int(bool(x_signed)), int(wc.dtype == torch.int8), int(bool(y_signed))
        q.x_zero_point, q.y_zero_point = int(x_zero_point), int(y_zero_point)
        q.x_scale, q.y_scale = float(x_scale), float(y_scale)
        q.w_zero_point, q.w_scale = wz.ctypes.data, ws.ctypes.data
        q.relu = int(bool(relu))
        self.handle = conv_fused_create_qlinear(self.desc, wc, b, q)
        self.out_shape = conv_fused_output_shape(self.desc)

    def new_output(self):
        import torch
        N, K, Ho, Wo = self.out_shape
        dt = torch.int8 if self.y_signed else torch.uint8
        return torch.empty((N, Ho, Wo, K), dtype=dt, device="cuda").permute(0, 3, 1, 2)


class InvertedResidualBlock(FusedConv):
    """A MobileNetV2 block as one fused kernel over torch tensors: ``w_expand`` (bf16 [Ch][Cin][1][1]
    or None), ``w_dw`` (bf16 [Ch][1][3][3]), ``w_project`` (bf16 [Cout][Ch][1][1]) and each stage's
    folded BN affine (scale, shift) as float arrays.  Calling it with x (bf16, channels-last) returns
    y (fp32, channels-last)."""

    def __init__(self, N, Cin, H, W, Ch, Cout, stride, w_expand, e_affine, w_dw, d_affine, w_project, p_affine,
                 residual=False):
        import numpy as np
        import torch
        d = BlockDesc()
        d.N, d.H, d.W, d.Cin, d.Ch, d.Cout, d.stride = N, H, W, Cin, Ch, Cout, stride
        d.expand = int(w_expand is not None)
        d.residual = int(bool(residual))
        self.block = d

        def bits(t):
            return None if t is None else t.contiguous().cpu().view(torch.int16)

        def f32(a):
            return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float32))

        es, et = (f32(e_affine[0]), f32(e_affine[1])) if e_affine is not None else (None, None)
        keep = [bits(w_expand), es, et, bits(w_dw), f32(d_affine[0]), f32(d_affine[1]), bits(w_project),
                f32(p_affine[0]), f32(p_affine[1])]
        self._keep = keep
        self.handle = conv_fused_create_mbv2_block(d, *keep)
        Ho = (H + 2 - 3) // stride + 1
        Wo = (W + 2 - 3) // stride + 1
        self.out_shape = (N, Cout, Ho, Wo)
        self.s8 = False
        self.out_bf16 = False
        self.residual = False


class ConvChain:
    """A sequence of FusedConv runs as one persistent launch (conv_fused_chain_*).

    ``steps`` is a sequence of ``(conv, x, y)`` or ``(conv, x, y, r)`` with ``conv`` a FusedConv
    (1x1-GEMM or im2col implicit-GEMM variant) and ``x``, ``y``, ``r`` CUDA tensors in
    channels-last storage.  A step whose ``x`` (or ``r``) is an earlier step's ``y`` reads that
    output.  The tensors and the convs must outlive the chain; calling it runs every step on the
    current torch stream."""

    def __init__(self, steps, cta_pairs: int = 0):
        self._keep = [tuple(st) for st in steps]
        items = []
        for st in self._keep:
            conv, x, y = st[0], st[1], st[2]
            r = st[3] if len(st) > 3 else None
            items.append((conv.handle, x.data_ptr(), None if r is None else r.data_ptr(), y.data_ptr()))
        self.handle = conv_fused_chain_create(items, cta_pairs)

    def describe(self) -> str:
        return conv_fused_chain_describe(self.handle)

    def __call__(self, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
        conv_fused_chain_run(self.handle, s)

    def status(self) -> int:
        return conv_fused_chain_status(self.handle)

    def clear_status(self):
        conv_fused_chain_clear_status(self.handle)

    def close(self):
        if self.handle:
            conv_fused_chain_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
