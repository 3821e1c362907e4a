/*
 * conv_fused.h -- fused ONNX Conv (+ folded inference BatchNorm, bias, ReLU/ReLU6/Clip)
 * on one GB300 GPU (sm_103a).  Plain C ABI: host/device pointers and sizes only.
 *
 * What the operation is
 * ---------------------
 *   ONNX Conv (public operator specification): X[N][C][H][W] (NCHW semantics),
 *   W[K][C/group][R][S], optional bias B[K], attributes strides, pads
 *   [h_begin, w_begin, h_end, w_end], dilations, group, auto_pad.
 *   Followed, per output channel k, by an affine y = scale[k]*z + shift[k] -- the inference
 *   BatchNorm folded offline into the conv ("tensorforge", section "ResNet fusion":
 *   Conv -> BN -> Relu becomes one fused conv epilogue, W' = scale*W, bias = shift) -- and by a
 *   clamp activation (ReLU, ReLU6 = min(max(u,0),6), Clip(lo,hi); consecutive relu/min/max fuse
 *   into one min+max, "Kyanite" README, section "Optimizer").
 *   The library selects one of four kernels per shape ("OxiONNX 0.1.7 Released", Technical
 *   Deep Dive 2, "Real Conv dispatch": ImplicitGemmConv / Conv1x1 / DepthwiseConv per shape),
 *   plus a static-int8 kernel ("onnx-vulkan-rs", feature list: static int8 convolutions on
 *   the tensor cores) -- and refuses, at create time, any node it cannot honour, naming the
 *   reason; there is no CPU fallback (the same page: refuse at load time, never answer wrongly).
 *
 * Storage layout
 * --------------
 *   Logical dimensions are always ONNX NCHW.  The kernels read and write channels-last storage
 *   (NHWC: x[n][h][w][c], y[n][oh][ow][k]), i.e. a torch channels_last tensor.  CONVF_NCHW
 *   storage is refused with CONVF_ERR_UNSUPPORTED.
 *
 * Numerics
 * --------
 *   CONVF_BF16: x and W are bf16 (raw uint16 bits), accumulation fp32, y fp32.  The BN scale
 *   is applied to the fp32 accumulator (y = clamp(scale*acc + bias', lo, hi), bias' =
 *   scale*B + shift), which equals conv(scale*W) + bias' without rounding scale*W to bf16.
 *   Depthwise folds scale into fp32 taps.
 *   CONVF_S8: x, W int8 (symmetric, zero point 0), int32 accumulation, int32 bias, then per
 *   output channel q = (v*mult + 2^(shift-1)) >> shift (int64, arithmetic shift), v = acc +
 *   bias, o = clamp(q + out_zero_point, relu ? max(zp,-128) : -128, 127) as int8.
 *
 * Ownership and errors
 * --------------------
 *   create copies every host array it is given (the library owns the device copies; the
 *   caller may free its arrays on return).  run reads caller-owned device x and writes
 *   caller-owned device y, asynchronously on the caller's stream; it allocates nothing and
 *   never synchronises.  Every call returns a convf_status; conv_fused_last_error() gives a
 *   thread-local message naming the offending argument.  A handle is used from one stream at a
 *   time.  Device waits inside the kernels are bounded: a wait that runs out sets a status bit
 *   that conv_fused_status reports as CONVF_ERR_TIMEOUT after the caller synchronises.
 */
#ifndef CONV_FUSED_H
#define CONV_FUSED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CONVF_OK = 0,
  CONVF_ERR_INVALID_ARG = -1,  /* malformed argument (named in conv_fused_last_error) */
  CONVF_ERR_UNSUPPORTED = -2,  /* well-formed but not served by any kernel: refused, no fallback */
  CONVF_ERR_OOM = -3,          /* device allocation failed at create */
  CONVF_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed */
  CONVF_ERR_TIMEOUT = -5,      /* a bounded device wait ran out during a run */
  CONVF_ERR_BOUNDS = -6        /* only in a library built with CONVF_DEBUG_BOUNDS: a kernel computed
                                  a global index outside the tensor its parameters describe and
                                  skipped that access (a library defect, never the caller's) */
} convf_status;

/* CONVF_Q8: ONNX QLinearConv -- 8-bit x, W and y with scales and zero points
 * (conv_fused_create_qlinear); the element types are given by its convf_qparams. */
typedef enum { CONVF_BF16 = 0, CONVF_S8 = 1, CONVF_Q8 = 2 } convf_dtype;
/* element type of y (and of the residual) on the bf16 path */
typedef enum { CONVF_OUT_F32 = 0, CONVF_OUT_BF16 = 1 } convf_out_dtype;
typedef enum { CONVF_NCHW = 0, CONVF_NHWC = 1 } convf_layout;
typedef enum {
  CONVF_ACT_NONE = 0, CONVF_ACT_RELU = 1, CONVF_ACT_RELU6 = 2, CONVF_ACT_CLIP = 3
} convf_act;
typedef enum {
  CONVF_AUTO_PAD_NOTSET = 0, CONVF_AUTO_PAD_SAME_UPPER = 1, CONVF_AUTO_PAD_SAME_LOWER = 2,
  CONVF_AUTO_PAD_VALID = 3
} convf_auto_pad;

/* Kernel variants.  CONVF_VARIANT_AUTO lets the shape-keyed selector choose; any other value
 * forces that kernel (refused with CONVF_ERR_UNSUPPORTED if it cannot serve the shape). */
typedef enum {
  CONVF_VARIANT_AUTO = 0,
  CONVF_VARIANT_IMPLICIT_GEMM = 1,   /* tcgen05 implicit GEMM, TMA im2col activation tiles */
  CONVF_VARIANT_GEMM_1X1 = 2,        /* same kernel, activations read as a [N*H*W][C] matrix */
  CONVF_VARIANT_DEPTHWISE = 3,       /* CUDA-core depthwise (group == C == K) */
  CONVF_VARIANT_INT8 = 4,            /* int8 warp-level MMA (mma.sync), int32 accumulate, requant;
                                        C % 64 == 0, K % 16 == 0.  Chosen only when the
                                        exact-integer tcgen05 variant cannot serve the shape */
  CONVF_VARIANT_IMPLICIT_GEMM_GATHER = 5, /* tcgen05 implicit GEMM, activation rows gathered by
                                            threads (any C, e.g. the 3-channel stem) */
  CONVF_VARIANT_IMPLICIT_GEMM_WINDOW = 6, /* tcgen05 implicit GEMM for C <= 8: a pre-pass pads the
                                            channels to 4 or 8 and the columns by the left pad,
                                            after which one filter row of one output pixel is a
                                            contiguous run and one TMA load (overlapping
                                            windows) brings a tile's whole activation operand;
                                            weights resident in shared memory.  Needs dilation
                                            1, sw*cpt*2 a multiple of 16 bytes, S*cpt <= 64,
                                            R*round_up(S*cpt,16) <= 256, K <= 256.  The selector
                                            takes it for outputs at least 32 pixels wide. */
  CONVF_VARIANT_IMPLICIT_GEMM_HALO = 7,   /* tcgen05 implicit GEMM for stride-1, dilation-1
                                            filters: output rows padded to the input width
                                            Wp = W + pl + pr <= 128, tiles of floor(128/Wp)
                                            output rows; per 64-channel block one TMA box of
                                            padded input rows serves every filter tap through
                                            shifted shared-memory descriptors (im2col reloads
                                            it once per tap).  The selector takes it when at
                                            least 60% of a tile's 128 rows are real outputs. */
  CONVF_VARIANT_INT8_TC = 8,         /* 8-bit convs (CONVF_S8, CONVF_Q8) on tcgen05: a pre-pass writes
                                        x - x_zero_point as bf16 (exact: |v| <= 255) into a handle
                                        workspace, the weights are prepacked as bf16 w - w_zero_point,
                                        and the tcgen05 implicit GEMM restarts its fp32 accumulator
                                        every chunk of reduction blocks small enough that no partial
                                        sum exceeds 2^24 (so every partial sum is an exact integer);
                                        the epilogue adds the chunks in int32 and requantises.
                                        Bit-exact.  C % 8 == 0, K % 16 == 0, group 1. */
  CONVF_VARIANT_GROUPED_DIRECT = 9,  /* CUDA-core direct conv for any group count and filter (one
                                        thread per output pixel and channel, fp32); chosen for the
                                        grouped convs the tensor-core kernels cannot take.  (Those
                                        take groups on CONVF_VARIANT_IMPLICIT_GEMM / _GEMM_1X1 when
                                        an output-channel tile covers whole groups or lies inside
                                        one: block-diagonal weights over the tile's input-channel
                                        window, at most 16x the grouped work.) */
  CONVF_VARIANT_MBV2_BLOCK = 10      /* a whole MobileNetV2 inverted-residual block in one kernel
                                        (conv_fused_create_mbv2_block); never selected for a single
                                        conv */
} convf_variant;

typedef struct {
  int N, C, H, W;          /* x: [N][C][H][W] logical; N may be 0 (empty run)                */
  int K, R, S;             /* W: [K][C/group][R][S]                                           */
  int stride[2];           /* (h, w), >= 1                                                    */
  int dilation[2];         /* (h, w), >= 1                                                    */
  int pads[4];             /* ONNX order h_begin, w_begin, h_end, w_end; ignored unless NOTSET */
  int auto_pad;            /* convf_auto_pad                                                  */
  int group;               /* C % group == 0 && K % group == 0                                */
  int dtype;               /* convf_dtype                                                     */
  int x_layout, y_layout;  /* convf_layout; only CONVF_NHWC is served                         */
  int act;                 /* convf_act                                                       */
  float clip_lo, clip_hi;  /* bounds for CONVF_ACT_CLIP (lo <= hi)                            */
  int variant;             /* convf_variant; 0 = selector                                     */
  int tile_n;              /* tcgen05 variants: output-channel tile width 32/64/128/256, 0 = auto */
  int cta_pair;            /* tcgen05 variants: 0 = auto, 1 = single-CTA 128-row tiles, 2 = CTA pairs
                              (cta_group::2, 256-row tiles, each CTA loads half the weight tile) */
  int stream_k;            /* TMA implicit-GEMM variants on single CTAs: 0 = auto, 1 = off (whole
                              tiles per CTA), 2 = on (each CTA takes an equal share of the tile x
                              reduction-block iterations; a split tile is finished by the CTA holding
                              its first reduction block, which adds the others' fp32 partials from a
                              handle-owned workspace).  Ignored where it does not apply. */
  int kblocks_per_step;    /* TMA implicit-GEMM variants (single CTAs, pairs, stream-K): 64-wide
                              reduction blocks per pipeline step, 0 = auto, else 1..4 (must divide
                              both the block count and the tile width's stage count).  A step's
                              weights are one TMA box, and so are its activations in the 1x1 mode
                              when C % 64 == 0; more bytes per TMA operation raise the operand
                              ingest rate.  Ignored where it does not apply. */
  int out_dtype;           /* convf_out_dtype of y on the bf16 path: CONVF_OUT_F32 (default) or
                              CONVF_OUT_BF16 (the fp32 result rounded to nearest-even bf16) */
  int residual;            /* 1: y = act(scale * conv + bias' + r) for a residual tensor r of
                              y's shape, layout and element type, passed to
                              conv_fused_run_residual (the skip connection of a bottleneck block,
                              added after the folded BN and before the activation, as in the
                              single fused conv, residual, bias and ReLU operation the "Kyanite"
                              README lists in section "Cuda Executor").  0: no residual.
                              Both options are served by the TMA implicit-GEMM and 1x1 kernels
                              (C % 8 == 0) and the direct grouped kernel; other kernels refuse them. */
} convf_desc;

typedef struct convf_handle convf_handle;

/* Quantisation parameters of ONNX QLinearConv (public operator specification): real x =
 * (x - x_zero_point) * x_scale, real w[k] = (w[k] - w_zero_point[k]) * w_scale[k], y =
 * saturate(round(conv_real / y_scale) + y_zero_point), bias int32 in units of x_scale *
 * w_scale[k].  Each zero point has its tensor's element type.  The rounding step is taken in
 * float32 (the specification fixes no precision): m[k] = float32(x_scale * w_scale[k] / y_scale)
 * formed in double, then y = saturate(round_half_even(float32(acc + bias[k]) * m[k]) + y_zp),
 * where acc = sum (x - x_zp)(w - w_zp[k]) is exact and the padded input stands for x_zp. */
typedef struct {
  int x_signed, w_signed, y_signed;  /* element types: 1 = int8, 0 = uint8                   */
  int32_t x_zero_point;              /* in x's range                                          */
  const int32_t* w_zero_point;       /* host [K], each in w's range (per output channel)     */
  float x_scale;                     /* > 0, finite                                           */
  const float* w_scale;              /* host [K], > 0, finite                                 */
  float y_scale;                     /* > 0, finite                                           */
  int32_t y_zero_point;              /* in y's range                                          */
  int relu;                          /* 1: clamp below at y_zero_point (a fused Relu)         */
} convf_qparams;

/* Output logical shape [N][K][Ho][Wo] of desc (ONNX Conv shape rule, auto_pad resolved).
 * CONVF_ERR_INVALID_ARG if the attributes are malformed or the window does not fit. */
convf_status conv_fused_output_shape(const convf_desc* desc, int out_nchw[4]);

/* Resolved explicit pads (h_begin, w_begin, h_end, w_end) for desc's auto_pad (ONNX rule:
 * SAME_* pads to ceil(in/stride) outputs, the odd element at the end for SAME_UPPER and at the
 * beginning for SAME_LOWER; VALID = no padding). */
convf_status conv_fused_resolve_pads(const convf_desc* desc, int pads_out[4]);

/* BN inference affine from its parameters, computed in double and rounded to float:
 *   scale[k] = gamma[k] / sqrt(var[k] + eps),  shift[k] = beta[k] - mean[k] * scale[k].
 * All arrays are host float[K]; eps > 0 (ONNX default 1e-5). */
convf_status conv_bn_scale_shift(int K, const float* gamma, const float* beta, const float* mean,
                                 const float* var, float eps, float* scale, float* shift);

/* Host-only view of the shape-keyed selector (no CUDA call): the variant create would pick
 * for desc, the tcgen05 tile width *tile_n (0 for the other kernels) and whether the tiles run on
 * CTA pairs (*cta_pair = 1: 256 x tile_n tiles; 0: 128 x tile_n) on a GPU with num_sms SMs, and
 * the prepacked weight row length *ktot (elements).  Any output pointer may be NULL.  Refusals
 * are the same as create's. */
convf_status conv_fused_plan(const convf_desc* desc, int num_sms, int* variant, int* tile_n,
                             int* ktot, int* cta_pair);

/* Host-only weight prepack for a tcgen05 variant (CONVF_VARIANT_GEMM_1X1, _IMPLICIT_GEMM or
 * _IMPLICIT_GEMM_GATHER): W [K][C][R][S] bf16 bits -> out [K][ktot] bf16 bits, reduction index
 * (r*S + s)*Cp + c with Cp = C rounded up to 64 for the im2col variant (each tap's channel run
 * is zero-padded); for the gather variant Cp = 4 (C <= 4) or 8 (C <= 8) when a tile's input rows
 * can be staged in shared memory (N*Ho*Wo tiles of 128 never straddle images, W*C*2 is a
 * multiple of 16 and the rows fit 32 KB), else Cp = C; the row tail is zero.
 * out_elems >= K*ktot. */
convf_status conv_fused_pack_weights(const convf_desc* desc, int variant, const uint16_t* W,
                                     uint16_t* out, size_t out_elems);

/* Build a handle: validate, resolve pads, fold BN into the epilogue, prepack W for the
 * selected kernel and upload it once (the only host->device crossing besides the launch).
 *   W:       host, ONNX layout [K][C/group][R][S]; uint16 bf16 bits (CONVF_BF16) or int8.
 *   bias:    host float[K] (bf16 path) or int32[K] (s8 path), or NULL (absent = 0).
 *   bn_scale, bn_shift: host float[K] each (the folded BN affine, see conv_bn_scale_shift),
 *            or NULL (identity).  Must be NULL on the s8 path.
 *   requant_mult (int32[K], > 0), requant_shift (int32[K], 1..62), out_zero_point: s8 path
 *            only (NULL / ignored on the bf16 path).
 *   *out receives the handle (NULL on failure; partial allocations are released). */
convf_status conv_fused_create(const convf_desc* desc, const void* W, const void* bias,
                               const float* bn_scale, const float* bn_shift,
                               const int32_t* requant_mult, const int32_t* requant_shift,
                               int32_t out_zero_point, convf_handle** out);

/* ONNX QLinearConv ("onnx-vulkan-rs", notes on the quantized kernels: zero-point corrected integer
 * sums, a +-1 LSB contract against other runtimes): desc->dtype must be CONVF_Q8 (act and the
 * performance knobs other than tile_n are ignored; use q->relu).
 *   W:    host [K][C/group][R][S], int8 or uint8 per q->w_signed.
 *   bias: host int32[K] or NULL.
 *   q:    the scales and zero points above (copied).
 * Served by CONVF_VARIANT_INT8_TC only.  run then takes 8-bit x and writes 8-bit y. */
convf_status conv_fused_create_qlinear(const convf_desc* desc, const void* W, const int32_t* bias,
                                       const convf_qparams* q, convf_handle** out);

/* conv_fused_create with a pre-activation prologue (the BN -> ReLU that a ResNet-v2 block
 * applies to its input before the first conv; "tensorforge", section "ResNet fusion"): the conv
 * reads u = clamp(pre_scale[c] * x + pre_shift[c]) per input channel c, the clamp of pre_act
 * (CONVF_ACT_NONE, _RELU or _RELU6), with the conv's zero padding applied to u, not to x.  u is
 * the conv's operand and is rounded to bf16 (nearest even).  It runs as a pre-pass into a
 * handle-owned bf16 copy of the input (one extra read and write of x per run) that every
 * kernel variant then reads.
 *   pre_scale, pre_shift: host float[C] (e.g. conv_bn_scale_shift of the input's BN), finite.
 * bf16 convs only (CONVF_ERR_UNSUPPORTED otherwise); the other arguments as for create. */
convf_status conv_fused_create_preact(const convf_desc* desc, const void* W, const void* bias,
                                      const float* bn_scale, const float* bn_shift, const float* pre_scale,
                                      const float* pre_shift, int pre_act, convf_handle** out);

/* A MobileNetV2 inverted-residual block as one fused kernel (the expanded "hidden" tensor stays
 * on chip; "tensorforge", section "ResNet fusion", taken to the whole block):
 *   h1 = ReLU6(e_scale * conv1x1(x, w_expand) + e_shift)      (absent when expand == 0: h1 = x)
 *   h2 = ReLU6(d_scale * dwconv3x3(h1, w_dw, stride, pad 1) + d_shift)
 *   y  = p_scale * conv1x1(h2, w_project) + p_shift  (+ x when residual)
 * per channel, the *_scale / *_shift being each stage's folded BN (conv_bn_scale_shift).  The
 * hidden values are kept in fp32 and the project GEMM reads h2 as two bf16 halves (hi + lo), so
 * the result meets the same bound as a single conv.  Run with conv_fused_run(h, x, y, stream):
 * x NHWC bf16 [N][H][W][Cin], y NHWC fp32 [N][Ho][Wo][Cout]. */
typedef struct {
  int N, H, W;         /* block input extent                                                  */
  int Cin, Ch, Cout;   /* input, hidden (expanded) and output channels; Cin % 8 == 0, Cin <= 192 */
  int stride;          /* depthwise stride: 1 or 2                                            */
  int expand;          /* 1: a 1x1 expand Cin -> Ch precedes the depthwise; 0: none (Ch == Cin) */
  int residual;        /* 1: y += x (stride 1 and Cin == Cout only)                           */
} convf_block_desc;

/* w_expand: host bf16 bits [Ch][Cin] (NULL when expand == 0); w_dw: [Ch][3][3]; w_project:
 * [Cout][Ch]; the six affine arrays host float ([Ch] or [Cout]; e_* NULL when expand == 0).
 * Refused (CONVF_ERR_UNSUPPORTED, named) when the tile geometry or the 512 TMEM columns cannot
 * hold the block. */
convf_status conv_fused_create_mbv2_block(const convf_block_desc* d, const uint16_t* w_expand,
                                          const float* e_scale, const float* e_shift, const uint16_t* w_dw,
                                          const float* d_scale, const float* d_shift,
                                          const uint16_t* w_project, const float* p_scale,
                                          const float* p_shift, convf_handle** out);

/* Run the fused conv: x (device, NHWC, bf16 bits or 8-bit) -> y (device, NHWC, float32 -- or bf16
 * bits with out_dtype = CONVF_OUT_BF16 -- for the bf16 path, 8-bit for the s8 and q8 paths).  Both must be 16-byte aligned and must not overlap.
 * `stream` is a cudaStream_t (NULL = legacy default stream).  Asynchronous: no allocation,
 * no synchronisation; launch errors are returned as CONVF_ERR_CUDA. */
convf_status conv_fused_run(convf_handle* h, const void* x, void* y, void* stream);

/* conv_fused_run for a handle created with residual = 1: y = act(scale * conv(x) + bias' + r).
 * r (device, NHWC, the element type of y, y's shape) must be 16-byte aligned; it may be y itself
 * (each element of the residual is read before the same element of y is written) but must not overlap y
 * otherwise, nor x.  conv_fused_run refuses residual handles and this call refuses the others
 * (CONVF_ERR_INVALID_ARG). */
convf_status conv_fused_run_residual(convf_handle* h, const void* x, const void* r, void* y, void* stream);

/* Device status of the handle's previous runs, read after the caller synchronised the
 * stream: CONVF_OK, or CONVF_ERR_TIMEOUT if a bounded wait ran out, or (bounds-checking build
 * only) CONVF_ERR_BOUNDS (the status is sticky
 * until conv_fused_clear_status). */
convf_status conv_fused_status(convf_handle* h);
convf_status conv_fused_clear_status(convf_handle* h);

/* Frees the handle's device memory.  The caller must have synchronised the stream. */
void conv_fused_destroy(convf_handle* h);

/* Selected kernel variant (convf_variant) of a handle, or a negative status. */
int conv_fused_variant(const convf_handle* h);

/* One-line description (variant, tile shape, grid) into buf[len]; returns the status. */
convf_status conv_fused_describe(const convf_handle* h, char* buf, size_t len);

/* Thread-local message for the last failing call on this thread ("" if none). */
const char* conv_fused_last_error(void);

/* Failure-detection self-test of the bounded device wait used by every kernel: launches one
 * CTA that waits on an mbarrier nobody arrives at, with a budget of `budget_cycles` SM
 * cycles, on `stream`.  *status_dev (device int32) receives CONVF_ERR_TIMEOUT's bit pattern
 * (1) when the wait ran out.  No other effect. */
convf_status conv_fused_watchdog_selftest(int32_t* status_dev, long long budget_cycles,
                                          void* stream);

/* Test hook for the allocation-failure path of the create calls (conv_fused_create,
 * _create_qlinear, _create_preact, _create_mbv2_block).  After conv_fused_debug_fail_alloc(n)
 * with n >= 1, the n-th allocation that create calls make from then on fails as if memory had
 * run out; host allocations (the handle) and device allocations (its one cudaMalloc) count
 * alike, in the order a call makes them: the handle first, before any CUDA call, then the
 * device block.  The failing call frees what it already holds and returns CONVF_ERR_OOM; its
 * conv_fused_last_error message ends in "(injected)".  The hook then disarms itself; n = 0
 * disarms it at once; a negative n is CONVF_ERR_INVALID_ARG.  Process-wide, for tests: calls
 * on other threads in the meantime draw on the same count.
 * conv_fused_debug_live_handles returns how many handles exist (created and not yet
 * destroyed), so a test can check that a failed create left nothing behind. */
convf_status conv_fused_debug_fail_alloc(int n);
int conv_fused_debug_live_handles(void);

/* Measurement helper (the int8 path's roofline denominator): times back-to-back
 * mma.sync.m16n8k32 int8 MMAs on register operands over every SM of the current device and
 * returns the rate in TOP/s (2 ops per multiply-add).  Synchronises `stream`. */
convf_status conv_fused_measure_int8_mma_rate(void* stream, double* tops);

/* Allocation-free run (this entry point has no counterpart in the method's sources; it serves
 * callers that cannot allocate device memory — e.g. code that runs while a CUDA graph is being
 * captured, inside a fixed device-memory budget that a host framework owns, or on a real-time
 * path where an allocation's latency or failure is not acceptable).  It runs the gathered-row
 * tcgen05 conv (convs with at most 8 input channels, such as an RGB stem, whose 128-row output
 * tiles stay inside one image) without a handle and without any allocation: the caller passes
 * every buffer, and the only scratch (the input with channels padded to whole taps, the padded
 * epilogue vectors and a status word) lives in a 16 MiB device array that the library reserves
 * on every GPU that loads it, until the process exits.
 *   desc:      as for create (NHWC storage; tile_n <= 128; cta_pair 0 or 1).
 *   x, y:      device, NHWC bf16 in / fp32 out, 16-byte aligned.
 *   w_packed:  device, the weights prepacked for CONVF_VARIANT_IMPLICIT_GEMM_GATHER exactly as
 *              conv_fused_pack_weights writes them ([K][ktot] bf16 bits), 16-byte aligned.
 *   scale, bias: device float[K], the folded epilogue y = clamp(scale*acc + bias, lo, hi)
 *              (bias = bn_scale*B + bn_shift).
 *   status_dev: optional device int32 that receives the timeout bit (1) if a bounded wait ran
 *              out.  With NULL a timeout is not reported to the caller at all (the bit lands in
 *              a word inside the scratch array, which every call clears first and nobody reads).
 *   desc options the gathered-row kernel cannot honour are refused (CONVF_ERR_UNSUPPORTED):
 *   tile_n > 128, cta_pair = 2, stream_k = 2, kblocks_per_step > 1, bf16 output, residual.
 * Sizes needing more scratch than 16 MiB are refused with CONVF_ERR_UNSUPPORTED.  The first call
 * on a device looks up the scratch array's device address (cudaGetSymbolAddress); make that
 * first call before any stream capture.  All calls share the one scratch array: calls whose
 * work overlaps on the GPU (other streams, or without ordering between them) race on it.
 * Asynchronous on `stream`; it never calls cudaMalloc, cudaFree or an allocating routine. */
convf_status conv_fused_run_noalloc(const convf_desc* desc, const void* x, const void* w_packed,
                                    const float* scale, const float* bias, void* y,
                                    int32_t* status_dev, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Conv chain: a sequence of conv runs executed by ONE persistent kernel launch.
 *
 * The steps compute exactly what conv_fused_run / conv_fused_run_residual would compute if they
 * were called one after another on one stream, with the same per-element arithmetic (fp32
 * accumulation of bf16 products, y = clamp(scale*acc + bias' (+ r), lo, hi), fp32 output or
 * bf16 rounded to nearest even).  A network's layers are short: a launch per layer pays the
 * kernel's start-up, its first operands' latency and its last tiles' epilogue (while other SMs
 * idle) every time.  A chain pays them once and lets a step's first tiles start while the
 * previous step's last ones are still running.
 *
 * Dependencies are taken from buffer identity: when a step's x (or residual) is exactly an
 * earlier step's y (same device pointer, same size and shape), the step reads that output, and
 * each of its 128-row output tiles waits (inside the kernel, bounded) only until the rows it
 * reads have been stored.  Every other x or residual is an input of the chain that no step
 * writes.  Refused (CONVF_ERR_UNSUPPORTED, named) at create: a step's x or residual partially
 * overlapping an output; a step reading an output that the same or a later step writes; two
 * steps writing overlapping outputs; an fp32 output read as a bf16 input.
 *
 * Steps: handles of CONVF_VARIANT_GEMM_1X1 or CONVF_VARIANT_IMPLICIT_GEMM (force the variant in
 * the desc if the selector would pick another), bf16, group 1, no pre-activation; C and K
 * multiples of 8; every step's output type the same (all fp32 or all bf16).  The chain chooses
 * its own tile shape per step (see conv_fused_chain_create_ex) and ignores the handles'
 * performance knobs.  The handles must outlive the chain (it reads their prepacked weights);
 * the buffers are fixed at create (the tensor maps are encoded for them).
 *
 * The chain's CTAs wait for one another's tiles, so they must all be resident at once: the
 * launch uses at most one CTA per SM (and, with CTA pairs, at most the clusters that fit).  A wait that runs out (or any error bit in the chain's
 * status word) makes every CTA give up; conv_fused_chain_status then reports it, and runs
 * after that give up at once until conv_fused_chain_clear_status.
 */
typedef struct convf_chain convf_chain;
typedef struct {
  convf_handle* conv;   /* the step's conv (see above)                                            */
  const void* x;        /* device NHWC bf16 input, 16-byte aligned                                */
  const void* r;        /* device residual of y's type and shape (handle created with residual =
                           1), else NULL                                                         */
  void* y;              /* device NHWC output, 16-byte aligned                                    */
} convf_chain_step;

/* Validates the n steps (host array, copied), finds their dependencies, encodes their tensor
 * maps and uploads the step table (one device allocation; synchronises the device once).
 * Equivalent to conv_fused_chain_create_ex(steps, n, 0, out). */
convf_status conv_fused_chain_create(const convf_chain_step* steps, int n, convf_chain** out);
/* The same with a choice of tiles: cta_pairs = 1 runs single CTAs (128-row tiles of 64 or 128
 * columns); 2 runs CTA pairs (clusters of two CTAs sharing tcgen05 MMAs of 256 rows: tiles of
 * 256 rows and 64, 128 or 256 columns, each CTA loading half the weight rows, which halves the
 * weight bytes per FLOP but also the number of tiles); 0 chooses pairs when no step reads another
 * step's output and every step has C and K of at least 256, single CTAs otherwise.  Results are
 * the same either way. */
convf_status conv_fused_chain_create_ex(const convf_chain_step* steps, int n, int cta_pairs, convf_chain** out);
/* One launch of the whole sequence on `stream` (a cudaStream_t, NULL = legacy default stream).
 * Asynchronous; allocates nothing; may be captured in a CUDA graph.  Runs of one chain must not
 * overlap in time (use one stream). */
convf_status conv_fused_chain_run(convf_chain* c, void* stream);
/* Device status of earlier runs (read after the caller synchronised): CONVF_OK, CONVF_ERR_TIMEOUT
 * or (bounds-checking build) CONVF_ERR_BOUNDS; sticky until conv_fused_chain_clear_status. */
convf_status conv_fused_chain_status(convf_chain* c);
convf_status conv_fused_chain_clear_status(convf_chain* c);
/* One line: step count, tiles, grid, and per step its filter, rows, channels, tile width,
 * reduction blocks and the steps it reads (src = x's producer, res = the residual's; -1 = an
 * input of the chain). */
convf_status conv_fused_chain_describe(const convf_chain* c, char* buf, size_t len);
/* Frees the chain's device memory (the caller must have synchronised); NULL is ignored. */
void conv_fused_chain_destroy(convf_chain* c);

#ifdef __cplusplus
}
#endif
#endif /* CONV_FUSED_H */
