// Internal interface between the host prep (api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

namespace convf {

// Bit set in a handle's device status word when a bounded device wait ran out.
constexpr int kStatusTimeout = 1;
// Bit set by a build with CONVF_DEBUG_BOUNDS when a kernel computed a global index outside the
// tensor its parameters describe; the access is skipped instead of made.
constexpr int kStatusBounds = 2;

// CONVF_IN_BOUNDS(ok, status): true when the checked condition holds.  Ordinary builds compile
// it to `true` (the kernels' own masks already keep every access inside its tensor); the
// CONVF_DEBUG_BOUNDS build evaluates the condition, and on failure sets kStatusBounds in the
// status word and returns false so that the caller skips the access.
#if defined(__CUDACC__)
__device__ __forceinline__ bool convf_bounds_ok(bool ok, int* status) {
  if (!ok && status) atomicOr(status, kStatusBounds);
  return ok;
}
#endif
#ifdef CONVF_DEBUG_BOUNDS
#define CONVF_IN_BOUNDS(ok, status) (::convf::convf_bounds_ok((ok), (status)))
#else
#define CONVF_IN_BOUNDS(ok, status) (true)
#endif

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel in the stream finishes; every kernel here waits (griddepcontrol.wait) before its
// first global-memory access, so stream order is kept for data.
// `cluster` > 1 launches clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- tcgen05 implicit GEMM
// GEMM view of the conv: rows m = (n, oh, ow) (M = N*Ho*Wo), columns = output channels,
// reduction j over (tap, channel).  A = activation rows (im2col on the fly), B = prepacked
// weights [K][Ktot] bf16 (Ktot = num_kb * 64), D = fp32 accumulator in TMEM.
enum AMode : int { kA2D = 0, kAIm2col = 1, kAGather = 2 };

struct TcConvParams {
  int M;            // output rows N*Ho*Wo
  int Kout;         // output channels
  int num_kb;       // 64-wide reduction blocks per tile
  int cblocks;      // channel blocks per tap (im2col mode)
  int R, S;         // filter taps
  int dh, dw;       // dilations
  int sh, sw;       // strides
  int pt, pl;       // leading pads
  int H, W, C;      // input extent (gather mode)
  int Ho, Wo;       // output extent
  int n_blocks;     // ceil(Kout / BN)
  int num_tiles;    // ceil(M / 128) * n_blocks
  int a_mode;       // AMode
  const float* scale;     // [Kpad] per-channel epilogue scale (BN scale)
  const float* bias;      // [Kpad] per-channel epilogue bias (scale*B + shift)
  const uint16_t* x;      // NHWC bf16 input (gather mode)
  int patch_rows;         // gather mode: input rows staged per tile in smem (0 = read global)
  int row_bytes;          // W*C*2, bytes of one input row
  int cpt;                // gather mode: channels per tap in the reduction layout (4, 8; 0 = C)
  float lo, hi;           // activation clamp
  float* y;               // NHWC output [M][Kout]: fp32, or bf16 bits when out_bf16
  const void* res;        // residual [M][Kout] of y's element type added before the clamp, or null
  int out_bf16;           // y (and res) hold bf16 (round to nearest even) instead of fp32
  int* status;            // device status word
  // stream-K: every CTA takes an equal share of the num_tiles x num_kb iterations; a tile split
  // across CTAs is finished by the CTA holding its k-block 0, which adds the others' fp32
  // partials (one workspace slot of 128 x BN floats and one flag per CTA, flags zero between
  // launches)
  int sk;                 // 0 = whole tiles per CTA
  float* sk_ws;
  int* sk_flags;
  // k-blocks per pipeline step (1, 2, 3 or 4; divides num_kb and the stage count): one weight
  // TMA box of kpb consecutive 64-wide blocks, and one activation box when a3d (2-D mode, C a
  // multiple of 64: the map is {64, M, C/64}); otherwise kpb activation loads shared by the two
  // producer warps.  1 in gather mode.
  int kpb;
  int a3d;
  // both epilogue warpgroups drain every tile (one column half each) instead of alternate tiles:
  // faster when a CTA has few tiles (its last tile's epilogue is the kernel's tail), slower
  // with many (twice the per-tile epilogue steps); 64+ column tiles without stream-K only
  int split_epi;
  // ---- integer-exact mode (the IQ instantiation): the operands are integers held exactly in
  // bf16 (8-bit values minus their zero points), so every product is an integer of at most 16
  // bits; the fp32 accumulator restarts every iq_chunk_kb reduction blocks, a count chosen so
  // that no partial sum exceeds 2^24 in magnitude (every partial sum is then an exactly
  // represented integer), and the epilogue converts each chunk to int32 and adds the chunks.
  // grouped convolution (1 < group): Kg output and Cg input channels per group; a tile of BN
  // output channels covers whole groups (BN % Kg == 0) or lies inside one (Kg % BN == 0), and
  // its activation loads read the channel window starting at (n0 / Kg) * Cg.  0 = dense.
  int grp_kg, grp_cg;
  int iq_chunk_kb;        // reduction blocks per exact chunk (a multiple of kpb)
  int iq_mode;            // requantisation: 0 fixed point (static int8), 1 float32 (QLinearConv)
  const int32_t* q_bias;  // [Kpad] int32 bias added to the exact sum
  const int32_t* q_mult;  // [Kpad] mode 0: multiplier M (> 0)
  const int32_t* q_shift; // [Kpad] mode 0: shift sh (1..62): q = (v*M + 2^(sh-1)) >> sh
  const float* q_scale;   // [Kpad] mode 1: float32 multiplier m: q = rint(float(v) * m)
  int q_zp;               // output zero point, added after the rounding
  int q_lo, q_hi;         // output clamp (the 8-bit type's range, the zero point below for ReLU)
  uint8_t* y8;            // NHWC 8-bit output [M][Kout] (int8 or uint8 bits)
};

// Pipeline stages (64-wide k-blocks held in shared memory) of the TMA implicit-GEMM kernel per
// tile width: operand ingest per SM does not grow with depth, so stages give way to the epilogue
// (and, with rsm, to the two bf16 residual tiles staged in shared memory: 32 or 64 KB).
constexpr int tc_conv_stages(int bn, bool gather, bool pair, bool rsm = false) {
  return gather ? (bn <= 64 ? 4 : 3)
         : rsm  ? (bn == 128 ? 4 : 6)
                : (pair ? (bn == 256 ? 6 : (bn == 128 ? 6 : 8)) : (bn == 256 ? 4 : (bn == 128 ? 6 : 8)));
}
// The bf16 residual is staged in shared memory by TMA (the tcgen05 kernel's EXTM 4) for single-CTA
// whole tiles of 64 or 128 columns with bf16 outputs of K % 8 == 0 channels.
constexpr bool tc_conv_rsm(int bn, bool pair, bool sk, bool res, bool out_bf16, int K) {
  return res && out_bf16 && (K % 8) == 0 && !pair && !sk && (bn == 64 || bn == 128);
}



// 8-bit NHWC (int8 when is_signed, else uint8) -> bf16 bits of (x - zp), exact (|x - zp| <= 255);
// n elements, n % 8 == 0, both pointers 16-byte aligned.
cudaError_t launch_q8_to_bf16(const uint8_t* x, uint16_t* out, long long n, int is_signed, int zp, int num_sms,
                              cudaStream_t stream);

// Pre-activation prologue: bf16 NHWC x -> bf16 bits of clamp(scale[c]*x + shift[c], lo, hi)
// (n elements, C channels; 16-byte aligned pointers).
cudaError_t launch_preact_bf16(const uint16_t* x, uint16_t* out, long long n, int C, const float* scale,
                               const float* shift, float lo, float hi, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- halo-tile implicit GEMM
// Stride-1, dilation-1 convolutions: the output is indexed in rows of Wp = W + pl + pr
// positions (Wp - Wo of them junk), so that every filter tap (r, s) reads the zero-padded
// input at a fixed offset r*Wp + s from the output position.  A tile is TR output rows of one
// image (TR*Wp <= 128 MMA rows); its activation operand for one 64-channel block is ONE TMA box
// of TR + R - 1 padded input rows, loaded once and read by all R*S taps through shifted
// shared-memory descriptors.  Weights stream per (tap, channel block) as in the im2col kernel.
struct HaloParams {
  int Ho, Wo, Wp, TR, R, S, pt, pl;
  int cblocks;            // 64-channel blocks
  int cpad;               // channels per tap in the packed weights (cblocks * 64)
  int Kout, n_blocks, tiles_per_img, num_tiles;
  uint32_t patch_bytes;   // one activation box
  int tpo;                // taps per weight load (divides R*S)
  int b_stages;           // weight stages (2..8) of tpo * BN x 64 bf16
  int resident;           // 1: one output-channel block whose weights fit the stages: loaded once
  const float* scale;     // [Kpad]
  const float* bias;      // [Kpad]
  float* y;               // NHWC fp32 [N*Ho*Wo][Kout], or bf16 bits when out_bf16
  float lo, hi;
  int* status;
  int out_bf16;           // y (and res) hold bf16, rounded to nearest even
  const void* res;        // residual of y's type and shape added before the clamp, or null
};
// BN in {64, 128, 256}; tmA: 4-D tiled {C, W, H, N} box {64, Wp, TR + R - 1, 1} (128 B swizzle),
// tmB: 3-D view {cpad, K, R*S taps} of the packed weights [K][R*S*cpad], box {64, BN, tpo}
// (128 B swizzle)
cudaError_t launch_tc_halo(const HaloParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int bn, int grid,
                           cudaStream_t stream);
// dynamic shared memory of the halo kernel besides its weight stages (total <= 232448)
size_t tc_halo_fixed_smem(int R, int S, int Wp, uint32_t patch_bytes);

// ---------------------------------------------------------------- window-mode implicit GEMM
// Small-C convolutions (C <= 8) whose filter row, for one output pixel, is one contiguous run
// of E bf16 in a channel- and column-padded copy of the input ([N][H][Wp][cpt], the first pl
// columns zero): tile = 128 output pixels of one output row; one 4-D TMA load brings the
// R x 128 overlapping windows of a tile, the weights stay resident in shared memory.
struct WinParams {
  int N, H, Ho, Wo, Kout;
  int sh, pt;             // row stride and top pad (the column offset is in the padded layout)
  int R;                  // filter rows (rows of the A box)
  int bnp;                // output channels rounded up to 32 (MMA N, B rows)
  int ow_blocks, num_tiles;
  int stages;             // A stages in shared memory
  uint32_t a_stage_bytes, b_bytes, b_region;
  uint32_t tmem_cols;
  int chunk0_per_block;   // row mode: 128-byte chunks between consecutive 128-window tiles
  int nchunk;             // row mode: 128-byte chunks of one filter row's input segment
  const uint16_t* w;      // row mode: weights in the no-swizzle core-matrix order (bulk copy)
  const float* scale;     // [>= bnp]
  const float* bias;      // [>= bnp]
  float* y;               // NHWC fp32 output
  float lo, hi;
  int* status;
};
// E = elements per window row (16, 32 or 64); rows = row mode (windows 16 bytes apart: the A
// operand is the plain input row segment, windows overlap through the MMA descriptor)
cudaError_t launch_tc_window(const WinParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int E, bool rows,
                             int grid, size_t smem, cudaStream_t stream);
// shared memory: [1 KB alignment][A stages][B, b_region bytes][epilogue: 8 warps x 4 KB]
// [scale, bias: 256 floats each][barriers and flags]
constexpr size_t kWinFixedSmem = 1024 + 8 * 4096 + 2 * 256 * 4 + 256;
// x [N][H][W][C] -> out [N][H][Wp][cpt] with out column j = x column j - shift (zero outside
// the image and in the channels past C)
cudaError_t launch_window_pad(const uint16_t* x, uint16_t* out, int N, int H, int W, int C, int cpt, int Wp,
                              int shift, int num_sms, cudaStream_t stream);

// NHWC bf16 with C <= 8 channels -> NHWC bf16 with cpt (4 or 8) channels, zero-padded.
cudaError_t launch_pad_channels(const uint16_t* x, uint16_t* out, long long pixels, int C, int cpt, int num_sms,
                                cudaStream_t stream);

// Division by a run-time invariant d >= 1 as a multiply-high, add and shift (the round-up
// method of Granlund and Montgomery, "Division by invariant integers using multiplication",
// 1994): with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, the quotient of any
// n < 2^31 is (umulhi(n, m) + n) >> l, and the sum cannot overflow 32 bits.
struct FastDiv {
  uint32_t d, m, l;
};
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f{d, 0, 0};
  while ((1ull << f.l) < d) ++f.l;
  f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.l) - d)) / d + 1);
  return f;
}
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) { return (__umulhi(n, f.m) + n) >> f.l; }
#endif

// ---------------------------------------------------------------- depthwise (CUDA cores)
struct DwParams {
  int N, C, H, W, Ho, Wo, R, S;
  int sh, sw, pt, pl, dh, dw;
  const uint16_t* x;      // NHWC bf16
  const float* taps;      // [R*S][C] fp32, BN scale folded in
  const float* bias;      // [C]
  float* y;               // NHWC fp32, or bf16 bits when out_bf16
  float lo, hi;
  int* status;            // device status word (watchdog bit)
  FastDiv f_slabs, f_owbs, f_ohbs;   // tile-index decoding (set by the launcher)
  int out_bf16;           // y (and res) hold bf16, rounded to nearest even
  const void* res;        // residual of y's type and shape added before the clamp, or null
};
// tmX: 4-D tiled map {C, W, H, N} of x with box {32, box_w, box_h, box_n} from dw_tile_box();
// used by the 3x3 dilation-1 strides-{1,2} kernel, ignored by the general one.
bool dw_uses_tma(const DwParams& p);
void dw_tile_box(int stride, int Wo, int* box_w, int* box_h, int* box_n);
cudaError_t launch_depthwise(const DwParams& p, const CUtensorMap* tmX, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- grouped conv, direct (CUDA cores)
// Any group count and filter: one thread per (output pixel, output channel), the reduction over
// its group's Cg input channels and the R x S taps in fp32.  The shapes the tensor-core kernels
// cannot take (group windows they cannot align, channel counts TMA cannot address).
struct GdParams {
  int N, C, H, W, K, R, S, Ho, Wo;
  int sh, sw, pt, pl, dh, dw;
  int Cg, Kg;
  const uint16_t* x;      // NHWC bf16
  const float* w;         // [R*S][Cg][K] fp32, BN scale folded in
  const float* bias;      // [K]
  void* y;                // NHWC fp32, or bf16 bits when out_bf16
  const void* res;        // residual of y's type and shape, or null
  int out_bf16;
  float lo, hi;
};
cudaError_t launch_grouped_direct(const GdParams& p, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- fused MobileNetV2 block
// expand 1x1 (+BN, ReLU6) -> depthwise 3x3 (+BN, ReLU6) -> project 1x1 (+BN, + x) in one kernel;
// tiles of TH x TW outputs of one image, the IH x IW input halo (P pixels, rb blocks of 128
// MMA rows) staged by TMA, hidden channels in chunks of 64 (k_mbblock.cu)
struct MbParams {
  int N, H, W, Cin, Ch, Ch_pad, Cout, Ho, Wo, st;
  int TH, TW, IH, IW, P, rb;
  int tiles_h, tiles_w, num_tiles;
  int cin_kb, nch, Np, nsplit;   // input 64-channel blocks, hidden chunks, project N (Cout to 16), N halves
  int expand, residual;          // expand == 0: the t = 1 block (hidden = input)
  int h1_stride;                 // floats per hidden row in shared memory (64 + 4: conflict-free)
  uint32_t x_kb_bytes;           // shared-memory bytes per input channel block (rb * 16 KB)
  uint32_t x_buf_bytes;          // one halo buffer (cin_kb * x_kb_bytes)
  int nxb;                       // halo buffers: 2 (the next tile's halo loads behind this one) or 1
  uint32_t we_buf, wp_buf;       // bytes per expand / project weight buffer (two of each)
  uint32_t x_bytes, we_bytes, wp_bytes;   // TMA transaction bytes
  uint32_t off_x, off_we, off_wp, off_h1, off_a, off_vec, off_bar;   // shared-memory layout (1 KB aligned)
  const float* vec;              // [nch][12][64]: per chunk expand scale, shift, 9 taps, dw shift
  const float* se;               // [Ch_pad] expand BN scale
  const float* be;               // [Ch_pad] expand BN shift
  const float* wd;               // [9][Ch_pad] depthwise taps, BN scale folded
  const float* bd;               // [Ch_pad] depthwise BN shift
  const float* sp;               // [Np] project BN scale
  const float* bp;               // [Np] project BN shift
  float* y;                      // NHWC fp32 [N][Ho][Wo][Cout]
  int* status;
};
// tmX: 4-D {Cin, W, H, N} box {64, IW, IH, 1}; tmWe: 2-D {Cin_pad, Ch_pad} box {64, 64};
// tmWp: 2-D {Ch_pad, Np} box {64, Np / nsplit}; all 128-byte swizzled, zero fill
cudaError_t launch_mbv2_block(const MbParams& p, const CUtensorMap& tmX, const CUtensorMap& tmWe,
                              const CUtensorMap& tmWp, int grid, cudaStream_t stream);
size_t mbv2_block_smem(const MbParams& p);

// ---------------------------------------------------------------- int8 implicit GEMM
struct S8Params {
  int M, Kout, C, H, W, Ho, Wo, R, S;
  int sh, sw, pt, pl, dh, dw;
  int num_kb;             // R*S*C/64
  const int8_t* x;        // NHWC int8
  const int8_t* w;        // [K][R][S][C] int8
  const int32_t* bias;    // [K]
  const int32_t* mult;    // [K]
  const int32_t* shift;  // [K]
  int8_t* y;              // NHWC int8
  int zp, relu;
  int* status;            // device status word (bounds-checking build)
};
cudaError_t launch_s8_conv(const S8Params& p, cudaStream_t stream);
cudaError_t measure_s8_mma_rate(int num_sms, cudaStream_t stream, double* tops);

// ---------------------------------------------------------------- watchdog self-test
cudaError_t launch_watchdog_selftest(int32_t* status, long long budget, cudaStream_t stream);

// ---------------------------------------------------------------- conv chain (tc_chain.cu)
// A sequence of tcgen05 convs (1x1-GEMM or im2col implicit-GEMM steps) run by one persistent
// launch.  Output tiles of 128 rows x bn channels are numbered step after step (row blocks
// major within a step); CTA b takes tiles b, b + grid, b + 2*grid, ...  A tile whose input (or
// residual) is an earlier step's output first waits until the 128-row blocks of that output it
// reads are complete: every 128-row block of every step has a counter, raised by one when one of
// the block's tiles has been stored and made visible (kChainArrivals per tile).  In launch e
// (0, 1, ...) a block is complete when its counter reaches (e + 1) * kChainArrivals * n_blocks
// of its step: the counters only grow, so no launch has to clear them.
constexpr int kChainArrivals = 1;
// The scalar description of one chain step (kept apart from its tensor maps so that a kernel
// role can hold the fields it uses in registers while it works on the step's tiles).
struct ChainGeom {
  int a_mode, a3d;           // AMode (kA2D or kAIm2col); a3d: one box per two k-blocks (2-D mode)
  int M, Kout, C, H, W, Ho, Wo, R, S, sh, sw, pt, pl, dh, dw;
  int cblocks, num_kb, bn, n_blocks, mtiles;
  int tile0, tile_end;       // this step's tiles [tile0, tile_end) in the launch-wide numbering
  uint32_t idesc;            // tcgen05 instruction descriptor: 128 x bn, bf16 inputs, fp32 sums
  float lo, hi;              // activation clamp
  const float* scale;        // [>= n_blocks * bn] epilogue scale (folded BN)
  const float* bias;         // [>= n_blocks * bn] epilogue bias
  const void* x;             // NHWC bf16 input [N][H][W][C] (the activation map's tensor)
  void* y;                   // NHWC [M][Kout], fp32 or bf16 bits (the chain's output type)
  const void* res;           // residual of y's type and shape added before the clamp, or null
  int src;                   // step whose y is this step's x, or -1 (x is written by no step)
  int rsrc;                  // step whose y is this step's residual, or -1
  int src_nb, rsrc_nb;       // n_blocks of those steps (their row blocks' tile counts)
  int consumed;              // a later step reads this step's output: its tiles are published
  uint32_t* done;            // [mtiles] arrival counters of this step's 128-row blocks
  const uint32_t* src_done;  // the source step's counters, or null
  const uint32_t* rsrc_done; // the residual's source step's counters, or null
};
struct ChainStep {
  CUtensorMap tmA;           // activations: 2-D {C, M} box {64, 128}; 3-D {64, M, C/64} box
                             // {64, 128, 2} (a3d); or im2col {C, W, H, N}, 128 pixels x 64 channels
  CUtensorMap tmB;           // weights: 3-D {64, K, num_kb} box {64, bn, 2} over [K][num_kb * 64]
  ChainGeom g;
};
struct ChainParams {
  const ChainStep* steps;    // device array [nsteps]
  int nsteps, total_tiles;
  uint32_t* counters;        // every step's done[] array, total_mtiles words in all
  int total_mtiles;
  uint32_t* state;           // [0] launches completed so far (the epoch), [1] CTAs done this launch
  int* status;               // device status word (timeout / bounds bits), sticky
};
// out_bf16: y and the residuals hold bf16 (else fp32).  pair: CTA pairs (clusters of two, 256-row
// tiles; the step table's tile numbering and weight maps must be made for them).  grid <= the
// CTAs that can be resident at once (tc_chain_max_ctas), even for pairs.
cudaError_t launch_tc_chain(const ChainParams& p, bool out_bf16, bool pair, int grid, cudaStream_t stream);
// CTAs of the chain kernel that can be resident at once on a GPU of num_sms SMs (0 if none)
int tc_chain_max_ctas(bool out_bf16, bool pair, int num_sms);

}  // namespace convf
