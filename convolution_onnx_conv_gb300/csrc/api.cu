// C-ABI of the fused ONNX Conv library: argument validation (refuse, never guess), ONNX
// attribute normalisation, BN fold, weight prepack, the shape-keyed variant selector, tensor
// map encoding and kernel dispatch.  Everything per-call is prepared in create; run only
// (re)encodes the two activation/output tensor maps when the caller's pointers change.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/conv_fused.h"
#include "api_internal.h"
#include "convf_internal.h"

namespace convf {
// defined once per tile width in tc_conv_inst.cu
cudaError_t launch_tc_conv_bn32(const TcConvParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap*, int,
                                bool, bool,
                               cudaStream_t);
cudaError_t launch_tc_conv_bn64(const TcConvParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap*, int,
                                bool, bool,
                               cudaStream_t);
cudaError_t launch_tc_conv_bn128(const TcConvParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap*, int,
                                bool, bool,
                               cudaStream_t);
cudaError_t launch_tc_conv_bn256(const TcConvParams&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap*, int,
                                bool, bool,
                               cudaStream_t);
}  // namespace convf

using namespace convf;

namespace {

constexpr uint32_t kMagic = 0xC0F5ED01u;
constexpr uint32_t kDeadMagic = 0xDEADC0F5u;

thread_local std::string g_last_error;

// Allocation-failure injection (conv_fused_debug_fail_alloc): the countdown reaching zero makes
// that allocation fail.  Live handles are counted by a member of the handle (below).
std::atomic<int> g_fail_countdown{0};
std::atomic<int> g_live_handles{0};

bool injected_alloc_failure() {
  int n = g_fail_countdown.load();
  while (n > 0) {
    if (g_fail_countdown.compare_exchange_weak(n, n - 1)) return n == 1;
  }
  return false;
}

struct LiveHandleCount {
  LiveHandleCount() { g_live_handles.fetch_add(1); }
  LiveHandleCount(const LiveHandleCount&) { g_live_handles.fetch_add(1); }
  LiveHandleCount& operator=(const LiveHandleCount&) = default;
  ~LiveHandleCount() { g_live_handles.fetch_sub(1); }
};

convf_status fail(convf_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}
convf_status ok() {
  g_last_error.clear();
  return CONVF_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------------ attribute normalisation
struct Shape {
  int N, C, H, W, K, R, S, Cg;
  int sh, sw, dh, dw;
  int pt, pl, pb, pr;
  int Ho, Wo;
  long long M;  // N*Ho*Wo
};

long long extent(long long in, long long k, long long st, long long pb, long long pe, long long d) {
  const long long span = in + pb + pe - d * (k - 1) - 1;
  return span < 0 ? 0 : span / st + 1;
}

convf_status resolve(const convf_desc* d, Shape* s) {
  if (!d) return fail(CONVF_ERR_INVALID_ARG, "desc is NULL");
  if (d->N < 0) return fail(CONVF_ERR_INVALID_ARG, "N=%d must be >= 0", d->N);
  const int dims[6] = {d->C, d->H, d->W, d->K, d->R, d->S};
  const char* names[6] = {"C", "H", "W", "K", "R", "S"};
  for (int i = 0; i < 6; ++i)
    if (dims[i] < 1) return fail(CONVF_ERR_INVALID_ARG, "%s=%d must be >= 1", names[i], dims[i]);
  if (d->stride[0] < 1 || d->stride[1] < 1)
    return fail(CONVF_ERR_INVALID_ARG, "strides (%d,%d) must be >= 1", d->stride[0], d->stride[1]);
  if (d->dilation[0] < 1 || d->dilation[1] < 1)
    return fail(CONVF_ERR_INVALID_ARG, "dilations (%d,%d) must be >= 1", d->dilation[0],
                d->dilation[1]);
  if (d->group < 1) return fail(CONVF_ERR_INVALID_ARG, "group=%d must be >= 1", d->group);
  if (d->C % d->group != 0 || d->K % d->group != 0)
    return fail(CONVF_ERR_INVALID_ARG, "group=%d must divide C=%d and K=%d", d->group, d->C, d->K);
  s->N = d->N; s->C = d->C; s->H = d->H; s->W = d->W; s->K = d->K; s->R = d->R; s->S = d->S;
  s->Cg = d->C / d->group;
  s->sh = d->stride[0]; s->sw = d->stride[1]; s->dh = d->dilation[0]; s->dw = d->dilation[1];
  switch (d->auto_pad) {
    case CONVF_AUTO_PAD_NOTSET:
      for (int i = 0; i < 4; ++i)
        if (d->pads[i] < 0) return fail(CONVF_ERR_INVALID_ARG, "pads[%d]=%d must be >= 0", i, d->pads[i]);
      s->pt = d->pads[0]; s->pl = d->pads[1]; s->pb = d->pads[2]; s->pr = d->pads[3];
      break;
    case CONVF_AUTO_PAD_VALID:
      s->pt = s->pl = s->pb = s->pr = 0;
      break;
    case CONVF_AUTO_PAD_SAME_UPPER:
    case CONVF_AUTO_PAD_SAME_LOWER: {
      const int in[2] = {d->H, d->W}, k[2] = {d->R, d->S}, st[2] = {s->sh, s->sw}, dl[2] = {s->dh, s->dw};
      int beg[2], end[2];
      for (int a = 0; a < 2; ++a) {
        const long long out = (in[a] + st[a] - 1) / st[a];
        long long total = (out - 1) * st[a] + (long long)(k[a] - 1) * dl[a] + 1 - in[a];
        if (total < 0) total = 0;
        const long long small = total / 2;
        beg[a] = (int)(d->auto_pad == CONVF_AUTO_PAD_SAME_UPPER ? small : total - small);
        end[a] = (int)(total - beg[a]);
      }
      s->pt = beg[0]; s->pl = beg[1]; s->pb = end[0]; s->pr = end[1];
      break;
    }
    default:
      return fail(CONVF_ERR_INVALID_ARG, "auto_pad=%d is not one of NOTSET/SAME_UPPER/SAME_LOWER/VALID",
                  d->auto_pad);
  }
  const long long Ho = extent(s->H, s->R, s->sh, s->pt, s->pb, s->dh);
  const long long Wo = extent(s->W, s->S, s->sw, s->pl, s->pr, s->dw);
  if (Ho < 1 || Wo < 1)
    return fail(CONVF_ERR_INVALID_ARG, "the %dx%d window (dilation %d,%d) does not fit the padded %dx%d input",
                s->R, s->S, s->dh, s->dw, s->H + s->pt + s->pb, s->W + s->pl + s->pr);
  s->Ho = (int)Ho;
  s->Wo = (int)Wo;
  s->M = (long long)s->N * Ho * Wo;
  const long long lim = 0x7FFFFFFFLL;
  if ((long long)s->N * s->H * s->W * s->C > lim || s->M * s->K > lim ||
      (long long)s->K * s->Cg * s->R * s->S > lim)
    return fail(CONVF_ERR_UNSUPPORTED, "tensor sizes exceed the 2^31-element indexing limit");
  return CONVF_OK;
}

convf_status check_misc(const convf_desc* d) {
  if (d->dtype != CONVF_BF16 && d->dtype != CONVF_S8 && d->dtype != CONVF_Q8)
    return fail(CONVF_ERR_INVALID_ARG, "dtype=%d is not CONVF_BF16, CONVF_S8 or CONVF_Q8", d->dtype);
  if ((d->x_layout != CONVF_NCHW && d->x_layout != CONVF_NHWC) ||
      (d->y_layout != CONVF_NCHW && d->y_layout != CONVF_NHWC))
    return fail(CONVF_ERR_INVALID_ARG, "layouts (%d,%d) must be CONVF_NCHW or CONVF_NHWC", d->x_layout,
                d->y_layout);
  if (d->x_layout != CONVF_NHWC || d->y_layout != CONVF_NHWC)
    return fail(CONVF_ERR_UNSUPPORTED, "only channels-last (CONVF_NHWC) storage is served");
  if (d->act < CONVF_ACT_NONE || d->act > CONVF_ACT_CLIP)
    return fail(CONVF_ERR_INVALID_ARG, "act=%d is not a convf_act", d->act);
  if (d->act == CONVF_ACT_CLIP && !(d->clip_lo <= d->clip_hi))
    return fail(CONVF_ERR_INVALID_ARG, "clip bounds (%g, %g) need lo <= hi", d->clip_lo, d->clip_hi);
  if (d->dtype == CONVF_S8 && (d->act == CONVF_ACT_RELU6 || d->act == CONVF_ACT_CLIP))
    return fail(CONVF_ERR_UNSUPPORTED, "the int8 path serves act NONE or RELU only");
  if (d->variant < CONVF_VARIANT_AUTO || d->variant > CONVF_VARIANT_GROUPED_DIRECT)
    return fail(CONVF_ERR_INVALID_ARG, "variant=%d is not a convf_variant", d->variant);
  if (d->tile_n != 0 && d->tile_n != 32 && d->tile_n != 64 && d->tile_n != 128 && d->tile_n != 256)
    return fail(CONVF_ERR_INVALID_ARG, "tile_n=%d is not 0, 32, 64, 128 or 256", d->tile_n);
  if (d->cta_pair < 0 || d->cta_pair > 2)
    return fail(CONVF_ERR_INVALID_ARG, "cta_pair=%d is not 0 (auto), 1 (single CTA) or 2 (CTA pair)", d->cta_pair);
  if (d->stream_k < 0 || d->stream_k > 2)
    return fail(CONVF_ERR_INVALID_ARG, "stream_k=%d is not 0 (auto), 1 (off) or 2 (on)", d->stream_k);
  if (d->kblocks_per_step < 0 || d->kblocks_per_step > 4)
    return fail(CONVF_ERR_INVALID_ARG, "kblocks_per_step=%d is not 0 (auto) or 1..4", d->kblocks_per_step);
  if (d->out_dtype != CONVF_OUT_F32 && d->out_dtype != CONVF_OUT_BF16)
    return fail(CONVF_ERR_INVALID_ARG, "out_dtype=%d is not CONVF_OUT_F32 (0) or CONVF_OUT_BF16 (1)", d->out_dtype);
  if (d->residual != 0 && d->residual != 1)
    return fail(CONVF_ERR_INVALID_ARG, "residual=%d is not 0 or 1", d->residual);
  return CONVF_OK;
}

// ------------------------------------------------------------------ window-mode geometry
// Padded input rows of Wp pixels x cpt channels with pl zero columns in front; windows of E
// elements (one filter row of one output pixel, zero-padded to 16/32/64); weights [R][bnp][E].
struct WinGeom {
  bool rows;        // row mode: windows exactly 16 bytes apart (sw * cpt == 8)
  int nchunk;       // row mode: 128-byte chunks of one filter row's input segment
  int cpt, E, Wp, bnp, stages, ow_blocks;
  long long tiles;
  uint32_t a_stage, b_bytes, b_region, tmem_cols;
  size_t smem;
};

std::string win_geom(const Shape& s, WinGeom* g) {
  if (s.C > 8) return "window mode needs C <= 8";
  if (s.dh != 1 || s.dw != 1) return "window mode needs dilation 1";
  g->cpt = s.C <= 4 ? 4 : 8;
  if ((s.sw * g->cpt * 2) % 16) return "window mode needs sw*cpt*2 to be a multiple of 16 bytes (stride_w even for C <= 4)";
  if (s.S * g->cpt > 64) return "window mode needs S*cpt <= 64";
  g->E = s.S * g->cpt <= 16 ? 16 : (s.S * g->cpt <= 32 ? 32 : 64);
  if (s.R * g->E > 256) return "window mode needs R*E <= 256 (one 64 KB activation stage)";
  if (s.K > 256) return "window mode needs K <= 256";
  g->bnp = (int)align_up((size_t)s.K, 32);
  g->rows = s.sw * g->cpt == 8;
  const long long need = std::max<long long>((long long)s.pl + s.W, (long long)(s.Wo - 1) * s.sw + g->E / g->cpt);
  // row mode reads whole 128-byte chunks of a row
  g->Wp = (int)align_up((size_t)need, (size_t)(g->rows ? 64 / g->cpt : 16 / (2 * g->cpt)));
  g->nchunk = (int)((127 * 8 + g->E + 63) / 64);
  if ((long long)s.N * s.H * g->Wp * g->cpt > 0x7FFFFFFFLL) return "window mode's padded input exceeds 2^31 elements";
  g->ow_blocks = (s.Wo + 127) / 128;
  g->tiles = (long long)s.N * s.Ho * g->ow_blocks;
  if (g->tiles > 0x7FFFFFFFLL) return "window mode tile count exceeds 2^31";
  g->a_stage = (uint32_t)(g->rows ? s.R * g->nchunk * 128 : s.R * 128 * g->E * 2);
  g->b_bytes = (uint32_t)(s.R * g->bnp * g->E * 2);
  g->b_region = (uint32_t)align_up(g->b_bytes, 1024);
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * g->bnp)) cols *= 2;
  g->tmem_cols = cols;
  const size_t budget = 232448;
  const size_t fixed = kWinFixedSmem + g->b_region;
  const size_t a_stride = align_up(g->a_stage, 1024);   // stages start on 1 KB boundaries
  if (fixed + 2 * a_stride > budget) return "window mode's stages and weights exceed shared memory";
  g->stages = (int)std::min<size_t>(4, (budget - fixed) / a_stride);
  g->smem = fixed + (size_t)g->stages * a_stride;
  return "";
}

// W[K][C][R][S] (bf16 bits) -> per filter row r a bnp x E operand, window element
// e = s*cpt + c, zero elsewhere: row-major [R][bnp][E] (the TMA swizzles it on load), or in row
// mode the no-swizzle core-matrix order: 8 channels x 8 elements per 128 bytes, K-adjacent
// core matrices 128 B apart, 8-channel groups E*16 B apart.
void pack_window(const uint16_t* W, const Shape& s, const WinGeom& g, uint16_t* out) {
  std::memset(out, 0, sizeof(uint16_t) * (size_t)s.R * g.bnp * g.E);
  for (int r = 0; r < s.R; ++r)
    for (int k = 0; k < s.K; ++k)
      for (int q = 0; q < s.S; ++q)
        for (int c = 0; c < s.C; ++c) {
          const int e = q * g.cpt + c;
          const size_t at = g.rows ? (size_t)r * g.bnp * g.E + (size_t)(k / 8) * g.E * 8 + (size_t)(e / 8) * 64 +
                                         (k % 8) * 8 + (e % 8)
                                   : ((size_t)r * g.bnp + k) * g.E + e;
          out[at] = W[(((size_t)k * s.C + c) * s.R + r) * s.S + q];
        }
}

// ------------------------------------------------------------------ halo-tile geometry
struct HaloGeom {
  int Wp, TR, tiles_per_img, cblocks, bn, tpo, b_stages;
  bool resident;    // the whole weight set (one output-channel block) stays in the stages
  uint32_t patch_bytes;
  double valid;     // fraction of the 128 MMA rows of a tile that are real outputs
};

// Tile width for the halo kernel: per 64-channel block a CTA ingests one patch plus R*S weight
// tiles (about 60 B/cycle per SM), issues R*S/tpo weight loads (about 600 cycles each on one
// warp; tpo = the most taps per load within 48 KB) and runs R*S*4 MMAs (48 / 64 / 128 cycles
// each for N = 64 / 128 / 256); minimise waves x the slowest of the three.
std::string halo_geom(const Shape& s, int num_sms, int forced_bn, HaloGeom* g) {
  if (s.sh != 1 || s.sw != 1) return "halo tiles need stride 1";
  if (s.dh != 1 || s.dw != 1) return "halo tiles need dilation 1";
  if (s.R * s.S < 2) return "halo tiles need a filter with more than one tap";
  if (s.R * s.S > 64) return "halo tiles need R*S <= 64";
  if (s.C % 8) return "halo tiles need C % 8 == 0 (16-byte TMA row stride)";
  g->Wp = s.W + s.pl + s.pr;
  if (g->Wp > 128) return "halo tiles need W + pl + pr <= 128";
  g->TR = std::min(128 / g->Wp, s.Ho);
  g->tiles_per_img = (s.Ho + g->TR - 1) / g->TR;
  g->cblocks = (s.C + 63) / 64;
  g->patch_bytes = (uint32_t)((g->TR + s.R - 1) * g->Wp * 128);
  if (g->TR + s.R - 1 > 256) return "halo tiles: patch taller than a TMA box";
  g->valid = (double)g->TR * s.Wo / 128.0;
  double best = 1e300;
  g->bn = 0;
  for (int bn : {64, 128, 256}) {
    if (forced_bn && bn != forced_bn) continue;
    if (!forced_bn && bn > 64 && bn / 2 >= s.K) continue;
    int tpo = 1;
    for (int t = 1; t <= s.R * s.S; ++t)
      if ((s.R * s.S) % t == 0 && (size_t)t * bn * 128 <= 49152) tpo = t;
    const size_t stage = (size_t)tpo * bn * 128;
    const size_t fixed = tc_halo_fixed_smem(s.R, s.S, g->Wp, g->patch_bytes);
    if (fixed + 2 * stage > 232448) continue;
    const int stages = (int)std::min<size_t>(8, (232448 - fixed) / stage);
    const bool res = (s.K + bn - 1) / bn == 1 && g->cblocks * (s.R * s.S / tpo) <= stages;
    const double ingest = g->cblocks * (g->patch_bytes + (res ? 0.0 : (double)s.R * s.S * bn * 128.0)) / 20.0;
    const double issue = res ? 0.0 : g->cblocks * (double)(s.R * s.S / tpo) * 600.0;
    const double mma = (double)g->cblocks * s.R * s.S * 4 * (bn == 64 ? 48.0 : bn == 128 ? 64.0 : 128.0);
    const long long tiles = (long long)s.N * g->tiles_per_img * ((s.K + bn - 1) / bn);
    const long long waves = (tiles + num_sms - 1) / num_sms;
    const double cost = (double)waves * std::max(std::max(ingest, issue), mma);
    if (cost < best * 0.999) {
      best = cost;
      g->bn = bn;
      g->tpo = tpo;
      g->b_stages = stages;
    }
  }
  if (!g->bn) return "halo tiles: the patch and weight stages exceed shared memory";
  g->resident = (s.K + g->bn - 1) / g->bn == 1 && g->cblocks * (s.R * s.S / g->tpo) <= g->b_stages;
  return "";
}

// ------------------------------------------------------------------ variant selector
// A 1x1 filter with unit strides and no padding: the activation operand is a plain matrix.
bool pure_1x1(const Shape& s) {
  return s.R == 1 && s.S == 1 && s.sh == 1 && s.sw == 1 && !s.pt && !s.pl && !s.pb && !s.pr;
}

// Grouped convolution on the tcgen05 kernels: an output-channel tile of bn channels must cover
// whole groups (bn % Kg == 0) or lie inside one (Kg % bn == 0); its reduction then runs over one
// window of input channels -- the groups' channels, cw = max(bn / Kg, 1) * Cg wide, padded to
// 64 -- starting at (n0 / Kg) * Cg, which must be a multiple of 8 channels (16-byte TMA
// coordinates).  The packed weights are block diagonal over that window (zero outside each
// output channel's own group), so the MMA does cwpad / Cg times the grouped conv's work: shapes
// where that exceeds 16 are left to the direct kernel.  The tile width minimises waves x
// per-tile cost, as pick_tile does for dense convs.
struct GroupTile {
  int bn, cwpad;
};

std::string grouped_tile(const Shape& s, int group, int num_sms, int forced_bn, GroupTile* g) {
  const int Kg = s.K / group, Cg = s.Cg;
  double best = 1e300;
  g->bn = 0;
  for (int bn : {32, 64, 128, 256}) {
    if (forced_bn && bn != forced_bn) continue;
    if (bn % Kg != 0 && Kg % bn != 0) continue;
    const int nb = (s.K + bn - 1) / bn;
    bool aligned = true;
    for (int j = 0; j < nb && aligned; ++j) aligned = ((long long)j * bn / Kg) * Cg % 8 == 0;
    if (!aligned) continue;
    const int cw = (bn % Kg == 0 ? bn / Kg : 1) * Cg;
    const int cwpad = (int)align_up((size_t)cw, 64);
    if (cwpad > 16 * Cg) continue;
    const long long tiles = (s.M + 127) / 128 * nb;
    const long long waves = (tiles + num_sms - 1) / num_sms;
    const double kb = bn == 32 ? 670.0 : bn == 64 ? 694.0 : bn == 128 ? 782.0 : 1620.0;
    const double cost = (double)waves * std::max((double)s.R * s.S * (cwpad / 64) * kb, 128.0 * bn * 4.0 / 20.0);
    if (cost < best * 0.999) {
      best = cost;
      g->bn = bn;
      g->cwpad = cwpad;
    }
  }
  if (!g->bn)
    return "grouped convs on the tensor cores need tiles that cover whole groups or lie inside one, 8-channel "
           "aligned group windows and at most 16x block-diagonal padding";
  return "";
}

// Why a shape cannot use a variant ("" = it can).
std::string cannot(int v, const convf_desc* d, const Shape& s) {
  const bool bf = d->dtype == CONVF_BF16;
  char b[256];
  if ((d->out_dtype != CONVF_OUT_F32 || d->residual) && v != CONVF_VARIANT_GEMM_1X1 &&
      v != CONVF_VARIANT_IMPLICIT_GEMM && v != CONVF_VARIANT_GROUPED_DIRECT && v != CONVF_VARIANT_DEPTHWISE &&
      v != CONVF_VARIANT_IMPLICIT_GEMM_HALO)
    return "bf16 output and the residual input are served by the TMA implicit-GEMM, 1x1, halo, depthwise and direct "
           "grouped kernels only";
  switch (v) {
    case CONVF_VARIANT_DEPTHWISE:
      if (!bf) return "depthwise serves bf16 only";
      if (!(d->group == s.C && s.K == s.C)) return "depthwise needs group == C == K";
      if (s.C % 8) return "depthwise needs C % 8 == 0 (16-byte channel vectors)";
      return "";
    case CONVF_VARIANT_GEMM_1X1:
      if (!bf) return "1x1 GEMM serves bf16 only";
      if (d->group != 1) {
        if (d->cta_pair == 2 || d->stream_k == 2) return "grouped convs run on single CTAs without stream-K";
        GroupTile g;
        const std::string why = grouped_tile(s, d->group, 148, d->tile_n, &g);
        if (!why.empty()) return why;
      }
      if (s.R != 1 || s.S != 1 || s.sh != 1 || s.sw != 1 || s.pt || s.pl || s.pb || s.pr)
        return "1x1 GEMM needs a 1x1 filter, unit strides and no padding";
      if (s.C % 8) return "1x1 GEMM needs C % 8 == 0 (16-byte TMA row stride)";
      if (s.K % 4) return "the tcgen05 kernels need K % 4 == 0 (16-byte TMA output row stride)";
      return "";
    case CONVF_VARIANT_IMPLICIT_GEMM:
      if (!bf) return "implicit GEMM serves bf16 only";
      if (d->group != 1) {
        if (d->cta_pair == 2 || d->stream_k == 2) return "grouped convs run on single CTAs without stream-K";
        GroupTile g;
        const std::string why = grouped_tile(s, d->group, 148, d->tile_n, &g);
        if (!why.empty()) return why;
      }
      if (s.C % 8) return "TMA im2col needs C % 8 == 0 (use the gather variant)";
      if (s.K % 4) return "the tcgen05 kernels need K % 4 == 0 (16-byte TMA output row stride)";
      if (s.sh > 8 || s.sw > 8) return "TMA im2col traversal strides are limited to 8";
      if (s.pt > 128 || s.pl > 128) return "TMA im2col box corners are limited to [-128, 127]";
      if ((long long)(s.R - 1) * s.dh - s.pb > 128 || (long long)(s.S - 1) * s.dw - s.pr > 128 ||
          s.pb - (long long)(s.R - 1) * s.dh > 127 || s.pr - (long long)(s.S - 1) * s.dw > 127)
        return "TMA im2col box corners are limited to [-128, 127]";
      if ((long long)(s.R - 1) * s.dh > 65535 || (long long)(s.S - 1) * s.dw > 65535)
        return "filter offsets exceed 16 bits";
      return "";
    case CONVF_VARIANT_IMPLICIT_GEMM_HALO: {
      if (!bf) return "implicit GEMM serves bf16 only";
      if (d->group != 1) return "implicit GEMM needs group == 1";
      if (s.K % 4) return "the tcgen05 kernels need K % 4 == 0 (16-byte output row stride)";
      if (d->tile_n == 32) return "halo tiles come 64, 128 or 256 channels wide";
      HaloGeom g;
      return halo_geom(s, 148, d->tile_n, &g);
    }
    case CONVF_VARIANT_IMPLICIT_GEMM_WINDOW: {
      if (!bf) return "implicit GEMM serves bf16 only";
      if (d->group != 1) return "implicit GEMM needs group == 1";
      if (s.K % 4) return "the tcgen05 kernels need K % 4 == 0 (16-byte TMA output row stride)";
      WinGeom g;
      return win_geom(s, &g);
    }
    case CONVF_VARIANT_IMPLICIT_GEMM_GATHER:
      if (!bf) return "implicit GEMM serves bf16 only";
      if (d->group != 1) return "implicit GEMM needs group == 1";
      if (s.K % 4) return "the tcgen05 kernels need K % 4 == 0 (16-byte TMA output row stride)";
      return "";
    case CONVF_VARIANT_GROUPED_DIRECT:
      if (!bf) return "the direct grouped kernel serves bf16 only";
      return "";
    case CONVF_VARIANT_INT8:
      if (d->dtype != CONVF_S8) return "the mma.sync int8 kernel serves CONVF_S8 only";
      if (d->group != 1) return "the int8 kernel needs group == 1";
      if (s.C % 64) return "the int8 kernel needs C % 64 == 0";
      if (s.K % 16) return "the int8 kernel needs K % 16 == 0";
      return "";
    case CONVF_VARIANT_INT8_TC:
      if (bf) return "the exact-integer tcgen05 kernel serves CONVF_S8 and CONVF_Q8 only";
      if (d->group != 1) return "the exact-integer tcgen05 kernel needs group == 1";
      if (s.C % 8) return "the exact-integer tcgen05 kernel needs C % 8 == 0 (16-byte rows of its bf16 staging copy)";
      if (s.K % 16) return "the exact-integer tcgen05 kernel needs K % 16 == 0 (16-byte 8-bit output groups)";
      if (pure_1x1(s)) return "";
      if (s.sh > 8 || s.sw > 8) return "TMA im2col traversal strides are limited to 8";
      if (s.pt > 128 || s.pl > 128) return "TMA im2col box corners are limited to [-128, 127]";
      if ((long long)(s.R - 1) * s.dh - s.pb > 128 || (long long)(s.S - 1) * s.dw - s.pr > 128 ||
          s.pb - (long long)(s.R - 1) * s.dh > 127 || s.pr - (long long)(s.S - 1) * s.dw > 127)
        return "TMA im2col box corners are limited to [-128, 127]";
      if ((long long)(s.R - 1) * s.dh > 65535 || (long long)(s.S - 1) * s.dw > 65535)
        return "filter offsets exceed 16 bits";
      return "";
  }
  snprintf(b, sizeof b, "unknown variant %d", v);
  return b;
}

convf_status select_variant(const convf_desc* d, const Shape& s, int* out) {
  if (d->variant != CONVF_VARIANT_AUTO) {
    std::string why = cannot(d->variant, d, s);
    if (!why.empty()) return fail(CONVF_ERR_UNSUPPORTED, "forced variant %d refused: %s", d->variant, why.c_str());
    *out = d->variant;
    return CONVF_OK;
  }
  // (the direct grouped kernel last: it takes only what no tensor-core kernel can)
  const int order_bf16[7] = {CONVF_VARIANT_DEPTHWISE, CONVF_VARIANT_GEMM_1X1, CONVF_VARIANT_IMPLICIT_GEMM_HALO,
                             CONVF_VARIANT_IMPLICIT_GEMM, CONVF_VARIANT_IMPLICIT_GEMM_WINDOW,
                             CONVF_VARIANT_IMPLICIT_GEMM_GATHER, CONVF_VARIANT_GROUPED_DIRECT};
  if (d->dtype == CONVF_S8 || d->dtype == CONVF_Q8) {
    // exact integers on tcgen05 first; static int8 falls back to the warp-level MMA kernel
    std::string why = cannot(CONVF_VARIANT_INT8_TC, d, s);
    if (why.empty()) {
      *out = CONVF_VARIANT_INT8_TC;
      return CONVF_OK;
    }
    if (d->dtype == CONVF_Q8) return fail(CONVF_ERR_UNSUPPORTED, "QLinearConv refused: %s", why.c_str());
    std::string why2 = cannot(CONVF_VARIANT_INT8, d, s);
    if (!why2.empty())
      return fail(CONVF_ERR_UNSUPPORTED, "int8 conv refused: %s; %s", why.c_str(), why2.c_str());
    *out = CONVF_VARIANT_INT8;
    return CONVF_OK;
  }
  std::string reasons;
  for (int v : order_bf16) {
    std::string why = cannot(v, d, s);
    // a tile is one output row segment of 128 pixels: narrower outputs leave most rows idle
    if (why.empty() && v == CONVF_VARIANT_IMPLICIT_GEMM_WINDOW && s.Wo < 32)
      why = "window mode is chosen automatically only for outputs at least 32 pixels wide";
    // the direct kernel is a fallback for grouped convs only: a dense conv the tensor-core kernels
    // refuse (e.g. a bf16-output stem) is refused rather than moved to CUDA cores
    if (why.empty() && v == CONVF_VARIANT_GROUPED_DIRECT && d->group == 1)
      why = "the direct grouped kernel is chosen automatically only for grouped convs";
    if (why.empty() && v == CONVF_VARIANT_IMPLICIT_GEMM_HALO) {
      HaloGeom g;
      halo_geom(s, 148, d->tile_n, &g);
      if (g.valid < 0.6) why = "halo tiles are chosen automatically only when 60% of a tile's rows are outputs";
      // measured: without resident weights the per-tile weight stream makes halo tiles no faster
      // than TMA im2col
      else if (!g.resident) why = "halo tiles are chosen automatically only when the weights stay resident";
      if (d->cta_pair == 2 || d->stream_k == 2) why = "halo tiles run on single CTAs without stream-K";
    }
    if (why.empty()) {
      *out = v;
      return CONVF_OK;
    }
    reasons += (reasons.empty() ? "" : "; ") + why;
  }
  return fail(CONVF_ERR_UNSUPPORTED, "no kernel serves this conv: %s", reasons.c_str());
}

// Tile shape for the tcgen05 kernels: minimise the time of the busiest CTA.  Per 64-wide
// reduction block a single CTA spends about {670, 694, 782, 1620} SM cycles for tile widths
// {32, 64, 128, 256} (measured on GB300 over the ResNet-50 layers: each SM ingests operands at
// about 43 B/cycle, plus pipeline overheads); a tile also writes 128 x bn fp32 outputs at about
// 20 B/cycle per SM; the busiest CTA runs ceil(tiles / CTAs) tiles.
// CTA pairs (256-row tiles, half the weight tile per CTA) cut the ingested bytes but measured
// slower on every ResNet-50 layer (longer cross-SM handshakes), so they are used only when
// requested: pair_mode 0 = auto (single CTAs), 1 = single, 2 = pairs.  Stream-K likewise
// measured slower on the ResNet-50 layers it would pick (the partial write-back and read-back
// run at the epilogue's store rate, about 13 B/cycle per SM, and sit on the critical path), so
// auto keeps whole tiles: sk_mode 0 = auto (off), 1 = off, 2 = on (single CTAs only; ignored
// with pairs or when sk_ok is false).
// k-blocks per pipeline step of the TMA implicit-GEMM kernel: the first of 4, 2, 3 that divides
// the stage count and the tile's k-blocks and still leaves two steps in flight (measured on the
// ResNet-50 layers: 4 beats 2 on 128 x 64 tiles, 2 matches or beats 3 on 128 x 128 tiles).
int auto_kblocks_per_step(int stages, int num_kb) {
  for (int k : {4, 2, 3})
    if (stages % k == 0 && num_kb % k == 0 && stages / k >= 2) return k;
  return 1;
}

void pick_tile(long long M, int K, int num_kb, int num_sms, int max_bn, int pair_mode, int sk_mode, bool sk_ok,
               int* bn_out, bool* pair_out, bool* sk_out) {
  const bool pair = pair_mode == 2;
  const long long tile_m = pair ? 256 : 128;
  const long long units = pair ? num_sms / 2 : num_sms;
  const bool sk_allowed = sk_ok && !pair && sk_mode != 1;
  int best_bn = max_bn;
  bool best_sk = false;
  double best_cost = 1e300;
  for (int bn : {256, 128, 64, 32}) {
    if (bn > max_bn) continue;
    if (bn > 32 && bn / 2 >= K && bn != max_bn) continue;  // no point in a tile twice as wide as K
    const long long tiles = (M + tile_m - 1) / tile_m * ((K + bn - 1) / bn);
    const long long waves = (tiles + units - 1) / units;
    const double kb_cycles = bn == 32 ? 670.0 : bn == 64 ? 694.0 : bn == 128 ? 782.0 : 1620.0;
    const double per_tile = std::max(num_kb * kb_cycles, 128.0 * bn * 4.0 / 20.0);
    double cost = (double)waves * per_tile;
    bool sk = false;
    if (sk_allowed && sk_mode == 2 && num_kb >= 2) sk = true;
    if (cost < best_cost * 0.999) {
      best_cost = cost;
      best_bn = bn;
      best_sk = sk;
    }
  }
  *bn_out = best_bn;
  *pair_out = pair;
  *sk_out = best_sk;
}

// Gather variant: input rows one 128-pixel tile reads, staged whole in shared memory, when
// tiles never straddle two images, rows are 16-byte multiples and the rows fit one 32 KB
// buffer; 0 means the gatherers read global memory directly.
int patch_rows_for(const Shape& s, int channels) {
  const long long hw = (long long)s.Ho * s.Wo;
  if (hw % 128 != 0) return 0;
  const long long row_bytes = (long long)s.W * channels * 2;
  if (row_bytes % 16 != 0) return 0;
  long long q = (127 + s.Wo - 1) / s.Wo + 1;   // output rows one tile can touch
  if (q > s.Ho) q = s.Ho;
  const long long rows = (q - 1) * s.sh + (long long)(s.R - 1) * s.dh + 1;
  if (rows * row_bytes > 32768) return 0;
  return (int)rows;
}

// Gather variant with at most 8 channels and staged rows: the reduction is laid out as whole
// taps of cpt = 4 or 8 channels (zero-padded), assembled with one vector read per tap; 0 keeps
// the channel-by-channel layout.
int gather_cpt(const Shape& s) {
  if (s.C > 8) return 0;
  const int cpt = s.C <= 4 ? 4 : 8;
  return patch_rows_for(s, cpt) > 0 ? cpt : 0;
}

// ------------------------------------------------------------------ driver entry points
EncodeTiledFn g_encode_tiled = nullptr;
EncodeIm2colFn g_encode_im2col = nullptr;
std::once_flag g_encode_once;

bool load_encoders() {
  std::call_once(g_encode_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode_tiled = reinterpret_cast<EncodeTiledFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode_im2col = reinterpret_cast<EncodeIm2colFn>(f);
  });
  return g_encode_tiled && g_encode_im2col;
}

}  // namespace

// ====================================================================== handle
struct convf_handle {
  LiveHandleCount live;   // counts the handles in existence (conv_fused_debug_live_handles)
  uint32_t magic;
  convf_desc desc;
  Shape s;
  int variant;
  int device;
  int num_sms;
  // one device allocation carved into the arrays below
  void* dev;
  size_t dev_bytes;
  uint16_t* w_bf16;
  int8_t* w_s8;
  float* taps;
  float* scale;
  float* bias;
  int32_t* qbias;
  int32_t* qmult;
  int32_t* qshift;
  uint16_t* xpad;   // gather variant with padded channels: x with cpt channels per pixel
  int* status;
  int32_t zp;
  float lo, hi;
  // tcgen05 configuration
  int bn, a_mode, num_kb, cblocks, ktot, grid, num_tiles, n_blocks, patch_rows, row_bytes, cpt;
  bool pair;        // CTA-pair (cta_group::2) 256-row tiles
  bool out_bf16;    // y (and the residual) are bf16
  bool has_res;     // runs add a residual tensor (conv_fused_run_residual)
  bool sk;          // stream-K work split
  int kpb;          // k-blocks per pipeline step (TcConvParams::kpb)
  bool a3d;         // 1x1 activation map is 3-D {64, M, C/64} (one box per step)
  float* sk_ws;     // stream-K: one 128 x bn fp32 partial per CTA
  int* sk_flags;    // stream-K: one flag per CTA (zero between launches)
  // exact-integer tcgen05 variant (8-bit convs)
  uint16_t* xq;     // bf16 staging copy of x - x_zero_point, written by the pre-pass each run
  int x_signed, x_zp, iq_chunk_kb, iq_mode, q_lo, q_hi;
  int32_t* q_bias;
  int32_t* q_mult;
  int32_t* q_shift;
  float* q_scale;
  // pre-activation prologue: a bf16 copy u = clamp(pre_scale*x + pre_shift) read instead of x
  bool preact;
  uint16_t* xs;
  float* pre_scale;
  float* pre_shift;
  float pre_lo, pre_hi;
  MbParams mb;      // fused MobileNetV2 block: geometry and device arrays
  CUtensorMap tmWe, tmWp;
  WinGeom wg;       // window variant geometry
  HaloGeom hg;      // halo variant geometry
  CUtensorMap tmB;
  CUtensorMap tmA;
  const void* map_x;
  bool rsm;         // the bf16 residual is staged in shared memory by TMA (its map: tmR)
  CUtensorMap tmR;
  const void* map_r;
};

namespace {

convf_status check_handle(const convf_handle* h) {
  if (!h) return fail(CONVF_ERR_INVALID_ARG, "handle is NULL");
  if (h->magic == kDeadMagic) return fail(CONVF_ERR_INVALID_ARG, "handle was destroyed");
  if (h->magic != kMagic) return fail(CONVF_ERR_INVALID_ARG, "not a convf handle");
  return CONVF_OK;
}

void act_bounds(const convf_desc* d, float* lo, float* hi) {
  switch (d->act) {
    case CONVF_ACT_RELU: *lo = 0.f; *hi = INFINITY; break;
    case CONVF_ACT_RELU6: *lo = 0.f; *hi = 6.f; break;
    case CONVF_ACT_CLIP: *lo = d->clip_lo; *hi = d->clip_hi; break;
    default: *lo = -INFINITY; *hi = INFINITY; break;
  }
}

// Prepacked weight layout for the tcgen05 variants: row length ktot (elements) and the
// channel stride cpad of each tap's run inside a row.
void tc_layout(int variant, const Shape& s, int* a_mode, int* cblocks, int* ktot, int* cpad) {
  if (variant == CONVF_VARIANT_GEMM_1X1) {
    *a_mode = kA2D;
    *cblocks = (s.C + 63) / 64;
    *ktot = *cblocks * 64;
    *cpad = *ktot;
  } else if (variant == CONVF_VARIANT_IMPLICIT_GEMM || variant == CONVF_VARIANT_IMPLICIT_GEMM_HALO) {
    *a_mode = kAIm2col;
    *cblocks = (s.C + 63) / 64;
    *cpad = *cblocks * 64;
    *ktot = s.R * s.S * *cpad;
  } else {
    *a_mode = kAGather;
    *cblocks = 0;
    const int cpt = gather_cpt(s);
    *cpad = cpt ? cpt : s.C;
    *ktot = (int)align_up((size_t)s.R * s.S * *cpad, 64);
  }
}

// W[K][C][R][S] (bf16 bits) -> [K][ktot]: reduction index (r*S + s)*cpad + c, zero elsewhere.
void pack_bf16(const uint16_t* W, const Shape& s, int cpad, int ktot, uint16_t* out) {
  std::memset(out, 0, sizeof(uint16_t) * (size_t)s.K * ktot);
  for (int k = 0; k < s.K; ++k)
    for (int c = 0; c < s.C; ++c)
      for (int r = 0; r < s.R; ++r)
        for (int q = 0; q < s.S; ++q)
          out[(size_t)k * ktot + (size_t)(r * s.S + q) * cpad + c] =
              W[(((size_t)k * s.C + c) * s.R + r) * s.S + q];
}

// Grouped: W[K][Cg][R][S] -> [K][ktot], row k = output channel of group k / Kg in the tile of bn
// channels whose window starts at input channel cb0 = (n0 / Kg) * Cg: element (r*S + s)*cpad + c
// holds W[k][cb0 + c - (k / Kg) * Cg][r][s] when that channel is in k's group, else zero.
void pack_bf16_grouped(const uint16_t* W, const Shape& s, int group, int bn, int cpad, int ktot, uint16_t* out) {
  std::memset(out, 0, sizeof(uint16_t) * (size_t)s.K * ktot);
  const int Kg = s.K / group, Cg = s.Cg;
  for (int k = 0; k < s.K; ++k) {
    const int cb0 = ((k / bn) * bn / Kg) * Cg;
    const int off = (k / Kg) * Cg - cb0;   // position of k's group inside the window
    for (int c = 0; c < Cg; ++c)
      for (int r = 0; r < s.R; ++r)
        for (int q = 0; q < s.S; ++q)
          out[(size_t)k * ktot + (size_t)(r * s.S + q) * cpad + off + c] = W[(((size_t)k * Cg + c) * s.R + r) * s.S + q];
  }
}

float bf16_to_f32(uint16_t v) {
  uint32_t u = (uint32_t)v << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

const char* conv_fused_last_error(void) { return g_last_error.c_str(); }

convf_status conv_fused_resolve_pads(const convf_desc* desc, int pads_out[4]) {
  Shape s;
  convf_status st = resolve(desc, &s);
  if (st != CONVF_OK) return st;
  if (!pads_out) return fail(CONVF_ERR_INVALID_ARG, "pads_out is NULL");
  pads_out[0] = s.pt; pads_out[1] = s.pl; pads_out[2] = s.pb; pads_out[3] = s.pr;
  return ok();
}

convf_status conv_fused_output_shape(const convf_desc* desc, int out_nchw[4]) {
  Shape s;
  convf_status st = resolve(desc, &s);
  if (st != CONVF_OK) return st;
  if (!out_nchw) return fail(CONVF_ERR_INVALID_ARG, "out_nchw is NULL");
  out_nchw[0] = s.N; out_nchw[1] = s.K; out_nchw[2] = s.Ho; out_nchw[3] = s.Wo;
  return ok();
}

convf_status conv_bn_scale_shift(int K, const float* gamma, const float* beta, const float* mean,
                                 const float* var, float eps, float* scale, float* shift) {
  if (K < 1) return fail(CONVF_ERR_INVALID_ARG, "K=%d must be >= 1", K);
  if (!gamma || !beta || !mean || !var || !scale || !shift)
    return fail(CONVF_ERR_INVALID_ARG, "a BN array is NULL");
  if (!(eps > 0.f)) return fail(CONVF_ERR_INVALID_ARG, "eps=%g must be > 0", eps);
  for (int k = 0; k < K; ++k) {
    const double v = (double)var[k] + (double)eps;
    if (!(v > 0.0)) return fail(CONVF_ERR_INVALID_ARG, "var[%d] + eps = %g is not positive", k, v);
    const double sc = (double)gamma[k] / std::sqrt(v);
    scale[k] = (float)sc;
    shift[k] = (float)((double)beta[k] - (double)mean[k] * sc);
  }
  return ok();
}

// Host-only view of the selector: the variant and tcgen05 tile width create would choose for
// `desc` on a GPU with `num_sms` SMs (no CUDA call).
convf_status conv_fused_plan(const convf_desc* desc, int num_sms, int* variant, int* tile_n, int* ktot,
                             int* cta_pair) {
  if (cta_pair) *cta_pair = 0;
  Shape s;
  convf_status st = resolve(desc, &s);
  if (st != CONVF_OK) return st;
  if ((st = check_misc(desc)) != CONVF_OK) return st;
  int v = 0;
  if ((st = select_variant(desc, s, &v)) != CONVF_OK) return st;
  if (variant) *variant = v;
  int bn = 0, kt = 0;
  if (v == CONVF_VARIANT_GEMM_1X1 || v == CONVF_VARIANT_IMPLICIT_GEMM || v == CONVF_VARIANT_IMPLICIT_GEMM_GATHER) {
    int am, cb, cp;
    tc_layout(v, s, &am, &cb, &kt, &cp);
    const bool gather = v == CONVF_VARIANT_IMPLICIT_GEMM_GATHER;
    const int max_bn = gather ? 128 : 256;
    if (desc->tile_n > max_bn)
      return fail(CONVF_ERR_UNSUPPORTED, "tile_n=%d exceeds %d for the gather variant", desc->tile_n, max_bn);
    if (gather && desc->cta_pair == 2)
      return fail(CONVF_ERR_UNSUPPORTED, "the gather variant runs on single CTAs");
    bool pair = false, sk = false;
    pick_tile(s.M, s.K, kt / 64, num_sms > 1 ? num_sms : 2, desc->tile_n ? desc->tile_n : max_bn,
              gather ? 1 : desc->cta_pair, desc->stream_k, !gather, &bn, &pair, &sk);
    if (desc->tile_n) bn = desc->tile_n;
    if (desc->group > 1) {
      GroupTile g;
      grouped_tile(s, desc->group, num_sms > 1 ? num_sms : 2, desc->tile_n, &g);
      bn = g.bn;
      kt = v == CONVF_VARIANT_GEMM_1X1 ? g.cwpad : s.R * s.S * g.cwpad;
      pair = false;
    }
    if (cta_pair) *cta_pair = pair ? 1 : 0;
  } else if (v == CONVF_VARIANT_IMPLICIT_GEMM_HALO) {
    HaloGeom g;
    halo_geom(s, num_sms > 1 ? num_sms : 2, desc->tile_n, &g);
    int am, cb, cp;
    tc_layout(v, s, &am, &cb, &kt, &cp);
    bn = g.bn;
  } else if (v == CONVF_VARIANT_IMPLICIT_GEMM_WINDOW) {
    WinGeom g;
    win_geom(s, &g);
    bn = g.bnp;
    kt = s.R * g.E;
  } else if (v == CONVF_VARIANT_INT8) {
    kt = s.R * s.S * s.C;
  } else if (v == CONVF_VARIANT_INT8_TC) {
    int am, cb, cp;
    tc_layout(pure_1x1(s) ? CONVF_VARIANT_GEMM_1X1 : CONVF_VARIANT_IMPLICIT_GEMM, s, &am, &cb, &kt, &cp);
    bool pair = false, sk = false;
    pick_tile(s.M, s.K, kt / 64, num_sms > 1 ? num_sms : 2, 128, 1, 1, false, &bn, &pair, &sk);
    if (bn < 64) bn = 64;
    if (desc->tile_n == 64 || desc->tile_n == 128) bn = desc->tile_n;
  }
  if (tile_n) *tile_n = bn;
  if (ktot) *ktot = kt;
  return ok();
}

// Host-only prepack of bf16 weights for a tcgen05 variant ([K][ktot], see pack_bf16).
convf_status conv_fused_pack_weights(const convf_desc* desc, int variant, const uint16_t* W, uint16_t* out,
                                     size_t out_elems) {
  Shape s;
  convf_status st = resolve(desc, &s);
  if (st != CONVF_OK) return st;
  if (!W || !out) return fail(CONVF_ERR_INVALID_ARG, "W/out is NULL");
  if (variant != CONVF_VARIANT_GEMM_1X1 && variant != CONVF_VARIANT_IMPLICIT_GEMM &&
      variant != CONVF_VARIANT_IMPLICIT_GEMM_GATHER && variant != CONVF_VARIANT_IMPLICIT_GEMM_HALO)
    return fail(CONVF_ERR_INVALID_ARG, "variant %d has no bf16 GEMM packing", variant);
  if (desc->group != 1) return fail(CONVF_ERR_UNSUPPORTED, "GEMM packing needs group == 1");
  int am, cb, kt, cp;
  tc_layout(variant, s, &am, &cb, &kt, &cp);
  if (out_elems < (size_t)s.K * kt) return fail(CONVF_ERR_INVALID_ARG, "out holds %zu < %zu elements", out_elems,
                                                (size_t)s.K * kt);
  pack_bf16(W, s, cp, kt, out);
  return ok();
}

namespace {
convf_status encode_a_map(convf_handle* h, const void* x);   // below, with the run path

int q8_lo(int is_signed) { return is_signed ? -128 : 0; }
int q8_hi(int is_signed) { return is_signed ? 127 : 255; }

convf_status create_impl(const convf_desc* desc, const void* W, const void* bias, const float* bn_scale,
                         const float* bn_shift, const int32_t* requant_mult, const int32_t* requant_shift,
                         int32_t out_zero_point, const convf_qparams* qp, convf_handle** out,
                         const float* pre_scale = nullptr, const float* pre_shift = nullptr, int pre_act = -1) {
  if (!out) return fail(CONVF_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  Shape s;
  convf_status st = resolve(desc, &s);
  if (st != CONVF_OK) return st;
  if ((st = check_misc(desc)) != CONVF_OK) return st;
  if (!W) return fail(CONVF_ERR_INVALID_ARG, "W is NULL");
  const bool s8 = desc->dtype == CONVF_S8;
  const bool q8 = desc->dtype == CONVF_Q8;
  if (q8 != (qp != nullptr))
    return fail(CONVF_ERR_INVALID_ARG, q8 ? "CONVF_Q8 handles are made by conv_fused_create_qlinear"
                                          : "conv_fused_create_qlinear needs desc->dtype == CONVF_Q8");
  if (q8) {
    if (!qp->w_zero_point || !qp->w_scale) return fail(CONVF_ERR_INVALID_ARG, "w_zero_point/w_scale is NULL");
    for (int v : {qp->x_signed, qp->w_signed, qp->y_signed, qp->relu})
      if (v != 0 && v != 1) return fail(CONVF_ERR_INVALID_ARG, "x_signed/w_signed/y_signed/relu must be 0 or 1");
    if (qp->x_zero_point < q8_lo(qp->x_signed) || qp->x_zero_point > q8_hi(qp->x_signed))
      return fail(CONVF_ERR_INVALID_ARG, "x_zero_point=%d is outside x's type", qp->x_zero_point);
    if (qp->y_zero_point < q8_lo(qp->y_signed) || qp->y_zero_point > q8_hi(qp->y_signed))
      return fail(CONVF_ERR_INVALID_ARG, "y_zero_point=%d is outside y's type", qp->y_zero_point);
    if (!(std::isfinite(qp->x_scale) && qp->x_scale > 0.f) || !(std::isfinite(qp->y_scale) && qp->y_scale > 0.f))
      return fail(CONVF_ERR_INVALID_ARG, "x_scale and y_scale must be finite and > 0");
    for (int k = 0; k < s.K; ++k) {
      if (qp->w_zero_point[k] < q8_lo(qp->w_signed) || qp->w_zero_point[k] > q8_hi(qp->w_signed))
        return fail(CONVF_ERR_INVALID_ARG, "w_zero_point[%d]=%d is outside w's type", k, qp->w_zero_point[k]);
      if (!(std::isfinite(qp->w_scale[k]) && qp->w_scale[k] > 0.f))
        return fail(CONVF_ERR_INVALID_ARG, "w_scale[%d] must be finite and > 0", k);
    }
    if (bn_scale || bn_shift || requant_mult || requant_shift)
      return fail(CONVF_ERR_INVALID_ARG, "BN and fixed-point requant arrays do not apply to QLinearConv");
  }
  if (s8) {
    if (bn_scale || bn_shift) return fail(CONVF_ERR_INVALID_ARG, "bn_scale/bn_shift must be NULL on the int8 path");
    if (!requant_mult || !requant_shift) return fail(CONVF_ERR_INVALID_ARG, "requant_mult/requant_shift are required on the int8 path");
    if (out_zero_point < -128 || out_zero_point > 127)
      return fail(CONVF_ERR_INVALID_ARG, "out_zero_point=%d is outside int8", out_zero_point);
    for (int k = 0; k < s.K; ++k) {
      if (requant_mult[k] <= 0) return fail(CONVF_ERR_INVALID_ARG, "requant_mult[%d]=%d must be > 0", k, requant_mult[k]);
      if (requant_shift[k] < 1 || requant_shift[k] > 62)
        return fail(CONVF_ERR_INVALID_ARG, "requant_shift[%d]=%d must be in 1..62", k, requant_shift[k]);
    }
  } else {
    if ((bn_scale == nullptr) != (bn_shift == nullptr))
      return fail(CONVF_ERR_INVALID_ARG, "bn_scale and bn_shift must be given together");
    if (bn_scale)
      for (int k = 0; k < s.K; ++k)
        if (!std::isfinite(bn_scale[k]) || !std::isfinite(bn_shift[k]))
          return fail(CONVF_ERR_INVALID_ARG, "bn_scale/bn_shift[%d] is not finite", k);
  }
  const bool preact = pre_act >= 0;
  if (preact) {
    if (desc->dtype != CONVF_BF16) return fail(CONVF_ERR_UNSUPPORTED, "the pre-activation prologue serves bf16 convs only");
    if (!pre_scale || !pre_shift) return fail(CONVF_ERR_INVALID_ARG, "pre_scale/pre_shift is NULL");
    if (pre_act != CONVF_ACT_NONE && pre_act != CONVF_ACT_RELU && pre_act != CONVF_ACT_RELU6)
      return fail(CONVF_ERR_INVALID_ARG, "pre_act=%d is not CONVF_ACT_NONE, _RELU or _RELU6", pre_act);
    for (int c = 0; c < s.C; ++c)
      if (!std::isfinite(pre_scale[c]) || !std::isfinite(pre_shift[c]))
        return fail(CONVF_ERR_INVALID_ARG, "pre_scale/pre_shift[%d] is not finite", c);
  }
  int variant = 0;
  if ((st = select_variant(desc, s, &variant)) != CONVF_OK) return st;

  // ---------------------------------------------------------------- host-side prep
  const bool host_injected = injected_alloc_failure();
  convf_handle* h = host_injected ? nullptr : new (std::nothrow) convf_handle();
  if (!h) return fail(CONVF_ERR_OOM, "host allocation failed%s", host_injected ? " (injected)" : "");
  h->desc = *desc;
  h->out_bf16 = desc->out_dtype == CONVF_OUT_BF16;
  h->has_res = desc->residual != 0;
  h->s = s;
  h->variant = variant;
  h->zp = out_zero_point;
  act_bounds(desc, &h->lo, &h->hi);

  cudaError_t ce = cudaGetDevice(&h->device);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (ce != cudaSuccess) {
    delete h;
    return fail(CONVF_ERR_CUDA, "no usable CUDA device: %s", cudaGetErrorString(ce));
  }
  int cc_major = 0, cc_minor = 0;
  cudaDeviceGetAttribute(&cc_major, cudaDevAttrComputeCapabilityMajor, h->device);
  cudaDeviceGetAttribute(&cc_minor, cudaDevAttrComputeCapabilityMinor, h->device);
  if (cc_major != 10 || cc_minor != 3) {
    delete h;
    return fail(CONVF_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a only", cc_major, cc_minor);
  }

  // BN fold: epilogue scale and bias' = scale*B + shift, in double, stored as float
  const int Kpad = (int)align_up((size_t)s.K, 256);
  std::vector<float> scale(Kpad, 0.f), biasf(Kpad, 0.f);
  for (int k = 0; k < s.K; ++k) {
    const double sc = bn_scale ? (double)bn_scale[k] : 1.0;
    const double sf = bn_shift ? (double)bn_shift[k] : 0.0;
    const double b = (!s8 && !q8 && bias) ? (double)static_cast<const float*>(bias)[k] : 0.0;
    scale[k] = (float)sc;
    biasf[k] = (float)(sc * b + sf);
  }

  // device layout
  size_t off = 0;
  auto carve = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  size_t o_w = 0, o_taps = 0, o_scale = 0, o_bias = 0, o_qb = 0, o_qm = 0, o_qs = 0, o_pad = 0, o_skws = 0,
         o_skflags = 0;
  std::vector<uint16_t> wpack;
  std::vector<float> taps;
  if (variant == CONVF_VARIANT_DEPTHWISE) {
    taps.assign((size_t)s.R * s.S * s.C, 0.f);
    const uint16_t* Wb = static_cast<const uint16_t*>(W);
    for (int c = 0; c < s.C; ++c)
      for (int r = 0; r < s.R; ++r)
        for (int q = 0; q < s.S; ++q)
          taps[(size_t)(r * s.S + q) * s.C + c] =
              (float)((double)scale[c] * (double)bf16_to_f32(Wb[((size_t)c * s.R + r) * s.S + q]));
    o_taps = carve(taps.size() * sizeof(float));
    o_bias = carve((size_t)Kpad * sizeof(float));
  } else if (variant == CONVF_VARIANT_IMPLICIT_GEMM_WINDOW) {
    win_geom(s, &h->wg);
    wpack.resize((size_t)s.R * h->wg.bnp * h->wg.E);
    pack_window(static_cast<const uint16_t*>(W), s, h->wg, wpack.data());
    h->ktot = s.R * h->wg.E;
    o_w = carve(wpack.size() * sizeof(uint16_t));
    o_scale = carve((size_t)Kpad * sizeof(float));
    o_bias = carve((size_t)Kpad * sizeof(float));
    o_pad = carve((size_t)s.N * s.H * h->wg.Wp * h->wg.cpt * sizeof(uint16_t));
  } else if (variant == CONVF_VARIANT_IMPLICIT_GEMM_HALO) {
    halo_geom(s, h->num_sms, desc->tile_n, &h->hg);
    int cpad = 0;
    tc_layout(variant, s, &h->a_mode, &h->cblocks, &h->ktot, &cpad);
    wpack.resize((size_t)s.K * h->ktot);
    pack_bf16(static_cast<const uint16_t*>(W), s, cpad, h->ktot, wpack.data());
    o_w = carve(wpack.size() * sizeof(uint16_t));
    o_scale = carve((size_t)Kpad * sizeof(float));
    o_bias = carve((size_t)Kpad * sizeof(float));
  } else if (variant == CONVF_VARIANT_GROUPED_DIRECT) {
    // [R*S][Cg][K] fp32 with the BN scale folded in (consecutive threads = consecutive k)
    taps.assign((size_t)s.R * s.S * s.Cg * s.K, 0.f);
    const uint16_t* Wb = static_cast<const uint16_t*>(W);
    for (int k = 0; k < s.K; ++k)
      for (int c = 0; c < s.Cg; ++c)
        for (int r = 0; r < s.R; ++r)
          for (int q = 0; q < s.S; ++q)
            taps[((size_t)(r * s.S + q) * s.Cg + c) * s.K + k] =
                (float)((double)scale[k] * (double)bf16_to_f32(Wb[(((size_t)k * s.Cg + c) * s.R + r) * s.S + q]));
    o_taps = carve(taps.size() * sizeof(float));
    o_bias = carve((size_t)Kpad * sizeof(float));
  } else if (variant == CONVF_VARIANT_INT8_TC) {
    // 8-bit operands as exact bf16 integers: w - w_zero_point[k] (|v| <= 255), prepacked like the
    // bf16 implicit GEMM (1x1 matrix rows or per-tap 64-channel runs)
    const bool wsig = q8 ? qp->w_signed != 0 : true;
    h->x_signed = q8 ? qp->x_signed : 1;
    h->x_zp = q8 ? qp->x_zero_point : 0;
    int cpad = 0;
    tc_layout(pure_1x1(s) ? CONVF_VARIANT_GEMM_1X1 : CONVF_VARIANT_IMPLICIT_GEMM, s, &h->a_mode, &h->cblocks,
              &h->ktot, &cpad);
    const size_t wn = (size_t)s.K * s.C * s.R * s.S;
    std::vector<uint16_t> wb(wn);
    const uint8_t* Wq = static_cast<const uint8_t*>(W);
    int maxb = 0;
    for (size_t i = 0; i < wn; ++i) {
      const int k = (int)(i / ((size_t)s.C * s.R * s.S));
      const int w = (wsig ? (int)(int8_t)Wq[i] : (int)Wq[i]) - (q8 ? qp->w_zero_point[k] : 0);
      maxb = std::max(maxb, std::abs(w));
      const float f = (float)w;   // |w| <= 255: exact in bf16, so the top half of the float is it
      uint32_t u;
      std::memcpy(&u, &f, 4);
      wb[i] = (uint16_t)(u >> 16);
    }
    wpack.resize((size_t)s.K * h->ktot);
    pack_bf16(wb.data(), s, cpad, h->ktot, wpack.data());
    // chunk of reduction blocks whose |partial sums| stay <= 2^24 (exact in the fp32 accumulator)
    const int lo = q8_lo(h->x_signed), hi = q8_hi(h->x_signed);
    const long long maxa = std::max(std::abs(lo - h->x_zp), std::abs(hi - h->x_zp));
    const int nkb = h->ktot / 64;
    long long bound = maxb == 0 || maxa == 0 ? nkb : (1LL << 24) / (maxa * maxb * 64);
    bool pair = false, sk = false;
    pick_tile(s.M, s.K, nkb, h->num_sms, 128, 1, 1, false, &h->bn, &pair, &sk);
    if (h->bn < 64) h->bn = 64;
    if (desc->tile_n == 64 || desc->tile_n == 128) h->bn = desc->tile_n;
    else if (desc->tile_n) {
      delete h;
      return fail(CONVF_ERR_UNSUPPORTED, "tile_n=%d: the exact-integer kernel comes 64 or 128 wide", desc->tile_n);
    }
    const int stg = tc_conv_stages(h->bn, false, false);
    if (desc->kblocks_per_step) {
      if (stg % desc->kblocks_per_step || nkb % desc->kblocks_per_step) {
        delete h;
        return fail(CONVF_ERR_UNSUPPORTED,
                    "kblocks_per_step=%d must divide both the %d reduction blocks and the %d pipeline stages of "
                    "%d-wide tiles", desc->kblocks_per_step, nkb, stg, h->bn);
      }
      h->kpb = desc->kblocks_per_step;
    } else {
      h->kpb = auto_kblocks_per_step(stg, nkb);
    }
    if (bound < h->kpb) {
      delete h;
      return fail(CONVF_ERR_UNSUPPORTED, "the exact-integer chunk (%lld blocks) is shorter than a pipeline step", bound);
    }
    h->iq_chunk_kb = (int)std::min<long long>(nkb, bound / h->kpb * h->kpb);
    h->a3d = h->a_mode == kA2D && h->kpb > 1 && s.C % 64 == 0;
    h->iq_mode = q8 ? 1 : 0;
    h->zp = q8 ? qp->y_zero_point : out_zero_point;
    const bool ysig = q8 ? qp->y_signed != 0 : true;
    const bool relu = q8 ? qp->relu != 0 : desc->act == CONVF_ACT_RELU;
    h->q_lo = relu ? std::max(h->zp, q8_lo(ysig)) : q8_lo(ysig);
    h->q_hi = q8_hi(ysig);
    o_w = carve(wpack.size() * sizeof(uint16_t));
    o_qb = carve((size_t)Kpad * 4);
    o_qm = carve((size_t)Kpad * 4);
    o_qs = carve((size_t)Kpad * 4);
    o_pad = carve((size_t)s.N * s.H * s.W * s.C * sizeof(uint16_t));
  } else if (variant == CONVF_VARIANT_INT8) {
    o_w = carve((size_t)s.K * s.R * s.S * s.C);
    o_qb = carve((size_t)s.K * 4);
    o_qm = carve((size_t)s.K * 4);
    o_qs = carve((size_t)s.K * 4);
  } else {
    int cpad = 0;
    GroupTile gt{0, 0};
    if (desc->group > 1) {
      // grouped: the tile width fixes the channel window; block-diagonal weights over it
      grouped_tile(s, desc->group, h->num_sms, desc->tile_n, &gt);
      h->a_mode = variant == CONVF_VARIANT_GEMM_1X1 ? kA2D : kAIm2col;
      h->cblocks = gt.cwpad / 64;
      cpad = gt.cwpad;
      h->ktot = variant == CONVF_VARIANT_GEMM_1X1 ? gt.cwpad : s.R * s.S * gt.cwpad;
      wpack.resize((size_t)s.K * h->ktot);
      pack_bf16_grouped(static_cast<const uint16_t*>(W), s, desc->group, gt.bn, cpad, h->ktot, wpack.data());
    } else {
      tc_layout(variant, s, &h->a_mode, &h->cblocks, &h->ktot, &cpad);
      wpack.resize((size_t)s.K * h->ktot);
      pack_bf16(static_cast<const uint16_t*>(W), s, cpad, h->ktot, wpack.data());
    }
    o_w = carve(wpack.size() * sizeof(uint16_t));
    o_scale = carve((size_t)Kpad * sizeof(float));
    o_bias = carve((size_t)Kpad * sizeof(float));
    const bool gather = variant == CONVF_VARIANT_IMPLICIT_GEMM_GATHER;
    const int max_bn = gather ? 128 : 256;
    if (desc->tile_n > max_bn || (gather && desc->cta_pair == 2)) {
      delete h;
      return fail(CONVF_ERR_UNSUPPORTED, "tile_n=%d / cta_pair=%d not served by the gather variant", desc->tile_n,
                  desc->cta_pair);
    }
    pick_tile(s.M, s.K, h->ktot / 64, h->num_sms, desc->tile_n ? desc->tile_n : max_bn, gather ? 1 : desc->cta_pair,
              desc->stream_k, !gather, &h->bn, &h->pair, &h->sk);
    if (desc->tile_n) h->bn = desc->tile_n;
    if (desc->group > 1) {
      h->bn = gt.bn;
      h->pair = h->sk = false;
    }
    h->kpb = 1;
    h->rsm = !gather && tc_conv_rsm(h->bn, h->pair, h->sk, h->has_res, h->out_bf16, s.K);
    if (!gather) {
      const int st = tc_conv_stages(h->bn, false, h->pair, h->rsm);
      const int nkb = h->ktot / 64;
      if (desc->kblocks_per_step) {
        if (st % desc->kblocks_per_step || nkb % desc->kblocks_per_step) {
          delete h;
          return fail(CONVF_ERR_UNSUPPORTED,
                      "kblocks_per_step=%d must divide both the %d reduction blocks and the %d pipeline stages of "
                      "%d-wide tiles", desc->kblocks_per_step, nkb, st, h->bn);
        }
        h->kpb = desc->kblocks_per_step;
      } else {
        h->kpb = auto_kblocks_per_step(st, nkb);
      }
    }
    h->a3d = h->a_mode == kA2D && !gather && h->kpb > 1 && s.C % 64 == 0 && desc->group == 1;
    if (h->sk) {
      o_skws = carve((size_t)h->num_sms * 128 * h->bn * sizeof(float));
      o_skflags = carve((size_t)h->num_sms * sizeof(int));
    }
    if (variant == CONVF_VARIANT_IMPLICIT_GEMM_GATHER && gather_cpt(s) > 0)
      o_pad = carve((size_t)s.N * s.H * s.W * gather_cpt(s) * sizeof(uint16_t));
  }
  size_t o_xs = 0, o_pre = 0;
  const size_t Cpad = align_up((size_t)s.C, 64);
  if (preact) {
    h->preact = true;
    o_xs = carve((size_t)s.N * s.H * s.W * s.C * sizeof(uint16_t));
    o_pre = carve(2 * Cpad * sizeof(float));
    convf_desc a{};
    a.act = pre_act;
    act_bounds(&a, &h->pre_lo, &h->pre_hi);
  }
  const size_t o_status = carve(sizeof(int));
  h->dev_bytes = off;
  const bool dev_injected = injected_alloc_failure();
  ce = dev_injected ? cudaErrorMemoryAllocation : cudaMalloc(&h->dev, h->dev_bytes);
  if (ce != cudaSuccess) {
    if (!dev_injected) cudaGetLastError();
    delete h;
    return fail(CONVF_ERR_OOM, "cudaMalloc(%zu) failed: %s%s", off, cudaGetErrorString(ce), dev_injected ? " (injected)" : "");
  }
  char* base = static_cast<char*>(h->dev);
  h->status = reinterpret_cast<int*>(base + o_status);
  std::vector<char> staging(h->dev_bytes, 0);
  if (variant == CONVF_VARIANT_DEPTHWISE || variant == CONVF_VARIANT_GROUPED_DIRECT) {
    h->taps = reinterpret_cast<float*>(base + o_taps);
    h->bias = reinterpret_cast<float*>(base + o_bias);
    std::memcpy(staging.data() + o_taps, taps.data(), taps.size() * sizeof(float));
    std::memcpy(staging.data() + o_bias, biasf.data(), (size_t)Kpad * sizeof(float));
  } else if (variant == CONVF_VARIANT_INT8_TC) {
    h->w_bf16 = reinterpret_cast<uint16_t*>(base + o_w);
    h->q_bias = reinterpret_cast<int32_t*>(base + o_qb);
    h->q_mult = reinterpret_cast<int32_t*>(base + o_qm);
    h->q_shift = reinterpret_cast<int32_t*>(base + o_qs);
    h->q_scale = reinterpret_cast<float*>(base + o_qm);   // mode 1 keeps its float multipliers here
    h->xq = reinterpret_cast<uint16_t*>(base + o_pad);
    std::memcpy(staging.data() + o_w, wpack.data(), wpack.size() * sizeof(uint16_t));
    int32_t* qb = reinterpret_cast<int32_t*>(staging.data() + o_qb);
    for (int k = 0; k < s.K; ++k) qb[k] = bias ? static_cast<const int32_t*>(bias)[k] : 0;
    if (q8) {
      // m[k] = float32(x_scale * w_scale[k] / y_scale), the quotient formed in double
      float* qm = reinterpret_cast<float*>(staging.data() + o_qm);
      for (int k = 0; k < s.K; ++k)
        qm[k] = (float)((double)qp->x_scale * (double)qp->w_scale[k] / (double)qp->y_scale);
    } else {
      std::memcpy(staging.data() + o_qm, requant_mult, (size_t)s.K * 4);
      std::memcpy(staging.data() + o_qs, requant_shift, (size_t)s.K * 4);
    }
  } else if (variant == CONVF_VARIANT_INT8) {
    h->w_s8 = reinterpret_cast<int8_t*>(base + o_w);
    h->qbias = reinterpret_cast<int32_t*>(base + o_qb);
    h->qmult = reinterpret_cast<int32_t*>(base + o_qm);
    h->qshift = reinterpret_cast<int32_t*>(base + o_qs);
    // [K][C][R][S] -> [K][R][S][C]
    const int8_t* Wi = static_cast<const int8_t*>(W);
    int8_t* dst = reinterpret_cast<int8_t*>(staging.data() + o_w);
    for (int k = 0; k < s.K; ++k)
      for (int c = 0; c < s.C; ++c)
        for (int r = 0; r < s.R; ++r)
          for (int q = 0; q < s.S; ++q)
            dst[(((size_t)k * s.R + r) * s.S + q) * s.C + c] = Wi[(((size_t)k * s.C + c) * s.R + r) * s.S + q];
    int32_t* qb = reinterpret_cast<int32_t*>(staging.data() + o_qb);
    for (int k = 0; k < s.K; ++k) qb[k] = bias ? static_cast<const int32_t*>(bias)[k] : 0;
    std::memcpy(staging.data() + o_qm, requant_mult, (size_t)s.K * 4);
    std::memcpy(staging.data() + o_qs, requant_shift, (size_t)s.K * 4);
  } else {
    h->w_bf16 = reinterpret_cast<uint16_t*>(base + o_w);
    h->xpad = o_pad ? reinterpret_cast<uint16_t*>(base + o_pad) : nullptr;
    h->sk_ws = o_skws ? reinterpret_cast<float*>(base + o_skws) : nullptr;
    h->sk_flags = o_skflags ? reinterpret_cast<int*>(base + o_skflags) : nullptr;   // zeroed by the upload
    h->scale = reinterpret_cast<float*>(base + o_scale);
    h->bias = reinterpret_cast<float*>(base + o_bias);
    std::memcpy(staging.data() + o_w, wpack.data(), wpack.size() * sizeof(uint16_t));
    std::memcpy(staging.data() + o_scale, scale.data(), (size_t)Kpad * sizeof(float));
    std::memcpy(staging.data() + o_bias, biasf.data(), (size_t)Kpad * sizeof(float));
  }
  if (preact) {
    h->xs = reinterpret_cast<uint16_t*>(base + o_xs);
    h->pre_scale = reinterpret_cast<float*>(base + o_pre);
    h->pre_shift = h->pre_scale + Cpad;
    std::memcpy(staging.data() + o_pre, pre_scale, (size_t)s.C * sizeof(float));
    std::memcpy(staging.data() + o_pre + Cpad * sizeof(float), pre_shift, (size_t)s.C * sizeof(float));
  }
  ce = cudaMemcpy(h->dev, staging.data(), h->dev_bytes, cudaMemcpyHostToDevice);
  if (ce != cudaSuccess) {
    cudaFree(h->dev);
    delete h;
    return fail(CONVF_ERR_CUDA, "weight upload failed: %s", cudaGetErrorString(ce));
  }

  if (variant == CONVF_VARIANT_IMPLICIT_GEMM_HALO) {
    const HaloGeom& g = h->hg;
    h->bn = g.bn;
    h->num_kb = h->ktot / 64;
    h->n_blocks = (s.K + g.bn - 1) / g.bn;
    h->num_tiles = (int)((long long)s.N * g.tiles_per_img * h->n_blocks);
    h->grid = (int)std::min<long long>(h->num_tiles, h->num_sms);
    CUresult r = load_encoders() ? CUDA_SUCCESS : CUDA_ERROR_NOT_SUPPORTED;
    if (r == CUDA_SUCCESS) {
      // {channels of one tap, output channel, tap}: a box brings tpo consecutive taps, each a
      // BN x 64 K-major tile
      const int cpad = g.cblocks * 64;
      const cuuint64_t dims[3] = {(cuuint64_t)cpad, (cuuint64_t)s.K, (cuuint64_t)(s.R * s.S)};
      const cuuint64_t strides[2] = {(cuuint64_t)h->ktot * 2, (cuuint64_t)cpad * 2};
      const cuuint32_t box[3] = {64, (cuuint32_t)g.bn, (cuuint32_t)g.tpo};
      const cuuint32_t es[3] = {1, 1, 1};
      r = g_encode_tiled(&h->tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, h->w_bf16, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) {
      cudaFree(h->dev);
      delete h;
      return fail(CONVF_ERR_CUDA, "halo weight tensor map encoding failed (CUresult %d)", (int)r);
    }
  }
  if (variant == CONVF_VARIANT_IMPLICIT_GEMM_WINDOW) {
    const WinGeom& g = h->wg;
    h->bn = g.bnp;
    h->num_tiles = (int)g.tiles;
    h->grid = (int)std::min<long long>(g.tiles, h->num_sms);
    h->cpt = g.cpt;
    CUresult r = CUDA_SUCCESS;
    if (!load_encoders()) r = CUDA_ERROR_NOT_SUPPORTED;
    const CUtensorMapSwizzle sw = g.E == 16 ? CU_TENSOR_MAP_SWIZZLE_32B
                                            : (g.E == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
    if (r == CUDA_SUCCESS && h->xpad && g.rows) {
      // row mode: {64-element chunks, chunks per row, rows, images}, box = nchunk chunks x R rows
      const size_t rowb = (size_t)g.Wp * g.cpt * 2;
      const cuuint64_t dims[4] = {64, (cuuint64_t)(rowb / 128), (cuuint64_t)s.H, (cuuint64_t)s.N};
      const cuuint64_t strides[3] = {128, (cuuint64_t)rowb, (cuuint64_t)s.H * rowb};
      const cuuint32_t box[4] = {64, (cuuint32_t)g.nchunk, (cuuint32_t)s.R, 1};
      const cuuint32_t es[4] = {1, 1, 1, 1};
      r = g_encode_tiled(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, h->xpad, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (r == CUDA_SUCCESS && h->xpad) {
      // overlapping windows: consecutive windows start sw*cpt elements apart, each E long
      const size_t px = (size_t)g.cpt * 2;
      const cuuint64_t dims[4] = {(cuuint64_t)g.E, (cuuint64_t)s.Wo, (cuuint64_t)s.H, (cuuint64_t)s.N};
      const cuuint64_t strides[3] = {(cuuint64_t)(s.sw * px), (cuuint64_t)(g.Wp * px), (cuuint64_t)s.H * g.Wp * px};
      const cuuint32_t box[4] = {(cuuint32_t)g.E, 128, (cuuint32_t)s.R, 1};
      const cuuint32_t es[4] = {1, 1, 1, 1};
      r = g_encode_tiled(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, h->xpad, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r == CUDA_SUCCESS && !g.rows) {
      const cuuint64_t dims[3] = {(cuuint64_t)g.E, (cuuint64_t)g.bnp, (cuuint64_t)s.R};
      const cuuint64_t strides[2] = {(cuuint64_t)g.E * 2, (cuuint64_t)g.bnp * g.E * 2};
      const cuuint32_t box[3] = {(cuuint32_t)g.E, (cuuint32_t)g.bnp, (cuuint32_t)s.R};
      const cuuint32_t es[3] = {1, 1, 1};
      r = g_encode_tiled(&h->tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, h->w_bf16, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) {
      cudaFree(h->dev);
      delete h;
      return fail(CONVF_ERR_CUDA, "window-mode tensor map encoding failed (CUresult %d)", (int)r);
    }
  }
  if (variant == CONVF_VARIANT_GEMM_1X1 || variant == CONVF_VARIANT_IMPLICIT_GEMM ||
      variant == CONVF_VARIANT_IMPLICIT_GEMM_GATHER || variant == CONVF_VARIANT_INT8_TC) {
    if (!load_encoders()) {
      cudaFree(h->dev);
      delete h;
      return fail(CONVF_ERR_CUDA, "cuTensorMapEncodeTiled/Im2col are unavailable from the driver");
    }
    h->cpt = variant == CONVF_VARIANT_IMPLICIT_GEMM_GATHER ? gather_cpt(s) : 0;
    h->patch_rows = variant == CONVF_VARIANT_IMPLICIT_GEMM_GATHER ? patch_rows_for(s, h->cpt ? h->cpt : s.C) : 0;
    h->row_bytes = s.W * (h->cpt ? h->cpt : s.C) * 2;
    h->num_kb = h->ktot / 64;
    h->n_blocks = (s.K + h->bn - 1) / h->bn;
    const long long tile_m = h->pair ? 256 : 128;
    const long long tiles = (s.M + tile_m - 1) / tile_m * h->n_blocks;
    h->num_tiles = (int)tiles;
    h->grid = h->pair ? 2 * (int)std::min<long long>(tiles, h->num_sms / 2)
                      // stream-K: every CTA needs at least one pipeline step of its own (a CTA
                      // with an empty share would be waited for as a contributor)
                      : (int)std::min<long long>(h->sk ? tiles * (h->num_kb / h->kpb) : tiles, h->num_sms);
    CUresult r;
    if (variant == CONVF_VARIANT_IMPLICIT_GEMM_GATHER || h->kpb == 1) {
      const cuuint64_t dims[2] = {(cuuint64_t)h->ktot, (cuuint64_t)s.K};
      const cuuint64_t strides[1] = {(cuuint64_t)h->ktot * 2};
      const cuuint32_t box[2] = {64, (cuuint32_t)(h->pair ? h->bn / 2 : h->bn)};
      const cuuint32_t es[2] = {1, 1};
      r = g_encode_tiled(&h->tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h->w_bf16, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      // {64 elements of a k-block, output channel, k-block}: one box = kpb consecutive bn x 64
      // K-major tiles
      const cuuint64_t dims[3] = {64, (cuuint64_t)s.K, (cuuint64_t)(h->ktot / 64)};
      const cuuint64_t strides[2] = {(cuuint64_t)h->ktot * 2, 128};
      const cuuint32_t box[3] = {64, (cuuint32_t)(h->pair ? h->bn / 2 : h->bn), (cuuint32_t)h->kpb};
      const cuuint32_t es[3] = {1, 1, 1};
      r = g_encode_tiled(&h->tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, h->w_bf16, dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) {
      cudaFree(h->dev);
      delete h;
      return fail(CONVF_ERR_CUDA, "weight tensor map encoding failed (CUresult %d)", (int)r);
    }
    if (variant == CONVF_VARIANT_INT8_TC) {
      // the activation operand is the handle's bf16 staging copy: its map is encoded once
      convf_status ms = encode_a_map(h, h->xq);
      if (ms != CONVF_OK) {
        cudaFree(h->dev);
        delete h;
        return ms;
      }
    }
  }
  h->magic = kMagic;
  *out = h;
  return ok();
}
}  // namespace

namespace {
// Tile geometry of the fused MobileNetV2 block: TW = min(Wo, 16 for stride 1, 8 for stride 2)
// output columns; among the row counts TH <= 8 whose input halo fits two 128-row MMA blocks
// (IH*IW <= 256), whose expand/project accumulators fit TMEM and whose buffers fit shared
// memory, the tallest that still gives every SM a tile, else the one with the most tiles.
std::string mb_geom(const convf_block_desc* d, int num_sms, MbParams* g) {
  std::memset(g, 0, sizeof *g);
  g->N = d->N; g->H = d->H; g->W = d->W; g->Cin = d->Cin; g->Ch = d->Ch; g->Cout = d->Cout; g->st = d->stride;
  g->Ho = (d->H + 2 - 3) / d->stride + 1;
  g->Wo = (d->W + 2 - 3) / d->stride + 1;
  g->Ch_pad = (int)align_up((size_t)d->Ch, 64);
  g->cin_kb = (d->Cin + 63) / 64;
  g->nch = g->Ch_pad / 64;
  g->Np = (int)align_up((size_t)d->Cout, 16);
  g->nsplit = 1;
  if (g->Np > 256) {
    g->Np = (int)align_up((size_t)d->Cout, 32);
    g->nsplit = 2;
  }
  if (g->Np > 512) return "fused block: Cout exceeds the project accumulator";
  g->expand = d->expand;
  g->residual = d->residual;
  g->h1_stride = 68;
  g->TW = std::min(g->Wo, d->stride == 1 ? 16 : 8);
  int best = -1;
  long long best_tiles = -1;
  for (int th = std::min(g->Ho, 8); th >= 1; --th) {
    const int IH = (th - 1) * d->stride + 3, IW = (g->TW - 1) * d->stride + 3;
    const int P = IH * IW;
    if (P > 256 || th * g->TW > 128) continue;
    const int rb = P > 128 ? 2 : 1;
    if (2 * rb * 64 + g->Np > 512) continue;
    const uint32_t xkb = rb * 16384u;
    const uint32_t sx = g->cin_kb * xkb;
    const uint32_t we = g->expand ? g->cin_kb * 8192u : 0u;
    const uint32_t wp = (uint32_t)align_up((size_t)g->Np * 128, 1024);
    const uint32_t h1 = (uint32_t)align_up((size_t)P * 68 * 4, 1024);
    const size_t total = 1024 + sx + 2 * we + 2 * wp + h1 + 32768 + 2 * 3072 + 256;   // one halo buffer
    if (total > 232448) continue;
    const long long tiles = (long long)d->N * ((g->Ho + th - 1) / th) * ((g->Wo + g->TW - 1) / g->TW);
    // rows go down from the tallest: stop at the first that gives every SM a tile, else keep
    // the one with the most tiles
    if (best < 0 || tiles > best_tiles) {
      best = th;
      best_tiles = tiles;
    }
    if (tiles >= num_sms) break;
  }
  if (best < 0) return "fused block: no tile of its output fits the shared memory and TMEM budgets";
  g->TH = best;
  g->IH = (best - 1) * d->stride + 3;
  g->IW = (g->TW - 1) * d->stride + 3;
  g->P = g->IH * g->IW;
  g->rb = g->P > 128 ? 2 : 1;
  g->tiles_h = (g->Ho + best - 1) / best;
  g->tiles_w = (g->Wo + g->TW - 1) / g->TW;
  g->num_tiles = (int)best_tiles;
  g->x_kb_bytes = g->rb * 16384u;
  g->x_buf_bytes = g->cin_kb * g->x_kb_bytes;
  g->we_buf = g->expand ? g->cin_kb * 8192u : 0u;
  g->wp_buf = (uint32_t)align_up((size_t)g->Np * 128, 1024);
  g->x_bytes = g->cin_kb * (uint32_t)g->P * 128u;
  g->we_bytes = g->cin_kb * 8192u;
  g->wp_bytes = (uint32_t)g->Np * 128u;
  // a second halo buffer when it fits: the next tile's halo then loads behind this tile's chunks
  {
    const size_t one = 1024 + (size_t)g->x_buf_bytes + 2 * (size_t)g->we_buf + 2 * (size_t)g->wp_buf +
                       align_up((size_t)g->P * 68 * 4, 1024) + 32768 + 2 * 3072 + 256;
    g->nxb = one + g->x_buf_bytes <= 232448 ? 2 : 1;
  }
  g->off_x = 0;
  g->off_we = g->nxb * g->x_buf_bytes;
  g->off_wp = g->off_we + 2 * g->we_buf;
  g->off_h1 = g->off_wp + 2 * g->wp_buf;
  g->off_a = g->off_h1 + (uint32_t)align_up((size_t)g->P * 68 * 4, 1024);
  g->off_vec = g->off_a + 32768;
  g->off_bar = g->off_vec + 2 * 3072;
  return "";
}

uint16_t f32_to_bf16_bits(float f) {   // round to nearest even (finite values)
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}
}  // namespace

convf_status conv_fused_create_mbv2_block(const convf_block_desc* d, const uint16_t* w_expand, const float* e_scale,
                                          const float* e_shift, const uint16_t* w_dw, const float* d_scale,
                                          const float* d_shift, const uint16_t* w_project, const float* p_scale,
                                          const float* p_shift, convf_handle** out) {
  if (!out) return fail(CONVF_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!d) return fail(CONVF_ERR_INVALID_ARG, "d is NULL");
  if (d->N < 0 || d->H < 1 || d->W < 1 || d->Cin < 1 || d->Ch < 1 || d->Cout < 1)
    return fail(CONVF_ERR_INVALID_ARG, "block extents (N=%d H=%d W=%d Cin=%d Ch=%d Cout=%d) must be positive", d->N,
                d->H, d->W, d->Cin, d->Ch, d->Cout);
  if (d->stride != 1 && d->stride != 2) return fail(CONVF_ERR_INVALID_ARG, "stride=%d is not 1 or 2", d->stride);
  if (d->expand != 0 && d->expand != 1) return fail(CONVF_ERR_INVALID_ARG, "expand=%d is not 0 or 1", d->expand);
  if (d->residual != 0 && d->residual != 1) return fail(CONVF_ERR_INVALID_ARG, "residual=%d is not 0 or 1", d->residual);
  if (!d->expand && d->Ch != d->Cin) return fail(CONVF_ERR_INVALID_ARG, "without an expand conv Ch (%d) must equal Cin (%d)",
                                                 d->Ch, d->Cin);
  if (d->residual && (d->stride != 1 || d->Cin != d->Cout))
    return fail(CONVF_ERR_INVALID_ARG, "the skip connection needs stride 1 and Cin == Cout");
  if (!w_dw || !d_scale || !d_shift || !w_project || !p_scale || !p_shift ||
      (d->expand && (!w_expand || !e_scale || !e_shift)))
    return fail(CONVF_ERR_INVALID_ARG, "a weight or affine array is NULL");
  if (d->Cin % 8) return fail(CONVF_ERR_UNSUPPORTED, "fused block: Cin %% 8 == 0 (16-byte TMA rows)");
  if (d->Cin > 192) return fail(CONVF_ERR_UNSUPPORTED, "fused block: Cin <= 192 (three 64-channel blocks of halo)");
  if (d->Cout % 4) return fail(CONVF_ERR_UNSUPPORTED, "fused block: Cout %% 4 == 0 (16-byte output stores)");
  if ((long long)d->N * d->H * d->W * d->Cin > 0x7FFFFFFFLL || (long long)d->N * d->H * d->W * d->Cout > 0x7FFFFFFFLL)
    return fail(CONVF_ERR_UNSUPPORTED, "tensor sizes exceed the 2^31-element indexing limit");
  const bool host_injected = injected_alloc_failure();
  convf_handle* h = host_injected ? nullptr : new (std::nothrow) convf_handle();
  if (!h) return fail(CONVF_ERR_OOM, "host allocation failed%s", host_injected ? " (injected)" : "");
  cudaError_t ce = cudaGetDevice(&h->device);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (ce != cudaSuccess) {
    delete h;
    return fail(CONVF_ERR_CUDA, "no usable CUDA device: %s", cudaGetErrorString(ce));
  }
  MbParams& g = h->mb;
  std::string why = mb_geom(d, h->num_sms, &g);
  if (!why.empty()) {
    delete h;
    return fail(CONVF_ERR_UNSUPPORTED, "%s", why.c_str());
  }
  h->variant = CONVF_VARIANT_MBV2_BLOCK;
  Shape& s = h->s;
  s.N = d->N; s.C = d->Cin; s.H = d->H; s.W = d->W; s.K = d->Cout; s.R = s.S = 3; s.Cg = 1;
  s.sh = s.sw = d->stride; s.dh = s.dw = 1; s.pt = s.pl = s.pb = s.pr = 1;
  s.Ho = g.Ho; s.Wo = g.Wo; s.M = (long long)d->N * g.Ho * g.Wo;
  std::memset(&h->desc, 0, sizeof h->desc);
  h->desc.group = 1;
  // device arrays: We [Ch_pad][Cin_pad] bf16, Wp [Np][Ch_pad] bf16, se/be/bd [Ch_pad], wd [9][Ch_pad],
  // sp/bp [Np] (zero padding everywhere)
  const int cin_pad = g.cin_kb * 64;
  size_t off = 0;
  auto carve = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  const size_t o_we = carve((size_t)g.Ch_pad * cin_pad * 2), o_wp = carve((size_t)g.Np * g.Ch_pad * 2);
  const size_t o_se = carve((size_t)g.Ch_pad * 4), o_be = carve((size_t)g.Ch_pad * 4);
  const size_t o_wd = carve((size_t)9 * g.Ch_pad * 4), o_bd = carve((size_t)g.Ch_pad * 4);
  const size_t o_sp = carve((size_t)g.Np * 4), o_bp = carve((size_t)g.Np * 4);
  const size_t o_vec = carve((size_t)g.nch * 12 * 64 * 4);
  const size_t o_status = carve(sizeof(int));
  h->dev_bytes = off;
  std::vector<char> st(off, 0);
  uint16_t* we = reinterpret_cast<uint16_t*>(st.data() + o_we);
  uint16_t* wp = reinterpret_cast<uint16_t*>(st.data() + o_wp);
  float* se = reinterpret_cast<float*>(st.data() + o_se);
  float* be = reinterpret_cast<float*>(st.data() + o_be);
  float* wd = reinterpret_cast<float*>(st.data() + o_wd);
  float* bd = reinterpret_cast<float*>(st.data() + o_bd);
  float* sp = reinterpret_cast<float*>(st.data() + o_sp);
  float* bp = reinterpret_cast<float*>(st.data() + o_bp);
  for (int c = 0; c < d->Ch; ++c) {
    if (d->expand) {
      for (int i = 0; i < d->Cin; ++i) we[(size_t)c * cin_pad + i] = w_expand[(size_t)c * d->Cin + i];
      se[c] = e_scale[c];
      be[c] = e_shift[c];
    }
    for (int t = 0; t < 9; ++t)
      wd[(size_t)t * g.Ch_pad + c] = (float)((double)d_scale[c] * (double)bf16_to_f32(w_dw[(size_t)c * 9 + t]));
    bd[c] = d_shift[c];
  }
  for (int k = 0; k < d->Cout; ++k) {
    for (int c = 0; c < d->Ch; ++c) wp[(size_t)k * g.Ch_pad + c] = w_project[(size_t)k * d->Ch + c];
    sp[k] = p_scale[k];
    bp[k] = p_shift[k];
  }
  // per chunk j: [12][64] = expand scale, expand shift, the nine depthwise taps, depthwise shift
  float* vec = reinterpret_cast<float*>(st.data() + o_vec);
  for (int j = 0; j < g.nch; ++j)
    for (int c = 0; c < 64; ++c) {
      const int ch = j * 64 + c;
      float* v = vec + (size_t)j * 12 * 64 + c;
      v[0] = se[ch];
      v[64] = be[ch];
      for (int t = 0; t < 9; ++t) v[(2 + t) * 64] = wd[(size_t)t * g.Ch_pad + ch];
      v[11 * 64] = bd[ch];
    }
  for (size_t i = 0; i < (size_t)g.Ch_pad; ++i)
    if (!std::isfinite(se[i]) || !std::isfinite(be[i]) || !std::isfinite(bd[i])) {
      delete h;
      return fail(CONVF_ERR_INVALID_ARG, "an expand or depthwise affine value is not finite");
    }
  const bool dev_injected = injected_alloc_failure();
  ce = dev_injected ? cudaErrorMemoryAllocation : cudaMalloc(&h->dev, h->dev_bytes);
  if (ce != cudaSuccess) {
    if (!dev_injected) cudaGetLastError();
    delete h;
    return fail(CONVF_ERR_OOM, "cudaMalloc(%zu) failed: %s%s", h->dev_bytes, cudaGetErrorString(ce), dev_injected ? " (injected)" : "");
  }
  ce = cudaMemcpy(h->dev, st.data(), h->dev_bytes, cudaMemcpyHostToDevice);
  char* base = static_cast<char*>(h->dev);
  g.se = reinterpret_cast<float*>(base + o_se); g.be = reinterpret_cast<float*>(base + o_be);
  g.wd = reinterpret_cast<float*>(base + o_wd); g.bd = reinterpret_cast<float*>(base + o_bd);
  g.sp = reinterpret_cast<float*>(base + o_sp); g.bp = reinterpret_cast<float*>(base + o_bp);
  g.vec = reinterpret_cast<float*>(base + o_vec);
  h->status = reinterpret_cast<int*>(base + o_status);
  g.status = h->status;
  CUresult r = ce == cudaSuccess && load_encoders() ? CUDA_SUCCESS : CUDA_ERROR_NOT_SUPPORTED;
  if (r == CUDA_SUCCESS) {
    const cuuint64_t dims[2] = {(cuuint64_t)cin_pad, (cuuint64_t)g.Ch_pad};
    const cuuint64_t strides[1] = {(cuuint64_t)cin_pad * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t es[2] = {1, 1};
    r = g_encode_tiled(&h->tmWe, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base + o_we, dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r == CUDA_SUCCESS) {
    const cuuint64_t dims[2] = {(cuuint64_t)g.Ch_pad, (cuuint64_t)g.Np};
    const cuuint64_t strides[1] = {(cuuint64_t)g.Ch_pad * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(g.Np / g.nsplit)};
    const cuuint32_t es[2] = {1, 1};
    r = g_encode_tiled(&h->tmWp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base + o_wp, dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    cudaFree(h->dev);
    delete h;
    return fail(ce != cudaSuccess ? CONVF_ERR_CUDA : CONVF_ERR_CUDA, "fused block set-up failed (%s, CUresult %d)",
                cudaGetErrorString(ce), (int)r);
  }
  h->grid = (int)std::min<long long>(g.num_tiles, h->num_sms);
  h->num_tiles = g.num_tiles;
  h->magic = kMagic;
  *out = h;
  return ok();
}

convf_status conv_fused_create(const convf_desc* desc, const void* W, const void* bias,
                               const float* bn_scale, const float* bn_shift,
                               const int32_t* requant_mult, const int32_t* requant_shift,
                               int32_t out_zero_point, convf_handle** out) {
  return create_impl(desc, W, bias, bn_scale, bn_shift, requant_mult, requant_shift, out_zero_point, nullptr, out);
}

convf_status conv_fused_create_preact(const convf_desc* desc, const void* W, const void* bias,
                                      const float* bn_scale, const float* bn_shift, const float* pre_scale,
                                      const float* pre_shift, int pre_act, convf_handle** out) {
  if (pre_act < 0) {
    if (out) *out = nullptr;
    return fail(CONVF_ERR_INVALID_ARG, "pre_act=%d is not CONVF_ACT_NONE, _RELU or _RELU6", pre_act);
  }
  return create_impl(desc, W, bias, bn_scale, bn_shift, nullptr, nullptr, 0, nullptr, out, pre_scale, pre_shift,
                     pre_act);
}

convf_status conv_fused_create_qlinear(const convf_desc* desc, const void* W, const int32_t* bias,
                                       const convf_qparams* q, convf_handle** out) {
  if (!q) {
    if (out) *out = nullptr;
    return fail(CONVF_ERR_INVALID_ARG, "q is NULL");
  }
  return create_impl(desc, W, bias, nullptr, nullptr, nullptr, nullptr, 0, q, out);
}

namespace {
convf_status encode_a_map(convf_handle* h, const void* x) {
  const Shape& s = h->s;
  CUresult r;
  if (h->a_mode == kA2D && h->a3d) {
    // {64 channels of a k-block, output row, k-block}: one box = kpb consecutive 128 x 64 tiles
    const cuuint64_t dims[3] = {64, (cuuint64_t)s.M, (cuuint64_t)(s.C / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)s.C * 2, 128};
    const cuuint32_t box[3] = {64, 128, (cuuint32_t)h->kpb};
    const cuuint32_t es[3] = {1, 1, 1};
    r = g_encode_tiled(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CONVF_ERR_CUDA, "activation tensor map encoding failed (CUresult %d)", (int)r);
  } else if (h->a_mode == kA2D) {
    const cuuint64_t dims[2] = {(cuuint64_t)s.C, (cuuint64_t)s.M};
    const cuuint64_t strides[1] = {(cuuint64_t)s.C * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t es[2] = {1, 1};
    r = g_encode_tiled(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CONVF_ERR_CUDA, "activation tensor map encoding failed (CUresult %d)", (int)r);
  } else if (h->a_mode == kAIm2col) {
    const cuuint64_t dims[4] = {(cuuint64_t)s.C, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)s.N};
    const cuuint64_t strides[3] = {(cuuint64_t)s.C * 2, (cuuint64_t)s.W * s.C * 2, (cuuint64_t)s.H * s.W * s.C * 2};
    const int lower[2] = {-s.pl, -s.pt};
    const int upper[2] = {s.pr - (s.S - 1) * s.dw, s.pb - (s.R - 1) * s.dh};
    const cuuint32_t es[4] = {1, (cuuint32_t)s.sw, (cuuint32_t)s.sh, 1};
    r = g_encode_im2col(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides, lower,
                        upper, 64, 128, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CONVF_ERR_CUDA, "im2col tensor map encoding failed (CUresult %d)", (int)r);
  } else {
    std::memset(&h->tmA, 0, sizeof h->tmA);
  }
  h->map_x = x;
  return CONVF_OK;
}
}  // namespace

namespace {
// staged residual (bf16 [M][K], K % 8 == 0): 2-D map {K, M}, 64 x 128 boxes of 128-byte rows in
// the 128-byte swizzle; out-of-range rows and channels read as zero
convf_status encode_r_map(convf_handle* h, const void* r) {
  const Shape& s = h->s;
  if (!load_encoders()) return fail(CONVF_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  const cuuint64_t dims[2] = {(cuuint64_t)s.K, (cuuint64_t)s.M};
  const cuuint64_t strides[1] = {(cuuint64_t)s.K * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  CUresult rc = g_encode_tiled(&h->tmR, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(r), dims, strides, box,
                               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (rc != CUDA_SUCCESS) return fail(CONVF_ERR_CUDA, "residual tensor map encoding failed (CUresult %d)", (int)rc);
  h->map_r = r;
  return CONVF_OK;
}

// depthwise 3x3: 4-D tiled map over x {C, W, H, N}, box = one tile's input window x 32 channels
convf_status encode_dw_map(convf_handle* h, const void* x) {
  const Shape& s = h->s;
  if (!load_encoders()) return fail(CONVF_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  int bw = 0, bh = 0, bn = 0;
  dw_tile_box(s.sh, s.Wo, &bw, &bh, &bn);
  const cuuint64_t dims[4] = {(cuuint64_t)s.C, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)s.N};
  const cuuint64_t strides[3] = {(cuuint64_t)s.C * 2, (cuuint64_t)s.W * s.C * 2, (cuuint64_t)s.H * s.W * s.C * 2};
  const cuuint32_t box[4] = {32, (cuuint32_t)bw, (cuuint32_t)bh, (cuuint32_t)bn};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode_tiled(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides, box,
                              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(CONVF_ERR_CUDA, "depthwise tensor map encoding failed (CUresult %d)", (int)r);
  h->map_x = x;
  return CONVF_OK;
}
}  // namespace

namespace {
convf_status run_impl(convf_handle* h, const void* x, const void* res, void* y, void* stream) {
  const Shape& s = h->s;
  convf_status st = CONVF_OK;
  if (s.M == 0) return ok();   // empty batch: nothing to compute
  if (!x || !y) return fail(CONVF_ERR_INVALID_ARG, "x/y is NULL");
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 15))
    return fail(CONVF_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  const bool q8bit = h->variant == CONVF_VARIANT_INT8 || h->variant == CONVF_VARIANT_INT8_TC;
  const size_t esz = q8bit ? 1 : 2;
  const size_t xb = (size_t)s.N * s.H * s.W * s.C * esz;
  const size_t yb = (size_t)s.M * s.K * (q8bit ? 1 : (h->out_bf16 ? 2 : 4));
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), y0 = reinterpret_cast<uintptr_t>(y);
  if (x0 < y0 + yb && y0 < x0 + xb) return fail(CONVF_ERR_INVALID_ARG, "x and y overlap");
  if (h->has_res) {
    if (!res) return fail(CONVF_ERR_INVALID_ARG, "the residual r is NULL");
    const uintptr_t r0 = reinterpret_cast<uintptr_t>(res);
    if (r0 & 15) return fail(CONVF_ERR_INVALID_ARG, "the residual r must be 16-byte aligned");
    if (r0 != y0 && r0 < y0 + yb && y0 < r0 + yb)
      return fail(CONVF_ERR_INVALID_ARG, "the residual r overlaps y without being y");
    if (r0 < x0 + xb && x0 < r0 + yb) return fail(CONVF_ERR_INVALID_ARG, "the residual r overlaps x");
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != h->device)
    return fail(CONVF_ERR_INVALID_ARG, "the current device (%d) is not the handle's device (%d)", dev, h->device);
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  cudaError_t ce = cudaSuccess;
  if (h->preact) {
    // the prologue's bf16 copy is what every variant reads (its tensor maps cache that pointer)
    ce = launch_preact_bf16(static_cast<const uint16_t*>(x), h->xs, (long long)s.N * s.H * s.W * s.C, s.C,
                            h->pre_scale, h->pre_shift, h->pre_lo, h->pre_hi, h->num_sms, strm);
    if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "pre-activation launch failed: %s", cudaGetErrorString(ce));
    x = h->xs;
  }
  switch (h->variant) {
    case CONVF_VARIANT_DEPTHWISE: {
      DwParams p{};
      p.N = s.N; p.C = s.C; p.H = s.H; p.W = s.W; p.Ho = s.Ho; p.Wo = s.Wo; p.R = s.R; p.S = s.S;
      p.sh = s.sh; p.sw = s.sw; p.pt = s.pt; p.pl = s.pl; p.dh = s.dh; p.dw = s.dw;
      p.x = static_cast<const uint16_t*>(x); p.taps = h->taps; p.bias = h->bias; p.y = static_cast<float*>(y);
      p.lo = h->lo; p.hi = h->hi; p.status = h->status;
      p.out_bf16 = h->out_bf16 ? 1 : 0; p.res = h->has_res ? res : nullptr;
      if (dw_uses_tma(p) && x != h->map_x) {
        if ((st = encode_dw_map(h, x)) != CONVF_OK) return st;
      }
      ce = launch_depthwise(p, &h->tmA, h->num_sms, strm);
      break;
    }
    case CONVF_VARIANT_IMPLICIT_GEMM_HALO: {
      const HaloGeom& g = h->hg;
      if (x != h->map_x) {
        // {C, W, H, N}, box = 64 channels x the padded row width x (TR + R - 1) rows of one image
        const cuuint64_t dims[4] = {(cuuint64_t)s.C, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)s.N};
        const cuuint64_t strides[3] = {(cuuint64_t)s.C * 2, (cuuint64_t)s.W * s.C * 2,
                                       (cuuint64_t)s.H * s.W * s.C * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)g.Wp, (cuuint32_t)(g.TR + s.R - 1), 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        CUresult r = g_encode_tiled(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(CONVF_ERR_CUDA, "halo activation tensor map encoding failed (CUresult %d)", (int)r);
        h->map_x = x;
      }
      HaloParams p{};
      p.Ho = s.Ho; p.Wo = s.Wo; p.Wp = g.Wp; p.TR = g.TR; p.R = s.R; p.S = s.S; p.pt = s.pt; p.pl = s.pl;
      p.cblocks = g.cblocks; p.cpad = g.cblocks * 64; p.Kout = s.K; p.n_blocks = h->n_blocks;
      p.tiles_per_img = g.tiles_per_img; p.num_tiles = h->num_tiles; p.patch_bytes = g.patch_bytes;
      p.tpo = g.tpo; p.b_stages = g.b_stages; p.resident = g.resident ? 1 : 0;
      p.scale = h->scale; p.bias = h->bias; p.y = static_cast<float*>(y); p.lo = h->lo; p.hi = h->hi;
      p.status = h->status;
      p.out_bf16 = h->out_bf16 ? 1 : 0; p.res = h->has_res ? res : nullptr;
      ce = launch_tc_halo(p, h->tmA, h->tmB, g.bn, h->grid, strm);
      break;
    }
    case CONVF_VARIANT_IMPLICIT_GEMM_WINDOW: {
      const WinGeom& g = h->wg;
      ce = launch_window_pad(static_cast<const uint16_t*>(x), h->xpad, s.N, s.H, s.W, s.C, g.cpt, g.Wp, s.pl,
                             h->num_sms, strm);
      if (ce != cudaSuccess) break;
      WinParams p{};
      p.N = s.N; p.H = s.H; p.Ho = s.Ho; p.Wo = s.Wo; p.Kout = s.K; p.sh = s.sh; p.pt = s.pt; p.R = s.R;
      p.bnp = g.bnp; p.ow_blocks = g.ow_blocks; p.num_tiles = h->num_tiles; p.stages = g.stages;
      p.a_stage_bytes = g.a_stage; p.b_bytes = g.b_bytes; p.b_region = g.b_region; p.tmem_cols = g.tmem_cols;
      p.chunk0_per_block = 128 * s.sw * g.cpt / 64; p.nchunk = g.nchunk; p.w = h->w_bf16;
      p.scale = h->scale; p.bias = h->bias; p.y = static_cast<float*>(y);
      p.lo = h->lo; p.hi = h->hi; p.status = h->status;
      ce = launch_tc_window(p, h->tmA, h->tmB, g.E, g.rows, h->grid, g.smem, strm);
      break;
    }
    case CONVF_VARIANT_MBV2_BLOCK: {
      MbParams p = h->mb;
      if (x != h->map_x) {
        // {C, W, H, N}, box = 64 channels x the tile's input halo (IW x IH pixels) of one image
        const cuuint64_t dims[4] = {(cuuint64_t)s.C, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)s.N};
        const cuuint64_t strides[3] = {(cuuint64_t)s.C * 2, (cuuint64_t)s.W * s.C * 2,
                                       (cuuint64_t)s.H * s.W * s.C * 2};
        const cuuint32_t box[4] = {64, (cuuint32_t)p.IW, (cuuint32_t)p.IH, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        CUresult r = g_encode_tiled(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(CONVF_ERR_CUDA, "fused block input tensor map failed (CUresult %d)", (int)r);
        h->map_x = x;
      }
      p.y = static_cast<float*>(y);
      ce = launch_mbv2_block(p, h->tmA, h->tmWe, h->tmWp, h->grid, strm);
      break;
    }
    case CONVF_VARIANT_GROUPED_DIRECT: {
      GdParams p{};
      p.N = s.N; p.C = s.C; p.H = s.H; p.W = s.W; p.K = s.K; p.R = s.R; p.S = s.S; p.Ho = s.Ho; p.Wo = s.Wo;
      p.sh = s.sh; p.sw = s.sw; p.pt = s.pt; p.pl = s.pl; p.dh = s.dh; p.dw = s.dw;
      p.Cg = s.Cg; p.Kg = s.K / h->desc.group;
      p.x = static_cast<const uint16_t*>(x); p.w = h->taps; p.bias = h->bias; p.y = y;
      p.res = h->has_res ? res : nullptr; p.out_bf16 = h->out_bf16 ? 1 : 0; p.lo = h->lo; p.hi = h->hi;
      ce = launch_grouped_direct(p, h->num_sms, strm);
      break;
    }
    case CONVF_VARIANT_INT8_TC: {
      // x - x_zero_point as exact bf16 into the handle's staging copy, then the tcgen05 GEMM in
      // its integer-exact mode (the staging copy's tensor map was encoded at create)
      ce = launch_q8_to_bf16(static_cast<const uint8_t*>(x), h->xq, (long long)s.N * s.H * s.W * s.C, h->x_signed,
                             h->x_zp, h->num_sms, strm);
      if (ce != cudaSuccess) break;
      TcConvParams p{};
      p.M = (int)s.M; p.Kout = s.K; p.num_kb = h->num_kb; p.cblocks = h->cblocks; p.R = s.R; p.S = s.S;
      p.dh = s.dh; p.dw = s.dw; p.sh = s.sh; p.sw = s.sw; p.pt = s.pt; p.pl = s.pl;
      p.H = s.H; p.W = s.W; p.C = s.C; p.Ho = s.Ho; p.Wo = s.Wo;
      p.n_blocks = h->n_blocks; p.num_tiles = h->num_tiles; p.a_mode = h->a_mode;
      p.x = h->xq; p.status = h->status; p.kpb = h->kpb; p.a3d = h->a3d ? 1 : 0; p.split_epi = 1;
      p.iq_chunk_kb = h->iq_chunk_kb; p.iq_mode = h->iq_mode;
      p.q_bias = h->q_bias; p.q_mult = h->q_mult; p.q_shift = h->q_shift; p.q_scale = h->q_scale;
      p.q_zp = h->zp; p.q_lo = h->q_lo; p.q_hi = h->q_hi; p.y8 = static_cast<uint8_t*>(y);
      if (h->bn == 64)
        ce = launch_tc_conv_bn64(p, h->tmA, h->tmB, nullptr, h->grid, false, false, strm);
      else
        ce = launch_tc_conv_bn128(p, h->tmA, h->tmB, nullptr, h->grid, false, false, strm);
      break;
    }
    case CONVF_VARIANT_INT8: {
      S8Params p{};
      p.M = (int)s.M; p.Kout = s.K; p.C = s.C; p.H = s.H; p.W = s.W; p.Ho = s.Ho; p.Wo = s.Wo; p.R = s.R; p.S = s.S;
      p.sh = s.sh; p.sw = s.sw; p.pt = s.pt; p.pl = s.pl; p.dh = s.dh; p.dw = s.dw;
      p.num_kb = s.R * s.S * s.C / 64;
      p.x = static_cast<const int8_t*>(x); p.w = h->w_s8; p.bias = h->qbias; p.mult = h->qmult;
      p.shift = h->qshift; p.y = static_cast<int8_t*>(y); p.zp = h->zp; p.relu = h->desc.act == CONVF_ACT_RELU;
      p.status = h->status;
      ce = launch_s8_conv(p, strm);
      break;
    }
    default: {
      if (x != h->map_x) {
        if ((st = encode_a_map(h, x)) != CONVF_OK) return st;
      }
      TcConvParams p{};   // (the integer-exact 8-bit path has its own case above)
      p.M = (int)s.M; p.Kout = s.K; p.num_kb = h->num_kb; p.cblocks = h->cblocks; p.R = s.R; p.S = s.S;
      p.dh = s.dh; p.dw = s.dw; p.sh = s.sh; p.sw = s.sw; p.pt = s.pt; p.pl = s.pl;
      p.H = s.H; p.W = s.W; p.C = s.C; p.Ho = s.Ho; p.Wo = s.Wo;
      p.n_blocks = h->n_blocks; p.num_tiles = h->num_tiles; p.a_mode = h->a_mode;
      p.scale = h->scale; p.bias = h->bias; p.x = static_cast<const uint16_t*>(x);
      p.patch_rows = h->patch_rows; p.row_bytes = h->row_bytes; p.cpt = h->cpt;
      if (h->cpt > 0) {
        // whole taps: pad the channels into the handle's scratch copy of x first
        ce = launch_pad_channels(static_cast<const uint16_t*>(x), h->xpad, (long long)s.N * s.H * s.W, s.C, h->cpt,
                                 h->num_sms, strm);
        if (ce != cudaSuccess) break;
        p.x = h->xpad;
        p.C = h->cpt;
      }
      p.lo = h->lo; p.hi = h->hi; p.status = h->status; p.y = static_cast<float*>(y);
      p.sk = h->sk ? 1 : 0; p.sk_ws = h->sk_ws; p.sk_flags = h->sk_flags;
      p.kpb = h->kpb; p.a3d = h->a3d ? 1 : 0;
      if (h->desc.group > 1) {
        p.grp_kg = s.K / h->desc.group;
        p.grp_cg = s.Cg;
      }
      p.res = h->has_res ? res : nullptr; p.out_bf16 = h->out_bf16 ? 1 : 0;
      // split epilogue columns when CTAs hold at most 8 tiles (measured on the ResNet-50 1x1
      // layers: 5 tiles per CTA gain, 10 and 20 lose)
      p.split_epi = h->num_tiles <= 8LL * h->grid ? 1 : 0;
      const bool gather = h->a_mode == kAGather;
      if (h->rsm && res != h->map_r) {
        if ((st = encode_r_map(h, res)) != CONVF_OK) return st;
      }
      const CUtensorMap* tmR = h->rsm ? &h->tmR : nullptr;
      switch (h->bn) {
        case 32: ce = launch_tc_conv_bn32(p, h->tmA, h->tmB, tmR, h->grid, gather, h->pair, strm); break;
        case 64: ce = launch_tc_conv_bn64(p, h->tmA, h->tmB, tmR, h->grid, gather, h->pair, strm); break;
        case 128: ce = launch_tc_conv_bn128(p, h->tmA, h->tmB, tmR, h->grid, gather, h->pair, strm); break;
        default: ce = launch_tc_conv_bn256(p, h->tmA, h->tmB, tmR, h->grid, gather, h->pair, strm); break;
      }
    }
  }
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(ce));
  return ok();
}
}  // namespace

convf_status conv_fused_run(convf_handle* h, const void* x, void* y, void* stream) {
  convf_status st = check_handle(h);
  if (st != CONVF_OK) return st;
  if (h->has_res) return fail(CONVF_ERR_INVALID_ARG, "this handle adds a residual: call conv_fused_run_residual");
  return run_impl(h, x, nullptr, y, stream);
}

convf_status conv_fused_run_residual(convf_handle* h, const void* x, const void* r, void* y, void* stream) {
  convf_status st = check_handle(h);
  if (st != CONVF_OK) return st;
  if (!h->has_res) return fail(CONVF_ERR_INVALID_ARG, "this handle was created without a residual (residual = 0)");
  return run_impl(h, x, r, y, stream);
}

convf_status conv_fused_status(convf_handle* h) {
  convf_status st = check_handle(h);
  if (st != CONVF_OK) return st;
  int v = 0;
  cudaError_t ce = cudaMemcpy(&v, h->status, sizeof v, cudaMemcpyDeviceToHost);
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "status read failed: %s", cudaGetErrorString(ce));
  if (v & kStatusTimeout) return fail(CONVF_ERR_TIMEOUT, "a bounded device wait ran out in an earlier run");
  if (v & kStatusBounds)
    return fail(CONVF_ERR_BOUNDS, "a kernel computed an index outside its tensor (bounds-checking build)");
  return ok();
}

convf_status conv_fused_clear_status(convf_handle* h) {
  convf_status st = check_handle(h);
  if (st != CONVF_OK) return st;
  cudaError_t ce = cudaMemset(h->status, 0, sizeof(int));
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "status clear failed: %s", cudaGetErrorString(ce));
  return ok();
}

void conv_fused_destroy(convf_handle* h) {
  if (!h || h->magic != kMagic) return;
  h->magic = kDeadMagic;
  cudaFree(h->dev);
  delete h;
}

convf_status conv_fused_debug_fail_alloc(int n) {
  if (n < 0) return fail(CONVF_ERR_INVALID_ARG, "n=%d is negative", n);
  g_fail_countdown.store(n);
  return ok();
}

int conv_fused_debug_live_handles(void) { return g_live_handles.load(); }

int conv_fused_variant(const convf_handle* h) {
  convf_status st = check_handle(h);
  if (st != CONVF_OK) return st;
  return h->variant;
}

convf_status conv_fused_describe(const convf_handle* h, char* buf, size_t len) {
  convf_status st = check_handle(h);
  if (st != CONVF_OK) return st;
  if (!buf || len == 0) return fail(CONVF_ERR_INVALID_ARG, "buf is NULL or empty");
  static const char* names[] = {"auto", "implicit_gemm_im2col", "gemm_1x1", "depthwise", "int8_mma",
                                "implicit_gemm_gather", "implicit_gemm_window", "implicit_gemm_halo",
                                "int8_tcgen05_exact", "grouped_direct", "mbv2_block"};
  const Shape& s = h->s;
  if (h->variant == CONVF_VARIANT_IMPLICIT_GEMM_HALO)
    snprintf(buf, len,
             "variant=%s M=%lld K=%d C=%d RxS=%dx%d stride=%d,%d tile=128x%d padded_row=%d tile_rows=%d "
             "taps_per_load=%d weight_stages=%d resident=%d kblocks=%d tiles=%d grid=%d weight_bytes=%zu",
             names[h->variant], s.M, s.K, s.C, s.R, s.S, s.sh, s.sw, h->hg.bn, h->hg.Wp, h->hg.TR, h->hg.tpo,
             h->hg.b_stages, h->hg.resident ? 1 : 0, h->num_kb, h->num_tiles, h->grid, h->dev_bytes);
  else if (h->variant == CONVF_VARIANT_IMPLICIT_GEMM_WINDOW)
    snprintf(buf, len,
             "variant=%s M=%lld K=%d C=%d RxS=%dx%d stride=%d,%d tile=128x%d window=%d row_mode=%d tap_channels=%d "
             "padded_row=%d stages=%d tiles=%d grid=%d weight_bytes=%zu",
             names[h->variant], s.M, s.K, s.C, s.R, s.S, s.sh, s.sw, h->wg.bnp, h->wg.E, h->wg.rows ? 1 : 0,
             h->wg.cpt, h->wg.Wp,
             h->wg.stages, h->num_tiles, h->grid, h->dev_bytes);
  else if (h->variant == CONVF_VARIANT_MBV2_BLOCK)
    snprintf(buf, len,
             "variant=%s N=%d Cin=%d Ch=%d Cout=%d HxW=%dx%d stride=%d expand=%d residual=%d tile=%dx%d halo=%dx%d "
             "halo_row_blocks=%d halo_buffers=%d hidden_chunks=%d project_n=%d tiles=%d grid=%d smem=%zu weight_bytes=%zu",
             names[h->variant], h->mb.N, h->mb.Cin, h->mb.Ch, h->mb.Cout, h->mb.H, h->mb.W, h->mb.st, h->mb.expand,
             h->mb.residual, h->mb.TH, h->mb.TW, h->mb.IH, h->mb.IW, h->mb.rb, h->mb.nxb, h->mb.nch, h->mb.Np,
             h->num_tiles,
             h->grid, mbv2_block_smem(h->mb), h->dev_bytes);
  else if (h->variant == CONVF_VARIANT_INT8_TC)
    snprintf(buf, len,
             "variant=%s M=%lld K=%d C=%d RxS=%dx%d stride=%d,%d tile=128x%d kblocks=%d kblocks_per_step=%d "
             "act_box_per_step=%d exact_chunk_kblocks=%d requant=%s tiles=%d grid=%d weight_bytes=%zu",
             names[h->variant], s.M, s.K, s.C, s.R, s.S, s.sh, s.sw, h->bn, h->num_kb, h->kpb, h->a3d ? 1 : 0,
             h->iq_chunk_kb, h->iq_mode ? "float32" : "fixed_point", h->num_tiles, h->grid, h->dev_bytes);
  else if (h->variant == CONVF_VARIANT_DEPTHWISE || h->variant == CONVF_VARIANT_INT8 ||
           h->variant == CONVF_VARIANT_GROUPED_DIRECT)
    snprintf(buf, len, "variant=%s M=%lld K=%d C=%d RxS=%dx%d stride=%d,%d group=%d out=%s residual=%d "
             "weight_bytes=%zu", names[h->variant], s.M, s.K, s.C, s.R, s.S, s.sh, s.sw, h->desc.group,
             h->out_bf16 ? "bf16" : "f32", h->has_res ? 1 : 0, h->dev_bytes);
  else
    snprintf(buf, len,
             "variant=%s M=%lld K=%d C=%d RxS=%dx%d stride=%d,%d group=%d preact=%d tile=%dx%d cta_pair=%d stream_k=%d kblocks=%d "
             "kblocks_per_step=%d act_box_per_step=%d split_epilogue=%d out=%s residual=%d residual_staged=%d "
             "tiles=%d grid=%d patch_rows=%d tap_channels=%d weight_bytes=%zu",
             names[h->variant], s.M, s.K, s.C, s.R, s.S, s.sh, s.sw, h->desc.group, h->preact ? 1 : 0,
             h->pair ? 256 : 128, h->bn,
             h->pair ? 1 : 0,
             h->sk ? 1 : 0, h->num_kb, h->kpb, h->a3d ? 1 : 0,
             (h->bn >= 64 && !h->sk && h->a_mode != kAGather && h->num_tiles <= 8LL * h->grid) ? 1 : 0,
             h->out_bf16 ? "bf16" : "f32", h->has_res ? 1 : 0, h->rsm ? 1 : 0, h->num_tiles,
             h->grid, h->patch_rows, h->cpt, h->dev_bytes);
  return ok();
}

convf_status conv_fused_measure_int8_mma_rate(void* stream, double* tops) {
  if (!tops) return fail(CONVF_ERR_INVALID_ARG, "tops is NULL");
  int dev = 0, sms = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce == cudaSuccess) ce = measure_s8_mma_rate(sms, static_cast<cudaStream_t>(stream), tops);
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "int8 MMA rate measurement failed: %s", cudaGetErrorString(ce));
  return ok();
}

convf_status conv_fused_watchdog_selftest(int32_t* status_dev, long long budget_cycles, void* stream) {
  if (!status_dev) return fail(CONVF_ERR_INVALID_ARG, "status_dev is NULL");
  if (budget_cycles < 1 || budget_cycles > 20000000000LL)
    return fail(CONVF_ERR_INVALID_ARG, "budget_cycles=%lld is outside 1..2e10", budget_cycles);
  cudaError_t ce = launch_watchdog_selftest(status_dev, budget_cycles, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "self-test launch failed: %s", cudaGetErrorString(ce));
  return ok();
}

}  // extern "C"

// ====================================================================== allocation-free run
// Scratch for conv_fused_run_noalloc: a file-scope device array, so the entry point needs no
// cudaMalloc.  Every GPU that loads this library reserves it until the process exits.  Host code
// must not use its name as a device address (on the host it is only a stand-in symbol); the
// device address is looked up with cudaGetSymbolAddress, once per device.
namespace {
constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on first use per device).
convf_status noalloc_scratch(void** out) {
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(ce));
  if (dev < 0 || dev >= kMaxDevices) return fail(CONVF_ERR_UNSUPPORTED, "device index %d beyond %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    ce = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (ce != cudaSuccess || !p)
      return fail(CONVF_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(ce));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return CONVF_OK;
}
}  // namespace

extern "C" convf_status conv_fused_run_noalloc(const convf_desc* desc, const void* x, const void* w_packed,
                                               const float* scale, const float* bias, void* y, int32_t* status_dev,
                                               void* stream) {
  Shape s;
  convf_status st = resolve(desc, &s);
  if (st != CONVF_OK) return st;
  if ((st = check_misc(desc)) != CONVF_OK) return st;
  if (desc->dtype != CONVF_BF16 || desc->group != 1)
    return fail(CONVF_ERR_UNSUPPORTED, "the allocation-free run serves bf16 convs with group == 1");
  if (!cannot(CONVF_VARIANT_IMPLICIT_GEMM_GATHER, desc, s).empty())
    return fail(CONVF_ERR_UNSUPPORTED, "allocation-free run refused: %s",
                cannot(CONVF_VARIANT_IMPLICIT_GEMM_GATHER, desc, s).c_str());
  const int cpt = gather_cpt(s);
  if (cpt == 0)
    return fail(CONVF_ERR_UNSUPPORTED,
                "the allocation-free run serves convs with at most 8 input channels whose 128-row tiles stay "
                "inside one image and whose input rows fit the 32 KB staging buffer");
  if (desc->tile_n > 128 || desc->cta_pair == 2)
    return fail(CONVF_ERR_UNSUPPORTED, "tile_n > 128 / CTA pairs are not served by the gathered-row kernel");
  if (desc->stream_k == 2)
    return fail(CONVF_ERR_UNSUPPORTED, "stream_k = 2 (on) is not served by the allocation-free run: it has no "
                                       "workspace for partial tiles");
  if (desc->kblocks_per_step > 1)
    return fail(CONVF_ERR_UNSUPPORTED, "kblocks_per_step = %d is not served by the gathered-row kernel (one "
                                       "reduction block per step)", desc->kblocks_per_step);
  if (desc->out_dtype != CONVF_OUT_F32 || desc->residual)
    return fail(CONVF_ERR_UNSUPPORTED, "the allocation-free run writes fp32 outputs without a residual");
  // scratch layout: [padded x][scale, padded to 256][bias, padded to 256][status word]; every
  // size refusal comes before any pointer is looked at
  const int Kpad = (int)align_up((size_t)s.K, 256);
  const size_t xpad_bytes = align_up((size_t)s.N * s.H * s.W * cpt * sizeof(uint16_t), 256);
  const size_t vec_bytes = (size_t)Kpad * sizeof(float);
  const size_t need = xpad_bytes + 2 * vec_bytes + 256;
  if (need > kNoAllocScratchBytes)
    return fail(CONVF_ERR_UNSUPPORTED, "the allocation-free run needs %zu bytes of scratch; its maximum is %zu",
                need, kNoAllocScratchBytes);
  if (s.M == 0) return ok();
  if (!x || !w_packed || !scale || !bias || !y) return fail(CONVF_ERR_INVALID_ARG, "x/w_packed/scale/bias/y is NULL");
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 15) ||
      (reinterpret_cast<uintptr_t>(w_packed) & 15))
    return fail(CONVF_ERR_INVALID_ARG, "x, w_packed and y must be 16-byte aligned");
  if (!load_encoders()) return fail(CONVF_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != CONVF_OK) return st;
  int dev = 0, num_sms = 0;
  cudaGetDevice(&dev);
  cudaError_t ce = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "device query failed: %s", cudaGetErrorString(ce));

  char* base = static_cast<char*>(scratch);
  uint16_t* xpad = reinterpret_cast<uint16_t*>(base);
  float* sc = reinterpret_cast<float*>(base + xpad_bytes);
  float* bi = reinterpret_cast<float*>(base + xpad_bytes + vec_bytes);
  int* status = status_dev ? reinterpret_cast<int*>(status_dev)
                           : reinterpret_cast<int*>(base + xpad_bytes + 2 * vec_bytes);
  cudaStream_t strm = static_cast<cudaStream_t>(stream);

  // the epilogue reads whole 32-column chunks: copy the vectors and zero their padding; the
  // internal status word (used when status_dev is NULL) starts every call at zero
  if ((ce = cudaMemsetAsync(sc, 0, 2 * vec_bytes + 256, strm)) != cudaSuccess ||
      (ce = cudaMemcpyAsync(sc, scale, (size_t)s.K * sizeof(float), cudaMemcpyDeviceToDevice, strm)) != cudaSuccess ||
      (ce = cudaMemcpyAsync(bi, bias, (size_t)s.K * sizeof(float), cudaMemcpyDeviceToDevice, strm)) != cudaSuccess)
    return fail(CONVF_ERR_CUDA, "scratch set-up copy failed: %s", cudaGetErrorString(ce));

  int am = 0, cblocks = 0, ktot = 0, cpad = 0;
  tc_layout(CONVF_VARIANT_IMPLICIT_GEMM_GATHER, s, &am, &cblocks, &ktot, &cpad);
  int bn = 0;
  bool pair = false;
  bool sk = false;
  pick_tile(s.M, s.K, ktot / 64, num_sms, desc->tile_n ? desc->tile_n : 128, 1, 1, false, &bn, &pair, &sk);
  if (desc->tile_n) bn = desc->tile_n;
  const int n_blocks = (s.K + bn - 1) / bn;
  const long long tiles = (s.M + 127) / 128 * n_blocks;
  const int grid = (int)std::min<long long>(tiles, num_sms);

  CUtensorMap tmA, tmB;
  std::memset(&tmA, 0, sizeof tmA);
  const cuuint32_t es[2] = {1, 1};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)ktot, (cuuint64_t)s.K};
    const cuuint64_t strides[1] = {(cuuint64_t)ktot * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)bn};
    CUresult r = g_encode_tiled(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w_packed), dims, strides,
                                box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(CONVF_ERR_CUDA, "weight tensor map encoding failed (CUresult %d)", (int)r);
  }

  ce = launch_pad_channels(static_cast<const uint16_t*>(x), xpad, (long long)s.N * s.H * s.W, s.C, cpt, num_sms, strm);
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "channel pre-pass launch failed: %s", cudaGetErrorString(ce));
  float lo, hi;
  act_bounds(desc, &lo, &hi);
  TcConvParams p{};
  p.M = (int)s.M; p.Kout = s.K; p.num_kb = ktot / 64; p.cblocks = 0; p.R = s.R; p.S = s.S;
  p.dh = s.dh; p.dw = s.dw; p.sh = s.sh; p.sw = s.sw; p.pt = s.pt; p.pl = s.pl;
  p.H = s.H; p.W = s.W; p.C = cpt; p.Ho = s.Ho; p.Wo = s.Wo;
  p.n_blocks = n_blocks; p.num_tiles = (int)tiles; p.a_mode = kAGather;
  p.kpb = 1; p.a3d = 0;
  p.scale = sc; p.bias = bi; p.x = xpad; p.lo = lo; p.hi = hi; p.status = status; p.y = static_cast<float*>(y);
  p.patch_rows = patch_rows_for(s, cpt); p.row_bytes = s.W * cpt * 2; p.cpt = cpt;
  switch (bn) {
    case 32: ce = launch_tc_conv_bn32(p, tmA, tmB, nullptr, grid, true, false, strm); break;
    case 64: ce = launch_tc_conv_bn64(p, tmA, tmB, nullptr, grid, true, false, strm); break;
    default: ce = launch_tc_conv_bn128(p, tmA, tmB, nullptr, grid, true, false, strm); break;
  }
  if (ce != cudaSuccess) return fail(CONVF_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(ce));
  return ok();
}

// ====================================================================== services for chain.cu
namespace convf {

convf_status record_error(convf_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}
convf_status record_ok() { return ok(); }
bool take_injected_alloc_failure() { return injected_alloc_failure(); }

bool tensor_map_encoders(EncodeTiledFn* tiled, EncodeIm2colFn* im2col) {
  if (!load_encoders()) return false;
  *tiled = g_encode_tiled;
  *im2col = g_encode_im2col;
  return true;
}

convf_status chain_conv_info(const convf_handle* h, ChainConvInfo* o) {
  convf_status st = check_handle(h);
  if (st != CONVF_OK) return st;
  if (h->variant != CONVF_VARIANT_GEMM_1X1 && h->variant != CONVF_VARIANT_IMPLICIT_GEMM)
    return fail(CONVF_ERR_UNSUPPORTED, "variant %d is not a tcgen05 1x1-GEMM or im2col implicit-GEMM conv",
                h->variant);
  if (h->desc.dtype != CONVF_BF16) return fail(CONVF_ERR_UNSUPPORTED, "only bf16 convs can be chain steps");
  if (h->desc.group != 1) return fail(CONVF_ERR_UNSUPPORTED, "grouped convs (group %d) cannot be chain steps", h->desc.group);
  if (h->preact) return fail(CONVF_ERR_UNSUPPORTED, "convs with a pre-activation prologue cannot be chain steps");
  const Shape& s = h->s;
  o->variant = h->variant;
  o->a_mode = h->a_mode;
  o->cblocks = h->cblocks;
  o->ktot = h->ktot;
  o->num_kb = h->ktot / 64;
  o->N = s.N; o->C = s.C; o->H = s.H; o->W = s.W; o->K = s.K; o->R = s.R; o->S = s.S;
  o->sh = s.sh; o->sw = s.sw; o->dh = s.dh; o->dw = s.dw;
  o->pt = s.pt; o->pl = s.pl; o->pb = s.pb; o->pr = s.pr;
  o->Ho = s.Ho; o->Wo = s.Wo; o->M = s.M;
  o->w = h->w_bf16;
  o->scale = h->scale;
  o->bias = h->bias;
  o->lo = h->lo;
  o->hi = h->hi;
  o->out_bf16 = h->out_bf16;
  o->has_res = h->has_res;
  o->device = h->device;
  return CONVF_OK;
}

}  // namespace convf
