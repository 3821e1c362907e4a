// Conv chain, host side (conv_fused_chain_*): validates a sequence of conv runs, finds each
// step's dependencies by buffer identity (a step's x or residual is an earlier step's y), fixes
// each step's tile width, encodes its tensor maps for its own buffers and uploads the step
// table; run is then a single launch of the persistent chain kernel (tc_chain.cu).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/conv_fused.h"
#include "api_internal.h"
#include "convf_internal.h"
#include "ptx.cuh"

using namespace convf;

namespace {
constexpr uint32_t kChainMagic = 0xC4A1F00Du;
constexpr uint32_t kChainDead = 0xDEADC4A1u;
constexpr int kMaxChainSteps = 4096;

struct Range {
  uintptr_t a, b;   // [a, b)
  bool overlaps(const Range& o) const { return a < o.b && o.a < b; }
};
Range range_of(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + bytes};
}
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

struct convf_chain {
  uint32_t magic;
  int device;
  int grid, nsteps, total_tiles, total_mtiles;
  bool out_bf16;
  bool pair;             // CTA pairs (256-row tiles)
  void* dev;             // one device allocation: step table, counters, state, status
  ChainStep* d_steps;
  uint32_t* d_counters;
  uint32_t* d_state;
  int* d_status;
  std::vector<ChainStep> steps;   // host copy (describe)
  std::vector<int> filter;        // 100 * R + S of each step (describe)
};

namespace {

convf_status check_chain(const convf_chain* c) {
  if (!c) return record_error(CONVF_ERR_INVALID_ARG, "chain is NULL");
  if (c->magic == kChainDead) return record_error(CONVF_ERR_INVALID_ARG, "chain was destroyed");
  if (c->magic != kChainMagic) return record_error(CONVF_ERR_INVALID_ARG, "not a convf chain");
  return CONVF_OK;
}

// the producing step of buffer `p` of `bytes` bytes read by step j: -1 (no step writes it), or
// i < j with y_i == p and the same size; -2 (message set) when the sequence cannot run as one
// launch (a partial overlap, or a later step writes what step j reads)
int find_source(const std::vector<Range>& outs, const convf_chain_step* steps, int j, const void* p, size_t bytes,
                const char* what) {
  const Range r = range_of(p, bytes);
  int src = -1;
  for (int i = 0; i < static_cast<int>(outs.size()); ++i) {
    if (!outs[i].overlaps(r)) continue;
    if (i >= j) {
      record_error(CONVF_ERR_UNSUPPORTED,
                   "step %d's %s overlaps the output of step %d, which does not come before it (one launch cannot "
                   "order a read before a later write)", j, what, i);
      return -2;
    }
    if (steps[i].y != p || outs[i].b - outs[i].a != bytes) {
      record_error(CONVF_ERR_UNSUPPORTED,
                   "step %d's %s overlaps step %d's output without being exactly that tensor", j, what, i);
      return -2;
    }
    if (src >= 0) {
      record_error(CONVF_ERR_UNSUPPORTED, "step %d's %s is written by two steps (%d and %d)", j, what, src, i);
      return -2;
    }
    src = i;
  }
  return src;
}

}  // namespace

extern "C" {

convf_status conv_fused_chain_create(const convf_chain_step* steps, int n, convf_chain** out) {
  return conv_fused_chain_create_ex(steps, n, 0, out);
}

convf_status conv_fused_chain_create_ex(const convf_chain_step* steps, int n, int cta_pairs, convf_chain** out) {
  if (!out) return record_error(CONVF_ERR_INVALID_ARG, "out is NULL");
  if (cta_pairs < 0 || cta_pairs > 2)
    return record_error(CONVF_ERR_INVALID_ARG, "cta_pairs=%d must be 0 (auto), 1 (single CTAs) or 2 (CTA pairs)",
                        cta_pairs);
  *out = nullptr;
  if (!steps) return record_error(CONVF_ERR_INVALID_ARG, "steps is NULL");
  if (n < 1 || n > kMaxChainSteps)
    return record_error(CONVF_ERR_INVALID_ARG, "n=%d must be in [1, %d]", n, kMaxChainSteps);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return record_error(CONVF_ERR_CUDA, "cudaGetDevice failed");
  EncodeTiledFn enc_tiled = nullptr;
  EncodeIm2colFn enc_im2col = nullptr;
  if (!tensor_map_encoders(&enc_tiled, &enc_im2col))
    return record_error(CONVF_ERR_CUDA, "cuTensorMapEncodeTiled/Im2col are unavailable from the driver");

  std::vector<ChainConvInfo> info(n);
  for (int j = 0; j < n; ++j) {
    const convf_status st = chain_conv_info(steps[j].conv, &info[j]);
    if (st != CONVF_OK) {
      const std::string why = conv_fused_last_error();
      return record_error(st, "step %d: %s", j, why.c_str());
    }
  }
  const bool out_bf16 = info[0].out_bf16;
  std::vector<Range> outs(n);
  for (int j = 0; j < n; ++j) {
    const ChainConvInfo& f = info[j];
    const convf_chain_step& st = steps[j];
    if (f.device != dev)
      return record_error(CONVF_ERR_INVALID_ARG, "step %d's handle lives on device %d, not the current device %d", j,
                          f.device, dev);
    if (f.out_bf16 != out_bf16)
      return record_error(CONVF_ERR_UNSUPPORTED, "step %d's output type differs from step 0's: one chain writes "
                                                 "either fp32 or bf16 outputs", j);
    if (!st.x || !st.y) return record_error(CONVF_ERR_INVALID_ARG, "step %d: x and y must not be NULL", j);
    if (f.has_res != (st.r != nullptr))
      return record_error(CONVF_ERR_INVALID_ARG, "step %d: a residual is %s but the handle was created with "
                                                 "residual = %d", j, st.r ? "given" : "missing", f.has_res ? 1 : 0);
    if (!aligned16(st.x) || !aligned16(st.y) || (st.r && !aligned16(st.r)))
      return record_error(CONVF_ERR_INVALID_ARG, "step %d: x, y and r must be 16-byte aligned", j);
    if (f.M < 1) return record_error(CONVF_ERR_UNSUPPORTED, "step %d has no output rows (empty batch)", j);
    if (f.M > (1LL << 31) - 256 || static_cast<long long>(f.N) * f.H * f.W > (1LL << 31) - 256)
      return record_error(CONVF_ERR_UNSUPPORTED, "step %d has more than 2^31 - 256 pixels", j);
    if (f.C % 8 != 0 || f.K % 8 != 0)
      return record_error(CONVF_ERR_UNSUPPORTED, "step %d: C=%d and K=%d must be multiples of 8", j, f.C, f.K);
    outs[j] = range_of(st.y, static_cast<size_t>(f.M) * f.K * (out_bf16 ? 2 : 4));
  }
  for (int j = 0; j < n; ++j)
    for (int i = 0; i < j; ++i)
      if (outs[i].overlaps(outs[j]))
        return record_error(CONVF_ERR_UNSUPPORTED, "steps %d and %d write overlapping outputs", i, j);

  std::vector<int> srcs(n, -1), rsrcs(n, -1);
  bool dependent = false;
  for (int j = 0; j < n; ++j) {
    const ChainConvInfo& f = info[j];
    const convf_chain_step& st = steps[j];
    const size_t esize = out_bf16 ? 2 : 4;
    const size_t xbytes = static_cast<size_t>(f.N) * f.H * f.W * f.C * 2;
    const Range xr = range_of(st.x, xbytes);
    if (xr.overlaps(outs[j]) || (st.r && range_of(st.r, static_cast<size_t>(f.M) * f.K * esize).overlaps(outs[j])))
      return record_error(CONVF_ERR_UNSUPPORTED, "step %d's output overlaps its own input or residual", j);
    const int src = find_source(outs, steps, j, st.x, xbytes, "x");
    if (src == -2) return CONVF_ERR_UNSUPPORTED;
    if (src >= 0) {
      const ChainConvInfo& g = info[src];
      if (!out_bf16)
        return record_error(CONVF_ERR_UNSUPPORTED, "step %d reads step %d's fp32 output as its bf16 input", j, src);
      if (g.N != f.N || g.Ho != f.H || g.Wo != f.W || g.K != f.C)
        return record_error(CONVF_ERR_INVALID_ARG, "step %d's input [%d,%d,%d,%d] is not step %d's output [%d,%d,%d,%d]",
                            j, f.N, f.C, f.H, f.W, src, g.N, g.K, g.Ho, g.Wo);
    }
    int rsrc = -1;
    if (st.r) {
      rsrc = find_source(outs, steps, j, st.r, static_cast<size_t>(f.M) * f.K * esize, "residual");
      if (rsrc == -2) return CONVF_ERR_UNSUPPORTED;
      if (rsrc >= 0 && (info[rsrc].M != f.M || info[rsrc].K != f.K))
        return record_error(CONVF_ERR_INVALID_ARG, "step %d's residual is not shaped like step %d's output", j, rsrc);
    }
    srcs[j] = src;
    rsrcs[j] = rsrc;
    dependent = dependent || src >= 0 || rsrc >= 0;
  }
  // CTA pairs: 256-row tiles of up to 256 columns, half the weight bytes per FLOP.  Per layer
  // shape (ResNet-50, batch 32, steady state) they were 6-25% faster on the wide compute-bound
  // steps (C and K >= 256 and at least ~150 FLOP per algorithmic byte) and up to 50% slower on
  // the narrow or HBM-bound ones; they also halve every step's tiles, which leaves SMs idle where
  // a step waits for a small predecessor.  The automatic choice takes them only for chains of
  // independent steps that are all wide.
  bool all_wide = true;
  for (int j = 0; j < n; ++j) all_wide = all_wide && info[j].C >= 256 && info[j].K >= 256;
  const bool pair = cta_pairs == 2 || (cta_pairs == 0 && !dependent && all_wide);
  const int tile_m = pair ? 256 : 128;

  std::vector<ChainStep> cs(n);
  std::vector<int> filter(n);
  long long tiles = 0, mtiles_total = 0;
  for (int j = 0; j < n; ++j) {
    const ChainConvInfo& f = info[j];
    const convf_chain_step& st = steps[j];
    const int src = srcs[j], rsrc = rsrcs[j];
    ChainStep& c = cs[j];
    std::memset(&c, 0, sizeof c);
    ChainGeom& g = c.g;
    g.a_mode = f.a_mode;
    g.M = static_cast<int>(f.M);
    g.Kout = f.K;
    g.C = f.C; g.H = f.H; g.W = f.W; g.Ho = f.Ho; g.Wo = f.Wo; g.R = f.R; g.S = f.S;
    g.sh = f.sh; g.sw = f.sw; g.pt = f.pt; g.pl = f.pl; g.dh = f.dh; g.dw = f.dw;
    g.cblocks = f.cblocks;
    g.num_kb = f.num_kb;
    g.mtiles = static_cast<int>((f.M + 127) / 128);   // 128-row blocks (the dependency counters)
    // single CTAs: 128 x 128 tiles (128 x 64 for K <= 64; narrower tiles for steps with fewer
    // tiles than SMs measured slower, in a chain of independent steps and in a dependent one
    // alike: an im2col tile's activation loads per FLOP double); pairs: 256 x 256 (256 x 128 for
    // K <= 128, 256 x 64 for K <= 64)
    g.bn = f.K <= 64 ? 64 : (f.K <= 128 || !pair ? 128 : 256);
    g.n_blocks = (f.K + g.bn - 1) / g.bn;
    g.tile0 = static_cast<int>(tiles);
    tiles += (f.M + tile_m - 1) / tile_m * g.n_blocks;
    if (tiles > (1LL << 30)) return record_error(CONVF_ERR_UNSUPPORTED, "more than 2^30 tiles in one chain");
    g.tile_end = static_cast<int>(tiles);
    g.idesc = idesc_bf16_f32(tile_m, g.bn);
    g.lo = f.lo;
    g.hi = f.hi;
    g.scale = f.scale;
    g.bias = f.bias;
    g.x = st.x;
    g.y = st.y;
    g.res = st.r;
    g.src = src;
    g.rsrc = rsrc;
    g.src_nb = src >= 0 ? cs[src].g.n_blocks : 0;
    g.rsrc_nb = rsrc >= 0 ? cs[rsrc].g.n_blocks : 0;
    g.done = reinterpret_cast<uint32_t*>(static_cast<uintptr_t>(mtiles_total));   // offsets until uploaded
    mtiles_total += g.mtiles;
    filter[j] = f.R * 100 + f.S;

    CUresult r;
    if (f.a_mode == kA2D) {
      g.a3d = f.C % 64 == 0 && f.num_kb % 2 == 0;
      if (g.a3d) {
        // {64 channels of a k-block, pixel, k-block}: one box = the two k-blocks of a step
        const cuuint64_t dims[3] = {64, (cuuint64_t)f.M, (cuuint64_t)(f.C / 64)};
        const cuuint64_t strides[2] = {(cuuint64_t)f.C * 2, 128};
        const cuuint32_t box[3] = {64, 128, 2};
        const cuuint32_t es[3] = {1, 1, 1};
        r = enc_tiled(&c.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(st.x), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      } else {
        const cuuint64_t dims[2] = {(cuuint64_t)f.C, (cuuint64_t)f.M};
        const cuuint64_t strides[1] = {(cuuint64_t)f.C * 2};
        const cuuint32_t box[2] = {64, 128};
        const cuuint32_t es[2] = {1, 1};
        r = enc_tiled(&c.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(st.x), dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      }
    } else {
      const cuuint64_t dims[4] = {(cuuint64_t)f.C, (cuuint64_t)f.W, (cuuint64_t)f.H, (cuuint64_t)f.N};
      const cuuint64_t strides[3] = {(cuuint64_t)f.C * 2, (cuuint64_t)f.W * f.C * 2, (cuuint64_t)f.H * f.W * f.C * 2};
      const int lower[2] = {-f.pl, -f.pt};
      const int upper[2] = {f.pr - (f.S - 1) * f.dw, f.pb - (f.R - 1) * f.dh};
      const cuuint32_t es[4] = {1, (cuuint32_t)f.sw, (cuuint32_t)f.sh, 1};
      r = enc_im2col(&c.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(st.x), dims, strides, lower, upper,
                     64, 128, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS)
      return record_error(CONVF_ERR_CUDA, "step %d: activation tensor map encoding failed (CUresult %d)", j, (int)r);
    {
      // {64 elements of a k-block, output channel, k-block}: one box = a step's two k-blocks
      // (one when the reduction is a single block)
      const cuuint64_t dims[3] = {64, (cuuint64_t)f.K, (cuuint64_t)f.num_kb};
      const cuuint64_t strides[2] = {(cuuint64_t)f.ktot * 2, 128};
      const cuuint32_t box[3] = {64, (cuuint32_t)(pair ? g.bn / 2 : g.bn), (cuuint32_t)std::min(2, f.num_kb)};
      const cuuint32_t es[3] = {1, 1, 1};
      r = enc_tiled(&c.tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(f.w), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS)
        return record_error(CONVF_ERR_CUDA, "step %d: weight tensor map encoding failed (CUresult %d)", j, (int)r);
    }
  }

  int num_sms = 0;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || num_sms < 1)
    return record_error(CONVF_ERR_CUDA, "cannot query the SM count");
  const int max_ctas = tc_chain_max_ctas(out_bf16, pair, num_sms);
  if (max_ctas < (pair ? 2 : 1)) return record_error(CONVF_ERR_CUDA, "the chain kernel cannot be resident on this device");

  const bool host_injected = take_injected_alloc_failure();
  convf_chain* c = host_injected ? nullptr : new (std::nothrow) convf_chain();
  if (!c) return record_error(CONVF_ERR_OOM, "chain allocation failed%s", host_injected ? " (injected)" : "");
  c->magic = kChainMagic;
  c->device = dev;
  c->nsteps = n;
  c->total_tiles = static_cast<int>(tiles);
  c->total_mtiles = static_cast<int>(mtiles_total);
  c->out_bf16 = out_bf16;
  c->pair = pair;
  // every CTA resident at once (they wait for one another's tiles); a pair takes a tile
  c->grid = pair ? 2 * static_cast<int>(std::min<long long>(tiles, max_ctas / 2))
                 : static_cast<int>(std::min<long long>(tiles, max_ctas));
  const size_t steps_bytes = (sizeof(ChainStep) * n + 255) / 256 * 256;
  const size_t ctr_bytes = (static_cast<size_t>(mtiles_total) * 4 + 255) / 256 * 256;
  const size_t bytes = steps_bytes + ctr_bytes + 256;
  const bool dev_injected = take_injected_alloc_failure();
  const cudaError_t me = dev_injected ? cudaErrorMemoryAllocation : cudaMalloc(&c->dev, bytes);
  if (me != cudaSuccess) {
    c->dev = nullptr;
    delete c;
    return record_error(CONVF_ERR_OOM, "device allocation of %zu bytes failed%s", bytes,
                        dev_injected ? " (injected)" : "");
  }
  uint8_t* base = static_cast<uint8_t*>(c->dev);
  c->d_steps = reinterpret_cast<ChainStep*>(base);
  c->d_counters = reinterpret_cast<uint32_t*>(base + steps_bytes);
  c->d_state = reinterpret_cast<uint32_t*>(base + steps_bytes + ctr_bytes);
  c->d_status = reinterpret_cast<int*>(base + steps_bytes + ctr_bytes + 16);
  for (ChainStep& s : cs) s.g.done = c->d_counters + reinterpret_cast<uintptr_t>(s.g.done);
  for (ChainStep& s : cs) {
    s.g.src_done = s.g.src >= 0 ? cs[s.g.src].g.done : nullptr;
    s.g.rsrc_done = s.g.rsrc >= 0 ? cs[s.g.rsrc].g.done : nullptr;
    if (s.g.src >= 0) cs[s.g.src].g.consumed = 1;
    if (s.g.rsrc >= 0) cs[s.g.rsrc].g.consumed = 1;
  }
  cudaError_t e = cudaMemcpy(c->d_steps, cs.data(), sizeof(ChainStep) * n, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemset(base + steps_bytes, 0, ctr_bytes + 256);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(c->dev);
    delete c;
    return record_error(CONVF_ERR_CUDA, "uploading the chain's step table failed: %s", cudaGetErrorString(e));
  }
  c->steps = std::move(cs);
  c->filter = std::move(filter);
  *out = c;
  return record_ok();
}

convf_status conv_fused_chain_run(convf_chain* c, void* stream) {
  convf_status st = check_chain(c);
  if (st != CONVF_OK) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device)
    return record_error(CONVF_ERR_INVALID_ARG, "the current device (%d) is not the chain's device (%d)", dev, c->device);
  ChainParams p{};
  p.steps = c->d_steps;
  p.nsteps = c->nsteps;
  p.total_tiles = c->total_tiles;
  p.counters = c->d_counters;
  p.total_mtiles = c->total_mtiles;
  p.state = c->d_state;
  p.status = c->d_status;
  const cudaError_t e = launch_tc_chain(p, c->out_bf16, c->pair, c->grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_error(CONVF_ERR_CUDA, "chain launch failed: %s", cudaGetErrorString(e));
  return record_ok();
}

convf_status conv_fused_chain_status(convf_chain* c) {
  convf_status st = check_chain(c);
  if (st != CONVF_OK) return st;
  int v = 0;
  if (cudaMemcpy(&v, c->d_status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return record_error(CONVF_ERR_CUDA, "reading the chain's status failed");
  if (v & kStatusTimeout)
    return record_error(CONVF_ERR_TIMEOUT, "a bounded device wait ran out in an earlier run of the chain");
  if (v & kStatusBounds)
    return record_error(CONVF_ERR_BOUNDS, "a chain kernel computed an out-of-range index (bounds-checking build)");
  return record_ok();
}

convf_status conv_fused_chain_clear_status(convf_chain* c) {
  convf_status st = check_chain(c);
  if (st != CONVF_OK) return st;
  if (cudaMemset(c->d_status, 0, sizeof(int)) != cudaSuccess)
    return record_error(CONVF_ERR_CUDA, "clearing the chain's status failed");
  return record_ok();
}

convf_status conv_fused_chain_describe(const convf_chain* c, char* buf, size_t len) {
  convf_status st = check_chain(c);
  if (st != CONVF_OK) return st;
  if (!buf || len == 0) return record_error(CONVF_ERR_INVALID_ARG, "buf is NULL or len is 0");
  std::string s;
  char line[160];
  snprintf(line, sizeof line, "steps=%d tiles=%d grid=%d cta_pairs=%d out=%s", c->nsteps, c->total_tiles, c->grid,
           c->pair ? 1 : 0, c->out_bf16 ? "bf16" : "f32");
  s += line;
  for (int j = 0; j < c->nsteps; ++j) {
    const ChainGeom& q = c->steps[j].g;
    char rs[16];
    if (!q.res)
      snprintf(rs, sizeof rs, "none");
    else
      snprintf(rs, sizeof rs, "%d", q.rsrc);
    snprintf(line, sizeof line, " | %d:%dx%d M=%d K=%d tile=%dx%d kb=%d%s src=%d res=%s", j, c->filter[j] / 100,
             c->filter[j] % 100, q.M, q.Kout, c->pair ? 256 : 128, q.bn, q.num_kb, q.a3d ? " a3d" : "", q.src, rs);
    s += line;
  }
  snprintf(buf, len, "%s", s.c_str());
  return record_ok();
}

void conv_fused_chain_destroy(convf_chain* c) {
  if (!c || c->magic != kChainMagic) return;
  cudaFree(c->dev);
  c->magic = kChainDead;
  delete c;
}

}  // extern "C"
