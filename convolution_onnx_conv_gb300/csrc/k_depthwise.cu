// Depthwise convolution (group == C == K) on CUDA cores: memory-bound (about 2-3 flop per
// byte), so no tensor cores.  NHWC bf16 in, fp32 taps with the BN scale folded in, fp32 out.
//
// 3x3, dilation 1, strides {1, 2}: persistent kernels over tiles of 7 output rows x 16 or 32
// output columns x 32 channels.  One thread per CTA streams each tile's input window (with its
// halo) into a ring of shared-memory stages with a single 4-D TMA load, so the loads of the next
// tiles are in flight while the current one is computed and no register holds a byte in flight;
// padding is the TMA's zero fill.  Each thread owns 4 channels of one output column (stride 2,
// and stride-1 images 16k but not 32k columns wide) or of two neighbouring output columns
// (stride 1 otherwise), walks the window's input rows once, scattering every converted row into
// the (up to three) output rows it feeds, then stores each output row as one 16-byte vector per
// column as soon as it is complete.  The taps of a CTA's first channel slab load, and its first
// tile's input window is prefetched into L2, before the wait for the previous kernel.
#include <cuda_bf16.h>

#include "convf_internal.h"
#include "ptx.cuh"

#include <mutex>

namespace convf {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float clampf(float v, float lo, float hi) { return fminf(fmaxf(v, lo), hi); }

// Two fp32 lanes in one 64-bit register pair, for the packed fp32 FMA of sm_100-class SMs
// (two independent round-to-nearest fused multiply-adds per instruction).
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack_f32x2(uint32_t lo_bits, uint32_t hi_bits) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo_bits), "r"(hi_bits));
  return r;
}
__device__ __forceinline__ f32x2 pack_f32x2(float lo, float hi) {
  return pack_f32x2(__float_as_uint(lo), __float_as_uint(hi));
}
__device__ __forceinline__ void unpack_f32x2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma_f32x2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// a 32-bit word holding two bf16 values (channel e in the low half) -> fp32 pair (e, e+1)
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w) { return pack_f32x2(w << 16, w & 0xFFFF0000u); }

// Column lanes per image in a stride-2 tile: 16, or 8 when the output is at most 8 columns
// wide, in which case one tile holds two images (the 16 lanes stay busy on 7-wide layers).
__host__ __device__ __forceinline__ int dw_tile_cols(int Wo) { return Wo <= 8 ? 8 : 16; }
// Stride-1 tiles of the two-column kernel have 32 column lanes: 32 columns of one image, or 16
// of two, or 8 of four.
__host__ __device__ __forceinline__ int dw_pair_cols(int Wo) { return Wo <= 8 ? 8 : Wo <= 16 ? 16 : 32; }
// Stride 1 runs on the two-column kernel unless its 32-column blocks leave more columns idle than
// the one-column kernel's 16-column blocks (e.g. 112 = 7 x 16 columns: measured 7 us faster per
// MobileNetV2 layer on 16-column tiles; 56-wide layers are faster on 32-column pairs).
__host__ __device__ __forceinline__ bool dw_use_pair(int Wo) {
  return Wo <= 16 || (Wo + 31) / 32 * 32 <= (Wo + 15) / 16 * 16;
}

// The nine taps and the bias of channels c..c+3 as fp32 pairs (zero past the last channel).
__device__ __forceinline__ void dw_load_taps(const DwParams& p, int c, f32x2 (&tap)[9][2], f32x2 (&bias)[2]) {
  const bool ok = c < p.C;
#pragma unroll
  for (int j = 0; j < 9; ++j) {
    const float4 v = ok ? __ldg(reinterpret_cast<const float4*>(p.taps + j * p.C + c)) : make_float4(0, 0, 0, 0);
    tap[j][0] = pack_f32x2(v.x, v.y);
    tap[j][1] = pack_f32x2(v.z, v.w);
  }
  const float4 b = ok ? __ldg(reinterpret_cast<const float4*>(p.bias + c)) : make_float4(0, 0, 0, 0);
  bias[0] = pack_f32x2(b.x, b.y);
  bias[1] = pack_f32x2(b.z, b.w);
}

// The input window of this CTA's first tile (tile index blockIdx.x: channel slab fastest, then
// column block, row block, image group) towards L2 before the wait for the previous kernel (a
// prefetch reads no stale data: what that kernel still writes lands in L2, which serves every
// read after the wait).  The box starts at column and row max(0, .): the padding holds no data.
__device__ __forceinline__ void dw_prefetch_first_window(const DwParams& p, const CUtensorMap* tm, int col_step,
                                                         int row_step, int nb, int cs) {
  const uint32_t u = blockIdx.x;
  const uint32_t t = fast_div(u, p.f_slabs);
  const int slab = static_cast<int>(u - t * p.f_slabs.d);
  const uint32_t t2 = fast_div(t, p.f_owbs);
  const int owb = static_cast<int>(t - t2 * p.f_owbs.d);
  const int ng = static_cast<int>(fast_div(t2, p.f_ohbs));
  const int ohb = static_cast<int>(t2 - ng * p.f_ohbs.d);
  if (ng * nb >= p.N) return;
  tma_prefetch_l2_4d(tm, slab * cs, max(0, owb * col_step - p.pl), max(0, ohb * row_step - p.pt), ng * nb);
}

// Epilogue of four channels of one output pixel at element offset e of y: clamp and a streaming
// 16-byte fp32 store, or (EXT) the residual added first and fp32 or bf16 (nearest even) stores.
template <bool EXT>
__device__ __forceinline__ void dw_store4(const DwParams& p, size_t e, f32x2 a0, f32x2 a1) {
  if (!CONVF_IN_BOUNDS(e + 4 <= static_cast<size_t>(p.N) * p.Ho * p.Wo * p.C, p.status)) return;
  float v0, v1, v2, v3;
  unpack_f32x2(a0, v0, v1);
  unpack_f32x2(a1, v2, v3);
  if (!EXT) {
    // streaming store: the output is not re-read here, keep L2 for the input windows
    __stcs(reinterpret_cast<float4*>(p.y + e), make_float4(clampf(v0, p.lo, p.hi), clampf(v1, p.lo, p.hi),
                                                           clampf(v2, p.lo, p.hi), clampf(v3, p.lo, p.hi)));
    return;
  }
  if (p.res != nullptr) {
    if (p.out_bf16) {
      const uint2 r = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.res) + e));
      v0 += __uint_as_float(r.x << 16);
      v1 += __uint_as_float(r.x & 0xFFFF0000u);
      v2 += __uint_as_float(r.y << 16);
      v3 += __uint_as_float(r.y & 0xFFFF0000u);
    } else {
      const float4 r = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.res) + e));
      v0 += r.x;
      v1 += r.y;
      v2 += r.z;
      v3 += r.w;
    }
  }
  v0 = clampf(v0, p.lo, p.hi);
  v1 = clampf(v1, p.lo, p.hi);
  v2 = clampf(v2, p.lo, p.hi);
  v3 = clampf(v3, p.lo, p.hi);
  if (p.out_bf16) {
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(v0, v1), b1 = __floats2bfloat162_rn(v2, v3);
    __stcs(reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.y) + e),
           make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1)));
  } else {
    __stcs(reinterpret_cast<float4*>(p.y + e), make_float4(v0, v1, v2, v3));
  }
}

template <int SW>
struct DwTile {
  static constexpr int kTH = 7;                          // output rows per tile
  static constexpr int kLanes = 16;                      // output columns per tile (all images)
  static constexpr int kCS = 32;                         // channels per tile (64-byte TMA rows)
  static constexpr int kThreads = kLanes * kCS / 4;      // 4 channels per thread: 128
  static constexpr int kInH = (kTH - 1) * SW + 3;        // input window rows: 9 or 15
  __host__ __device__ static constexpr int in_w(int cols) { return (cols - 1) * SW + 3; }
  __host__ __device__ static constexpr int bytes(int cols) { return (kLanes / cols) * kInH * in_w(cols) * kCS * 2; }
  static constexpr int kMaxBytes = bytes(16) > bytes(8) ? bytes(16) : bytes(8);
  static constexpr int kStageBytes = (kMaxBytes + 127) / 128 * 128;
  static constexpr int kStages = SW == 1 ? 3 : 2;
  static constexpr int kSlots = SW == 1 ? 3 : 2;         // output rows accumulated at once
  static constexpr int kSmem = kStages * kStageBytes + 128 + 2 * 8 * kStages;
};

// EXT: bf16 output and/or a residual (DwParams::out_bf16, res), its own instantiation so the
// fp32 store path keeps its code
template <int SW, int TCOLS, bool EXT>
__global__ void __launch_bounds__(DwTile<SW>::kThreads) dw3x3_tma_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                         const DwParams p) {
  using T = DwTile<SW>;
  extern __shared__ uint8_t dw_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dw_smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::kStages * T::kStageBytes);
  uint64_t* empty = full + T::kStages;
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;

  const int tid = threadIdx.x;
  const int cq = tid & 7;                  // 4-channel group within the tile's 32 channels
  const int lane = tid >> 3;               // output column lane of the tile
  constexpr int tcols = TCOLS;
  constexpr int nb = T::kLanes / tcols;    // images per tile
  constexpr int in_w = T::in_w(tcols);
  constexpr uint32_t tile_bytes = T::bytes(tcols);
  const int img = lane / tcols;            // this lane's image within the tile
  const int col = lane - img * tcols;      // and its output column within the column block
  if (tid == 0) {
#pragma unroll
    for (int st = 0; st < T::kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], T::kThreads / 32);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    abort_flag = 0;
  }
  __syncthreads();
  pdl_launch_dependents();
  // the taps and bias of this CTA's first channel slab (the slab index varies fastest in the
  // tile order) are constants of the handle, so they load before the wait for the previous kernel
  f32x2 tap[9][2], bias[2];    // channel pairs (c, c+1), (c+2, c+3)
  int cur_slab = static_cast<int>(blockIdx.x - fast_div(blockIdx.x, p.f_slabs) * p.f_slabs.d);
  dw_load_taps(p, cur_slab * T::kCS + cq * 4, tap, bias);
  if (tid == 0) dw_prefetch_first_window(p, &tmX, tcols * SW, T::kTH * SW, nb, T::kCS);
  pdl_wait_prior();

  const int slabs = p.f_slabs.d;
  const int owbs = p.f_owbs.d;
  const int ohbs = p.f_ohbs.d;
  const int units = (p.N + nb - 1) / nb * ohbs * owbs * slabs;
  const int G = gridDim.x;
  int issued = 0, waited = 0;   // tiles whose loads this thread issued / saw land (thread 0's count)

  // tile u -> (slab fastest, then column block, row block, image group)
  auto decode = [&](uint32_t u, int& slab, int& owb, int& ohb, int& ng) {
    const uint32_t t = fast_div(u, p.f_slabs);
    slab = static_cast<int>(u - t * p.f_slabs.d);
    const uint32_t t2 = fast_div(t, p.f_owbs);
    owb = static_cast<int>(t - t2 * p.f_owbs.d);
    ng = static_cast<int>(fast_div(t2, p.f_ohbs));
    ohb = static_cast<int>(t2 - ng * p.f_ohbs.d);
  };
  // load this CTA's j-th tile (tile index u) into stage j % kStages, once every warp has
  // released that stage's previous tile (j - kStages)
  auto issue = [&](int j, int u) {
    const int stage = j % T::kStages;
    if (j >= T::kStages && !mbar_wait(&empty[stage], ((j / T::kStages) - 1) & 1, abort_v, p.status)) return;
    int slab, owb, ohb, ng;
    decode(u, slab, owb, ohb, ng);
    mbar_arrive_expect_tx(&full[stage], tile_bytes);
    tma_load_4d(smem + stage * T::kStageBytes, &tmX, &full[stage], slab * T::kCS, owb * tcols * SW - p.pl,
                ohb * T::kTH * SW - p.pt, ng * nb);
    ++issued;
  };
  if (tid == 0) {
#pragma unroll
    for (int j = 0; j < T::kStages - 1; ++j)
      if (static_cast<int>(blockIdx.x) + j * G < units) issue(j, blockIdx.x + j * G);
  }

  int k = 0;
  for (int u = blockIdx.x; u < units; u += G, ++k) {
    if (*abort_v) break;
    const int stage = k % T::kStages;
    if (tid == 0 && u + (T::kStages - 1) * G < units) issue(k + T::kStages - 1, u + (T::kStages - 1) * G);
    if (!mbar_wait(&full[stage], (k / T::kStages) & 1, abort_v, p.status)) break;
    waited = k + 1;
    int slab, owb, ohb, n;
    decode(u, slab, owb, ohb, n);
    n = n * nb + img;
    const int c = slab * T::kCS + cq * 4;
    const bool c_ok = c < p.C;
    if (slab != cur_slab) {
      cur_slab = slab;
      dw_load_taps(p, c, tap, bias);
    }
    const int ow = owb * tcols + col;
    const bool col_ok = c_ok && ow < p.Wo && n < p.N;
    const int oh0 = ohb * T::kTH;
    float* ybase = p.y + ((static_cast<size_t>(n) * p.Ho + oh0) * p.Wo + ow) * p.C + c;
    const size_t yrow = static_cast<size_t>(p.Wo) * p.C;
    // this thread's 4 channels of window column col*SW of its image, as 8-byte words; the
    // window is [image][row][column][32 channels], one pixel = 8 words
    const uint2* win = reinterpret_cast<const uint2*>(smem + stage * T::kStageBytes) +
                       (img * T::kInH * in_w + col * SW) * 8 + cq;

    f32x2 acc[T::kSlots][2];
#pragma unroll
    for (int q = 0; q < T::kSlots; ++q) {
      acc[q][0] = bias[0];
      acc[q][1] = bias[1];
    }
#pragma unroll
    for (int i = 0; i < T::kInH; ++i) {
      f32x2 xv[3][2];
#pragma unroll
      for (int s = 0; s < 3; ++s) {
        const uint2 v = win[(i * in_w + s) * 8];
        xv[s][0] = bf16x2_to_f32x2(v.x);
        xv[s][1] = bf16x2_to_f32x2(v.y);
      }
      // input row i feeds output row o through filter row r = i - o*SW
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        if (i - r < 0 || (i - r) % SW != 0) continue;
        const int o = (i - r) / SW;
        if (o >= T::kTH) continue;
#pragma unroll
        for (int s = 0; s < 3; ++s)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            acc[o % T::kSlots][e] = fma_f32x2(xv[s][e], tap[r * 3 + s][e], acc[o % T::kSlots][e]);
      }
      // output row o is complete after input row o*SW + 2
      if (i >= 2 && (i - 2) % SW == 0) {
        const int o = (i - 2) / SW;
        f32x2 (&a)[2] = acc[o % T::kSlots];
        if (col_ok && oh0 + o < p.Ho)
          dw_store4<EXT>(p, static_cast<size_t>(ybase - p.y) + static_cast<size_t>(o) * yrow, a[0], a[1]);
        a[0] = bias[0];
        a[1] = bias[1];
      }
    }
    // this warp is done with the stage
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(&empty[stage]);
  }
  // on a timeout, let the loads still in flight land (bounded) before the CTA's smem goes away
  if (tid == 0 && *abort_v) {
    for (int j = waited; j < issued; ++j) {
      int quiet = 0;
      mbar_wait(&full[j % T::kStages], (j / T::kStages) & 1, &quiet, nullptr, 20000000LL);
    }
  }
}

// Stride 1: tiles of 7 output rows x 32 output columns (one image, or 16 columns of two, or 8
// of four) x 32 channels, 128 threads; each thread owns two neighbouring output columns x 4
// channels, so one input row's four pixels (loaded and converted once) feed both columns' three
// taps: a third fewer shared-memory loads and conversions per output than one column per thread.
template <int TCOLS>
struct DwPairTile {
  static constexpr int kTH = 7;
  static constexpr int kLanes = 32;
  static constexpr int kCS = 32;
  static constexpr int kThreads = kLanes / 2 * kCS / 4;   // 128
  static constexpr int kInH = kTH + 2;
  static constexpr int kNb = kLanes / TCOLS;             // images per tile
  static constexpr int kInW = TCOLS + 2;
  static constexpr int kBytes = kNb * kInH * kInW * kCS * 2;
  static constexpr int kStageBytes = (kBytes + 127) / 128 * 128;
  static constexpr int kStages = 2;
  static constexpr int kSlots = 3;
  static constexpr int kSmem = kStages * kStageBytes + 128 + 2 * 8 * kStages;
};

template <int TCOLS, bool EXT>
__global__ void __launch_bounds__(128) dw3x3_pair_kernel(const __grid_constant__ CUtensorMap tmX, const DwParams p) {
  using T = DwPairTile<TCOLS>;
  extern __shared__ uint8_t dw_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dw_smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + T::kStages * T::kStageBytes);
  uint64_t* empty = full + T::kStages;
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;

  const int tid = threadIdx.x;
  const int cq = tid & 7;                  // 4-channel group within the tile's 32 channels
  const int lane = (tid >> 3) * 2;         // first of the thread's two column lanes
  const int img = lane / TCOLS;            // its image within the tile
  const int col = lane - img * TCOLS;      // and its first output column within the column block
  if (tid == 0) {
#pragma unroll
    for (int st = 0; st < T::kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], T::kThreads / 32);
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    abort_flag = 0;
  }
  __syncthreads();
  pdl_launch_dependents();
  f32x2 tap[9][2], bias[2];
  int cur_slab = static_cast<int>(blockIdx.x - fast_div(blockIdx.x, p.f_slabs) * p.f_slabs.d);
  dw_load_taps(p, cur_slab * T::kCS + cq * 4, tap, bias);
  if (tid == 0) dw_prefetch_first_window(p, &tmX, TCOLS, T::kTH, T::kNb, T::kCS);
  pdl_wait_prior();

  const int units = (p.N + T::kNb - 1) / T::kNb * p.f_ohbs.d * p.f_owbs.d * p.f_slabs.d;
  const int G = gridDim.x;
  int issued = 0, waited = 0;
  auto decode = [&](uint32_t u, int& slab, int& owb, int& ohb, int& ng) {
    const uint32_t t = fast_div(u, p.f_slabs);
    slab = static_cast<int>(u - t * p.f_slabs.d);
    const uint32_t t2 = fast_div(t, p.f_owbs);
    owb = static_cast<int>(t - t2 * p.f_owbs.d);
    ng = static_cast<int>(fast_div(t2, p.f_ohbs));
    ohb = static_cast<int>(t2 - ng * p.f_ohbs.d);
  };
  auto issue = [&](int j, int u) {
    const int stage = j % T::kStages;
    if (j >= T::kStages && !mbar_wait(&empty[stage], ((j / T::kStages) - 1) & 1, abort_v, p.status)) return;
    int slab, owb, ohb, ng;
    decode(u, slab, owb, ohb, ng);
    mbar_arrive_expect_tx(&full[stage], T::kBytes);
    tma_load_4d(smem + stage * T::kStageBytes, &tmX, &full[stage], slab * T::kCS, owb * TCOLS - p.pl,
                ohb * T::kTH - p.pt, ng * T::kNb);
    ++issued;
  };
  if (tid == 0 && static_cast<int>(blockIdx.x) < units) issue(0, blockIdx.x);

  int k = 0;
  for (int u = blockIdx.x; u < units; u += G, ++k) {
    if (*abort_v) break;
    const int stage = k % T::kStages;
    if (tid == 0 && u + G < units) issue(k + 1, u + G);
    if (!mbar_wait(&full[stage], (k / T::kStages) & 1, abort_v, p.status)) break;
    waited = k + 1;
    int slab, owb, ohb, n;
    decode(u, slab, owb, ohb, n);
    n = n * T::kNb + img;
    const int c = slab * T::kCS + cq * 4;
    if (slab != cur_slab) {
      cur_slab = slab;
      dw_load_taps(p, c, tap, bias);
    }
    const int ow = owb * TCOLS + col;
    const bool ok0 = c < p.C && n < p.N && ow < p.Wo;
    const bool ok1 = ok0 && ow + 1 < p.Wo;
    const int oh0 = ohb * T::kTH;
    const size_t ebase = ((static_cast<size_t>(n) * p.Ho + oh0) * p.Wo + ow) * p.C + c;
    const size_t yrow = static_cast<size_t>(p.Wo) * p.C;
    // this thread's 4 channels of window column col of its image, as 8-byte words; the window
    // is [image][row][column][32 channels], one pixel = 8 words
    const uint2* win = reinterpret_cast<const uint2*>(smem + stage * T::kStageBytes) +
                       (img * T::kInH * T::kInW + col) * 8 + cq;

    f32x2 acc[T::kSlots][2][2];   // [output row slot][column][channel pair]
#pragma unroll
    for (int q = 0; q < T::kSlots; ++q)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        acc[q][j][0] = bias[0];
        acc[q][j][1] = bias[1];
      }
#pragma unroll
    for (int i = 0; i < T::kInH; ++i) {
      f32x2 xv[4][2];
#pragma unroll
      for (int s2 = 0; s2 < 4; ++s2) {
        const uint2 v = win[(i * T::kInW + s2) * 8];
        xv[s2][0] = bf16x2_to_f32x2(v.x);
        xv[s2][1] = bf16x2_to_f32x2(v.y);
      }
      // input row i feeds output row o = i - r through filter row r
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        const int o = i - r;
        if (o < 0 || o >= T::kTH) continue;
#pragma unroll
        for (int s2 = 0; s2 < 3; ++s2)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            acc[o % T::kSlots][0][e] = fma_f32x2(xv[s2][e], tap[r * 3 + s2][e], acc[o % T::kSlots][0][e]);
            acc[o % T::kSlots][1][e] = fma_f32x2(xv[s2 + 1][e], tap[r * 3 + s2][e], acc[o % T::kSlots][1][e]);
          }
      }
      // output row o = i - 2 is complete
      if (i >= 2) {
        const int o = i - 2;
        f32x2 (&a)[2][2] = acc[o % T::kSlots];
        if (oh0 + o < p.Ho) {
          const size_t e0 = ebase + static_cast<size_t>(o) * yrow;
          if (ok0) dw_store4<EXT>(p, e0, a[0][0], a[0][1]);
          if (ok1) dw_store4<EXT>(p, e0 + p.C, a[1][0], a[1][1]);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          a[j][0] = bias[0];
          a[j][1] = bias[1];
        }
      }
    }
    // this warp is done with the stage
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(&empty[stage]);
  }
  // on a timeout, let the loads still in flight land (bounded) before the CTA's smem goes away
  if (tid == 0 && *abort_v) {
    for (int j = waited; j < issued; ++j) {
      int quiet = 0;
      mbar_wait(&full[j % T::kStages], (j / T::kStages) & 1, &quiet, nullptr, 20000000LL);
    }
  }
}

// Any filter size, strides and dilations: one output pixel x 8 channels per thread.
__global__ void __launch_bounds__(256) dw_generic_kernel(const DwParams p) {
  pdl_launch_dependents();
  pdl_wait_prior();
  const int C8 = p.C >> 3;
  const long long total = static_cast<long long>(p.N) * p.Ho * p.Wo * C8;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c8 = static_cast<int>(idx % C8);
    long long t = idx / C8;
    const int ow = static_cast<int>(t % p.Wo);
    t /= p.Wo;
    const int oh = static_cast<int>(t % p.Ho);
    const int n = static_cast<int>(t / p.Ho);
    const int c0 = c8 * 8;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __ldg(p.bias + c0 + e);
    for (int r = 0; r < p.R; ++r) {
      const int ih = oh * p.sh - p.pt + r * p.dh;
      if (ih < 0 || ih >= p.H) continue;
      for (int s = 0; s < p.S; ++s) {
        const int iw = ow * p.sw - p.pl + s * p.dw;
        if (iw < 0 || iw >= p.W) continue;
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
            p.x + ((static_cast<size_t>(n) * p.H + ih) * p.W + iw) * p.C + c0));
        float xv[8];
        bf16x8_to_f32(raw, xv);
        const float* tp = p.taps + (r * p.S + s) * p.C + c0;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(xv[e], __ldg(tp + e), acc[e]);
      }
    }
    const size_t e = ((static_cast<size_t>(n) * p.Ho + oh) * p.Wo + ow) * p.C + c0;
    if (!CONVF_IN_BOUNDS(e + 8 <= static_cast<size_t>(p.N) * p.Ho * p.Wo * p.C, p.status)) continue;
    if (p.res != nullptr) {
      if (p.out_bf16) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.res) + e));
        float rf[8];
        bf16x8_to_f32(r, rf);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += rf[i];
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] += __ldg(static_cast<const float*>(p.res) + e + i);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = clampf(acc[i], p.lo, p.hi);
    if (p.out_bf16) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        w[i] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.y) + e) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      float4* dst = reinterpret_cast<float4*>(p.y + e);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}

// Grouped convolution, direct: consecutive threads take consecutive output channels of one
// pixel, so the weight reads ([tap][c][k]) and the output stores are coalesced and threads of one
// group read the same input values (broadcast).
__global__ void __launch_bounds__(256) grouped_direct_kernel(const GdParams p) {
  pdl_launch_dependents();
  pdl_wait_prior();
  const long long total = static_cast<long long>(p.N) * p.Ho * p.Wo * p.K;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int k = static_cast<int>(idx % p.K);
    long long t = idx / p.K;
    const int ow = static_cast<int>(t % p.Wo);
    t /= p.Wo;
    const int oh = static_cast<int>(t % p.Ho);
    const int n = static_cast<int>(t / p.Ho);
    const int cb = (k / p.Kg) * p.Cg;
    float acc = __ldg(p.bias + k);
    for (int r = 0; r < p.R; ++r) {
      const int ih = oh * p.sh - p.pt + r * p.dh;
      if (ih < 0 || ih >= p.H) continue;
      for (int s = 0; s < p.S; ++s) {
        const int iw = ow * p.sw - p.pl + s * p.dw;
        if (iw < 0 || iw >= p.W) continue;
        const uint16_t* xp = p.x + ((static_cast<size_t>(n) * p.H + ih) * p.W + iw) * p.C + cb;
        const float* wp = p.w + static_cast<size_t>(r * p.S + s) * p.Cg * p.K + k;
        for (int c = 0; c < p.Cg; ++c)
          acc = fmaf(__uint_as_float(static_cast<uint32_t>(__ldg(xp + c)) << 16), __ldg(wp + static_cast<size_t>(c) * p.K),
                     acc);
      }
    }
    if (p.res != nullptr)
      acc += p.out_bf16 ? __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p.res)[idx]) << 16)
                        : static_cast<const float*>(p.res)[idx];
    const float v = clampf(acc, p.lo, p.hi);
    if (p.out_bf16) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      static_cast<uint16_t*>(p.y)[idx] = *reinterpret_cast<const uint16_t*>(&b);
    } else {
      static_cast<float*>(p.y)[idx] = v;
    }
  }
}

cudaError_t launch_grouped_direct(const GdParams& p, int num_sms, cudaStream_t stream) {
  const long long total = static_cast<long long>(p.N) * p.Ho * p.Wo * p.K;
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(grouped_direct_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, p);
}

bool dw_uses_tma(const DwParams& p) {
  return p.R == 3 && p.S == 3 && p.dh == 1 && p.dw == 1 && p.sh == p.sw && (p.sh == 1 || p.sh == 2);
}

void dw_tile_box(int stride, int Wo, int* box_w, int* box_h, int* box_n) {
  if (stride == 1 && dw_use_pair(Wo)) {
    const int cols = dw_pair_cols(Wo);
    *box_w = cols + 2;
    *box_h = DwPairTile<32>::kInH;
    *box_n = DwPairTile<32>::kLanes / cols;
    return;
  }
  const int cols = dw_tile_cols(Wo);
  *box_w = stride == 1 ? DwTile<1>::in_w(cols) : DwTile<2>::in_w(cols);
  *box_h = stride == 1 ? DwTile<1>::kInH : DwTile<2>::kInH;
  *box_n = DwTile<2>::kLanes / cols;
}

namespace {
template <int SW, int TCOLS, bool EXT>
cudaError_t launch_dw_tma(const DwParams& p, const CUtensorMap* tmX, int num_sms, cudaStream_t stream) {
  using T = DwTile<SW>;
  static std::once_flag once;
  static cudaError_t set_err = cudaSuccess;
  static int occ = 0;
  std::call_once(once, [] {
    set_err = cudaFuncSetAttribute(dw3x3_tma_kernel<SW, TCOLS, EXT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   T::kSmem);
    if (set_err == cudaSuccess)
      set_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dw3x3_tma_kernel<SW, TCOLS, EXT>, T::kThreads,
                                                              T::kSmem);
    if (set_err == cudaSuccess && occ < 1) set_err = cudaErrorInvalidConfiguration;
  });
  if (set_err != cudaSuccess) return set_err;
  const long long slabs = (p.C + T::kCS - 1) / T::kCS;
  constexpr int cols = TCOLS;
  constexpr int nb = T::kLanes / cols;
  const long long units = static_cast<long long>((p.N + nb - 1) / nb) * ((p.Ho + T::kTH - 1) / T::kTH) *
                          ((p.Wo + cols - 1) / cols) * slabs;
  if (units >= (1LL << 31)) return cudaErrorInvalidValue;
  DwParams q = p;
  q.f_slabs = make_fastdiv(static_cast<uint32_t>(slabs));
  q.f_owbs = make_fastdiv(static_cast<uint32_t>((p.Wo + cols - 1) / cols));
  q.f_ohbs = make_fastdiv(static_cast<uint32_t>((p.Ho + T::kTH - 1) / T::kTH));
  long long grid = std::min<long long>(units, static_cast<long long>(num_sms) * occ);
  // a multiple of the channel-slab count keeps every CTA on one slab (taps loaded once)
  if (grid < units && grid >= slabs) grid -= grid % slabs;
  return launch_pdl(dw3x3_tma_kernel<SW, TCOLS, EXT>, dim3(static_cast<unsigned>(grid)), dim3(T::kThreads), T::kSmem, stream, 1,
                    *tmX, q);
}

template <int TCOLS, bool EXT>
cudaError_t launch_dw_pair(const DwParams& p, const CUtensorMap* tmX, int num_sms, cudaStream_t stream) {
  using T = DwPairTile<TCOLS>;
  static std::once_flag once;
  static cudaError_t set_err = cudaSuccess;
  static int occ = 0;
  std::call_once(once, [] {
    set_err = cudaFuncSetAttribute(dw3x3_pair_kernel<TCOLS, EXT>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmem);
    if (set_err == cudaSuccess)
      set_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dw3x3_pair_kernel<TCOLS, EXT>, T::kThreads, T::kSmem);
    if (set_err == cudaSuccess && occ < 1) set_err = cudaErrorInvalidConfiguration;
  });
  if (set_err != cudaSuccess) return set_err;
  const long long slabs = (p.C + T::kCS - 1) / T::kCS;
  const long long units = static_cast<long long>((p.N + T::kNb - 1) / T::kNb) * ((p.Ho + T::kTH - 1) / T::kTH) *
                          ((p.Wo + TCOLS - 1) / TCOLS) * slabs;
  if (units >= (1LL << 31)) return cudaErrorInvalidValue;
  DwParams q = p;
  q.f_slabs = make_fastdiv(static_cast<uint32_t>(slabs));
  q.f_owbs = make_fastdiv(static_cast<uint32_t>((p.Wo + TCOLS - 1) / TCOLS));
  q.f_ohbs = make_fastdiv(static_cast<uint32_t>((p.Ho + T::kTH - 1) / T::kTH));
  long long grid = std::min<long long>(units, static_cast<long long>(num_sms) * occ);
  // a multiple of the channel-slab count keeps every CTA on one slab (taps loaded once)
  if (grid < units && grid >= slabs) grid -= grid % slabs;
  return launch_pdl(dw3x3_pair_kernel<TCOLS, EXT>, dim3(static_cast<unsigned>(grid)), dim3(T::kThreads), T::kSmem,
                    stream, 1, *tmX, q);
}
}  // namespace

cudaError_t launch_depthwise(const DwParams& p, const CUtensorMap* tmX, int num_sms, cudaStream_t stream) {
  const long long C8 = p.C / 8;
  if (static_cast<long long>(p.N) * p.Ho * p.Wo * C8 == 0) return cudaSuccess;
  if (dw_uses_tma(p)) {
    if (!tmX) return cudaErrorInvalidValue;
    const bool ext = p.out_bf16 || p.res != nullptr;
    if (p.sh == 1 && dw_use_pair(p.Wo)) {
      const int cols = dw_pair_cols(p.Wo);
      if (ext)
        return cols == 8 ? launch_dw_pair<8, true>(p, tmX, num_sms, stream)
               : cols == 16 ? launch_dw_pair<16, true>(p, tmX, num_sms, stream)
                            : launch_dw_pair<32, true>(p, tmX, num_sms, stream);
      return cols == 8 ? launch_dw_pair<8, false>(p, tmX, num_sms, stream)
             : cols == 16 ? launch_dw_pair<16, false>(p, tmX, num_sms, stream)
                          : launch_dw_pair<32, false>(p, tmX, num_sms, stream);
    }
    const bool narrow = dw_tile_cols(p.Wo) == 8;
    if (p.sh == 1) {
      // wide images whose width is a multiple of 16 but not of 32: 16-column tiles
      if (ext) return launch_dw_tma<1, 16, true>(p, tmX, num_sms, stream);
      return launch_dw_tma<1, 16, false>(p, tmX, num_sms, stream);
    }
    if (ext)
      return narrow ? launch_dw_tma<2, 8, true>(p, tmX, num_sms, stream)
                    : launch_dw_tma<2, 16, true>(p, tmX, num_sms, stream);
    return narrow ? launch_dw_tma<2, 8, false>(p, tmX, num_sms, stream)
                  : launch_dw_tma<2, 16, false>(p, tmX, num_sms, stream);
  }
  const dim3 b(256);
  const long long work = static_cast<long long>(p.N) * p.Ho * p.Wo * C8;
  long long blocks = (work + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 3 * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(dw_generic_kernel, dim3(static_cast<unsigned>(blocks)), b, 0, stream, 1, p);
}

}  // namespace convf
