// Window-mode tcgen05 implicit GEMM for convolutions with few input channels (a 3-channel
// stem, say), which TMA im2col cannot address (it needs 16-byte channel runs).
//
// A pre-pass writes the input with its channels padded to cpt (4 or 8) and pl zero columns in
// front, rows Wp pixels long.  In that layout the cpt*S elements one filter row of one output
// pixel reads are contiguous, and the runs of neighbouring output pixels start sw*cpt elements
// apart, so a 4-D tensor map with dims {E window elements, Wo windows, H rows, N images} and
// a window stride (sw*cpt*2 bytes) smaller than the window (E*2 bytes) presents each tile's
// A operand -- 128 windows x R filter rows, K-major, swizzled -- as ONE box.  Rows above and
// below the image and windows past Wo are TMA zero fill.  The weights ([R][bnp][E], window
// element e = s*cpt + c) stay resident in shared memory for the whole kernel.
//
// Row mode, when consecutive windows start exactly 16 bytes apart (4 channels at stride 2, or
// 8 channels at stride 1: both stems): the tile's A operand is read straight from the plain
// input row segment.  In the no-swizzle K-major layout a core matrix is 8 rows x 16 bytes and
// element (i, k) of the operand sits at (i%8)*16 + (i/8)*SBO + (k%8)*2 + (k/8)*LBO; with
// LBO = 16 and SBO = 128 that is 16*i + 2*k, i.e. window i of the contiguous row.  The TMA box
// is then R rows x nchunk 128-byte chunks (about a quarter of the window bytes, in 128-byte
// requests), and the weights are bulk-copied in the matching core-matrix order.
//
// Warp roles: 0 activation producer (one TMA load per tile), 1 TMEM allocation and MMA issue
// (R * E/16 MMAs of 128 x bnp x 16 per tile), 2 weight load, 3-10 two epilogue warpgroups that
// take alternate tiles (TMEM accumulator buffer = tile parity), each warp on its own 32 rows:
// tcgen05.ld -> per-warp smem transpose -> clamp(scale*acc + bias) -> coalesced stores.
#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {

namespace {
constexpr int kWinBM = 128;
constexpr int kWinEpiCols = 32;
constexpr int kWinWarpStage = 32 * kWinEpiCols * 4;   // one epilogue warp's 32 x 32 fp32
constexpr int kWinThreads = 96 + 256;

// Shared-memory descriptor of a K-major operand whose rows are E bf16 (32, 64 or 128 bytes)
// with the matching swizzle: 8-row atoms, SBO = 8 rows, LBO unused.
template <int E>
__device__ __forceinline__ uint64_t sdesc_kmajor_win(uint32_t saddr) {
  constexpr uint64_t layout = E == 16 ? 6 : (E == 32 ? 4 : 2);   // 32B, 64B, 128B swizzle
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>((8 * E * 2) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= layout << 61;
  return d;
}
// No-swizzle K-major descriptor with explicit leading (K) and stride (M/N) byte offsets.
__device__ __forceinline__ uint64_t sdesc_kmajor_none(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(lbo >> 4) << 16;
  d |= static_cast<uint64_t>(sbo >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}
}  // namespace

template <int E, bool ROWS>
__global__ void __launch_bounds__(kWinThreads, 1)
    tc_window_kernel(const WinParams p, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t win_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(win_smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // stages start on 1 KB boundaries (swizzled operands and the swizzled epilogue staging after
  // them depend on address bits 7-9); a row-mode box is only a multiple of 128 bytes
  const uint32_t a_stride = (p.a_stage_bytes + 1023u) & ~1023u;
  uint8_t* sA = smem;
  uint8_t* sB = sA + p.stages * a_stride;
  uint8_t* sEpi = sB + p.b_region;
  float* sScale = reinterpret_cast<float*>(sEpi + 8 * kWinWarpStage);
  float* sBias = sScale + 256;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sBias + 256);
  uint64_t* full = bars;          // [4] A stage landed
  uint64_t* empty = bars + 4;     // [4] A stage consumed by the MMAs
  uint64_t* tfull = bars + 8;     // [2] accumulator ready
  uint64_t* tempty = bars + 10;   // [2] accumulator drained
  uint64_t* bfull = bars + 12;    // weights landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tstep = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);   // one arrival per warp of the group that drains buffer b
    }
    mbar_init(bfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // scale and bias are the handle's own constant arrays (nothing earlier in the stream writes them)
  for (int i = threadIdx.x; i < p.bnp; i += blockDim.x) {
    sScale[i] = p.scale[i];
    sBias[i] = p.bias[i];
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the weights are constant too: start their load before waiting on the previous kernel
  if (warp == 2 && lane == 0) {
    mbar_arrive_expect_tx(bfull, p.b_bytes);
    if (ROWS)
      bulk_load(sB, p.w, p.b_bytes, bfull);
    else
      tma_load_3d(sB, &tmB, bfull, 0, 0, 0);
  }
  pdl_launch_dependents();
  pdl_wait_prior();

  if (warp == 0) {
    // ------------------------------------------------------------------ activation producer
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += tstep, ++it) {
        const int stage = it % p.stages;
        const uint32_t ph = (it / p.stages) & 1;
        if (!mbar_wait(&empty[stage], ph ^ 1, abort_flag, p.status)) goto teardown;
        const int owb = tile % p.ow_blocks;
        const int row = tile / p.ow_blocks;   // n * Ho + oh
        const int n = row / p.Ho;
        const int oh = row - n * p.Ho;
        mbar_arrive_expect_tx(&full[stage], p.a_stage_bytes);
        if (ROWS)
          tma_load_4d(sA + stage * a_stride, &tmA, &full[stage], 0, owb * p.chunk0_per_block,
                      oh * p.sh - p.pt, n);
        else
          tma_load_4d(sA + stage * a_stride, &tmA, &full[stage], 0, owb * kWinBM, oh * p.sh - p.pt, n);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kWinBM, p.bnp);
      if (!mbar_wait(bfull, 0, abort_flag, p.status)) goto teardown;
      int it = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += tstep, ++it) {
        const int acc = it & 1;
        if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) goto teardown;
        const int stage = it % p.stages;
        if (!mbar_wait(&full[stage], (it / p.stages) & 1, abort_flag, p.status)) goto teardown;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.bnp);
        for (int r = 0; r < p.R; ++r) {
          if (ROWS) {
            // A: window i = bytes 16 i .. of the row segment; B: core matrices 8 channels x 8
            // elements, K-adjacent ones 128 B apart, 8-channel groups E*16 B apart
            const uint32_t a0 = smem_u32(sA + stage * a_stride + r * p.nchunk * 128);
            const uint32_t b0 = smem_u32(sB + r * (p.bnp * E * 2));
#pragma unroll
            for (int k = 0; k < E / 16; ++k)
              tc_mma_bf16(d_tmem, sdesc_kmajor_none(a0 + 32 * k, 16, 128),
                          sdesc_kmajor_none(b0 + 256 * k, 128, E * 16), idesc, (r | k) != 0);
          } else {
            const uint64_t adesc =
                sdesc_kmajor_win<E>(smem_u32(sA + stage * a_stride + r * (kWinBM * E * 2)));
            const uint64_t bdesc = sdesc_kmajor_win<E>(smem_u32(sB + r * (p.bnp * E * 2)));
#pragma unroll
            for (int k = 0; k < E / 16; ++k)   // 16 bf16 (32 B) along K inside the swizzled row
              tc_mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (r | k) != 0);
          }
        }
        tc_commit(&empty[stage]);
        tc_commit(&tfull[acc]);
      }
    }
  } else if (warp >= 3) {
    // ------------------------------------------------------------------ epilogue
    // group eg (warps 3-6 / 7-10) drains the tiles this CTA computes into accumulator buffer eg
    // (odd/even tiles).  Each warp owns TMEM lanes 32q..32q+31 = tile rows = 32 output pixels
    // and works alone: tcgen05.ld of 32 columns (thread = row) -> its own 4 KB of smem ->
    // read back as thread = (row, 4 channels), scale/bias/clamp, coalesced 16-byte stores that
    // cover four whole 128-byte row segments per instruction.
    const int eg = (warp - 3) >> 2;
    const int q = warp & 3;                // TMEM lane quadrant this warp may access
    float* wst = reinterpret_cast<float*>(sEpi + (warp - 3) * kWinWarpStage);
    const int sub = lane >> 3;             // row within each group of four in the store phase
    const int c4 = lane & 7;               // 4-channel column group
    const int nchunks = p.bnp / kWinEpiCols;
    int n_it = 0;
    for (int tile = blockIdx.x + eg * tstep; tile < p.num_tiles; tile += 2 * tstep, ++n_it) {
      if (!mbar_wait(&tfull[eg], n_it & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const int owb = tile % p.ow_blocks;
      const int orow = tile / p.ow_blocks;   // n * Ho + oh
      const int ow0 = owb * kWinBM + q * 32;
      float* yw = p.y + (static_cast<size_t>(orow) * p.Wo + ow0) * p.Kout;
      // two 32-column chunks per TMEM read round, so the buffer is released as early as possible
      for (int ch = 0; ch < nchunks; ch += 2) {
        const bool two = ch + 1 < nchunks;
        uint32_t v[2][32];
        const uint32_t tcol = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(eg * p.bnp + ch * kWinEpiCols);
        tmem_ld_32x32b_x32(tcol, v[0]);
        if (two) tmem_ld_32x32b_x32(tcol + kWinEpiCols, v[1]);
        tmem_ld_wait();
        if (ch + 2 >= nchunks) {
          // the warp's last TMEM read of the tile (tcgen05.ld is warp-collective)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[eg]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !two) break;
          const int nc = (ch + h) * kWinEpiCols;
          // row `lane` -> smem, 16-byte chunks XOR-swizzled by row: both phases conflict-free
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(wst + lane * 32 + ((c ^ (lane & 7)) << 2)) =
                make_float4(__uint_as_float(v[h][4 * c]), __uint_as_float(v[h][4 * c + 1]),
                            __uint_as_float(v[h][4 * c + 2]), __uint_as_float(v[h][4 * c + 3]));
          __syncwarp();
          const bool col_ok = nc + 4 * c4 < p.Kout;
          const float4 sc = *reinterpret_cast<const float4*>(sScale + nc + 4 * c4);
          const float4 bi = *reinterpret_cast<const float4*>(sBias + nc + 4 * c4);
          // rows read back four at a time ahead of their math, so the shared-memory loads issue
          // back to back (four, not eight: this kernel has fewer registers to spare)
#pragma unroll
          for (int i0 = 0; i0 < 8; i0 += 4) {
            float4 a[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = 4 * (i0 + i) + sub;
              a[i] = *reinterpret_cast<const float4*>(wst + r * 32 + ((c4 ^ (r & 7)) << 2));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = 4 * (i0 + i) + sub;
              if (col_ok && ow0 + r < p.Wo &&
                  CONVF_IN_BOUNDS((static_cast<size_t>(orow) * p.Wo + ow0 + r) * p.Kout + nc + 4 * c4 + 4 <=
                                      static_cast<size_t>(p.num_tiles / p.ow_blocks) * p.Wo * p.Kout,
                                  p.status))
                *reinterpret_cast<float4*>(yw + static_cast<size_t>(r) * p.Kout + nc + 4 * c4) =
                    make_float4(fminf(fmaxf(fmaf(a[i].x, sc.x, bi.x), p.lo), p.hi),
                                fminf(fmaxf(fmaf(a[i].y, sc.y, bi.y), p.lo), p.hi),
                                fminf(fmaxf(fmaf(a[i].z, sc.z, bi.z), p.lo), p.hi),
                                fminf(fmaxf(fmaf(a[i].w, sc.w, bi.w), p.lo), p.hi));
            }
          }
          __syncwarp();
        }
      }
    }
  }

teardown:
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // a wait ran out: give copies and MMAs already in flight time to land before TMEM is freed
    for (int i = 0; i < 2000; ++i) __nanosleep(100000);
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

cudaError_t launch_tc_window(const WinParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int E, bool rows,
                             int grid, size_t smem, cudaStream_t stream) {
  void (*k)(WinParams, CUtensorMap, CUtensorMap) = nullptr;
  if (E == 16) k = rows ? tc_window_kernel<16, true> : tc_window_kernel<16, false>;
  else if (E == 32) k = rows ? tc_window_kernel<32, true> : tc_window_kernel<32, false>;
  else if (E == 64) k = rows ? tc_window_kernel<64, true> : tc_window_kernel<64, false>;
  else return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(kWinThreads), smem, stream, 1, p, tmA, tmB);
}

// ------------------------------------------------------------------ pre-pass
// grid.y walks groups of four image rows (n, h), grid.x x threads the Wp padded columns: the
// four rows' loads are issued together, and no thread divides
__global__ void __launch_bounds__(256) window_pad_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ out,
                                                         long long rows, int W, int C, int cpt, int Wp, int shift) {
  pdl_launch_dependents();
  pdl_wait_prior();
  constexpr int kRows = 4;
  for (long long row0 = static_cast<long long>(blockIdx.y) * kRows; row0 < rows;
       row0 += static_cast<long long>(gridDim.y) * kRows) {
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < Wp; j += gridDim.x * blockDim.x) {
      const int col = j - shift;
      const bool in = col >= 0 && col < W;
      uint32_t v[kRows][8];
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        const bool ok = in && row0 + i < rows;
        const uint16_t* xr = x + ((row0 + i) * W + col) * C;
#pragma unroll
        for (int c = 0; c < 8; ++c) v[i][c] = (ok && c < C) ? xr[c] : 0u;
      }
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        if (row0 + i >= rows) break;
        uint16_t* o = out + ((row0 + i) * Wp + j) * cpt;
        if (cpt == 4)
          *reinterpret_cast<uint2*>(o) = make_uint2(v[i][0] | (v[i][1] << 16), v[i][2] | (v[i][3] << 16));
        else
          *reinterpret_cast<uint4*>(o) = make_uint4(v[i][0] | (v[i][1] << 16), v[i][2] | (v[i][3] << 16),
                                                    v[i][4] | (v[i][5] << 16), v[i][6] | (v[i][7] << 16));
      }
    }
  }
}

cudaError_t launch_window_pad(const uint16_t* x, uint16_t* out, int N, int H, int W, int C, int cpt, int Wp,
                              int shift, int num_sms, cudaStream_t stream) {
  (void)num_sms;
  const long long rows = static_cast<long long>(N) * H;
  if (rows == 0) return cudaSuccess;
  const long long groups = (rows + 3) / 4;
  const dim3 grid(static_cast<unsigned>((Wp + 255) / 256), static_cast<unsigned>(groups < 65535 ? groups : 65535));
  return launch_pdl(window_pad_kernel, grid, dim3(256), 0, stream, 1, x, out, rows, W, C, cpt, Wp, shift);
}

}  // namespace convf
