// Static-int8 implicit-GEMM convolution: int8 x int8 -> int32 on the tensor cores with the
// warp-level m16n8k32 MMA (sm_103a has no int8 kind for tcgen05.mma), a 4-stage cp.async
// pipeline that gathers the activation rows (zero-fill for padding taps), and a fused
// epilogue: + int32 bias, per-channel fixed-point requantisation
// q = (v*M + 2^(sh-1)) >> sh in int64, + output zero point, clamp (ReLU at the zero point),
// int8 store staged through shared memory for 16-byte coalesced writes.
// Tile: 128 (rows m = n,oh,ow) x 128 (output channels) x 64 (channels of one filter tap).
#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {

constexpr int kS8BM = 128, kS8BN = 128, kS8BK = 64, kS8Stages = 4;
constexpr int kS8TileBytes = kS8BM * kS8BK;           // 8 KB (A and B tiles alike)
constexpr int kS8Smem = kS8Stages * 2 * kS8TileBytes;  // 64 KB

// Row `row`, 16-byte chunk `ch` (0..3) of a 64-byte-row tile; XOR swizzle keeps the 8 rows an
// ldmatrix reads on distinct banks.
__device__ __forceinline__ uint32_t s8_off(int row, int ch) {
  return static_cast<uint32_t>(row * 64 + ((ch ^ ((row >> 1) & 3)) << 4));
}

__global__ void __launch_bounds__(256, 1) s8_conv_kernel(const S8Params p) {
  extern __shared__ __align__(128) uint8_t s8_smem[];
  uint8_t* sA = s8_smem;
  uint8_t* sB = s8_smem + kS8Stages * kS8TileBytes;

  pdl_launch_dependents();
  pdl_wait_prior();
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 2;   // 0..1 : 64-row slab
  const int wn = warp & 3;    // 0..3 : 32-column slab
  const int m0 = blockIdx.x * kS8BM;
  const int n0 = blockIdx.y * kS8BN;

  // each thread copies two 16-byte chunks of one A row and of one B row per stage
  const int ld_row = tid >> 1;
  const int ld_ch = (tid & 1) * 2;
  const int m = m0 + ld_row;
  const bool m_ok = m < p.M;
  const int hw = p.Ho * p.Wo;
  const int img = m_ok ? m / hw : 0;
  const int rem = m - img * hw;
  const int oh = rem / p.Wo, ow = rem - (rem / p.Wo) * p.Wo;
  const int ih0 = oh * p.sh - p.pt, iw0 = ow * p.sw - p.pl;
  const int8_t* ximg = p.x + static_cast<size_t>(img) * p.H * p.W * p.C;
  const int nrow = n0 + ld_row;
  const bool n_ok = nrow < p.Kout;
  const size_t ktot = static_cast<size_t>(p.R) * p.S * p.C;
  const int8_t* wrow = p.w + static_cast<size_t>(n_ok ? nrow : 0) * ktot;
  const int cblocks = p.C / kS8BK;

  auto load_stage = [&](int kb, int stage) {
    const int tap = kb / cblocks;
    const int cb = kb - tap * cblocks;
    const int r = tap / p.S, s = tap - (tap / p.S) * p.S;
    const int ih = ih0 + r * p.dh, iw = iw0 + s * p.dw;
    const bool ok = m_ok && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W;
    const int8_t* src = ok ? ximg + (static_cast<size_t>(ih) * p.W + iw) * p.C + cb * kS8BK : p.x;
    uint8_t* dA = sA + stage * kS8TileBytes;
    uint8_t* dB = sB + stage * kS8TileBytes;
    const int8_t* wsrc = wrow + static_cast<size_t>(kb) * kS8BK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      cp_async_16(dA + s8_off(ld_row, ld_ch + i), ok ? src + (ld_ch + i) * 16 : p.x, ok ? 16u : 0u);
      cp_async_16(dB + s8_off(ld_row, ld_ch + i), n_ok ? wsrc + (ld_ch + i) * 16 : p.w,
                  n_ok ? 16u : 0u);
    }
  };

  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][j][e] = 0;

#pragma unroll
  for (int s = 0; s < kS8Stages - 1; ++s) {
    if (s < p.num_kb) load_stage(s, s);
    cp_async_commit();
  }

  // ldmatrix lane addressing: matrix index = lane / 8, row within matrix = lane % 8
  const int lm_mat = lane >> 3, lm_row = lane & 7;
  for (int kb = 0; kb < p.num_kb; ++kb) {
    cp_async_wait<kS8Stages - 2>();
    __syncthreads();
    const int stage = kb % kS8Stages;
    const uint32_t aBase = smem_u32(sA + stage * kS8TileBytes);
    const uint32_t bBase = smem_u32(sB + stage * kS8TileBytes);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {   // two k32 steps per 64-byte block
      uint32_t af[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // matrices: (rows 0-7, k 0-15), (rows 8-15, k 0-15), (rows 0-7, k 16-31), (rows 8-15, k 16-31)
        const int row = wm * 64 + i * 16 + (lm_mat & 1) * 8 + lm_row;
        const int ch = ks * 2 + (lm_mat >> 1);
        ldmatrix_x4(aBase + s8_off(row, ch), af[i][0], af[i][1], af[i][2], af[i][3]);
      }
      uint32_t bf[4][2];
#pragma unroll
      for (int j2 = 0; j2 < 2; ++j2) {
        // matrices: (n 0-7, k 0-15), (n 0-7, k 16-31), (n 8-15, k 0-15), (n 8-15, k 16-31)
        const int row = wn * 32 + j2 * 16 + (lm_mat >> 1) * 8 + lm_row;
        const int ch = ks * 2 + (lm_mat & 1);
        ldmatrix_x4(bBase + s8_off(row, ch), bf[2 * j2][0], bf[2 * j2][1], bf[2 * j2 + 1][0],
                    bf[2 * j2 + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_s8_16832(acc[i][j], af[i], bf[j][0], bf[j][1]);
    }
    const int next = kb + kS8Stages - 1;
    if (next < p.num_kb) load_stage(next, next % kS8Stages);
    cp_async_commit();
  }
  cp_async_wait<0>();
  __syncthreads();

  // epilogue: requantise into a 128 x 128 int8 tile in shared memory, then coalesced stores
  int8_t* sOut = reinterpret_cast<int8_t*>(s8_smem);
  const int g = lane >> 2, tg = lane & 3;
  const int lo = p.relu ? (p.zp > -128 ? p.zp : -128) : -128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int col = wn * 32 + j * 8 + tg * 2;
    int64_t bias2[2], mult2[2];
    int sh2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = n0 + col + e;
      const bool ok = n < p.Kout;
      bias2[e] = ok ? __ldg(p.bias + n) : 0;
      mult2[e] = ok ? __ldg(p.mult + n) : 1;
      sh2[e] = ok ? __ldg(p.shift + n) : 1;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int hv = 0; hv < 2; ++hv) {
        const int row = wm * 64 + i * 16 + g + hv * 8;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int64_t v = static_cast<int64_t>(acc[i][j][hv * 2 + e]) + bias2[e];
          int64_t q = (v * mult2[e] + (static_cast<int64_t>(1) << (sh2[e] - 1))) >> sh2[e];
          q += p.zp;
          q = q < lo ? lo : (q > 127 ? 127 : q);
          sOut[row * kS8BN + col + e] = static_cast<int8_t>(q);
        }
      }
    }
  }
  __syncthreads();
  // 128 rows x 8 chunks of 16 bytes
  for (int idx = tid; idx < kS8BM * (kS8BN / 16); idx += 256) {
    const int row = idx >> 3, ch = idx & 7;
    const int mm = m0 + row, nn = n0 + ch * 16;
    if (mm < p.M && nn < p.Kout &&
        CONVF_IN_BOUNDS(static_cast<size_t>(mm) * p.Kout + nn + 16 <= static_cast<size_t>(p.M) * p.Kout, p.status))
      *reinterpret_cast<uint4*>(p.y + static_cast<size_t>(mm) * p.Kout + nn) =
          *reinterpret_cast<const uint4*>(sOut + row * kS8BN + ch * 16);
  }
}

// Rate of the int8 warp-level MMA on this GPU: every warp issues back-to-back m16n8k32 MMAs on
// register operands into 8 independent accumulators (no memory traffic), the roofline
// denominator of the int8 path.
__global__ void __launch_bounds__(256) s8_mma_rate_kernel(int iters, int* sink) {
  int acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0;
  const uint32_t t = threadIdx.x;
  const uint32_t a[4] = {t * 0x01010101u, t * 0x02030405u, t ^ 0x7F7F7F7Fu, t + 0x11111111u};
  const uint32_t b0 = t * 0x03050709u, b1 = t ^ 0x55AA55AAu;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) mma_s8_16832(acc[j], a, b0, b1);
  }
  int sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) sum += acc[j][e];
  if (sum == 0x7FFFFFFF) sink[0] = sum;   // keeps the MMAs live
}

cudaError_t measure_s8_mma_rate(int num_sms, cudaStream_t stream, double* tops) {
  int* sink = nullptr;
  cudaError_t e = cudaSuccess;
  const int iters = 4096, blocks = num_sms * 4;
  cudaEvent_t e0, e1;
  if ((e = cudaEventCreate(&e0)) != cudaSuccess) return e;
  if ((e = cudaEventCreate(&e1)) != cudaSuccess) return e;
  s8_mma_rate_kernel<<<blocks, 256, 0, stream>>>(64, sink);   // warm-up
  cudaEventRecord(e0, stream);
  s8_mma_rate_kernel<<<blocks, 256, 0, stream>>>(iters, sink);
  cudaEventRecord(e1, stream);
  e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return e;
  const double ops = 2.0 * 16 * 8 * 32 * 8.0 * iters * (blocks * 8.0);
  *tops = ops / (ms * 1e-3) / 1e12;
  return cudaGetLastError();
}

cudaError_t launch_s8_conv(const S8Params& p, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(s8_conv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kS8Smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (p.M == 0) return cudaSuccess;
  dim3 grid((p.M + kS8BM - 1) / kS8BM, (p.Kout + kS8BN - 1) / kS8BN);
  return launch_pdl(s8_conv_kernel, grid, dim3(256), kS8Smem, stream, 1, p);
}

}  // namespace convf
