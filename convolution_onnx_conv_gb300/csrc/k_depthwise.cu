// Depthwise convolution (group == C == K) on CUDA cores: memory-bound (about 2-3 flop per
// byte), so no tensor cores.  NHWC bf16 in, fp32 taps with the BN scale folded in, fp32 out.
// Each thread owns 8 channels (one 16-byte vector) x kOW = 2 consecutive outputs of a column
// strip; consecutive threads take consecutive channel vectors of the same pixel, so every load
// and store is a coalesced 128-bit access.  Inputs shared by neighbouring columns are re-read
// through L1/L2, not from HBM; inputs shared by neighbouring rows stay in registers.
#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {

constexpr int kOW = 2;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float clampf(float v, float lo, float hi) { return fminf(fmaxf(v, lo), hi); }

// 3x3, dilation 1, equal strides SW in {1, 2}.  Each thread owns 8 channels x kOW outputs of a
// column and walks down p.th output rows, keeping the 3 input rows it needs in registers: per
// new output row it loads only the SW new input rows (NCOL 16-byte vectors each), all issued
// before the arithmetic.  Padding reads as zero without a branch.  The strip height p.th is
// chosen by the host so that enough threads run to keep the memory system busy.
template <int SW>
__global__ void __launch_bounds__(256, 2) dw3x3_kernel(const DwParams p) {
  pdl_launch_dependents();
  pdl_wait_prior();
  // grid.y walks (image, strip of kTH output rows); grid.x x 256 threads cover (output column
  // block, channel vector) of a row, with 32-bit index arithmetic
  const int C8 = p.C >> 3;
  const int owb_n = (p.Wo + kOW - 1) / kOW;
  const int row_items = owb_n * C8;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= row_items) return;
  const int c8 = j % C8;
  const int owb = j / C8;
  const int c0 = c8 * 8;
  const int ow0 = owb * kOW;
  const int iw_base = ow0 * SW - p.pl;
  constexpr int NCOL = (kOW - 1) * SW + 3;
  const int strips = (p.Ho + p.th - 1) / p.th;

  float bias[8];
  {
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(p.bias + c0));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(p.bias + c0 + 4));
    bias[0] = b0.x; bias[1] = b0.y; bias[2] = b0.z; bias[3] = b0.w;
    bias[4] = b1.x; bias[5] = b1.y; bias[6] = b1.z; bias[7] = b1.w;
  }

  for (int ns = blockIdx.y; ns < p.N * strips; ns += gridDim.y) {
    const int n = ns / strips;
    const int oh_begin = (ns - n * strips) * p.th;
    const int oh_end = min(oh_begin + p.th, p.Ho);
    const uint16_t* ximg = p.x + static_cast<size_t>(n) * p.H * p.W * p.C + c0;
    auto load_row = [&](int ih, uint4 (&dst)[NCOL]) {
      const bool row_ok = ih >= 0 && ih < p.H;
      const uint16_t* xrow = ximg + static_cast<size_t>(row_ok ? ih : 0) * p.W * p.C;
#pragma unroll
      for (int col = 0; col < NCOL; ++col) {
        const int iw = iw_base + col;
        dst[col] = (row_ok && iw >= 0 && iw < p.W)
                       ? __ldg(reinterpret_cast<const uint4*>(xrow + static_cast<size_t>(iw) * p.C))
                       : make_uint4(0, 0, 0, 0);
      }
    };
    // window rows: win[0..2] = input rows oh*SW - pt + 0..2
    uint4 win[3][NCOL];
    const int ih0 = oh_begin * SW - p.pt;
    if (SW == 1) {
      load_row(ih0, win[0]);
      load_row(ih0 + 1, win[1]);
    } else {
      load_row(ih0, win[0]);
    }
    for (int oh = oh_begin; oh < oh_end; ++oh) {
      const int ihb = oh * SW - p.pt;
      if (SW == 1) {
        load_row(ihb + 2, win[2]);
      } else {
        load_row(ihb + 1, win[1]);
        load_row(ihb + 2, win[2]);
      }
      float acc[kOW][8];
#pragma unroll
      for (int jj = 0; jj < kOW; ++jj)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[jj][e] = bias[e];
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        float tap[3][8];
#pragma unroll
        for (int s = 0; s < 3; ++s) {
          const float4 t0 = __ldg(reinterpret_cast<const float4*>(p.taps + (r * 3 + s) * p.C + c0));
          const float4 t1 = __ldg(reinterpret_cast<const float4*>(p.taps + (r * 3 + s) * p.C + c0 + 4));
          tap[s][0] = t0.x; tap[s][1] = t0.y; tap[s][2] = t0.z; tap[s][3] = t0.w;
          tap[s][4] = t1.x; tap[s][5] = t1.y; tap[s][6] = t1.z; tap[s][7] = t1.w;
        }
#pragma unroll
        for (int col = 0; col < NCOL; ++col) {
          float xv[8];
          bf16x8_to_f32(win[r][col], xv);
#pragma unroll
          for (int jj = 0; jj < kOW; ++jj) {
            const int s = col - jj * SW;
            if (s >= 0 && s < 3) {
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[jj][e] = fmaf(xv[e], tap[s][e], acc[jj][e]);
            }
          }
        }
      }
      float* yrow = p.y + ((static_cast<size_t>(n) * p.Ho + oh) * p.Wo) * p.C + c0;
#pragma unroll
      for (int jj = 0; jj < kOW; ++jj) {
        if (ow0 + jj < p.Wo) {
          float4* dst = reinterpret_cast<float4*>(yrow + static_cast<size_t>(ow0 + jj) * p.C);
          dst[0] = make_float4(clampf(acc[jj][0], p.lo, p.hi), clampf(acc[jj][1], p.lo, p.hi),
                               clampf(acc[jj][2], p.lo, p.hi), clampf(acc[jj][3], p.lo, p.hi));
          dst[1] = make_float4(clampf(acc[jj][4], p.lo, p.hi), clampf(acc[jj][5], p.lo, p.hi),
                               clampf(acc[jj][6], p.lo, p.hi), clampf(acc[jj][7], p.lo, p.hi));
        }
      }
      // slide the window down by SW input rows
#pragma unroll
      for (int col = 0; col < NCOL; ++col) {
        if (SW == 1) {
          win[0][col] = win[1][col];
          win[1][col] = win[2][col];
        } else {
          win[0][col] = win[2][col];
        }
      }
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
    float4* dst = reinterpret_cast<float4*>(p.y + ((static_cast<size_t>(n) * p.Ho + oh) * p.Wo + ow) * p.C + c0);
    dst[0] = make_float4(clampf(acc[0], p.lo, p.hi), clampf(acc[1], p.lo, p.hi),
                         clampf(acc[2], p.lo, p.hi), clampf(acc[3], p.lo, p.hi));
    dst[1] = make_float4(clampf(acc[4], p.lo, p.hi), clampf(acc[5], p.lo, p.hi),
                         clampf(acc[6], p.lo, p.hi), clampf(acc[7], p.lo, p.hi));
  }
}

cudaError_t launch_depthwise(const DwParams& p, int num_sms, cudaStream_t stream) {
  const bool fast = p.R == 3 && p.S == 3 && p.dh == 1 && p.dw == 1 && p.sh == p.sw &&
                    (p.sh == 1 || p.sh == 2);
  const long long C8 = p.C / 8;
  if (static_cast<long long>(p.N) * p.Ho * p.Wo * C8 == 0) return cudaSuccess;
  const dim3 b(256);
  if (fast) {
    const long long row_items = ((p.Wo + kOW - 1) / kOW) * C8;
    // tallest strip (fewest redundant row loads) that still leaves >= 1024 threads per SM
    DwParams q = p;
    q.th = 1;
    for (int th : {8, 4, 2}) {
      const long long threads = static_cast<long long>(p.N) * ((p.Ho + th - 1) / th) * row_items;
      if (threads >= static_cast<long long>(num_sms) * 1024) {
        q.th = th;
        break;
      }
    }
    const long long strips = static_cast<long long>(p.N) * ((p.Ho + q.th - 1) / q.th);
    const dim3 g(static_cast<unsigned>((row_items + 255) / 256), static_cast<unsigned>(strips < 65535 ? strips : 65535));
    return p.sh == 1 ? launch_pdl(dw3x3_kernel<1>, g, b, 0, stream, 1, q)
                     : launch_pdl(dw3x3_kernel<2>, g, b, 0, stream, 1, q);
  }
  const long long work = static_cast<long long>(p.N) * p.Ho * p.Wo * C8;
  long long blocks = (work + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 3 * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(dw_generic_kernel, dim3(static_cast<unsigned>(blocks)), b, 0, stream, 1, p);
}

}  // namespace convf
