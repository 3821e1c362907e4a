// Channel padding for the gathered-row implicit GEMM: NHWC bf16 with C channels (C <= 8) ->
// NHWC bf16 with cpt channels (4 or 8), the extra channels zero, so that each filter tap of a
// pixel is one aligned 8- or 16-byte vector.  One thread per pixel; reads and writes are
// consecutive across the warp.
#include <cuda_bf16.h>

#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {

__global__ void __launch_bounds__(256) pad_channels_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ out,
                                                           long long pixels, int C, int cpt) {
  pdl_launch_dependents();
  pdl_wait_prior();
  for (long long px = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; px < pixels;
       px += static_cast<long long>(gridDim.x) * blockDim.x) {
    uint32_t v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = c < C ? x[px * C + c] : 0u;
    if (cpt == 4)
      *reinterpret_cast<uint2*>(out + px * 4) = make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
    else
      *reinterpret_cast<uint4*>(out + px * 8) =
          make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
  }
}

cudaError_t launch_pad_channels(const uint16_t* x, uint16_t* out, long long pixels, int C, int cpt, int num_sms,
                                cudaStream_t stream) {
  if (pixels == 0) return cudaSuccess;
  long long blocks = (pixels + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(pad_channels_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, x, out, pixels,
                    C, cpt);
}

// 8-bit activations for the integer-exact tcgen05 path: each byte b (int8 or uint8) becomes the
// bf16 bits of b - zp, an integer of magnitude at most 255 and therefore exact in bf16 (8
// significant bits).  Zero-filled padding taps then stand for the zero point, as ONNX's
// quantized convolutions pad.  16 bytes in, 32 bytes out per thread and step.
__device__ __forceinline__ uint32_t q8pair_to_bf16x2(uint32_t b0, uint32_t b1, int is_signed, int zp) {
  const int v0 = (is_signed ? static_cast<int>(static_cast<int8_t>(b0)) : static_cast<int>(b0)) - zp;
  const int v1 = (is_signed ? static_cast<int>(static_cast<int8_t>(b1)) : static_cast<int>(b1)) - zp;
  const __nv_bfloat162 h = __floats2bfloat162_rn(static_cast<float>(v0), static_cast<float>(v1));
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(256) q8_to_bf16_kernel(const uint8_t* __restrict__ x, uint16_t* __restrict__ out,
                                                         long long n, int is_signed, int zp) {
  pdl_launch_dependents();
  pdl_wait_prior();
  const long long groups = n >> 3;   // 8 elements per group (n % 8 == 0)
  for (long long g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 2; g < groups;
       g += static_cast<long long>(gridDim.x) * blockDim.x * 2) {
    if (g + 1 < groups) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + g * 8));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        o[2 * i] = q8pair_to_bf16x2(w[i] & 0xff, (w[i] >> 8) & 0xff, is_signed, zp);
        o[2 * i + 1] = q8pair_to_bf16x2((w[i] >> 16) & 0xff, w[i] >> 24, is_signed, zp);
      }
      *reinterpret_cast<uint4*>(out + g * 8) = make_uint4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<uint4*>(out + g * 8 + 8) = make_uint4(o[4], o[5], o[6], o[7]);
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(x + g * 8));
      const uint32_t w[2] = {v.x, v.y};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        o[2 * i] = q8pair_to_bf16x2(w[i] & 0xff, (w[i] >> 8) & 0xff, is_signed, zp);
        o[2 * i + 1] = q8pair_to_bf16x2((w[i] >> 16) & 0xff, w[i] >> 24, is_signed, zp);
      }
      *reinterpret_cast<uint4*>(out + g * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// Pre-activation prologue: u = clamp(scale[c] * x + shift[c], lo, hi) per channel, rounded to
// bf16 (nearest even), into the handle's staging copy that the conv kernels then read; the
// conv's zero padding is therefore applied to u.  8 channels (16 bytes) per thread when
// C % 8 == 0, else one element per thread.
__global__ void __launch_bounds__(256) preact_bf16_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ out,
                                                          long long n, int C, const float* __restrict__ scale,
                                                          const float* __restrict__ shift, float lo, float hi) {
  pdl_launch_dependents();
  pdl_wait_prior();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  if ((C & 7) == 0) {
    for (long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; g < n / 8; g += stride) {
      const int c0 = static_cast<int>((g * 8) % C);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + g * 8));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = fminf(fmaxf(fmaf(__uint_as_float(w[i] << 16), __ldg(scale + c0 + 2 * i), __ldg(shift + c0 + 2 * i)), lo), hi);
        const float b = fminf(fmaxf(fmaf(__uint_as_float(w[i] & 0xffff0000u), __ldg(scale + c0 + 2 * i + 1),
                                         __ldg(shift + c0 + 2 * i + 1)), lo), hi);
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        o[i] = *reinterpret_cast<const uint32_t*>(&h);
      }
      *reinterpret_cast<uint4*>(out + g * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  } else {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
      const int c = static_cast<int>(i % C);
      const float a = fminf(fmaxf(fmaf(__uint_as_float(static_cast<uint32_t>(x[i]) << 16), __ldg(scale + c), __ldg(shift + c)), lo), hi);
      const __nv_bfloat16 h = __float2bfloat16_rn(a);
      out[i] = *reinterpret_cast<const uint16_t*>(&h);
    }
  }
}

cudaError_t launch_preact_bf16(const uint16_t* x, uint16_t* out, long long n, int C, const float* scale,
                               const float* shift, float lo, float hi, int num_sms, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const long long work = (C & 7) == 0 ? n / 8 : n;
  long long blocks = (work + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(preact_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, x, out, n, C,
                    scale, shift, lo, hi);
}

cudaError_t launch_q8_to_bf16(const uint8_t* x, uint16_t* out, long long n, int is_signed, int zp, int num_sms,
                              cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const long long pairs = (n / 8 + 1) / 2;
  long long blocks = (pairs + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  return launch_pdl(q8_to_bf16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, 1, x, out, n,
                    is_signed, zp);
}

}  // namespace convf
