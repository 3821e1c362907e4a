// Channel padding for the gathered-row implicit GEMM: NHWC bf16 with C channels (C <= 8) ->
// NHWC bf16 with cpt channels (4 or 8), the extra channels zero, so that each filter tap of a
// pixel is one aligned 8- or 16-byte vector.  One thread per pixel; reads and writes are
// consecutive across the warp.
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

}  // namespace convf
