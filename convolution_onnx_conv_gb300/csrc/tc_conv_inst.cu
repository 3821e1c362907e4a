// One tile width of the tcgen05 implicit-GEMM kernel per translation unit (compiled with
// -DCONVF_BN=32/64/128/256) so the instantiations build in parallel.
#include "tc_conv.cuh"

#ifndef CONVF_BN
#error "compile with -DCONVF_BN=<tile width>"
#endif
#define CONVF_CAT2(a, b) a##b
#define CONVF_CAT(a, b) CONVF_CAT2(a, b)

namespace convf {
cudaError_t CONVF_CAT(launch_tc_conv_bn, CONVF_BN)(const TcConvParams& p, const CUtensorMap& tmA,
                                                   const CUtensorMap& tmB, const CUtensorMap* tmR, int grid,
                                                   bool gather, bool pair, cudaStream_t stream) {
  const CUtensorMap& tmR_ = tmR ? *tmR : tmB;   // unused unless the residual is staged
  if (p.y8 != nullptr) {
    // integer-exact 8-bit convolution: single CTAs, whole tiles, 64- or 128-wide tiles
    if (gather || pair || p.sk) return cudaErrorInvalidValue;
#if CONVF_BN == 64 || CONVF_BN == 128
    return launch_tc_conv_t<CONVF_BN, false, false, false, 0, true>(p, tmA, tmB, tmR_, grid, stream);
#else
    return cudaErrorInvalidValue;
#endif
  }
  if (p.res != nullptr || p.out_bf16) {
    // residual and/or bf16 output: the extended-epilogue instantiations
    if (gather) return cudaErrorInvalidValue;
    if (p.res != nullptr && p.out_bf16 && (p.Kout & 7) == 0 && !p.sk) {
      // residual with bf16 output on 16-byte rows (staged in shared memory by TMA when the
      // caller encoded its map: single CTAs, 64- or 128-wide tiles)
      if (pair) return launch_tc_conv_t<CONVF_BN, false, true, false, 3>(p, tmA, tmB, tmR_, grid, stream);
#if CONVF_BN == 64 || CONVF_BN == 128
      if (tmR) return launch_tc_conv_t<CONVF_BN, false, false, false, 4>(p, tmA, tmB, tmR_, grid, stream);
#endif
      return launch_tc_conv_t<CONVF_BN, false, false, false, 3>(p, tmA, tmB, tmR_, grid, stream);
    }
    if (p.res != nullptr) {
      if (p.sk) return launch_tc_conv_t<CONVF_BN, false, false, true, 1>(p, tmA, tmB, tmR_, grid, stream);
      if (pair) return launch_tc_conv_t<CONVF_BN, false, true, false, 1>(p, tmA, tmB, tmR_, grid, stream);
      return launch_tc_conv_t<CONVF_BN, false, false, false, 1>(p, tmA, tmB, tmR_, grid, stream);
    }
    // bf16 output without a residual
    if (p.sk) return launch_tc_conv_t<CONVF_BN, false, false, true, 2>(p, tmA, tmB, tmR_, grid, stream);
    if (pair) return launch_tc_conv_t<CONVF_BN, false, true, false, 2>(p, tmA, tmB, tmR_, grid, stream);
    return launch_tc_conv_t<CONVF_BN, false, false, false, 2>(p, tmA, tmB, tmR_, grid, stream);
  }
  if (p.sk) {
    // stream-K: single CTAs with TMA activation loads only
    if (gather || pair) return cudaErrorInvalidValue;
    return launch_tc_conv_t<CONVF_BN, false, false, true>(p, tmA, tmB, tmR_, grid, stream);
  }
  if (pair) {
    if (gather) return cudaErrorInvalidValue;
    return launch_tc_conv_t<CONVF_BN, false, true>(p, tmA, tmB, tmR_, grid, stream);
  }
#if CONVF_BN == 256
  // gather mode needs room for the input-row patch: tile widths up to 128 only
  if (gather) return cudaErrorInvalidValue;
  return launch_tc_conv_t<CONVF_BN, false, false>(p, tmA, tmB, tmR_, grid, stream);
#else
  return gather ? launch_tc_conv_t<CONVF_BN, true, false>(p, tmA, tmB, tmR_, grid, stream)
                : launch_tc_conv_t<CONVF_BN, false, false>(p, tmA, tmB, tmR_, grid, stream);
#endif
}
}  // namespace convf
