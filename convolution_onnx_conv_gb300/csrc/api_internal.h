// Host-side services of api.cu for the library's other host translation units (the conv chain,
// chain.cu): the thread-local error message, the allocation-failure test hook, the driver's
// tensor-map encoders, and a read-only view of a handle's tcgen05 configuration.
#pragma once
#include <cuda.h>

#include "conv_fused.h"
#include "convf_internal.h"

namespace convf {

// Sets conv_fused_last_error's message (printf format) and returns st.
convf_status record_error(convf_status st, const char* fmt, ...);
// Clears the message and returns CONVF_OK.
convf_status record_ok();
// conv_fused_debug_fail_alloc's countdown: true when the allocation about to be made is to fail.
bool take_injected_alloc_failure();

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*EncodeIm2colFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const int*, const int*, cuuint32_t, cuuint32_t,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled / cuTensorMapEncodeIm2col from the driver (false if unavailable)
bool tensor_map_encoders(EncodeTiledFn* tiled, EncodeIm2colFn* im2col);

// What a conv chain needs of a handle: its resolved shape and its device-resident prepacked
// weights and epilogue vectors (owned by the handle, which must outlive the chain).
struct ChainConvInfo {
  int variant;             // CONVF_VARIANT_GEMM_1X1 or CONVF_VARIANT_IMPLICIT_GEMM
  int a_mode;              // kA2D or kAIm2col
  int cblocks, ktot, num_kb;
  int N, C, H, W, K, R, S, sh, sw, dh, dw, pt, pl, pb, pr, Ho, Wo;
  long long M;
  const uint16_t* w;       // [K][ktot] bf16 bits
  const float* scale;      // [round_up(K, 256)]
  const float* bias;       // [round_up(K, 256)]
  float lo, hi;            // activation clamp
  bool out_bf16, has_res;
  int device;
};
// Fills *out for a handle that can be a chain step (a dense bf16 tcgen05 1x1-GEMM or im2col
// implicit-GEMM conv without a pre-activation prologue); otherwise returns
// CONVF_ERR_UNSUPPORTED (or the handle's own error) with a message naming the reason.
convf_status chain_conv_info(const convf_handle* h, ChainConvInfo* out);

}  // namespace convf
