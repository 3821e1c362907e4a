// Fused MobileNetV2 inverted-residual block: 1x1 expand + BN + ReLU6 -> depthwise 3x3 + BN +
// ReLU6 -> 1x1 project + BN (+ the block input, for stride-1 blocks with equal channel counts)
// in one kernel; the expanded ("hidden") tensor never leaves the SM.
//
// One CTA per tile of TH x TW output pixels of one image.  Its input halo (IH x IW pixels,
// IH = (TH-1)*st + 3) comes in once per 64-channel block as one 4-D TMA box (out-of-image pixels
// are zero fill) and is the A operand of the expand GEMM, whose rows are the halo pixels.  The
// hidden channels go in chunks of 64:
//   warp 0, lane 0   TMA (input halo per tile, weights per chunk, double-buffered) and the
//                    tcgen05 MMAs: expand into a double-buffered TMEM accumulator (up to two
//                    128-row blocks of halo pixels), project into one TMEM accumulator of
//                    Cout columns summed over the chunks
//   warps 1-8        hidden epilogue (TMEM -> BN + ReLU6 -> fp32 rows in shared memory, zero
//                    for halo pixels outside the image: the depthwise conv pads the hidden
//                    tensor with zeros), depthwise 3x3 on CUDA cores (thread = output column x
//                    4 channels, walking the input rows once), BN + ReLU6, and the result split
//                    into two bf16 halves hi + lo (about 16 significant bits) as the project
//                    GEMM's A operands, so the project sees the hidden values at nearly fp32
//                    precision; after the last chunk, the project epilogue (BN, skip
//                    connection, fp32 stores)
// Every wait is bounded (the handle's status word reports a timeout).
#include <cuda_bf16.h>

#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {

namespace {

constexpr int kMbWorkers = 256;   // warps 1-8
constexpr int kMbThreads = 32 + kMbWorkers;
constexpr int kMbTHMax = 8;       // output rows per tile, at most

__device__ __forceinline__ float relu6(float v) { return fminf(fmaxf(v, 0.f), 6.f); }

// two fp32 lanes in one 64-bit register pair for the packed fp32 FMA (two fused multiply-adds,
// each rounded to nearest, per instruction)
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(f32x2 v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// per hidden chunk, the per-channel vectors in one contiguous 3 KB block (one bulk copy):
// rows of 64 floats: expand BN scale, expand BN shift, the nine depthwise taps, depthwise shift
constexpr int kVecRows = 12;
constexpr uint32_t kVecBytes = kVecRows * 64 * 4;

template <int ST>
__global__ void __launch_bounds__(kMbThreads, 1)
    mbv2_block_kernel(const MbParams p, const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWe,
                      const __grid_constant__ CUtensorMap tmWp) {
  extern __shared__ uint8_t mb_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(mb_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = smem + p.off_x;
  uint8_t* sWe = smem + p.off_we;
  uint8_t* sWp = smem + p.off_wp;
  float* sH1 = reinterpret_cast<float*>(smem + p.off_h1);
  uint8_t* sAhi = smem + p.off_a;
  uint8_t* sAlo = sAhi + 16384;
  float* sVec = reinterpret_cast<float*>(smem + p.off_vec);   // [2][kVecRows][64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* bx = bars;          // [2] input halo landed (per halo buffer use)
  uint64_t* bwe = bars + 2;     // [2] expand weights landed (per buffer use)
  uint64_t* bwp = bars + 4;     // [2] project weights landed
  uint64_t* bexp = bars + 6;    // [2] expand MMAs of a chunk complete
  uint64_t* bdw = bars + 8;     // depthwise of a chunk written (8 worker warps)
  uint64_t* bprj = bars + 9;    // project MMAs of a chunk complete
  uint64_t* btile = bars + 10;  // project epilogue of a tile done (8 worker warps)
  uint64_t* bvec = bars + 11;   // [2] per-channel vectors of a chunk landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bx[b], 1);
      mbar_init(&bvec[b], 1);
      mbar_init(&bwe[b], 1);
      mbar_init(&bwp[b], 1);
      mbar_init(&bexp[b], 1);
    }
    mbar_init(bdw, kMbWorkers / 32);
    mbar_init(bprj, 1);
    mbar_init(btile, kMbWorkers / 32);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmWe);
    tma_prefetch_desc(&tmWp);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait_prior();

  const int de_stride = p.rb * 64;            // TMEM columns of one expand buffer
  const uint32_t dp_col = 2u * de_stride;     // project accumulator
  const int tiles_per_img = p.tiles_h * p.tiles_w;
  auto tile_pos = [&](int tile, int& n, int& oy0, int& ox0) {
    n = tile / tiles_per_img;
    const int rem = tile - n * tiles_per_img;
    const int ty = rem / p.tiles_w;
    oy0 = ty * p.TH;
    ox0 = (rem - ty * p.tiles_w) * p.TW;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA + MMA issue
    if (lane == 0) {
      const uint32_t idesc_e = idesc_bf16_f32(128, 64);
      const int nh = p.Np / p.nsplit;
      const uint32_t idesc_p = idesc_bf16_f32(128, nh);
      const uint64_t dX = sdesc_kmajor_sw128(smem_u32(sX));
      const uint64_t dWe = sdesc_kmajor_sw128(smem_u32(sWe));
      const uint64_t dWp = sdesc_kmajor_sw128(smem_u32(sWp));
      const uint64_t dAhi = sdesc_kmajor_sw128(smem_u32(sAhi));
      const uint64_t dAlo = sdesc_kmajor_sw128(smem_u32(sAlo));
      int gc = 0;   // chunks issued so far (all tiles): weight buffer gc % 2, phases
      int ti = 0;   // tiles done by this CTA
      // expand weights of chunk j into buffer g % 2; project weights likewise
      auto load_we = [&](int g, int j) {
        const int b = g & 1;
        mbar_arrive_expect_tx(&bwe[b], p.we_bytes);
        for (int kb = 0; kb < p.cin_kb; ++kb)
          tma_load_2d(sWe + b * p.we_buf + kb * 8192, &tmWe, &bwe[b], kb * 64, j * 64);
      };
      auto load_vec = [&](int g, int j) {
        const int b = g & 1;
        mbar_arrive_expect_tx(&bvec[b], kVecBytes);
        bulk_load(sVec + b * kVecRows * 64, p.vec + static_cast<size_t>(j) * kVecRows * 64, kVecBytes, &bvec[b]);
      };
      auto load_wp = [&](int g, int j) {
        const int b = g & 1;
        mbar_arrive_expect_tx(&bwp[b], p.wp_bytes);
        for (int h = 0; h < p.nsplit; ++h)
          tma_load_2d(sWp + b * p.wp_buf + h * nh * 128, &tmWp, &bwp[b], j * 64, h * nh);
      };
      // the input halo of tile number t (this CTA's t-th) into halo buffer t % nxb
      auto load_x = [&](int t) {
        int n, oy0, ox0;
        tile_pos(blockIdx.x + t * gridDim.x, n, oy0, ox0);
        const int xb = t % p.nxb;
        mbar_arrive_expect_tx(&bx[xb], p.x_bytes);
        for (int kb = 0; kb < p.cin_kb; ++kb)
          tma_load_4d(sX + xb * p.x_buf_bytes + kb * p.x_kb_bytes, &tmX, &bx[xb], kb * 64, ox0 * ST - 1,
                      oy0 * ST - 1, n);
      };
      auto expand = [&](int g, int xb) -> bool {
        const int b = g & 1;
        if (!mbar_wait(&bwe[b], (g >> 1) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        for (int rbk = 0; rbk < p.rb; ++rbk)
          for (int kb = 0; kb < p.cin_kb; ++kb)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_bf16(tmem + b * de_stride + rbk * 64,
                          dX + ((xb * p.x_buf_bytes + kb * p.x_kb_bytes + rbk * 16384) >> 4) + 2 * k,
                          dWe + ((b * p.we_buf + kb * 8192) >> 4) + 2 * k, idesc_e, (kb | k) != 0);
        tc_commit(&bexp[b]);
        return true;
      };
      const int ntiles = blockIdx.x < static_cast<unsigned>(p.num_tiles)
                             ? (p.num_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
      if (ntiles > 0) load_x(0);
      bool okk = true;
      for (ti = 0; ti < ntiles && okk; ++ti) {
        const int xb = ti % p.nxb;
        const int g0 = gc;
        if (ti > 0) {
          // every MMA of the previous tile is complete: its weight buffers are free
          if (!mbar_wait(bprj, (g0 - 1) & 1, abort_flag, p.status)) break;
          if (p.nxb == 1) {
            // one halo buffer: the previous tile's project epilogue must be done with it first
            if (!mbar_wait(btile, (ti - 1) & 1, abort_flag, p.status)) break;
            load_x(ti);
          }
        }
        for (int j = 0; j < p.nch && j < 2; ++j) {
          if (p.expand) load_we(g0 + j, j);
          load_wp(g0 + j, j);
          load_vec(g0 + j, j);   // (the workers of chunk g0 + j - 2 are done with the buffer)
        }
        if (p.expand) {
          if (!mbar_wait(&bx[xb], (ti / p.nxb) & 1, abort_flag, p.status)) break;
          for (int j = 0; j < p.nch && j < 2 && okk; ++j) okk = expand(g0 + j, xb);
          if (!okk) break;
        }
        // the project accumulator (and, with two halo buffers, the other halo buffer) is free once
        // the previous tile's project epilogue is done; then the next tile's halo loads behind
        // this one's chunks
        if (ti > 0 && p.nxb == 2 && !mbar_wait(btile, (ti - 1) & 1, abort_flag, p.status)) break;
        if (p.nxb == 2 && ti + 1 < ntiles) load_x(ti + 1);
        for (int j = 0; j < p.nch && okk; ++j) {
          const int g = g0 + j;
          const int b = g & 1;
          // expand weights of chunk j + 2 as soon as expand j has released their buffer
          if (p.expand && j + 2 < p.nch) {
            if (!mbar_wait(&bexp[b], (g >> 1) & 1, abort_flag, p.status)) { okk = false; break; }
            load_we(g + 2, j + 2);
          }
          // project chunk j once its depthwise output is in shared memory
          if (!mbar_wait(bdw, g & 1, abort_flag, p.status) || !mbar_wait(&bwp[b], (g >> 1) & 1, abort_flag, p.status)) {
            okk = false;
            break;
          }
          tc_fence_after();
          for (int h = 0; h < p.nsplit; ++h)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t bd = dWp + ((b * p.wp_buf + h * nh * 128) >> 4) + 2 * k;
              tc_mma_bf16(tmem + dp_col + h * nh, dAhi + 2 * k, bd, idesc_p, (j | k) != 0);
              tc_mma_bf16(tmem + dp_col + h * nh, dAlo + 2 * k, bd, idesc_p, 1u);
            }
          tc_commit(bprj);
          // the workers are done with chunk j's vectors (its depthwise is written)
          if (j + 2 < p.nch) load_vec(g + 2, j + 2);
          if (j + 2 < p.nch) {
            // project weights of chunk j + 2 once project j has released their buffer
            if (!mbar_wait(bprj, g & 1, abort_flag, p.status)) { okk = false; break; }
            load_wp(g + 2, j + 2);
            if (p.expand && !expand(g + 2, xb)) okk = false;
          }
        }
        gc += p.nch;
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- workers (warps 1-8)
    const int wt = threadIdx.x - 32;          // 0..255
    const int q = warp & 3;                   // TMEM lane quadrant
    const int grp = (warp - 1) >> 2;          // 0: warps 1-4, 1: warps 5-8
    const int cg = wt & 15;                   // depthwise: 4-channel group
    const int dox = wt >> 4;                  // depthwise: output column
    int gc = 0, ti = 0;
    bool okk = true;
    for (int tile = blockIdx.x; tile < p.num_tiles && okk; tile += gridDim.x, ++ti) {
      int n, oy0, ox0;
      tile_pos(tile, n, oy0, ox0);
      const int iy0 = oy0 * ST - 1, ix0 = ox0 * ST - 1;   // halo origin in the input (pad 1)
      for (int j = 0; j < p.nch; ++j) {
        const int g = gc + j;
        const int b = g & 1;
        if (p.expand) {
          if (!mbar_wait(&bexp[b], (g >> 1) & 1, abort_flag, p.status)) { okk = false; break; }
          tc_fence_after();
        } else if (j == 0) {
          if (!mbar_wait(&bx[ti % p.nxb], (ti / p.nxb) & 1, abort_flag, p.status)) { okk = false; break; }
        }
        if (!mbar_wait(&bvec[b], (g >> 1) & 1, abort_flag, p.status)) { okk = false; break; }
        const float* vec = sVec + b * kVecRows * 64;
        named_barrier(1, kMbWorkers);         // the previous chunk's depthwise is done with sH1
        // ---- hidden epilogue: pixel rows of the halo -> fp32 rows of sH1
        {
          const int pix = p.rb == 2 ? grp * 128 + q * 32 + lane : q * 32 + lane;
          const int c_beg = p.rb == 2 ? 0 : grp * 32;
          const int c_cnt = p.rb == 2 ? 64 : 32;
          const int hy = pix / p.IW, hx = pix - (pix / p.IW) * p.IW;
          const bool valid = pix < p.P && iy0 + hy >= 0 && iy0 + hy < p.H && ix0 + hx >= 0 && ix0 + hx < p.W;
          float* hrow = sH1 + static_cast<size_t>(pix) * p.h1_stride;
          if (p.expand) {
            const uint32_t tcol = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * de_stride +
                                  (p.rb == 2 ? grp * 64 : 0) + c_beg;
            for (int cc = 0; cc < c_cnt; cc += 32) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tcol + cc, v);
              tmem_ld_wait();
              if (pix < p.P) {
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                  const int c = c_beg + cc + e;
                  const float4 s4 = *reinterpret_cast<const float4*>(vec + c);
                  const float4 b4 = *reinterpret_cast<const float4*>(vec + 64 + c);
                  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                  if (valid)
                    o = make_float4(relu6(fmaf(__uint_as_float(v[e]), s4.x, b4.x)),
                                    relu6(fmaf(__uint_as_float(v[e + 1]), s4.y, b4.y)),
                                    relu6(fmaf(__uint_as_float(v[e + 2]), s4.z, b4.z)),
                                    relu6(fmaf(__uint_as_float(v[e + 3]), s4.w, b4.w)));
                  *reinterpret_cast<float4*>(hrow + c) = o;
                }
              }
            }
          } else if (pix < p.P) {
            // no expand (t = 1): the hidden tensor is the input itself, bf16 in the halo's
            // 128-byte-swizzled rows (k-block j)
            const uint8_t* xrow = sX + (ti % p.nxb) * p.x_buf_bytes + j * p.x_kb_bytes + (pix >> 3) * 1024 + (pix & 7) * 128;
            for (int c = c_beg; c < c_beg + c_cnt; c += 8) {
              uint4 w = *reinterpret_cast<const uint4*>(xrow + ((((c >> 3) ^ (pix & 7))) << 4));
              if (!valid) w = make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<float4*>(hrow + c) = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                                                                  __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
              *reinterpret_cast<float4*>(hrow + c + 4) = make_float4(__uint_as_float(w.z << 16),
                                                                      __uint_as_float(w.z & 0xffff0000u),
                                                                      __uint_as_float(w.w << 16),
                                                                      __uint_as_float(w.w & 0xffff0000u));
            }
          }
        }
        if (p.expand) tc_fence_before();
        named_barrier(1, kMbWorkers);         // sH1 complete
        // the previous chunk's project MMAs are done reading the A operands
        if (g > 0 && !mbar_wait(bprj, (g - 1) & 1, abort_flag, p.status)) { okk = false; break; }
        // ---- depthwise 3x3 (stride ST, pad 1) + BN + ReLU6 -> bf16 hi/lo A operands
        if (dox < p.TW) {
          f32x2 tp[9][2];
#pragma unroll
          for (int t = 0; t < 9; ++t) {
            const float4 w4 = *reinterpret_cast<const float4*>(vec + (2 + t) * 64 + 4 * cg);
            tp[t][0] = pk2(w4.x, w4.y);
            tp[t][1] = pk2(w4.z, w4.w);
          }
          const float4 bb = *reinterpret_cast<const float4*>(vec + 11 * 64 + 4 * cg);
          f32x2 acc2[kMbTHMax][2];
#pragma unroll
          for (int o = 0; o < kMbTHMax; ++o) {
            acc2[o][0] = pk2(bb.x, bb.y);
            acc2[o][1] = pk2(bb.z, bb.w);
          }
          constexpr int kIHMax = (kMbTHMax - 1) * ST + 3;
#pragma unroll
          for (int iy = 0; iy < kIHMax; ++iy) {
            if (iy >= p.IH) continue;          // (predicates, not breaks: the loops stay unrolled)
            f32x2 v[3][2];
#pragma unroll
            for (int s = 0; s < 3; ++s) {
              const float4 f = *reinterpret_cast<const float4*>(sH1 + static_cast<size_t>(iy * p.IW + dox * ST + s) * p.h1_stride +
                                                               4 * cg);
              v[s][0] = pk2(f.x, f.y);
              v[s][1] = pk2(f.z, f.w);
            }
#pragma unroll
            for (int o = 0; o < kMbTHMax; ++o) {
              const int r = iy - o * ST;
              if (r < 0 || r > 2) continue;
#pragma unroll
              for (int s = 0; s < 3; ++s) {
                acc2[o][0] = fma2(v[s][0], tp[r * 3 + s][0], acc2[o][0]);
                acc2[o][1] = fma2(v[s][1], tp[r * 3 + s][1], acc2[o][1]);
              }
            }
          }
          float4 acc[kMbTHMax];
#pragma unroll
          for (int o = 0; o < kMbTHMax; ++o) {
            upk2(acc2[o][0], acc[o].x, acc[o].y);
            upk2(acc2[o][1], acc[o].z, acc[o].w);
          }
#pragma unroll
          for (int o = 0; o < kMbTHMax; ++o) {
            if (o >= p.TH) continue;
            const float h[4] = {relu6(acc[o].x), relu6(acc[o].y), relu6(acc[o].z), relu6(acc[o].w)};
            uint32_t hi[2], lo[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const __nv_bfloat162 a = __floats2bfloat162_rn(h[2 * e], h[2 * e + 1]);
              const float2 af = __bfloat1622float2(a);
              const __nv_bfloat162 l = __floats2bfloat162_rn(h[2 * e] - af.x, h[2 * e + 1] - af.y);
              hi[e] = *reinterpret_cast<const uint32_t*>(&a);
              lo[e] = *reinterpret_cast<const uint32_t*>(&l);
            }
            const int m = o * p.TW + dox;     // A row = output pixel of the tile
            const uint32_t off = (m >> 3) * 1024 + (m & 7) * 128 + ((((cg >> 1) ^ (m & 7))) << 4) + (cg & 1) * 8;
            *reinterpret_cast<uint2*>(sAhi + off) = make_uint2(hi[0], hi[1]);
            *reinterpret_cast<uint2*>(sAlo + off) = make_uint2(lo[0], lo[1]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bdw);
      }
      if (!okk) break;
      gc += p.nch;
      // ---- project epilogue: TMEM rows = output pixels -> BN (+ skip) -> fp32 NHWC
      if (!mbar_wait(bprj, (gc - 1) & 1, abort_flag, p.status)) break;
      tc_fence_after();
      {
        const int m = q * 32 + lane;
        const int oy = m / p.TW, ox = m - (m / p.TW) * p.TW;
        const bool pix_ok = m < p.TH * p.TW && oy0 + oy < p.Ho && ox0 + ox < p.Wo;
        float* yrow = p.y + ((static_cast<size_t>(n) * p.Ho + oy0 + oy) * p.Wo + ox0 + ox) * p.Cout;
        const int hp = (oy + 1) * p.IW + ox + 1;   // the same pixel in the halo (skip connection, stride 1)
        const int n16 = p.Np / 16;
        const int half = (n16 + 1) / 2;
        const int c_beg = grp == 0 ? 0 : half, c_end = grp == 0 ? half : n16;
        for (int c16 = c_beg; c16 < c_end; ++c16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(q * 32) << 16) + dp_col + c16 * 16, v);
          tmem_ld_wait();
          if (!pix_ok) continue;
          for (int e = 0; e < 16; e += 4) {
            const int k = c16 * 16 + e;
            if (k >= p.Cout) break;
            const float4 s4 = __ldg(reinterpret_cast<const float4*>(p.sp + k));
            const float4 b4 = __ldg(reinterpret_cast<const float4*>(p.bp + k));
            float4 o = make_float4(fmaf(__uint_as_float(v[e]), s4.x, b4.x), fmaf(__uint_as_float(v[e + 1]), s4.y, b4.y),
                                   fmaf(__uint_as_float(v[e + 2]), s4.z, b4.z), fmaf(__uint_as_float(v[e + 3]), s4.w, b4.w));
            if (p.residual && CONVF_IN_BOUNDS(hp < p.P && k < p.cin_kb * 64, p.status)) {
              const uint8_t* xr = sX + (ti % p.nxb) * p.x_buf_bytes + (k >> 6) * p.x_kb_bytes + (hp >> 3) * 1024 +
                                  (hp & 7) * 128;
              const uint2 w = *reinterpret_cast<const uint2*>(xr + (((((k & 63) >> 3) ^ (hp & 7))) << 4) + (k & 4) * 2);
              o.x += __uint_as_float(w.x << 16);
              o.y += __uint_as_float(w.x & 0xffff0000u);
              o.z += __uint_as_float(w.y << 16);
              o.w += __uint_as_float(w.y & 0xffff0000u);
            }
            if (CONVF_IN_BOUNDS(((static_cast<size_t>(n) * p.Ho + oy0 + oy) * p.Wo + ox0 + ox) * p.Cout + k + 4 <=
                                    static_cast<size_t>(p.N) * p.Ho * p.Wo * p.Cout,
                                p.status))
              *reinterpret_cast<float4*>(yrow + k) = o;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(btile);
    }
  }

  // teardown
  __syncwarp();
  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // a wait ran out: give copies and MMAs in flight time to land before TMEM and smem go away
    for (int i = 0; i < 2000; ++i) __nanosleep(100000);
  }
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// at least 120 KB so that a second CTA never shares the SM (each holds all 512 TMEM columns)
size_t mbv2_block_smem(const MbParams& p) {
  const size_t need = 1024 + p.off_bar + 256;
  return need < 122880 ? 122880 : need;
}

cudaError_t launch_mbv2_block(const MbParams& p, const CUtensorMap& tmX, const CUtensorMap& tmWe,
                              const CUtensorMap& tmWp, int grid, cudaStream_t stream) {
  const size_t smem = mbv2_block_smem(p);
  auto* k = p.st == 1 ? mbv2_block_kernel<1> : mbv2_block_kernel<2>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(kMbThreads), smem, stream, 1, p, tmX, tmWe, tmWp);
}

}  // namespace convf
