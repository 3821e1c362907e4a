// Halo-tile tcgen05 implicit GEMM for stride-1, dilation-1 convolutions.
//
// Output positions are indexed in rows of Wp = W + pl + pr (the zero-padded input width), so
// the input of filter tap (r, s) for output position i of a tile is padded-input position
// i + r*Wp + s: every tap's A operand is the same shared-memory patch read at a row offset.  A
// tile is TR = floor(128 / Wp) output rows of one image; per 64-channel block the CTA loads ONE
// TMA box of TR + R - 1 padded input rows (out-of-image rows and columns are TMA zero fill,
// 128-byte swizzle) and issues R*S*4 MMAs against it, where the im2col kernel loads R*S boxes.
// The 128-byte swizzle of tcgen05 operands follows absolute shared-memory address bits, so a
// descriptor starting at any 128-byte row of a 1 KB-aligned patch reads it correctly.
// MMA rows past TR*Wp and columns past Wo compute junk the epilogue drops.
//
// Warp roles: 0 activation patches (ring of two) and odd weight loads, 1 TMEM + MMA issue, 2 even
// weight loads, 3-10 two epilogue warpgroups taking alternate tiles.  A TMA operation holds
// its issuing warp for a few hundred cycles whatever its size, so one weight load brings tpo
// consecutive taps (a 3-D box {64 channels, BN rows, tpo taps}: each tap lands as its own
// K-major 128-byte-swizzled BN x 64 operand).
#include <cuda_bf16.h>

#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {

namespace {
constexpr int kHBM = 128;
constexpr int kHBK = 64;
constexpr int kHEpiCols = 32;
constexpr int kHEpiWarpBytes = 32 * kHEpiCols * 4;
constexpr int kHThreads = 96 + 256;
constexpr int kHMaxTaps = 64;

template <int BN>
struct HaloCfg {
  static constexpr int kBBytes = BN * kHBK * 2;   // one tap's weight tile
  static constexpr int kTmemCols = 2 * BN;
};

// patch slot: the box, plus room for the junk MMA rows that read past it
uint32_t patch_stride(int R, int S, int Wp, uint32_t patch_bytes) {
  const uint32_t reach = static_cast<uint32_t>(kHBM + (R - 1) * Wp + S - 1) * 128u;
  const uint32_t b = patch_bytes > reach ? patch_bytes : reach;
  return (b + 1023u) & ~1023u;
}
}  // namespace

size_t tc_halo_fixed_smem(int R, int S, int Wp, uint32_t patch_bytes) {
  return 1024 + 2 * static_cast<size_t>(patch_stride(R, S, Wp, patch_bytes)) + 8 * kHEpiWarpBytes + 2 * kHBM * 4 +
         kHMaxTaps * 4 + 512;
}

// EXT: bf16 output and/or a residual (HaloParams::out_bf16, res) in its own instantiation
template <int BN, bool EXT>
__global__ void __launch_bounds__(kHThreads, 1)
    tc_halo_kernel(const HaloParams p, const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   uint32_t pstride) {
  using Cfg = HaloCfg<BN>;
  const int kStages = p.b_stages;
  const uint32_t bstage = static_cast<uint32_t>(p.tpo) * Cfg::kBBytes;
  extern __shared__ uint8_t halo_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(halo_smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sB = smem;
  uint8_t* sP = sB + kStages * bstage;
  uint8_t* sEpi = sP + 2 * pstride;
  int* rm_off = reinterpret_cast<int*>(sEpi + 8 * kHEpiWarpBytes);   // tile row -> pixel offset or -1
  int* rm_dr = rm_off + kHBM;                                         // tile row -> output row offset
  uint32_t* toff = reinterpret_cast<uint32_t*>(rm_dr + kHBM);         // tap -> patch row offset (16 B units)
  uint64_t* bars = reinterpret_cast<uint64_t*>(toff + kHMaxTaps);
  uint64_t* bfull = bars;
  uint64_t* bempty = bars + kStages;
  uint64_t* afull = bars + 2 * kStages;
  uint64_t* aempty = afull + 2;
  uint64_t* tfull = aempty + 2;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 1);
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);   // one arrival per warp of the group that drains buffer b
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < p.R * p.S) {
    const int t = threadIdx.x;
    toff[t] = static_cast<uint32_t>(((t / p.S) * p.Wp + t % p.S) * 8);
  }
  if (threadIdx.x < kHBM) {
    const int i = threadIdx.x;
    const int dr = i / p.Wp;
    const int ow = i - dr * p.Wp;
    rm_off[i] = (dr < p.TR && ow < p.Wo) ? dr * p.Wo + ow : -1;
    rm_dr[i] = dr;
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tmA);
  if (warp == 2 && lane == 0) tma_prefetch_desc(&tmB);
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();
  // the input rows of this CTA's first two tiles start towards L2 behind the previous kernel's
  // tail (a prefetch reads no stale data: what that kernel still writes lands in L2); the boxes
  // start at column 0 and row max(0, .): the padding columns and rows hold no data
  if (warp == 0 && lane == 0) {
    for (int tile = blockIdx.x, j = 0; j < 2 && tile < p.num_tiles; tile += gridDim.x, ++j) {
      const int rt = tile / p.n_blocks;
      const int img = rt / p.tiles_per_img;
      const int oh0 = (rt - img * p.tiles_per_img) * p.TR;
      for (int cb = 0; cb < p.cblocks; ++cb) tma_prefetch_l2_4d(&tmA, cb * kHBK, 0, max(0, oh0 - p.pt), img);
    }
  }
  pdl_wait_prior();

  const int taps = p.R * p.S;
  // Every CTA reads the same weights: walk the channel blocks and tap groups in an order
  // rotated by the CTA index, so that concurrent CTAs spread over different weight tiles
  // instead of all hitting the same L2 lines at once.  Producers and MMA use the same order.
  const int ngroups = taps / p.tpo;
  const int rot_g = static_cast<int>(blockIdx.x) % ngroups;
  const int rot_c = (static_cast<int>(blockIdx.x) / ngroups) % p.cblocks;
  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------------ producers
    // Loads issued by one thread complete one after another, so the weight loads alternate
    // between two issuing warps: warp 2 takes the even ones, warp 0 the odd ones plus the
    // activation patches.  Both walk the whole sequence to keep their ring positions in step.
    if (lane == 0) {
      const int me = warp == 2 ? 0 : 1;
      int slot = 0, stage = 0, bi = 0;
      uint32_t ph = 0, phase = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
        const int n0 = (tile % p.n_blocks) * BN;
        const int rt = tile / p.n_blocks;
        const int img = rt / p.tiles_per_img;
        const int oh0 = (rt - img * p.tiles_per_img) * p.TR;
        for (int cbi = 0; cbi < p.cblocks; ++cbi) {
          const int cb = cbi + rot_c < p.cblocks ? cbi + rot_c : cbi + rot_c - p.cblocks;
          if (warp == 0) {
            if (!mbar_wait(&aempty[slot], ph ^ 1, abort_flag, p.status)) goto teardown;
            mbar_arrive_expect_tx(&afull[slot], p.patch_bytes);
            tma_load_4d(sP + slot * pstride, &tmA, &afull[slot], cb * kHBK, -p.pl, oh0 - p.pt, img);
            if (++slot == 2) {
              slot = 0;
              ph ^= 1;
            }
          }
          for (int gi = 0; gi < ngroups; ++gi, ++bi) {
            const int g = gi + rot_g < ngroups ? gi + rot_g : gi + rot_g - ngroups;
            if (p.resident) {
              // the whole weight set stays in stage cb * ngroups + g: load it with the first tile
              if (tile == static_cast<int>(blockIdx.x) && (bi & 1) == me) {
                const int st = cb * ngroups + g;
                mbar_arrive_expect_tx(&bfull[st], bstage);
                tma_load_3d(sB + st * bstage, &tmB, &bfull[st], cb * kHBK, n0, g * p.tpo);
              }
              continue;
            }
            if ((bi & 1) == me) {
              if (!mbar_wait(&bempty[stage], phase ^ 1, abort_flag, p.status)) goto teardown;
              mbar_arrive_expect_tx(&bfull[stage], bstage);
              tma_load_3d(sB + stage * bstage, &tmB, &bfull[stage], cb * kHBK, n0, g * p.tpo);
            }
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kHBM, BN);
      const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(sP));
      const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(sB));
      int stage = 0, slot = 0;
      uint32_t phase = 0, ph = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        if (!mbar_wait(&tempty[acc], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) goto teardown;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int cbi = 0; cbi < p.cblocks; ++cbi) {
          if (!mbar_wait(&afull[slot], ph, abort_flag, p.status)) goto teardown;
          tc_fence_after();
          // descriptors are built once; taps and stages move them by whole 16-byte units (the
          // issuing thread's per-MMA work is what bounds short MMAs)
          const uint64_t apatch = adesc0 + ((slot * pstride) >> 4);
          const int cb = cbi + rot_c < p.cblocks ? cbi + rot_c : cbi + rot_c - p.cblocks;
          for (int gi = 0; gi < ngroups; ++gi) {
            const int g = gi + rot_g < ngroups ? gi + rot_g : gi + rot_g - ngroups;
            const int t0 = g * p.tpo;
            // resident weights: stage cb * ngroups + g, landed once (phase 0) and never released
            const int bs = p.resident ? cb * ngroups + g : stage;
            if (!mbar_wait(&bfull[bs], p.resident ? 0u : phase, abort_flag, p.status)) goto teardown;
            tc_fence_after();
            const uint64_t bst = bdesc0 + ((bs * bstage) >> 4);
            for (int j = 0; j < p.tpo; ++j) {
              // tap t0 + j: the patch read r*Wp + s rows further on; its weights are tile j
              const uint64_t adesc = apatch + toff[t0 + j];
              const uint64_t bdesc = bst + j * (Cfg::kBBytes >> 4);
              tc_mma_bf16(d_tmem, adesc, bdesc, idesc, (cbi | gi | j) != 0);
#pragma unroll
              for (int k = 1; k < kHBK / 16; ++k) tc_mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, 1u);
            }
            if (!p.resident) {
              tc_commit(&bempty[stage]);
              if (++stage == kStages) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
          tc_commit(&aempty[slot]);
          if (++slot == 2) {
            slot = 0;
            ph ^= 1;
          }
        }
        tc_commit(&tfull[acc]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    // group eg drains the CTA's tiles it with it % 2 == eg (accumulator buffer eg).  Each warp
    // owns TMEM lanes 32q..32q+31 = tile rows; rows map to output pixels through rm_off/rm_dr.
    const int eg = (warp - 3) >> 2;
    const int q = warp & 3;
    float* wst = reinterpret_cast<float*>(sEpi + (warp - 3) * kHEpiWarpBytes);
    const int sub = lane >> 3;
    const int c4 = lane & 7;
    int n_it = 0;
    for (int tile = blockIdx.x + eg * gridDim.x; tile < p.num_tiles; tile += 2 * gridDim.x, ++n_it) {
      if (!mbar_wait(&tfull[eg], n_it & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const int n0 = (tile % p.n_blocks) * BN;
      const int rt = tile / p.n_blocks;
      const int img = rt / p.tiles_per_img;
      const int oh0 = (rt - img * p.tiles_per_img) * p.TR;
      const int left = p.Kout - n0;
      const int nchunks = left >= BN ? BN / kHEpiCols : (left + kHEpiCols - 1) / kHEpiCols;
      float* ybase = p.y + (static_cast<size_t>(img) * p.Ho + oh0) * p.Wo * p.Kout + n0;
      // elements of y (bounds-checking build): images x Ho x Wo x Kout
      const size_t ytotal = static_cast<size_t>(p.num_tiles / p.n_blocks / p.tiles_per_img) * p.Ho * p.Wo * p.Kout;
      (void)ytotal;
      for (int ch = 0; ch < nchunks; ch += 2) {
        const bool two = ch + 1 < nchunks;
        uint32_t v[2][32];
        const uint32_t tcol = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(eg * BN + ch * kHEpiCols);
        tmem_ld_32x32b_x32(tcol, v[0]);
        if (two) tmem_ld_32x32b_x32(tcol + kHEpiCols, v[1]);
        tmem_ld_wait();
        if (ch + 2 >= nchunks) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[eg]);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !two) break;
          const int nc = (ch + h) * kHEpiCols;
          const bool col_ok = nc + 4 * c4 < left;
          // this thread's 4 channels, fetched before the transpose so their latency overlaps it
          const float4 sc = __ldg(reinterpret_cast<const float4*>(p.scale + n0 + nc + 4 * c4));
          const float4 bi = __ldg(reinterpret_cast<const float4*>(p.bias + n0 + nc + 4 * c4));
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(wst + lane * 32 + ((c ^ (lane & 7)) << 2)) =
                make_float4(__uint_as_float(v[h][4 * c]), __uint_as_float(v[h][4 * c + 1]),
                            __uint_as_float(v[h][4 * c + 2]), __uint_as_float(v[h][4 * c + 3]));
          __syncwarp();
          // all eight rows read back first, so the shared-memory loads issue back to back
          float4 a[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + sub;
            a[i] = *reinterpret_cast<const float4*>(wst + r * 32 + ((c4 ^ (r & 7)) << 2));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int tr = q * 32 + 4 * i + sub;
            const int off = rm_off[tr];
            if (!col_ok || off < 0 || oh0 + rm_dr[tr] >= p.Ho) continue;
            if (!CONVF_IN_BOUNDS(static_cast<size_t>(ybase - p.y) + static_cast<size_t>(off) * p.Kout + nc + 4 * c4 + 4 <=
                                     ytotal, p.status))
              continue;
            if (!EXT) {
              *reinterpret_cast<float4*>(ybase + static_cast<size_t>(off) * p.Kout + nc + 4 * c4) =
                  make_float4(fminf(fmaxf(fmaf(a[i].x, sc.x, bi.x), p.lo), p.hi),
                              fminf(fmaxf(fmaf(a[i].y, sc.y, bi.y), p.lo), p.hi),
                              fminf(fmaxf(fmaf(a[i].z, sc.z, bi.z), p.lo), p.hi),
                              fminf(fmaxf(fmaf(a[i].w, sc.w, bi.w), p.lo), p.hi));
              continue;
            }
            // residual (added after the folded BN, before the clamp) and/or bf16 output
            const size_t e = static_cast<size_t>(ybase - p.y) + static_cast<size_t>(off) * p.Kout + nc + 4 * c4;
            float4 o = make_float4(fmaf(a[i].x, sc.x, bi.x), fmaf(a[i].y, sc.y, bi.y), fmaf(a[i].z, sc.z, bi.z),
                                   fmaf(a[i].w, sc.w, bi.w));
            if (p.res != nullptr) {
              if (p.out_bf16) {
                const uint2 r = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.res) + e));
                o.x += __uint_as_float(r.x << 16);
                o.y += __uint_as_float(r.x & 0xffff0000u);
                o.z += __uint_as_float(r.y << 16);
                o.w += __uint_as_float(r.y & 0xffff0000u);
              } else {
                const float4 r = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.res) + e));
                o.x += r.x;
                o.y += r.y;
                o.z += r.z;
                o.w += r.w;
              }
            }
            o = make_float4(fminf(fmaxf(o.x, p.lo), p.hi), fminf(fmaxf(o.y, p.lo), p.hi),
                            fminf(fmaxf(o.z, p.lo), p.hi), fminf(fmaxf(o.w, p.lo), p.hi));
            if (p.out_bf16) {
              const __nv_bfloat162 b0 = __floats2bfloat162_rn(o.x, o.y), b1 = __floats2bfloat162_rn(o.z, o.w);
              *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.y) + e) =
                  make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
            } else {
              *reinterpret_cast<float4*>(p.y + e) = o;
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
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

namespace {
template <int BN, bool EXT>
cudaError_t launch_bn(const HaloParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int grid,
                      cudaStream_t stream) {
  const uint32_t ps = patch_stride(p.R, p.S, p.Wp, p.patch_bytes);
  const size_t smem = tc_halo_fixed_smem(p.R, p.S, p.Wp, p.patch_bytes) +
                      static_cast<size_t>(p.b_stages) * p.tpo * HaloCfg<BN>::kBBytes;
  if (smem > 232448 || p.b_stages < 2 || p.b_stages > 8) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(tc_halo_kernel<BN, EXT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return launch_pdl(tc_halo_kernel<BN, EXT>, dim3(grid), dim3(kHThreads), smem, stream, 1, p, tmA, tmB, ps);
}
}  // namespace

cudaError_t launch_tc_halo(const HaloParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB, int bn, int grid,
                           cudaStream_t stream) {
  const bool ext = p.out_bf16 || p.res != nullptr;
  switch (bn) {
    case 64: return ext ? launch_bn<64, true>(p, tmA, tmB, grid, stream) : launch_bn<64, false>(p, tmA, tmB, grid, stream);
    case 128:
      return ext ? launch_bn<128, true>(p, tmA, tmB, grid, stream) : launch_bn<128, false>(p, tmA, tmB, grid, stream);
    case 256:
      return ext ? launch_bn<256, true>(p, tmA, tmB, grid, stream) : launch_bn<256, false>(p, tmA, tmB, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace convf
