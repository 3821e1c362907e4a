// Persistent tcgen05 implicit-GEMM convolution with a fused scale + bias + clamp epilogue.
//
// GEMM view (the "tensorforge" page does im2col + GEMM, section "Status"; here the im2col is
// never materialised): rows m = (n, oh, ow), M = N*Ho*Wo; columns = output channels K;
// reduction over (tap r,s; channel c) in 64-wide blocks.  One CTA per SM loops over 128 x BN
// output tiles.  Warp roles:
//   warp 0      activation producer: TMA activation tiles (2D/3D tiled loads for
//               1x1/stride-1/pad-0, else im2col loads whose tap offsets select the filter
//               position; padding is TMA zero fill); in gather mode the per-tile bulk copies of
//               input rows
//   warp 1      TMEM allocation + single-thread tcgen05.mma issue into a double-buffered
//               fp32 accumulator (2 x BN TMEM columns)
//   warp 2      weight producer: TMA weight boxes of one or several k-blocks (plus half of the
//               im2col activation loads when a pipeline step holds several k-blocks)
//   warps 3-10  epilogue, two warpgroups on the two column halves of every tile (alternate
//               tiles for 32-wide tiles and stream-K; warps 3-6 only in gather mode):
//               tcgen05.ld -> per-warp smem transpose -> y = clamp(scale[k]*acc + bias[k],
//               lo, hi) -> 16-byte global stores (the ragged M and K edges masked)
//   warps 7-14  (gather mode only) activation rows gathered by threads, for channel counts
//               that TMA cannot address (C not a multiple of 8, e.g. a 3-channel stem)
#pragma once
#include <cuda_bf16.h>

#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kATileBytes = kBM * kBK * 2;
constexpr int kEpiCols = 32;
constexpr int kEpiWarpBytes = 32 * kEpiCols * 4;   // one epilogue warp's 32 x 32 fp32 transpose
constexpr int kPatchBufBytes = 32768;
constexpr int kResAhead = 3;   // staged residual: tiles of L2 prefetch ahead of the smem load
constexpr int kActAhead = 4;   // tiles whose input rows are prefetched into L2 before the wait
constexpr int kGatherThreads = 256;

template <int BN, bool GATHER, bool PAIR, bool RSM = false>
struct TcCfg {
  // with a CTA pair each CTA holds half of the weight tile (BN/2 rows)
  static constexpr int kBTileBytes = (PAIR ? BN / 2 : BN) * kBK * 2;
  // two epilogue warpgroups (alternate tiles, or the two column halves of every tile) except
  // in gather mode, whose extra warps take the register and smem room
  static constexpr int kEpiGroups = GATHER ? 1 : 2;
  // tiles of 64+ columns: both groups can drain every tile, one column half each
  static constexpr bool kSplitEpiOk = kEpiGroups == 2 && BN >= 64;
  static constexpr int kThreads = 96 + 128 * kEpiGroups + (GATHER ? kGatherThreads : 0);
  static constexpr int kStages = tc_conv_stages(BN, GATHER, PAIR, RSM);
  // RSM: two bf16 residual tiles (one per accumulator buffer), 128 rows of BN columns each, as
  // 64-column boxes of 128-byte rows in the 128-byte swizzle
  static constexpr int kResTileBytes = RSM ? kBM * BN * 2 : 0;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kBarBytes = 256;
  // gather mode: two buffers for the input rows one tile needs (TcConvParams::patch_rows)
  static constexpr int kPatchBytes = GATHER ? 2 * kPatchBufBytes : 0;
  static constexpr int kSmem = 1024 + kStages * (kATileBytes + kBTileBytes) + 4 * kEpiGroups * kEpiWarpBytes +
                               2 * kResTileBytes + kPatchBytes + kBarBytes;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512, "TMEM columns");
};

// Work of one CTA as a sequence of segments (tile, k-blocks [ka, kend)): whole tiles tstart,
// tstart + tstep, ... or, with stream-K, this CTA's contiguous share [it0, it1) of the
// num_tiles x (num_kb / kpb) pipeline steps, cut at tile boundaries (so segments start and end on
// step boundaries).  Every role walks the same sequence.
template <bool SK>
struct SegSched {
  int num_kb, num_tiles, tstep, tile, kpb, spt;
  long long it, it1;
  __device__ SegSched(const TcConvParams& p, int tstart, int tstep_)
      : num_kb(p.num_kb), num_tiles(p.num_tiles), tstep(tstep_), tile(tstart), kpb(p.kpb), spt(p.num_kb / p.kpb),
        it(0), it1(0) {
    if (SK) {
      const long long total = static_cast<long long>(p.num_tiles) * spt;
      it = total * blockIdx.x / gridDim.x;
      it1 = total * (blockIdx.x + 1) / gridDim.x;
    }
  }
  __device__ bool next(int& t, int& ka, int& kend) {
    if (!SK) {
      if (tile >= num_tiles) return false;
      t = tile;
      ka = 0;
      kend = num_kb;
      tile += tstep;
      return true;
    }
    if (it >= it1) return false;
    t = static_cast<int>(it / spt);
    const long long base = static_cast<long long>(t) * spt;
    const int s0 = static_cast<int>(it - base);
    const int s1 = static_cast<int>(min(base + spt, it1) - base);
    ka = s0 * kpb;
    kend = s1 * kpb;
    it = base + s1;
    return true;
  }
};

// EXTM: 0 the plain fp32 epilogue; 1 a residual (fp32 or bf16 y); 2 bf16 y without a residual;
// 3 a residual with bf16 y and K % 8 == 0 (the 16-byte mapping known at compile time, four
// prefetched residual vectors instead of eight); 4 the same with the residual tile loaded by TMA
// into shared memory while the tile's MMAs run (the activation producer issues it after the
// tile's operands; the epilogue reads it from shared memory instead of waiting on global loads,
// whose latency bounded the HBM-heavy residual layers).
// Each its own instantiation: a shared epilogue cost the fp32 one 1.3% of the ResNet-50 step, and
// the residual's prefetched rows (32 registers) made the bf16-only epilogue spill.
// IQ: integer-exact mode for 8-bit convolutions (TcConvParams::iq_*): the accumulator restarts
// every iq_chunk_kb reduction blocks into alternating TMEM buffers; both epilogue warpgroups
// drain every chunk (one column half each), add it to int32 sums held in registers and, after a
// tile's last chunk, requantise and store 8-bit outputs.
template <int BN, bool GATHER, bool PAIR, bool SK, int EXTM, bool IQ = false>
__global__ void __launch_bounds__(TcCfg<BN, GATHER, PAIR>::kThreads, 1)
    tc_conv_kernel(const TcConvParams p, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmR) {
  static_assert(!(GATHER && PAIR), "the gathered-row mode runs on single CTAs");
  static_assert(!(SK && (GATHER || PAIR)), "stream-K runs on single CTAs with TMA activation loads");
  constexpr bool EXT = EXTM != 0;   // residual and/or bf16 output
  constexpr bool RES = EXTM == 1 || EXTM == 3 || EXTM == 4;   // a residual may be added
  constexpr bool RSM = EXTM == 4;   // the bf16 residual tile staged in shared memory by TMA
  static_assert(!RSM || (!PAIR && !SK && !GATHER && (BN == 64 || BN == 128)), "staged residual: single CTAs, whole tiles");
  static_assert(!(EXT && GATHER), "residual and bf16 output are served with TMA activation loads only");
  static_assert(!(IQ && (GATHER || PAIR || SK || EXT)), "the integer-exact mode runs whole tiles on single CTAs");
  static_assert(!IQ || BN == 64 || BN == 128, "the integer-exact epilogue holds 32 or 64 int32 sums per thread");
  using Cfg = TcCfg<BN, GATHER, PAIR, RSM>;
  // TcConvParams::split_epi on whole tiles of 64+ columns: both epilogue groups drain every
  // tile, one column half each (a tile's epilogue takes half as long, which shortens the last
  // tile of every CTA); otherwise (many tiles per CTA, stream-K segments, 32-column tiles,
  // gather mode) the groups take alternate tiles
  // (the integer-exact mode always splits: both groups then wait on every chunk in order)
  const bool split_epi = Cfg::kSplitEpiOk && !SK && (IQ || p.split_epi);
  // CTA pair (cluster of 2): the leader (rank 0) issues M = 256 MMAs over both CTAs' smem into
  // both CTAs' TMEM; each CTA loads its own 128 activation rows and half of the weight tile.
  const uint32_t crank = PAIR ? cluster_ctarank() : 0;
  const bool leader = !PAIR || crank == 0;
  constexpr int kTileM = PAIR ? 2 * kBM : kBM;
  const int tstart = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tstep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int mrow_off = PAIR ? static_cast<int>(crank) * kBM : 0;
  constexpr int kStages = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kStages * kATileBytes;
  uint8_t* sEpi = sB + kStages * Cfg::kBTileBytes;
  uint8_t* sRes = sEpi + 4 * Cfg::kEpiGroups * kEpiWarpBytes;   // RSM: [2][BN/64][128 rows][128 B]
  uint8_t* sPatch = sRes + 2 * Cfg::kResTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sPatch + Cfg::kPatchBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = bars + 2 * kStages + 2;
  uint64_t* pfull = bars + 2 * kStages + 4;    // input-row patch landed (gather mode)
  uint64_t* pempty = bars + 2 * kStages + 6;   // input-row patch consumed (gather mode)
  uint64_t* rfull = bars + 2 * kStages + 8;    // RSM: residual tile landed (per buffer)
  uint64_t* rempty = bars + 2 * kStages + 10;  // RSM: residual tile read (per buffer)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // gather mode: go/abort decisions broadcast by a leader thread through a named barrier; two
  // slots used alternately so the leader never overwrites a flag another thread has yet to read
  volatile int* gat_go = abort_flag + 5;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // weight producer + (activation producer | one arrival per gather warp)
      mbar_init(&full[s], GATHER ? 1 + kGatherThreads / 32 : 2);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      // one arrival per warp that drains the buffer (both groups when they split the columns)
      mbar_init(&tempty[b], (PAIR ? 2 : 1) * 4 * (split_epi ? 2 : 1));
      mbar_init(&pfull[b], 1);
      mbar_init(&pempty[b], 1);
      mbar_init(&rfull[b], 1);
      mbar_init(&rempty[b], 4 * (split_epi ? 2 : 1));
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (!GATHER) tma_prefetch_desc(&tmA);
    if (RSM) tma_prefetch_desc(&tmR);
  }
  if (warp == 2 && lane == 0) tma_prefetch_desc(&tmB);
  // the integer-exact mode keeps its running int32 sums in a third BN-column region
  constexpr uint32_t kTmemAlloc = IQ ? 512u : static_cast<uint32_t>(Cfg::kTmemCols);
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, kTmemAlloc);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemAlloc);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();   // the peer's barriers and TMEM exist before any cross-CTA operation
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // setup above touched only smem/TMEM: overlap it with the previous kernel's tail
  pdl_launch_dependents();
  // The weights are not written by the previous kernel: the weight producer issues the weight
  // boxes of its first pipeline steps (one pass over the free stages) before waiting for it, so
  // only the activations are on the critical path when it completes.  Those stages get the
  // weight bytes as expected transactions without an arrival; the producer arrives on them
  // after the wait (with its share of the activation bytes), so no phase can complete early.
  int pre_steps = 0;
  if (!PAIR && warp == 2 && lane == 0) {
    SegSched<SK> sched(p, tstart, tstep);
    int tile, ka, kend;
    if (sched.next(tile, ka, kend)) {
      const int n0 = (tile % p.n_blocks) * BN;
      const int kpb0 = GATHER ? 1 : p.kpb;
      for (int kb = ka; kb < kend && (pre_steps + 1) * kpb0 <= kStages; kb += kpb0, ++pre_steps) {
        const int stage = pre_steps * kpb0;
        mbar_expect_tx(&full[stage], static_cast<uint32_t>(kpb0 * Cfg::kBTileBytes));
        if (kpb0 == 1)
          tma_load_2d(sB + stage * Cfg::kBTileBytes, &tmB, &full[stage], kb * kBK, n0);
        else
          tma_load_3d(sB + stage * Cfg::kBTileBytes, &tmB, &full[stage], 0, n0, kb);
      }
    }
  }
  // The input rows of this CTA's first kActAhead tiles start towards L2 now, behind the previous
  // kernel's tail (a prefetch reads no stale data: whatever the previous kernel still writes
  // lands in L2, which serves every read after the wait).  Whole NHWC rows of one image: the
  // tile's pixels (1x1) or the input rows its output rows read (im2col).
  if (!GATHER && warp == 0 && lane == 0) {
    SegSched<SK> sched(p, tstart, tstep);
    int tile, ka, kend;
    for (int j = 0; j < kActAhead && sched.next(tile, ka, kend); ++j) {
      const int m0 = (tile / p.n_blocks) * kTileM + mrow_off;
      if (m0 >= p.M) break;
      const int m1 = min(m0 + kBM, p.M) - 1;
      if (p.a_mode == kA2D) {
        bulk_prefetch_l2(p.x + static_cast<size_t>(m0) * p.C, static_cast<uint32_t>(m1 - m0 + 1) * p.C * 2);
      } else {
        const int hw = p.Ho * p.Wo;
        const int img = m0 / hw;
        const int last = min(m1 - img * hw, hw - 1);   // within the tile's first image
        const int ih0 = max(0, ((m0 - img * hw) / p.Wo) * p.sh - p.pt);
        const int ih1 = min(p.H - 1, (last / p.Wo) * p.sh - p.pt + (p.R - 1) * p.dh);
        if (ih0 <= ih1)
          bulk_prefetch_l2(p.x + (static_cast<size_t>(img) * p.H + ih0) * p.W * p.C,
                           static_cast<uint32_t>(ih1 - ih0 + 1) * p.W * p.C * 2);
      }
    }
  }
  // RSM: the residual boxes of this CTA's first tiles start towards L2 now (as above)
  if (RSM && warp == 0 && lane == 0) {
    for (int j = 0; j < kResAhead; ++j) {
      const int ft = tstart + j * tstep;
      if (ft >= p.num_tiles) break;
      for (int h = 0; h < BN / 64; ++h) tma_prefetch_l2_2d(&tmR, (ft % p.n_blocks) * BN + h * 64, (ft / p.n_blocks) * kTileM);
    }
  }
  pdl_wait_prior();

  // One pipeline step moves kpb k-blocks (TcConvParams::kpb) through kpb consecutive stage
  // slots under the first slot's barriers.  A TMA operation holds its issuing warp for several
  // hundred cycles and an SM takes a new one only every few hundred cycles, so the bytes per
  // operation and the number of issuing warps set the operand ingest rate: the weights of a
  // step are one box, and the activations one box (3-D map) or kpb loads split between the two
  // producer warps (even k-blocks on warp 0, odd ones on warp 2).
  const int kpb = GATHER ? 1 : p.kpb;
  const bool a3d = !GATHER && p.a3d;
  const bool a_odd = !GATHER && !a3d && kpb > 1;
  const uint32_t a_bytes0 = static_cast<uint32_t>((a3d ? kpb : (kpb + 1) / 2) * kATileBytes);
  const uint32_t b_bytes2 = static_cast<uint32_t>(kpb * Cfg::kBTileBytes + (a_odd ? kpb / 2 : 0) * kATileBytes);
  // first output pixel's input window origin (im2col mode)
  auto tile_origin = [&](int m0, int& img, int& hb, int& wb) {
    if (p.a_mode == kAIm2col) {
      const int hw = p.Ho * p.Wo;
      img = m0 / hw;
      const int rem = m0 - img * hw;
      const int oh = rem / p.Wo;
      const int ow = rem - oh * p.Wo;
      hb = oh * p.sh - p.pt;
      wb = ow * p.sw - p.pl;
    }
  };
  // filter tap (r, s) and channel block cb of a k-block (im2col mode): computed once per tile,
  // then stepped one k-block at a time (the issuing thread's scalar work delays its next copy)
  struct KPos {
    int r, s, cb;
  };
  auto kpos_at = [&](int kb) {
    KPos q{0, 0, 0};
    if (p.a_mode == kAIm2col) {
      const int tap = kb / p.cblocks;
      q.cb = kb - tap * p.cblocks;
      q.r = tap / p.S;
      q.s = tap - q.r * p.S;
    }
    return q;
  };
  auto kpos_next = [&](KPos& q) {
    if (++q.cb == p.cblocks) {
      q.cb = 0;
      if (++q.s == p.S) {
        q.s = 0;
        ++q.r;
      }
    }
  };
  // activation tile of k-block kb at position q: a 2-D tile, or the im2col column of its filter
  // tap and channel block (padding is TMA zero fill)
  // (cbase: first input channel of the tile's channel window -- nonzero only for grouped convs,
  // whose output-channel tiles read the input channels of their own groups)
  auto load_a = [&](int kb, const KPos& q, uint8_t* dA, uint64_t* bar, int m0, int img, int hb, int wb, int cbase) {
    if (p.a_mode == kA2D) {
      if (PAIR)
        tma_load_2d_pair(dA, &tmA, map_to_rank(smem_u32(bar), 0), cbase + kb * kBK, m0);
      else
        tma_load_2d(dA, &tmA, bar, cbase + kb * kBK, m0);
    } else {
      if (PAIR)
        tma_load_im2col_4d_pair(dA, &tmA, map_to_rank(smem_u32(bar), 0), cbase + q.cb * kBK, wb, hb, img,
                                static_cast<uint16_t>(q.s * p.dw), static_cast<uint16_t>(q.r * p.dh));
      else
        tma_load_im2col_4d(dA, &tmA, bar, cbase + q.cb * kBK, wb, hb, img, static_cast<uint16_t>(q.s * p.dw),
                           static_cast<uint16_t>(q.r * p.dh));
    }
  };
  // grouped convs (TcConvParams::grp_kg > 0): a tile of output channels n0.. covers whole groups
  // or lies inside one, and its channel window starts at group n0 / Kg's first input channel
  auto tile_cbase = [&](int tile) {
    return p.grp_kg > 0 ? ((tile % p.n_blocks) * BN / p.grp_kg) * p.grp_cg : 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ activation producer
    // (TMA activation tiles; in gather mode the per-tile input-row bulk copies instead)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      SegSched<SK> sched(p, tstart, tstep);
      int tile, ka, kend;
      for (; sched.next(tile, ka, kend); ++it) {
        const int m0 = (tile / p.n_blocks) * kTileM + mrow_off;
        if (GATHER) {
          if (p.patch_rows > 0) {
            // bulk-copy the input rows this tile reads (whole rows of W*C bf16) into smem
            const int pb = it & 1;
            if (!mbar_wait(&pempty[pb], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) goto teardown;
            const int hw = p.Ho * p.Wo;
            const int img = m0 / hw;
            const int ih_first = ((m0 - img * hw) / p.Wo) * p.sh - p.pt;
            int valid = 0;
            for (int i = 0; i < p.patch_rows; ++i) valid += (ih_first + i >= 0 && ih_first + i < p.H);
            mbar_arrive_expect_tx(&pfull[pb], static_cast<uint32_t>(valid * p.row_bytes));
            for (int i = 0; i < p.patch_rows; ++i) {
              const int ih = ih_first + i;
              if (ih >= 0 && ih < p.H)
                bulk_load(sPatch + pb * kPatchBufBytes + i * p.row_bytes,
                          p.x + (static_cast<size_t>(img) * p.H + ih) * p.W * p.C, p.row_bytes, &pfull[pb]);
            }
          }
          continue;
        }
        int img = 0, hb = 0, wb = 0;
        tile_origin(m0, img, hb, wb);
        const int cbase = tile_cbase(tile);
        KPos q = kpos_at(ka);
        for (int kb = ka; kb < kend; kb += kpb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) goto teardown;
          // a pair's loads all complete on the leader's barrier, which expects both CTAs' bytes
          if (!PAIR || leader)
            mbar_arrive_expect_tx(&full[stage], PAIR ? 2 * a_bytes0 : a_bytes0);
          if (a3d) {
            if (PAIR)
              tma_load_3d_pair(sA + stage * kATileBytes, &tmA, map_to_rank(smem_u32(&full[stage]), 0), 0, m0, kb);
            else
              tma_load_3d(sA + stage * kATileBytes, &tmA, &full[stage], 0, m0, kb);
          } else {
            for (int j = 0; j < kpb; ++j) {
              if (!(j & 1)) load_a(kb + j, q, sA + (stage + j) * kATileBytes, &full[stage], m0, img, hb, wb, cbase);
              kpos_next(q);
            }
          }
          stage += kpb;
          if (stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (RSM) {
          // the tile's residual, behind its operands: into buffer it & 1 once the epilogue has
          // read that buffer's previous tile (rows past M and channels past K are zero fill)
          const int rb = it & 1;
          if (!mbar_wait(&rempty[rb], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) goto teardown;
          const int n0 = (tile % p.n_blocks) * BN;
          mbar_arrive_expect_tx(&rfull[rb], static_cast<uint32_t>(Cfg::kResTileBytes));
          for (int h = 0; h < BN / 64; ++h)
            tma_load_2d(sRes + rb * Cfg::kResTileBytes + h * (kBM * 128), &tmR, &rfull[rb], n0 + h * 64, m0);
          // and the residual of this CTA's tile kResAhead tiles on into L2, so that the shared-
          // memory load above finds it there (two buffers alone leave too few bytes in flight)
          const int ft = tile + kResAhead * tstep;
          if (ft < p.num_tiles) {
            const int fn0 = (ft % p.n_blocks) * BN, fm0 = (ft / p.n_blocks) * kTileM;
            for (int h = 0; h < BN / 64; ++h) tma_prefetch_l2_2d(&tmR, fn0 + h * 64, fm0);
          }
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ weight producer
    // (plus the odd-numbered activation loads of a step when the activation is not one box)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      SegSched<SK> sched(p, tstart, tstep);
      int tile, ka, kend;
      while (sched.next(tile, ka, kend)) {
        const int n0 = (tile % p.n_blocks) * BN;
        const int m0 = (tile / p.n_blocks) * kTileM + mrow_off;
        int img = 0, hb = 0, wb = 0;
        if (a_odd) tile_origin(m0, img, hb, wb);
        const int cbase = tile_cbase(tile);
        KPos q = kpos_at(a_odd ? ka : 0);
        for (int kb = ka; kb < kend; kb += kpb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) goto teardown;
          if (pre_steps > 0) {
            // weights already issued before the dependent-launch wait: arrive with the rest
            --pre_steps;
            mbar_arrive_expect_tx(&full[stage], b_bytes2 - static_cast<uint32_t>(kpb * Cfg::kBTileBytes));
            if (a_odd) {
              for (int j = 0; j < kpb; ++j) {
                if (j & 1) load_a(kb + j, q, sA + (stage + j) * kATileBytes, &full[stage], m0, img, hb, wb, cbase);
                kpos_next(q);
              }
            }
            stage += kpb;
            if (stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          if (!PAIR || leader)
            mbar_arrive_expect_tx(&full[stage], PAIR ? 2 * b_bytes2 : b_bytes2);
          if (PAIR && kpb == 1)
            tma_load_2d_pair(sB + stage * Cfg::kBTileBytes, &tmB, map_to_rank(smem_u32(&full[stage]), 0), kb * kBK,
                             n0 + static_cast<int>(crank) * (BN / 2));
          else if (PAIR)
            tma_load_3d_pair(sB + stage * Cfg::kBTileBytes, &tmB, map_to_rank(smem_u32(&full[stage]), 0), 0,
                             n0 + static_cast<int>(crank) * (BN / 2), kb);
          else if (kpb == 1)
            tma_load_2d(sB + stage * Cfg::kBTileBytes, &tmB, &full[stage], kb * kBK, n0);
          else
            tma_load_3d(sB + stage * Cfg::kBTileBytes, &tmB, &full[stage], 0, n0, kb);
          if (a_odd) {
            for (int j = 0; j < kpb; ++j) {
              if (j & 1) load_a(kb + j, q, sA + (stage + j) * kATileBytes, &full[stage], m0, img, hb, wb, cbase);
              kpos_next(q);
            }
          }
          stage += kpb;
          if (stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, BN);
      // descriptors built once; stages move them by whole 16-byte units (the issuing thread's
      // per-MMA work is what bounds short MMAs)
      const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(sA));
      const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(sB));
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      SegSched<SK> sched(p, tstart, tstep);
      int tile, ka, kend;
      while (sched.next(tile, ka, kend)) {
        if (IQ) {
          // exact chunks: the accumulator restarts every iq_chunk_kb blocks, each chunk into the
          // next TMEM buffer (the epilogue adds the chunks in int32)
          for (int c0 = ka; c0 < kend; c0 += p.iq_chunk_kb) {
            if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.status)) goto teardown;
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            const int c1 = min(c0 + p.iq_chunk_kb, kend);
            for (int kb = c0; kb < c1; kb += kpb) {
              if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) goto teardown;
              tc_fence_after();
              for (int j = 0; j < kpb; ++j) {
                const uint64_t adesc = adesc0 + (((stage + j) * kATileBytes) >> 4);
                const uint64_t bdesc = bdesc0 + (((stage + j) * Cfg::kBTileBytes) >> 4);
                const uint32_t first = kb + j != c0;
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                  tc_mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k == 0 ? first : 1u);
              }
              tc_commit(&empty[stage]);
              stage += kpb;
              if (stage == kStages) {
                stage = 0;
                phase ^= 1;
              }
            }
            tc_commit(&tfull[acc]);
            if (++acc == 2) {
              acc = 0;
              acc_phase ^= 1;
            }
          }
          continue;
        }
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.status)) goto teardown;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        // one k-block per iteration: wait at the first slot of a step, release the step's
        // slots after its last k-block
        // one wait and one release per step; the k-blocks of a step issue back to back (a
        // per-k-block branch on the step position measured 30% slower on 128 x 64 tiles)
        for (int kb = ka; kb < kend; kb += kpb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) goto teardown;
          tc_fence_after();
          for (int j = 0; j < kpb; ++j) {
            const uint64_t adesc = adesc0 + (((stage + j) * kATileBytes) >> 4);
            const uint64_t bdesc = bdesc0 + (((stage + j) * Cfg::kBTileBytes) >> 4);
            const uint32_t first = kb + j != ka;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              // advance 16 bf16 (32 B) along K inside the 128 B swizzle atom
              if (PAIR)
                tc_mma_bf16_pair(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k == 0 ? first : 1u);
              else
                tc_mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k == 0 ? first : 1u);
            }
          }
          if (PAIR)
            tc_commit_pair(&empty[stage], 3);
          else
            tc_commit(&empty[stage]);
          stage += kpb;
          if (stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (PAIR)
          tc_commit_pair(&tfull[acc], 3);
        else
          tc_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
    }
  } else if (warp < 3 + 4 * Cfg::kEpiGroups) {
    // ------------------------------------------------------------------ epilogue
    // Two warpgroups split every tile's columns (split_epi), or take alternate tiles.  Each
    // warp owns TMEM lanes 32q..32q+31 = 32 tile rows and works alone:
    // tcgen05.ld of two 32-column chunks at a time (the buffer is released after the last
    // read) -> its own 4 KB of smem (thread = row) -> read back as thread = (row, 4 channels),
    // scale/bias/clamp, 16-byte stores that cover four whole 128-byte row segments.
    // With stream-K a segment that covers only part of a tile's reduction is a contributor
    // (k-block 0 not in it, always its CTA's first segment: the raw fp32 partial goes to this
    // CTA's workspace slot with plain stores, then the CTA's flag is raised) or the tile's
    // owner (k-block 0 in it, its CTA's last segment: waits for the contributors' flags, adds
    // their partials -- eight loads in flight per contributor and chunk -- applies the
    // epilogue and lowers the flags for the next launch).
    constexpr int G = Cfg::kEpiGroups;
    const int eg = (warp - 3) >> 2;        // epilogue group
    const int q = warp & 3;                // TMEM lane quadrant this warp may access
    if constexpr (IQ) {
      // ---- integer-exact epilogue: thread = tile row 32q + lane, columns [eg*BN/2, (eg+1)*BN/2).
      // The running int32 sums live in TMEM columns [2*BN, 3*BN) (this warp's lanes), so a thread
      // only ever holds 16 columns in registers.
      constexpr int HC = BN / 2;           // this group's columns of a tile
      const int nch = (p.num_kb + p.iq_chunk_kb - 1) / p.iq_chunk_kb;
      const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const uint32_t sums = lane_base + static_cast<uint32_t>(2 * BN + eg * HC);
      SegSched<false> sched(p, tstart, tstep);
      int tile, ka, kend;
      int chunk = 0;                       // chunks drained by this CTA so far (buffer, phase)
      while (sched.next(tile, ka, kend)) {
        const int row = (tile / p.n_blocks) * kBM + q * 32 + lane;
        const int n0 = (tile % p.n_blocks) * BN;
        const int c0 = n0 + eg * HC;       // this group's first output channel
        const bool has_cols = c0 < p.Kout;
        for (int c = 0; c < nch; ++c, ++chunk) {
          const int acc = chunk & 1;
          if (!mbar_wait(&tfull[acc], (chunk >> 1) & 1, abort_flag, p.status)) goto teardown;
          tc_fence_after();
          if (has_cols) {
            const uint32_t buf = lane_base + static_cast<uint32_t>(acc * BN + eg * HC);
#pragma unroll 1
            for (int h = 0; h < HC / 16; ++h) {
              uint32_t v[16], t[16];
              tmem_ld_32x32b_x16(buf + 16 * h, v);
              if (c > 0) tmem_ld_32x32b_x16(sums + 16 * h, t);
              tmem_ld_wait();
              // every chunk sum is an integer of magnitude <= 2^24: the conversion is exact
#pragma unroll
              for (int i = 0; i < 16; ++i)
                t[i] = static_cast<uint32_t>((c > 0 ? static_cast<int>(t[i]) : 0) + __float2int_rn(__uint_as_float(v[i])));
              tmem_st_32x32b_x16(sums + 16 * h, t);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);   // the chunk buffer is free for the MMA again
        }
        if (!has_cols) continue;
        uint8_t* yrow = p.y8 + static_cast<size_t>(row) * p.Kout;
#pragma unroll 1
        for (int g = 0; g < HC / 16; ++g) {
          const int col = c0 + 16 * g;
          uint32_t t[16];
          tmem_ld_32x32b_x16(sums + 16 * g, t);   // warp-collective: before any per-thread exit
          tmem_ld_wait();
          if (col >= p.Kout || row >= p.M) continue;   // Kout % 16 == 0: whole 16-channel groups
          uint32_t packed[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int4 bv = __ldg(reinterpret_cast<const int4*>(p.q_bias + col + 4 * h));
            const int bb[4] = {bv.x, bv.y, bv.z, bv.w};
            int qv[4];
            if (p.iq_mode == 0) {
              const int4 mv = __ldg(reinterpret_cast<const int4*>(p.q_mult + col + 4 * h));
              const int4 sv = __ldg(reinterpret_cast<const int4*>(p.q_shift + col + 4 * h));
              const int mm[4] = {mv.x, mv.y, mv.z, mv.w};
              const int ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // q = (v*M + 2^(sh-1)) >> sh in 64 bits (arithmetic shift: rounds half up)
                const long long v = static_cast<long long>(static_cast<int>(t[4 * h + e])) + bb[e];
                const long long r = (v * mm[e] + (1LL << (ss[e] - 1))) >> ss[e];
                const long long o = r + p.q_zp;
                qv[e] = static_cast<int>(o < p.q_lo ? p.q_lo : (o > p.q_hi ? p.q_hi : o));
              }
            } else {
              const float4 fv = __ldg(reinterpret_cast<const float4*>(p.q_scale + col + 4 * h));
              const float ff[4] = {fv.x, fv.y, fv.z, fv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // float32 steps, each rounded to nearest even: float(v) * m, then to an integer
                const long long v = static_cast<long long>(static_cast<int>(t[4 * h + e])) + bb[e];
                const float pr = __fmul_rn(__ll2float_rn(v), ff[e]);
                const long long o = static_cast<long long>(__float2int_rn(fminf(fmaxf(pr, -1.0e9f), 1.0e9f))) + p.q_zp;
                qv[e] = static_cast<int>(o < p.q_lo ? p.q_lo : (o > p.q_hi ? p.q_hi : o));
              }
            }
            packed[h] = (static_cast<uint32_t>(qv[0]) & 0xffu) | ((static_cast<uint32_t>(qv[1]) & 0xffu) << 8) |
                        ((static_cast<uint32_t>(qv[2]) & 0xffu) << 16) | ((static_cast<uint32_t>(qv[3]) & 0xffu) << 24);
          }
          if (CONVF_IN_BOUNDS(static_cast<size_t>(row) * p.Kout + col + 16 <= static_cast<size_t>(p.M) * p.Kout, p.status))
            *reinterpret_cast<uint4*>(yrow + col) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
      }
      goto teardown;
    }
    const bool glead = warp == 3 + 4 * eg && lane == 0;   // group leader thread
    float* wst = reinterpret_cast<float*>(sEpi + (warp - 3) * kEpiWarpBytes);
    const int sub = lane >> 3;             // row within each group of four in the store phase
    constexpr bool plain_out = !EXT;   // fp32 y, no residual
    const int c4 = lane & 7;               // 4-channel column group
    const long long total_it = static_cast<long long>(p.num_tiles) * (p.num_kb / p.kpb);   // in steps
    // alternate whole tiles: group eg visits only its own tiles; split columns: every tile;
    // stream-K: every segment, keeping its own
    const bool kAll = SK || split_epi;
    SegSched<SK> sched(p, tstart + (kAll ? 0 : eg * tstep), kAll ? tstep : G * tstep);
    int tile, ka, kend;
    for (int seg = kAll ? 0 : eg; sched.next(tile, ka, kend); seg += kAll ? 1 : G) {
      if (SK && seg % G != eg) continue;
      const int acc = seg & 1;                         // accumulator buffer of segment seg
      const uint32_t acc_phase = (seg >> 1) & 1;
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      // 0 whole tile, 1 owner, 2 contributor (always 0 without stream-K)
      const int mode = !SK ? 0 : (ka > 0 ? 2 : (kend < p.num_kb ? 1 : 0));
      int d0 = 0, d1 = 0;                              // owner: contributing CTAs [d0, d1)
      if (SK && mode == 1) {
        // contributors: the CTAs after this one whose share starts inside the tile
        const long long tend = static_cast<long long>(tile + 1) * (p.num_kb / p.kpb);
        d0 = blockIdx.x + 1;
        d1 = d0;
        while (d1 < static_cast<int>(gridDim.x) && total_it * d1 / gridDim.x < tend) ++d1;
        if (glead) {
          for (int d = d0; d < d1; ++d) {
            const long long t0 = clock64();
            while (ld_acquire_gpu(p.sk_flags + d) == 0) {
              if (*abort_flag) break;
              if (clock64() - t0 > kWatchdogCycles) {
                *abort_flag = 1;
                atomicOr(p.status, kStatusTimeout);
                break;
              }
            }
          }
        }
        named_barrier(1 + 2 * eg, 128);
      }
      const int mt = (tile / p.n_blocks) * kTileM + mrow_off + q * 32;   // this warp's first row
      const int n0 = (tile % p.n_blocks) * BN;
      const int left = p.Kout - n0;
      const int nchunks = left >= BN ? BN / kEpiCols : (left + kEpiCols - 1) / kEpiCols;
      float* yw = p.y + static_cast<size_t>(mt) * p.Kout + n0;
      // workspace: one [128][BN] fp32 slot per CTA; this warp's rows of slot d start at ws(d)
      const size_t slot = static_cast<size_t>(kBM) * BN;
      float* wsw = p.sk_ws + slot * blockIdx.x + static_cast<size_t>(q * 32) * BN;
      // two 32-column chunks per TMEM read round (one in gather mode, whose 480 threads have
      // fewer registers each), so the buffer is released as early as possible
      constexpr int kRead = GATHER ? 1 : 2;
      // this group's chunks [cbeg, cend): all of them, or one half when the groups split columns
      const int chalf = (nchunks + 1) >> 1;
      const int cbeg = split_epi ? (eg == 0 ? 0 : chalf) : 0;
      const int cend = split_epi ? (eg == 0 ? chalf : nchunks) : nchunks;
      if (cbeg >= cend && lane == 0) {
        // nothing of this tile to drain (ragged last column block): release at once
        if (PAIR && !leader)
          mbar_arrive_remote(map_to_rank(smem_u32(&tempty[acc]), 0));
        else
          mbar_arrive(&tempty[acc]);
      }
      // RSM: this tile's residual (buffer acc) in shared memory
      if (RSM && !mbar_wait(&rfull[acc], acc_phase, abort_flag, p.status)) break;
      const uint8_t* sResT = sRes + acc * Cfg::kResTileBytes;
      for (int ch = cbeg; ch < cend; ch += kRead) {
        const bool two = kRead == 2 && ch + 1 < cend;
        uint32_t v[kRead][32];
        const uint32_t tcol = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(acc * BN + ch * kEpiCols);
        tmem_ld_32x32b_x32(tcol, v[0]);
        if (two) tmem_ld_32x32b_x32(tcol + kEpiCols, v[kRead - 1]);
        tmem_ld_wait();
        if (ch + kRead >= cend) {
          // the warp's last TMEM read of the tile (tcgen05.ld is warp-collective)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (PAIR && !leader)
              mbar_arrive_remote(map_to_rank(smem_u32(&tempty[acc]), 0));
            else
              mbar_arrive(&tempty[acc]);
          }
        }
#pragma unroll
        for (int h = 0; h < kRead; ++h) {
          if (h == 1 && !two) break;
          const int nc = (ch + h) * kEpiCols;
          const bool col_ok = nc + 4 * c4 < left;
          // this thread's 4 channels (loaded before the transpose so their latency overlaps it)
          const float4 sc = __ldg(reinterpret_cast<const float4*>(p.scale + n0 + nc + 4 * c4));
          const float4 bi = __ldg(reinterpret_cast<const float4*>(p.bias + n0 + nc + 4 * c4));
          // the 16-byte bf16 mapping (EXTM >= 3 at compile time): its 8 channels' scale and bias,
          // likewise in flight before the transpose
          float4 w16s0, w16s1, w16b0, w16b1;
          if constexpr (EXTM >= 3) {
            const int wcol = n0 + nc + 8 * (lane & 3);
            w16s0 = __ldg(reinterpret_cast<const float4*>(p.scale + wcol));
            w16s1 = __ldg(reinterpret_cast<const float4*>(p.scale + wcol + 4));
            w16b0 = __ldg(reinterpret_cast<const float4*>(p.bias + wcol));
            w16b1 = __ldg(reinterpret_cast<const float4*>(p.bias + wcol + 4));
          }
          // EXT: the residual of this thread's eight (row, 4 channels), all eight loads in flight
          // before the transpose (one memory latency per chunk, not one per row).  bf16 output with
          // K % 8 == 0 (w16) maps threads to (row, 8 channels) instead, so that every load and
          // store moves 16 bytes; its residual bits sit in rv[0..3].
          const bool w16 = EXTM >= 3 || (EXT && !SK && p.out_bf16 && (p.Kout & 7) == 0);
          const int sub8 = lane >> 2;   // w16: row within each group of eight
          const int c8 = lane & 3;      // w16: 8-channel column group
          float4 rv[EXTM >= 3 ? 4 : (RES ? 8 : 1)];
          if (RSM) {
            // from the staged tile: row R's 16-byte chunk j sits at chunk j ^ (R & 7) of its
            // 128-byte row (the 128-byte swizzle), one 64-column box after another
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = q * 32 + 8 * i + sub8;
              const int col = nc + 8 * c8;
              const uint4 w = *reinterpret_cast<const uint4*>(sResT + (col >> 6) * (kBM * 128) + rr * 128 +
                                                              ((((col & 63) >> 3) ^ (rr & 7)) << 4));
              rv[i] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z),
                                  __uint_as_float(w.w));
            }
          } else if (RES && w16) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              rv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              const int r = 8 * i + sub8;
              const int col = nc + 8 * c8;
              if (p.res == nullptr || col >= left || mt + r >= p.M) continue;
              const uint16_t* rp = static_cast<const uint16_t*>(p.res) + static_cast<size_t>(mt + r) * p.Kout + n0 + col;
              if (!CONVF_IN_BOUNDS(static_cast<size_t>(mt + r) * p.Kout + n0 + col + (col + 8 <= left ? 8 : 4) <=
                                       static_cast<size_t>(p.M) * p.Kout, p.status))
                continue;
              if (col + 8 <= left) {
                const uint4 q = __ldg(reinterpret_cast<const uint4*>(rp));
                rv[i] = make_float4(__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z),
                                    __uint_as_float(q.w));
              } else {   // the last 4 channels of the row (K % 8 == 0 leaves none; kept for safety)
                const uint2 q = __ldg(reinterpret_cast<const uint2*>(rp));
                rv[i] = make_float4(__uint_as_float(q.x), __uint_as_float(q.y), 0.f, 0.f);
              }
            }
          } else if (RES && EXTM < 3) {
#pragma unroll
            for (int i = 0; i < (EXTM >= 3 ? 0 : 8); ++i) {
              rv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              const int r = 4 * i + sub;
              if (p.res == nullptr || (SK && mode == 2) || !col_ok || mt + r >= p.M) continue;
              const size_t e = static_cast<size_t>(mt + r) * p.Kout + n0 + nc + 4 * c4;
              if (!CONVF_IN_BOUNDS(e + 4 <= static_cast<size_t>(p.M) * p.Kout, p.status)) continue;
              if (p.out_bf16) {
                const uint2 rb = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.res) + e));
                rv[i] = make_float4(__uint_as_float(rb.x << 16), __uint_as_float(rb.x & 0xffff0000u),
                                    __uint_as_float(rb.y << 16), __uint_as_float(rb.y & 0xffff0000u));
              } else {
                rv[i] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.res) + e));
              }
            }
          }
          // row `lane` -> smem, 16-byte chunks XOR-swizzled by row: both phases conflict-free
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(wst + lane * 32 + ((c ^ (lane & 7)) << 2)) =
                make_float4(__uint_as_float(v[h][4 * c]), __uint_as_float(v[h][4 * c + 1]),
                            __uint_as_float(v[h][4 * c + 2]), __uint_as_float(v[h][4 * c + 3]));
          __syncwarp();
          if (EXT && w16) {
            // bf16 output, thread = (row 8i + sub8, channels 8*c8 .. +7): two 16-byte smem reads,
            // one 16-byte residual load (prefetched) and one 16-byte store per row
            const int col = nc + 8 * c8;
            float4 s0, s1, b0, b1;
            if constexpr (EXTM >= 3) {
              s0 = w16s0;
              s1 = w16s1;
              b0 = w16b0;
              b1 = w16b1;
            } else {
              s0 = __ldg(reinterpret_cast<const float4*>(p.scale + n0 + col));
              s1 = __ldg(reinterpret_cast<const float4*>(p.scale + n0 + col + 4));
              b0 = __ldg(reinterpret_cast<const float4*>(p.bias + n0 + col));
              b1 = __ldg(reinterpret_cast<const float4*>(p.bias + n0 + col + 4));
            }
            float4 x0[4], x1[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = 8 * i + sub8;
              x0[i] = *reinterpret_cast<const float4*>(wst + r * 32 + (((2 * c8) ^ (r & 7)) << 2));
              x1[i] = *reinterpret_cast<const float4*>(wst + r * 32 + (((2 * c8 + 1) ^ (r & 7)) << 2));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = 8 * i + sub8;
              if (col >= left || mt + r >= p.M) continue;
              float o[8] = {fmaf(x0[i].x, s0.x, b0.x), fmaf(x0[i].y, s0.y, b0.y), fmaf(x0[i].z, s0.z, b0.z),
                            fmaf(x0[i].w, s0.w, b0.w), fmaf(x1[i].x, s1.x, b1.x), fmaf(x1[i].y, s1.y, b1.y),
                            fmaf(x1[i].z, s1.z, b1.z), fmaf(x1[i].w, s1.w, b1.w)};
              uint32_t pk[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                // residual (zero bits when there is none) added before the clamp, then RNE to bf16
                float a0 = o[2 * j], a1 = o[2 * j + 1];
                if constexpr (RES) {
                  const uint32_t rb = __float_as_uint(j == 0 ? rv[i].x : j == 1 ? rv[i].y : j == 2 ? rv[i].z : rv[i].w);
                  a0 += __uint_as_float(rb << 16);
                  a1 += __uint_as_float(rb & 0xffff0000u);
                }
                const float lo = fminf(fmaxf(a0, p.lo), p.hi);
                const float hi = fminf(fmaxf(a1, p.lo), p.hi);
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                pk[j] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              uint16_t* yp = reinterpret_cast<uint16_t*>(p.y) + static_cast<size_t>(mt + r) * p.Kout + n0 + col;
              if (!CONVF_IN_BOUNDS(static_cast<size_t>(mt + r) * p.Kout + n0 + col + (col + 8 <= left ? 8 : 4) <=
                                       static_cast<size_t>(p.M) * p.Kout, p.status))
                continue;
              if (col + 8 <= left)
                *reinterpret_cast<uint4*>(yp) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              else
                *reinterpret_cast<uint2*>(yp) = make_uint2(pk[0], pk[1]);
            }
            __syncwarp();
            continue;
          }
          // all eight of this thread's (row, 4 channels) read back first: the shared-memory loads
          // issue back to back instead of one load latency per row
          float4 a[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + sub;
            a[i] = *reinterpret_cast<const float4*>(wst + r * 32 + ((c4 ^ (r & 7)) << 2));
          }
          float4 part[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) part[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (SK)
            for (int d = d0; d < d1; ++d) {
            // one contributor's partial for these rows: all eight loads in flight at once
            const float* wd = p.sk_ws + slot * d + static_cast<size_t>(q * 32) * BN + nc + 4 * c4;
            float4 b[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + sub;
              b[i] = (col_ok && mt + r < p.M) ? __ldcg(reinterpret_cast<const float4*>(wd + static_cast<size_t>(r) * BN))
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              part[i].x += b[i].x;
              part[i].y += b[i].y;
              part[i].z += b[i].z;
              part[i].w += b[i].w;
            }
          }
          if (!plain_out && !(SK && mode == 2)) {
            // residual and/or bf16 output: v = scale*acc + bias' (+ r), clamp, store as fp32 or
            // as four round-to-nearest-even bf16 (8 bytes)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + sub;
              if (!col_ok || mt + r >= p.M) continue;
              if (SK) {
                a[i].x += part[i].x;
                a[i].y += part[i].y;
                a[i].z += part[i].z;
                a[i].w += part[i].w;
              }
              const size_t e = static_cast<size_t>(mt + r) * p.Kout + n0 + nc + 4 * c4;   // element index
              float4 v = make_float4(fmaf(a[i].x, sc.x, bi.x), fmaf(a[i].y, sc.y, bi.y), fmaf(a[i].z, sc.z, bi.z),
                                     fmaf(a[i].w, sc.w, bi.w));
              if (RES && EXTM < 3) {   // zero where there is no residual
                v.x += rv[EXTM == 1 ? i : 0].x;
                v.y += rv[EXTM == 1 ? i : 0].y;
                v.z += rv[EXTM == 1 ? i : 0].z;
                v.w += rv[EXTM == 1 ? i : 0].w;
              }
              v = make_float4(fminf(fmaxf(v.x, p.lo), p.hi), fminf(fmaxf(v.y, p.lo), p.hi),
                              fminf(fmaxf(v.z, p.lo), p.hi), fminf(fmaxf(v.w, p.lo), p.hi));
              if (!CONVF_IN_BOUNDS(e + 4 <= static_cast<size_t>(p.M) * p.Kout, p.status)) continue;
              if (p.out_bf16) {
                const __nv_bfloat162 lo2 = __floats2bfloat162_rn(v.x, v.y);
                const __nv_bfloat162 hi2 = __floats2bfloat162_rn(v.z, v.w);
                *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.y) + e) =
                    make_uint2(*reinterpret_cast<const uint32_t*>(&lo2), *reinterpret_cast<const uint32_t*>(&hi2));
              } else {
                *reinterpret_cast<float4*>(p.y + e) = v;
              }
            }
          } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = 4 * i + sub;
            if (!col_ok || mt + r >= p.M) continue;
            if (SK) {
              if (mode == 2) {
                if (CONVF_IN_BOUNDS(static_cast<size_t>(q * 32 + r) * BN + nc + 4 * c4 + 4 <= static_cast<size_t>(kBM) * BN,
                                    p.status))
                  __stcg(reinterpret_cast<float4*>(wsw + static_cast<size_t>(r) * BN + nc + 4 * c4), a[i]);
                continue;
              }
              a[i].x += part[i].x;
              a[i].y += part[i].y;
              a[i].z += part[i].z;
              a[i].w += part[i].w;
            }
            if (!CONVF_IN_BOUNDS(static_cast<size_t>(mt + r) * p.Kout + n0 + nc + 4 * c4 + 4 <=
                                     static_cast<size_t>(p.M) * p.Kout, p.status))
              continue;
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
      if (RSM) {
        // this warp has read its rows of the staged residual: the producer may refill the buffer
        __syncwarp();
        if (lane == 0) mbar_arrive(&rempty[acc]);
      }
      if (SK && mode == 2) {
        // partial published: every thread's stores are visible before the flag
        __threadfence();
        named_barrier(1 + 2 * eg, 128);
        if (glead) st_release_gpu(p.sk_flags + blockIdx.x, 1);
      } else if (SK && mode == 1) {
        // every partial has been read: lower the contributors' flags for the next launch
        named_barrier(1 + 2 * eg, 128);
        if (glead)
          for (int d = d0; d < d1; ++d) p.sk_flags[d] = 0;
      }
    }
  } else if (GATHER) {
    // ------------------------------------------------------------------ row gatherers
    // 256 threads, two per tile row: thread gt assembles half gh of row gr in every k-block
    // (16-byte chunks 4*gh .. 4*gh+3 of the row's 128 bytes).  Reduction index
    // j = (r*S + s)*Cp + c.  With p.patch_rows > 0 the rows come from the tile's input rows that
    // the producer bulk-copied into smem; with cpt > 0 the input already holds whole taps of
    // cpt channels (zero-padded by pad_channels_kernel) and each tap is one vector read.
    const int gt = threadIdx.x - 96 - 128 * Cfg::kEpiGroups;
    const int gr = gt & 127;
    const int gh = gt >> 7;
    int stage = 0;
    uint32_t phase = 0;
    int gi = 0;                            // broadcast counter (selects the go slot)
    const int hw = p.Ho * p.Wo;
    const bool use_patch = p.patch_rows > 0;
    int it = 0;
    for (int tile = tstart; tile < p.num_tiles; tile += tstep, ++it) {
      const int m0 = (tile / p.n_blocks) * kBM;
      const int m = m0 + gr;
      const bool row_ok = m < p.M;
      const int img = row_ok ? m / hw : 0;
      const int rem = m - img * hw;
      const int oh = rem / p.Wo;
      const int ow = rem - oh * p.Wo;
      const int ih0 = oh * p.sh - p.pt;
      const int iw0 = ow * p.sw - p.pl;
      const int pb = it & 1;
      int ih_first = 0;
      const uint16_t* src;
      if (use_patch) {
        if (gt == 0) gat_go[gi & 1] = mbar_wait(&pfull[pb], (it >> 1) & 1, abort_flag, p.status) ? 1 : 0;
        named_barrier(2, kGatherThreads);  // also: every thread has finished the previous tile
        if (!gat_go[gi & 1]) goto teardown;
        ++gi;
        const int img0 = m0 / hw;
        ih_first = ((m0 - img0 * hw) / p.Wo) * p.sh - p.pt;
        src = reinterpret_cast<const uint16_t*>(sPatch + pb * kPatchBufBytes);
      } else {
        src = p.x + static_cast<size_t>(img) * p.H * p.W * p.C;
      }
      for (int kb = 0; kb < p.num_kb; ++kb) {
        if (gt == 0) gat_go[gi & 1] = mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status) ? 1 : 0;
        named_barrier(2, kGatherThreads);
        if (!gat_go[gi & 1]) goto teardown;
        ++gi;
        uint8_t* dst = sA + stage * kATileBytes + gr * 128;
        if (p.cpt == 4) {
          // 8 whole taps of 4 channels (8 bytes each) -> chunks 4*gh .. 4*gh+3
          const int t0 = kb * 16 + gh * 8;
          int r = t0 / p.S, s = t0 - (t0 / p.S) * p.S;
          uint2 v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            v[i] = make_uint2(0, 0);
            const int ih = ih0 + r * p.dh, iw = iw0 + s * p.dw;
            if (row_ok && r < p.R && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W &&
                CONVF_IN_BOUNDS(!use_patch || (ih >= ih_first && ih - ih_first < p.patch_rows), p.status))
              v[i] = *reinterpret_cast<const uint2*>(src + ((ih - ih_first) * p.W + iw) * 4);
            if (++s == p.S) {
              s = 0;
              ++r;
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(dst + (((gh * 4 + q) ^ (gr & 7)) << 4)) =
                make_uint4(v[2 * q].x, v[2 * q].y, v[2 * q + 1].x, v[2 * q + 1].y);
        } else if (p.cpt == 8) {
          // 4 whole taps of 8 channels (16 bytes each)
          const int t0 = kb * 8 + gh * 4;
          int r = t0 / p.S, s = t0 - (t0 / p.S) * p.S;
          uint4 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[i] = make_uint4(0, 0, 0, 0);
            const int ih = ih0 + r * p.dh, iw = iw0 + s * p.dw;
            if (row_ok && r < p.R && ih >= 0 && ih < p.H && iw >= 0 && iw < p.W &&
                CONVF_IN_BOUNDS(!use_patch || (ih >= ih_first && ih - ih_first < p.patch_rows), p.status))
              v[i] = *reinterpret_cast<const uint4*>(src + ((ih - ih_first) * p.W + iw) * 8);
            if (++s == p.S) {
              s = 0;
              ++r;
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(dst + (((gh * 4 + q) ^ (gr & 7)) << 4)) = v[q];
        } else {
          // channel by channel: elements j0 .. j0+31 of the row
          const int j0 = kb * 64 + gh * 32;
          int c = j0 % p.C;
          const int t = j0 / p.C;
          int s = t % p.S;
          int r = t / p.S;
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              uint32_t val = 0;
              if (row_ok && r < p.R) {
                const int ih = ih0 + r * p.dh;
                const int iw = iw0 + s * p.dw;
                if (ih >= 0 && ih < p.H && iw >= 0 && iw < p.W &&
                    CONVF_IN_BOUNDS(!use_patch || (ih >= ih_first && ih - ih_first < p.patch_rows), p.status))
                  val = use_patch ? src[((ih - ih_first) * p.W + iw) * p.C + c]
                                  : __ldg(src + (static_cast<size_t>(ih) * p.W + iw) * p.C + c);
              }
              if (e & 1)
                pk[e >> 1] |= val << 16;
              else
                pk[e >> 1] = val;
              if (++c == p.C) {
                c = 0;
                if (++s == p.S) {
                  s = 0;
                  ++r;
                }
              }
            }
            *reinterpret_cast<uint4*>(dst + (((gh * 4 + q) ^ (gr & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);   // one arrival per gather warp
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (use_patch) {
        named_barrier(2, kGatherThreads);  // every row of this tile has been assembled
        if (gt == 0) mbar_arrive(&pempty[pb]);
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
  if (PAIR) cluster_sync();   // no CTA of the pair leaves while the other may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemAlloc);
    else
      tmem_dealloc(tmem_base, kTmemAlloc);
  }
}

// tmR: the residual's tensor map (EXTM 4 only; any map otherwise, unused)
template <int BN, bool GATHER, bool PAIR, bool SK = false, int EXTM = 0, bool IQ = false>
cudaError_t launch_tc_conv_t(const TcConvParams& p, const CUtensorMap& tmA, const CUtensorMap& tmB,
                             const CUtensorMap& tmR, int grid, cudaStream_t stream) {
  using Cfg = TcCfg<BN, GATHER, PAIR, EXTM == 4>;
  static bool configured = false;
  auto* k = tc_conv_kernel<BN, GATHER, PAIR, SK, EXTM, IQ>;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    if (PAIR) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
      if (e != cudaSuccess) return e;
    }
    configured = true;
  }
  return launch_pdl(k, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmem, stream, PAIR ? 2 : 1, p, tmA, tmB, tmR);
}

}  // namespace convf
