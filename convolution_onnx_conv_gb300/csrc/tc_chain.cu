// Conv chain: a sequence of tcgen05 convolutions (1x1 GEMM or im2col implicit GEMM) in one
// persistent launch.
//
// Each step is the same fused operation as one run of the tcgen05 kernel (implicit GEMM with
// the folded BN + bias + clamp epilogue, "tensorforge", section "ResNet fusion"; an optional
// residual added before the clamp, "Kyanite" README, section "Cuda Executor"), but the steps
// share one launch: the per-launch costs of a short layer (CTA start, TMEM allocation, the
// first operands' latency, the last tiles' epilogue while other SMs idle) are paid once for
// the whole sequence, and a step's first tiles start while the previous step's last tiles are
// still in flight.  A step that reads an earlier step's output waits only for the 128-row
// blocks it reads (ChainStep::done), so a network's layers pipeline through the GPU.
//
// Warp roles (one CTA per SM, tiles b, b + grid, ... of the launch-wide numbering):
//   warp 0      activation producer: the dependency wait of each tile, then TMA activation
//               loads (one box per k-block, or one per pipeline step in the 3-D 1x1 mode)
//   warp 1      TMEM allocation + single-thread tcgen05.mma issue into four 128-column fp32
//               accumulators (two of 256 columns in a CTA pair)
//   warp 2      weight producer: one TMA box per pipeline step (two k-blocks)
//   warps 3-10  epilogue, two warpgroups on the two column halves of every tile:
//               tcgen05.ld -> smem transpose -> clamp(scale*acc + bias (+ r)) -> 16-byte stores
//   warp 11     publisher: per stored tile of a step whose output a later step reads, a
//               gpu-scope fence and the increment of the tile's row-block counter (off the
//               epilogue warps' path)
// Pipeline: 3 steps of two 64-wide k-blocks each in shared memory (a step's odd k-block is
// zero fill past a step's last block).
#include <cuda_bf16.h>

#include "convf_internal.h"
#include "ptx.cuh"

namespace convf {
namespace {

constexpr int kQM = 128;                    // tile rows
constexpr int kQK = 64;                     // reduction block
constexpr int kQSlots = 6;                  // k-block slots
constexpr int kQSteps = kQSlots / 2;        // pipeline steps of two k-blocks
constexpr int kQATile = kQM * kQK * 2;      // 16 KB
constexpr int kQBTile = 128 * kQK * 2;      // 16 KB: one k-block of up to 128 weight rows
constexpr int kQEpiWarpBytes = 32 * 32 * 4;
constexpr int kQThreads = 96 + 256 + 32;     // producer, MMA, weight producer, 8 epilogue warps, publisher
constexpr int kQPub = 4;                    // tiles a CTA may have stored but not yet published
constexpr int kQSmem = 1024 + kQSlots * (kQATile + kQBTile) + 8 * kQEpiWarpBytes + 256;
static_assert(kQSmem <= 232448, "shared memory budget");
// the barrier block after the epilogue staging: full/empty per step, tfull/tempty per
// accumulator (4), stored/pubfree per publication slot, then the TMEM slot, abort flag and epoch
static_assert((2 * kQSteps + 2 * 4 + 2 * kQPub) * 8 + 3 * 4 <= 256, "barrier block");
static_assert(kChainArrivals == 1, "one arrival per tile (the publisher's)");

// Single CTAs (128-row tiles, up to 128 columns) or CTA pairs (cta_group::2: 256-row tiles of up
// to 256 columns, each CTA of the cluster holding its own 128 rows of activations and of the
// accumulator and half of the weight rows).  A pair moves half the weight bytes per FLOP of a
// single CTA's 128 x 128 tile and issues M = 256 MMAs.
template <bool PAIR>
struct ChainShape {
  // TMEM accumulators, all 512 columns: the MMA issuer may run that many tiles minus one ahead of
  // the epilogue (four on single CTAs measured 4% faster over ResNet-50's 52 layers than two,
  // the MMA running ahead through compute-bound steps while the epilogue drains HBM-bound ones)
  static constexpr int kAcc = PAIR ? 2 : 4;
  static constexpr int kTileM = PAIR ? 256 : 128;   // output rows per tile
  static constexpr int kBNMax = PAIR ? 256 : 128;   // widest tile (TMEM buffer stride)
};

// The tiles of this CTA (or CTA pair) and this CTA's first row within a tile.
template <bool PAIR>
struct ChainSched {
  int tstart, tstep, rowoff;
  uint32_t crank;
  __device__ ChainSched() {
    crank = PAIR ? cluster_ctarank() : 0u;
    tstart = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    tstep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    rowoff = static_cast<int>(crank) * kQM;
  }
};

// Wait until the counter reaches `target` (wrap-safe).  Gives up, raising the CTA's abort flag,
// when another role of this CTA aborted, when any CTA flagged an error in the status word, or
// after the watchdog budget (then the timeout bit is set).
__device__ bool chain_wait(const uint32_t* ctr, uint32_t target, int* status, volatile int* abort_flag) {
  if (static_cast<int>(ld_acquire_gpu_u32(ctr) - target) >= 0) return true;
  const long long t0 = clock64();
  uint32_t ns = 32;
  while (true) {
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
    if (static_cast<int>(ld_acquire_gpu_u32(ctr) - target) >= 0) return true;
    if (*abort_flag || *reinterpret_cast<volatile int*>(status) != 0) {
      *abort_flag = 1;
      return false;
    }
    if (clock64() - t0 > kWatchdogCycles) {
      *abort_flag = 1;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
}

// Input pixels (flat NHWC row indices of the step's x, which are the producing step's output
// rows) that the tile of output rows [m0, m0 + 128) reads: whole input rows, conservatively.
__device__ __forceinline__ void chain_input_rows(const ChainGeom& g, int m0, int& lo, int& hi) {
  const int m1 = min(m0 + kQM, g.M) - 1;
  if (g.a_mode == kA2D) {
    lo = m0;
    hi = m1;
    return;
  }
  const int hw = g.Ho * g.Wo;
  const int i0 = m0 / hw, i1 = m1 / hw;
  const int oh0 = (m0 - i0 * hw) / g.Wo, oh1 = (m1 - i1 * hw) / g.Wo;
  const int h0 = min(max(0, oh0 * g.sh - g.pt), g.H - 1);
  const int h1 = max(min(g.H - 1, oh1 * g.sh - g.pt + (g.R - 1) * g.dh), 0);
  lo = (i0 * g.H + h0) * g.W;
  hi = (i1 * g.H + h1) * g.W + g.W - 1;
}

// Walks the launch-wide tile numbering in increasing order, keeping the step that holds it.
struct ChainCursor {
  const ChainStep* steps;
  int L, end;
  __device__ explicit ChainCursor(const ChainStep* s) : steps(s), L(0), end(s[0].g.tile_end) {}
  __device__ int at(int t) {
    while (t >= end) end = steps[++L].g.tile_end;
    return L;
  }
};

// filter tap (r, s) and channel block of a k-block (im2col mode), stepped one block at a time
struct ChainKPos {
  int r, s, cb;
  __device__ void next(int cblocks, int S) {
    if (++cb == cblocks) {
      cb = 0;
      if (++s == S) {
        s = 0;
        ++r;
      }
    }
  }
};

// Producer roles.  ROLE 0 (warp 0): the dependency wait of each tile, then the activation loads
// of both k-blocks of every pipeline step (one box in the 3-D mode, else one per k-block).
// ROLE 2 (warp 2): the weight box of each step.  (Moving the odd k-block's activation load from
// the weight producer to the activation producer measured 2-5% faster on every layer shape.)
// Every role keeps the current step's fields in registers (ChainGeom, reloaded when the step
// changes): the issuing thread's scalar work delays its next copy.  In a CTA pair both CTAs load
// their own operands; every load completes on the leader's full barrier, which the leader's
// producers arm with both CTAs' bytes.
template <int ROLE, bool PAIR>
__device__ void chain_producer(const ChainParams& p, uint8_t* sA, uint8_t* sB, uint64_t* full, uint64_t* empty,
                               uint32_t epoch1, volatile int* abort_flag) {
  const ChainStep* steps = p.steps;
  const ChainSched<PAIR> sch;
  const bool leader = sch.crank == 0;
  ChainCursor cur(steps);
  int stage = 0;
  uint32_t phase = 0;
  int dep_done = -1;   // row blocks of the source verified for the current step
  int last = -1;
  ChainGeom g;
  const CUtensorMap* tmA = nullptr;
  const CUtensorMap* tmB = nullptr;
  uint32_t b_bytes = 0, target = 0;
  int bcol = 0;        // this CTA's first weight row within a tile (half of the tile in a pair)
  for (int t = sch.tstart; t < p.total_tiles; t += sch.tstep) {
    const int L = cur.at(t);
    if (L != last) {
      last = L;
      g = steps[L].g;
      tmA = &steps[L].tmA;
      tmB = &steps[L].tmB;
      tma_prefetch_desc(ROLE == 0 ? tmA : tmB);
      dep_done = -1;
      // this CTA's weight box: two k-blocks (zero fill past the last), one if the step has one,
      // of bn rows (bn / 2 in a pair)
      const int brows = PAIR ? g.bn / 2 : g.bn;
      b_bytes = static_cast<uint32_t>((g.num_kb > 1 ? 2 : 1) * brows * kQK * 2);
      bcol = static_cast<int>(sch.crank) * brows;
      target = epoch1 * static_cast<uint32_t>(kChainArrivals * g.src_nb);
    }
    const int local = t - g.tile0;
    const int mt = local / g.n_blocks;
    const int n0 = (local - mt * g.n_blocks) * g.bn;
    const int m0 = mt * ChainShape<PAIR>::kTileM + sch.rowoff;   // this CTA's first output row
    const bool a3d = g.a3d != 0, a2d = g.a_mode == kA2D;
    if (ROLE == 0 && g.src >= 0 && m0 < g.M) {
      int lo, hi;
      chain_input_rows(g, m0, lo, hi);
      // this CTA's tiles of one step visit increasing rows, so the blocks below dep_done that
      // the range still covers were verified for an earlier tile
      for (int b = max(lo / kQM, dep_done + 1); b <= hi / kQM; ++b)
        if (!chain_wait(g.src_done + b, target, p.status, abort_flag)) return;
      dep_done = max(dep_done, hi / kQM);
      fence_proxy_async_global();   // the source's stores before this thread's TMA reads
    }
    int img = 0, hb = 0, wb = 0;
    if (ROLE == 0 && !a2d) {
      const int hw = g.Ho * g.Wo;
      img = m0 / hw;
      const int rem = m0 - img * hw;
      const int oh = rem / g.Wo;
      hb = oh * g.sh - g.pt;
      wb = (rem - oh * g.Wo) * g.sw - g.pl;
    }
    ChainKPos q{0, 0, 0};
    for (int kb = 0; kb < g.num_kb; kb += 2) {
      const bool two = kb + 1 < g.num_kb;
      if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) return;
      uint8_t* a0 = sA + stage * 2 * kQATile;
      uint64_t* fb = &full[stage];
      const uint32_t fbar = PAIR ? map_to_rank(smem_u32(fb), 0) : smem_u32(fb);   // the leader's
      if constexpr (ROLE == 0) {
        ChainKPos q1 = q;   // k-block kb + 1
        q1.next(g.cblocks, g.S);
        const uint32_t a_bytes = a3d || two ? 2u * kQATile : static_cast<uint32_t>(kQATile);
        if (leader) mbar_arrive_expect_tx(fb, PAIR ? 2 * a_bytes : a_bytes);
        if (a3d) {
          if (PAIR)
            tma_load_3d_pair(a0, tmA, fbar, 0, m0, kb);
          else
            tma_load_3d(a0, tmA, fb, 0, m0, kb);
        } else {
          for (int jk = 0; jk < (two ? 2 : 1); ++jk) {
            const ChainKPos& qq = jk == 0 ? q : q1;
            uint8_t* dst = a0 + jk * kQATile;
            if (a2d) {
              if (PAIR)
                tma_load_2d_pair(dst, tmA, fbar, (kb + jk) * kQK, m0);
              else
                tma_load_2d(dst, tmA, fb, (kb + jk) * kQK, m0);
            } else {
              const uint16_t ow = static_cast<uint16_t>(qq.s * g.dw), oh = static_cast<uint16_t>(qq.r * g.dh);
              if (PAIR)
                tma_load_im2col_4d_pair(dst, tmA, fbar, qq.cb * kQK, wb, hb, img, ow, oh);
              else
                tma_load_im2col_4d(dst, tmA, fb, qq.cb * kQK, wb, hb, img, ow, oh);
            }
          }
        }
        q = q1;
        q.next(g.cblocks, g.S);
      } else {
        if (leader) mbar_arrive_expect_tx(fb, PAIR ? 2 * b_bytes : b_bytes);
        if (PAIR)
          tma_load_3d_pair(sB + stage * 2 * kQBTile, tmB, fbar, 0, n0 + bcol, kb);
        else
          tma_load_3d(sB + stage * 2 * kQBTile, tmB, fb, 0, n0, kb);
      }
      if (++stage == kQSteps) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
}

// MMA issuer (one thread; the leader's in a CTA pair): per tile, one kTileM x bn accumulator
// buffer (in turn), four K = 16 MMAs per k-block.  A pair's MMAs read both CTAs' operands and
// write both CTAs' TMEM; their commits arrive on the barriers of both CTAs.
template <bool PAIR>
__device__ void chain_mma(const ChainParams& p, uint8_t* sA, uint8_t* sB, uint64_t* full, uint64_t* empty,
                          uint64_t* tfull, uint64_t* tempty, uint32_t tmem_base, volatile int* abort_flag) {
  const ChainStep* steps = p.steps;
  const ChainSched<PAIR> sch;
  ChainCursor cur(steps);
  const uint64_t adesc0 = sdesc_kmajor_sw128(smem_u32(sA));
  const uint64_t bdesc0 = sdesc_kmajor_sw128(smem_u32(sB));
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  int last = -1;
  uint32_t idesc = 0, bblock = 0;
  int num_kb = 0;
  for (int t = sch.tstart; t < p.total_tiles; t += sch.tstep) {
    const int L = cur.at(t);
    if (L != last) {
      last = L;
      idesc = steps[L].g.idesc;
      num_kb = steps[L].g.num_kb;
      // bytes of one k-block's weights in this CTA's shared memory
      bblock = static_cast<uint32_t>((PAIR ? steps[L].g.bn / 2 : steps[L].g.bn) * kQK * 2);
    }
    if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.status)) return;
    tc_fence_after();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ChainShape<PAIR>::kBNMax);
    for (int kb = 0; kb < num_kb; kb += 2) {
      if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) return;
      tc_fence_after();
      const uint64_t a = adesc0 + (static_cast<uint32_t>(stage * 2 * kQATile) >> 4);
      const uint64_t b = bdesc0 + (static_cast<uint32_t>(stage * 2 * kQBTile) >> 4);
      // straight-line issue: each MMA's descriptors are a register plus a constant (about 0.5%
      // faster over the chain than computing them in a loop)
      const uint32_t first = kb > 0 ? 1u : 0u;
      if (PAIR) {
        tc_mma_bf16_pair(d_tmem, a, b, idesc, first);
#pragma unroll
        for (int k = 1; k < 4; ++k) tc_mma_bf16_pair(d_tmem, a + 2 * k, b + 2 * k, idesc, 1u);
      } else {
        tc_mma_bf16(d_tmem, a, b, idesc, first);
#pragma unroll
        for (int k = 1; k < 4; ++k) tc_mma_bf16(d_tmem, a + 2 * k, b + 2 * k, idesc, 1u);
      }
      if (kb + 1 < num_kb) {
        const uint64_t a2 = a + (kQATile >> 4), b2 = b + (bblock >> 4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (PAIR)
            tc_mma_bf16_pair(d_tmem, a2 + 2 * k, b2 + 2 * k, idesc, 1u);
          else
            tc_mma_bf16(d_tmem, a2 + 2 * k, b2 + 2 * k, idesc, 1u);
        }
      }
      if (PAIR)
        tc_commit_pair(&empty[stage], 3);
      else
        tc_commit(&empty[stage]);
      if (++stage == kQSteps) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (PAIR)
      tc_commit_pair(&tfull[acc], 3);
    else
      tc_commit(&tfull[acc]);
    if (++acc == ChainShape<PAIR>::kAcc) {
      acc = 0;
      acc_phase ^= 1;
    }
  }
}

// Epilogue warp (two warpgroups; group eg drains columns [eg*bn/2, (eg+1)*bn/2) of every tile,
// the warp its TMEM lane quadrant q = rows 32q..32q+31).  Both of a tile's 32-column chunks are
// read from TMEM at once (the buffer goes back to the MMA issuer after one wait), then per
// chunk: this warp's 4 KB of smem (thread = row) -> read back as thread = (row, 4 or 8 channels)
// -> clamp(scale*acc + bias (+ r)) -> 16-byte stores; a chunk's epilogue vectors and residual
// are loaded before its accumulator is needed.  After a tile's stores the warp arrives on the
// tile's publication barrier (stored[j % kQPub] for the CTA's j-th tile) and moves on: the
// publisher warp makes the stores visible at gpu scope and raises the row-block counter, so no
// epilogue warp waits for its stores to reach L2.
template <bool OUT_BF16>
struct ChainEpiChunk;
template <>
struct ChainEpiChunk<true> {   // bf16 y: thread = (rows 8i + sub8, channels col .. col + 7)
  float4 s0, s1, b0, b1;
  uint4 rv[4];
  int col;
  bool col_ok;
  __device__ void load(const ChainGeom& g, int col0, int row0, int lane, int* status) {
    const int sub8 = lane >> 2, c8 = lane & 3;
    col = col0 + 8 * c8;
    col_ok = col < g.Kout;   // Kout % 8 == 0: whole 8-channel groups
    s0 = s1 = b0 = b1 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col_ok) {
      s0 = __ldg(reinterpret_cast<const float4*>(g.scale + col));
      s1 = __ldg(reinterpret_cast<const float4*>(g.scale + col + 4));
      b0 = __ldg(reinterpret_cast<const float4*>(g.bias + col));
      b1 = __ldg(reinterpret_cast<const float4*>(g.bias + col + 4));
    }
    [[maybe_unused]] const size_t total = static_cast<size_t>(g.M) * g.Kout;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      rv[i] = make_uint4(0u, 0u, 0u, 0u);
      const int r = row0 + 8 * i + sub8;
      const size_t e = static_cast<size_t>(r) * g.Kout + col;
      // written by an earlier step of this launch: read through L2 (not the read-only path)
      if (g.res != nullptr && col_ok && r < g.M && CONVF_IN_BOUNDS(e + 8 <= total, status))
        rv[i] = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(g.res) + e));
    }
  }
  __device__ void store(const ChainGeom& g, const float* wst, int row0, int lane, int* status) const {
    const int sub8 = lane >> 2, c8 = lane & 3;
    [[maybe_unused]] const size_t total = static_cast<size_t>(g.M) * g.Kout;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rr = 8 * i + sub8;
      const int r = row0 + rr;
      const float4 x0 = *reinterpret_cast<const float4*>(wst + rr * 32 + (((2 * c8) ^ (rr & 7)) << 2));
      const float4 x1 = *reinterpret_cast<const float4*>(wst + rr * 32 + (((2 * c8 + 1) ^ (rr & 7)) << 2));
      if (!col_ok || r >= g.M) continue;
      const float o[8] = {fmaf(x0.x, s0.x, b0.x), fmaf(x0.y, s0.y, b0.y), fmaf(x0.z, s0.z, b0.z),
                          fmaf(x0.w, s0.w, b0.w), fmaf(x1.x, s1.x, b1.x), fmaf(x1.y, s1.y, b1.y),
                          fmaf(x1.z, s1.z, b1.z), fmaf(x1.w, s1.w, b1.w)};
      const uint32_t rw[4] = {rv[i].x, rv[i].y, rv[i].z, rv[i].w};
      uint32_t pk[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // residual (zero bits when there is none) before the clamp, then RNE to bf16
        const float a0 = fminf(fmaxf(o[2 * j] + __uint_as_float(rw[j] << 16), g.lo), g.hi);
        const float a1 = fminf(fmaxf(o[2 * j + 1] + __uint_as_float(rw[j] & 0xffff0000u), g.lo), g.hi);
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
        pk[j] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      const size_t e = static_cast<size_t>(r) * g.Kout + col;
      if (CONVF_IN_BOUNDS(e + 8 <= total, status))
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(g.y) + e) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
};
template <>
struct ChainEpiChunk<false> {   // fp32 y: thread = (rows 4i + sub, channels col .. col + 3)
  float4 sc, bi;
  float4 rv[8];
  int col;
  bool col_ok;
  __device__ void load(const ChainGeom& g, int col0, int row0, int lane, int* status) {
    const int sub = lane >> 3, c4 = lane & 7;
    col = col0 + 4 * c4;
    col_ok = col < g.Kout;   // Kout % 4 == 0
    sc = bi = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col_ok) {
      sc = __ldg(reinterpret_cast<const float4*>(g.scale + col));
      bi = __ldg(reinterpret_cast<const float4*>(g.bias + col));
    }
    [[maybe_unused]] const size_t total = static_cast<size_t>(g.M) * g.Kout;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      rv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      const int r = row0 + 4 * i + sub;
      const size_t e = static_cast<size_t>(r) * g.Kout + col;
      if (g.res != nullptr && col_ok && r < g.M && CONVF_IN_BOUNDS(e + 4 <= total, status))
        rv[i] = __ldcg(reinterpret_cast<const float4*>(static_cast<const float*>(g.res) + e));
    }
  }
  __device__ void store(const ChainGeom& g, const float* wst, int row0, int lane, int* status) const {
    const int sub = lane >> 3, c4 = lane & 7;
    [[maybe_unused]] const size_t total = static_cast<size_t>(g.M) * g.Kout;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + sub;
      const int r = row0 + rr;
      const float4 a = *reinterpret_cast<const float4*>(wst + rr * 32 + ((c4 ^ (rr & 7)) << 2));
      if (!col_ok || r >= g.M) continue;
      const float4 o = make_float4(fminf(fmaxf(fmaf(a.x, sc.x, bi.x) + rv[i].x, g.lo), g.hi),
                                   fminf(fmaxf(fmaf(a.y, sc.y, bi.y) + rv[i].y, g.lo), g.hi),
                                   fminf(fmaxf(fmaf(a.z, sc.z, bi.z) + rv[i].z, g.lo), g.hi),
                                   fminf(fmaxf(fmaf(a.w, sc.w, bi.w) + rv[i].w, g.lo), g.hi));
      const size_t e = static_cast<size_t>(r) * g.Kout + col;
      if (CONVF_IN_BOUNDS(e + 4 <= total, status)) *reinterpret_cast<float4*>(static_cast<float*>(g.y) + e) = o;
    }
  }
};

// one 32 x 32 fp32 chunk, row `lane` of the accumulator -> smem, 16-byte chunks XOR-swizzled by
// row (both the write and the read-back are conflict-free)
__device__ __forceinline__ void chain_stage_chunk(float* wst, const uint32_t (&v)[32], int lane) {
#pragma unroll
  for (int cc = 0; cc < 8; ++cc)
    *reinterpret_cast<float4*>(wst + lane * 32 + ((cc ^ (lane & 7)) << 2)) =
        make_float4(__uint_as_float(v[4 * cc]), __uint_as_float(v[4 * cc + 1]), __uint_as_float(v[4 * cc + 2]),
                    __uint_as_float(v[4 * cc + 3]));
}

template <bool OUT_BF16, bool PAIR>
__device__ void chain_epilogue(const ChainParams& p, uint8_t* sEpi, uint64_t* tfull, uint64_t* tempty,
                               uint64_t* stored, uint64_t* pubfree, uint32_t tmem_base, uint32_t epoch1,
                               volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int eg = (warp - 3) >> 2;
  const int q = warp & 3;   // TMEM lane quadrant this warp may access
  float* wst = reinterpret_cast<float*>(sEpi + (warp - 3) * kQEpiWarpBytes);
  const ChainStep* steps = p.steps;
  const ChainSched<PAIR> sch;
  ChainCursor cur(steps);
  int acc = 0;
  uint32_t acc_phase = 0;
  int last = -1;
  ChainGeom g;
  uint32_t rtarget = 0;
  int j = 0;   // tiles of this CTA handed to the publisher so far
  for (int t = sch.tstart; t < p.total_tiles; t += sch.tstep) {
    const int L = cur.at(t);
    if (L != last) {
      last = L;
      g = steps[L].g;
      rtarget = epoch1 * static_cast<uint32_t>(kChainArrivals * g.rsrc_nb);
    }
    const int local = t - g.tile0;
    const int mt = local / g.n_blocks;
    const int n0 = (local - mt * g.n_blocks) * g.bn;
    const int m0 = mt * ChainShape<PAIR>::kTileM + sch.rowoff;   // this CTA's first row of the tile
    const int rb = m0 / kQM;                                     // its 128-row block
    const bool rows = m0 < g.M;                                  // a pair's second half may lie past M
    const int row0 = m0 + q * 32;
    const int half = g.bn >> 1;   // this group's columns: 32, 64 or 128
    const int nch = half >> 5;
    const int col0 = n0 + eg * half;
    if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status)) return;
    tc_fence_after();
    if (rows && g.res != nullptr && g.rsrc >= 0) {
      // the residual rows of this tile are the producing step's row block rb (same shape)
      int ok = 1;
      if (lane == 0) ok = chain_wait(g.rsrc_done + rb, rtarget, p.status, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    }
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                           static_cast<uint32_t>(acc * ChainShape<PAIR>::kBNMax + eg * half);
    // chunk pairs: both chunks of a pair read from TMEM at once; after the last pair's reads the
    // buffer goes back to the MMA issuer (the leader's barrier in a CTA pair)
    auto release_tmem = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && sch.crank != 0)
          mbar_arrive_remote(map_to_rank(smem_u32(&tempty[acc]), 0));
        else
          mbar_arrive(&tempty[acc]);
      }
    };
    if constexpr (!PAIR) {
      // at most one pair (128-column tiles): straight-line code, as few registers as possible
      const bool two = nch > 1;
      uint32_t v0[32], v1[32];
      tmem_ld_32x32b_x32(taddr, v0);
      if (two) tmem_ld_32x32b_x32(taddr + 32, v1);
      ChainEpiChunk<OUT_BF16> ch;
      ch.load(g, col0, row0, lane, p.status);
      tmem_ld_wait();
      release_tmem();
      chain_stage_chunk(wst, v0, lane);
      __syncwarp();
      ch.store(g, wst, row0, lane, p.status);
      __syncwarp();   // the chunk's smem reads are done before the next chunk is written
      if (two) {
        ch.load(g, col0 + 32, row0, lane, p.status);
        chain_stage_chunk(wst, v1, lane);
        __syncwarp();
        ch.store(g, wst, row0, lane, p.status);
        __syncwarp();
      }
    } else {
#pragma unroll 1
      for (int c = 0; c < nch; c += 2) {
        const bool two = c + 1 < nch;
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(taddr + 32 * c, v0);
        if (two) tmem_ld_32x32b_x32(taddr + 32 * c + 32, v1);
        ChainEpiChunk<OUT_BF16> ch;
        ch.load(g, col0 + 32 * c, row0, lane, p.status);
        tmem_ld_wait();
        if (c + 2 >= nch) release_tmem();
        chain_stage_chunk(wst, v0, lane);
        __syncwarp();
        ch.store(g, wst, row0, lane, p.status);
        __syncwarp();
        if (two) {
          ch.load(g, col0 + 32 * c + 32, row0, lane, p.status);
          chain_stage_chunk(wst, v1, lane);
          __syncwarp();
          ch.store(g, wst, row0, lane, p.status);
          __syncwarp();
        }
      }
    }
    // the tile is stored: hand it to the publisher (once it has taken the slot's previous tile),
    // unless no later step reads this step's output
    if (g.consumed && rows) {
      if (lane == 0) {
        const int slot = j % kQPub;
        const bool ok = j < kQPub ||
                        mbar_wait(&pubfree[slot], static_cast<uint32_t>((j / kQPub - 1) & 1), abort_flag, p.status);
        if (ok) mbar_arrive(&stored[slot]);
      }
      ++j;
    }
    if (++acc == ChainShape<PAIR>::kAcc) {
      acc = 0;
      acc_phase ^= 1;
    }
  }
}

// Publisher (one thread): for each of the CTA's tiles whose step's output a later step reads,
// in order, once all eight epilogue warps have arrived (their stores ordered before their
// arrivals), a gpu-scope fence makes those stores visible -- the fence is cumulative over what
// the barrier let this thread observe -- and the counter of the CTA's 128-row block of the tile
// is raised by one.  (Sharing one fence among tiles already stored when their turn comes saved
// nothing on the independent steps and delayed the dependent ones' consumers: one fence per
// tile.)
template <bool PAIR>
__device__ void chain_publisher(const ChainParams& p, uint64_t* stored, uint64_t* pubfree, volatile int* abort_flag) {
  const ChainStep* steps = p.steps;
  const ChainSched<PAIR> sch;
  ChainCursor cur(steps);
  int last = -1, tile0 = 0, nb = 1, M = 0;
  bool consumed = false;
  uint32_t* done = nullptr;
  int j = 0;
  for (int t = sch.tstart; t < p.total_tiles; t += sch.tstep) {
    const int L = cur.at(t);
    if (L != last) {
      last = L;
      tile0 = steps[L].g.tile0;
      nb = steps[L].g.n_blocks;
      done = steps[L].g.done;
      M = steps[L].g.M;
      consumed = steps[L].g.consumed != 0;
    }
    const int m0 = ((t - tile0) / nb) * ChainShape<PAIR>::kTileM + sch.rowoff;
    if (!consumed || m0 >= M) continue;
    const int slot = j % kQPub;
    if (!mbar_wait(&stored[slot], static_cast<uint32_t>((j / kQPub) & 1), abort_flag, p.status)) return;
    fence_acq_rel_gpu();
    fence_proxy_async_global();   // ... and ordered before later async-proxy (TMA) reads of them
    red_relaxed_gpu_add(done + m0 / kQM, 1u);
    mbar_arrive(&pubfree[slot]);
    ++j;
  }
}

template <bool OUT_BF16, bool PAIR>
__global__ void __launch_bounds__(kQThreads, 1) tc_chain_kernel(const ChainParams p) {
  constexpr uint32_t kTmemCols = ChainShape<PAIR>::kAcc * ChainShape<PAIR>::kBNMax;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kQSlots * kQATile;
  uint8_t* sEpi = sB + kQSlots * kQBTile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + 8 * kQEpiWarpBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kQSteps;
  uint64_t* tfull = bars + 2 * kQSteps;
  uint64_t* tempty = tfull + 4;        // tfull, tempty: [kAcc <= 4] per accumulator
  uint64_t* stored = tempty + 4;       // [kQPub] a tile's stores are done (eight epilogue warps)
  uint64_t* pubfree = stored + kQPub;  // [kQPub] the publisher has taken the slot's tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pubfree + kQPub);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* epoch_slot = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQSteps; ++s) {
      mbar_init(&full[s], 2);    // activation producer + weight producer (the leader's, in a pair)
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < ChainShape<PAIR>::kAcc; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], PAIR ? 16 : 8);  // every epilogue warp (of both CTAs of a pair)
    }
    for (int b = 0; b < kQPub; ++b) {
      mbar_init(&stored[b], 8);  // every epilogue warp
      mbar_init(&pubfree[b], 1); // the publisher
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();   // the peer's barriers and TMEM exist before any cross-CTA operation
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // the next kernel may launch once every CTA of this grid has started (so none of this
  // grid's CTAs can be kept from an SM by it: the CTAs wait for one another's tiles)
  pdl_launch_dependents();
  // The first tile's operands start towards L2 behind the previous kernel's tail: its weight
  // boxes, and its input rows when no step of this chain writes them (a prefetch reads no stale
  // data: whatever the previous kernel still writes lands in L2, which serves every read after
  // the wait).
  if (lane == 0 && (warp == 0 || warp == 2)) {
    const ChainSched<PAIR> sch;
    const int t = sch.tstart;
    int L = 0;
    while (t >= p.steps[L].g.tile_end) ++L;
    const ChainGeom& g = p.steps[L].g;
    const int local = t - g.tile0;
    const int mt = local / g.n_blocks;
    const int m0 = mt * ChainShape<PAIR>::kTileM + sch.rowoff;
    if (warp == 2) {
      const int brows = PAIR ? g.bn / 2 : g.bn;
      tma_prefetch_desc(&p.steps[L].tmB);
      for (int kb = 0; kb < min(g.num_kb, 4); kb += 2)
        tma_prefetch_l2_3d(&p.steps[L].tmB, 0, (local - mt * g.n_blocks) * g.bn + static_cast<int>(sch.crank) * brows,
                           kb);
    } else if (g.src < 0 && m0 < g.M) {
      tma_prefetch_desc(&p.steps[L].tmA);
      int lo, hi;
      chain_input_rows(g, m0, lo, hi);
      bulk_prefetch_l2(static_cast<const uint16_t*>(g.x) + static_cast<size_t>(lo) * g.C,
                       static_cast<uint32_t>(hi - lo + 1) * g.C * 2);
    }
  }
  pdl_wait_prior();
  if (threadIdx.x == 0) *epoch_slot = *reinterpret_cast<volatile uint32_t*>(p.state);
  __syncthreads();
  const uint32_t epoch1 = *epoch_slot + 1u;
  const bool leader = !PAIR || cluster_ctarank() == 0;

  if (warp == 0) {
    if (lane == 0) chain_producer<0, PAIR>(p, sA, sB, full, empty, epoch1, abort_flag);
  } else if (warp == 2) {
    if (lane == 0) chain_producer<2, PAIR>(p, sA, sB, full, empty, epoch1, abort_flag);
  } else if (warp == 1) {
    if (lane == 0 && leader) chain_mma<PAIR>(p, sA, sB, full, empty, tfull, tempty, tmem_base, abort_flag);
  } else if (warp == 11) {
    if (lane == 0) chain_publisher<PAIR>(p, stored, pubfree, abort_flag);
  } else {
    chain_epilogue<OUT_BF16, PAIR>(p, sEpi, tfull, tempty, stored, pubfree, tmem_base, epoch1, abort_flag);
  }

  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) {
    // a wait ran out: give copies and MMAs already in flight time to land before TMEM is freed
    for (int i = 0; i < 2000; ++i) __nanosleep(100000);
  }
  __syncthreads();
  if (PAIR) cluster_sync();   // no CTA of a pair leaves while the other may still signal it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // the last CTA out advances the epoch (or, after an error, restarts the counters at zero)
    __threadfence();
    const uint32_t prev = atomicAdd(p.state + 1, 1u);
    if (prev == gridDim.x - 1) {
      __threadfence();
      if (*reinterpret_cast<volatile int*>(p.status) != 0) {
        for (int i = 0; i < p.total_mtiles; ++i) p.counters[i] = 0u;
        p.state[0] = 0u;
      } else {
        p.state[0] = epoch1;
      }
      p.state[1] = 0u;
      __threadfence();
    }
  }
}

template <bool OUT_BF16, bool PAIR>
cudaError_t chain_configure() {
  static cudaError_t e = [] {
    cudaError_t r = cudaFuncSetAttribute(tc_chain_kernel<OUT_BF16, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kQSmem);
    if (r == cudaSuccess && PAIR)
      r = cudaFuncSetAttribute(tc_chain_kernel<OUT_BF16, PAIR>, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    return r;
  }();
  return e;
}

template <bool OUT_BF16, bool PAIR>
cudaError_t chain_launch(const ChainParams& p, int grid, cudaStream_t stream) {
  const cudaError_t e = chain_configure<OUT_BF16, PAIR>();
  if (e != cudaSuccess) return e;
  return launch_pdl(tc_chain_kernel<OUT_BF16, PAIR>, dim3(grid), dim3(kQThreads), kQSmem, stream, PAIR ? 2 : 1, p);
}

// CTAs that can be resident at once: one per SM, or (pairs) two per co-resident cluster
template <bool OUT_BF16, bool PAIR>
int chain_max_ctas(int num_sms) {
  if (chain_configure<OUT_BF16, PAIR>() != cudaSuccess) return 0;
  if (!PAIR) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tc_chain_kernel<OUT_BF16, PAIR>, kQThreads, kQSmem) !=
        cudaSuccess)
      return 0;
    return n * num_sms;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = kQSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, tc_chain_kernel<OUT_BF16, PAIR>, &cfg) != cudaSuccess) return 0;
  return 2 * clusters;
}

}  // namespace

cudaError_t launch_tc_chain(const ChainParams& p, bool out_bf16, bool pair, int grid, cudaStream_t stream) {
  if (pair) return out_bf16 ? chain_launch<true, true>(p, grid, stream) : chain_launch<false, true>(p, grid, stream);
  return out_bf16 ? chain_launch<true, false>(p, grid, stream) : chain_launch<false, false>(p, grid, stream);
}

int tc_chain_max_ctas(bool out_bf16, bool pair, int num_sms) {
  if (pair) return out_bf16 ? chain_max_ctas<true, true>(num_sms) : chain_max_ctas<false, true>(num_sms);
  return out_bf16 ? chain_max_ctas<true, false>(num_sms) : chain_max_ctas<false, false>(num_sms);
}

}  // namespace convf
