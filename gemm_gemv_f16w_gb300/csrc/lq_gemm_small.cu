// The prefill GEMM for a few rows of A (M = 2..48): C = A W^T on the tensor
// cores with warp-level MMAs, every weight read from HBM once.
//
// For so few tokens the weight stream sets the pace, as in the decode GEMV,
// and the tcgen05 kernel (lq_gemm_tma.cu) spends most of a call on fixed
// costs: the TMEM allocation, a K split over clusters of CTAs and the
// reduction of their partial tiles, and the MMA pipeline's fill and drain.
// This kernel keeps everything in registers instead:
//
//  * one CTA per SM owns a contiguous range of W rows (at most 128), streamed
//    as stages of two 256-K pieces through a ring in shared memory by TMA
//    tensor copies (a piece: Q8_0 / Q4_0 one box of the rows' 272 / 144
//    bytes of that K; f16 four 128-byte-swizzled boxes of 64 halves), the
//    first stages' weights issued at kernel start (weights depend on nothing);
//  * each stage also holds the same K of A (the M rows, f32, one box a
//    piece), copied once the previous kernel on the stream has completed;
//    the lanes round their A values to bf16 (nearest even) as they build the
//    MMA operands (rows of the MMA past M are zeros);
//  * warp w takes block w % 8 (32 K) of piece w / 8 of every stage, for
//    every 8-row tile of the CTA, two tiles at a time: each lane dequantises
//    8 weights of one row (lane / 4) exactly in f32 and rounds them once to
//    bf16, the same operand as the tcgen05 kernel's, and two mma.m16n8k16
//    (bf16 x bf16 -> f32; A = 16 tokens, B = 8 W rows) add the block to the
//    tile's accumulator, for each group of 16 tokens (more than 16 rows of
//    A: two or three groups share every converted weight, for CTAs of at
//    most 64 or 48 W rows, whose accumulators fit in registers; where two
//    pieces' A rows and weights do not fit twice in shared memory, stages of
//    one piece, its 8 block positions shared by the warps' two halves, each
//    taking every other tile pair). Within a block lane q =
//    lane % 4 takes 8 codes (f16
//    elements 8q .. 8q+7; Q8_0 codes 4q .. 4q+3 and 16+4q .. 19+4q; Q4_0 the
//    low and high nibbles of bytes 4q .. 4q+3, the same codes), so the MMA's
//    K order is a fixed permutation of the block, and each lane reads the A
//    values of the same positions;
//  * after the last stage the 16 block positions' partial tiles are added in
//    a fixed order through shared memory and C (plus R with the residual
//    epilogue) is stored.
//
// The tolerance is the tensor-core route's (A and W rounded to bf16, f32
// accumulation). Every wait is bounded (LQ_ERR_DEVICE_TIMEOUT on expiry).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "lq_device.cuh"
#include "lq_epilogue.cuh"
#include "lq_internal.h"
#include "lq_tcgen05.cuh"

namespace lq {
namespace {

__device__ unsigned g_small_err;
__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_small_err, 0u, code); }

constexpr int kSWarps = 16, kSThreads = kSWarps * 32;
constexpr int kSPos = 16;  // block positions of a two-piece stage (8 blocks x 2 pieces)
constexpr int kPieceK = 256;      // K of one weight stage: 8 blocks of 32
constexpr int kSMaxStages = 8;
constexpr int kSMaxTiles = 16;    // 8-row W tiles of a CTA (128 rows)
constexpr int kSTokens = 16;      // the MMA's M: rows of A, zero-padded
constexpr int kSMaxM = 48;        // up to three token groups of 16 share every converted weight
constexpr int kSMaxPairs2 = 4;    // tile pairs a CTA with two token groups (64 W rows)
constexpr int kSMaxPairs3 = 3;    // with three (48 W rows: more lost to the tcgen05 kernel)

// Bytes of one W row's 256 K in a stage.
__host__ __device__ constexpr int piece_row_bytes(int fmt) {
  return fmt == LQ_FMT_F16 ? 512 : (fmt == LQ_FMT_Q8_0 ? 272 : 144);
}

// pieces a stage (the last stage may hold fewer): 2, or 1 where two pieces'
// A rows and weights would not fit twice in shared memory (M > 32; f16 at
// M = 25..32 on wide CTAs)
constexpr unsigned kARowBytes = kPieceK * 4;  // one row of A in a piece: 256 f32

struct SmallParams {
  float* C;
  const float* R;       // residual epilogue: added to every output
  int M, N, K;
  int rows_box;         // W rows of a stage (the copy's box), at most 128
  int stages;           // ring depth
  unsigned w_bytes;     // weight bytes of a piece (the copy's box)
  unsigned w_pitch;     // their space in the slot (a multiple of 128)
  unsigned slot_bytes;  // ring slot: A of its pieces (M rows each), then their weights; a multiple of 1024
  unsigned ring_bytes;  // ring (reused for the partial tiles at the end)
  unsigned long long wait_ns;
  unsigned wait_iters;
};

struct SmallBars {
  uint64_t full[kSMaxStages];  // the stage's bytes landed
  int done[kSMaxStages];       // warps finished with the slot's current stage
  int last[kSMaxStages];       // last stage issued into each slot (-1: none)
  volatile int abort;
};
constexpr int kSBarsBytes = 256;
static_assert(sizeof(SmallBars) <= kSBarsBytes, "barrier block");

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The lane's 8 weights of W row `row` (of the stage), block bp, as four bf16
// pairs in the MMA's K order: f16 elements 8q .. 8q+7; Q8_0 codes 8q ..
// 8q+7, or with BIG (more than 8 rows of A) codes 4q .. 4q+3 and 16+4q ..
// 19+4q; Q4_0 the low nibbles of bytes 4q .. 4q+3 (the same codes), then
// their high nibbles. Reading words q (and q + 4) of a row's codes, the 32
// lanes hit 32 different banks (rows 68 or 36 words apart, 4 banks); BIG
// Q8_0 does so at the cost of a fourth load for unaligned blocks, which only
// pays when the A loads are conflict-free too. Each weight is formed exactly in f32
// (an f16 widened; d * q, or d * (q - 8), from the code placed in the
// mantissa of 2^23 by one byte-permute and one exact packed add) and rounded
// once to bf16 (nearest even).
template <int FMT, bool BIG>
__device__ __forceinline__ void load_weights(uint32_t stage, int rows_box, int row, int bp, int q,
                                             uint32_t (&bw)[4]) {
  if constexpr (FMT == LQ_FMT_F16) {
    // box bp / 2: rows x 128 bytes, 16-byte chunk c of row r at chunk c ^ (r % 8)
    const uint32_t c = static_cast<uint32_t>((bp & 1) * 4 + q) ^ static_cast<uint32_t>(row & 7);
    const uint4 v = lds128(stage + static_cast<uint32_t>((bp >> 1) * rows_box * 128 + row * 128) + (c << 4));
    const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
      bw[j] = pack_bf16x2(f.x, f.y);
    }
  } else if constexpr (FMT == LQ_FMT_Q8_0) {
    // block bp at byte 34 bp of the row's 272: scale, then 32 codes; even
    // blocks' codes start 2 bytes into a word, odd blocks' on a word
    const uint32_t rowa = stage + static_cast<uint32_t>(row) * 272u;
    const bool mis = (bp & 1) == 0;
    const uint32_t sh = mis ? 16u : 0u;
    uint32_t x0, x1;  // four codes each, sign bits flipped
    if constexpr (BIG) {
      // codes 4q .. 4q+3 and 16+4q .. 19+4q: words q (and q + 1) and q + 4
      // (q + 5) of the codes, one bank each (four loads when unaligned)
      const uint32_t o = 34u * static_cast<uint32_t>(bp) + 2u + 4u * static_cast<uint32_t>(q);
      const uint32_t wa = rowa + (o & ~3u);
      const uint32_t w0 = lds32(wa), w1 = mis ? lds32(wa + 4u) : 0u;
      const uint32_t w4 = lds32(wa + 16u), w5 = mis ? lds32(wa + 20u) : 0u;
      x0 = __funnelshift_r(w0, w1, sh) ^ 0x80808080u;
      x1 = __funnelshift_r(w4, w5, sh) ^ 0x80808080u;
    } else {
      // codes 8q .. 8q+7: three words (two when aligned), two lanes a bank
      const uint32_t o = 34u * static_cast<uint32_t>(bp) + 2u + 8u * static_cast<uint32_t>(q);
      const uint32_t wa = rowa + (o & ~3u);
      const uint32_t w0 = lds32(wa), w1 = lds32(wa + 4u), w2 = mis ? lds32(wa + 8u) : 0u;
      x0 = __funnelshift_r(w0, w1, sh) ^ 0x80808080u;
      x1 = __funnelshift_r(w1, w2, sh) ^ 0x80808080u;
    }
    const uint32_t dw = lds32(rowa + ((34u * static_cast<uint32_t>(bp)) & ~3u));
    const float d = f16_lo(mis ? dw : (dw >> 16));
    const float2 dd = make_float2(d, d), mb = make_float2(-kMagicS8, -kMagicS8);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x = j < 2 ? x0 : x1;
      const int i = 2 * (j & 1);
      const float2 w = fmul2(fadd2(make_float2(s8_to_magic(x, i), s8_to_magic(x, i + 1)), mb), dd);
      bw[j] = pack_bf16x2(w.x, w.y);
    }
  } else {
    // block bp at byte 18 bp of the row's 144: scale, then 16 bytes of
    // nibbles (byte j: code j low, code j + 16 high)
    const uint32_t rowa = stage + static_cast<uint32_t>(row) * 144u;
    const bool mis = (bp & 1) == 0;
    const uint32_t o = 18u * static_cast<uint32_t>(bp) + 2u + 4u * static_cast<uint32_t>(q);
    const uint32_t wa = rowa + (o & ~3u);
    const uint32_t w0 = lds32(wa), w1 = mis ? lds32(wa + 4u) : 0u;
    const uint32_t x = __funnelshift_r(w0, w1, mis ? 16u : 0u);  // bytes 4q .. 4q+3
    const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
    const uint32_t dw = lds32(rowa + ((18u * static_cast<uint32_t>(bp)) & ~3u));
    const float d = f16_lo(mis ? dw : (dw >> 16));
    const float2 dd = make_float2(d, d), m8 = make_float2(-kMagicQ4, -kMagicQ4);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t x2 = j < 2 ? lo : hi;
      const int i = 2 * (j & 1);
      const float2 w = fmul2(fadd2(make_float2(s8_to_magic(x2, i), s8_to_magic(x2, i + 1)), m8), dd);
      bw[j] = pack_bf16x2(w.x, w.y);
    }
  }
}

// The lane's A values of token row `row` (0..15) for block bp of a stage, in
// the order of its weights (elements 8q .. 8q+7 of the block, 16-byte
// chunks 2q and 2q+1; Q4_0, and Q8_0 with BIG: 4q .. 4q+3 and 16+4q ..
// 19+4q, chunks q and 4+q), as four bf16 pairs (nearest even). The piece's
// A is M rows of 256 values (1 KB each), so every row's chunk c sits in the
// same banks and a quarter-warp's eight lanes, two rows, read each bank
// twice. With BIG the odd row reads its two chunks in the other order (the
// first load of all eight lanes then covers the 32 banks once); with 8 rows
// or fewer the swap measured slower (Q8_0 M=8 2048x2048 4.24 against 3.73
// us). (One box a stage: eight 128-byte-swizzled boxes issued eight times as
// many copies and measured slower.)
template <int FMT, bool BIG>
__device__ __forceinline__ void load_a(uint32_t sa, int row, int M, int bp, int q, uint32_t (&a)[4]) {
  const uint32_t rbase = sa + static_cast<uint32_t>(row * 1024 + bp * 128);
  const bool quarters = FMT == LQ_FMT_Q4_0 || (FMT == LQ_FMT_Q8_0 && BIG);
  const uint32_t c0 = quarters ? q : 2 * q, c1 = quarters ? 4 + q : 2 * q + 1;
  const bool odd = BIG && (row & 1) != 0;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 x = row < M ? lds128f(rbase + ((odd ? c1 : c0) << 4)) : z;  // rows past M: zeros (not in the slot)
  const float4 y = row < M ? lds128f(rbase + ((odd ? c0 : c1) << 4)) : z;
  const uint32_t p0 = pack_bf16x2(x.x, x.y), p1 = pack_bf16x2(x.z, x.w);
  const uint32_t p2 = pack_bf16x2(y.x, y.y), p3 = pack_bf16x2(y.z, y.w);
  a[0] = odd ? p2 : p0;
  a[1] = odd ? p3 : p1;
  a[2] = odd ? p0 : p2;
  a[3] = odd ? p1 : p3;
}

// NP: pairs of 8-row tiles a CTA (its T tiles, 2 NP - 1 <= T <= 2 NP), so the
// tile loop is unrolled without branches. BIG: more than 8 rows of A
// (otherwise the MMA's rows 8..15 are zeros, never loaded). TG: groups of 16
// tokens (rows 16 tg ..), each weight pair converted once and multiplied with
// every group. PPS: pieces a stage. With 2, warp w takes block w % 8 of piece
// w / 8 for every pair; with 1, block w % 8 of the piece for the pairs w / 8,
// w / 8 + 2, ... (half of them: fewer accumulators, A loaded a group at a
// time), and a tile's partial sums come from 8 positions instead of 16.
template <int FMT, int EPI, int NP, bool BIG, int TG, int PPS>
__global__ void __launch_bounds__(kSThreads, 1)
    gemm_small_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                      const SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);  // 1024-aligned (swizzled boxes)
  SmallBars& b = *reinterpret_cast<SmallBars*>(ring + p.ring_bytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.stages, npieces = p.K / kPieceK, nstages = (npieces + PPS - 1) / PPS;
  const int r0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.N / gridDim.x);
  const int nrows = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.N / gridDim.x) - r0;
  const int T = (nrows + 7) / 8;  // 8-row tiles

  // stage st (pieces PPS st .. PPS st + PPS - 1) into ring slot `slot`: the
  // weights, then (once the previous kernel has completed) A; one barrier
  // counts both. Slot layout: A of piece 0, A of piece 1, W of piece 0, W of
  // piece 1.
  auto issue_w = [&](int st, int slot) {
    const int np = min(PPS, npieces - PPS * st);
    mbar_arrive_expect_tx(&b.full[slot], static_cast<unsigned>(np) * (p.w_bytes + static_cast<unsigned>(p.M) * kARowBytes));
    for (int sp = 0; sp < np; ++sp) {
      const int piece = PPS * st + sp;
      uint8_t* dst = ring + static_cast<size_t>(slot) * p.slot_bytes + PPS * p.M * kARowBytes + sp * p.w_pitch;
      if constexpr (FMT == LQ_FMT_F16) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          tc::tma_load_2d(dst + i * p.rows_box * 128, &tmW, kPieceK * piece + 64 * i, r0, &b.full[slot]);
      } else {
        tc::tma_load_3d(dst, &tmW, 0, piece, r0, &b.full[slot]);
      }
    }
    b.last[slot] = st;
  };
  auto issue_a = [&](int st, int slot) {
    const int np = min(PPS, npieces - PPS * st);
    for (int sp = 0; sp < np; ++sp)
      tc::tma_load_2d(ring + static_cast<size_t>(slot) * p.slot_bytes + sp * p.M * kARowBytes, &tmA,
                      kPieceK * (PPS * st + sp), 0, &b.full[slot]);
  };
  const int first = min(S, nstages);
  if (threadIdx.x == 0) {
    for (int k = 0; k < S; ++k) {
      mbar_init(&b.full[k], 1);
      b.done[k] = 0;
      b.last[k] = -1;
    }
    b.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  // the first stages' copies from two threads at once: the weights (they
  // depend on nothing) and, once the previous kernel on the stream has
  // completed, A (a slot's barrier may see A's bytes land before the
  // weights' thread has announced them: the transaction count dips below
  // zero and the phase still completes only after that announcement)
  if (threadIdx.x == 0) {
    tc::prefetch_tmap(&tmW);
    for (int j = 0; j < first; ++j) issue_w(j, j);
  } else if (threadIdx.x == 32) {
    tc::prefetch_tmap(&tmA);
    pdl_wait();
    for (int j = 0; j < first; ++j) issue_a(j, j);
  }
  pdl_wait();  // (C and R)

  // ---- main loop: warp w takes block w % 8 of piece w / 8 of each stage,
  // for every tile, two tiles at a time (PPS 2; PPS 1: block w % 8 of the
  // piece, pairs w / 8, w / 8 + 2, ...), each pair an independent chain of
  // loads, conversions and MMAs; lane (g, q): W row 8t + wr, its 8 codes,
  // and the A values of tokens 16 tg + g and 16 tg + g + 8 in the same order
  const int bp = warp & 7, sp = PPS == 2 ? warp >> 3 : 0, half = warp >> 3, g = lane >> 2, q = lane & 3;
  // f16: MMA column g of a tile is W row wr = g / 2 + 4 (g % 2) of it, so
  // the two rows a quarter-warp reads sit in different halves of the boxes'
  // 128-byte swizzle (conflict-free 16-byte loads: f16 M=16 6144x2048 6.89
  // -> 6.66 us; the block formats keep column g = row g, measured 1 % ahead)
  const int wr = FMT == LQ_FMT_F16 ? (g >> 1) + 4 * (g & 1) : g;
  constexpr int NPA = PPS == 2 ? NP : (NP + 1) / 2;  // pairs a warp
  float acc[2 * NPA][TG][4];
#pragma unroll
  for (int i = 0; i < 2 * NPA; ++i)
#pragma unroll
    for (int j = 0; j < 4 * TG; ++j) acc[i][j >> 2][j & 3] = 0.f;
  int s = 0;
  uint32_t ph = 0;
#pragma unroll 1
  for (int st = 0; st < nstages; ++st) {
    const bool ok = mbar_wait(&b.full[s], ph, p.wait_ns, p.wait_iters);
    if (!__all_sync(0xffffffffu, ok) || b.abort) {
      if (lane == 0) {
        record_error(kDevErrTimeout);
        b.abort = 1;
      }
      break;
    }
    if (PPS * st + sp < npieces) {
      const uint32_t slot = smem_u32(ring) + static_cast<uint32_t>(s) * p.slot_bytes;
      const uint32_t sa = slot + static_cast<uint32_t>(sp * p.M) * kARowBytes;
      const uint32_t wst = slot + static_cast<uint32_t>(PPS * p.M) * kARowBytes + static_cast<uint32_t>(sp) * p.w_pitch;
      uint32_t alo[PPS == 2 ? TG : 1][4], ahi[PPS == 2 ? TG : 1][4];
      if constexpr (PPS == 2) {
#pragma unroll
        for (int tg = 0; tg < TG; ++tg) {
          load_a<FMT, BIG>(sa, 16 * tg + g, p.M, bp, q, alo[tg]);
          if constexpr (BIG)
            load_a<FMT, BIG>(sa, 16 * tg + g + 8, p.M, bp, q, ahi[tg]);
          else
            ahi[tg][0] = ahi[tg][1] = ahi[tg][2] = ahi[tg][3] = 0u;
        }
      }
#pragma unroll
      for (int m = 0; m < NPA; ++m) {
        const int pr = PPS == 2 ? m : half + 2 * m;  // the pair
        if (PPS == 1 && pr >= NP) break;
        // with an odd tile count the last pair repeats its first tile into
        // the second accumulator; a CTA with fewer rows than the largest
        // computes its pairs past T on bytes of the ring or its tail;
        // neither is ever stored
        const int t0 = 2 * pr, t1 = min(t0 + 1, T - 1);
        uint32_t b0[4], b1[4];
        load_weights<FMT, BIG>(wst, p.rows_box, 8 * t0 + wr, bp, q, b0);
        load_weights<FMT, BIG>(wst, p.rows_box, 8 * t1 + wr, bp, q, b1);
#pragma unroll
        for (int tg = 0; tg < TG; ++tg) {
          uint32_t al[4], ah[4];
          if constexpr (PPS == 2) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              al[j] = alo[tg][j];
              ah[j] = ahi[tg][j];
            }
          } else {
            load_a<FMT, BIG>(sa, 16 * tg + g, p.M, bp, q, al);
            if constexpr (BIG)
              load_a<FMT, BIG>(sa, 16 * tg + g + 8, p.M, bp, q, ah);
            else
              ah[0] = ah[1] = ah[2] = ah[3] = 0u;
          }
          mma_bf16_16816(acc[2 * m][tg], al[0], ah[0], al[1], ah[1], b0[0], b0[1]);  // the lane's values 0 .. 3
          mma_bf16_16816(acc[2 * m + 1][tg], al[0], ah[0], al[1], ah[1], b1[0], b1[1]);
          mma_bf16_16816(acc[2 * m][tg], al[2], ah[2], al[3], ah[3], b0[2], b0[3]);  // values 4 .. 7
          mma_bf16_16816(acc[2 * m + 1][tg], al[2], ah[2], al[3], ah[3], b1[2], b1[3]);
        }
      }
    }
    // The last warp done with the slot refills it (every warp's reads of it
    // have returned: their values went into the MMAs above).
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&b.done[s], 1) == kSWarps - 1) {
        b.done[s] = 0;
        if (st + S < nstages) {
          fence_proxy_async_smem();  // the generic reads above, before the copies' writes
          issue_w(st + S, s);
          issue_a(st + S, s);
        }
      }
    }
    if (++s == S) {
      s = 0;
      ph ^= 1u;
    }
  }
  __syncthreads();
  if (b.abort) {
    // no copy may still be in flight when the CTA exits
    if (threadIdx.x == 0)
      for (int k = 0; k < S; ++k)
        if (b.last[k] >= 0) mbar_wait(&b.full[k], static_cast<uint32_t>(b.last[k] / S) & 1u, kDrainWaitNs);
    return;
  }

  // ---- the block positions' partial tiles (16, or 8 with PPS 1), added in
  // a fixed order (shared memory of the ring, every stage consumed):
  // red[t][position][m][n], 16 TG tokens x 8 columns a tile
  constexpr int kTileF = 128 * TG;
  constexpr int kNPos = 8 * PPS;
  const int pos = PPS == 2 ? warp : bp;
  float* red = reinterpret_cast<float*>(ring);
#pragma unroll
  for (int m = 0; m < NPA; ++m) {
    const int pr = PPS == 2 ? m : half + 2 * m;
    if (PPS == 1 && pr >= NP) break;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int t = 2 * pr + h2;
      if (t < T) {
        float* tile = red + (t * kNPos + pos) * kTileF;
        const int a = 2 * m + h2;
#pragma unroll
        for (int tg = 0; tg < TG; ++tg) {
          *reinterpret_cast<float2*>(tile + (16 * tg + g) * 8 + 2 * q) = make_float2(acc[a][tg][0], acc[a][tg][1]);
          *reinterpret_cast<float2*>(tile + (16 * tg + g + 8) * 8 + 2 * q) =
              make_float2(acc[a][tg][2], acc[a][tg][3]);
        }
      }
    }
  }
  __syncthreads();
#pragma unroll 1
  for (int idx = threadIdx.x; idx < T * kTileF; idx += kSThreads) {
    const int t = idx / kTileF, e = idx - t * kTileF, mrow = e >> 3, c = e & 7;  // c: MMA column
    const int n = 8 * t + (FMT == LQ_FMT_F16 ? (c >> 1) + 4 * (c & 1) : c);
    if (mrow < p.M && n < nrows && LQ_IN_BOUNDS(r0 + n < p.N)) {
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < kNPos; ++k) sum += red[(t * kNPos + k) * kTileF + e];
      const long long o = static_cast<long long>(mrow) * p.N + r0 + n;
      if constexpr (EPI == epi::kResidual)
        p.C[o] = sum + p.R[o];
      else
        p.C[o] = sum;
    }
  }
}

template <int FMT, int EPI, int NP, bool BIG, int TG, int PPS>
lq_status launch_small_k(const MatmulArgs& a, const CUtensorMap& tw, const CUtensorMap& ta, const SmallParams& p,
                         int G, size_t smem) {
  auto kern = gemm_small_kernel<FMT, EPI, NP, BIG, TG, PPS>;
  static int configured[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_CUDA;
  if (!configured[dev]) {
    const int mx = std::min(device_info().max_smem_optin, 227 * 1024);
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e != cudaSuccess) return cuda_status(e);
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G));
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tw, ta, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

template <int FMT, int EPI, int NP>
lq_status launch_small_t(const MatmulArgs& a, const CUtensorMap& tw, const CUtensorMap& ta, const SmallParams& p,
                         int G, size_t smem, int pps) {
  const int tg = (p.M + kSTokens - 1) / kSTokens;
  if (tg > 1) {
    // two or three token groups: the accumulators of up to 4 tile pairs
    // (3 with three groups; half of them a warp with single-piece stages)
    // fit the 128 registers of 512 threads (the plan refuses more). Four
    // groups spilled and lost to the tcgen05 kernel (Q8_0 6144x2048 M = 64
    // 14.9 against 14.2 us); three on 64-row CTAs too (8192x2048 M = 33
    // 14.7 against 14.2).
    if constexpr (NP <= kSMaxPairs2) {
      if (pps == 2) return tg == 2 ? launch_small_k<FMT, EPI, NP, true, 2, 2>(a, tw, ta, p, G, smem) : LQ_ERR_UNSUPPORTED;
      if (tg == 2) return launch_small_k<FMT, EPI, NP, true, 2, 1>(a, tw, ta, p, G, smem);
      if constexpr (NP <= kSMaxPairs3)
        if (tg == 3) return launch_small_k<FMT, EPI, NP, true, 3, 1>(a, tw, ta, p, G, smem);
      return LQ_ERR_UNSUPPORTED;
    }
    return LQ_ERR_UNSUPPORTED;
  }
  if (pps != 2) return LQ_ERR_UNSUPPORTED;
  return p.M > 8 ? launch_small_k<FMT, EPI, NP, true, 1, 2>(a, tw, ta, p, G, smem)
                 : launch_small_k<FMT, EPI, NP, false, 1, 2>(a, tw, ta, p, G, smem);
}

// the kernel for the CTAs' tile count: the largest CTA holds ceil(N / G)
// rows, ceil(rows / 8) tiles, NP = ceil(tiles / 2) pairs
template <int FMT, int EPI>
lq_status launch_small_np(const MatmulArgs& a, const CUtensorMap& tw, const CUtensorMap& ta, const SmallParams& p,
                          int G, size_t smem, int pps) {
  const int rows = static_cast<int>((static_cast<long long>(p.N) + G - 1) / G);
  switch ((rows + 15) / 16) {
    case 1: return launch_small_t<FMT, EPI, 1>(a, tw, ta, p, G, smem, pps);
    case 2: return launch_small_t<FMT, EPI, 2>(a, tw, ta, p, G, smem, pps);
    case 3: return launch_small_t<FMT, EPI, 3>(a, tw, ta, p, G, smem, pps);
    case 4: return launch_small_t<FMT, EPI, 4>(a, tw, ta, p, G, smem, pps);
    case 5: return launch_small_t<FMT, EPI, 5>(a, tw, ta, p, G, smem, pps);
    case 6: return launch_small_t<FMT, EPI, 6>(a, tw, ta, p, G, smem, pps);
    case 7: return launch_small_t<FMT, EPI, 7>(a, tw, ta, p, G, smem, pps);
    case 8: return launch_small_t<FMT, EPI, 8>(a, tw, ta, p, G, smem, pps);
    default: return LQ_ERR_UNSUPPORTED;
  }
}

template <int FMT>
lq_status launch_small_fmt(const MatmulArgs& a, const CUtensorMap& tw, const CUtensorMap& ta, const SmallParams& p,
                           int G, size_t smem, int pps) {
  if (a.epi == epi::kResidual) return launch_small_np<FMT, epi::kResidual>(a, tw, ta, p, G, smem, pps);
  return launch_small_np<FMT, epi::kPlain>(a, tw, ta, p, G, smem, pps);
}

struct SmallPlan {
  int G = 0, rows_box = 0, stages = 0, pps = 0;
  unsigned w_bytes = 0, w_pitch = 0, slot_bytes = 0, ring_bytes = 0;
  size_t smem = 0;
};

bool plan_small(const MatmulArgs& a, SmallPlan& pl) {
  if (a.fmt != LQ_FMT_F16 && a.fmt != LQ_FMT_Q8_0 && a.fmt != LQ_FMT_Q4_0) return false;
  if (a.a_perm || (a.epi != epi::kPlain && a.epi != epi::kResidual)) return false;
  if (a.M < 2 || a.M > kSMaxM || a.K % kPieceK != 0 || a.K > (1 << 20) || a.N < 1 || a.N >= (1LL << 30))
    return false;
  if (!aligned_to(a.A, 16) || !aligned_to(a.W, 16)) return false;
  if (!tma_encode_tiled()) return false;
  const DeviceInfo& di = device_info();
  if (di.cc_major < 10) return false;
  const int64_t G = std::min<int64_t>(di.sm_count, (a.N + 7) / 8);
  const int64_t rows = (a.N + G - 1) / G;
  if (rows > 8 * kSMaxTiles) return false;
  const int tg = (a.M + kSTokens - 1) / kSTokens;
  if (tg > 1 && rows > 16 * kSMaxPairs2) return false;
  if (tg > 2 && rows > 16 * kSMaxPairs3) return false;
  pl.G = static_cast<int>(G);
  // the box covers the CTA's rows (f16: whole 8-row groups, for the
  // swizzled boxes' 1024-byte alignment); a tile's rows past the box read
  // other bytes of shared memory, into outputs that are not stored
  pl.rows_box = static_cast<int>(a.fmt == LQ_FMT_F16 ? (rows + 7) / 8 * 8 : rows);
  pl.w_bytes = static_cast<unsigned>(pl.rows_box * piece_row_bytes(a.fmt));  // f16: a multiple of 4096
  pl.w_pitch = (pl.w_bytes + 127u) / 128u * 128u;
  const long long budget = std::min(di.max_smem_optin, 227 * 1024) - 1024 - kSBarsBytes;
  // the last tile's rows past the box read up to 7 rows beyond the last slot
  const long long tail = 7LL * piece_row_bytes(a.fmt);
  // two pieces a stage where they fit twice (one or two token groups), else
  // one (two or three token groups); a ring of one slot would not overlap
  // copies and MMAs
  int S = 0, pps = 0, nstages = 0;
  for (const int cand : {2, 1}) {
    if ((cand == 2 && tg > 2) || (cand == 1 && tg < 2)) continue;  // (one group: two pieces or nothing)
    // (A's M KB a piece keeps the weights 1024-aligned, as f16's swizzled boxes need)
    const unsigned slot = (cand * (static_cast<unsigned>(a.M) * kARowBytes + pl.w_pitch) + 1023u) / 1024u * 1024u;
    const int ns = static_cast<int>((a.K / kPieceK + cand - 1) / cand);
    const int s = static_cast<int>(std::min<long long>({kSMaxStages, ns, (budget - tail) / slot}));
    if (s >= std::min(2, ns)) {
      S = s;
      pps = cand;
      nstages = ns;
      pl.slot_bytes = slot;
      break;
    }
  }
  if (!pps) return false;
  (void)nstages;
  const long long red = static_cast<long long>((rows + 7) / 8) * (8 * pps) * 128 * tg * 4;  // partial tiles
  pl.stages = S;
  pl.pps = pps;
  pl.ring_bytes = static_cast<unsigned>(std::max<long long>(static_cast<long long>(S) * pl.slot_bytes + tail, red));
  pl.ring_bytes = (pl.ring_bytes + 127u) / 128u * 128u;
  if (static_cast<long long>(pl.ring_bytes) > budget) return false;
  pl.smem = 1024 + pl.ring_bytes + kSBarsBytes;
  return true;
}

}  // namespace

bool gemm_small_eligible(const MatmulArgs& a) {
  SmallPlan pl;
  return plan_small(a, pl);
}

unsigned read_clear_small_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_small_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_small_err, &z, sizeof(z));
  return v;
}

lq_status launch_gemm_small(const MatmulArgs& a) {
  SmallPlan pl;
  if (!plan_small(a, pl)) return LQ_ERR_UNSUPPORTED;
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  Encode enc = reinterpret_cast<Encode>(tma_encode_tiled());
  CUtensorMap tw, ta;
  const uint64_t rb = static_cast<uint64_t>(row_bytes(a.fmt, a.K));
  if (a.fmt == LQ_FMT_F16) {
    // W as [N][K] halves; boxes of 64 halves x rows_box rows, 128B-swizzled
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.N)};
    cuuint64_t strides[1] = {rb};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(pl.rows_box)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(a.W), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return LQ_ERR_UNSUPPORTED;
  } else {
    // W as [N][K/256][bytes of 256 K / 4] words; a box is one such piece of rows_box rows
    const int prb = piece_row_bytes(a.fmt);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(prb / 4), static_cast<cuuint64_t>(a.K / kPieceK),
                          static_cast<cuuint64_t>(a.N)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(prb), rb};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(prb / 4), 1, static_cast<cuuint32_t>(pl.rows_box)};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(a.W), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return LQ_ERR_UNSUPPORTED;
  }
  {
    // A as [M][K] f32; boxes of 256 values x M rows
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kPieceK), static_cast<cuuint32_t>(a.M)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(a.A), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return LQ_ERR_UNSUPPORTED;
  }
  SmallParams p = {};
  p.C = a.C;
  p.R = a.R;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.rows_box = pl.rows_box;
  p.stages = pl.stages;
  p.w_bytes = pl.w_bytes;
  p.w_pitch = pl.w_pitch;
  p.slot_bytes = pl.slot_bytes;
  p.ring_bytes = pl.ring_bytes;
  p.wait_ns = wait_limit_ns();
  p.wait_iters = wait_limit_iters();
  lq_status st;
  if (a.fmt == LQ_FMT_F16)
    st = launch_small_fmt<LQ_FMT_F16>(a, tw, ta, p, pl.G, pl.smem, pl.pps);
  else if (a.fmt == LQ_FMT_Q8_0)
    st = launch_small_fmt<LQ_FMT_Q8_0>(a, tw, ta, p, pl.G, pl.smem, pl.pps);
  else
    st = launch_small_fmt<LQ_FMT_Q4_0>(a, tw, ta, p, pl.G, pl.smem, pl.pps);
  if (st == LQ_OK) count_route(5);
  return st;
}

}  // namespace lq
