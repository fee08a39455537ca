// Prefill GEMM, fast path: TMA-fed tcgen05 kernel with the weight operand in
// tensor memory.
//
// Counterparts on the source pages: gemm_q4_tiled / gemm_q8_tiled
// (lattice-inference, metal_qwen35.rs and dispatch.rs: W dequantised inside
// the tile loop) and gemm_f32a_f16w_v2 (ferrum-kernels pipelines.rs: f16
// weights widened on load). The GB300 design:
//
//  1. a pre-pass rounds A (f32) to bf16, to nearest even: exactly the
//     operand the tensor-core tolerance is defined on, over the whole f32
//     range (bf16 keeps f32's exponent);
//  2. the GEMM kernel, one CTA per SM, owns 128 rows of W and a tile of BT
//     tokens. Raw W (f16 / Q8_0 / Q4_0 bytes) arrives by TMA, one box of
//     full-width rows per stage, each slot refilled by a warp of its own as
//     soon as the converters have read it: Q8_0 rows of 256 K are 272
//     bytes and Q4_0 rows 144 bytes, both odd multiples of 16, so eight
//     threads reading 16-byte chunks of eight consecutive rows hit eight
//     different bank groups; f16 rows (64 K = 128 bytes per box) use the
//     TMA's 128-byte swizzle for the same effect. The bf16 A tile arrives the
//     same way in the swizzled K-major layout of the MMA's B operand;
//  3. eight converter warps (thread = W row = TMEM lane) dequantise 64 K of
//     their row at a time: each weight is formed exactly in f32 (Q8_0: q*d,
//     Q4_0: (q-8)*d, an 11-bit scale times a code of at most 8 bits; f16:
//     widened) and rounded once to bf16, for any block scale, and written
//     into tensor memory with tcgen05.st;
//  4. one thread issues tcgen05.mma kind::f16 (bf16 x bf16) with A (= W) from
//     tensor memory and B (= tokens) from shared memory, accumulating f32 in
//     TMEM;
//  5. four warps read the accumulator (tcgen05.ld) and store C with
//     coalesced stores.
// Every wait is bounded; on timeout the kernel records LQ_ERR_DEVICE_TIMEOUT,
// lets its copies and MMAs finish, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "lq_device.cuh"
#include "lq_epilogue.cuh"
#include "lq_internal.h"
#include "lq_q4i.cuh"
#include "lq_tcgen05.cuh"

namespace lq {
namespace {

__device__ unsigned g_tma_err;

constexpr int kNumConv = 8;                        // converter warps (kGroups groups of 4)
constexpr int kGroups = kNumConv / 4;              // a group's 4 warps cover the 128 TMEM lanes
constexpr int kConvThreads = kNumConv * 32;
constexpr int kRawWarp = 2 + kNumConv;             // raw W refills
constexpr int kTmaThreads = (3 + kNumConv) * 32;   // producer, MMA, converters, raw W
constexpr int kGateWarp = 3 + kNumConv;            // CTA pairs: the stage relay (rank 1) / gate (rank 0)
constexpr int kPairThreads = kTmaThreads + 32;
constexpr int kBN = 128;                           // W rows per CTA
constexpr int kKS = 128;                           // K per pipeline stage (8 MMAs of K=16)
constexpr int kMaxStages = 4, kMaxRawStages = 8;  // A ring (streamed A), raw W ring
constexpr int kMaxSlots = 7;                       // TMEM weight slots (resident A: up to 7)
constexpr uint32_t kTmemCols = 512;                // D: [0, w_col0), W slots: [w_col0, w_col0 + 64 * stages)

// Pipeline stages per raw stage, and bytes of one W row per raw stage (Q
// formats: 256 K in one box; f16: 128 K as two boxes of 64 K, each 128 rows
// x 128 bytes, swizzled).
template <int FMT> constexpr int kSub = FMT == LQ_FMT_F16 ? 1 : 2;
template <int FMT> constexpr int kRowBytes = FMT == LQ_FMT_F16 ? 256 : (FMT == LQ_FMT_Q8_0 ? 272 : 144);

struct TmaGemmParams {
  const float* A;      // resident-A mode: the f32 activations themselves
  float* C;
  const float* R;      // residual epilogue: added to every output
  int M, N, K;
  int bt;              // tokens per CTA (multiple of 16, <= 256)
  int split;           // CTAs of a cluster splitting K (1: no split)
  int stages;          // pipeline depth = TMEM weight slots (2..kMaxStages, resident A up to kMaxSlots)
  int w_col0;          // first TMEM column of the weight slots (the accumulator's bt columns lie below)
  int raw_stages;      // raw W ring depth (2..kMaxRawStages)
  unsigned long long wait_ns;
  unsigned wait_iters;
  int a_res;           // 1: the CTA rounds its whole A slice to bf16 into shared memory itself
  int a_tiles;         // A tiles in shared memory: the ring's stages, or (resident) the K-steps of a rank
  int a_perm;          // resident A, Q4_0 with interleaved nibbles: the slot order of lq_q4i.cuh
};

struct Bars {
  uint64_t raw_full[kMaxRawStages], raw_empty[kMaxRawStages];
  uint64_t full[kMaxSlots];    // A tile landed (TMA bytes) + the group's 4 converter warps wrote W
  uint64_t pfull[kMaxSlots];   // CTA pairs, rank 0: rank 1's half of the stage is ready (its relay warp)
  uint64_t empty[kMaxSlots];   // the stage's MMAs completed (commit)
  uint64_t tmem_full;
  uint64_t a_ready;            // resident A: the converter warps stored every stage's A tile
  uint32_t tmem_base;
  volatile int abort;
};

__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_tma_err, 0u, code); }

// Bounded wait by all 32 lanes of a warp, with one outcome for the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const TmaGemmParams& p) {
  const bool ok = mbar_wait(bar, parity, p.wait_ns, p.wait_iters);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// Pre-pass: A f32 [M,K] -> bf16 [M,K], every value rounded to nearest even
// (cvt.rn.bf16x2.f32). Elementwise: thread i converts elements 8i .. 8i+7
// (K is a multiple of 128 on this route, so eight never straddle a row or a
// block of 32). With perm (Q4_0 with interleaved nibbles) each block's
// elements go to the slots of lq_q4i.cuh: element 2j to slot j, 2j+1 to
// slot 16+j.
// ---------------------------------------------------------------------------
constexpr int kPreThreads = 256;

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x (low half) = lo
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __launch_bounds__(kPreThreads) a_to_bf16_kernel(const float* __restrict__ A,
                                                                uint32_t* __restrict__ A16, long long n8,
                                                                int perm) {
  pdl_launch_dependents();
  pdl_wait();
  const long long stride = static_cast<long long>(gridDim.x) * kPreThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kPreThreads + threadIdx.x; i < n8; i += stride) {
    const float4 x = ldg128f(A + 8 * i), y = ldg128f(A + 8 * i + 4);
    if (!perm) {
      const uint4 o = make_uint4(bf16x2(x.x, x.y), bf16x2(x.z, x.w), bf16x2(y.x, y.y), bf16x2(y.z, y.w));
      *reinterpret_cast<uint4*>(A16 + 4 * i) = o;
    } else {
      // chunk c of block b: even elements 8c, 8c+2, 8c+4, 8c+6 -> slots
      // 4c .. 4c+3 (words 2c, 2c+1); odd ones -> slots 16+4c .. (words 8+2c, 9+2c)
      uint32_t* blk = A16 + 16 * (i >> 2);
      const int c = static_cast<int>(i & 3);
      *reinterpret_cast<uint2*>(blk + 2 * c) = make_uint2(bf16x2(x.x, x.z), bf16x2(y.x, y.z));
      *reinterpret_cast<uint2*>(blk + 8 + 2 * c) = make_uint2(bf16x2(x.y, x.w), bf16x2(y.y, y.w));
    }
  }
}

// ---------------------------------------------------------------------------
// Converters: 64 K of W row r (raw stage in shared memory at `stage`) ->
// 32 words of packed bf16 pairs (word j = elements 2j, 2j+1; low half = even
// element). Each weight is formed exactly in f32 and rounded once: a code
// byte goes into the low mantissa byte of 2^23 (one byte-permute), one
// packed add takes the bias off exactly (q, or q - 8), and one packed
// multiply by the f16 scale is exact too (11 x 8 significant bits); the
// f16 weights widen exactly. cvt.rn.bf16x2.f32 then rounds to nearest even.
// ---------------------------------------------------------------------------
template <int FMT, int SUB>
__device__ __forceinline__ void convert64(uint32_t stage, uint32_t r, uint32_t (&out)[32]) {
  if constexpr (FMT == LQ_FMT_F16) {
    // box SUB: 128 rows x 128 bytes, 16-byte chunk c of row r at chunk c ^ (r % 8)
    const uint32_t row = stage + SUB * (kBN * 128u) + r * 128u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 v = lds128(row + ((static_cast<uint32_t>(i) ^ (r & 7u)) << 4));
      const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[j]));
        out[4 * i + j] = bf16x2(f.x, f.y);
      }
    }
  } else if constexpr (FMT == LQ_FMT_Q8_0) {
    // two 34-byte blocks at byte 68*SUB of the row's 272 raw bytes
    constexpr int s0 = (68 * SUB) / 16, off = SUB;  // first 16-byte chunk, word offset in it
    const uint32_t row = stage + r * 272u;
    uint32_t w[20];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
      const uint4 v = lds128(row + static_cast<uint32_t>(s0 + i) * 16u);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
    const float2 bias = make_float2(-kMagicS8, -kMagicS8);
    const float d0 = f16_lo(w[off]), d1 = f16_lo(w[off + 8] >> 16);
    const float2 dd0 = make_float2(d0, d0), dd1 = make_float2(d1, d1);
#pragma unroll
    for (int p = 0; p < 16; ++p) {
      // block 0: bytes 2+2p, 3+2p; block 1: bytes 36+2p, 37+2p
      const int b0 = 2 + 2 * p, b1 = 36 + 2 * p;
      const uint32_t x0 = w[off + (b0 >> 2)] ^ 0x80808080u;  // sign bits flipped: byte = q + 128
      const uint32_t x1 = w[off + (b1 >> 2)] ^ 0x80808080u;
      const float2 q0 = fadd2(make_float2(s8_to_magic(x0, b0 & 3), s8_to_magic(x0, (b0 & 3) + 1)), bias);
      const float2 q1 = fadd2(make_float2(s8_to_magic(x1, b1 & 3), s8_to_magic(x1, (b1 & 3) + 1)), bias);
      const float2 v0 = fmul2(q0, dd0), v1 = fmul2(q1, dd1);
      out[p] = bf16x2(v0.x, v0.y);
      out[16 + p] = bf16x2(v1.x, v1.y);
    }
  } else {
    // two 18-byte blocks at byte 36*SUB of the row's 144 raw bytes
    constexpr int s0 = (36 * SUB) / 16, off = SUB;
    const uint32_t row = stage + r * 144u;
    uint32_t w[12];
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      const uint4 v = lds128(row + static_cast<uint32_t>(s0 + i) * 16u);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
    const float2 bias = make_float2(-kMagicQ4, -kMagicQ4);
    const float d0 = f16_lo(w[off]), d1 = f16_lo(w[off + 4] >> 16);
    const float2 dd0 = make_float2(d0, d0), dd1 = make_float2(d1, d1);
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      // bytes j = 2+2p, 3+2p of block 0 (and 20+2p.. of block 1) hold
      // q_{2p}, q_{2p+1} (low nibbles) and q_{16+2p}, q_{17+2p} (high)
      const int b0 = 2 + 2 * p, b1 = 20 + 2 * p;
      const uint32_t x0 = w[off + (b0 >> 2)], x1 = w[off + (b1 >> 2)];
      const uint32_t lo0 = x0 & 0x0F0F0F0Fu, hi0 = (x0 >> 4) & 0x0F0F0F0Fu;
      const uint32_t lo1 = x1 & 0x0F0F0F0Fu, hi1 = (x1 >> 4) & 0x0F0F0F0Fu;
      const int i0 = b0 & 3, i1 = b1 & 3;
      const float2 l0 = fmul2(fadd2(make_float2(s8_to_magic(lo0, i0), s8_to_magic(lo0, i0 + 1)), bias), dd0);
      const float2 h0 = fmul2(fadd2(make_float2(s8_to_magic(hi0, i0), s8_to_magic(hi0, i0 + 1)), bias), dd0);
      const float2 l1 = fmul2(fadd2(make_float2(s8_to_magic(lo1, i1), s8_to_magic(lo1, i1 + 1)), bias), dd1);
      const float2 h1 = fmul2(fadd2(make_float2(s8_to_magic(hi1, i1), s8_to_magic(hi1, i1 + 1)), bias), dd1);
      out[p] = bf16x2(l0.x, l0.y);
      out[8 + p] = bf16x2(h0.x, h0.y);
      out[16 + p] = bf16x2(l1.x, l1.y);
      out[24 + p] = bf16x2(h1.x, h1.y);
    }
  }
}

// One K-step of W row r: pieces P0 and P1 (compile-time, so that the two
// conversions form one straight-line block the scheduler can interleave)
// into the step's TMEM slot columns tcol .. tcol + 63.
template <int FMT, int P0, int P1>
__device__ __forceinline__ void convert_step(uint32_t stage, uint32_t r, uint32_t tcol) {
  uint32_t out0[32], out1[32];
  convert64<FMT, P0>(stage, r, out0);
  convert64<FMT, P1>(stage, r, out1);
  tc::st_32x32b_x32(tcol, out0);
  tc::st_32x32b_x32(tcol + 32u, out1);
}


// ---------------------------------------------------------------------------
// Split-K support: cluster barrier and loads from a peer CTA's shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t peer_addr(uint32_t local_addr, uint32_t peer) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(peer));
  return remote;
}
// Arrive on a barrier of another CTA of the cluster (address from peer_addr),
// releasing this thread's prior writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}
// Polls of a barrier that another CTA arrives on (acquire at cluster scope).
__device__ __forceinline__ bool mbar_test_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait as mbar_wait with acquire at cluster scope, by all 32 lanes,
// with one outcome for the warp.
__device__ __forceinline__ bool warp_wait_cl(uint64_t* bar, uint32_t parity, const TmaGemmParams& p) {
  bool ok = false;
  if (p.wait_iters < 1024u) {
    for (uint32_t it = 0; it < p.wait_iters && !ok; ++it) ok = mbar_test_wait_cl(bar, parity);
  } else {
    ok = mbar_try_wait_cl(bar, parity);
    const long long t0 = clock64(), limit = static_cast<long long>(p.wait_ns) * 4;
    for (uint32_t it = 1; !ok && it < p.wait_iters; ++it) {
      ok = mbar_try_wait_cl(bar, parity);
      if (!ok && (it & 15u) == 15u && clock64() - t0 > limit) break;
    }
  }
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ float ld_peer_f32(uint32_t local_addr, uint32_t peer) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(peer));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote));
  return v;
}

// Epilogue of one TMEM lane (W row r of the tile): the accumulator columns
// of 32-column chunks c0, c0 + 2, ..., plus the partial tiles of peers
// 1 .. split-1 (token-major f32 at `red` in their shared memory) when
// split > 1, stored to C[m0 + j, n0 + r].
template <int FMT, int EPI>
__device__ __forceinline__ void store_tile(const TmaGemmParams& p, uint32_t tcol, int r, int n0, int m0,
                                           int bt, uint32_t red, int split, int c0) {
  const int n = n0 + r;
#pragma unroll
  for (int i = 0; i < (8 + kGroups - 1) / kGroups; ++i) {
    const int c = c0 + kGroups * i;
    if (c >= (bt + 31) / 32) break;
    uint32_t v[32];
    tc::ld_32x32b_x32(tcol + 32u * c, v);
    tc::wait_ld();
#pragma unroll 1
    for (int q = 1; q < split; ++q) {
      // all 32 loads first, so that they are in flight together
      float t[32];
#pragma unroll
      for (int jj = 0; jj < 32; ++jj)
        t[jj] = 32 * c + jj < bt ? ld_peer_f32(red + 4u * static_cast<uint32_t>((32 * c + jj) * kBN + r),
                                               static_cast<uint32_t>(q))
                                 : 0.f;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) v[jj] = __float_as_uint(__uint_as_float(v[jj]) + t[jj]);
    }
    // residual: 16 values of R first (R may be C, so no load could move
    // past a store), then their stores
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float rv[16];
      if constexpr (EPI == epi::kResidual) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int m = m0 + 32 * c + 16 * h + jj;
          rv[jj] = (n < p.N && 32 * c + 16 * h + jj < bt && m < p.M && LQ_IN_BOUNDS(n >= 0 && m >= 0))
                       ? p.R[static_cast<long long>(m) * p.N + n]
                       : 0.f;
        }
      }
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int m = m0 + 32 * c + 16 * h + jj;
        if (n < p.N && 32 * c + 16 * h + jj < bt && m < p.M && LQ_IN_BOUNDS(n >= 0 && m >= 0)) {
          const long long o = static_cast<long long>(m) * p.N + n;
          if constexpr (EPI == epi::kResidual)
            p.C[o] = __uint_as_float(v[16 * h + jj]) + rv[jj];
          else
            p.C[o] = __uint_as_float(v[16 * h + jj]);
        }
      }
    }
  }
}

// Resident A: thread t of the kConvThreads converter threads stores 16-byte
// chunks t, t + kConvThreads, ... of the CTA's A slice: chunk q = (token r, K-step s, chunk cc
// of 16 in the step); tokens past M are zeros. The eight bf16 values of a
// chunk are A[m0 + r][128 (ks0 + s) + 8 cc ..] rounded to nearest even, or,
// with perm (Q4_0 with interleaved nibbles), the slots 8u .. 8u+7 of their
// block of 32 (u = cc % 4): elements 16 (u % 2) + 2 i + u / 2 of the block.
__device__ __forceinline__ void load_resident_a(const TmaGemmParams& p, uint8_t* a_ring, uint32_t a_stage_bytes,
                                                uint32_t atom_bytes, int bt, int m0, int ks0, int nk, int t) {
  const int per_row = nk * 16, total = bt * per_row;
  const uint32_t ring = smem_u32(a_ring);
#pragma unroll 1
  for (int q0 = t; q0 < total; q0 += kConvThreads * 4) {
    float v[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0 + kConvThreads * u;
      const int r = q / per_row, c = q - r * per_row;
      const int m = m0 + r;
      if (q < total && m < p.M && LQ_IN_BOUNDS(m >= 0)) {
        const float* row = p.A + static_cast<long long>(m) * p.K + 128LL * ks0;
        const int kb = 8 * c;  // first K of the chunk within the slice
        if (!p.a_perm) {
          const float4 x = ldg128f(row + kb), y = ldg128f(row + kb + 4);
          v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
          v[u][4] = y.x; v[u][5] = y.y; v[u][6] = y.z; v[u][7] = y.w;
        } else {
          const int blk = kb & ~31, w = (kb >> 3) & 3;
          const float* src = row + blk + 16 * (w & 1) + (w >> 1);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[u][i] = __ldg(src + 2 * i);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0 + kConvThreads * u;
      if (q >= total) break;
      const int r = q / per_row, c = q - r * per_row;
      const int s = c >> 4, cc = c & 15;
      const uint32_t addr = ring + static_cast<uint32_t>(s) * a_stage_bytes + static_cast<uint32_t>(cc >> 3) * atom_bytes +
                            tc::sw128_offset(static_cast<uint32_t>(r), static_cast<uint32_t>(cc & 7));
      sts128(addr, make_uint4(bf16x2(v[u][0], v[u][1]), bf16x2(v[u][2], v[u][3]), bf16x2(v[u][4], v[u][5]),
                              bf16x2(v[u][6], v[u][7])));
    }
  }
}

// ---------------------------------------------------------------------------
// The GEMM kernel. Warp 0: TMA producer of the A stages (and of the first
// raw W stages). Warp 1: TMEM owner and MMA issuer. Warp 2 + kNumConv: the
// raw W refills.
// Warps 2..: converters in kGroups groups of four (group g converts the
// pipeline stages ks with ks % kGroups == g: 128 K of its W rows into the
// stage's 64 TMEM columns); then every group runs the epilogue, group g
// taking the 32-column chunks g, g + kGroups, ... With split K (a cluster of CTAs sharing one
// output tile), the other ranks leave their partial tiles in their own
// shared memory and the leader adds them over distributed shared memory
// before storing C. Per stage one barrier
// says "A tile and W operand ready" (1 arrival with the TMA bytes + 4
// converter warps) and one commit says "the stage's MMAs are done". The
// producer and MMA warps run their loops with all 32 lanes (every lane
// waits, lane 0 issues); a lone active lane beside parked lanes issues very
// slowly. Every waiter sees the phases of the barriers it waits on in order.
// ---------------------------------------------------------------------------
//
// EPI (lq_epilogue.cuh): kResidual adds R in the store. kSwiglu: tmW views W
// as [2][N][row] (gate rows, then up rows) and one box brings 64 gate rows
// and the 64 matching up rows (tile rows 0-63 and 64-127, the same bytes and
// layout as a 128-row box), so a tile covers 64 outputs; the epilogue warps
// put the scaled accumulators into the idle A ring and then combine gate and
// up pairs in one short loop (a fully unrolled combine made the kernel's
// code large enough to stall on instruction fetch). No K split with kSwiglu.
//
// PAIR (opt-in, lq_debug_gemm_pairs): the two CTAs of a cluster of two (W
// row tiles 2i and 2i + 1, the same tokens) run as one CTA pair. Each loads
// half of the token tile (bt / 2 rows) and converts its own 128 W rows into
// its own tensor memory; rank 0's MMA thread issues M = 256 MMAs over both
// (cta_group::2), so each SM pulls half the token bytes per MMA FLOP. A warp
// of its own (kGateWarp) carries each stage's readiness across: in rank 1 it
// waits for its own full barrier and arrives on rank 0's pfull (release at
// cluster scope); in rank 0 it waits for pfull (acquire at cluster scope)
// and arrives on rank 0's full, which then counts six arrivals, so that the
// MMA thread only waits at CTA scope. Rank 0's commits arrive on both CTAs'
// barriers. No K split, streamed A only. Slower than single CTAs on every
// shape measured (Q8_0 512 x 6144 x 2048: 23.2 against 17.6 us): in a
// %globaltimer timeline the half tiles land no sooner than whole ones
// (about 1.4 us after issue), the hop from rank 1 to rank 0 adds about
// 0.8 us to every stage and the setup's cluster barrier about 2.5 us, while
// the pair's MMAs alone run at the single CTAs' rate.
template <int FMT, int EPI, bool PAIR = false>
__global__ void __launch_bounds__(PAIR ? kPairThreads : kTmaThreads, 1)
    gemm_tma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                    const TmaGemmParams p) {
  constexpr int SUB = kSub<FMT>;
  constexpr bool SWIGLU = EPI == epi::kSwiglu;
  static_assert(!(PAIR && SWIGLU), "no CTA pairs with the SwiGLU epilogue");
  constexpr int kRawBytes = kRowBytes<FMT> * kBN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base_u = (raw_u + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u - raw_u);
  const int bt = p.bt, S = p.stages;
  const int prank = PAIR ? static_cast<int>(blockIdx.x & 1u) : 0;  // rank in the CTA pair
  const int bta = PAIR ? bt / 2 : bt;                               // token rows of this CTA's A tiles
  const uint32_t atom_bytes = static_cast<uint32_t>(bta) * 128u;  // 64 K of the A tile
  const uint32_t a_stage_bytes = 2u * atom_bytes;                  // 128 K
  uint8_t* a_ring = base;                                          // S x A tiles (swizzled)
  const int RR = p.raw_stages;
  // resident A: one A tile per K-step of the CTA instead of a ring of S
  uint8_t* w_ring = base + p.a_tiles * a_stage_bytes;              // RR x raw W stages
  Bars& b = *reinterpret_cast<Bars*>(w_ring + RR * kRawBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Split K: the `split` CTAs of a cluster share one output tile, rank r
  // taking raw W stages [jr0, jr0 + nraw); stage indices below are local to
  // the CTA, the K coordinates of its loads add ks0.
  const int split = p.split, rank = static_cast<int>(blockIdx.x) % split;
  const int n0 = (static_cast<int>(blockIdx.x) / split) * (SWIGLU ? kBN / 2 : kBN), m0 = blockIdx.y * bt;
  const int nraw_all = p.K / kKS / SUB;
  const int jr0 = rank * nraw_all / split;
  const int nraw = (rank + 1) * nraw_all / split - jr0, nk = nraw * SUB, ks0 = jr0 * SUB;
  bool epi = false;  // this CTA's accumulator is complete and may be used

  // W does not depend on the previous kernel or on the TMEM allocation:
  // with streamed A its first stages are issued as soon as their barriers
  // exist (M = 512: 18.5 against 18.6 us, f16 17.7 against 18.0); with
  // resident A after the allocation, by the producer (f16 M = 16: 10.6
  // against 10.9 us).
  auto issue_raw = [&](int j, int slot) {
    mbar_arrive_expect_tx(&b.raw_full[slot], kRawBytes);
    if (FMT == LQ_FMT_F16) {
      for (int h = 0; h < 2; ++h) {  // two boxes of 64 halves x 128 rows (128B-swizzled)
        if constexpr (SWIGLU)
          tc::tma_load_3d(w_ring + slot * kRawBytes + h * (kBN * 128), &tmW, 128 * (jr0 + j) + 64 * h, n0, 0,
                          &b.raw_full[slot]);
        else
          tc::tma_load_2d(w_ring + slot * kRawBytes + h * (kBN * 128), &tmW, 128 * (jr0 + j) + 64 * h, n0,
                          &b.raw_full[slot]);
      }
    } else {  // one box of (row bytes of 256 K) / 4 words x 128 rows
      if constexpr (SWIGLU)
        tc::tma_load_3d(w_ring + slot * kRawBytes, &tmW, (kRowBytes<FMT> / 4) * (jr0 + j), n0, 0,
                        &b.raw_full[slot]);
      else
        tc::tma_load_2d(w_ring + slot * kRawBytes, &tmW, (kRowBytes<FMT> / 4) * (jr0 + j), n0,
                        &b.raw_full[slot]);
    }
  };
  const int raw_first = min(nraw, RR);
  if (threadIdx.x == 0) {
    for (int i = 0; i < RR; ++i) {
      mbar_init(&b.raw_full[i], 1);
      mbar_init(&b.raw_empty[i], 4 * SUB);
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(&b.full[i], 1 + 4 + (PAIR && prank == 0 ? 1 : 0));
      mbar_init(&b.empty[i], 1);
      mbar_init(&b.pfull[i], 1);
    }
    mbar_init(&b.tmem_full, 1);
    mbar_init(&b.a_ready, 1);
    b.abort = 0;
    fence_barrier_init();
    if (!p.a_res) {
      tc::prefetch_tmap(&tmW);
      for (int j = 0; j < raw_first; ++j) issue_raw(j, j);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tc::tmem_alloc_pair(&b.tmem_base, kTmemCols);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(&b.tmem_base, kTmemCols);
      tc::tmem_relinquish();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote arrive or commit
  tc::fence_after_sync();
  const uint32_t tmem = b.tmem_base;
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- producer ----------------
    if (lane == 0) {
      if (p.a_res) {
        tc::prefetch_tmap(&tmW);
        for (int j = 0; j < raw_first; ++j) issue_raw(j, j);
      } else {
        tc::prefetch_tmap(&tmA);
      }
    }
    __syncwarp();
    int issued = 0;
    bool ok = true;
    pdl_wait();
    int st = 0, lap = 0;  // stage ring position
    for (int ks = 0; ks < nk; ++ks) {
      if (ks >= S && (!warp_wait(&b.empty[st], (lap - 1) & 1, p) || b.abort)) {
        ok = false;
        break;
      }
      if (p.a_res) {
        // resident A: every stage's tile is in place once the converter
        // warps say so; the stage's producer arrival carries no bytes
        if (ks == 0 && (!warp_wait(&b.a_ready, 0, p) || b.abort)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive(&b.full[st]);
      } else if (lane == 0) {
        const int ma = m0 + prank * bta;  // CTA pairs: this CTA's half of the token tile
        mbar_arrive_expect_tx(&b.full[st], a_stage_bytes);
        tc::tma_load_2d(a_ring + st * a_stage_bytes, &tmA, kKS * (ks0 + ks), ma, &b.full[st]);
        tc::tma_load_2d(a_ring + st * a_stage_bytes + atom_bytes, &tmA, kKS * (ks0 + ks) + 64, ma,
                        &b.full[st]);
      }
      __syncwarp();
      ++issued;
      if (++st == S) { st = 0; ++lap; }
    }
    if (!ok && lane == 0) {
      record_error(kDevErrTimeout);
      b.abort = 1;
    }
    // never leave copies in flight (waits for the last use of every slot)
    if (!p.a_res)
      for (int ks = max(0, issued - S); ks < issued; ++ks)
        mbar_wait(&b.full[ks % S], (ks / S) & 1, kDrainWaitNs);
  } else if (PAIR && warp == kGateWarp) {
    // ---------------- CTA pair: stage readiness across the pair ----------------
    // rank 1: full[st] (its A half landed, its converters wrote its W rows)
    // -> one arrival on rank 0's pfull[st]; rank 0: pfull[st] -> one
    // arrival on its own full[st]. Phases advance in order: rank 1's next
    // phase of full[st] needs the commit of this one's MMAs, which rank 0
    // issues only after its full[st] completed.
    bool ok = true;
    int st = 0, lap = 0;
    const uint32_t pfull0 = peer_addr(smem_u32(&b.pfull[0]), 0u);
    for (int ks = 0; ks < nk; ++ks) {
      if (prank == 1 ? !warp_wait(&b.full[st], lap & 1, p) : !warp_wait_cl(&b.pfull[st], lap & 1, p)) {
        ok = false;
        break;
      }
      if (b.abort) {
        ok = false;
        break;
      }
      if (lane == 0) {
        if (prank == 1)
          mbar_arrive_remote(pfull0 + 8u * static_cast<uint32_t>(st));
        else
          mbar_arrive(&b.full[st]);
      }
      __syncwarp();
      if (++st == S) { st = 0; ++lap; }
    }
    if (!ok && lane == 0) {
      record_error(kDevErrTimeout);
      b.abort = 1;
    }
  } else if (warp == 1 && PAIR && prank == 1) {
    // rank 1 issues no MMAs
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = tc::idesc_bf16_f32(PAIR ? 2 * kBN : kBN, static_cast<uint32_t>(bt));
    bool ok = true;
    int st = 0, lap = 0;
    auto issue_stage = [&](int ks, int sst) {
      const uint32_t abase = smem_u32(a_ring + (p.a_res ? ks : sst) * a_stage_bytes);
      const uint32_t wcol = tmem + static_cast<uint32_t>(p.w_col0) + 64u * sst;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t bdesc = tc::desc_sw128_kmajor(abase + (kk >> 2) * atom_bytes) + 2u * (kk & 3);
        if constexpr (PAIR)
          tc::mma_f16_ts_pair(tmem, wcol + 8u * kk, bdesc, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
        else
          tc::mma_f16_ts(tmem, wcol + 8u * kk, bdesc, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
      }
      if constexpr (PAIR)
        tc::commit_pair(&b.empty[sst], 0x3);
      else
        tc::commit(&b.empty[sst]);
    };
    for (int ks = 0; ks < nk;) {
      if (!warp_wait(&b.full[st], lap & 1, p)) {
        ok = false;
        break;
      }
      // Issue this stage and, without a blocking wait, any following stages
      // that are already complete (the pipeline usually runs ahead).
      int cnt = 1;
      int st2 = st + 1 == S ? 0 : st + 1, lap2 = st + 1 == S ? lap + 1 : lap;
      while (ks + cnt < nk && cnt < S - 1 && __all_sync(0xffffffffu, mbar_test_wait(&b.full[st2], lap2 & 1))) {
        ++cnt;
        if (++st2 == S) { st2 = 0; ++lap2; }
      }
      tc::fence_after_sync();
      if (lane == 0) {
        int sst = st;
        for (int i = 0; i < cnt; ++i) {
          issue_stage(ks + i, sst);
          if (++sst == S) sst = 0;
        }
      }
      __syncwarp();
      ks += cnt;
      for (int i = 0; i < cnt; ++i)
        if (++st == S) { st = 0; ++lap; }
    }
    if (!ok && lane == 0) {
      record_error(kDevErrTimeout);
      b.abort = 1;
    }
    if (lane == 0) {
      if constexpr (PAIR)
        tc::commit_pair(&b.tmem_full, 0x3);
      else
        tc::commit(&b.tmem_full);
    }
    __syncwarp();
    if (b.abort) mbar_wait(&b.tmem_full, 0, kDrainWaitNs);
  } else if (warp == kRawWarp) {
    // ---------------- raw W refills ----------------
    // slot j % RR gets raw stage j once its 4 SUB converter warps have read
    // stage j - RR. A warp of its own: in the producer's loop a refill
    // waited behind the A stages, which wait for the MMAs (Q8_0 M = 512
    // 18.1 -> 17.5 us on taking it out of that loop); issued by the last
    // converter warp instead it stalled that warp's conversions (f16 17.5 ->
    // 18.1 us).
    int issued = raw_first;
    bool ok = true;
    int rslot = 0, rlap = 0;
    for (int j = RR; j < nraw; ++j) {
      if (!warp_wait(&b.raw_empty[rslot], rlap & 1, p) || b.abort) {
        ok = false;
        break;
      }
      if (lane == 0) issue_raw(j, rslot);
      __syncwarp();
      ++issued;
      if (++rslot == RR) { rslot = 0; ++rlap; }
    }
    if (!ok && lane == 0) {
      record_error(kDevErrTimeout);
      b.abort = 1;
    }
    // never leave copies in flight
    for (int j = max(0, issued - RR); j < issued; ++j)
      mbar_wait(&b.raw_full[j % RR], (j / RR) & 1, kDrainWaitNs);
  } else {
    // ---------------- converters ----------------
    const int cw = warp - 2, g = cw >> 2, q4 = warp & 3;
    const int r = 32 * q4 + lane;  // W row in the tile = TMEM lane
    const uint32_t tlane = static_cast<uint32_t>(32 * q4) << 16;
    bool ok = true;
    if (p.a_res) {
      // Resident A: the converter threads round this CTA's A slice (bt
      // tokens x its nk K-steps) to bf16 and store it in the layout the TMA
      // would have written (per K-step two 64-K atoms of bt rows x 128
      // bytes, 16-byte chunks swizzled by row % 8), once the previous kernel
      // has completed; W keeps streaming meanwhile. (Converting the weights
      // that had landed first and loading A later measured no faster.)
      pdl_wait();
      load_resident_a(p, a_ring, a_stage_bytes, atom_bytes, bt, m0, ks0, nk, static_cast<int>(threadIdx.x) - 64);
      fence_proxy_async_smem();  // generic-proxy stores, read by the tensor core
      named_barrier(4, kConvThreads);
      if (threadIdx.x == 64) mbar_arrive(&b.a_ready);
    }
    // positions advance incrementally (no runtime divisions in the loop):
    // slot st = ks % S and its lap ks / S; raw stage j = ks / SUB, its slot
    // j % RR and lap j / RR
    int st = g % S, slap = g / S, j = g / SUB, rslot = j % RR, rlap = j / RR;
    for (int ks = g; ks < nk; ks += kGroups) {
      const int half = ks % SUB;
      if (!warp_wait(&b.raw_full[rslot], rlap & 1, p) || b.abort) {
        ok = false;
        break;
      }
      if (ks >= S && (!warp_wait(&b.empty[st], (slap - 1) & 1, p) || b.abort)) {
        ok = false;
        break;
      }
      const uint32_t stage = smem_u32(w_ring + rslot * kRawBytes);
      const uint32_t tcol = tmem + tlane + static_cast<uint32_t>(p.w_col0) + 64u * st;
      if (SUB == 1 || half == 0)
        convert_step<FMT, 0, 1>(stage, static_cast<uint32_t>(r), tcol);
      else
        convert_step<FMT, 2, 3>(stage, static_cast<uint32_t>(r), tcol);
      tc::wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&b.full[st]);
        mbar_arrive(&b.raw_empty[rslot]);
      }
      st += kGroups;
      while (st >= S) { st -= S; ++slap; }
      const int j2 = (ks + kGroups) / SUB;
      rslot += j2 - j;
      j = j2;
      while (rslot >= RR) { rslot -= RR; ++rlap; }
    }
    if (!ok && lane == 0) {
      record_error(kDevErrTimeout);
      b.abort = 1;
    }
    {
      // ---------------- epilogue (every group: 32-column chunks g, g + kGroups, ...) ----------------
      // C (and R) are touched only once the previous kernel on the stream
      // has completed (by now griddepcontrol.wait returns at once)
      pdl_wait();
      const bool have = warp_wait(&b.tmem_full, 0, p);
      tc::fence_after_sync();
      if (!have && lane == 0) {
        record_error(kDevErrTimeout);
        b.abort = 1;
      }
      epi = have && !b.abort;
      if constexpr (SWIGLU) {
        // gate (lanes 0-63) and up (lanes 64-127) accumulators
        // -> the A ring as [token][gate 64 | up 64]; then all converter warps
        // combine (token, output) pairs in one rolled loop and store 64
        // consecutive outputs of a token together
        float* xch = reinterpret_cast<float*>(a_ring);
        if (epi) {
#pragma unroll
          for (int i = 0; i < (8 + kGroups - 1) / kGroups; ++i) {
            const int c = g + kGroups * i;
            if (c >= (bt + 31) / 32) break;
            uint32_t v[32];
            tc::ld_32x32b_x32(tmem + tlane + 32u * c, v);
            tc::wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              if (32 * c + jj < bt) xch[(32 * c + jj) * 128 + r] = __uint_as_float(v[jj]);
          }
        }
        named_barrier(3, kConvThreads);  // the epilogue warps, whatever their outcome
        if (epi) {
          const int t0 = static_cast<int>(threadIdx.x) - 64;  // 0 .. kConvThreads - 1 over the converter warps
          const int rows = min(bt, p.M - m0);
#pragma unroll 1
          for (int idx = t0; idx < rows * 64; idx += kConvThreads) {
            const int tok = idx >> 6, j = idx & 63, n = n0 + j;
            if (n < p.N && LQ_IN_BOUNDS(m0 + tok < p.M && m0 + tok >= 0))
              p.C[static_cast<long long>(m0 + tok) * p.N + n] = epi::swiglu(xch[tok * 128 + j], xch[tok * 128 + 64 + j]);
          }
        }
      } else if (epi && split == 1) {
        store_tile<FMT, EPI>(p, tmem + tlane, r, n0, m0, bt, 0u, 1, g);
      } else if (epi && rank != 0) {
        // this rank's partial tile -> its own shared memory (the A ring is
        // idle now), token-major so that the 32 lanes write 32 rows in a row
        float* red = reinterpret_cast<float*>(a_ring);
#pragma unroll 1
        for (int c = g; c < (bt + 31) / 32; c += kGroups) {
          uint32_t v[32];
          tc::ld_32x32b_x32(tmem + tlane + 32u * c, v);
          tc::wait_ld();
#pragma unroll
          for (int jj = 0; jj < 32; ++jj)
            if (32 * c + jj < bt) red[(32 * c + jj) * kBN + r] = __uint_as_float(v[jj]);
        }
      }
    }
  }
  // ---------------- teardown ----------------
  tc::fence_before_sync();
  __syncthreads();
  if (split > 1) {
    // the peers' partial tiles are in their shared memory; the leader adds
    // them to its own (rank order: a fixed summation order) and stores C
    cluster_sync();
    if (rank == 0 && epi && warp >= 2 && warp < kRawWarp) {
      tc::fence_after_sync();
      const int q4 = warp & 3, r = 32 * q4 + lane, g = (warp - 2) >> 2;
      store_tile<FMT, EPI>(p, tmem + (static_cast<uint32_t>(32 * q4) << 16), r, n0, m0, bt, smem_u32(a_ring),
                           split, g);
    }
    cluster_sync();  // the peers keep their shared memory until the leader read it
  }
  // CTA pairs: rank 0's MMAs read both CTAs' shared and tensor memory, and
  // both free the pair's columns together
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc::fence_after_sync();
    if constexpr (PAIR)
      tc::tmem_dealloc_pair(tmem, kTmemCols);
    else
      tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// Launch with programmatic dependent launch and, when cluster_x > 1,
// clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                               unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  cfg.numAttrs = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  return launch_pdl_cluster(kern, grid, block, smem, st, 1u, std::forward<Args>(args)...);
}

bool aligned(const void* p, unsigned al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; }

int kstep_multiple(int fmt) { return fmt == LQ_FMT_F16 ? 128 : 256; }  // one raw stage

// Token-tile width. Up to 256 tokens: one tile (W is streamed once; the SMs
// are filled by splitting K). Beyond: enough tiles to put about one CTA on
// every SM, at most 256 tokens (the MMA's N limit).
int pick_bt(int64_t M, int64_t N) {
  if (M <= 256) return static_cast<int>((M + 15) / 16 * 16);
  const DeviceInfo& di = device_info();
  const int64_t ntn = (N + kBN - 1) / kBN;
  int64_t t = std::max<int64_t>(1, (di.sm_count + ntn / 2) / ntn);
  t = std::max<int64_t>(t, (M + 255) / 256);
  t = std::min<int64_t>(t, (M + 15) / 16);
  const int64_t per = (M + t - 1) / t;
  return static_cast<int>(std::min<int64_t>(256, (per + 15) / 16 * 16));
}

int raw_stage_bytes(int fmt) { return kBN * (fmt == LQ_FMT_F16 ? 256 : (fmt == LQ_FMT_Q8_0 ? 272 : 144)); }

// Ring depths for a token tile of bt: the raw W ring first (W comes from
// HBM: up to 6 raw stages of f16, 4 of Q8_0 / Q4_0, i.e. 6 to 8 pipeline
// stages of lookahead), then as many A stages (bt rows x 128 K halves, from
// L2) as fit, at least two of each; where that leaves two A stages, three A
// stages over fewer raw stages.
struct RingPlan {
  int a_stages = 0, raw_stages = 0;
};
std::atomic<int> g_ring_a{0}, g_ring_raw{0};  // debug override (0 = automatic)
std::atomic<int> g_pair{0};                    // CTA pairs: 1 = where they fit, 0 = never (the default)

// Raw W ring depth from the number of stages that fit. A converter group
// waits on a raw slot's next phase by parity, which is sound only if it has
// itself seen the slot's previous phase complete (copies may land out of
// order). With SUB = 2 both groups take every raw stage in order; with
// SUB = 1 (f16) group g takes the stages j with j % kGroups == g, so the
// depth is a multiple of kGroups and every slot has a single group.
int raw_ring_depth(int fmt, long long fit) {
  const long long unit = fmt == LQ_FMT_F16 ? kGroups : (kGroups + 1) / 2;
  return static_cast<int>(fit / unit * unit);
}

RingPlan ring_plan(int fmt, int bt) {
  const DeviceInfo& di = device_info();
  const long long budget = std::min(di.max_smem_optin, 227 * 1024) - 1024 -
                           static_cast<long long>(sizeof(Bars)) - 64;
  const long long a_stage = static_cast<long long>(bt) * 256, raw = raw_stage_bytes(fmt);
  RingPlan rp;
  const int raw_cap = fmt == LQ_FMT_F16 ? 6 : 4;
  rp.raw_stages = raw_ring_depth(fmt, std::min<long long>(raw_cap, (budget - 2 * a_stage) / raw));
  if (rp.raw_stages < 2) return RingPlan{};
  rp.a_stages = static_cast<int>(std::min<long long>(kMaxStages, (budget - rp.raw_stages * raw) / a_stage));
  if (rp.a_stages < 2) return RingPlan{};
  // Large token tiles leave room for two A stages only: three A stages over
  // two raw stages measured about 5 % faster at M = 512 (f16 and Q8_0).
  if (rp.a_stages == 2 && 3 * a_stage + 2 * raw <= budget) {
    rp.a_stages = 3;
    rp.raw_stages = raw_ring_depth(fmt, std::min<long long>(raw_cap, (budget - 3 * a_stage) / raw));
  }
  const int oa = g_ring_a.load(), orr = g_ring_raw.load();
  if (oa || orr) {
    const int a2 = oa ? oa : rp.a_stages, r2 = orr ? orr : rp.raw_stages;
    if (a2 >= 2 && a2 <= kMaxStages && r2 >= 2 && r2 <= kMaxRawStages && r2 == raw_ring_depth(fmt, r2) &&
        a2 * a_stage + r2 * raw <= budget)
      return RingPlan{a2, r2};
  }
  return rp;
}

size_t tma_smem_bytes(int fmt, int bt, int a_stages, int raw_stages) {
  const size_t need = 1024 + static_cast<size_t>(a_stages) * bt * 256 +
                      static_cast<size_t>(raw_stages) * raw_stage_bytes(fmt) + sizeof(Bars) + 64;
  // at least 116 KB, so that no two CTAs share an SM (each holds all of TMEM)
  return std::max<size_t>(need, 116 * 1024);
}

// Clusters of `split` CTAs along K: the largest split (up to 8, the portable
// cluster size) whose clusters all fit on the GPU at once, or 1.
template <int FMT>
int pick_split_query(int64_t tiles, int nraw_all, size_t smem);

template <int FMT>
int pick_split(int64_t tiles, int nraw_all, size_t smem) {
  const DeviceInfo& di = device_info();
  if (2 * tiles > di.sm_count) return 1;
  // the answer depends on (tiles, K, shared memory) only: remember it
  static std::mutex mu;
  static std::map<std::tuple<int, int64_t, int, size_t>, int> cache;
  const auto key = std::make_tuple(current_device(), tiles, nraw_all, smem);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const int s = pick_split_query<FMT>(tiles, nraw_all, smem);
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = s;
  return s;
}

// Lets a kernel instance use up to the per-block opt-in limit of shared
// memory (once per device); the occupancy queries and launches below then
// see the real request.
template <int FMT, int EPI, bool PAIR = false>
cudaError_t allow_full_smem() {
  static int configured[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    const int mx = std::min(device_info().max_smem_optin, 227 * 1024);
    const cudaError_t e =
        cudaFuncSetAttribute(gemm_tma_kernel<FMT, EPI, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return cudaSuccess;
}

template <int FMT>
int pick_split_query(int64_t tiles, int nraw_all, size_t smem) {
  const DeviceInfo& di = device_info();
  if (allow_full_smem<FMT, epi::kPlain>() != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  int s = static_cast<int>(std::min<int64_t>({8, di.sm_count / std::max<int64_t>(tiles, 1), nraw_all}));
  for (; s >= 2; --s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * s));
    cfg.blockDim = dim3(kTmaThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(s);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, gemm_tma_kernel<FMT, epi::kPlain>, &cfg) == cudaSuccess &&
        active >= tiles)
      return s;
    cudaGetLastError();  // a refused query is not an error of the call
  }
  return 1;
}

// CTA pairs: how many clusters of two CTAs with `smem` bytes each are
// resident at once (a GPC with an odd number of free SMs leaves one idle).
// Remembered per (device, shared memory).
template <int FMT>
int pair_slots(size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, size_t>, int> cache;
  const auto key = std::make_tuple(current_device(), smem);
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int active = 0;
  if (allow_full_smem<FMT, epi::kPlain, true>() == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(device_info().sm_count));
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&active, gemm_tma_kernel<FMT, epi::kPlain, true>, &cfg) != cudaSuccess)
      active = 0;
  }
  cudaGetLastError();  // a refused query is not an error of the call
  std::lock_guard<std::mutex> lk(mu);
  cache[key] = active;
  return active;
}

int pair_slots_fmt(int fmt, size_t smem) {
  if (fmt == LQ_FMT_F16) return pair_slots<LQ_FMT_F16>(smem);
  if (fmt == LQ_FMT_Q8_0) return pair_slots<LQ_FMT_Q8_0>(smem);
  return pair_slots<LQ_FMT_Q4_0>(smem);
}

int pick_split_fmt(int fmt, int64_t tiles, int nraw_all, size_t smem) {
  if (fmt == LQ_FMT_F16) return pick_split<LQ_FMT_F16>(tiles, nraw_all, smem);
  if (fmt == LQ_FMT_Q8_0) return pick_split<LQ_FMT_Q8_0>(tiles, nraw_all, smem);
  return pick_split<LQ_FMT_Q4_0>(tiles, nraw_all, smem);
}

// The launch plan of a call: token tile, K split, ring depths and whether A
// is resident. Resident A: when the CTA's whole A slice (bt tokens x its
// share of K, bf16) fits in shared memory beside two raw W stages, the CTA
// rounds it itself and no pre-pass, workspace or A ring is needed (small M);
// otherwise the pre-pass writes the bf16 copy of A to the workspace and the
// CTAs stream its tiles with TMA.
struct TmaLaunch {
  int bt = 0, split = 1, stages = 0, raw_stages = 0, a_res = 0, a_tiles = 0, w_col0 = 256;
  int pair = 0;  // CTA pairs (each CTA's A tiles hold bt / 2 token rows)
};

TmaLaunch plan_tma(const MatmulArgs& a) {
  TmaLaunch pl;
  const bool sw = a.epi == epi::kSwiglu;
  // swiglu tiles hold 64 outputs (128 W rows): as many tiles as 2N rows
  pl.bt = pick_bt(a.M, sw ? 2 * a.N : a.N);
  const RingPlan rp = ring_plan(a.fmt, pl.bt);
  if (rp.a_stages < 2) return TmaLaunch{};
  pl.stages = rp.a_stages;
  pl.raw_stages = rp.raw_stages;
  pl.a_tiles = rp.a_stages;
  const int sub = a.fmt == LQ_FMT_F16 ? 1 : 2;
  const int nraw_all = static_cast<int>(a.K / kKS / sub);
  const int bn = sw ? kBN / 2 : kBN;
  const int64_t tiles = ((a.N + bn - 1) / bn) * ((a.M + pl.bt - 1) / pl.bt);
  pl.split = sw ? 1 : pick_split_fmt(a.fmt, tiles, nraw_all, tma_smem_bytes(a.fmt, pl.bt, pl.a_tiles, pl.raw_stages));
  const DeviceInfo& di = device_info();
  const long long budget = std::min(di.max_smem_optin, 227 * 1024) - 1024 -
                           static_cast<long long>(sizeof(Bars)) - 64;
  // at least two tiles: the epilogue reuses the area for bt x 128 floats
  const int a_tiles = std::max(2, (nraw_all + pl.split - 1) / pl.split * sub);
  const long long a_bytes = static_cast<long long>(a_tiles) * pl.bt * 256, raw = raw_stage_bytes(a.fmt);
  // The CTA loads its slice before its first MMA, so only small slices pay:
  // up to 64 KB of bf16 (a_tiles x bt <= 256) it saves 2 to 2.6 us per call
  // at M = 5..16 (N = 6144, K = 2048, graph replay) and 0.3 to 0.9 us at
  // M = 32; at M = 64 (96 KB) it cost 1.5 to 1.8 us. An explicit A-ring
  // depth from lq_debug_gemm_rings keeps the streamed A.
  if (a_bytes + 2 * raw <= budget && a_tiles * pl.bt <= 256 && g_ring_a.load() == 0) {
    pl.a_res = 1;
    pl.a_tiles = a_tiles;
    // the accumulator needs bt columns; the weight slots take the rest of
    // the 512 in steps of 64 (7 slots up to bt = 64, 4 at bt = 256)
    pl.w_col0 = (pl.bt + 63) / 64 * 64;
    pl.stages = std::min(kMaxSlots, (512 - pl.w_col0) / 64);
    pl.raw_stages = raw_ring_depth(a.fmt, std::min<long long>(a.fmt == LQ_FMT_F16 ? 6 : 4, (budget - a_bytes) / raw));
  }
  // CTA pairs: streamed A without a K split, an even number of W row tiles
  // (tiles 2i and 2i + 1 pair up), and no more waves of pairs than of
  // single CTAs (one an SM). Each CTA's A tiles then hold bt / 2 rows, so
  // the rings are planned for that.
  const int64_t row_tiles = (a.N + bn - 1) / bn;
  if (!sw && !pl.a_res && pl.split == 1 && row_tiles % 2 == 0 && g_pair.load() != 0) {
    const RingPlan hp = ring_plan(a.fmt, pl.bt / 2);
    const int slots =
        hp.a_stages >= 2 ? pair_slots_fmt(a.fmt, tma_smem_bytes(a.fmt, pl.bt / 2, hp.a_stages, hp.raw_stages)) : 0;
    const int64_t sms = std::max(di.sm_count, 1);
    if (slots > 0 && (tiles / 2 + slots - 1) / slots <= (tiles + sms - 1) / sms) {
      pl.pair = 1;
      pl.stages = hp.a_stages;
      pl.raw_stages = hp.raw_stages;
      pl.a_tiles = hp.a_stages;
    }
  }
  return pl;
}

template <int FMT, int EPI, bool PAIR = false>
lq_status launch_gemm_kernel(const MatmulArgs& a, const CUtensorMap& tmW, const CUtensorMap& tmA,
                             TmaGemmParams p);

template <int FMT>
lq_status launch_gemm_fmt(const MatmulArgs& a, const CUtensorMap& tmW, const CUtensorMap& tmA,
                          const TmaGemmParams& p, bool pair) {
  switch (a.epi) {
    case epi::kPlain:
      return pair ? launch_gemm_kernel<FMT, epi::kPlain, true>(a, tmW, tmA, p)
                  : launch_gemm_kernel<FMT, epi::kPlain>(a, tmW, tmA, p);
    case epi::kResidual:
      return pair ? launch_gemm_kernel<FMT, epi::kResidual, true>(a, tmW, tmA, p)
                  : launch_gemm_kernel<FMT, epi::kResidual>(a, tmW, tmA, p);
    case epi::kSwiglu: return launch_gemm_kernel<FMT, epi::kSwiglu>(a, tmW, tmA, p);
    default: return LQ_ERR_UNSUPPORTED;
  }
}

lq_status launch_gemm_epi(const MatmulArgs& a, const CUtensorMap& tmW, const CUtensorMap& tmA,
                          const TmaGemmParams& p, bool pair) {
  if (a.fmt == LQ_FMT_F16) return launch_gemm_fmt<LQ_FMT_F16>(a, tmW, tmA, p, pair);
  if (a.fmt == LQ_FMT_Q8_0) return launch_gemm_fmt<LQ_FMT_Q8_0>(a, tmW, tmA, p, pair);
  return launch_gemm_fmt<LQ_FMT_Q4_0>(a, tmW, tmA, p, pair);
}

template <int FMT, int EPI, bool PAIR>
lq_status launch_gemm_kernel(const MatmulArgs& a, const CUtensorMap& tmW, const CUtensorMap& tmA,
                             TmaGemmParams p) {
  auto kern = gemm_tma_kernel<FMT, EPI, PAIR>;
  const int bn = EPI == epi::kSwiglu ? kBN / 2 : kBN;  // outputs per tile
  const size_t smem = tma_smem_bytes(FMT, PAIR ? p.bt / 2 : p.bt, p.a_tiles, p.raw_stages);
  {
    const cudaError_t e = allow_full_smem<FMT, EPI, PAIR>();
    if (e != cudaSuccess) return cuda_status(e);
  }
  const dim3 grid(static_cast<unsigned>((a.N + bn - 1) / bn * p.split),
                  static_cast<unsigned>((a.M + p.bt - 1) / p.bt));
  cudaError_t e = launch_pdl_cluster(kern, grid, dim3(PAIR ? kPairThreads : kTmaThreads), smem, a.stream,
                                     PAIR ? 2u : static_cast<unsigned>(p.split), tmW, tmA, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

}  // namespace

void* tma_encode_tiled() { return reinterpret_cast<void*>(encode_fn()); }

unsigned read_clear_gemm_tma_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_tma_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_tma_err, &z, sizeof(z));
  return v;
}


void set_gemm_rings(int a_stages, int raw_stages) {
  g_ring_a.store(a_stages);
  g_ring_raw.store(raw_stages);
}

void set_gemm_pairs(bool on) { g_pair.store(on ? 1 : 0); }

bool gemm_tma_eligible(const MatmulArgs& a) {
  if (a.M < 2 || a.K % kstep_multiple(a.fmt) != 0) return false;
  if (!aligned(a.A, 16) || !aligned(a.W, 16)) return false;
  if (a.M > (1LL << 24) || a.N > (1LL << 24)) return false;
  if (!encode_fn()) return false;
  const DeviceInfo& di = device_info();
  return di.cc_major >= 10 && ring_plan(a.fmt, 256).a_stages >= 2;
}

// The library's own stream-ordered memory pool on the current device: freed
// blocks stay in the pool (release threshold = max), so repeated calls and
// CUDA-graph replays do not map and unmap memory each time.
cudaMemPool_t workspace_pool() {
  static std::mutex mu;
  static cudaMemPool_t pools[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
    uint64_t thr = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
    pools[dev] = pool;
  }
  return pools[dev];
}

// The B operand of the tensor-core kernel (the bf16 copy of A) lives in a
// stream-ordered workspace from the library's pool for the duration of the
// call, unless A is resident (small M: no workspace, no pre-pass).
lq_status launch_gemm_tma(const MatmulArgs& a) {
  const size_t ws_bytes = gemm_tma_workspace_bytes(a);
  void* ws = nullptr;
  if (ws_bytes) {
    cudaMemPool_t pool = workspace_pool();
    if (!pool) return LQ_ERR_CUDA;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, ws_bytes, pool, a.stream);
    if (e != cudaSuccess) return LQ_ERR_CUDA;
  }
  lq_status st = launch_gemm_tma_ws(a, ws);
  if (ws) {
    cudaError_t ef = cudaFreeAsync(ws, a.stream);
    if (st == LQ_OK && ef != cudaSuccess) st = LQ_ERR_CUDA;
  }
  if (st == LQ_OK) count_route(2);
  return st;
}

size_t gemm_tma_workspace_bytes(const MatmulArgs& a) {
  const TmaLaunch pl = plan_tma(a);
  if (pl.a_res) return 0;
  return (static_cast<size_t>(a.M) * static_cast<size_t>(a.K) * 2 + 255) / 256 * 256;
}

// Pre-pass + GEMM given a workspace of gemm_tma_workspace_bytes(a) bytes
// (the bf16 copy of A, 256-byte aligned); the GEMM alone when A is resident.
lq_status launch_gemm_tma_ws(const MatmulArgs& a, void* a16) {
  const int M = static_cast<int>(a.M), N = static_cast<int>(a.N), K = static_cast<int>(a.K);
  const TmaLaunch pl = plan_tma(a);
  if (pl.bt == 0) return LQ_ERR_UNSUPPORTED;
  const int bt = pl.bt;
  // 1. A -> bf16 (round to nearest even), unless the CTAs do it themselves
  if (!pl.a_res) {
    if (!a16) return LQ_ERR_INVALID_ARG;
    const long long n8 = static_cast<long long>(M) * K / 8;
    const long long want = (n8 + kPreThreads - 1) / kPreThreads;
    const long long cap = static_cast<long long>(std::max(device_info().sm_count, 1)) * 8;
    const unsigned grid = static_cast<unsigned>(std::max<long long>(1, std::min(want, cap)));
    cudaError_t e = launch_pdl(a_to_bf16_kernel, dim3(grid), dim3(kPreThreads), 0, a.stream, a.A,
                               static_cast<uint32_t*>(a16), n8, a.a_perm ? 1 : 0);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return LQ_ERR_CUDA;
    count_route(6);  // the pre-pass launch
  }

  // 2. tensor maps. Q formats: raw W as [N][row_bytes/4] 32-bit words, one
  //    box = the bytes of 256 K (68 or 36 words) x 128 rows. f16: W as
  //    [N][K] halves, boxes of 64 x 128 with the 128-byte swizzle. The bf16
  //    A as [M][K], boxes of 64 x bt with the 128-byte swizzle.
  EncodeTiled enc = encode_fn();
  if (!enc) return LQ_ERR_UNSUPPORTED;
  const uint64_t rb = static_cast<uint64_t>(row_bytes(a.fmt, a.K));
  CUtensorMap tmW, tmA;
  std::memset(&tmA, 0, sizeof(tmA));  // resident A: never read
  {
    // swiglu: a third dimension of 2 (gate rows, up rows N rows further on)
    // and boxes of 64 + 64 rows; otherwise boxes of 128 rows
    const bool sw = a.epi == epi::kSwiglu;
    const cuuint32_t rank = sw ? 3 : 2;
    const bool f16 = a.fmt == LQ_FMT_F16;
    cuuint64_t dims[3] = {f16 ? static_cast<cuuint64_t>(K) : rb / 4, static_cast<cuuint64_t>(N), 2};
    cuuint64_t strides[2] = {rb, rb * static_cast<cuuint64_t>(N)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(f16 ? 64 : (a.fmt == LQ_FMT_Q8_0 ? 68 : 36)),
                         static_cast<cuuint32_t>(sw ? kBN / 2 : kBN), 2};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&tmW, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT32, rank,
            const_cast<void*>(a.W), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            f16 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return LQ_ERR_UNSUPPORTED;
  }
  if (!pl.a_res) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(pl.pair ? bt / 2 : bt)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a16, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return LQ_ERR_UNSUPPORTED;
  }
  TmaGemmParams p;
  p.A = a.A;
  p.C = a.C;
  p.R = a.R;
  p.M = M;
  p.N = N;
  p.K = K;
  p.bt = bt;
  p.split = pl.split;
  p.stages = pl.stages;
  p.w_col0 = pl.w_col0;
  p.raw_stages = pl.raw_stages;
  p.a_res = pl.a_res;
  p.a_tiles = pl.a_tiles;
  p.a_perm = a.a_perm ? 1 : 0;
  p.wait_ns = wait_limit_ns();
  p.wait_iters = wait_limit_iters();
  const lq_status st = launch_gemm_epi(a, tmW, tmA, p, pl.pair != 0);
  if (st == LQ_OK && pl.pair) count_route(7);
  return st;
}

}  // namespace lq
