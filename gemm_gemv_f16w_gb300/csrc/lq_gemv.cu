// Decode GEMV (M == 1): C[n] = sum_k A[k] * w(n, k) for f16, Q8_0 and Q4_0 W.
//
// Counterparts on the source pages (lattice-inference 0.1.2,
// src/forward/metal_qwen35.rs): gemv_decode_m1 / gemv_decode_core (f16),
// gemv_q8_decode and gemv_q4_decode (NR=2 rows per threadgroup, per-lane block
// slices, simd_sum). Those kernels read W with vector loads straight from
// unified memory and rely on many small threadgroups. On GB300 the weight
// stream has to keep ~7 TB/s of HBM busy, so this kernel is built around the
// copy engine instead:
//
//  * one persistent CTA per SM owns a contiguous range of W rows;
//  * a producer thread moves stages of up to 8 whole rows into a ring of
//    shared-memory slots, one 1-D bulk copy (cp.async.bulk) per stage, with
//    mbarrier transaction counts; small copies are slow, so stages are large;
//  * eight consumer warps each cover a K-slice of every row of a stage, so a
//    lane holds only its few activations in registers and has eight
//    independent rows of work per stage;
//  * dequantisation happens in registers without int->float conversions:
//    a quantised value is dropped into the mantissa of 2^23 and unbiased with
//    one exact add/fma; dot products use packed f32x2 fma;
//  * each warp reduces its eight row partials across lanes with one
//    transposed shuffle tree; the stage's finisher warp adds the eight warps'
//    partials in a fixed order and writes C.
//
// Every wait is bounded (lq_device.cuh); on timeout the kernel records
// LQ_ERR_DEVICE_TIMEOUT, its producer drains its own copies and it returns.
#include <algorithm>

#include "lq_device.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

__device__ unsigned g_gemv_err;

constexpr int kConsumerWarps = 8;              // each owns a K-slice of every row
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kRowsPerStage = 8;               // rows moved by one bulk copy
constexpr int kMaxStages = 16;
constexpr int kGemvFastMaxK = 16384;
constexpr int kHeaderBytes = 5120;             // barriers + reduction buffers

struct GemvParams {
  const float* A;
  const uint8_t* W;
  float* C;
  int N, K;
  int row_bytes;
  int rows_per_stage;        // <= kRowsPerStage
  int stages;                // ring depth
  int a_bytes;               // K * 4 (a multiple of 16)
  unsigned long long wait_ns;
  unsigned wait_iters;
};

struct Header {
  uint64_t full[kMaxStages];       // stage landed (TMA transaction bytes)
  uint64_t empty[kMaxStages];      // every consumer warp is done with the stage
  uint64_t red_full[kMaxStages];   // every consumer warp wrote its row partials
  uint64_t a_bar;
  volatile int abort;
  float red[kMaxStages][kConsumerWarps][kRowsPerStage];  // per ring slot
};
static_assert(sizeof(Header) <= kHeaderBytes, "header too large");

__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_gemv_err, 0u, code); }

// ---------------------------------------------------------------------------
// Per-format slices. A "chunk" is the part of a row that one warp covers in
// one pass: 32 lanes x 8 elements (f16, Q8_0) or 32 lanes x 16 elements
// (Q4_0). Warp w takes chunks w, w+8, w+16, ... of every row; a lane holds
// the activations of its part of each of its chunks in registers.
// ---------------------------------------------------------------------------

// f16: chunk = 256 halves = 512 bytes; lane l reads bytes [16l, 16l+16).
template <int CPW>
struct F16Slice {
  float2 a[CPW][4];
  uint32_t off[CPW];  // byte offset of the lane's 16 bytes within a row
  bool ok[CPW];
  __device__ __forceinline__ void init(uint32_t As, int warp, int lane, int K) {
    const int nch = (K + 255) / 256;
#pragma unroll
    for (int i = 0; i < CPW; ++i) {
      const int c = warp + kConsumerWarps * i;
      const int e = 256 * c + 8 * lane;
      ok[i] = c < nch && e < K;
      off[i] = 2u * static_cast<uint32_t>(e);
      if (ok[i]) {
        const float4 x = lds128f(As + 4u * e), y = lds128f(As + 4u * e + 16u);
        a[i][0] = make_float2(x.x, x.y);
        a[i][1] = make_float2(x.z, x.w);
        a[i][2] = make_float2(y.x, y.y);
        a[i][3] = make_float2(y.z, y.w);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) a[i][t] = make_float2(0.f, 0.f);
      }
    }
  }
  __device__ __forceinline__ float dot(uint32_t row, int i) const {
    const uint4 v = lds128(row + off[i]);
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&v.z));
    const float2 f3 = __half22float2(*reinterpret_cast<const __half2*>(&v.w));
    float2 acc = ffma2(f0, a[i][0], make_float2(0.f, 0.f));
    float2 acc1 = ffma2(f1, a[i][1], make_float2(0.f, 0.f));
    acc = ffma2(f2, a[i][2], acc);
    acc1 = ffma2(f3, a[i][3], acc1);
    return (acc.x + acc1.x) + (acc.y + acc1.y);
  }
};

// Q8_0: chunk = 8 blocks = 272 bytes. Lane l takes block l/4 of the chunk
// and its 8 values 8*(l%4) .. 8*(l%4)+7 (bytes 2+8*(l%4) .. of the block).
// Those 8 bytes start 2 bytes past a word boundary for even blocks, so such
// a lane reads 3 words and realigns them with one byte-permute each.
template <int CPW>
struct Q8Slice {
  float2 a[CPW][4];
  uint32_t qoff[CPW], doff[CPW];  // word-aligned byte offsets of quants / scale word
  uint32_t sel, dshift, w2off;
  bool ok[CPW];
  __device__ __forceinline__ void init(uint32_t As, int warp, int lane, int K) {
    const int nb = K / 32;
    const int bl = lane >> 2, seg = lane & 3;
    const uint32_t qb = 34u * bl + 2u + 8u * seg;   // byte offset within the chunk
    sel = (qb & 2u) ? 0x5432u : 0x3210u;
    w2off = (qb & 2u) ? 8u : 4u;  // aligned lanes re-read word 1: never past the block
    dshift = (bl & 1) ? 16u : 0u;
#pragma unroll
    for (int i = 0; i < CPW; ++i) {
      const int c = warp + kConsumerWarps * i;
      const int b = 8 * c + bl;
      ok[i] = b < nb;
      qoff[i] = 272u * c + (qb & ~3u);
      doff[i] = 272u * c + ((34u * bl) & ~3u);
      const int e = 32 * b + 8 * seg;
      if (ok[i]) {
        const float4 x = lds128f(As + 4u * e), y = lds128f(As + 4u * e + 16u);
        a[i][0] = make_float2(x.x, x.y);
        a[i][1] = make_float2(x.z, x.w);
        a[i][2] = make_float2(y.x, y.y);
        a[i][3] = make_float2(y.z, y.w);
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) a[i][t] = make_float2(0.f, 0.f);
      }
    }
  }
  __device__ __forceinline__ float dot(uint32_t row, int i) const {
    const uint32_t w0 = lds32(row + qoff[i]), w1 = lds32(row + qoff[i] + 4u),
                   w2 = lds32(row + qoff[i] + w2off);
    const uint32_t dw = lds32(row + doff[i]);
    const uint32_t x0 = __byte_perm(w0, w1, sel) ^ 0x80808080u;
    const uint32_t x1 = __byte_perm(w1, w2, sel) ^ 0x80808080u;
    const float d = f16_lo(dw >> dshift);
    const float2 mb = make_float2(-kMagicS8, -kMagicS8);
    const float2 q0 = fadd2(make_float2(s8_to_magic(x0, 0), s8_to_magic(x0, 1)), mb);
    const float2 q1 = fadd2(make_float2(s8_to_magic(x0, 2), s8_to_magic(x0, 3)), mb);
    const float2 q2 = fadd2(make_float2(s8_to_magic(x1, 0), s8_to_magic(x1, 1)), mb);
    const float2 q3 = fadd2(make_float2(s8_to_magic(x1, 2), s8_to_magic(x1, 3)), mb);
    float2 acc = ffma2(q0, a[i][0], make_float2(0.f, 0.f));
    float2 acc1 = ffma2(q1, a[i][1], make_float2(0.f, 0.f));
    acc = ffma2(q2, a[i][2], acc);
    acc1 = ffma2(q3, a[i][3], acc1);
    return d * ((acc.x + acc1.x) + (acc.y + acc1.y));
  }
};

// Q4_0: chunk = 16 blocks = 288 bytes = 512 values. Lane l takes block l/2
// of the chunk and nibble bytes 8*(l%2) .. 8*(l%2)+7 of it, i.e. values
// q_{8s+j} (low nibbles) and q_{16+8s+j} (high nibbles), s = l%2, j < 8.
// Taking each word as two half-words of two bytes (B0, B1), the nibble at
// bit 4p of a half-word is, for p = 0..3: B0.lo, B0.hi, B1.lo, B1.hi. A
// nibble at bit 4p dropped into the mantissa of 2^23 gives 2^23 + q*16^p; one
// fma with (16^-p, -(2^(23-4p)+8)) turns that into q - 8 exactly.
template <int CPW>
struct Q4Slice {
  float2 a[CPW][8];  // pair j: (a_{8s+j}, a_{16+8s+j})
  uint32_t qoff[CPW], doff[CPW];
  uint32_t sel, dshift, w2off;
  bool ok[CPW];
  __device__ __forceinline__ void init(uint32_t As, int warp, int lane, int K) {
    const int nb = K / 32;
    const int bl = lane >> 1, hs = lane & 1;
    const uint32_t qb = 18u * bl + 2u + 8u * hs;
    sel = (qb & 2u) ? 0x5432u : 0x3210u;
    w2off = (qb & 2u) ? 8u : 4u;
    dshift = (bl & 1) ? 16u : 0u;
#pragma unroll
    for (int i = 0; i < CPW; ++i) {
      const int c = warp + kConsumerWarps * i;
      const int b = 16 * c + bl;
      ok[i] = b < nb;
      qoff[i] = 288u * c + (qb & ~3u);
      doff[i] = 288u * c + ((18u * bl) & ~3u);
      const int e = 32 * b + 8 * hs;
      if (ok[i]) {
        const float4 l0 = lds128f(As + 4u * e), l1 = lds128f(As + 4u * e + 16u);
        const float4 h0 = lds128f(As + 4u * (e + 16)), h1 = lds128f(As + 4u * (e + 16) + 16u);
        a[i][0] = make_float2(l0.x, h0.x);
        a[i][1] = make_float2(l0.y, h0.y);
        a[i][2] = make_float2(l0.z, h0.z);
        a[i][3] = make_float2(l0.w, h0.w);
        a[i][4] = make_float2(l1.x, h1.x);
        a[i][5] = make_float2(l1.y, h1.y);
        a[i][6] = make_float2(l1.z, h1.z);
        a[i][7] = make_float2(l1.w, h1.w);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) a[i][t] = make_float2(0.f, 0.f);
      }
    }
  }
  // One half-word (bytes j, j+1 of the lane's eight) into two f32x2 sums.
  __device__ __forceinline__ static void halfword(uint32_t x, float2 a01, float2 a23, float2& acc0,
                                                  float2& acc1) {
    const float2 s01 = make_float2(1.0f, 0.0625f);
    const float2 c01 = make_float2(-8388616.0f, -524296.0f);
    const float2 s23 = make_float2(0.00390625f, 0.000244140625f);
    const float2 c23 = make_float2(-32776.0f, -2056.0f);
    float2 v01 = make_float2(__uint_as_float((x & 0x000Fu) | 0x4B000000u),
                             __uint_as_float((x & 0x00F0u) | 0x4B000000u));
    float2 v23 = make_float2(__uint_as_float((x & 0x0F00u) | 0x4B000000u),
                             __uint_as_float((x & 0xF000u) | 0x4B000000u));
    v01 = ffma2(v01, s01, c01);  // (q_{8s+j} - 8, q_{16+8s+j} - 8)
    v23 = ffma2(v23, s23, c23);  // (q_{8s+j+1} - 8, q_{16+8s+j+1} - 8)
    acc0 = ffma2(v01, a01, acc0);
    acc1 = ffma2(v23, a23, acc1);
  }
  __device__ __forceinline__ float dot(uint32_t row, int i) const {
    const uint32_t w0 = lds32(row + qoff[i]), w1 = lds32(row + qoff[i] + 4u),
                   w2 = lds32(row + qoff[i] + w2off);
    const uint32_t dw = lds32(row + doff[i]);
    const uint32_t x0 = __byte_perm(w0, w1, sel), x1 = __byte_perm(w1, w2, sel);
    const float d = f16_lo(dw >> dshift);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
    halfword(x0, a[i][0], a[i][1], acc0, acc1);
    halfword(x0 >> 16, a[i][2], a[i][3], acc0, acc1);
    halfword(x1, a[i][4], a[i][5], acc0, acc1);
    halfword(x1 >> 16, a[i][6], a[i][7], acc0, acc1);
    return d * ((acc0.x + acc1.x) + (acc0.y + acc1.y));
  }
};

template <int FMT, int CPW>
struct SliceOf;
template <int CPW> struct SliceOf<LQ_FMT_F16, CPW> { using T = F16Slice<CPW>; };
template <int CPW> struct SliceOf<LQ_FMT_Q8_0, CPW> { using T = Q8Slice<CPW>; };
template <int CPW> struct SliceOf<LQ_FMT_Q4_0, CPW> { using T = Q4Slice<CPW>; };

// Sums acc[0..7] over the 32 lanes with 9 shuffles: after the three halving
// steps lane l holds row ((l>>4)&1)*4 + ((l>>3)&1)*2 + ((l>>2)&1) summed over
// 8 lanes, and the last two steps finish the sum. Returns the value; `row`
// receives the row it belongs to.
__device__ __forceinline__ float transpose_reduce8(const float (&acc)[8], int lane, int& row) {
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
  float v4[4], v2[2];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = b4 ? acc[i] : acc[i + 4];
    const float keep = b4 ? acc[i + 4] : acc[i];
    v4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = b3 ? v4[i] : v4[i + 2];
    const float keep = b3 ? v4[i + 2] : v4[i];
    v2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float send = b2 ? v2[0] : v2[1];
  const float keep = b2 ? v2[1] : v2[0];
  float v = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  row = (b4 ? 4 : 0) + (b3 ? 2 : 0) + (b2 ? 1 : 0);
  return v;
}

// ---------------------------------------------------------------------------
// The streaming kernel. Ring slot s holds stage st (st % S == s); the full
// barrier of a slot completes once per stage and every consumer warp waits
// for every stage in order, so no waiter can mistake an older phase. A slot
// is released (empty barrier, 8 arrivals) only after the stage's finisher
// has read the slot's reduction buffer.
// ---------------------------------------------------------------------------
template <int FMT, int CPW>
__global__ void __launch_bounds__(kGemvThreads, CPW >= 4 ? 1 : 2) gemv_stream_kernel(const GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Header& hd = *reinterpret_cast<Header*>(smem);
  float* As = reinterpret_cast<float*>(smem + kHeaderBytes);
  uint8_t* ring = smem + kHeaderBytes + p.a_bytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int r0 = static_cast<int>((static_cast<long long>(blockIdx.x) * p.N) / G);
  const int r1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * p.N) / G);
  const int nrows = r1 - r0;
  const int RS = p.rows_per_stage, S = p.stages;
  const int nst = (nrows + RS - 1) / RS;
  const uint32_t stage_bytes = static_cast<uint32_t>(RS) * p.row_bytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hd.full[s], 1);
      mbar_init(&hd.empty[s], kConsumerWarps);
      mbar_init(&hd.red_full[s], kConsumerWarps);
    }
    mbar_init(&hd.a_bar, 1);
    hd.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    const uint8_t* wbase = p.W + static_cast<long long>(r0) * p.row_bytes;
    int issued = 0;
    bool a_issued = false, ok = true;
    for (int st = 0; st < nst; ++st) {
      const int s = st % S;
      if (st >= S) {
        if (!mbar_wait(&hd.empty[s], ((st / S) - 1) & 1, p.wait_ns, p.wait_iters) || hd.abort) {
          ok = false;
          break;
        }
      }
      const int rows = min(RS, nrows - st * RS);
      const uint32_t bytes = static_cast<uint32_t>(rows) * p.row_bytes;
      mbar_arrive_expect_tx(&hd.full[s], bytes);
      bulk_g2s(ring + static_cast<size_t>(s) * stage_bytes,
               wbase + static_cast<long long>(st) * RS * p.row_bytes, bytes, &hd.full[s], pol);
      ++issued;
      if (st == 0) {
        // A may come from the previous kernel on the stream: wait for it only
        // now, with the first weight stage already on its way.
        pdl_wait();
        mbar_arrive_expect_tx(&hd.a_bar, p.a_bytes);
        bulk_g2s(As, p.A, p.a_bytes, &hd.a_bar, policy_evict_last());
        a_issued = true;
      }
    }
    if (nst == 0) pdl_wait();
    if (!ok) {
      record_error(kDevErrTimeout);
      hd.abort = 1;
    }
    // Never leave copies in flight: consumers may have given up already.
    for (int st = max(0, issued - S); st < issued; ++st)
      mbar_wait(&hd.full[st % S], (st / S) & 1, kDrainWaitNs);
    if (a_issued) mbar_wait(&hd.a_bar, 0, kDrainWaitNs);
    return;
  }

  // ---------------- consumers ----------------
  pdl_wait();
  if (nrows == 0) return;
  if (!mbar_wait(&hd.a_bar, 0, p.wait_ns, p.wait_iters)) {
    record_error(kDevErrTimeout);
    hd.abort = 1;
    return;
  }
  typename SliceOf<FMT, CPW>::T sl;
  sl.init(smem_u32(As), warp, lane, p.K);
  const uint32_t ring_u = smem_u32(ring);
  for (int st = 0; st < nst; ++st) {
    const int s = st % S;
    const uint32_t ph = (st / S) & 1;
    if (!mbar_wait(&hd.full[s], ph, p.wait_ns, p.wait_iters) || hd.abort) {
      record_error(kDevErrTimeout);
      hd.abort = 1;
      return;
    }
    const int rows = min(RS, nrows - st * RS);
    const uint32_t base = ring_u + static_cast<uint32_t>(s) * stage_bytes;
    float acc[kRowsPerStage];
#pragma unroll
    for (int r = 0; r < kRowsPerStage; ++r) acc[r] = 0.f;
#pragma unroll
    for (int i = 0; i < CPW; ++i) {
      if (sl.ok[i]) {
#pragma unroll
        for (int r = 0; r < kRowsPerStage; ++r)
          if (r < rows) acc[r] += sl.dot(base + static_cast<uint32_t>(r) * p.row_bytes, i);
      }
    }
    int row;
    const float v = transpose_reduce8(acc, lane, row);
    if ((lane & 3) == 0) hd.red[s][warp][row] = v;
    __syncwarp();
    if (lane == 0) mbar_arrive(&hd.red_full[s]);
    if (warp == st % kConsumerWarps) {
      // finisher of this stage: the eight warps' partials, in a fixed order
      if (!mbar_wait(&hd.red_full[s], ph, p.wait_ns, p.wait_iters) || hd.abort) {
        record_error(kDevErrTimeout);
        hd.abort = 1;
        return;
      }
      if (lane < rows) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) sum += hd.red[s][w][lane];
        p.C[r0 + st * RS + lane] = sum;
      }
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(&hd.empty[s]);
  }
}

// ---------------------------------------------------------------------------
// Generic kernel: any M, N, K (quantised K % 32 == 0), any W byte alignment.
// One warp per output element C[m, n]; W is read with byte loads. It is the
// correctness net under the fast kernels, not a performance path.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_f16_bytes(const uint8_t* p) {
  const unsigned short b = static_cast<unsigned short>(p[0]) | (static_cast<unsigned short>(p[1]) << 8);
  return __half2float(__ushort_as_half(b));
}

template <int FMT>
__global__ void __launch_bounds__(256) generic_matmul_kernel(const float* __restrict__ A,
                                                             const uint8_t* __restrict__ W,
                                                             float* __restrict__ C, int M, int N,
                                                             int K, long long row_bytes) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  pdl_wait();
  if (n >= N) return;
  const uint8_t* w = W + static_cast<long long>(n) * row_bytes;
  for (int m = blockIdx.y; m < M; m += gridDim.y) {
    const float* a = A + static_cast<long long>(m) * K;
    float acc = 0.f;
    if (FMT == LQ_FMT_F16) {
      const __half* wh = reinterpret_cast<const __half*>(w);
      for (int k = lane; k < K; k += 32) acc = fmaf(a[k], __half2float(wh[k]), acc);
    } else if (FMT == LQ_FMT_Q8_0) {
      for (int b = lane; b < K / 32; b += 32) {
        const uint8_t* blk = w + 34LL * b;
        float s = 0.f;
        for (int i = 0; i < 32; ++i)
          s = fmaf(static_cast<float>(static_cast<int8_t>(blk[2 + i])), a[32 * b + i], s);
        acc = fmaf(load_f16_bytes(blk), s, acc);
      }
    } else {
      for (int b = lane; b < K / 32; b += 32) {
        const uint8_t* blk = w + 18LL * b;
        float s = 0.f;
        for (int i = 0; i < 16; ++i) {
          const int byte = blk[2 + i];
          s = fmaf(static_cast<float>((byte & 0xF) - 8), a[32 * b + i], s);
          s = fmaf(static_cast<float>((byte >> 4) - 8), a[32 * b + 16 + i], s);
        }
        acc = fmaf(load_f16_bytes(blk), s, acc);
      }
    }
    acc = warp_sum(acc);
    if (lane == 0) C[static_cast<long long>(m) * N + n] = acc;
  }
}

// ---------------------------------------------------------------------------
// launch helpers
// ---------------------------------------------------------------------------
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                   Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Chunks per warp (template set 1, 2, 4, 8) that cover K for this format.
int pick_cpw(int fmt, int K) {
  const int chunk = fmt == LQ_FMT_Q4_0 ? 512 : 256;
  const int nch = (K + chunk - 1) / chunk;
  const int need = (nch + kConsumerWarps - 1) / kConsumerWarps;
  for (int c : {1, 2, 4, 8})
    if (c >= need) return c;
  return 0;
}

template <int FMT, int CPW>
lq_status launch_stream_t(const MatmulArgs& a, const GemvParams& p, int G, size_t smem) {
  auto kern = gemv_stream_kernel<FMT, CPW>;
  static int configured_smem[kMaxDevices] = {};  // per instantiation and device
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_CUDA;
  if (configured_smem[dev] < static_cast<int>(smem)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e);
    configured_smem[dev] = static_cast<int>(smem);
  }
  cudaError_t e = launch(kern, dim3(G), dim3(kGemvThreads), smem, a.stream, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

template <int FMT>
lq_status launch_stream_fmt(const MatmulArgs& a, int cpw, const GemvParams& p, int G, size_t smem) {
  switch (cpw) {
    case 1: return launch_stream_t<FMT, 1>(a, p, G, smem);
    case 2: return launch_stream_t<FMT, 2>(a, p, G, smem);
    case 4: return launch_stream_t<FMT, 4>(a, p, G, smem);
    case 8: return launch_stream_t<FMT, 8>(a, p, G, smem);
    default: return LQ_ERR_UNSUPPORTED;
  }
}

}  // namespace

unsigned read_clear_gemv_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_err, &z, sizeof(z));
  return v;
}

lq_status launch_gemv_generic(const MatmulArgs& a) {
  const dim3 grid(static_cast<unsigned>((a.N + 7) / 8),
                  static_cast<unsigned>(std::min<int64_t>(a.M, 65535)));
  const long long rb = row_bytes(a.fmt, a.K);
  const auto* W = static_cast<const uint8_t*>(a.W);
  const int M = static_cast<int>(a.M), N = static_cast<int>(a.N), K = static_cast<int>(a.K);
  cudaError_t e;
  if (a.fmt == LQ_FMT_F16)
    e = launch(generic_matmul_kernel<LQ_FMT_F16>, grid, dim3(256), 0, a.stream, a.A, W, a.C, M, N, K, rb);
  else if (a.fmt == LQ_FMT_Q8_0)
    e = launch(generic_matmul_kernel<LQ_FMT_Q8_0>, grid, dim3(256), 0, a.stream, a.A, W, a.C, M, N, K, rb);
  else
    e = launch(generic_matmul_kernel<LQ_FMT_Q4_0>, grid, dim3(256), 0, a.stream, a.A, W, a.C, M, N, K, rb);
  if (e == cudaSuccess) e = cudaGetLastError();
  count_route(3);
  return cuda_status(e);
}

// Launch plan of the streaming kernel: grid, ring geometry and shared memory.
struct GemvPlan {
  GemvParams p;
  int grid = 0, cpw = 0;
  size_t smem = 0;
  bool ok = false;
};

// `ctas_per_sm` CTAs share an SM (each gets 1/ctas_per_sm of the usable
// shared memory); stages hold up to `max_rows` rows.
GemvPlan plan_gemv(const MatmulArgs& a, int ctas_per_sm, int max_rows) {
  GemvPlan pl;
  const int K = static_cast<int>(a.K);
  const int rb = static_cast<int>(row_bytes(a.fmt, a.K));
  // Fast path: every stage start and A are 16-byte aligned for the bulk
  // copies (rows a multiple of 16 bytes), and the per-lane slices cover K.
  const bool shape_ok = a.K <= kGemvFastMaxK &&
                        (a.fmt == LQ_FMT_F16 ? (K % 8 == 0) : (K % 256 == 0)) && a.N < (1LL << 30);
  const bool align_ok = aligned(a.W, 16) && aligned(a.A, 16);
  pl.cpw = shape_ok ? pick_cpw(a.fmt, K) : 0;
  if (!shape_ok || !align_ok || pl.cpw == 0) return pl;

  const DeviceInfo& di = device_info();
  const int G = static_cast<int>(std::min<int64_t>(a.N, static_cast<int64_t>(di.sm_count) * ctas_per_sm));
  const int a_bytes = K * 4;  // a multiple of 16 on this path
  const int per_cta = std::min(di.max_smem_optin, (226 * 1024) / ctas_per_sm - 1024);
  const int budget = per_cta - kHeaderBytes - a_bytes;
  const int rows_per_cta = static_cast<int>((a.N + G - 1) / G);
  // up to max_rows rows per bulk copy, and room for at least two stages
  const int rs = std::min({max_rows, kRowsPerStage, std::max(1, budget / (2 * rb)),
                           std::max(1, rows_per_cta)});
  const int stage_bytes = rs * rb;
  const int need_stages = (rows_per_cta + rs - 1) / rs;
  const int stages = std::min({kMaxStages, budget / std::max(stage_bytes, 1), std::max(need_stages, 2)});
  if (G < 1 || budget <= 0 || stages < 2) return pl;

  GemvParams& p = pl.p;
  p.A = a.A;
  p.W = static_cast<const uint8_t*>(a.W);
  p.C = a.C;
  p.N = static_cast<int>(a.N);
  p.K = K;
  p.row_bytes = rb;
  p.rows_per_stage = rs;
  p.stages = stages;
  p.a_bytes = a_bytes;
  p.wait_ns = wait_limit_ns();
  p.wait_iters = wait_limit_iters();
  pl.grid = G;
  pl.smem = kHeaderBytes + a_bytes + static_cast<size_t>(stages) * stage_bytes;
  pl.ok = true;
  return pl;
}

lq_status launch_plan(const MatmulArgs& a, const GemvPlan& pl) {
  if (a.fmt == LQ_FMT_F16) return launch_stream_fmt<LQ_FMT_F16>(a, pl.cpw, pl.p, pl.grid, pl.smem);
  if (a.fmt == LQ_FMT_Q8_0) return launch_stream_fmt<LQ_FMT_Q8_0>(a, pl.cpw, pl.p, pl.grid, pl.smem);
  return launch_stream_fmt<LQ_FMT_Q4_0>(a, pl.cpw, pl.p, pl.grid, pl.smem);
}

lq_status launch_gemv(const MatmulArgs& a) {
  // Two CTAs per SM: twice the warps to hide shared-memory and ALU latency,
  // and room for the next kernel's CTAs to start while this one drains
  // (programmatic dependent launch). Measured on GB300 against one CTA per
  // SM: LM head 4.45 -> 6.57 TB/s, Q8_0 4096x4096 1.79 -> 2.49 TB/s.
  GemvPlan pl = plan_gemv(a, 2, kRowsPerStage);
  // very long rows: half the shared memory cannot hold two stages
  if (!pl.ok) pl = plan_gemv(a, 1, kRowsPerStage);
  if (!pl.ok) return launch_gemv_generic(a);
  const lq_status st = launch_plan(a, pl);
  if (st == LQ_ERR_UNSUPPORTED) return launch_gemv_generic(a);
  if (st == LQ_OK) count_route(0);
  return st;
}

}  // namespace lq
