// Per-format GEMV slices and the warp reduction, shared by the streaming
// GEMV (lq_gemv.cu) and the persistent chain engine (lq_gemv_chain.cu).
#pragma once

#include "lq.h"
#include "lq_device.cuh"

namespace lq {
namespace gemv {

// ---------------------------------------------------------------------------
// Per-format slices. A "chunk" is the part of a row that one warp covers in
// one pass: 32 lanes x 8 elements (f16, Q8_0) or 32 lanes x 16 elements
// (Q4_0). The warp of K-group kg (of nk) takes chunks kg, kg+nk, kg+2nk, ...
// of each of its rows; a lane holds the activations of its part of each of
// its chunks in registers (read once from global memory).
// ---------------------------------------------------------------------------

// f16: chunk = 256 halves = 512 bytes; lane l reads bytes [16l, 16l+16).
template <int CPW>
struct F16Slice {
  float2 a[CPW][4];
  uint32_t off[CPW];  // byte offset of the lane's 16 bytes within a row
  bool ok[CPW];
  // sA: the activations in shared memory, in order (a_layout_f16).
  __device__ __forceinline__ void init(uint32_t sA, int kg, int nk, int lane, int K) {
    const int nch = (K + 255) / 256;
#pragma unroll
    for (int i = 0; i < CPW; ++i) {
      const int c = kg + nk * i;
      const int e = 256 * c + 8 * lane;
      ok[i] = c < nch && e < K;
      off[i] = 2u * static_cast<uint32_t>(e);
      if (ok[i]) {
        const float4 x = lds128f(sA + 4u * e), y = lds128f(sA + 4u * e + 16u);
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
  }};

// Quantised formats, one whole block per lane. K-group kg covers segments
// kg/2 + (nk/2)*c (c < CPW; 64 blocks = 2048 values each) and, of them, the
// blocks of parity kg%2: lane l takes block 64*seg + 2l + parity, so a
// warp's 32 blocks of a segment are every other block of it. Their activations sit in shared memory
// at slot (2*seg + parity)*32 + l, 144 bytes apart (a_slot_q): 144 is an odd
// multiple of 16, so the lanes' 16-byte loads fall in eight different bank
// groups.
__host__ __device__ __forceinline__ int a_slot_q(int b) { return (2 * (b >> 6) + (b & 1)) * 32 + ((b & 63) >> 1); }
constexpr int kASlotBytes = 144;

// Q8_0 (34-byte blocks): the lane's block spans nine 32-bit words starting
// at word 17l of the segment (+8 for odd blocks, whose scale sits in the
// upper half of that first word). 17 is odd, so for each of the nine loads
// the 32 lanes hit 32 different banks: every byte is read once, with no bank
// conflicts. Even blocks start with their scale, so their quants are 2 bytes
// past a word boundary; odd blocks' quants are word-aligned. One code path
// serves both parities (the parity is the same for the whole warp): each
// word of quants is a funnel shift of two loaded words by 16 bits (even) or
// 32 (odd: the second word as is). Per-parity code saves those eight shifts
// a block but doubles the dot's instructions in the kernel, and the smaller
// footprint measured faster in every kernel that uses the slices (the
// decode chain: Q8_0 4096x4096 3.72 against 4.05 us a GEMV).
template <int CPW>
struct Q8Slice {
  float2 a[CPW][16];       // the blocks' activations
  uint32_t woff[CPW];      // byte offset of the lane's first word in the row
  bool odd;                // block parity (warp-uniform)
  bool ok[CPW];
  __device__ __forceinline__ void init(uint32_t sA, int kg, int nk, int lane, int K) {
    const int par = kg & 1;
    odd = par != 0;
#pragma unroll
    for (int c = 0; c < CPW; ++c) {
      const int seg = (kg >> 1) + (nk >> 1) * c;
      const int b = 64 * seg + 2 * lane + par;
      ok[c] = b < K / 32;
      woff[c] = 2176u * seg + 68u * lane + (par ? 32u : 0u);
      const uint32_t src = sA + static_cast<uint32_t>(a_slot_q(b)) * kASlotBytes;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float4 x = ok[c] ? lds128f(src + 16u * t) : make_float4(0.f, 0.f, 0.f, 0.f);
        a[c][2 * t] = make_float2(x.x, x.y);
        a[c][2 * t + 1] = make_float2(x.z, x.w);
      }
    }
  }
  __device__ __forceinline__ float dot(uint32_t row, int c) const {
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = lds32(row + woff[c] + 4u * i);
    const float d = f16_lo(w[0] >> (odd ? 16 : 0));
    const uint32_t sh = odd ? 32u : 16u;
    const float2 mb = make_float2(-kMagicS8, -kMagicS8);
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t x = __funnelshift_rc(w[i], w[i + 1], sh) ^ 0x80808080u;  // q_{4i..4i+3}, sign flipped
      const float2 q01 = fadd2(make_float2(s8_to_magic(x, 0), s8_to_magic(x, 1)), mb);
      const float2 q23 = fadd2(make_float2(s8_to_magic(x, 2), s8_to_magic(x, 3)), mb);
      acc[(2 * i) & 3] = ffma2(q01, a[c][2 * i], acc[(2 * i) & 3]);
      acc[(2 * i + 1) & 3] = ffma2(q23, a[c][2 * i + 1], acc[(2 * i + 1) & 3]);
    }
    const float2 s = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
    return d * (s.x + s.y);
  }
};

// Q4_0 (18-byte blocks): the lane's block spans five words starting at word
// 9l of the segment (+4 for odd blocks); 9 is odd, so again conflict-free.
// Byte j of the 16 nibble bytes holds q_j (low nibble) and q_{j+16} (high).
// For a word of four such bytes, masking with 0x0F0F0F0F leaves the four low
// codes as bytes and masking with 0xF0F0F0F0 the four high codes times 16
// (no shift); each byte goes into the mantissa of 2^23 with one byte-permute
// as in Q8_0, and one packed add per pair gives q - 8 exactly, or 16 (q - 8)
// with Q8_0's bias of 2^23 + 128. The high half's partial sums are thus 16
// times the products' and come back at the block's end with one exact
// packed multiply-add by 1/16 in place of the add: scaling by 16 commutes
// with rounding, so the sums are the same bits as with the codes themselves
// (outside f32's subnormal range, where they are closer), for activations
// below about 2^119 in magnitude (2^123 with the codes themselves). (Pulling
// each nibble in place with its own scale, one fma per pair, needs four
// constant pairs per word and measured about 30 % more instructions.) The
// words are aligned by the same funnel shift as Q8_0's, one code path for
// both parities.
template <int CPW>
struct Q4Slice {
  float2 a[CPW][16];       // a[2t], a[2t+1]: elements 4t .. 4t+3; a[8+2t], a[9+2t]: 16+4t ..
  uint32_t woff[CPW];
  bool odd;
  bool ok[CPW];
  __device__ __forceinline__ void init(uint32_t sA, int kg, int nk, int lane, int K) {
    const int par = kg & 1;
    odd = par != 0;
#pragma unroll
    for (int c = 0; c < CPW; ++c) {
      const int seg = (kg >> 1) + (nk >> 1) * c;
      const int b = 64 * seg + 2 * lane + par;
      ok[c] = b < K / 32;
      woff[c] = 1152u * seg + 36u * lane + (par ? 16u : 0u);
      const uint32_t src = sA + static_cast<uint32_t>(a_slot_q(b)) * kASlotBytes;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float4 lo = ok[c] ? lds128f(src + 16u * t) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 hi = ok[c] ? lds128f(src + 64u + 16u * t) : make_float4(0.f, 0.f, 0.f, 0.f);
        a[c][2 * t] = make_float2(lo.x, lo.y);
        a[c][2 * t + 1] = make_float2(lo.z, lo.w);
        a[c][8 + 2 * t] = make_float2(hi.x, hi.y);
        a[c][9 + 2 * t] = make_float2(hi.z, hi.w);
      }
    }
  }
  __device__ __forceinline__ float dot(uint32_t row, int c) const {
    uint32_t w[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) w[i] = lds32(row + woff[c] + 4u * i);
    const float d = f16_lo(w[0] >> (odd ? 16 : 0));
    const uint32_t sh = odd ? 32u : 16u;
    const float2 m8 = make_float2(-kMagicQ4, -kMagicQ4);
    const float2 m128 = make_float2(-kMagicS8, -kMagicS8);  // 2^23 + 16 q - (2^23 + 128) = 16 (q - 8)
    float2 acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = __funnelshift_rc(w[i], w[i + 1], sh);  // bytes 4i .. 4i+3
      const uint32_t lo = x & 0x0F0F0F0Fu, hi16 = x & 0xF0F0F0F0u;
      const float2 l01 = fadd2(make_float2(s8_to_magic(lo, 0), s8_to_magic(lo, 1)), m8);
      const float2 l23 = fadd2(make_float2(s8_to_magic(lo, 2), s8_to_magic(lo, 3)), m8);
      const float2 h01 = fadd2(make_float2(s8_to_magic(hi16, 0), s8_to_magic(hi16, 1)), m128);
      const float2 h23 = fadd2(make_float2(s8_to_magic(hi16, 2), s8_to_magic(hi16, 3)), m128);
      acc[0] = ffma2(l01, a[c][2 * i], acc[0]);
      acc[1] = ffma2(l23, a[c][2 * i + 1], acc[1]);
      acc[2] = ffma2(h01, a[c][8 + 2 * i], acc[2]);  // 16 x the high codes' products
      acc[3] = ffma2(h23, a[c][9 + 2 * i], acc[3]);
    }
    const float2 s = ffma2(fadd2(acc[2], acc[3]), make_float2(0.0625f, 0.0625f), fadd2(acc[0], acc[1]));
    return d * (s.x + s.y);
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

}  // namespace gemv
}  // namespace lq
