// Multi-token slices of the batched decode kernel (lq_gemv_batch.cu): the
// lane mapping of the one-token slices in lq_gemv_slices.cuh, with the weights
// dequantised once and multiplied with up to eight activation rows.
#pragma once
#include "lq_gemv_slices.cuh"

namespace lq {
namespace gemv {

// ---------------------------------------------------------------------------
// Multi-token slices for the batched decode kernel (M = 2..8 activation
// rows): the lane mapping of the one-token slices, one chunk per warp, the
// weights dequantised once and multiplied with MT activation rows. Token t's
// activations sit at sA + t * a_stride in the layout of the one-token slice.
// ---------------------------------------------------------------------------
template <int MT>
struct F16SliceM {
  float2 a[MT][4];
  uint32_t off;
  bool ok;
  __device__ __forceinline__ void init(uint32_t sA, uint32_t a_stride, int kg, int lane, int K) {
    const int nch = (K + 255) / 256;
    const int e = 256 * kg + 8 * lane;
    ok = kg < nch && e < K;
    off = 2u * static_cast<uint32_t>(e);
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const uint32_t src = sA + a_stride * t + 4u * e;
      const float4 x = ok ? lds128f(src) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 y = ok ? lds128f(src + 16u) : make_float4(0.f, 0.f, 0.f, 0.f);
      a[t][0] = make_float2(x.x, x.y);
      a[t][1] = make_float2(x.z, x.w);
      a[t][2] = make_float2(y.x, y.y);
      a[t][3] = make_float2(y.z, y.w);
    }
  }
  __device__ __forceinline__ void dot(uint32_t row, float (&out)[MT]) const {
    const uint4 v = lds128(row + off);
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&v.z));
    const float2 f3 = __half22float2(*reinterpret_cast<const __half2*>(&v.w));
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      float2 acc = ffma2(f0, a[t][0], make_float2(0.f, 0.f));
      float2 acc1 = ffma2(f1, a[t][1], make_float2(0.f, 0.f));
      acc = ffma2(f2, a[t][2], acc);
      acc1 = ffma2(f3, a[t][3], acc1);
      out[t] = (acc.x + acc1.x) + (acc.y + acc1.y);
    }
  }};

// Q8_0 / Q4_0: one whole block per lane (see Q8Slice / Q4Slice for the
// mapping and the bank argument); the block's 32 values are dequantised into
// registers once, then dotted with each token's 32 activations.
template <int MT>
struct Q8SliceM {
  float2 a[MT][16];
  uint32_t woff;
  bool odd, ok;
  __device__ __forceinline__ void init(uint32_t sA, uint32_t a_stride, int kg, int lane, int K) {
    const int seg = kg >> 1, par = kg & 1;
    const int b = 64 * seg + 2 * lane + par;
    ok = b < K / 32;
    odd = par != 0;
    woff = 2176u * seg + 68u * lane + (par ? 32u : 0u);
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const uint32_t src = sA + a_stride * t + static_cast<uint32_t>(a_slot_q(b)) * kASlotBytes;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = ok ? lds128f(src + 16u * u) : make_float4(0.f, 0.f, 0.f, 0.f);
        a[t][2 * u] = make_float2(x.x, x.y);
        a[t][2 * u + 1] = make_float2(x.z, x.w);
      }
    }
  }
  // the block's codes q (paired as a[t]) times each token's activations
  __device__ __forceinline__ void fma_tokens(const float2 (&q)[16], float d, float (&out)[MT]) const {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      float2 acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i & 3] = ffma2(q[i], a[t][i], acc[i & 3]);
      const float2 s = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
      out[t] = d * (s.x + s.y);
    }
  }
  // one code path for both block parities (as Q8Slice::dot)
  __device__ __forceinline__ void dot(uint32_t row, float (&out)[MT]) const {
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = lds32(row + woff + 4u * i);
    const float d = f16_lo(w[0] >> (odd ? 16 : 0));
    const uint32_t sh = odd ? 32u : 16u;
    const float2 mb = make_float2(-kMagicS8, -kMagicS8);
    float2 q[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t x = __funnelshift_rc(w[i], w[i + 1], sh) ^ 0x80808080u;
      q[2 * i] = fadd2(make_float2(s8_to_magic(x, 0), s8_to_magic(x, 1)), mb);
      q[2 * i + 1] = fadd2(make_float2(s8_to_magic(x, 2), s8_to_magic(x, 3)), mb);
    }
    fma_tokens(q, d, out);
  }
};

template <int MT>
struct Q4SliceM {
  float2 a[MT][16];  // a[t][2u], a[t][2u+1]: elements 4u .. 4u+3; a[t][8+2u], a[t][9+2u]: 16+4u ..
  uint32_t woff;
  bool odd, ok;
  __device__ __forceinline__ void init(uint32_t sA, uint32_t a_stride, int kg, int lane, int K) {
    const int seg = kg >> 1, par = kg & 1;
    const int b = 64 * seg + 2 * lane + par;
    ok = b < K / 32;
    odd = par != 0;
    woff = 1152u * seg + 36u * lane + (par ? 16u : 0u);
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const uint32_t src = sA + a_stride * t + static_cast<uint32_t>(a_slot_q(b)) * kASlotBytes;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 lo = ok ? lds128f(src + 16u * u) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 hi = ok ? lds128f(src + 64u + 16u * u) : make_float4(0.f, 0.f, 0.f, 0.f);
        a[t][2 * u] = make_float2(lo.x, lo.y);
        a[t][2 * u + 1] = make_float2(lo.z, lo.w);
        a[t][8 + 2 * u] = make_float2(hi.x, hi.y);
        a[t][9 + 2 * u] = make_float2(hi.z, hi.w);
      }
    }
  }
  // the codes once (as Q4Slice: masked into bytes, each into the 2^23
  // magic), then one set of packed fmas per token
  // the block's codes q (paired as a[t]) times each token's activations
  __device__ __forceinline__ void fma_tokens(const float2 (&q)[16], float d, float (&out)[MT]) const {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      float2 acc[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i & 3] = ffma2(q[i], a[t][i], acc[i & 3]);
      const float2 s = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
      out[t] = d * (s.x + s.y);
    }
  }
  // one code path for both block parities (as Q8Slice::dot)
  __device__ __forceinline__ void dot(uint32_t row, float (&out)[MT]) const {
    uint32_t w[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) w[i] = lds32(row + woff + 4u * i);
    const float d = f16_lo(w[0] >> (odd ? 16 : 0));
    const uint32_t sh = odd ? 32u : 16u;
    const float2 m8 = make_float2(-kMagicQ4, -kMagicQ4);
    float2 q[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = __funnelshift_rc(w[i], w[i + 1], sh);
      const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
      q[2 * i] = fadd2(make_float2(s8_to_magic(lo, 0), s8_to_magic(lo, 1)), m8);
      q[2 * i + 1] = fadd2(make_float2(s8_to_magic(lo, 2), s8_to_magic(lo, 3)), m8);
      q[8 + 2 * i] = fadd2(make_float2(s8_to_magic(hi, 0), s8_to_magic(hi, 1)), m8);
      q[9 + 2 * i] = fadd2(make_float2(s8_to_magic(hi, 2), s8_to_magic(hi, 3)), m8);
    }
    fma_tokens(q, d, out);
  }
};

// ---------------------------------------------------------------------------
// Half-block slices for five to eight activation rows (MT = 8): a lane holds
// 16 weights of a block for every token, so eight tokens' activations take
// the registers four tokens' whole blocks take. K-group kg covers segment
// kg/4, block parity kg%2 and half (kg/2)%2 of every block: lane l takes
// block 64*seg + 2l + parity, as the whole-block slices (the 17-word (Q8_0)
// and 9-word (Q4_0) lane strides stay conflict-free), and of it one half.
// Each weight is still dequantised once, by the lane that owns its half.
// ---------------------------------------------------------------------------
// Q8_0: half h holds codes 16h .. 16h+15. Relative to the lane's first word
// (woff, as Q8SliceM), the codes start at byte 2 + 16h (even blocks) or
// 4 + 16h (odd: the block starts 2 bytes into its first word); in both cases
// words 4h .. 4h+4 hold them, aligned by the same funnel shift (16 bits even,
// 32 odd) as the whole-block slices. The scale sits in word 0.
template <int MT>
struct Q8HalfSliceM {
  float2 a[MT][8];
  uint32_t woff, woff_h;  // the block's first word; the first word of the half's codes
  bool odd, ok;
  __device__ __forceinline__ void init(uint32_t sA, uint32_t a_stride, int kg, int lane, int K) {
    const int seg = kg >> 2, par = kg & 1, h = (kg >> 1) & 1;
    const int b = 64 * seg + 2 * lane + par;
    ok = b < K / 32;
    odd = par != 0;
    woff = 2176u * seg + 68u * lane + (par ? 32u : 0u);
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const uint32_t src = sA + a_stride * t + static_cast<uint32_t>(a_slot_q(b)) * kASlotBytes + 64u * h;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 x = ok ? lds128f(src + 16u * u) : make_float4(0.f, 0.f, 0.f, 0.f);
        a[t][2 * u] = make_float2(x.x, x.y);
        a[t][2 * u + 1] = make_float2(x.z, x.w);
      }
    }
    woff_h = woff + 16u * h;
  }
  __device__ __forceinline__ void fma_tokens(const float2 (&q)[8], float d, float (&out)[MT]) const {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        acc0 = ffma2(q[i], a[t][i], acc0);
        acc1 = ffma2(q[i + 1], a[t][i + 1], acc1);
      }
      const float2 s = fadd2(acc0, acc1);
      out[t] = d * (s.x + s.y);
    }
  }
  __device__ __forceinline__ void dot(uint32_t row, float (&out)[MT]) const {
    const uint32_t w0 = lds32(row + woff);
    uint32_t w[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) w[i] = lds32(row + woff_h + 4u * i);
    const float d = f16_lo(w0 >> (odd ? 16 : 0));
    const uint32_t sh = odd ? 32u : 16u;
    const float2 mb = make_float2(-kMagicS8, -kMagicS8);
    float2 q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = __funnelshift_rc(w[i], w[i + 1], sh) ^ 0x80808080u;
      q[2 * i] = fadd2(make_float2(s8_to_magic(x, 0), s8_to_magic(x, 1)), mb);
      q[2 * i + 1] = fadd2(make_float2(s8_to_magic(x, 2), s8_to_magic(x, 3)), mb);
    }
    fma_tokens(q, d, out);
  }
};

// Q4_0: half h holds nibble bytes 8h .. 8h+7, i.e. codes 8h .. 8h+7 (low
// nibbles) and 16+8h .. 16+8h+7 (high). Relative to woff (as Q4SliceM) the
// bytes start at 2 + 8h (even) or 4 + 8h (odd), inside words 2h .. 2h+2,
// aligned by the same funnel shift; the scale sits in word 0.
template <int MT>
struct Q4HalfSliceM {
  float2 a[MT][8];  // a[t][0..3]: codes 8h .. 8h+7; a[t][4..7]: codes 16+8h ..
  uint32_t woff, woff_h;
  bool odd, ok;
  __device__ __forceinline__ void init(uint32_t sA, uint32_t a_stride, int kg, int lane, int K) {
    const int seg = kg >> 2, par = kg & 1, h = (kg >> 1) & 1;
    const int b = 64 * seg + 2 * lane + par;
    ok = b < K / 32;
    odd = par != 0;
    woff = 1152u * seg + 36u * lane + (par ? 16u : 0u);
    woff_h = woff + 8u * h;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      const uint32_t src = sA + a_stride * t + static_cast<uint32_t>(a_slot_q(b)) * kASlotBytes;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float4 lo = ok ? lds128f(src + 32u * h + 16u * u) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 hi = ok ? lds128f(src + 64u + 32u * h + 16u * u) : make_float4(0.f, 0.f, 0.f, 0.f);
        a[t][2 * u] = make_float2(lo.x, lo.y);
        a[t][2 * u + 1] = make_float2(lo.z, lo.w);
        a[t][4 + 2 * u] = make_float2(hi.x, hi.y);
        a[t][5 + 2 * u] = make_float2(hi.z, hi.w);
      }
    }
  }
  __device__ __forceinline__ void fma_tokens(const float2 (&q)[8], float d, float (&out)[MT]) const {
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        acc0 = ffma2(q[i], a[t][i], acc0);
        acc1 = ffma2(q[i + 1], a[t][i + 1], acc1);
      }
      const float2 s = fadd2(acc0, acc1);
      out[t] = d * (s.x + s.y);
    }
  }
  __device__ __forceinline__ void dot(uint32_t row, float (&out)[MT]) const {
    const uint32_t w0 = lds32(row + woff);
    uint32_t w[3];
#pragma unroll
    for (int i = 0; i < 3; ++i) w[i] = lds32(row + woff_h + 4u * i);
    const float d = f16_lo(w0 >> (odd ? 16 : 0));
    const uint32_t sh = odd ? 32u : 16u;
    const float2 m8 = make_float2(-kMagicQ4, -kMagicQ4);
    float2 q[8];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t x = __funnelshift_rc(w[i], w[i + 1], sh);  // nibble bytes 8h+4i .. 8h+4i+3
      const uint32_t lo = x & 0x0F0F0F0Fu, hi = (x >> 4) & 0x0F0F0F0Fu;
      q[2 * i] = fadd2(make_float2(s8_to_magic(lo, 0), s8_to_magic(lo, 1)), m8);
      q[2 * i + 1] = fadd2(make_float2(s8_to_magic(lo, 2), s8_to_magic(lo, 3)), m8);
      q[4 + 2 * i] = fadd2(make_float2(s8_to_magic(hi, 0), s8_to_magic(hi, 1)), m8);
      q[5 + 2 * i] = fadd2(make_float2(s8_to_magic(hi, 2), s8_to_magic(hi, 3)), m8);
    }
    fma_tokens(q, d, out);
  }
};

// K-groups a segment of 64 blocks takes: two parities, and for the
// half-block slices two halves each.
__host__ __device__ constexpr int kgroups_per_segment(int mt) { return mt > 4 ? 4 : 2; }

template <int FMT, int MT>
struct SliceM;
template <int MT> struct SliceM<LQ_FMT_F16, MT> { using T = F16SliceM<MT>; };
template <int MT> struct SliceM<LQ_FMT_Q8_0, MT> { using T = Q8SliceM<MT>; };
template <int MT> struct SliceM<LQ_FMT_Q4_0, MT> { using T = Q4SliceM<MT>; };
template <> struct SliceM<LQ_FMT_Q8_0, 8> { using T = Q8HalfSliceM<8>; };
template <> struct SliceM<LQ_FMT_Q4_0, 8> { using T = Q4HalfSliceM<8>; };

}  // namespace gemv
}  // namespace lq
