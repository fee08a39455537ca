// Host-side packers: f32 weights -> f16 / Q8_0 / Q4_0 bytes (CPU only).
//
// Counterparts: make_buffer_f16, quantize_row_q8_0 and make_buffer_q4_0 in
// lattice-inference 0.1.2, src/forward/metal_qwen35.rs (packing happens once
// at model load, off the decode path). The Q4_0 rule, which the page imports
// but does not print, is the matmul statement's: m = the signed element of
// largest magnitude (first index on ties), d = m / -8, q = min(15,
// (int)(x/d + 8.5)), low nibbles = elements 0-15, high nibbles = 16-31.
// Q8_0 divides x by the float32 d (d = max|x| / 127) and rounds halves away
// from zero; both formats store the f16 of the float32 d, little-endian.
//
// Narrowing to f16 uses the compiler's IEEE conversion (_Float16, round to
// nearest even). Large inputs are packed on several host threads; the result
// does not depend on the thread count. Compiled without fp contraction.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "../../include/lq.h"

namespace {

inline uint16_t to_f16_bits(float x) {
  const _Float16 h = static_cast<_Float16>(x);
  uint16_t b;
  std::memcpy(&b, &h, 2);
  return b;
}

inline void put_d(uint8_t* dst, float d) {
  const uint16_t b = to_f16_bits(d);
  dst[0] = static_cast<uint8_t>(b & 0xFF);
  dst[1] = static_cast<uint8_t>(b >> 8);
}

// reciprocal: q = round(x * (1/d)) as quantize_row_q8_0 computes it;
// otherwise q = round(x / d) as the matmul statement writes it
void q8_0_block(const float* x, uint8_t* out, bool reciprocal) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) amax = std::fmax(amax, std::fabs(x[i]));
  const float d = amax / 127.0f;
  const float id = d != 0.0f ? 1.0f / d : 0.0f;
  put_d(out, d);
  for (int i = 0; i < 32; ++i) {
    int q = 0;
    if (d != 0.0f) {
      const float v = reciprocal ? x[i] * id : x[i] / d;
      float r = std::round(v);  // halves away from zero
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      q = static_cast<int>(r);
    }
    out[2 + i] = static_cast<uint8_t>(static_cast<int8_t>(q));
  }
}

// interleaved: byte j holds elements 2j (low nibble) and 2j+1 (high), the
// order gemv_q4_decode reads; otherwise elements j and j+16
void q4_0_block(const float* x, uint8_t* out, bool interleaved) {
  float m = x[0], amax = std::fabs(x[0]);
  for (int i = 1; i < 32; ++i) {
    const float a = std::fabs(x[i]);
    if (a > amax) {
      amax = a;
      m = x[i];
    }
  }
  const float d = m / -8.0f;
  put_d(out, d);
  uint8_t q[32];
  for (int i = 0; i < 32; ++i) {
    if (d == 0.0f) {
      q[i] = 8;
    } else {
      const float t = x[i] / d + 8.5f;
      int v = static_cast<int>(t);  // t >= 0.5: truncation is floor
      if (v > 15) v = 15;
      q[i] = static_cast<uint8_t>(v);
    }
  }
  for (int j = 0; j < 16; ++j) {
    const int lo = interleaved ? q[2 * j] : q[j], hi = interleaved ? q[2 * j + 1] : q[j + 16];
    out[2 + j] = static_cast<uint8_t>((lo & 0xF) | ((hi & 0xF) << 4));
  }
}

bool all_finite(const float* W, int64_t n) {
  for (int64_t i = 0; i < n; ++i)
    if (!std::isfinite(W[i])) return false;
  return true;
}

// Runs body(row_begin, row_end) over [0, N) on up to hardware_concurrency threads.
template <typename F>
void parallel_rows(int64_t N, int64_t work_per_row, F body) {
  const int64_t total = N * work_per_row;
  unsigned nt = std::thread::hardware_concurrency();
  if (nt == 0) nt = 1;
  if (total < (1 << 22)) nt = 1;
  if (nt > 64) nt = 64;
  if (static_cast<int64_t>(nt) > N) nt = static_cast<unsigned>(N);
  if (nt <= 1) {
    body(0, N);
    return;
  }
  std::vector<std::thread> th;
  for (unsigned t = 0; t < nt; ++t) {
    const int64_t b = N * t / nt, e = N * (t + 1) / nt;
    th.emplace_back([=] { body(b, e); });
  }
  for (auto& x : th) x.join();
}

bool shape_ok(int64_t N, int64_t K, bool quant) {
  if (N < 0 || K < 0) return false;
  if (quant && (K == 0 || K % 32 != 0)) return false;
  return true;
}

}  // namespace

namespace {
lq_status pack_q8(const float* W, int64_t N, int64_t K, void* out, bool reciprocal) {
  if (!shape_ok(N, K, true) || (N > 0 && (!W || !out))) return LQ_ERR_INVALID_ARG;
  if (!all_finite(W, N * K)) return LQ_ERR_INVALID_ARG;
  const int64_t nb = K / 32;
  auto* o = static_cast<uint8_t*>(out);
  parallel_rows(N, K, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n)
      for (int64_t j = 0; j < nb; ++j) q8_0_block(W + n * K + 32 * j, o + (n * nb + j) * 34, reciprocal);
  });
  return LQ_OK;
}

lq_status pack_q4(const float* W, int64_t N, int64_t K, void* out, bool interleaved) {
  if (!shape_ok(N, K, true) || (N > 0 && (!W || !out))) return LQ_ERR_INVALID_ARG;
  if (!all_finite(W, N * K)) return LQ_ERR_INVALID_ARG;
  const int64_t nb = K / 32;
  auto* o = static_cast<uint8_t*>(out);
  parallel_rows(N, K, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n)
      for (int64_t j = 0; j < nb; ++j) q4_0_block(W + n * K + 32 * j, o + (n * nb + j) * 18, interleaved);
  });
  return LQ_OK;
}
}  // namespace

extern "C" {

size_t lq_packed_bytes(int fmt, int64_t N, int64_t K) {
  if (fmt == LQ_FMT_F16) return shape_ok(N, K, false) ? static_cast<size_t>(N * K * 2) : 0;
  if (fmt == LQ_FMT_Q8_0) return shape_ok(N, K, true) ? static_cast<size_t>(N * (K / 32) * 34) : 0;
  if (fmt == LQ_FMT_Q4_0 || fmt == LQ_FMT_Q4_0I) return shape_ok(N, K, true) ? static_cast<size_t>(N * (K / 32) * 18) : 0;
  return 0;
}

lq_status lq_pack_f16(const float* W, int64_t N, int64_t K, void* out) {
  if (!shape_ok(N, K, false) || (N * K > 0 && (!W || !out))) return LQ_ERR_INVALID_ARG;
  if (!all_finite(W, N * K)) return LQ_ERR_INVALID_ARG;
  auto* o = static_cast<uint8_t*>(out);
  parallel_rows(N, K, [&](int64_t b, int64_t e) {
    for (int64_t i = b * K; i < e * K; ++i) {
      const uint16_t h = to_f16_bits(W[i]);
      o[2 * i] = static_cast<uint8_t>(h & 0xFF);
      o[2 * i + 1] = static_cast<uint8_t>(h >> 8);
    }
  });
  return LQ_OK;
}


lq_status lq_pack_q8_0(const float* W, int64_t N, int64_t K, void* out) { return pack_q8(W, N, K, out, false); }
lq_status lq_pack_q8_0_rcp(const float* W, int64_t N, int64_t K, void* out) { return pack_q8(W, N, K, out, true); }
lq_status lq_pack_q4_0(const float* W, int64_t N, int64_t K, void* out) { return pack_q4(W, N, K, out, false); }
lq_status lq_pack_q4_0i(const float* W, int64_t N, int64_t K, void* out) { return pack_q4(W, N, K, out, true); }

}  // extern "C"
