// Device helpers of the argmax entry points (lq_gemv_argmax, lq_argmax_f32).
//
// The order is the one of topk_better in the source pages (lattice-inference
// 0.1.2, src/forward/metal_qwen35.rs, the top-k kernels): the larger value
// ranks first, equal values rank by the lower index, NaN never ranks first;
// the "nothing found" result is the pages' sentinel (-inf, UINT_MAX), which
// reads as index -1 here.
//
// A candidate (v, i) is packed into one 64-bit key whose unsigned order is
// that ranking, so that the merge is a plain atomicMax:
//   high word: the f32 bits of v mapped to an unsigned order (negative
//              values flipped, positive ones offset by the sign bit), with
//              -0 taken as +0 so that the two compare equal as floats do;
//   low word : 0xFFFFFFFF - i (the lower index has the larger word).
// NaN gets key 0, below every real candidate; a real -inf at index i keeps a
// non-zero low word, so it still beats "nothing".
//
// The merge across CTAs needs no barrier: each warp folds its best key into
// the result with one atomicMax, then counts itself done; the warp that
// counts last reads the key back and writes (value, index). Warps that gave
// up on a timed-out wait never count, so the result is left unwritten and
// the device status word holds the timeout.
#pragma once
#include <cstdint>

#include "../../include/lq.h"

namespace lq {
namespace amax {

__device__ __forceinline__ unsigned long long make_key(float v, unsigned idx) {
  if (v != v) return 0ull;
  v += 0.0f;  // -0 -> +0
  const unsigned u = __float_as_uint(v);
  const unsigned hi = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(hi) << 32) | (0xFFFFFFFFu - idx);
}

__device__ __forceinline__ unsigned long long warp_max(unsigned long long k) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, k, off);
    k = o > k ? o : k;
  }
  return k;
}

__device__ __forceinline__ void decode(unsigned long long key, lq_argmax_result* out) {
  if (key == 0ull) {
    out->value = -__int_as_float(0x7f800000);  // -inf
    out->index = -1;
    return;
  }
  const unsigned hi = static_cast<unsigned>(key >> 32);
  const unsigned lo = static_cast<unsigned>(key);
  const unsigned u = (hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi;
  out->value = __uint_as_float(u);
  out->index = static_cast<int32_t>(0xFFFFFFFFu - lo);
}

// Called by all 32 lanes of a warp that has finished its share; `key` is the
// lane's best candidate key (0 if none). `total` is the number of warps that
// call this for the result `out` (whose work words were zeroed before the
// launch).
__device__ __forceinline__ void warp_done(unsigned long long key, lq_argmax_result* out,
                                          unsigned total, int lane) {
  key = warp_max(key);
  if (lane == 0) {
    unsigned long long* best = reinterpret_cast<unsigned long long*>(&out->work[0]);
    unsigned* count = reinterpret_cast<unsigned*>(&out->work[1]);
    if (key) atomicMax(best, key);
    __threadfence();
    if (atomicAdd(count, 1u) == total - 1u) {
      __threadfence();
      decode(atomicAdd(best, 0ull), out);
    }
  }
  __syncwarp();
}

}  // namespace amax
}  // namespace lq
