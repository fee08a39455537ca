// lq_topk_f32 / lq_gemv_topk: the k best entries of a vector (k <= 64),
// best first, in the order of topk_better (lattice-inference 0.1.2,
// src/forward/metal_qwen35.rs): the larger value first, equal values by the
// lower index, NaN never chosen; missing entries are the pages' sentinel
// (-inf, index -1).
//
// The pages sort 1280-logit tiles (padded to 2048) per threadgroup
// (logits_topk_first_pass) and merge groups of top-k candidates sixteen at a
// time (logits_topk_merge_pass) until one group is left. Here each entry is
// the 64-bit ordered key of lq_argmax.cuh, so that one unsigned comparison
// ranks two candidates, and two launches do the work:
//
//  1. a grid of CTAs (at most one tile of the input each, as many CTAs as
//     tiles up to a cap) keeps a running top-64 of its tiles in shared
//     memory: slots 0..63 hold the best keys so far, slots 64..2047 take the
//     next 1984 inputs, and a bitonic sort of the 2048 keys brings the best
//     64 back to the front; each CTA writes its best k keys to the work
//     buffer;
//  2. one CTA runs the same loop over the CTAs' candidates and writes the k
//     results.
#include <algorithm>

#include "lq_argmax.cuh"
#include "lq_device.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int kTopkThreads = 256;
constexpr int kTopkTile = 2048;                 // keys sorted together
constexpr int kTopkMaxK = 64;                   // kept between tiles
constexpr int kTopkNew = kTopkTile - kTopkMaxK; // fresh keys per tile
constexpr int kTopkMaxCtas = 512;

// Bitonic sort of s[0 .. kTopkTile) into descending order by all threads of
// the CTA (compare-exchange pair i joins lo and lo + stride; blocks of `size`
// with (lo & size) == 0 run descending, so the last merge sorts the whole
// array descending).
__device__ void sort_desc(unsigned long long* s) {
  for (int size = 2; size <= kTopkTile; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < kTopkTile / 2; i += kTopkThreads) {
        const int lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long a = s[lo], b = s[hi];
        if (desc ? a < b : a > b) {
          s[lo] = b;
          s[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

// The running top-64 over tiles t = first, first + step, ... of `count`
// inputs; key(j) gives the key of input j. Leaves the best keys, sorted, in
// s[0 .. kTopkMaxK).
template <typename KeyOf>
__device__ void running_topk(unsigned long long* s, long long count, long long first, long long step,
                             KeyOf key) {
  for (int j = threadIdx.x; j < kTopkMaxK; j += kTopkThreads) s[j] = 0ull;
  for (long long t = first; t * kTopkNew < count; t += step) {
    const long long base = t * kTopkNew;
    for (int j = threadIdx.x; j < kTopkNew; j += kTopkThreads)
      s[kTopkMaxK + j] = base + j < count ? key(base + j) : 0ull;
    __syncthreads();
    sort_desc(s);
  }
}

__global__ void __launch_bounds__(kTopkThreads) topk_first_kernel(const float* __restrict__ x, long long n,
                                                                  int k, unsigned long long* work) {
  __shared__ unsigned long long s[kTopkTile];
  pdl_wait();  // x may come from the previous kernel on the stream
  running_topk(s, n, blockIdx.x, gridDim.x,
               [&](long long j) { return amax::make_key(x[j], static_cast<unsigned>(j)); });
  pdl_launch_dependents();
  for (int j = threadIdx.x; j < k; j += kTopkThreads) work[static_cast<long long>(blockIdx.x) * k + j] = s[j];
}

__global__ void __launch_bounds__(kTopkThreads) topk_merge_kernel(const unsigned long long* __restrict__ work,
                                                                  long long count, int k, float* values,
                                                                  int32_t* indices) {
  __shared__ unsigned long long s[kTopkTile];
  pdl_wait();  // the candidates of the first pass
  running_topk(s, count, 0, 1, [&](long long j) { return work[j]; });
  for (int j = threadIdx.x; j < k; j += kTopkThreads) {
    const unsigned long long key = s[j];
    if (key == 0ull) {  // fewer than k candidates: the sentinel
      values[j] = -__int_as_float(0x7f800000);
      indices[j] = -1;
    } else {
      const unsigned hi = static_cast<unsigned>(key >> 32), lo = static_cast<unsigned>(key);
      values[j] = __uint_as_float((hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi);
      indices[j] = static_cast<int32_t>(0xFFFFFFFFu - lo);
    }
  }
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_topk(void (*kern)(KArgs...), unsigned grid, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace

int64_t topk_ctas(int64_t n) { return std::min<int64_t>(kTopkMaxCtas, (n + kTopkNew - 1) / kTopkNew); }

lq_status launch_topk_f32(const float* x, int64_t n, int k, float* values, int32_t* indices, void* work,
                          cudaStream_t stream) {
  const int64_t G = topk_ctas(n);
  auto* w = static_cast<unsigned long long*>(work);
  cudaError_t e = launch_pdl_topk(topk_first_kernel, static_cast<unsigned>(G), stream, x,
                                  static_cast<long long>(n), k, w);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_status(e);
  e = launch_pdl_topk(topk_merge_kernel, 1u, stream, static_cast<const unsigned long long*>(w),
                      static_cast<long long>(G * k), k, values, indices);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

}  // namespace lq
