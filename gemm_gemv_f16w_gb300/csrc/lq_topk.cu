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
// ranks two candidates:
//
//  1. a grid of CTAs (one tile of the input each, as many CTAs as tiles up
//     to a cap) keeps a running top-64 of its tiles in shared memory: slots
//     0..63 hold the best keys so far, slots 64..2047 take the next 1984
//     inputs, and a bitonic sort of the 2048 keys (1024 threads, two keys
//     each in registers; shared memory only for strides of 64 and more)
//     brings the best 64 back to the front;
//     each CTA writes its best k keys to the work buffer;
//  2. merge passes, each CTA sorting up to 1984 / k groups of k candidates
//     into one group, until one group is left; the last pass writes the k
//     results.
#include <algorithm>

#include "lq_argmax.cuh"
#include "lq_device.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int kTopkThreads = 1024;              // two keys a thread
constexpr int kTopkLog = 11;
constexpr int kTopkTile = 1 << kTopkLog;        // keys sorted together (2048)
constexpr int kTopkMaxK = 64;                   // kept between tiles
constexpr int kTopkNew = kTopkTile - kTopkMaxK; // fresh keys per tile
constexpr int kTopkMaxCtas = 512;

// Bitonic sort of s[0 .. 2048) into descending order. Thread t holds
// positions 2t and 2t+1 in registers; a step of stride 1 compares the two,
// strides 2..32 pair the thread with lane t ^ (stride / 2) of its warp by
// shuffles, and only strides of 64 and more go through shared memory (pair
// t joins lo and lo + stride, lo = t with a zero bit inserted at
// log2(stride)). Blocks of `size` with (lo & size) == 0 run descending, so
// the last merge sorts the whole array descending. Reads s after a barrier
// and leaves it written, followed by one.
__device__ void sort_desc(unsigned long long* s) {
  const int t = threadIdx.x, p0 = 2 * t;
  unsigned long long e0 = s[p0], e1 = s[p0 + 1];
  for (int ls = 1; ls <= kTopkLog; ++ls) {
    const int size = 1 << ls;
    int lst = ls - 1;
    if ((1 << lst) >= 64) {
      s[p0] = e0;  // this thread's own positions: nobody else reads them now
      s[p0 + 1] = e1;
      __syncthreads();
      for (; (1 << lst) >= 64; --lst) {
        const int stride = 1 << lst;
        const int lo = ((t >> lst) << (lst + 1)) | (t & (stride - 1)), hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long a = s[lo], b = s[hi];
        if (desc ? a < b : a > b) {
          s[lo] = b;
          s[hi] = a;
        }
        __syncthreads();
      }
      e0 = s[p0];
      e1 = s[p0 + 1];
    }
    for (; lst >= 1; --lst) {
      const int stride = 1 << lst;
      const unsigned long long q0 = __shfl_xor_sync(0xffffffffu, e0, stride >> 1);
      const unsigned long long q1 = __shfl_xor_sync(0xffffffffu, e1, stride >> 1);
      // both positions share bit lst (stride >= 2) and bit ls (size >= 4)
      const bool keep_max = ((p0 & stride) == 0) == (((p0 & ~stride) & size) == 0);
      e0 = keep_max ? (e0 > q0 ? e0 : q0) : (e0 < q0 ? e0 : q0);
      e1 = keep_max ? (e1 > q1 ? e1 : q1) : (e1 < q1 ? e1 : q1);
    }
    const bool desc = (p0 & size) == 0;  // stride 1, inside the thread
    if (desc ? e0 < e1 : e0 > e1) {
      const unsigned long long x = e0;
      e0 = e1;
      e1 = x;
    }
  }
  s[p0] = e0;
  s[p0 + 1] = e1;
  __syncthreads();
}

// Leaves in s[0 .. kTopkMaxK) the best keys of inputs key(0 .. count),
// sorted, taking tiles t = first, first + step, ... of kTopkNew inputs.
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
                                                                  int k, unsigned long long* out) {
  __shared__ unsigned long long s[kTopkTile];
  pdl_wait();  // x may come from the previous kernel on the stream
  running_topk(s, n, blockIdx.x, gridDim.x,
               [&](long long j) { return amax::make_key(x[j], static_cast<unsigned>(j)); });
  pdl_launch_dependents();
  for (int j = threadIdx.x; j < k; j += kTopkThreads) out[static_cast<long long>(blockIdx.x) * k + j] = s[j];
}

// One merge pass: CTA b sorts groups [b * fan_in, (b + 1) * fan_in) of k
// candidates (fan_in * k <= kTopkNew) into one group; with one CTA left it
// writes the final values and indices.
__global__ void __launch_bounds__(kTopkThreads) topk_merge_kernel(const unsigned long long* __restrict__ in,
                                                                  int groups, int k, int fan_in,
                                                                  unsigned long long* out, float* values,
                                                                  int32_t* indices) {
  __shared__ unsigned long long s[kTopkTile];
  pdl_wait();  // the candidates of the previous pass
  const long long g0 = static_cast<long long>(blockIdx.x) * fan_in;
  const long long count = (min(static_cast<long long>(groups), g0 + fan_in) - g0) * k;
  const unsigned long long* src = in + g0 * k;
  running_topk(s, count, 0, 1, [&](long long j) { return src[j]; });
  pdl_launch_dependents();
  if (gridDim.x > 1) {
    for (int j = threadIdx.x; j < k; j += kTopkThreads) out[static_cast<long long>(blockIdx.x) * k + j] = s[j];
    return;
  }
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

// Work: two regions of topk_ctas(n) * k keys (the passes alternate).
int64_t topk_ctas(int64_t n) { return 2 * std::min<int64_t>(kTopkMaxCtas, (n + kTopkNew - 1) / kTopkNew); }

lq_status launch_topk_f32(const float* x, int64_t n, int k, float* values, int32_t* indices, void* work,
                          cudaStream_t stream) {
  const int G = static_cast<int>(std::min<int64_t>(kTopkMaxCtas, (n + kTopkNew - 1) / kTopkNew));
  auto* a = static_cast<unsigned long long*>(work);
  auto* b = a + static_cast<size_t>(G) * k;
  cudaError_t e = launch_pdl_topk(topk_first_kernel, static_cast<unsigned>(G), stream, x,
                                  static_cast<long long>(n), k, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  const int fan_in = kTopkNew / k;
  int groups = G;
  while (e == cudaSuccess) {
    const int next = (groups + fan_in - 1) / fan_in;
    e = launch_pdl_topk(topk_merge_kernel, static_cast<unsigned>(next), stream,
                        static_cast<const unsigned long long*>(a), groups, k, fan_in, b, values, indices);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (next == 1) break;
    groups = next;
    std::swap(a, b);
  }
  return cuda_status(e);
}

}  // namespace lq
