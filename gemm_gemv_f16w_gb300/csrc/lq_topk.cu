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
//     inputs, and a partial bitonic sort (runs of 64 sorted in registers,
//     then rounds that keep the best half of each pair of runs) brings the
//     best 64 of the 2048 keys back to the front;
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

// One compare-exchange step of a bitonic network on the warp's keys, thread
// holding positions p and p + 1 (p even): strides 2..32 pair lanes by
// shuffles, stride 1 is inside the thread. keep_max for the lower position
// of each pair is decided by the caller's direction.
__device__ __forceinline__ void cx_step(unsigned long long& e0, unsigned long long& e1, int p, int stride,
                                        bool desc) {
  if (stride == 1) {
    if (desc ? e0 < e1 : e0 > e1) {
      const unsigned long long x = e0;
      e0 = e1;
      e1 = x;
    }
    return;
  }
  const unsigned long long q0 = __shfl_xor_sync(0xffffffffu, e0, stride >> 1);
  const unsigned long long q1 = __shfl_xor_sync(0xffffffffu, e1, stride >> 1);
  const bool keep_max = ((p & stride) == 0) == desc;  // both positions share bit log2(stride)
  e0 = keep_max ? (e0 > q0 ? e0 : q0) : (e0 < q0 ? e0 : q0);
  e1 = keep_max ? (e1 > q1 ? e1 : q1) : (e1 < q1 ? e1 : q1);
}

// The best 64 of s[0 .. 2048), sorted descending into s[0 .. 64) (the rest
// of s is left undefined). Warp w holds the run of positions 64w .. 64w+63,
// two keys a lane. (1) Each run is sorted by the bitonic network on the
// global positions, which leaves even runs descending and odd runs
// ascending. (2) Five rounds halve the runs: warp w, a multiple of 2^(r+1),
// takes the elementwise maximum of its run and the run of warp w + 2^r
// (read through shared memory): a descending run against an ascending one,
// this is the half-cleaner of their bitonic concatenation and keeps the best
// 64 as a bitonic sequence, which six steps sort in the direction the next
// round needs (descending when w / 2^(r+1) is even).
__device__ void top64_desc(unsigned long long* s) {
  const int t = threadIdx.x, w = t >> 5, p0 = 2 * t;
  unsigned long long e0 = s[p0], e1 = s[p0 + 1];
  for (int ls = 1; ls <= 6; ++ls)
    for (int lst = ls - 1; lst >= 0; --lst) {
      const int stride = 1 << lst;
      cx_step(e0, e1, p0, stride, (((p0 & ~stride) & (1 << ls)) == 0));
    }
  for (int r = 0; r < 5; ++r) {
    s[p0] = e0;  // this thread's own positions
    s[p0 + 1] = e1;
    __syncthreads();
    if ((w & ((2 << r) - 1)) == 0) {
      const int q = p0 + (64 << r);  // the same lane of warp w + 2^r
      const unsigned long long b0 = s[q], b1 = s[q + 1];
      e0 = e0 > b0 ? e0 : b0;
      e1 = e1 > b1 ? e1 : b1;
      const bool desc = ((w >> (r + 1)) & 1) == 0;
      for (int lst = 5; lst >= 0; --lst) cx_step(e0, e1, p0 & 63, 1 << lst, desc);
    }
    __syncthreads();
  }
  if (w == 0) {
    s[p0] = e0;
    s[p0 + 1] = e1;
  }
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
    top64_desc(s);
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
