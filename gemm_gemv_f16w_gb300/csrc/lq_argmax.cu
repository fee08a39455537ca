// lq_argmax_f32: the argmax of a device vector in one launch.
//
// The pages reduce materialised logits in two dispatches, one 1024-thread
// group per 1024 logits (logits_argmax_first) and one group over the group
// winners (logits_argmax_merge), lattice-inference 0.1.2,
// src/forward/metal_qwen35.rs. Here a grid of a few CTAs per SM strides over
// the vector with coalesced loads, every warp folds its lanes' best
// candidates with shuffles and merges its winner into the result with one
// 64-bit atomicMax; the warp that finishes last writes (value, index)
// (lq_argmax.cuh). The GEMV falls back to this kernel for the shapes its
// fused argmax does not take.
#include <algorithm>

#include "lq_argmax.cuh"
#include "lq_device.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int kArgmaxThreads = 256;

__global__ void __launch_bounds__(kArgmaxThreads) argmax_f32_kernel(const float* __restrict__ x, int n,
                                                                    lq_argmax_result* out,
                                                                    unsigned total_warps) {
  pdl_wait();  // x may come from the previous kernel on the stream
  const int lane = threadIdx.x & 31;
  const int stride = gridDim.x * kArgmaxThreads;
  unsigned long long best = 0ull;
  for (int i = blockIdx.x * kArgmaxThreads + threadIdx.x; i < n; i += stride) {
    const unsigned long long k = amax::make_key(x[i], static_cast<unsigned>(i));
    best = k > best ? k : best;
  }
  pdl_launch_dependents();
  amax::warp_done(best, out, total_warps, lane);
}

}  // namespace

lq_status launch_argmax_f32(const float* x, int64_t n, lq_argmax_result* out, cudaStream_t stream) {
  const DeviceInfo& di = device_info();
  const int64_t want = (n + kArgmaxThreads * 8 - 1) / (kArgmaxThreads * 8);  // ~8 values a thread
  const int G = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 4LL * std::max(di.sm_count, 1))));
  cudaError_t e = cudaMemsetAsync(out->work, 0, sizeof(out->work), stream);
  if (e != cudaSuccess) return cuda_status(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G));
  cfg.blockDim = dim3(kArgmaxThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const unsigned warps = static_cast<unsigned>(G) * (kArgmaxThreads / 32);
  e = cudaLaunchKernelEx(&cfg, argmax_f32_kernel, x, static_cast<int>(n), out, warps);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

}  // namespace lq
