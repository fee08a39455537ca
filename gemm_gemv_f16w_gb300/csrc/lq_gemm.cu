// Prefill GEMM (M > 1). Until the tensor-core kernel is in place both GEMM
// routes run on the generic CUDA-core kernel.
#include "lq_device.cuh"
#include "lq_internal.h"

namespace lq {
namespace {
__device__ unsigned g_gemm_err;
}

unsigned read_clear_gemm_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemm_err, &z, sizeof(z));
  return v;
}

bool gemm_tc_eligible(const MatmulArgs&) { return false; }
lq_status launch_gemm_tc(const MatmulArgs&) { return LQ_ERR_UNSUPPORTED; }
lq_status launch_gemm_stream(const MatmulArgs& a) { return launch_gemv_generic(a); }

}  // namespace lq
