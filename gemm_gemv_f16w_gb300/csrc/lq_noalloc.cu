// lq_gemm_noalloc: the tensor-core GEMM for callers that must not allocate
// device memory.
//
// The regular tensor-core GEMM takes a short-lived workspace (a bf16 copy of
// A) from a stream-ordered memory pool on every call.
// Some callers cannot allow that: runtimes that own all device memory
// themselves and give the library none, services whose memory budget is fixed
// at start-up, and hard real-time paths where an allocation (and the pool
// growth behind it) is an unacceptable latency or failure point. For them
// this entry point runs the same kernels
// on a workspace that is a fixed array in this library's device memory,
// allocated once when the library is loaded on a device and held until the
// process exits. (Calls small enough for the GEMM to round A in shared
// memory itself use no workspace on either entry point.)
#include <mutex>

#include "lq_internal.h"

namespace lq {
namespace {

// 8 MiB: enough for the M*K*2 bytes of bf16 activations when M*K is at most
// 4 Mi elements (e.g. 512 x 8192 or 2048 x 2048).
constexpr size_t kNoAllocBytes = 8u << 20;
static __device__ __align__(256) unsigned char g_noalloc_ws[kNoAllocBytes];

std::mutex g_mu;
void* g_ws_ptr[kMaxDevices];  // device address of g_noalloc_ws, per device

// Device address of the array on the current device. The array's name in
// host code is only a host-side handle, so the address is looked up once per
// device (with that device current) and cached.
lq_status workspace_address(void** out) {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ws_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || !p) return LQ_ERR_CUDA;
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return LQ_OK;
}

}  // namespace
}  // namespace lq

using namespace lq;

extern "C" lq_status lq_gemm_noalloc(int fmt, const float* A, const void* W, float* C, int64_t M,
                                     int64_t N, int64_t K, void* stream) {
  if (fmt != LQ_FMT_F16 && fmt != LQ_FMT_Q8_0 && fmt != LQ_FMT_Q4_0) return LQ_ERR_INVALID_ARG;
  // the same argument checks as lq_gemm_<fmt> (sizes, null pointers, the
  // 4-byte alignment of A and C), before anything else
  bool noop = false;
  const lq_status vs = validate(fmt, A, W, C, M, N, K, &noop);
  if (vs != LQ_OK || noop) return vs;
  MatmulArgs a{A, W, C, M, N, K, fmt, static_cast<cudaStream_t>(stream)};
  // Only the tensor-core kernel that needs the workspace is offered here.
  if (!gemm_tma_eligible(a)) return LQ_ERR_UNSUPPORTED;
  // Beyond the fixed workspace: a clear refusal, never a larger allocation.
  // Calls whose A is resident (small M) need no workspace at all.
  const size_t need = gemm_tma_workspace_bytes(a);
  if (need > kNoAllocBytes) return LQ_ERR_UNSUPPORTED;
  void* ws = nullptr;
  if (need) {
    const lq_status st = workspace_address(&ws);
    if (st != LQ_OK) return st;
  }
  // Every byte the kernels read from the workspace (the bf16 rows of the M
  // tokens) is written earlier in the same call, so nothing needs clearing
  // between calls.
  return launch_gemm_tma_ws(a, ws);
}
