// C-ABI entry points: argument validation, the M==1 / M>1 router and the
// route hooks used by the tests.
//
// The router mirrors dispatch_gemm_q8 / dispatch_gemm_q4 / dispatch_matmul_half
// (lattice-inference, src/forward/metal_qwen35/inner/dispatch.rs): M == 0 or
// N == 0 returns without launching; quantised formats need K > 0 and
// K % 32 == 0 (the page asserts, this library returns LQ_ERR_INVALID_ARG);
// M == 1 goes to the GEMV; M > 1 goes to a GEMM, the tensor-core kernel when
// it can take the shape and the CUDA-core kernel otherwise.
#include <atomic>
#include <mutex>

#include "lq_epilogue.cuh"
#include "lq_internal.h"

namespace lq {

namespace {
std::atomic<int> g_force_route{0};
std::atomic<uint64_t> g_route_count[8];
std::atomic<unsigned long long> g_wait_ns{0};
std::mutex g_info_mu;
DeviceInfo g_info[kMaxDevices];
bool g_info_valid[kMaxDevices];
}  // namespace

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

const DeviceInfo& device_info() {
  static DeviceInfo empty;
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return empty;
  std::lock_guard<std::mutex> lk(g_info_mu);
  if (!g_info_valid[dev]) {
    DeviceInfo d;
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    g_info[dev] = d;
    g_info_valid[dev] = true;
  }
  return g_info[dev];
}

unsigned long long wait_limit_ns() {
  const unsigned long long v = g_wait_ns.load();
  return v ? v : kDefaultWaitNsHost;
}

unsigned wait_limit_iters() {
  const unsigned long long v = g_wait_ns.load();
  if (v == 0 || v >= 1000000ull) return 1u << 30;
  const unsigned long long it = v / 1000ull;
  return it < 1 ? 1u : static_cast<unsigned>(it);
}

void count_route(int route) {
  if (route >= 0 && route < 8) g_route_count[route].fetch_add(1);
}

namespace {
std::atomic<bool> g_use_pdl{true};
}
bool use_pdl() { return g_use_pdl.load(); }
void set_use_pdl(bool on) { g_use_pdl.store(on); }

lq_status cuda_status(cudaError_t e) { return e == cudaSuccess ? LQ_OK : LQ_ERR_CUDA; }

bool aligned_to(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shared argument checks. Returns LQ_OK to proceed, or the status to return;
// `*noop` is set when the call is a valid no-op.
lq_status validate(int fmt, const float* A, const void* W, float* C, int64_t M, int64_t N,
                   int64_t K, bool* noop) {
  *noop = false;
  if (M < 0 || N < 0 || K < 0) return LQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) {
    *noop = true;
    return LQ_OK;
  }
  if (fmt != LQ_FMT_F16 && (K == 0 || K % 32 != 0)) return LQ_ERR_INVALID_ARG;
  if (K == 0) return LQ_ERR_INVALID_ARG;
  if (!A || !W || !C) return LQ_ERR_INVALID_ARG;
  if (!aligned_to(A, 4) || !aligned_to(C, 4)) return LQ_ERR_INVALID_ARG;
  if (fmt == LQ_FMT_F16 && !aligned_to(W, 2)) return LQ_ERR_INVALID_ARG;
  // 32-bit indexing inside the kernels
  if (M > (1LL << 31) - 1 || N > (1LL << 30) || K > (1LL << 30)) return LQ_ERR_UNSUPPORTED;
  return LQ_OK;
}

namespace {

// Arguments for the launchers: LQ_FMT_Q4_0I runs the Q4_0 kernels with A
// reordered within each block (lq_q4i.cuh).
MatmulArgs make_args(int fmt, const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K,
                     void* stream) {
  MatmulArgs a{A, W, C, M, N, K, fmt, static_cast<cudaStream_t>(stream)};
  if (fmt == LQ_FMT_Q4_0I) {
    a.fmt = LQ_FMT_Q4_0;
    a.a_perm = true;
  }
  return a;
}

bool known_format(int fmt) {
  return fmt == LQ_FMT_F16 || fmt == LQ_FMT_Q8_0 || fmt == LQ_FMT_Q4_0 || fmt == LQ_FMT_Q4_0I;
}

lq_status do_gemv(int fmt, const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K,
                  void* stream) {
  bool noop;
  lq_status st = validate(fmt, A, W, C, M, N, K, &noop);
  if (st != LQ_OK || noop) return st;
  if (M != 1) return LQ_ERR_INVALID_ARG;
  MatmulArgs a = make_args(fmt, A, W, C, M, N, K, stream);
  if (g_force_route.load() == 3) return launch_gemv_generic(a);
  return launch_gemv(a);
}

lq_status do_gemm(int fmt, const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K,
                  void* stream) {
  bool noop;
  lq_status st = validate(fmt, A, W, C, M, N, K, &noop);
  if (st != LQ_OK || noop) return st;
  MatmulArgs a = make_args(fmt, A, W, C, M, N, K, stream);
  switch (g_force_route.load()) {
    case 1:
      st = launch_gemv_batch(a);
      return st == LQ_ERR_UNSUPPORTED ? launch_gemm_stream(a) : st;
    case 2:
      if (gemm_tma_eligible(a)) return launch_gemm_tma(a);
      return gemm_tc_eligible(a) ? launch_gemm_tc(a) : LQ_ERR_UNSUPPORTED;
    case 3: return launch_gemv_generic(a);
    case 5: return launch_gemm_small(a);
    default: break;
  }
  // M = 2..48: the warp-MMA tensor-core kernel (N = 6144, K = 2048, Q8_0 /
  // f16 / Q4_0: 7.1 / 6.8 / 6.4 us at M = 2 against 7.7 / 9.2 / 7.0 on the
  // batched CUDA-core kernel and 10.6 / 10.1 / 10.6 on the tcgen05 kernel;
  // at M = 16 7.7 / 7.2 / 7.2 against 11.4 / 10.8 / 11.3 on tcgen05; from 17
  // rows two or three token groups share each converted weight, for CTAs of
  // up to 64 / 48 W rows: M = 32 8.3 / 9.9 / 7.7 against 12.9 / 12.3 / 12.7,
  // M = 48 12.1 / 11.9 / 12.2 against 14.0 / 13.2 / 13.3). The batched kernel
  // takes the shapes the warp-MMA kernel does not (up to four rows), and two
  // to eight rows by a forced route (lq_debug_force_route(1)).
  if (M <= 48) {
    st = launch_gemm_small(a);
    if (st != LQ_ERR_UNSUPPORTED) return st;
  }
  if (M <= 4) {
    st = launch_gemv_batch(a);
    if (st != LQ_ERR_UNSUPPORTED) return st;
  }
  if (gemm_tma_eligible(a)) return launch_gemm_tma(a);
  if (gemm_tc_eligible(a)) return launch_gemm_tc(a);
  return launch_gemm_stream(a);
}

// The matmul with an epilogue (residual add or gate/up SwiGLU): the same
// routes as do_matmul, each kernel applying the epilogue before its store;
// the tensor-core kernel of lq_gemm.cu and the small-M stream kernel do not
// take epilogues, so those shapes go to the generic kernel.
lq_status do_epilogue(int fmt, const float* A, const void* W, const float* R, float* C, int64_t M,
                      int64_t N, int64_t K, int epi_kind, void* stream) {
  bool noop;
  lq_status st = validate(fmt, A, W, C, M, N, K, &noop);
  if (st != LQ_OK || noop) return st;
  if (epi_kind == epi::kResidual && (!R || !aligned_to(R, 4))) return LQ_ERR_INVALID_ARG;
  if (epi_kind == epi::kSwiglu && 2 * N >= (1LL << 30)) return LQ_ERR_UNSUPPORTED;
  MatmulArgs a = make_args(fmt, A, W, C, M, N, K, stream);
  a.epi = epi_kind;
  a.R = R;
  switch (g_force_route.load()) {
    case 1:
      st = launch_gemv_batch(a);
      return st == LQ_ERR_UNSUPPORTED ? launch_gemv_generic(a) : st;
    case 2:
      return gemm_tma_eligible(a) ? launch_gemm_tma(a) : LQ_ERR_UNSUPPORTED;
    case 3: return launch_gemv_generic(a);
    case 5: return launch_gemm_small(a);
    default: break;
  }
  if (M == 1) return launch_gemv(a);  // falls back to the generic kernel itself
  // as do_gemm; the warp-MMA kernel has no SwiGLU epilogue, which keeps the
  // batched kernel up to four rows
  if (M <= 48) {
    st = launch_gemm_small(a);
    if (st != LQ_ERR_UNSUPPORTED) return st;
  }
  if (M <= 4) {
    st = launch_gemv_batch(a);
    if (st != LQ_ERR_UNSUPPORTED) return st;
  }
  if (gemm_tma_eligible(a)) return launch_gemm_tma(a);
  return launch_gemv_generic(a);
}

lq_status do_matmul(int fmt, const float* A, const void* W, float* C, int64_t M, int64_t N,
                    int64_t K, void* stream) {
  if (M == 1) return do_gemv(fmt, A, W, C, M, N, K, stream);
  return do_gemm(fmt, A, W, C, M, N, K, stream);
}

}  // namespace
}  // namespace lq

using namespace lq;

extern "C" {

lq_status lq_gemv_f16(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_gemv(LQ_FMT_F16, A, W, C, M, N, K, s);
}
lq_status lq_gemv_q8_0(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_gemv(LQ_FMT_Q8_0, A, W, C, M, N, K, s);
}
lq_status lq_gemv_q4_0(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_gemv(LQ_FMT_Q4_0, A, W, C, M, N, K, s);
}
lq_status lq_gemm_f16(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_gemm(LQ_FMT_F16, A, W, C, M, N, K, s);
}
lq_status lq_gemm_q8_0(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_gemm(LQ_FMT_Q8_0, A, W, C, M, N, K, s);
}
lq_status lq_gemm_q4_0(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_gemm(LQ_FMT_Q4_0, A, W, C, M, N, K, s);
}
lq_status lq_matmul_f16(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_matmul(LQ_FMT_F16, A, W, C, M, N, K, s);
}
lq_status lq_matmul_q8_0(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_matmul(LQ_FMT_Q8_0, A, W, C, M, N, K, s);
}
lq_status lq_matmul_q4_0(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_matmul(LQ_FMT_Q4_0, A, W, C, M, N, K, s);
}

lq_status lq_gemv_q4_0i(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_gemv(LQ_FMT_Q4_0I, A, W, C, M, N, K, s);
}
lq_status lq_gemm_q4_0i(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_gemm(LQ_FMT_Q4_0I, A, W, C, M, N, K, s);
}
lq_status lq_matmul_q4_0i(const float* A, const void* W, float* C, int64_t M, int64_t N, int64_t K, void* s) {
  return do_matmul(LQ_FMT_Q4_0I, A, W, C, M, N, K, s);
}

const char* lq_status_string(lq_status s) {
  switch (s) {
    case LQ_OK: return "LQ_OK";
    case LQ_ERR_INVALID_ARG: return "LQ_ERR_INVALID_ARG: bad pointer, size or alignment";
    case LQ_ERR_UNSUPPORTED: return "LQ_ERR_UNSUPPORTED: no kernel for this request";
    case LQ_ERR_CUDA: return "LQ_ERR_CUDA: a CUDA call or launch failed";
    case LQ_ERR_DEVICE_TIMEOUT: return "LQ_ERR_DEVICE_TIMEOUT: a bounded device wait ran out";
    case LQ_ERR_BOUNDS: return "LQ_ERR_BOUNDS: an index check of the debug build failed (access skipped)";
  }
  return "unknown lq_status";
}

lq_status lq_last_device_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return LQ_ERR_CUDA;
  const unsigned a = read_clear_gemv_error();
  const unsigned b = read_clear_gemm_error();
  const unsigned c = read_clear_gemm_tma_error();
  const unsigned d = read_clear_chain_error();
  const unsigned e = read_clear_batch_error();
  const unsigned f = read_clear_small_error();
  const unsigned v = a ? a : (b ? b : (c ? c : (d ? d : (e ? e : f))));
  if (v == 0) return LQ_OK;
  return static_cast<lq_status>(v);
}

lq_status lq_gemv_chain(int fmt, const lq_gemv_problem* problems, int count, void* stream) {
  if (!known_format(fmt)) return LQ_ERR_INVALID_ARG;
  if (!problems || count < 1) return LQ_ERR_INVALID_ARG;
  for (int j = 0; j < count; ++j) {
    const lq_gemv_problem& q = problems[j];
    if (q.N < 0 || q.K < 1) return LQ_ERR_INVALID_ARG;
    if (fmt != LQ_FMT_F16 && q.K % 32 != 0) return LQ_ERR_INVALID_ARG;
    if (!q.A || !q.W || !q.C) return LQ_ERR_INVALID_ARG;
    if (!aligned_to(q.A, 4) || !aligned_to(q.C, 4)) return LQ_ERR_INVALID_ARG;
    if (fmt == LQ_FMT_F16 && !aligned_to(q.W, 2)) return LQ_ERR_INVALID_ARG;
  }
  return lq::launch_gemv_chain(fmt, problems, count, static_cast<cudaStream_t>(stream));
}

lq_status lq_gemv_argmax(int fmt, const float* A, const void* W, float* C, int64_t N, int64_t K,
                         lq_argmax_result* out, void* stream) {
  if (!known_format(fmt)) return LQ_ERR_INVALID_ARG;
  if (N < 1 || N >= (1LL << 30)) return LQ_ERR_INVALID_ARG;
  if (!out || !aligned_to(out, 8)) return LQ_ERR_INVALID_ARG;
  float* C_check = C ? C : reinterpret_cast<float*>(out);  // C may be null
  bool noop;
  lq_status st = validate(fmt, A, W, C_check, 1, N, K, &noop);
  if (st != LQ_OK) return st;
  MatmulArgs a = make_args(fmt, A, W, C, 1, N, K, stream);
  if (g_force_route.load() != 3) {
    st = launch_gemv_argmax(a, out);
    if (st != LQ_ERR_UNSUPPORTED) return st;
  }
  // unfused: the GEMV into C, then the argmax of C
  if (!C) return LQ_ERR_UNSUPPORTED;
  st = g_force_route.load() == 3 ? launch_gemv_generic(a) : launch_gemv(a);
  if (st != LQ_OK) return st;
  return launch_argmax_f32(C, N, out, a.stream);
}

lq_status lq_matmul_residual(int fmt, const float* A, const void* W, const float* R, float* C, int64_t M,
                             int64_t N, int64_t K, void* stream) {
  if (!known_format(fmt)) return LQ_ERR_INVALID_ARG;
  return do_epilogue(fmt, A, W, R, C, M, N, K, epi::kResidual, stream);
}

lq_status lq_matmul_swiglu(int fmt, const float* A, const void* W, float* H, int64_t M, int64_t I, int64_t K,
                           void* stream) {
  if (!known_format(fmt)) return LQ_ERR_INVALID_ARG;
  return do_epilogue(fmt, A, W, nullptr, H, M, I, K, epi::kSwiglu, stream);
}

lq_status lq_argmax_f32(const float* x, int64_t n, lq_argmax_result* out, void* stream) {
  if (!x || !aligned_to(x, 4) || n < 1 || n >= (1LL << 31)) return LQ_ERR_INVALID_ARG;
  if (!out || !aligned_to(out, 8)) return LQ_ERR_INVALID_ARG;
  return launch_argmax_f32(x, n, out, static_cast<cudaStream_t>(stream));
}

size_t lq_topk_work_bytes(int64_t n, int k) {
  if (n < 1 || n >= (1LL << 31) || k < 1 || k > 64) return 0;
  return static_cast<size_t>(topk_ctas(n)) * static_cast<size_t>(k) * 8u;
}

lq_status lq_topk_f32(const float* x, int64_t n, int k, float* values, int32_t* indices, void* work,
                      void* stream) {
  if (!x || !aligned_to(x, 4) || n < 1 || n >= (1LL << 31) || k < 1 || k > 64) return LQ_ERR_INVALID_ARG;
  if (!values || !aligned_to(values, 4) || !indices || !aligned_to(indices, 4)) return LQ_ERR_INVALID_ARG;
  if (!work || !aligned_to(work, 8)) return LQ_ERR_INVALID_ARG;
  return launch_topk_f32(x, n, k, values, indices, work, static_cast<cudaStream_t>(stream));
}

lq_status lq_gemv_topk(int fmt, const float* A, const void* W, float* C, int64_t N, int64_t K, int k,
                       float* values, int32_t* indices, void* work, void* stream) {
  if (!known_format(fmt) || !C) return LQ_ERR_INVALID_ARG;
  if (N < 1 || N >= (1LL << 30) || k < 1 || k > 64) return LQ_ERR_INVALID_ARG;
  if (!values || !aligned_to(values, 4) || !indices || !aligned_to(indices, 4)) return LQ_ERR_INVALID_ARG;
  if (!work || !aligned_to(work, 8)) return LQ_ERR_INVALID_ARG;
  const lq_status st = do_gemv(fmt, A, W, C, 1, N, K, stream);
  if (st != LQ_OK) return st;
  return launch_topk_f32(C, N, k, values, indices, work, static_cast<cudaStream_t>(stream));
}

#ifdef LQ_DEBUG_BOUNDS
const char* lq_version(void) { return "lq 0.2.0 (sm_103a, debug bounds checks)"; }
#else
const char* lq_version(void) { return "lq 0.2.0 (sm_103a)"; }
#endif

lq_status lq_debug_force_route(int route) {
  if (route < 0 || route > 5 || route == 4) return LQ_ERR_INVALID_ARG;
  g_force_route.store(route);
  return LQ_OK;
}
uint64_t lq_debug_route_count(int route) {
  if (route < 0 || route > 7) return 0;
  return g_route_count[route].load();
}
void lq_debug_reset_counts(void) {
  for (auto& c : g_route_count) c.store(0);
}
void lq_debug_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns); }
lq_status lq_debug_gemm_rings(int a_stages, int raw_stages) {
  if (a_stages < 0 || a_stages > 4 || raw_stages < 0 || raw_stages > 8) return LQ_ERR_INVALID_ARG;
  lq::set_gemm_rings(a_stages, raw_stages);
  return LQ_OK;
}
void lq_debug_chain_waits(int on) { lq::set_chain_waits(on != 0); }
void lq_debug_gemm_pairs(int on) { lq::set_gemm_pairs(on != 0); }
lq_status lq_debug_gemv_plan(int ctas_per_sm, int rows_per_stage, int smem_bytes) {
  if (ctas_per_sm < 0 || ctas_per_sm > 2 || rows_per_stage < 0 || rows_per_stage > 8 ||
      smem_bytes < 0)
    return LQ_ERR_INVALID_ARG;
  lq::set_gemv_tuning(ctas_per_sm, rows_per_stage, smem_bytes);
  return LQ_OK;
}

}  // extern "C"
