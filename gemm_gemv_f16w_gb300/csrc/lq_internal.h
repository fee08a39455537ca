// Host-side declarations shared by the translation units of liblq.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/lq.h"

namespace lq {

// Problem handed from the C-ABI layer (already validated) to a launcher.
// With epilogue kSwiglu (lq_epilogue.cuh) W holds 2N rows (gate, then up)
// and C receives the N SwiGLU outputs of each row of A; with kResidual C =
// A W^T + R.
struct MatmulArgs {
  const float* A;
  const void* W;
  float* C;
  int64_t M, N, K;
  int fmt;            // lq_format
  cudaStream_t stream;
  int epi = 0;        // lq::epi kind (0: plain)
  const float* R = nullptr;
  // Q4_0 weights with interleaved nibbles (LQ_FMT_Q4_0I, fmt is then
  // LQ_FMT_Q4_0): the kernels read A reordered within each block of 32
  // (lq_q4i.cuh); launchers that cannot do so return LQ_ERR_UNSUPPORTED
  bool a_perm = false;
};

// Per-device facts cached on first use.
struct DeviceInfo {
  int sm_count = 0;
  int max_smem_optin = 0;
  int cc_major = 0, cc_minor = 0;
};
const DeviceInfo& device_info();
constexpr int kMaxDevices = 64;
int current_device();

constexpr unsigned long long kDefaultWaitNsHost = 2000000000ull;
unsigned long long wait_limit_ns();
// Poll budget of a device wait: unlimited by default; with an overridden
// limit below 1 ms, one non-blocking poll per microsecond (at least one).
unsigned wait_limit_iters();
void count_route(int route);
bool use_pdl();
void set_use_pdl(bool on);  // kernels may overlap their predecessor (default on)

// Bytes of one packed W row.
inline int64_t row_bytes(int fmt, int64_t K) {
  return fmt == LQ_FMT_F16 ? 2 * K : (fmt == LQ_FMT_Q8_0 ? K / 32 * 34 : K / 32 * 18);
}

// Launchers (return LQ_OK, LQ_ERR_CUDA or LQ_ERR_UNSUPPORTED; arguments were
// checked by the C-ABI layer).
lq_status launch_gemv(const MatmulArgs& a);            // M == 1, picks fast or generic
lq_status launch_gemv_generic(const MatmulArgs& a);    // any M, K, alignment
// GEMV launch-plan override (0 = automatic): CTAs per SM, rows per stage,
// shared memory per CTA.
void set_gemv_tuning(int ctas_per_sm, int rows_per_stage, int smem_cap);
lq_status launch_gemm_stream(const MatmulArgs& a);     // CUDA-core, small M
// CUDA-core batched decode for M = 2..8 (W streamed once, every row of A
// multiplied with each dequantised block); LQ_ERR_UNSUPPORTED outside its shapes
lq_status launch_gemv_batch(const MatmulArgs& a);
lq_status launch_gemm_tc(const MatmulArgs& a);         // tcgen05, operands via shared memory
bool gemm_tc_eligible(const MatmulArgs& a);
// tcgen05 with TMA loads and W in tensor memory; takes its workspace (the
// bf16 copy of A) from the library's pool unless A is resident (small M)
lq_status launch_gemm_tma(const MatmulArgs& a);
// workspace bytes of a call (0: A is resident, no workspace and no pre-pass)
size_t gemm_tma_workspace_bytes(const MatmulArgs& a);
// the same given that workspace (256-byte aligned; may be null when 0)
lq_status launch_gemm_tma_ws(const MatmulArgs& a, void* ws);
bool gemm_tma_eligible(const MatmulArgs& a);
// cuTensorMapEncodeTiled from the driver (null when unavailable)
void* tma_encode_tiled();
// tensor cores with warp-level MMAs for M = 2..48 (W streamed once, every
// operand in registers); LQ_ERR_UNSUPPORTED outside its shapes
lq_status launch_gemm_small(const MatmulArgs& a);
bool gemm_small_eligible(const MatmulArgs& a);
// TMA GEMM ring-depth override (0 = automatic): A stages, raw W stages.
void set_gemm_rings(int a_stages, int raw_stages);
void set_gemm_pairs(bool on);

// Argmax (lq_gemv_argmax, lq_argmax_f32). launch_gemv_argmax returns
// LQ_ERR_UNSUPPORTED, launching nothing, outside the streaming GEMV's fast
// path. Both zero out->work on the stream first.
lq_status launch_gemv_argmax(const MatmulArgs& a, lq_argmax_result* out);
lq_status launch_argmax_f32(const float* x, int64_t n, lq_argmax_result* out, cudaStream_t stream);

// Top-k (lq_topk_f32): the work buffer holds topk_ctas(n) * k keys of 8
// bytes (two regions for the first pass's CTAs), and the launches.
int64_t topk_ctas(int64_t n);
lq_status launch_topk_f32(const float* x, int64_t n, int k, float* values, int32_t* indices, void* work,
                          cudaStream_t stream);

// Decode chain (lq_gemv_chain); LQ_ERR_UNSUPPORTED when the problems do not
// fit its fast path.
lq_status launch_gemv_chain(int fmt, const lq_gemv_problem* problems, int count, cudaStream_t stream);
// Debug: dependent problems wait inside one chain launch (device-wide
// counter) instead of starting a new launch (the default).
void set_chain_waits(bool on);

// Device status words of each translation unit (read-and-clear).
unsigned read_clear_gemv_error();
unsigned read_clear_gemm_error();
unsigned read_clear_gemm_tma_error();
unsigned read_clear_chain_error();
unsigned read_clear_batch_error();
unsigned read_clear_small_error();

lq_status cuda_status(cudaError_t e);

bool aligned_to(const void* p, unsigned a);
// The argument checks every matmul entry point makes before launching
// anything: LQ_OK to proceed (with *noop set for M == 0 or N == 0), else the
// status to return.
lq_status validate(int fmt, const float* A, const void* W, float* C, int64_t M, int64_t N,
                   int64_t K, bool* noop);

}  // namespace lq
