// Epilogues the matmul kernels can apply to their outputs before storing
// them (lq_matmul_residual, lq_matmul_swiglu, lq_gemv_argmax).
//
//  * residual: C = A W^T + R, as gemm_q1_v7_residual (oxibonsai-kernels
//    0.1.4, src/gpu_backend/metal_prefill/functions.rs) adds the hidden
//    state to the projection; R may be C itself;
//  * swiglu: W is gate_up, the gate rows followed by the up rows (2I rows),
//    and output j of a token is silu(g_j) * u_j with g_j, u_j the outputs
//    of rows j and I + j: fused_gate_up_swiglu_gemm on the same page, and
//    silu_mul (lattice-inference 0.1.2, src/forward/metal_qwen35.rs), which
//    computes silu(g) = g / (1 + exp(-g)) and multiplies by up.
#pragma once
#include <cstdint>

namespace lq {
namespace epi {

enum : int { kPlain = 0, kArgmax = 1, kResidual = 2, kSwiglu = 3 };

// silu(g) * u, evaluated as silu_mul writes it (expf is CUDA's, within 2 ulp)
__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.0f + expf(-g)) * u; }

}  // namespace epi
}  // namespace lq
