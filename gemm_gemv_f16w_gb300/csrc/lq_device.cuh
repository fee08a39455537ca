// Device-side building blocks for sm_103a: mbarriers, 1-D bulk copies (TMA),
// programmatic dependent launch, packed f32x2 math and the bounded waits that
// every kernel in this library uses instead of unbounded spins.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace lq {

// Device status codes (mirror lq_status).
constexpr unsigned kDevErrTimeout = 4u;
constexpr unsigned kDevErrBounds = 5u;

// ---- debug bounds checks ----------------------------------------------------
// Built with -DLQ_DEBUG_BOUNDS (liblq_debug.so), each global index a kernel
// computes for a plain load or store, and each byte range of a bulk copy of
// W rows, is checked against its extent first: a failed check records
// kDevErrBounds in the translation unit's status word (lq_last_device_error
// reports LQ_ERR_BOUNDS) and the access is skipped, so nothing faults or
// traps (a skipped copy leaves its waiters to their time limits). Release
// builds compile the checks away. A translation unit that uses LQ_IN_BOUNDS
// defines record_error(unsigned) first. Tensor-map copies need no check:
// the TMA unit clips them to the tensor's extents.
#ifdef LQ_DEBUG_BOUNDS
#define LQ_IN_BOUNDS(cond) ((cond) ? true : (record_error(::lq::kDevErrBounds), false))
#else
#define LQ_IN_BOUNDS(cond) true
#endif

// Limit for draining copies that are still in flight when a kernel gives up
// (not affected by the debugging override of the normal wait limit).
constexpr unsigned long long kDrainWaitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// Makes mbarrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete, for at most about
// `limit_ns` nanoseconds and `max_iters` polls. Returns false on timeout.
// The deadline is kept in SM clock cycles (clock64 is cheap to read; the
// limit is converted at 4 cycles per ns, so at clocks up to 4 GHz the wait
// lasts at least `limit_ns`). A small poll budget (a debugging override)
// polls without blocking, so that the wait gives up deterministically;
// otherwise the hardware's potentially blocking try_wait is used.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns,
                                          uint32_t max_iters = (1u << 30)) {
  if (max_iters < 1024u) {
    for (uint32_t it = 0; it < max_iters; ++it)
      if (mbar_test_wait(bar, parity)) return true;
    return false;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  const long long limit = static_cast<long long>(limit_ns) * 4;
  for (uint32_t it = 1; it < max_iters; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && clock64() - t0 > limit) return false;
  }
  return false;
}

// ---- 1-D bulk copy global -> shared (TMA, no tensor map) -------------------
// dst, src 16-byte aligned; bytes a multiple of 16. Completion is signalled
// as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Prefetch of [src, src + bytes) into L2 (16-byte aligned, bytes a multiple
// of 16); no completion to wait for.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- shared-memory loads by 32-bit shared address --------------------------
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// ---- 16-byte asynchronous copies global -> shared (per thread) -------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
}
// Barrier over the first `threads` threads of the block (a multiple of 32)
// on hardware barrier `id` (1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- read-only global loads -------------------------------------------------
// For data that no thread writes while the kernel runs (inputs produced by an
// earlier, completed kernel).
__device__ __forceinline__ float4 ldg128f(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// ---- programmatic dependent launch ----------------------------------------
// Blocks until the preceding kernel on the stream has completed and its
// memory is visible (no-op when the kernel was not launched with PDL).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream start launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- packed f32x2 arithmetic (sm_100+) -------------------------------------
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

// ---- small integer -> exact float without I2F ------------------------------
// Byte i of w, placed as the low mantissa byte of 2^23: the float equals
// 2^23 + that byte exactly. For an int8 q with its sign bit flipped the byte
// is q + 128; for a Q4_0 code masked into a byte it is the code itself.
__device__ __forceinline__ float s8_to_magic(uint32_t w_xor80, int i) {
  // result bytes: [w.byte_i, 0x00, 0x00, 0x4B]
  const uint32_t sel = 0x7540u | static_cast<uint32_t>(i);
  return __uint_as_float(__byte_perm(w_xor80, 0x4B000000u, sel));
}
constexpr float kMagicS8 = 8388608.0f + 128.0f;  // 2^23 + 128
constexpr float kMagicQ4 = 8388608.0f + 8.0f;    // 2^23 + 8: a nibble code's offset

__device__ __forceinline__ float f16_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}

// Warp-wide sum.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace lq
