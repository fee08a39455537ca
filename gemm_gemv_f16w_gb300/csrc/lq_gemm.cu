// Prefill GEMM (M > 1): C[M,N] = A[M,K] @ W[N,K]^T on the tensor cores.
//
// Counterparts on the source pages: gemm_q4_tiled (lattice-inference 0.1.2,
// src/forward/metal_qwen35.rs: 64x32 tiles, W dequantised to f32 in
// threadgroup memory, simdgroup 8x8 matrices), gemm_q8_tiled and the f16
// gemm_f32a_f16w_v2 (ferrum-kernels, pipelines.rs). Here the contraction runs
// on GB300's 5th-generation tensor cores:
//
//  * a CTA owns 128 rows of W and a tile of BT tokens ("swap AB": W rows are
//    the MMA's M side, tokens its N side), so small batches waste no MMA
//    rows and the TMEM accumulator maps W row n to TMEM lane n;
//  * four converter warps read raw W (f16 / Q8_0 / Q4_0 bytes) and f32 A,
//    dequantise W and round A to bf16 (round to nearest even), and write both
//    as 128-byte-swizzled K-major tiles into a 3-stage shared-memory ring;
//  * one thread issues tcgen05.mma kind::f16 (bf16 x bf16 -> f32 in TMEM),
//    64 K per stage as 4 MMAs of K=16, and tcgen05.commit releases the stage;
//  * after the last stage the same four warps read the accumulator with
//    tcgen05.ld and store C with coalesced f32 stores (32 W rows per warp).
//
// Every wait is bounded; on timeout the kernel records
// LQ_ERR_DEVICE_TIMEOUT, waits for its own MMAs, frees TMEM and returns.
#include <algorithm>

#include "lq_device.cuh"
#include "lq_internal.h"
#include "lq_tcgen05.cuh"

namespace lq {
namespace {

__device__ unsigned g_gemm_err;

constexpr int kConvWarps = 4;                      // converters, then epilogue
constexpr int kTcThreads = (kConvWarps + 1) * 32;  // + the MMA warp
constexpr int kBN = 128;                           // W rows per CTA (MMA M)
constexpr int kBK = 64;                            // K per stage (one 128-byte swizzle atom)
constexpr int kStages = 3;
constexpr int kWTileBytes = kBN * kBK * 2;         // 16 KB of bf16

struct TcParams {
  const float* A;
  const uint8_t* W;
  float* C;
  int M, N, K;
  long long rb;  // bytes of one packed W row
  unsigned long long wait_ns;
  unsigned wait_iters;
};

struct TcBars {
  uint64_t full[kStages];   // converters wrote the stage (128 arrivals)
  uint64_t empty[kStages];  // the MMAs that read the stage completed (commit)
  uint64_t tmem_full;       // all MMAs completed (commit)
  uint32_t tmem_base;
  volatile int abort;
};

__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_gemm_err, 0u, code); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 64 dequantised weights w(n, k0 .. k0+63) of one W row, as f32.
template <int FMT>
__device__ __forceinline__ void load_w64(const uint8_t* row, int ks, float (&v)[64]) {
  if constexpr (FMT == LQ_FMT_F16) {
    const uint4* src = reinterpret_cast<const uint4*>(row + 128LL * ks);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 x = __ldg(src + c);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        v[8 * c + 2 * i] = f.x;
        v[8 * c + 2 * i + 1] = f.y;
      }
    }
  } else if constexpr (FMT == LQ_FMT_Q8_0) {
    // two 34-byte blocks = 17 words, 4-byte aligned (K % 64 == 0)
    const uint32_t* src = reinterpret_cast<const uint32_t*>(row + 68LL * ks);
    uint32_t w[17];
#pragma unroll
    for (int i = 0; i < 17; ++i) w[i] = __ldg(src + i);
    const float d0 = f16_lo(w[0]), d1 = f16_lo(w[8] >> 16);
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int b0 = 2 + e, b1 = 36 + e;
      const float q0 = static_cast<float>(static_cast<int8_t>((w[b0 >> 2] >> (8 * (b0 & 3))) & 0xFFu));
      const float q1 = static_cast<float>(static_cast<int8_t>((w[b1 >> 2] >> (8 * (b1 & 3))) & 0xFFu));
      v[e] = d0 * q0;
      v[32 + e] = d1 * q1;
    }
  } else {
    // two 18-byte blocks = 9 words; byte j of a block's 16 holds q_j | q_{j+16} << 4
    const uint32_t* src = reinterpret_cast<const uint32_t*>(row + 36LL * ks);
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = __ldg(src + i);
    const float d0 = f16_lo(w[0]), d1 = f16_lo(w[4] >> 16);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int b0 = 2 + j, b1 = 20 + j;
      const uint32_t x0 = (w[b0 >> 2] >> (8 * (b0 & 3))) & 0xFFu;
      const uint32_t x1 = (w[b1 >> 2] >> (8 * (b1 & 3))) & 0xFFu;
      v[j] = d0 * static_cast<float>(static_cast<int>(x0 & 0xF) - 8);
      v[16 + j] = d0 * static_cast<float>(static_cast<int>(x0 >> 4) - 8);
      v[32 + j] = d1 * static_cast<float>(static_cast<int>(x1 & 0xF) - 8);
      v[48 + j] = d1 * static_cast<float>(static_cast<int>(x1 >> 4) - 8);
    }
  }
}

// Writes 64 f32 values as one bf16 row of a 128B-swizzled K-major tile.
__device__ __forceinline__ void store_row_bf16(uint32_t tile, uint32_t r, const float (&v)[64]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t a = tile + tc::sw128_offset(r, c);
    const uint32_t x = pack_bf16x2(v[8 * c], v[8 * c + 1]);
    const uint32_t y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
    const uint32_t z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
    const uint32_t t = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(t)
                 : "memory");
  }
}

template <int FMT, int BT>
__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled tiles
  const uint32_t raw_u = smem_u32(smem_raw);
  const uint32_t base_u = (raw_u + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u - raw_u);
  constexpr int kTokTileBytes = BT * kBK * 2;
  constexpr int kStageBytes = kWTileBytes + kTokTileBytes;
  TcBars& bars = *reinterpret_cast<TcBars*>(base + kStages * kStageBytes);
  constexpr uint32_t kTmemCols = BT <= 32 ? 32u : (BT <= 64 ? 64u : (BT <= 128 ? 128u : 256u));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * BT;
  const int nk = p.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.full[s], kConvWarps * 32);
      mbar_init(&bars.empty[s], 1);
    }
    mbar_init(&bars.tmem_full, 1);
    bars.abort = 0;
    fence_barrier_init();
  }
  if (warp == kConvWarps) {
    tc::tmem_alloc(&bars.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars.tmem_base;
  pdl_launch_dependents();
  pdl_wait();  // A (and C) may belong to the previous kernel on the stream

  if (warp < kConvWarps) {
    // ---------------- converters ----------------
    const int t = threadIdx.x;  // 0..127: W row of the tile, and token row(s)
    const int n = n0 + t;
    const uint8_t* wrow = p.W + static_cast<long long>(n < p.N ? n : 0) * p.rb;
    bool ok = true;
    for (int ks = 0; ks < nk && ok; ++ks) {
      const int s = ks % kStages;
      if (ks >= kStages &&
          (!mbar_wait(&bars.empty[s], ((ks / kStages) - 1) & 1, p.wait_ns, p.wait_iters) || bars.abort)) {
        ok = false;
        break;
      }
      const uint32_t wtile = base_u + s * kStageBytes;
      const uint32_t ttile = wtile + kWTileBytes;
      float v[64];
      if (n < p.N && LQ_IN_BOUNDS(kBK * ks + kBK <= p.K)) {
        load_w64<FMT>(wrow, ks, v);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = 0.f;
      }
      store_row_bf16(wtile, t, v);
#pragma unroll
      for (int rr = 0; rr < (BT + 127) / 128; ++rr) {
        const int r = t + 128 * rr;
        if (r < BT) {
          const int m = m0 + r;
          if (m < p.M && LQ_IN_BOUNDS(kBK * ks + kBK <= p.K)) {
            const float4* src = reinterpret_cast<const float4*>(p.A + static_cast<long long>(m) * p.K + kBK * ks);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float4 x = __ldg(src + i);
              v[4 * i] = x.x;
              v[4 * i + 1] = x.y;
              v[4 * i + 2] = x.z;
              v[4 * i + 3] = x.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) v[i] = 0.f;
          }
          store_row_bf16(ttile, r, v);
        }
      }
      fence_proxy_async_smem();  // make the generic-proxy stores visible to the tensor core
      mbar_arrive(&bars.full[s]);
    }
    if (!ok) {
      record_error(kDevErrTimeout);
      bars.abort = 1;
    }
    // ---------------- epilogue ----------------
    const bool have = mbar_wait(&bars.tmem_full, 0, p.wait_ns, p.wait_iters);
    if (!have) {
      record_error(kDevErrTimeout);
      bars.abort = 1;
    }
    tc::fence_after_sync();
    if (have && !bars.abort) {
      const int nrow = n0 + 32 * warp + lane;
#pragma unroll 1
      for (int c = 0; c < (BT + 31) / 32; ++c) {
        uint32_t r[32];
        tc::ld_32x32b_x32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 32u * c, r);
        tc::wait_ld();
        if (nrow < p.N) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = m0 + 32 * c + j;
            if (32 * c + j < BT && m < p.M && LQ_IN_BOUNDS(m >= 0 && nrow >= 0))
              p.C[static_cast<long long>(m) * p.N + nrow] = __uint_as_float(r[j]);
          }
        }
      }
    }
  } else if (lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = tc::idesc_bf16_f32(kBN, BT);
    int issued = 0;
    for (int ks = 0; ks < nk; ++ks) {
      const int s = ks % kStages;
      if (!mbar_wait(&bars.full[s], (ks / kStages) & 1, p.wait_ns, p.wait_iters) || bars.abort) {
        record_error(kDevErrTimeout);
        bars.abort = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t wtile = base_u + s * kStageBytes;
      const uint64_t adesc = tc::desc_sw128_kmajor(wtile);
      const uint64_t bdesc = tc::desc_sw128_kmajor(wtile + kWTileBytes);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        // +32 bytes along K inside the swizzle atom = +2 in the address field
        tc::mma_bf16(tmem, adesc + 2u * kk, bdesc + 2u * kk, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
      }
      tc::commit(&bars.empty[s]);
      ++issued;
    }
    // Completion of every issued MMA (or nothing, when none was issued).
    tc::commit(&bars.tmem_full);
    if (bars.abort) mbar_wait(&bars.tmem_full, 0, kDrainWaitNs);
    (void)issued;
  }
  // ---------------- teardown ----------------
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kConvWarps) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                   Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int FMT, int BT>
lq_status launch_tc_t(const MatmulArgs& a) {
  auto kern = gemm_tc_kernel<FMT, BT>;
  const size_t smem = 1024 + static_cast<size_t>(kStages) * (kWTileBytes + BT * kBK * 2) + 256;
  static int configured[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_CUDA;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e);
    configured[dev] = 1;
  }
  TcParams p;
  p.A = a.A;
  p.W = static_cast<const uint8_t*>(a.W);
  p.C = a.C;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.rb = row_bytes(a.fmt, a.K);
  p.wait_ns = wait_limit_ns();
  p.wait_iters = wait_limit_iters();
  const dim3 grid(static_cast<unsigned>((a.N + kBN - 1) / kBN), static_cast<unsigned>((a.M + BT - 1) / BT));
  cudaError_t e = launch(kern, grid, dim3(kTcThreads), smem, a.stream, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

template <int FMT>
lq_status launch_tc_fmt(const MatmulArgs& a) {
  if (a.M <= 16) return launch_tc_t<FMT, 16>(a);
  if (a.M <= 32) return launch_tc_t<FMT, 32>(a);
  if (a.M <= 64) return launch_tc_t<FMT, 64>(a);
  if (a.M <= 128) return launch_tc_t<FMT, 128>(a);
  return launch_tc_t<FMT, 256>(a);
}

bool aligned(const void* p, unsigned al) { return (reinterpret_cast<uintptr_t>(p) % al) == 0; }

}  // namespace

unsigned read_clear_gemm_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemm_err, &z, sizeof(z));
  return v;
}

bool gemm_tc_eligible(const MatmulArgs& a) {
  if (a.a_perm || a.epi != 0) return false;  // neither interleaved Q4_0 nor epilogues here
  if (a.M < 2 || a.K % kBK != 0) return false;
  if (!aligned(a.A, 16)) return false;
  // W rows: 16-byte loads for f16, 4-byte loads for the block formats
  if (!aligned(a.W, a.fmt == LQ_FMT_F16 ? 16 : 4)) return false;
  const DeviceInfo& di = device_info();
  return di.cc_major >= 10;
}

lq_status launch_gemm_tc(const MatmulArgs& a) {
  if (!gemm_tc_eligible(a)) return LQ_ERR_UNSUPPORTED;
  lq_status st;
  if (a.fmt == LQ_FMT_F16)
    st = launch_tc_fmt<LQ_FMT_F16>(a);
  else if (a.fmt == LQ_FMT_Q8_0)
    st = launch_tc_fmt<LQ_FMT_Q8_0>(a);
  else
    st = launch_tc_fmt<LQ_FMT_Q4_0>(a);
  if (st == LQ_OK) count_route(2);
  return st;
}

lq_status launch_gemm_stream(const MatmulArgs& a) { return launch_gemv_generic(a); }

}  // namespace lq
