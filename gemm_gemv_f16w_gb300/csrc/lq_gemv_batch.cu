// Batched decode: C[m, n] = sum_k A[m, k] * w(n, k) for M = 2..8 rows of A
// (several sequences decoded together; route 1, the CUDA-core streaming
// GEMM). The pages' counterpart is the NR x NM multi-row GEMV pattern of
// gemm_q4 / gemm_q8 (lattice-inference 0.1.2, src/forward/metal_qwen35.rs),
// which reads each weight block once for several rows of A.
//
// The streaming GEMV (lq_gemv.cu) with the weights dequantised once per lane
// and multiplied with all M activation rows:
//
//  * one CTA per SM owns a contiguous range of W rows, streamed in stages of
//    up to 8 rows through a ring of shared-memory slots (one bulk copy per
//    stage, mbarrier transaction counts);
//  * every ring slot gets its first weight stage at kernel start (weights
//    depend on nothing); A (all M rows) is read once the previous kernel on
//    the stream completed: f16 with one bulk copy into place, the quantised
//    formats by the consumers with plain loads (up to 16 in flight per
//    thread) straight into the 144-byte block slots the slices read;
//  * the warps form the K-groups x row-groups grid of the GEMV, a row-group
//    taking whole stages (ring depth a multiple of the row-group count);
//    every lane holds its chunk of all M activation rows (five to eight
//    rows: half a quantised block per lane, lq_gemv_slices_batch.cuh);
//  * per stage each warp reduces its row partials per token with the
//    transposed shuffle tree; the stage's finisher adds the K-groups in a
//    fixed order and writes the M outputs of each row.
//
// f32 activations and exact dequantisation: the results meet the GEMV
// tolerance. Every wait is bounded (LQ_ERR_DEVICE_TIMEOUT on expiry).
#include <algorithm>

#include "lq_device.cuh"
#include "lq_epilogue.cuh"
#include "lq_gemv_slices_batch.cuh"
#include "lq_internal.h"
#include "lq_q4i.cuh"

namespace lq {
namespace {

using namespace gemv;

__device__ unsigned g_batch_err;

constexpr int kBKGroups = 8;   // K-groups at most (reduction buffer width)
constexpr int kBRows = 8;      // rows per stage at most
constexpr int kBMaxStages = 16;
constexpr int kBMaxTokens = 8;

// Warps per CTA, all of them consumers. The f16 slices up to four tokens and
// the two-token quantised slices fit in 128 registers, so 16 warps; the
// quantised four-token slices and every eight-token slice (with eight
// tokens' partial sums of a stage) need up to 255, so 8 (two per SM
// sub-partition).
__host__ __device__ constexpr int batch_warps(int fmt, int mt) {
  return mt > 4 ? 8 : (fmt == LQ_FMT_F16 || mt == 2 ? 16 : 8);
}

struct BatchParams {
  const float* A;
  const uint8_t* W;
  float* C;
  int M, N, K;
  int row_bytes;
  int rows_per_stage;     // at most kBRows
  int stages;             // ring depth, a multiple of nr
  int nk, nr;             // K-groups x row-groups
  int a_slot;             // bytes of one token's A as the slices read it
  unsigned long long wait_ns;
  unsigned wait_iters;
  const float* R;         // residual epilogue: added to every output
  long long up_off;       // swiglu epilogue: bytes from a gate row to its up row
  int a_perm;             // Q4_0 with interleaved nibbles: A reordered per block
};

template <int MT>
struct BatchHeader {
  uint64_t full[kBMaxStages];
  uint64_t red_full[kBMaxStages];
  uint64_t a_bar;
  int last[kBMaxStages];  // last stage issued into each slot (-1: none)
  volatile int abort;
  int row0, nrows;        // this CTA's rows
  float red[kBMaxStages][MT][kBRows][kBKGroups];
};
template <int MT>
__host__ __device__ constexpr int batch_header_bytes() {
  return (static_cast<int>(sizeof(BatchHeader<MT>)) + 127) / 128 * 128;
}

__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_batch_err, 0u, code); }

// No producer warp. The ring is refilled by the finisher of a stage: once
// every K-group has posted its partials for slot s no warp reads the slot's
// weights any more, and once the finisher has summed the partials its lane 0
// issues the stage S further on into the slot.
//
// EPI (lq_epilogue.cuh): kResidual adds R[m, n]; a kSwiglu stage of n
// outputs holds their n gate rows followed by their n up rows (two bulk
// copies), and output j of the stage is swiglu(gate sum j, up sum j).
template <int FMT, int MT, int EPI>
__global__ void __launch_bounds__(batch_warps(FMT, MT) * 32, 1) gemv_batch_kernel(const BatchParams p) {
  constexpr int NW = batch_warps(FMT, MT);
  constexpr bool SWIGLU = EPI == epi::kSwiglu;
  extern __shared__ __align__(1024) uint8_t smem[];
  BatchHeader<MT>& hd = *reinterpret_cast<BatchHeader<MT>*>(smem);
  uint8_t* sA = smem + batch_header_bytes<MT>();  // MT x a_slot
  uint8_t* ring = sA + MT * p.a_slot;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int RS = p.rows_per_stage, S = p.stages, nk = p.nk, nr = p.nr, active = nk * nr;
  const uint32_t stage_bytes = static_cast<uint32_t>(SWIGLU ? 2 * RS : RS) * p.row_bytes;
  if (S % nr != 0 || S > kBMaxStages || nk > kBKGroups || active > NW || (SWIGLU ? 2 * RS : RS) > kBRows ||
      p.M > MT) {
    if (threadIdx.x == 0) record_error(LQ_ERR_UNSUPPORTED);
    return;
  }
  // this CTA's rows: worked out by thread 0 (64-bit divisions are long
  // sequences), which issues the first stages, and read by the rest after
  // the block barrier
  int r0 = 0, nrows = 0, nst = 0;
  const uint8_t* wbase = p.W;
  auto set_rows = [&](int a, int n) {
    r0 = a;
    nrows = n;
    nst = (n + RS - 1) / RS;
    wbase = p.W + static_cast<long long>(a) * p.row_bytes;
  };
  auto issue = [&](int st, int s, uint64_t pol) {  // stage st into slot s
    if (!LQ_IN_BOUNDS(st >= 0 && r0 + st * RS + min(RS, nrows - st * RS) <= p.N)) return;
    const uint32_t bytes = static_cast<uint32_t>(min(RS, nrows - st * RS)) * p.row_bytes;
    uint8_t* dst = ring + static_cast<size_t>(s) * stage_bytes;
    const uint8_t* src = wbase + static_cast<long long>(st) * RS * p.row_bytes;
    hd.last[s] = st;
    if constexpr (SWIGLU) {
      mbar_arrive_expect_tx(&hd.full[s], 2u * bytes);
      bulk_g2s(dst, src, bytes, &hd.full[s], pol);
      bulk_g2s(dst + bytes, src + p.up_off, bytes, &hd.full[s], pol);  // up rows right after
    } else {
      mbar_arrive_expect_tx(&hd.full[s], bytes);
      bulk_g2s(dst, src, bytes, &hd.full[s], pol);
    }
  };

  if (threadIdx.x == 0) {
    const long long G = gridDim.x;
    const int a = static_cast<int>((static_cast<long long>(blockIdx.x) * p.N) / G);
    const int n = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * p.N) / G) - a;
    hd.row0 = a;
    hd.nrows = n;
    set_rows(a, n);
    for (int s = 0; s < S; ++s) {
      mbar_init(&hd.full[s], 1);
      mbar_init(&hd.red_full[s], nk);
      hd.last[s] = -1;
    }
    mbar_init(&hd.a_bar, 1);
    hd.abort = 0;
    fence_barrier_init();
    const uint64_t pol = policy_evict_first();
    for (int st = 0; st < min(nst, S); ++st) issue(st, st, pol);  // weights depend on nothing
    if (FMT == LQ_FMT_F16) {
      // A (M rows, contiguous, in place) once the previous kernel on the
      // stream completed
      pdl_wait();
      const uint32_t a_bytes = static_cast<uint32_t>(p.M) * static_cast<uint32_t>(p.K) * 4u;
      mbar_arrive_expect_tx(&hd.a_bar, a_bytes);
      bulk_g2s(sA, p.A, a_bytes, &hd.a_bar, policy_evict_last());
    }
  }
  __syncthreads();
  pdl_launch_dependents();
  set_rows(hd.row0, hd.nrows);

  if (warp < active && nrows > 0) {
    if (FMT == LQ_FMT_F16) {
      // One lead thread waits for the copy of A under the time limit; the
      // other consumers follow its outcome (a named barrier has no time
      // limit, so every consumer has to reach it) and then observe the
      // landed copy themselves.
      if (threadIdx.x == 0 && !mbar_wait(&hd.a_bar, 0, p.wait_ns, p.wait_iters)) {
        record_error(kDevErrTimeout);
        hd.abort = 1;
      }
      named_barrier(1, static_cast<uint32_t>(active) * 32u);
      if (!hd.abort && threadIdx.x != 0) mbar_wait(&hd.a_bar, 0, kDrainWaitNs);
    } else {
      // A (M rows) straight from global memory into the block slots the
      // slices read, once the previous kernel on the stream completed: each
      // thread issues up to 16 loads of 16 bytes before storing any
      pdl_wait();
      const uint32_t sa = smem_u32(sA);
      const int per = p.K / 4, total = p.M * per, nthr = active * 32;
      const float* A = p.A;
#pragma unroll 1
      for (int q0 = warp * 32 + lane; q0 < total; q0 += 16 * nthr) {
        float4 v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int q = q0 + u * nthr;
          if (q < total && LQ_IN_BOUNDS(q >= 0)) v[u] = ldg128f(A + 4LL * q);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int q = q0 + u * nthr;
          if (q >= total) break;
          const int t = q / per, c = q - t * per;
          const uint32_t blk =
              sa + static_cast<uint32_t>(t * p.a_slot) + static_cast<uint32_t>(a_slot_q(c >> 3)) * kASlotBytes;
          const uint4 w = make_uint4(__float_as_uint(v[u].x), __float_as_uint(v[u].y), __float_as_uint(v[u].z),
                                     __float_as_uint(v[u].w));
          if (p.a_perm)
            q4i::store_chunk(blk, c & 7, w);
          else
            sts128(blk + 16u * (c & 7), w);
        }
      }
      named_barrier(2, static_cast<uint32_t>(active) * 32u);
    }
    if (!hd.abort) {
      pdl_wait();  // returns at once: the previous kernel has completed
      const uint64_t pol = policy_evict_first();
      const int kg = warp % nk, rg = warp / nk;
      typename SliceM<FMT, MT>::T sl;
      sl.init(smem_u32(sA), static_cast<uint32_t>(p.a_slot), kg, lane, p.K);
      const uint32_t ring_u = smem_u32(ring);
      // stages rg, rg + nr, ...: slot st mod S, ring phase (st / S) mod 2 and
      // finisher (st / nr) mod nk, advanced incrementally
      int s = rg, kf = 0;
      uint32_t ph = 0;
      for (int st = rg; st < nst; st += nr) {
        if (!mbar_wait(&hd.full[s], ph, p.wait_ns, p.wait_iters) || hd.abort) {
          record_error(kDevErrTimeout);
          hd.abort = 1;
          break;
        }
        const int rows = min(RS, nrows - st * RS);
        const uint32_t base = ring_u + static_cast<uint32_t>(s) * stage_bytes;
        float acc[MT][kBRows];
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int r = 0; r < kBRows; ++r) acc[t][r] = 0.f;
        if (sl.ok) {
#pragma unroll
          for (int r = 0; r < kBRows; ++r) {
            // swiglu: slot rows 0 .. rows-1 are gate rows, rows .. 2rows-1 up rows
            if (r < (SWIGLU ? 2 * rows : rows)) {
              float o[MT];
              sl.dot(base + static_cast<uint32_t>(r) * p.row_bytes, o);
#pragma unroll
              for (int t = 0; t < MT; ++t) acc[t][r] = o[t];
            }
          }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          int r;
          const float v = transpose_reduce8(acc[t], lane, r);
          if ((lane & 3) == 0) hd.red[s][t][r][kg] = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hd.red_full[s]);
        if (kg == kf) {
          // finisher: adds the K-groups' partials in a fixed order, one
          // output per token, then refills slot s. The refill comes last: its
          // landing releases the row-group's next stage in this slot, whose
          // partials overwrite red[s]. (Residual: R is fetched while the
          // other K-groups finish.)
          float rres[MT];
#pragma unroll
          for (int t = 0; t < MT; ++t)
            rres[t] = EPI == epi::kResidual && lane < rows && t < p.M &&
                              LQ_IN_BOUNDS(r0 + st * RS + lane < p.N)
                          ? p.R[static_cast<long long>(t) * p.N + r0 + st * RS + lane]
                          : 0.f;
          if (!mbar_wait(&hd.red_full[s], ph, p.wait_ns, p.wait_iters) || hd.abort) {
            record_error(kDevErrTimeout);
            hd.abort = 1;
            break;
          }
          const bool row_ok = lane < rows && LQ_IN_BOUNDS(r0 + st * RS + lane < p.N);
          if (SWIGLU && row_ok) {
            // one token at a time: a copy of silu per token would bloat the loop
#pragma unroll 1
            for (int t = 0; t < p.M; ++t) {
              float sum = 0.f, up = 0.f;
              for (int g = 0; g < nk; ++g) {
                sum += hd.red[s][t][lane][g];
                up += hd.red[s][t][rows + lane][g];
              }
              p.C[static_cast<long long>(t) * p.N + r0 + st * RS + lane] = epi::swiglu(sum, up);
            }
          } else if (row_ok) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              if (t < p.M) {
                float sum = 0.f;
                for (int g = 0; g < nk; ++g) sum += hd.red[s][t][lane][g];
                const long long o = static_cast<long long>(t) * p.N + r0 + st * RS + lane;
                if constexpr (EPI == epi::kResidual) {
                  p.C[o] = sum + rres[t];
                } else {
                  p.C[o] = sum;
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0 && st + S < nst) issue(st + S, s, pol);
        }
        s += nr;
        if (s >= S) {
          s -= S;
          ph ^= 1u;
        }
        if (++kf == nk) kf = 0;
      }
    }
  }
  // Every warp gets here (all waits are bounded); no copy may still be in
  // flight when the CTA exits.
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s)
      if (hd.last[s] >= 0) mbar_wait(&hd.full[s], (hd.last[s] / S) & 1, kDrainWaitNs);
    if (FMT == LQ_FMT_F16) mbar_wait(&hd.a_bar, 0, kDrainWaitNs);
  }
}

template <int FMT, int MT, int EPI>
lq_status launch_batch_t(const MatmulArgs& a, const BatchParams& p, int G, size_t smem) {
  auto kern = gemv_batch_kernel<FMT, MT, EPI>;
  static int configured[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_CUDA;
  if (configured[dev] < static_cast<int>(smem)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e);
    configured[dev] = static_cast<int>(smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G));
  cfg.blockDim = dim3(static_cast<unsigned>(batch_warps(FMT, MT) * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

template <int FMT, int EPI>
lq_status launch_batch_mt(const MatmulArgs& a, const BatchParams& p, int G, size_t smem, int MT) {
  if (MT == 2) return launch_batch_t<FMT, 2, EPI>(a, p, G, smem);
  if (MT == 4) return launch_batch_t<FMT, 4, EPI>(a, p, G, smem);
  return launch_batch_t<FMT, 8, EPI>(a, p, G, smem);
}

template <int FMT>
lq_status launch_batch_fmt(const MatmulArgs& a, const BatchParams& p, int G, size_t smem, int MT) {
  switch (a.epi) {
    case epi::kPlain: return launch_batch_mt<FMT, epi::kPlain>(a, p, G, smem, MT);
    case epi::kResidual: return launch_batch_mt<FMT, epi::kResidual>(a, p, G, smem, MT);
    case epi::kSwiglu: return launch_batch_mt<FMT, epi::kSwiglu>(a, p, G, smem, MT);
    default: return LQ_ERR_UNSUPPORTED;
  }
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

unsigned read_clear_batch_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_batch_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_batch_err, &z, sizeof(z));
  return v;
}

lq_status launch_gemv_batch(const MatmulArgs& a) {
  const int64_t M = a.M, N = a.N, K = a.K;
  // the streaming GEMV's shapes, one chunk per warp
  const bool shape_ok = M >= 2 && M <= kBMaxTokens && K <= 16384 && N < (1LL << 30) &&
                        (a.fmt == LQ_FMT_F16 ? (K % 8 == 0) : (K % 256 == 0));
  if (!shape_ok || !aligned16(a.A) || !aligned16(a.W)) return LQ_ERR_UNSUPPORTED;
  const int MT = M <= 2 ? 2 : (M <= 4 ? 4 : 8);
  int nk;
  if (a.fmt == LQ_FMT_F16) {
    const int nch = static_cast<int>((K + 255) / 256);
    if (nch > kBKGroups) return LQ_ERR_UNSUPPORTED;
    nk = 1;
    while (nk < nch) nk *= 2;
  } else {
    const int nseg = static_cast<int>((K / 32 + 63) / 64);
    if (kgroups_per_segment(MT) * nseg > kBKGroups) return LQ_ERR_UNSUPPORTED;
    nk = kgroups_per_segment(MT) * nseg;
  }
  const int NW = batch_warps(a.fmt, MT);
  const DeviceInfo& di = device_info();
  const int G = static_cast<int>(std::min<int64_t>(N, di.sm_count));
  // a swiglu "row" is a gate row and its up row, moved together
  const bool swiglu = a.epi == epi::kSwiglu;
  if (a.epi != epi::kPlain && a.epi != epi::kResidual && !swiglu) return LQ_ERR_UNSUPPORTED;
  const int wrb = static_cast<int>(row_bytes(a.fmt, K));
  const int rb = swiglu ? 2 * wrb : wrb;
  const int max_rows = swiglu ? kBRows / 2 : kBRows;
  const int a_slot = a.fmt == LQ_FMT_F16 ? static_cast<int>(K * 4)
                                         : static_cast<int>((K / 32 + 63) / 64) * 64 * kASlotBytes;
  const int hdr = MT == 2 ? batch_header_bytes<2>() : (MT == 4 ? batch_header_bytes<4>() : batch_header_bytes<8>());
  const int budget = std::min(di.max_smem_optin, 227 * 1024) - hdr - MT * a_slot;
  const int rows_per_cta = static_cast<int>((N + G - 1) / G);
  if (budget < 2 * rb) return LQ_ERR_UNSUPPORTED;
  // Stage height: as large as 8 rows while two stages fit; then as many
  // row-groups as there are stages (up to the warps over the K-groups), and
  // the height balanced so that every row-group gets the same number of
  // stages. The ring takes as many slots as fit, a multiple of nr and never
  // more than the CTA's stages rounded up to nr.
  const int rs_max = std::max(1, std::min({max_rows, budget / (2 * rb), rows_per_cta}));
  const int need_max = (rows_per_cta + rs_max - 1) / rs_max;
  int nr = std::max(1, std::min(NW / nk, need_max));
  const int cap_slots = std::min(kBMaxStages, budget / (rs_max * rb));
  while (nr > 1 && cap_slots < nr) --nr;
  const int total = nr * ((need_max + nr - 1) / nr);
  const int RS = std::max(1, (rows_per_cta + total - 1) / total);
  const int need = (rows_per_cta + RS - 1) / RS;
  int S = std::min(kBMaxStages, budget / (RS * rb));
  S -= S % nr;
  S = std::min(S, nr * ((need + nr - 1) / nr));
  if (S < 1) return LQ_ERR_UNSUPPORTED;
  const int ring = S * RS * rb;
  BatchParams p = {};
  p.A = a.A;
  p.W = static_cast<const uint8_t*>(a.W);
  p.C = a.C;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.row_bytes = wrb;
  p.rows_per_stage = RS;
  p.R = a.R;
  p.up_off = static_cast<long long>(N) * wrb;
  p.a_perm = a.a_perm ? 1 : 0;
  p.nk = nk;
  p.nr = nr;
  p.stages = S;
  p.a_slot = a_slot;
  p.wait_ns = wait_limit_ns();
  p.wait_iters = wait_limit_iters();
  const size_t smem = static_cast<size_t>(hdr) + MT * static_cast<size_t>(a_slot) + ring;
  lq_status st;
  if (a.fmt == LQ_FMT_F16)
    st = launch_batch_fmt<LQ_FMT_F16>(a, p, G, smem, MT);
  else if (a.fmt == LQ_FMT_Q8_0)
    st = launch_batch_fmt<LQ_FMT_Q8_0>(a, p, G, smem, MT);
  else
    st = launch_batch_fmt<LQ_FMT_Q4_0>(a, p, G, smem, MT);
  if (st == LQ_OK) count_route(1);
  return st;
}

}  // namespace lq
