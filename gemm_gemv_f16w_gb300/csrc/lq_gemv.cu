// Decode GEMV (M == 1): C[n] = sum_k A[k] * w(n, k) for f16, Q8_0 and Q4_0 W.
//
// Counterparts on the source pages (lattice-inference 0.1.2,
// src/forward/metal_qwen35.rs): gemv_decode_m1 / gemv_decode_core (f16),
// gemv_q8_decode and gemv_q4_decode (NR=2 rows per threadgroup, per-lane block
// slices, simd_sum). Those kernels read W with vector loads straight from
// unified memory and rely on many small threadgroups. On GB300 the weight
// stream has to keep ~7 TB/s of HBM busy, so this kernel is built around the
// copy engine instead:
//
//  * persistent CTAs (one or two per SM) each own a contiguous range of W
//    rows; a CTA stays within half an SM (<= 112 KB of shared memory, 288
//    threads of <= 112 registers) so that the next GEMV on the stream can be
//    resident beside it and start streaming its own weights while this one
//    finishes (programmatic dependent launch; weights never depend on the
//    previous kernel, activations and outputs are touched only after it
//    completed);
//  * a producer thread moves stages of up to 8 whole rows into a ring of
//    shared-memory slots, one 1-D bulk copy (cp.async.bulk) per stage, with
//    mbarrier transaction counts; small copies are slow, so stages are large;
//  * eight consumer warps form a grid of K-groups x row-groups: a warp
//    covers its K-slice of every row of its stages, keeps that slice of A in
//    registers, and has up to eight independent rows of work per stage;
//  * dequantisation happens in registers without int->float conversions:
//    a quantised value is dropped into the mantissa of 2^23 and unbiased with
//    one exact add/fma; dot products use packed f32x2 fma;
//  * each warp reduces its row partials across lanes with one transposed
//    shuffle tree; the stage's finisher warp adds the K-groups' partials in a
//    fixed order and writes C.
//
// Every wait is bounded (lq_device.cuh); on timeout the kernel records
// LQ_ERR_DEVICE_TIMEOUT, its producer drains its own copies and it returns.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "lq_argmax.cuh"
#include "lq_device.cuh"
#include "lq_epilogue.cuh"
#include "lq_gemv_slices.cuh"
#include "lq_internal.h"
#include "lq_q4i.cuh"

namespace lq {
namespace {

using namespace gemv;

__device__ unsigned g_gemv_err;

constexpr int kConsumerWarps = 8;              // K-groups x row-groups
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kRowsPerStage = 8;               // rows moved by one bulk copy
constexpr int kMaxStages = 12;
constexpr int kGemvFastMaxK = 16384;
constexpr int kHalfSmSmem = 112 * 1024;        // two CTAs fit on one SM
constexpr int64_t kL2PrefetchMaxBytes = 32LL << 20;

struct GemvParams {
  const float* A;
  const uint8_t* W;
  float* C;
  int N, K;
  int row_bytes;
  int rows_per_stage;        // <= kRowsPerStage
  int stages;                // ring depth
  int nk, nr;                // consumer warp grid: nk K-groups x nr row-groups
  int a_region;              // bytes of shared memory for A (a multiple of 128)
  int a_stage;               // bytes of the staging area for A (0 for f16)
  int l2_prefetch;           // prefetch the rows beyond the first ring-full into L2
  unsigned long long wait_ns;
  unsigned wait_iters;
  lq_argmax_result* amax;    // argmax variant: the result (C may then be null)
  unsigned amax_warps;       // argmax variant: consumer warps of the grid
  const float* R;            // residual variant: added to every output
  long long up_off;          // swiglu variant: bytes from a gate row to its up row
  int a_perm;                // Q4_0 with interleaved nibbles: A reordered per block
};

struct Header {
  uint64_t full[kMaxStages];       // stage landed (TMA transaction bytes)
  uint64_t empty[kMaxStages];      // every consumer warp is done with the stage
  uint64_t red_full[kMaxStages];   // every consumer warp wrote its row partials
  uint64_t a_bar;                  // A landed in the staging area
  volatile int abort;
  int row0, nrows;                 // this CTA's rows
  float red[kMaxStages][kRowsPerStage][kConsumerWarps];  // [slot][row][K-group]
};
constexpr int kHeaderBytes = (static_cast<int>(sizeof(Header)) + 127) / 128 * 128;

__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_gemv_err, 0u, code); }

// ---------------------------------------------------------------------------
// The streaming kernel. Consumer warp w < nk*nr is K-group kg = w % nk of
// row-group rg = w / nk; row-group rg takes stages rg, rg + nr, rg + 2nr,
// ..., all rows of each. Ring slot s holds stage st (st % S == s), and S is
// a multiple of nr, so each slot serves one row-group only. Its full barrier
// completes once per stage, and a slot is refilled only after the nk warps
// of its stage released it (empty barrier, after the stage's finisher read
// the slot's reduction buffer), so a waiter sees either the phase it waits
// for or the one before it, never an older one.
//
// EPI (lq_epilogue.cuh) picks what the finisher does with a row's sum:
//  * kArgmax (lq_gemv_argmax): a finisher lane ranks each row it writes, and
//    every consumer warp merges its best row into the result once its stages
//    are done (lq_argmax.cuh);
//  * kResidual: adds R[n];
//  * kSwiglu: a stage of n outputs holds their n gate rows followed by their
//    n up rows (two bulk copies, the up rows up_off bytes further on in W);
//    output j of the stage is swiglu(sum of slot row j, sum of slot row
//    n + j).
// ---------------------------------------------------------------------------
template <int FMT, int CPW, int EPI>
__global__ void __launch_bounds__(kGemvThreads, CPW <= 2 ? 2 : 1)
    gemv_stream_kernel(const GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Header& hd = *reinterpret_cast<Header*>(smem);
  uint8_t* sA = smem + kHeaderBytes;            // A as the slices read it
  uint8_t* stage_a = sA + p.a_region;           // A as copied (quantised formats)
  uint8_t* ring = stage_a + p.a_stage;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int RS = p.rows_per_stage, S = p.stages;
  const int nk = p.nk, nr = p.nr, active = nk * nr;
  constexpr bool AMAX = EPI == epi::kArgmax, SWIGLU = EPI == epi::kSwiglu;
  const uint32_t stage_bytes = static_cast<uint32_t>(SWIGLU ? 2 * RS : RS) * p.row_bytes;
  // The host plans S as a multiple of nr (see plan_gemv); refuse anything else.
  if (S % nr != 0 || S > kMaxStages || active > kConsumerWarps || (SWIGLU && 2 * RS > kRowsPerStage)) {
    if (threadIdx.x == 0) record_error(LQ_ERR_UNSUPPORTED);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hd.full[s], 1);
      mbar_init(&hd.empty[s], nk);
      mbar_init(&hd.red_full[s], nk);
    }
    mbar_init(&hd.a_bar, 1);
    hd.abort = 0;
    // this CTA's rows (one thread: 64-bit divisions are long sequences)
    const long long G = gridDim.x;
    const int a = static_cast<int>((static_cast<long long>(blockIdx.x) * p.N) / G);
    hd.row0 = a;
    hd.nrows = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * p.N) / G) - a;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  const int r0 = hd.row0, nrows = hd.nrows;
  const int nst = (nrows + RS - 1) / RS;

  if (warp == kConsumerWarps) {
    // ---------------- producer ----------------
    const uint64_t pol = policy_evict_first();
    const uint8_t* wbase = p.W + static_cast<long long>(r0) * p.row_bytes;
    auto issue = [&](int st, int s) {  // stage st into slot s
      const int rows = min(RS, nrows - st * RS);
      if (!LQ_IN_BOUNDS(st >= 0 && rows > 0 && r0 + st * RS + rows <= p.N)) return;
      const uint32_t bytes = static_cast<uint32_t>(rows) * p.row_bytes;
      uint8_t* dst = ring + static_cast<size_t>(s) * stage_bytes;
      const uint8_t* src = wbase + static_cast<long long>(st) * RS * p.row_bytes;
      if constexpr (SWIGLU) {
        mbar_arrive_expect_tx(&hd.full[s], 2u * bytes);
        bulk_g2s(dst, src, bytes, &hd.full[s], pol);
        bulk_g2s(dst + bytes, src + p.up_off, bytes, &hd.full[s], pol);  // up rows right after
      } else {
        mbar_arrive_expect_tx(&hd.full[s], bytes);
        bulk_g2s(dst, src, bytes, &hd.full[s], pol);
      }
    };
    // W never depends on the previous kernel: fill the ring at once. The
    // rows that do not fit in it are prefetched into L2 at the same time, so
    // that the refills later hit L2 (only when the whole matrix is small next
    // to L2; otherwise the prefetched lines would not survive).
    if (lane != 0) return;
    const int first = min(nst, S);
    for (int st = 0; st < first; ++st) issue(st, st);
    if (p.l2_prefetch && nst > S) {
      const long long done = static_cast<long long>(S) * RS * p.row_bytes;
      const long long rest = static_cast<long long>(nrows) * p.row_bytes - done;
      bulk_prefetch_l2(wbase + done, static_cast<uint32_t>(rest));
    }
    // A may come from the previous kernel: one bulk copy once that one has
    // completed (f16 straight into place; quantised formats into the staging
    // area, which the consumers spread into the block slots).
    pdl_wait();
    mbar_arrive_expect_tx(&hd.a_bar, static_cast<uint32_t>(p.K) * 4u);
    bulk_g2s(FMT == LQ_FMT_F16 ? sA : stage_a, p.A, static_cast<uint32_t>(p.K) * 4u, &hd.a_bar,
             policy_evict_last());
    int issued = first;
    bool ok = true;
    // stages past the first S (first == S here): slot s of ring lap `lap`
    // once the consumers released the slot's previous lap
    int s = 0, lap = 1;
    for (int st = first; st < nst; ++st) {
      if (!mbar_wait(&hd.empty[s], static_cast<uint32_t>(lap - 1) & 1, p.wait_ns, p.wait_iters) || hd.abort) {
        ok = false;
        break;
      }
      issue(st, s);
      ++issued;
      if (++s == S) {
        s = 0;
        ++lap;
      }
    }
    if (!ok) {
      record_error(kDevErrTimeout);
      hd.abort = 1;
    }
    // Never leave copies in flight: consumers may have given up already.
    for (int st = max(0, issued - S); st < issued; ++st)
      mbar_wait(&hd.full[st % S], (st / S) & 1, kDrainWaitNs);
    mbar_wait(&hd.a_bar, 0, kDrainWaitNs);
    return;
  }
  if (warp >= active) return;

  // ---------------- consumers ----------------
  // A arrives through the producer, which copies it only after the previous
  // kernel on the stream completed; C is written after that too.
  if (nrows == 0) return;
  if (!mbar_wait(&hd.a_bar, 0, p.wait_ns, p.wait_iters)) {
    record_error(kDevErrTimeout);
    hd.abort = 1;
    return;
  }
  pdl_wait();  // returns at once: the previous kernel has completed
  if (FMT != LQ_FMT_F16) {
    // staging area -> block slots: each warp moves 512 contiguous bytes per
    // step, and the four blocks they hold land in different bank groups
    const uint32_t sa = smem_u32(sA), sg = smem_u32(stage_a);
    for (int q = warp * 32 + lane; q < p.K / 4; q += active * 32) {
      const uint4 v = lds128(sg + 16u * q);
      const uint32_t blk = sa + static_cast<uint32_t>(a_slot_q(q >> 3)) * kASlotBytes;
      if (p.a_perm)
        q4i::store_chunk(blk, q & 7, v);
      else
        sts128(blk + 16u * (q & 7), v);
    }
    named_barrier(1, static_cast<uint32_t>(active) * 32u);
  }
  const int kg = warp % nk, rg = warp / nk;
  typename SliceOf<FMT, CPW>::T sl;
  sl.init(smem_u32(sA), kg, nk, lane, p.K);
  const uint32_t ring_u = smem_u32(ring);
  unsigned long long best = 0ull;  // argmax variant: this lane's best row
  // stages rg, rg + nr, ...: slot st mod S, ring phase (st / S) mod 2 and
  // finisher (st / nr) mod nk, advanced incrementally
  int s = rg, kf = 0;
  uint32_t ph = 0;
  for (int st = rg; st < nst; st += nr) {
    if (!mbar_wait(&hd.full[s], ph, p.wait_ns, p.wait_iters) || hd.abort) {
      record_error(kDevErrTimeout);
      hd.abort = 1;
      return;
    }
    const int rows = min(RS, nrows - st * RS);
    const uint32_t base = ring_u + static_cast<uint32_t>(s) * stage_bytes;
    float acc[kRowsPerStage];
#pragma unroll
    for (int r = 0; r < kRowsPerStage; ++r) acc[r] = 0.f;
    // swiglu: slot rows 0 .. rows-1 are gate rows, rows .. 2rows-1 up rows
    const int live = SWIGLU ? 2 * rows : rows;
#pragma unroll
    for (int i = 0; i < CPW; ++i) {
      if (sl.ok[i]) {
        if (FMT == LQ_FMT_F16 && CPW == 1 && live == kRowsPerStage) {
          // f16, a full stage: no per-row guard, so the rows' loads can
          // overlap (measured faster for f16 only; the quantised slices,
          // with their longer dequantisation, ran slower this way)
#pragma unroll
          for (int r = 0; r < kRowsPerStage; ++r) acc[r] += sl.dot(base + static_cast<uint32_t>(r) * p.row_bytes, i);
        } else {
#pragma unroll
          for (int r = 0; r < kRowsPerStage; ++r)
            if (r < live) acc[r] += sl.dot(base + static_cast<uint32_t>(r) * p.row_bytes, i);
        }
      }
    }
    int r;
    const float v = transpose_reduce8(acc, lane, r);
    if ((lane & 3) == 0) hd.red[s][r][kg] = v;
    __syncwarp();
    if (lane == 0) mbar_arrive(&hd.red_full[s]);
    if (kg == kf) {
      // finisher of this stage: the K-groups' partials, in a fixed order
      // (residual: R is fetched while the other K-groups finish)
      float rres = 0.f;
      if constexpr (EPI == epi::kResidual)
        if (lane < rows && LQ_IN_BOUNDS(r0 + st * RS + lane < p.N)) rres = p.R[r0 + st * RS + lane];
      if (!mbar_wait(&hd.red_full[s], ph, p.wait_ns, p.wait_iters) || hd.abort) {
        record_error(kDevErrTimeout);
        hd.abort = 1;
        return;
      }
      if (lane < rows && LQ_IN_BOUNDS(r0 + st * RS + lane < p.N)) {
        float sum = 0.f;
        for (int g = 0; g < nk; ++g) sum += hd.red[s][lane][g];
        const int row = r0 + st * RS + lane;
        if constexpr (AMAX) {
          const unsigned long long key = amax::make_key(sum, static_cast<unsigned>(row));
          best = key > best ? key : best;
          if (p.C) p.C[row] = sum;
        } else if constexpr (EPI == epi::kResidual) {
          p.C[row] = sum + rres;
        } else if constexpr (SWIGLU) {
          float up = 0.f;
          for (int g = 0; g < nk; ++g) up += hd.red[s][rows + lane][g];
          p.C[row] = epi::swiglu(sum, up);
        } else {
          p.C[row] = sum;
        }
      }
      __syncwarp();
    }
    if (lane == 0) mbar_arrive(&hd.empty[s]);
    s += nr;
    if (s >= S) {
      s -= S;
      ph ^= 1u;
    }
    if (++kf == nk) kf = 0;
  }
  if constexpr (AMAX) amax::warp_done(best, p.amax, p.amax_warps, lane);
}

// ---------------------------------------------------------------------------
// Generic kernel: any M, N, K (quantised K % 32 == 0), any W byte alignment.
// One warp per output element C[m, n]; W is read with byte loads. It is the
// correctness net under the fast kernels, not a performance path.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_f16_bytes(const uint8_t* p) {
  const unsigned short b = static_cast<unsigned short>(p[0]) | (static_cast<unsigned short>(p[1]) << 8);
  return __half2float(__ushort_as_half(b));
}

// The dot product of one W row with one row of A, summed over the warp
// (il: Q4_0 with interleaved nibbles, byte j = elements 2j and 2j+1).
template <int FMT>
__device__ __forceinline__ float generic_row_dot(const float* a, const uint8_t* w, int K, int lane, bool il) {
  float acc = 0.f;
  if (FMT == LQ_FMT_F16) {
    const __half* wh = reinterpret_cast<const __half*>(w);
    for (int k = lane; k < K; k += 32) acc = fmaf(a[k], __half2float(wh[k]), acc);
  } else if (FMT == LQ_FMT_Q8_0) {
    for (int b = lane; b < K / 32; b += 32) {
      const uint8_t* blk = w + 34LL * b;
      float s = 0.f;
      for (int i = 0; i < 32; ++i)
        s = fmaf(static_cast<float>(static_cast<int8_t>(blk[2 + i])), a[32 * b + i], s);
      acc = fmaf(load_f16_bytes(blk), s, acc);
    }
  } else {
    for (int b = lane; b < K / 32; b += 32) {
      const uint8_t* blk = w + 18LL * b;
      float s = 0.f;
      for (int i = 0; i < 16; ++i) {
        const int byte = blk[2 + i];
        s = fmaf(static_cast<float>((byte & 0xF) - 8), a[32 * b + (il ? 2 * i : i)], s);
        s = fmaf(static_cast<float>((byte >> 4) - 8), a[32 * b + (il ? 2 * i + 1 : 16 + i)], s);
      }
      acc = fmaf(load_f16_bytes(blk), s, acc);
    }
  }
  return warp_sum(acc);
}

// EPI as in the streaming kernel (no argmax here): residual adds R[m, n];
// swiglu reads rows n (gate) and N + n (up) of W.
template <int FMT, int EPI>
__global__ void __launch_bounds__(256) generic_matmul_kernel(const float* __restrict__ A,
                                                             const uint8_t* __restrict__ W,
                                                             float* __restrict__ C, int M, int N,
                                                             int K, long long row_bytes,
                                                             const float* __restrict__ R, int il) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  pdl_wait();
  if (n >= N) return;
  const uint8_t* w = W + static_cast<long long>(n) * row_bytes;
  for (int m = blockIdx.y; m < M; m += gridDim.y) {
    const float* a = A + static_cast<long long>(m) * K;
    const long long o = static_cast<long long>(m) * N + n;
    if (!LQ_IN_BOUNDS(o < static_cast<long long>(M) * N)) break;
    const float acc = generic_row_dot<FMT>(a, w, K, lane, il != 0);
    if constexpr (EPI == epi::kSwiglu) {
      const float up = generic_row_dot<FMT>(a, w + static_cast<long long>(N) * row_bytes, K, lane, il != 0);
      if (lane == 0) C[o] = epi::swiglu(acc, up);
    } else if constexpr (EPI == epi::kResidual) {
      if (lane == 0) C[o] = acc + R[o];
    } else {
      if (lane == 0) C[o] = acc;
    }
  }
}

// ---------------------------------------------------------------------------
// launch helpers
// ---------------------------------------------------------------------------
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

bool aligned(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Consumer warp grid for this format and K: nk K-groups x nr row-groups
// (nk * nr <= 8) and cpw chunks per warp. f16: chunks of 256 values, nk a
// power of two up to 8, cpw 1, 2, 4 or 8. Q8_0 / Q4_0: two K-groups (even and
// odd blocks) per segment of 64 blocks, up to four segments at a time, cpw
// 1 or 2.
struct WarpGrid {
  int nk = 0, nr = 0, cpw = 0;
};
WarpGrid pick_grid(int fmt, int K) {
  WarpGrid g;
  if (fmt == LQ_FMT_F16) {
    const int nch = (K + 255) / 256;
    g.nk = 1;
    while (g.nk < nch && g.nk < kConsumerWarps) g.nk *= 2;
    const int need = (nch + g.nk - 1) / g.nk;
    for (int c : {1, 2, 4, 8})
      if (c >= need) {
        g.cpw = c;
        break;
      }
  } else {
    const int nseg = (K / 32 + 63) / 64;
    g.nk = 2 * std::min(nseg, kConsumerWarps / 2);
    const int need = (nseg + g.nk / 2 - 1) / (g.nk / 2);
    g.cpw = need <= 1 ? 1 : (need <= 2 ? 2 : 0);
  }
  g.nr = g.cpw ? kConsumerWarps / g.nk : 0;
  return g;
}

template <int FMT, int CPW, int EPI>
lq_status launch_stream_t(const MatmulArgs& a, const GemvParams& p, int G, size_t smem) {
  auto kern = gemv_stream_kernel<FMT, CPW, EPI>;
  static int configured_smem[kMaxDevices] = {};  // per instantiation and device
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_CUDA;
  if (configured_smem[dev] < static_cast<int>(smem)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e);
    configured_smem[dev] = static_cast<int>(smem);
  }
  cudaError_t e = launch(kern, dim3(G), dim3(kGemvThreads), smem, a.stream, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

template <int FMT, int EPI>
lq_status launch_stream_fmt(const MatmulArgs& a, int cpw, const GemvParams& p, int G, size_t smem) {
  if constexpr (FMT != LQ_FMT_F16) {
    return cpw == 1 ? launch_stream_t<FMT, 1, EPI>(a, p, G, smem)
                    : (cpw == 2 ? launch_stream_t<FMT, 2, EPI>(a, p, G, smem) : LQ_ERR_UNSUPPORTED);
  } else {
    switch (cpw) {
      case 1: return launch_stream_t<FMT, 1, EPI>(a, p, G, smem);
      case 2: return launch_stream_t<FMT, 2, EPI>(a, p, G, smem);
      case 4: return launch_stream_t<FMT, 4, EPI>(a, p, G, smem);
      case 8: return launch_stream_t<FMT, 8, EPI>(a, p, G, smem);
      default: return LQ_ERR_UNSUPPORTED;
    }
  }
}

}  // namespace

unsigned read_clear_gemv_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemv_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_gemv_err, &z, sizeof(z));
  return v;
}

lq_status launch_gemv_generic(const MatmulArgs& a) {
  const dim3 grid(static_cast<unsigned>((a.N + 7) / 8),
                  static_cast<unsigned>(std::min<int64_t>(a.M, 65535)));
  const long long rb = row_bytes(a.fmt, a.K);
  const auto* W = static_cast<const uint8_t*>(a.W);
  const int M = static_cast<int>(a.M), N = static_cast<int>(a.N), K = static_cast<int>(a.K);
  if (a.epi != epi::kPlain && a.epi != epi::kResidual && a.epi != epi::kSwiglu) return LQ_ERR_UNSUPPORTED;
  auto go = [&](auto kern) {
    return launch(kern, grid, dim3(256), 0, a.stream, a.A, W, a.C, M, N, K, rb, a.R, a.a_perm ? 1 : 0);
  };
  auto by_epi = [&](auto fmt_tag) {
    constexpr int F = decltype(fmt_tag)::value;
    if (a.epi == epi::kResidual) return go(generic_matmul_kernel<F, epi::kResidual>);
    if (a.epi == epi::kSwiglu) return go(generic_matmul_kernel<F, epi::kSwiglu>);
    return go(generic_matmul_kernel<F, epi::kPlain>);
  };
  cudaError_t e;
  if (a.fmt == LQ_FMT_F16)
    e = by_epi(std::integral_constant<int, LQ_FMT_F16>{});
  else if (a.fmt == LQ_FMT_Q8_0)
    e = by_epi(std::integral_constant<int, LQ_FMT_Q8_0>{});
  else
    e = by_epi(std::integral_constant<int, LQ_FMT_Q4_0>{});
  if (e == cudaSuccess) e = cudaGetLastError();
  count_route(3);
  return cuda_status(e);
}

namespace {

// Launch plan of the streaming kernel: grid, warp grid, ring geometry and
// shared memory.
struct GemvPlan {
  GemvParams p;
  int grid = 0, cpw = 0;
  size_t smem = 0;
  bool ok = false;
};

// `ctas_per_sm` CTAs per SM, each with at most `smem_cap` bytes of shared
// memory; stages hold up to `max_rows` rows.
GemvPlan plan_gemv(const MatmulArgs& a, int ctas_per_sm, int max_rows, int smem_cap) {
  GemvPlan pl;
  const int K = static_cast<int>(a.K);
  // a swiglu "row" is a gate row and its up row, moved together
  const bool swiglu = a.epi == epi::kSwiglu;
  const int wrb = static_cast<int>(row_bytes(a.fmt, a.K));
  const int rb = swiglu ? 2 * wrb : wrb;
  if (swiglu) max_rows = std::min(max_rows, kRowsPerStage / 2);
  // Fast path: every stage start is 16-byte aligned for the bulk copies
  // (rows a multiple of 16 bytes), A is 16-byte aligned for vector loads,
  // and the per-lane slices cover K.
  const bool shape_ok = a.K <= kGemvFastMaxK &&
                        (a.fmt == LQ_FMT_F16 ? (K % 8 == 0) : (K % 256 == 0)) && a.N < (1LL << 30);
  const bool align_ok = aligned(a.W, 16) && aligned(a.A, 16);
  if (!shape_ok || !align_ok) return pl;
  const WarpGrid wg = pick_grid(a.fmt, K);
  if (wg.cpw == 0) return pl;

  const DeviceInfo& di = device_info();
  const int G = static_cast<int>(std::min<int64_t>(a.N, static_cast<int64_t>(di.sm_count) * ctas_per_sm));
  const int per_cta = std::min(di.max_smem_optin, smem_cap);
  // A in shared memory: in order for f16; for the quantised formats one
  // 144-byte slot per block, two parities x 32 slots per 64-block segment.
  const int a_bytes = a.fmt == LQ_FMT_F16 ? K * 4 : ((K / 32 + 63) / 64) * 64 * kASlotBytes;
  const int a_region = (a_bytes + 127) / 128 * 128;
  const int a_stage = a.fmt == LQ_FMT_F16 ? 0 : (K * 4 + 127) / 128 * 128;
  const int budget = per_cta - kHeaderBytes - a_region - a_stage;
  const int rows_per_cta = static_cast<int>((a.N + G - 1) / G);
  if (G < 1 || budget < 2 * rb) return pl;
  // up to max_rows rows per bulk copy, and room for at least two stages
  const int rs_max = std::max(1, std::min({max_rows, kRowsPerStage, budget / (2 * rb), rows_per_cta}));
  int stages = std::min({kMaxStages, budget / (rs_max * rb), std::max((rows_per_cta + rs_max - 1) / rs_max, 2)});
  if (stages < 2) return pl;
  // Row-groups take whole stages, and every ring slot must serve a single
  // row-group (stage st goes to slot st % S and to row-group st % nr): with
  // S a multiple of nr the warps of a slot see each of its phases in turn.
  // Otherwise a warp could wait on a slot whose previous use belonged to
  // another row-group, and with copies landing out of order the parity of
  // an older phase would satisfy its wait.
  // Prefer all eight warps; give up row-groups rather than drop below
  // three stages in flight.
  const int need_max = (rows_per_cta + rs_max - 1) / rs_max;
  int nr = std::max(1, std::min({wg.nr, need_max, stages}));
  while (nr > 1 && stages - stages % nr < std::min(3, stages)) --nr;
  // Even out the row-groups: a multiple of nr stages, rows spread over them.
  const int total = nr * ((need_max + nr - 1) / nr);
  const int rs = std::max(1, (rows_per_cta + total - 1) / total);
  const int stage_bytes = rs * rb;
  const int need_stages = (rows_per_cta + rs - 1) / rs;
  stages = std::min({kMaxStages, budget / stage_bytes, std::max(need_stages, 2)});
  const int ring = stages - stages % nr;
  if (ring < 1) return pl;

  GemvParams& p = pl.p;
  p.A = a.A;
  p.W = static_cast<const uint8_t*>(a.W);
  p.C = a.C;
  p.N = static_cast<int>(a.N);
  p.K = K;
  p.row_bytes = wrb;
  p.rows_per_stage = rs;
  p.stages = ring;
  p.nk = wg.nk;
  p.nr = nr;
  p.a_region = a_region;
  p.a_stage = a_stage;
  // L2 keeps a whole weight matrix of up to a quarter of its size
  p.l2_prefetch = !swiglu && static_cast<int64_t>(a.N) * rb <= kL2PrefetchMaxBytes ? 1 : 0;
  p.R = a.R;
  p.up_off = static_cast<long long>(a.N) * wrb;
  p.a_perm = a.a_perm ? 1 : 0;
  p.wait_ns = wait_limit_ns();
  p.wait_iters = wait_limit_iters();
  pl.cpw = wg.cpw;
  pl.grid = G;
  pl.smem = kHeaderBytes + a_region + a_stage + static_cast<size_t>(ring) * stage_bytes;
  pl.ok = true;
  return pl;
}

template <int EPI>
lq_status launch_plan_epi(const MatmulArgs& a, const GemvPlan& pl) {
  if (a.fmt == LQ_FMT_F16) return launch_stream_fmt<LQ_FMT_F16, EPI>(a, pl.cpw, pl.p, pl.grid, pl.smem);
  if (a.fmt == LQ_FMT_Q8_0) return launch_stream_fmt<LQ_FMT_Q8_0, EPI>(a, pl.cpw, pl.p, pl.grid, pl.smem);
  return launch_stream_fmt<LQ_FMT_Q4_0, EPI>(a, pl.cpw, pl.p, pl.grid, pl.smem);
}

lq_status launch_plan(const MatmulArgs& a, const GemvPlan& pl, int epi_kind) {
  switch (epi_kind) {
    case epi::kPlain: return launch_plan_epi<epi::kPlain>(a, pl);
    case epi::kArgmax: return launch_plan_epi<epi::kArgmax>(a, pl);
    case epi::kResidual: return launch_plan_epi<epi::kResidual>(a, pl);
    case epi::kSwiglu: return launch_plan_epi<epi::kSwiglu>(a, pl);
    default: return LQ_ERR_UNSUPPORTED;
  }
}

std::atomic<int> g_tune_ctas{0}, g_tune_rows{0}, g_tune_smem{0};

}  // namespace

void set_gemv_tuning(int ctas_per_sm, int rows_per_stage, int smem_cap) {
  g_tune_ctas.store(ctas_per_sm);
  g_tune_rows.store(rows_per_stage);
  g_tune_smem.store(smem_cap);
}

namespace {

// The launch plan launch_gemv uses (ok == false: the shape or the alignment
// is outside the streaming kernel's fast path).
GemvPlan plan_for(const MatmulArgs& a) {
  const WarpGrid wg = pick_grid(a.fmt, static_cast<int>(std::min<int64_t>(a.K, kGemvFastMaxK)));
  const DeviceInfo& di = device_info();
  // Kernels with one or two chunks per warp fit in half an SM (registers
  // and shared memory): two CTAs per SM, each streaming its own rows, give
  // the SM sixteen consumer warps and twice the bytes in flight (measured
  // faster than one CTA per SM that leaves room for the next kernel). With
  // fewer rows than that, one CTA per SM.
  int ctas = 1, smem_cap = di.max_smem_optin;
  if (wg.cpw <= 2) {
    smem_cap = kHalfSmSmem;
    ctas = a.N >= 2LL * kRowsPerStage * std::max(di.sm_count, 1) ? 2 : 1;
  }
  int rows = kRowsPerStage;
  if (const int c = g_tune_ctas.load()) ctas = c;
  if (const int r = g_tune_rows.load()) rows = r;
  if (const int m = g_tune_smem.load()) smem_cap = m;
  GemvPlan pl = plan_gemv(a, ctas, rows, smem_cap);
  // very long rows: two stages need more than half an SM
  if (!pl.ok) pl = plan_gemv(a, 1, kRowsPerStage, di.max_smem_optin);
  return pl;
}

}  // namespace

lq_status launch_gemv(const MatmulArgs& a) {
  const GemvPlan pl = plan_for(a);
  if (!pl.ok) return launch_gemv_generic(a);
  const lq_status st = launch_plan(a, pl, a.epi);
  if (st == LQ_ERR_UNSUPPORTED) return launch_gemv_generic(a);
  if (st == LQ_OK) count_route(0);
  return st;
}

lq_status launch_gemv_argmax(const MatmulArgs& a, lq_argmax_result* out) {
  GemvPlan pl = plan_for(a);
  if (!pl.ok) return LQ_ERR_UNSUPPORTED;
  // every CTA owns at least one row (grid <= N), so every consumer warp of
  // the grid reaches the merge
  pl.p.amax = out;
  pl.p.amax_warps = static_cast<unsigned>(pl.grid) * static_cast<unsigned>(pl.p.nk * pl.p.nr);
  cudaError_t e = cudaMemsetAsync(out->work, 0, sizeof(out->work), a.stream);
  if (e != cudaSuccess) return cuda_status(e);
  const lq_status st = launch_plan(a, pl, epi::kArgmax);
  if (st == LQ_OK) count_route(0);
  return st;
}

}  // namespace lq
