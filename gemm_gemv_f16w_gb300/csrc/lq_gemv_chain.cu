// Decode engine: a chain of M = 1 GEMVs of one weight format in a single
// persistent launch (lq_gemv_chain).
//
// A decode step runs many GEMVs back to back, each reading the output of an
// earlier one (q/k/v and o projections, gate/up and down, the LM head). As
// separate launches, every GEMV pays its launch, the release of the
// dependent kernel after the previous one drained, and a cold start of its
// weight stream. Here one CTA per SM walks the whole list (a launch of
// independent problems starts early after the previous kernel on the
// stream, its weights streaming at once and its A read once that kernel has
// completed; with the in-kernel waits below it is a cooperative launch, so
// that all CTAs are resident together):
//
//  * the producer warp streams every problem's weight rows through one ring
//    of shared-memory slots, running ahead into later problems as soon as
//    slots free up (weights never depend on anything);
//  * three activation warps bring each problem's A into one of two areas in
//    the layout the slices read, after the previous problem is complete on
//    every CTA when the problem says it reads that output ("after"): a
//    device-wide counter of finished (CTA, problem) pairs, polled with
//    acquire loads, with a time limit;
//  * sixteen consumer warps (K-groups x row-groups, the slices of the
//    streaming GEMV) compute each problem's rows; each stage's finisher
//    writes its C rows, and the last finisher of a problem on the CTA adds
//    one to the counter (release).
//
// Every wait is bounded. On a timeout the CTA records LQ_ERR_DEVICE_TIMEOUT,
// raises a device-wide abort flag that every other wait also checks, drains
// its own copies and returns.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "lq_device.cuh"
#include "lq_gemv_slices.cuh"
#include "lq_internal.h"
#include "lq_q4i.cuh"

namespace lq {
namespace {

using namespace gemv;

__device__ unsigned g_chain_err;
// Completion counter and abort flag, one pair per call in flight.
constexpr int kSyncSlots = 64;
__device__ unsigned g_chain_sync[kSyncSlots][2];

constexpr int kChainMax = 64;                 // problems per call
constexpr int kCW = 16;                       // consumer warps
constexpr int kProducerWarp = kCW;
constexpr int kAWarp = kCW + 1;               // first of the activation warps
constexpr int kAWarps = 3;
constexpr int kChainThreads = (kCW + 1 + kAWarps) * 32;
constexpr int kChainRows = 8;                 // rows per stage (at most)
constexpr int kChainMaxStages = 32;
// Ring slots each row-group cycles through: the rows of its later slots are
// in flight while it computes the current one. Independent problems gain
// from two (the next problem's rows stream in while this one's are
// computed: Q8_0 2048x2048 1.87 against 2.28 us); a chain whose problems wait
// for each other does better with one slot of more rows, fewer stages per
// problem (Q8_0 4096x4096: 8.3 against 9.2 us).
constexpr int kSlotsIndependent = 2;
constexpr int kSlotsDependent = 1;

struct ChainProblem {
  const float* A;
  const uint8_t* W;
  float* C;
  int N, K;
  int row_bytes;
  int after;
};

struct ChainParams {
  ChainProblem pr[kChainMax];
  int count;
  int nk, nr;             // consumer warp grid (from the largest K)
  int rows_per_stage;
  int stages;             // ring depth, a multiple of nr
  unsigned slot_bytes;    // ring slot: rows_per_stage x the largest row
  int a_slots;            // bytes of one of the two A areas the slices read
  int a_stage;            // bytes of the A staging area (quantised formats), else 0
  unsigned* sync;         // [0] finished (CTA, problem) pairs, [1] abort
  int publish;            // some problem waits for an earlier one
  unsigned long long wait_ns;
  unsigned wait_iters;
  int a_perm;             // Q4_0 with interleaved nibbles: A reordered per block
  int red_bytes;          // the K-groups' partials: [2 phases][stages][kChainRows][nk] floats
};

struct ChainHeader {
  uint64_t full[kChainMaxStages];
  uint64_t empty[kChainMaxStages];
  uint64_t red_full[kChainMaxStages];
  uint64_t a_landed;               // A_j in the staging area (quantised formats)
  uint64_t a_full[2], a_empty[2];  // A_j ready for the slices / every consumer warp read it
  volatile int a_go;               // the lead activation thread's outcome for the problem
  unsigned fin[kChainMax];         // finished stages of each problem on this CTA
  int row0[kChainMax], nrows[kChainMax], nstage[kChainMax];  // each problem's rows and stages here
  volatile int abort;
};
constexpr int kChainHeaderBytes = (static_cast<int>(sizeof(ChainHeader)) + 127) / 128 * 128;

__device__ __forceinline__ void record_error(unsigned code) { atomicCAS(&g_chain_err, 0u, code); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Gives up the whole launch: this CTA's waits see hd.abort, the other CTAs'
// activation warps see sync[1].
__device__ __forceinline__ void abort_all(ChainHeader& hd, const ChainParams& p) {
  record_error(kDevErrTimeout);
  hd.abort = 1;
  atomicExch(p.sync + 1, 1u);
}

// The CTA's own flag: cheap, checked after every wait. The device-wide flag
// is read only by the activation warp's dependency poll, which copies it
// into the CTA's flag; everything else is bounded by its own wait limit.
__device__ __forceinline__ bool aborted(const ChainHeader& hd) { return hd.abort != 0; }
__device__ __forceinline__ bool aborted_anywhere(ChainHeader& hd, const ChainParams& p) {
  if (*reinterpret_cast<volatile unsigned*>(p.sync + 1) != 0) hd.abort = 1;
  return hd.abort != 0;
}

// Rows of problem j owned by this CTA.
__device__ __forceinline__ void cta_rows(const ChainProblem& q, int& r0, int& nrows) {
  const int G = gridDim.x;
  r0 = static_cast<int>((static_cast<long long>(blockIdx.x) * q.N) / G);
  const int r1 = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * q.N) / G);
  nrows = r1 - r0;
}

template <int FMT>
__global__ void __launch_bounds__(kChainThreads, 1) gemv_chain_kernel(const __grid_constant__ ChainParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  ChainHeader& hd = *reinterpret_cast<ChainHeader*>(smem);
  uint8_t* slots_a = smem + kChainHeaderBytes;          // 2 x a_slots: A as the slices read it
  uint8_t* stage_a = slots_a + 2 * p.a_slots;           // A as copied (quantised formats)
  float* red = reinterpret_cast<float*>(stage_a + p.a_stage);
  uint8_t* ring = stage_a + p.a_stage + p.red_bytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int RS = p.rows_per_stage, S = p.stages, nk = p.nk, nr = p.nr, active = nk * nr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&hd.full[s], 1);
      mbar_init(&hd.empty[s], nk);
      mbar_init(&hd.red_full[s], nk);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&hd.a_full[b], 1);
      mbar_init(&hd.a_empty[b], active);
    }
    mbar_init(&hd.a_landed, 1);
    for (int i = 0; i < kChainMax; ++i) hd.fin[i] = 0;
    hd.abort = 0;
    fence_barrier_init();
  }
  // this CTA's share of every problem, worked out once (the divisions would
  // otherwise cost each consumer warp more than a row's dot per problem)
  for (int j = threadIdx.x; j < p.count; j += blockDim.x) {
    int r0, n;
    cta_rows(p.pr[j], r0, n);
    hd.row0[j] = r0;
    hd.nrows[j] = n;
    hd.nstage[j] = (n + RS - 1) / RS;
  }
  __syncthreads();
  // the next kernel on the stream may start streaming its weights as this
  // one's CTAs leave; A is read only once the previous kernel has completed
  // (below)
  pdl_launch_dependents();

  if (warp == kProducerWarp) {
    // ---------------- weight stream ----------------
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int g = 0, s = 0, lap = 0;  // global stage, its slot and ring lap
    bool ok = true;
    for (int j = 0; j < p.count && ok; ++j) {
      const ChainProblem& q = p.pr[j];
      const int r0 = hd.row0[j], nrows = hd.nrows[j], nst = hd.nstage[j];
      for (int st = 0; st < nst; ++st) {
        if (lap > 0 && (!mbar_wait(&hd.empty[s], static_cast<uint32_t>(lap - 1) & 1, p.wait_ns,
                                   p.wait_iters) ||
                        aborted(hd))) {
          ok = false;
          break;
        }
        const uint32_t bytes = static_cast<uint32_t>(min(RS, nrows - st * RS)) * q.row_bytes;
        if (!LQ_IN_BOUNDS(r0 + st * RS + min(RS, nrows - st * RS) <= q.N)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&hd.full[s], bytes);
        bulk_g2s(ring + static_cast<size_t>(s) * p.slot_bytes,
                 q.W + (static_cast<long long>(r0) + static_cast<long long>(st) * RS) * q.row_bytes, bytes,
                 &hd.full[s], pol);
        ++g;
        if (++s == S) {
          s = 0;
          ++lap;
        }
      }
    }
    if (!ok) abort_all(hd, p);
    for (int d = max(0, g - S); d < g; ++d)
      mbar_wait(&hd.full[d % S], static_cast<uint32_t>(d / S) & 1, kDrainWaitNs);
    return;
  }

  if (warp >= kAWarp) {
    // ---------------- activations ----------------
    // A_j goes to slot area j % 2 in the layout the slices read (f16: as
    // is, by the bulk copy itself; quantised: staged, then moved into the
    // block slots by this warp), once every consumer warp has read problem
    // j - 2's and, for a dependent problem, every CTA has finished j - 1.
    const unsigned G = gridDim.x;
    const bool lead = warp == kAWarp && lane == 0;
    const int at = (warp - kAWarp) * 32 + lane;  // 0 .. 32 * kAWarps - 1
    int issued = 0, landed = 0;
    bool ok = true;
    // every A (and, after it, every C) only once the previous kernel on the
    // stream has completed (at once in a cooperative launch, which never
    // starts early); the weight stream above does not wait
    if (lead) pdl_wait();
    for (int j = 0; j < p.count; ++j) {
      const ChainProblem& q = p.pr[j];
      const int b = j & 1;
      // The lead thread waits; the activation warps follow its outcome,
      // passed through shared memory at a named barrier (they stay in step).
      const uint32_t nthr = 32u * kAWarps;
      if (lead) {
        bool w = true;
        if (j >= 2)
          w = mbar_wait(&hd.a_empty[b], static_cast<uint32_t>((j >> 1) - 1) & 1, p.wait_ns, p.wait_iters) &&
              !aborted(hd);
        if (w && j > 0 && q.after) {
          // every CTA has finished problems 0 .. j-1
          const unsigned target = G * static_cast<unsigned>(j);
          const long long t0 = clock64(), limit = static_cast<long long>(p.wait_ns) * 4;
          unsigned it = 0;
          while (ld_acquire(p.sync) < target) {
            if (aborted_anywhere(hd, p) || ++it >= p.wait_iters || clock64() - t0 > limit) {
              w = false;
              break;
            }
            __nanosleep(64);
          }
          // the bulk copy below reads what other CTAs wrote with ordinary stores
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        const uint32_t bytes = static_cast<uint32_t>(q.K) * 4u;
        if (w) {
          if (FMT == LQ_FMT_F16) {
            mbar_arrive_expect_tx(&hd.a_full[b], bytes);
            bulk_g2s(slots_a + b * p.a_slots, q.A, bytes, &hd.a_full[b], policy_evict_last());
          } else {
            mbar_arrive_expect_tx(&hd.a_landed, bytes);
            bulk_g2s(stage_a, q.A, bytes, &hd.a_landed, policy_evict_last());
          }
          ++issued;
          if (FMT != LQ_FMT_F16) {
            w = mbar_wait(&hd.a_landed, static_cast<uint32_t>(j) & 1, p.wait_ns, p.wait_iters) && !aborted(hd);
            if (w) ++landed;
          }
        }
        hd.a_go = w ? 1 : 0;
      }
      named_barrier(2, nthr);
      if (!hd.a_go) {
        ok = false;
        break;
      }
      if (FMT != LQ_FMT_F16) {
        // the copy has landed (the lead saw it): observe it here too
        if (!lead) mbar_wait(&hd.a_landed, static_cast<uint32_t>(j) & 1, kDrainWaitNs);
        // staging -> block slots (see a_slot_q): 512 contiguous bytes per
        // warp step, the four blocks they hold land in different bank groups
        const uint32_t sg = smem_u32(stage_a), sa = smem_u32(slots_a + b * p.a_slots);
        for (int c = at; c < q.K / 4; c += static_cast<int>(nthr)) {
          const uint4 v = lds128(sg + 16u * c);
          const uint32_t blk = sa + static_cast<uint32_t>(a_slot_q(c >> 3)) * kASlotBytes;
          if (p.a_perm)
            q4i::store_chunk(blk, c & 7, v);
          else
            sts128(blk + 16u * (c & 7), v);
        }
        named_barrier(2, nthr);
        if (lead) mbar_arrive(&hd.a_full[b]);
      }
    }
    if (!ok && lead) abort_all(hd, p);
    if (lead) {
      if (FMT == LQ_FMT_F16) {
        for (int d = max(0, issued - 2); d < issued; ++d)
          mbar_wait(&hd.a_full[d & 1], static_cast<uint32_t>(d >> 1) & 1, kDrainWaitNs);
      } else if (issued > landed) {
        mbar_wait(&hd.a_landed, static_cast<uint32_t>(issued - 1) & 1, kDrainWaitNs);
      }
    }
    return;
  }

  if (warp >= active) return;

  // ---------------- consumers ----------------
  const int kg = warp % nk, rg = warp / nk;
  // this row-group's global stages are rg, rg + nr, rg + 2 nr, ... through all
  // the problems; slot, ring phase and finisher advance with them, nr stages
  // at a time: slot g mod S, phase (g / S) mod 2, finisher (g / nr) mod nk
  int gw = rg;     // the warp's next global stage
  int s = rg;      // its slot (rg < nr <= S)
  uint32_t ph = 0;
  int kf = 0;
  int g0 = 0;      // first global stage of problem j on this CTA
  for (int j = 0; j < p.count; ++j) {
    const ChainProblem& q = p.pr[j];
    const int r0 = hd.row0[j], nrows = hd.nrows[j], nst = hd.nstage[j];
    const int b = j & 1;
    if (!mbar_wait(&hd.a_full[b], static_cast<uint32_t>(j >> 1) & 1, p.wait_ns, p.wait_iters) ||
        aborted(hd)) {
      abort_all(hd, p);
      return;
    }
    typename SliceOf<FMT, 1>::T sl;
    sl.init(smem_u32(slots_a + b * p.a_slots), kg, nk, lane, q.K);
    __syncwarp();
    if (lane == 0) mbar_arrive(&hd.a_empty[b]);  // this warp has read A_j

    for (int st = gw - g0; st < nst; st += nr) {
      if (!mbar_wait(&hd.full[s], ph, p.wait_ns, p.wait_iters) || aborted(hd)) {
        abort_all(hd, p);
        return;
      }
      const int rows = min(RS, nrows - st * RS);
      const uint32_t base = smem_u32(ring + static_cast<size_t>(s) * p.slot_bytes);
      float acc[kChainRows];
#pragma unroll
      for (int r = 0; r < kChainRows; ++r) acc[r] = 0.f;
      if (sl.ok[0]) {
        if constexpr (FMT == LQ_FMT_F16) {
          // f16 rows in pairs under one guard (their loads overlap); past
          // the last row the pair's second half repeats the first, into a
          // partial nobody reads. Measured on 10 independent f16
          // 4096x4096 GEMVs: 5.85 against 6.23 us a GEMV; the quantised
          // dots, whose dequantisation is the longer part, ran no faster
          // (Q4_0) or slower (Q8_0 3.90 against 3.71 us) paired.
#pragma unroll
          for (int r = 0; r < kChainRows; r += 2)
            if (r < rows) {
              const uint32_t row0 = base + static_cast<uint32_t>(r) * q.row_bytes;
              const uint32_t row1 = r + 1 < rows ? row0 + q.row_bytes : row0;
              acc[r] += sl.dot(row0, 0);
              acc[r + 1] += sl.dot(row1, 0);
            }
        } else {
#pragma unroll
          for (int r = 0; r < kChainRows; ++r)
            if (r < rows) acc[r] += sl.dot(base + static_cast<uint32_t>(r) * q.row_bytes, 0);
        }
      }
      int r;
      const float v = transpose_reduce8(acc, lane, r);
      // partials of this use of the slot: double-buffered by the ring phase,
      // so the slot itself is handed back as soon as its rows are read (the
      // refill overlaps the reduction); the partials of this phase are not
      // written again before this stage's finisher has moved on to its next
      // stage, whose slot release the second refill waits for
      float* red_s = red + (static_cast<size_t>(ph) * S + s) * kChainRows * nk;
      if ((lane & 3) == 0) red_s[r * nk + kg] = v;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&hd.red_full[s]);
        mbar_arrive(&hd.empty[s]);  // this warp has read the slot
      }
      if (kg == kf) {
        // finisher: the K-groups' partials in a fixed order, then C
        if (!mbar_wait(&hd.red_full[s], ph, p.wait_ns, p.wait_iters) || aborted(hd)) {
          abort_all(hd, p);
          return;
        }
        float sum = 0.f;
        if (lane < rows)
          for (int k = 0; k < nk; ++k) sum += red_s[lane * nk + k];
        if (lane < rows && LQ_IN_BOUNDS(r0 + st * RS + lane < q.N)) q.C[r0 + st * RS + lane] = sum;
        if (p.publish) {
          __syncwarp();
          if (lane == 0) {
            __threadfence();  // the warp's C stores, before the count below
            if (atomicAdd(&hd.fin[j], 1u) == static_cast<unsigned>(nst - 1))
              add_release(p.sync, 1u);  // last stage of problem j on this CTA
          }
          __syncwarp();
        }
      }
      s += nr;
      if (s >= S) {
        s -= S;
        ph ^= 1u;
      }
      if (++kf == nk) kf = 0;
      gw += nr;
    }
    if (p.publish && nst == 0 && warp == 0 && lane == 0) add_release(p.sync, 1u);  // no rows here
    g0 += nst;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
std::mutex g_sync_mu;
unsigned* g_sync_ptr[kMaxDevices];
std::atomic<unsigned> g_sync_next{0};

lq_status sync_slot(unsigned** out) {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_sync_mu);
    if (!g_sync_ptr[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_chain_sync) != cudaSuccess || !ptr) return LQ_ERR_CUDA;
      g_sync_ptr[dev] = static_cast<unsigned*>(ptr);
    }
  }
  *out = g_sync_ptr[dev] + 2 * (g_sync_next.fetch_add(1) % kSyncSlots);
  return LQ_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// A launch whose problems wait for earlier ones inside it (the in-kernel
// device-wide wait) is cooperative: every CTA resident at once. Otherwise
// the CTAs never wait for each other and the launch may start early after
// the previous kernel on the stream (programmatic dependent launch).
template <int FMT>
lq_status launch_chain_t(const ChainParams& p, size_t smem, cudaStream_t stream) {
  auto kern = gemv_chain_kernel<FMT>;
  static int configured[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return LQ_ERR_CUDA;
  if (configured[dev] < static_cast<int>(smem)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_status(e);
    configured[dev] = static_cast<int>(smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(device_info().sm_count));
  cfg.blockDim = dim3(kChainThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (p.publish) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_status(e);
}

}  // namespace

unsigned read_clear_chain_error() {
  unsigned v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_chain_err, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_chain_err, &z, sizeof(z));
  return v;
}

// The launch plan of one chain launch (no launch): LQ_ERR_UNSUPPORTED when
// the problems do not fit its fast path.
lq_status plan_chain(int fmt, const lq_gemv_problem* problems, int count, ChainParams& p, size_t& smem) {
  if (count < 1 || count > kChainMax) return LQ_ERR_UNSUPPORTED;
  p = ChainParams{};
  if (fmt == LQ_FMT_Q4_0I) {  // the Q4_0 kernel with A reordered per block (lq_q4i.cuh)
    fmt = LQ_FMT_Q4_0;
    p.a_perm = 1;
  }
  int kmax = 0, rb_max = 0;
  for (int j = 0; j < count; ++j) {
    const lq_gemv_problem& u = problems[j];
    const int64_t K = u.K, N = u.N;
    // the streaming fast path's shapes: 16-byte rows and A, the slices' K
    const bool shape_ok = K >= 1 && K <= 16384 && N >= 0 && N < (1LL << 30) &&
                          (fmt == LQ_FMT_F16 ? (K % 8 == 0) : (K % 256 == 0));
    if (!shape_ok || !aligned16(u.A) || !aligned16(u.W)) return LQ_ERR_UNSUPPORTED;
    ChainProblem& q = p.pr[j];
    q.A = u.A;
    q.W = static_cast<const uint8_t*>(u.W);
    q.C = u.C;
    q.N = static_cast<int>(N);
    q.K = static_cast<int>(K);
    q.row_bytes = static_cast<int>(row_bytes(fmt, K));
    q.after = u.after ? 1 : 0;
    kmax = std::max(kmax, q.K);
    rb_max = std::max(rb_max, q.row_bytes);
  }
  p.count = count;
  p.publish = 0;
  for (int j = 1; j < count; ++j) p.publish |= p.pr[j].after;
  // warp grid for the largest K: f16 chunks of 256 values, quantised formats
  // two K-groups (block parities) per 64-block segment, one chunk per warp
  if (fmt == LQ_FMT_F16) {
    const int nch = (kmax + 255) / 256;
    if (nch > kCW) return LQ_ERR_UNSUPPORTED;
    int nk = 1;
    while (nk < nch) nk *= 2;
    p.nk = nk;
  } else {
    const int nseg = (kmax / 32 + 63) / 64;
    if (2 * nseg > kCW) return LQ_ERR_UNSUPPORTED;
    p.nk = 2 * nseg;
  }
  p.nr = kCW / p.nk;
  const DeviceInfo& di = device_info();
  // two slot areas of A as the slices read it (f16: in order; quantised: the
  // block slots) and, for the quantised formats, one staging area
  const int a_linear = (kmax * 4 + 127) / 128 * 128;
  p.a_slots = fmt == LQ_FMT_F16 ? a_linear : ((kmax / 32 + 63) / 64) * 64 * kASlotBytes;
  p.a_stage = fmt == LQ_FMT_F16 ? 0 : a_linear;
  const long long fixed = kChainHeaderBytes + 2LL * p.a_slots + p.a_stage;
  const long long budget = std::min(di.max_smem_optin, 227 * 1024) - fixed - 128;
  // a ring slot costs its rows plus two phases of the K-groups' partials;
  // rows per stage: the most (up to kChainRows) that still give every
  // row-group its slots, and the ring at least two
  const long long red_slot = 2LL * kChainRows * p.nk * static_cast<long long>(sizeof(float));
  const int slots_per_group = p.publish ? kSlotsDependent : kSlotsIndependent;
  // independent problems keep at least three slots in the ring: with a single
  // row-group (f16 beyond K = 2048) two slots per group meant two stages of
  // eight rows; three of seven measured 5.10 against 5.55 us a 4096 x 4096
  // f16 GEMV (the quantised plans, four row-groups, are unchanged)
  const int min_slots = p.publish ? 2 : 3;
  const long long per_slot = budget / std::max(min_slots, slots_per_group * p.nr);
  p.rows_per_stage = static_cast<int>(std::min<long long>(kChainRows, (per_slot - red_slot) / rb_max));
  if (p.rows_per_stage < 1)
    p.rows_per_stage = static_cast<int>(std::min<long long>(kChainRows, (budget / 2 - red_slot) / rb_max));
  if (p.rows_per_stage < 1) return LQ_ERR_UNSUPPORTED;
  p.slot_bytes = static_cast<unsigned>(p.rows_per_stage * rb_max);
  int stages = static_cast<int>(std::min<long long>(kChainMaxStages, budget / (p.slot_bytes + red_slot)));
  // every ring slot serves one row-group: S a multiple of nr
  while (p.nr > 1 && stages - stages % p.nr < 2) p.nr /= 2;
  stages -= stages % p.nr;
  if (stages < 2) return LQ_ERR_UNSUPPORTED;
  p.stages = stages;
  p.red_bytes = static_cast<int>((stages * red_slot + 127) / 128 * 128);
  p.wait_ns = wait_limit_ns();
  p.wait_iters = wait_limit_iters();
  smem = static_cast<size_t>(fixed) + p.red_bytes + static_cast<size_t>(stages) * p.slot_bytes;
  return LQ_OK;
}

lq_status launch_planned_chain(int fmt, ChainParams& p, size_t smem, cudaStream_t stream) {
  if (fmt == LQ_FMT_Q4_0I) fmt = LQ_FMT_Q4_0;
  unsigned* sync = nullptr;
  lq_status st = sync_slot(&sync);
  if (st != LQ_OK) return st;
  p.sync = sync;
  if (p.publish) {  // the completion count and the abort word, read only by the in-kernel waits
    const cudaError_t e = cudaMemsetAsync(sync, 0, 2 * sizeof(unsigned), stream);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (fmt == LQ_FMT_F16) st = launch_chain_t<LQ_FMT_F16>(p, smem, stream);
  else if (fmt == LQ_FMT_Q8_0) st = launch_chain_t<LQ_FMT_Q8_0>(p, smem, stream);
  else st = launch_chain_t<LQ_FMT_Q4_0>(p, smem, stream);
  if (st == LQ_OK) count_route(4);
  return st;
}

}  // namespace lq

namespace lq {
namespace {
std::atomic<int> g_chain_waits{0};  // debug: dependent problems wait inside one launch
}

void set_chain_waits(bool on) { g_chain_waits.store(on ? 1 : 0); }

// A chain whose problems wait for earlier ones runs, by default, as one
// launch per run of independent problems, in order on the stream: a run of
// several problems is a chain launch, a single problem the streaming GEMV
// (programmatic dependent launch: its weights stream in while the previous
// run finishes, its A is read after). Measured on Q8_0 4096x4096 GEMVs each
// reading the previous one's output, that beats the in-kernel device-wide
// wait (kept behind lq_debug_chain_waits): 6.1 against 8.0 us a GEMV.
// Every run is planned before anything is launched, so a problem outside
// the fast path still refuses the whole call.
lq_status launch_gemv_chain(int fmt, const lq_gemv_problem* problems, int count, cudaStream_t stream) {
  if (count < 1 || count > kChainMax) return LQ_ERR_UNSUPPORTED;
  bool dependent = false;
  for (int j = 1; j < count; ++j) dependent |= problems[j].after != 0;
  if (!dependent || g_chain_waits.load()) {
    ChainParams p;
    size_t smem = 0;
    lq_status st = plan_chain(fmt, problems, count, p, smem);
    if (st != LQ_OK) return st;
    return launch_planned_chain(fmt, p, smem, stream);
  }
  lq_gemv_problem runs[kChainMax];
  for (int j = 0; j < count; ++j) {
    runs[j] = problems[j];
    runs[j].after = 0;
  }
  // plan every run first
  std::vector<ChainParams> plans(count);
  std::vector<size_t> smems(count);
  for (int s0 = 0; s0 < count;) {
    int e = s0 + 1;
    while (e < count && !problems[e].after) ++e;
    const lq_status st = plan_chain(fmt, runs + s0, e - s0, plans[s0], smems[s0]);
    if (st != LQ_OK) return st;
    s0 = e;
  }
  for (int s0 = 0; s0 < count;) {
    int e = s0 + 1;
    while (e < count && !problems[e].after) ++e;
    lq_status st = LQ_OK;
    if (e - s0 == 1) {
      const lq_gemv_problem& q = runs[s0];
      if (q.N > 0) {
        MatmulArgs a{q.A, q.W, q.C, 1, q.N, q.K, fmt == LQ_FMT_Q4_0I ? LQ_FMT_Q4_0 : fmt, stream};
        a.a_perm = fmt == LQ_FMT_Q4_0I;
        st = launch_gemv(a);
      }
    } else {
      st = launch_planned_chain(fmt, plans[s0], smems[s0], stream);
    }
    if (st != LQ_OK) return st;
    s0 = e;
  }
  return LQ_OK;
}

}  // namespace lq
