// lq_topk_f32 / lq_gemv_topk: the k best entries of a vector (k <= 64),
// best first, in the order of topk_better (lattice-inference 0.1.2,
// src/forward/metal_qwen35.rs): the larger value first, equal values by the
// lower index, NaN never chosen; missing entries are the pages' sentinel
// (-inf, index -1).
//
// The pages sort 1280-logit tiles (padded to 2048) per threadgroup
// (logits_topk_first_pass) and merge groups of top-k candidates sixteen at a
// time (logits_topk_merge_pass) until one group is left. Here each entry is
// the 64-bit ordered key of lq_argmax.cuh, so that one unsigned comparison
// ranks two candidates:
//
//  1. a grid of CTAs (one tile of the input each, as many CTAs as tiles up
//     to a cap) keeps a running top-64 of its tiles in shared memory: slots
//     0..63 hold the best keys so far, slots 64..2047 take the next 1984
//     inputs, and a partial bitonic sort (runs of 64 sorted in registers,
//     then rounds that keep the best half of each pair of runs) brings the
//     best 64 of the 2048 keys back to the front;
//     each CTA writes its best k keys to the work buffer;
//  2. merge passes, each CTA sorting up to 1984 / k groups of k candidates
//     into one group, until one group is left; the last pass writes the k
//     results.
//
// Inputs of up to 4 Mi entries take a radix selection instead (two
// launches): every CTA holds 4096 keys in registers (16384 beyond 1 Mi
// entries) and finds the k-th
// largest a byte at a time from the top (a histogram of the byte among the
// keys that share the bytes found so far, then the byte where the count from
// the top reaches the number of keys still wanted; once that byte's bucket
// holds exactly that number, all of it is in), gathers the keys at or above
// it and sorts those k with one warp; one CTA does the same over the CTAs'
// candidates. On the LM head (151936 logits, k = 50) the sorting passes
// took about 29 us.
#include <algorithm>

#include "lq_argmax.cuh"
#include "lq_device.cuh"
#include "lq_internal.h"

namespace lq {
namespace {

constexpr int kTopkThreads = 1024;              // two keys a thread
constexpr int kTopkLog = 11;
constexpr int kTopkTile = 1 << kTopkLog;        // keys sorted together (2048)
constexpr int kTopkMaxK = 64;                   // kept between tiles
constexpr int kTopkNew = kTopkTile - kTopkMaxK; // fresh keys per tile
constexpr int kTopkMaxCtas = 512;

// One compare-exchange step of a bitonic network on the warp's keys, thread
// holding positions p and p + 1 (p even): strides 2..32 pair lanes by
// shuffles, stride 1 is inside the thread. keep_max for the lower position
// of each pair is decided by the caller's direction.
__device__ __forceinline__ void cx_step(unsigned long long& e0, unsigned long long& e1, int p, int stride,
                                        bool desc) {
  if (stride == 1) {
    if (desc ? e0 < e1 : e0 > e1) {
      const unsigned long long x = e0;
      e0 = e1;
      e1 = x;
    }
    return;
  }
  const unsigned long long q0 = __shfl_xor_sync(0xffffffffu, e0, stride >> 1);
  const unsigned long long q1 = __shfl_xor_sync(0xffffffffu, e1, stride >> 1);
  const bool keep_max = ((p & stride) == 0) == desc;  // both positions share bit log2(stride)
  e0 = keep_max ? (e0 > q0 ? e0 : q0) : (e0 < q0 ? e0 : q0);
  e1 = keep_max ? (e1 > q1 ? e1 : q1) : (e1 < q1 ? e1 : q1);
}

// The best 64 of s[0 .. 2048), sorted descending into s[0 .. 64) (the rest
// of s is left undefined). Warp w holds the run of positions 64w .. 64w+63,
// two keys a lane. (1) Each run is sorted by the bitonic network on the
// global positions, which leaves even runs descending and odd runs
// ascending. (2) Five rounds halve the runs: warp w, a multiple of 2^(r+1),
// takes the elementwise maximum of its run and the run of warp w + 2^r
// (read through shared memory): a descending run against an ascending one,
// this is the half-cleaner of their bitonic concatenation and keeps the best
// 64 as a bitonic sequence, which six steps sort in the direction the next
// round needs (descending when w / 2^(r+1) is even).
__device__ void top64_desc(unsigned long long* s) {
  const int t = threadIdx.x, w = t >> 5, p0 = 2 * t;
  unsigned long long e0 = s[p0], e1 = s[p0 + 1];
  for (int ls = 1; ls <= 6; ++ls)
    for (int lst = ls - 1; lst >= 0; --lst) {
      const int stride = 1 << lst;
      cx_step(e0, e1, p0, stride, (((p0 & ~stride) & (1 << ls)) == 0));
    }
  for (int r = 0; r < 5; ++r) {
    s[p0] = e0;  // this thread's own positions
    s[p0 + 1] = e1;
    __syncthreads();
    if ((w & ((2 << r) - 1)) == 0) {
      const int q = p0 + (64 << r);  // the same lane of warp w + 2^r
      const unsigned long long b0 = s[q], b1 = s[q + 1];
      e0 = e0 > b0 ? e0 : b0;
      e1 = e1 > b1 ? e1 : b1;
      const bool desc = ((w >> (r + 1)) & 1) == 0;
      for (int lst = 5; lst >= 0; --lst) cx_step(e0, e1, p0 & 63, 1 << lst, desc);
    }
    __syncthreads();
  }
  if (w == 0) {
    s[p0] = e0;
    s[p0 + 1] = e1;
  }
  __syncthreads();
}

// Leaves in s[0 .. kTopkMaxK) the best keys of inputs key(0 .. count),
// sorted, taking tiles t = first, first + step, ... of kTopkNew inputs.
template <typename KeyOf>
__device__ void running_topk(unsigned long long* s, long long count, long long first, long long step,
                             KeyOf key) {
  for (int j = threadIdx.x; j < kTopkMaxK; j += kTopkThreads) s[j] = 0ull;
  for (long long t = first; t * kTopkNew < count; t += step) {
    const long long base = t * kTopkNew;
    for (int j = threadIdx.x; j < kTopkNew; j += kTopkThreads)
      s[kTopkMaxK + j] = base + j < count ? key(base + j) : 0ull;
    __syncthreads();
    top64_desc(s);
  }
}

__global__ void __launch_bounds__(kTopkThreads) topk_first_kernel(const float* __restrict__ x, long long n,
                                                                  int k, unsigned long long* out) {
  __shared__ unsigned long long s[kTopkTile];
  pdl_wait();  // x may come from the previous kernel on the stream
  running_topk(s, n, blockIdx.x, gridDim.x,
               [&](long long j) { return amax::make_key(x[j], static_cast<unsigned>(j)); });
  pdl_launch_dependents();
  for (int j = threadIdx.x; j < k; j += kTopkThreads) out[static_cast<long long>(blockIdx.x) * k + j] = s[j];
}

// The result entry j from a key (0: the pages' sentinel, -inf and -1).
__device__ __forceinline__ void write_result(unsigned long long key, int j, float* values, int32_t* indices) {
  if (key == 0ull) {
    values[j] = -__int_as_float(0x7f800000);
    indices[j] = -1;
  } else {
    const unsigned hi = static_cast<unsigned>(key >> 32), lo = static_cast<unsigned>(key);
    values[j] = __uint_as_float((hi & 0x80000000u) ? (hi & 0x7FFFFFFFu) : ~hi);
    indices[j] = static_cast<int32_t>(0xFFFFFFFFu - lo);
  }
}

// One merge pass: CTA b sorts groups [b * fan_in, (b + 1) * fan_in) of k
// candidates (fan_in * k <= kTopkNew) into one group; with one CTA left it
// writes the final values and indices.
__global__ void __launch_bounds__(kTopkThreads) topk_merge_kernel(const unsigned long long* __restrict__ in,
                                                                  int groups, int k, int fan_in,
                                                                  unsigned long long* out, float* values,
                                                                  int32_t* indices) {
  __shared__ unsigned long long s[kTopkTile];
  pdl_wait();  // the candidates of the previous pass
  const long long g0 = static_cast<long long>(blockIdx.x) * fan_in;
  const long long count = (min(static_cast<long long>(groups), g0 + fan_in) - g0) * k;
  const unsigned long long* src = in + g0 * k;
  running_topk(s, count, 0, 1, [&](long long j) { return src[j]; });
  pdl_launch_dependents();
  if (gridDim.x > 1) {
    for (int j = threadIdx.x; j < k; j += kTopkThreads) out[static_cast<long long>(blockIdx.x) * k + j] = s[j];
    return;
  }
  for (int j = threadIdx.x; j < k; j += kTopkThreads) write_result(s[j], j, values, indices);  // 0: fewer than k
}

// ---------------------------------------------------------------------------
// Radix selection (n <= kRadixMaxN).
// ---------------------------------------------------------------------------
// A pass costs each thread a ballot, a match and a compare per key it holds:
// the first launch takes 4 keys a thread (16 for inputs beyond 1 Mi), the
// final one as few as hold the candidates.
constexpr int kRadixThreads = 1024;
constexpr int kRadixMaxKpt = 16;                                // keys a thread, at most
constexpr int kRadixMaxCand = kRadixThreads * kRadixMaxKpt;     // candidates the final CTA takes
constexpr int kRadixMaxCtas = kRadixMaxCand / kTopkMaxK;        // 256
constexpr long long kRadixMaxN = static_cast<long long>(kRadixMaxCtas) * kRadixThreads * kRadixMaxKpt;

constexpr int kRadixGather = 128;  // candidates ranked directly once this few remain

struct RadixShared {
  unsigned hist[kRadixThreads / 32][256];  // one histogram a warp
  unsigned tot[256];
  unsigned long long gath[kRadixGather];   // the keys at or above the final prefix
  unsigned rank[kRadixGather];
  unsigned long long sel[kTopkMaxK];
  unsigned long long prefix;               // the bytes found so far (lower bytes zero)
  int remaining, done, count, total;
};

// The k largest of the CTA's keys (0 = no key), sorted descending, into
// s.sel[0 .. k); entries past the valid keys are 0. Bytes are found from the
// top until the keys at or above the prefix number at most kRadixGather
// (always true once the last byte is found: keys are unique); those are
// gathered and each one's rank among them decides its place.
template <int KPT>
__device__ void radix_topk_block(const unsigned long long (&keys)[KPT], int k, RadixShared& s) {
  const int t = threadIdx.x, w = t >> 5, lane = t & 31;
  int mine = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) mine += keys[i] != 0ull;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, off);
  if (t == 0) {
    s.total = 0;
    s.count = 0;
    s.prefix = 0ull;
    s.remaining = k;
    s.done = 0;
  }
  if (t < kTopkMaxK) s.sel[t] = 0ull;
  if (t < kRadixGather) s.rank[t] = 0u;
  __syncthreads();
  if (lane == 0) atomicAdd(&s.total, mine);
  __syncthreads();
  unsigned long long T = 1ull;  // keys >= T are gathered (every valid key when few)
  if (s.total > kRadixGather) {
    for (int d = 7; d >= 0; --d) {
      for (int b = lane; b < 256; b += 32) s.hist[w][b] = 0u;
      __syncwarp();
      const unsigned long long pre = s.prefix;
      const int sh = 8 * d;
#pragma unroll
      for (int i = 0; i < KPT; ++i) {
        const unsigned long long x = keys[i];
        const bool in = x != 0ull && (d == 7 || (x >> (sh + 8)) == (pre >> (sh + 8)));
        const unsigned act = __ballot_sync(0xffffffffu, in);
        if (in) {
          const unsigned dig = static_cast<unsigned>(x >> sh) & 255u;
          const unsigned peers = __match_any_sync(act, dig);  // lanes with the same byte add once
          if (lane == __ffs(peers) - 1) atomicAdd(&s.hist[w][dig], static_cast<unsigned>(__popc(peers)));
        }
      }
      __syncthreads();
      if (t < 256) {
        unsigned v = 0;
#pragma unroll 8
        for (int ww = 0; ww < kRadixThreads / 32; ++ww) v += s.hist[ww][t];
        s.tot[t] = v;
      }
      __syncthreads();
      if (w == 0) {
        // lane l: bins 255 - 8l - j, j = 0..7 (from the top)
        unsigned c[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = s.tot[255 - 8 * lane - j];
          sum += c[j];
        }
        unsigned incl = sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += y;
        }
        const unsigned rem = static_cast<unsigned>(s.remaining);
        unsigned above = incl - sum;  // keys in the bins above this lane's
        if (above < rem && incl >= rem) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (above + c[j] >= rem) {
              const unsigned dig = static_cast<unsigned>(255 - 8 * lane - j);
              s.prefix = pre | (static_cast<unsigned long long>(dig) << sh);
              s.remaining = static_cast<int>(rem - above);
              // keys at or above the new prefix: those taken so far and the bucket
              s.done = static_cast<unsigned>(k) - (rem - above) + c[j] <= static_cast<unsigned>(kRadixGather);
              break;
            }
            above += c[j];
          }
        }
      }
      __syncthreads();
      if (s.done) break;
    }
    T = s.prefix;
  }
#pragma unroll
  for (int i = 0; i < KPT; ++i)
    if (keys[i] != 0ull && keys[i] >= T) {
      const int slot = atomicAdd(&s.count, 1);
      if (slot < kRadixGather) s.gath[slot] = keys[i];
    }
  __syncthreads();
  // rank of gathered key i: the gathered keys above it (thread t counts
  // over the j of one of eight ranges for key t % kRadixGather)
  const int cnt = min(s.count, kRadixGather);
  {
    const int i = t % kRadixGather, c0 = (t / kRadixGather) * (kRadixGather / 8);
    if (i < cnt) {
      const unsigned long long key = s.gath[i];
      unsigned r = 0;
      for (int j = c0; j < min(cnt, c0 + kRadixGather / 8); ++j) r += s.gath[j] > key;
      if (r) atomicAdd(&s.rank[i], r);
    }
  }
  __syncthreads();
  if (t < cnt && s.rank[t] < static_cast<unsigned>(k)) s.sel[s.rank[t]] = s.gath[t];
  __syncthreads();
}

// CTA b: keys of x[T b .. T (b + 1)) (T = 1024 KPT), its k best to
// out[b k ..]; a grid of one CTA writes the results itself.
template <int KPT>
__global__ void __launch_bounds__(kRadixThreads) radix_first_kernel(const float* __restrict__ x, long long n, int k,
                                                                    unsigned long long* out, float* values,
                                                                    int32_t* indices) {
  __shared__ RadixShared s;
  pdl_wait();  // x may come from the previous kernel on the stream
  unsigned long long keys[KPT];
  const long long base = static_cast<long long>(blockIdx.x) * (kRadixThreads * KPT) + threadIdx.x;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const long long j = base + static_cast<long long>(i) * kRadixThreads;
    keys[i] = j < n ? amax::make_key(x[j], static_cast<unsigned>(j)) : 0ull;
  }
  radix_topk_block(keys, k, s);
  pdl_launch_dependents();
  for (int j = threadIdx.x; j < k; j += kRadixThreads) {
    if (gridDim.x == 1)
      write_result(s.sel[j], j, values, indices);
    else
      out[static_cast<long long>(blockIdx.x) * k + j] = s.sel[j];
  }
}

// One CTA over the count = G k <= 1024 KPT candidates of radix_first_kernel.
template <int KPT>
__global__ void __launch_bounds__(kRadixThreads) radix_final_kernel(const unsigned long long* __restrict__ in,
                                                                    int count, int k, float* values,
                                                                    int32_t* indices) {
  __shared__ RadixShared s;
  pdl_wait();  // the candidates of the first launch
  unsigned long long keys[KPT];
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const int j = static_cast<int>(threadIdx.x) + i * kRadixThreads;
    keys[i] = j < count ? in[j] : 0ull;
  }
  radix_topk_block(keys, k, s);
  for (int j = threadIdx.x; j < k; j += kRadixThreads) write_result(s.sel[j], j, values, indices);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_topk(void (*kern)(KArgs...), unsigned grid, cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTopkThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = use_pdl() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace

// Work: two regions of topk_ctas(n) * k keys (the passes alternate).
int64_t topk_ctas(int64_t n) { return 2 * std::min<int64_t>(kTopkMaxCtas, (n + kTopkNew - 1) / kTopkNew); }

lq_status launch_topk_f32(const float* x, int64_t n, int k, float* values, int32_t* indices, void* work,
                          cudaStream_t stream) {
  if (n <= kRadixMaxN) {
    // radix selection: G CTAs of 1024 KPT keys, then one CTA over their G k
    // candidates (G <= 256, so G k <= 16384; the work buffer holds
    // topk_ctas(n) k >= G k keys)
    const bool small = n <= static_cast<long long>(kRadixMaxCtas) * kRadixThreads * 4;
    const long long tile = static_cast<long long>(kRadixThreads) * (small ? 4 : kRadixMaxKpt);
    const int G = static_cast<int>((n + tile - 1) / tile);
    auto* cand = static_cast<unsigned long long*>(work);
    cudaError_t e = small ? launch_pdl_topk(radix_first_kernel<4>, static_cast<unsigned>(G), stream, x,
                                            static_cast<long long>(n), k, cand, values, indices)
                          : launch_pdl_topk(radix_first_kernel<kRadixMaxKpt>, static_cast<unsigned>(G), stream,
                                            x, static_cast<long long>(n), k, cand, values, indices);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess && G > 1) {
      const int count = G * k, kpt = (count + kRadixThreads - 1) / kRadixThreads;
      const auto* c = static_cast<const unsigned long long*>(cand);
      if (kpt <= 1)
        e = launch_pdl_topk(radix_final_kernel<1>, 1u, stream, c, count, k, values, indices);
      else if (kpt <= 2)
        e = launch_pdl_topk(radix_final_kernel<2>, 1u, stream, c, count, k, values, indices);
      else if (kpt <= 4)
        e = launch_pdl_topk(radix_final_kernel<4>, 1u, stream, c, count, k, values, indices);
      else if (kpt <= 8)
        e = launch_pdl_topk(radix_final_kernel<8>, 1u, stream, c, count, k, values, indices);
      else
        e = launch_pdl_topk(radix_final_kernel<kRadixMaxKpt>, 1u, stream, c, count, k, values, indices);
      if (e == cudaSuccess) e = cudaGetLastError();
    }
    return cuda_status(e);
  }
  const int G = static_cast<int>(std::min<int64_t>(kTopkMaxCtas, (n + kTopkNew - 1) / kTopkNew));
  auto* a = static_cast<unsigned long long*>(work);
  auto* b = a + static_cast<size_t>(G) * k;
  cudaError_t e = launch_pdl_topk(topk_first_kernel, static_cast<unsigned>(G), stream, x,
                                  static_cast<long long>(n), k, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  const int fan_in = kTopkNew / k;
  int groups = G;
  while (e == cudaSuccess) {
    const int next = (groups + fan_in - 1) / fan_in;
    e = launch_pdl_topk(topk_merge_kernel, static_cast<unsigned>(next), stream,
                        static_cast<const unsigned long long*>(a), groups, k, fan_in, b, values, indices);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (next == 1) break;
    groups = next;
    std::swap(a, b);
  }
  return cuda_status(e);
}

}  // namespace lq
