/*
 * lq.h - weight-only mixed-precision matmul for GB300 (sm_103a).
 *
 *     C[M,N] (f32) = A[M,K] (f32) @ W[N,K]^T,   W in {f16, Q8_0, Q4_0}
 *
 * Operation and formats follow the docs.rs source pages of lattice-inference
 * (src/forward/metal_qwen35.rs: kernels gemv_decode_m1, gemv_q8_decode,
 * gemv_q4_decode, gemm_q8, gemm_q4, gemm_q4_tiled; host packers f32_to_f16,
 * quantize_row_q8_0; src/forward/metal_qwen35/inner/dispatch.rs: routers
 * dispatch_matmul_half, dispatch_gemm_q8, dispatch_gemm_q4) and ferrum-kernels
 * (src/attention/metal/pipelines.rs: gemm_f32a_f16w_v2, gemv_f32a_f16w).
 *
 * Layouts (all row-major, tightly packed, little-endian):
 *   A : float[M*K]                      activations, row m at A + m*K
 *   C : float[M*N]                      outputs, row m at C + m*N
 *   W f16  : uint16_t[N*K]              IEEE binary16 bits, row n at W + n*K
 *   W q8_0 : uint8_t[N*(K/32)*34]       per 32-element block: f16 scale d
 *                                       (2 bytes) then 32 x int8 q; x = d*q
 *   W q4_0 : uint8_t[N*(K/32)*18]       per block: f16 scale d then 16 bytes;
 *                                       byte j holds q_j (low nibble) and
 *                                       q_{j+16} (high nibble); x = d*(q-8)
 *
 * Conventions shared by every compute entry point:
 *   - A, W and C are DEVICE pointers on the current CUDA device; the caller
 *     owns them. C must not overlap A or W.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Calls are
 *     asynchronous: nothing is synchronised, results are ready when the
 *     stream reaches them.
 *   - M == 0 or N == 0: LQ_OK, nothing is launched (as the page's routers
 *     return early).
 *   - Quantised formats need K > 0 and K % 32 == 0, else LQ_ERR_INVALID_ARG
 *     (the page's routers assert this). f16 takes any K >= 1.
 *   - NULL pointers, negative sizes, pointers not aligned to their element
 *     size (4 bytes for A and C, 2 for f16 W) -> LQ_ERR_INVALID_ARG, before
 *     any launch.
 *   - Shapes or alignments that the fastest kernel cannot take run on a
 *     slower, correct kernel; no call silently computes less.
 *   - A launch failure returns LQ_ERR_CUDA (cudaGetLastError after launch).
 *   - Kernels never trap: every wait inside a kernel is bounded; a wait that
 *     runs out records LQ_ERR_DEVICE_TIMEOUT in a per-device status word,
 *     read and cleared by lq_last_device_error().
 *   - Sub-matrices (e.g. the gate or up half of a fused weight) are addressed
 *     by pointer offsets; a W row offset is always block-aligned.
 *   - Memory: the library allocates nothing per call and holds no workspace,
 *     with one exception: the tcgen05 route of the GEMM entry points
 *     (lq_gemm_<fmt>, lq_matmul_<fmt> and the epilogue fusions; M > 48, or
 *     shapes the warp-MMA kernel does not take), when a CTA's token tile is
 *     too large to stay in its shared memory, takes an M*K*2-byte
 *     stream-ordered buffer from a memory pool the library owns (described
 *     at lq_gemm_f16); lq_gemm_noalloc runs the same kernels on a fixed
 *     array instead. Caller-provided scratch
 *     (lq_topk_f32's work) is named in the call.
 *   - Kernels launched on a stream may begin streaming W before the previous
 *     kernel on that stream has finished (programmatic dependent launch); A
 *     and C are touched only after it has. Do not write W on the same stream
 *     with a kernel that itself allows early launch of its successors.
 */
#ifndef LQ_H
#define LQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LQ_OK = 0,
  LQ_ERR_INVALID_ARG = 1,    /* bad pointer, size or alignment; nothing ran   */
  LQ_ERR_UNSUPPORTED = 2,    /* no kernel exists for this request             */
  LQ_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed          */
  LQ_ERR_DEVICE_TIMEOUT = 4, /* a bounded device-side wait ran out            */
  LQ_ERR_BOUNDS = 5          /* debug build (liblq_debug.so, LQ_DEBUG_BOUNDS)
                                only: a kernel's index check failed and the
                                access was skipped                            */
} lq_status;

/* Weight formats. LQ_FMT_Q4_0I is Q4_0 with the nibble order the pages' own
 * Q4 kernels read (gemv_q4_decode, gemm_q4: the low nibble of byte j is
 * element 2j, the high nibble element 2j+1); LQ_FMT_Q4_0 keeps elements
 * 0-15 in the low nibbles and 16-31 in the high ones. Same 18-byte blocks,
 * same scale, same values. */
typedef enum { LQ_FMT_F16 = 0, LQ_FMT_Q8_0 = 1, LQ_FMT_Q4_0 = 2, LQ_FMT_Q4_0I = 3 } lq_format;

/* ---- decode GEMV, M == 1 (M != 1 -> LQ_ERR_INVALID_ARG) -----------------
 * One pass over W: each output C[0,n] = sum_k A[0,k] * w(n,k), accumulated
 * in f32 (Q formats: sum of q*a per block slice, times d, as gemv_q8_decode /
 * gemv_q4_decode do). Bound by HBM bandwidth: a decode step streams every
 * weight once, the point the page's dispatcher makes for decode (dispatch.rs,
 * dispatch_gemm_q3). */
lq_status lq_gemv_f16 (const float* A, const void* W, float* C,
                       int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_gemv_q8_0(const float* A, const void* W, float* C,
                       int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_gemv_q4_0(const float* A, const void* W, float* C,
                       int64_t M, int64_t N, int64_t K, void* stream);

/* ---- prefill GEMM, any M >= 1 -----------------------------------------
 * Counterparts: gemm_q8 / gemm_q4 / gemm_q4_tiled (metal_qwen35.rs),
 * gemm_f32a_f16w_v2 (ferrum-kernels pipelines.rs). Up to four rows of the
 * shapes the warp-MMA kernel below does not take stream W on the CUDA cores
 * in f32 (GEMV accuracy); everything else runs on the tensor cores
 * with bf16 operands: A rounded to bf16 (round to nearest even, over f32's
 * whole range), each weight formed exactly in f32 and rounded once to bf16
 * (any finite block scale), products accumulated in f32 -- up to 48 rows
 * with warp-level MMAs on W streamed once (K a multiple of 256; up to 128
 * W rows per SM, 64 beyond 16 rows of A, 48 beyond 32, and stages that fit
 * twice in shared memory), beyond with tcgen05 MMAs and TMEM accumulators. Tolerance: 5e-3 times
 * sum_k |a_k w_k| plus 1e-5, against A rounded to bf16 (the weights'
 * rounding contributes at most 2^-8 of the sum).
 * Workspace: the tcgen05 route converts A once per call into a
 * stream-ordered buffer of M*K*2 bytes taken from the library's own memory
 * pool (cudaMallocFromPoolAsync; the pool keeps freed blocks, so repeated
 * calls and CUDA-graph replays reuse the same memory without a driver
 * call). This departs from "the library allocates nothing": every one of
 * the N/128 tiles reads its token tile from that one copy, where converting
 * f32 A inside the GEMM would double the bytes each SM pulls for its token
 * tiles. Callers that may not allocate use lq_gemm_noalloc. */
lq_status lq_gemm_f16 (const float* A, const void* W, float* C,
                       int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_gemm_q8_0(const float* A, const void* W, float* C,
                       int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_gemm_q4_0(const float* A, const void* W, float* C,
                       int64_t M, int64_t N, int64_t K, void* stream);

/* ---- dispatcher: M == 1 -> GEMV, M > 1 -> GEMM ---------------------------
 * The matmul entry point model code calls (dispatch_matmul / dispatch_gemm
 * in dispatch.rs). */
lq_status lq_matmul_f16 (const float* A, const void* W, float* C,
                         int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_matmul_q8_0(const float* A, const void* W, float* C,
                         int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_matmul_q4_0(const float* A, const void* W, float* C,
                         int64_t M, int64_t N, int64_t K, void* stream);

/* ---- Q4_0 with interleaved nibbles (LQ_FMT_Q4_0I) -----------------------
 * As lq_gemv_q4_0 / lq_gemm_q4_0 / lq_matmul_q4_0, for weights packed by
 * lq_pack_q4_0i (byte j of a block: element 2j low, 2j+1 high). Same routes,
 * results and tolerances; A is read in the reordered sequence the nibble
 * order needs (lq_gemv_chain takes the format too). lq_gemm_noalloc does not
 * (LQ_ERR_INVALID_ARG). */
lq_status lq_gemv_q4_0i(const float* A, const void* W, float* C,
                        int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_gemm_q4_0i(const float* A, const void* W, float* C,
                        int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_matmul_q4_0i(const float* A, const void* W, float* C,
                          int64_t M, int64_t N, int64_t K, void* stream);

/* ---- host-side packers (HOST memory in, HOST memory out) ----------------
 * make_buffer_f16 / quantize_row_q8_0 (metal_qwen35.rs) and the Q4_0 rule:
 *   f16 : RNE narrowing of every element.
 *   q8_0: per 32-block d = max|x|/127 (f32), q = round(x/d) halves away from
 *         zero, clamped to [-127,127]; d == 0 -> q = 0.
 *   q4_0: per block m = first element of largest |x|, d = m/-8 (f32),
 *         q = min(15, (int)(x/d + 8.5)); d == 0 -> q = 8.
 * `out` must hold lq_packed_bytes(fmt, N, K) bytes. Non-finite input or a
 * bad shape -> LQ_ERR_INVALID_ARG (out may be partly written). The packers
 * are plain CPU code and need no GPU. */
size_t    lq_packed_bytes(int fmt, int64_t N, int64_t K); /* 0 if invalid */
lq_status lq_pack_f16 (const float* W_host, int64_t N, int64_t K, void* out_host);
lq_status lq_pack_q8_0(const float* W_host, int64_t N, int64_t K, void* out_host);
lq_status lq_pack_q4_0(const float* W_host, int64_t N, int64_t K, void* out_host);
/* The pages' own variants: Q4_0 with interleaved nibbles (LQ_FMT_Q4_0I), and
 * Q8_0 rounded as quantize_row_q8_0 computes it, q = round(x * (1/d)) with
 * 1/d in float32 (ordinary Q8_0 bytes; a code can differ by one from
 * lq_pack_q8_0's where x/d is within an ulp of a half). */
lq_status lq_pack_q4_0i(const float* W_host, int64_t N, int64_t K, void* out_host);
lq_status lq_pack_q8_0_rcp(const float* W_host, int64_t N, int64_t K, void* out_host);

/* ---- decode chain: many M = 1 GEMVs in one launch ------------------------
 * (An addition of this library for the decode step the source pages run as
 * a sequence of gemv_decode_m1 / gemv_q8_decode / gemv_q4_decode
 * dispatches, one per projection; the pages have no such engine.)
 * Computes, for j = 0 .. count-1 in order, C_j[n] = sum_k A_j[k] w_j(n, k)
 * with every W_j in format `fmt`; W_j, A_j, C_j are device pointers laid
 * out as for lq_gemv_<fmt> (M = 1). If problems[j].after is non-zero,
 * problem j reads A_j only after problems 0 .. j-1 are complete, so A_j may
 * be (or depend on) an earlier C; otherwise A_j must not be written by this
 * call. Weights are streamed ahead of the computation in every case. Each
 * run of problems that wait for nothing is one launch (one CTA per SM, or
 * the streaming GEMV for a run of one problem), the runs in order on the
 * stream, each streaming its weights while the previous kernel finishes and
 * reading A after it; the problems array is read during the call (host
 * memory, caller-owned).
 *   - count in 1..64; N_j >= 0; K_j % 8 == 0 (f16) or K_j % 256 == 0
 *     (quantised) with the largest K_j at most 4096 (f16), 14336 (Q8_0) or
 *     15616 (Q4_0, Q4_0I) so that A and the ring fit in shared memory;
 *     A_j and W_j 16-byte aligned. Anything else returns
 *     LQ_ERR_UNSUPPORTED without launching anything (use lq_gemv_<fmt>).
 *   - Device-side waits are bounded; lq_last_device_error reports a
 *     timeout. At most 64 calls may be in flight at once across streams. */
typedef struct {
  const float* A;
  const void*  W;
  float*       C;
  int64_t      N;
  int64_t      K;
  int32_t      after;
} lq_gemv_problem;
lq_status lq_gemv_chain(int fmt, const lq_gemv_problem* problems, int count, void* stream);

/* ---- tensor-core GEMM without device allocation ---------------------------
 * (An addition of this library; the source pages have no counterpart.)
 * Same result as lq_gemm_<fmt> on its tensor-core route (fmt: LQ_FMT_*), for
 * callers that must not allocate device memory during the call: runtimes
 * that own all device memory and hand the library none, services that fix
 * their memory budget at start-up, real-time paths where an allocation is a
 * stall or a failure point they cannot accept. Its
 * workspace is a fixed 8 MiB array inside this library, held on every GPU
 * that loads the library until the process exits; it holds the bf16 copy
 * of A, round_up(M*K*2, 256) bytes, so M*K up to 4 Mi elements.
 *   - LQ_ERR_UNSUPPORTED: larger than the fixed workspace, or a shape or
 *     alignment the tensor-core kernel does not take (K % 256 for Q8_0/Q4_0,
 *     K % 128 for f16, A and W 16-byte aligned, M >= 2). Nothing runs.
 *   - Other argument errors as for lq_gemm_<fmt>.
 *   - The first call on a device looks up the array's device address (a
 *     CUDA runtime query); make that first call before any stream capture.
 *   - All calls share the one array: calls whose executions overlap on the
 *     GPU (different streams or host threads) race and give wrong
 *     results; serialise them. Nothing carries over between calls. */
lq_status lq_gemm_noalloc(int fmt, const float* A, const void* W, float* C,
                          int64_t M, int64_t N, int64_t K, void* stream);

/* ---- argmax: LM-head GEMV fused with the selection of its best row --------
 * lm_head block-top-k stage 1 and 2 (lattice-inference, src/forward/
 * metal_qwen35/inner/dispatch.rs: dispatch_lm_head_block_stage1_enc,
 * dispatch_block_topk_merge_enc) for k = 1, with the candidate order of
 * topk_better and the merge of logits_argmax_first / logits_argmax_merge
 * (lattice-inference 0.1.2, src/forward/metal_qwen35.rs):
 *   index = the n with the largest y[n]; equal values -> the lowest n;
 *   NaN is never chosen; -0 and +0 are equal (a winning zero is reported
 *   as +0). If every y[n] is NaN the result is the pages' sentinel:
 *   value = -inf, index = -1.
 * `out` is a DEVICE pointer to one caller-owned lq_argmax_result, 8-byte
 * aligned. The call zeroes its work words on `stream` before the kernel and
 * writes value and index when the kernel completes; work is undefined
 * afterwards. Calls in flight at the same time need distinct results. */
typedef struct {
  float    value;    /* y[index], or -inf when nothing was chosen */
  int32_t  index;    /* the chosen row, or -1 */
  uint64_t work[2];  /* scratch of the call */
} lq_argmax_result;

/* y = A W^T for M = 1 (A: K floats; W: N rows in format `fmt`, as for
 * lq_gemv_<fmt>), then the argmax of y, in one kernel: each row's output is
 * ranked where it is produced and the per-warp winners are merged with one
 * 64-bit atomic each. C (N floats, device) receives y when non-NULL; with C
 * NULL the logits are never stored.
 *   - N >= 1 and N < 2^30, else LQ_ERR_INVALID_ARG; K as for lq_gemv_<fmt>.
 *   - Shapes outside the streaming GEMV's fast path (K or alignment) run the
 *     GEMV into C followed by lq_argmax_f32 on C; with C NULL they return
 *     LQ_ERR_UNSUPPORTED and launch nothing.
 *   - A device-side timeout (lq_last_device_error) leaves `out` unwritten. */
lq_status lq_gemv_argmax(int fmt, const float* A, const void* W, float* C,
                         int64_t N, int64_t K, lq_argmax_result* out, void* stream);

/* The argmax of x[0 .. n-1] (device floats), the same order and result as
 * lq_gemv_argmax: the unfused pair logits_argmax_first + logits_argmax_merge
 * of the pages as one launch. n >= 1 and n < 2^31, else LQ_ERR_INVALID_ARG;
 * x 4-byte aligned. */
lq_status lq_argmax_f32(const float* x, int64_t n, lq_argmax_result* out, void* stream);

/* ---- top-k --------------------------------------------------------------
 * The k best entries (1 <= k <= 64), best first, in the order of the argmax
 * above (larger value first, equal values by the lower index, NaN never
 * chosen); when fewer than k entries are not NaN the rest are the pages'
 * sentinel (value -inf, index -1). logits_topk_first_pass /
 * logits_topk_merge_pass (lattice-inference 0.1.2, src/forward/
 * metal_qwen35.rs), as two launches: per-CTA candidates, then one merge.
 * values (k floats), indices (k int32) and work (lq_topk_work_bytes(n, k)
 * bytes, 8-byte aligned) are caller-owned device buffers; work is scratch.
 *
 * lq_topk_f32: over x[0 .. n-1] (device floats), 1 <= n < 2^31.
 * lq_gemv_topk: the GEMV (M = 1, as lq_gemv_<fmt>) into C (required, N
 *   floats), then the top-k of C.
 * lq_topk_work_bytes: 0 for arguments out of range. */
size_t    lq_topk_work_bytes(int64_t n, int k);
lq_status lq_topk_f32(const float* x, int64_t n, int k, float* values, int32_t* indices,
                      void* work, void* stream);
lq_status lq_gemv_topk(int fmt, const float* A, const void* W, float* C, int64_t N, int64_t K,
                       int k, float* values, int32_t* indices, void* work, void* stream);

/* ---- epilogue fusions -----------------------------------------------------
 * The matmul with its output combined before it is stored, for any M (the
 * M = 1, M = 2..4 and tensor-core kernels apply it in their store; shapes
 * outside their fast paths use the generic kernel with the same epilogue).
 *
 * lq_matmul_residual: C = A W^T + R (R: M*N floats, device), as
 *   gemm_q1_v7_residual adds the hidden state to the output projection
 *   (oxibonsai-kernels 0.1.4, src/gpu_backend/metal_prefill/functions.rs).
 *   R may be C itself (in-place update of the residual stream); any other
 *   overlap of R with C is not allowed. Arguments otherwise as lq_matmul_<fmt>;
 *   R NULL or not 4-byte aligned -> LQ_ERR_INVALID_ARG.
 *
 * lq_matmul_swiglu: W is gate_up, 2*I rows in format `fmt` (gate rows
 *   0 .. I-1, then up rows I .. 2I-1, as the pages lay out gate_up and index
 *   it by offset); H (M*I floats, device) receives
 *       H[m, j] = silu(g) * u,  g = (A W^T)[m, j],  u = (A W^T)[m, I + j],
 *       silu(g) = g / (1 + exp(-g)),
 *   fused_gate_up_swiglu_gemm (same page) and silu_mul / silu_mul_fused
 *   (lattice-inference). The 2I x K gate/up products are never stored.
 *   Arguments as lq_matmul_<fmt> with N = I; 2I >= 2^30 -> LQ_ERR_UNSUPPORTED.
 *
 * Tolerances: as the underlying matmul route for the products, then the
 * float32 epilogue (one add; silu with CUDA's expf, a divide and a multiply). */
lq_status lq_matmul_residual(int fmt, const float* A, const void* W, const float* R, float* C,
                             int64_t M, int64_t N, int64_t K, void* stream);
lq_status lq_matmul_swiglu(int fmt, const float* A, const void* W, float* H,
                           int64_t M, int64_t I, int64_t K, void* stream);

/* ---- status ---------------------------------------------------------- */
const char* lq_status_string(lq_status s);
/* Synchronises the current device, then reads and clears its device status
 * word. LQ_OK if no kernel recorded an error. */
lq_status   lq_last_device_error(void);
/* Library version string. */
const char* lq_version(void);

/* ---- test hooks (the forced-route idea of the page's
 * force_q4_gemm_fallback_for_test and its fallback dispatch counter) ------
 * route: 0 = automatic, 1 = CUDA-core streaming GEMM (any M),
 *        2 = tensor-core GEMM (tcgen05), 3 = generic fallback kernels (any
 *        shape), 5 = tensor-core GEMM with warp-level MMAs for M = 2..48
 *        (LQ_ERR_UNSUPPORTED outside its shapes).
 * lq_debug_route_count(r) counts launches taken by route r (r = 0 counts
 * the fast GEMV, r = 4 the decode chain, r = 6 the A pre-pass launches of
 * route 2, r = 7 the route-2 GEMMs run as CTA pairs); counters are
 * process-wide. */
lq_status lq_debug_force_route(int route);
uint64_t  lq_debug_route_count(int route);
void      lq_debug_reset_counts(void);
/* Overrides the device-side wait limit in nanoseconds (0 = default, 2 s).
 * Below one millisecond the waits also stop blocking and give up after
 * ns/1000 polls (at least one), which exercises the LQ_ERR_DEVICE_TIMEOUT
 * path deterministically without any real hang. */
void      lq_debug_set_wait_limit_ns(uint64_t ns);
/* on != 0: lq_gemv_chain keeps problems that wait for earlier ones in one
 * launch, waiting on a device-wide counter (the default starts a new launch
 * at each such problem; both give the same results). For comparisons. */
void      lq_debug_chain_waits(int on);
/* Overrides the decode GEMV's launch plan (0 = automatic for each field):
 * CTAs per SM (1 or 2), rows per bulk-copy stage (1..8), shared memory per
 * CTA in bytes. For tuning sweeps; results do not change. Returns
 * LQ_ERR_INVALID_ARG for values out of range. */
lq_status lq_debug_gemv_plan(int ctas_per_sm, int rows_per_stage, int smem_bytes);
/* Overrides the tensor-core GEMM's ring depths (0 = automatic): A-tile
 * stages (2..4) and raw-weight stages (2..8); ignored when they do not fit
 * in shared memory. A non-zero a_stages also keeps A streamed through the
 * ring where it would otherwise be resident (small M), so that the two ways
 * of staging A can be compared. For tuning sweeps; results do not change. */
lq_status lq_debug_gemm_rings(int a_stages, int raw_stages);
/* on != 0: the tensor-core GEMM runs its CTAs in pairs (W row tiles 2i and
 * 2i + 1 on one 256-row cta_group::2 MMA, each CTA holding half of the
 * token tile) wherever A is streamed without a K split, the tile count is
 * even and the pairs need no more waves than single CTAs; on = 0 (the
 * default): never. Both give the same results; pairs measured slower, so
 * this is for comparisons. */
void      lq_debug_gemm_pairs(int on);

#ifdef __cplusplus
}
#endif
#endif /* LQ_H */
