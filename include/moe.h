/*
 * moe.h -- C ABI of a GB300 (sm_103a) MoE expert layer for one serving step.
 *
 * One MoE layer on a batch of T tokens (a prefill chunk of `quantum` rows plus a few decode
 * or speculative-verify rows):
 *   router logits -> top-k with normalised gates -> expert histogram, exclusive scan and
 *   stable permutation -> grouped gate/up projection with SwiGLU -> down projection ->
 *   gate-weighted unpermute-combine, plus the always-on shared expert(s).
 * Sources (web pages, by title):
 *   "moe-prefill-quantum" (ds4-server on M3 Ultra): the cause section, the expected
 *     unique-experts formula, Table 9 (tokens per expert = Q*k/E, cost flattens at 48).
 *   "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra": Decode paragraph (router and
 *     top-k in one dispatch, fused shared-expert gate+up+SwiGLU, bf16 rounding inside the
 *     producer kernel) and DSpark paragraph (6 verify rows share one weight stream).
 *   "Why SSD-streamed MoE was slow: 8GB Jetson Orin Nano, part 2": gate -> up -> down as
 *     SwiGLU(gate, up); `mul_mat_id` grouped expert matmul; every chosen expert must be
 *     computed exactly once (the section on generated text changing between runs).
 *
 * Conventions for every entry point below:
 *   - Tensor pointers are DEVICE pointers unless stated otherwise.  They are borrowed: the
 *     caller owns them and keeps them alive until the work queued on `stream` has finished.
 *   - Layouts are row-major with the last index contiguous.  bf16 tensors are passed as
 *     `void*` holding IEEE bfloat16 bit patterns.
 *   - The activation tensors x, y, shared_y and out of moe_layer_forward, moe_route,
 *     moe_experts and moe_combine are moved as 16-byte vectors: their base addresses must be
 *     16-byte aligned (MOE_ERR_INVALID_ARG otherwise).
 *   - Calls that take a plan and a stream only enqueue work; they never synchronise the host,
 *     never allocate device memory and are safe to capture in a CUDA graph once the plan has its
 *     weights and workspace.  T == 0 is a no-op that returns MOE_OK.
 *   - A non-MOE_OK status means nothing was enqueued (argument errors are found before any
 *     launch) or, for MOE_ERR_CUDA, that a launch failed; moe_last_error() explains it.
 *   - Problems found on the device (an expert id out of range in moe_permute input, a
 *     non-finite router logit, a wait that timed out) never trap: they set bits of the
 *     plan's device error word, read with moe_plan_get_device_error().
 *   - A plan is not thread-safe: one host thread issues its calls, and calls that share the
 *     plan's workspace must be ordered on one stream.
 *   - moe_layer_forward may run part of its work on a second stream the plan owns: forked from
 *     `stream` (an event recorded on it) and joined back (`stream` waits for an event of the
 *     second stream) before the call's last launch, so every effect is ordered on `stream` as
 *     if all of it ran there, and a graph capture of `stream` captures both.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as the CUDA runtime's cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef struct moe_plan moe_plan; /* opaque */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, n_prefill outside [0, T] ... */
  MOE_ERR_UNSUPPORTED = 2, /* shape the kernels do not handle (see moe_plan_create) */
  MOE_ERR_NOT_READY = 3,   /* weights or workspace not set yet */
  MOE_ERR_WORKSPACE = 4,   /* workspace too small for this T, or misaligned */
  MOE_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_DEVICE = 6,      /* moe_plan_get_device_error found device-side error bits */
  MOE_ERR_TIMEOUT = 7      /* (device error bit) a bounded wait inside a kernel gave up */
} moe_status;

typedef enum {
  MOE_W_BF16 = 0,  /* routed expert weights in bf16 */
  MOE_W_MXFP4 = 1  /* routed expert weights block-scaled 4-bit: e2m1 codes, two per byte
                      (even element in the low nibble, bit 3 = sign), one e8m0 scale byte
                      2^(s-127) per 32 consecutive K elements (OCP MX v1.0) */
} moe_wdtype;

/* Which kernels run the expert FFN (gate/up + SwiGLU + down). */
typedef enum {
  MOE_PATH_AUTO = 0, /* chosen by T: a step of at most 8 tokens with bf16 routed weights runs the
                        whole layer in one launch that streams the weights (a GEMV on the CUDA
                        cores); larger steps, and 4-bit weights, the tensor-core path where the
                        shape allows it */
  MOE_PATH_SIMT = 1, /* plain CUDA-core grouped FFN (debug/reference path, slow) */
  MOE_PATH_TC = 2    /* tcgen05/TMEM grouped GEMM at every T (requires d % 128 == 0, d_ff % 64 == 0) */
} moe_path;

/* Device error bits (moe_plan_get_device_error). */
#define MOE_DEVERR_EXPERT_RANGE 0x1u /* moe_permute saw an id outside [0, E) */
#define MOE_DEVERR_NONFINITE 0x2u    /* a selected router logit was NaN or infinite */
#define MOE_DEVERR_TIMEOUT 0x4u      /* a bounded in-kernel wait expired */
#define MOE_DEVERR_SEGMENT 0x8u      /* internal work-list overflow (should not happen) */
#define MOE_DEVERR_RANGE 0x10u       /* an intermediate (h or y) exceeded the fp16 range and was
                                        clamped to +-65504 */

/*
 * Create a plan for E routed experts, top-k, model width d_model, expert hidden width d_ff,
 * n_shared always-on shared experts (0 allowed; their width is set by moe_plan_set_shared) and
 * routed-weight format weight_dtype.  Source: the layer shapes of "moe-prefill-quantum" (cause
 * section: 256 experts, k chosen per token) and "DeepSeek V4.1F Q4 with native DSpark MTP on M3
 * Ultra" (Decode paragraph: a 384-expert router and an always-run shared expert).
 * Host-side only; no device memory is touched.
 * Limits: 1 <= k <= E <= 1024, k <= 32, d_model and d_ff multiples of 8 (multiples of 32
 * for MOE_W_MXFP4).  Returns NULL on bad arguments (moe_last_error() says why).
 */
moe_plan* moe_plan_create(int E, int k, int d_model, int d_ff, int n_shared, moe_wdtype weight_dtype);

/* Free the plan and the device memory it owns (its weight copies).  NULL is a no-op.
   Synchronises the device first so no queued work still reads the plan's memory.  (No
   counterpart on the pages: resource management of this library.) */
void moe_plan_destroy(moe_plan* plan);

/* Message for the most recent failing call on this host thread ("" if none).  (No counterpart
   on the pages: error reporting of this library.) */
const char* moe_last_error(void);

/*
 * Source: the expert FFN weights gate, up, down of "Why SSD-streamed MoE was slow: 8GB Jetson
 * Orin Nano, part 2" (section re-checking part 1) and their block-scaled 4-bit form ("moe-prefill-
 * quantum", hardware-check paragraph: MXFP4 unpack times scale).
 * Copy the layer's weights into plan-owned device memory (repacked for the kernels); the
 * caller's buffers may be freed when this returns.  Synchronous.  All pointers are device
 * pointers.  bf16 down-projection weights are held as fp16 (the down GEMM multiplies them with
 * the fp16 hidden vector): exact for 2^-17 <= |w| <= 65504 and zero, smaller magnitudes land
 * on the fp16 subnormal grid (absolute error <= 2^-25); a weight above 65504 in magnitude
 * makes the call fail with MOE_ERR_UNSUPPORTED.
 *   w_router  fp32 [E][d_model]                 router weight (logit = x . w_router[e] + b[e])
 *   b_router  fp32 [E] or NULL (zero bias)
 *   w_gate    [E][d_ff][d_model]                bf16, or e2m1 codes [E][d_ff][d_model/2]
 *   w_up      [E][d_ff][d_model]                same format as w_gate
 *   w_down    [E][d_model][d_ff]                bf16, or codes [E][d_model][d_ff/2]
 *   s_gate, s_up  uint8 [E][d_ff][d_model/32]   e8m0 scales (MOE_W_MXFP4), else NULL
 *   s_down        uint8 [E][d_model][d_ff/32]
 */
moe_status moe_plan_set_weights(moe_plan* plan, const float* w_router, const float* b_router,
                                const void* w_gate, const void* w_up, const void* w_down,
                                const uint8_t* s_gate, const uint8_t* s_up, const uint8_t* s_down);

/*
 * Source: "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra", Decode paragraph (the shared
 * expert's gate+up+SwiGLU runs for every token).
 * Shared experts (bf16), added to every token with weight 1:
 *   w_gate, w_up [n_shared][d_ff_shared][d_model],  w_down [n_shared][d_model][d_ff_shared].
 * Required before forward when n_shared > 0 (and before moe_plan_set_workspace, whose size
 * depends on d_ff_shared).  Copies into plan memory (w_down as fp16, as above); synchronous.
 */
moe_status moe_plan_set_shared(moe_plan* plan, int d_ff_shared, const void* w_gate,
                               const void* w_up, const void* w_down);

/* Bytes of device workspace forward/route/permute/experts need for up to T_max tokens (no
   counterpart on the pages: the library's memory contract, so that no call allocates). */
size_t moe_plan_workspace_bytes(const moe_plan* plan, int T_max);

/*
 * (No counterpart on the pages: the library's memory contract.)
 * Give the plan a caller-owned device workspace of `bytes` (>= moe_plan_workspace_bytes(T_max),
 * 256-byte aligned).  The plan keeps the pointer until the next call or destroy; it never
 * allocates device memory itself after this point.
 */
moe_status moe_plan_set_workspace(moe_plan* plan, void* dev_ptr, size_t bytes, int T_max);

/* Choose the expert-FFN kernels (default MOE_PATH_AUTO; env MOE_FORCE_PATH=simt|tc overrides
   the default at plan creation).  No counterpart on the pages: a testing and debugging switch. */
moe_status moe_plan_set_path(moe_plan* plan, moe_path path);

/*
 * The kernels the expert FFN will actually run on (no counterpart on the pages): MOE_PATH_TC
 * or MOE_PATH_SIMT, as MOE_PATH_AUTO (or a forced path) resolves for the plan's shapes and
 * weights -- the tensor-core path needs d_model % 128 == 0, d_ff % 64 == 0, d_ff_shared % 64
 * == 0 and, for MOE_W_MXFP4, every e8m0 scale byte in [104, 140] (where e2m1 x 2^(s-127) is exact
 * in fp16).  MOE_PATH_SIMT is the CUDA-core reference path, orders of magnitude slower; a caller
 * that must not run it checks this after moe_plan_set_weights / moe_plan_set_shared, and
 * moe_last_error() then names the reason.  Returns -1 for a NULL plan.
 */
int moe_plan_resolved_path(const moe_plan* plan);

/*
 * The whole layer on one serving step.  Source: "moe-prefill-quantum", the cause section and
 * Table 9 (a step's batch is a prefill chunk of `quantum` rows plus the decode rows of the
 * generating sessions, and every row goes through the MoE layer) and "DeepSeek V4.1F Q4 with
 * native DSpark MTP on M3 Ultra", Decode and DSpark paragraphs (decode and 6-row verify steps).
 * x bf16 [T][d_model] -> out bf16 [T][d_model]:
 *   out[t] = sum_j g[t,j] * FFN_{ids[t,j]}(x[t]) + sum_s FFN_shared_s(x[t]),
 * the sum taken in fp32 in slot order j = 0..k-1, then the shared term, then one
 * round-to-nearest-even to bf16.  Rows [0, n_prefill) are prefill rows and the rest decode or
 * verify rows; the layer is per token, so the result does not depend on n_prefill.
 * 0 <= T <= T_max of the workspace.
 */
moe_status moe_layer_forward(moe_plan* plan, const void* x, int T, int n_prefill, void* out,
                             moe_stream_t stream);

/*
 * Router + top-k.  Source: "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra", Decode
 * paragraph (router logits and top-k selection, one dispatch); "moe-prefill-quantum", cause
 * section (k of E experts per token).  The tie rule (lower index first) is this library's.
 * logits fp32 [T][E] (may be NULL: then kept in the workspace),
 * ids int32 [T][k], gates fp32 [T][k].  Slot j holds the (j+1)-th largest logit under the
 * order (value desc, index asc; +0 == -0; NaN lowest); gates are the softmax of the k
 * selected logits, computed in fp32.
 */
moe_status moe_route(moe_plan* plan, const void* x, int T, float* logits, int32_t* ids,
                     float* gates, moe_stream_t stream);

/* Top-k and gates from given fp32 logits [T][E] (the same selection code as moe_route; the
   Decode paragraph's top-k step of "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra").
   Exists so that selection can be compared bit for bit on identical logits. */
moe_status moe_route_logits(moe_plan* plan, const float* logits, int T, int32_t* ids,
                            float* gates, moe_stream_t stream);

/*
 * Grouping of the T*k assignments a = t*k + j by expert.  Source: "Why SSD-streamed MoE was
 * slow: 8GB Jetson Orin Nano, part 2" -- the grouped expert matmul (`mul_mat_id`, first-cache
 * section) needs the rows of each expert together, and the section on generated text changing
 * between runs requires every chosen expert to be computed exactly once (a bijection here):
 *   counts int32 [E], offsets int32 [E+1] (exclusive scan, offsets[E] = T*k),
 *   perm int32 [T*k] (perm[r] = a, a stable counting sort: rows of one expert ascend by a),
 *   inv_perm int32 [T*k] (inv_perm[perm[r]] = r).
 * An id outside [0, E), or one that repeats an earlier slot of the same token, sets
 * MOE_DEVERR_EXPERT_RANGE and is dropped: it is not counted, gets no row, and its inv_perm entry
 * is -1; perm then holds offsets[E] < T*k rows and its tail is left untouched.  With T == 0,
 * counts and offsets are zeroed and ids, perm, inv_perm may be NULL.
 */
moe_status moe_permute(moe_plan* plan, const int32_t* ids, int T, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv_perm, moe_stream_t stream);

/*
 * moe_permute without a plan and without any device allocation.  The pages have no counterpart
 * to this call; it exists for callers that cannot allocate device memory: engines whose memory
 * planner owns the whole device and forbids components from allocating outside its pool, and
 * code on a latency-critical path, where cudaMalloc would synchronise the device.  Same inputs and outputs as moe_permute
 * (ids int32 [T][k] -> counts [E], offsets [E+1], perm and inv_perm [T*k], all device
 * pointers; invalid or repeated ids are dropped with inv_perm = -1, but there is no error word).
 * Scratch is a fixed 1 MiB device array inside the library, present on every GPU that loads it
 * until the process exits; ceil(ceil(T / 32) / 4) * 4 * E must not exceed 262144 (T <= 32768 at
 * E = 256),
 * else MOE_ERR_WORKSPACE and nothing is enqueued.  The first call in a CUDA context (the first
 * on a device, and the first after that device's context was destroyed and re-created, e.g. by
 * cudaDeviceReset) looks up the array's device address (cudaGetSymbolAddress); make that first
 * call before any stream capture.  All calls share the array: two calls that may run at the same time on the GPU
 * (unordered streams) race; calls ordered on one stream do not.  Every scratch word a call
 * reads is rewritten by that call, so no clearing is needed between calls.
 */
moe_status moe_permute_static(int E, int k, const int32_t* ids, int T, int32_t* counts,
                              int32_t* offsets, int32_t* perm, int32_t* inv_perm, moe_stream_t stream);

/*
 * Self-test of the bounded waits' expiry path (failure detection; the pages have no counterpart).
 * Launches one CTA whose first warp waits on an mbarrier phase nothing completes, with the same
 * bounded wait the layer's kernels use, while its second warp holds a TMEM allocation: after
 * about one second (the kernels' wait limit) the wait gives up, sets MOE_DEVERR_TIMEOUT in *err
 * and raises the CTA's abort flag, and the CTA takes the GEMM kernels' abort teardown (waits out
 * in-flight copies, frees TMEM) and returns, leaving the context usable.
 *   err     device uint32, OR-ed with the error bits (the caller clears it first);
 *   result  device uint32 [3]: [0] = 2 when the wait expired (1 if it completed), [1] = the
 *           milliseconds it waited, [2] = 1 if the abort flag was raised.
 * Returns MOE_ERR_INVALID_ARG for NULL pointers, MOE_ERR_CUDA if the launch fails.
 */
moe_status moe_selftest_wait_expiry(uint32_t* err, uint32_t* result, moe_stream_t stream);

/*
 * Expert FFNs on grouped rows (testing entry point for the grouped GEMMs).  Source: "Why
 * SSD-streamed MoE was slow: 8GB Jetson Orin Nano, part 2", section re-checking part 1 (gate ->
 * up -> down, SwiGLU(gate, up)); "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra", Decode
 * paragraph (intermediates rounded inside the producing kernel):
 *   y[r] = FFN_e(x[perm[r] / k]) for r in [offsets[e], offsets[e+1]),  fp16 [T*k][d_model],
 *   shared_y[t] = sum_s FFN_shared_s(x[t]) fp16 [T][d_model] (may be NULL if n_shared == 0).
 * FFN(x) = W_d (silu(W_g x) * (W_u x)) with fp32 accumulation; the hidden vector is rounded to
 * fp16 (it is the fp16 operand of the down GEMM) and y is rounded to fp16.  Values beyond the
 * fp16 range are clamped and set MOE_DEVERR_RANGE.  offsets and perm as produced by
 * moe_permute (device pointers).
 */
moe_status moe_experts(moe_plan* plan, const void* x, int T, const int32_t* offsets,
                       const int32_t* perm, void* y, void* shared_y, moe_stream_t stream);

/*
 * Gate-weighted unpermute-combine.  Source: the combine is implicit in the pages -- every token's
 * output is the gate-weighted sum of its chosen experts' outputs ("moe-prefill-quantum", cause
 * section: each token is sent to k of the E experts; "Why SSD-streamed MoE was slow", part 2,
 * the section on generated text changing between runs: each chosen expert counted exactly once).
 *   out[t] = sum_{j<k} gates[t,j] * y[inv_perm[t*k+j]]  (+ shared_y[t]),
 * fp32 accumulation in slot order, then the shared term, one round-to-nearest-even to bf16.
 *   y         fp32 [T*k][d_model] in grouped (permuted) row order (device);
 *   gates     fp32 [T][k];  inv_perm int32 [T*k] (entries < 0 are skipped);
 *   shared_y  fp32 [T][d_model] or NULL;  out bf16 [T][d_model].
 * Needs no workspace and no weights (only the plan's k and d_model).  d_model % 8 != 0 gives
 * MOE_ERR_UNSUPPORTED.  (moe_layer_forward runs the same kernel on its own fp16 intermediates.)
 */
moe_status moe_combine(moe_plan* plan, const float* y, const float* gates, const int32_t* inv_perm,
                       const float* shared_y, int T, void* out, moe_stream_t stream);

/* Synchronise the device, return the device error word in *code (host pointer) and clear
   it.  Returns MOE_ERR_DEVICE when *code != 0.  No counterpart on the pages (failure detection
   of this library: device-side problems never trap). */
moe_status moe_plan_get_device_error(moe_plan* plan, uint32_t* code);

/*
 * Per-kernel timing for profiling (no counterpart on the pages).  When enabled, every kernel launched by the calls above
 * is bracketed by CUDA events recorded on the launching stream (a few microseconds of
 * overhead per launch).  moe_plan_timing_report synchronises, writes one line per kernel
 * name, "name launches total_ms\n", into buf (host memory, NUL-terminated, truncated to
 * len) and resets the counters.  Returns the number of bytes the full report needs.
 */
moe_status moe_plan_enable_timing(moe_plan* plan, int enable);
size_t moe_plan_timing_report(moe_plan* plan, char* buf, size_t len);

/* Number of kernels the most recent moe_layer_forward call launched (no counterpart on the
   pages; the Decode paragraph of "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra" counts
   dispatches per layer the same way). */
int moe_plan_last_launch_count(const moe_plan* plan);

/*
 * Step composer: the layer calls (serving steps) a prompt's prefill is cut into.
 * Source: "moe-prefill-quantum" -- the cause section's source excerpt (the server hands the
 * prompt over in pieces of `quantum` tokens while any request is generating, else of 2048) and
 * the section on prefill_cap boundaries with its code excerpt and Table 11 (the engine cuts a
 * piece where the absolute context position crosses a multiple of prefill_cap; a prompt that
 * starts off a boundary keeps being cut, e.g. 2048, 509, 1539, ... from 1539 mod 4096).
 * Reading where the excerpt is silent: no call exceeds prefill_cap tokens.
 *
 * Host-only and pure (no device work, no plan).  Prefilling n_tokens prompt tokens from
 * context position start_pos: writes the first min(total, max_calls) calls, in order, to
 * `calls` (host memory; may be NULL when max_calls == 0) and the total number of calls to
 * *n_calls (host pointer).  Each call's `n` prompt rows go to moe_layer_forward as its
 * n_prefill rows, followed by one row per generating request.
 * MOE_ERR_INVALID_ARG when start_pos < 0, n_tokens < 0, quantum < 1, prefill_cap < 1 or
 * n_calls is NULL.
 */
typedef struct {
  int64_t pos;   /* context position of the call's first prompt token */
  int32_t n;     /* prompt tokens in the call, 1 <= n <= prefill_cap */
  int32_t piece; /* index of the server piece the call belongs to */
} moe_prefill_call;

moe_status moe_compose_prefill(int64_t start_pos, int64_t n_tokens, int32_t quantum,
                               int32_t generation_active, int32_t prefill_cap,
                               moe_prefill_call* calls, int64_t max_calls, int64_t* n_calls);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
