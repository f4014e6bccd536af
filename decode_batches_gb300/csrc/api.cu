// C ABI of the MoE layer: plan, validation, weight set-up, workspace carving and the launch
// sequence of each entry point (see include/moe.h for the contract of every call).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"

using namespace moe;

// ============================================================================================
// errors
// ============================================================================================
static thread_local std::string g_last_error;

static moe_status fail(moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

#define MOE_CUDA_TRY(expr)                                                                  \
  do {                                                                                      \
    cudaError_t _e = (expr);                                                                \
    if (_e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(_e)); \
  } while (0)

extern "C" const char* moe_last_error(void) { return g_last_error.c_str(); }

moe_status moe::fail_message(moe_status s, const char* msg) {
  g_last_error = msg;
  return s;
}

// ============================================================================================
// plan
// ============================================================================================
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t logits, parts, ids, gates, masks, counts, offsets, perm, inv, segs, n_segs, h, h_s, y, y_s, x16;
  size_t touched, y32;  // the one-launch small-step layer: touched-expert list, fp32 expert outputs
  size_t xq, xs;        // the block-scaled 4-bit gate/up: x as two e4m3 terms and their e8m0 scales
  size_t hq, hs;        // ... and down: h as two e4m3 terms and their e8m0 scales
  size_t total;
  int max_segs;
};

struct TimedLaunch {
  const char* name;
  cudaEvent_t start, stop;
};

}  // namespace

struct moe_plan {
  int E = 0, k = 0, d = 0, f = 0, n_shared = 0, f_s = 0;
  moe_wdtype wdtype = MOE_W_BF16;
  moe_path path = MOE_PATH_AUTO;
  int device = 0, num_sms = 0;
  // plan-owned device memory
  float* w_router = nullptr;
  float* b_router = nullptr;
  uint16_t* w_router3 = nullptr;  // W_r split into three bf16 pieces [3][E][d] (tensor-core router)
  CUtensorMap map_router3{};
  CUtensorMap map_x{};  // the current call's x [T][d] (tensor-core router), encoded per call
  bool router_tc = false;
  uint8_t* w_gu = nullptr;
  uint8_t* s_gu = nullptr;
  uint8_t* w_down = nullptr;
  uint8_t* s_down = nullptr;
  uint16_t* w_gu_s = nullptr;
  uint16_t* w_down_s = nullptr;
  uint32_t* err = nullptr;
  uint32_t* ls_sync = nullptr;  // launch-wide words of the one-launch small-step layer (zero between launches)
  bool weights_set = false, shared_set = false;
  bool tiled = false, tiled_s = false;  // weights stored in the tile-contiguous layouts
  bool fp4_tiled = false;  // 4-bit routed weights in the tile-contiguous layout
  bool fp4_tc = false;     // ... and every scale in the fp16-exact range: tensor-core path allowed
  // 4-bit gate/up and down on the block-scaled MMA (e2m1 weights x two e4m3 terms of x or h)
  // instead of the dequantising kernels (the default, faster as measured); env MOE_FP4_GATEUP /
  // MOE_FP4_DOWN = mx selects the former at plan creation
  bool fp4_mx = false, fp4_mx_down = false;
  // steps of at most 8 tokens with bf16 weights: the one-launch layer (layer_small.cu) instead of
  // the routing launch + tensor-core GEMMs + combine; env MOE_SMALL_STEP = fused | multi
  bool small_fused = false;
  // workspace (caller-owned)
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  int T_max = 0;
  WsLayout L{};
  TcMaps maps{};
  bool maps_weights = false, maps_ws = false;
  // plan-owned second stream: the shared expert's gate/up runs there, beside the routing, when
  // it occupies at most half of the SMs; forked from and joined back into the caller's stream
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // timing
  bool timing = false;
  std::vector<TimedLaunch> timed;
  std::vector<cudaEvent_t> event_pool;
  int launch_count = 0;

  bool router_tc_capable() const { return E % 128 == 0 && d % 64 == 0; }
};

static WsLayout layout_for(const moe_plan* p, int T_max) {
  WsLayout L{};
  const size_t T = static_cast<size_t>(T_max > 0 ? T_max : 1);
  const size_t R = T * p->k;
  const size_t n_chunks = (T + kChunk - 1) / kChunk;
  L.max_segs = p->E + static_cast<int>((R + kSegRowsMax - 1) / kSegRowsMax) + 1;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  L.logits = take(T * p->E * sizeof(float));
  // partial router logits of the tensor-core router: splits(T') * T' rows for the worst T' <= T
  size_t part_rows = 0;
  if (p->router_tc_capable())
    for (size_t m = 1; 128 * (m - 1) < T; ++m) {  // the largest T' of each 128-token tile count
      const size_t tt = 128 * m < T ? 128 * m : T;
      const size_t r = static_cast<size_t>(router_tc_splits(static_cast<int>(tt), p->E, p->d, p->num_sms)) * tt;
      if (r > part_rows) part_rows = r;
    }
  if (p->d % 128 == 0) {  // the small-T router's K-split partials
    const size_t r = static_cast<size_t>(router_small_splits(p->d)) * (T < 128 ? T : 128);
    if (r > part_rows) part_rows = r;
  }
  L.parts = take(part_rows * p->E * sizeof(float));
  L.ids = take(R * sizeof(int32_t));
  L.gates = take(R * sizeof(float));
  L.masks = take(static_cast<size_t>(group_mask_stride(static_cast<int>(n_chunks))) * p->E * sizeof(uint32_t));
  L.counts = take(p->E * sizeof(int32_t));
  L.offsets = take((p->E + 1) * sizeof(int32_t));
  L.perm = take(R * sizeof(int32_t));
  L.inv = take(R * sizeof(int32_t));
  L.segs = take(static_cast<size_t>(L.max_segs) * sizeof(Seg));
  L.n_segs = take(sizeof(int32_t));
  L.h = take(R * p->f * 2);
  L.h_s = take(T * static_cast<size_t>(p->n_shared) * p->f_s * 2);
  L.y = take(R * p->d * 2);
  L.y_s = take(T * p->d * 2);
  L.x16 = take(p->wdtype == MOE_W_MXFP4 ? T * p->d * 2 : 0);
  const size_t T8 = T < static_cast<size_t>(kLsTMax) ? T : static_cast<size_t>(kLsTMax);
  L.touched = take((p->E + 1) * sizeof(int32_t));
  L.xq = take(p->wdtype == MOE_W_MXFP4 ? T * 2 * p->d : 0);
  L.xs = take(p->wdtype == MOE_W_MXFP4 ? T * 2 * (p->d / 32) : 0);
  L.hq = take(p->wdtype == MOE_W_MXFP4 ? R * 2 * p->f : 0);
  L.hs = take(p->wdtype == MOE_W_MXFP4 ? R * 2 * static_cast<size_t>(mx_scale_bytes(p->f)) : 0);
  L.y32 = take(p->wdtype == MOE_W_BF16 ? T8 * (p->k + 1) * p->d * sizeof(float) : 0);
  L.total = o;
  return L;
}

template <typename Tp>
static Tp* ws_ptr(const moe_plan* p, size_t off) {
  return reinterpret_cast<Tp*>(p->ws + off);
}

// The tensor-core path: bf16 routed weights with d % 128 == 0 and d_ff % 64 == 0, or 4-bit
// routed weights in the tiled layout whose scales all allow exact fp16 dequantisation; shared
// experts need d_ff_shared % 64 == 0.
static bool tc_shape_ok(const moe_plan* p) {
  const bool routed = p->wdtype == MOE_W_BF16 ? (p->d % 128 == 0 && p->f % 64 == 0) : p->fp4_tc;
  return routed && (p->n_shared == 0 || p->f_s % 64 == 0);
}

static bool use_tc(const moe_plan* p) {
  if (p->path == MOE_PATH_SIMT) return false;
  return tc_shape_ok(p);
}

// The one-launch small-step layer (layer_small.cu): MOE_PATH_AUTO at T <= 8 with bf16 routed
// weights in the tensor-core tile layout (the kernel streams those tiles).
static bool use_small_layer(const moe_plan* p, int T) {
  return p->small_fused && p->path == MOE_PATH_AUTO && p->wdtype == MOE_W_BF16 && tc_shape_ok(p) && p->tiled &&
         (p->n_shared == 0 || p->tiled_s) && p->ls_sync &&
         layer_small_ok(T, p->E, p->k, p->d, p->f, p->n_shared, p->f_s);
}

// ---- timing -----------------------------------------------------------------------------------
static cudaEvent_t pool_event(moe_plan* p) {
  if (!p->event_pool.empty()) {
    cudaEvent_t e = p->event_pool.back();
    p->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

struct LaunchScope {
  moe_plan* p;
  const char* name;
  cudaStream_t st;
  cudaEvent_t start = nullptr;
  LaunchScope(moe_plan* p_, const char* n, cudaStream_t s) : p(p_), name(n), st(s) {
    ++p->launch_count;
    if (p->timing) {
      start = pool_event(p);
      if (start) cudaEventRecord(start, st);
    }
  }
  ~LaunchScope() {
    if (p->timing && start) {
      cudaEvent_t stop = pool_event(p);
      if (stop) {
        cudaEventRecord(stop, st);
        p->timed.push_back(TimedLaunch{name, start, stop});
      } else {
        p->event_pool.push_back(start);
      }
    }
  }
};

#define LAUNCH(plan, name, stream, call)                                                    \
  do {                                                                                      \
    LaunchScope _ls(plan, name, stream);                                                    \
    cudaError_t _e = (call);                                                                \
    if (_e != cudaSuccess) return fail(MOE_ERR_CUDA, "%s launch: %s", name, cudaGetErrorString(_e)); \
  } while (0)

// ---- tensor maps --------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D 16-bit tensor [rows][inner] (row pitch inner*2 bytes), box {64, box_rows}, 128-byte
// swizzle; dtype is CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 or _FLOAT16.
static moe_status make_map_16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                              uint32_t box_rows, CUtensorMapDataType dtype) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return MOE_OK;
}

static moe_status build_weight_maps(moe_plan* p) {
  // the tensor-core path reads the tile-contiguous weights directly (bulk copies, no maps)
  const bool routed = p->wdtype == MOE_W_BF16 ? p->tiled : p->fp4_tc;
  p->maps_weights = tc_shape_ok(p) && p->weights_set && routed && (p->n_shared == 0 || (p->shared_set && p->tiled_s));
  return MOE_OK;
}

static moe_status build_ws_maps(moe_plan* p) {
  p->maps_ws = false;
  if (!tc_shape_ok(p) || !p->ws) return MOE_OK;
  const uint64_t R = static_cast<uint64_t>(p->T_max) * p->k;
  moe_status s;
  const CUtensorMapDataType F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if ((s = make_map_16(&p->maps.h, p->ws + p->L.h, p->f, R, 32, F16)) != MOE_OK) return s;
  if (p->n_shared > 0 && p->f_s > 0) {
    if ((s = make_map_16(&p->maps.h_s, p->ws + p->L.h_s, static_cast<uint64_t>(p->n_shared) * p->f_s, p->T_max, 32, F16)) != MOE_OK)
      return s;
  }
  p->maps_ws = true;
  return MOE_OK;
}

// ============================================================================================
// creation / destruction
// ============================================================================================
extern "C" moe_plan* moe_plan_create(int E, int k, int d_model, int d_ff, int n_shared, moe_wdtype weight_dtype) {
  if (E < 1 || E > 1024 || k < 1 || k > 32 || k > E) {
    fail(MOE_ERR_INVALID_ARG, "need 1 <= k <= E <= 1024 and k <= 32 (E=%d k=%d)", E, k);
    return nullptr;
  }
  if (weight_dtype != MOE_W_BF16 && weight_dtype != MOE_W_MXFP4) {
    fail(MOE_ERR_INVALID_ARG, "unknown weight dtype %d", static_cast<int>(weight_dtype));
    return nullptr;
  }
  const int mult = weight_dtype == MOE_W_MXFP4 ? 32 : 8;
  if (d_model <= 0 || d_ff <= 0 || d_model % mult || d_ff % mult) {
    fail(MOE_ERR_INVALID_ARG, "d_model and d_ff must be positive multiples of %d (d=%d f=%d)", mult, d_model, d_ff);
    return nullptr;
  }
  if (n_shared < 0 || n_shared > 64) {
    fail(MOE_ERR_INVALID_ARG, "n_shared must be in [0, 64] (%d)", n_shared);
    return nullptr;
  }
  moe_plan* p = new moe_plan();
  p->E = E;
  p->k = k;
  p->d = d_model;
  p->f = d_ff;
  p->n_shared = n_shared;
  p->wdtype = weight_dtype;
  cudaGetDevice(&p->device);
  cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
  if (p->num_sms <= 0) p->num_sms = 1;
  if (const char* env = getenv("MOE_FP4_GATEUP")) p->fp4_mx = strcmp(env, "mx") == 0;
  if (const char* env = getenv("MOE_FP4_DOWN")) p->fp4_mx_down = strcmp(env, "mx") == 0;
  if (const char* env = getenv("MOE_SMALL_STEP")) p->small_fused = strcmp(env, "fused") == 0;
  if (const char* env = getenv("MOE_FORCE_PATH")) {
    if (!strcmp(env, "simt")) p->path = MOE_PATH_SIMT;
    else if (!strcmp(env, "tc")) p->path = MOE_PATH_TC;
  }
  g_last_error.clear();
  return p;
}

static void free_weights(moe_plan* p) {
  cudaFree(p->w_router3);
  p->w_router3 = nullptr;
  p->router_tc = false;
  cudaFree(p->w_router);
  cudaFree(p->b_router);
  cudaFree(p->w_gu);
  cudaFree(p->s_gu);
  cudaFree(p->w_down);
  cudaFree(p->s_down);
  p->w_router = p->b_router = nullptr;
  p->w_gu = p->s_gu = p->w_down = p->s_down = nullptr;
  p->weights_set = false;
}

extern "C" void moe_plan_destroy(moe_plan* p) {
  if (!p) return;
  cudaDeviceSynchronize();
  free_weights(p);
  cudaFree(p->w_gu_s);
  cudaFree(p->w_down_s);
  cudaFree(p->err);
  cudaFree(p->ls_sync);
  for (auto& t : p->timed) {
    cudaEventDestroy(t.start);
    cudaEventDestroy(t.stop);
  }
  for (auto e : p->event_pool) cudaEventDestroy(e);
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  if (p->side) cudaStreamDestroy(p->side);
  delete p;
}

// Plan-owned device words: [0] the error bits, [1] the small-step routing counter, [2..3] and
// [4..5] the unit hand-out words of the 4-bit gate/up and down kernels (all counters 0 between
// launches), kept out of the caller's workspace, whose contents may change between calls.
constexpr int kPlanWords = 6;
constexpr int kSchedFp4GateUp = 2, kSchedFp4Down = 4;
static moe_status ensure_err_word(moe_plan* p) {
  if (p->err) return MOE_OK;
  MOE_CUDA_TRY(cudaMalloc(&p->err, kPlanWords * sizeof(uint32_t)));
  MOE_CUDA_TRY(cudaMemset(p->err, 0, kPlanWords * sizeof(uint32_t)));
  return MOE_OK;
}

// The plan's second stream (highest priority, so that its few blocks start ahead of queued ones)
// and its fork/join events.
static moe_status ensure_side_stream(moe_plan* p) {
  if (p->side) return MOE_OK;
  int lo = 0, hi = 0;
  MOE_CUDA_TRY(cudaDeviceGetStreamPriorityRange(&lo, &hi));
  if (!p->ev_fork) MOE_CUDA_TRY(cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming));
  if (!p->ev_join) MOE_CUDA_TRY(cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming));
  MOE_CUDA_TRY(cudaStreamCreateWithPriority(&p->side, cudaStreamNonBlocking, hi));
  return MOE_OK;
}

// ============================================================================================
// weights
// ============================================================================================
// Down weights (n bf16 matrices [rows][K]) into the fp16 tile-contiguous layout.
static moe_status tile_down_f16(uint16_t* dst, const void* src, int n, int rows, int K, int by_matrix) {
  uint32_t* flag = nullptr;
  MOE_CUDA_TRY(cudaMalloc(&flag, sizeof(uint32_t)));
  cudaMemset(flag, 0, sizeof(uint32_t));
  cudaError_t e = launch_tile_down(static_cast<const uint16_t*>(src), dst, n, rows, K, by_matrix, flag, 0);
  uint32_t bad = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&bad, flag, sizeof bad, cudaMemcpyDeviceToHost);
  cudaFree(flag);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "down weight tiling: %s", cudaGetErrorString(e));
  if (bad) return fail(MOE_ERR_UNSUPPORTED, "a down-projection weight is outside the fp16 range (|w| > 65504)");
  return MOE_OK;
}

// Copy n bf16 values into an fp16 plan buffer; MOE_ERR_UNSUPPORTED if any is outside the fp16
// range (the down projection runs fp16 x fp16 on the tensor cores).
static moe_status copy_bf16_as_f16(uint16_t* dst, const void* src, size_t n) {
  uint32_t* flag = nullptr;
  MOE_CUDA_TRY(cudaMalloc(&flag, sizeof(uint32_t)));
  cudaMemset(flag, 0, sizeof(uint32_t));
  cudaError_t e = launch_bf16_to_f16(static_cast<const uint16_t*>(src), dst, n, flag, 0);
  uint32_t bad = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&bad, flag, sizeof bad, cudaMemcpyDeviceToHost);
  cudaFree(flag);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, "bf16 -> fp16 weight copy: %s", cudaGetErrorString(e));
  if (bad) return fail(MOE_ERR_UNSUPPORTED, "a down-projection weight is outside the fp16 range (|w| > 65504)");
  return MOE_OK;
}
extern "C" moe_status moe_plan_set_weights(moe_plan* p, const float* w_router, const float* b_router,
                                           const void* w_gate, const void* w_up, const void* w_down,
                                           const uint8_t* s_gate, const uint8_t* s_up, const uint8_t* s_down) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (!w_router || !w_gate || !w_up || !w_down)
    return fail(MOE_ERR_INVALID_ARG, "w_router, w_gate, w_up and w_down are required");
  const bool fp4 = p->wdtype == MOE_W_MXFP4;
  if (fp4 && (!s_gate || !s_up || !s_down))
    return fail(MOE_ERR_INVALID_ARG, "MOE_W_MXFP4 needs s_gate, s_up and s_down");
  if (!fp4 && (s_gate || s_up || s_down))
    return fail(MOE_ERR_INVALID_ARG, "scales are only valid with MOE_W_MXFP4");
  moe_status s = ensure_err_word(p);
  if (s != MOE_OK) return s;
  cudaDeviceSynchronize();
  free_weights(p);
  const size_t E = p->E, d = p->d, f = p->f;
  MOE_CUDA_TRY(cudaMalloc(&p->w_router, E * d * sizeof(float)));
  MOE_CUDA_TRY(cudaMemcpy(p->w_router, w_router, E * d * sizeof(float), cudaMemcpyDeviceToDevice));
  if (p->router_tc_capable()) {
    MOE_CUDA_TRY(cudaMalloc(&p->w_router3, 3 * E * d * sizeof(uint16_t)));
    MOE_CUDA_TRY(launch_split_router(p->w_router, p->w_router3, E * d, 0));
    s = make_map_16(&p->map_router3, p->w_router3, d, 3 * E, 128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    if (s != MOE_OK) {
      free_weights(p);
      return s;
    }
    p->router_tc = true;
  }
  MOE_CUDA_TRY(cudaMalloc(&p->b_router, E * sizeof(float)));
  if (b_router)
    MOE_CUDA_TRY(cudaMemcpy(p->b_router, b_router, E * sizeof(float), cudaMemcpyDeviceToDevice));
  else
    MOE_CUDA_TRY(cudaMemset(p->b_router, 0, E * sizeof(float)));
  const size_t gu_row = fp4 ? d / 2 : d * 2;     // bytes per gate/up row
  const size_t dn_row = fp4 ? f / 2 : f * 2;     // bytes per down row
  p->tiled = !fp4 && d % 128 == 0 && f % 64 == 0;
  p->fp4_tiled = fp4 && d % 128 == 0 && f % 64 == 0;
  p->fp4_tc = false;
  if (p->fp4_tiled) {
    // codes and scales go together into kFp4BlockBytes blocks; no separate scale arrays
    const size_t gu_blocks = E * (f / 64) * (d / 64), dn_blocks = E * (d / 128) * (f / 64);
    MOE_CUDA_TRY(cudaMalloc(&p->w_gu, gu_blocks * kFp4BlockBytes));
    MOE_CUDA_TRY(cudaMalloc(&p->w_down, dn_blocks * kFp4BlockBytes));
    uint32_t* flag = nullptr;
    MOE_CUDA_TRY(cudaMalloc(&flag, sizeof(uint32_t)));
    cudaMemset(flag, 0, sizeof(uint32_t));
    cudaError_t e = launch_tile_fp4(static_cast<const uint8_t*>(w_gate), s_gate, static_cast<const uint8_t*>(w_up), s_up,
                                    p->w_gu, p->E, p->f, p->d, 1, flag, 0);
    if (e == cudaSuccess)
      e = launch_tile_fp4(static_cast<const uint8_t*>(w_down), s_down, nullptr, nullptr, p->w_down, p->E, p->d, p->f, 0,
                          flag, 0);
    uint32_t oor = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&oor, flag, sizeof oor, cudaMemcpyDeviceToHost);
    cudaFree(flag);
    if (e != cudaSuccess) {
      free_weights(p);
      return fail(MOE_ERR_CUDA, "4-bit weight tiling: %s", cudaGetErrorString(e));
    }
    p->fp4_tc = oor == 0;  // otherwise the CUDA-core path runs the same layout
    MOE_CUDA_TRY(cudaDeviceSynchronize());
    p->weights_set = true;
    return build_weight_maps(p);
  }
  MOE_CUDA_TRY(cudaMalloc(&p->w_gu, E * 2 * f * gu_row));
  MOE_CUDA_TRY(cudaMalloc(&p->w_down, E * d * dn_row));
  if (p->tiled) {
    MOE_CUDA_TRY(launch_tile_gate_up(static_cast<const uint16_t*>(w_gate), static_cast<const uint16_t*>(w_up),
                                     reinterpret_cast<uint16_t*>(p->w_gu), p->E, p->f, p->d, 0, 0));
    s = tile_down_f16(reinterpret_cast<uint16_t*>(p->w_down), w_down, p->E, p->d, p->f, 1);
    if (s != MOE_OK) {
      free_weights(p);
      return s;
    }
  } else {
    MOE_CUDA_TRY(launch_interleave_gate_up(static_cast<const uint8_t*>(w_gate), static_cast<const uint8_t*>(w_up),
                                           p->w_gu, p->E, p->f, gu_row, 0));
    if (fp4) {
      MOE_CUDA_TRY(cudaMemcpy(p->w_down, w_down, E * d * dn_row, cudaMemcpyDeviceToDevice));
    } else {
      s = copy_bf16_as_f16(reinterpret_cast<uint16_t*>(p->w_down), w_down, E * d * f);
      if (s != MOE_OK) {
        free_weights(p);
        return s;
      }
    }
  }
  if (fp4) {
    MOE_CUDA_TRY(cudaMalloc(&p->s_gu, E * 2 * f * (d / 32)));
    MOE_CUDA_TRY(launch_interleave_gate_up(s_gate, s_up, p->s_gu, p->E, p->f, d / 32, 0));
    MOE_CUDA_TRY(cudaMalloc(&p->s_down, E * d * (f / 32)));
    MOE_CUDA_TRY(cudaMemcpy(p->s_down, s_down, E * d * (f / 32), cudaMemcpyDeviceToDevice));
  }
  MOE_CUDA_TRY(cudaDeviceSynchronize());
  p->weights_set = true;
  return build_weight_maps(p);
}

extern "C" moe_status moe_plan_set_shared(moe_plan* p, int d_ff_shared, const void* w_gate, const void* w_up,
                                          const void* w_down) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (p->n_shared == 0) return fail(MOE_ERR_INVALID_ARG, "plan was created with n_shared = 0");
  if (d_ff_shared <= 0 || d_ff_shared % 8) return fail(MOE_ERR_INVALID_ARG, "d_ff_shared must be a positive multiple of 8");
  if (!w_gate || !w_up || !w_down) return fail(MOE_ERR_INVALID_ARG, "shared weights are required");
  if (p->ws && d_ff_shared != p->f_s)
    return fail(MOE_ERR_INVALID_ARG, "d_ff_shared changed after the workspace was set; set the workspace again");
  moe_status s = ensure_err_word(p);
  if (s != MOE_OK) return s;
  cudaDeviceSynchronize();
  cudaFree(p->w_gu_s);
  cudaFree(p->w_down_s);
  p->w_gu_s = p->w_down_s = nullptr;
  p->f_s = d_ff_shared;
  const size_t n = p->n_shared, d = p->d, fs = d_ff_shared;
  MOE_CUDA_TRY(cudaMalloc(&p->w_gu_s, n * 2 * fs * d * 2));
  MOE_CUDA_TRY(cudaMalloc(&p->w_down_s, n * d * fs * 2));
  p->tiled_s = d % 128 == 0 && fs % 64 == 0;
  if (p->tiled_s) {
    MOE_CUDA_TRY(launch_tile_gate_up(static_cast<const uint16_t*>(w_gate), static_cast<const uint16_t*>(w_up), p->w_gu_s,
                                     p->n_shared, p->f_s, p->d, 1, 0));
    s = tile_down_f16(p->w_down_s, w_down, p->n_shared, p->d, p->f_s, 0);
  } else {
    MOE_CUDA_TRY(launch_interleave_gate_up(static_cast<const uint8_t*>(w_gate), static_cast<const uint8_t*>(w_up),
                                           reinterpret_cast<uint8_t*>(p->w_gu_s), p->n_shared, p->f_s, d * 2, 0));
    s = copy_bf16_as_f16(p->w_down_s, w_down, n * d * fs);
  }
  if (s != MOE_OK) return s;
  MOE_CUDA_TRY(cudaDeviceSynchronize());
  p->shared_set = true;
  return build_weight_maps(p);
}

// ============================================================================================
// workspace and options
// ============================================================================================
extern "C" size_t moe_plan_workspace_bytes(const moe_plan* p, int T_max) {
  if (!p || T_max < 0) return 0;
  if (p->n_shared > 0 && p->f_s == 0) {
    // width of the shared experts unknown yet: size for the routed width
    moe_plan tmp = *p;
    tmp.f_s = p->f;
    return layout_for(&tmp, T_max).total;
  }
  return layout_for(p, T_max).total;
}

extern "C" moe_status moe_plan_set_workspace(moe_plan* p, void* dev_ptr, size_t bytes, int T_max) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (!dev_ptr || T_max < 1) return fail(MOE_ERR_INVALID_ARG, "workspace pointer and T_max >= 1 required");
  if (reinterpret_cast<uintptr_t>(dev_ptr) & 255) return fail(MOE_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (p->n_shared > 0 && !p->shared_set)
    return fail(MOE_ERR_NOT_READY, "set the shared experts before the workspace (their width sizes it)");
  const WsLayout L = layout_for(p, T_max);
  if (bytes < L.total)
    return fail(MOE_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed for T_max=%d", bytes, L.total, T_max);
  p->ws = static_cast<uint8_t*>(dev_ptr);
  p->ws_bytes = bytes;
  p->T_max = T_max;
  p->L = L;
  moe_status s = ensure_err_word(p);
  if (s != MOE_OK) return s;
  if ((s = ensure_side_stream(p)) != MOE_OK) return s;
  if (!p->ls_sync) {
    MOE_CUDA_TRY(cudaMalloc(&p->ls_sync, kLsSyncWords * sizeof(uint32_t)));
    MOE_CUDA_TRY(cudaMemset(p->ls_sync, 0, kLsSyncWords * sizeof(uint32_t)));
  }
  return build_ws_maps(p);
}

extern "C" moe_status moe_plan_set_path(moe_plan* p, moe_path path) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (path != MOE_PATH_AUTO && path != MOE_PATH_SIMT && path != MOE_PATH_TC)
    return fail(MOE_ERR_INVALID_ARG, "unknown path %d", static_cast<int>(path));
  if (path == MOE_PATH_TC && !tc_shape_ok(p))
    return fail(MOE_ERR_UNSUPPORTED, "tensor-core path needs bf16 weights, d %% 128 == 0, d_ff %% 64 == 0, d_ff_shared %% 64 == 0");
  p->path = path;
  return MOE_OK;
}

extern "C" int moe_plan_resolved_path(const moe_plan* p) {
  if (!p) return -1;
  if (use_tc(p)) return MOE_PATH_TC;
  if (p->path == MOE_PATH_SIMT) {
    fail(MOE_OK, "the CUDA-core path was chosen with moe_plan_set_path or MOE_FORCE_PATH");
  } else if (p->wdtype == MOE_W_MXFP4 && p->weights_set && p->fp4_tiled && !p->fp4_tc) {
    fail(MOE_OK, "an e8m0 scale byte is outside [%d, %d]: the 4-bit weights cannot be dequantised exactly "
                 "into fp16, so the CUDA-core path runs", kFp4ScaleMin, kFp4ScaleMax);
  } else {
    fail(MOE_OK, "shape without tensor-core tiles (need d_model %% 128 == 0, d_ff %% 64 == 0, d_ff_shared %% 64 == 0)");
  }
  return MOE_PATH_SIMT;
}

// ============================================================================================
// step entry points
// ============================================================================================
static moe_status check_ready(moe_plan* p, int T, bool need_ws) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T must be >= 0 (%d)", T);
  if (!p->weights_set) return fail(MOE_ERR_NOT_READY, "weights not set");
  if (p->n_shared > 0 && !p->shared_set) return fail(MOE_ERR_NOT_READY, "shared experts not set");
  if (need_ws) {
    if (!p->ws) return fail(MOE_ERR_NOT_READY, "workspace not set");
    if (T > p->T_max) return fail(MOE_ERR_WORKSPACE, "T=%d exceeds the workspace's T_max=%d", T, p->T_max);
  }
  return MOE_OK;
}

static FfnWeights ffn_weights(const moe_plan* p) {
  FfnWeights w;
  w.w_gu = p->w_gu;
  w.s_gu = p->s_gu;
  w.w_down = p->w_down;
  w.s_down = p->s_down;
  w.fp4 = p->wdtype == MOE_W_MXFP4;
  w.w_gu_s = p->w_gu_s;
  w.w_down_s = p->w_down_s;
  w.n_shared = p->n_shared;
  w.f_s = p->f_s;
  w.E = p->E;
  w.k = p->k;
  w.d = p->d;
  w.f = p->f;
  w.err = p->err;
  w.tiled = p->tiled ? 1 : 0;
  w.tiled_s = p->tiled_s ? 1 : 0;
  w.fp4_tiled = p->fp4_tiled ? 1 : 0;
  return w;
}

// Expert FFN over grouped rows; y/y_s outputs, h/h_s in the workspace.  For the tensor-core
// path `segs`/`n_segs` must already describe the routed segments.
// Weight tiles per unit of the 16-bit grouped GEMMs: 2 (the pair shares each token-row stage:
// half the activation traffic, and twice the weight bytes in flight per stage) unless that
// leaves fewer units than a quarter of the SMs, where single tiles double the parallelism.  The
// routed unit count is estimated from the number of segments, about min(E, T k) + T k / 128.
static int tc_pair(const moe_plan* p, int T, bool routed, bool gate_up) {
  const long tiles_r = gate_up ? p->f / 64 : p->d / 128;
  const long tiles_s = gate_up ? static_cast<long>(p->n_shared) * p->f_s / 64 : p->d / 128;
  const long R = static_cast<long>(T) * p->k;
  const long segs_r = routed ? std::min<long>(p->E, R) + R / kSegRowsMax : 0;
  const long segs_s = p->n_shared > 0 ? (T + kSegRowsMax - 1) / kSegRowsMax : 0;
  const long units2 = segs_r * ((tiles_r + 1) / 2) + segs_s * ((tiles_s + 1) / 2);
  return 4 * units2 >= p->num_sms ? 2 : 1;
}

// Arguments of the grouped tensor-core kernels for one step.
static TcArgs tc_args(const moe_plan* p, const uint16_t* x, int T, const int32_t* perm, uint16_t* y, uint16_t* y_s) {
  TcArgs a;
  a.w_gu = reinterpret_cast<const uint16_t*>(p->w_gu);
  a.w_gu_s = p->w_gu_s;
  a.w_down = reinterpret_cast<const uint16_t*>(p->w_down);
  a.w_down_s = p->w_down_s;
  a.segs = ws_ptr<Seg>(p, p->L.segs);
  a.n_segs = ws_ptr<int32_t>(p, p->L.n_segs);
  a.perm = perm;
  a.x = x;
  a.h = ws_ptr<uint16_t>(p, p->L.h);
  a.h_s = ws_ptr<uint16_t>(p, p->L.h_s);
  a.y = y;
  a.y_s = y_s;
  a.err = p->err;
  a.T = T;
  a.E = p->E;
  a.k = p->k;
  a.d = p->d;
  a.f = p->f;
  a.n_shared = p->n_shared;
  a.f_s = p->f_s;
  a.n_shared_segs = p->n_shared > 0 ? (T + kSegRowsMax - 1) / kSegRowsMax : 0;
  if (p->wdtype == MOE_W_MXFP4) {
    a.q_gu = p->w_gu;
    a.q_down = p->w_down;
    a.x16 = ws_ptr<uint16_t>(p, p->L.x16);
  }
  return a;
}

// The shared experts' arguments: the 16-bit kernels restricted to their units.
static TcArgs shared_args(const moe_plan* p, const TcArgs& a, int T, bool gate_up) {
  TcArgs sh = a;
  sh.routed = 0;
  sh.pair = tc_pair(p, T, false, gate_up);
  return sh;
}

// With 4-bit routed weights the shared experts run on their own launches.  Their gate/up
// depends on x alone, so when it fills at most half of the SMs it runs on the plan's second
// stream beside the router and the grouping (which leave most SMs idle at such T) instead of
// after them.  The shared down projection follows it there when kSharedDownBeside (it needs h_s
// alone; its blocks take the SMs the routed gate/up's last, partial round of units leaves idle,
// the side stream having the higher priority), and the caller's stream joins before the combine.
constexpr bool kSharedDownBeside = true;

static bool shared_gate_up_beside(const moe_plan* p, int T) {
  if (!use_tc(p) || p->wdtype != MOE_W_MXFP4 || p->n_shared == 0 || !p->side) return false;
  const long tiles = static_cast<long>(p->n_shared) * p->f_s / 64;
  const int pair = tc_pair(p, T, false, true);
  const long units = static_cast<long>((T + kSegRowsMax - 1) / kSegRowsMax) * ((tiles + pair - 1) / pair);
  return 2 * units <= p->num_sms;
}

// Fork the shared gate/up onto the side stream (after everything already queued on st).
static moe_status launch_shared_gate_up_beside(moe_plan* p, const uint16_t* x, int T, cudaStream_t st) {
  if (!p->maps_weights || !p->maps_ws) return fail(MOE_ERR_NOT_READY, "tensor maps not built");
  MOE_CUDA_TRY(cudaEventRecord(p->ev_fork, st));
  MOE_CUDA_TRY(cudaStreamWaitEvent(p->side, p->ev_fork, 0));
  const TcArgs sh = shared_args(p, tc_args(p, x, T, nullptr, nullptr, nullptr), T, true);
  LAUNCH(p, "tc_gateup_shared", p->side, launch_tc_gateup(&p->maps, sh, p->num_sms, p->side));
  if (kSharedDownBeside) {
    const TcArgs shd = shared_args(p, tc_args(p, x, T, nullptr, nullptr, ws_ptr<uint16_t>(p, p->L.y_s)), T, false);
    LAUNCH(p, "tc_down_shared", p->side, launch_tc_down(&p->maps, shd, p->num_sms, p->side));
  }
  MOE_CUDA_TRY(cudaEventRecord(p->ev_join, p->side));
  return MOE_OK;
}

// Expert FFN over grouped rows; y/y_s outputs, h/h_s in the workspace.  For the tensor-core
// path `segs`/`n_segs` must already describe the routed segments.  shared_forked: the shared
// expert was launched on the side stream (launch_shared_gate_up_beside); unless its down
// projection went there too, st joins the side stream before launching it.  x16_ready: the
// routing already wrote the 4-bit path's fp16 copy of x.
static moe_status run_experts(moe_plan* p, const uint16_t* x, int T, const int32_t* offsets, const int32_t* perm,
                              uint16_t* y, uint16_t* y_s, cudaStream_t st, bool shared_forked = false,
                              bool x16_ready = false) {
  if (use_tc(p)) {
    if (!p->maps_weights || !p->maps_ws) return fail(MOE_ERR_NOT_READY, "tensor maps not built");
    TcArgs a = tc_args(p, x, T, perm, y, y_s);
    if (p->wdtype == MOE_W_MXFP4) {
      // routed experts on the 4-bit kernels (fp16 activations), shared experts on the 16-bit
      // kernels restricted to their units
      uint16_t* x16 = ws_ptr<uint16_t>(p, p->L.x16);
      a.sched = p->err + kSchedFp4GateUp;
      if (p->fp4_mx) {
        a.xq = ws_ptr<uint8_t>(p, p->L.xq);
        a.xs = ws_ptr<uint8_t>(p, p->L.xs);
        LAUNCH(p, "x_to_mx", st, launch_x_to_mx(x, ws_ptr<uint8_t>(p, p->L.xq), ws_ptr<uint8_t>(p, p->L.xs), T, p->d, st));
        LAUNCH(p, "mx_gateup", st, launch_mx_gateup(a, p->num_sms, st));
      } else {
        if (!x16_ready)
          LAUNCH(p, "x_to_f16", st, launch_x_to_f16(x, x16, static_cast<size_t>(T) * p->d, p->err, st));
        LAUNCH(p, "fp4_gateup", st, launch_fp4_gateup(&p->maps, a, p->num_sms, st));
      }
      if (p->n_shared > 0 && !shared_forked) {
        const TcArgs sh = shared_args(p, a, T, true);
        LAUNCH(p, "tc_gateup_shared", st, launch_tc_gateup(&p->maps, sh, p->num_sms, st));
      }
      a.sched = p->err + kSchedFp4Down;
      if (p->fp4_mx_down) {
        const int R = T * p->k;
        uint8_t* hq = ws_ptr<uint8_t>(p, p->L.hq);
        uint8_t* hs = ws_ptr<uint8_t>(p, p->L.hs);
        LAUNCH(p, "h_to_mx", st, launch_h_to_mx(ws_ptr<uint16_t>(p, p->L.h), hq, hs, R, p->f, st));
        TcArgs ad = a;
        ad.xq = hq;
        ad.xs = hs;
        LAUNCH(p, "mx_down", st, launch_mx_down(ad, p->num_sms, st));
      } else {
        LAUNCH(p, "fp4_down", st, launch_fp4_down(&p->maps, a, p->num_sms, st));
      }
      if (p->n_shared > 0 && !(shared_forked && kSharedDownBeside)) {
        if (shared_forked) MOE_CUDA_TRY(cudaStreamWaitEvent(st, p->ev_join, 0));
        const TcArgs sh = shared_args(p, a, T, false);
        LAUNCH(p, "tc_down_shared", st, launch_tc_down(&p->maps, sh, p->num_sms, st));
      }
    } else {
      a.pair = tc_pair(p, T, true, true);
      LAUNCH(p, "tc_gateup", st, launch_tc_gateup(&p->maps, a, p->num_sms, st));
      a.pair = tc_pair(p, T, true, false);
      LAUNCH(p, "tc_down", st, launch_tc_down(&p->maps, a, p->num_sms, st));
    }
  } else {
    FfnWeights w = ffn_weights(p);
    uint16_t* h = ws_ptr<uint16_t>(p, p->L.h);
    uint16_t* h_s = ws_ptr<uint16_t>(p, p->L.h_s);
    LAUNCH(p, "simt_ffn", st, launch_ffn_simt(w, x, T, offsets, perm, h, h_s, y, y_s, st));
    p->launch_count += 1;  // the SIMT FFN is two kernels
  }
  return MOE_OK;
}

// Router logits as nsplit partial matrices [nsplit][T][E] for the top-k to add (in split order,
// plus *bias when not null).  T > kRouterTcMinT with a tensor-core-capable shape: the
// tensor-core router; T <= 128 and d % 128 == 0: the small-T K-split router; otherwise the
// CUDA-core router (bias included).
static moe_status router_step(moe_plan* p, const uint16_t* x, int T, const float** parts_out, int* nsplit,
                              const float** bias, cudaStream_t st) {
  float* parts = ws_ptr<float>(p, p->L.parts);
  if (p->router_tc && T > kRouterTcMinT) {
    const int ns = router_tc_splits(T, p->E, p->d, p->num_sms);
    moe_status s = make_map_16(&p->map_x, x, p->d, T, 128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    if (s != MOE_OK) return s;
    LAUNCH(p, "router_tc", st, launch_router_tc(&p->map_router3, &p->map_x, T, p->E, p->d, ns, parts, p->err, p->num_sms, st));
    *parts_out = parts, *nsplit = ns, *bias = p->b_router;
  } else if (T <= 128 && p->d % 128 == 0) {
    LAUNCH(p, "router_logits", st, launch_router_parts_small(x, p->w_router, T, p->E, p->d, parts, st));
    *parts_out = parts, *nsplit = router_small_splits(p->d), *bias = p->b_router;
  } else {
    float* lg = ws_ptr<float>(p, p->L.logits);
    LAUNCH(p, "router_logits", st, launch_router_logits(x, p->w_router, p->b_router, T, p->E, p->d, lg, st));
    *parts_out = lg, *nsplit = 1, *bias = nullptr;
  }
  return MOE_OK;
}

// The nsplit router_step will produce for T tokens.
static int router_nsplit(const moe_plan* p, int T) {
  if (p->router_tc && T > kRouterTcMinT) return router_tc_splits(T, p->E, p->d, p->num_sms);
  if (T <= 128 && p->d % 128 == 0) return router_small_splits(p->d);
  return 1;
}

// Router logits + top-k (+ masks).
static moe_status route_step(moe_plan* p, const uint16_t* x, int T, float* logits_out, int32_t* ids, float* gates,
                             uint32_t* masks, cudaStream_t st, const XConv& xc = XConv{}) {
  const float* parts = nullptr;
  const float* bias = nullptr;
  int ns = 1;
  moe_status s = router_step(p, x, T, &parts, &ns, &bias, st);
  if (s != MOE_OK) return s;
  LAUNCH(p, "topk", st, launch_topk(parts, ns, bias, logits_out, T, p->E, p->k, ids, gates, masks, p->err, st, xc));
  return MOE_OK;
}

// Device rows are read and written as 16-byte vectors (cp.async, TMA, uint4 stores).
static bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }

extern "C" moe_status moe_layer_forward(moe_plan* p, const void* x, int T, int n_prefill, void* out,
                                        moe_stream_t stream) {
  moe_status s = check_ready(p, T, true);
  if (s != MOE_OK) return s;
  if (n_prefill < 0 || n_prefill > T) return fail(MOE_ERR_INVALID_ARG, "n_prefill=%d outside [0, T=%d]", n_prefill, T);
  p->launch_count = 0;
  if (T == 0) return MOE_OK;
  if (!x || !out) return fail(MOE_ERR_INVALID_ARG, "x and out are required");
  if (!aligned16(x) || !aligned16(out)) return fail(MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  if (use_small_layer(p, T)) {
    LsArgs a;
    a.x = xb;
    a.w_router = p->w_router;
    a.b_router = p->b_router;
    a.w_gu = reinterpret_cast<const uint16_t*>(p->w_gu);
    a.w_down = reinterpret_cast<const uint16_t*>(p->w_down);
    a.w_gu_s = p->w_gu_s;
    a.w_down_s = p->w_down_s;
    a.logits = ws_ptr<float>(p, p->L.logits);
    a.ids = ws_ptr<int32_t>(p, p->L.ids);
    a.gates = ws_ptr<float>(p, p->L.gates);
    a.counts = ws_ptr<int32_t>(p, p->L.counts);
    a.offsets = ws_ptr<int32_t>(p, p->L.offsets);
    a.perm = ws_ptr<int32_t>(p, p->L.perm);
    a.inv = ws_ptr<int32_t>(p, p->L.inv);
    a.touched = ws_ptr<int32_t>(p, p->L.touched);
    a.n_touched = a.touched + p->E;
    a.h = ws_ptr<uint16_t>(p, p->L.h);
    a.h_s = ws_ptr<uint16_t>(p, p->L.h_s);
    a.y32 = ws_ptr<float>(p, p->L.y32);
    a.ys32 = a.y32 + static_cast<size_t>(T) * p->k * p->d;
    a.out = static_cast<uint16_t*>(out);
    a.sync = p->ls_sync;
    a.err = p->err;
    a.T = T, a.E = p->E, a.k = p->k, a.d = p->d, a.f = p->f, a.n_shared = p->n_shared, a.f_s = p->f_s;
    LAUNCH(p, "layer_small", st, launch_layer_small(a, p->num_sms, st));
    return MOE_OK;
  }
  int32_t* ids = ws_ptr<int32_t>(p, p->L.ids);
  float* gates = ws_ptr<float>(p, p->L.gates);
  uint32_t* masks = ws_ptr<uint32_t>(p, p->L.masks);
  int32_t* counts = ws_ptr<int32_t>(p, p->L.counts);
  int32_t* offsets = ws_ptr<int32_t>(p, p->L.offsets);
  int32_t* perm = ws_ptr<int32_t>(p, p->L.perm);
  int32_t* inv = ws_ptr<int32_t>(p, p->L.inv);
  uint16_t* y = ws_ptr<uint16_t>(p, p->L.y);
  uint16_t* y_s = p->n_shared > 0 ? ws_ptr<uint16_t>(p, p->L.y_s) : nullptr;
  const bool tc = use_tc(p);
  Seg* segs = tc ? ws_ptr<Seg>(p, p->L.segs) : nullptr;
  const bool forked = shared_gate_up_beside(p, T);
  if (forked && (s = launch_shared_gate_up_beside(p, xb, T, st)) != MOE_OK) return s;
  struct Join {  // an error return between the fork and the join still joins the side stream
    cudaStream_t st;
    cudaEvent_t ev;
    bool armed;
    ~Join() {
      if (armed) cudaStreamWaitEvent(st, ev, 0);
    }
  } join{st, p->ev_join, forked};
  // At T <= 64 the 4-bit path's fp16 copy of x is made on the side by the one routing launch
  // that precedes the expert kernels (every thread of its grid takes a share); above, the top-k
  // kernel would carry T·d conversions on few threads, so x_to_f16 keeps its own launch.
  XConv xc;
  if (tc && p->wdtype == MOE_W_MXFP4 && !p->fp4_mx) {
    xc.x = xb;
    xc.x16 = ws_ptr<uint16_t>(p, p->L.x16);
    xc.n8 = static_cast<size_t>(T) * p->d / 8;
  }
  if (router_nsplit(p, T) == router_small_splits(p->d) && !(p->router_tc && T > kRouterTcMinT) &&
      router_route_tiny_ok(T, p->E, p->d, p->k)) {
    // tiny step: router, top-k and grouping in one launch
    LAUNCH(p, "router_route", st,
           launch_router_route_tiny(xb, p->w_router, p->b_router, T, p->E, p->d, ws_ptr<float>(p, p->L.parts), p->k,
                                    ids, gates, counts, offsets, perm, inv, segs, ws_ptr<int32_t>(p, p->L.n_segs),
                                    p->L.max_segs, p->err + 1, p->err, st, xc));
  } else if (route_small_ok(T, p->E, p->k, router_nsplit(p, T))) {
    // small step: the whole routing and grouping in one block after the router
    const float* parts = nullptr;
    const float* bias = nullptr;
    int ns = 1;
    s = router_step(p, xb, T, &parts, &ns, &bias, st);
    if (s != MOE_OK) return s;
    LAUNCH(p, "route_small", st,
           launch_route_small(parts, ns, bias, T, p->E, p->k, ids, gates, counts, offsets, perm, inv, segs,
                              ws_ptr<int32_t>(p, p->L.n_segs), p->L.max_segs, p->err + 1, p->err, st, xc));
  } else {
    xc = XConv{};
    s = route_step(p, xb, T, nullptr, ids, gates, masks, st);
    if (s != MOE_OK) return s;
    LAUNCH(p, "group", st,
           launch_group(ids, masks, T, p->E, p->k, counts, offsets, perm, inv, segs, ws_ptr<int32_t>(p, p->L.n_segs),
                        p->L.max_segs, p->err, st));
  }
  s = run_experts(p, xb, T, offsets, perm, y, y_s, st, forked, xc.x16 != nullptr);
  if (s != MOE_OK) return s;
  if (forked && kSharedDownBeside) MOE_CUDA_TRY(cudaStreamWaitEvent(st, p->ev_join, 0));
  join.armed = false;  // joined (before the shared down projection or here)
  LAUNCH(p, "combine", st, launch_combine(y, gates, inv, y_s, T, p->k, p->d, static_cast<uint16_t*>(out), st));
  return MOE_OK;
}

extern "C" moe_status moe_route(moe_plan* p, const void* x, int T, float* logits, int32_t* ids, float* gates,
                                moe_stream_t stream) {
  moe_status s = check_ready(p, T, true);
  if (s != MOE_OK) return s;
  p->launch_count = 0;
  if (T == 0) return MOE_OK;
  if (!x || !ids || !gates) return fail(MOE_ERR_INVALID_ARG, "x, ids and gates are required");
  if (!aligned16(x)) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return route_step(p, static_cast<const uint16_t*>(x), T, logits, ids, gates, nullptr, st);
  return MOE_OK;
}

extern "C" moe_status moe_route_logits(moe_plan* p, const float* logits, int T, int32_t* ids, float* gates,
                                       moe_stream_t stream) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T must be >= 0");
  moe_status s = ensure_err_word(p);
  if (s != MOE_OK) return s;
  p->launch_count = 0;
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !gates) return fail(MOE_ERR_INVALID_ARG, "logits, ids and gates are required");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LAUNCH(p, "topk", st, launch_topk(logits, 1, nullptr, nullptr, T, p->E, p->k, ids, gates, nullptr, p->err, st));
  return MOE_OK;
}

extern "C" moe_status moe_permute(moe_plan* p, const int32_t* ids, int T, int32_t* counts, int32_t* offsets,
                                  int32_t* perm, int32_t* inv_perm, moe_stream_t stream) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T must be >= 0");
  if (!p->ws) return fail(MOE_ERR_NOT_READY, "workspace not set");
  if (T > p->T_max) return fail(MOE_ERR_WORKSPACE, "T=%d exceeds the workspace's T_max=%d", T, p->T_max);
  if (!counts || !offsets || (T > 0 && (!ids || !perm || !inv_perm)))
    return fail(MOE_ERR_INVALID_ARG, "ids, counts, offsets, perm and inv_perm are required (ids, perm, inv_perm "
                                     "may be NULL when T == 0)");
  moe_status s = ensure_err_word(p);
  if (s != MOE_OK) return s;
  p->launch_count = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* masks = ws_ptr<uint32_t>(p, p->L.masks);
  if (T > 0) LAUNCH(p, "masks_from_ids", st, launch_masks_from_ids(ids, T, p->E, p->k, masks, p->err, st));
  LAUNCH(p, "group", st,
         launch_group(ids, masks, T, p->E, p->k, counts, offsets, perm, inv_perm, nullptr, nullptr, 0, p->err, st));
  return MOE_OK;
}

extern "C" moe_status moe_experts(moe_plan* p, const void* x, int T, const int32_t* offsets, const int32_t* perm,
                                  void* y, void* shared_y, moe_stream_t stream) {
  moe_status s = check_ready(p, T, true);
  if (s != MOE_OK) return s;
  p->launch_count = 0;
  if (T == 0) return MOE_OK;
  if (!x || !offsets || !perm || !y) return fail(MOE_ERR_INVALID_ARG, "x, offsets, perm and y are required");
  if (p->n_shared > 0 && !shared_y) return fail(MOE_ERR_INVALID_ARG, "shared_y is required when n_shared > 0");
  if (!aligned16(x) || !aligned16(y) || (p->n_shared > 0 && !aligned16(shared_y)))
    return fail(MOE_ERR_INVALID_ARG, "x, y and shared_y must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (use_tc(p))
    LAUNCH(p, "segments", st,
           launch_segments_from_offsets(offsets, p->E, ws_ptr<Seg>(p, p->L.segs), ws_ptr<int32_t>(p, p->L.n_segs),
                                        p->L.max_segs, p->err, st));
  return run_experts(p, static_cast<const uint16_t*>(x), T, offsets, perm, static_cast<uint16_t*>(y),
                     p->n_shared > 0 ? static_cast<uint16_t*>(shared_y) : nullptr, st);
}

extern "C" moe_status moe_combine(moe_plan* p, const float* y, const float* gates, const int32_t* inv_perm,
                                  const float* shared_y, int T, void* out, moe_stream_t stream) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T must be >= 0");
  p->launch_count = 0;
  if (T == 0) return MOE_OK;
  if (!y || !gates || !inv_perm || !out) return fail(MOE_ERR_INVALID_ARG, "y, gates, inv_perm and out are required");
  if (p->d % 8) return fail(MOE_ERR_UNSUPPORTED, "moe_combine needs d_model %% 8 == 0");
  if (!aligned16(y) || !aligned16(out) || (shared_y && !aligned16(shared_y)))
    return fail(MOE_ERR_INVALID_ARG, "y, shared_y and out must be 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LAUNCH(p, "combine", st, launch_combine_f32(y, gates, inv_perm, shared_y, T, p->k, p->d, static_cast<uint16_t*>(out), st));
  return MOE_OK;
}

extern "C" moe_status moe_plan_get_device_error(moe_plan* p, uint32_t* code) {
  if (!p || !code) return fail(MOE_ERR_INVALID_ARG, "plan and code are required");
  *code = 0;
  MOE_CUDA_TRY(cudaDeviceSynchronize());
  if (!p->err) return MOE_OK;
  MOE_CUDA_TRY(cudaMemcpy(code, p->err, sizeof(uint32_t), cudaMemcpyDeviceToHost));
  MOE_CUDA_TRY(cudaMemset(p->err, 0, sizeof(uint32_t)));
  if (*code) return fail(MOE_ERR_DEVICE, "device error bits 0x%x", *code);
  return MOE_OK;
}

extern "C" moe_status moe_plan_enable_timing(moe_plan* p, int enable) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "plan is NULL");
  p->timing = enable != 0;
  return MOE_OK;
}

extern "C" size_t moe_plan_timing_report(moe_plan* p, char* buf, size_t len) {
  if (!p) return 0;
  std::map<std::string, std::pair<long, double>> agg;
  std::vector<std::string> order;
  for (auto& t : p->timed) {
    float ms = 0.f;
    cudaEventSynchronize(t.stop);
    cudaEventElapsedTime(&ms, t.start, t.stop);
    auto it = agg.find(t.name);
    if (it == agg.end()) {
      order.push_back(t.name);
      agg[t.name] = {1, ms};
    } else {
      it->second.first += 1;
      it->second.second += ms;
    }
    p->event_pool.push_back(t.start);
    p->event_pool.push_back(t.stop);
  }
  p->timed.clear();
  std::string rep;
  for (auto& n : order) {
    char line[256];
    snprintf(line, sizeof line, "%s %ld %.6f\n", n.c_str(), agg[n].first, agg[n].second);
    rep += line;
  }
  if (buf && len > 0) {
    const size_t n = rep.size() < len - 1 ? rep.size() : len - 1;
    memcpy(buf, rep.data(), n);
    buf[n] = '\0';
  }
  return rep.size() + 1;
}

extern "C" int moe_plan_last_launch_count(const moe_plan* p) { return p ? p->launch_count : 0; }
