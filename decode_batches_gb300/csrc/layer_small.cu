// The whole MoE layer of a small step (at most 8 tokens) in ONE launch: router logits, top-k and
// grouping, the shared and routed experts' gate/up with SwiGLU, their down projections and the
// gate-weighted combine -- the GB300 counterpart of the single command buffer per layer of the
// Decode paragraph of "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra" (router and top-k
// merged into one dispatch, shared-expert gate+up+SwiGLU fused).
//
// At this T the layer is a weight stream: every touched expert's weights are read once and each
// weight meets at most T token rows.  Persistent CTAs (one per SM) of kWarps warps; each warp owns
// whole tasks -- 64 weight rows of one matrix over the whole K -- and streams their rows through
// its own ring of kSlots 8 KB shared-memory slots with one bulk copy per 64-K chunk (the 64 rows'
// 128-byte lines are contiguous in the tile-contiguous weight layout), kSlots - 1 pieces ahead of
// its arithmetic.  The arithmetic is mma.sync m16n8k16 (fp32 accumulate): 4 fragments of 16 rows
// x 8 token columns per warp, so no cross-warp reduction exists.  Tasks have equal sizes and are
// dealt round-robin over all the launch's warps (gate/up task i to warp i mod NW, down task j to
// warp NW - 1 - j mod NW, so warps with one gate/up task more get one down task less).
//
//   router  every CTA computes the logits of experts blockIdx.x, blockIdx.x + G, ... (full K, so
//           no partial sums).  Once every CTA's logits are written (a launch-wide counter), each
//           CTA selects the top k of every token (topk.cuh, the same selection as every other
//           front end; one warp per token) and warp 0 groups the assignments (counts, offsets,
//           the stable permutation, the touched experts) in shared memory: the same result in
//           every CTA, with no further hop.  Shared-expert gate/up tasks need no routing and
//           stream from the start.
//   gate/up task = one matrix (an expert, or the shared experts) x 64 interleaved rows (32
//           features: four groups of 8 gate rows and their 8 up rows): the m16n8k16 fragment puts
//           gate row g and up row g + 8 of a group in the same lane, so SwiGLU runs in registers
//           and h (fp16, as the tensor-core path rounds it) goes straight to the workspace.
//   down    task = one matrix x 64 output features; after every CTA's gate/up tasks are done (a
//           launch-wide counter, one addition per CTA) each CTA copies all of h into shared memory
//           once; y (fp32) goes to the workspace.
//   combine after every down task (one addition per CTA), out[t] = sum_j g[t,j] y[t,j] + y_s[t]
//           in fp32, slot order, one rounding to bf16, 8-column chunks spread over the CTAs.
// Every sum has a fixed order: the result does not depend on which CTA or warp did what.  Every
// wait is bounded (1 s); an expired wait sets MOE_DEVERR_TIMEOUT and the CTA stops.  The last CTA
// to leave resets the launch-wide counters for the next launch.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace ls {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kSlots = 4;                // per warp
constexpr int kRowsPerTask = 64;
constexpr int kRowBytes = 128;           // 64 bf16 / fp16 elements of one row in one K chunk
constexpr int kSlotBytes = kRowsPerTask * kRowBytes;  // 8 KB: the task's rows of one 64-K chunk
constexpr int kUnionBytes = kLsUnionBytes;
constexpr int kMaxR = 256;               // T * k
constexpr int kEMax = 1024;
constexpr int kSmemBytes = kWarps * kSlots * kSlotBytes + kUnionBytes + kWarps * kLsTMax * 4 /*red*/ +
                           (kEMax + 1) * 4 /*off*/ + 3 * kMaxR * 4 /*perm, gates, ids*/ + (kEMax + 1) * 4 /*touched*/ +
                           kWarps * kSlots * 8 /*barriers*/ + 64 /*flags*/ + 1024 /*alignment*/;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

enum Kind : int { kEnd = -1, kGuShared = 0, kGuRouted = 1, kDnShared = 2, kDnRouted = 3 };

// Launch-wide words (plan-owned, zero between launches; kLsSyncWords of them).
struct Sync {
  uint32_t router_done, gu_done, dn_done, exited, pad0, pad1, pad2, pad3;
};

struct Smem {
  uint8_t* ring;     // [kWarps][kSlots][8 KB], 1024-aligned
  uint16_t* uni;     // x (bf16 [T][d + 8]) during gate/up, then h (fp16) during down
  float* red;        // [kWarps][kLsTMax] (router logits)
  int32_t* off;      // [E + 1] offsets of the grouping (counts while it is built)
  int32_t* perm;     // [T k]
  float* gates;      // [T k]
  int32_t* ids;      // [T k]
  int32_t* touched;  // [E] touched experts, ascending; touched[E] = their number
  uint64_t* full;    // [kWarps][kSlots]
  volatile int* flags;  // [0] abort, [1] gate/up tasks done here, [2] down tasks done here,
                        // [4] routing ready, [5] h complete, [6] down complete
};

MOE_DEVICE Smem carve(uint8_t* raw) {
  Smem s;
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  s.ring = p;
  p += kWarps * kSlots * kSlotBytes;
  s.uni = reinterpret_cast<uint16_t*>(p);
  p += kUnionBytes;
  s.red = reinterpret_cast<float*>(p);
  p += kWarps * kLsTMax * 4;
  s.off = reinterpret_cast<int32_t*>(p);
  p += (kEMax + 1) * 4;
  s.perm = reinterpret_cast<int32_t*>(p);
  p += kMaxR * 4;
  s.gates = reinterpret_cast<float*>(p);
  p += kMaxR * 4;
  s.ids = reinterpret_cast<int32_t*>(p);
  p += kMaxR * 4;
  s.touched = reinterpret_cast<int32_t*>(p);
  p += (kEMax + 1) * 4;
  p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 7) & ~uintptr_t(7));
  s.full = reinterpret_cast<uint64_t*>(p);
  s.flags = reinterpret_cast<volatile int*>(s.full + kWarps * kSlots);
  return s;
}

// Barrier of the CTA's warps.
MOE_DEVICE void cta_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// The same barrier returning the AND of every thread's predicate.
MOE_DEVICE bool cta_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kThreads)
      : "memory");
  return r != 0;
}

MOE_DEVICE uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *p >= target (one thread).  false: gave up (MOE_DEVERR_TIMEOUT set).
MOE_DEVICE bool wait_counter(const uint32_t* p, uint32_t target, volatile int* abort_flag, uint32_t* err) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire(p) >= target) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > MOE_WAIT_LIMIT_NS) {
      set_error(err, MOE_DEVERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// Warp-level tensor-core fragments (mma.sync m16n8k16, fp32 accumulate): 16 weight rows x 16 K
// (A, row-major in the slot) times 16 K x 8 tokens (B, token rows of x or h).  At this T the MMA
// replaces a few CUDA-core instructions per weight; the weights still stream once.
MOE_DEVICE void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
MOE_DEVICE void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
template <bool kBf16>
MOE_DEVICE void mma_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  if (kBf16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Bounded wait until the shared-memory flag is set (one thread).
MOE_DEVICE bool wait_flag(volatile int* flag, volatile int* abort_flag, uint32_t* err) {
  if (*flag) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (*flag) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > MOE_WAIT_LIMIT_NS) {
      set_error(err, MOE_DEVERR_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
  }
}

// Top k and gates of token t by one warp, from the logits every CTA wrote (read through L2), into
// the shared-memory ids / gates.
template <int PL>
MOE_DEVICE void select_token(const LsArgs& a, int t, int32_t* ids, float* gates) {
  const int lane = threadIdx.x & 31;
  float v[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < a.E ? __ldcg(a.logits + static_cast<size_t>(t) * a.E + e) : 0.f;
  }
  topk_select<PL>(v, t, a.E, a.k, ids, gates, a.err);
}

// The grouping of the step by one warp (warp 0), into shared memory, from the selected ids:
// counts -> offsets, the stable permutation (rows of an expert ascend by assignment index) and
// the touched experts in ascending order.  Returns the number of touched experts.
MOE_DEVICE int group_step(const LsArgs& a, const Smem& S) {
  const int lane = threadIdx.x & 31;
  const int E = a.E, R = a.T * a.k;
  int32_t* cnt = S.off;  // counts first, then turned into offsets
  for (int e = lane; e <= E; e += 32) cnt[e] = 0;
  __syncwarp();
  for (int q = lane; q < R; q += 32) atomicAdd(&cnt[S.ids[q]], 1);
  __syncwarp();
  int run = 0, trun = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    const int c = e < E ? cnt[e] : 0;
    const unsigned used = __ballot_sync(0xffffffffu, c > 0);
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += up;
    }
    if (e < E) {
      if (c > 0) S.touched[trun + __popc(used & ((1u << lane) - 1u))] = e;
      cnt[e] = run + inc - c;  // the exclusive offset
    }
    run += __shfl_sync(0xffffffffu, inc, 31);
    trun += __popc(used);
  }
  if (lane == 0) {
    cnt[E] = run;
    S.touched[E] = trun;
  }
  __syncwarp();
  for (int q = lane; q < R; q += 32) {
    const int e = S.ids[q];
    int r = cnt[e];
    for (int q2 = 0; q2 < q; ++q2) r += S.ids[q2] == e ? 1 : 0;
    S.perm[r] = q;
  }
  __syncwarp();
  return trun;
}

__global__ void __launch_bounds__(kThreads, 1) layer_small_kernel(const LsArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem S = carve(smem_raw);
  Sync* sy = reinterpret_cast<Sync*>(a.sync);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, k = a.k, d = a.d, f = a.f;
  const int R = T * k;
  const int G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  const int NW = G * kWarps, W = b * kWarps + warp;        // warps of the launch, this one
  const int fs_all = a.n_shared * a.f_s;                   // shared experts' hidden width, concatenated
  const int n_gu_s = fs_all / 32;                          // shared gate/up tasks (they come first)
  const int nk_gu = d / 64;                                // K chunks of a gate/up row
  uint64_t* full = S.full + warp * kSlots;
  uint8_t* ring = S.ring + warp * kSlots * kSlotBytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWarps * kSlots; ++i) mbar_init(&S.full[i], 1);
    for (int i = 0; i < 8; ++i) S.flags[i] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  volatile int* abort_flag = S.flags;
  const uint64_t pol = l2_policy_evict_first();
  bool ok = true;
  int n_touched = -1;

  // ---- the warp's task sequence ----
  struct Task {
    int kind, m, blk, nk;  // blk: 64-row block of the matrix
  };
  struct Seq {
    int gu_i, dn_i, kc;    // next gate/up / down task of this warp, K chunk within the current one
    Task cur;
  };
  auto task_at = [&](Seq& q) -> int {  // the next task into q.cur; 1 a task, 0 none, -1 routing unknown
    if (q.gu_i < n_gu_s) {
      q.cur = Task{kGuShared, -1, q.gu_i, nk_gu};
      q.gu_i += NW;
      return 1;
    }
    if (n_touched < 0) return -1;
    const int n_gu = n_gu_s + n_touched * (f / 32);
    const int nmat = n_touched + (a.n_shared > 0 ? 1 : 0);
    if (q.gu_i < n_gu) {
      const int v = q.gu_i - n_gu_s;
      q.cur = Task{kGuRouted, S.touched[v / (f / 32)], v % (f / 32), nk_gu};
      q.gu_i += NW;
      return 1;
    }
    if (q.dn_i < nmat * (d / 64)) {
      const int g = q.dn_i / nmat, mi = q.dn_i % nmat;  // feature-block major
      if (a.n_shared > 0 && mi == 0)
        q.cur = Task{kDnShared, -1, g, fs_all / 64};
      else
        q.cur = Task{kDnRouted, S.touched[mi - (a.n_shared > 0 ? 1 : 0)], g, f / 64};
      q.dn_i += NW;
      return 1;
    }
    q.cur = Task{kEnd, -1, 0, 0};
    return 0;
  };
  auto advance = [&](Seq& q) -> int {  // 1 a piece, 0 the end, -1 routing unknown (q unchanged)
    if (q.cur.kind == kEnd) return 0;
    if (q.kc >= 0 && q.kc + 1 < q.cur.nk) {
      ++q.kc;
      return 1;
    }
    Seq save = q;
    const int r = task_at(q);
    if (r < 0) {
      q = save;
      return -1;
    }
    q.kc = 0;
    return r;
  };
  // piece (task t, K chunk kc) into slot sl: one 8 KB bulk copy of the task's 64 rows
  auto issue = [&](const Task& t, int kc, int sl) {
    if (t.kind == kEnd) return;
    const bool gu = t.kind == kGuShared || t.kind == kGuRouted;
    int tiles;
    const uint16_t* base;
    if (gu) {
      tiles = (t.kind == kGuShared ? fs_all : f) / 64;
      base = t.kind == kGuShared ? a.w_gu_s : a.w_gu + static_cast<size_t>(t.m) * tiles * t.nk * kTileElems;
    } else {
      tiles = d / 128;
      base = t.kind == kDnShared ? a.w_down_s : a.w_down + static_cast<size_t>(t.m) * tiles * t.nk * kTileElems;
    }
    const uint16_t* src =
        base + tile_chunk_offset(t.blk / 2, kc, tiles, t.nk) + static_cast<size_t>(kRowsPerTask * (t.blk % 2)) * 64;
    if (elect_one()) {
      mbar_arrive_expect_tx(&full[sl], kSlotBytes);
      bulk_load(ring + sl * kSlotBytes, src, kSlotBytes, &full[sl], pol);
    }
    __syncwarp();
  };

  // ---- x into shared memory (rows padded by 16 bytes against ldmatrix bank conflicts) ----
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.x);
    for (int i = threadIdx.x; i < T * d / 8; i += kThreads) {
      const int t = i / (d / 8), c = i % (d / 8);
      reinterpret_cast<uint4*>(S.uni + static_cast<size_t>(t) * (d + 8))[c] = __ldg(src + i);
    }
  }
  // the first pieces that need no routing stream while the logits are computed
  Seq iq{W, (NW - 1) - W, -1, Task{kGuShared, -1, 0, 0}};  // issue cursor
  int issued = 0;
  Task pend_t[kSlots];
  int pend_kc[kSlots];
  while (issued < kSlots) {
    const int r = advance(iq);
    if (r < 0) break;
    pend_t[issued % kSlots] = iq.cur;
    pend_kc[issued % kSlots] = iq.kc;
    issue(iq.cur, iq.kc, issued % kSlots);
    ++issued;
    if (r == 0) break;
  }
  cta_sync();
  // ---- router logits of this CTA's experts (full K: no partial sums) ----
  {
    const int ks = d / kWarps;  // K slice per warp (a multiple of 32)
    for (int e = b; e < E; e += G) {
      float acc[kLsTMax];
#pragma unroll
      for (int t = 0; t < kLsTMax; ++t) acc[t] = 0.f;
      const float* wr = a.w_router + static_cast<size_t>(e) * d + warp * ks;
      for (int i = lane * 4; i < ks; i += 128) {
        const float4 w4 = __ldg(reinterpret_cast<const float4*>(wr + i));
#pragma unroll
        for (int t = 0; t < kLsTMax; ++t) {
          if (t < T) {
            const uint2 xv = *reinterpret_cast<const uint2*>(S.uni + static_cast<size_t>(t) * (d + 8) + warp * ks + i);
            acc[t] = fmaf(w4.x, __uint_as_float(xv.x << 16), acc[t]);
            acc[t] = fmaf(w4.y, __uint_as_float(xv.x & 0xFFFF0000u), acc[t]);
            acc[t] = fmaf(w4.z, __uint_as_float(xv.y << 16), acc[t]);
            acc[t] = fmaf(w4.w, __uint_as_float(xv.y & 0xFFFF0000u), acc[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kLsTMax; ++t) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
        if (lane == 0) S.red[warp * kLsTMax + t] = acc[t];
      }
      cta_sync();
      if (threadIdx.x < T) {
        float v = 0.f;
        for (int w = 0; w < kWarps; ++w) v += S.red[w * kLsTMax + threadIdx.x];
        if (a.b_router) v += a.b_router[e];
        a.logits[static_cast<size_t>(threadIdx.x) * E + e] = v;
      }
      cta_sync();
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&sy->router_done, 1u);
  }
  // ---- every CTA's logits written: top k of every token (a warp per token), grouping by warp 0 ----
  if (threadIdx.x == 0) S.flags[4] = wait_counter(&sy->router_done, static_cast<uint32_t>(G), abort_flag, a.err) ? 1 : 0;
  cta_sync();
  ok = S.flags[4] != 0;
  if (ok) {
    ld_acquire(&sy->router_done);  // every thread's own acquire of the logits
    for (int t = warp; t < T; t += kWarps) {
      if (E <= 256)
        select_token<8>(a, t, S.ids, S.gates);
      else if (E <= 512)
        select_token<16>(a, t, S.ids, S.gates);
      else
        select_token<32>(a, t, S.ids, S.gates);
    }
    cta_sync();
    if (warp == 0) group_step(a, S);
    cta_sync();
    n_touched = S.touched[E];
  }
  // ---- the rest of the prologue, now that routed tasks are known ----
  while (ok && issued < kSlots && iq.cur.kind != kEnd) {
    const int r = advance(iq);
    pend_t[issued % kSlots] = iq.cur;
    pend_kc[issued % kSlots] = iq.kc;
    issue(iq.cur, iq.kc, issued % kSlots);
    ++issued;
    if (r == 0) break;
  }
  const int hr_ld = f + 8, hs_ld = fs_all + 8;             // h row strides in shared memory (padded)
  uint16_t* h_r = S.uni;                                   // routed h rows [R][f + 8]
  uint16_t* h_s = S.uni + static_cast<size_t>(R) * hr_ld;  // shared h rows [T][n_s f_s + 8]
  float dacc[4][4];   // 4 fragments (rows 16 j .. 16 j + 15) x 8 token columns
  int brow = 0;       // per task: the x row (gate/up) or h row (down) of token lane % 8
  int n_tok = 0, r0 = 0;
  bool gu_done_here = false;  // this warp has passed the gate/up -> down barrier
  // The gate/up -> down barrier of the CTA: every warp passes it exactly once (before its first
  // down piece, or at its end), whatever its state, so that no warp waits for another forever.
  // Then the CTA's gate/up count goes out, every CTA's is awaited, and all of h comes into shared
  // memory (x is no longer needed).
  auto gate_up_barrier = [&](bool ok_in) -> bool {
    gu_done_here = true;
    if (!cta_all(ok_in)) return false;
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(&sy->gu_done, static_cast<uint32_t>(S.flags[1]));
      const uint32_t n_gu = static_cast<uint32_t>(n_gu_s + n_touched * (f / 32));
      S.flags[5] = wait_counter(&sy->gu_done, n_gu, abort_flag, a.err) ? 1 : 0;
    }
    cta_sync();
    if (!S.flags[5]) return false;
    __threadfence();
    const uint4* src_r = reinterpret_cast<const uint4*>(a.h);
    for (int i = threadIdx.x; i < R * f / 8; i += kThreads)
      reinterpret_cast<uint4*>(h_r + static_cast<size_t>(i / (f / 8)) * hr_ld)[i % (f / 8)] = __ldcg(src_r + i);
    const uint4* src_s = reinterpret_cast<const uint4*>(a.h_s);
    for (int i = threadIdx.x; i < T * fs_all / 8; i += kThreads)
      reinterpret_cast<uint4*>(h_s + static_cast<size_t>(i / (fs_all / 8)) * hs_ld)[i % (fs_all / 8)] =
          __ldcg(src_s + i);
    cta_sync();
    return true;
  };
  for (int p = 0; ok && p < issued; ++p) {
    const int sl = p % kSlots;
    const Task t = pend_t[sl];
    const int kc = pend_kc[sl];
    if (t.kind == kEnd) break;
    const bool gu = t.kind == kGuShared || t.kind == kGuRouted;
    const bool routed = t.kind == kGuRouted || t.kind == kDnRouted;
    if (!gu && !gu_done_here) {
      ok = gate_up_barrier(true);
      if (!ok) break;
    }
    if (!(ok = mbar_wait_warp(&full[sl], static_cast<uint32_t>(p / kSlots) & 1u, abort_flag, a.err))) break;
    if (kc == 0) {  // a new task: its tokens, and fresh accumulators
      const int n = lane & 7;  // the B row (token) whose address this lane gives ldmatrix
      if (routed) {
        r0 = S.off[t.m];
        n_tok = S.off[t.m + 1] - r0;
        const int nn = n < n_tok ? n : 0;  // columns past the task's tokens repeat its first (ignored)
        brow = gu ? S.perm[r0 + nn] / k : r0 + nn;
      } else {
        n_tok = T;
        brow = n < T ? n : 0;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) dacc[j][0] = dacc[j][1] = dacc[j][2] = dacc[j][3] = 0.f;
    }
    // ---- 64 rows x 64 K on the tensor core: 4 K steps x 4 row fragments (m16n8k16) ----
    {
      const uint32_t slot_a = smem_u32(ring + sl * kSlotBytes);
      // A: lane i gives row (i % 8) + 8 ((i / 8) % 2) of the fragment, K half i / 16; rows keep the
      // weight layout's 16-byte chunk swizzle (chunk c of row r at c ^ (r % 8))
      const int ar = (lane & 7) + 8 * ((lane >> 3) & 1), ah = lane >> 4;
      // B: lane i (< 16) gives token row i % 8, K half i / 8
      const uint16_t* bb = gu ? S.uni + static_cast<size_t>(brow) * (d + 8)
                              : (t.kind == kDnRouted ? h_r + static_cast<size_t>(brow) * hr_ld
                                                     : h_s + static_cast<size_t>(brow) * hs_ld);
      const uint32_t b_addr = smem_u32(bb + kc * 64 + 8 * ((lane >> 3) & 1));
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t bf[2];
        ldsm_x2(b_addr + ks * 32, bf);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t af[4];
          ldsm_x4(slot_a + (16 * j + ar) * kRowBytes + ((((2 * ks + ah) ^ (ar & 7))) << 4), af);
          if (gu)
            mma_16816<true>(dacc[j], af, bf);
          else
            mma_16816<false>(dacc[j], af, bf);
        }
      }
    }
    __syncwarp();  // every lane is done with the slot: refill it with the piece kSlots ahead
    if (iq.cur.kind != kEnd) {
      advance(iq);  // the routing is known by now: never blocks
      pend_t[issued % kSlots] = iq.cur;
      pend_kc[issued % kSlots] = iq.kc;
      issue(iq.cur, iq.kc, issued % kSlots);
      ++issued;
    }
    if (kc + 1 < t.nk) continue;
    // ---- end of the task, inside the warp: lane (g, c) holds rows g and g + 8 of each fragment,
    // token columns 2c and 2c + 1 ----
    const int g = lane >> 2, tc = 2 * (lane & 3);
    if (gu) {
      // fragment j = interleave group 4 blk + j: rows g (gate) and g + 8 (up) of feature 8 (4 blk + j) + g
      bool sat = false;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int feat = 8 * (4 * t.blk + j) + g;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int tk = tc + c;
          if (tk < n_tok) {
            float hv = swiglu(dacc[j][c], dacc[j][2 + c]);
            if (!(fabsf(hv) <= kF16Max)) {
              sat = true;
              hv = fminf(fmaxf(hv, -kF16Max), kF16Max);
            }
            if (t.kind == kGuRouted)
              a.h[static_cast<size_t>(r0 + tk) * f + feat] = f32_to_f16_bits_rn(hv);
            else
              a.h_s[static_cast<size_t>(tk) * fs_all + feat] = f32_to_f16_bits_rn(hv);
          }
        }
      }
      if (sat) set_error(a.err, MOE_DEVERR_RANGE);
      __syncwarp();
      if (lane == 0) atomicAdd(const_cast<int*>(&S.flags[1]), 1);
    } else {
      // output features 64 blk + 16 j + g and + 8 of tokens tc, tc + 1
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int feat = 64 * t.blk + 16 * j + g;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int tk = tc + c;
          if (tk < n_tok) {
            float* yr = t.kind == kDnRouted ? a.y32 + static_cast<size_t>(S.perm[r0 + tk]) * d
                                            : a.ys32 + static_cast<size_t>(tk) * d;
            yr[feat] = dacc[j][c];
            yr[feat + 8] = dacc[j][2 + c];
          }
        }
      }
      __syncwarp();
      if (lane == 0) atomicAdd(const_cast<int*>(&S.flags[2]), 1);
    }
  }
  // a warp without down pieces (or one that stopped) passes the gate/up barrier here
  if (!gu_done_here) ok = gate_up_barrier(ok);
  ok = cta_all(ok);
  // ---- every CTA's down tasks done (one addition per CTA), then this CTA's share of the combine ----
  if (ok) {
    if (threadIdx.x == 0) {
      __threadfence();
      if (S.flags[2]) atomicAdd(&sy->dn_done, static_cast<uint32_t>(S.flags[2]));
      const uint32_t nmat = static_cast<uint32_t>(n_touched) + (a.n_shared > 0 ? 1u : 0u);
      S.flags[6] = wait_counter(&sy->dn_done, nmat * static_cast<uint32_t>(d / 64), abort_flag, a.err) ? 1 : 0;
    }
    cta_sync();
    ok = S.flags[6] != 0;
  }
  if (ok) {
    // out[t][8c .. 8c + 7] for the 8-column chunks c of this CTA: slot order, then the shared term
    __threadfence();
    const int n8 = T * d / 8;
    for (int c = b + G * static_cast<int>(threadIdx.x); c < n8; c += G * kThreads) {
      const int t = (8 * c) / d, j = (8 * c) % d;
      float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int sl = 0; sl < k; ++sl) {
        const float gt = S.gates[t * k + sl];
        const float4* yp = reinterpret_cast<const float4*>(a.y32 + static_cast<size_t>(t * k + sl) * d + j);
        const float4 y0 = __ldcg(yp), y1 = __ldcg(yp + 1);
        o[0] = fmaf(gt, y0.x, o[0]), o[1] = fmaf(gt, y0.y, o[1]), o[2] = fmaf(gt, y0.z, o[2]);
        o[3] = fmaf(gt, y0.w, o[3]), o[4] = fmaf(gt, y1.x, o[4]), o[5] = fmaf(gt, y1.y, o[5]);
        o[6] = fmaf(gt, y1.z, o[6]), o[7] = fmaf(gt, y1.w, o[7]);
      }
      if (a.n_shared > 0) {
        const float4* sp = reinterpret_cast<const float4*>(a.ys32 + static_cast<size_t>(t) * d + j);
        const float4 s0 = __ldcg(sp), s1 = __ldcg(sp + 1);
        o[0] += s0.x, o[1] += s0.y, o[2] += s0.z, o[3] += s0.w;
        o[4] += s1.x, o[5] += s1.y, o[6] += s1.z, o[7] += s1.w;
      }
      uint4 v;
      v.x = pack_bf16x2(o[0], o[1]);
      v.y = pack_bf16x2(o[2], o[3]);
      v.z = pack_bf16x2(o[4], o[5]);
      v.w = pack_bf16x2(o[6], o[7]);
      *reinterpret_cast<uint4*>(a.out + static_cast<size_t>(t) * d + j) = v;
    }
  }
  if (!ok) *abort_flag = 1;

  // ---- leave: CTA 0 leaves the routing in the workspace; the last CTA out resets the counters ----
  __syncthreads();
  if (b == 0 && n_touched >= 0) {
    for (int q = threadIdx.x; q < R; q += kThreads) {
      a.ids[q] = S.ids[q];
      a.gates[q] = S.gates[q];
      a.perm[q] = S.perm[q];
      a.inv[S.perm[q]] = q;
    }
    for (int e = threadIdx.x; e <= E; e += kThreads) {
      a.offsets[e] = S.off[e];
      if (e < E) a.counts[e] = S.off[e + 1] - S.off[e];
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&sy->exited, 1u) == gridDim.x - 1) {
      sy->router_done = 0u;
      sy->gu_done = 0u;
      sy->dn_done = 0u;
      sy->exited = 0u;
      __threadfence();
    }
  }
  abort_quiesce(abort_flag);  // bulk copies of a stopped warp land before the CTA exits
}

}  // namespace ls

bool layer_small_ok(int T, int E, int k, int d, int f, int n_shared, int f_s) {
  if (T < 1 || T > kLsTMax || E > ls::kEMax || T * k > ls::kMaxR) return false;
  if (d % 128 || f % 64 || (n_shared > 0 && (n_shared * f_s) % 64)) return false;
  const size_t x_bytes = static_cast<size_t>(T) * (d + 8) * 2;  // rows padded by 16 bytes
  const size_t h_bytes = (static_cast<size_t>(T) * k * (f + 8) + static_cast<size_t>(T) * (n_shared * f_s + 8)) * 2;
  return x_bytes <= ls::kUnionBytes && h_bytes <= ls::kUnionBytes;
}

cudaError_t launch_layer_small(const LsArgs& a, int num_sms, cudaStream_t st) {
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(ls::layer_small_kernel), ls::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(ls::layer_small_kernel, dim3(num_sms), dim3(ls::kThreads), ls::kSmemBytes, st, a);
}

}  // namespace moe
