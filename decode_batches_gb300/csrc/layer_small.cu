// The whole MoE layer of a small step (at most 8 tokens) in ONE launch: router logits, top-k and
// grouping, the shared and routed experts' gate/up with SwiGLU, their down projections and the
// gate-weighted combine -- the GB300 counterpart of the single command buffer per layer of the
// Decode paragraph of "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra" (router and top-k
// merged into one dispatch, shared-expert gate+up+SwiGLU fused).
//
// At this T the layer is a weight stream: every touched expert's weights are read once and each
// weight meets at most T token rows, so the tensor cores have nothing to do.  This kernel streams
// the weights through shared memory with bulk copies and multiplies on the CUDA cores (fp32
// accumulation), the weight-streaming GEMV of the small-T regime.
//
// Persistent CTAs, one per SM.  Warp 0 is the producer: it takes tasks from two launch-wide
// counters (gate/up tasks first, then down tasks) and streams each task's weight rows into a
// ring of kSlots shared-memory slots (one 32 KB piece per slot; bulk copies of whole 128-byte
// rows of the tile-contiguous weight layout).  Warps 1..16 consume the pieces in ring order.
//
//   router  every CTA computes the logits of experts blockIdx.x, blockIdx.x + gridDim.x, ...
//           (full K, so no partial sums); the last CTA to finish selects the top k of each token
//           (topk.cuh, the same selection as every other front end), groups the assignments
//           (counts, offsets, the stable permutation) and raises the routed flag.
//   gate/up task = one matrix (an expert, or the shared experts) x 8 features: its 16
//           interleaved rows (8 gate, 8 up) over the whole K; consumer warp w takes K chunk w of
//           each 16-chunk piece, the 16 warps' partial sums are added in warp order, SwiGLU, h
//           rounded to fp16 (as the tensor-core path does) into the workspace.
//   down    task = one matrix x 32 output features (32 rows of W_d over the whole K); after every
//           gate/up task is done (a launch-wide counter) each CTA copies all of h into shared
//           memory once; y (fp32) goes to the workspace.  The last down task of a 32-feature
//           group (a per-group counter) combines those features of every token:
//           out[t] = sum_j g[t,j] y[t,j] + y_s[t] in fp32, slot order, one rounding to bf16.
// Shared-expert gate/up tasks come first and need no routing, so they stream while the router
// finishes.  Every sum has a fixed order: the result does not depend on which CTA did what.
// Every wait is bounded (1 s); an expired wait sets MOE_DEVERR_TIMEOUT and the CTA stops.  The
// last CTA to leave resets the launch-wide counters for the next launch.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace ls {

constexpr int kConsumerWarps = 16;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kSlots = 4;
constexpr int kSlotBytes = 32 * 1024;   // one piece: 16 rows x 16 K chunks (gate/up), 32 x 8 (down)
constexpr int kRowBytes = 128;          // 64 bf16 / fp16 elements of one row in one K chunk
constexpr int kUnionBytes = kLsUnionBytes;
constexpr int kMaxR = 256;              // T * k
constexpr int kEMax = 1024;
constexpr int kSmemBytes = kSlots * kSlotBytes + kUnionBytes + kConsumerWarps * 16 * kLsTMax * 4 /*red*/ +
                           32 * kLsTMax * 4 /*sums*/ + (kEMax + 1) * 4 + 2 * kMaxR * 4 + (kEMax + 1) * 4 /*touched*/ +
                           1024 /*barriers, descriptors, flags*/;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

enum Kind : int { kEnd = -1, kGuShared = 0, kGuRouted = 1, kDnShared = 2, kDnRouted = 3 };

struct Piece {
  int kind;      // Kind
  int m;         // routed expert (kinds 1, 3), else -1
  int group;     // 8-feature group (gate/up) or 32-feature group (down)
  int kc0, nkc;  // K chunks of this piece
  int last;      // 1 on the task's last piece
  int pad0, pad1;
};

// Launch-wide words (plan-owned, zero between launches): see kLsSyncWords.
struct Sync {
  uint32_t gu_next, dn_next, router_done, routed, gu_done, exited, pad0, pad1;
  uint32_t fg_done[1];  // [d / 32]
};

struct Smem {
  uint8_t* ring;
  uint16_t* uni;  // x (bf16 [T][d]) during gate/up, then h (fp16) during down
  float* red;     // [kConsumerWarps][16][kLsTMax]
  float* sums;    // [32][kLsTMax]
  int32_t* off;   // [E + 1]
  int32_t* perm;  // [T k]
  float* gates;   // [T k]
  int32_t* touched;  // producer's copy: [E] (+ count in touched[E])
  uint64_t* full;
  uint64_t* empty;
  Piece* desc;
  volatile int* flags;  // [0] abort, [3] last router CTA, [4] routing published, [5] h complete,
                        // [6] last task of a down group (each written by one thread, read after a barrier)
};

MOE_DEVICE Smem carve(uint8_t* base) {
  Smem s;
  uint8_t* p = base;
  s.ring = p;
  p += kSlots * kSlotBytes;
  s.uni = reinterpret_cast<uint16_t*>(p);
  p += kUnionBytes;
  s.red = reinterpret_cast<float*>(p);
  p += kConsumerWarps * 16 * kLsTMax * 4;
  s.sums = reinterpret_cast<float*>(p);
  p += 32 * kLsTMax * 4;
  s.off = reinterpret_cast<int32_t*>(p);
  p += (kEMax + 1) * 4;
  s.perm = reinterpret_cast<int32_t*>(p);
  p += kMaxR * 4;
  s.gates = reinterpret_cast<float*>(p);
  p += kMaxR * 4;
  s.touched = reinterpret_cast<int32_t*>(p);
  p += (kEMax + 1) * 4;
  s.full = reinterpret_cast<uint64_t*>(p);
  s.empty = s.full + kSlots;
  s.desc = reinterpret_cast<Piece*>(s.empty + kSlots);
  s.flags = reinterpret_cast<volatile int*>(s.desc + kSlots);
  return s;
}

// Named barrier of the consumer warps only (the producer never joins it).
MOE_DEVICE void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

// The same barrier returning the AND of every consumer thread's predicate.
MOE_DEVICE bool consumers_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kConsumers)
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

// dot of 8 bf16 weights with 8 bf16 activations, accumulated into acc
MOE_DEVICE float dot8_bf16(const uint4& w, const uint4& x, float acc) {
  float wf[8], xf[8];
  bf16x8_to_f32(w, wf);
  bf16x8_to_f32(x, xf);
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf(wf[i], xf[i], acc);
  return acc;
}
MOE_DEVICE float dot8_f16(const uint4& w, const uint4& h, float acc) {
  float wf[8], hf[8];
  f16x8_to_f32(w, wf);
  f16x8_to_f32(h, hf);
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf(wf[i], hf[i], acc);
  return acc;
}

// Top k and gates of token t by one warp, from the logits the CTAs wrote (read through L2).
template <int PL>
MOE_DEVICE void select_token(const LsArgs& a, int t) {
  const int lane = threadIdx.x & 31;
  float v[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < a.E ? __ldcg(a.logits + static_cast<size_t>(t) * a.E + e) : 0.f;
  }
  topk_select<PL>(v, t, a.E, a.k, a.ids, a.gates, a.err);
}

__global__ void __launch_bounds__(kThreads, 1) layer_small_kernel(const LsArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Smem S = carve(smem_raw);
  Sync* sy = reinterpret_cast<Sync*>(a.sync);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, k = a.k, d = a.d, f = a.f;
  const int R = T * k;
  const int fs_all = a.n_shared * a.f_s;                     // shared experts' hidden width, concatenated
  const int n_gu_s = fs_all / 8;                             // shared gate/up tasks
  const int nk_gu = d / 64;                                  // K chunks of a gate/up row
  const int n_dn_groups = d / 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    for (int i = 0; i < 8; ++i) S.flags[i] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  volatile int* abort_flag = S.flags;

  if (warp == 0) {
    // ================================ producer ================================
    const uint64_t pol = l2_policy_evict_first();
    int n_touched = -1;  // known once the routing is published
    bool gu_phase = true, ok = true;
    uint32_t slot = 0, phase = 0;
    while (ok) {
      // ---- next task ----
      int kind = kEnd, m = -1, group = 0;
      if (gu_phase) {
        uint32_t id = 0;
        if (lane == 0) id = atomicAdd(&sy->gu_next, 1u);
        id = __shfl_sync(0xffffffffu, id, 0);
        if (static_cast<int>(id) < n_gu_s) {
          kind = kGuShared, group = static_cast<int>(id);
        } else {
          if (n_touched < 0) {
            bool okw = true;
            if (lane == 0) okw = wait_counter(&sy->routed, 1u, abort_flag, a.err);
            if (!__shfl_sync(0xffffffffu, okw, 0)) break;
            ld_acquire(&sy->routed);  // every lane's own acquire of the published routing
            n_touched = static_cast<int>(__ldcg(a.n_touched));
            for (int i = lane; i < n_touched; i += 32) S.touched[i] = __ldcg(a.touched + i);
            __syncwarp();
          }
          const int v = static_cast<int>(id) - n_gu_s;
          if (v < n_touched * (f / 8)) {
            kind = kGuRouted, m = S.touched[v / (f / 8)], group = v % (f / 8);
          } else {
            gu_phase = false;
          }
        }
      }
      if (!gu_phase) {
        if (n_touched < 0) {  // no gate/up task reached the routed ones: wait for the routing here
          bool okw = true;
          if (lane == 0) okw = wait_counter(&sy->routed, 1u, abort_flag, a.err);
          if (!__shfl_sync(0xffffffffu, okw, 0)) break;
          ld_acquire(&sy->routed);
          n_touched = static_cast<int>(__ldcg(a.n_touched));
          for (int i = lane; i < n_touched; i += 32) S.touched[i] = __ldcg(a.touched + i);
          __syncwarp();
        }
        const int nmat = n_touched + (a.n_shared > 0 ? 1 : 0);
        uint32_t id = 0;
        if (lane == 0) id = atomicAdd(&sy->dn_next, 1u);
        id = __shfl_sync(0xffffffffu, id, 0);
        if (static_cast<int>(id) < nmat * n_dn_groups) {
          group = static_cast<int>(id) / nmat;  // feature-group major: groups complete one by one
          const int mi = static_cast<int>(id) % nmat;
          if (a.n_shared > 0 && mi == 0) {
            kind = kDnShared;
          } else {
            kind = kDnRouted, m = S.touched[mi - (a.n_shared > 0 ? 1 : 0)];
          }
        }
      }
      // ---- its pieces ----
      const bool gu = kind == kGuShared || kind == kGuRouted;
      int nk = 1, tiles = 1, tile = 0, r0 = 0, rows = 0;
      const uint16_t* base = nullptr;
      if (kind == kGuShared || kind == kGuRouted) {
        tiles = (kind == kGuShared ? fs_all : f) / 64;
        nk = nk_gu;
        tile = group / 8, r0 = 16 * (group % 8), rows = 16;
        base = kind == kGuShared ? a.w_gu_s : a.w_gu + static_cast<size_t>(m) * tiles * nk * kTileElems;
      } else if (kind == kDnShared || kind == kDnRouted) {
        tiles = d / 128;
        nk = (kind == kDnShared ? fs_all : f) / 64;
        tile = group / 4, r0 = 32 * (group % 4), rows = 32;
        base = kind == kDnShared ? a.w_down_s : a.w_down + static_cast<size_t>(m) * tiles * nk * kTileElems;
      }
      const int per_piece = gu ? 16 : 8;  // K chunks per 32 KB piece
      const int npieces = kind == kEnd ? 1 : (nk + per_piece - 1) / per_piece;
      for (int pc = 0; pc < npieces; ++pc) {
        if (!(ok = mbar_wait_warp(&S.empty[slot], phase ^ 1u, abort_flag, a.err))) break;
        const int kc0 = pc * per_piece;
        const int nkc = kind == kEnd ? 0 : min(per_piece, nk - kc0);
        if (lane == 0) {
          S.desc[slot] = Piece{kind, m, group, kc0, nkc, pc == npieces - 1 ? 1 : 0, 0, 0};
          mbar_arrive_expect_tx(&S.full[slot], static_cast<uint32_t>(nkc * rows * kRowBytes));
        }
        __syncwarp();
        if (lane < nkc) {  // one bulk copy per K chunk: `rows` consecutive 128-byte rows
          const uint16_t* src = base + tile_chunk_offset(tile, kc0 + lane, tiles, nk) + static_cast<size_t>(r0) * 64;
          bulk_load(S.ring + slot * kSlotBytes + lane * rows * kRowBytes, src, rows * kRowBytes, &S.full[slot], pol);
        }
        __syncwarp();
        if (++slot == kSlots) slot = 0, phase ^= 1u;
      }
      if (kind == kEnd) break;
    }
    if (!ok || *abort_flag) {
      // wake the consumers so that they see the abort (their waits also give up on the flag)
      *abort_flag = 1;
    }
  } else {
    // ================================ consumers ================================
    const int cw = warp - 1;              // consumer warp 0..15
    const int ct = threadIdx.x - 32;      // consumer thread 0..511
    bool ok = true;
    // ---- x into shared memory ----
    {
      const uint4* src = reinterpret_cast<const uint4*>(a.x);
      uint4* dst = reinterpret_cast<uint4*>(S.uni);
      for (int i = ct; i < T * d / 8; i += kConsumers) dst[i] = __ldg(src + i);
    }
    consumers_sync();
    // ---- router logits of this CTA's experts (full K: no partial sums) ----
    {
      const int ks = d / kConsumerWarps;  // K slice per warp (a multiple of 8)
      for (int e = blockIdx.x; e < E; e += gridDim.x) {
        float acc[kLsTMax];
#pragma unroll
        for (int t = 0; t < kLsTMax; ++t) acc[t] = 0.f;
        const float* wr = a.w_router + static_cast<size_t>(e) * d + cw * ks;
        for (int i = lane * 4; i < ks; i += 128) {
          const float4 w4 = __ldg(reinterpret_cast<const float4*>(wr + i));
#pragma unroll
          for (int t = 0; t < kLsTMax; ++t) {
            if (t < T) {
              const uint16_t* xr = S.uni + static_cast<size_t>(t) * d + cw * ks + i;
              const uint2 xv = *reinterpret_cast<const uint2*>(xr);
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
          if (lane == 0) S.red[cw * kLsTMax + t] = acc[t];
        }
        consumers_sync();
        if (ct < T) {
          float v = 0.f;
          for (int w = 0; w < kConsumerWarps; ++w) v += S.red[w * kLsTMax + ct];
          if (a.b_router) v += a.b_router[e];
          a.logits[static_cast<size_t>(ct) * E + e] = v;
        }
        consumers_sync();
      }
    }
    // ---- the last CTA to finish its logits routes and groups the step ----
    if (ct == 0) {
      __threadfence();
      const uint32_t prev = atomicAdd(&sy->router_done, 1u);
      S.flags[3] = prev == gridDim.x - 1 ? 1 : 0;
    }
    consumers_sync();
    if (S.flags[3]) {
      __threadfence();
      int32_t* cnt = S.off;  // counts first, then turned into offsets
      for (int e = ct; e <= E; e += kConsumers) cnt[e] = 0;
      consumers_sync();
      for (int t = cw; t < T; t += kConsumerWarps) {  // one warp per token: logits -> top k + gates
        if (E <= 256)
          select_token<8>(a, t);
        else if (E <= 512)
          select_token<16>(a, t);
        else
          select_token<32>(a, t);
      }
      __threadfence_block();
      consumers_sync();
      // counts (order-independent), then offsets, the stable permutation and the touched list
      for (int q = ct; q < R; q += kConsumers) {
        S.perm[q] = a.ids[q];
        atomicAdd(&cnt[a.ids[q]], 1);
      }
      consumers_sync();
      if (cw == 0) {  // one warp scans E counts: exclusive offsets and touched-expert positions
        int run = 0, trun = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
          const int e = e0 + lane;
          const int c = e < E ? cnt[e] : 0;
          int inc = c;
          const unsigned used = __ballot_sync(0xffffffffu, c > 0);
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int up = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += up;
          }
          if (e < E) {
            a.counts[e] = c;
            const int ex = run + inc - c;
            if (c > 0) a.touched[trun + __popc(used & ((1u << lane) - 1u))] = e;
            cnt[e] = ex;  // now the exclusive offset
          }
          run += __shfl_sync(0xffffffffu, inc, 31);
          trun += __popc(used);
        }
        if (lane == 0) {
          cnt[E] = run;
          *a.n_touched = trun;
        }
      }
      consumers_sync();
      for (int e = ct; e <= E; e += kConsumers) a.offsets[e] = cnt[e];
      for (int q = ct; q < R; q += kConsumers) {  // row of assignment q: stable by assignment index
        const int e = S.perm[q];
        int r = cnt[e];
        for (int q2 = 0; q2 < q; ++q2) r += S.perm[q2] == e ? 1 : 0;
        a.perm[r] = q;
        a.inv[q] = r;
      }
      __threadfence();
      consumers_sync();
      if (ct == 0) {
        __threadfence();
        atomicExch(&sy->routed, 1u);
      }
    }
    // ---- pieces ----
    float acc[4][kLsTMax];
    int tok[kLsTMax];  // per task: x row (gate/up) or h row (down) of each of its tokens
    int n_tok = 0;
    bool routing = false, h_loaded = false;
    uint32_t slot = 0, phase = 0;
    const int hr_ld = f, hs_ld = fs_all;                   // h row strides in shared memory
    uint16_t* h_r = S.uni;                                 // routed h rows [R][f]
    uint16_t* h_s = S.uni + static_cast<size_t>(R) * f;    // shared h rows [T][n_s f_s]
    while (ok) {
      // every consumer warp waits for the piece, then all agree (a warp whose wait gave up still
      // reaches this barrier, so no consumer is left waiting at a later one)
      ok = consumers_all(mbar_wait_warp(&S.full[slot], phase, abort_flag, a.err));
      if (!ok) break;
      const Piece pc = S.desc[slot];
      if (pc.kind == kEnd) break;
      const bool gu = pc.kind == kGuShared || pc.kind == kGuRouted;
      const bool routed = pc.kind == kGuRouted || pc.kind == kDnRouted;
      if ((routed || !gu) && !routing) {
        // the routing: offsets, permutation and gates into shared memory (once)
        if (ct == 0) S.flags[4] = wait_counter(&sy->routed, 1u, abort_flag, a.err) ? 1 : 0;
        consumers_sync();
        if (!S.flags[4]) {
          ok = false;
          break;
        }
        for (int e = ct; e <= E; e += kConsumers) S.off[e] = __ldcg(a.offsets + e);
        for (int q = ct; q < R; q += kConsumers) {
          S.perm[q] = __ldcg(a.perm + q);
          S.gates[q] = __ldcg(a.gates + q);
        }
        consumers_sync();
        routing = true;
      }
      if (!gu && !h_loaded) {
        // every gate/up task of the launch is done: all of h into shared memory (x is no longer needed)
        if (ct == 0) {
          const uint32_t n_gu = static_cast<uint32_t>(n_gu_s + static_cast<int>(__ldcg(a.n_touched)) * (f / 8));
          S.flags[5] = wait_counter(&sy->gu_done, n_gu, abort_flag, a.err) ? 1 : 0;
        }
        consumers_sync();
        if (!S.flags[5]) {
          ok = false;
          break;
        }
        __threadfence();
        const uint4* src_r = reinterpret_cast<const uint4*>(a.h);
        uint4* dst_r = reinterpret_cast<uint4*>(h_r);
        for (int i = ct; i < R * f / 8; i += kConsumers) dst_r[i] = __ldcg(src_r + i);
        const uint4* src_s = reinterpret_cast<const uint4*>(a.h_s);
        uint4* dst_s = reinterpret_cast<uint4*>(h_s);
        for (int i = ct; i < T * fs_all / 8; i += kConsumers) dst_s[i] = __ldcg(src_s + i);
        consumers_sync();
        h_loaded = true;
      }
      if (pc.kc0 == 0) {  // a new task: its tokens, and fresh accumulators
        if (routed) {
          const int r0 = S.off[pc.m];
          n_tok = S.off[pc.m + 1] - r0;
#pragma unroll
          for (int t = 0; t < kLsTMax; ++t) tok[t] = t < n_tok ? (gu ? S.perm[r0 + t] / k : r0 + t) : 0;
        } else {
          n_tok = T;
#pragma unroll
          for (int t = 0; t < kLsTMax; ++t) tok[t] = t;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int t = 0; t < kLsTMax; ++t) acc[i][t] = 0.f;
      }
      // ---- this warp's K chunk of the piece: 16 rows x 128 bytes, 4 vectors per lane ----
      const int rows = gu ? 16 : 32;
      const int kci = gu ? cw : (cw & 7);           // K chunk within the piece
      const int rb = gu ? 0 : 16 * (cw >> 3);       // first row of this warp's 16
      if (kci < pc.nkc) {
        const int kc = pc.kc0 + kci;
        const uint8_t* base = S.ring + slot * kSlotBytes + kci * rows * kRowBytes;
        const int p = lane & 7;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rho = rb + (lane >> 3) + 4 * i;            // row within the task's rows
          const uint4 w = *reinterpret_cast<const uint4*>(base + rho * kRowBytes + p * 16);
          const int c = p ^ (rho & 7);                          // logical 8-element chunk of the row
          const int k0 = kc * 64 + c * 8;
          if (gu) {
#pragma unroll
            for (int t = 0; t < kLsTMax; ++t)
              if (t < n_tok)
                acc[i][t] = dot8_bf16(w, *reinterpret_cast<const uint4*>(S.uni + static_cast<size_t>(tok[t]) * d + k0),
                                      acc[i][t]);
          } else {
            const uint16_t* hb = pc.kind == kDnRouted ? h_r : h_s;
            const int ld = pc.kind == kDnRouted ? hr_ld : hs_ld;
#pragma unroll
            for (int t = 0; t < kLsTMax; ++t)
              if (t < n_tok)
                acc[i][t] = dot8_f16(w, *reinterpret_cast<const uint4*>(hb + static_cast<size_t>(tok[t]) * ld + k0),
                                     acc[i][t]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      if (++slot == kSlots) slot = 0, phase ^= 1u;
      if (!pc.last) continue;
      // ---- end of task: add the 8 lanes of each row, then the warps in K order ----
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int t = 0; t < kLsTMax; ++t) {
          float v = acc[i][t];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          if ((lane & 7) == 0) S.red[(cw * 16 + (lane >> 3) + 4 * i) * kLsTMax + t] = v;
        }
      consumers_sync();
      if (gu) {
        if (ct < 16 * kLsTMax) {  // (row, token): the 16 warps' partial sums in K order
          const int rho = ct / kLsTMax, t = ct % kLsTMax;
          float v = 0.f;
          for (int w = 0; w < kConsumerWarps; ++w) v += S.red[(w * 16 + rho) * kLsTMax + t];
          S.sums[rho * kLsTMax + t] = v;
        }
        consumers_sync();
        if (ct < 8 * kLsTMax) {  // rows i (gate) and 8 + i (up) of feature 8 group + i
          const int i = ct / kLsTMax, t = ct % kLsTMax;
          if (t < n_tok) {
            float hv = swiglu(S.sums[i * kLsTMax + t], S.sums[(8 + i) * kLsTMax + t]);
            if (!(fabsf(hv) <= kF16Max)) {
              set_error(a.err, MOE_DEVERR_RANGE);
              hv = fminf(fmaxf(hv, -kF16Max), kF16Max);
            }
            const int feat = 8 * pc.group + i;
            if (pc.kind == kGuRouted)
              a.h[static_cast<size_t>(S.off[pc.m] + t) * f + feat] = f32_to_f16_bits_rn(hv);
            else
              a.h_s[static_cast<size_t>(t) * fs_all + feat] = f32_to_f16_bits_rn(hv);
          }
        }
        consumers_sync();
        if (ct == 0) {
          __threadfence();
          atomicAdd(&sy->gu_done, 1u);
        }
      } else {
        if (ct < 32 * kLsTMax) {  // (row, token): the 8 warps of the row's half in K order
          const int rho = ct / kLsTMax, t = ct % kLsTMax;
          const int half = rho >> 4;
          float v = 0.f;
          for (int w = 0; w < 8; ++w) v += S.red[((8 * half + w) * 16 + (rho & 15)) * kLsTMax + t];
          if (t < n_tok) {
            const int feat = 32 * pc.group + rho;
            if (pc.kind == kDnRouted)
              a.y32[static_cast<size_t>(S.perm[S.off[pc.m] + t]) * d + feat] = v;
            else
              a.ys32[static_cast<size_t>(t) * d + feat] = v;
          }
        }
        consumers_sync();
        if (ct == 0) {
          __threadfence();
          const uint32_t nmat = static_cast<uint32_t>(__ldcg(a.n_touched)) + (a.n_shared > 0 ? 1u : 0u);
          S.flags[6] = atomicAdd(&sy->fg_done[pc.group], 1u) == nmat - 1 ? 1 : 0;
        }
        consumers_sync();
        if (S.flags[6]) {  // the group's last task: combine its 32 features of every token
          __threadfence();
          if (ct < 32 * T) {
            const int t = ct / 32, j = 32 * pc.group + (ct & 31);
            float o = 0.f;
            for (int s = 0; s < k; ++s)
              o = fmaf(S.gates[t * k + s], __ldcg(a.y32 + static_cast<size_t>(t * k + s) * d + j), o);
            if (a.n_shared > 0) o += __ldcg(a.ys32 + static_cast<size_t>(t) * d + j);
            a.out[static_cast<size_t>(t) * d + j] = f32_to_bf16_bits_rn(o);
          }
        }
      }
    }
    if (!ok) *abort_flag = 1;
  }

  // ---- leave; the last CTA out resets the launch-wide words ----
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&sy->exited, 1u) == gridDim.x - 1) {
      sy->gu_next = 0u;
      sy->dn_next = 0u;
      sy->router_done = 0u;
      sy->routed = 0u;
      sy->gu_done = 0u;
      for (int g = 0; g < n_dn_groups; ++g) sy->fg_done[g] = 0u;
      sy->exited = 0u;
      __threadfence();
    }
  }
  abort_quiesce(abort_flag);
}

}  // namespace ls

bool layer_small_ok(int T, int E, int k, int d, int f, int n_shared, int f_s) {
  if (T < 1 || T > kLsTMax || E > ls::kEMax || T * k > ls::kMaxR) return false;
  if (d % 128 || f % 64 || (n_shared > 0 && (n_shared * f_s) % 64)) return false;
  const size_t x_bytes = static_cast<size_t>(T) * d * 2;
  const size_t h_bytes = (static_cast<size_t>(T) * k * f + static_cast<size_t>(T) * n_shared * f_s) * 2;
  return x_bytes <= ls::kUnionBytes && h_bytes <= ls::kUnionBytes && d / 32 <= kLsMaxGroups;
}

cudaError_t launch_layer_small(const LsArgs& a, int num_sms, cudaStream_t st) {
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(ls::layer_small_kernel), ls::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(ls::layer_small_kernel, dim3(num_sms), dim3(ls::kThreads), ls::kSmemBytes, st, a);
}

}  // namespace moe
