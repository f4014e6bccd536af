// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// The grouped problem is a list of segments: consecutive grouped rows of one routed expert
// (at most 128), or consecutive tokens for the shared experts.  Each unit of work is one
// segment times a pair of 128-row tiles of that expert's weight matrix (two MMAs per K step
// share the segment's B stage, which halves the token-row traffic).  The MMA computes
//     D[weight row][token] = W[128 x K] . X[N x K]^T
// ("swap-AB": the weight tile is the M=128 operand, the segment's tokens are N <= 128), so the
// weights -- the bytes that bound this layer -- stream through shared memory exactly once per
// segment, whatever the number of rows routed to the expert.
//
//   gate/up kernel (bf16 x bf16): A = 128 interleaved rows of W_gate|W_up (8 gate rows, then
//     the same 8 features' up rows, repeated); B = the segment's token rows of x, gathered
//     with cp.async (the permutation is applied on the fly, x is never copied);
//     epilogue: h = fp16(silu(gate) * up), the gate-first SwiGLU of "Why SSD-streamed MoE was
//     slow: 8GB Jetson Orin Nano, part 2" (section re-checking part 1), rounded inside the
//     producer as in the Decode paragraph of "DeepSeek V4.1F Q4 with native DSpark MTP on M3
//     Ultra" (there in bf16; fp16 here keeps 3 more bits for the same bytes).
//   down kernel (fp16 x fp16): A = 128 rows of W_down (held as fp16 by the plan), B = the
//     segment's rows of h (TMA); epilogue writes y (fp16) in grouped row order for the combine.
//   Intermediates that leave the fp16 range are clamped and flag MOE_DEVERR_RANGE.
//   Weights are stored tile-contiguous and pre-swizzled (16 KB per 128 x 64 tile, a unit's K
//   loop consecutive), so each A stage is one bulk copy and a unit streams one run of HBM.
//
// Roles (persistent CTAs, one per SM, every role walks the same unit sequence):
//   warp 0      producer: A by bulk copy; B by TMA (down kernel)
//   warp 1      TMEM owner and MMA issuer
//   warps 2-9   epilogue (TMEM lanes 32*(warp%4) .. +31; the two warps of a lane quarter take
//               alternate 16-column chunks, so the epilogue keeps pace with 128-row segments)
//   warps 10-17 gate/up only: cp.async gather of the token rows, two warps per stage slot
// Producer and MMA loops run converged and issue under elect_one() (warp-uniform operands: an
// MMA issues in a few tens of cycles), and the MMA warp probes the next stage's barrier before
// issuing the current stage, so the barrier round trip hides behind the issue.
// Pipeline: 4 shared-memory stages of (2 x A 16 KB + B up to 16 KB); two TMEM accumulator pairs
// (2 x 2 x 128 fp32 columns, all 512) so the epilogue of one unit overlaps the main loop of the
// next.  An
// expert with more than 128 rows is split into parts; the units of its parts are ordered
// tile-major (tile 0 of every part, then tile 1, ...) so that CTAs working on the same
// weight tile run side by side and the second read of the tile is served by L2.
// The gather warps of a slot wait for their own copies and arrive themselves, so every stage
// of the ring can be in flight at once (a lagged arrive would leave only part of it).
// Every wait is bounded (see common.cuh); on a timeout the CTA stops issuing work, drains its
// MMAs, frees TMEM and returns with MOE_DEVERR_TIMEOUT set.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace tc {

constexpr int BM = 128;                          // weight rows per tile (MMA M)
constexpr int BK = 64;                           // K elements per stage (128-byte rows)
constexpr int kPair = 2;                         // weight tiles per unit (sharing the B stage)
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;             // 16 KB per tile
constexpr int kBBytes = kSegRowsMax * BK * 2;    // 16 KB (N <= 128)
constexpr int kStageBytes = kPair * kABytes + kBBytes;  // 48 KB
constexpr int kAccCols = kSegRowsMax;
constexpr int kTmemCols = 2 * kPair * kAccCols;  // 2 buffers x 2 tiles x 128 columns = 512
constexpr int kGatherPerSlot = 2;                // gate/up B producers per stage slot
constexpr int kGatherWarps = kGatherPerSlot * kStages;
constexpr int kTokBytes = kGatherWarps * kSegRowsMax * 4;  // per gather warp: token of each row
constexpr int kEpiStageBytes = 16 * 32 * 2;     // per epilogue warp: 16 columns x 32 fp16 rows
constexpr int kEpiWarps = 8;                     // two per TMEM lane quarter, alternate 16-column chunks
constexpr int kFirstGather = 2 + kEpiWarps;      // gate/up: first gather warp
constexpr int kBaseThreads = 32 * kFirstGather;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*barriers*/ + 1024 /*align slack*/ + kTokBytes +
                           kEpiWarps * kEpiStageBytes;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct Unit {
  int shared;     // 1: shared-expert segment
  int expert;     // routed expert (shared: -1)
  int row_start;  // grouped row (routed) or token (shared) of column 0
  int rows;       // valid columns
  int tile;       // first 128-row weight tile (even)
  int ntile;      // 1 or 2 tiles
};

MOE_DEVICE Seg load_seg(const Seg* p) {
  const int4 lo = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 hi = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  return Seg{lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
}

// A unit is one segment times a.pair (1 or 2) consecutive weight tiles (the last group of an
// odd tile count has one).  groups(tiles): tile groups of one weight matrix.
MOE_DEVICE int groups(int tiles, int pair) { return (tiles + pair - 1) / pair; }

template <bool kL2 = false>
MOE_DEVICE Unit decode_unit(int u, const TcArgs& a, int tiles_r, int tiles_s, int n_shared_units) {
  Unit un;
  if (u < n_shared_units) {
    const int pairs_s = groups(tiles_s, a.pair);
    const int ss = u / pairs_s;
    const int nss = a.n_shared_segs;
    const int q = a.T / nss, rem = a.T % nss;
    un.shared = 1;
    un.expert = -1;
    un.tile = a.pair * (u % pairs_s);
    un.ntile = min(a.pair, tiles_s - un.tile);
    un.row_start = ss * q + min(ss, rem);
    un.rows = q + (ss < rem ? 1 : 0);
  } else {
    // The parts [first, first + nparts) of one expert own units [first, first + nparts) * pairs;
    // inside that range the pair index is the slow one and the part the fast one.
    // kL2: read the segment records through L2 (the down kernel's producer reads them before
    // its grid-dependency wait, so nothing may come from a stale L1 line)
    const int pairs_r = groups(tiles_r, a.pair);
    const int v = u - n_shared_units;
    const Seg any = kL2 ? load_seg(a.segs + v / pairs_r) : a.segs[v / pairs_r];
    const int o = v - any.first * pairs_r;
    const Seg s = kL2 ? load_seg(a.segs + any.first + o % any.nparts) : a.segs[any.first + o % any.nparts];
    un.shared = 0;
    un.expert = s.expert;
    un.tile = a.pair * (o / any.nparts);
    un.ntile = min(a.pair, tiles_r - un.tile);
    un.row_start = s.row_start;
    un.rows = s.rows;
  }
  return un;
}

MOE_DEVICE int pad16(int rows) { return rows <= 16 ? 16 : ((rows + 15) & ~15); }

template <bool kGateUp>
__global__ void __launch_bounds__(kGateUp ? kBaseThreads + 32 * kGatherWarps : kBaseThreads, 1)
    tc_ffn_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* tok_tab = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + 1024);
  uint16_t* epi_stage = reinterpret_cast<uint16_t*>(smem + kStages * kStageBytes + 1024 + kTokBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], kGateUp ? 1 + kGatherPerSlot : 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0 && !kGateUp) {
    tma_prefetch_map(&maps.h);
    if (a.n_shared) tma_prefetch_map(&maps.h_s);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // gate/up lets its dependents start only once its own predecessors (the routing) are
  // complete, so the down kernel may read the unit list -- and stream its first weight stages
  // -- before its grid-dependency wait; everything that reads h waits.
  if (kGateUp) {
    pdl_wait();
    pdl_trigger();
  } else {
    pdl_trigger();
    if (warp != 0) pdl_wait();
  }

  const int tiles_r = kGateUp ? a.f / 64 : a.d / BM;
  const int tiles_s = kGateUp ? (a.n_shared * a.f_s) / 64 : a.d / BM;
  const int n_shared_units = a.n_shared ? a.n_shared_segs * groups(tiles_s, a.pair) : 0;
  const int n_routed_units = a.routed ? __ldcg(a.n_segs) * groups(tiles_r, a.pair) : 0;
  const int total_units = n_shared_units + n_routed_units;
  const int nk_r = kGateUp ? a.d / BK : a.f / BK;
  const int nk_s = kGateUp ? a.d / BK : (a.n_shared * a.f_s) / BK;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_act = l2_policy_evict_last();
    uint32_t pre = 0;  // down: stages whose weights were requested before the dependency wait
    if (!kGateUp) {
      for (int u = blockIdx.x; u < total_units && pre < static_cast<uint32_t>(kStages); u += gridDim.x) {
        const Unit un = decode_unit<true>(u, a, tiles_r, tiles_s, n_shared_units);
        const int nk = un.shared ? nk_s : nk_r;
        const int tiles_m = un.shared ? tiles_s : tiles_r;
        const uint16_t* mbase = un.shared ? a.w_down_s : a.w_down + static_cast<size_t>(un.expert) * tiles_r * nk * kTileElems;
        for (int kk = 0; kk < nk && pre < static_cast<uint32_t>(kStages); ++kk, ++pre) {
          if (elect_one()) {  // a fresh slot: no wait; the arrival comes with the h rows below
            mbar_expect_tx(&full[pre], un.ntile * kABytes);
            bulk_load(smem + pre * kStageBytes, mbase + tile_chunk_offset(un.tile, kk, tiles_m, nk), un.ntile * kABytes,
                      &full[pre], pol_w);
          }
          __syncwarp();
        }
      }
      pdl_wait();
    }
    uint32_t g = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
      const Unit un = decode_unit(u, a, tiles_r, tiles_s, n_shared_units);
      const int nk = un.shared ? nk_s : nk_r;
      const int nbox = kGateUp ? 0 : (pad16(un.rows) + 31) / 32;
      // the unit's weight matrix (an expert, or all shared experts); with the paired tile layout
      // both tiles of a pair unit at one K chunk are one contiguous 32 KB run
      const int tiles_m = un.shared ? tiles_s : tiles_r;
      const uint16_t* mbase =
          kGateUp ? (un.shared ? a.w_gu_s : a.w_gu + static_cast<size_t>(un.expert) * tiles_r * nk * kTileElems)
                  : (un.shared ? a.w_down_s : a.w_down + static_cast<size_t>(un.expert) * tiles_r * nk * kTileElems);
      const CUtensorMap* hm = un.shared ? &maps.h_s : &maps.h;
      for (int kk = 0; kk < nk; ++kk, ++g) {
        const int slot = g % kStages;
        if (!(ok = mbar_wait_warp(&empty[slot], ((g / kStages) & 1u) ^ 1u, abort_flag, a.err))) break;
        if (elect_one()) {
          uint8_t* sa = smem + slot * kStageBytes;
          const bool early = g < pre;  // weights already requested
          mbar_arrive_expect_tx(&full[slot], (early ? 0 : un.ntile * kABytes) + nbox * 32 * BK * 2);
          if (!early)
            bulk_load(sa, mbase + tile_chunk_offset(un.tile, kk, tiles_m, nk), un.ntile * kABytes, &full[slot], pol_w);
          if (!kGateUp)
            for (int i = 0; i < nbox; ++i)
              tma_load_2d(sa + kPair * kABytes + i * 32 * BK * 2, hm, &full[slot], kk * BK, un.row_start + 32 * i,
                          pol_act);
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: the warp waits, one elected lane issues ----------------
    uint32_t g = 0, j = 0;
    bool ok = true, ready = false;  // ready: full[g % kStages] already seen complete for stage g
    for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x, ++j) {
      const Unit un = decode_unit(u, a, tiles_r, tiles_s, n_shared_units);
      const int nk = un.shared ? nk_s : nk_r;
      const uint32_t N = static_cast<uint32_t>(pad16(un.rows));
      const uint32_t buf = j & 1u, use_acc = j >> 1;
      if (!(ok = mbar_wait_warp(&acc_empty[buf], (use_acc & 1u) ^ 1u, abort_flag, a.err))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + buf * (kPair * kAccCols);  // tile t: + t * kAccCols
      // gate/up: bf16 weights x bf16 tokens; down: fp16 weights x fp16 hidden vectors
      const uint32_t idesc = kGateUp ? idesc_bf16_f32(BM, N) : idesc_f16_f32(BM, N);
      for (int kk = 0; kk < nk; ++kk, ++g) {
        const int slot = g % kStages;
        if (!ready && !(ok = mbar_wait_warp(&full[slot], (g / kStages) & 1u, abort_flag, a.err))) break;
        const uint32_t gn = g + 1;  // probe the next stage now, use the answer next iteration
        const bool next = mbar_test(&full[gn % kStages], (gn / kStages) & 1u);
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + slot * kStageBytes);
        const uint64_t adesc0 = smem_desc_sw128(sa);
        const uint64_t adesc1 = smem_desc_sw128(sa + kABytes);
        const uint64_t bdesc = smem_desc_sw128(sa + kPair * kABytes);
        const bool two = un.ntile > 1;
        if (elect_one()) {
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {  // K = 16 per MMA: +32 bytes = +2 in the address field
            mma_f16_ss(d_tmem, adesc0 + 2 * ks, bdesc + 2 * ks, idesc, (kk | ks) != 0);
            if (two) mma_f16_ss(d_tmem + kAccCols, adesc1 + 2 * ks, bdesc + 2 * ks, idesc, (kk | ks) != 0);
          }
          mma_commit(&empty[slot]);
        }
        ready = __all_sync(0xffffffffu, next);
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&acc_full[buf]);
      __syncwarp();
    }
    // all MMAs issued by this warp have finished once `drain` completes
    if (elect_one()) mma_commit(drain);
    __syncwarp();
    mbar_wait_warp(drain, 0, nullptr, a.err);
  } else if (warp < kFirstGather) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // h and y are read back by the next launch: keep them in L2 ahead of the streamed weights
    const uint64_t pol_out = l2_policy_evict_last();
    uint32_t j = 0;
    for (int u = blockIdx.x; u < total_units && !*abort_flag; u += gridDim.x, ++j) {
      const Unit un = decode_unit(u, a, tiles_r, tiles_s, n_shared_units);
      const uint32_t buf = j & 1u, use_acc = j >> 1;
      if (!mbar_wait(&acc_full[buf], use_acc & 1u, abort_flag, a.err)) break;
      tc_fence_after();
      const int L = 32 * q + lane;  // accumulator row (= weight row of the tile)
      // Each 16-column chunk goes through a per-warp shared tile [column][row] so that the
      // global stores are 16-byte vectors of 8 consecutive features of one token.
      uint16_t* stg = epi_stage + (warp - 2) * (kEpiStageBytes / 2);
      const int c_first = 16 * ((warp - 2) / 4);  // this warp's 16-column chunks: c_first + 32 i
      bool sat = false;
      for (int t = 0; t < un.ntile; ++t) {
        const int tile = un.tile + t;
        const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + (buf * kPair + t) * kAccCols;
        if (kGateUp) {
          // lanes L and L ^ 8 hold the gate and up rows of one feature: each computes h for 8 of
          // the 16 columns (gate lane the even ones); the warp covers 16 consecutive features
          const int w16 = L & 15;
          const bool is_gate = w16 < 8;
          const int fl = 8 * ((L >> 4) & 1) + (w16 & 7);  // feature within the warp's 16
          const int feat0 = tile * 64 + 16 * q;
          uint16_t* hout;
          int ldh;
          if (un.shared) {
            hout = a.h_s;
            ldh = a.n_shared * a.f_s;
          } else {
            hout = a.h;
            ldh = a.f;
          }
          for (int c0 = c_first; c0 < un.rows; c0 += 32) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(tbase + c0, r);
            tmem_wait_ld();
  #pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const uint32_t send = is_gate ? r[2 * jj + 1] : r[2 * jj];
              const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 8);
              const int cl = 2 * jj + (is_gate ? 0 : 1);
              const float gv = __uint_as_float(is_gate ? r[2 * jj] : recv);
              const float uv = __uint_as_float(is_gate ? recv : r[2 * jj + 1]);
              float hv = swiglu(gv, uv);
              if (c0 + cl < un.rows && !(fabsf(hv) <= kF16Max)) {  // padding columns never count
                sat = true;
                hv = fminf(fmaxf(hv, -kF16Max), kF16Max);
              }
              stg[cl * 16 + fl] = f32_to_f16_bits_rn(hv);
            }
            __syncwarp();
            {  // lane i: column i / 2, features 8 (i % 2) .. + 7
              const int cl = lane >> 1, half = lane & 1;
              if (c0 + cl < un.rows) {
                const uint4 v = *reinterpret_cast<const uint4*>(stg + cl * 16 + 8 * half);
                st_global_v4_hint(hout + static_cast<size_t>(un.row_start + c0 + cl) * ldh + feat0 + 8 * half, v, pol_out);
              }
            }
            __syncwarp();
          }
        } else {
          const int feat0 = tile * BM + 32 * q;
          uint16_t* yout = un.shared ? a.y_s : a.y;
          for (int c0 = c_first; c0 < un.rows; c0 += 32) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(tbase + c0, r);
            tmem_wait_ld();
  #pragma unroll
            for (int c = 0; c < 16; ++c) {
              float v = __uint_as_float(r[c]);
              if (c0 + c < un.rows && !(fabsf(v) <= kF16Max)) {
                sat = true;
                v = fminf(fmaxf(v, -kF16Max), kF16Max);
              }
              stg[c * 32 + lane] = f32_to_f16_bits_rn(v);
            }
            __syncwarp();
  #pragma unroll
            for (int pass = 0; pass < 2; ++pass) {  // column (16 pass + lane) / 4, features 8 (lane % 4) .. + 7
              const int idx = 32 * pass + lane;
              const int cl = idx >> 2, g = idx & 3;
              if (c0 + cl < un.rows) {
                const uint4 v = *reinterpret_cast<const uint4*>(stg + cl * 32 + 8 * g);
                st_global_v4_hint(yout + static_cast<size_t>(un.row_start + c0 + cl) * a.d + feat0 + 8 * g, v, pol_out);
              }
            }
            __syncwarp();
          }
        }
      }  // tiles of the unit
      if (__any_sync(0xffffffffu, sat) && lane == 0) set_error(a.err, MOE_DEVERR_RANGE);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  } else if (kGateUp) {
    // ---------------- token-row gather (cp.async) ----------------
    // Warps w and w + kStages own stage slot w: they fill every stage g with g % kStages == w
    // (each half of the rows), wait for their own copies, fence them for the tensor core and
    // arrive.  8 consecutive lanes copy the 8 16-byte chunks of one row (a 128-byte line).
    const int gw = warp - kFirstGather;
    const int slot = gw % kStages, half = gw / kStages;
    int32_t* tok = tok_tab + kSegRowsMax * gw;  // token of each row of this warp's unit
    const int ch = lane & 7;
    const int rs = (lane >> 3) + 4 * half;      // first row; rows rs + 8 i
    const uint64_t pol_x = l2_policy_evict_last();  // each x row is gathered once per weight tile
    uint32_t g = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
      const Unit un = decode_unit(u, a, tiles_r, tiles_s, n_shared_units);
      const int nk = un.shared ? nk_s : nk_r;
      bool have_tok = false;
      for (int kk = 0; kk < nk; ++kk, ++g) {
        const int s = g % kStages;
        if (s != slot) continue;
        if (!have_tok) {
          for (int n = lane; n < un.rows; n += 32) tok[n] = un.shared ? un.row_start + n : a.perm[un.row_start + n] / a.k;
          __syncwarp();
          have_tok = true;
        }
        if (!(ok = mbar_wait_warp(&empty[s], ((g / kStages) & 1u) ^ 1u, abort_flag, a.err))) break;
        const uint32_t sb = smem_u32(smem + s * kStageBytes + kPair * kABytes);
        const int k0 = kk * BK + ch * 8;
        for (int n = rs; n < un.rows; n += 8)
          cp_async_16_hint(sb + n * 128 + ((ch ^ (n & 7)) << 4), a.x + static_cast<size_t>(tok[n]) * a.d + k0, pol_x);
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  abort_quiesce(abort_flag);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tc

template <bool kGateUp>
static cudaError_t launch_tc(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st) {
  auto kern = tc::tc_ffn_kernel<kGateUp>;
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), tc::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(num_sms), dim3(kGateUp ? tc::kBaseThreads + 32 * tc::kGatherWarps : tc::kBaseThreads),
                    tc::kSmemBytes, st,
                    *maps, a);
}

cudaError_t launch_tc_gateup(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st) {
  return launch_tc<true>(maps, a, num_sms, st);
}

cudaError_t launch_tc_down(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st) {
  return launch_tc<false>(maps, a, num_sms, st);
}

}  // namespace moe
