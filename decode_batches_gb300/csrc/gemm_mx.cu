// Grouped gate/up projection with block-scaled 4-bit weights on the block-scaled tensor-core MMA
// (tcgen05.mma kind::mxf8f6f4.block_scale, sm_103a): the weights' e2m1 codes and e8m0 scales go
// to the tensor core as they are stored, no dequantisation.
//
// Source: "moe-prefill-quantum", hardware-check paragraph (MXFP4 unpack x scale x accumulate is the
// operation that must run at bandwidth) and "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra",
// DSpark paragraph (verify rows are bound by weight bytes per committed token).
//
// The activation operand must be 8-bit for this MMA (the e2m1 x e2m1 form would round x to 4
// bits).  One e4m3 rounding of x costs 2^-4 relative per element -- far above the layer's error
// budget -- so x is split in two e4m3 terms with their own e8m0 block scales (32 consecutive K):
//     x = hi + lo,  hi = s1 * e4m3(x / s1),  lo = s2 * e4m3((x - hi) / s2),
// and both terms go through the MMA as two rows of the B operand (row 2n = hi, 2n + 1 = lo of the
// unit's n-th token); the epilogue adds the two accumulator columns.  The split is exact to about
// 2^-8 of the residual, i.e. ~2^-12 of x: the measured layer error stays ~0.005 RMS (bound 0.06).
//
// Operands per 128-deep K stage (swap-AB as everywhere: 128 weight rows as M):
//   A  128 rows x 128 bytes, 128-byte swizzled K-major: the e2m1 codes, 16 per 16-byte chunk in its
//      low 8 bytes (the MMA's layout of 4-bit elements), expanded from the raw 4-bit blocks by one
//      warp quartet (one warp per TMEM lane quarter), which also writes the scale factors;
//   B  up to 128 rows (64 tokens x hi/lo) x 128 bytes of e4m3, gathered with cp.async;
//   scale factors in TMEM, 8 columns per stage after the two accumulators: SFA (row m of A at lane
//      m, column + m / 32, one byte per 32-K block) and SFB (row n of B at column 4 + n / 32 and
//      lane n % 32 of EVERY lane quarter) -- the layout the MMA reads, established by a probe.
//   4 MMAs of K = 32 per stage, the byte of each block picked by the scale-factor ids.
// A unit is (segment, 128-row weight tile, half): a segment of up to 128 rows is worked in halves
// of up to 64 tokens (N = 2 x rows <= 128), so both accumulators (2 x 128 columns) and the scale
// factors fit the 512 TMEM columns.  Units are handed out at run time as in gemm_fp4.cu; a half
// without rows is skipped by the producer and never published.
//
// Roles: warp 0 raw producer + unit hand-out; warp 1 TMEM owner and MMA issuer; warps 2-5 epilogue
// (SwiGLU, h in fp16 for the down projection); warps 6-15 gather (two per B stage); warps 16-23
// expand the codes and write the scale factors, two quartets (one warp per TMEM lane quarter
// each) taking alternate stages.  Every wait is bounded (common.cuh).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace mx {

constexpr int BM = 128;
constexpr int kStageK = 128;                      // K per stage: two 64-K raw blocks
constexpr int kRawBytes = 2 * kFp4BlockBytes;     // 8704 B per stage
constexpr int kRawSlots = 10;                    // 87 KB of 4-bit weights in flight per SM
constexpr int kAStages = 3;                       // expanded A tiles + their scale factors (TMEM)
constexpr int kStages = 5;                        // B (activation) ring
constexpr int kTokMax = 64;                       // tokens per unit
constexpr int kNMax = 2 * kTokMax;                // B rows (hi / lo) per unit
constexpr int kABytes = BM * kStageK;             // 16 KB
constexpr int kBBytes = kNMax * kStageK;          // 16 KB
constexpr int kGatherPerSlot = 2;
constexpr int kGatherWarps = kGatherPerSlot * kStages;   // 10 (two per B slot)
constexpr int kFirstGather = 6;
constexpr int kFirstExpand = kFirstGather + kGatherWarps;  // 16: warps 16..23, two quartets
constexpr int kExpandSets = 2;                             // quartet e takes the stages g % 2 == e
constexpr int kThreads = 32 * (kFirstExpand + 4 * kExpandSets);  // 768
constexpr int kAccCols = kNMax;                   // 128 fp32 columns per accumulator
constexpr int kSfBase = 2 * kAccCols;             // scale factors after the two accumulators
constexpr int kSfCols = 8;                        // per stage: SFA 4, SFB 4
constexpr int kTmemCols = 512;
constexpr int kEpiStageBytes = 16 * 32 * 2;       // per epilogue warp: 16 columns x 32 fp16 rows
constexpr int kUnitRing = 8;
constexpr int kTokBytes = kGatherWarps * kTokMax * 4;
constexpr int kSmemBytes = kAStages * kABytes + kStages * kBBytes + kStages * kNMax * 4 /*SFB words*/ +
                           kRawSlots * kRawBytes + 1024 /*barriers*/ + 1024 /*align*/ + kTokBytes + 4 * kEpiStageBytes;
static_assert(kSfBase + kAStages * kSfCols <= kTmemCols, "TMEM columns");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kFirstExpand % 4 == 0, "expander warps cover lane quarters 0..3 in order");

struct Unit {
  int expert, row_start, rows, tile;
};

MOE_DEVICE Seg load_seg_l2(const Seg* p) {
  const int4 lo = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 hi = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  return Seg{lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
}

// Unit u = 2 v + h: v as in gemm_fp4.cu (the parts of one expert tile-major), h the half of the
// segment (rows [64 h, 64 h + 64)); rows == 0 for an empty half.
MOE_DEVICE Unit decode_unit(int u, const Seg* segs, int tiles) {
  const int v = u >> 1, h = u & 1;
  const Seg any = load_seg_l2(segs + v / tiles);
  const int o = v - any.first * tiles;
  const Seg s = load_seg_l2(segs + any.first + o % any.nparts);
  const int rows = min(max(s.rows - kTokMax * h, 0), kTokMax);
  return Unit{s.expert, s.row_start + kTokMax * h, rows, o / any.nparts};
}

MOE_DEVICE int pad16(int n) { return n <= 16 ? 16 : ((n + 15) & ~15); }

// Scale bytes per quantised row of K elements: K / 32, rounded up to a multiple of 4 so that a
// stage's four block scales are one aligned 32-bit word.
__host__ __device__ inline int mx_scale_stride(int K) { return ((K / 32) + 3) & ~3; }

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A e2m1 (5), B e4m3 (0), K-major
// both, N >> 3 at bit 17, e8m0 scale factors (bit 23), M >> 4 at bit 24, scale-factor byte ids of
// B (bits 4-5) and A (bits 29-30).
MOE_DEVICE uint32_t idesc_mx(uint32_t N, uint32_t sf_id) {
  return (sf_id << 4) | (5u << 7) | (0u << 10) | ((N >> 3) << 17) | (1u << 23) | ((BM >> 4) << 24) | (sf_id << 29);
}

MOE_DEVICE void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

MOE_DEVICE void tmem_st_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
MOE_DEVICE void tmem_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3)
               : "memory");
}
MOE_DEVICE void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

MOE_DEVICE void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,"
      "%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

MOE_DEVICE void cp_async_4(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst_smem), "l"(src) : "memory");
}

// Unit i of this CTA for a non-producer warp: waits for ring slot i, reads it, releases the slot.
MOE_DEVICE int ring_unit(const int32_t* ring, uint64_t* unit_full, uint64_t* unit_empty, uint32_t i,
                         volatile int* abort_flag, uint32_t* err) {
  const uint32_t s = i % kUnitRing;
  if (!mbar_wait_warp(&unit_full[s], (i / kUnitRing) & 1u, abort_flag, err)) return -1;
  const int u = ring[s];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&unit_empty[s]);
  return u;
}

// kGateUp: gate/up (A = W_gate|W_up interleaved, B = x in two e4m3 terms gathered by token, SwiGLU
// epilogue, h fp16); else down (A = W_down, B = h in two e4m3 terms, grouped rows, y fp16).  In both
// the B operand comes as xq [rows][2][K] e4m3 and xs [rows][2][sstride] e8m0.
template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 1) mx_ffn_kernel(const TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring_a = smem;                                        // kAStages x 16 KB (1024-aligned)
  uint8_t* ring_b = ring_a + kAStages * kABytes;                 // kStages x 16 KB
  uint32_t* sfb_words = reinterpret_cast<uint32_t*>(ring_b + kStages * kBBytes);  // [kStages][kNMax]
  uint8_t* ring_raw = reinterpret_cast<uint8_t*>(sfb_words + kStages * kNMax);   // kRawSlots x 8704 B
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(ring_raw + kRawSlots * kRawBytes);
  uint64_t* raw_empty = raw_full + kRawSlots;
  uint64_t* a_full = raw_empty + kRawSlots;
  uint64_t* a_empty = a_full + kAStages;
  uint64_t* b_full = a_empty + kAStages;
  uint64_t* b_empty = b_full + kStages;
  uint64_t* acc_full = b_empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* unit_full = drain + 1;
  uint64_t* unit_empty = unit_full + kUnitRing;
  int32_t* unit_ring = reinterpret_cast<int32_t*>(unit_empty + kUnitRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(unit_ring + kUnitRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* tok_tab = reinterpret_cast<int32_t*>(ring_raw + kRawSlots * kRawBytes + 1024);
  uint16_t* epi_stage = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(tok_tab) + kTokBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawSlots; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&b_full[s], kGatherPerSlot);
      mbar_init(&b_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kUnitRing; ++s) {
      mbar_init(&unit_full[s], 1);
      mbar_init(&unit_empty[s], kThreads / 32 - 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  const int K = kGateUp ? a.d : a.f;         // reduction length
  const int tiles = kGateUp ? a.f / 64 : a.d / BM;
  const int nblk = K / 64;                   // 64-K raw blocks per unit
  const int nst = (nblk + 1) / 2;            // stages per unit (the last one may hold one block)
  const int sstride = mx_scale_stride(K);    // scale bytes per B-source row
  const uint8_t* wq = kGateUp ? a.q_gu : a.q_down;
  const int total_units = 2 * __ldcg(a.n_segs) * tiles;

  if (warp == 0) {
    // ---------------- raw 4-bit blocks (one bulk copy per stage) and the unit hand-out ----------
    const uint64_t pol_w = l2_policy_evict_first();
    uint32_t p = 0;
    bool ok = true;
    int u = static_cast<int>(blockIdx.x);
    for (uint32_t i = 0; ok; ++i) {
      // skip empty halves: take tickets until a unit with rows (or the end)
      Unit un{0, 0, 0, 0};
      while (u < total_units) {
        un = decode_unit(u, a.segs, tiles);
        if (un.rows > 0) break;
        uint32_t ticket = 0;
        if (lane == 0) ticket = atomicAdd(a.sched, 1u);
        u = static_cast<int>(gridDim.x + __shfl_sync(0xffffffffu, ticket, 0));
      }
      const uint32_t rs = i % kUnitRing;
      if (!(ok = mbar_wait_warp(&unit_empty[rs], ((i / kUnitRing) & 1u) ^ 1u, abort_flag, a.err))) break;
      if (lane == 0) {
        unit_ring[rs] = u;
        mbar_arrive(&unit_full[rs]);
      }
      __syncwarp();
      if (u >= total_units) break;
      uint32_t ticket = 0;
      if (lane == 0) ticket = atomicAdd(a.sched, 1u);  // the next unit's, read after this unit's copies
      const uint8_t* w0 = wq + (static_cast<size_t>(un.expert) * tiles + un.tile) * nblk * kFp4BlockBytes;
      for (int kk = 0; kk < nst; ++kk, ++p) {
        const int slot = p % kRawSlots;
        const uint32_t bytes = static_cast<uint32_t>(min(2, nblk - 2 * kk)) * kFp4BlockBytes;
        if (!(ok = mbar_wait_warp(&raw_empty[slot], ((p / kRawSlots) & 1u) ^ 1u, abort_flag, a.err))) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&raw_full[slot], bytes);
          bulk_load(ring_raw + slot * kRawBytes, w0 + static_cast<size_t>(2 * kk) * kFp4BlockBytes, bytes,
                    &raw_full[slot], pol_w);
        }
        __syncwarp();
      }
      u = static_cast<int>(gridDim.x + __shfl_sync(0xffffffffu, ticket, 0));
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: 4 block-scaled MMAs of K = 32 per stage ----------------
    uint32_t g = 0, j = 0;
    bool ok = true;
    const uint64_t a_base = smem_desc_sw128(smem_u32(ring_a));
    const uint64_t b_base = smem_desc_sw128(smem_u32(ring_b));
    for (uint32_t ui = 0; ok; ++ui, ++j) {
      const int u = ring_unit(unit_ring, unit_full, unit_empty, ui, abort_flag, a.err);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= total_units) break;
      const Unit un = decode_unit(u, a.segs, tiles);
      const uint32_t N = static_cast<uint32_t>(pad16(2 * un.rows));
      const uint32_t buf = j & 1u, use_acc = j >> 1;
      if (!(ok = mbar_wait_warp(&acc_empty[buf], (use_acc & 1u) ^ 1u, abort_flag, a.err))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + buf * kAccCols;
      for (int kk = 0; kk < nst; ++kk, ++g) {
        // a_full of the stage implies its B rows (the expander waited for them before its arrival)
        const uint32_t sa = g % kAStages, sb = g % kStages;
        if (!(ok = mbar_wait_warp(&a_full[sa], (g / kAStages) & 1u, abort_flag, a.err))) break;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t ad = a_base + sa * (kABytes >> 4), bd = b_base + sb * (kBBytes >> 4);
          const uint32_t sf = tmem + kSfBase + sa * kSfCols;
          const uint32_t nkb = 2u * static_cast<uint32_t>(min(2, nblk - 2 * kk));  // 32-K blocks of the stage
          for (uint32_t kb = 0; kb < nkb; ++kb)  // K = 32 per MMA: +32 bytes = +2 in the address field
            mma_mx(d_tmem, ad + 2 * kb, bd + 2 * kb, idesc_mx(N, kb), sf, sf + 4, (kk | kb) != 0);
          mma_commit(&a_empty[sa]);
          mma_commit(&b_empty[sb]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&acc_full[buf]);
      __syncwarp();
    }
    if (elect_one()) mma_commit(drain);  // completes once every MMA issued above has finished
    __syncwarp();
    mbar_wait_warp(drain, 0, nullptr, a.err);
  } else if (warp < 6) {
    // ---------------- epilogue: hi + lo columns; gate/up: SwiGLU, h (fp16); down: y (fp16) ----------------
    const int q = warp & 3;
    uint32_t j = 0;
    for (uint32_t ui = 0; !*abort_flag; ++ui, ++j) {
      const int u = ring_unit(unit_ring, unit_full, unit_empty, ui, abort_flag, a.err);
      if (u < 0 || u >= total_units) break;
      const Unit un = decode_unit(u, a.segs, tiles);
      const uint32_t buf = j & 1u, use_acc = j >> 1;
      if (!mbar_wait(&acc_full[buf], use_acc & 1u, abort_flag, a.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * kAccCols;
      const int L = 32 * q + lane;
      uint16_t* stg = epi_stage + (warp - 2) * (kEpiStageBytes / 2);
      bool sat = false;
      if (!kGateUp) {
        const int feat0 = un.tile * BM + 32 * q;
        for (int c0 = 0; c0 < un.rows; c0 += 16) {
          uint32_t rr[32];
          tmem_ld_32x32b_x32(tbase + 2 * c0, rr);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float v = __uint_as_float(rr[2 * c]) + __uint_as_float(rr[2 * c + 1]);
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
            const int cl = idx >> 2, g4 = idx & 3;
            if (c0 + cl < un.rows) {
              const uint4 v = *reinterpret_cast<const uint4*>(stg + cl * 32 + 8 * g4);
              *reinterpret_cast<uint4*>(a.y + static_cast<size_t>(un.row_start + c0 + cl) * a.d + feat0 + 8 * g4) = v;
            }
          }
          __syncwarp();
        }
        if (__any_sync(0xffffffffu, sat) && lane == 0) set_error(a.err, MOE_DEVERR_RANGE);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        continue;
      }
      const int w16 = L & 15;
      const bool is_gate = w16 < 8;
      const int fl = 8 * ((L >> 4) & 1) + (w16 & 7);
      const int feat0 = un.tile * 64 + 16 * q;
      for (int c0 = 0; c0 < un.rows; c0 += 16) {  // 16 tokens = 32 accumulator columns (hi, lo)
        uint32_t rr[32];
        tmem_ld_32x32b_x32(tbase + 2 * c0, rr);
        tmem_wait_ld();
        uint32_t r[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) r[t] = __float_as_uint(__uint_as_float(rr[2 * t]) + __uint_as_float(rr[2 * t + 1]));
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const uint32_t send = is_gate ? r[2 * jj + 1] : r[2 * jj];
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 8);
          const int cl = 2 * jj + (is_gate ? 0 : 1);
          const float gv = __uint_as_float(is_gate ? r[2 * jj] : recv);
          const float uv = __uint_as_float(is_gate ? recv : r[2 * jj + 1]);
          float hv = swiglu(gv, uv);
          if (c0 + cl < un.rows && !(fabsf(hv) <= kF16Max)) {
            sat = true;
            hv = fminf(fmaxf(hv, -kF16Max), kF16Max);
          }
          stg[cl * 16 + fl] = f32_to_f16_bits_rn(hv);
        }
        __syncwarp();
        {
          const int cl = lane >> 1, half = lane & 1;
          if (c0 + cl < un.rows) {
            const uint4 v = *reinterpret_cast<const uint4*>(stg + cl * 16 + 8 * half);
            *reinterpret_cast<uint4*>(a.h + static_cast<size_t>(un.row_start + c0 + cl) * a.f + feat0 + 8 * half) = v;
          }
        }
        __syncwarp();
      }
      if (__any_sync(0xffffffffu, sat) && lane == 0) set_error(a.err, MOE_DEVERR_RANGE);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  } else if (warp < kFirstExpand) {
    // ---------------- gather: hi / lo rows of x (e4m3) and their scale words ----------------
    const int gw = warp - kFirstGather;
    const int slot = gw % kStages, half = gw / kStages;
    int32_t* tok = tok_tab + kTokMax * gw;
    const int ch = lane & 7;
    const int rs0 = (lane >> 3) + 4 * half;  // B rows rs0 + 8 i
    const uint64_t pol_x = l2_policy_evict_last();
    const int dbytes = K;  // per B-source row: e4m3 bytes (scale bytes: sstride)
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t ui = 0; ok; ++ui) {
      const int u = ring_unit(unit_ring, unit_full, unit_empty, ui, abort_flag, a.err);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= total_units) break;
      const Unit un = decode_unit(u, a.segs, tiles);
      bool have_tok = false;
      const int nrow = 2 * un.rows;
      for (int kk = 0; kk < nst; ++kk, ++g) {
        const int s = g % kStages;
        if (s != slot) continue;
        if (!have_tok) {  // gate/up: the token of each row; down: the grouped row itself
          for (int n = lane; n < un.rows; n += 32) tok[n] = kGateUp ? a.perm[un.row_start + n] / a.k : un.row_start + n;
          __syncwarp();
          have_tok = true;
        }
        const int nch = min(2, nblk - 2 * kk) * 4;  // 16-byte chunks of this stage's K
        if (!(ok = mbar_wait_warp(&b_empty[s], ((g / kStages) & 1u) ^ 1u, abort_flag, a.err))) break;
        const uint32_t sb = smem_u32(ring_b + s * kBBytes);
        if (ch < nch)
          for (int n = rs0; n < nrow; n += 8) {
            const int qrow = 2 * tok[n >> 1] + (n & 1);  // row of the quantised source: token / row, hi / lo
            const uint8_t* src = a.xq + static_cast<size_t>(qrow) * dbytes + kk * kStageK + ch * 16;
            cp_async_16_hint(sb + n * 128 + ((ch ^ (n & 7)) << 4), src, pol_x);
          }
        for (int n = half * 64 + lane; n < min(nrow, half * 64 + 64); n += 32) {
          const int qrow = 2 * tok[n >> 1] + (n & 1);
          cp_async_4(smem_u32(sfb_words + s * kNMax + n), a.xs + static_cast<size_t>(qrow) * sstride + kk * 4);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&b_full[s]);
      }
    }
  } else {
    // ---------------- expand the codes into the MMA's layout; scale factors into TMEM ----------------
    const int q = warp & 3;           // TMEM lane quarter
    const int r = 32 * q + lane;      // weight row of the tile owned by this thread
    const uint32_t set = static_cast<uint32_t>(warp - kFirstExpand) / 4;
    uint32_t g = 0, p = 0;
    bool ok = true;
    for (uint32_t ui = 0; ok; ++ui) {
      const int u = ring_unit(unit_ring, unit_full, unit_empty, ui, abort_flag, a.err);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= total_units) break;
      for (int kk = 0; kk < nst; ++kk, ++g, ++p) {
        if (g % kExpandSets != set) continue;
        const int rsl = p % kRawSlots, s = g % kStages, sa = g % kAStages;
        if (!(ok = mbar_wait_warp(&raw_full[rsl], (p / kRawSlots) & 1u, abort_flag, a.err))) break;
        const uint8_t* raw = ring_raw + rsl * kRawBytes;
        const int nb = min(2, nblk - 2 * kk);  // raw blocks in this stage
        uint4 c[2][2];
        uint32_t sc[2] = {0u, 0u};
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          if (b < nb) {
            const uint8_t* blk = raw + b * kFp4BlockBytes;
            c[b][0] = *reinterpret_cast<const uint4*>(blk + r * 16);
            c[b][1] = *reinterpret_cast<const uint4*>(blk + 2048 + r * 16);
            sc[b] = *reinterpret_cast<const uint16_t*>(blk + 4096 + 2 * r);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rsl]);
        if (!(ok = mbar_wait_warp(&a_empty[sa], ((g / kAStages) & 1u) ^ 1u, abort_flag, a.err))) break;
        // row r: logical 16-element chunk j = 4 b + 2 half + sub holds the codes in its low 8 bytes
        uint8_t* arow = ring_a + sa * kABytes + r * 128;
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            if (b >= nb) continue;  // a one-block stage: the MMAs read chunks 0..3 only
            const int j0 = 4 * b + 2 * hf;
            *reinterpret_cast<uint4*>(arow + ((j0 ^ (r & 7)) << 4)) = make_uint4(c[b][hf].x, c[b][hf].y, 0u, 0u);
            *reinterpret_cast<uint4*>(arow + (((j0 + 1) ^ (r & 7)) << 4)) = make_uint4(c[b][hf].z, c[b][hf].w, 0u, 0u);
          }
        fence_proxy_async_smem();
        const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16) + kSfBase + sa * kSfCols;
        tmem_st_x1(tq + q, sc[0] | (sc[1] << 16));  // SFA: row r's four block scales, column + r / 32
        if (!(ok = mbar_wait_warp(&b_full[s], (g / kStages) & 1u, abort_flag, a.err))) break;
        const uint32_t* w = sfb_words + s * kNMax;  // SFB: B row n at column 4 + n / 32, lane n % 32
        tmem_st_x4(tq + 4, w[lane], w[32 + lane], w[64 + lane], w[96 + lane]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[sa]);
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
  // the last CTA to leave resets the hand-out words for the next launch
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
      a.sched[0] = 0u;
      a.sched[1] = 0u;
      __threadfence();
    }
  }
}

// x (bf16 [T][d]) -> two e4m3 terms with e8m0 scales per 32 consecutive elements:
//   xq [T][2][d] (row 2t = hi, 2t + 1 = lo of token t), xs [T][2][d / 32].
// One thread per 32-element block.  The hi scale makes the block's largest magnitude land in
// [128, 256) (below e4m3's 448, no saturation); the residual x - hi is exact in fp32 and gets its
// own scale the same way.  An all-zero block gets scale byte 0 and zero codes.
MOE_DEVICE uint32_t e8m0_for(float amax) {
  const uint32_t eb = (__float_as_uint(amax) >> 23) & 0xFFu;  // biased exponent (0: zero / subnormal)
  const int s = eb == 0 ? 0 : static_cast<int>(eb) - 7;         // 2^(E - 7): E + 120 as a biased byte
  return static_cast<uint32_t>(s < 0 ? 0 : (s > 254 ? 254 : s));
}
MOE_DEVICE float inv_pow2(uint32_t s) { return __uint_as_float((254u - s) << 23); }   // 2^(127 - s), s in [1, 253]
MOE_DEVICE float pow2(uint32_t s) { return s == 0 ? 0.f : __uint_as_float(s << 23); }  // 2^(s - 127)

// two floats -> packed e4m3x2 (RNE, saturating): element a in the low byte
MOE_DEVICE uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}
MOE_DEVICE float2 e4m3x2_to_f32(uint32_t v) {  // low byte -> .x
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(v));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

template <bool kBf16>
__global__ void __launch_bounds__(256) to_mx_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ xq,
                                                   uint8_t* __restrict__ xs, int T, int d) {
  pdl_wait();
  pdl_trigger();
  const int nb = d / 32, ss = mx_scale_stride(d);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * nb; i += gridDim.x * blockDim.x) {
    const int t = i / nb, j = i % nb;
    float v[32];
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d + 32 * j);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f8[8];
      if (kBf16)
        bf16x8_to_f32(src[q], f8);
      else
        f16x8_to_f32(src[q], f8);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[8 * q + e] = f8[e];
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
    const uint32_t s1 = e8m0_for(amax);
    const float m1 = s1 == 0 ? 0.f : inv_pow2(s1), b1 = pow2(s1);
    uint32_t hi[8];
    float amax2 = 0.f;
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const uint32_t p0 = e4m3x2(v[e] * m1, v[e + 1] * m1), p1 = e4m3x2(v[e + 2] * m1, v[e + 3] * m1);
      hi[e / 4] = p0 | (p1 << 16);
      const float2 f0 = e4m3x2_to_f32(p0), f1 = e4m3x2_to_f32(p1);
      v[e] -= f0.x * b1, v[e + 1] -= f0.y * b1, v[e + 2] -= f1.x * b1, v[e + 3] -= f1.y * b1;  // exact residual
      amax2 = fmaxf(amax2, fmaxf(fmaxf(fabsf(v[e]), fabsf(v[e + 1])), fmaxf(fabsf(v[e + 2]), fabsf(v[e + 3]))));
    }
    const uint32_t s2 = e8m0_for(amax2);
    const float m2 = s2 == 0 ? 0.f : inv_pow2(s2);
    uint32_t lo[8];
#pragma unroll
    for (int e = 0; e < 32; e += 4)
      lo[e / 4] = e4m3x2(v[e] * m2, v[e + 1] * m2) | (e4m3x2(v[e + 2] * m2, v[e + 3] * m2) << 16);
    uint4* dh = reinterpret_cast<uint4*>(xq + (static_cast<size_t>(2 * t) * d + 32 * j));
    uint4* dl = reinterpret_cast<uint4*>(xq + (static_cast<size_t>(2 * t + 1) * d + 32 * j));
    dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    xs[static_cast<size_t>(2 * t) * ss + j] = static_cast<uint8_t>(s1);
    xs[static_cast<size_t>(2 * t + 1) * ss + j] = static_cast<uint8_t>(s2);
  }
}

}  // namespace mx

template <bool kGateUp>
static cudaError_t launch_mx(const TcArgs& a, int num_sms, cudaStream_t st) {
  if (!a.sched || !a.xq || !a.xs) return cudaErrorInvalidValue;
  auto kern = mx::mx_ffn_kernel<kGateUp>;
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), mx::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(num_sms), dim3(mx::kThreads), mx::kSmemBytes, st, a);
}

cudaError_t launch_mx_gateup(const TcArgs& a, int num_sms, cudaStream_t st) { return launch_mx<true>(a, num_sms, st); }
cudaError_t launch_mx_down(const TcArgs& a, int num_sms, cudaStream_t st) { return launch_mx<false>(a, num_sms, st); }

cudaError_t launch_x_to_mx(const uint16_t* x, uint8_t* xq, uint8_t* xs, int T, int d, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int n = T * (d / 32);
  const int blocks = (n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024;
  return launch_pdl(mx::to_mx_kernel<true>, dim3(blocks), dim3(256), 0, st, x, xq, xs, T, d);
}

cudaError_t launch_h_to_mx(const uint16_t* h, uint8_t* hq, uint8_t* hs, int R, int f, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  const int n = R * (f / 32);
  const int blocks = (n + 255) / 256 < 2048 ? (n + 255) / 256 : 2048;
  return launch_pdl(mx::to_mx_kernel<false>, dim3(blocks), dim3(256), 0, st, h, hq, hs, R, f);
}

int mx_scale_bytes(int K) { return mx::mx_scale_stride(K); }

}  // namespace moe
