// Grouped expert GEMMs with block-scaled 4-bit weights on the tensor cores (sm_103a).
//
// Same grouped problem, units and epilogues as gemm_tc.cu (swap-AB: 128 weight rows as M, the
// segment's tokens as N <= 128), for routed experts whose weights are e2m1 codes with one e8m0
// scale per 32 K elements (OCP MX v1.0; the "moe-prefill-quantum" page's hardware check and
// the Jetson page's model are MXFP4).  The weights are dequantised in the kernel:
//
//   raw 4-bit blocks (4352 B per 128 x 64 tile chunk) --bulk copy--> shared memory
//   --4 dequant warps, one TMEM lane quarter each: cvt.rn.f16x2.e2m1x2, times the block scale
//     (one HMUL2, exact in fp16 for the scale range checked at set-up)--> TMEM (tcgen05.st)
//   --tcgen05.mma kind::f16 with A read from TMEM, B (fp16 token / hidden rows) from shared
//     memory--> fp32 accumulator in TMEM --> the same SwiGLU / down epilogues.
//
// The dequantised tile never touches shared memory: shared-memory traffic per weight byte stays
// close to the 16-bit kernel's, and the weights -- 4.25 bits each -- stream from HBM once.
// Activations are fp16 (x converted once per step; h is fp16 already), matching the fp16 A.
//
// Roles: warp 0 raw producer; warp 1 TMEM owner and MMA issuer; warps 2-5 epilogue; gate/up:
// warps 6-13 gather the fp16 token rows (cp.async), warps 14-21 dequantise; down: warp 6 loads
// rows of h by TMA, warps 7-14 dequantise.  The dequant warps form two quartets (one warp per
// TMEM lane quarter each) that take alternate stages.  A stage is 128 deep in K (two 4-bit
// blocks, two 64-wide swizzled B slices, 8 MMAs), so the single-thread MMA issue -- one barrier
// wait and one commit per stage -- keeps ahead of the weight stream.  Producer and MMA loops run
// converged and issue under elect_one().  Every wait is bounded (common.cuh).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace fq {

constexpr int BM = 128;
constexpr int kSubK = 64;                        // one 128-byte-swizzled K slice / one 4-bit block
constexpr int kSubs = 2;                         // K slices per pipeline stage (K = 128)
constexpr int kDqSets = 2;                       // dequant quartets; quartet q takes the stages kk % 2 == q
constexpr int kRawBytes = kSubs * kFp4BlockBytes;          // 8704 B per stage
constexpr int kRawPer = 2;                       // stages per raw bulk copy (one per quartet)
constexpr int kRawSlotBytes = kRawPer * kRawBytes;
constexpr int kACols = kSubs * kSubK / 2;        // 64 columns (fp16 pairs) per A stage
constexpr int kTmemCols = 512;                   // accumulators + A stages
constexpr int kEpiStageBytes = 16 * 32 * 2;     // per epilogue warp: 16 columns x 32 fp16 rows

// Geometry for segments of at most kN rows (128, or 64 for steps of at most 64 tokens): the two
// accumulators take 2 kN TMEM columns and the rest of the 512 hold A stages, so small segments
// get a deeper A ring (6 stages instead of 4).  With 128-row segments the activation (B) stages
// have their own, deeper ring in shared memory: a B stage can be requested before the A slot of
// its stage is free, so the gathered rows' L2 latency hides behind several stages of MMAs.
template <int kN>
struct Geo {
  static constexpr int kStages = (kTmemCols - 2 * kN) / kACols;  // A stages (TMEM)
  // 128-row activation stages get their own ring (5 stages); 64-row ones share the A ring's
  // barriers (the second pair of barrier operations per stage costs more than it hides there)
  static constexpr bool kSplitB = kN > 64;
  static constexpr int kBStages = kSplitB ? 5 : kStages;         // B stages (shared memory)
  static constexpr int kStagesRaw = kN > 64 ? 6 : 8;             // 4-bit stages in shared memory
  static constexpr int kRawSlots = kStagesRaw / kRawPer;         // raw ring slots of kRawPer stages
  static constexpr int kSubBytes = kN * kSubK * 2;                // one K slice of up to kN rows
  static constexpr int kBBytes = kSubs * kSubBytes;
  static constexpr int kAccCols = kN;
  static constexpr int kAStart = 2 * kAccCols;                   // A stages after the accumulators
  static constexpr int kGatherPerSlot = kN > 64 ? 2 : 1;         // gate/up B producers per B slot
  static constexpr int kGatherWarps = kGatherPerSlot * kBStages;
  static constexpr int kTokBytes = kGatherWarps * kN * 4;         // per gather warp: token per row
  static constexpr int kSmemBytes =
      kBStages * kBBytes + kStagesRaw * kRawBytes + 1024 + 1024 + kTokBytes + 4 * kEpiStageBytes;
  static constexpr int kBProducers = 4;                           // down: warps issuing the TMA loads of h
  static constexpr int threads(bool gate_up) { return 32 * (gate_up ? 6 + kGatherWarps + 8 : 6 + kBProducers + 8); }
  static_assert(kRawPer == kDqSets && kStagesRaw % kRawPer == 0, "one stage of each raw copy per quartet");
  static_assert(kAStart + kStages * kACols <= kTmemCols, "TMEM columns");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kN <= kSegRowsMax && kN % 32 == 0, "segment rows");
};

MOE_DEVICE int pad16(int rows) { return rows <= 16 ? 16 : ((rows + 15) & ~15); }

// Units are handed out at run time: each CTA's first unit is blockIdx.x, later ones come from a
// per-launch counter (gridDim.x + the counter's old value), so a CTA that starts late -- its SM
// still busy with another kernel -- does fewer units instead of holding the end of the launch.
// Warp 0 fetches them and publishes each CTA's sequence in a ring of kUnitRing slots; every
// other warp reads the same sequence from the ring.  An index >= the unit count ends it.
constexpr int kUnitRing = 8;

// Unit i of this CTA for a consumer warp (converged): waits for ring slot i, reads it and
// releases the slot.  -1 when the wait gave up.
MOE_DEVICE int ring_unit(const int32_t* ring, uint64_t* unit_full, uint64_t* unit_empty, uint32_t i,
                         volatile int* abort_flag, uint32_t* err) {
  const uint32_t s = i % kUnitRing;
  if (!mbar_wait_warp(&unit_full[s], (i / kUnitRing) & 1u, abort_flag, err)) return -1;
  const int u = ring[s];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&unit_empty[s]);
  return u;
}

struct Unit {
  int expert, row_start, rows, tile;
};

// Routed units only; the parts of one expert are tile-major (see gemm_tc.cu).
// kL2: read the segment records through L2 (the down kernel's raw producer reads them before its
// grid-dependency wait, when nothing may come from a stale L1 line).
MOE_DEVICE Seg load_seg_l2(const Seg* p) {
  const int4 lo = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 hi = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  return Seg{lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
}
template <bool kL2 = false>
MOE_DEVICE Unit decode_unit(int u, const Seg* segs, int tiles) {
  const Seg any = kL2 ? load_seg_l2(segs + u / tiles) : segs[u / tiles];
  const int o = u - any.first * tiles;
  const Seg s = kL2 ? load_seg_l2(segs + any.first + o % any.nparts) : segs[any.first + o % any.nparts];
  return Unit{s.expert, s.row_start, s.rows, o / any.nparts};
}

// e8m0 scale byte -> fp16 2^(s-127) for s in [kFp4ScaleMin, kFp4ScaleMax] (subnormal below 2^-14).
MOE_DEVICE uint32_t scale_half2(uint32_t s) {
  const int e = static_cast<int>(s) - 127;
  const uint32_t h = e >= -14 ? static_cast<uint32_t>(e + 15) << 10 : 1u << (e + 24);
  return h | (h << 16);
}

// 16 code bytes (32 e2m1 values, element 2i in the low nibble of byte i) -> 16 fp16x2 words times
// the scale: word j holds elements (2j, 2j+1) in its (low, high) halves.
MOE_DEVICE void dequant16(const uint4 c, uint32_t sc2, uint32_t* w) {
  const uint32_t src[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(src[i]));
    const uint32_t hv[4] = {h0, h1, h2, h3};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t o;
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o) : "r"(hv[q]), "r"(sc2));
      w[4 * i + q] = o;
    }
  }
}

MOE_DEVICE void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
MOE_DEVICE void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16.
MOE_DEVICE void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The MMAs of one 128-deep stage in one block: `two` ? 8 : 4 MMAs of K = 16, D += A x B^T with A
// in TMEM (+8 columns per step, +32 per 64-wide slice) and B in shared memory (descriptor +2 per
// step, +kSubDesc per slice).  Only the first MMA may start a fresh accumulation (acc == 0); the
// offsets are added inside the block, off the issuing lane's dependency chain.
template <uint32_t kSubDesc>
MOE_DEVICE void mma_stage_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc, bool two) {
  if (two)
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
        ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, %4, %4;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\tadd.u32 a4, %1, 32;\n\t"
        "add.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
        "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\tadd.u64 b4, %2, %5;\n\t"
        "add.u64 b5, b4, 2;\n\tadd.u64 b6, b4, 4;\n\tadd.u64 b7, b4, 6;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, t;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc), "n"(static_cast<uint64_t>(kSubDesc))
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t.reg .b32 a1, a2, a3;\n\t.reg .b64 b1, b2, b3;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, %4, %4;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
        "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// tcgen05.commit / mbarrier.test_wait on a barrier given by its shared-memory address.
MOE_DEVICE void mma_commit_u32(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
MOE_DEVICE bool mbar_test_u32(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Pipeline.  Stage g covers K slices [2g, 2g + 2) of the unit (the last stage of an odd K/64
// has one).  Rings:
//   raw[p % kRawSlots]   the 4-bit blocks of stages 2p', 2p' + 1 of a unit (p' the pair within the
//                        unit, p counting pairs): one bulk copy per pair (a fixed cost per bulk
//                        operation makes fewer, larger copies stream faster); quartet q reads
//                        stage 2p' + q, and both quartets free the slot
//   A[g % kStages]       dequantised weights in TMEM: full when the quartet (4 arrivals) is done,
//                        empty when the MMAs reading it finish
//   B[g % kBStages]      activation rows in shared memory: full when the slot's gather warps (or
//                        one arrive.expect_tx for TMA) are done, empty when the MMAs finish.
//                        Without kSplitB the B slots are the A slots' and share their barriers.
// The MMA lane tests one or two barriers and commits once or twice per 128 K.
template <bool kGateUp, int kN>
__global__ void __launch_bounds__(Geo<kN>::threads(kGateUp), 1)
    fp4_ffn_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
  constexpr int kStages = Geo<kN>::kStages;
  constexpr int kSubBytes = Geo<kN>::kSubBytes;
  constexpr int kBBytes = Geo<kN>::kBBytes;
  constexpr int kAccCols = Geo<kN>::kAccCols;
  constexpr int kAStart = Geo<kN>::kAStart;
  constexpr int kGatherPerSlot = Geo<kN>::kGatherPerSlot;
  constexpr int kGatherWarps = Geo<kN>::kGatherWarps;
  constexpr int kTokBytes = Geo<kN>::kTokBytes;
  constexpr int kBStages = Geo<kN>::kBStages;
  constexpr bool kSplitB = Geo<kN>::kSplitB;
  constexpr int kStagesRaw = Geo<kN>::kStagesRaw;
  constexpr int kRawSlots = Geo<kN>::kRawSlots;
  constexpr int kBProducers = Geo<kN>::kBProducers;
  constexpr int kDqWarp = kGateUp ? 6 + kGatherWarps : 6 + kBProducers;  // first dequant warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring_b = smem;                                  // kBStages x kBBytes, 1024-aligned
  uint8_t* ring_raw = smem + kBStages * kBBytes;           // kStagesRaw x 8704 B
  uint64_t* raw_full = reinterpret_cast<uint64_t*>(ring_raw + kStagesRaw * kRawBytes);
  uint64_t* raw_empty = raw_full + kRawSlots;
  uint64_t* full = raw_empty + kRawSlots;
  uint64_t* empty = full + kStages;
  uint64_t* b_full = kSplitB ? empty + kStages : full;
  uint64_t* b_empty = kSplitB ? b_full + kBStages : empty;
  uint64_t* acc_full = empty + kStages + 2 * kBStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* unit_full = reinterpret_cast<uint64_t*>(tmem_slot + 2);
  uint64_t* unit_empty = unit_full + kUnitRing;
  int32_t* unit_ring = reinterpret_cast<int32_t*>(unit_empty + kUnitRing);
  static_assert((2 * kRawSlots + 2 * kStages + 2 * kBStages + 5) * 8 + 8 + kUnitRing * 20 <= 1024,
                "barriers, TMEM slot, abort flag and unit ring fit the 1 KB area");
  int32_t* tok_tab = reinterpret_cast<int32_t*>(ring_raw + kStagesRaw * kRawBytes + 1024);
  uint16_t* epi_stage = reinterpret_cast<uint16_t*>(ring_raw + kStagesRaw * kRawBytes + 1024 + kTokBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRawSlots; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], 4 * kDqSets);
    }
    const int b_arrivals = kGateUp ? kGatherPerSlot : 1;  // the slot's gather warps, or one TMA arrival
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 4 + (kSplitB ? 0 : b_arrivals));  // the dequant quartet (+ the B producers)
      mbar_init(&empty[s], 1);
    }
    if (kSplitB)
      for (int s = 0; s < kBStages; ++s) {
        mbar_init(&b_full[s], b_arrivals);
        mbar_init(&b_empty[s], 1);
      }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kUnitRing; ++s) {
      mbar_init(&unit_full[s], 1);                                    // warp 0 publishes
      mbar_init(&unit_empty[s], static_cast<int>(blockDim.x / 32) - 1);  // every other warp reads
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (!kGateUp && warp == 6 && lane == 0) tma_prefetch_map(&maps.h);
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // gate/up lets its dependents start only once its own predecessors (the routing) are complete,
  // so the down kernel's raw producer may read the unit list -- and request its first weight
  // stages -- before its grid-dependency wait; everything that reads h waits.
  if (kGateUp) {
    pdl_wait();
    pdl_trigger();
  } else {
    pdl_trigger();
    if (warp != 0) pdl_wait();
  }

  const int tiles = kGateUp ? a.f / 64 : a.d / BM;
  const int nsub = (kGateUp ? a.d : a.f) / kSubK;          // K slices (4-bit blocks) per unit
  const int nst = (nsub + kSubs - 1) / kSubs;              // stages per unit
  const int npair = (nst + kRawPer - 1) / kRawPer;         // raw copies per unit
  const int total_units = __ldcg(a.n_segs) * tiles;
  const uint8_t* wq = kGateUp ? a.q_gu : a.q_down;

  if (warp == 0) {
    // ---------------- raw 4-bit blocks: one bulk copy per stage (the blocks are adjacent) -----
    // ---------------- also the unit hand-out: publishes this CTA's units in the ring ----------
    const uint64_t pol_w = l2_policy_evict_first();
    uint32_t p = 0;
    bool ok = true, waited = kGateUp;  // down: the first kRawSlots copies go out before the wait
    int u = static_cast<int>(blockIdx.x);
    for (uint32_t i = 0; ok; ++i) {
      const uint32_t rs = i % kUnitRing;
      if (!(ok = mbar_wait_warp(&unit_empty[rs], ((i / kUnitRing) & 1u) ^ 1u, abort_flag, a.err))) break;
      if (lane == 0) {
        unit_ring[rs] = u;
        mbar_arrive(&unit_full[rs]);
      }
      __syncwarp();
      if (u >= total_units) break;
      // the next unit's ticket is requested now and read once this unit's copies are out (the
      // counter is only touched after the grid-dependency wait: it is reset by the previous launch)
      uint32_t ticket = 0;
      bool requested = false;
      if (waited) {
        if (lane == 0) ticket = atomicAdd(a.sched, 1u);
        requested = true;
      }
      const Unit un = waited ? decode_unit(u, a.segs, tiles) : decode_unit<true>(u, a.segs, tiles);
      const uint8_t* w0 = wq + (static_cast<size_t>(un.expert) * tiles + un.tile) * nsub * kFp4BlockBytes;
      for (int kp = 0; kp < npair; ++kp, ++p) {
        if (!waited && p >= static_cast<uint32_t>(kRawSlots)) {
          pdl_wait();
          waited = true;
        }
        const int slot = p % kRawSlots;
        const int sub0 = kRawPer * kSubs * kp;
        const uint32_t bytes = static_cast<uint32_t>(min(kRawPer * kSubs, nsub - sub0)) * kFp4BlockBytes;
        if (!(ok = mbar_wait_warp(&raw_empty[slot], ((p / kRawSlots) & 1u) ^ 1u, abort_flag, a.err))) break;
        if (elect_one()) {
          mbar_arrive_expect_tx(&raw_full[slot], bytes);
          bulk_load(ring_raw + slot * kRawSlotBytes, w0 + static_cast<size_t>(sub0) * kFp4BlockBytes, bytes,
                    &raw_full[slot], pol_w);
        }
        __syncwarp();
      }
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      if (!requested && lane == 0) ticket = atomicAdd(a.sched, 1u);
      u = static_cast<int>(gridDim.x + __shfl_sync(0xffffffffu, ticket, 0));
    }
    if (!waited) pdl_wait();
  } else if (warp == 1) {
    // ---------------- MMA issuer (A from TMEM): the warp waits, one elected lane issues -------
    const uint32_t a_base = tmem + kAStart;
    const uint64_t b_base = smem_desc_sw128(smem_u32(ring_b));
    const uint32_t full_u32 = smem_u32(full), empty_u32 = smem_u32(empty);
    const uint32_t bfull_u32 = smem_u32(b_full), bempty_u32 = smem_u32(b_empty);
    uint32_t g = 0, j = 0;
    bool ok = true, ready = false;  // ready: stage g's A and B barriers already seen complete
    for (uint32_t ui = 0; ok; ++ui, ++j) {
      const int u = ring_unit(unit_ring, unit_full, unit_empty, ui, abort_flag, a.err);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= total_units) break;
      const Unit un = decode_unit(u, a.segs, tiles);
      const uint32_t N = static_cast<uint32_t>(pad16(un.rows));
      const uint32_t buf = j & 1u, use_acc = j >> 1;
      if (!(ok = mbar_wait_warp(&acc_empty[buf], (use_acc & 1u) ^ 1u, abort_flag, a.err))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + buf * kAccCols;
      const uint32_t idesc = idesc_f16_f32(BM, N);
      // The elected lane issues a run of consecutive stages that are already full (testing each
      // next pair of barriers itself), so the warp-wide bookkeeping is paid once per run.
      for (int kk = 0; kk < nst;) {
        const uint32_t s = g % kStages, sb = g % kBStages;
        if (!ready && !(ok = mbar_wait_warp(&full[s], (g / kStages) & 1u, abort_flag, a.err) &&
                             (!kSplitB || mbar_wait_warp(&b_full[sb], (g / kBStages) & 1u, abort_flag, a.err))))
          break;
        tc_fence_after();
        int issued = 0;
        if (elect_one()) {
          // slots and phases advance incrementally: the lane's dependency chain per stage is the
          // address arithmetic, the MMA block, the commits and the next barriers' tests
          uint32_t ss = s, ph = (g / kStages) & 1u, sbb = sb, phb = (g / kBStages) & 1u;
          int k2 = kk;
          while (true) {
            mma_stage_ts<(kSubBytes >> 4)>(d_tmem, a_base + ss * kACols, b_base + sbb * (kBBytes >> 4), idesc,
                                           static_cast<uint32_t>(k2), nsub - kSubs * k2 >= kSubs);
            mma_commit_u32(empty_u32 + 8 * ss);
            if (kSplitB) mma_commit_u32(bempty_u32 + 8 * sbb);
            ++k2, ++issued;
            if (++ss == static_cast<uint32_t>(kStages)) ss = 0, ph ^= 1u;
            if (++sbb == static_cast<uint32_t>(kBStages)) sbb = 0, phb ^= 1u;
            if (k2 >= nst || !mbar_test_u32(full_u32 + 8 * ss, ph) ||
                (kSplitB && !mbar_test_u32(bfull_u32 + 8 * sbb, phb)))
              break;
            tc_fence_after();
          }
        }
        issued = static_cast<int>(__reduce_max_sync(0xffffffffu, static_cast<uint32_t>(issued)));
        kk += issued;
        g += static_cast<uint32_t>(issued);
        // probe the next stage (possibly the next unit's first) now, use the answer next iteration
        ready = __all_sync(0xffffffffu, mbar_test(&full[g % kStages], (g / kStages) & 1u) &&
                                            (!kSplitB || mbar_test(&b_full[g % kBStages], (g / kBStages) & 1u)));
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&acc_full[buf]);
      __syncwarp();
    }
    if (elect_one()) mma_commit(drain);  // completes once every MMA issued above has finished
    __syncwarp();
    mbar_wait_warp(drain, 0, nullptr, a.err);
  } else if (warp < 6) {
    // ---------------- epilogue (as in gemm_tc.cu) ----------------
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
      // 16-column chunks go through a per-warp shared tile [column][row]: the global stores
      // are 16-byte vectors of 8 consecutive features of one token (as in gemm_tc.cu)
      uint16_t* stg = epi_stage + (warp - 2) * (kEpiStageBytes / 2);
      bool sat = false;
      if (kGateUp) {
        const int w16 = L & 15;
        const bool is_gate = w16 < 8;
        const int fl = 8 * ((L >> 4) & 1) + (w16 & 7);
        const int feat0 = un.tile * 64 + 16 * q;
        for (int c0 = 0; c0 < un.rows; c0 += 16) {
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
      } else {
        const int feat0 = un.tile * BM + 32 * q;
        for (int c0 = 0; c0 < un.rows; c0 += 16) {
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
          for (int pass = 0; pass < 2; ++pass) {
            const int idx = 32 * pass + lane;
            const int cl = idx >> 2, g = idx & 3;
            if (c0 + cl < un.rows) {
              const uint4 v = *reinterpret_cast<const uint4*>(stg + cl * 32 + 8 * g);
              *reinterpret_cast<uint4*>(a.y + static_cast<size_t>(un.row_start + c0 + cl) * a.d + feat0 + 8 * g) = v;
            }
          }
          __syncwarp();
        }
      }
      if (__any_sync(0xffffffffu, sat) && lane == 0) set_error(a.err, MOE_DEVERR_RANGE);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  } else if (warp >= kDqWarp) {
    // ---------------- dequantisation into TMEM ----------------
    const int q = warp & 3;       // TMEM lane quarter
    const int r = 32 * q + lane;  // weight row of the tile owned by this thread
    const uint32_t set = static_cast<uint32_t>(warp - kDqWarp) >> 2;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q) << 16) + kAStart;
    uint32_t p = 0, uidx = 0;
    bool ok = true;
    for (uint32_t ui = 0; ok; ++ui, ++uidx) {
      const int u = ring_unit(unit_ring, unit_full, unit_empty, ui, abort_flag, a.err);
      if (u < 0) {
        ok = false;
        break;
      }
      if (u >= total_units) break;
      for (int kp = 0; kp < npair; ++kp, ++p) {
        const int kk = kRawPer * kp + static_cast<int>(set);
        const bool have = kk < nst;  // the last pair of an odd stage count has one stage
        const int sr = p % kRawSlots;
        const uint32_t g = uidx * static_cast<uint32_t>(nst) + static_cast<uint32_t>(kk);
        const int s = g % kStages;
        const int subs = have ? min(kSubs, nsub - kSubs * kk) : 0;
        if (!(ok = mbar_wait_warp(&raw_full[sr], (p / kRawSlots) & 1u, abort_flag, a.err))) break;
        const uint8_t* blk = ring_raw + sr * kRawSlotBytes + set * kRawBytes;
        uint4 c[kSubs][2];
        uint32_t sc[kSubs];
#pragma unroll
        for (int j2 = 0; j2 < kSubs; ++j2) {
          if (j2 < subs) {
            const uint8_t* b = blk + j2 * kFp4BlockBytes;
            c[j2][0] = *reinterpret_cast<const uint4*>(b + r * 16);
            c[j2][1] = *reinterpret_cast<const uint4*>(b + 2048 + r * 16);
            sc[j2] = *reinterpret_cast<const uint16_t*>(b + 4096 + 2 * r);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[sr]);  // the raw bytes are in registers now
        if (!have) continue;
        if (!(ok = mbar_wait_warp(&empty[s], ((g / kStages) & 1u) ^ 1u, abort_flag, a.err))) break;
#pragma unroll
        for (int j2 = 0; j2 < kSubs; ++j2) {
          if (j2 < subs) {
            uint32_t w[32];
            dequant16(c[j2][0], scale_half2(sc[j2] & 0xFFu), w);
            dequant16(c[j2][1], scale_half2(sc[j2] >> 8), w + 16);
            tmem_st_32x32b_x32(trow + s * kACols + 32 * j2, w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
    }
  } else if (!kGateUp) {
    // ---------------- B producer (down): rows of h by TMA ----------------
    // kBProducers warps take turns (stage g: warp 6 + g % kBProducers): each stage needs up to
    // 2 x 4 box loads, and one issuing thread would pace the whole pipeline.
    {
      const int bp = warp - 6;
      const uint64_t pol_act = l2_policy_evict_last();
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
        const int nbox = (pad16(un.rows) + 31) / 32;
        for (int kk = 0; kk < nst; ++kk, ++g) {
          if (static_cast<int>(g % kBProducers) != bp) continue;
          const int sb = g % kBStages;
          const int subs = min(kSubs, nsub - kSubs * kk);
          if (!(ok = mbar_wait_warp(&b_empty[sb], ((g / kBStages) & 1u) ^ 1u, abort_flag, a.err))) break;
          if (elect_one()) {
            mbar_arrive_expect_tx(&b_full[sb], subs * nbox * 32 * kSubK * 2);
            for (int j2 = 0; j2 < subs; ++j2)
              for (int i = 0; i < nbox; ++i)
                tma_load_2d(ring_b + sb * kBBytes + j2 * kSubBytes + i * 32 * kSubK * 2, &maps.h, &b_full[sb],
                            (kSubs * kk + j2) * kSubK, un.row_start + 32 * i, pol_act);
          }
          __syncwarp();
        }
      }
    }
  } else {
    // ---------------- B producer (gate/up): fp16 token rows gathered with cp.async ----------
    // Gather warps w and w + kBStages own B slot w: they fill every stage g with
    // g % kBStages == w (each half of the rows), wait for their own copies, fence them for the
    // tensor core and arrive.  All kBStages slots can be in flight at once, and no copy waits
    // behind the issue of a later stage.
    const int gw = warp - 6;
    const int slot = gw % kBStages, half = gw / kBStages;
    int32_t* tok = tok_tab + kN * gw;           // token row of each row of this warp's unit
    const int ch = lane & 7;                    // 16-byte chunk
    const int rs = (lane >> 3) + 4 * half;      // first row; rows rs + 4 kGatherPerSlot i
    const uint64_t pol_x = l2_policy_evict_last();
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
      for (int kk = 0; kk < nst; ++kk, ++g) {
        const int s = g % kBStages;
        if (s != slot) continue;
        if (!have_tok) {
          for (int n = lane; n < un.rows; n += 32) tok[n] = a.perm[un.row_start + n] / a.k;
          __syncwarp();
          have_tok = true;
        }
        const int subs = min(kSubs, nsub - kSubs * kk);
        if (!(ok = mbar_wait_warp(&b_empty[s], ((g / kBStages) & 1u) ^ 1u, abort_flag, a.err))) break;
        const uint32_t sb = smem_u32(ring_b + s * kBBytes);
        const int k0 = kSubs * kk * kSubK + ch * 8;
        for (int n = rs; n < un.rows; n += 4 * kGatherPerSlot) {
          const uint16_t* src = a.x16 + static_cast<size_t>(tok[n]) * a.d + k0;
          const uint32_t dst = sb + n * 128 + ((ch ^ (n & 7)) << 4);
          cp_async_16_hint(dst, src, pol_x);
          if (subs > 1) cp_async_16_hint(dst + kSubBytes, src + kSubK, pol_x);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&b_full[s]);
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
  // The last CTA to leave resets the hand-out words for the next launch: every CTA's tickets
  // were taken by its thread 0 before this point.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.sched + 1, 1u) == gridDim.x - 1) {
      a.sched[0] = 0u;
      a.sched[1] = 0u;
      __threadfence();
    }
  }
}

}  // namespace fq

template <bool kGateUp, int kN>
static cudaError_t launch_fq_n(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st) {
  auto kern = fq::fp4_ffn_kernel<kGateUp, kN>;
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), fq::Geo<kN>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(num_sms), dim3(fq::Geo<kN>::threads(kGateUp)), fq::Geo<kN>::kSmemBytes, st, *maps, a);
}

// Steps of at most 64 tokens have segments of at most 64 rows: the deeper-ring geometry.
template <bool kGateUp>
static cudaError_t launch_fq(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st) {
  if (!a.sched) return cudaErrorInvalidValue;  // the unit hand-out words are required
  if (a.T <= 64) return launch_fq_n<kGateUp, 64>(maps, a, num_sms, st);
  return launch_fq_n<kGateUp, 128>(maps, a, num_sms, st);
}

cudaError_t launch_fp4_gateup(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st) {
  return launch_fq<true>(maps, a, num_sms, st);
}

cudaError_t launch_fp4_down(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st) {
  return launch_fq<false>(maps, a, num_sms, st);
}

// x (bf16) -> fp16 for the 4-bit path's B operand; exact for 2^-17 <= |x| <= 65504 (and 0),
// larger magnitudes are clamped and flag MOE_DEVERR_RANGE.
__global__ void __launch_bounds__(256) x_to_f16_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ x16,
                                                       size_t n8, uint32_t* err) {
  pdl_trigger();
  pdl_wait();
  XConv c;
  c.x = x, c.x16 = x16, c.n8 = n8;
  convert_x16(c, err);
}

cudaError_t launch_x_to_f16(const uint16_t* x, uint16_t* x16, size_t n, uint32_t* err, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const size_t n8 = n / 8;
  const int blocks = static_cast<int>(n8 / 256 + 1 < 1024 ? n8 / 256 + 1 : 1024);
  return launch_pdl(x_to_f16_kernel, dim3(blocks), dim3(256), 0, st, x, x16, n8, err);
}

}  // namespace moe
