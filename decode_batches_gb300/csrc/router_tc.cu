// Router logits on the tensor cores for large T.
//
// l[t, e] = x[t] . W_r[e] + b[e] with fp32 router weights.  W_r is split once, at set-up, into
// three bf16 matrices W_r = W1 + W2 + W3 exactly (W1 = bf16(W_r), W2 = bf16(W_r - W1),
// W3 = W_r - W1 - W2, which has at most 8 significant bits left).  x is bf16, so every product
// x * Wp is exact in fp32 and the MMAs accumulate, in fp32 TMEM, the sum an fp32 FMA loop
// would form -- at bf16 tensor-core rate instead of CUDA-core FMA rate.
//
// Tile: 128 experts (M, the A operand) x up to 128 tokens (N, the B operand) x a K range of at
// most 512; both operands arrive by TMA (rows past T are zero-filled).  The tensor core's internal fp32 accumulation loses about 2^-24 of the
// running sum per MMA step, so chains are kept short: W1 accumulates in one TMEM accumulator
// (<= 32 steps per K range) and W2 + W3, 2^-8 smaller, in a second one; the epilogue adds the
// two in IEEE fp32.  Partial sums land in parts[split][t][e] and the top-k kernel adds them in a
// fixed order (deterministic).
// The router of the "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra" post (Decode
// paragraph) is one dispatch; here it is one GEMM launch plus the top-k launch.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace rt {

constexpr int BM = 128;                 // experts per tile
constexpr int BN = 128;                 // tokens per tile
constexpr int BK = 64;
constexpr int kPieces = 3;
constexpr int kStages = 3;
constexpr int kABytes = BM * BK * 2;    // one piece
constexpr int kBBytes = BN * BK * 2;
constexpr int kStageBytes = kPieces * kABytes + kBBytes;  // 64 KB
constexpr int kAccCols = 2 * BN;        // one item: [0, BN) W1 chain, [BN, 2 BN) W2 + W3 chain
constexpr int kTmemCols = 2 * kAccCols;  // two items in flight: 512 columns
constexpr int kSmemBytes = kStages * kStageBytes + 1024 + 1024;
constexpr int kThreads = 192;

// Work item i: expert tile i % tiles_e, then K split, then token tile.
struct Item {
  int e0, t0, rows, split, kc0, kc1;
};

MOE_DEVICE Item decode_item(int i, int tiles_e, int nsplit, int nk, int T) {
  Item it;
  const int rest = i / tiles_e;
  it.e0 = (i % tiles_e) * BM;
  it.split = rest % nsplit;
  it.t0 = (rest / nsplit) * BN;
  it.rows = min(BN, T - it.t0);
  it.kc0 = it.split * nk / nsplit;
  it.kc1 = (it.split + 1) * nk / nsplit;
  return it;
}

// Persistent CTAs (at most one per SM) walk the items b, b + gridDim.x, ...; the stage ring runs
// on across items and the two TMEM accumulator pairs let the epilogue of one item overlap the
// main loop of the next.  Roles: warp 0 TMA producer (the W pieces and the token rows), warp 1
// TMEM owner and MMA issuer, warps 2-5 epilogue (TMEM lanes 32 (warp % 4) ..).
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap w3, const __grid_constant__ CUtensorMap xm, int T, int E,
                     int d, int nsplit, float* __restrict__ parts, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_e = E / BM;
  const int nk = d / BK;
  const int items = tiles_e * ((T + BN - 1) / BN) * nsplit;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&w3);
    tma_prefetch_map(&xm);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();
  pdl_wait();  // x and the previous step's readers of `parts` are done from here on

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();  // W pieces are re-read by every token tile
      uint32_t g = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < items && ok; i += gridDim.x) {
        const Item it = decode_item(i, tiles_e, nsplit, nk, T);
        for (int kc = it.kc0; kc < it.kc1; ++kc, ++g) {
          const int slot = g % kStages;
          if (!(ok = mbar_wait(&empty[slot], ((g / kStages) & 1u) ^ 1u, abort_flag, err))) break;
          uint8_t* sa = smem + slot * kStageBytes;
          mbar_arrive_expect_tx(&full[slot], kPieces * kABytes + kBBytes);
          for (int p = 0; p < kPieces; ++p) tma_load_2d(sa + p * kABytes, &w3, &full[slot], kc * BK, p * E + it.e0, pol);
          tma_load_2d(sa + kPieces * kABytes, &xm, &full[slot], kc * BK, it.t0, pol);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t g = 0, j = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < items && ok; i += gridDim.x, ++j) {
        const Item it = decode_item(i, tiles_e, nsplit, nk, T);
        const uint32_t buf = j & 1u;
        if (!(ok = mbar_wait(&acc_empty[buf], ((j >> 1) & 1u) ^ 1u, abort_flag, err))) break;
        tc_fence_after();
        const uint32_t d1 = tmem + buf * kAccCols;
        const uint32_t N = it.rows <= 16 ? 16u : static_cast<uint32_t>((it.rows + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(BM, N);
        for (int kc = it.kc0; kc < it.kc1; ++kc, ++g) {
          const int slot = g % kStages;
          if (!(ok = mbar_wait(&full[slot], (g / kStages) & 1u, abort_flag, err))) break;
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + slot * kStageBytes);
          const uint64_t bdesc = smem_desc_sw128(sa + kPieces * kABytes);
#pragma unroll
          for (int p = 0; p < kPieces; ++p) {
            const uint64_t adesc = smem_desc_sw128(sa + p * kABytes);
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks) {
              const bool first = kc == it.kc0 && ks == 0 && p != 2;  // p = 2 adds onto the p = 1 chain
              mma_f16_ss(p == 0 ? d1 : d1 + BN, adesc + 2 * ks, bdesc + 2 * ks, idesc, first ? 0u : 1u);
            }
          }
          mma_commit(&empty[slot]);
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
      mma_commit(drain);  // completes once every MMA issued above has
      mbar_wait(drain, 0, nullptr, err);
      if (!ok) *abort_flag = 1;
    }
  } else if (warp < 6) {
    const int q = warp & 3;
    uint32_t j = 0;
    for (int i = blockIdx.x; i < items; i += gridDim.x, ++j) {
      const Item it = decode_item(i, tiles_e, nsplit, nk, T);
      const uint32_t buf = j & 1u;
      if (!mbar_wait(&acc_full[buf], (j >> 1) & 1u, abort_flag, err)) break;
      tc_fence_after();
      const int e = it.e0 + 32 * q + lane;
      float* out = parts + (static_cast<size_t>(it.split) * T + it.t0) * E + e;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * kAccCols;
      for (int c0 = 0; c0 < it.rows; c0 += 16) {
        uint32_t r[16], r2[16];
        tmem_ld_32x32b_x16(tbase + c0, r);
        tmem_ld_32x32b_x16(tbase + BN + c0, r2);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (c0 + c < it.rows) out[static_cast<size_t>(c0 + c) * E] = __uint_as_float(r[c]) + __uint_as_float(r2[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
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

}  // namespace rt

// K splits: at least ceil(d / 512) (short accumulation chains), more while the grid is below
// one CTA per SM (up to 8; 16 for a single token tile, where the whole grid is a few CTAs), at
// most one split per 64-wide K chunk.
int router_tc_splits(int T, int E, int d, int num_sms) {
  const int tiles = (E / rt::BM) * ((T + rt::BN - 1) / rt::BN);
  const int nk = d / rt::BK;
  int s = tiles > 0 ? num_sms / tiles : 1;
  const int s_min = (nk + 7) / 8;
  const int s_cap = T <= rt::BN ? 16 : 8;  // the top-k reads every partial
  if (s > s_cap) s = s_cap;
  if (s < s_min) s = s_min;
  if (s > nk) s = nk;
  if (s < 1) s = 1;
  return s;
}

cudaError_t launch_router_tc(const CUtensorMap* w3, const CUtensorMap* xm, int T, int E, int d, int nsplit,
                             float* parts, uint32_t* err, int num_sms, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(rt::router_tc_kernel), rt::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int items = (E / rt::BM) * ((T + rt::BN - 1) / rt::BN) * nsplit;
  return launch_pdl(rt::router_tc_kernel, dim3(items < num_sms ? items : num_sms), dim3(rt::kThreads), rt::kSmemBytes,
                    st, *w3, *xm, T, E, d, nsplit, parts, err);
}

// W_r (fp32 [E][d]) -> three bf16 matrices [3][E][d] with W1 + W2 + W3 == W_r exactly.
__global__ void split_router_kernel(const float* __restrict__ w, uint16_t* __restrict__ w3, size_t n) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float v = w[i];
    const uint16_t h1 = f32_to_bf16_bits_rn(v);
    const float r1 = v - bf16_bits_to_f32(h1);
    const uint16_t h2 = f32_to_bf16_bits_rn(r1);
    const float r2 = r1 - bf16_bits_to_f32(h2);
    w3[i] = h1;
    w3[n + i] = h2;
    w3[2 * n + i] = f32_to_bf16_bits_rn(r2);
  }
}

cudaError_t launch_split_router(const float* w, uint16_t* w3, size_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  split_router_kernel<<<1024, 256, 0, st>>>(w, w3, n);
  return cudaGetLastError();
}

}  // namespace moe
