// Top-k selection of one token by one warp, shared by the routing kernels (route.cu) and the
// one-launch small-step layer (layer_small.cu), so that every front end selects identically:
// the total order (value desc, index asc), +0 == -0, NaN below -inf, and softmax gates over the
// k selected logits in fp32.
#pragma once

#include "common.cuh"

namespace moe {

// Ordered 32-bit key of a logit: a larger key ranks first.  A float maps to an unsigned integer
// that grows with its value (-0 is first turned into +0, so the two compare equal); every real
// value maps above 2.  NaN maps to 2, below -inf; 1 marks a padding lane (e >= E) and 0 a
// candidate already taken.  Equal keys rank by expert index, lower first.
MOE_DEVICE uint32_t rank_key(float v) {
  if (isnan(v)) return 2u;
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Selection and gates of token t by one warp from its logits v (lane l holds experts
// l + 32 i): writes ids / gates of the token and returns, in lane j < k, the expert chosen in
// round j.  Each round every lane offers its best remaining candidate (largest key, then lowest
// index); the warp takes the largest key and, among the lanes offering it, the lowest expert.
template <int PL>
MOE_DEVICE int topk_select(const float (&v)[PL], int t, int E, int k, int32_t* __restrict__ ids,
                           float* __restrict__ gates, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  uint32_t key[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) key[i] = lane + 32 * i < E ? rank_key(v[i]) : 1u;
  int sel_i = 0;  // lane j keeps the expert chosen in round j
  for (int j = 0; j < k; ++j) {
    uint32_t best = key[0];
    int bi = 0;
#pragma unroll
    for (int i = 1; i < PL; ++i) {
      const bool gt = key[i] > best;  // strict: the lowest index keeps a tie
      best = gt ? key[i] : best;
      bi = gt ? i : bi;
    }
    const uint32_t win_key = __reduce_max_sync(0xffffffffu, best);
    const uint32_t cand = best == win_key ? static_cast<uint32_t>(lane + 32 * bi) : 0xffffffffu;
    const int win_e = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
    // the owner lane retires the winner (a select per key: the keys stay in registers)
    const bool owner = (win_e & 31) == lane;
#pragma unroll
    for (int i = 0; i < PL; ++i) key[i] = (owner && i == bi) ? 0u : key[i];
    if (lane == j) sel_i = win_e;
  }
  // gates: softmax over the k selected logits, slot 0 holds the maximum
  float sel_v = 0.f;
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const float vi = __shfl_sync(0xffffffffu, v[i], sel_i & 31);
    if (i == (sel_i >> 5)) sel_v = vi;
  }
  const float vmax = __shfl_sync(0xffffffffu, sel_v, 0);
  const float ex = (lane < k) ? expf(sel_v - vmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const bool bad = (lane < k) && !isfinite(sel_v);
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(err, MOE_DEVERR_NONFINITE);
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = sel_i;
    gates[static_cast<size_t>(t) * k + lane] = ex / sum;
  }
  return sel_i;
}

}  // namespace moe
