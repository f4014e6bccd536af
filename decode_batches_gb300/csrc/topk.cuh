// Top-k selection of one token by one warp, shared by the routing kernels (route.cu) and the
// one-launch small-step layer (layer_small.cu), so that every front end selects identically:
// the total order (value desc, index asc), +0 == -0, NaN below -inf, and softmax gates over the
// k selected logits in fp32.
#pragma once

#include "common.cuh"

namespace moe {

// Sortable 64-bit key of (logit v, expert e): a larger key ranks first.  The high word maps the
// float to an unsigned integer that grows with v (-0 is first turned into +0, so the two
// compare equal); NaN maps to 0, below -inf.  The low word is ~e, so on equal values the lower
// index ranks first.  Padding lanes (e >= E) get key 0, below every real candidate.
MOE_DEVICE uint64_t rank_key(float v, int e) {
  uint32_t hi = 0u;
  if (!isnan(v)) {
    const uint32_t b = __float_as_uint(v + 0.0f);
    hi = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  return (static_cast<uint64_t>(hi) << 32) | static_cast<uint32_t>(~e);
}

// Selection and gates of token t by one warp from its logits v (lane l holds experts
// l + 32 i): writes ids / gates of the token and returns, in lane j < k, the expert chosen in
// round j.
template <int PL>
MOE_DEVICE int topk_select(const float (&v)[PL], int t, int E, int k, int32_t* __restrict__ ids,
                           float* __restrict__ gates, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  uint64_t key[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? rank_key(v[i], e) : 0ull;
  }
  int sel_i = 0;  // lane j keeps the expert chosen in round j
  for (int j = 0; j < k; ++j) {
    uint64_t best = key[0];
#pragma unroll
    for (int i = 1; i < PL; ++i) best = key[i] > best ? key[i] : best;
    const uint32_t hi = static_cast<uint32_t>(best >> 32);
    const uint32_t win_hi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t win_lo = __reduce_max_sync(0xffffffffu, hi == win_hi ? static_cast<uint32_t>(best) : 0u);
    const int win_e = static_cast<int>(~win_lo);
    // the owner lane retires the winner (a select per key: the keys stay in registers)
    const int win_slot = (win_e & 31) == lane ? (win_e >> 5) : -1;
#pragma unroll
    for (int i = 0; i < PL; ++i) key[i] = i == win_slot ? 0ull : key[i];
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
