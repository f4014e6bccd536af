// Routing and grouping kernels of the MoE layer.
//
//   router logits      l[t,e] = x[t] . W_r[e] + b[e]        (fp32 accumulation)
//   top-k + gates      warp per token; total order (value desc, index asc), NaN lowest;
//                      gates = softmax of the k selected logits (fp32)
//   grouping           per 32-token chunk a 32-bit mask per expert; one launch reads the
//                      masks for counts, exclusive offsets and chunk bases and ranks each
//                      assignment inside its chunk with one popcount, so the permutation is a
//                      stable counting sort with no atomics-order dependence (identical on
//                      every run).  Steps of at most 64 assignments
//                      sort unique (expert, assignment) keys in one warp instead (group_tiny):
//                      the same permutation, with one block barrier.
// Sources: "DeepSeek V4.1F Q4 with native DSpark MTP on M3 Ultra", Decode paragraph (the
// 384-expert router and its top-k in one dispatch); "Why SSD-streamed MoE was slow: 8GB Jetson
// Orin Nano, part 2", the `mul_mat_id` grouped matmul and the section on generated text
// changing between runs (every chosen expert computed exactly once -> bijection checks).
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

// ============================================================================================
// Router logits
// ============================================================================================

// Small T: one warp per expert and up to kTokTile tokens per block row (grid.y covers T).
// Each lane walks its 8-element slices of d; W_r[e] is read once per block row.
template <int kTokTile>
__global__ void __launch_bounds__(256) router_logits_small_kernel(const uint16_t* __restrict__ x,
                                                                  const float* __restrict__ wr,
                                                                  const float* __restrict__ br, int T,
                                                                  int E, int d,
                                                                  float* __restrict__ logits) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const int t0 = blockIdx.y * kTokTile;
  if (e >= E) return;
  const int nt = min(kTokTile, T - t0);
  float acc[kTokTile];
#pragma unroll
  for (int t = 0; t < kTokTile; ++t) acc[t] = 0.f;
  const float* w = wr + static_cast<size_t>(e) * d;
  for (int i = lane * 8; i < d; i += 256) {
    const float4 w0 = *reinterpret_cast<const float4*>(w + i);
    const float4 w1 = *reinterpret_cast<const float4*>(w + i + 4);
#pragma unroll
    for (int t = 0; t < kTokTile; ++t) {
      if (t < nt) {
        const uint4 xv = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + t) * d + i);
        float xf[8];
        bf16x8_to_f32(xv, xf);
        float a = acc[t];
        a = fmaf(xf[0], w0.x, a);
        a = fmaf(xf[1], w0.y, a);
        a = fmaf(xf[2], w0.z, a);
        a = fmaf(xf[3], w0.w, a);
        a = fmaf(xf[4], w1.x, a);
        a = fmaf(xf[5], w1.y, a);
        a = fmaf(xf[6], w1.z, a);
        a = fmaf(xf[7], w1.w, a);
        acc[t] = a;
      }
    }
  }
  const float bias = br ? br[e] : 0.f;
#pragma unroll
  for (int t = 0; t < kTokTile; ++t) {
    if (t < nt) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) logits[static_cast<size_t>(t0 + t) * E + e] = v + bias;
    }
  }
}

// Large T: 64 tokens x 64 experts per block, 32-deep K slices staged in shared memory,
// 4 x 4 outputs per thread.
__global__ void __launch_bounds__(256) router_logits_tiled_kernel(const uint16_t* __restrict__ x,
                                                                  const float* __restrict__ wr,
                                                                  const float* __restrict__ br, int T,
                                                                  int E, int d,
                                                                  float* __restrict__ logits) {
  constexpr int BM = 64, BN = 64, BK = 32;
  pdl_trigger();
  pdl_wait();
  __shared__ float xs[BK][BM + 4];
  __shared__ float ws[BK][BN + 4];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * BM, e0 = blockIdx.y * BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += BK) {
    // x tile: 64 rows x 32 bf16 = 256 chunks of 8
    {
      const int r = tid >> 2, c = (tid & 3) * 8;
      float xf[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (t0 + r < T) {
        const uint4 xv = *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + r) * d + k0 + c);
        bf16x8_to_f32(xv, xf);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) xs[c + q][r] = xf[q];
    }
    // w tile: 64 rows x 32 fp32 = 512 float4
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int idx = tid + rep * 256;
      const int r = idx >> 3, c = (idx & 7) * 4;
      float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + r < E) wv = *reinterpret_cast<const float4*>(wr + static_cast<size_t>(e0 + r) * d + k0 + c);
      ws[c + 0][r] = wv.x;
      ws[c + 1][r] = wv.y;
      ws[c + 2][r] = wv.z;
      ws[c + 3][r] = wv.w;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) logits[static_cast<size_t>(t) * E + e] = acc[i][j] + (br ? br[e] : 0.f);
    }
  }
}

// Small T, K split: block (8 experts, one 512-wide K slice); the slice of every token's x is
// staged in shared memory (G tokens at a time) and each warp forms its expert's partial dot
// products: lane l holds W_r[e][k0 + 4 l + 128 q + c], q < 4, c < 4.  Partials go to
// parts[split][t][e] and the top-k adds them in split order (deterministic).  d % 128 == 0.
constexpr int kRouterKS = 512;

int router_small_splits(int d) { return (d + kRouterKS - 1) / kRouterKS; }

template <int G>  // tokens per group, a power of two <= 32; xs: G * kRouterKS shared elements
MOE_DEVICE void router_parts_block(const uint16_t* __restrict__ x, const float* __restrict__ wr, int T, int E, int d,
                                   float* __restrict__ parts, uint16_t* xs) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const int sp = blockIdx.y;
  const int k0 = sp * kRouterKS;
  const int ks = min(kRouterKS, d - k0);  // multiple of 128
  float4 w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int kk = 4 * lane + 128 * q;
    w[q] = (e < E && kk < ks) ? *reinterpret_cast<const float4*>(wr + static_cast<size_t>(e) * d + k0 + kk)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int t0 = 0; t0 < T; t0 += G) {
    const int nt = min(G, T - t0);
    __syncthreads();  // the previous group's readers are done
    for (int i = threadIdx.x; i < nt * (ks / 8); i += blockDim.x) {
      const int tl = i / (ks / 8), c8 = i % (ks / 8);
      *reinterpret_cast<uint4*>(xs + tl * kRouterKS + 8 * c8) =
          *reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + tl) * d + k0 + 8 * c8);
    }
    __syncthreads();
    if (e < E) {
      // lane-partial dot products of the group's G tokens (rows past nt read stale shared
      // memory and are never stored)
      float acc[G];
#pragma unroll
      for (int tl = 0; tl < G; ++tl) {
        float a = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int kk = 4 * lane + 128 * q;
          if (kk < ks) {
            const uint2 xv = *reinterpret_cast<const uint2*>(xs + tl * kRouterKS + kk);
            a = fmaf(bf16_bits_to_f32(static_cast<uint16_t>(xv.x & 0xFFFFu)), w[q].x, a);
            a = fmaf(bf16_bits_to_f32(static_cast<uint16_t>(xv.x >> 16)), w[q].y, a);
            a = fmaf(bf16_bits_to_f32(static_cast<uint16_t>(xv.y & 0xFFFFu)), w[q].z, a);
            a = fmaf(bf16_bits_to_f32(static_cast<uint16_t>(xv.y >> 16)), w[q].w, a);
          }
        }
        acc[tl] = a;
      }
      // transposing butterfly over lane bits below G: after the level for offset o a lane
      // keeps the half of its values whose index has the lane's bit o, so lane l ends with
      // token (l mod G) summed over the lanes that agree with it above bit log2(G); plain
      // butterflies over the remaining bits finish the sums
#pragma unroll
      for (int o = G / 2; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
          const float send = upper ? acc[i] : acc[i + o];
          const float keep = upper ? acc[i + o] : acc[i];
          acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
#pragma unroll
      for (int o = G; o < 32; o <<= 1) acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], o);
      if (lane < nt) parts[(static_cast<size_t>(sp) * T + t0 + lane) * E + e] = acc[0];
    }
  }
}

template <int G>
__global__ void __launch_bounds__(256, 1) router_parts_small_kernel(const uint16_t* __restrict__ x,
                                                                 const float* __restrict__ wr, int T, int E, int d,
                                                                 float* __restrict__ parts) {
  __shared__ __align__(16) uint16_t xs[G * kRouterKS];
  pdl_trigger();
  pdl_wait();
  router_parts_block<G>(x, wr, T, E, d, parts, xs);
}

cudaError_t launch_router_parts_small(const uint16_t* x, const float* w_router, int T, int E, int d, float* parts,
                                      cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  dim3 grid((E + 7) / 8, router_small_splits(d));
  if (T <= 8) return launch_pdl(router_parts_small_kernel<8>, grid, dim3(256), 0, st, x, w_router, T, E, d, parts);
  if (T <= 16) return launch_pdl(router_parts_small_kernel<16>, grid, dim3(256), 0, st, x, w_router, T, E, d, parts);
  return launch_pdl(router_parts_small_kernel<32>, grid, dim3(256), 0, st, x, w_router, T, E, d, parts);
}

cudaError_t launch_router_logits(const uint16_t* x, const float* w_router, const float* b_router, int T,
                                 int E, int d, float* logits, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  if (T <= 128) {
    dim3 grid((E + 7) / 8, (T + 15) / 16);
    return launch_pdl(router_logits_small_kernel<16>, grid, dim3(256), 0, st, x, w_router, b_router, T, E, d, logits);
  } else {
    dim3 grid((T + 63) / 64, (E + 63) / 64);
    return launch_pdl(router_logits_tiled_kernel, grid, dim3(256), 0, st, x, w_router, b_router, T, E, d, logits);
  }
}

// ============================================================================================
// Top-k with gates
// ============================================================================================

// Two blocks per 32-token chunk (16 tokens each), one warp per token.  Lane l holds the
// logits of experts l, l + 32, ..., l + 32 (PL - 1); topk_select takes k rounds of a warp-wide
// maximum.  Masks are stored expert-major, masks[e * mstride + c], bit tl for token tl of the
// chunk: each block writes its 16-bit half of the word.  The logits are the sum of `nsplit`
// partial matrices parts[s][T][E] (s ascending) plus the optional bias; they are written to
// logits_out if given.
constexpr int kTopkTokens = kChunk / 2;       // tokens per block
constexpr int kTopkThreads = 32 * kTopkTokens;

// Top-k of token t by one warp: sums the partial logits (split order fixed) and the bias,
// optionally stores the logits, then selects (topk_select).
template <int PL>
MOE_DEVICE int topk_token(const float* __restrict__ parts, int nsplit, const float* __restrict__ bias,
                          float* __restrict__ logits_out, int t, int T, int E, int k, int32_t* __restrict__ ids,
                          float* __restrict__ gates, uint32_t* err) {
  const int lane = threadIdx.x & 31;
  // U partial matrices in flight at a time (one L2 round trip per U splits), added in order
  constexpr int U = PL <= 8 ? 4 : (PL <= 16 ? 2 : 1);
  float v[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) v[i] = 0.f;
  for (int sp = 0; sp < nsplit; sp += U) {
    float w[U][PL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float* ps = parts + (static_cast<size_t>(sp + u) * T + t) * E;
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane + 32 * i;
        w[u][i] = (e < E && sp + u < nsplit) ? ps[e] : 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int i = 0; i < PL; ++i)
        if (sp + u < nsplit) v[i] = (sp + u == 0) ? w[u][i] : v[i] + w[u][i];
  }
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      if (bias) v[i] += bias[e];
      if (logits_out) logits_out[static_cast<size_t>(t) * E + e] = v[i];
    }
  }
  return topk_select<PL>(v, t, E, k, ids, gates, err);
}

template <int PL>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const float* __restrict__ parts, int nsplit,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits_out, int T, int E, int k,
                                                            int n_chunks, int32_t* __restrict__ ids,
                                                            float* __restrict__ gates,
                                                            uint32_t* __restrict__ masks, uint32_t* err,
                                                            const XConv xc) {
  extern __shared__ uint32_t smask[];  // [E]: bits of this block's 16 tokens
  pdl_trigger();
  pdl_wait();
  convert_x16(xc, err);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x >> 1, half = blockIdx.x & 1;
  if (masks)
    for (int e = threadIdx.x; e < E; e += blockDim.x) smask[e] = 0u;
  __syncthreads();
  const int t = c * kChunk + kTopkTokens * half + warp;
  if (t < T) {
    const int sel = topk_token<PL>(parts, nsplit, bias, logits_out, t, T, E, k, ids, gates, err);
    if (masks && lane < k) atomicOr(&smask[sel], 1u << warp);
  }
  if (masks) {
    __syncthreads();
    // little-endian: half h of the 32-bit mask word is the 16-bit word 2 w + h
    uint16_t* m16 = reinterpret_cast<uint16_t*>(masks);
    const size_t mstride = group_mask_stride(n_chunks);
    for (int e = threadIdx.x; e < E; e += blockDim.x)
      m16[2 * (static_cast<size_t>(e) * mstride + c) + half] = static_cast<uint16_t>(smask[e]);
  }
}

template <int PL>
static cudaError_t launch_topk_pl(const float* parts, int nsplit, const float* bias, float* logits_out, int T, int E,
                                  int k, int n_chunks, int32_t* ids, float* gates, uint32_t* masks, uint32_t* err,
                                  const XConv& xc, cudaStream_t st) {
  return launch_pdl(topk_kernel<PL>, dim3(2 * n_chunks), dim3(kTopkThreads), masks ? E * sizeof(uint32_t) : 0, st,
                    parts, nsplit, bias, logits_out, T, E, k, n_chunks, ids, gates, masks, err, xc);
}

cudaError_t launch_topk(const float* parts, int nsplit, const float* bias, float* logits_out, int T, int E, int k,
                        int32_t* ids, float* gates, uint32_t* masks, uint32_t* err, cudaStream_t st, const XConv& xc) {
  if (T <= 0) return cudaSuccess;
  const int n_chunks = (T + kChunk - 1) / kChunk;
  const int pl = (E + 31) / 32;
#define MOE_TOPK(PLV) \
  launch_topk_pl<PLV>(parts, nsplit, bias, logits_out, T, E, k, n_chunks, ids, gates, masks, err, xc, st)
  if (pl <= 1) return MOE_TOPK(1);
  if (pl <= 2) return MOE_TOPK(2);
  if (pl <= 4) return MOE_TOPK(4);
  if (pl <= 8) return MOE_TOPK(8);
  if (pl <= 12) return MOE_TOPK(12);
  if (pl <= 16) return MOE_TOPK(16);
  return MOE_TOPK(32);
#undef MOE_TOPK
}

// ============================================================================================
// Grouping
// ============================================================================================

// Assignment (t, j) is used iff its id is in range and no earlier slot of the token has it.
MOE_DEVICE bool assignment_valid(const int32_t* __restrict__ ids_row, int j, int e, int E) {
  if (e < 0 || e >= E) return false;
  for (int q = 0; q < j; ++q)
    if (ids_row[q] == e) return false;
  return true;
}

__global__ void __launch_bounds__(256) masks_from_ids_kernel(const int32_t* __restrict__ ids, int T, int E,
                                                             int k, int n_chunks, uint32_t* __restrict__ masks,
                                                             uint32_t* err) {
  extern __shared__ uint32_t smask[];
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) smask[e] = 0u;
  __syncthreads();
  for (int a = threadIdx.x; a < kChunk * k; a += blockDim.x) {
    const int tl = a / k, j = a % k;
    const int t = c * kChunk + tl;
    if (t >= T) continue;
    const int32_t* row = ids + static_cast<size_t>(t) * k;
    const int e = row[j];
    if (!assignment_valid(row, j, e, E)) {
      set_error(err, MOE_DEVERR_EXPERT_RANGE);
      continue;
    }
    atomicOr(&smask[e], 1u << tl);
  }
  __syncthreads();
  const size_t mstride = group_mask_stride(n_chunks);
  for (int e = threadIdx.x; e < E; e += blockDim.x) masks[static_cast<size_t>(e) * mstride + c] = smask[e];
}

cudaError_t launch_masks_from_ids(const int32_t* ids, int T, int E, int k, uint32_t* masks,
                                  uint32_t* err, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int n_chunks = (T + kChunk - 1) / kChunk;
  return launch_pdl(masks_from_ids_kernel, dim3(n_chunks), dim3(256), E * sizeof(uint32_t), st, ids, T, E, k, n_chunks,
                    masks, err);
}

// Exclusive scan over the block (blockDim.x a multiple of 32, <= 1024) of v; *total = block sum.
MOE_DEVICE int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int warp_excl = warp == 0 ? 0 : warp_sums[warp - 1];
  *total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return warp_excl + inc - v;
}

// Split `total` rows of expert e (starting at grouped row `start`) into near-equal segments of
// at most kSegRowsMax rows; `base` is the index of the expert's first segment.
MOE_DEVICE int num_segments(int total) { return (total + kSegRowsMax - 1) / kSegRowsMax; }

MOE_DEVICE void write_segments(Seg* segs, int base, int max_segs, int e, int start, int total,
                               uint32_t* err) {
  const int ns = num_segments(total);
  if (ns == 0) return;
  const int q = total / ns, rem = total % ns;
  int r = start;
  for (int s = 0; s < ns; ++s) {
    const int rows = q + (s < rem ? 1 : 0);
    if (base + s < max_segs) {
      segs[base + s] = Seg{e, r, rows, base, ns, 0, 0, 0};
    } else {
      set_error(err, MOE_DEVERR_SEGMENT);
    }
    r += rows;
  }
}

constexpr int kScanThreads = 256;
constexpr int kScanPerThread = 1024 / kScanThreads;  // E <= 1024

// Block-wide exclusive scan of counts[0..E) into s_off[0..E]; returns the total.
MOE_DEVICE int block_offsets(const int32_t* __restrict__ counts, int E, int* s_off) {
  int c[kScanPerThread];
  int mine = 0;
#pragma unroll
  for (int q = 0; q < kScanPerThread; ++q) {
    const int e = threadIdx.x * kScanPerThread + q;
    c[q] = e < E ? counts[e] : 0;
    mine += c[q];
  }
  int total;
  int run = block_exclusive_scan(mine, &total);
#pragma unroll
  for (int q = 0; q < kScanPerThread; ++q) {
    const int e = threadIdx.x * kScanPerThread + q;
    if (e < E) s_off[e] = run;
    run += c[q];
  }
  if (threadIdx.x == 0) s_off[E] = total;
  __syncthreads();
  return total;
}

// Grouping from the per-chunk expert masks in one launch.  masks[e * mstride + c] holds bit tl
// for token 32 c + tl of chunk c when that token chose expert e (valid assignments only);
// mstride is a multiple of 4, so a mask row is read as 16-byte vectors.  Block b owns the
// chunks [b cpb, (b + 1) cpb).  Every block first reads the whole mask matrix (a few threads
// per expert): each expert's total, its count in the chunks before the block's, and the block's
// own mask words; a block scan of the totals gives the offsets.  Each assignment of the block's
// chunks then takes its row from shared memory alone -- a stable counting sort:
//   row = offsets[e] + (rows of e before the block) + (rows of e in the block's earlier chunks)
//         + popc(mask word & bits of the earlier tokens of the chunk).
// An assignment whose id is out of range or repeats an earlier slot gets inv = -1 (the mask
// builder flags it).  Block 0 also writes counts, offsets and, if segs is given, the segment
// list of the grouped GEMMs.
constexpr int kGroupThreads = 1024;
constexpr int kGroupBlocksMax = 256;
constexpr int kGroupLoads = 8;  // 16-byte mask loads in flight per thread

static int group_cpb(int n_chunks) {
  return n_chunks <= kGroupBlocksMax ? 1 : (n_chunks + kGroupBlocksMax - 1) / kGroupBlocksMax;
}

__global__ void __launch_bounds__(kGroupThreads) group_kernel(
    const int32_t* __restrict__ ids, const uint32_t* __restrict__ masks, int mstride, int T, int E, int k,
    int n_chunks, int cpb, int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, Seg* segs, int32_t* n_segs, int max_segs, uint32_t* err) {
  extern __shared__ int g_sm[];
  int* s_tot = g_sm;                                            // [E]
  int* s_pre = s_tot + E;                                       // [E]: rows of e before chunk c0
  int* s_off = s_pre + E;                                       // [E + 1]
  uint32_t* s_w = reinterpret_cast<uint32_t*>(s_off + E + 1);  // [cpb][E]: the block's mask words
  int32_t* s_ids = reinterpret_cast<int32_t*>(s_w + cpb * E);  // [cpb * 32][k]: the block's ids
  pdl_trigger();
  pdl_wait();
  const int c0 = blockIdx.x * cpb, c1 = min(c0 + cpb, n_chunks);
  // the block's ids: the first share is requested now and lands while the masks are read
  const int nt = max(0, min(cpb * kChunk, T - c0 * kChunk));  // tokens of the block
  const int na = nt * k;
  const int32_t* ids_blk = ids + static_cast<size_t>(c0) * kChunk * k;
  const int id0 = static_cast<int>(threadIdx.x) < na ? ids_blk[threadIdx.x] : 0;
  // threads per expert: a power of two <= 32 (consecutive lanes of one warp)
  int tpe = 1;
  while (tpe < 32 && 2 * tpe * E <= kGroupThreads) tpe *= 2;
  const int e = threadIdx.x / tpe, q = threadIdx.x % tpe;
  int tot = 0, pre = 0;
  if (e < E) {
    const uint4* row = reinterpret_cast<const uint4*>(masks + static_cast<size_t>(e) * mstride);
    const int n4 = (n_chunks + 3) / 4;
    for (int i0 = q; i0 < n4; i0 += kGroupLoads * tpe) {
      uint4 v[kGroupLoads];
#pragma unroll
      for (int u = 0; u < kGroupLoads; ++u) {  // every load of the batch before any use
        const int i = i0 + u * tpe;
        v[u] = i < n4 ? __ldcg(row + i) : make_uint4(0u, 0u, 0u, 0u);  // written by the previous launch
      }
#pragma unroll
      for (int u = 0; u < kGroupLoads; ++u) {
        const int cb = 4 * (i0 + u * tpe);  // chunk of the vector's first word
        if (cb + 3 < n_chunks && (cb + 3 < c0 || cb >= c1)) {
          // the common case: four mask words, none of them the block's own or padding
          const int pc = __popc(v[u].x) + __popc(v[u].y) + __popc(v[u].z) + __popc(v[u].w);
          tot += pc;
          if (cb < c0) pre += pc;
        } else if (cb < n_chunks) {
          const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int c = cb + b;
            const int pc = c < n_chunks ? __popc(w[b]) : 0;  // the row's padding words are not masks
            tot += pc;
            if (c < c0) pre += pc;
            else if (c < c1) s_w[(c - c0) * E + e] = w[b];
          }
        }
      }
    }
  }
  for (int o = 1; o < tpe; o <<= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    pre += __shfl_xor_sync(0xffffffffu, pre, o);
  }
  if (q == 0 && e < E) {
    s_tot[e] = tot;
    s_pre[e] = pre;
  }
  if (static_cast<int>(threadIdx.x) < na) s_ids[threadIdx.x] = id0;
  for (int a = threadIdx.x + blockDim.x; a < na; a += blockDim.x) s_ids[a] = ids_blk[a];
  __syncthreads();
  int total;
  const int mine = static_cast<int>(threadIdx.x) < E ? s_tot[threadIdx.x] : 0;
  const int ex = block_exclusive_scan(mine, &total);
  if (static_cast<int>(threadIdx.x) < E) s_off[threadIdx.x] = ex;
  if (threadIdx.x == 0) s_off[E] = total;
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int x = threadIdx.x; x <= E; x += blockDim.x) {
      offsets[x] = s_off[x];
      if (x < E) counts[x] = s_tot[x];
    }
    if (segs) {
      const int ns = static_cast<int>(threadIdx.x) < E ? num_segments(mine) : 0;
      int seg_total;
      const int base = block_exclusive_scan(ns, &seg_total);
      if (static_cast<int>(threadIdx.x) < E) write_segments(segs, base, max_segs, threadIdx.x, ex, mine, err);
      if (threadIdx.x == 0) *n_segs = min(seg_total, max_segs);
    }
  }
  for (int a = threadIdx.x; a < na; a += blockDim.x) {
    const int tb = a / k, j = a % k;  // token within the block, slot
    const int32_t* id_row = s_ids + tb * k;
    const int ee = id_row[j];
    const size_t ai = (static_cast<size_t>(c0) * kChunk + tb) * k + j;
    if (!assignment_valid(id_row, j, ee, E)) {
      inv[ai] = -1;
      continue;
    }
    const int cc = tb / kChunk, tl = tb % kChunk;
    int r = s_off[ee] + s_pre[ee];
    for (int c2 = 0; c2 < cc; ++c2) r += __popc(s_w[c2 * E + ee]);
    r += __popc(s_w[cc * E + ee] & ((1u << tl) - 1u));
    perm[r] = static_cast<int32_t>(ai);
    inv[ai] = r;
  }
}

cudaError_t launch_group(const int32_t* ids, const uint32_t* masks, int T, int E, int k, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv, Seg* segs, int32_t* n_segs, int max_segs,
                         uint32_t* err, cudaStream_t st) {
  const int n_chunks = (T + kChunk - 1) / kChunk;
  const int cpb = group_cpb(n_chunks);
  const int blocks = n_chunks > 0 ? (n_chunks + cpb - 1) / cpb : 1;
  const size_t smem =
      (3 * static_cast<size_t>(E) + 1 + static_cast<size_t>(cpb) * E + static_cast<size_t>(cpb) * kChunk * k) *
      sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(group_kernel), static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(group_kernel, dim3(blocks), dim3(kGroupThreads), smem, st, ids, masks, group_mask_stride(n_chunks),
                    T, E, k, n_chunks, cpb, counts, offsets, perm, inv, segs, n_segs, max_segs, err);
}

// Routing and grouping of a small step in one launch.  One block per token adds its partial
// logits (every load of the block issued at once; split order fixed, then the bias: the same
// arithmetic as the top-k kernel) into shared memory, and one warp selects the top k and
// publishes ids / gates.  The last block to finish (a counter the plan owns, reset by that
// block) groups the step: per-chunk expert masks from the ids, counts, chunk bases, offsets,
// segments and the stable scatter -- the steps of the masks and group launches, without their
// launches.  Needs route_small_ok(T, E, k, nsplit).
constexpr int kSmallSplitsMax = 16;
constexpr int kRgThreads = 256;
constexpr int kRgPer = 4;  // experts per thread (E <= 1024)

size_t route_small_smem(int T, int E, int k) {
  const int nch = (T + kChunk - 1) / kChunk;
  const size_t grouping = (2 * static_cast<size_t>(nch) * E + static_cast<size_t>(T) * k + E + 1) * 4;
  const size_t logits = static_cast<size_t>(E) * 4;
  return grouping > logits ? grouping : logits;
}

// Grouping of a small step by one block of kRgThreads threads, from the step's ids held in
// shared memory: per-chunk expert masks, counts, chunk bases, offsets, segments and the
// stable scatter (the steps of the group launch).  sm: [2 n_chunks E] words of scratch, then
// ids [T][k], then [E + 1] words.
MOE_DEVICE void group_small(int T, int E, int k, uint32_t* sm, int32_t* __restrict__ counts,
                            int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                            Seg* segs, int32_t* n_segs, int max_segs, uint32_t* err) {
  const int nch = (T + kChunk - 1) / kChunk;
  uint32_t* smask = sm;                                        // [e][c]: bit tl = token c*32+tl chose e
  int32_t* scb = reinterpret_cast<int32_t*>(smask + nch * E);  // [e][c]: rows of e before chunk c
  int32_t* sids = scb + nch * E;                               // [T][k]
  int* s_off = sids + T * k;                                   // [E + 1]
  for (int i = threadIdx.x; i < nch * E; i += kRgThreads) smask[i] = 0u;
  __syncthreads();
  for (int a = threadIdx.x; a < T * k; a += kRgThreads) {
    const int tt = a / k, j = a % k;
    const int e = sids[a];
    if (assignment_valid(sids + tt * k, j, e, E)) atomicOr(&smask[e * nch + tt / kChunk], 1u << (tt % kChunk));
  }
  __syncthreads();
  // experts threadIdx.x * per + q, q < per (contiguous, so one block scan orders them)
  const int per = (E + kRgThreads - 1) / kRgThreads;  // <= kRgPer
  int cl[kRgPer], mine = 0;
#pragma unroll
  for (int q = 0; q < kRgPer; ++q) {
    cl[q] = 0;
    const int e = threadIdx.x * per + q;
    if (q < per && e < E) {
      int run = 0;
      for (int c = 0; c < nch; ++c) {
        scb[e * nch + c] = run;
        run += __popc(smask[e * nch + c]);
      }
      counts[e] = run;
      cl[q] = run;
      mine += run;
    }
  }
  int total;
  int base = block_exclusive_scan(mine, &total);
#pragma unroll
  for (int q = 0; q < kRgPer; ++q) {
    const int e = threadIdx.x * per + q;
    if (q < per && e < E) s_off[e] = base;
    base += cl[q];
  }
  if (threadIdx.x == 0) s_off[E] = total;
  if (segs) {
    int nsl[kRgPer], ns_mine = 0;
#pragma unroll
    for (int q = 0; q < kRgPer; ++q) {
      const int e = threadIdx.x * per + q;
      nsl[q] = (q < per && e < E) ? num_segments(cl[q]) : 0;
      ns_mine += nsl[q];
    }
    int seg_total;
    int sbase = block_exclusive_scan(ns_mine, &seg_total);  // also publishes s_off (barriers)
#pragma unroll
    for (int q = 0; q < kRgPer; ++q) {
      const int e = threadIdx.x * per + q;
      if (q < per && e < E) write_segments(segs, sbase, max_segs, e, s_off[e], cl[q], err);
      sbase += nsl[q];
    }
    if (threadIdx.x == 0) *n_segs = min(seg_total, max_segs);
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += kRgThreads) offsets[e] = s_off[e];
  for (int a = threadIdx.x; a < T * k; a += kRgThreads) {
    const int tt = a / k, j = a % k;
    const int32_t* row = sids + tt * k;
    const int e = row[j];
    if (!assignment_valid(row, j, e, E)) {
      inv[a] = -1;
      continue;
    }
    const int c = tt / kChunk, tl = tt % kChunk;
    const int r = s_off[e] + scb[e * nch + c] + __popc(smask[e * nch + c] & ((1u << tl) - 1u));
    perm[r] = a;
    inv[a] = r;
  }
}

// Largest step that group_tiny takes: its 64 sort keys, two per lane of one warp.
constexpr int kTinyGroupRows = 64;

// One compare-exchange stage of a bitonic network over the warp: this lane's key and the key
// of lane ^ d; the lower lane of the pair keeps the smaller key when the run ascends.
MOE_DEVICE uint32_t bitonic_ce_shfl(uint32_t v, int lane, int d, bool ascending) {
  const uint32_t o = __shfl_xor_sync(0xffffffffu, v, d);
  const bool lower = (lane & d) == 0;
  return (lower == ascending) ? min(v, o) : max(v, o);
}

// The same grouping as group_small for steps of at most kTinyGroupRows assignments (T·k <= 64,
// so every expert has at most 64 rows and one segment).  group_small takes about a dozen
// block-wide steps, each a barrier apart; here one warp does the ordering in registers and the
// block meets once.  Each valid assignment a = t·k + j becomes the key (expert << 8) | a
// (invalid ones -- an id out of range or repeated within the token -- 0xFFFFFFFF), and a bitonic
// network sorts the 64 keys (lane l holds positions l and l + 32).  The keys are unique, so the
// sorted position of a key is exactly its row in the stable counting sort by expert: rows of one
// expert ascend by a.  Segments start where the expert changes; counts and offsets come from
// a binary search of the sorted keys by every thread of the block.  sids: the step's ids [T][k]
// in shared memory.  Every thread of the block calls it.
MOE_DEVICE void group_tiny(int T, int E, int k, const int32_t* sids, int32_t* __restrict__ counts,
                           int32_t* __restrict__ offsets, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                           Seg* segs, int32_t* n_segs, int max_segs, uint32_t* err) {
  constexpr uint32_t kNone = 0xFFFFFFFFu;
  __shared__ uint32_t s_keys[kTinyGroupRows];
  const int R = T * k;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t key[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int a = lane + 32 * h;
      key[h] = kNone;
      if (a < R) {
        const int t = a / k, j = a - t * k;
        const int e = sids[a];
        if (assignment_valid(sids + t * k, j, e, E))
          key[h] = (static_cast<uint32_t>(e) << 8) | static_cast<uint32_t>(a);
        else
          inv[a] = -1;
      }
    }
    // bitonic sort of positions p = lane + 32 h, ascending: runs of length s, partners p ^ d
#pragma unroll
    for (int s = 2; s <= 32; s <<= 1) {
#pragma unroll
      for (int d = s >> 1; d >= 1; d >>= 1) {
        const bool asc0 = (lane & s) == 0;                 // p = lane
        const bool asc1 = s == 32 ? false : asc0;          // p = lane + 32
        key[0] = bitonic_ce_shfl(key[0], lane, d, asc0);
        key[1] = bitonic_ce_shfl(key[1], lane, d, asc1);
      }
    }
    {  // s = 64: the halves at distance 32 sit in one lane, then every run ascends
      const uint32_t lo = min(key[0], key[1]), hi = max(key[0], key[1]);
      key[0] = lo;
      key[1] = hi;
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) {
        key[0] = bitonic_ce_shfl(key[0], lane, d, true);
        key[1] = bitonic_ce_shfl(key[1], lane, d, true);
      }
    }
    s_keys[lane] = key[0];
    s_keys[lane + 32] = key[1];
    // segment starts: a valid key whose expert differs from the key before it
    const uint32_t v0 = __ballot_sync(0xffffffffu, key[0] != kNone);
    const uint32_t v1 = __ballot_sync(0xffffffffu, key[1] != kNone);
    const int n_valid = __popc(v0) + __popc(v1);
    const uint32_t before0 = __shfl_sync(0xffffffffu, key[0], (lane + 31) & 31);  // p - 1 for p = lane >= 1
    const uint32_t last0 = __shfl_sync(0xffffffffu, key[0], 31);                  // p = 31
    const uint32_t before1 = __shfl_sync(0xffffffffu, key[1], (lane + 31) & 31);  // p - 1 for p = lane + 32, lane >= 1
    const uint32_t prev[2] = {before0, lane == 0 ? last0 : before1};
    bool start[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
      start[h] = key[h] != kNone && ((lane == 0 && h == 0) || (prev[h] >> 8) != (key[h] >> 8));
    const uint64_t S = static_cast<uint64_t>(__ballot_sync(0xffffffffu, start[0])) |
                       (static_cast<uint64_t>(__ballot_sync(0xffffffffu, start[1])) << 32);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (key[h] == kNone) continue;
      const int p = lane + 32 * h;
      const int a = static_cast<int>(key[h] & 0xFFu);
      perm[p] = a;
      inv[a] = p;
      if (start[h] && segs) {
        const int idx = __popcll(S & ((1ull << p) - 1ull));
        const uint64_t upto = p == 63 ? ~0ull : ((2ull << p) - 1ull);  // bits 0..p
        const uint64_t above = S & ~upto;
        const int next = above ? __ffsll(static_cast<long long>(above)) - 1 : n_valid;
        if (idx < max_segs)
          segs[idx] = Seg{static_cast<int>(key[h] >> 8), p, next - p, idx, 1, 0, 0, 0};
        else
          set_error(err, MOE_DEVERR_SEGMENT);
      }
    }
    if (lane == 0 && segs) *n_segs = min(__popcll(S), max_segs);
  }
  __syncthreads();
  // offsets[e] = number of keys below expert e (the invalid keys sort above every expert)
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    int lo = 0, hi = 0;
    const uint32_t t_lo = static_cast<uint32_t>(e) << 8, t_hi = static_cast<uint32_t>(e + 1) << 8;
#pragma unroll
    for (int step = kTinyGroupRows / 2; step >= 1; step >>= 1) {
      if (s_keys[lo + step - 1] < t_lo) lo += step;
      if (s_keys[hi + step - 1] < t_hi) hi += step;
    }
    lo += s_keys[lo] < t_lo ? 1 : 0;  // lo <= 63 here
    hi += s_keys[hi] < t_hi ? 1 : 0;
    offsets[e] = lo;
    if (e < E) counts[e] = hi - lo;
  }
}

template <int PL>
__global__ void __launch_bounds__(kRgThreads) route_group_kernel(
    const float* __restrict__ parts, int nsplit, const float* __restrict__ bias, int T, int E, int k,
    int32_t* __restrict__ ids, float* __restrict__ gates, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, Seg* segs, int32_t* n_segs, int max_segs,
    uint32_t* done, uint32_t* err, const XConv xc) {
  extern __shared__ uint32_t sm[];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  convert_x16(xc, err);
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x;
  {
    float* slog = reinterpret_cast<float*>(sm);  // [E]
    float w[kRgPer][kSmallSplitsMax];
#pragma unroll
    for (int q = 0; q < kRgPer; ++q) {
      const int e = threadIdx.x + kRgThreads * q;
#pragma unroll
      for (int sp = 0; sp < kSmallSplitsMax; ++sp)
        w[q][sp] = (e < E && sp < nsplit) ? parts[(static_cast<size_t>(sp) * T + t) * E + e] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kRgPer; ++q) {
      const int e = threadIdx.x + kRgThreads * q;
      if (e < E) {
        float v = w[q][0];
#pragma unroll
        for (int sp = 1; sp < kSmallSplitsMax; ++sp)
          if (sp < nsplit) v += w[q][sp];
        if (bias) v += bias[e];
        slog[e] = v;
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      float v[PL];
#pragma unroll
      for (int i = 0; i < PL; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? slog[e] : 0.f;
      }
      topk_select<PL>(v, t, E, k, ids, gates, err);
    }
  }
  // publish this token's ids, then count finished blocks
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- grouping, by the last block ----
  const int nch = (T + kChunk - 1) / kChunk;
  int32_t* sids = reinterpret_cast<int32_t*>(sm) + 2 * nch * E;
  for (int i = threadIdx.x; i < T * k; i += kRgThreads) sids[i] = __ldcg(ids + i);
  __syncthreads();
  if (T * k <= kTinyGroupRows)
    group_tiny(T, E, k, sids, counts, offsets, perm, inv, segs, n_segs, max_segs, err);
  else
    group_small(T, E, k, sm, counts, offsets, perm, inv, segs, n_segs, max_segs, err);
  if (threadIdx.x == 0) *done = 0u;  // ready for the next launch (stream-ordered)
}

// Router, top-k and grouping of a step of at most 8 tokens in one launch: every block forms its
// K-split partial logits (router_parts_block); the last block to finish adds them (split order,
// then the bias, as the top-k kernel does), selects each token's top k with one warp per token
// and groups the step (group_tiny, or group_small above 64 assignments).
template <int PL>
__global__ void __launch_bounds__(kRgThreads, 1) router_route_tiny_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias, int T, int E,
    int d, float* __restrict__ parts, int k, int32_t* __restrict__ ids, float* __restrict__ gates,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, Seg* segs, int32_t* n_segs, int max_segs, uint32_t* done, uint32_t* err,
    const XConv xc) {
  extern __shared__ __align__(16) uint32_t sm[];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  convert_x16(xc, err);
  router_parts_block<8>(x, wr, T, E, d, parts, reinterpret_cast<uint16_t*>(sm));
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == gridDim.x * gridDim.y - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int nsplit = gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* sids = reinterpret_cast<int32_t*>(sm) + 2 * E;  // one chunk: T <= 8
  if (warp < T) {
    const int t = warp;
    float v[PL], bv[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      v[i] = 0.f;
      bv[i] = (bias && lane + 32 * i < E) ? bias[lane + 32 * i] : 0.f;  // in flight with the partials
    }
    for (int sp = 0; sp < nsplit; sp += 4) {  // partials of other blocks: read through L2
      float w[4][PL];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < PL; ++i) {
          const int e = lane + 32 * i;
          w[u][i] = (e < E && sp + u < nsplit) ? __ldcg(parts + (static_cast<size_t>(sp + u) * T + t) * E + e) : 0.f;
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < PL; ++i)
          if (sp + u < nsplit) v[i] = (sp + u == 0) ? w[u][i] : v[i] + w[u][i];
    }
    if (bias)
#pragma unroll
      for (int i = 0; i < PL; ++i) v[i] += bv[i];
    const int sel = topk_select<PL>(v, t, E, k, ids, gates, err);
    if (lane < k) sids[t * k + lane] = sel;
  }
  __syncthreads();
  if (T * k <= kTinyGroupRows)
    group_tiny(T, E, k, sids, counts, offsets, perm, inv, segs, n_segs, max_segs, err);
  else
    group_small(T, E, k, sm, counts, offsets, perm, inv, segs, n_segs, max_segs, err);
  if (threadIdx.x == 0) *done = 0u;  // ready for the next launch (stream-ordered)
}

bool router_route_tiny_ok(int T, int E, int d, int k) {
  return T > 0 && T <= 8 && d % 128 == 0 && E <= kRgThreads * kRgPer && router_small_splits(d) <= kSmallSplitsMax &&
         route_small_smem(T, E, k) <= 48 * 1024;
}

template <int PL>
static cudaError_t launch_rrt_pl(const uint16_t* x, const float* wr, const float* bias, int T, int E, int d,
                                 float* parts, int k, int32_t* ids, float* gates, int32_t* counts, int32_t* offsets,
                                 int32_t* perm, int32_t* inv, Seg* segs, int32_t* n_segs, int max_segs, uint32_t* done,
                                 uint32_t* err, const XConv& xc, cudaStream_t st) {
  const size_t xs_bytes = 8 * kRouterKS * 2;
  const size_t g_bytes = route_small_smem(T, E, k);
  dim3 grid((E + 7) / 8, router_small_splits(d));
  return launch_pdl(router_route_tiny_kernel<PL>, grid, dim3(kRgThreads), xs_bytes > g_bytes ? xs_bytes : g_bytes, st,
                    x, wr, bias, T, E, d, parts, k, ids, gates, counts, offsets, perm, inv, segs, n_segs, max_segs,
                    done, err, xc);
}

cudaError_t launch_router_route_tiny(const uint16_t* x, const float* w_router, const float* bias, int T, int E, int d,
                                     float* parts, int k, int32_t* ids, float* gates, int32_t* counts,
                                     int32_t* offsets, int32_t* perm, int32_t* inv, Seg* segs, int32_t* n_segs,
                                     int max_segs, uint32_t* done, uint32_t* err, cudaStream_t st,
                                     const XConv& xc) {
  if (!router_route_tiny_ok(T, E, d, k)) return cudaErrorInvalidValue;
  const int pl = (E + 31) / 32;
#define MOE_RRT(PLV)                                                                                            \
  launch_rrt_pl<PLV>(x, w_router, bias, T, E, d, parts, k, ids, gates, counts, offsets, perm, inv, segs, n_segs, \
                     max_segs, done, err, xc, st)
  if (pl <= 1) return MOE_RRT(1);
  if (pl <= 2) return MOE_RRT(2);
  if (pl <= 4) return MOE_RRT(4);
  if (pl <= 8) return MOE_RRT(8);
  if (pl <= 12) return MOE_RRT(12);
  if (pl <= 16) return MOE_RRT(16);
  return MOE_RRT(32);
#undef MOE_RRT
}

bool route_small_ok(int T, int E, int k, int nsplit) {
  return T > 0 && T <= kSmallRouteT && E <= kRgThreads * kRgPer && nsplit <= kSmallSplitsMax &&
         route_small_smem(T, E, k) <= 48 * 1024;
}

template <int PL>
static cudaError_t launch_route_small_pl(const float* parts, int nsplit, const float* bias, int T, int E, int k,
                                         int32_t* ids, float* gates, int32_t* counts, int32_t* offsets, int32_t* perm,
                                         int32_t* inv, Seg* segs, int32_t* n_segs, int max_segs, uint32_t* done,
                                         uint32_t* err, const XConv& xc, cudaStream_t st) {
  return launch_pdl(route_group_kernel<PL>, dim3(T), dim3(kRgThreads), route_small_smem(T, E, k), st, parts, nsplit,
                    bias, T, E, k, ids, gates, counts, offsets, perm, inv, segs, n_segs, max_segs, done, err, xc);
}

cudaError_t launch_route_small(const float* parts, int nsplit, const float* bias, int T, int E, int k, int32_t* ids,
                               float* gates, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, Seg* segs,
                               int32_t* n_segs, int max_segs, uint32_t* done, uint32_t* err, cudaStream_t st,
                               const XConv& xc) {
  if (!route_small_ok(T, E, k, nsplit)) return cudaErrorInvalidValue;
  const int pl = (E + 31) / 32;
#define MOE_RS(PLV)                                                                                             \
  launch_route_small_pl<PLV>(parts, nsplit, bias, T, E, k, ids, gates, counts, offsets, perm, inv, segs, n_segs, \
                             max_segs, done, err, xc, st)
  if (pl <= 1) return MOE_RS(1);
  if (pl <= 2) return MOE_RS(2);
  if (pl <= 4) return MOE_RS(4);
  if (pl <= 8) return MOE_RS(8);
  if (pl <= 12) return MOE_RS(12);
  if (pl <= 16) return MOE_RS(16);
  return MOE_RS(32);
#undef MOE_RS
}

// Segment list from offsets only (the separate experts entry point).  One block of 256 threads.
__global__ void __launch_bounds__(kScanThreads) segments_from_offsets_kernel(const int32_t* __restrict__ offsets,
                                                                           int E, Seg* segs, int32_t* n_segs,
                                                                           int max_segs, uint32_t* err) {
  pdl_trigger();
  pdl_wait();
  int ns[kScanPerThread];
  int mine = 0;
#pragma unroll
  for (int q = 0; q < kScanPerThread; ++q) {
    const int e = threadIdx.x * kScanPerThread + q;
    ns[q] = e < E ? num_segments(offsets[e + 1] - offsets[e]) : 0;
    mine += ns[q];
  }
  int seg_total;
  int base = block_exclusive_scan(mine, &seg_total);
#pragma unroll
  for (int q = 0; q < kScanPerThread; ++q) {
    const int e = threadIdx.x * kScanPerThread + q;
    if (e < E) write_segments(segs, base, max_segs, e, offsets[e], offsets[e + 1] - offsets[e], err);
    base += ns[q];
  }
  if (threadIdx.x == 0) *n_segs = min(seg_total, max_segs);
}

cudaError_t launch_segments_from_offsets(const int32_t* offsets, int E, Seg* segs, int32_t* n_segs,
                                         int max_segs, uint32_t* err, cudaStream_t st) {
  return launch_pdl(segments_from_offsets_kernel, dim3(1), dim3(kScanThreads), 0, st, offsets, E, segs, n_segs, max_segs,
                    err);
}

}  // namespace moe
