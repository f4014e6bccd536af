// Expert FFN on CUDA cores: one block per grouped row, one warp per output feature.
//
// This is the plain reference path (MOE_PATH_SIMT), kept for debugging and for shapes the
// tensor-core path does not tile.  It computes what the tensor-core path computes: fp32
// accumulation of bf16 (or decoded 4-bit) products, SwiGLU(gate, up) rounded to fp16 into h,
// then the down projection (fp16 weights held by the plan, or decoded 4-bit) rounded to fp16
// into y.  It re-reads each expert's weights for every row, so it is slow by design.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__constant__ float c_e2m1[16] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f,
                                 -0.f, -0.5f, -1.f, -1.5f, -2.f, -3.f, -4.f, -6.f};

// Row index of (feature F, gate = 0 / up = 1) in the gate/up interleaved layout.
MOE_DEVICE int gu_row(int F, int which) { return 16 * (F >> 3) + 8 * which + (F & 7); }

// Dot product of a bf16 activation row (length K, in shared memory as fp32) with one weight row,
// reduced across the warp.  bf16 weights.
MOE_DEVICE float warp_dot_bf16(const float* act, const uint16_t* wrow, int K, int lane) {
  float acc = 0.f;
  for (int i = lane * 8; i < K; i += 256) {
    const uint4 wv = *reinterpret_cast<const uint4*>(wrow + i);
    float wf[8];
    bf16x8_to_f32(wv, wf);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc = fmaf(act[i + q], wf[q], acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// Same with an fp16 weight row.
MOE_DEVICE float warp_dot_f16(const float* act, const uint16_t* wrow, int K, int lane) {
  float acc = 0.f;
  for (int i = lane * 8; i < K; i += 256) {
    const uint4 wv = *reinterpret_cast<const uint4*>(wrow + i);
    float wf[8];
    f16x8_to_f32(wv, wf);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc = fmaf(act[i + q], wf[q], acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// Dot product with one row of a tile-contiguous matrix: `blocks` points at the row's first
// 128 x 64 block, consecutive K chunks are `stride` elements apart (tile_chunk_stride), r is the
// row inside the block.
template <bool kF16>
MOE_DEVICE float warp_dot_tiled(const float* act, const uint16_t* blocks, size_t stride, int r, int K, int lane) {
  float acc = 0.f;
  for (int k = lane * 8; k < K; k += 256) {
    const uint4 wv = *reinterpret_cast<const uint4*>(blocks + static_cast<size_t>(k >> 6) * stride +
                                                     tile_elem_offset(r, k & 63));
    float wf[8];
    if (kF16)
      f16x8_to_f32(wv, wf);
    else
      bf16x8_to_f32(wv, wf);
#pragma unroll
    for (int q = 0; q < 8; ++q) acc = fmaf(act[k + q], wf[q], acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// Row of (feature F, gate 0 / up 1) inside its 128-row gate/up tile.
MOE_DEVICE int gu_tile_row(int F, int which) { return 16 * ((F & 63) >> 3) + 8 * which + (F & 7); }

MOE_DEVICE uint16_t to_f16_sat(float v, bool& sat) {
  if (!(fabsf(v) <= kF16Max)) {
    sat = true;
    v = fminf(fmaxf(v, -kF16Max), kF16Max);
  }
  return f32_to_f16_bits_rn(v);
}

// Same with a 4-bit row: codes (K/2 bytes) and e8m0 scales (K/32 bytes).  Each lane takes one
// 32-element block (16 code bytes) at a time.
MOE_DEVICE float warp_dot_fp4(const float* act, const uint8_t* crow, const uint8_t* srow, int K, int lane) {
  float acc = 0.f;
  for (int b = lane; b < K / 32; b += 32) {
    const uint4 cv = *reinterpret_cast<const uint4*>(crow + b * 16);
    const float scale = ldexpf(1.0f, static_cast<int>(srow[b]) - 127);
    const uint32_t w[4] = {cv.x, cv.y, cv.z, cv.w};
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int el = b * 32 + q * 8 + n;
        part = fmaf(act[el], c_e2m1[(w[q] >> (4 * n)) & 0xF], part);
      }
    }
    acc = fmaf(part, scale, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// Same with a row of the 4-bit tile-contiguous layout: `blocks` is the row's first block (K
// chunk 0), r its row inside the blocks; 32-element scale block b lives in chunk b / 2, half b % 2.
MOE_DEVICE float warp_dot_fp4_tiled(const float* act, const uint8_t* blocks, int r, int K, int lane) {
  float acc = 0.f;
  for (int b = lane; b < K / 32; b += 32) {
    const uint8_t* blk = blocks + static_cast<size_t>(b >> 1) * kFp4BlockBytes;
    const uint4 cv = *reinterpret_cast<const uint4*>(blk + (b & 1) * 2048 + r * 16);
    const float scale = ldexpf(1.0f, static_cast<int>(blk[4096 + 2 * r + (b & 1)]) - 127);
    const uint32_t w[4] = {cv.x, cv.y, cv.z, cv.w};
    float part = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int n = 0; n < 8; ++n) part = fmaf(act[b * 32 + q * 8 + n], c_e2m1[(w[q] >> (4 * n)) & 0xF], part);
    }
    acc = fmaf(part, scale, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// Expert of grouped row r: the e with offsets[e] <= r < offsets[e+1] (binary search).
MOE_DEVICE int expert_of_row(const int32_t* offsets, int E, int r) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offsets[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Blocks [0, R) are routed rows, blocks [R, R + T) are shared rows (if any).
__global__ void __launch_bounds__(256) simt_gateup_kernel(FfnWeights w, const uint16_t* __restrict__ x,
                                                          int T, const int32_t* __restrict__ offsets,
                                                          const int32_t* __restrict__ perm,
                                                          uint16_t* __restrict__ h, uint16_t* __restrict__ h_s) {
  extern __shared__ float act[];  // [d]
  pdl_trigger();
  pdl_wait();
  const int R = T * w.k;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tok, e = -1;
  if (b < R) {
    if (b >= offsets[w.E]) return;
    e = expert_of_row(offsets, w.E, b);
    tok = perm[b] / w.k;
  } else {
    tok = b - R;
  }
  for (int i = threadIdx.x; i < w.d; i += blockDim.x) act[i] = bf16_bits_to_f32(x[static_cast<size_t>(tok) * w.d + i]);
  __syncthreads();
  if (e >= 0) {
    for (int F = warp; F < w.f; F += 8) {
      float g, u;
      if (w.fp4 && w.fp4_tiled) {
        const uint8_t* blocks = static_cast<const uint8_t*>(w.w_gu) +
                                (static_cast<size_t>(e) * (w.f / 64) + F / 64) * (w.d / 64) * kFp4BlockBytes;
        g = warp_dot_fp4_tiled(act, blocks, gu_tile_row(F, 0), w.d, lane);
        u = warp_dot_fp4_tiled(act, blocks, gu_tile_row(F, 1), w.d, lane);
      } else if (w.fp4) {
        const uint8_t* c = static_cast<const uint8_t*>(w.w_gu) + static_cast<size_t>(e) * 2 * w.f * (w.d / 2);
        const uint8_t* s = w.s_gu + static_cast<size_t>(e) * 2 * w.f * (w.d / 32);
        g = warp_dot_fp4(act, c + static_cast<size_t>(gu_row(F, 0)) * (w.d / 2), s + static_cast<size_t>(gu_row(F, 0)) * (w.d / 32), w.d, lane);
        u = warp_dot_fp4(act, c + static_cast<size_t>(gu_row(F, 1)) * (w.d / 2), s + static_cast<size_t>(gu_row(F, 1)) * (w.d / 32), w.d, lane);
      } else if (w.tiled) {
        const int tiles = w.f / 64, t = F / 64;
        const uint16_t* blocks = static_cast<const uint16_t*>(w.w_gu) + static_cast<size_t>(e) * tiles * (w.d / 64) * kTileElems +
                                 tile_chunk_offset(t, 0, tiles, w.d / 64);
        const size_t stride = tile_chunk_stride(t, tiles);
        g = warp_dot_tiled<false>(act, blocks, stride, gu_tile_row(F, 0), w.d, lane);
        u = warp_dot_tiled<false>(act, blocks, stride, gu_tile_row(F, 1), w.d, lane);
      } else {
        const uint16_t* base = static_cast<const uint16_t*>(w.w_gu) + static_cast<size_t>(e) * 2 * w.f * w.d;
        g = warp_dot_bf16(act, base + static_cast<size_t>(gu_row(F, 0)) * w.d, w.d, lane);
        u = warp_dot_bf16(act, base + static_cast<size_t>(gu_row(F, 1)) * w.d, w.d, lane);
      }
      bool sat = false;
      const uint16_t hv = to_f16_sat(swiglu(g, u), sat);
      if (lane == 0) {
        h[static_cast<size_t>(b) * w.f + F] = hv;
        if (sat) set_error(w.err, MOE_DEVERR_RANGE);
      }
    }
  } else {
    const int fs_tot = w.n_shared * w.f_s;
    for (int F = warp; F < fs_tot; F += 8) {
      const int s = F / w.f_s, Fl = F % w.f_s;
      float g, u;
      if (w.tiled_s) {
        const int tiles = w.n_shared * (w.f_s / 64), t = s * (w.f_s / 64) + Fl / 64;  // one matrix
        const uint16_t* blocks = w.w_gu_s + tile_chunk_offset(t, 0, tiles, w.d / 64);
        const size_t stride = tile_chunk_stride(t, tiles);
        g = warp_dot_tiled<false>(act, blocks, stride, gu_tile_row(Fl, 0), w.d, lane);
        u = warp_dot_tiled<false>(act, blocks, stride, gu_tile_row(Fl, 1), w.d, lane);
      } else {
        const uint16_t* base = w.w_gu_s + static_cast<size_t>(s) * 2 * w.f_s * w.d;
        g = warp_dot_bf16(act, base + static_cast<size_t>(gu_row(Fl, 0)) * w.d, w.d, lane);
        u = warp_dot_bf16(act, base + static_cast<size_t>(gu_row(Fl, 1)) * w.d, w.d, lane);
      }
      bool sat = false;
      const uint16_t hv = to_f16_sat(swiglu(g, u), sat);
      if (lane == 0) {
        h_s[static_cast<size_t>(tok) * fs_tot + F] = hv;
        if (sat) set_error(w.err, MOE_DEVERR_RANGE);
      }
    }
  }
}

__global__ void __launch_bounds__(256) simt_down_kernel(FfnWeights w, int T, const int32_t* __restrict__ offsets,
                                                        const uint16_t* __restrict__ h,
                                                        const uint16_t* __restrict__ h_s,
                                                        uint16_t* __restrict__ y, uint16_t* __restrict__ y_s) {
  extern __shared__ float act[];  // [max(f, n_s * f_s)]
  pdl_trigger();
  pdl_wait();
  const int R = T * w.k;
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (b < R) {
    if (b >= offsets[w.E]) return;
    const int e = expert_of_row(offsets, w.E, b);
    for (int i = threadIdx.x; i < w.f; i += blockDim.x) act[i] = f16_bits_to_f32(h[static_cast<size_t>(b) * w.f + i]);
    __syncthreads();
    for (int n = warp; n < w.d; n += 8) {
      float v;
      if (w.fp4 && w.fp4_tiled) {
        const uint8_t* blocks = static_cast<const uint8_t*>(w.w_down) +
                                (static_cast<size_t>(e) * (w.d / 128) + n / 128) * (w.f / 64) * kFp4BlockBytes;
        v = warp_dot_fp4_tiled(act, blocks, n & 127, w.f, lane);
      } else if (w.fp4) {
        const uint8_t* c = static_cast<const uint8_t*>(w.w_down) + (static_cast<size_t>(e) * w.d + n) * (w.f / 2);
        const uint8_t* s = w.s_down + (static_cast<size_t>(e) * w.d + n) * (w.f / 32);
        v = warp_dot_fp4(act, c, s, w.f, lane);
      } else if (w.tiled) {
        const int tiles = w.d / 128, t = n / 128;
        const uint16_t* blocks = static_cast<const uint16_t*>(w.w_down) + static_cast<size_t>(e) * tiles * (w.f / 64) * kTileElems +
                                 tile_chunk_offset(t, 0, tiles, w.f / 64);
        v = warp_dot_tiled<true>(act, blocks, tile_chunk_stride(t, tiles), n & 127, w.f, lane);
      } else {
        v = warp_dot_f16(act, static_cast<const uint16_t*>(w.w_down) + (static_cast<size_t>(e) * w.d + n) * w.f, w.f, lane);
      }
      bool sat = false;
      const uint16_t yv = to_f16_sat(v, sat);
      if (lane == 0) {
        y[static_cast<size_t>(b) * w.d + n] = yv;
        if (sat) set_error(w.err, MOE_DEVERR_RANGE);
      }
    }
  } else {
    const int tok = b - R;
    const int fs_tot = w.n_shared * w.f_s;
    for (int i = threadIdx.x; i < fs_tot; i += blockDim.x) act[i] = f16_bits_to_f32(h_s[static_cast<size_t>(tok) * fs_tot + i]);
    __syncthreads();
    for (int n = warp; n < w.d; n += 8) {
      float v = 0.f;
      for (int s = 0; s < w.n_shared; ++s)
        v += w.tiled_s ? warp_dot_tiled<true>(act + s * w.f_s,
                                              w.w_down_s + tile_chunk_offset(n / 128, s * (w.f_s / 64), w.d / 128,
                                                                             w.n_shared * (w.f_s / 64)),
                                              tile_chunk_stride(n / 128, w.d / 128), n & 127, w.f_s, lane)
                       : warp_dot_f16(act + s * w.f_s, w.w_down_s + (static_cast<size_t>(s) * w.d + n) * w.f_s, w.f_s, lane);
      bool sat = false;
      const uint16_t yv = to_f16_sat(v, sat);
      if (lane == 0) {
        y_s[static_cast<size_t>(tok) * w.d + n] = yv;
        if (sat) set_error(w.err, MOE_DEVERR_RANGE);
      }
    }
  }
}

cudaError_t launch_ffn_simt(const FfnWeights& w, const uint16_t* x, int T, const int32_t* offsets,
                            const int32_t* perm, uint16_t* h, uint16_t* h_s, uint16_t* y,
                            uint16_t* y_s, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  const int blocks = T * w.k + (w.n_shared > 0 ? T : 0);
  cudaError_t e = launch_pdl(simt_gateup_kernel, dim3(blocks), dim3(256), w.d * sizeof(float), st, w, x, T, offsets,
                             perm, h, h_s);
  if (e != cudaSuccess) return e;
  const int kmax = w.f > w.n_shared * w.f_s ? w.f : w.n_shared * w.f_s;
  return launch_pdl(simt_down_kernel, dim3(blocks), dim3(256), kmax * sizeof(float), st, w, T, offsets,
                    static_cast<const uint16_t*>(h), static_cast<const uint16_t*>(h_s), y, y_s);
}

}  // namespace moe
