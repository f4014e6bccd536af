// Set-up time weight repacking (not on the per-step path).
//
// Gate and up projections are stored together with their rows interleaved in groups of 8:
// rows 16q..16q+7 are gate rows 8q..8q+7 and rows 16q+8..16q+15 are the up rows of the same
// features.  A 128-row tile then holds the gate and up rows of 64 features, so one tensor-core
// accumulator holds both and a single lane exchange (lane ^ 8) pairs them for SwiGLU.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void interleave_gate_up_kernel(const uint8_t* __restrict__ gate, const uint8_t* __restrict__ up,
                                          uint8_t* __restrict__ dst, int f, size_t row_bytes) {
  const size_t drow = blockIdx.x;      // destination row over [n][2f]
  const size_t e = drow / (2 * f);
  const int rr = static_cast<int>(drow % (2 * f));
  const int q = rr >> 4, w = rr & 15;
  const int which = w >> 3;
  const int F = 8 * q + (w & 7);
  const uint8_t* src = (which ? up : gate) + (e * f + F) * row_bytes;
  uint8_t* out = dst + drow * row_bytes;
  if ((row_bytes & 15) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    for (size_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x)
      reinterpret_cast<uint4*>(out)[i] = reinterpret_cast<const uint4*>(src)[i];
  } else {
    for (size_t i = threadIdx.x; i < row_bytes; i += blockDim.x) out[i] = src[i];
  }
}

cudaError_t launch_interleave_gate_up(const uint8_t* gate, const uint8_t* up, uint8_t* dst, int n,
                                      int f, size_t row_bytes, cudaStream_t st) {
  const size_t rows = static_cast<size_t>(n) * 2 * f;
  if (rows == 0) return cudaSuccess;
  interleave_gate_up_kernel<<<static_cast<unsigned>(rows), 128, 0, st>>>(gate, up, dst, f, row_bytes);
  return cudaGetLastError();
}

// bf16 -> fp16 for the down-projection weights.  Exact for 2^-17 <= |w| <= 65504 (and 0);
// smaller magnitudes land on the fp16 subnormal grid (absolute error <= 2^-25).
__global__ void bf16_to_f16_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, size_t n,
                                   uint32_t* bad) {
  bool oor = false;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float v = bf16_bits_to_f32(src[i]);
    if (!(fabsf(v) <= kF16Max)) oor = true;
    dst[i] = f32_to_f16_bits_rn(v);
  }
  if (oor) atomicOr(bad, 1u);
}

cudaError_t launch_bf16_to_f16(const uint16_t* src, uint16_t* dst, size_t n, uint32_t* bad, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  bf16_to_f16_kernel<<<1024, 256, 0, st>>>(src, dst, n, bad);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// Tile-contiguous layouts for the tensor-core path.  A block is 128 weight rows x 64 K elements
// (16 KB) stored exactly as the MMA reads it from shared memory: row r at r * 128 bytes, its
// 16-byte chunk c at ((c ^ (r % 8)) * 16) (the 128-byte swizzle).  Blocks of one unit's K loop
// are consecutive, so a unit streams its weights as one contiguous run of HBM.
// ---------------------------------------------------------------------------------------------
// Gate/up of n experts ([n][f][d] each) -> blocks [n][f/64][d/64]; block row r of feature tile t
// is gate row 64t + 8(r/16) + r%8 when r%16 < 8, else the up row of that feature.
__global__ void tile_gate_up_kernel(const uint16_t* __restrict__ gate, const uint16_t* __restrict__ up,
                                    uint16_t* __restrict__ dst, int n, int f, int d, int one_matrix,
                                    size_t n_chunks16) {
  const int nk = d / 64, tiles = f / 64;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_chunks16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    // logical 16-byte chunk i: block b = i / 1024 = (e * tiles + t) * nk + kc, row r, physical chunk pc
    const size_t b = i >> 10;
    const int r = static_cast<int>((i >> 3) & 127), pc = static_cast<int>(i & 7);
    const int kc = static_cast<int>(b % nk);
    const size_t et = b / nk;
    const int t = static_cast<int>(et % tiles);
    const size_t e = et / tiles;
    const int F = 64 * t + 8 * (r >> 4) + (r & 7);
    const uint16_t* src = ((r & 15) < 8 ? gate : up) + (e * f + F) * static_cast<size_t>(d) + kc * 64 + 8 * (pc ^ (r & 7));
    const size_t blk = one_matrix ? tile_chunk_offset(static_cast<int>(e) * tiles + t, kc, n * tiles, nk)
                                  : e * tiles * nk * kTileElems + tile_chunk_offset(t, kc, tiles, nk);
    reinterpret_cast<uint4*>(dst + blk + r * 64)[pc] = *reinterpret_cast<const uint4*>(src);
  }
}

cudaError_t launch_tile_gate_up(const uint16_t* gate, const uint16_t* up, uint16_t* dst, int n, int f, int d,
                                int one_matrix, cudaStream_t st) {
  const size_t chunks = static_cast<size_t>(n) * 2 * f * d / 8;
  if (chunks == 0) return cudaSuccess;
  tile_gate_up_kernel<<<2048, 256, 0, st>>>(gate, up, dst, n, f, d, one_matrix, chunks);
  return cudaGetLastError();
}

// Down projections of n matrices ([n][rows][K] bf16) -> fp16 blocks.  Routed (by_matrix): one
// tile-contiguous matrix per m (rows/128 tiles, K/64 chunks).  Shared: one matrix of rows/128
// tiles whose K chunks run over all n matrices (chunk m * K/64 + kc), so one output tile's K loop
// covers every shared expert.
__global__ void tile_down_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int n, int rows, int K,
                                 int by_matrix, size_t n_chunks16, uint32_t* bad) {
  const int nk = K / 64, dts = rows / 128;
  bool oor = false;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_chunks16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t b = i >> 10;
    const int r = static_cast<int>((i >> 3) & 127), pc = static_cast<int>(i & 7);
    const int kc = static_cast<int>(b % nk);
    const size_t rest = b / nk;
    int m, dt;
    if (by_matrix) {
      dt = static_cast<int>(rest % dts);
      m = static_cast<int>(rest / dts);
    } else {
      m = static_cast<int>(rest % n);
      dt = static_cast<int>(rest / n);
    }
    const uint16_t* s = src + (static_cast<size_t>(m) * rows + dt * 128 + r) * K + kc * 64 + 8 * (pc ^ (r & 7));
    const uint4 v = *reinterpret_cast<const uint4*>(s);
    const size_t blk = by_matrix ? static_cast<size_t>(m) * dts * nk * kTileElems + tile_chunk_offset(dt, kc, dts, nk)
                                 : tile_chunk_offset(dt, m * nk + kc, dts, n * nk);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = bf16_bits_to_f32(static_cast<uint16_t>(w[q] & 0xFFFFu));
      const float hi = bf16_bits_to_f32(static_cast<uint16_t>(w[q] >> 16));
      if (!(fabsf(lo) <= kF16Max) || !(fabsf(hi) <= kF16Max)) oor = true;
      o[q] = static_cast<uint32_t>(f32_to_f16_bits_rn(lo)) | (static_cast<uint32_t>(f32_to_f16_bits_rn(hi)) << 16);
    }
    reinterpret_cast<uint4*>(dst + blk + r * 64)[pc] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (oor) atomicOr(bad, 1u);
}

cudaError_t launch_tile_down(const uint16_t* src, uint16_t* dst, int n, int rows, int K, int by_matrix, uint32_t* bad,
                             cudaStream_t st) {
  const size_t chunks = static_cast<size_t>(n) * rows * K / 8;
  if (chunks == 0) return cudaSuccess;
  tile_down_kernel<<<2048, 256, 0, st>>>(src, dst, n, rows, K, by_matrix, chunks, bad);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// 4-bit weights: one block per (matrix, 128-row tile, 64-K chunk), kFp4BlockBytes = 4352 bytes:
//   [0, 2048)     codes of K elements 0..31 of the chunk, row r at r * 16
//   [2048, 4096)  codes of K elements 32..63, row r at 2048 + r * 16
//   [4096, 4352)  e8m0 scales, row r at 4096 + 2 r (+0: elements 0..31, +1: 32..63)
// so that a thread owning one row reads its 16-byte halves without bank conflicts.  Gate/up rows
// are interleaved by 8 as in the 16-bit layout.  *scale_oor gets 1 if a scale byte lies outside
// [kFp4ScaleMin, kFp4ScaleMax], where the fp16 dequantisation would not be exact.
// ---------------------------------------------------------------------------------------------
__global__ void tile_fp4_kernel(const uint8_t* __restrict__ codes_a, const uint8_t* __restrict__ scales_a,
                                const uint8_t* __restrict__ codes_b, const uint8_t* __restrict__ scales_b,
                                uint8_t* __restrict__ dst, int rows, int K, int gate_up, size_t n_rows_total,
                                uint32_t* scale_oor) {
  const int nk = K / 64;
  const int tiles = gate_up ? rows / 64 : rows / 128;  // gate/up: 64 features per tile
  bool oor = false;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_rows_total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    // work item i: block b = i / 128, row r = i % 128
    const size_t b = i >> 7;
    const int r = static_cast<int>(i & 127);
    const int kc = static_cast<int>(b % nk);
    const size_t mt = b / nk;
    const int t = static_cast<int>(mt % tiles);
    const size_t m = mt / tiles;
    const uint8_t* codes;
    const uint8_t* scales;
    size_t src_row;
    if (gate_up) {
      const int F = 64 * t + 8 * (r >> 4) + (r & 7);
      const bool up = (r & 15) >= 8;
      codes = up ? codes_b : codes_a;
      scales = up ? scales_b : scales_a;
      src_row = m * rows + F;
    } else {
      codes = codes_a;
      scales = scales_a;
      src_row = m * rows + 128 * t + r;
    }
    const uint8_t* c = codes + src_row * (K / 2) + kc * 32;
    const uint8_t* sc = scales + src_row * (K / 32) + kc * 2;
    uint8_t* blk = dst + b * kFp4BlockBytes;
    *reinterpret_cast<uint4*>(blk + r * 16) = *reinterpret_cast<const uint4*>(c);
    *reinterpret_cast<uint4*>(blk + 2048 + r * 16) = *reinterpret_cast<const uint4*>(c + 16);
    blk[4096 + 2 * r] = sc[0];
    blk[4096 + 2 * r + 1] = sc[1];
    if (sc[0] < kFp4ScaleMin || sc[0] > kFp4ScaleMax || sc[1] < kFp4ScaleMin || sc[1] > kFp4ScaleMax) oor = true;
  }
  if (oor) atomicOr(scale_oor, 1u);
}

cudaError_t launch_tile_fp4(const uint8_t* codes_a, const uint8_t* scales_a, const uint8_t* codes_b,
                            const uint8_t* scales_b, uint8_t* dst, int n, int rows, int K, int gate_up,
                            uint32_t* scale_oor, cudaStream_t st) {
  // gate/up: n experts x (2 * rows) interleaved rows; down: n matrices x rows rows
  const size_t total_rows = static_cast<size_t>(n) * (gate_up ? 2 * rows : rows) * (K / 64);
  if (total_rows == 0) return cudaSuccess;
  tile_fp4_kernel<<<2048, 256, 0, st>>>(codes_a, scales_a, codes_b, scales_b, dst, rows, K, gate_up, total_rows,
                                        scale_oor);
  return cudaGetLastError();
}

}  // namespace moe
