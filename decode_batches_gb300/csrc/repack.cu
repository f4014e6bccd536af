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

}  // namespace moe
