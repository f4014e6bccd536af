// Gate-weighted unpermute-combine (y, y_s fp16; out bf16):
//   out[t] = sum_{j<k} g[t,j] * y[inv[t*k+j]]  (+ y_s[t]),
// accumulated in fp32 in slot order j = 0..k-1, then the shared term, then one
// round-to-nearest-even to bf16.  One block per token, 8 bf16 columns (16 bytes) per thread
// per step, so every read of y and y_s is a coalesced 16-byte load.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y, const float* __restrict__ gates,
                                                      const int32_t* __restrict__ inv,
                                                      const uint16_t* __restrict__ ys, int T, int k, int d,
                                                      uint16_t* __restrict__ out) {
  __shared__ int s_row[32];
  __shared__ float s_g[32];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    s_row[threadIdx.x] = inv[static_cast<size_t>(t) * k + threadIdx.x];
    s_g[threadIdx.x] = gates[static_cast<size_t>(t) * k + threadIdx.x];
  }
  __syncthreads();
  const uint64_t pol = l2_policy_evict_first();  // y and y_s are read once, here
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < k; j0 += 8) {  // the loads of 8 slots are in flight together
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int r = j0 + u < k ? s_row[j0 + u] : -1;
        v[u] = r >= 0 ? ld_global_v4_hint(y + static_cast<size_t>(r) * d + c, pol) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u >= k || s_row[j0 + u] < 0) continue;
        float yf[8];
        f16x8_to_f32(v[u], yf);
        const float g = s_g[j0 + u];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(g, yf[q], acc[q]);
      }
    }
    if (ys) {
      const uint4 v = ld_global_v4_hint(ys + static_cast<size_t>(t) * d + c, pol);
      float sf[8];
      f16x8_to_f32(v, sf);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += sf[q];
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(out + static_cast<size_t>(t) * d + c) = o;
  }
}

cudaError_t launch_combine(const uint16_t* y, const float* gates, const int32_t* inv,
                           const uint16_t* shared_y, int T, int k, int d, uint16_t* out,
                           cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  int threads = d / 8;
  if (threads > 256) threads = 256;
  threads = (threads + 31) / 32 * 32;
  return launch_pdl(combine_kernel, dim3(T), dim3(threads), 0, st, y, gates, inv, shared_y, T, k, d, out);
}

}  // namespace moe
