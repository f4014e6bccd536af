// Gate-weighted unpermute-combine (out bf16):
//   out[t] = sum_{j<k} g[t,j] * y[inv[t*k+j]]  (+ y_s[t]),
// accumulated in fp32 in slot order j = 0..k-1, then the shared term, then one
// round-to-nearest-even to bf16.  One block per token, 8 output columns per thread per step, so
// every read of y and y_s is a coalesced 16-byte (fp16) or 2 x 16-byte (fp32) load.
// Two element types of y / y_s: fp16 (the layer's own intermediates, written by the down GEMMs)
// and fp32 (the separate moe_combine entry point's contract).
#include "common.cuh"
#include "kernels.h"

namespace moe {

template <typename Y>
struct Row8;

template <>
struct Row8<uint16_t> {  // 8 fp16 values
  uint4 v;
  MOE_DEVICE void load(const uint16_t* p, uint64_t pol) { v = ld_global_v4_hint(p, pol); }
  MOE_DEVICE void zero() { v = make_uint4(0u, 0u, 0u, 0u); }
  MOE_DEVICE void to_f32(float (&o)[8]) const { f16x8_to_f32(v, o); }
};

template <>
struct Row8<float> {  // 8 fp32 values
  uint4 a, b;
  MOE_DEVICE void load(const float* p, uint64_t pol) {
    a = ld_global_v4_hint(p, pol);
    b = ld_global_v4_hint(p + 4, pol);
  }
  MOE_DEVICE void zero() { a = b = make_uint4(0u, 0u, 0u, 0u); }
  MOE_DEVICE void to_f32(float (&o)[8]) const {
    o[0] = __uint_as_float(a.x), o[1] = __uint_as_float(a.y), o[2] = __uint_as_float(a.z), o[3] = __uint_as_float(a.w);
    o[4] = __uint_as_float(b.x), o[5] = __uint_as_float(b.y), o[6] = __uint_as_float(b.z), o[7] = __uint_as_float(b.w);
  }
};

template <typename Y>
__global__ void __launch_bounds__(256) combine_kernel(const Y* __restrict__ y, const float* __restrict__ gates,
                                                      const int32_t* __restrict__ inv, const Y* __restrict__ ys, int T,
                                                      int k, int d, uint16_t* __restrict__ out) {
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
    Row8<Y> vs;  // the shared term: requested with the first slots, added last
    if (ys) vs.load(ys + static_cast<size_t>(t) * d + c, pol);
    for (int j0 = 0; j0 < k; j0 += 8) {  // the loads of 8 slots are in flight together
      Row8<Y> v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int r = j0 + u < k ? s_row[j0 + u] : -1;
        if (r >= 0)
          v[u].load(y + static_cast<size_t>(r) * d + c, pol);
        else
          v[u].zero();
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (j0 + u >= k || s_row[j0 + u] < 0) continue;
        float yf[8];
        v[u].to_f32(yf);
        const float g = s_g[j0 + u];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = fmaf(g, yf[q], acc[q]);
      }
    }
    if (ys) {
      float sf[8];
      vs.to_f32(sf);
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

template <typename Y>
static cudaError_t launch_combine_t(const Y* y, const float* gates, const int32_t* inv, const Y* shared_y, int T, int k,
                                    int d, uint16_t* out, cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  int threads = d / 8;
  if (threads > 256) threads = 256;
  threads = (threads + 31) / 32 * 32;
  return launch_pdl(combine_kernel<Y>, dim3(T), dim3(threads), 0, st, y, gates, inv, shared_y, T, k, d, out);
}

cudaError_t launch_combine(const uint16_t* y, const float* gates, const int32_t* inv, const uint16_t* shared_y, int T,
                           int k, int d, uint16_t* out, cudaStream_t st) {
  return launch_combine_t(y, gates, inv, shared_y, T, k, d, out, st);
}

cudaError_t launch_combine_f32(const float* y, const float* gates, const int32_t* inv, const float* shared_y, int T,
                               int k, int d, uint16_t* out, cudaStream_t st) {
  return launch_combine_t(y, gates, inv, shared_y, T, k, d, out, st);
}

}  // namespace moe
