// Shared device helpers for the MoE layer kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers, TMA (cp.async.bulk.tensor), cp.async, and the
// tcgen05 tensor-core / TMEM instructions, plus bf16 helpers.  Every wait on an mbarrier is
// bounded by wall time (the %globaltimer register): a wait that expires sets a bit in the
// caller's device error word and returns false, so a kernel can never spin forever.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

#include "../../include/moe.h"
#include "kernels.h"

#define MOE_DEVICE __device__ __forceinline__

// Bounded-wait limit for any in-kernel spin (nanoseconds).  Legitimate waits here are
// microseconds; one second means something is wrong.
#ifndef MOE_WAIT_LIMIT_NS
#define MOE_WAIT_LIMIT_NS 1000000000ull
#endif

namespace moe {

MOE_DEVICE uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEVICE uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

MOE_DEVICE void set_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// ------------------------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of a layer step is launched with programmatic
// stream serialization: it may start while its predecessor in the stream is still running,
// runs its shared-memory / TMEM prologue, then waits in pdl_wait() -- before its first global
// memory access -- until the predecessor has completed and its writes are visible.  pdl_trigger()
// at kernel entry lets the successor launch early.  Without the launch attribute both are no-ops.
// ------------------------------------------------------------------------------------------
MOE_DEVICE void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MOE_DEVICE void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Host side: the unique id of the CUDA context current on this thread (cuCtxGetId; ids are never
// reused within a process).  With no context current yet, the runtime's primary context of the
// current device is made current first.  Driver entry points come through the runtime, so the
// library does not link libcuda.
inline cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  if (!get_current || !get_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1);
    if (e != cudaSuccess || q1 != cudaDriverEntryPointSuccess) return cudaErrorNotSupported;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
    if (e != cudaSuccess || q2 != cudaDriverEntryPointSuccess) return cudaErrorNotSupported;
    get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
    get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (!ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);  // initialises and binds the primary context
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  }
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Host side: raise the kernel's dynamic shared-memory limit to `bytes`, once per (context,
// kernel).  The attribute belongs to the kernel's module in one context, so a plan on a second
// device, or a context re-created after cudaDeviceReset, sets it again.
inline cudaError_t ensure_max_dynamic_smem(const void* kern, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<unsigned long long, const void*>> done;
  unsigned long long ctx = 0;
  cudaError_t e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({ctx, kern})) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({ctx, kern});
  return e;
}

// Host side: launch `kern` with the programmatic-stream-serialization attribute.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
MOE_DEVICE void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

MOE_DEVICE void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEVICE void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

MOE_DEVICE void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

MOE_DEVICE bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and sets
// MOE_DEVERR_TIMEOUT) if it does not complete within MOE_WAIT_LIMIT_NS, or if another thread
// of the CTA already flagged an abort.
MOE_DEVICE bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (((++spins) & 63u) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (global_timer_ns() - t0 > MOE_WAIT_LIMIT_NS) {
        set_error(err, MOE_DEVERR_TIMEOUT);
        if (abort_flag) *abort_flag = 1;
        return false;
      }
    }
  }
}

// Teardown after an aborted pipeline (a bounded wait expired somewhere in the CTA).  A role that
// gave up may leave bulk / TMA copies it issued still in flight into this CTA's shared memory;
// their completion cannot be observed once the barrier phases they feed will never complete (the
// other arrivals are missing).  Every such copy is a bounded read of device memory that lands
// within microseconds, so the CTA waits a fixed 50 us of %globaltimer before it frees TMEM and
// exits: no copy outlives the CTA's shared memory.  Called by every thread of the CTA after the
// final barrier; a no-op unless the abort flag is set.
MOE_DEVICE void abort_quiesce(volatile int* abort_flag) {
  if (!abort_flag || !*abort_flag) return;
  const uint64_t t0 = global_timer_ns();
  while (global_timer_ns() - t0 < 50000ull) {
  }
}

// Non-blocking probe of the phase with the given parity (mbarrier.test_wait).  Issue it early
// and consume the result late: the probe's latency then overlaps other work.
MOE_DEVICE bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same wait for a whole converged warp: every lane waits, the result is warp-uniform.
MOE_DEVICE bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* err) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, err));
}

// One lane of a converged warp (the same lane every time the full warp calls it).  Role loops
// that issue tcgen05.mma / TMA run converged and issue under elect_one(): the operands then stay
// warp-uniform, and a single MMA issues in a few tens of cycles instead of a few hundred.
MOE_DEVICE bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------------------------------------
// TMA (tensor maps live in kernel parameter space: __grid_constant__ const CUtensorMap)
// ------------------------------------------------------------------------------------------
MOE_DEVICE uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MOE_DEVICE uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MOE_DEVICE void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load: coordinates (c0 = innermost, c1 = row).  c0 * element size must be a
// multiple of 16 bytes (callers pass multiples of 64 bf16 elements / 32 bytes of codes).
MOE_DEVICE void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Raise the phase's expected transaction bytes without arriving (the arrival comes later).
MOE_DEVICE void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// 16-byte global load / store with an L2 eviction policy (intermediates that should stay in,
// or leave, L2 between the kernel that writes them and the one that reads them).
MOE_DEVICE uint4 ld_global_v4_hint(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
MOE_DEVICE void st_global_v4_hint(void* p, const uint4& v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(policy)
               : "memory");
}

// Bulk copy of `bytes` contiguous bytes (multiple of 16, both addresses 16-byte aligned) into
// shared memory, completing `bytes` transactions on the mbarrier.
MOE_DEVICE void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------------------------------
// cp.async (16-byte, L2 only) for gathered rows
// ------------------------------------------------------------------------------------------
MOE_DEVICE void cp_async_16(uint32_t dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
// Same with an L2 cache-eviction policy (e.g. evict_last for activations re-read by many CTAs).
MOE_DEVICE void cp_async_16_hint(uint32_t dst_smem, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst_smem), "l"(src), "l"(policy)
               : "memory");
}
MOE_DEVICE void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
MOE_DEVICE void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Make this thread's completed generic-proxy shared-memory writes visible to the async
// proxy (the tensor core reads operands through it).
MOE_DEVICE void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads
// ------------------------------------------------------------------------------------------
// Warp-wide: allocates ncols (power of two >= 32) TMEM columns, writes the address to *slot.
MOE_DEVICE void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
MOE_DEVICE void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MOE_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
MOE_DEVICE void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MOE_DEVICE void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 inputs, fp32 accumulate).
MOE_DEVICE void mma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier when all previously issued tcgen05.mma of this thread finish.
MOE_DEVICE void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns: thread i of the warp gets lane (base + i).
MOE_DEVICE void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
MOE_DEVICE void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile stored with the 128-byte
// swizzle: rows of 128 bytes (64 bf16), groups of 8 rows 1024 bytes apart (stride byte
// offset), tile base 1024-byte aligned.  Fields: start address >> 4 in bits [0,14), leading
// byte offset >> 4 in [16,30) (unused for swizzled K-major; set to 1), stride byte offset
// >> 4 in [32,46), descriptor version 1 in [46,48), layout 2 (128-byte swizzle) in [61,64).
MOE_DEVICE uint64_t smem_desc_sw128(uint32_t smem_addr) {
  return (static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu)) | (1ull << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B type in bits 7-9 and
// 10-12 (0 = fp16, 1 = bf16; both operands must have the same type), both K-major (bits 15,
// 16 = 0), N >> 3 in bits [17,23), M >> 4 in bits [24,29).
MOE_DEVICE uint32_t idesc_bf16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
MOE_DEVICE uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ------------------------------------------------------------------------------------------
// bf16 helpers
// ------------------------------------------------------------------------------------------
MOE_DEVICE float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

MOE_DEVICE uint16_t f32_to_bf16_bits_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

MOE_DEVICE void bf16x8_to_f32(const uint4& v, float (&o)[8]) {
  o[0] = __uint_as_float(v.x << 16);
  o[1] = __uint_as_float(v.x & 0xFFFF0000u);
  o[2] = __uint_as_float(v.y << 16);
  o[3] = __uint_as_float(v.y & 0xFFFF0000u);
  o[4] = __uint_as_float(v.z << 16);
  o[5] = __uint_as_float(v.z & 0xFFFF0000u);
  o[6] = __uint_as_float(v.w << 16);
  o[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// fp16 storage of the layer's intermediates (hidden vector h, expert outputs y).
constexpr float kF16Max = 65504.0f;
MOE_DEVICE uint16_t f32_to_f16_bits_rn(float f) { return __half_as_ushort(__float2half_rn(f)); }

// Grid-stride part of an XConv: values outside the fp16 range clamp and flag MOE_DEVERR_RANGE.
MOE_DEVICE void convert_x16(const XConv& c, uint32_t* err) {
  if (!c.x16) return;
  bool sat = false;
  const size_t stride = static_cast<size_t>(gridDim.x) * gridDim.y * gridDim.z * blockDim.x;
  const size_t b = (static_cast<size_t>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
  for (size_t i = b * blockDim.x + threadIdx.x; i < c.n8; i += stride) {
    const uint4 v = reinterpret_cast<const uint4*>(c.x)[i];
    float f[8];
    bf16x8_to_f32(v, f);
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float lo = f[2 * q], hi = f[2 * q + 1];
      if (!(fabsf(lo) <= kF16Max) || !(fabsf(hi) <= kF16Max)) {
        sat = true;
        lo = fminf(fmaxf(lo, -kF16Max), kF16Max);
        hi = fminf(fmaxf(hi, -kF16Max), kF16Max);
      }
      o[q] = static_cast<uint32_t>(f32_to_f16_bits_rn(lo)) | (static_cast<uint32_t>(f32_to_f16_bits_rn(hi)) << 16);
    }
    reinterpret_cast<uint4*>(c.x16)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (sat) set_error(err, MOE_DEVERR_RANGE);
}
MOE_DEVICE float f16_bits_to_f32(uint16_t b) { return __half2float(__ushort_as_half(b)); }

MOE_DEVICE void f16x8_to_f32(const uint4& v, float (&o)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}

MOE_DEVICE uint32_t pack_bf16x2(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16_bits_rn(lo)) |
         (static_cast<uint32_t>(f32_to_bf16_bits_rn(hi)) << 16);
}

// silu(g) * u in fp32 (the SwiGLU of the gate and up projections).  Fast exp and division:
// the result is rounded to fp16 (11 bits) right after, far coarser than their ~2-ulp error.
MOE_DEVICE float swiglu(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

}  // namespace moe
