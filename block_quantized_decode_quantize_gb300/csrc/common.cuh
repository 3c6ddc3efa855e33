// Device helpers and host plumbing shared by the memra CUDA translation units.
// sm_103a only.  Nothing here is shared with the CPU oracle.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "memra.h"

namespace memra {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// Loads.
// ---------------------------------------------------------------------------

// One Q8_0 block of quants (32 bytes) per lane, streamed: a single 256-bit
// non-coherent load that does not allocate in L1 (the weights are read once per
// call).  The pointer must be 32-byte aligned.
struct Quants32 {
  uint32_t w[8];
};

__device__ __forceinline__ Quants32 ld_stream_32B(const int8_t* p) {
  Quants32 r;
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
        "=r"(r.w[6]), "=r"(r.w[7])
      : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p) {
  unsigned short v;
  asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Shared-memory barriers and bulk (TMA) copies, sm_90+ PTX.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for barrier phase `parity`.  Gives up when `*abort` is set by
// another thread or after ~2^31 SM cycles (about a second), setting `*abort`;
// returns whether the phase completed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort) return false;
      if (clock64() - t0 > (1ll << 31)) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Bulk copy global -> this CTA's shared memory, completing `bytes` of the
// barrier's transaction count.  Addresses and size must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Same, with an L2 eviction-priority policy (weights are streamed once).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  wait: block until the preceding kernel on the
// stream has completed and its writes are visible (a no-op when the kernel was
// not launched as a dependent).  launch_dependents: allow the next kernel on the
// stream to begin launching.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// The exact int32 block dot of 32 int8 pairs: 8 dp4a (4 signed byte products
// each, accumulated in int32).  |result| <= 32 * 127 * 127.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int block_dot(const Quants32& w, const uint4& xlo, const uint4& xhi) {
  int s = 0;
  s = __dp4a((int)w.w[0], (int)xlo.x, s);
  s = __dp4a((int)w.w[1], (int)xlo.y, s);
  s = __dp4a((int)w.w[2], (int)xlo.z, s);
  s = __dp4a((int)w.w[3], (int)xlo.w, s);
  s = __dp4a((int)w.w[4], (int)xhi.x, s);
  s = __dp4a((int)w.w[5], (int)xhi.y, s);
  s = __dp4a((int)w.w[6], (int)xhi.z, s);
  s = __dp4a((int)w.w[7], (int)xhi.w, s);
  return s;
}

// ---------------------------------------------------------------------------
// Quantisation of one value with a given scale: clamp(round-half-away(v / d)).
// `/` is the IEEE round-to-nearest division (the library is built without
// fast-math), roundf rounds halves away from zero.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int quant_value(float v, float d) {
  if (d == 0.0f) return 0;
  float r = roundf(v / d);
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return (int)r;
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) |
         ((uint32_t)(d & 0xff) << 24);
}

// ---------------------------------------------------------------------------
// Host side: per-device properties (cached) and launch helpers.
// ---------------------------------------------------------------------------
struct DeviceInfo {
  int sms;
  int max_smem_optin;
};

// Returns false and records the error if the CUDA runtime fails.
bool device_info(DeviceInfo* info);

// Record a CUDA error for memra_last_cuda_error() and return MEMRA_ERR_CUDA.
memra_status cuda_fail(cudaError_t e);

// Check the launch that was just made.
memra_status check_launch();

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// Programmatic dependent launch is on unless the environment sets MEMRA_PDL=0
// (read once per process).
bool pdl_enabled();

// Launch `kernel` on `stream`, as a programmatic dependent of the preceding kernel
// when PDL is enabled.  Returns the launch's cudaError_t.
template <typename... ExpTypes, typename... ActTypes>
cudaError_t launch_kernel(void (*kernel)(ExpTypes...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, ActTypes&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<ActTypes>(args)...);
}

}  // namespace memra
