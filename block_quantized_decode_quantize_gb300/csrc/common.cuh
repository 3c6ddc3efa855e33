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
// call).  The pointer must be 32-byte aligned.  Volatile, so that loads issued
// before a grid-dependency wait stay before it.
struct Quants32 {
  uint32_t w[8];
};

__device__ __forceinline__ Quants32 ld_stream_32B(const int8_t* p) {
  Quants32 r;
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
        "=r"(r.w[6]), "=r"(r.w[7])
      : "l"(p));
  return r;
}

// 16 bytes cached in L2 only (never a stale L1 line): for data written by the
// preceding kernel, read after the grid-dependency wait.
__device__ __forceinline__ uint4 ld_cg_16B(const void* p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Shared-memory barriers and bulk (TMA) copies, sm_90+ PTX.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Loads from this CTA's shared memory at a 32-bit shared-window address.
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(a));
  return r;
}
__device__ __forceinline__ uint16_t lds_u16(uint32_t a) {
  uint16_t r;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float r;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(a));
  return r;
}
__device__ __forceinline__ int lds_s32(uint32_t a) {
  int r;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(r) : "r"(a));
  return r;
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

// The same test, letting the hardware suspend the thread for up to `ns` nanoseconds
// while the phase is incomplete; the thread resumes as soon as the phase completes.
// A waiting warp then retries a few times per wait instead of polling, which leaves
// the issue slots to the warps with work.
__device__ __forceinline__ bool mbar_try_wait_for(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

#ifndef MEMRA_WAIT_SUSPEND_NS
#define MEMRA_WAIT_SUSPEND_NS 8192
#endif

// The default limit of a bounded wait: about a second of SM cycles.
constexpr long long kWaitLimitCycles = 1ll << 31;

// Bounded wait for barrier phase `parity`.  Gives up when `*abort` is set by
// another thread or after `limit` SM cycles, setting `*abort`; returns whether the
// phase completed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_for(bar, parity, MEMRA_WAIT_SUSPEND_NS)) return true;
    if (*abort) return false;
    if (clock64() - t0 > limit) {
      *abort = 1;
      return false;
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

// Quantise 8 values with scale d: the same integers as quant_value, computed by a
// multiply with an approximate reciprocal `inv` of d.  round-half-away only changes
// at k + 1/2, and r = v * inv differs from the correctly rounded quotient fl(v / d)
// by less than 5e-5 (|v/d| <= 254 and at most four roundings of relative size 2^-24
// separate them), so whenever r is farther than 1e-4 from every k + 1/2 both round
// to the same integer.  Values closer than that (exact ties included) take the IEEE
// quotient; the warp votes so that the division runs only when some lane needs it.
// Every lane of the warp must call this.
__device__ __forceinline__ void quant8_fast(const float v[8], float d, float inv, int q[8]) {
  unsigned near = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float r = __fmul_rn(v[i], inv);
    const float a = fabsf(r);
    const float frac = __fsub_rn(a, floorf(a));
    near |= (fabsf(__fsub_rn(frac, 0.5f)) <= 1e-4f ? 1u : 0u) << i;
    q[i] = (int)fminf(fmaxf(roundf(r), -127.0f), 127.0f);
  }
  if (d == 0.0f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = 0;
    near = 0;
  }
  if (__any_sync(kFullMask, near != 0)) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (near & (1u << i)) q[i] = quant_value(v[i], d);
  }
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
  return (uint32_t)(a & 0xff) | ((uint32_t)(b & 0xff) << 8) | ((uint32_t)(c & 0xff) << 16) |
         ((uint32_t)(d & 0xff) << 24);
}

// ---------------------------------------------------------------------------
// q8_1 quantisation of one 32-value block held by four consecutive lanes (8
// values each).  Every lane of the warp must call it (two xor-shuffles).
// Returns the lane's 8 quants packed in 8 bytes and the block scale
// d = max|v| / 127 (fp32, IEEE division).  Used by the standalone quantiser and by
// the products that quantise their activation in the prologue, so both give the
// same bits.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint2 q8_1_group8(const float v[8], float* d_out) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
  a = fmaxf(a, __shfl_xor_sync(kFullMask, a, 1));
  a = fmaxf(a, __shfl_xor_sync(kFullMask, a, 2));
  const float d = a / 127.0f;
  const float inv = a == 0.0f ? 0.0f : 127.0f / a;  // within 2 roundings of 1/d
  int q[8];
  quant8_fast(v, d, inv, q);
  uint2 r;
  r.x = pack4(q[0], q[1], q[2], q[3]);
  r.y = pack4(q[4], q[5], q[6], q[7]);
  *d_out = d;
  return r;
}

__device__ __forceinline__ void load8_f32(const float* p, float v[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// exp by Cody & Waite's range reduction ("Software Manual for the Elementary
// Functions", 1980) and a degree-7 Taylor polynomial: k = rint(x log2 e),
// r = (x - k*C1) - k*C2 with C1 = 0.693359375 (exact product with k) and C2 =
// ln 2 - C1, p = sum_{i<=7} r^i / i! in Horner form, result p * 2^k.  Every
// operation is an explicitly rounded fp32 operation (no contraction), and the
// argument is clamped to [-87, 88] so 2^k is a normal number.
__device__ __forceinline__ float exp_cody_waite(float x) {
  x = fminf(fmaxf(x, -87.0f), 88.0f);
  const float kf = rintf(__fmul_rn(x, 1.44269504088896341f));
  float r = __fsub_rn(x, __fmul_rn(kf, 0.693359375f));
  r = __fsub_rn(r, __fmul_rn(kf, -2.12194440e-4f));
  float p = 1.0f / 5040.0f;
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 720.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 120.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 24.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 6.0f);
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const int k = (int)kf;
  return __fmul_rn(p, __int_as_float((k + 127) << 23));
}

// h = (g / (1 + exp(-g))) * u, each fp32 operation rounded once in that order (SwiGLU
// of the routed-expert FFN).
__device__ __forceinline__ float swiglu1(float g, float u) {
  const float den = __fadd_rn(1.0f, exp_cody_waite(-g));
  return __fmul_rn(__fdiv_rn(g, den), u);
}

// swiglu1 of 8 consecutive values.
__device__ __forceinline__ void swiglu8(const float* g, const float* u, float h[8]) {
  const float4 g0 = *reinterpret_cast<const float4*>(g);
  const float4 g1 = *reinterpret_cast<const float4*>(g + 4);
  const float4 u0 = *reinterpret_cast<const float4*>(u);
  const float4 u1 = *reinterpret_cast<const float4*>(u + 4);
  const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) h[i] = swiglu1(gv[i], uv[i]);
}

// 8 bf16 values (16 bytes) to fp32, exactly.
__device__ __forceinline__ void load8_bf16(const uint16_t* p, float v[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
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

// Let `kernel` take more than 48 KB of dynamic shared memory.  The attribute goes to
// the device's opt-in maximum, never to one launch's size: a CUDA graph captured
// earlier can hold launches of the same kernel with larger sizes, and lowering the
// attribute would make those launches invalid wherever they are checked again (a
// profiler re-issues graph nodes as single launches).
template <typename Kern>
cudaError_t allow_dynamic_smem(Kern kernel, size_t smem, const DeviceInfo& info) {
  if (smem <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              info.max_smem_optin);
}

// The tensor-core product of M = 1..8 activation rows (mma.cu).  Returns
// MEMRA_ERR_UNSUPPORTED, having launched nothing, when the shape or the alignment does
// not suit it (K a multiple of 1024, N >= 16, 16-byte aligned planes and activations).
memra_status run_mma_product(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K, int M,
                             const int8_t* xq, const float* xd, float* y, cudaStream_t stream);

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
