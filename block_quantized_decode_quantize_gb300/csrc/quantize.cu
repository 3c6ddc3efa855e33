// Block quantisers: Q8_0 weight ingest, q8_1 activation quantisation and the
// fused SwiGLU + q8_1 quantisation of the routed-expert FFN.
//
// Thread mapping (all three kernels): a thread owns 8 consecutive values, four
// consecutive lanes own one 32-value block.  The block's max|v| is combined with
// two xor-shuffles, every lane quantises its 8 values and stores them as one 8-byte
// word, and the first lane of the four stores the block scale.  The kernels are
// HBM/L2 bound and tiny next to the weight stream; a grid-stride loop over warps
// keeps every shuffle warp-uniform.
#include "common.cuh"

namespace memra {
namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ void load8(const float* p, float v[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const uint16_t* p, float v[8]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);             // bf16 -> fp32 is exact
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ float group4_amax(const float v[8]) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
  a = fmaxf(a, __shfl_xor_sync(kFullMask, a, 1));
  a = fmaxf(a, __shfl_xor_sync(kFullMask, a, 2));
  return a;
}

__device__ __forceinline__ uint2 quant8(const float v[8], float d) {
  uint2 r;
  r.x = pack4(quant_value(v[0], d), quant_value(v[1], d), quant_value(v[2], d),
              quant_value(v[3], d));
  r.y = pack4(quant_value(v[4], d), quant_value(v[5], d), quant_value(v[6], d),
              quant_value(v[7], d));
  return r;
}

// Activations: d = amax / 127 in fp32.  T = float or uint16_t (bf16 bits).
template <typename T>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_q8_1_kernel(const T* __restrict__ x, int64_t groups, int8_t* __restrict__ q,
                         float* __restrict__ d) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < groups;
       base += stride) {
    const int64_t g = base + lane;
    const bool valid = g < groups;
    float v[8];
    if (valid) {
      load8(x + g * 8, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    const float amax = group4_amax(v);
    const float dv = amax / 127.0f;
    const uint2 packed = quant8(v, dv);
    if (valid) {
      *reinterpret_cast<uint2*>(q + g * 8) = packed;
      if ((lane & 3) == 0) d[g >> 2] = dv;
    }
  }
}

// Weights: d16 = fp16_rne(amax / 127); quants use the stored fp16 value.  This
// kernel does not let its dependents start early: the products stream weights
// before waiting on their predecessor, so they must never overlap the ingest.
__global__ void __launch_bounds__(kQuantThreads)
    quantize_q8_0_kernel(const float* __restrict__ w, int64_t groups, int8_t* __restrict__ q,
                         uint16_t* __restrict__ d) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < groups;
       base += stride) {
    const int64_t g = base + lane;
    const bool valid = g < groups;
    float v[8];
    if (valid) {
      load8(w + g * 8, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    const float amax = group4_amax(v);
    const __half d16 = __float2half_rn(amax / 127.0f);
    const float dv = __half2float(d16);
    const uint2 packed = quant8(v, dv);
    if (valid) {
      *reinterpret_cast<uint2*>(q + g * 8) = packed;
      if ((lane & 3) == 0) d[g >> 2] = __half_as_ushort(d16);
    }
  }
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

// h = (g / (1 + exp(-g))) * u, one rounding per operation, then q8_1 of h.
// gu: [R][2F] (gate columns first), F % 32 == 0, so a thread's 8 values never
// straddle a row.
__global__ void __launch_bounds__(kQuantThreads)
    swiglu_quantize_kernel(const float* __restrict__ gu, int64_t F, int64_t groups,
                           int8_t* __restrict__ q, float* __restrict__ d) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t gpr = F / 8;  // groups per row
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); base < groups;
       base += stride) {
    const int64_t g = base + lane;
    const bool valid = g < groups;
    float h[8];
    if (valid) {
      const int64_t r = g / gpr;
      const int64_t f0 = (g - r * gpr) * 8;
      float gv[8], uv[8];
      load8(gu + r * 2 * F + f0, gv);
      load8(gu + r * 2 * F + F + f0, uv);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float den = __fadd_rn(1.0f, exp_cody_waite(-gv[i]));
        const float sg = __fdiv_rn(gv[i], den);
        h[i] = __fmul_rn(sg, uv[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = 0.0f;
    }
    const float amax = group4_amax(h);
    const float dv = amax / 127.0f;
    const uint2 packed = quant8(h, dv);
    if (valid) {
      *reinterpret_cast<uint2*>(q + g * 8) = packed;
      if ((lane & 3) == 0) d[g >> 2] = dv;
    }
  }
}

int quant_grid(int64_t groups, const DeviceInfo& info) {
  const int64_t warps = (groups + 31) / 32;
  const int64_t blocks = (warps * 32 + kQuantThreads - 1) / kQuantThreads;
  const int64_t cap = (int64_t)info.sms * 8;  // 8 resident 256-thread CTAs per SM
  return (int)(blocks < cap ? blocks : cap);
}

}  // namespace
}  // namespace memra

using namespace memra;

extern "C" memra_status memra_quantize_q8_0(const float* w, int64_t N, int64_t K, int8_t* wq,
                                            uint16_t* wd, cudaStream_t stream) {
  if (N < 0 || K < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return MEMRA_OK;
  if (!w || !wq || !wd) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(wq, 16) || !aligned(wd, 2)) return MEMRA_ERR_ALIGNMENT;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  const int64_t groups = N * K / 8;
  cudaError_t e = launch_kernel(quantize_q8_0_kernel, dim3(quant_grid(groups, info)),
                                dim3(kQuantThreads), 0, stream, w, groups, wq, wd);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

extern "C" memra_status memra_quantize_q8_1(const void* x, int32_t dtype, int64_t M, int64_t K,
                                            int8_t* xq, float* xd, cudaStream_t stream) {
  if (M < 0 || K < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (dtype != MEMRA_BF16 && dtype != MEMRA_F32) return MEMRA_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return MEMRA_OK;
  if (!x || !xq || !xd) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xq, 16) || !aligned(xd, 4)) return MEMRA_ERR_ALIGNMENT;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  const int64_t groups = M * K / 8;
  const dim3 grid(quant_grid(groups, info));
  cudaError_t e;
  if (dtype == MEMRA_BF16) {
    e = launch_kernel(quantize_q8_1_kernel<uint16_t>, grid, dim3(kQuantThreads), 0, stream,
                      static_cast<const uint16_t*>(x), groups, xq, xd);
  } else {
    e = launch_kernel(quantize_q8_1_kernel<float>, grid, dim3(kQuantThreads), 0, stream,
                      static_cast<const float*>(x), groups, xq, xd);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

extern "C" memra_status memra_swiglu_quantize_q8_1(const float* gu, int64_t R, int64_t F,
                                                   int8_t* hq, float* hd, cudaStream_t stream) {
  if (R < 0 || F < 0 || F % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (R == 0 || F == 0) return MEMRA_OK;
  if (!gu || !hq || !hd) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(gu, 16) || !aligned(hq, 16) || !aligned(hd, 4)) return MEMRA_ERR_ALIGNMENT;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  const int64_t groups = R * F / 8;
  cudaError_t e = launch_kernel(swiglu_quantize_kernel, dim3(quant_grid(groups, info)),
                                dim3(kQuantThreads), 0, stream, gu, F, groups, hq, hd);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}
