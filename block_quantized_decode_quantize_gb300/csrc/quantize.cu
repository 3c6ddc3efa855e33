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

__device__ __forceinline__ void load8(const float* p, float v[8]) { load8_f32(p, v); }
__device__ __forceinline__ void load8(const uint16_t* p, float v[8]) { load8_bf16(p, v); }

__device__ __forceinline__ float group4_amax(const float v[8]) {
  float a = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
  a = fmaxf(a, __shfl_xor_sync(kFullMask, a, 1));
  a = fmaxf(a, __shfl_xor_sync(kFullMask, a, 2));
  return a;
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
    float dv;
    const uint2 packed = q8_1_group8(v, &dv);
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
    const float inv = dv == 0.0f ? 0.0f : 1.0f / dv;
    int qv[8];
    quant8_fast(v, dv, inv, qv);
    uint2 packed;
    packed.x = pack4(qv[0], qv[1], qv[2], qv[3]);
    packed.y = pack4(qv[4], qv[5], qv[6], qv[7]);
    if (valid) {
      *reinterpret_cast<uint2*>(q + g * 8) = packed;
      if ((lane & 3) == 0) d[g >> 2] = __half_as_ushort(d16);
    }
  }
}

// Weights to Q4_0: per 32-block m = the element of largest |w| (the first one on a
// tie), d16 = fp16_rne(m / -8) (+0 for an all-zero block), code = clamp(round-half-
// away(w / float(d16)) + 8, 0, 15).  Packed split plane: byte j < 16 of a block holds
// element j's code in its low nibble and element j+16's in its high nibble.  Four
// lanes own a block (8 values each); like the Q8_0 ingest this kernel does not let
// its dependents start early.
__global__ void __launch_bounds__(kQuantThreads)
    quantize_q4_0_kernel(const float* __restrict__ w, int64_t groups, uint8_t* __restrict__ q4,
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
    // The lane's first largest-magnitude value, then the block's: a larger
    // magnitude wins, an equal one from the lower lane (earlier elements) wins.
    float am = 0.0f, m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (fabsf(v[i]) > am) {
        am = fabsf(v[i]);
        m = v[i];
      }
    }
#pragma unroll
    for (int mask = 1; mask <= 2; mask <<= 1) {
      const float om = __shfl_xor_sync(kFullMask, m, mask);
      const float oam = fabsf(om);
      const bool other_first = (lane & mask) != 0;
      if (oam > am || (oam == am && other_first)) {
        am = oam;
        m = om;
      }
    }
    const uint16_t d16 = am == 0.0f ? (uint16_t)0 : __half_as_ushort(__float2half_rn(m / -8.0f));
    const float dv = __half2float(__ushort_as_half(d16));
    const float inv = dv == 0.0f ? 0.0f : 1.0f / dv;
    int qv[8];
    quant8_fast(v, dv, inv, qv);  // clamp(round-half-away(v / dv), +-127), exactly
    int c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = min(max(qv[i] + 8, 0), 15);
    uint2 own;
    own.x = pack4(c[0], c[1], c[2], c[3]);
    own.y = pack4(c[4], c[5], c[6], c[7]);
    // Lanes 0 and 1 of the block (elements 0..15) take the codes of lanes 2 and 3
    // (elements 16..31) as their high nibbles.
    uint2 high;
    high.x = __shfl_xor_sync(kFullMask, own.x, 2);
    high.y = __shfl_xor_sync(kFullMask, own.y, 2);
    if (valid && (lane & 2) == 0) {
      uint2 out;
      out.x = own.x | (high.x << 4);
      out.y = own.y | (high.y << 4);
      *reinterpret_cast<uint2*>(q4 + (g >> 2) * 16 + (lane & 1) * 8) = out;
    }
    if (valid && (lane & 3) == 0) d[g >> 2] = d16;
  }
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
      swiglu8(gu + r * 2 * F + f0, gu + r * 2 * F + F + f0, h);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = 0.0f;
    }
    float dv;
    const uint2 packed = q8_1_group8(h, &dv);
    if (valid) {
      *reinterpret_cast<uint2*>(q + g * 8) = packed;
      if ((lane & 3) == 0) d[g >> 2] = dv;
    }
  }
}

// GGUF block arrays -> planes, one thread per block.  A block starts on a 2-byte
// boundary only (34 or 18 bytes long), so it is read as 16-bit words; word 0 is the
// fp16 scale (little-endian, as on the device) and the quant bytes follow in order.
// The quants leave in 16-byte stores: block i of the flattened [N][K/32] array is
// bytes [32 i, 32 i + 32) of the Q8_0 plane and [16 i, 16 i + 16) of the Q4_0 plane.
// Like the weight quantisers, these kernels let no dependent start early.
template <int WORDS>
__device__ __forceinline__ void load_block_words(const uint16_t* blk, uint32_t* w) {
#pragma unroll
  for (int j = 0; j < WORDS / 2; ++j)
    w[j] = (uint32_t)blk[1 + 2 * j] | ((uint32_t)blk[2 + 2 * j] << 16);
}

__global__ void __launch_bounds__(kQuantThreads)
    repack_q8_0_kernel(const uint16_t* __restrict__ blocks, int64_t nblk,
                       int8_t* __restrict__ q, uint16_t* __restrict__ d) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblk; i += stride) {
    const uint16_t* blk = blocks + i * 17;
    uint32_t w[8];
    load_block_words<16>(blk, w);
    uint4* dst = reinterpret_cast<uint4*>(q + i * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    d[i] = blk[0];
  }
}

__global__ void __launch_bounds__(kQuantThreads)
    repack_q4_0_kernel(const uint16_t* __restrict__ blocks, int64_t nblk,
                       uint8_t* __restrict__ q4, uint16_t* __restrict__ d) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblk; i += stride) {
    const uint16_t* blk = blocks + i * 9;
    uint32_t w[4];
    load_block_words<8>(blk, w);
    *reinterpret_cast<uint4*>(q4 + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    d[i] = blk[0];
  }
}

// ---------------------------------------------------------------------------
// NVFP4 weight ingest: per-tensor fp32 scale g = amax / (6 * 448), per 16-block
// FP8 E4M3 scale s = e4m3(amax_block / (6 g)), FP4 E2M1 codes of w / (s g), all
// rounded to nearest even with saturation; element 2j in the low nibble of byte j.
// Three launches: the tensor's amax (as fp32 bits, atomicMax: non-negative floats
// order as their bit patterns), the blocks, then g.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3_rn_satfinite(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;  // the second source lands in the low byte
}

__device__ __forceinline__ float e4m3_value(uint32_t b) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)b));
  return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
}

// E2M1 code of v: the sign bit of v, and the magnitude code of the nearest grid value
// (0, .5, 1, 1.5, 2, 3, 4, 6) with ties to the even mantissa, saturating at 6.  The
// thresholds are the midpoints; a midpoint goes to the neighbour with mantissa 0.
__device__ __forceinline__ uint32_t e2m1_code(float v) {
  const float a = fabsf(v);
  const uint32_t m = a <= 0.25f ? 0u : a < 0.75f ? 1u : a <= 1.25f ? 2u : a < 1.75f ? 3u
                   : a <= 2.5f  ? 4u : a < 3.5f  ? 5u : a <= 5.0f  ? 6u : 7u;
  return (__float_as_uint(v) >> 31) << 3 | m;
}

__global__ void __launch_bounds__(kQuantThreads)
    amax_kernel(const float4* __restrict__ w, int64_t n4, unsigned int* __restrict__ amax_bits) {
  pdl_wait();
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = w[i];
    m = fmaxf(fmaxf(m, fabsf(v.x)), fmaxf(fabsf(v.y), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));
}

__global__ void __launch_bounds__(kQuantThreads)
    quantize_nvfp4_kernel(const float4* __restrict__ w, int64_t nblk,
                          const unsigned int* __restrict__ amax_bits, uint2* __restrict__ codes,
                          uint8_t* __restrict__ scales) {
  pdl_wait();
  const float g = __fdiv_rn(__uint_as_float(__ldcg(amax_bits)), 2688.0f);
  const float g6 = __fmul_rn(6.0f, g);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblk;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 t = w[i * 4 + q];
      v[4 * q] = t.x;
      v[4 * q + 1] = t.y;
      v[4 * q + 2] = t.z;
      v[4 * q + 3] = t.w;
    }
    float bmax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) bmax = fmaxf(bmax, fabsf(v[j]));
    const uint32_t sc = g == 0.0f ? 0u : e4m3_rn_satfinite(__fdiv_rn(bmax, g6));
    const float denom = __fmul_rn(e4m3_value(sc), g);
    uint32_t lo = 0, hi = 0;
    if (denom != 0.0f) {
#pragma unroll
      for (int j = 0; j < 8; ++j) lo |= e2m1_code(__fdiv_rn(v[j], denom)) << (4 * j);
#pragma unroll
      for (int j = 0; j < 8; ++j) hi |= e2m1_code(__fdiv_rn(v[8 + j], denom)) << (4 * j);
    }
    codes[i] = make_uint2(lo, hi);
    scales[i] = (uint8_t)sc;
  }
}

__global__ void nvfp4_scale_kernel(float* __restrict__ g) {
  pdl_wait();
  *g = __fdiv_rn(__uint_as_float(*reinterpret_cast<const unsigned int*>(g)), 2688.0f);
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

extern "C" memra_status memra_quantize_q4_0(const float* w, int64_t N, int64_t K, uint8_t* wq4,
                                            uint16_t* wd, cudaStream_t stream) {
  if (N < 0 || K < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return MEMRA_OK;
  if (!w || !wq4 || !wd) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(wq4, 16) || !aligned(wd, 2)) return MEMRA_ERR_ALIGNMENT;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  const int64_t groups = N * K / 8;
  cudaError_t e = launch_kernel(quantize_q4_0_kernel, dim3(quant_grid(groups, info)),
                                dim3(kQuantThreads), 0, stream, w, groups, wq4, wd);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

extern "C" memra_status memra_quantize_nvfp4(const float* w, int64_t N, int64_t K,
                                             uint8_t* codes, uint8_t* scales, float* g,
                                             cudaStream_t stream) {
  if (N < 0 || K < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return MEMRA_OK;
  if (!w || !codes || !scales || !g) return MEMRA_ERR_INVALID_ARG;
  if (N > INT64_MAX / K) return MEMRA_ERR_UNSUPPORTED;
  if (!aligned(w, 16) || !aligned(codes, 8) || !aligned(g, 4)) return MEMRA_ERR_ALIGNMENT;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float), stream);
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int* amax_bits = reinterpret_cast<unsigned int*>(g);
  const int64_t n4 = N * K / 4;
  e = launch_kernel(amax_kernel, dim3(quant_grid(n4, info)), dim3(kQuantThreads), 0, stream,
                    reinterpret_cast<const float4*>(w), n4, amax_bits);
  if (e != cudaSuccess) return cuda_fail(e);
  const int64_t nblk = N * K / 16;
  e = launch_kernel(quantize_nvfp4_kernel, dim3(quant_grid(nblk, info)), dim3(kQuantThreads), 0,
                    stream, reinterpret_cast<const float4*>(w), nblk,
                    static_cast<const unsigned int*>(amax_bits), reinterpret_cast<uint2*>(codes),
                    scales);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_kernel(nvfp4_scale_kernel, dim3(1), dim3(1), 0, stream, g);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

// Shared argument checks of the two repacks; *nblk receives N * K / 32.
static memra_status repack_args(const void* blocks, int64_t N, int64_t K, const void* q,
                                const void* d, int64_t block_bytes, int64_t* nblk) {
  *nblk = 0;
  if (N < 0 || K < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (N == 0 || K == 0) return MEMRA_OK;
  if (!blocks || !q || !d) return MEMRA_ERR_INVALID_ARG;
  if (N > INT64_MAX / block_bytes / (K / 32)) return MEMRA_ERR_UNSUPPORTED;
  if (!aligned(blocks, 2) || !aligned(q, 16) || !aligned(d, 2)) return MEMRA_ERR_ALIGNMENT;
  *nblk = N * (K / 32);
  return MEMRA_OK;
}

extern "C" memra_status memra_repack_q8_0(const void* blocks, int64_t N, int64_t K, int8_t* wq,
                                          uint16_t* wd, cudaStream_t stream) {
  int64_t nblk;
  memra_status st = repack_args(blocks, N, K, wq, wd, 34, &nblk);
  if (st != MEMRA_OK || nblk == 0) return st;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  cudaError_t e = launch_kernel(repack_q8_0_kernel, dim3(quant_grid(nblk, info)),
                                dim3(kQuantThreads), 0, stream,
                                static_cast<const uint16_t*>(blocks), nblk, wq, wd);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

extern "C" memra_status memra_repack_q4_0(const void* blocks, int64_t N, int64_t K, uint8_t* wq4,
                                          uint16_t* wd, cudaStream_t stream) {
  int64_t nblk;
  memra_status st = repack_args(blocks, N, K, wq4, wd, 18, &nblk);
  if (st != MEMRA_OK || nblk == 0) return st;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  cudaError_t e = launch_kernel(repack_q4_0_kernel, dim3(quant_grid(nblk, info)),
                                dim3(kQuantThreads), 0, stream,
                                static_cast<const uint16_t*>(blocks), nblk, wq4, wd);
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
