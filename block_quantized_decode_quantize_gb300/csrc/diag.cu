// Diagnostic: a plain read stream over device memory, the ceiling a weight-streaming
// product can approach on this GPU.  Not on the hot path.  sm_103a.
#include "common.cuh"

namespace memra {
namespace {

constexpr int kStreamThreads = 512;
constexpr int kStreamUnroll = 4;  // 16-byte loads in flight per thread per round

// Every 16-byte word of buf is read once; a thread folds its words with xor and the
// CTA's lanes combine them, so no load can be dropped.  Rounds of kStreamUnroll
// loads are issued before any is used.
__global__ void __launch_bounds__(kStreamThreads)
    read_stream_kernel(const uint4* __restrict__ buf, int64_t words,
                       uint32_t* __restrict__ sink) {
  uint32_t acc = 0;
  const int64_t stride = (int64_t)gridDim.x * kStreamThreads;
  int64_t i = (int64_t)blockIdx.x * kStreamThreads + threadIdx.x;
  for (; i + (kStreamUnroll - 1) * stride < words; i += kStreamUnroll * stride) {
    uint4 v[kStreamUnroll];
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u) v[u] = __ldcs(buf + i + u * stride);
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  for (; i < words; i += stride) {
    const uint4 v = __ldcs(buf + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(kFullMask, acc, o);
  if ((threadIdx.x & 31) == 0) atomicXor(sink + blockIdx.x, acc);
}

}  // namespace
}  // namespace memra

using namespace memra;

extern "C" memra_status memra_read_stream(const void* buf, int64_t bytes, uint32_t* sink,
                                          int32_t ctas_per_sm, cudaStream_t stream) {
  if (bytes < 0 || bytes % 16 != 0 || ctas_per_sm < 1 || ctas_per_sm > 4)
    return MEMRA_ERR_INVALID_ARG;
  if (bytes == 0) return MEMRA_OK;
  if (!buf || !sink) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(buf, 16) || !aligned(sink, 4)) return MEMRA_ERR_ALIGNMENT;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  const cudaError_t e =
      launch_kernel(read_stream_kernel, dim3((unsigned)(info.sms * ctas_per_sm)),
                    dim3(kStreamThreads), 0, stream, static_cast<const uint4*>(buf), bytes / 16,
                    sink);
  return e == cudaSuccess ? MEMRA_OK : cuda_fail(e);
}
