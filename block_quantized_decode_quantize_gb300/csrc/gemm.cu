// Q8_0 x q8_1 products: the M = 1 decode GEMV, the M <= 8 verify skinny GEMM and
// the routed-expert (MoE) GEMV, all from one weight-streaming kernel template.
//
// Work decomposition.  A "virtual row" is one weight row paired with the
// activation row(s) it multiplies: row n of W for the dense product, (expert k,
// row n) for the routed product.  Each CTA owns a contiguous range of virtual rows
// (balanced to within one row, or one group of top_k rows for the gated MoE), and
// splits it into chunks of R rows x 32 blocks: lane l of the warp that takes a
// chunk streams block 32p + l of each of the R rows (one 32-byte load per row),
// so a chunk is R contiguous 1-KB runs of the weight plane.  Chunks are dealt
// round-robin to the CTA's warps and each warp keeps U chunks of loads in flight
// in a register ring, so a CTA's share of HBM bandwidth does not depend on how
// its rows divide among warps.
//
// Arithmetic (fixed order, deterministic):
//   term  = (float(d_w) * d_x) * float(s_b)   s_b from 8 dp4a, exact int32
//   part  = xor-butterfly sum of the 32 lanes' terms (masks 16, 8, 4, 2, 1)
//   y     = sum over the parts of the row, sequential in part index.
// A row's value depends only on K, never on M, R, U, the grid or the other rows,
// so the M-row verify result equals the M = 1 GEMV bit for bit.
//
// Activations are staged once per CTA in shared memory in a half-block-split
// layout (xs[row][half][block] of 16 bytes) so that lane-consecutive blocks read
// consecutive 16-byte words without bank conflicts.  The weights never touch
// shared memory.  With programmatic dependent launch the weight loads of the
// first U chunks are issued before the wait on the preceding kernel.
#include <algorithm>

#include "common.cuh"

namespace memra {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kPartFloats = 8192;  // 32 KB of per-part partial sums per tile
constexpr int kMaxTopK = MEMRA_MAX_TOP_K;

enum Mode { kDense = 0, kMoeUngated = 1, kMoeGated = 2 };

struct Params {
  const int8_t* wq;       // dense weights or the expert bank
  const uint16_t* wd;
  int64_t N;              // rows of one weight matrix
  int64_t K;
  int nb;                 // blocks per row (K / 32)
  int cpr;                // parts (32-block runs) per row
  const int8_t* xq;
  const float* xd;
  int xrows;              // activation rows staged in shared memory
  float* y;
  int64_t vrows;          // virtual rows
  int unit;               // CTA ranges are multiples of this many virtual rows
  int tile_rows;          // virtual rows per partial-sum tile (multiple of unit and R)
  // routed experts
  const int32_t* ids;
  const float* gate_w;
  int top_k;
  int64_t E;
  int x_per_expert;
  int32_t* status;
};

template <int R>
struct ChunkRegs {
  Quants32 w[R];
  uint16_t d[R];
};

__host__ __device__ constexpr int next_pow2(int v) { return v <= 1 ? 1 : 2 * next_pow2((v + 1) / 2); }
__host__ __device__ constexpr int log2i(int v) { return v <= 1 ? 0 : 1 + log2i(v / 2); }

// Sum V = 2^t values across the warp with the xor-butterfly tree (masks 16, 8, 4,
// 2, 1), exchanging half of the remaining values at each of the first t stages.
// Every value goes through the same tree of pairwise sums as a plain butterfly.
// Afterwards lane l holds the total of value (l >> (5 - t)).
template <int V>
__device__ __forceinline__ void warp_sum_transposed(float (&v)[V], int lane) {
  constexpr int t = log2i(V);
#pragma unroll
  for (int s = 0; s < t; ++s) {
    const int mask = 16 >> s;
    const int half = V >> (s + 1);
    const bool upper = (lane & mask) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(kFullMask, send, mask);
    }
  }
#pragma unroll
  for (int s = t; s < 5; ++s) v[0] += __shfl_xor_sync(kFullMask, v[0], 16 >> s);
}

template <int M, int R, int U, int MODE>
__global__ void __launch_bounds__(kThreads, 2) q8_gemm_kernel(const Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int V = next_pow2(R * M);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nb = p.nb;
  const int cpr = p.cpr;

  // Shared memory: xs | xds | partial sums | expert ids | gate weights.
  uint4* xs = reinterpret_cast<uint4*>(smem);
  float* xds = reinterpret_cast<float*>(smem + (size_t)p.xrows * p.K);
  float* part = xds + (((size_t)p.xrows * nb + 3) & ~(size_t)3);
  int32_t* s_ids = reinterpret_cast<int32_t*>(part + (size_t)p.tile_rows * cpr * M);
  float* s_gate = reinterpret_cast<float*>(s_ids + kMaxTopK);

  const int64_t units = p.vrows / p.unit;
  const int64_t v_begin = units * blockIdx.x / gridDim.x * p.unit;
  const int64_t v_end = units * (blockIdx.x + 1) / gridDim.x * p.unit;

  pdl_launch_dependents();

  if (MODE != kDense) {
    // Expert ids and gate weights may come from the preceding kernel.
    pdl_wait();
    if (threadIdx.x < p.top_k) {
      const int32_t e = p.ids[threadIdx.x];
      const bool ok = e >= 0 && e < p.E;
      s_ids[threadIdx.x] = ok ? e : -1;
      s_gate[threadIdx.x] = (MODE == kMoeGated) ? p.gate_w[threadIdx.x] : 1.0f;
      if (!ok && p.status && blockIdx.x == 0) atomicOr(p.status, 1);
    }
    __syncthreads();
  }

  // Weight row of virtual row v (nullptr for an invalid expert) and its x row.
  auto row_of = [&](int64_t v, const int8_t*& q, const uint16_t*& d, int& xrow) -> bool {
    if (MODE == kDense) {
      q = p.wq + v * p.K;
      d = p.wd + v * nb;
      xrow = 0;
      return true;
    }
    int64_t k, n;
    if (MODE == kMoeUngated) {
      k = v / p.N;
      n = v - k * p.N;
    } else {
      n = v / p.top_k;
      k = v - n * p.top_k;
    }
    const int e = s_ids[k];
    xrow = p.x_per_expert ? (int)k : 0;
    if (e < 0) return false;
    const int64_t row = (int64_t)e * p.N + n;
    q = p.wq + row * p.K;
    d = p.wd + row * nb;
    return true;
  };

  bool staged = false;
  for (int64_t tile_v0 = v_begin; tile_v0 < v_end; tile_v0 += p.tile_rows) {
    const int tile_n = (int)min((int64_t)p.tile_rows, v_end - tile_v0);
    const int groups = (tile_n + R - 1) / R;
    const int nchunks = groups * cpr;

    auto load_chunk = [&](ChunkRegs<R>& regs, int c) {
      const int g = c / cpr;
      const int pt = c - g * cpr;
      const int b = pt * 32 + lane;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int vi = g * R + r;
        const int8_t* q;
        const uint16_t* d;
        int xrow;
        bool ok = b < nb && vi < tile_n;
        if (ok) ok = row_of(tile_v0 + vi, q, d, xrow);
        if (ok) {
          regs.w[r] = ld_stream_32B(q + (int64_t)b * 32);
          regs.d[r] = ld_stream_u16(d + b);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) regs.w[r].w[i] = 0u;
          regs.d[r] = 0;
        }
      }
    };

    auto compute_chunk = [&](const ChunkRegs<R>& regs, int c) {
      const int g = c / cpr;
      const int pt = c - g * cpr;
      const int b = pt * 32 + lane;
      float vals[V];
#pragma unroll
      for (int i = 0; i < V; ++i) vals[i] = 0.0f;
      if (b < nb) {
        int xrow0 = 0;
        if (MODE != kDense) {
          const int8_t* q;
          const uint16_t* d;
          row_of(tile_v0 + g * R, q, d, xrow0);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const int xr = (MODE == kDense) ? m : xrow0;
          const uint4 lo = xs[((size_t)xr * 2 + 0) * nb + b];
          const uint4 hi = xs[((size_t)xr * 2 + 1) * nb + b];
          const float dx = xds[(size_t)xr * nb + b];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int s = block_dot(regs.w[r], lo, hi);
            const float c_b = __half2float(__ushort_as_half(regs.d[r])) * dx;
            vals[r * M + m] = c_b * (float)s;
          }
        }
      }
      warp_sum_transposed<V>(vals, lane);
      constexpr int t = log2i(V);
      if ((lane & ((32 >> t) - 1)) == 0) {
        const int idx = lane >> (5 - t);
        if (idx < R * M) {
          const int r = idx / M;
          const int m = idx - r * M;
          const int vi = g * R + r;
          if (vi < tile_n) part[((size_t)vi * cpr + pt) * M + m] = vals[0];
        }
      }
    };

    ChunkRegs<R> ring[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = warp + u * kWarps;
      if (c < nchunks) load_chunk(ring[u], c);
    }

    if (!staged) {
      if (MODE == kDense) pdl_wait();
      // Stage the activation rows: 16-byte words into the half-block-split layout.
      const int64_t words = (int64_t)p.xrows * p.K / 16;
      for (int64_t i = threadIdx.x; i < words; i += kThreads) {
        const int64_t row = i / (p.K / 16);
        const int64_t j = i - row * (p.K / 16);
        const int64_t blk = j >> 1;
        const int64_t h = j & 1;
        xs[(row * 2 + h) * nb + blk] = reinterpret_cast<const uint4*>(p.xq)[i];
      }
      const int64_t nd = (int64_t)p.xrows * nb;
      for (int64_t i = threadIdx.x; i < nd; i += kThreads) xds[i] = p.xd[i];
      __syncthreads();
      staged = true;
    }

    for (int c = warp; c < nchunks; c += U * kWarps) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int cc = c + u * kWarps;
        if (cc < nchunks) {
          compute_chunk(ring[u], cc);
          const int nc = cc + U * kWarps;
          if (nc < nchunks) load_chunk(ring[u], nc);
        }
      }
    }
    __syncthreads();

    // Epilogue: sum each row's parts in order and store.
    if (MODE == kMoeGated) {
      const int rows_n = tile_n / p.top_k;
      for (int i = threadIdx.x; i < rows_n; i += kThreads) {
        float acc = 0.0f;
        for (int k = 0; k < p.top_k; ++k) {
          if (s_ids[k] < 0) continue;
          const int vi = i * p.top_k + k;
          float yk = 0.0f;
          for (int pt = 0; pt < cpr; ++pt) yk += part[(size_t)vi * cpr + pt];
          acc += s_gate[k] * yk;
        }
        p.y[tile_v0 / p.top_k + i] = acc;
      }
    } else {
      for (int i = threadIdx.x; i < tile_n * M; i += kThreads) {
        const int vi = i / M;
        const int m = i - vi * M;
        float acc = 0.0f;
        for (int pt = 0; pt < cpr; ++pt) acc += part[((size_t)vi * cpr + pt) * M + m];
        p.y[(int64_t)m * p.vrows + tile_v0 + vi] = acc;
      }
    }
    __syncthreads();
  }
}

// Test export: exact int32 block sums with the same dp4a routine.
__global__ void __launch_bounds__(256)
    block_dots_kernel(const int8_t* __restrict__ wq, int64_t N, int64_t K,
                      const int8_t* __restrict__ xq, int64_t M, int32_t* __restrict__ s) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t nb = K / 32;
  const int64_t total = M * N * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / (N * nb);
    const int64_t rem = i - m * N * nb;
    const int64_t n = rem / nb;
    const int64_t b = rem - n * nb;
    const Quants32 w = ld_stream_32B(wq + n * K + b * 32);
    const uint4* xp = reinterpret_cast<const uint4*>(xq + m * K + b * 32);
    s[i] = block_dot(w, xp[0], xp[1]);
  }
}

// ----------------------------------------------------------------------------
// Host dispatch.
// ----------------------------------------------------------------------------

size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }

size_t smem_bytes(const Params& p, int M) {
  size_t b = align16((size_t)p.xrows * p.K);                            // xs
  b += ((size_t)p.xrows * p.nb + 3) / 4 * 16;                           // xds
  b += align16((size_t)p.tile_rows * p.cpr * M * sizeof(float));        // partial sums
  b += 2 * kMaxTopK * sizeof(int32_t);                                  // ids, gates
  return b;
}

template <int M, int R, int U, int MODE>
memra_status launch_gemm(Params p, cudaStream_t stream) {
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  p.nb = (int)(p.K / 32);
  p.cpr = (p.nb + 31) / 32;
  const int64_t units = p.vrows / p.unit;
  // Tile: as many rows as the partial-sum budget allows, a multiple of both the
  // range unit and R.
  int64_t step = p.unit;
  while (step % R) step += p.unit;
  int64_t tile = kPartFloats / ((int64_t)p.cpr * M);
  tile = std::max<int64_t>(step, tile / step * step);
  // Resident CTAs per SM from the shared-memory footprint (registers allow two).
  p.tile_rows = (int)tile;
  size_t smem = smem_bytes(p, M);
  if (smem > (size_t)info.max_smem_optin) return MEMRA_ERR_UNSUPPORTED;
  const int per_sm = (2 * (smem + 1024) <= 228 * 1024) ? 2 : 1;
  int64_t grid = std::min<int64_t>(units, (int64_t)info.sms * per_sm);
  // Shrink the tile to the CTA's row range when that is smaller.
  const int64_t rows_per_cta = (units + grid - 1) / grid * p.unit;
  if (rows_per_cta < tile) {
    tile = (rows_per_cta + step - 1) / step * step;
    p.tile_rows = (int)tile;
    smem = smem_bytes(p, M);
  }
  auto kernel = q8_gemm_kernel<M, R, U, MODE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cudaError_t e = launch_kernel(kernel, dim3((unsigned)grid), dim3(kThreads), smem, stream, p);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

template <int MODE>
memra_status dispatch_m(const Params& p, int M, cudaStream_t s) {
  switch (M) {
    case 1: return launch_gemm<1, 1, 8, MODE>(p, s);
    case 2: return launch_gemm<2, 1, 8, MODE>(p, s);
    case 3: return launch_gemm<3, 1, 8, MODE>(p, s);
    case 4: return launch_gemm<4, 2, 4, MODE>(p, s);
    case 5: return launch_gemm<5, 2, 4, MODE>(p, s);
    case 6: return launch_gemm<6, 2, 4, MODE>(p, s);
    case 7: return launch_gemm<7, 2, 4, MODE>(p, s);
    case 8: return launch_gemm<8, 4, 2, MODE>(p, s);
  }
  return MEMRA_ERR_UNSUPPORTED;
}

memra_status zero_fill(float* y, int64_t count, cudaStream_t s) {
  if (count == 0) return MEMRA_OK;
  cudaError_t e = cudaMemsetAsync(y, 0, (size_t)count * sizeof(float), s);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

bool x_fits(int64_t xrows, int64_t K) {
  return xrows * K + xrows * (K / 32) * 4 <= MEMRA_MAX_X_BYTES;
}

}  // namespace
}  // namespace memra

using namespace memra;

extern "C" memra_status memra_q8_0_gemm_small_m(const int8_t* wq, const uint16_t* wd, int64_t N,
                                                int64_t K, int64_t M, const int8_t* xq,
                                                const float* xd, float* y, cudaStream_t stream) {
  if (N < 0 || K < 0 || M < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (M > MEMRA_MAX_M) return MEMRA_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (N == 0 || M == 0) return MEMRA_OK;
  if (!y) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4)) return MEMRA_ERR_ALIGNMENT;
  if (K == 0) return zero_fill(y, M * N, stream);
  if (!wq || !wd || !xq || !xd) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(wq, 32) || !aligned(wd, 2) || !aligned(xq, 16) || !aligned(xd, 4))
    return MEMRA_ERR_ALIGNMENT;
  if (!x_fits(M, K)) return MEMRA_ERR_UNSUPPORTED;
  Params p{};
  p.wq = wq;
  p.wd = wd;
  p.N = N;
  p.K = K;
  p.xq = xq;
  p.xd = xd;
  p.xrows = (int)M;
  p.y = y;
  p.vrows = N;
  p.unit = 1;
  return dispatch_m<kDense>(p, (int)M, stream);
}

extern "C" memra_status memra_q8_0_gemv(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K,
                                        const int8_t* xq, const float* xd, float* y,
                                        cudaStream_t stream) {
  return memra_q8_0_gemm_small_m(wq, wd, N, K, 1, xq, xd, y, stream);
}

extern "C" memra_status memra_q8_0_moe_gemv(const int8_t* wq_bank, const uint16_t* wd_bank,
                                            int64_t E, int64_t N, int64_t K, const int32_t* ids,
                                            const float* gate_w, int64_t top_k, const int8_t* xq,
                                            const float* xd, int32_t x_per_expert, float* y,
                                            int32_t* dev_status, cudaStream_t stream) {
  if (E < 1 || N < 0 || K < 0 || K % 32 != 0 || top_k < 1) return MEMRA_ERR_INVALID_ARG;
  if (x_per_expert != 0 && x_per_expert != 1) return MEMRA_ERR_INVALID_ARG;
  if (top_k > MEMRA_MAX_TOP_K) return MEMRA_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX || E > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (N == 0) return MEMRA_OK;
  if (!y || !ids) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4) || !aligned(ids, 4) || (gate_w && !aligned(gate_w, 4)) ||
      (dev_status && !aligned(dev_status, 4)))
    return MEMRA_ERR_ALIGNMENT;
  if (K == 0) return zero_fill(y, gate_w ? N : top_k * N, stream);
  if (!wq_bank || !wd_bank || !xq || !xd) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(wq_bank, 32) || !aligned(wd_bank, 2) || !aligned(xq, 16) || !aligned(xd, 4))
    return MEMRA_ERR_ALIGNMENT;
  const int64_t xrows = x_per_expert ? top_k : 1;
  if (!x_fits(xrows, K)) return MEMRA_ERR_UNSUPPORTED;
  Params p{};
  p.wq = wq_bank;
  p.wd = wd_bank;
  p.N = N;
  p.K = K;
  p.xq = xq;
  p.xd = xd;
  p.xrows = (int)xrows;
  p.y = y;
  p.vrows = top_k * N;
  p.ids = ids;
  p.gate_w = gate_w;
  p.top_k = (int)top_k;
  p.E = E;
  p.x_per_expert = x_per_expert;
  p.status = dev_status;
  if (gate_w) {
    p.unit = (int)top_k;
    return launch_gemm<1, 1, 8, kMoeGated>(p, stream);
  }
  p.unit = 1;
  return launch_gemm<1, 1, 8, kMoeUngated>(p, stream);
}

extern "C" memra_status memra_q8_0_block_dots(const int8_t* wq, int64_t N, int64_t K,
                                              const int8_t* xq, int64_t M, int32_t* s,
                                              cudaStream_t stream) {
  if (N < 0 || K < 0 || M < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (N == 0 || K == 0 || M == 0) return MEMRA_OK;
  if (!wq || !xq || !s) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(wq, 32) || !aligned(xq, 16) || !aligned(s, 4)) return MEMRA_ERR_ALIGNMENT;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  const int64_t total = M * N * (K / 32);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)info.sms * 8);
  cudaError_t e = launch_kernel(block_dots_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                                wq, N, K, xq, M, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}
