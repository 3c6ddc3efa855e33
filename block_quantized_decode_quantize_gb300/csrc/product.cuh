// Device routines of the product kernels (gemm.cu): the one fp32 summation order of a
// row, the exact dp4a block dot, and the in-kernel q8_1 quantisation of activations.
// sm_103a only.
#pragma once

#include "common.cuh"

namespace memra {

#ifndef MEMRA_SLICE_PARTS
#define MEMRA_SLICE_PARTS 4
#endif
constexpr int kSlicePartsMax = MEMRA_SLICE_PARTS;

__host__ __device__ constexpr int next_pow2(int v) { return v <= 1 ? 1 : 2 * next_pow2((v + 1) / 2); }
__host__ __device__ constexpr int log2i(int v) { return v <= 1 ? 0 : 1 + log2i(v / 2); }

__host__ __device__ inline int slices_for(int cpr) {
  return (cpr + kSlicePartsMax - 1) / kSlicePartsMax;
}

// Sum V = 2^t values across the warp with the xor-butterfly tree (masks 16, 8, 4,
// 2, 1), exchanging half of the remaining values at each of the first t stages.
// Every value goes through the same tree of pairwise sums as a plain butterfly
// (fp32 addition is commutative).  Afterwards lane l holds value (l >> (5 - t)).
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
      v[i] = __fadd_rn(keep, __shfl_xor_sync(kFullMask, send, mask));
    }
  }
#pragma unroll
  for (int s = t; s < 5; ++s) v[0] = __fadd_rn(v[0], __shfl_xor_sync(kFullMask, v[0], 16 >> s));
}

// Reduce acc[R][M] of every lane and store the slice partials:
// part[(row * S + s) * M + m] for rows < nrows.
template <int R, int M>
__device__ __forceinline__ void store_partials(float (&acc)[R][M], int lane, float* part,
                                               int row0, int nrows, int s, int S) {
  constexpr int V = next_pow2(R * M);
  float v[V];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) v[r * M + m] = acc[r][m];
#pragma unroll
  for (int i = R * M; i < V; ++i) v[i] = 0.0f;
  warp_sum_transposed<V>(v, lane);
  constexpr int t = log2i(V);
  if ((lane & ((32 >> t) - 1)) == 0) {
    const int idx = lane >> (5 - t);
    if (idx < R * M) {
      const int r = idx / M;
      const int m = idx - r * M;
      if (r < nrows) part[((size_t)(row0 + r) * S + s) * M + m] = v[0];
    }
  }
}

// One block of one weight row against an x block: the exact int32 sum from two
// 16-byte halves (in either order: integer addition is exact).
__device__ __forceinline__ int dot_halves(const uint4& w0, const uint4& w1, const uint4& x0,
                                          const uint4& x1) {
  int s = 0;
  s = __dp4a((int)w0.x, (int)x0.x, s);
  s = __dp4a((int)w0.y, (int)x0.y, s);
  s = __dp4a((int)w0.z, (int)x0.z, s);
  s = __dp4a((int)w0.w, (int)x0.w, s);
  s = __dp4a((int)w1.x, (int)x1.x, s);
  s = __dp4a((int)w1.y, (int)x1.y, s);
  s = __dp4a((int)w1.z, (int)x1.z, s);
  s = __dp4a((int)w1.w, (int)x1.w, s);
  return s;
}

__device__ __forceinline__ float block_term_acc(float acc, uint16_t dw_bits, float dx, int s) {
  const float c = __fmul_rn(__half2float(__ushort_as_half(dw_bits)), dx);
  return __fmaf_rn(c, (float)s, acc);
}

// Activation input of a product: q8_1 planes, or values quantised in the kernel's
// prologue (bf16, fp32, SwiGLU of an fp32 gate|up row pair, or the first K floats of
// fp32 rows of 2K floats: the SwiGLU rows a paired gate|up product writes).
enum XIn { kXq8 = 0, kXbf16 = 1, kXf32 = 2, kXswiglu = 3, kXhalf = 4 };

// The 8 activation values of group g (row-major [rows][K], K % 8 == 0).
template <int XIN>
__device__ __forceinline__ void load_x_group(const void* xin, int g, int K, float v[8]) {
  if (XIN == kXbf16) {
    load8_bf16(static_cast<const uint16_t*>(xin) + (size_t)g * 8, v);
  } else if (XIN == kXf32) {
    load8_f32(static_cast<const float*>(xin) + (size_t)g * 8, v);
  } else if (XIN == kXhalf) {
    const int gpr = K / 8;
    const int row = g / gpr;
    load8_f32(static_cast<const float*>(xin) + (size_t)row * 2 * K + (g - row * gpr) * 8, v);
  } else {
    const int gpr = K / 8;
    const int row = g / gpr;
    const int f0 = (g - row * gpr) * 8;
    const float* gu = static_cast<const float*>(xin) + (size_t)row * 2 * K;
    swiglu8(gu + f0, gu + K + f0, v);
  }
}

// Quantise `rows` activation rows of K values (bf16 bits, fp32, or SwiGLU of gate|up
// pairs) into the shared-memory q8_1 planes (natural layout).  Called by `nwarps`
// whole warps (warp index w).  Thread t = 32w + lane takes groups t, t + T, t + 2T,
// ... (T = 32 nwarps; four consecutive lanes hold one 32-value block) and issues the
// loads of up to U of them before quantising any, so the prologue pays one memory
// latency per U T groups; bf16 rows are loaded raw (16 bytes a group), which lets U
// reach 6, enough for any K <= 18432 in a single round with 12 warps.
template <int XIN>
__device__ __forceinline__ void quantize_rows_to_smem(const void* xin, int rows, int K,
                                                      int8_t* xs, float* xds, int w, int nwarps,
                                                      int lane) {
  constexpr int U = XIN == kXbf16 ? 6 : 2;
  const int groups = rows * K / 8;  // fits: rows * K is bounded by MEMRA_MAX_X_BYTES
  const int T = nwarps * 32;
  const int t = w * 32 + lane;
  auto store = [&](int g, const float (&v)[8]) {
    float d;
    const uint2 q = q8_1_group8(v, &d);
    if (g < groups) {
      *reinterpret_cast<uint2*>(xs + (size_t)g * 8) = q;
      if ((lane & 3) == 0) xds[g >> 2] = d;
    }
  };
  for (int base = 0; base < groups; base += U * T) {
    if (base + w * 32 >= groups) break;  // warp-uniform: no group of this warp is left
    if (XIN == kXbf16) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = base + u * T + t;
        raw[u] = g < groups
                     ? *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(xin) +
                                                       (size_t)g * 8)
                     : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (base + u * T + w * 32 >= groups) break;  // warp-uniform
        const uint32_t wv[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[2 * i] = __uint_as_float(wv[i] << 16);
          v[2 * i + 1] = __uint_as_float(wv[i] & 0xffff0000u);
        }
        store(base + u * T + t, v);
      }
    } else {
      float v[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = base + u * T + t;
        if (g < groups) {
          load_x_group<XIN>(xin, g, K, v[u]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) v[u][i] = 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (base + u * T + w * 32 >= groups) break;  // warp-uniform
        store(base + u * T + t, v[u]);
      }
    }
  }
}

// Copy q8_1 activation planes (xq: qbytes, xd: dbytes; both multiples of 16 and
// 16-byte aligned) into shared memory with L2-only 16-byte loads, U loads in flight
// per thread before any store.  Called by `nt` threads (index t).
template <int U>
__device__ __forceinline__ void copy_x_to_smem(const int8_t* xq, const float* xd, int qbytes,
                                               int dbytes, int8_t* xs, float* xds, int t,
                                               int nt) {
  const int nq = qbytes / 16;
  const int total = nq + dbytes / 16;
  for (int base = t; base < total; base += nt * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * nt;
      if (i < total)
        v[u] = i < nq ? ld_cg_16B(xq + (size_t)i * 16)
                      : ld_cg_16B(reinterpret_cast<const int8_t*>(xd) + (size_t)(i - nq) * 16);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * nt;
      if (i < total) {
        if (i < nq)
          reinterpret_cast<uint4*>(xs)[i] = v[u];
        else
          reinterpret_cast<uint4*>(xds)[i - nq] = v[u];
      }
    }
  }
}

// Slice boundaries (in parts) for the row's S slices: tab[s] = s*cpr/S.
__device__ __forceinline__ void fill_slice_table(int* tab, int cpr, int S, int tid, int nthreads) {
  for (int s = tid; s <= S; s += nthreads) tab[s] = (int)(((long long)s * cpr) / S);
}

}  // namespace memra
