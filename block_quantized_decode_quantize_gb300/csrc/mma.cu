// Q8_0 x q8_1 products of 1..8 activation rows with the exact int32 block sums formed
// on the tensor cores: the verify skinny GEMM of memra_q8_0_gemm_small_m (and each
// pass of a batched call).
//
// The arithmetic is the library's one definition (gemm.cu): per row, nb = K/32
// blocks in parts of 32 blocks; slices of up to 4 parts; "lane class" l of a part is
// its block l.  Within a slice the sum of class l runs over the slice's parts in
// ascending order, acc = fma(fl(d_w * d_x), float(s_b), acc) from 0; the 32 class
// sums are added by the xor-butterfly tree (pairs l, l^16, then ^8, ^4, ^2, ^1); the
// row is the slice values summed in slice order.  Here s_b comes from one int8
// mma.sync m16n8k32: A = the block's 32 quants of 16 weight rows, B = the same block
// of 8 activation rows (rows past M are zero), D = 16 x 8 exact int32 sums (|s_b| <=
// 32 * 127^2).  So every output is bit-identical to the CUDA-core kernels', for any M
// and grid.
//
// Layout.  One CTA per SM owns a contiguous range of weight rows, streamed by warp 0
// in stages of 8 full rows: one bulk copy per row (a copy of K bytes keeps the copy
// engine near the HBM rate) into shared rows K + 16 bytes apart, so that the 8 rows
// of an ldmatrix phase fall in distinct banks, and the rows' scales as one 3-D tensor
// box (32 scales x 8 rows x the row's parts, 64-byte swizzle: scale loads of 8 rows
// are conflict-free too).  Two consecutive stages form a 16-row tile (a lone last
// stage stands for both halves; its repeated rows are not stored).  Eight consumer
// warps each own four lane classes {c, c+8, c+16, c+24} of every part: per tile and
// part 4 MMAs, all parts of a tile in flight.  At a slice's end each warp adds its
// four classes (the first two levels of the tree), the eight results meet in shared
// memory, and 128 threads finish the tree and add the slice into their output (row,
// activation row) in slice order.  Eight full rows and the activation must fit in
// shared memory, so K is limited (about 10000 at M = 8); larger K, and everything
// the tensor-core kernel does not take, runs on the CUDA-core kernels.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "product.cuh"

namespace memra {
namespace {

constexpr int kMmaConsumerWarps = 8;
constexpr int kMmaThreads = 32 * (1 + kMmaConsumerWarps);
constexpr int kMmaTileRows = 16;
constexpr int kMmaStageRows = 8;
constexpr int kMmaMaxStages = 16;
constexpr int kMmaPad = 8;                          // activation rows of the B operand
constexpr int kMmaMaxParts = 5;                     // K <= 5120: each warp's x in registers
constexpr uint32_t kMmaHeader = 1024;
constexpr int kHdrEmpty = 8 * kMmaMaxStages;
constexpr int kHdrXdone = 16 * kMmaMaxStages;
constexpr int kHdrAbort = kHdrXdone + 16;
constexpr int kHdrSlice = kHdrAbort + 16;
constexpr int kMmaMaxSlices = (int)((kMmaHeader - kHdrSlice) / 4) - 1;

size_t align_up_sz(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct MmaParams {
  CUtensorMap wd_map;  // uint16 scales viewed as [parts][N rows][32]: box 32 x 8 rows x cpr
  const int8_t* wq;    // [N][K]
  const int8_t* xq;    // [M][K]
  const float* xd;     // [M][K/32]
  float* y;            // [M][N]
  int64_t N;
  int K, nb, cpr, S, M;
  int ns;              // ring stages
  uint32_t stage_bytes;
  uint32_t scale_off;  // the stage's scale box, after its 8 quant rows
  int ws;              // bytes between weight rows of a stage (K + 16)
  uint32_t off_ubuf, off_ring;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar),
        "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&a)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}

// D = A * B over one 32-element block: A 16 x 32 int8 (row-major fragments), B 32 x 8
// int8 (column-major fragments), D int32, exact.
__device__ __forceinline__ void mma_block(const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          int (&d)[4]) {
  asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%10, %10, %10, %10};"
      : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

__global__ void __launch_bounds__(kMmaThreads, 1) q8_mma_kernel(const __grid_constant__ MmaParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // Swizzled tensor copies need 1024-byte aligned destinations.
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kHdrAbort);
  int* s_slice = reinterpret_cast<int*>(smem + kHdrSlice);
  float* ubuf = reinterpret_cast<float*>(smem + p.off_ubuf);
  unsigned char* ring = smem + p.off_ring;
  auto full_bar = [&](int i) { return smem_addr(smem + 8 * i); };
  auto empty_bar = [&](int i) { return smem_addr(smem + kHdrEmpty + 8 * i); };
  // The activation is staged in the ring's last slot; the producer fills that slot
  // only once every consumer warp has taken its fragments into registers.
  const uint32_t xdone_bar = smem_addr(smem + kHdrXdone);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ns = p.ns;
  const int64_t r0 = p.N * blockIdx.x / gridDim.x;
  const int64_t r1 = p.N * (blockIdx.x + 1) / gridDim.x;
  // Stages of up to 8 rows; stage j holds rows [r0 + 8j, min(r0 + 8j + 8, r1)).
  const int nst = (int)((r1 - r0 + kMmaStageRows - 1) / kMmaStageRows);
  const int ntiles = (nst + 1) / 2;
  auto stage_rows = [&](int j) -> int {
    const int64_t left = r1 - r0 - (int64_t)j * kMmaStageRows;
    return (int)(left < kMmaStageRows ? left : kMmaStageRows);
  };

  // Weights do not depend on the preceding kernel: let the next one launch at once.
  pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < ns; ++i) {
        mbar_init(full_bar(i), 1);
        mbar_init(empty_bar(i), kMmaConsumerWarps);
      }
      mbar_init(xdone_bar, kMmaConsumerWarps);
      *abort_flag = 0;
      mbar_init_fence();
    }
    __syncwarp();
    asm volatile("bar.arrive 2, %0;" ::"n"(kMmaThreads) : "memory");
  } else {
    fill_slice_table(s_slice, p.cpr, p.S, threadIdx.x - 32, kMmaThreads - 32);
    asm volatile("bar.sync 2, %0;" ::"n"(kMmaThreads) : "memory");
  }

  int issued = 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the stages (so that it reaches the final barrier
    // converged); lane 0 waits for free slots and issues the copies.
    const uint64_t policy = l2_evict_first_policy();
    const uint32_t scale_bytes = (uint32_t)kMmaStageRows * 64u * (uint32_t)p.cpr;
    for (int j = 0; j < nst; ++j) {
      const int slot = j % ns;
      bool ok = true;
      if (lane == 0 && j == ns - 1) ok = mbar_wait(xdone_bar, 0, abort_flag);
      if (lane == 0 && j >= ns) ok = mbar_wait(empty_bar(slot), ((j / ns) - 1) & 1, abort_flag);
      if (!__shfl_sync(kFullMask, ok ? 1 : 0, 0)) break;
      if (lane == 0) {
        const int nr = stage_rows(j);
        const int64_t row0 = r0 + (int64_t)j * kMmaStageRows;
        const uint32_t dst = smem_addr(ring + (size_t)slot * p.stage_bytes);
        // The scale box always lands 8 rows (past N: zeros; past r1: unused).
        mbar_arrive_expect_tx(full_bar(slot), (uint32_t)nr * (uint32_t)p.K + scale_bytes);
        for (int r = 0; r < nr; ++r)
          bulk_g2s_hint(dst + (uint32_t)(r * p.ws), p.wq + (row0 + r) * (int64_t)p.K,
                        (uint32_t)p.K, full_bar(slot), policy);
        tma_load_3d(dst + p.scale_off, &p.wd_map, 0, (int)row0, 0, full_bar(slot), policy);
      }
      __syncwarp();
      issued = j + 1;
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;  // lane classes cw, cw + 8, cw + 16, cw + 24 of every part
    const int ct = threadIdx.x - 32;
    const int g = lane >> 2;
    const int tq = lane & 3;
    // The activation comes from the preceding kernel.  It is staged once, with
    // coalesced 16-byte loads: the quants into the ring's last slot (rows K + 16 bytes
    // apart, so that 8 rows at one column fall in distinct banks; rows M..7 zero), the
    // scales into the slice buffer (rows nb + 4 floats apart).  A warp only ever reads
    // its own lane classes of it, 4 blocks per part, and keeps them in registers: B
    // operands (activation row g, bytes 4 tq .. and 16 + 4 tq .. of the block) and the
    // scales of activation rows 2 tq and 2 tq + 1.
    pdl_wait();
    const int xs_stride = p.K + 16;
    const int ds_stride = p.nb + 4;
    int8_t* xs = reinterpret_cast<int8_t*>(ring + (size_t)(ns - 1) * p.stage_bytes);
    float* xds = ubuf;
    {
      constexpr int U = 8;
      constexpr int T = kMmaConsumerWarps * 32;
      const int qw = p.K / 16;
      const int nq = kMmaPad * qw;
      const int dw4 = p.nb / 4;
      const int nd = kMmaPad * dw4;
      for (int base = ct; base < nq + nd; base += U * T) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = base + u * T;
          v[u] = make_uint4(0u, 0u, 0u, 0u);
          if (i < nq) {
            const int m = i / qw;
            if (m < p.M) v[u] = ld_cg_16B(p.xq + (size_t)m * p.K + (size_t)(i - m * qw) * 16);
          } else if (i < nq + nd) {
            const int m = (i - nq) / dw4;
            if (m < p.M)
              v[u] = ld_cg_16B(p.xd + (size_t)m * p.nb + (size_t)(i - nq - m * dw4) * 4);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int i = base + u * T;
          if (i < nq) {
            const int m = i / qw;
            *reinterpret_cast<uint4*>(xs + (size_t)m * xs_stride + (size_t)(i - m * qw) * 16) = v[u];
          } else if (i < nq + nd) {
            const int m = (i - nq) / dw4;
            *reinterpret_cast<uint4*>(xds + (size_t)m * ds_stride + (size_t)(i - nq - m * dw4) * 4) =
                v[u];
          }
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kMmaConsumerWarps * 32) : "memory");
    uint32_t xb0[kMmaMaxParts][4], xb1[kMmaMaxParts][4];
    float xa[kMmaMaxParts][4], xc[kMmaMaxParts][4];
#pragma unroll
    for (int pt = 0; pt < kMmaMaxParts; ++pt) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int b = pt * 32 + cw + 8 * q;
        const bool in = pt < p.cpr;
        const int8_t* xp = xs + (size_t)g * xs_stride + (size_t)b * 32 + 4 * tq;
        xb0[pt][q] = in ? *reinterpret_cast<const uint32_t*>(xp) : 0u;
        xb1[pt][q] = in ? *reinterpret_cast<const uint32_t*>(xp + 16) : 0u;
        xa[pt][q] = in ? xds[(size_t)(2 * tq) * ds_stride + b] : 0.0f;
        xc[pt][q] = in ? xds[(size_t)(2 * tq + 1) * ds_stride + b] : 0.0f;
      }
    }
    // Every consumer is done with the staged activation before the slot and the slice
    // buffer are reused.
    asm volatile("bar.sync 1, %0;" ::"n"(kMmaConsumerWarps * 32) : "memory");
    if (lane == 0) mbar_arrive(xdone_bar);

    // ldmatrix: lane i addresses tile row (i & 7) + 8 ((i >> 3) & 1) (rows 8..15 in the
    // tile's second stage) at the block's first (i < 16) or second 16 bytes.
    const int ri = lane & 7;
    const bool hi_row = ((lane >> 3) & 1) != 0;
    const uint32_t a_lane = (uint32_t)(ri * p.ws + (lane >> 4) * 16 + cw * 32);
    // Scales of row g (and row g of the second stage): part p, element j = cw + 8q:
    // p * 256 + g * 32 + ((q ^ ((g >> 1) & 3)) << 3) + cw halves into the box.
    const int swz = (g >> 1) & 3;

    int ub = 0;
    bool live = true;  // false once a wait gave up: the control flow goes on, the work stops
    for (int t = 0; t < ntiles; ++t) {
      const int ja = 2 * t;
      const bool two = ja + 1 < nst;
      const int sa_slot = ja % ns;
      const int sb_slot = two ? (ja + 1) % ns : sa_slot;
      if (live && !mbar_wait(full_bar(sa_slot), (ja / ns) & 1, abort_flag)) live = false;
      if (two && live && !mbar_wait(full_bar(sb_slot), ((ja + 1) / ns) & 1, abort_flag))
        live = false;
      const uint32_t st_a = smem_addr(ring + (size_t)sa_slot * p.stage_bytes);
      const uint32_t st_b = smem_addr(ring + (size_t)sb_slot * p.stage_bytes);
      const uint32_t a_base = (hi_row ? st_b : st_a) + a_lane;
      const uint16_t* sc_a =
          reinterpret_cast<const uint16_t*>(ring + (size_t)sa_slot * p.stage_bytes + p.scale_off);
      const uint16_t* sc_b =
          reinterpret_cast<const uint16_t*>(ring + (size_t)sb_slot * p.stage_bytes + p.scale_off);
      float yacc = 0.0f;
      for (int s = 0; s < p.S; ++s) {
        float acc[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[q][i] = 0.0f;
        if (live) {
          const int plo = s_slice[s];
          const int phi = s_slice[s + 1];
#pragma unroll
          for (int pt = 0; pt < kMmaMaxParts; ++pt) {
            if (pt < plo || pt >= phi) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t a[4];
              ldsm_x4(a_base + (uint32_t)(pt * 1024 + q * 256), a);
              int d[4];
              mma_block(a, xb0[pt][q], xb1[pt][q], d);
              const int e = pt * 256 + g * 32 + ((q ^ swz) << 3) + cw;
              const float wlo = __half2float(__ushort_as_half(sc_a[e]));
              const float whi = __half2float(__ushort_as_half(sc_b[e]));
              acc[q][0] = __fmaf_rn(__fmul_rn(wlo, xa[pt][q]), (float)d[0], acc[q][0]);
              acc[q][1] = __fmaf_rn(__fmul_rn(wlo, xc[pt][q]), (float)d[1], acc[q][1]);
              acc[q][2] = __fmaf_rn(__fmul_rn(whi, xa[pt][q]), (float)d[2], acc[q][2]);
              acc[q][3] = __fmaf_rn(__fmul_rn(whi, xc[pt][q]), (float)d[3], acc[q][3]);
            }
          }
        }
        // This warp's classes c, c+16 (pair of the first level) and c+8, c+24, then the
        // second level: the tree's node over classes {c, c+8, c+16, c+24}.
        float4 u;
        u.x = __fadd_rn(__fadd_rn(acc[0][0], acc[2][0]), __fadd_rn(acc[1][0], acc[3][0]));
        u.y = __fadd_rn(__fadd_rn(acc[0][1], acc[2][1]), __fadd_rn(acc[1][1], acc[3][1]));
        u.z = __fadd_rn(__fadd_rn(acc[0][2], acc[2][2]), __fadd_rn(acc[1][2], acc[3][2]));
        u.w = __fadd_rn(__fadd_rn(acc[0][3], acc[2][3]), __fadd_rn(acc[1][3], acc[3][3]));
        *reinterpret_cast<float4*>(ubuf + ((size_t)(ub * 8 + cw) * 32 + lane) * 4) = u;
        asm volatile("bar.sync 1, %0;" ::"n"(kMmaConsumerWarps * 32) : "memory");
        if (ct < kMmaTileRows * kMmaPad) {
          // Output (row r of the tile, activation row m): D element of lane
          // 4 (r & 7) + m / 2, register 2 (r >> 3) + (m & 1).
          const int r = ct >> 3;
          const int m = ct & 7;
          const float* src = ubuf + ((size_t)(ub * 8) * 32 + (r & 7) * 4 + (m >> 1)) * 4 +
                             (r >> 3) * 2 + (m & 1);
          float v[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) v[c] = src[c * 32 * 4];
          const float u30 = __fadd_rn(v[0], v[4]);
          const float u31 = __fadd_rn(v[1], v[5]);
          const float u32 = __fadd_rn(v[2], v[6]);
          const float u33 = __fadd_rn(v[3], v[7]);
          const float tot = __fadd_rn(__fadd_rn(u30, u32), __fadd_rn(u31, u33));
          yacc = s == 0 ? tot : __fadd_rn(yacc, tot);
        }
        ub ^= 1;
      }
      // Every warp is past its last read of the tile's stages (the slice barrier).
      if (lane == 0 && live) {
        mbar_arrive(empty_bar(sa_slot));
        if (two) mbar_arrive(empty_bar(sb_slot));
      }
      if (ct < kMmaTileRows * kMmaPad && live) {
        const int r = ct >> 3;
        const int m = ct & 7;
        const int j = ja + (r >> 3);
        if (m < p.M && (r < 8 || two) && (r & 7) < stage_rows(j))
          p.y[(int64_t)m * p.N + r0 + (int64_t)j * kMmaStageRows + (r & 7)] = yacc;
      }
    }
  }
  asm volatile("bar.sync 3, %0;" ::"n"(kMmaThreads) : "memory");
  if (*abort_flag && warp == 0) {
    // A wait gave up: let the copies this CTA issued land (bounded), then mark its
    // outputs invalid.
    if (lane == 0) {
      for (int j = issued > ns ? issued - ns : 0; j < issued; ++j) {
        const long long t0 = clock64();
        while (!mbar_try_wait(full_bar(j % ns), (j / ns) & 1) && clock64() - t0 < (1ll << 30)) {
        }
      }
    }
    __syncwarp();
    const float nan = __int_as_float(0x7fc00000);
    for (int m = 0; m < p.M; ++m)
      for (int64_t i = r0 + lane; i < r1; i += 32) p.y[(int64_t)m * p.N + i] = nan;
  }
}

// ----------------------------------------------------------------------------
// Host side.
// ----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// The scale plane uint16 [N][K/32] viewed as [K/1024 parts][N rows][32 scales] (strides
// K/16 and 64 bytes): one box of 32 scales x 8 rows x cpr parts per stage, with the
// 64-byte swizzle.
bool encode_scales(CUtensorMap* map, const uint16_t* wd, int64_t N, int64_t K) {
  const auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[3] = {32, (cuuint64_t)N, (cuuint64_t)(K / 1024)};
  const cuuint64_t strides[2] = {(cuuint64_t)(K / 16), 64};
  const cuuint32_t box[3] = {32, (cuuint32_t)kMmaStageRows, (cuuint32_t)(K / 1024)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(wd), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

// The tensor-core product of M (1..8) activation rows, or MEMRA_ERR_UNSUPPORTED
// (nothing launched) when the shape or alignment does not suit it.
memra_status run_mma_product(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K, int M,
                             const int8_t* xq, const float* xd, float* y, cudaStream_t stream) {
  if (M < 1 || M > kMmaPad || K < 1024 || K % 1024 != 0 || K > 1024 * kMmaMaxParts ||
      N < kMmaTileRows)
    return MEMRA_ERR_UNSUPPORTED;
  if (N > INT32_MAX - kMmaTileRows) return MEMRA_ERR_UNSUPPORTED;
  if (!aligned(wq, 16) || !aligned(wd, 16) || !aligned(xq, 16) || !aligned(xd, 16))
    return MEMRA_ERR_UNSUPPORTED;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  MmaParams p{};
  p.wq = wq;
  p.xq = xq;
  p.xd = xd;
  p.y = y;
  p.N = N;
  p.K = (int)K;
  p.nb = (int)(K / 32);
  p.cpr = p.nb / 32;
  p.S = slices_for(p.cpr);
  if (p.S > kMmaMaxSlices) return MEMRA_ERR_UNSUPPORTED;
  p.M = M;
  p.ws = p.K + 16;
  // Stages are 512-byte aligned (the scale box's 64-byte swizzle repeats every 512
  // bytes; the quant rows need 16).
  p.scale_off = (uint32_t)align_up_sz((size_t)kMmaStageRows * p.ws, 512);
  p.stage_bytes = (uint32_t)align_up_sz(p.scale_off + (size_t)kMmaStageRows * 64 * p.cpr, 512);
  size_t off = kMmaHeader;
  p.off_ubuf = (uint32_t)off;
  off += 2 * kMmaConsumerWarps * 32 * 4 * sizeof(float);
  off = align_up_sz(off, 1024);
  p.off_ring = (uint32_t)off;
  // 1024 bytes of slack realign the dynamic shared memory inside the kernel.  A tile
  // needs two stages.
  const size_t budget = (size_t)info.max_smem_optin;
  if (off + 1024 + 2 * (size_t)p.stage_bytes > budget) return MEMRA_ERR_UNSUPPORTED;
  p.ns = (int)std::min<size_t>(kMmaMaxStages, (budget - off - 1024) / p.stage_bytes);
  const size_t smem = off + 1024 + (size_t)p.ns * p.stage_bytes;
  if (!encode_scales(&p.wd_map, wd, N, K)) return cuda_fail(cudaErrorInvalidValue);
  const int64_t grid = std::min<int64_t>(info.sms, std::max<int64_t>(1, N / kMmaTileRows));
  cudaError_t e = allow_dynamic_smem(q8_mma_kernel, smem, info);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_kernel(q8_mma_kernel, dim3((unsigned)grid), dim3(kMmaThreads), smem, stream, p);
  return e == cudaSuccess ? MEMRA_OK : cuda_fail(e);
}

}  // namespace memra
