// Block-quantised weight x q8_1 activation products: the M = 1 decode GEMV, the
// M <= 8 verify skinny GEMM (two passes up to 16 rows), the routed-expert (MoE)
// GEMVs and the routed FFN layer, on Q8_0, Q4_0 and NVFP4 weights.
//
// Arithmetic (one definition for every kernel below, so that a row's result is
// the same bit for bit whichever kernel, M, grid or batch produced it):
//   nb = K/32 blocks, cpr = ceil(nb/32) parts of 32 blocks, S = ceil(cpr/4)
//   slices; slice s covers parts [s*cpr/S, (s+1)*cpr/S).
//   Within a slice, lane l owns blocks b = 32p + l and accumulates, in ascending
//   p:  acc = fma(fl(float(d_w[b]) * d_x[b]), float(s_b), acc), from acc = 0,
//   where s_b is the exact int32 block dot (8 dp4a for Q8_0; the 4-bit formats'
//   exact forms are at their block dots below).
//   part[s] = xor-butterfly sum over the 32 lanes (masks 16, 8, 4, 2, 1).
//   y = part[0] + part[1] + ... + part[S-1], sequentially.
//
// Two kernels implement it (a third, the tensor-core verify kernel, is mma.cu).
//
// q8_tma_kernel (the GB300 path; K % 256 == 0 and 16-byte aligned planes): two
//   CTAs per SM for M = 1 (one, with a deeper ring and more registers per thread,
//   for M > 1), each owning a contiguous range of weight rows (or, for the routed
//   product, a few contiguous row ranges, one per selected expert).  Warp 0 is the
//   producer: one lane streams whole rows of the quant and scale planes into a ring
//   of shared-memory stages with cp.async.bulk, completing on per-stage mbarriers,
//   records each stage's rows in shared memory, closes the stream with a sentinel
//   stage, and reduces each finished stage's slice partials into y.  Warps 1..12
//   consume stages: each task is (R rows, one slice), dealt round-robin, and each
//   32-block part of it runs through one routine (add_part) whose shared-memory
//   loads are 128-bit at 32-bit shared-window addresses.  The HBM stream is set by
//   the ring (about 208 KB in flight per SM), not by how tasks divide among warps.
//   With programmatic dependent launch the producer starts the ring as soon as the
//   CTA is resident, before the preceding kernel has finished (dense weights do not
//   depend on it), but issues only the first two stages until its consumers, which
//   wait for that kernel, have staged the activation with plain loads: those loads
//   then wait behind a short queue of weight copies.
//
// q8_reg_kernel (Q8_0 products below about 24 MB, K % 256 != 0, unaligned planes):
//   the same tasks with weights loaded straight into registers (256-bit loads, a
//   slice's blocks issued together), activations staged in shared memory.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "product.cuh"

// Ring and stage sizes measured on GB300: two CTAs per SM, each streaming through
// about 104 KB of 34-KB stages, keep HBM busiest (bulk copies below ~16 KB stream
// markedly slower per CTA).  From 28 KB in 88 KB: 64-layer sweep 4.133 -> 4.089 ms per
// token, top-8 MoE batches of 8 / 16 tokens 3.00 -> 2.83 / 5.45 -> 4.94 ms (32 in 96
// and 36 in 108 the same; the LM head 0.6 % slower).  Each can be overridden at run
// time by the environment variable of the same name (read once per process; see
// TmaTuning).
#ifndef MEMRA_TMA_RING_KB
#define MEMRA_TMA_RING_KB 104
#endif
#ifndef MEMRA_TMA_STAGE_KB
#define MEMRA_TMA_STAGE_KB 34
#endif
// Routed experts at M = 1 for one token move a few tens of rows per CTA: smaller
// stages keep more of them in flight (top-8 MoE layer: 0.967 ms per 48-layer token
// at 28 KB, 0.926 at 24, 0.938 at 20).
#ifndef MEMRA_TMA_ROUTED_STAGE_KB
#define MEMRA_TMA_ROUTED_STAGE_KB 24
#endif
#ifndef MEMRA_TMA_CTAS_PER_SM
#define MEMRA_TMA_CTAS_PER_SM 2
#endif
#ifndef MEMRA_TMA_SMEM_LIMIT_KB
#define MEMRA_TMA_SMEM_LIMIT_KB 113
#endif
// M > 1 products: one CTA per SM (the consumers need more registers) with a deeper
// ring of larger stages (measured on GB300: 200 KB of 44 KB stages).
#ifndef MEMRA_TMA_MULTI_RING_KB
#define MEMRA_TMA_MULTI_RING_KB 200
#endif
#ifndef MEMRA_TMA_MULTI_STAGE_KB
#define MEMRA_TMA_MULTI_STAGE_KB 44
#endif
// Dense products below this many MB of weights use the register kernel.
#ifndef MEMRA_TMA_DENSE_MIN_MB
#define MEMRA_TMA_DENSE_MIN_MB 24
#endif
#ifndef MEMRA_TMA_MIN_BLOCKS
#define MEMRA_TMA_MIN_BLOCKS 2
#endif
// Dense products: stages a CTA issues before its consumers have staged the activation
// (0: no limit).  The activation's loads, issued after the grid-dependency wait, queue
// behind the weight copies already in flight to the SM; with two stages per CTA
// instead of the whole ring they return sooner, and the dependent chain of products
// and quantise launches moves faster (64-layer sweep: 4.28 -> 4.12 ms per token; one
// stage: 4.33 ms).
#ifndef MEMRA_TMA_PREFILL
#define MEMRA_TMA_PREFILL 2
#endif
#ifndef MEMRA_TMA_ROUTED_PREFILL
#define MEMRA_TMA_ROUTED_PREFILL 1
#endif
// Dense M = 1 products on 4-bit weights, whose consumers take longer per byte than
// Q8_0's, issue one stage before the activation is staged (64-layer sweeps with 34 KB
// stages in 104 KB: Q4_0 3.00 -> 2.92 ms per token, NVFP4 3.46 -> 3.35; Q8_0 is best
// with two).
#ifndef MEMRA_TMA_PREFILL_4BIT
#define MEMRA_TMA_PREFILL_4BIT 1
#endif

namespace memra {
namespace {

// Routed slots one launch holds in shared memory: a batch's tokens x top_k.
constexpr int kMaxTopK = MEMRA_MAX_PAIRS;
static_assert(MEMRA_MAX_TOP_K <= MEMRA_MAX_PAIRS, "a single token's slots fit");

enum Mode { kDense = 0, kMoeUngated = 1, kMoeGated = 2 };

// Weight formats: Q8_0 (32 int8 quants a block, K bytes a row), Q4_0 (32 4-bit
// codes a block, K/2 bytes a row; byte j of a block holds elements j and j+16), and
// NVFP4 (E2M1 codes, K/2 bytes a row, byte j holding elements 2j and 2j+1; an E4M3
// scale per 16 elements, so a 32-block's two scales fill the 2-byte scale slot).
enum Fmt { kQ8 = 0, kQ4 = 1, kNv4 = 2 };

// dp4a with unsigned bytes in a and signed bytes in b (the Q4_0 codes against q8_1
// activations): exact int32.
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// NVFP4: the exact sum over 16 elements of (twice the E2M1 value of the code) times
// the int8 activation.  Codes c0 (elements 0..7) and c1 (8..15), one nibble each in
// element order; x: the 16 activation bytes.  prmt looks up each nibble of its
// 16-bit selector in the 8 bytes {kLo, kHi} (twice the magnitudes 0, .5, 1, 1.5, 2,
// 3, 4, 6); a nibble with bit 3 set (a negative code) takes the sign-replicated
// byte instead, 0 for these bytes.  So the lookup of the codes gives the magnitudes
// of the positive codes, that of the codes with every sign flipped the magnitudes of
// the negative ones, and the sum is the difference of their two dp4a sums.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// The lookup bytes: kNv4Lo | kNv4Hi.  The kernels read them from shared memory into
// registers once, so that the compiler keeps them there rather than rebuilding the
// two constants for every lookup.
constexpr uint32_t kNv4Lo = 0x03020100u, kNv4Hi = 0x0C080604u;

__device__ __forceinline__ int nv4_dot16(uint32_t c0, uint32_t c1, const uint4& x, uint32_t kLo,
                                         uint32_t kHi) {
  const uint32_t n0 = c0 ^ 0x88888888u;
  const uint32_t n1 = c1 ^ 0x88888888u;
  int p = __dp4a((int)prmt(kLo, kHi, c0), (int)x.x, 0);
  int q = __dp4a((int)prmt(kLo, kHi, n0), (int)x.x, 0);
  p = __dp4a((int)prmt(kLo, kHi, c0 >> 16), (int)x.y, p);
  q = __dp4a((int)prmt(kLo, kHi, n0 >> 16), (int)x.y, q);
  p = __dp4a((int)prmt(kLo, kHi, c1), (int)x.z, p);
  q = __dp4a((int)prmt(kLo, kHi, n1), (int)x.z, q);
  p = __dp4a((int)prmt(kLo, kHi, c1 >> 16), (int)x.w, p);
  q = __dp4a((int)prmt(kLo, kHi, n1 >> 16), (int)x.w, q);
  return p - q;
}

// The two E4M3 scales of a 32-element block (low byte: elements 0..15), exactly.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t bits) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(bits));
  return make_float2(__half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half((uint16_t)(h2 >> 16))));
}

// ----------------------------------------------------------------------------
// Work description shared by both kernels: a CTA's rows come as segments, each a
// contiguous run of weight rows multiplied by one activation row set.
// ----------------------------------------------------------------------------
struct Params {
  const int8_t* wq;        // dense weights or the expert bank
  const uint16_t* wd;
  int64_t N;               // rows of one weight matrix
  int64_t K;
  int64_t qrow;            // bytes of one row of the quant plane (K, or K/2 for Q4_0)
  int nb, cpr, S;
  const int8_t* xq;
  const float* xd;
  const void* xin;         // unquantised activation (fused-quantisation entry point)
  int xrows;               // activation rows held in shared memory
  float* y;
  int64_t units;           // dense/gated: N; ungated: top_k * N
  // routed experts
  const int32_t* ids;
  const float* gate_w;
  int top_k;
  int64_t E;
  int xpe;                 // one activation row per expert (per routed slot)
  // Routed slots that share one activation row (xpe): slot k reads row k / xdiv.  A
  // batch of tokens routes top_k slots each and shares each token's row among them.
  int xdiv;
  // NVFP4: half the tensor scale (the block sums use twice the E2M1 values); routed
  // products take each expert's tensor scale from gexp[id] (fp32 [E], device).
  float gscale;
  const float* gexp;
  // Slots of a batched routed product (> 0): the grid gives every slot the same
  // number of CTAs at the same row offsets, so that slots routed to the same expert
  // stream its rows at the same time and the repeats are served from L2.
  int lockstep;
  int32_t* status;
  // The routing was already waited for by the preceding kernel of the same call, and
  // that kernel let this one launch only after its own wait: read it at once.
  int routing_ready;
  // Gated routed product whose CTA takes all of its top_k segments (rps rows each at
  // most) in one packed stage: segment k's rows at stage rows [k*n, (k+1)*n).
  int packed;
  // Ungated routed product over gate|up pairs (the routed FFN's first launch): each
  // expert has 2N rows, gate rows 0..N-1 and up rows N..2N-1, and unit (k, j) is the pair
  // (gate j, up j) of slot k.  A stage holds n gate rows, then the same n up rows; the
  // epilogue writes y[k][j] = silu(g) u and y[k][N + j] = u (y: [slots][2N]).
  int pairs;
  // Bounded waits give up after wait_limit SM cycles.  stall_after >= 0 (test hook):
  // each CTA's producer stops after that many stages and leaves one more stage that
  // nothing completes, so that the waits run out and the abort path runs.
  long long wait_limit;
  int stall_after;
  // Dense products: stages a CTA's producer issues before its consumers have staged the
  // activation (0: no limit).  A short queue of weight copies in flight lets the
  // activation's loads, issued after the grid-dependency wait, return sooner.
  int prefill_stages;
  // TMA kernel layout
  int rps;                 // rows per stage
  int ns;                  // stages in the ring
  uint32_t stage_bytes;    // bytes per stage (quants, then scales at wd_off)
  uint32_t wd_off;
  uint32_t off_x, off_xd, off_ring, off_part, off_yacc, off_slice;
  uint32_t off_xsum;       // Q4_0: int32 per-block sums of the activation quants
  // register kernel layout
  int tile_rows;
};

// Unquantised activation row `row` (K values; SwiGLU input rows hold gate|up, 2K).
template <int XIN>
__device__ __forceinline__ const void* xin_row(const void* xin, int64_t row, int64_t K) {
  if (XIN == kXbf16) return static_cast<const uint16_t*>(xin) + row * K;
  if (XIN == kXf32) return static_cast<const float*>(xin) + row * K;
  return static_cast<const float*>(xin) + row * 2 * K;  // kXswiglu, kXhalf: rows of 2K
}

// The unit range [u0, u1) of CTA b of G: units * b / G with 32-bit arithmetic when the
// products fit (every workload here), else 64-bit.
__device__ __forceinline__ int64_t cta_unit(int64_t units, unsigned b, unsigned G) {
  if (units <= (int64_t)(0xffffffffu / G)) return (int64_t)((uint32_t)units * b / G);
  return units * b / G;
}

struct Seg {
  int64_t row0;   // first weight row (absolute row index into the plane)
  int nrows;
  int xrow;       // first activation row used
  int k;          // routed slot (0 for dense)
  int64_t out0;   // first output row (dense/ungated)
  bool valid;
};

// The slot of a CTA's first unit (ungated routed products; 0 otherwise): the one
// 64-bit division a CTA needs, taken once.
template <int MODE>
__device__ __forceinline__ int64_t first_slot(const Params& p, int64_t u0) {
  return MODE == kMoeUngated ? u0 / p.N : 0;
}

template <int MODE>
__device__ __forceinline__ int num_segs(const Params& p, int64_t u0, int64_t u1, int64_t k0) {
  if (MODE == kDense) return 1;
  if (MODE == kMoeGated) return p.top_k;
  // slots k0 .. k with k N <= u1 - 1 < (k + 1) N
  int64_t k = k0;
  while ((k + 1) * p.N <= u1 - 1) ++k;
  return (int)(k - k0 + 1);
}

template <int MODE>
__device__ __forceinline__ Seg get_seg(const Params& p, int64_t u0, int64_t u1, int si,
                                       const int32_t* s_ids, int64_t k0) {
  Seg g;
  if (MODE == kDense) {
    g.row0 = u0;
    g.nrows = (int)(u1 - u0);
    g.xrow = 0;
    g.k = 0;
    g.out0 = u0;
    g.valid = true;
  } else if (MODE == kMoeGated) {
    const int e = s_ids[si];
    g.k = si;
    g.valid = e >= 0;
    g.row0 = (int64_t)(e < 0 ? 0 : e) * p.N + u0;
    g.nrows = (int)(u1 - u0);
    g.xrow = p.xpe ? si : 0;
    g.out0 = u0;
  } else {
    const int64_t k = k0 + si;
    const int64_t lo = (u0 > k * p.N ? u0 : k * p.N) - k * p.N;
    const int64_t hi = (u1 < (k + 1) * p.N ? u1 : (k + 1) * p.N) - k * p.N;
    const int e = s_ids[k];
    const int64_t er = p.pairs ? 2 * p.N : p.N;  // weight rows (and outputs) per slot
    g.k = (int)k;
    g.valid = e >= 0;
    g.row0 = (int64_t)(e < 0 ? 0 : e) * er + lo;
    g.nrows = (int)(hi - lo);
    g.xrow = p.xpe ? (int)(p.xdiv > 1 ? k / p.xdiv : k) : 0;
    g.out0 = k * er + lo;
  }
  return g;
}

// Load ids (validated) and gate weights into shared memory; flag bad ids.
template <int MODE>
__device__ __forceinline__ void load_routing(const Params& p, int32_t* s_ids, float* s_gate,
                                             int tid, int nthreads) {
  for (int k = tid; k < p.top_k; k += nthreads) {
    const int32_t e = __ldcg(p.ids + k);
    const bool ok = e >= 0 && e < p.E;
    s_ids[k] = ok ? e : -1;
    s_gate[k] = (MODE == kMoeGated) ? __ldcg(p.gate_w + k) : 1.0f;
    if (!ok && p.status && blockIdx.x == 0) atomicOr(p.status, 1);
  }
}

// ============================================================================
// TMA producer/consumer kernel.
// ============================================================================
#ifndef MEMRA_TMA_CONSUMER_WARPS
#define MEMRA_TMA_CONSUMER_WARPS 12
#endif
// M > 1 products run one CTA per SM, where dp4a issue rather than the stream limits
// them.  With M <= 3 a task holds few accumulators and more consumer warps help
// (measured: M = 2 at 20 warps 4.72 ms per sweep token, at 12 warps 5.01 ms); from
// M = 4 on, more warps only shrink the register budget (M = 8 spills from 16 warps).
#ifndef MEMRA_TMA_FEW_M_CONSUMER_WARPS
#define MEMRA_TMA_FEW_M_CONSUMER_WARPS 20
#endif
__host__ __device__ constexpr int tma_consumer_warps(int M) {
  return M == 1 || M > 3 ? MEMRA_TMA_CONSUMER_WARPS : MEMRA_TMA_FEW_M_CONSUMER_WARPS;
}
__host__ __device__ constexpr int tma_threads(int M) { return 32 * (1 + tma_consumer_warps(M)); }
constexpr int kMaxStages = 16;
// Shared-memory header: full[kMaxStages] | empty[kMaxStages] mbarriers, the abort
// flag, the stage metadata, the routed ids and gate weights.
constexpr int kOffAbort = 8 * 2 * kMaxStages;
constexpr int kOffXready = kOffAbort + 8;  // mbarrier: the consumers staged the activation
constexpr int kOffMeta = kOffAbort + 16;
constexpr int kOffIds = kOffMeta + 16 * kMaxStages;
constexpr int kOffGate = kOffIds + 4 * kMaxTopK;
constexpr int kOffGsc = kOffGate + 4 * kMaxTopK;  // NVFP4 routed: half each slot's g
constexpr int kOffTab = kOffGsc + 4 * kMaxTopK;  // NVFP4: the lookup bytes
constexpr int kHeaderBytes = (kOffTab + 8 + 127) / 128 * 128;

// What the producer put in a ring slot: rows [r0, r0 + nr) of segment `seg`, with
// activation row `xrow`.  nr == 0 marks the end of the CTA's stages.  A packed stage
// (seg < 0) holds every routed segment of the CTA, xrow rows each, segment after
// segment.
struct StageMeta {
  int seg;
  int r0;
  int nr;
  int xrow;
};

// Add one 32-block part of R weight rows against M activation rows to acc: this lane's
// block q parts past wl[r] (quants) and dl[r] (scales), and past xl / xdl / xsl (the
// activation row's quants, scales and Q4_0 block sums; further rows Ki bytes and nb
// blocks on).  All are 32-bit shared-window addresses, so that each part's offsets are
// immediates of its loads.  h1: which 16-byte half of a Q8_0 block this lane loads first; xh: the
// same for the activation (0 for NVFP4, which reads both halves in element order).
// Format constants: Q4_0 nibble masks q4m0 / q4m1 and shift q4s0 of this lane; NVFP4
// lookup bytes tlo | thi.
struct PartConsts {
  uint32_t q4m0, q4m1;
  int q4s0;
  uint32_t tlo, thi;
};

template <int M, int R, int FMT>
__device__ __forceinline__ void add_part(float (&acc)[R][M], const uint32_t (&wl)[R],
                                         const uint32_t (&dl)[R], uint32_t xl, uint32_t xdl,
                                         uint32_t xsl, int q, int Ki, int nb, int h1, int xh,
                                         const PartConsts& pc) {
  constexpr int kBlockBytes = FMT == kQ8 ? 32 : 16;
  constexpr int kPartBytes = 32 * kBlockBytes;
  uint4 w0[R], w1[R];
  uint16_t dw[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    // Q8_0: the two halves in this lane quad's order (see the file comment).
    // Q4_0 and NVFP4: the block's 16 bytes of codes in one load.
    w0[r] = lds_v4(wl[r] + q * kPartBytes);
    if (FMT == kQ8) w1[r] = lds_v4(wl[r] + q * kPartBytes + 16 - 32 * h1);
    dw[r] = lds_u16(dl[r] + q * 64);
  }
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const uint32_t xm = xl + m * Ki + q * 1024;
    const uint4 x0 = lds_v4(xm);
    const uint4 x1 = lds_v4(xm + 16 - 32 * xh);
    const float dx = lds_f32(xdl + (m * nb + q * 32) * 4);
    if (FMT == kQ4) {
      // x0 holds half h1 of the block (elements 16*h1 ..), x1 the other half.  The
      // lane pairs x0 with the nibbles of half h1 (mask m0) and x1 with the other
      // nibbles (m1).  A high-nibble mask leaves 16 times the codes in place, which
      // makes that dp4a exactly 16 times the half's dot (a multiple of 16 below 2^19),
      // undone by the shift.
      const uint32_t q4m0 = pc.q4m0, q4m1 = pc.q4m1;
      const int q4s0 = pc.q4s0;
      const int sx = lds_s32(xsl + (m * nb + q * 32) * 4);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint4 c = w0[r];
        int a = dp4a_us(c.x & q4m0, (int)x0.x, 0);
        a = dp4a_us(c.y & q4m0, (int)x0.y, a);
        a = dp4a_us(c.z & q4m0, (int)x0.z, a);
        a = dp4a_us(c.w & q4m0, (int)x0.w, a);
        int b = dp4a_us(c.x & q4m1, (int)x1.x, 0);
        b = dp4a_us(c.y & q4m1, (int)x1.y, b);
        b = dp4a_us(c.z & q4m1, (int)x1.z, b);
        b = dp4a_us(c.w & q4m1, (int)x1.w, b);
        const int dot = (a >> q4s0) + (b >> (4 - q4s0));
        acc[r][m] = block_term_acc(acc[r][m], dw[r], dx, dot - 8 * sx);
      }
    } else if (FMT == kNv4) {
      // Code bytes 0..7 are the block's elements 0..15 (first E4M3 scale), bytes 8..15
      // elements 16..31; x0 and x1 hold the same halves (xh = 0).  Each half's exact
      // sum, then the two terms in element order.
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint4 c = w0[r];
        const int sa = nv4_dot16(c.x, c.y, x0, pc.tlo, pc.thi);  // elements 0..15
        const int sb = nv4_dot16(c.z, c.w, x1, pc.tlo, pc.thi);  // elements 16..31
        const float2 sc = e4m3x2_to_float2(dw[r]);
        acc[r][m] = __fmaf_rn(__fmul_rn(sc.x, dx), (float)sa, acc[r][m]);
        acc[r][m] = __fmaf_rn(__fmul_rn(sc.y, dx), (float)sb, acc[r][m]);
      }
    } else {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int sb = dot_halves(w0[r], w1[r], x0, x1);
        acc[r][m] = block_term_acc(acc[r][m], dw[r], dx, sb);
      }
    }
  }
}

template <int M, int R, int MODE, int XIN, int FMT = kQ8>
__global__ void __launch_bounds__(tma_threads(M), M == 1 ? MEMRA_TMA_MIN_BLOCKS : 1)
    q8_tma_kernel(const Params p) {
  constexpr int kConsumerWarps = tma_consumer_warps(M);
  constexpr int kTmaThreads = tma_threads(M);
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[8] | empty[8]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  StageMeta* meta = reinterpret_cast<StageMeta*>(smem + kOffMeta);
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem + kOffIds);
  float* s_gate = reinterpret_cast<float*>(smem + kOffGate);
  float* s_gsc = reinterpret_cast<float*>(smem + kOffGsc);
  int8_t* xs = reinterpret_cast<int8_t*>(smem + p.off_x);
  float* xds = reinterpret_cast<float*>(smem + p.off_xd);
  unsigned char* ring = smem + p.off_ring;
  float* part = reinterpret_cast<float*>(smem + p.off_part);
  float* yacc = reinterpret_cast<float*>(smem + p.off_yacc);
  int* s_slice = reinterpret_cast<int*>(smem + p.off_slice);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nb = p.nb;
  const int S = p.S;
  const int ns = p.ns;
  const int64_t u0 = cta_unit(p.units, blockIdx.x, gridDim.x);
  const int64_t u1 = cta_unit(p.units, blockIdx.x + 1, gridDim.x);
  // Activation rows this CTA stages: [xlo, xlo + nxr).  An ungated routed product
  // with an activation row per slot group stages only the rows of its own segments.
  const int64_t k0 = first_slot<MODE>(p, u0);
  const int nseg = num_segs<MODE>(p, u0, u1, k0);
  int xlo = 0, nxr = p.xrows;
  if (MODE == kMoeUngated && p.xpe) {
    const int d = p.xdiv > 1 ? p.xdiv : 1;
    xlo = (int)k0 / d;
    nxr = (int)(k0 + nseg - 1) / d - xlo + 1;
  }
  auto full_bar = [&](int i) { return smem_addr(bars + i); };
  auto empty_bar = [&](int i) { return smem_addr(bars + kMaxStages + i); };
  const uint32_t xready_bar = smem_addr(smem + kOffXready);

  if (MODE == kDense) pdl_launch_dependents();
  // Start-up.  The producer warp initialises the barriers (and, for routed
  // products, loads the routing), signals the consumers with a non-blocking arrive
  // on named barrier 2 and starts streaming at once; the consumers build the slice
  // table and wait there before touching any barrier.
  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < ns; ++i) {
        mbar_init(full_bar(i), 1);
        mbar_init(empty_bar(i), kConsumerWarps);
      }
      mbar_init(xready_bar, 1);
      *abort_flag = 0;
      if (FMT == kNv4) {
        reinterpret_cast<uint32_t*>(smem + kOffTab)[0] = kNv4Lo;
        reinterpret_cast<uint32_t*>(smem + kOffTab)[1] = kNv4Hi;
      }
      mbar_init_fence();
    }
    if (MODE != kDense) {
      // ids and gate weights may come from the preceding kernel (L2 reads: never a
      // stale L1 line).
      if (!p.routing_ready) pdl_wait();
      load_routing<MODE>(p, s_ids, s_gate, lane, 32);
      if (FMT == kNv4)  // the same lane wrote s_ids[k] just above
        for (int k = lane; k < p.top_k; k += 32)
          s_gsc[k] = s_ids[k] >= 0 ? __fmul_rn(0.5f, __ldcg(p.gexp + s_ids[k])) : 0.0f;
    }
    if (MODE == kMoeGated) {
      for (int64_t i = lane; i < u1 - u0; i += 32) yacc[i] = 0.0f;
    }
    __syncwarp();
    asm volatile("bar.arrive 2, %0;" ::"n"(kTmaThreads) : "memory");
  } else {
    fill_slice_table(s_slice, p.cpr, S, threadIdx.x - 32, kTmaThreads - 32);
    asm volatile("bar.sync 2, %0;" ::"n"(kTmaThreads) : "memory");
  }
  // A routed product lets the next kernel launch only once its routing has been
  // read after the wait for its own predecessor, so that a following kernel of the
  // same call (routing_ready) can read the same routing before it waits.
  if (MODE != kDense) pdl_launch_dependents();

  auto seg_of = [&](int si) { return get_seg<MODE>(p, u0, u1, si, s_ids, k0); };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_evict_first_policy();
    uint32_t issued = 0;  // ring slots filled, the closing sentinel included
    bool ok = true;

    // Stage source: the CTA's own segments in order, rps rows at a time.
    int cur_si = 0, cur_r0 = 0;
    auto static_next = [&](StageMeta& m) -> bool {
      while (cur_si < nseg) {
        const Seg g = get_seg<MODE>(p, u0, u1, cur_si, s_ids, k0);
        if (!g.valid || cur_r0 >= g.nrows) {
          if (!g.valid && MODE == kMoeUngated)
            for (int i = lane; i < g.nrows; i += 32) {
              p.y[g.out0 + i] = 0.0f;
              if (p.pairs) p.y[g.out0 + p.N + i] = 0.0f;
            }
          ++cur_si;
          cur_r0 = 0;
          continue;
        }
        // A pairs stage takes rps / 2 pairs: rps rows.
        const int step = MODE == kMoeUngated && p.pairs ? p.rps / 2 : p.rps;
        m.seg = cur_si;
        m.r0 = cur_r0;
        m.nr = min(step, g.nrows - cur_r0) * (MODE == kMoeUngated && p.pairs ? 2 : 1);
        m.xrow = g.xrow - xlo;
        cur_r0 += step;
        return true;
      }
      return false;
    };

    // Reduce the slice partials of the stage in `slot` into the outputs.
    auto epilogue = [&](int slot) {
      const StageMeta mt = meta[slot];
      const float* pp = part + (size_t)slot * p.rps * S * M;
      if (MODE == kMoeGated && mt.seg < 0) {
        // Packed stage: each output accumulates its segments in ascending k.
        const int n = mt.xrow;
        for (int i = lane; i < n; i += 32) {
          float acc = yacc[i];
          for (int k = 0; k < p.top_k; ++k) {
            if (s_ids[k] < 0) continue;
            const float* q = pp + (size_t)(k * n + i) * S;
            float tot = q[0];
            for (int s = 1; s < S; ++s) tot = __fadd_rn(tot, q[s]);
            if (FMT == kNv4) tot = __fmul_rn(s_gsc[k], tot);
            acc = __fadd_rn(acc, __fmul_rn(s_gate[k], tot));
          }
          yacc[i] = acc;
        }
        __syncwarp();
        return;
      }
      const Seg g = seg_of(mt.seg);
      if (MODE == kMoeUngated && p.pairs) {
        // Rows [0, n) are gate rows j, rows [n, 2n) the same up rows (M == 1).
        const int n = mt.nr / 2;
        for (int i = lane; i < n; i += 32) {
          float tg = pp[(size_t)i * S];
          float tu = pp[(size_t)(n + i) * S];
          for (int s = 1; s < S; ++s) {
            tg = __fadd_rn(tg, pp[(size_t)i * S + s]);
            tu = __fadd_rn(tu, pp[(size_t)(n + i) * S + s]);
          }
          if (FMT == kNv4) {
            tg = __fmul_rn(s_gsc[g.k], tg);
            tu = __fmul_rn(s_gsc[g.k], tu);
          }
          p.y[g.out0 + mt.r0 + i] = swiglu1(tg, tu);
          p.y[g.out0 + p.N + mt.r0 + i] = tu;
        }
        __syncwarp();
        return;
      }
      for (int i = lane; i < mt.nr * M; i += 32) {
        const int r = i / M;
        const int m = i - r * M;
        float tot = pp[((size_t)r * S) * M + m];
        for (int s = 1; s < S; ++s) tot = __fadd_rn(tot, pp[((size_t)r * S + s) * M + m]);
        if (FMT == kNv4) tot = __fmul_rn(MODE == kDense ? p.gscale : s_gsc[g.k], tot);
        if (MODE == kMoeGated) {
          const int n = mt.r0 + r;
          yacc[n] = __fadd_rn(yacc[n], __fmul_rn(s_gate[g.k], tot));
        } else {
          p.y[(int64_t)m * p.units + g.out0 + mt.r0 + r] = tot;
        }
      }
      __syncwarp();
    };

    // Make ring slot issued % ns free: wait until its previous stage is consumed
    // and reduce it.
    bool acquired = false;
    auto acquire = [&]() -> bool {
      if (acquired) return true;
      const int slot = issued % ns;
      if (issued >= (uint32_t)ns) {
        if (!mbar_wait(empty_bar(slot), ((issued / ns) - 1) & 1, abort_flag, p.wait_limit))
          return false;
        epilogue(slot);
      }
      acquired = true;
      return true;
    };
    // Fill the acquired slot with stage `m`, or with the closing sentinel.
    auto fill = [&](const StageMeta* m) {
      const int slot = issued % ns;
      if (lane == 0) {
        if (m) {
          meta[slot] = *m;
          const Seg g = seg_of(m->seg);
          const uint32_t qb = (uint32_t)(m->nr * p.qrow);
          const uint32_t db = (uint32_t)(m->nr * nb * 2);
          const uint32_t dst = smem_addr(ring + (size_t)slot * p.stage_bytes);
          mbar_arrive_expect_tx(full_bar(slot), qb + db);
          if (MODE == kMoeUngated && p.pairs) {
            // n gate rows, then the n up rows N further on.
            const int n = m->nr / 2;
            const int64_t gr = g.row0 + m->r0;
            const int64_t ur = gr + p.N;
            bulk_g2s_hint(dst, p.wq + gr * p.qrow, qb / 2, full_bar(slot), policy);
            bulk_g2s_hint(dst + (uint32_t)(n * p.qrow), p.wq + ur * p.qrow, qb / 2, full_bar(slot),
                          policy);
            bulk_g2s_hint(dst + p.wd_off, p.wd + gr * nb, db / 2, full_bar(slot), policy);
            bulk_g2s_hint(dst + p.wd_off + (uint32_t)(n * nb * 2), p.wd + ur * nb, db / 2,
                          full_bar(slot), policy);
          } else {
            bulk_g2s_hint(dst, p.wq + (g.row0 + m->r0) * p.qrow, qb, full_bar(slot), policy);
            bulk_g2s_hint(dst + p.wd_off, p.wd + (g.row0 + m->r0) * nb, db, full_bar(slot),
                          policy);
          }
        } else {
          meta[slot] = StageMeta{0, 0, 0, 0};  // sentinel: no more stages
          mbar_arrive(full_bar(slot));
        }
      }
      __syncwarp();
      ++issued;
      acquired = false;
    };

    if (MODE == kMoeGated && p.packed) {
      // One stage with every valid segment's rows, completing on one barrier: a
      // stage costs its round trip through the consumers and the epilogue whatever
      // its size, and the CTA's segments are only a few rows each.
      const int n = (int)(u1 - u0);
      if (acquire()) {
        const int slot = issued % ns;
        if (lane == 0) {
          meta[slot] = StageMeta{-1, 0, p.top_k * n, n};
          uint32_t bytes = 0;
          for (int k = 0; k < p.top_k; ++k)
            if (s_ids[k] >= 0) bytes += (uint32_t)(n * (p.qrow + nb * 2));
          const uint32_t dst = smem_addr(ring + (size_t)slot * p.stage_bytes);
          // With no valid segment (bytes == 0) this arrival alone completes the stage.
          mbar_arrive_expect_tx(full_bar(slot), bytes);
          for (int k = 0; k < p.top_k; ++k) {
            if (s_ids[k] < 0) continue;
            const int64_t row0 = (int64_t)s_ids[k] * p.N + u0;
            bulk_g2s_hint(dst + (uint32_t)(k * n) * (uint32_t)p.qrow, p.wq + row0 * p.qrow,
                          (uint32_t)(n * p.qrow), full_bar(slot), policy);
            bulk_g2s_hint(dst + p.wd_off + (uint32_t)(k * n * nb * 2), p.wd + row0 * nb,
                          (uint32_t)(n * nb * 2), full_bar(slot), policy);
          }
        }
        __syncwarp();
        ++issued;
        acquired = false;
      } else {
        ok = false;
      }
    }
    bool stalled = false;
    for (;;) {
      StageMeta m;
      if ((MODE == kMoeGated && p.packed) || !static_next(m)) break;
      if (!acquire()) {
        ok = false;
        break;
      }
      if (p.prefill_stages > 0 && issued == (uint32_t)p.prefill_stages) {
        bool ready = true;
        if (lane == 0) ready = mbar_wait(xready_bar, 0, abort_flag, p.wait_limit);
        if (!__shfl_sync(kFullMask, ready ? 1 : 0, 0)) {
          ok = false;
          break;
        }
      }
      if (p.stall_after >= 0 && issued == (uint32_t)p.stall_after) {
        // Test hook: a stage that no copy and no arrival will ever complete.
        ++issued;
        acquired = false;
        stalled = true;
        break;
      }
      fill(&m);
    }
    if (ok && !stalled) {
      if (acquire()) {
        fill(nullptr);
      } else {
        ok = false;
      }
    }
    // Drain: the partials of the stages still in the ring (after a normal end the
    // last slot filled holds the sentinel).
    const uint32_t first = issued > (uint32_t)ns ? issued - ns : 0;
    const uint32_t last = ok && !stalled ? issued - 1 : issued;
    for (uint32_t j = first; j < last && ok; ++j) {
      const int slot = j % ns;
      if (!mbar_wait(empty_bar(slot), (j / ns) & 1, abort_flag, p.wait_limit)) {
        ok = false;
        break;
      }
      epilogue(slot);
    }
    if (!ok || *abort_flag) {
      // A wait gave up: let the copies already issued land (bounded), then mark the
      // outputs this CTA owns invalid with NaN (after the preceding kernel, which
      // may still read them).
      *abort_flag = 1;
      pdl_wait();
      for (uint32_t j = first; j < issued; ++j) {
        const int slot = j % ns;
        const long long t0 = clock64();
        while (!mbar_try_wait(full_bar(slot), (j / ns) & 1) && clock64() - t0 < p.wait_limit) {
        }
      }
      if (p.status && lane == 0) atomicOr(p.status, 2);
      const float nan = __int_as_float(0x7fc00000);
      if (MODE == kMoeGated) {
        for (int64_t i = lane; i < u1 - u0; i += 32) p.y[u0 + i] = nan;
      } else if (MODE == kMoeUngated && p.pairs) {
        for (int64_t i = u0 + lane; i < u1; i += 32) {
          const int64_t k = i / p.N;
          p.y[i + k * p.N] = nan;          // k * 2N + j
          p.y[i + k * p.N + p.N] = nan;
        }
      } else if (MODE == kMoeUngated) {
        for (int64_t i = u0 + lane; i < u1; i += 32) p.y[i] = nan;
      } else {
        for (int m = 0; m < M; ++m)
          for (int64_t i = u0 + lane; i < u1; i += 32) p.y[m * p.units + i] = nan;
      }
    } else if (MODE == kMoeGated) {
      for (int64_t i = lane; i < u1 - u0; i += 32) p.y[u0 + i] = yacc[i];
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int cw = warp - 1;
    const int h1 = (lane >> 2) & 1;  // which half this lane loads first
    const int Ki = (int)p.K;
    const bool last_ok = lane < nb - (p.cpr - 1) * 32;
    // The activation comes from the preceding kernel.  The consumers stage it with
    // plain loads: a bulk copy would queue behind the weight stages already issued
    // and land only after all of them.
    pdl_wait();
    if (XIN == kXq8) {
      copy_x_to_smem<4>(p.xq + (size_t)xlo * Ki, p.xd + (size_t)xlo * nb, nxr * Ki, nxr * nb * 4,
                        xs, xds, threadIdx.x - 32, kConsumerWarps * 32);
    } else {
      quantize_rows_to_smem<XIN>(xin_row<XIN>(p.xin, xlo, p.K), nxr, (int)p.K, xs, xds, cw,
                                 kConsumerWarps, lane);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    if (threadIdx.x == 32) mbar_arrive(xready_bar);
    // Q4_0: s_b = sum_i (c_i - 8) x_i = (sum_i c_i x_i) - 8 sum_i x_i, with the
    // activation's per-block sums taken once here.
    int32_t* xsum = reinterpret_cast<int32_t*>(smem + p.off_xsum);
    if (FMT == kQ4) {
      for (int i = threadIdx.x - 32; i < nxr * nb; i += kConsumerWarps * 32) {
        const uint4 a = *reinterpret_cast<const uint4*>(xs + (size_t)i * 32);
        const uint4 b = *reinterpret_cast<const uint4*>(xs + (size_t)i * 32 + 16);
        const int ones = 0x01010101;
        int t = __dp4a(ones, (int)a.x, 0);
        t = __dp4a(ones, (int)a.y, t);
        t = __dp4a(ones, (int)a.z, t);
        t = __dp4a(ones, (int)a.w, t);
        t = __dp4a(ones, (int)b.x, t);
        t = __dp4a(ones, (int)b.y, t);
        t = __dp4a(ones, (int)b.z, t);
        xsum[i] = __dp4a(ones, (int)b.w, t);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    }
    // Bytes of one block in the ring's quant rows.
    constexpr int kBlockBytes = FMT == kQ8 ? 32 : 16;
    const int Qrow = (int)p.qrow;
    // Q4_0 nibble masks and shift of this lane (see add_part); the NVFP4 lookup bytes.
    PartConsts pc;
    pc.q4m0 = h1 ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
    pc.q4m1 = ~pc.q4m0;
    pc.q4s0 = h1 ? 4 : 0;
    pc.tlo = FMT == kNv4 ? reinterpret_cast<const uint32_t*>(smem + kOffTab)[0] : 0u;
    pc.thi = FMT == kNv4 ? reinterpret_cast<const uint32_t*>(smem + kOffTab)[1] : 0u;
    // NVFP4 reads the activation halves in element order (xh = 0): it is issue-bound,
    // and the half order's selects cost more there than a 2-way bank conflict.
    const int xh = FMT == kNv4 ? 0 : h1;
    const uint32_t ring_a = smem_addr(ring);
    const uint32_t xs_a = smem_addr(xs);
    const uint32_t xds_a = smem_addr(xds);
    const uint32_t xsum_a = smem_addr(xsum);
    uint32_t tbase = 0;  // tasks in all earlier stages: deals tasks round-robin over warps
    // A warp's tasks are kConsumerWarps apart: in (group, slice) form a step of
    // (dgi, dsl) with a carry, so no task needs a division.
    const int dgi = kConsumerWarps / S;
    const int dsl = kConsumerWarps - dgi * S;
    // t0 / S for a warp's first task in a stage (t0 < kConsumerWarps) as a multiply-high
    // by ceil(2^32 / S), exact for t0 < 2^17 and S <= 256.
    const uint32_t sinv = S > 1 ? (uint32_t)((0x100000000ull + S - 1) / S) : 0u;
    int slot = 0;
    uint32_t phase = 0;
    for (;;) {
      // Every warp waits for every stage, tasks or not: an arrival on the stage's
      // empty barrier must never run ahead of the stage itself.
      if (!mbar_wait(full_bar(slot), phase, abort_flag, p.wait_limit)) return;
      const StageMeta mt = meta[slot];
      if (mt.nr <= 0) break;
      const int nr = mt.nr;
      const bool packed_stage = MODE == kMoeGated && mt.seg < 0;  // R == 1 there
      const int groups = (nr + R - 1) / R;
      const int ntasks = groups * S;
      const int t0 =
          (int)((cw + kConsumerWarps - (int)(tbase % kConsumerWarps)) % kConsumerWarps);
      tbase += ntasks;
      const uint32_t ws = ring_a + slot * p.stage_bytes;
      const uint32_t ds = ws + p.wd_off;
      float* pp = part + (size_t)slot * p.rps * S * M;
      int ngi = S > 1 ? (int)__umulhi((uint32_t)t0, sinv) : t0;
      int nsl = t0 - ngi * S;
      for (int t = t0; t < ntasks; t += kConsumerWarps) {
        const int gi = ngi;
        const int s = nsl;
        ngi += dgi;
        nsl += dsl;
        if (nsl >= S) {
          nsl -= S;
          ++ngi;
        }
        const int rbase = gi * R;
        int xrow = mt.xrow;
        if (packed_stage) {
          const int k = rbase / mt.xrow;
          if (s_ids[k] < 0) continue;  // not copied; its partials are never read
          xrow = p.xpe ? k : 0;
        }
        const int plo = s_slice[s];
        const int phi = s_slice[s + 1];
        // Per-lane shared-window addresses at the task's first block; add_part reaches
        // part q of the slice at an immediate offset from them.
        uint32_t wl[R], dl[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          // Rows past the stage's end reuse a valid row; their sums are dropped.
          const int row = rbase + r < nr ? rbase + r : rbase;
          wl[r] = ws + row * Qrow + (plo * 32 + lane) * kBlockBytes + (FMT == kQ8 ? h1 * 16 : 0);
          dl[r] = ds + (row * nb + plo * 32 + lane) * 2;
        }
        const int xb = xrow * nb + plo * 32 + lane;  // the task's first activation block
        const uint32_t xl = xs_a + xb * 32 + xh * 16;
        const uint32_t xdl = xds_a + xb * 4;
        const uint32_t xsl = xsum_a + xb * 4;
        float acc[R][M];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;
        // A slice has at most kSlicePartsMax parts.  Unrolled over that bound, every
        // part's offsets are constants; the parts are still taken in order, so each
        // lane's sum is unchanged.
#pragma unroll
        for (int q = 0; q < kSlicePartsMax; ++q) {
          const int pt = plo + q;
          if (pt < phi && (pt < p.cpr - 1 || last_ok))
            add_part<M, R, FMT>(acc, wl, dl, xl, xdl, xsl, q, Ki, nb, h1, xh, pc);
        }
        store_partials<R, M>(acc, lane, pp, rbase, nr - rbase, s, S);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(slot));
      if (++slot == ns) {
        slot = 0;
        phase ^= 1;
      }
    }
  }
}

// ============================================================================
// Register kernel (fallback): the same tasks, weights loaded into registers.
// ============================================================================
#ifndef MEMRA_REG_WARPS
#define MEMRA_REG_WARPS 16
#endif
constexpr int kRegWarps = MEMRA_REG_WARPS;
constexpr int kRegThreads = kRegWarps * 32;
// 32 resident warps per SM (64 registers a thread): plain 256-bit streaming needs
// about that many loads in flight to approach the HBM read ceiling.
constexpr int kRegCtasPerSm = kRegWarps >= 32 ? 1 : 32 / kRegWarps;
// Several activation rows need more registers than 64 a thread: those products
// run half as many warps (128 registers a thread).
__host__ __device__ constexpr int reg_ctas_per_sm(int M) {
  return M == 1 ? kRegCtasPerSm : (kRegCtasPerSm > 1 ? kRegCtasPerSm / 2 : 1);
}
constexpr int kPartFloats = 8192;  // 32 KB of slice partials per tile

// Activation rows in shared memory for the register kernel: half-block planes
// xs[row][half][block][16 bytes], so that lane-consecutive blocks read
// consecutive 16-byte words (no bank conflicts) with the halves in register order.
__device__ __forceinline__ int split_offset(int row, int byte, int nb) {
  const int blk = byte >> 5;
  const int h = (byte >> 4) & 1;
  return ((row * 2 + h) * nb + blk) * 16 + (byte & 15);
}

template <int XIN>
__device__ __forceinline__ void stage_x_split(const Params& p, int8_t* xs, float* xds, int w,
                                              int nwarps, int lane, int tid, int nthreads) {
  const int nb = p.nb;
  // rows * K is bounded by MEMRA_MAX_X_BYTES, so 32-bit indices suffice.
  const int K = (int)p.K;
  if (XIN == kXq8) {
    const int wpr = K / 16;  // 16-byte words per row
    const int words = p.xrows * wpr;
    for (int i = tid; i < words; i += nthreads) {
      const int row = i / wpr;
      const int j = i - row * wpr;
      *reinterpret_cast<uint4*>(xs + split_offset(row, j * 16, nb)) =
          reinterpret_cast<const uint4*>(p.xq)[i];
    }
    const int nd = p.xrows * nb;
    for (int i = tid; i < nd; i += nthreads) xds[i] = p.xd[i];
  } else {
    // Quantise 8-value groups; a warp handles 2 groups per lane per round with both
    // loads issued first (the prefetched weights still hold registers here).
    constexpr int U = 2;
    const int gpr = K / 8;
    const int groups = p.xrows * gpr;
    for (int base = w * 32 * U; base < groups; base += nwarps * 32 * U) {
      float v[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = base + u * 32 + lane;
        if (g < groups) {
          load_x_group<XIN>(p.xin, g, K, v[u]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) v[u][i] = 0.0f;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int g = base + u * 32 + lane;
        float d;
        const uint2 q = q8_1_group8(v[u], &d);
        if (g < groups) {
          const int row = g / gpr;
          const int byte = (g - row * gpr) * 8;
          *reinterpret_cast<uint2*>(xs + split_offset(row, byte, nb)) = q;
          if ((lane & 3) == 0) xds[g >> 2] = d;
        }
      }
    }
  }
}

template <int M, int R, int MODE, int XIN>
__global__ void __launch_bounds__(kRegThreads, reg_ctas_per_sm(M)) q8_reg_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nb = p.nb;
  const int S = p.S;
  const int64_t K = p.K;

  // Shared memory: xs | xds | partials | ids | gates | slice table.
  int8_t* xs = reinterpret_cast<int8_t*>(smem);
  float* xds = reinterpret_cast<float*>(smem + p.off_xd);
  float* part = reinterpret_cast<float*>(smem + p.off_part);
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem + p.off_yacc);
  float* s_gate = reinterpret_cast<float*>(s_ids + kMaxTopK);
  int* s_slice = reinterpret_cast<int*>(s_gate + kMaxTopK);

  const int64_t u0 = cta_unit(p.units, blockIdx.x, gridDim.x);
  const int64_t u1 = cta_unit(p.units, blockIdx.x + 1, gridDim.x);
  // Lanes past the end of a row's last part hold no block.
  const bool last_ok = lane < nb - (p.cpr - 1) * 32;

  // Parts in groups of G: every load of a group is issued before its math.
  constexpr int G = R >= 4 ? 1 : (R == 2 || MODE != kDense ? 2 : kSlicePartsMax);
  Quants32 w[G][R];
  uint16_t dw[G][R];

  // wt/dt: this lane's first block of the task's first part in row rbase.
  auto load_group = [&](const int8_t* wt, const uint16_t* dt, int q0, int npart, int plo,
                        int rows_left) {
#pragma unroll
    for (int q = 0; q < G; ++q) {
      const int pq = q0 + q;
      const bool inb = pq < npart && (plo + pq < p.cpr - 1 || last_ok);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (inb && r < rows_left) {
          w[q][r] = ld_stream_32B(wt + r * K + pq * 1024);
          dw[q][r] = ld_stream_u16(dt + r * nb + pq * 32);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[q][r].w[i] = 0u;
          dw[q][r] = 0;
        }
      }
    }
  };

  // Routed products signal their dependents only after the routing has been read
  // behind the wait (a following kernel of the same call may rely on that).
  if (MODE == kDense) pdl_launch_dependents();
  // Dense products stream weights that the preceding kernel does not write: the
  // first group of this warp's first task is requested before waiting for it.
  bool prefetched = false;
  if (MODE == kDense) {
    const int nr = (int)min((int64_t)p.tile_rows, u1 - u0);
    if (warp < ((nr + R - 1) / R) * S) {
      const int gi = warp / S;
      const int s = warp - gi * S;
      const int plo = (int)(((long long)s * p.cpr) / S);
      const int phi = (int)(((long long)(s + 1) * p.cpr) / S);
      const int64_t row = u0 + gi * R;
      load_group(p.wq + row * K + (plo * 32 + lane) * 32, p.wd + row * nb + plo * 32 + lane, 0,
                 phi - plo, plo, nr - gi * R);
      prefetched = true;
    }
  }
  fill_slice_table(s_slice, p.cpr, S, threadIdx.x, kRegThreads);
  pdl_wait();
  if (MODE != kDense) {
    load_routing<MODE>(p, s_ids, s_gate, threadIdx.x, kRegThreads);
    pdl_launch_dependents();
  }
  stage_x_split<XIN>(p, xs, xds, warp, kRegWarps, lane, threadIdx.x, kRegThreads);
  __syncthreads();

  const int64_t k0 = first_slot<MODE>(p, u0);
  const int nseg = num_segs<MODE>(p, u0, u1, k0);
  bool any_valid = false;
  for (int si = 0; si < nseg; ++si) {
    const Seg g = get_seg<MODE>(p, u0, u1, si, s_ids, k0);
    if (!g.valid) {
      if (MODE == kMoeUngated)
        for (int i = threadIdx.x; i < g.nrows; i += kRegThreads) p.y[g.out0 + i] = 0.0f;
      continue;
    }
    const int xrow = (MODE == kDense) ? 0 : g.xrow;
    const int8_t* xlo = xs + ((size_t)xrow * 2) * nb * 16 + lane * 16;       // half 0
    const int8_t* xhi = xs + ((size_t)xrow * 2 + 1) * nb * 16 + lane * 16;   // half 1
    const float* xdl = xds + (size_t)xrow * nb + lane;
    for (int r0 = 0; r0 < g.nrows; r0 += p.tile_rows) {
      const int nr = min(p.tile_rows, g.nrows - r0);
      const int groups = (nr + R - 1) / R;
      const int ntasks = groups * S;
      for (int t = warp; t < ntasks; t += kRegWarps) {
        const int gi = t / S;
        const int s = t - gi * S;
        const int rbase = gi * R;
        const int plo = s_slice[s];
        const int npart = s_slice[s + 1] - plo;
        const int64_t row = g.row0 + r0 + rbase;
        const int8_t* wt = p.wq + row * K + (plo * 32 + lane) * 32;
        const uint16_t* dt = p.wd + row * nb + plo * 32 + lane;
        float acc[R][M];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;
        for (int q0 = 0; q0 < npart; q0 += G) {
          if (prefetched) {
            prefetched = false;  // the prologue already requested this group
          } else {
            load_group(wt, dt, q0, npart, plo, nr - rbase);
          }
#pragma unroll
          for (int q = 0; q < G; ++q) {
            const int pq = q0 + q;
            if (pq < npart && (plo + pq < p.cpr - 1 || last_ok)) {
              const int off = (plo + pq) * 32;  // block index of lane 0
#pragma unroll
              for (int m = 0; m < M; ++m) {
                const uint4 x0 = *reinterpret_cast<const uint4*>(xlo + ((size_t)m * 2 * nb + off) * 16);
                const uint4 x1 = *reinterpret_cast<const uint4*>(xhi + ((size_t)m * 2 * nb + off) * 16);
                const float dx = xdl[(size_t)m * nb + off];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                  const uint4 w0 =
                      make_uint4(w[q][r].w[0], w[q][r].w[1], w[q][r].w[2], w[q][r].w[3]);
                  const uint4 w1 =
                      make_uint4(w[q][r].w[4], w[q][r].w[5], w[q][r].w[6], w[q][r].w[7]);
                  const int sb = dot_halves(w0, w1, x0, x1);
                  acc[r][m] = block_term_acc(acc[r][m], dw[q][r], dx, sb);
                }
              }
            }
          }
        }
        store_partials<R, M>(acc, lane, part, rbase, nr - rbase, s, S);
      }
      __syncthreads();
      // Tile epilogue: slice sums in order.
      for (int i = threadIdx.x; i < nr * M; i += kRegThreads) {
        const int r = i / M;
        const int m = i - r * M;
        float tot = part[((size_t)r * S) * M + m];
        for (int s = 1; s < S; ++s) tot = __fadd_rn(tot, part[((size_t)r * S + s) * M + m]);
        if (MODE == kMoeGated) {
          // Gated tiles cover the CTA's whole n-range, so each output accumulates
          // over k (ascending) in its own y word, starting from the first valid k.
          const int64_t n = u0 + r0 + r;
          const float prev = any_valid ? p.y[n] : 0.0f;
          p.y[n] = __fadd_rn(prev, __fmul_rn(s_gate[g.k], tot));
        } else {
          p.y[(int64_t)m * p.units + g.out0 + r0 + r] = tot;
        }
      }
      __syncthreads();
    }
    any_valid = true;
  }
  if (MODE == kMoeGated && !any_valid) {
    for (int64_t i = u0 + threadIdx.x; i < u1; i += kRegThreads) p.y[i] = 0.0f;
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
    const uint4 w0 = make_uint4(w.w[0], w.w[1], w.w[2], w.w[3]);
    const uint4 w1 = make_uint4(w.w[4], w.w[5], w.w[6], w.w[7]);
    s[i] = dot_halves(w0, w1, xp[0], xp[1]);
  }
}

// Gated sum of a batch's routed slots: y[t][n] = sum over the valid slots k of token
// t, in ascending k, of gate[t][k] * yp[t][k][n], from 0 with one rounding per
// multiply and per add.  That is the gated routed product's own order, so token t's
// row equals, bit for bit, the gated product of that token alone.
__global__ void __launch_bounds__(256)
    moe_combine_kernel(const float* __restrict__ yp, const int32_t* __restrict__ ids,
                       const float* __restrict__ gate_w, int64_t T, int top_k, int64_t N,
                       int64_t E, float* __restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t total = T * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / N;
    const int64_t n = i - t * N;
    float acc = 0.0f;
    for (int k = 0; k < top_k; ++k) {
      const int64_t slot = t * top_k + k;
      const int32_t e = __ldcg(ids + slot);
      if (e < 0 || e >= E) continue;
      acc = __fadd_rn(acc, __fmul_rn(__ldcg(gate_w + slot), yp[slot * N + n]));
    }
    y[i] = acc;
  }
}

// ----------------------------------------------------------------------------
// Host dispatch.
// ----------------------------------------------------------------------------

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Sizes of the bulk-copy kernel.  The compiled-in defaults can be overridden per
// process by environment variables of the same names (MEMRA_TMA_RING_KB, ...), read
// on first use; a value that is not a non-negative integer keeps the default.
struct TmaTuning {
  size_t stage_target;    // bytes per ring stage (rounded to whole rows)
  size_t ring_budget;     // bytes of ring per CTA
  size_t smem_pair_limit; // shared memory of one CTA when two must fit on an SM
  int ctas_per_sm;
  size_t packed_max;         // gated routed: largest packed stage (bytes)
  size_t multi_ring_budget;  // M > 1: bytes of ring per CTA (one CTA per SM)
  size_t multi_stage_target; // M > 1: bytes per ring stage
  size_t routed_stage_target; // M = 1 routed experts: bytes per ring stage
  bool multi_default;        // M > 1 products use this kernel by default
  int64_t dense_min_bytes;  // smaller dense products use the register kernel
  int prefill_stages;       // dense: stages issued before the activation is staged (0: all)
  int routed_prefill;       // the same for routed products
  int prefill_4bit;         // the same for dense M = 1 products on 4-bit weights
};

long env_long(const char* name, long dflt, long lo) {
  const char* e = std::getenv(name);
  if (!e || !*e) return dflt;
  char* end = nullptr;
  const long v = std::strtol(e, &end, 10);
  if (*end != '\0' || v < lo || v > (1L << 20)) return dflt;
  return v;
}

const TmaTuning& tma_tuning() {
  static const TmaTuning t = [] {
    TmaTuning r;
    r.stage_target = (size_t)env_long("MEMRA_TMA_STAGE_KB", MEMRA_TMA_STAGE_KB, 1) * 1024;
    r.ring_budget = (size_t)env_long("MEMRA_TMA_RING_KB", MEMRA_TMA_RING_KB, 1) * 1024;
    r.smem_pair_limit =
        (size_t)env_long("MEMRA_TMA_SMEM_LIMIT_KB", MEMRA_TMA_SMEM_LIMIT_KB, 1) * 1024;
    r.packed_max = (size_t)env_long("MEMRA_TMA_PACKED_KB", 48, 0) * 1024;
    r.multi_ring_budget =
        (size_t)env_long("MEMRA_TMA_MULTI_RING_KB", MEMRA_TMA_MULTI_RING_KB, 1) * 1024;
    r.routed_stage_target =
        (size_t)env_long("MEMRA_TMA_ROUTED_STAGE_KB", MEMRA_TMA_ROUTED_STAGE_KB, 1) * 1024;
    r.multi_stage_target =
        (size_t)env_long("MEMRA_TMA_MULTI_STAGE_KB", MEMRA_TMA_MULTI_STAGE_KB, 1) * 1024;
    r.multi_default = env_long("MEMRA_TMA_MULTI", 1, 0) != 0;
    r.ctas_per_sm = (int)env_long("MEMRA_TMA_CTAS_PER_SM", MEMRA_TMA_CTAS_PER_SM, 1);
    r.dense_min_bytes =
        (int64_t)env_long("MEMRA_TMA_DENSE_MIN_MB", MEMRA_TMA_DENSE_MIN_MB, 0) * 1024 * 1024;
    r.prefill_stages = (int)env_long("MEMRA_TMA_PREFILL", MEMRA_TMA_PREFILL, 0);
    r.routed_prefill = (int)env_long("MEMRA_TMA_ROUTED_PREFILL", MEMRA_TMA_ROUTED_PREFILL, 0);
    r.prefill_4bit = (int)env_long("MEMRA_TMA_PREFILL_4BIT", MEMRA_TMA_PREFILL_4BIT, 0);
    return r;
  }();
  return t;
}

// Kernel selection seam for tests and benchmarks (read once per process):
// MEMRA_GEMV_PATH=reg forces the register kernel; MEMRA_GEMV_PATH=tma uses the
// bulk-copy kernel wherever it applies, whatever the size.  By default the bulk-copy
// kernel serves products of at least ~24 MB of weights (M = 1 and M > 1), routed
// experts, and the register kernel the rest (small products, K % 256 != 0, planes
// not 16-byte aligned).
int gemv_path_override() {
  static const int v = [] {
    const char* e = std::getenv("MEMRA_GEMV_PATH");
    if (e && std::strcmp(e, "reg") == 0) return 1;
    if (e && std::strcmp(e, "tma") == 0) return 2;
    if (e && std::strcmp(e, "mma") == 0) return 3;
    return 0;
  }();
  return v;
}

// The tensor-core kernel (mma.cu) takes dense products only when MEMRA_GEMV_PATH=mma:
// on GB300 it does not beat the CUDA-core kernels (memra_q8_0_gemm_small_m_mma).
bool use_mma() { return gemv_path_override() == 3; }

int64_t max_units_per_cta(int64_t units, int64_t grid) { return (units + grid - 1) / grid; }

template <int M, int R, int MODE, int XIN, int FMT = kQ8>
bool plan_tma(Params& p, const DeviceInfo& info, int64_t grid, size_t* smem_out) {
  const int path = gemv_path_override();
  const TmaTuning& tune = tma_tuning();
  if (FMT == kQ8 && (path == 1 || (path == 0 && M > 1 && !tune.multi_default))) return false;
  // Per-shape dispatch: below a few tens of MB of weights the register kernel's
  // faster start wins over the deeper bulk-copy stream (measured on GB300).
  if (FMT == kQ8 && path == 0 && MODE == kDense && p.units * p.K < tune.dense_min_bytes)
    return false;
  if (p.K % 256 != 0) return false;
  if (!aligned(p.wd, 16) || !aligned(p.wq, 16)) return false;
  if (XIN == kXq8 && (!aligned(p.xd, 16) || !aligned(p.xq, 16))) return false;
  const size_t row_bytes = (size_t)p.qrow + (size_t)p.nb * 2;
  const int64_t maxu = max_units_per_cta(p.units, grid);
  const bool pairs = MODE == kMoeUngated && p.pairs;
  const int64_t upr = pairs ? 2 : 1;  // weight rows per unit
  // A routed product whose CTA share is a few stages long (one token's slots) takes
  // smaller stages; batches of tokens, with shares many stages long, keep the
  // dense size.
  const bool short_routed =
      MODE != kDense && (size_t)(maxu * upr) * row_bytes <= 4 * tune.stage_target;
  const size_t target = M > 1 ? tune.multi_stage_target
                        : (short_routed ? tune.routed_stage_target : tune.stage_target);
  int rps = (int)std::max<size_t>(1, target /
                                          row_bytes);
  // A stage never spans two segments, and no segment is longer than a CTA's share
  // of the units (routed: of one expert's rows): size stages, and so the ring's
  // depth, by what a stage can actually hold.
  rps = (int)std::min<int64_t>(
      rps, MODE == kMoeUngated ? upr * std::min<int64_t>(maxu, p.N) : maxu);
  rps = std::max(R, rps / R * R);
  if (pairs) rps = std::max(2, rps / 2 * 2);  // whole pairs: n gate rows and n up rows
  // Gated routed products whose segments are a few rows each pack all of a CTA's
  // segments into one stage.
  p.packed = 0;
  if (MODE == kMoeGated && R == 1 && (size_t)p.top_k * maxu * row_bytes <= tune.packed_max) {
    p.packed = 1;
    rps = (int)(p.top_k * maxu);
  }
  size_t stage = align_up((size_t)rps * p.qrow, 128) + align_up((size_t)rps * p.nb * 2, 128);
  // Activation rows a CTA stages: an ungated routed product with a row per slot group
  // needs only those of the slots its unit range touches (at most ceil(maxu/N) + 1).
  const int64_t xr = MODE == kMoeUngated && p.xpe
                         ? std::min<int64_t>(p.xrows, (maxu + p.N - 1) / p.N + 1)
                         : p.xrows;
  const size_t xsum_bytes = FMT == kQ4 ? align_up((size_t)xr * p.nb * 4, 128) : 0;
  const size_t xbytes = align_up((size_t)xr * p.K, 128) + align_up((size_t)xr * p.nb * 4, 128) +
                        xsum_bytes;
  const size_t yacc = MODE == kMoeGated ? align_up((size_t)maxu * 4, 16) : 0;
  const size_t fixed = kHeaderBytes + xbytes + yacc + align_up((size_t)(p.S + 1) * 4, 16);
  size_t part_per_stage = align_up((size_t)rps * p.S * M * 4, 16);
  // Ring: up to the budget, and within the two-CTAs-per-SM limit when possible.  M > 1
  // products run one CTA per SM (their consumers need more registers) with a deeper
  // ring.
  size_t limit = M > 1 ? (size_t)info.max_smem_optin
                       : std::max<size_t>(tune.smem_pair_limit, fixed + 2 * (stage + part_per_stage));
  limit = std::min<size_t>(limit, (size_t)info.max_smem_optin);
  const size_t budget = M > 1 ? tune.multi_ring_budget : tune.ring_budget;
  int ns = (int)std::min<size_t>(kMaxStages, std::max<size_t>(2, budget / stage));
  // A dense product whose CTA share is a little more than the ring holds: stretch the
  // stages so that the whole share is in flight at once (no stage waits for a slot).
  if (MODE == kDense && maxu > (int64_t)ns * rps) {
    const int wide = (int)((maxu + ns - 1) / ns + R - 1) / R * R;
    const size_t wstage =
        align_up((size_t)wide * p.qrow, 128) + align_up((size_t)wide * p.nb * 2, 128);
    const size_t wpart = align_up((size_t)wide * p.S * M * 4, 16);
    if (wide <= 2 * rps && fixed + ns * (wstage + wpart) <= limit) {
      rps = wide;
      stage = wstage;
      part_per_stage = wpart;
    }
  }
  while (ns > 2 && fixed + ns * (stage + part_per_stage) > limit) --ns;
  if (ns < 2 || fixed + ns * (stage + part_per_stage) > (size_t)info.max_smem_optin) return false;
  p.rps = rps;
  p.ns = ns;
  p.stage_bytes = (uint32_t)stage;
  p.wd_off = (uint32_t)align_up((size_t)rps * p.qrow, 128);
  size_t off = kHeaderBytes;
  p.off_x = (uint32_t)off;
  p.off_xd = (uint32_t)(off + align_up((size_t)xr * p.K, 128));
  p.off_xsum = (uint32_t)(p.off_xd + align_up((size_t)xr * p.nb * 4, 128));
  off += xbytes;
  p.off_ring = (uint32_t)off;
  off += (size_t)ns * stage;
  p.off_part = (uint32_t)off;
  off += (size_t)ns * part_per_stage;
  p.off_yacc = (uint32_t)off;
  off += yacc;
  p.off_slice = (uint32_t)off;
  off += align_up((size_t)(p.S + 1) * 4, 16);
  *smem_out = off;
  return true;
}

template <int M, int R, int MODE, int XIN>
bool plan_reg(Params& p, const DeviceInfo& info, int64_t grid, size_t* smem_out) {
  const int64_t maxu = max_units_per_cta(p.units, grid);
  int64_t tile;
  if (MODE == kMoeGated) {
    tile = maxu;  // the gated epilogue needs the whole n-range in one tile
  } else {
    tile = std::max<int64_t>(R, kPartFloats / ((int64_t)p.S * M) / R * R);
    tile = std::min<int64_t>(tile, (maxu + R - 1) / R * R);
  }
  p.tile_rows = (int)std::max<int64_t>(tile, 1);
  const size_t xb = align_up((size_t)p.xrows * p.K, 16);
  const size_t db = align_up((size_t)p.xrows * p.nb * 4, 16);
  const size_t pb = align_up((size_t)p.tile_rows * p.S * M * 4, 16);
  p.off_xd = (uint32_t)xb;
  p.off_part = (uint32_t)(xb + db);
  p.off_yacc = (uint32_t)(xb + db + pb);
  const size_t total = xb + db + pb + 2 * kMaxTopK * 4 + align_up((size_t)(p.S + 1) * 4, 16);
  if (total > (size_t)info.max_smem_optin) return false;
  *smem_out = total;
  return true;
}

template <typename Kern>
memra_status launch(Kern kernel, int64_t grid, int threads, size_t smem, cudaStream_t stream,
                    const DeviceInfo& info, const Params& p) {
  cudaError_t e = allow_dynamic_smem(kernel, smem, info);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_kernel(kernel, dim3((unsigned)grid), dim3(threads), smem, stream, p);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

// CTAs per SM in a register-kernel grid: the occupancy the kernel is built for,
// or fewer (MEMRA_REG_CTAS_PER_SM, read once per process).
int reg_grid_ctas_per_sm(int M) {
  static const long v = env_long("MEMRA_REG_CTAS_PER_SM", 0, 0);
  const int built = reg_ctas_per_sm(M);
  return v > 0 && v < built ? (int)v : built;
}

// The wait test hook (memra_debug_set_wait_test): 0 and -1 when off.
std::atomic<long long> g_test_wait_limit{0};
std::atomic<long long> g_test_stall_after{-1};

template <int M, int R, int MODE, int XIN, int FMT = kQ8>
memra_status run_product(Params p, cudaStream_t stream) {
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  p.prefill_stages = MODE != kDense ? tma_tuning().routed_prefill
                     : (FMT != kQ8 && M == 1 ? tma_tuning().prefill_4bit
                                             : tma_tuning().prefill_stages);
  const long long wl = g_test_wait_limit.load(std::memory_order_relaxed);
  p.wait_limit = wl > 0 ? wl : kWaitLimitCycles;
  p.stall_after = (int)g_test_stall_after.load(std::memory_order_relaxed);
  p.qrow = FMT == kQ8 ? p.K : p.K / 2;
  p.nb = (int)(p.K / 32);
  p.cpr = (p.nb + 31) / 32;
  p.S = slices_for(p.cpr);
  // A single wave of `slots` CTAs; a batched routed product takes a multiple of its
  // slot count, so that every slot's rows split at the same offsets.
  auto wave = [&](int64_t slots) {
    if (p.lockstep > 0 && p.lockstep <= slots) slots = slots / p.lockstep * p.lockstep;
    return std::min<int64_t>(p.units, slots);
  };
  int64_t grid = wave((int64_t)info.sms * (M > 1 ? 1 : tma_tuning().ctas_per_sm));
  size_t smem = 0;
  if (plan_tma<M, R, MODE, XIN, FMT>(p, info, grid, &smem)) {
    if (grid > info.sms && smem > tma_tuning().smem_pair_limit) {
      // Only one such CTA fits per SM: one per SM, so the grid stays a single wave.
      grid = wave(info.sms);
      if (!plan_tma<M, R, MODE, XIN, FMT>(p, info, grid, &smem)) return MEMRA_ERR_UNSUPPORTED;
    }
    return launch(q8_tma_kernel<M, R, MODE, XIN, FMT>, grid, tma_threads(M), smem, stream, info,
                  p);
  }
  // 4-bit formats and gate|up pairs run on the bulk-copy kernel only.
  if (FMT != kQ8 || p.pairs) return MEMRA_ERR_UNSUPPORTED;
  grid = std::min<int64_t>(p.units, (int64_t)info.sms * reg_grid_ctas_per_sm(M));
  if (plan_reg<M, R, MODE, XIN>(p, info, grid, &smem))
    return launch(q8_reg_kernel<M, R, MODE, XIN>, grid, kRegThreads, smem, stream, info, p);
  return MEMRA_ERR_UNSUPPORTED;
}

// Q4_0 and NVFP4 products (dense, q8_1 input).  A 4-bit block costs as many dp4a as
// a Q8_0 block (NVFP4 twice as many) in half the bytes, so the consumers, not the
// stream, set the pace: M = 1 takes 3-row tasks, which share each block's activation
// loads between three rows, and whose 34 KB stages hold 12 rows at K = 5120 and 3 at
// K = 17408 (64-layer sweeps, Q4_0 / NVFP4 ms per token: 1-row tasks 3.00 / 3.55,
// 2-row 2.91 / 3.36, 3-row 2.86 / 3.33, 4-row 3.01 / 3.51).  M = 8 takes 2-row tasks:
// with K = 17408 the activation planes and their block sums leave room for 2-row
// stages only.
template <int FMT>
memra_status dispatch_m_4bit(const Params& p, int M, cudaStream_t s) {
  switch (M) {
    case 1: return run_product<1, 3, kDense, kXq8, FMT>(p, s);
    case 2: return run_product<2, 1, kDense, kXq8, FMT>(p, s);
    case 3: return run_product<3, 1, kDense, kXq8, FMT>(p, s);
    case 4: return run_product<4, 2, kDense, kXq8, FMT>(p, s);
    case 5: return run_product<5, 2, kDense, kXq8, FMT>(p, s);
    case 6: return run_product<6, 2, kDense, kXq8, FMT>(p, s);
    case 7: return run_product<7, 2, kDense, kXq8, FMT>(p, s);
    case 8: return run_product<8, 2, kDense, kXq8, FMT>(p, s);
  }
  return MEMRA_ERR_UNSUPPORTED;
}

template <int MODE, int XIN>
memra_status dispatch_m(const Params& p, int M, cudaStream_t s) {
  switch (M) {
    case 1: return run_product<1, 1, MODE, XIN>(p, s);
    case 2: return run_product<2, 1, MODE, XIN>(p, s);
    case 3: return run_product<3, 1, MODE, XIN>(p, s);
    case 4: return run_product<4, 2, MODE, XIN>(p, s);
    case 5: return run_product<5, 2, MODE, XIN>(p, s);
    case 6: return run_product<6, 2, MODE, XIN>(p, s);
    case 7: return run_product<7, 2, MODE, XIN>(p, s);
    case 8: return run_product<8, 4, MODE, XIN>(p, s);
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

// A batch of up to MEMRA_MAX_M activation rows runs as passes over the weights of at
// most kPassRows rows each: one pass up to kPassRows, else ceil(M/2) then floor(M/2)
// rows.  Every row's arithmetic is the M = 1 arithmetic, so the split changes no bit
// of y.  From M = 8 on the dp4a issue rate, not the weight stream, sets a pass's time
// (the 27B verify sweep: 4.33 ms per token at M = 1, 6.85 ms at M = 8), so a second
// stream of the weights costs little next to the block dots.
constexpr int64_t kPassRows = 8;
static_assert(MEMRA_MAX_M <= 2 * kPassRows, "two passes at most");

int64_t pass_rows(int64_t M) { return M <= kPassRows ? M : (M + 1) / 2; }

template <typename Pass>
memra_status in_passes(int64_t M, Pass&& pass) {
  if (M <= kPassRows) return pass(0, M);
  const int64_t m1 = (M + 1) / 2;
  const memra_status st = pass(0, m1);
  if (st != MEMRA_OK) return st;
  return pass(m1, M - m1);
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
  if (!x_fits(pass_rows(M), K)) return MEMRA_ERR_UNSUPPORTED;
  return in_passes(M, [&](int64_t m0, int64_t rows) {
    if (use_mma()) {
      const memra_status st = run_mma_product(wq, wd, N, K, (int)rows, xq + m0 * K,
                                              xd + m0 * (K / 32), y + m0 * N, stream);
      if (st != MEMRA_ERR_UNSUPPORTED) return st;
    }
    Params p{};
    p.wq = wq;
    p.wd = wd;
    p.N = N;
    p.K = K;
    p.xq = xq + m0 * K;
    p.xd = xd + m0 * (K / 32);
    p.xrows = (int)rows;
    p.y = y + m0 * N;
    p.units = N;
    return dispatch_m<kDense, kXq8>(p, (int)rows, stream);
  });
}

extern "C" memra_status memra_q8_0_gemm_small_m_mma(const int8_t* wq, const uint16_t* wd,
                                                    int64_t N, int64_t K, int64_t M,
                                                    const int8_t* xq, const float* xd, float* y,
                                                    cudaStream_t stream) {
  if (N < 0 || K < 0 || M < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (M > MEMRA_MAX_M) return MEMRA_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (N == 0 || M == 0) return MEMRA_OK;
  if (!y) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4)) return MEMRA_ERR_ALIGNMENT;
  if (K == 0) return zero_fill(y, M * N, stream);
  if (!wq || !wd || !xq || !xd) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(wq, 16) || !aligned(wd, 16) || !aligned(xq, 16) || !aligned(xd, 16))
    return MEMRA_ERR_ALIGNMENT;
  return in_passes(M, [&](int64_t m0, int64_t rows) {
    return run_mma_product(wq, wd, N, K, (int)rows, xq + m0 * K, xd + m0 * (K / 32),
                           y + m0 * N, stream);
  });
}

extern "C" memra_status memra_q8_0_gemv(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K,
                                        const int8_t* xq, const float* xd, float* y,
                                        cudaStream_t stream) {
  return memra_q8_0_gemm_small_m(wq, wd, N, K, 1, xq, xd, y, stream);
}

extern "C" memra_status memra_q4_0_gemm_small_m(const uint8_t* wq4, const uint16_t* wd, int64_t N,
                                                int64_t K, int64_t M, const int8_t* xq,
                                                const float* xd, float* y, cudaStream_t stream) {
  if (N < 0 || K < 0 || M < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (M > MEMRA_MAX_M) return MEMRA_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (N == 0 || M == 0) return MEMRA_OK;
  if (!y) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4)) return MEMRA_ERR_ALIGNMENT;
  if (K == 0) return zero_fill(y, M * N, stream);
  if (!wq4 || !wd || !xq || !xd) return MEMRA_ERR_INVALID_ARG;
  if (K % 256 != 0) return MEMRA_ERR_UNSUPPORTED;
  if (!aligned(wq4, 16) || !aligned(wd, 16) || !aligned(xq, 16) || !aligned(xd, 16))
    return MEMRA_ERR_ALIGNMENT;
  if (!x_fits(pass_rows(M), K)) return MEMRA_ERR_UNSUPPORTED;
  return in_passes(M, [&](int64_t m0, int64_t rows) {
    Params p{};
    p.wq = reinterpret_cast<const int8_t*>(wq4);
    p.wd = wd;
    p.N = N;
    p.K = K;
    p.xq = xq + m0 * K;
    p.xd = xd + m0 * (K / 32);
    p.xrows = (int)rows;
    p.y = y + m0 * N;
    p.units = N;
    return dispatch_m_4bit<kQ4>(p, (int)rows, stream);
  });
}

extern "C" memra_status memra_nvfp4_gemm_small_m(const uint8_t* codes, const uint8_t* scales,
                                                 float g, int64_t N, int64_t K, int64_t M,
                                                 const int8_t* xq, const float* xd, float* y,
                                                 cudaStream_t stream) {
  if (N < 0 || K < 0 || M < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (M > MEMRA_MAX_M) return MEMRA_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (N == 0 || M == 0) return MEMRA_OK;
  if (!y) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4)) return MEMRA_ERR_ALIGNMENT;
  if (K == 0) return zero_fill(y, M * N, stream);
  if (!codes || !scales || !xq || !xd) return MEMRA_ERR_INVALID_ARG;
  if (K % 256 != 0) return MEMRA_ERR_UNSUPPORTED;
  if (!aligned(codes, 16) || !aligned(scales, 16) || !aligned(xq, 16) || !aligned(xd, 16))
    return MEMRA_ERR_ALIGNMENT;
  if (!x_fits(pass_rows(M), K)) return MEMRA_ERR_UNSUPPORTED;
  return in_passes(M, [&](int64_t m0, int64_t rows) {
    Params p{};
    p.wq = reinterpret_cast<const int8_t*>(codes);
    p.wd = reinterpret_cast<const uint16_t*>(scales);
    p.gscale = g * 0.5f;
    p.N = N;
    p.K = K;
    p.xq = xq + m0 * K;
    p.xd = xd + m0 * (K / 32);
    p.xrows = (int)rows;
    p.y = y + m0 * N;
    p.units = N;
    return dispatch_m_4bit<kNv4>(p, (int)rows, stream);
  });
}

extern "C" memra_status memra_nvfp4_gemv(const uint8_t* codes, const uint8_t* scales, float g,
                                         int64_t N, int64_t K, const int8_t* xq, const float* xd,
                                         float* y, cudaStream_t stream) {
  return memra_nvfp4_gemm_small_m(codes, scales, g, N, K, 1, xq, xd, y, stream);
}

extern "C" memra_status memra_q4_0_gemv(const uint8_t* wq4, const uint16_t* wd, int64_t N, int64_t K,
                                        const int8_t* xq, const float* xd, float* y,
                                        cudaStream_t stream) {
  return memra_q4_0_gemm_small_m(wq4, wd, N, K, 1, xq, xd, y, stream);
}

extern "C" memra_status memra_q8_0_quant_gemm(const int8_t* wq, const uint16_t* wd, int64_t N,
                                              int64_t K, int64_t M, const void* x, int32_t dtype,
                                              float* y, cudaStream_t stream) {
  if (N < 0 || K < 0 || M < 0 || K % 32 != 0) return MEMRA_ERR_INVALID_ARG;
  if (dtype != MEMRA_BF16 && dtype != MEMRA_F32) return MEMRA_ERR_INVALID_ARG;
  if (M > MEMRA_MAX_M) return MEMRA_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (N == 0 || M == 0) return MEMRA_OK;
  if (!y) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4)) return MEMRA_ERR_ALIGNMENT;
  if (K == 0) return zero_fill(y, M * N, stream);
  if (!wq || !wd || !x) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(wq, 32) || !aligned(wd, 2) || !aligned(x, 16)) return MEMRA_ERR_ALIGNMENT;
  if (!x_fits(pass_rows(M), K)) return MEMRA_ERR_UNSUPPORTED;
  const int64_t x_row_bytes = K * (dtype == MEMRA_BF16 ? 2 : 4);
  return in_passes(M, [&](int64_t m0, int64_t rows) {
    Params p{};
    p.wq = wq;
    p.wd = wd;
    p.N = N;
    p.K = K;
    p.xin = static_cast<const char*>(x) + m0 * x_row_bytes;
    p.xrows = (int)rows;
    p.y = y + m0 * N;
    p.units = N;
    if (dtype == MEMRA_BF16) return dispatch_m<kDense, kXbf16>(p, (int)rows, stream);
    return dispatch_m<kDense, kXf32>(p, (int)rows, stream);
  });
}

namespace memra {
namespace {
// The routed-expert GEMV for either weight format (wq_bank: int8 [E][N][K] for Q8_0,
// packed uint8 [E][N][K/2] for Q4_0).
template <int FMT>
memra_status moe_gemv(const int8_t* wq_bank, const uint16_t* wd_bank, int64_t E, int64_t N,
                      int64_t K, const int32_t* ids, const float* gate_w, int64_t top_k,
                      const int8_t* xq, const float* xd, int32_t x_per_expert, float* y,
                      int32_t* dev_status, cudaStream_t stream, const float* gexp = nullptr) {
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
  if (FMT != kQ8) {
    if (FMT == kNv4 && !gexp) return MEMRA_ERR_INVALID_ARG;
    if (K % 256 != 0) return MEMRA_ERR_UNSUPPORTED;
    if (!aligned(wq_bank, 16) || !aligned(wd_bank, 16) || !aligned(xq, 16) || !aligned(xd, 16) ||
        (gexp && !aligned(gexp, 4)))
      return MEMRA_ERR_ALIGNMENT;
  } else if (!aligned(wq_bank, 32) || !aligned(wd_bank, 2) || !aligned(xq, 16) ||
             !aligned(xd, 4)) {
    return MEMRA_ERR_ALIGNMENT;
  }
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
  p.ids = ids;
  p.gate_w = gate_w;
  p.top_k = (int)top_k;
  p.E = E;
  p.xpe = x_per_expert;
  p.status = dev_status;
  p.gexp = gexp;
  if (gate_w) {
    p.units = N;
    return run_product<1, 1, kMoeGated, kXq8, FMT>(p, stream);
  }
  p.units = top_k * N;
  return run_product<1, 1, kMoeUngated, kXq8, FMT>(p, stream);
}

memra_status launch_combine(const float* yp, const int32_t* ids, const float* gate_w, int64_t T,
                            int64_t top_k, int64_t N, int64_t E, float* y, cudaStream_t stream) {
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>((T * N + 255) / 256, (int64_t)info.sms * 8);
  const cudaError_t e = launch_kernel(moe_combine_kernel, dim3((unsigned)blocks), dim3(256), 0,
                                      stream, yp, ids, gate_w, T, (int)top_k, N, E, y);
  return e == cudaSuccess ? MEMRA_OK : cuda_fail(e);
}

// Routed experts for a batch of T tokens, top_k slots each: every (token, slot) pair is
// one segment of the ungated routed product (the single-token arithmetic), and the
// grid gives every pair the same row split (lockstep), so that pairs routed to the
// same expert read its rows from HBM once and from L2 after.
template <int FMT>
memra_status moe_gemv_tokens(const int8_t* wq_bank, const uint16_t* wd_bank, int64_t E,
                             int64_t N, int64_t K, const int32_t* ids, const float* gate_w,
                             int64_t T, int64_t top_k, const int8_t* xq, const float* xd,
                             int32_t x_per_expert, float* y, float* workspace,
                             int32_t* dev_status, cudaStream_t stream,
                             const float* gexp = nullptr) {
  if (E < 1 || N < 0 || K < 0 || K % 32 != 0 || top_k < 1 || T < 0) return MEMRA_ERR_INVALID_ARG;
  if (x_per_expert != 0 && x_per_expert != 1) return MEMRA_ERR_INVALID_ARG;
  if (top_k > MEMRA_MAX_TOP_K || T > MEMRA_MAX_PAIRS || T * top_k > MEMRA_MAX_PAIRS)
    return MEMRA_ERR_UNSUPPORTED;
  if (N > INT32_MAX || K > INT32_MAX || E > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (N == 0 || T == 0) return MEMRA_OK;
  if (!y || !ids || (gate_w && !workspace)) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4) || !aligned(ids, 4) || (gate_w && !aligned(gate_w, 4)) ||
      (gate_w && !aligned(workspace, 4)) || (dev_status && !aligned(dev_status, 4)))
    return MEMRA_ERR_ALIGNMENT;
  const int64_t P = T * top_k;
  if (K == 0) return zero_fill(y, gate_w ? T * N : P * N, stream);
  if (!wq_bank || !wd_bank || !xq || !xd) return MEMRA_ERR_INVALID_ARG;
  if (FMT != kQ8) {
    if (FMT == kNv4 && !gexp) return MEMRA_ERR_INVALID_ARG;
    if (K % 256 != 0) return MEMRA_ERR_UNSUPPORTED;
    if (!aligned(wq_bank, 16) || !aligned(wd_bank, 16) || !aligned(xq, 16) || !aligned(xd, 16) ||
        (gexp && !aligned(gexp, 4)))
      return MEMRA_ERR_ALIGNMENT;
  } else if (!aligned(wq_bank, 32) || !aligned(wd_bank, 2) || !aligned(xq, 16) ||
             !aligned(xd, 4)) {
    return MEMRA_ERR_ALIGNMENT;
  }
  const int64_t xrows = x_per_expert ? P : T;
  if (!x_fits(xrows, K)) return MEMRA_ERR_UNSUPPORTED;
  Params p{};
  p.wq = wq_bank;
  p.wd = wd_bank;
  p.N = N;
  p.K = K;
  p.xq = xq;
  p.xd = xd;
  p.xrows = (int)xrows;
  p.y = gate_w ? workspace : y;
  p.ids = ids;
  p.top_k = (int)P;
  p.E = E;
  p.xpe = 1;
  p.xdiv = x_per_expert ? 1 : (int)top_k;
  p.lockstep = (int)P;
  p.status = dev_status;
  p.gexp = gexp;
  p.units = P * N;
  const memra_status st = run_product<1, 1, kMoeUngated, kXq8, FMT>(p, stream);
  if (st != MEMRA_OK || !gate_w) return st;
  return launch_combine(workspace, ids, gate_w, T, top_k, N, E, y, stream);
}
}  // namespace
}  // namespace memra

extern "C" memra_status memra_q8_0_moe_gemv(const int8_t* wq_bank, const uint16_t* wd_bank,
                                            int64_t E, int64_t N, int64_t K, const int32_t* ids,
                                            const float* gate_w, int64_t top_k, const int8_t* xq,
                                            const float* xd, int32_t x_per_expert, float* y,
                                            int32_t* dev_status, cudaStream_t stream) {
  return moe_gemv<kQ8>(wq_bank, wd_bank, E, N, K, ids, gate_w, top_k, xq, xd, x_per_expert, y,
                       dev_status, stream);
}

extern "C" memra_status memra_q4_0_moe_gemv(const uint8_t* wq4_bank, const uint16_t* wd_bank,
                                            int64_t E, int64_t N, int64_t K, const int32_t* ids,
                                            const float* gate_w, int64_t top_k, const int8_t* xq,
                                            const float* xd, int32_t x_per_expert, float* y,
                                            int32_t* dev_status, cudaStream_t stream) {
  return moe_gemv<kQ4>(reinterpret_cast<const int8_t*>(wq4_bank), wd_bank, E, N, K, ids, gate_w,
                       top_k, xq, xd, x_per_expert, y, dev_status, stream);
}

extern "C" memra_status memra_nvfp4_moe_gemv(const uint8_t* codes_bank,
                                             const uint8_t* scales_bank, const float* gexp,
                                             int64_t E, int64_t N, int64_t K, const int32_t* ids,
                                             const float* gate_w, int64_t top_k,
                                             const int8_t* xq, const float* xd,
                                             int32_t x_per_expert, float* y, int32_t* dev_status,
                                             cudaStream_t stream) {
  return moe_gemv<kNv4>(reinterpret_cast<const int8_t*>(codes_bank),
                        reinterpret_cast<const uint16_t*>(scales_bank), E, N, K, ids, gate_w,
                        top_k, xq, xd, x_per_expert, y, dev_status, stream, gexp);
}

extern "C" memra_status memra_nvfp4_moe_gemv_tokens(const uint8_t* codes_bank,
                                                    const uint8_t* scales_bank,
                                                    const float* gexp, int64_t E, int64_t N,
                                                    int64_t K, const int32_t* ids,
                                                    const float* gate_w, int64_t T,
                                                    int64_t top_k, const int8_t* xq,
                                                    const float* xd, int32_t x_per_expert,
                                                    float* y, float* workspace,
                                                    int32_t* dev_status, cudaStream_t stream) {
  return moe_gemv_tokens<kNv4>(reinterpret_cast<const int8_t*>(codes_bank),
                               reinterpret_cast<const uint16_t*>(scales_bank), E, N, K, ids,
                               gate_w, T, top_k, xq, xd, x_per_expert, y, workspace, dev_status,
                               stream, gexp);
}

extern "C" memra_status memra_q8_0_moe_gemv_tokens(const int8_t* wq_bank, const uint16_t* wd_bank,
                                                   int64_t E, int64_t N, int64_t K,
                                                   const int32_t* ids, const float* gate_w,
                                                   int64_t T, int64_t top_k, const int8_t* xq,
                                                   const float* xd, int32_t x_per_expert,
                                                   float* y, float* workspace,
                                                   int32_t* dev_status, cudaStream_t stream) {
  return moe_gemv_tokens<kQ8>(wq_bank, wd_bank, E, N, K, ids, gate_w, T, top_k, xq, xd,
                              x_per_expert, y, workspace, dev_status, stream);
}

extern "C" memra_status memra_q4_0_moe_gemv_tokens(const uint8_t* wq4_bank,
                                                   const uint16_t* wd_bank, int64_t E, int64_t N,
                                                   int64_t K, const int32_t* ids,
                                                   const float* gate_w, int64_t T, int64_t top_k,
                                                   const int8_t* xq, const float* xd,
                                                   int32_t x_per_expert, float* y,
                                                   float* workspace, int32_t* dev_status,
                                                   cudaStream_t stream) {
  return moe_gemv_tokens<kQ4>(reinterpret_cast<const int8_t*>(wq4_bank), wd_bank, E, N, K, ids,
                              gate_w, T, top_k, xq, xd, x_per_expert, y, workspace, dev_status,
                              stream);
}

namespace memra {
namespace {
// The routed FFN's two banks: present for their format (NVFP4 also needs each bank's
// per-expert tensor scales), and aligned for the bulk copies.
template <int FMT>
bool banks_ok(const int8_t* gu_q, const uint16_t* gu_d, const int8_t* dn_q,
              const uint16_t* dn_d, int64_t, int64_t, const float* ggu, const float* gdn) {
  if (!gu_q || !gu_d || !dn_q || !dn_d) return false;
  return FMT != kNv4 || (ggu && gdn);
}

template <int FMT>
bool banks_aligned(const int8_t* gu_q, const uint16_t* gu_d, const int8_t* dn_q,
                   const uint16_t* dn_d, const float* ggu, const float* gdn) {
  if (FMT == kQ8)
    return aligned(gu_q, 32) && aligned(gu_d, 2) && aligned(dn_q, 32) && aligned(dn_d, 2);
  return aligned(gu_q, 16) && aligned(gu_d, 16) && aligned(dn_q, 16) && aligned(dn_d, 16) &&
         (!ggu || aligned(ggu, 4)) && (!gdn || aligned(gdn, 4));
}

template <int FMT>
memra_status moe_ffn(const int8_t* gu_q, const uint16_t* gu_d, const int8_t* dn_q,
                     const uint16_t* dn_d, int64_t E, int64_t H, int64_t F, const int32_t* ids,
                     const float* gate_w, int64_t top_k, const void* x, int32_t dtype, float* y,
                     float* workspace, int32_t* dev_status, cudaStream_t stream,
                     const float* ggu = nullptr, const float* gdn = nullptr) {
  if (E < 1 || H < 0 || F < 0 || H % 32 != 0 || F % 32 != 0 || top_k < 1)
    return MEMRA_ERR_INVALID_ARG;
  if (dtype != MEMRA_BF16 && dtype != MEMRA_F32) return MEMRA_ERR_INVALID_ARG;
  if (top_k > MEMRA_MAX_TOP_K) return MEMRA_ERR_UNSUPPORTED;
  if (H > INT32_MAX / 2 || F > INT32_MAX / 2 || E > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (H == 0) return MEMRA_OK;
  if (!y || !ids || !gate_w) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4) || !aligned(ids, 4) || !aligned(gate_w, 4) ||
      (dev_status && !aligned(dev_status, 4)))
    return MEMRA_ERR_ALIGNMENT;
  if (F == 0) return zero_fill(y, H, stream);
  if (!gu_q || !gu_d || !dn_q || !dn_d || !x || !workspace) return MEMRA_ERR_INVALID_ARG;
  if (!banks_ok<FMT>(gu_q, gu_d, dn_q, dn_d, H, F, ggu, gdn)) return MEMRA_ERR_INVALID_ARG;
  if (FMT != kQ8 && (H % 256 != 0 || F % 256 != 0)) return MEMRA_ERR_UNSUPPORTED;
  if (!banks_aligned<FMT>(gu_q, gu_d, dn_q, dn_d, ggu, gdn) || !aligned(x, 16) ||
      !aligned(workspace, 16))
    return MEMRA_ERR_ALIGNMENT;
  if (!x_fits(1, H) || !x_fits(top_k, F)) return MEMRA_ERR_UNSUPPORTED;
  // gate|up of every selected expert, as (gate j, up j) pairs: workspace[k][j] =
  // silu(g_j) u_j and workspace[k][F + j] = u_j, with (g, u) = W_gu[ids[k]] x.
  Params a{};
  a.wq = gu_q;
  a.wd = gu_d;
  a.N = F;
  a.K = H;
  a.xin = x;
  a.xrows = 1;
  a.y = workspace;
  a.ids = ids;
  a.top_k = (int)top_k;
  a.E = E;
  a.xpe = 0;
  a.status = dev_status;
  a.gexp = ggu;
  a.pairs = 1;
  a.units = top_k * F;
  auto gate_up = [&](const Params& q) {
    return dtype == MEMRA_BF16 ? run_product<1, 1, kMoeUngated, kXbf16, FMT>(q, stream)
                               : run_product<1, 1, kMoeUngated, kXf32, FMT>(q, stream);
  };
  memra_status st = gate_up(a);
  const bool paired = st != MEMRA_ERR_UNSUPPORTED;
  if (!paired) {
    // Shapes the bulk-copy kernel does not take: plain gate|up rows (workspace[k][0, 2F)
    // = W_gu[ids[k]] x), SwiGLU in the down launch's prologue.
    a.N = 2 * F;
    a.pairs = 0;
    a.units = top_k * 2 * F;
    st = gate_up(a);
  }
  if (st != MEMRA_OK) return st;
  // down rows with q8_1 of each expert's SwiGLU row (paired) or SwiGLU + q8_1 of its
  // gate|up row in the prologue.
  Params b{};
  b.wq = dn_q;
  b.wd = dn_d;
  b.N = H;
  b.K = F;
  b.xin = workspace;
  b.xrows = (int)top_k;
  b.y = y;
  b.ids = ids;
  b.gate_w = gate_w;
  b.top_k = (int)top_k;
  b.E = E;
  b.xpe = 1;
  b.status = dev_status;
  b.routing_ready = 1;  // the gate|up kernel above waited for the routing
  b.gexp = gdn;
  b.units = H;
  if (paired) return run_product<1, 1, kMoeGated, kXhalf, FMT>(b, stream);
  return run_product<1, 1, kMoeGated, kXswiglu, FMT>(b, stream);
}

template <int FMT>
memra_status moe_ffn_tokens(const int8_t* gu_q, const uint16_t* gu_d, const int8_t* dn_q,
                            const uint16_t* dn_d, int64_t E, int64_t H, int64_t F,
                            const int32_t* ids, const float* gate_w, int64_t T, int64_t top_k,
                            const void* x, int32_t dtype, float* y, float* workspace,
                            int32_t* dev_status, cudaStream_t stream,
                            const float* ggu = nullptr, const float* gdn = nullptr) {
  if (E < 1 || H < 0 || F < 0 || H % 32 != 0 || F % 32 != 0 || top_k < 1 || T < 0)
    return MEMRA_ERR_INVALID_ARG;
  if (dtype != MEMRA_BF16 && dtype != MEMRA_F32) return MEMRA_ERR_INVALID_ARG;
  if (top_k > MEMRA_MAX_TOP_K || T > MEMRA_MAX_PAIRS || T * top_k > MEMRA_MAX_PAIRS)
    return MEMRA_ERR_UNSUPPORTED;
  if (H > INT32_MAX / 2 || F > INT32_MAX / 2 || E > INT32_MAX) return MEMRA_ERR_UNSUPPORTED;
  if (H == 0 || T == 0) return MEMRA_OK;
  if (!y || !ids || !gate_w) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(y, 4) || !aligned(ids, 4) || !aligned(gate_w, 4) ||
      (dev_status && !aligned(dev_status, 4)))
    return MEMRA_ERR_ALIGNMENT;
  if (F == 0) return zero_fill(y, T * H, stream);
  if (!gu_q || !gu_d || !dn_q || !dn_d || !x || !workspace) return MEMRA_ERR_INVALID_ARG;
  if (!banks_ok<FMT>(gu_q, gu_d, dn_q, dn_d, H, F, ggu, gdn)) return MEMRA_ERR_INVALID_ARG;
  if (FMT != kQ8 && (H % 256 != 0 || F % 256 != 0)) return MEMRA_ERR_UNSUPPORTED;
  if (!banks_aligned<FMT>(gu_q, gu_d, dn_q, dn_d, ggu, gdn) || !aligned(x, 16) ||
      !aligned(workspace, 16))
    return MEMRA_ERR_ALIGNMENT;
  const int64_t P = T * top_k;
  if (!x_fits(T, H) || !x_fits(P, F)) return MEMRA_ERR_UNSUPPORTED;
  float* gu = workspace;              // [P][2F]: gate|up rows of every (token, slot)
  float* yp = workspace + P * 2 * F;  // [P][H]: down rows of every (token, slot)
  // gate|up, with each token's row quantised in the prologue.
  Params a{};
  a.wq = gu_q;
  a.wd = gu_d;
  a.N = 2 * F;
  a.K = H;
  a.xin = x;
  a.xrows = (int)T;
  a.y = gu;
  a.ids = ids;
  a.top_k = (int)P;
  a.E = E;
  a.xpe = 1;
  a.xdiv = (int)top_k;
  a.lockstep = (int)P;
  a.status = dev_status;
  a.gexp = ggu;
  a.units = P * 2 * F;
  memra_status st = dtype == MEMRA_BF16
                        ? run_product<1, 1, kMoeUngated, kXbf16, FMT>(a, stream)
                        : run_product<1, 1, kMoeUngated, kXf32, FMT>(a, stream);
  if (st != MEMRA_OK) return st;
  // down, with SwiGLU + q8_1 of each pair's gate|up row in the prologue.
  Params b{};
  b.wq = dn_q;
  b.wd = dn_d;
  b.N = H;
  b.K = F;
  b.xin = gu;
  b.xrows = (int)P;
  b.y = yp;
  b.ids = ids;
  b.top_k = (int)P;
  b.E = E;
  b.xpe = 1;
  b.xdiv = 1;
  b.lockstep = (int)P;
  b.status = dev_status;
  b.routing_ready = 1;  // the gate|up kernel above waited for the routing
  b.gexp = gdn;
  b.units = P * H;
  st = run_product<1, 1, kMoeUngated, kXswiglu, FMT>(b, stream);
  if (st != MEMRA_OK) return st;
  return launch_combine(yp, ids, gate_w, T, top_k, H, E, y, stream);
}

}  // namespace
}  // namespace memra

extern "C" memra_status memra_q8_0_moe_ffn(const int8_t* gu_q, const uint16_t* gu_d,
                                           const int8_t* dn_q, const uint16_t* dn_d, int64_t E,
                                           int64_t H, int64_t F, const int32_t* ids,
                                           const float* gate_w, int64_t top_k, const void* x,
                                           int32_t dtype, float* y, float* workspace,
                                           int32_t* dev_status, cudaStream_t stream) {
  return moe_ffn<kQ8>(gu_q, gu_d, dn_q, dn_d, E, H, F, ids, gate_w, top_k, x, dtype, y,
                      workspace, dev_status, stream);
}

extern "C" memra_status memra_q4_0_moe_ffn(const uint8_t* gu_q4, const uint16_t* gu_d,
                                           const uint8_t* dn_q4, const uint16_t* dn_d, int64_t E,
                                           int64_t H, int64_t F, const int32_t* ids,
                                           const float* gate_w, int64_t top_k, const void* x,
                                           int32_t dtype, float* y, float* workspace,
                                           int32_t* dev_status, cudaStream_t stream) {
  return moe_ffn<kQ4>(reinterpret_cast<const int8_t*>(gu_q4), gu_d,
                      reinterpret_cast<const int8_t*>(dn_q4), dn_d, E, H, F, ids, gate_w, top_k,
                      x, dtype, y, workspace, dev_status, stream);
}

extern "C" memra_status memra_nvfp4_moe_ffn(const uint8_t* gu_codes, const uint8_t* gu_scales,
                                            const float* gu_g, const uint8_t* dn_codes,
                                            const uint8_t* dn_scales, const float* dn_g,
                                            int64_t E, int64_t H, int64_t F, const int32_t* ids,
                                            const float* gate_w, int64_t top_k, const void* x,
                                            int32_t dtype, float* y, float* workspace,
                                            int32_t* dev_status, cudaStream_t stream) {
  return moe_ffn<kNv4>(reinterpret_cast<const int8_t*>(gu_codes),
                       reinterpret_cast<const uint16_t*>(gu_scales),
                       reinterpret_cast<const int8_t*>(dn_codes),
                       reinterpret_cast<const uint16_t*>(dn_scales), E, H, F, ids, gate_w, top_k,
                       x, dtype, y, workspace, dev_status, stream, gu_g, dn_g);
}

extern "C" memra_status memra_q8_0_moe_ffn_tokens(const int8_t* gu_q, const uint16_t* gu_d,
                                                  const int8_t* dn_q, const uint16_t* dn_d,
                                                  int64_t E, int64_t H, int64_t F,
                                                  const int32_t* ids, const float* gate_w,
                                                  int64_t T, int64_t top_k, const void* x,
                                                  int32_t dtype, float* y, float* workspace,
                                                  int32_t* dev_status, cudaStream_t stream) {
  return moe_ffn_tokens<kQ8>(gu_q, gu_d, dn_q, dn_d, E, H, F, ids, gate_w, T, top_k, x, dtype,
                             y, workspace, dev_status, stream);
}

extern "C" memra_status memra_q4_0_moe_ffn_tokens(const uint8_t* gu_q4, const uint16_t* gu_d,
                                                  const uint8_t* dn_q4, const uint16_t* dn_d,
                                                  int64_t E, int64_t H, int64_t F,
                                                  const int32_t* ids, const float* gate_w,
                                                  int64_t T, int64_t top_k, const void* x,
                                                  int32_t dtype, float* y, float* workspace,
                                                  int32_t* dev_status, cudaStream_t stream) {
  return moe_ffn_tokens<kQ4>(reinterpret_cast<const int8_t*>(gu_q4), gu_d,
                             reinterpret_cast<const int8_t*>(dn_q4), dn_d, E, H, F, ids, gate_w,
                             T, top_k, x, dtype, y, workspace, dev_status, stream);
}

extern "C" memra_status memra_nvfp4_moe_ffn_tokens(
    const uint8_t* gu_codes, const uint8_t* gu_scales, const float* gu_g,
    const uint8_t* dn_codes, const uint8_t* dn_scales, const float* dn_g, int64_t E, int64_t H,
    int64_t F, const int32_t* ids, const float* gate_w, int64_t T, int64_t top_k, const void* x,
    int32_t dtype, float* y, float* workspace, int32_t* dev_status, cudaStream_t stream) {
  return moe_ffn_tokens<kNv4>(reinterpret_cast<const int8_t*>(gu_codes),
                              reinterpret_cast<const uint16_t*>(gu_scales),
                              reinterpret_cast<const int8_t*>(dn_codes),
                              reinterpret_cast<const uint16_t*>(dn_scales), E, H, F, ids, gate_w,
                              T, top_k, x, dtype, y, workspace, dev_status, stream, gu_g, dn_g);
}





// ----------------------------------------------------------------------------
// memra_q8_0_moe_ffn_noalloc: the routed FFN with its gate|up workspace in a
// fixed device array owned by this library instead of caller memory.
// ----------------------------------------------------------------------------

// The array lives on every GPU that loads the library, until the process exits.
static __device__ __align__(256) float g_moe_ffn_scratch[MEMRA_MOE_NOALLOC_SCRATCH_FLOATS];

namespace memra {
namespace {
constexpr int kScratchDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_addr[kScratchDevices] = {};

// The scratch array's device address on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
memra_status moe_scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kScratchDevices) return MEMRA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_moe_ffn_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_scratch_addr[dev] = static_cast<float*>(ptr);
  }
  *out = g_scratch_addr[dev];
  return MEMRA_OK;
}
}  // namespace
}  // namespace memra

extern "C" memra_status memra_q8_0_moe_ffn_noalloc(const int8_t* gu_q, const uint16_t* gu_d,
                                                   const int8_t* dn_q, const uint16_t* dn_d,
                                                   int64_t E, int64_t H, int64_t F,
                                                   const int32_t* ids, const float* gate_w,
                                                   int64_t top_k, const void* x, int32_t dtype,
                                                   float* y, int32_t* dev_status,
                                                   cudaStream_t stream) {
  // top_k * 2F > the array's size, tested without forming the product (top_k and F
  // are not range-checked yet, so the product could overflow).  Other out-of-range
  // sizes are refused by the workspace entry point below.
  const bool top_k_ok = top_k >= 1 && top_k <= MEMRA_MAX_TOP_K;
  if (top_k_ok && F > MEMRA_MOE_NOALLOC_SCRATCH_FLOATS / (2 * top_k))
    return MEMRA_ERR_UNSUPPORTED;
  float* ws = nullptr;
  if (H > 0 && F > 0 && top_k_ok) {
    const memra_status st = memra::moe_scratch_address(&ws);
    if (st != MEMRA_OK) return st;
  }
  // Same checks and kernels as the workspace entry point.  Calls that return before
  // launching (empty or invalid sizes) never look at the workspace pointer.
  return memra_q8_0_moe_ffn(gu_q, gu_d, dn_q, dn_d, E, H, F, ids, gate_w, top_k, x, dtype, y,
                            ws, dev_status, stream);
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

extern "C" memra_status memra_debug_set_wait_test(int64_t wait_limit_cycles,
                                                  int64_t stall_after_stages) {
  if (stall_after_stages > INT32_MAX) return MEMRA_ERR_INVALID_ARG;
  memra::g_test_wait_limit.store(wait_limit_cycles > 0 ? wait_limit_cycles : 0);
  memra::g_test_stall_after.store(stall_after_stages >= 0 ? stall_after_stages : -1);
  return MEMRA_OK;
}
