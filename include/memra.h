/*
 * memra.h -- C ABI of the GB300 (sm_103a) block-quantised decode library.
 *
 * The single-user decode step of an LLM streams block-quantised weights through
 * a fused dequantise matrix-vector (M = 1) or skinny matrix (M <= 16: speculative
 * verify, batched decode) product, plus a routed-expert (MoE) variant for one token
 * or a batch of tokens.  Weights come as Q8_0 (below), Q4_0 or NVFP4 (declared with
 * their entry points).  The memra pages name this path: Q8_0 decode through split-plane repacked matvecs with warp-level dp4a and
 * per-shape dispatch (memra wiki, github.com/avifenesh/memra/wiki, feature list);
 * one batched K+1 verify for MTP speculative decoding (same list); routed MoE
 * experts (same list); Q8_0 27B plain decode as a measured cell ("memra
 * performance", docs/PERFORMANCE.md, historical 27B board).  They print no block
 * layout or formula; the arithmetic stated here is GGUF's Q8_0 format as the
 * workloads define it.
 *
 * Formats (all row-major, "split-plane": quants and scales in separate arrays):
 *   Q8_0 weights   wq int8 [N][K] and wd fp16 (IEEE binary16 bits) [N][K/32].
 *                  Block b of row n covers k in [32b, 32b+32):
 *                  w[n][k] ~= float(wd[n][b]) * wq[n][k].
 *   q8_1 activation xq int8 [M][K] and xd fp32 [M][K/32]:
 *                  x[m][k] ~= xd[m][b] * xq[m][k].
 *   Quantisation of a block: amax = max|v|; weights d = fp16_rne(amax/127) and
 *   q = clamp(round_half_away(v / float(d)), -127, 127); activations d = amax/127
 *   in fp32 and q = clamp(round_half_away(v / d), -127, 127); amax = 0 gives
 *   d = 0 and q = 0.  Division is IEEE fp32 division.
 *   Product:       s_b = sum_{i<32} wq*xq (exact int32, |s_b| <= 516128) and
 *                  y[m][n] = sum_b (float(wd[n][b]) * xd[m][b]) * float(s_b) in fp32.
 *                  The int32 block sums are exact; the fp32 sum order is fixed by
 *                  the kernel (deterministic, no atomics) and a row's result does
 *                  not depend on M or on the other rows in the call.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers, allocated and owned by the caller.
 *     The library allocates nothing and keeps no state beyond a per-device cache
 *     of the SM count and shared-memory limit.
 *   - Work is enqueued on `stream` (0 = legacy default stream); no call
 *     synchronises.  Kernels may be launched with programmatic dependent launch,
 *     so a kernel may start streaming weights before the preceding kernel on the
 *     stream has finished; it reads activations, ids and gate weights and writes
 *     its outputs only after that kernel has completed.  Weights must therefore
 *     not be written by the immediately preceding kernel on the same stream.
 *   - Sizes are int64_t.  K must be a multiple of 32.  N, M, K may be 0 (an empty
 *     product writes zeros where an output row exists, nothing otherwise).
 *   - A violated precondition returns an error status and launches nothing.  A
 *     launch failure returns MEMRA_ERR_CUDA; memra_last_cuda_error() gives the
 *     cudaError_t of the calling thread's last failure.
 *   - Alignment: wq and wq_bank 32 bytes; xq, hq (outputs of the quantisers) and
 *     the quantiser inputs 16 bytes; wd 2 bytes; xd, y, ids, gate_w 4 bytes.  The
 *     4-bit formats' planes and their q8_1 inputs: 16 bytes.
 *   - Inputs must be finite.
 *
 * Run-time switches.  The defaults are the configurations measured best on GB300;
 * the environment variables below override them for benchmarking and tests.  Each is
 * read once per process, on the first call that needs it; a value that does not parse
 * keeps the default.  No result bit depends on them (every kernel computes the same
 * fp32 order), only the kernel choice and launch shapes.
 *   MEMRA_GEMV_PATH   "reg": dense Q8_0 products on the register-stream kernel;
 *                     "tma": on the bulk-copy kernel wherever it applies (also below
 *                     the size threshold); "mma": memra_q8_0_gemm_small_m on the
 *                     tensor-core kernel where it applies (as
 *                     memra_q8_0_gemm_small_m_mma).  Unset: per-shape dispatch.
 *   MEMRA_PDL         "0": launch without programmatic dependent launch.
 *   MEMRA_TMA_STAGE_KB, MEMRA_TMA_RING_KB, MEMRA_TMA_ROUTED_STAGE_KB,
 *   MEMRA_TMA_SMEM_LIMIT_KB, MEMRA_TMA_CTAS_PER_SM, MEMRA_TMA_PACKED_KB,
 *   MEMRA_TMA_MULTI_RING_KB, MEMRA_TMA_MULTI_STAGE_KB, MEMRA_TMA_MULTI,
 *   MEMRA_TMA_DENSE_MIN_MB, MEMRA_REG_CTAS_PER_SM
 *                     stage, ring and shared-memory sizes (KB), CTAs per SM, the
 *                     M > 1 bulk-copy switch and the register/bulk-copy size
 *                     threshold (MB) of the product kernels.
 *   MEMRA_TMA_PREFILL, MEMRA_TMA_ROUTED_PREFILL, MEMRA_TMA_PREFILL_4BIT
 *                     stages a dense (routed; dense M = 1 4-bit) product's producer
 *                     issues before its consumers have staged the activation (0: the
 *                     whole ring).
 * The same names, defined as macros when the library is compiled, change the
 * compiled-in defaults (also MEMRA_TMA_CONSUMER_WARPS,
 * MEMRA_TMA_FEW_M_CONSUMER_WARPS, MEMRA_TMA_MIN_BLOCKS, MEMRA_WAIT_SUSPEND_NS (the
 * suspend-time hint of a barrier wait's retries, ns), MEMRA_SLICE_PARTS; the last
 * changes the fp32 summation order and with it the result bits).
 */
#ifndef MEMRA_H
#define MEMRA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum memra_status {
  MEMRA_OK = 0,
  MEMRA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, K % 32 != 0, bad enum */
  MEMRA_ERR_ALIGNMENT = 2,     /* a pointer violates the alignment above */
  MEMRA_ERR_UNSUPPORTED = 3,   /* a size beyond the documented limits (M > 16, ...) */
  MEMRA_ERR_CUDA = 4           /* the CUDA runtime reported an error */
} memra_status;

typedef enum memra_dtype { MEMRA_BF16 = 0, MEMRA_F32 = 1 } memra_dtype;

/* Limits. */
#define MEMRA_MAX_M 16           /* activation rows per small-M call */
#define MEMRA_MAX_TOP_K 64       /* experts per routed call (per token) */
#define MEMRA_MAX_PAIRS 128      /* (token, slot) pairs per batched routed call */
/* Bytes of q8_1 activation a pass over the weights holds on chip: P*K*(1 + 4/32)
 * with P the rows of one pass (M up to 8, else ceil(M/2)). */
#define MEMRA_MAX_X_BYTES 196608

/*
 * Weight ingest: fp32 W [N][K] -> Q8_0 planes wq [N][K], wd [N][K/32].
 * The pages have memra repack checkpoints into its own internal layout (agentlens
 * summary of memra, "Design boundaries"); this is that repack for Q8_0 from fp32.
 * w: 16-byte aligned.  Bit-exact with the block definition above.
 */
memra_status memra_quantize_q8_0(const float* w, int64_t N, int64_t K, int8_t* wq, uint16_t* wd,
                                 cudaStream_t stream);

/*
 * Activation quantisation to int8 blocks with fp32 scales, the operand of the
 * dp4a block dot (memra wiki, feature list: warp-level dp4a).
 * x: [M][K] of `dtype` (MEMRA_BF16: uint16 bf16 bits, MEMRA_F32: float), 16-byte
 * aligned.  Outputs xq [M][K] (16-byte aligned), xd [M][K/32].
 * The block carries an fp32 scale and no sum term (Q8_0 weights have no offset).
 */
memra_status memra_quantize_q8_1(const void* x, int32_t dtype, int64_t M, int64_t K, int8_t* xq,
                                 float* xd, cudaStream_t stream);

/*
 * Plain decode GEMV (M = 1): y[n] = sum_b d_w[n][b] d_x[b] s_b[n].
 * memra wiki, feature list (Q8_0 split-plane dp4a matvec); memra performance,
 * historical 27B board (Q8_0 plain decode).  y: fp32 [N].
 */
memra_status memra_q8_0_gemv(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K,
                             const int8_t* xq, const float* xd, float* y, cudaStream_t stream);

/*
 * Speculative / MTP verify skinny GEMM and batched decode: M in [0, 16] activation
 * rows (memra wiki, feature list: one batched K+1 verify; memra performance,
 * "Serving performance": batched decode in 16-wide chunks on a kernel class whose
 * 16-batch results are bit-exact).  Up to 8 rows share one pass over the weights;
 * 9..16 rows take two passes, of ceil(M/2) and floor(M/2) rows.
 * xq [M][K], xd [M][K/32], y fp32 [M][N].  Row m of y equals, bit for bit, the
 * memra_q8_0_gemv result for activation row m, whatever M.
 */
memra_status memra_q8_0_gemm_small_m(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K,
                                     int64_t M, const int8_t* xq, const float* xd, float* y,
                                     cudaStream_t stream);

/*
 * memra_q8_0_gemm_small_m with the exact int32 block sums formed on the tensor cores
 * (one int8 mma.sync m16n8k32 per 32-element block of 16 weight rows and up to 8
 * activation rows) instead of dp4a.  The pages credit memra with an int8 tensor-core
 * GEMM (memra wiki, feature list); the workload definition allows tensor cores for the
 * verify GEMM only where they beat the CUDA-core path.  On GB300 they do not (the
 * int8 MMA rate equals the dp4a rate, and the kernel is latency-bound), so
 * memra_q8_0_gemm_small_m does not use this kernel; it is kept as an explicit entry
 * point for comparison.  The fp32 arithmetic around the block sums is the library's
 * one order, so y is bit-identical to memra_q8_0_gemm_small_m for every row.
 * Same arguments and results as memra_q8_0_gemm_small_m, with narrower support:
 * K a multiple of 1024 and at most 5120, N >= 16, wq, wd, xq, xd 16-byte aligned;
 * other shapes return MEMRA_ERR_UNSUPPORTED (misaligned pointers MEMRA_ERR_ALIGNMENT)
 * and launch nothing.  Empty sizes and K = 0 behave as in memra_q8_0_gemm_small_m.
 */
memra_status memra_q8_0_gemm_small_m_mma(const int8_t* wq, const uint16_t* wd, int64_t N,
                                         int64_t K, int64_t M, const int8_t* xq,
                                         const float* xd, float* y, cudaStream_t stream);

/*
 * Q4_0 weights, the pages' other split-plane decode format (memra wiki, feature
 * list, which names NVFP4, Q4_0 and Q8_0 decode through split-plane matvecs).  The
 * pages print nothing of it; this library's reading is GGUF's Q4_0 block: 32 consecutive
 * weights of a row share one fp16 scale d and carry 4-bit codes c in [0, 15] with
 * w ~= d * (c - 8).
 *   Planes: wq4 uint8 [N][K/2] and wd fp16 [N][K/32].  Byte j < 16 of a block holds
 *   element j's code in its low nibble and element j+16's in its high nibble.
 *   Quantisation: m = the element of largest |w| (the first one on a tie);
 *   d = fp16_rne(m / -8) (+0 for an all-zero block); c = clamp(round_half_away(
 *   w / float(d)) + 8, 0, 15).  w: fp32 [N][K], 16-byte aligned; wq4 16-byte aligned.
 */
memra_status memra_quantize_q4_0(const float* w, int64_t N, int64_t K, uint8_t* wq4, uint16_t* wd,
                                 cudaStream_t stream);

/*
 * NVFP4 weights, the pages' third split-plane decode format (memra wiki, feature
 * list; their safetensors loader reads NVIDIA ModelOpt NVFP4 checkpoints byte for
 * byte).  The pages print nothing of it; this library's reading is ModelOpt's NVFP4:
 * 16 consecutive weights of a row share one FP8 E4M3 scale s, each weight is an FP4
 * E2M1 code e (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 and a sign), and the tensor has
 * one fp32 scale g: w ~= g * s * e.
 *   Planes: codes uint8 [N][K/2], byte j holding element 2j in its low nibble and
 *   element 2j+1 in its high nibble; scales E4M3 bits uint8 [N][K/16].
 *   Quantisation: g = amax|W| / (6 * 448); s = e4m3(amax_block / (6 g)); e =
 *   e2m1(w / (float(s) g)), a block with s == 0 gets code 0; every conversion rounds
 *   to nearest, ties to even, saturating at 448 and 6; the code's sign is w's sign bit.
 * memra_quantize_nvfp4 writes g to device memory (*g, fp32); w 16-byte aligned,
 * codes 8-byte aligned.  It makes three launches and uses *g as its amax scratch.
 */
memra_status memra_quantize_nvfp4(const float* w, int64_t N, int64_t K, uint8_t* codes,
                                  uint8_t* scales, float* g, cudaStream_t stream);

/*
 * NVFP4 x q8_1 products (W4A8: every block sum exact in int32):
 *   y[m][n] = (g / 2) * sum_b [ (s_lo d_x[m][b]) S_lo + (s_hi d_x[m][b]) S_hi ],
 * S_lo, S_hi the sums of (twice the E2M1 value) * xq over elements 0..15 and 16..31
 * of activation block b, s_lo, s_hi their two E4M3 scales; the fp32 terms accumulate
 * in this library's one summation order, so a row does not depend on M.  g is the
 * tensor scale (host value).  M in [0, 16] (passes as memra_q8_0_gemm_small_m).  K a
 * multiple of 256 (MEMRA_ERR_UNSUPPORTED otherwise); codes, scales, xq, xd 16-byte
 * aligned.
 */
memra_status memra_nvfp4_gemm_small_m(const uint8_t* codes, const uint8_t* scales, float g,
                                      int64_t N, int64_t K, int64_t M, const int8_t* xq,
                                      const float* xd, float* y, cudaStream_t stream);

/* The decode GEMV on NVFP4 weights: memra_nvfp4_gemm_small_m with M = 1, y fp32 [N]. */
memra_status memra_nvfp4_gemv(const uint8_t* codes, const uint8_t* scales, float g, int64_t N,
                              int64_t K, const int8_t* xq, const float* xd, float* y,
                              cudaStream_t stream);

/*
 * Repack from GGUF's interleaved block arrays into the split planes (memra wiki,
 * feature list: decode runs on split-plane repacked weights).  The pages print no
 * block layout; the reading is GGUF's:
 *   Q8_0 block, 34 bytes: fp16 scale (little-endian), then 32 int8 quants;
 *   Q4_0 block, 18 bytes: fp16 scale (little-endian), then 16 bytes, byte j holding
 *   element j's code in its low nibble and element j+16's in its high nibble (the
 *   same byte layout as this library's Q4_0 plane).
 * blocks: N * K/32 blocks, row after row (device memory, 2-byte aligned).  Outputs:
 * wq int8 [N][K] or wq4 uint8 [N][K/2] (16-byte aligned) and wd fp16 bits [N][K/32]
 * (2-byte aligned), all allocated by the caller.  Byte for byte: no value changes.
 * Errors: K % 32 != 0 or a null pointer -> MEMRA_ERR_INVALID_ARG; misaligned
 * pointers -> MEMRA_ERR_ALIGNMENT; N * K/32 * block bytes beyond int64 ->
 * MEMRA_ERR_UNSUPPORTED.  N == 0 or K == 0 launches nothing.
 */
memra_status memra_repack_q8_0(const void* blocks, int64_t N, int64_t K, int8_t* wq,
                               uint16_t* wd, cudaStream_t stream);
memra_status memra_repack_q4_0(const void* blocks, int64_t N, int64_t K, uint8_t* wq4,
                               uint16_t* wd, cudaStream_t stream);

/*
 * Q4_0 x q8_1 products: y[m][n] = sum_b (d_w[n][b] * d_x[m][b]) * s_b with the exact
 * int32 block sum s_b = sum_i (c_i - 8) * xq_i, in the same fp32 summation order as
 * the Q8_0 products (so the result equals the Q8_0 product of the unpacked codes,
 * bit for bit).  M in [0, 16], in passes as for memra_q8_0_gemm_small_m; xq [M][K],
 * xd [M][K/32], y fp32 [M][N].
 * K must be a multiple of 256 (MEMRA_ERR_UNSUPPORTED otherwise); wq4, wd, xq and xd
 * 16-byte aligned.  The 4-bit formats stream through shared memory only: a pass whose
 * activation rows and two weight rows do not fit a CTA's shared memory (at M = 1, K
 * above about 96,000) returns MEMRA_ERR_UNSUPPORTED.
 */
memra_status memra_q4_0_gemm_small_m(const uint8_t* wq4, const uint16_t* wd, int64_t N, int64_t K,
                                     int64_t M, const int8_t* xq, const float* xd, float* y,
                                     cudaStream_t stream);

/* The decode GEMV on Q4_0 weights: memra_q4_0_gemm_small_m with M = 1, y fp32 [N]. */
memra_status memra_q4_0_gemv(const uint8_t* wq4, const uint16_t* wd, int64_t N, int64_t K,
                             const int8_t* xq, const float* xd, float* y, cudaStream_t stream);

/*
 * The verify GEMM (or, with M = 1, the decode GEMV) with the activation's q8_1
 * quantisation done in the kernel's prologue: each CTA quantises x [M][K] (bf16
 * bits or fp32, 16-byte aligned) into on-chip memory while the weight stream is
 * already in flight, instead of a separate memra_quantize_q8_1 launch.  This is
 * the pages' m=1 fusion chain applied to the quantise-then-matvec pair (memra
 * performance, "Serving performance": the B=1 decode path that keeps the m=1
 * fusion chain).  Bit-identical to
 * memra_quantize_q8_1 followed by memra_q8_0_gemm_small_m.  y fp32 [M][N].
 */
memra_status memra_q8_0_quant_gemm(const int8_t* wq, const uint16_t* wd, int64_t N, int64_t K,
                                   int64_t M, const void* x, int32_t dtype, float* y,
                                   cudaStream_t stream);

/*
 * Routed-expert GEMV for one token (memra wiki, feature list: MoE routed experts).
 * Bank: wq_bank [E][N][K], wd_bank [E][N][K/32] (expert e's planes are the slices
 * at e*N*K and e*N*(K/32)).  ids: device int32 [top_k]; gate_w: device fp32
 * [top_k] or NULL.  x_per_expert = 0: one shared activation xq [K], xd [K/32];
 * x_per_expert = 1: row k of xq [top_k][K], xd [top_k][K/32] feeds expert k.
 *   gate_w == NULL: y fp32 [top_k][N], row k = W_{ids[k]} x_k.
 *   gate_w != NULL: y fp32 [N] = sum_k gate_w[k] * (W_{ids[k]} x_k), k ascending.
 * An id outside [0, E) is detected on the device: that expert is skipped (its
 * ungated row is written as zeros; it adds nothing to the gated sum) and, if
 * dev_status is not NULL, the int32 word *dev_status is OR-ed with 1.  The word is
 * never cleared by the library.  E >= 1 and 1 <= top_k <= MEMRA_MAX_TOP_K.  With
 * K = 0 the outputs are zero-filled and the ids are not examined.
 */
memra_status memra_q8_0_moe_gemv(const int8_t* wq_bank, const uint16_t* wd_bank, int64_t E,
                                 int64_t N, int64_t K, const int32_t* ids, const float* gate_w,
                                 int64_t top_k, const int8_t* xq, const float* xd,
                                 int32_t x_per_expert, float* y, int32_t* dev_status,
                                 cudaStream_t stream);

/*
 * memra_q8_0_moe_gemv on a Q4_0 expert bank (the pages credit wide loads of Q4_0
 * expert weights for part of their MoE margins: memra performance, docs/
 * PERFORMANCE.md, Gemma-4 QAT Q4_0 board; memra wiki, the same board): wq4_bank uint8 [E][N][K/2]
 * packed as memra_quantize_q4_0 packs a weight matrix, wd_bank fp16 [E][N][K/32].
 * Same arguments, outputs, id handling and dev_status as memra_q8_0_moe_gemv; the
 * block sums are those of memra_q4_0_gemm_small_m.  K must be a multiple of 256
 * (MEMRA_ERR_UNSUPPORTED otherwise); wq4_bank, wd_bank, xq and xd 16-byte aligned.
 */
memra_status memra_q4_0_moe_gemv(const uint8_t* wq4_bank, const uint16_t* wd_bank, int64_t E,
                                 int64_t N, int64_t K, const int32_t* ids, const float* gate_w,
                                 int64_t top_k, const int8_t* xq, const float* xd,
                                 int32_t x_per_expert, float* y, int32_t* dev_status,
                                 cudaStream_t stream);

/*
 * SwiGLU between the routed gate/up and down projections, followed by q8_1
 * quantisation (the MoE FFN's activation; the pages put the routed experts in the
 * qwen/silu MoE class: memra performance, "Shipped on the sm_90a build").  The
 * gate/up split below is this library's reading.  gu: fp32 [R][2F], gate in
 * columns [0, F), up in [F, 2F); F % 32 == 0.  h = (g / (1 + exp(-g))) * u with
 * each fp32 operation rounded once in that order and exp computed by Cody-Waite
 * reduction (ln 2 = 0.693359375 + -2.12194440e-4, k = rint(x*log2(e)), argument
 * clamped to [-87, 88]) and the degree-7 Taylor polynomial in Horner form; then
 * hq [R][F], hd [R][F/32] as memra_quantize_q8_1.
 */
memra_status memra_swiglu_quantize_q8_1(const float* gu, int64_t R, int64_t F, int8_t* hq,
                                        float* hd, cudaStream_t stream);

/*
 * One routed-expert FFN layer for one token, in two kernels:
 *   y = sum_k gate_w[k] * W_dn[ids[k]] q8_1( swiglu( W_gu[ids[k]] q8_1(x) ) ).
 * The gate|up product quantises x in its prologue and streams each expert's gate row
 * j together with its up row j, so that its epilogue computes h_j = silu(g_j) u_j once
 * per row (the arithmetic of memra_swiglu_quantize_q8_1); the down product quantises
 * the h rows to q8_1 in its prologue.  Bit-identical to memra_quantize_q8_1,
 * memra_q8_0_moe_gemv (no gate weights, shared x), memra_swiglu_quantize_q8_1 and
 * memra_q8_0_moe_gemv (gate weights, x per expert) run in sequence.
 *   gu_q [E][2F][H], gu_d [E][2F][H/32]: gate rows [0, F), up rows [F, 2F).
 *   dn_q [E][H][F], dn_d [E][H][F/32].  x [H] (dtype bf16 bits or fp32, 16-byte
 *   aligned).  ids, gate_w [top_k] (device).  y fp32 [H].
 *   workspace: caller-allocated device fp32 [top_k][2F], 16-byte aligned.  After the
 *   call row k holds [h (F floats) | up (F floats)] of slot k, h = silu(gate) * up.
 *   (Shapes the bulk-copy kernel does not take, K % 256 != 0 or planes not 16-byte
 *   aligned, run unpaired: row k then holds [gate | up] and the down product computes
 *   SwiGLU in its prologue; the result y is the same.)
 * Bad ids behave as in memra_q8_0_moe_gemv.  H % 32 == 0, F % 32 == 0.
 */
memra_status memra_q8_0_moe_ffn(const int8_t* gu_q, const uint16_t* gu_d, const int8_t* dn_q,
                                const uint16_t* dn_d, int64_t E, int64_t H, int64_t F,
                                const int32_t* ids, const float* gate_w, int64_t top_k,
                                const void* x, int32_t dtype, float* y, float* workspace,
                                int32_t* dev_status, cudaStream_t stream);

/*
 * Routed experts for a batch of T tokens (the pages' expert-major MoE batching,
 * memra wiki, feature list; here for speculative verify or batched decode of
 * routed layers).  Token t routes ids[t][0..top_k) with gates gate_w[t][..].
 * Every (token, slot) pair is computed with the single-token arithmetic, and pairs
 * that route to the same expert stream its rows at the same time, so the expert's
 * weights come from HBM once and from L2 after (not a guarantee: a timing effect).
 *   ids: device int32 [T][top_k]; gate_w: device fp32 [T][top_k] or NULL.
 *   x_per_expert == 0: xq [T][K], xd [T][K/32], one row per token;
 *   x_per_expert == 1: xq [T][top_k][K], xd [T][top_k][K/32], one row per pair.
 *   gate_w == NULL: y fp32 [T][top_k][N], y[t][k] = W[ids[t][k]] x; workspace unused.
 *   gate_w given:   y fp32 [T][N], y[t] = sum_k gate_w[t][k] y[t][k] in ascending k;
 *                   workspace: caller-allocated fp32 [T][top_k][N] (4-byte aligned),
 *                   which keeps the per-pair rows after the call.
 * Row t of the result equals, bit for bit, memra_q8_0_moe_gemv on token t alone.
 * Limits: top_k <= MEMRA_MAX_TOP_K, T * top_k <= MEMRA_MAX_PAIRS, and the
 * activation rows (T, or T * top_k per pair) within MEMRA_MAX_X_BYTES.  Bad ids,
 * alignment and dev_status as memra_q8_0_moe_gemv.  T == 0 or N == 0 launches nothing.
 */
memra_status memra_q8_0_moe_gemv_tokens(const int8_t* wq_bank, const uint16_t* wd_bank, int64_t E,
                                        int64_t N, int64_t K, const int32_t* ids,
                                        const float* gate_w, int64_t T, int64_t top_k,
                                        const int8_t* xq, const float* xd, int32_t x_per_expert,
                                        float* y, float* workspace, int32_t* dev_status,
                                        cudaStream_t stream);

/* memra_q8_0_moe_gemv_tokens on a Q4_0 expert bank (layout and limits as
 * memra_q4_0_moe_gemv). */
memra_status memra_q4_0_moe_gemv_tokens(const uint8_t* wq4_bank, const uint16_t* wd_bank,
                                        int64_t E, int64_t N, int64_t K, const int32_t* ids,
                                        const float* gate_w, int64_t T, int64_t top_k,
                                        const int8_t* xq, const float* xd, int32_t x_per_expert,
                                        float* y, float* workspace, int32_t* dev_status,
                                        cudaStream_t stream);

/*
 * Routed experts on an NVFP4 bank: codes_bank uint8 [E][N][K/2] and scales_bank E4M3
 * bits [E][N][K/16] as memra_quantize_nvfp4 lays out one matrix, and gexp: fp32 [E]
 * (device), each expert's tensor scale (ModelOpt stores one per expert).  Slot k's
 * output is expert ids[k]'s memra_nvfp4_gemv result, bit for bit; the rest (gated
 * sum, ids, outputs, dev_status) as memra_q8_0_moe_gemv.  K a multiple of 256;
 * banks, xq, xd 16-byte aligned, gexp 4-byte aligned.
 */
memra_status memra_nvfp4_moe_gemv(const uint8_t* codes_bank, const uint8_t* scales_bank,
                                  const float* gexp, int64_t E, int64_t N, int64_t K,
                                  const int32_t* ids, const float* gate_w, int64_t top_k,
                                  const int8_t* xq, const float* xd, int32_t x_per_expert,
                                  float* y, int32_t* dev_status, cudaStream_t stream);

/* memra_q8_0_moe_gemv_tokens on an NVFP4 bank (layout as memra_nvfp4_moe_gemv). */
memra_status memra_nvfp4_moe_gemv_tokens(const uint8_t* codes_bank, const uint8_t* scales_bank,
                                         const float* gexp, int64_t E, int64_t N, int64_t K,
                                         const int32_t* ids, const float* gate_w, int64_t T,
                                         int64_t top_k, const int8_t* xq, const float* xd,
                                         int32_t x_per_expert, float* y, float* workspace,
                                         int32_t* dev_status, cudaStream_t stream);

/*
 * memra_q8_0_moe_ffn for a batch of T tokens, in three kernels: gate|up of every
 * (token, slot) pair with each token's row quantised in the prologue, down of every
 * pair with its SwiGLU + q8_1 in the prologue, and the gated sum per token.
 *   x [T][H] (bf16 bits or fp32, 16-byte aligned); ids, gate_w [T][top_k]; y fp32 [T][H].
 *   workspace: caller-allocated device fp32 [T * top_k * (2F + H)], 16-byte aligned:
 *   the pairs' gate|up rows [T][top_k][2F], then their down rows [T][top_k][H].
 * Row t of y equals, bit for bit, memra_q8_0_moe_ffn on token t alone.  Limits as
 * memra_q8_0_moe_gemv_tokens (x: T rows of H; h: T * top_k rows of F).
 */
memra_status memra_q8_0_moe_ffn_tokens(const int8_t* gu_q, const uint16_t* gu_d,
                                       const int8_t* dn_q, const uint16_t* dn_d, int64_t E,
                                       int64_t H, int64_t F, const int32_t* ids,
                                       const float* gate_w, int64_t T, int64_t top_k,
                                       const void* x, int32_t dtype, float* y, float* workspace,
                                       int32_t* dev_status, cudaStream_t stream);

/*
 * memra_q8_0_moe_ffn and memra_q8_0_moe_ffn_tokens on Q4_0 banks (gu_q4 uint8
 * [E][2F][H/2], gu_d fp16 [E][2F][H/32], dn_q4 uint8 [E][H][F/2], dn_d fp16
 * [E][H][F/32], packed as memra_quantize_q4_0 packs a matrix) and on NVFP4 banks
 * (codes uint8 [E][rows][K/2], E4M3 scales uint8 [E][rows][K/16], and each bank's
 * per-expert tensor scales gu_g, dn_g: fp32 [E], device).  Same arithmetic, outputs,
 * workspace and id handling as the Q8_0 entry points, with the block sums of the
 * format's products; each token's output is bit-identical to the format's routed
 * GEMVs (gate|up ungated, SwiGLU + q8_1, down gated) run in sequence.  H and F must be
 * multiples of 256 (MEMRA_ERR_UNSUPPORTED otherwise); banks 16-byte aligned.
 */
memra_status memra_q4_0_moe_ffn(const uint8_t* gu_q4, const uint16_t* gu_d, const uint8_t* dn_q4,
                                const uint16_t* dn_d, int64_t E, int64_t H, int64_t F,
                                const int32_t* ids, const float* gate_w, int64_t top_k,
                                const void* x, int32_t dtype, float* y, float* workspace,
                                int32_t* dev_status, cudaStream_t stream);
memra_status memra_nvfp4_moe_ffn(const uint8_t* gu_codes, const uint8_t* gu_scales,
                                 const float* gu_g, const uint8_t* dn_codes,
                                 const uint8_t* dn_scales, const float* dn_g, int64_t E,
                                 int64_t H, int64_t F, const int32_t* ids, const float* gate_w,
                                 int64_t top_k, const void* x, int32_t dtype, float* y,
                                 float* workspace, int32_t* dev_status, cudaStream_t stream);
memra_status memra_q4_0_moe_ffn_tokens(const uint8_t* gu_q4, const uint16_t* gu_d,
                                       const uint8_t* dn_q4, const uint16_t* dn_d, int64_t E,
                                       int64_t H, int64_t F, const int32_t* ids,
                                       const float* gate_w, int64_t T, int64_t top_k,
                                       const void* x, int32_t dtype, float* y, float* workspace,
                                       int32_t* dev_status, cudaStream_t stream);
memra_status memra_nvfp4_moe_ffn_tokens(const uint8_t* gu_codes, const uint8_t* gu_scales,
                                        const float* gu_g, const uint8_t* dn_codes,
                                        const uint8_t* dn_scales, const float* dn_g, int64_t E,
                                        int64_t H, int64_t F, const int32_t* ids,
                                        const float* gate_w, int64_t T, int64_t top_k,
                                        const void* x, int32_t dtype, float* y, float* workspace,
                                        int32_t* dev_status, cudaStream_t stream);

/*
 * memra_q8_0_moe_ffn without caller memory.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory when they call
 * -- code running under a fixed memory arena or budget, plug-ins and embedded
 * runtimes that are handed device pointers but no allocator, and real-time decode
 * loops that must not pay for (or risk failing) an allocation per layer.  It takes
 * the same arguments minus `workspace` and returns bit-identical results.
 *
 * The gate|up outputs go to a fixed array of MEMRA_MOE_NOALLOC_SCRATCH_FLOATS
 * floats (256 KB) inside the library, which every GPU that loads the library holds
 * until the process exits.  Calls whose top_k * 2F exceeds that size return
 * MEMRA_ERR_UNSUPPORTED and launch nothing.  The call itself allocates nothing
 * (no cudaMalloc, no library allocation).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before
 *     any stream capture on the device.
 *   - That address is kept for the life of the process.  A cudaDeviceReset destroys
 *     the context that holds the array, so after one this entry point must not be
 *     called again in the same process (it would write to the old address).
 *   - Every call shares the one array.  Calls that may overlap on the GPU (on
 *     different streams, or before an earlier one has finished on another stream)
 *     race on it; keep such calls on one stream.  The array keeps the last call's
 *     workspace rows; nothing in it needs clearing because each call writes every
 *     element it later reads.
 */
#define MEMRA_MOE_NOALLOC_SCRATCH_FLOATS 65536
memra_status memra_q8_0_moe_ffn_noalloc(const int8_t* gu_q, const uint16_t* gu_d,
                                        const int8_t* dn_q, const uint16_t* dn_d, int64_t E,
                                        int64_t H, int64_t F, const int32_t* ids,
                                        const float* gate_w, int64_t top_k, const void* x,
                                        int32_t dtype, float* y, int32_t* dev_status,
                                        cudaStream_t stream);

/*
 * Exact int32 block sums s[m][n][b] = sum_{i<32} wq[n][32b+i] * xq[m][32b+i],
 * computed with the same dp4a block-dot routine as the product kernels.  For
 * verification of the integer stage.  s: int32 [M][N][K/32], 4-byte aligned.
 */
memra_status memra_q8_0_block_dots(const int8_t* wq, int64_t N, int64_t K, const int8_t* xq,
                                   int64_t M, int32_t* s, cudaStream_t stream);

/*
 * Diagnostic, not part of the decode path: read `bytes` of device memory once (every
 * 16-byte word, streaming loads) with sms * ctas_per_sm CTAs of 512 threads, and fold
 * them into sink[blockIdx]: sink is uint32 [sms * ctas_per_sm] (sms = the device's
 * multiprocessor count), xor-accumulated, so the caller zeroes it to compare runs.  Timing it gives the read-only stream ceiling that the weight-
 * streaming products approach.  bytes % 16 == 0; buf 16-byte aligned; ctas_per_sm in
 * [1, 4].
 */
memra_status memra_read_stream(const void* buf, int64_t bytes, uint32_t* sink,
                               int32_t ctas_per_sm, cudaStream_t stream);

/*
 * Test hook for the device-side failure handling; the pages have no counterpart.  The
 * bulk-copy product kernel bounds every wait on its shared-memory barriers (about a
 * second of SM cycles by default): when a wait runs out, the CTA raises an abort flag
 * that releases its other warps, lets the copies it issued land, writes NaN into the
 * outputs it owns, ORs 2 into *dev_status (routed entry points, when given) and
 * returns; nothing traps.  This hook lets a test make those waits run out without a
 * fault: launches made after it, in this process, give up waiting after
 * wait_limit_cycles SM cycles (<= 0: the default), and, with stall_after_stages >= 0,
 * each CTA's producer stops after that many stages and leaves one more stage that no
 * copy completes.  Set both off again (0, -1) for normal operation.  Launches already
 * enqueued or captured in a CUDA graph keep the settings they were made with; calls
 * made from several host threads at once see whichever setting was current.
 */
memra_status memra_debug_set_wait_test(int64_t wait_limit_cycles, int64_t stall_after_stages);

/* Static text for a status code. */
const char* memra_status_string(memra_status status);

/* The cudaError_t (as int) of the calling thread's last MEMRA_ERR_CUDA, else 0. */
int32_t memra_last_cuda_error(void);

/* Library version string. */
const char* memra_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MEMRA_H */
