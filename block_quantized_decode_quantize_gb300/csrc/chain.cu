// Chained decode GEMVs in one persistent launch: memra_q8_0_gemv_chain.
//
// A decode step is a chain of M = 1 products, each reading an activation that
// (in a model) depends on the products before it.  Launched one kernel per
// product, every launch pays a ramp (first weights in flight) and a drain (last
// rows computed while no new weights stream) of about 3 us on GB300.  Here one
// cooperative grid runs the whole chain:
//   - warp 0 of each CTA claims stages (a few consecutive rows of one step) from a
//     per-step counter, in step order, and streams their weight rows into a ring of
//     shared-memory stages with cp.async.bulk.  Weights do not depend on
//     activations, so the stream runs on across step boundaries.  With each stage
//     it writes, into shared memory, all the consumers need to know about the
//     stage's step;
//   - warps 1..12 compute whole rows of the stages (each row with the slices and
//     fp32 summation order of the single-product kernels, so every output is
//     bit-identical to memra_q8_0_quant_gemm of that step) and write y.  After a
//     CTA's last rows of a step, one thread adds their count to the step's
//     completion counter (a release reduction).  On their first stage of step i
//     the warps wait until the counters show every row of the earlier steps
//     written, then quantise x_i (q8_1, into shared memory).
// Claiming rows on demand keeps the CTAs' finishing times within about a stage of
// each other.  All waits are bounded (mbarriers and counters alike): on timeout the
// kernel raises a shared abort word that releases the other CTAs, lets its own
// copies land, reports through dev_status and returns.
#include <algorithm>

#include "common.cuh"
#include "product.cuh"

namespace memra {
namespace {

constexpr int kChainConsumers = 12;
constexpr int kChainThreads = 32 * (1 + kChainConsumers);
constexpr int kChainMaxStages = 8;
constexpr int kChainHeader = 1024;                     // barriers, abort flag, stage metadata
constexpr int kChainMetaOffset = 256;
constexpr size_t kChainStageTarget = 28 * 1024;
constexpr size_t kChainRingBudget = 88 * 1024;
constexpr size_t kChainSmemLimit = 113 * 1024;          // two CTAs per SM
constexpr long long kChainWaitCycles = 1ll << 31;       // about a second at 2 GHz

struct ChainParams {
  const memra_q8_0_step* steps;
  int n_steps;
  uint32_t slot_bytes;
  int ns;
  uint32_t off_x, off_xd, off_ring, off_slice;
  unsigned int* claim;  // [n_steps] rows claimed
  unsigned int* done;   // [n_steps] rows written
  unsigned int* abort;  // grid-wide abort word
  int32_t* status;
};

// A ring stage, written by the producer before the stage's copies are issued and
// read by the consumers once its full barrier completes: everything the consumers
// need about the stage's step, so that none of it is fetched from global memory
// while the weight stream keeps the memory system busy.
struct ChainMeta {
  float* y;             // the step's output at the stage's first row
  const void* x;        // the step's activation
  int K;
  int x_dtype;
  int nr;               // rows in the stage (0: no rows, only the end of the CTA's work)
  int step;             // -1: the CTA has no more stages
  int dep_step;         // last earlier step with rows (-1: none) ...
  unsigned int dep_rows;  // ... and its row count: x may be read once they are written
  int pub_step;         // before this stage: the CTA's rows of pub_step are complete
  unsigned int pub_rows;  // (0: nothing to publish)
};
static_assert(sizeof(ChainMeta) * kChainMaxStages + kChainMetaOffset <= kChainHeader,
              "stage metadata must fit the header");

// Rows per ring stage for a step of width K (same on host and device).
__host__ __device__ inline int chain_rows_per_stage(int64_t K) {
  const int64_t row = K + K / 16;
  const int64_t r = (int64_t)kChainStageTarget / row;
  return (int)(r < 1 ? 1 : r);
}

__host__ __device__ inline uint32_t chain_align(uint64_t v, uint64_t a) {
  return (uint32_t)((v + a - 1) / a * a);
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16 bytes from global memory through L2 only: activations may have been written
// during this launch by other SMs.
__device__ __forceinline__ uint4 ld_cg_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Wait (one thread) until step j's `need` rows are written.  Returns false if it
// gave up: the abort word was raised elsewhere, or the bounded wait ran out (then
// this thread raises it).
__device__ bool wait_rows(const ChainParams& p, int j, unsigned int need,
                          volatile int* abort_flag) {
  if (ld_acquire_u32(&p.done[j]) >= need) return true;
  const long long t0 = clock64();
  for (;;) {
    if (ld_acquire_u32(&p.done[j]) >= need) return true;
    if (*abort_flag || ld_acquire_u32(p.abort) != 0u) break;
    if (clock64() - t0 > kChainWaitCycles) {
      atomicExch(p.abort, 1u);
      break;
    }
    __nanosleep(20);
  }
  *abort_flag = 1;
  return false;
}

// Quantise one activation row of K values into the shared-memory q8_1 planes.  All
// consumer threads take part; each loads up to U groups of 8 values before
// quantising any, so a row of up to U * 8 * nthreads values costs one memory
// latency.  Thread t handles groups t, t + nthreads, ...; nthreads is a multiple of
// 4, so the four groups of a block sit in one lane quad.
template <bool BF16, int U>
__device__ __forceinline__ void chain_quantize_x(const void* xin, int K, int8_t* xs, float* xds,
                                                 int t, int nthreads) {
  const int groups = K / 8;
  for (int base = 0; base < groups; base += U * nthreads) {
    uint4 raw[U][BF16 ? 1 : 2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = base + u * nthreads + t;
      if (g < groups) {
        if (BF16) {
          raw[u][0] = ld_cg_16(static_cast<const uint16_t*>(xin) + (size_t)g * 8);
        } else {
          raw[u][0] = ld_cg_16(static_cast<const float*>(xin) + (size_t)g * 8);
          raw[u][BF16 ? 0 : 1] = ld_cg_16(static_cast<const float*>(xin) + (size_t)g * 8 + 4);
        }
      } else {
#pragma unroll
        for (int h = 0; h < (BF16 ? 1 : 2); ++h) raw[u][h] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = base + u * nthreads + t;
      if (base + u * nthreads >= groups) break;  // uniform across the CTA
      float v[8];
      if (BF16) {
        const uint32_t w[4] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[2 * i] = __uint_as_float(w[i] << 16);
          v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
      } else {
        const uint4 lo = raw[u][0], hi = raw[u][BF16 ? 0 : 1];
        v[0] = __uint_as_float(lo.x); v[1] = __uint_as_float(lo.y);
        v[2] = __uint_as_float(lo.z); v[3] = __uint_as_float(lo.w);
        v[4] = __uint_as_float(hi.x); v[5] = __uint_as_float(hi.y);
        v[6] = __uint_as_float(hi.z); v[7] = __uint_as_float(hi.w);
      }
      float d;
      const uint2 q = q8_1_group8(v, &d);
      if (g < groups) {
        *reinterpret_cast<uint2*>(xs + (size_t)g * 8) = q;
        if ((t & 3) == 0) xds[g >> 2] = d;
      }
    }
  }
}

__global__ void __launch_bounds__(kChainThreads, 2) q8_chain_kernel(const ChainParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  // full[8] | empty[8] | allin | go | xready, then the abort flag
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 8 * (2 * kChainMaxStages + 3));
  ChainMeta* meta = reinterpret_cast<ChainMeta*>(smem + kChainMetaOffset);
  int8_t* xs = reinterpret_cast<int8_t*>(smem + p.off_x);
  float* xds = reinterpret_cast<float*>(smem + p.off_xd);
  unsigned char* ring = smem + p.off_ring;
  int* s_slice = reinterpret_cast<int*>(smem + p.off_slice);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ns = p.ns;
  auto full_bar = [&](int i) { return smem_addr(bars + i); };
  auto empty_bar = [&](int i) { return smem_addr(bars + kChainMaxStages + i); };
  // allin: every consumer warp has written its rows of the CTA's last stage of a
  // step (one thread then publishes the step); go: the next step's inputs are
  // written (one thread checks); xready: every consumer warp has quantised its
  // share of that step's x.
  const uint32_t allin_bar = smem_addr(bars + 2 * kChainMaxStages);
  const uint32_t go_bar = smem_addr(bars + 2 * kChainMaxStages + 1);
  const uint32_t xready_bar = smem_addr(bars + 2 * kChainMaxStages + 2);

  if (threadIdx.x == 0) {
    for (int i = 0; i < ns; ++i) {
      mbar_init(full_bar(i), 1);
      mbar_init(empty_bar(i), kChainConsumers);
    }
    mbar_init(allin_bar, kChainConsumers);
    mbar_init(go_bar, 1);
    mbar_init(xready_bar, kChainConsumers);
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_evict_first_policy();
    uint32_t issued = 0;
    bool ok = true;
    // A free slot for stage `issued`: the consumers are done with the stage that
    // used it before.
    auto free_slot = [&]() -> bool {
      if (issued < (uint32_t)ns) return true;
      return mbar_wait(empty_bar(issued % ns), ((issued / ns) - 1) & 1, abort_flag);
    };
    // Claims (lane 0) run one stage ahead: the next claim is issued with the current
    // stage, so its latency overlaps the wait for a free slot.
    int cs = 0;                 // step being claimed
    unsigned int cr = 0;        // outstanding claim: first row
    memra_q8_0_step st{};
    int rps = 1;
    int dep_step = -1;          // last step before cs with rows
    unsigned int dep_rows = 0;
    unsigned int rows_here = 0;  // rows of cs this CTA has issued
    int pub_step = -1;
    unsigned int pub_rows = 0;
    auto begin_step = [&]() {
      st = p.steps[cs];
      rps = chain_rows_per_stage(st.K);
      cr = atomicAdd(&p.claim[cs], (unsigned int)rps);
      // One CTA warms L2 with the next step's activation while this one streams:
      // harmless if that activation is still being written (L2 is where writes
      // land), and it saves the consumers a trip to HBM behind the weight stream.
      if (cs + 1 < p.n_steps && blockIdx.x == (unsigned)((cs + 1) % (int)gridDim.x)) {
        const memra_q8_0_step nx = p.steps[cs + 1];
        if (nx.N > 0) prefetch_l2(nx.x, (uint32_t)(nx.K * (nx.x_dtype == MEMRA_BF16 ? 2 : 4)));
      }
    };
    if (lane == 0 && p.n_steps > 0) begin_step();
    for (;;) {
      if (!free_slot()) {
        ok = false;
        break;
      }
      const int slot = issued % ns;
      int have = 0;
      if (lane == 0) {
        // Resolve the outstanding claim, moving on while steps are exhausted.
        while (cs < p.n_steps) {
          if ((int64_t)cr < st.N) {
            have = 1;
            break;
          }
          if (rows_here > 0) {
            pub_step = cs;
            pub_rows = rows_here;
            rows_here = 0;
          }
          if (st.N > 0) {
            dep_step = cs;
            dep_rows = (unsigned int)st.N;
          }
          if (++cs < p.n_steps) begin_step();
        }
        ChainMeta m{};
        m.pub_step = pub_step;
        m.pub_rows = pub_rows;
        pub_rows = 0;
        if (have) {
          const int nb = (int)(st.K / 32);
          const int64_t r = cr;
          const int nr = (int)min((int64_t)rps, st.N - r);
          m.y = st.y + r;
          m.x = st.x;
          m.K = (int)st.K;
          m.x_dtype = st.x_dtype;
          m.nr = nr;
          m.step = cs;
          m.dep_step = dep_step;
          m.dep_rows = dep_rows;
          meta[slot] = m;
          const uint32_t wd_off = chain_align((uint64_t)rps * st.K, 128);
          const uint32_t qb = (uint32_t)(nr * st.K);
          const uint32_t db = (uint32_t)(nr * nb * 2);
          const uint32_t dst = smem_addr(ring + (size_t)slot * p.slot_bytes);
          mbar_arrive_expect_tx(full_bar(slot), qb + db);
          bulk_g2s_hint(dst, st.wq + r * st.K, qb, full_bar(slot), policy);
          bulk_g2s_hint(dst + wd_off, st.wd + r * nb, db, full_bar(slot), policy);
          rows_here += (unsigned int)nr;
          cr = atomicAdd(&p.claim[cs], (unsigned int)rps);
        } else {
          m.step = -1;  // the end marker (it may still carry a publication)
          meta[slot] = m;
          mbar_arrive(full_bar(slot));
        }
      }
      have = __shfl_sync(0xffffffffu, have, 0);
      __syncwarp();
      if (!have) break;
      ++issued;
    }
    if (!ok || *abort_flag) {
      // Let the copies already issued land (bounded) before the CTA can exit.
      *abort_flag = 1;
      const uint32_t first = issued > (uint32_t)ns ? issued - ns : 0;
      for (uint32_t j = first; j < issued; ++j) {
        const long long t0 = clock64();
        while (!mbar_try_wait(full_bar(j % ns), (j / ns) & 1) && clock64() - t0 < (1ll << 30)) {
        }
      }
      if (lane == 0) {
        atomicExch(p.abort, 1u);  // release the other CTAs from their waits
        if (p.status) atomicOr(p.status, 2);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int cw = warp - 1;
  const int ctid = threadIdx.x - 32;
  const int h1 = (lane >> 2) & 1;  // which half this lane loads first (bank-conflict free)
  uint32_t it = 0;
  uint32_t rbase = 0;  // rows in all earlier stages: deals rows round-robin over warps
  uint32_t phase = 0;   // steps this CTA has had rows in (parity of go and xready)
  uint32_t pphase = 0;  // steps this CTA has published (parity of allin)
  int cur = -1;
  int K = 0, nb = 0, cpr = 0, S = 0;
  uint32_t wd_off = 0;
  bool last_ok = false;
  for (;; ++it) {
    const int slot = it % ns;
    // Every warp waits for every stage, rows or not: an arrival on the stage's
    // empty barrier must never run ahead of the stage itself.
    if (!mbar_wait(full_bar(slot), (it / ns) & 1, abort_flag)) break;
    const ChainMeta mt = meta[slot];
    if (mt.pub_rows > 0) {
      // The CTA has no more rows of step pub_step, and every consumer warp is past
      // them: once all have arrived, one thread publishes the rows (a release, so
      // they are visible to whoever sees the count).
      if (lane == 0) mbar_arrive(allin_bar);
      if (ctid == 0 && mbar_wait(allin_bar, pphase & 1, abort_flag))
        red_release_add(&p.done[mt.pub_step], mt.pub_rows);
      ++pphase;
    }
    if (mt.step < 0) break;
    if (mt.step != cur) {
      // First stage of a step in this CTA.  x of that step may depend on every
      // output of the steps before it: one thread waits until the last earlier step
      // with rows is fully written (rows of a step are only computed once its
      // predecessors are, so that covers them all); then every consumer warp
      // quantises its share of the new x.  (All of them are done with the previous
      // x: they are all at this stage.)
      if (ctid == 0 && (mt.dep_step < 0 || wait_rows(p, mt.dep_step, mt.dep_rows, abort_flag)))
        mbar_arrive(go_bar);
      if (!mbar_wait(go_bar, phase & 1, abort_flag)) break;
      cur = mt.step;
      K = mt.K;
      nb = K / 32;
      cpr = (nb + 31) / 32;
      S = slices_for(cpr);
      wd_off = chain_align((uint64_t)chain_rows_per_stage(K) * K, 128);
      last_ok = lane < nb - (cpr - 1) * 32;
      if (mt.x_dtype == MEMRA_BF16)
        chain_quantize_x<true, 3>(mt.x, K, xs, xds, ctid, kChainConsumers * 32);
      else
        chain_quantize_x<false, 1>(mt.x, K, xs, xds, ctid, kChainConsumers * 32);
      fill_slice_table(s_slice, cpr, S, ctid, kChainConsumers * 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(xready_bar);
      if (!mbar_wait(xready_bar, phase & 1, abort_flag)) break;
      ++phase;
    }
    // Whole rows per warp: the slices of a row in order, each reduced across the
    // warp, then summed in slice order (the one summation order of a row).
    const int t0 = (int)((cw + kChainConsumers - (int)(rbase % kChainConsumers)) % kChainConsumers);
    rbase += mt.nr;
    const int8_t* ws = reinterpret_cast<const int8_t*>(ring + (size_t)slot * p.slot_bytes);
    const uint16_t* ds =
        reinterpret_cast<const uint16_t*>(ring + (size_t)slot * p.slot_bytes + wd_off);
    for (int row = t0; row < mt.nr; row += kChainConsumers) {
      float tot = 0.0f;
      for (int s = 0; s < S; ++s) {
        const int plo = s_slice[s];
        const int phi = s_slice[s + 1];
        const int8_t* wl = ws + row * K + (plo * 32 + lane) * 32 + h1 * 16;
        const uint16_t* dl = ds + row * nb + plo * 32 + lane;
        const int8_t* xl = xs + (plo * 32 + lane) * 32 + h1 * 16;
        const float* xdl = xds + plo * 32 + lane;
        float acc[1] = {0.0f};
        for (int pt = plo; pt < phi; ++pt) {
          const int q = pt - plo;
          if (pt < cpr - 1 || last_ok) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(wl + q * 1024);
            const uint4 w1 = *reinterpret_cast<const uint4*>(wl + q * 1024 + 16 - 32 * h1);
            const uint4 x0 = *reinterpret_cast<const uint4*>(xl + q * 1024);
            const uint4 x1 = *reinterpret_cast<const uint4*>(xl + q * 1024 + 16 - 32 * h1);
            const int sb = dot_halves(w0, w1, x0, x1);
            acc[0] = block_term_acc(acc[0], dl[q * 32], xdl[q * 32], sb);
          }
        }
        warp_sum_transposed<1>(acc, lane);
        tot = s == 0 ? acc[0] : __fadd_rn(tot, acc[0]);
      }
      if (lane == 0) mt.y[row] = tot;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(slot));
  }
  if (*abort_flag && ctid == 0) {
    atomicExch(p.abort, 1u);  // release the other CTAs from their waits
    if (p.status) atomicOr(p.status, 2);
  }
}

}  // namespace
}  // namespace memra

using namespace memra;

extern "C" size_t memra_q8_0_gemv_chain_sync_bytes(int32_t n_steps) {
  // claim[n_steps] | done[n_steps] | abort, rounded up to 16 bytes
  const size_t words = 2 * (size_t)(n_steps < 0 ? 0 : n_steps) + 1;
  return (words * sizeof(uint32_t) + 15) / 16 * 16;
}

extern "C" memra_status memra_q8_0_gemv_chain(const memra_q8_0_step* steps,
                                              const memra_q8_0_step* host_steps, int32_t n_steps,
                                              uint32_t* sync_words, int32_t* dev_status,
                                              cudaStream_t stream) {
  if (n_steps < 0) return MEMRA_ERR_INVALID_ARG;
  if (n_steps == 0) return MEMRA_OK;
  if (!steps || !host_steps || !sync_words) return MEMRA_ERR_INVALID_ARG;
  if (!aligned(steps, 16) || !aligned(sync_words, 16) || (dev_status && !aligned(dev_status, 4)))
    return MEMRA_ERR_ALIGNMENT;
  int64_t max_k = 0;
  size_t slot = 0;
  for (int32_t i = 0; i < n_steps; ++i) {
    const memra_q8_0_step& s = host_steps[i];
    if (s.N < 0 || s.K < 256 || s.K % 256 != 0) return MEMRA_ERR_INVALID_ARG;
    if (s.x_dtype != MEMRA_BF16 && s.x_dtype != MEMRA_F32) return MEMRA_ERR_INVALID_ARG;
    if (s.N > INT32_MAX / 2) return MEMRA_ERR_UNSUPPORTED;
    if (s.N > 0 && (!s.wq || !s.wd || !s.x || !s.y)) return MEMRA_ERR_INVALID_ARG;
    if (!s.x) return MEMRA_ERR_INVALID_ARG;
    if (!aligned(s.wq, 32) || !aligned(s.wd, 16) || !aligned(s.x, 16) || !aligned(s.y, 4))
      return MEMRA_ERR_ALIGNMENT;
    max_k = std::max(max_k, s.K);
    const int rps = chain_rows_per_stage(s.K);
    const size_t bytes = chain_align((uint64_t)rps * s.K, 128) +
                         chain_align((uint64_t)rps * (s.K / 16), 128);
    slot = std::max(slot, bytes);
  }
  if (max_k + max_k / 8 > MEMRA_MAX_X_BYTES) return MEMRA_ERR_UNSUPPORTED;
  DeviceInfo info;
  if (!device_info(&info)) return MEMRA_ERR_CUDA;
  ChainParams p{};
  p.steps = steps;
  p.n_steps = n_steps;
  p.slot_bytes = (uint32_t)slot;
  p.claim = sync_words;
  p.done = sync_words + n_steps;
  p.abort = sync_words + 2 * (size_t)n_steps;
  p.status = dev_status;
  const int max_cpr = (int)((max_k / 32 + 31) / 32);
  const size_t xbytes = chain_align(max_k, 128) + chain_align((max_k / 32) * 4, 128);
  const size_t fixed = kChainHeader + xbytes + chain_align((slices_for(max_cpr) + 1) * 4, 16);
  int ns = (int)std::min<size_t>(kChainMaxStages, std::max<size_t>(2, kChainRingBudget / slot));
  while (ns > 2 && fixed + ns * slot > kChainSmemLimit) --ns;
  const size_t smem = fixed + ns * slot;
  if (smem > (size_t)info.max_smem_optin) return MEMRA_ERR_UNSUPPORTED;
  p.ns = ns;
  size_t off = kChainHeader;
  p.off_x = (uint32_t)off;
  p.off_xd = (uint32_t)(off + chain_align(max_k, 128));
  off += xbytes;
  p.off_ring = (uint32_t)off;
  off += (size_t)ns * slot;
  p.off_slice = (uint32_t)off;
  // Every CTA must be resident at once (the grid barrier waits for all of them):
  // a cooperative launch of as many CTAs as fit, up to two per SM.
  cudaError_t e = allow_dynamic_smem(q8_chain_kernel, smem, info);
  if (e != cudaSuccess) return cuda_fail(e);
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q8_chain_kernel, kChainThreads,
                                                    smem);
  if (e != cudaSuccess) return cuda_fail(e);
  if (per_sm < 1) return MEMRA_ERR_UNSUPPORTED;
  const int grid = info.sms * std::min(per_sm, 2);
  e = cudaMemsetAsync(sync_words, 0, memra_q8_0_gemv_chain_sync_bytes(n_steps), stream);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kChainThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, q8_chain_kernel, p);
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}
