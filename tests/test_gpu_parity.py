"""GPU parity: the sm_103a library against the CPU oracle, through the C ABI.

Integer stages (quantised weights and activations, block sums) must match bit for
bit; fp32 outputs within |y - y_ref| <= 1e-4 * sum_b |d_w d_x s_b| + 1e-6.  Each
side runs its own pipeline from the same seeded fp32/bf16 inputs: the oracle never
sees a value the GPU produced.
"""
import numpy as np
import pytest
import torch

import synth
from _util import Guarded, abs_terms, assert_within, bf16_bits_np, np_, wd_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_decode_quantize_gb300 as m
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    m.lib()
    return m


def gpu_weights(mem, w_cpu):
    wq, wd = mem.memra_quantize_q8_0(w_cpu.cuda())
    return wq, wd


def check_weights(orc, w_cpu, wq, wd):
    oq, od = orc.quantize_q8_0(np_(w_cpu))
    assert np.array_equal(np_(wq), oq)
    assert np.array_equal(wd_bits(wd), od)
    return oq, od


def check_acts(orc, x_cpu, xq, xd):
    if x_cpu.dtype == torch.bfloat16:
        oq, od = orc.quantize_q8_1(bf16_bits_np(x_cpu))
    else:
        oq, od = orc.quantize_q8_1(np_(x_cpu))
    assert np.array_equal(np_(xq), oq)
    assert np.array_equal(np_(xd).view(np.uint32), od.view(np.uint32))
    return oq, od


# ----------------------------------------------------------------------------
# Quantisers and block sums: bit-exact.
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("N,K,seed", [(37, 96, 1), (4096, 4096, 0), (3, 17408, 2)])
def test_quantize_q8_0_bit_exact(mem, orc, N, K, seed):
    w = synth.weights_fp32(N, K, seed, 0)
    wq, wd = gpu_weights(mem, w)
    check_weights(orc, w, wq, wd)


def test_quantize_q8_0_special_blocks(mem, orc):
    w = synth.weights_fp32(64, 512, 7, 1)
    synth.perturb_blocks(w, 7, 2, zero_frac=0.05, scale_frac=0.05, scale=50.0)
    w[3, :32] = torch.tensor(1.4 * 2 ** -24 * 127)       # subnormal fp16 scale, clamped quants
    w[3, 1] = -w[3, 0] / 2
    w[4, :32] = 0.0
    w[5, 32:64] = torch.linspace(-127.0, 127.0, 32)       # d = 1 exactly, ties at .5 steps
    w[6, 64:96] = 300.0 * torch.randn(32)                # scale far above the others
    wq, wd = gpu_weights(mem, w)
    check_weights(orc, w, wq, wd)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (8, 17408), (5, 5120)])
def test_quantize_q8_1_bit_exact(mem, orc, dtype, M, K):
    x = synth.activations_fp32(M, K, 11, M, K, outlier_frac=0.001).to(dtype)
    if K >= 64:
        x[0, 32:64] = 0.0                                # all-zero block
        x[0, :32] = torch.tensor([127.0, 63.5, -63.5, 2.5, -2.5, 0.5, -0.5, 1.5] * 4)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    check_acts(orc, x, xq, xd)


def test_block_dots_bit_exact(mem, orc):
    g = torch.Generator().manual_seed(5)
    N, K, M = 50, 1184, 3
    wq = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int8)
    xq = torch.randint(-127, 128, (M, K), generator=g, dtype=torch.int8)
    wq[0, :32] = -127
    xq[0, :32] = -127
    s = mem.memra_q8_0_block_dots(wq.cuda(), xq.cuda())
    ref = orc.block_dots(np_(wq), np_(xq))
    assert np.array_equal(np_(s), ref)
    assert int(ref[0, 0, 0]) == 32 * 127 * 127


# ----------------------------------------------------------------------------
# GEMV and the verify skinny GEMM.
# ----------------------------------------------------------------------------

def run_pair(mem, orc, N, K, M, seed, x_dtype=torch.bfloat16, outliers=0.001):
    w = synth.weights_fp32(N, K, seed, 100)
    x = synth.activations_fp32(M, K, seed, 200, outlier_frac=outliers).to(x_dtype)
    wq, wd = gpu_weights(mem, w)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oq, od = check_weights(orc, w, wq, wd)
    oxq, oxd = check_acts(orc, x, xq, xd)
    return (wq, wd, xq, xd), (oq, od, oxq, oxd)


@pytest.mark.parametrize("N,K", [(1003, 1184), (257, 17408), (4096, 4096), (64, 32),
                                 (130, 768), (1, 5120), (1000, 3072), (40, 2048)])
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_gemm_parity(mem, orc, N, K, M):
    (wq, wd, xq, xd), (oq, od, oxq, oxd) = run_pair(mem, orc, N, K, M, seed=N * 31 + K + M)
    y = Guarded((M, N), torch.float32)
    if M == 1:
        mem.memra_q8_0_gemv(wq, wd, xq[0], xd[0], y=y.view[0])
    else:
        mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd, y=y.view)
    torch.cuda.synchronize()
    assert y.intact()
    y_ref = orc.gemm(oq, od, oxq, oxd)
    terms = abs_terms(orc.block_dots(oq, oxq), od, oxd)
    assert_within(np_(y.view), y_ref, terms, "gemm N=%d K=%d M=%d" % (N, K, M))


@pytest.mark.parametrize("N,K", [(4096, 4096), (1000, 3072), (40, 2048), (777, 5120),
                                 (17, 1024), (16, 2048)])
@pytest.mark.parametrize("M", [1, 2, 5, 8, 11, 16])
def test_tensor_core_gemm_parity(mem, orc, N, K, M):
    """The tensor-core entry point: against the oracle, and bit for bit the CUDA-core
    product (every row, one and two weight passes; tiles of 16 rows moved back at the
    end of a CTA's rows, N = 16 and 17 included)."""
    (wq, wd, xq, xd), (oq, od, oxq, oxd) = run_pair(mem, orc, N, K, M, seed=N * 7 + K + M)
    y = Guarded((M, N), torch.float32)
    mem.memra_q8_0_gemm_small_m_mma(wq, wd, xq, xd, y=y.view)
    ref = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)
    torch.cuda.synchronize()
    assert y.intact()
    assert_within(np_(y.view), orc.gemm(oq, od, oxq, oxd),
                  abs_terms(orc.block_dots(oq, oxq), od, oxd), "mma N=%d K=%d M=%d" % (N, K, M))
    assert torch.equal(y.view.view(torch.int32), ref.view(torch.int32))


@pytest.mark.parametrize("N,K", [(4096, 17408), (15, 1024), (100, 1056)])
def test_tensor_core_gemm_refuses_other_shapes(mem, N, K):
    wq = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    wd = torch.zeros((N, K // 32), dtype=torch.float16, device="cuda")
    xq = torch.zeros((2, K), dtype=torch.int8, device="cuda")
    xd = torch.zeros((2, K // 32), dtype=torch.float32, device="cuda")
    y = torch.full((2, N), 5.0, device="cuda")
    with pytest.raises(mem.MemraError) as e:
        mem.memra_q8_0_gemm_small_m_mma(wq, wd, xq, xd, y=y)
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert bool((y == 5.0).all())


def test_rows_do_not_depend_on_m(mem, orc):
    N, K = 777, 5120
    (wq, wd, xq, xd), _ = run_pair(mem, orc, N, K, 8, seed=9)
    y8 = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)
    for m in range(8):
        y1 = mem.memra_q8_0_gemv(wq, wd, xq[m], xd[m])
        assert torch.equal(y1.view(torch.int32), y8[m].view(torch.int32)), m
    for M in (2, 3, 5):
        yM = mem.memra_q8_0_gemm_small_m(wq, wd, xq[:M].contiguous(), xd[:M].contiguous())
        assert torch.equal(yM.view(torch.int32), y8[:M].view(torch.int32)), M


@pytest.mark.parametrize("N,K", [(1003, 1184), (257, 17408), (4096, 4096), (130, 768)])
@pytest.mark.parametrize("M", [9, 12, 16])
def test_batched_decode_parity(mem, orc, N, K, M):
    """M = 9..16 rows (two passes over the weights): against the oracle, and every row
    bit for bit the M = 1 product of that row."""
    (wq, wd, xq, xd), (oq, od, oxq, oxd) = run_pair(mem, orc, N, K, M, seed=N * 17 + K + M)
    y = Guarded((M, N), torch.float32)
    mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd, y=y.view)
    torch.cuda.synchronize()
    assert y.intact()
    assert_within(np_(y.view), orc.gemm(oq, od, oxq, oxd),
                  abs_terms(orc.block_dots(oq, oxq), od, oxd), "batch N=%d K=%d M=%d" % (N, K, M))
    for m in range(M):
        y1 = mem.memra_q8_0_gemv(wq, wd, xq[m], xd[m])
        assert torch.equal(y1.view(torch.int32), y.view[m].view(torch.int32)), m


def test_batched_decode_limits(mem):
    K = 17408
    wq = torch.zeros((64, K), dtype=torch.int8, device="cuda")
    wd = torch.zeros((64, K // 32), dtype=torch.float16, device="cuda")
    xq = torch.zeros((17, K), dtype=torch.int8, device="cuda")
    xd = torch.zeros((17, K // 32), dtype=torch.float32, device="cuda")
    with pytest.raises(mem.MemraError) as e:
        mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)        # M = 17
    assert e.value.status == 3
    y = mem.memra_q8_0_gemm_small_m(wq, wd, xq[:16], xd[:16])  # two passes of 8 rows
    torch.cuda.synchronize()
    assert not y.any()


def test_deterministic_repeat(mem, orc):
    (wq, wd, xq, xd), _ = run_pair(mem, orc, 2048, 5120, 4, seed=3)
    a = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)
    b = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_zero_and_scaled_blocks(mem, orc):
    N, K = 300, 2048
    w = synth.weights_fp32(N, K, 4, 4)
    synth.perturb_blocks(w, 4, 5, zero_frac=0.01, scale_frac=0.01, scale=50.0)
    w[17] = 0.0
    x = synth.activations_bf16(8, K, 4, 6)
    wq, wd = gpu_weights(mem, w)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oq, od = check_weights(orc, w, wq, wd)
    oxq, oxd = check_acts(orc, x, xq, xd)
    y = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)
    y_ref = orc.gemm(oq, od, oxq, oxd)
    assert_within(np_(y), y_ref, abs_terms(orc.block_dots(oq, oxq), od, oxd), "perturbed")
    assert torch.all(y[:, 17] == 0)


# ----------------------------------------------------------------------------
# Routed experts.
# ----------------------------------------------------------------------------

def make_bank(mem, E, N, K, seed):
    w = torch.stack([synth.weights_fp32(N, K, seed, 300, e) for e in range(E)])
    wq, wd = mem.memra_quantize_q8_0(w.view(E * N, K).cuda())
    return w, wq.view(E, N, K), wd.view(E, N, K // 32)


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("per_expert", [False, True])
def test_moe_gemv_parity(mem, orc, gated, per_expert):
    E, N, K, top_k = 12, 200, 768, 8
    w, wq, wd = make_bank(mem, E, N, K, 21)
    oq, od = orc.quantize_q8_0(np_(w).reshape(E * N, K))
    assert np.array_equal(np_(wq).reshape(E * N, K), oq)
    oq = oq.reshape(E, N, K)
    od = od.reshape(E, N, K // 32)
    ids, gw = synth.routing(E, top_k, 22, int(gated), int(per_expert))
    x = synth.activations_bf16(top_k if per_expert else 1, K, 23)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oxq, oxd = check_acts(orc, x, xq, xd)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    xq_in, xd_in = (xq, xd) if per_expert else (xq[0], xd[0])
    y = mem.memra_q8_0_moe_gemv(wq, wd, ids.cuda(), gw.cuda() if gated else None, xq_in, xd_in,
                                per_expert, dev_status=status)
    y_ref, bad = orc.moe_gemv(oq, od, np_(ids), np_(gw) if gated else None,
                              oxq if per_expert else oxq[:1], oxd if per_expert else oxd[:1],
                              int(per_expert))
    assert bad == 0 and int(status.item()) == 0
    terms = np.zeros((top_k, N))
    for k, e in enumerate(np_(ids)):
        xr = k if per_expert else 0
        terms[k] = abs_terms(orc.block_dots(oq[e], oxq[xr:xr + 1]), od[e], oxd[xr:xr + 1])[0]
    if gated:
        terms = (np.abs(np_(gw))[:, None] * terms).sum(axis=0)
    assert_within(np_(y), y_ref, terms, "moe gated=%s per_expert=%s" % (gated, per_expert))


def test_moe_bad_ids_flagged_and_skipped(mem, orc):
    E, N, K = 4, 64, 256
    w, wq, wd = make_bank(mem, E, N, K, 31)
    oq, od = orc.quantize_q8_0(np_(w).reshape(E * N, K))
    oq = oq.reshape(E, N, K)
    od = od.reshape(E, N, K // 32)
    x = synth.activations_bf16(1, K, 32)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oxq, oxd = check_acts(orc, x, xq, xd)
    ids = torch.tensor([2, 7, -3], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mem.memra_q8_0_moe_gemv(wq, wd, ids.cuda(), None, xq[0], xd[0], False, dev_status=status)
    assert int(status.item()) == 1
    assert torch.all(y[1] == 0) and torch.all(y[2] == 0)
    y_ref, bad = orc.moe_gemv(oq, od, np_(ids), None, oxq, oxd, 0)
    assert bad == 2
    terms = abs_terms(orc.block_dots(oq[2], oxq), od[2], oxd)[0]
    assert_within(np_(y[0]), y_ref[0], terms, "moe bad ids")
    status.zero_()
    gw = torch.tensor([0.5, 0.25, 0.25], dtype=torch.float32)
    yg = mem.memra_q8_0_moe_gemv(wq, wd, ids.cuda(), gw.cuda(), xq[0], xd[0], False,
                                 dev_status=status)
    assert int(status.item()) == 1
    yg_ref, _ = orc.moe_gemv(oq, od, np_(ids), np_(gw), oxq, oxd, 0)
    assert_within(np_(yg), yg_ref, 0.5 * terms, "moe bad ids gated")


def test_moe_gated_packed_stage_with_bad_ids(mem, orc):
    """Gated routed products pack all of a CTA's expert segments into one ring stage.
    Here each CTA owns several rows per segment, one id in the middle is out of range
    and one is negative (both skipped), and a second call has no valid id at all (its
    stage carries no bytes; the output must be exact zeros)."""
    E, N, K = 8, 1000, 512
    w, wq, wd = make_bank(mem, E, N, K, 41)
    oq, od = orc.quantize_q8_0(np_(w).reshape(E * N, K))
    oq = oq.reshape(E, N, K)
    od = od.reshape(E, N, K // 32)
    x = synth.activations_bf16(5, K, 42)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oxq, oxd = check_acts(orc, x, xq, xd)
    ids = torch.tensor([3, -1, 5, 99, 0], dtype=torch.int32)
    gw = torch.tensor([0.3, 0.1, 0.25, 0.15, 0.2], dtype=torch.float32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mem.memra_q8_0_moe_gemv(wq, wd, ids.cuda(), gw.cuda(), xq, xd, True, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    y_ref, bad = orc.moe_gemv(oq, od, np_(ids), np_(gw), oxq, oxd, 1)
    assert bad == 2
    terms = np.zeros(N)
    for k, e in enumerate(np_(ids)):
        if 0 <= e < E:
            t = abs_terms(orc.block_dots(oq[e], oxq[k:k + 1]), od[e], oxd[k:k + 1])[0]
            terms += abs(float(gw[k])) * t
    assert_within(np_(y), y_ref, terms, "gated packed stage, bad ids")
    bad_ids = torch.tensor([-4, 8, 1 << 20], dtype=torch.int32, device="cuda")
    status.zero_()
    y0 = mem.memra_q8_0_moe_gemv(wq, wd, bad_ids, gw[:3].contiguous().cuda(), xq[:3].contiguous(),
                                 xd[:3].contiguous(), True, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert torch.all(y0 == 0)


@pytest.mark.parametrize("R,F", [(8, 768), (1, 32), (3, 2048)])
def test_swiglu_quantize_bit_exact(mem, orc, R, F):
    gu = synth.normal((R, 2 * F), 41, R, F, std=3.0)
    gu[0, :6] = torch.tensor([0.0, -30.0, 30.0, -95.0, 95.0, 1e-3])
    hq, hd = mem.memra_swiglu_quantize_q8_1(gu.cuda())
    oq, od = orc.swiglu_quantize_q8_1(np_(gu))
    assert np.array_equal(np_(hq), oq)
    assert np.array_equal(np_(hd).view(np.uint32), od.view(np.uint32))


def test_moe_ffn_layer_composition(mem, orc):
    """One routed FFN layer: quantise x, gate/up experts, SwiGLU + quantise, down experts
    with gate weights.  The GPU's fp32 gate/up outputs differ from the oracle's in the
    last bits, so h may quantise one step differently; the bound allows one h quantum
    per element on top of the stated product tolerance."""
    E, H, F, top_k = 16, 2048, 768, 8
    wgu, gq, gd = make_bank(mem, E, 2 * F, H, 51)
    wdn, dq, dd = make_bank(mem, E, H, F, 52)
    ogq, ogd = orc.quantize_q8_0(np_(wgu).reshape(-1, H))
    odq, odd = orc.quantize_q8_0(np_(wdn).reshape(-1, F))
    ogq, ogd = ogq.reshape(E, 2 * F, H), ogd.reshape(E, 2 * F, H // 32)
    odq, odd = odq.reshape(E, H, F), odd.reshape(E, H, F // 32)
    ids, gw = synth.routing(E, top_k, 53)
    x = synth.normal((H,), 54)
    xq, xd = mem.memra_quantize_q8_1(x.cuda()[None])
    ygu = mem.memra_q8_0_moe_gemv(gq, gd, ids.cuda(), None, xq[0], xd[0], False)
    hq, hd = mem.memra_swiglu_quantize_q8_1(ygu)
    y = mem.memra_q8_0_moe_gemv(dq, dd, ids.cuda(), gw.cuda(), hq, hd, True)
    y_ref, bad = orc.moe_ffn(np_(x), ogq, ogd, odq, odd, np_(ids), np_(gw))
    assert bad == 0
    # one quantum of h per element: sum_k w_k sum_f |W_dn[n, f]| * hd_k[f/32]
    _, ohd = orc.swiglu_quantize_q8_1(orc.moe_gemv(ogq, ogd, np_(ids), None,
                                                   *orc.quantize_q8_1(np_(x)[None]), 0)[0])
    bound = np.zeros(H)
    for k, e in enumerate(np_(ids)):
        wabs = np.abs(odq[e].astype(np.float64) *
                      np.repeat(odd[e].view(np.float16).astype(np.float64), 32, axis=1))
        bound += gw[k].item() * (wabs @ np.repeat(2.0 * ohd[k].astype(np.float64), 32))
    err = np.abs(np_(y).astype(np.float64) - y_ref)
    assert np.all(err <= bound + 1e-4 * np.abs(y_ref).max() + 1e-6)


# ----------------------------------------------------------------------------
# Edge cases and errors.
# ----------------------------------------------------------------------------

def test_empty_and_degenerate_sizes(mem, orc):
    dev = "cuda"
    wq = torch.zeros((5, 0), dtype=torch.int8, device=dev)
    wd = torch.zeros((5, 0), dtype=torch.float16, device=dev)
    xq = torch.zeros((2, 0), dtype=torch.int8, device=dev)
    xd = torch.zeros((2, 0), dtype=torch.float32, device=dev)
    y = torch.full((2, 5), 7.0, device=dev)
    mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd, y=y)       # K = 0: empty sums
    assert torch.all(y == 0)
    y0 = mem.memra_q8_0_gemm_small_m(torch.zeros((0, 64), dtype=torch.int8, device=dev),
                                     torch.zeros((0, 2), dtype=torch.float16, device=dev),
                                     torch.zeros((3, 64), dtype=torch.int8, device=dev),
                                     torch.zeros((3, 2), dtype=torch.float32, device=dev))
    assert y0.shape == (3, 0)
    # N = 1, K = 32: one block
    (wq, wd, xq, xd), (oq, od, oxq, oxd) = run_pair(mem, orc, 1, 32, 1, seed=61)
    y = mem.memra_q8_0_gemv(wq, wd, xq[0], xd[0])
    assert_within(np_(y)[None], orc.gemm(oq, od, oxq, oxd),
                  abs_terms(orc.block_dots(oq, oxq), od, oxd), "1x32")
    # all-zero activation: every output exactly zero
    z = torch.zeros((1, 4096), dtype=torch.bfloat16, device=dev)
    zq, zd = mem.memra_quantize_q8_1(z)
    assert torch.all(zd == 0) and torch.all(zq == 0)


def test_misaligned_views_are_rejected(mem):
    dev = "cuda"
    N, K = 64, 256
    base = torch.zeros(N * K + 16, dtype=torch.int8, device=dev)
    wq_bad = base[16:16 + N * K].view(N, K)             # 16-byte aligned, not 32
    wd = torch.zeros((N, K // 32), dtype=torch.float16, device=dev)
    xq = torch.zeros((1, K), dtype=torch.int8, device=dev)
    xd = torch.zeros((1, K // 32), dtype=torch.float32, device=dev)
    y = torch.full((1, N), 3.0, device=dev)
    with pytest.raises(mem.MemraError) as ei:
        mem.memra_q8_0_gemm_small_m(wq_bad, wd, xq, xd, y=y)
    assert ei.value.status == 2
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)                          # nothing launched
    with pytest.raises(mem.MemraError) as ei:
        mem.memra_q8_0_gemm_small_m(torch.zeros((N, K), dtype=torch.int8, device=dev), wd,
                                    torch.zeros((17, K), dtype=torch.int8, device=dev),
                                    torch.zeros((17, K // 32), dtype=torch.float32, device=dev))
    assert ei.value.status == 3                         # M > 16


# ----------------------------------------------------------------------------
# Quantisation fused into the product's prologue.
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("N,K,M", [(1003, 1184, 1), (4096, 4096, 1), (257, 17408, 1),
                                   (513, 5120, 3), (130, 768, 8), (64, 32, 2), (300, 5120, 13)])
def test_fused_quant_gemm_matches_two_step(mem, orc, dtype, N, K, M):
    w = synth.weights_fp32(N, K, 80, N, K)
    x = synth.activations_fp32(M, K, 81, N, K, M, outlier_frac=0.001).to(dtype).cuda()
    wq, wd = mem.memra_quantize_q8_0(w.cuda())
    xq, xd = mem.memra_quantize_q8_1(x)
    y2 = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)
    y = Guarded((M, N), torch.float32)
    mem.memra_q8_0_quant_gemm(wq, wd, x, y=y.view)
    torch.cuda.synchronize()
    assert y.intact()
    assert torch.equal(y.view.view(torch.int32), y2.view(torch.int32))
    # and against the oracle's own pipeline
    oq, od = orc.quantize_q8_0(np_(w))
    xo = bf16_bits_np(x.cpu()) if dtype == torch.bfloat16 else np_(x)
    oxq, oxd = orc.quantize_q8_1(xo)
    assert_within(np_(y.view), orc.gemm(oq, od, oxq, oxd),
                  abs_terms(orc.block_dots(oq, oxq), od, oxd), "fused N=%d K=%d M=%d" % (N, K, M))


@pytest.mark.parametrize("scale", [0.1, 1.0 / 3.0, 7.77e-3, 3.3e4])
def test_quantizers_near_rounding_boundaries(mem, orc, scale):
    """Values within +-3e-5 (and just outside 1e-4) of k + 1/2 quanta, where a
    quotient computed by reciprocal could round differently from the IEEE one."""
    rng = np.random.default_rng(int(scale * 1e6) % 1000)
    d = np.float32(scale)
    blocks = []
    for eps in (-2e-4, -3e-5, -1e-6, 0.0, 1e-6, 3e-5, 2e-4):
        k = rng.integers(-126, 126, size=31)
        v = ((k + 0.5 + eps) * np.float64(d)).astype(np.float32)
        blocks.append(np.concatenate([[np.float32(127.0) * d], v]))   # max sets d = 127*d/127
    x = np.stack(blocks).astype(np.float32).reshape(1, -1)
    xt = torch.from_numpy(x).cuda()
    xq, xd = mem.memra_quantize_q8_1(xt)
    oq, od = orc.quantize_q8_1(x)
    assert np.array_equal(np_(xq), oq)
    assert np.array_equal(np_(xd).view(np.uint32), od.view(np.uint32))
    # the fused product quantises the same way
    wq, wd = mem.memra_quantize_q8_0(torch.from_numpy(x).repeat(3, 1).cuda())
    y1 = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)
    y2 = mem.memra_q8_0_quant_gemm(wq, wd, xt)
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    # weights: fp16 scales, same construction
    owq, owd = orc.quantize_q8_0(np.repeat(x, 3, axis=0))
    assert np.array_equal(np_(wq), owq)
    assert np.array_equal(wd_bits(wd), owd)



@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("E,H,F,top_k", [(16, 2048, 768, 8), (5, 256, 96, 3), (3, 512, 32, 1)])
def test_moe_ffn_matches_four_step_pipeline(mem, orc, dtype, E, H, F, top_k):
    """The two-kernel FFN entry point against the four calls it fuses (bit for bit),
    and against the oracle's layer."""
    _, gq, gd = make_bank(mem, E, 2 * F, H, 90 + H)
    _, dq, dd = make_bank(mem, E, H, F, 91 + F)
    ids, gw = synth.routing(E, top_k, 92, E, H)
    ids, gw = ids.cuda(), gw.cuda()
    x = synth.normal((H,), 93, H).to(dtype).cuda()
    st1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.full((top_k, 2 * F), 5.0, device="cuda")
    y = mem.memra_q8_0_moe_ffn(gq, gd, dq, dd, ids, gw, x, workspace=ws, dev_status=st1)
    xq, xd = mem.memra_quantize_q8_1(x[None])
    ygu = mem.memra_q8_0_moe_gemv(gq, gd, ids, None, xq[0], xd[0], False)
    hq, hd = mem.memra_swiglu_quantize_q8_1(ygu)
    y4 = mem.memra_q8_0_moe_gemv(dq, dd, ids, gw, hq, hd, True)
    torch.cuda.synchronize()
    assert int(st1.item()) == 0
    # the workspace keeps each slot's [silu(gate) up | up]: the up rows are the routed
    # GEMV's bit for bit, the SwiGLU rows the oracle's SwiGLU of the same gate|up bits
    assert torch.equal(ws[:, F:].contiguous().view(torch.int32),
                       ygu[:, F:].contiguous().view(torch.int32))
    h_ref = orc.swiglu(np_(ygu))
    assert np.array_equal(np_(ws[:, :F]).view(np.uint32), h_ref.view(np.uint32))
    assert torch.equal(y.view(torch.int32), y4.view(torch.int32))
    xo = bf16_bits_np(x.cpu()) if dtype == torch.bfloat16 else np_(x)
    oxq, oxd = orc.quantize_q8_1(xo[None])
    assert np.array_equal(np_(xq), oxq)
    ygu_ref, _ = orc.moe_gemv(np_(gq), wd_bits(gd), np_(ids), None, oxq, oxd, 0)
    ohq, ohd = orc.swiglu_quantize_q8_1(ygu_ref)
    y_ref, bad = orc.moe_gemv(np_(dq), wd_bits(dd), np_(ids), np_(gw), ohq, ohd, 1)
    assert bad == 0
    err = np.abs(np_(y).astype(np.float64) - y_ref)
    assert np.all(err <= 0.02 * np.abs(y_ref).max() + 1e-5)


def test_moe_ffn_bad_ids(mem):
    E, H, F = 4, 256, 64
    _, gq, gd = make_bank(mem, E, 2 * F, H, 94)
    _, dq, dd = make_bank(mem, E, H, F, 95)
    ids = torch.tensor([1, 9], dtype=torch.int32, device="cuda")
    gw = torch.tensor([0.6, 0.4], device="cuda")
    x = synth.normal((H,), 96).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mem.memra_q8_0_moe_ffn(gq, gd, dq, dd, ids, gw, x, dev_status=st)
    y1 = mem.memra_q8_0_moe_ffn(gq, gd, dq, dd, ids[:1].contiguous(), gw[:1].contiguous(), x)
    torch.cuda.synchronize()
    assert int(st.item()) == 1
    assert torch.equal(y.view(torch.int32), y1.view(torch.int32))


def test_activation_at_the_size_limit(mem, orc):
    """M = 1 with K = 174752, the largest multiple of 32 whose q8_1 activation fits
    MEMRA_MAX_X_BYTES (K + K/8 <= 196608): parity; one block more is refused."""
    K = 174752
    assert K + K // 8 <= 196608 < (K + 32) + (K + 32) // 8
    (wq, wd, xq, xd), (oq, od, oxq, oxd) = run_pair(mem, orc, 40, K, 1, seed=97)
    y = Guarded((1, 40), torch.float32)
    mem.memra_q8_0_gemv(wq, wd, xq[0], xd[0], y=y.view[0])
    torch.cuda.synchronize()
    assert y.intact()
    assert_within(np_(y.view), orc.gemm(oq, od, oxq, oxd),
                  abs_terms(orc.block_dots(oq, oxq), od, oxd), "K at the limit")
    K2 = K + 32
    with pytest.raises(mem.MemraError) as e:
        mem.memra_q8_0_gemv(torch.zeros((4, K2), dtype=torch.int8, device="cuda"),
                            torch.zeros((4, K2 // 32), dtype=torch.float16, device="cuda"),
                            torch.zeros((K2,), dtype=torch.int8, device="cuda"),
                            torch.zeros((K2 // 32,), dtype=torch.float32, device="cuda"))
    assert e.value.status == 3


def test_four_bit_rows_beyond_shared_memory_are_refused(mem):
    """The 4-bit formats stream through shared memory only: a row of K = 131072 with its
    activation cannot fit a CTA, and the call returns MEMRA_ERR_UNSUPPORTED."""
    K = 131072
    wq4 = torch.zeros((8, K // 2), dtype=torch.uint8, device="cuda")
    xq = torch.zeros((1, K), dtype=torch.int8, device="cuda")
    xd = torch.zeros((1, K // 32), dtype=torch.float32, device="cuda")
    with pytest.raises(mem.MemraError) as e:
        mem.memra_q4_0_gemm_small_m(wq4, torch.zeros((8, K // 32), dtype=torch.float16,
                                                     device="cuda"), xq, xd)
    assert e.value.status == 3
    with pytest.raises(mem.MemraError) as e:
        mem.memra_nvfp4_gemm_small_m(wq4, torch.zeros((8, K // 16), dtype=torch.uint8,
                                                      device="cuda"), 1.0, xq, xd)
    assert e.value.status == 3
