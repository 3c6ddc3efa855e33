"""GPU parity for NVFP4 weights, through the C ABI.

The weight ingest must match the oracle bit for bit (codes, E4M3 scales and the tensor
scale).  Products must match the oracle within |y - y_ref| <= 1e-4 * sum |term| + 1e-6,
with one term per 16-element half-block, |(g/2) s d_x S|, twice over: against the
oracle's fp32 product (exact half-block sums, the scale terms in block order), and
against the plain definition summed element by element in fp64, sum_e g s e2m1 d_x q_x,
which shares no grouping with the kernel.  Each row must equal, bit for bit, the M = 1
product of that row.  Each side runs its own pipeline from the same seeded inputs.
"""
import json
import os

import numpy as np
import pytest
import torch

import synth
from _util import Guarded, assert_within, bf16_bits_np, np_, nvfp4_terms

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def mem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_decode_quantize_gb300 as m
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    m.lib()
    return m


def check_nvfp4_weights(orc, mem, w_cpu):
    codes, scales, g = mem.memra_quantize_nvfp4(w_cpu.cuda())
    torch.cuda.synchronize()
    oc, os_, og = orc.quantize_nvfp4(np_(w_cpu))
    assert np_(g)[0].view(np.uint32) == np.float32(og).view(np.uint32)
    assert np.array_equal(np_(scales), os_)
    assert np.array_equal(np_(codes), oc)
    return codes, scales, float(np_(g)[0]), oc, os_, og


@pytest.mark.parametrize("N,K,seed,std", [(37, 96, 1, 0.02), (4096, 4096, 0, 0.02),
                                          (3, 17408, 2, 1.0), (64, 1024, 3, 300.0)])
def test_quantize_nvfp4_bit_exact(mem, orc, N, K, seed, std):
    w = synth.weights_fp32(N, K, seed, 600, std=std)
    check_nvfp4_weights(orc, mem, w)


def test_quantize_nvfp4_special_values(mem, orc):
    with open(os.path.join(GOLDEN, "nvfp4_hand_row.json")) as f:
        hand = json.load(f)
    w = synth.weights_fp32(8, 256, 9, 601, std=0.3)
    w[0, :64] = torch.tensor(hand["w"])                 # every E2M1 tie, -0, amax 2688
    w[1, 0:16] = 0.0                                    # a zero block
    w[2, 16:32] = -0.0                                  # negative zeros
    w[3, 32:48] = 1e-30                                 # a block whose scale underflows
    w[4, 48:64] = -0.03                                 # scale 0.03/6 -> E4M3 subnormal 3 * 2^-9
    codes, scales, g, *_ = check_nvfp4_weights(orc, mem, w)
    assert g == 1.0
    assert np_(scales)[1, 0] == 0 and np_(scales)[3, 2] == 0
    zero = np.zeros((1, 4096), np.float32)
    check_nvfp4_weights(orc, mem, torch.from_numpy(zero))  # all zero: g = 0


@pytest.mark.parametrize("N,K,M", [(1003, 4096, 1), (777, 5120, 1), (300, 5120, 8),
                                   (64, 17408, 1), (130, 17408, 8), (12289, 4096, 2),
                                   (5120, 17408, 1), (513, 2048, 4), (1, 256, 3),
                                   (700, 5120, 16), (129, 17408, 11)])
def test_nvfp4_gemm_parity(mem, orc, N, K, M):
    seed = N * 29 + K + M
    w = synth.weights_fp32(N, K, seed, 602)
    x = synth.activations_fp32(M, K, seed, 603, outlier_frac=0.001).to(torch.bfloat16)
    codes, scales, g, oc, os_, og = check_nvfp4_weights(orc, mem, w)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x))
    assert np.array_equal(np_(xq), oxq)
    y = Guarded((M, N), torch.float32)
    if M == 1:
        mem.memra_nvfp4_gemv(codes, scales, g, xq[0], xd[0], y=y.view[0])
    else:
        mem.memra_nvfp4_gemm_small_m(codes, scales, g, xq, xd, y=y.view)
    torch.cuda.synchronize()
    assert y.intact()
    y_ref = orc.gemm_nvfp4(oc, os_, og, oxq, oxd)
    terms = nvfp4_terms(orc, oc, os_, og, oxq, oxd)
    assert_within(np_(y.view), y_ref, terms, "nvfp4 N=%d K=%d M=%d" % (N, K, M))
    y64 = orc.nvfp4_dequant_gemm_f64(oc, os_, og, oxq, oxd)
    assert_within(np_(y.view), y64, terms, "nvfp4 vs element-order fp64 N=%d K=%d M=%d" % (N, K, M))
    for m in sorted({0, M - 1}):
        y1 = mem.memra_nvfp4_gemv(codes, scales, g, xq[m], xd[m])
        torch.cuda.synchronize()
        assert torch.equal(y.view[m].view(torch.int32), y1.view(torch.int32)), m


def test_nvfp4_hand_row_through_the_product(mem, orc):
    """The hand-worked row and activation: y = 342120 exactly (every term is exact)."""
    with open(os.path.join(GOLDEN, "nvfp4_hand_row.json")) as f:
        hand = json.load(f)
    K = 256
    w = torch.zeros((2, K))
    w[0, :64] = torch.tensor(hand["w"])
    x = torch.zeros((1, K))
    x[0, :64] = torch.tensor(hand["x"])
    codes, scales, g, *_ = check_nvfp4_weights(orc, mem, w)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    y = mem.memra_nvfp4_gemv(codes, scales, g, xq[0], xd[0])
    torch.cuda.synchronize()
    assert float(y[0]) == hand["y"] and float(y[1]) == 0.0


def test_nvfp4_rejects_k_not_multiple_of_256(mem):
    codes = torch.zeros((4, 48), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((4, 6), dtype=torch.uint8, device="cuda")
    xq = torch.zeros((1, 96), dtype=torch.int8, device="cuda")
    xd = torch.zeros((1, 3), dtype=torch.float32, device="cuda")
    with pytest.raises(mem.MemraError) as e:
        mem.memra_nvfp4_gemm_small_m(codes, scales, 1.0, xq, xd)
    assert e.value.status == 3


def nvfp4_bank(mem, E, N, K, seed, orc=None):
    """Each expert quantised on its own (its own tensor scale), stacked into a bank.  With
    the oracle given, each expert's GPU ingest is checked bit for bit against the oracle's
    quantisation of the same fp32 weights, and the oracle's bank is returned as well."""
    ws = [synth.weights_fp32(N, K, seed, e, std=0.01 * (1 + e % 3)) for e in range(E)]
    if orc is not None:
        parts = [check_nvfp4_weights(orc, mem, w) for w in ws]
        obank = (np.stack([p[3] for p in parts]), np.stack([p[4] for p in parts]),
                 np.array([p[5] for p in parts], np.float32))
        parts = [(p[0], p[1], torch.tensor([p[2]], dtype=torch.float32, device="cuda"))
                 for p in parts]
    else:
        parts = [mem.memra_quantize_nvfp4(w.cuda()) for w in ws]
    codes = torch.stack([c for c, _, _ in parts])
    scales = torch.stack([s for _, s, _ in parts])
    gexp = torch.cat([g for _, _, g in parts])
    if orc is not None:
        return codes, scales, gexp, obank
    return codes, scales, gexp


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("per_expert", [False, True])
def test_nvfp4_moe_gemv_parity(mem, orc, gated, per_expert):
    E, N, K, top_k = 10, 200, 1024, 8
    codes, scales, gexp, (oc, os_, og) = nvfp4_bank(mem, E, N, K, 610, orc)
    ids = torch.tensor([3, 9, 0, 7, 3, 5, 12, 1], dtype=torch.int32)   # 12 is out of range
    gw = torch.tensor([0.2, 0.15, 0.1, 0.1, 0.15, 0.1, 0.1, 0.1], dtype=torch.float32)
    x = synth.activations_bf16(top_k if per_expert else 1, K, 611)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    xq_in, xd_in = (xq, xd) if per_expert else (xq[0], xd[0])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mem.memra_nvfp4_moe_gemv(codes, scales, gexp, ids.cuda(), gw.cuda() if gated else None,
                                 xq_in, xd_in, per_expert, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 1
    g_np = np_(gexp)
    if not gated:
        for k, e in enumerate(ids.tolist()):
            if e >= E:
                assert not y[k].any()
                continue
            one = mem.memra_nvfp4_gemv(codes[e], scales[e], float(g_np[e]),
                                       xq[k if per_expert else 0], xd[k if per_expert else 0])
            torch.cuda.synchronize()
            assert torch.equal(one.view(torch.int32), y[k].view(torch.int32)), k
    # the oracle on its own quantisation of the generator's values (equal to the GPU's)
    oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x))
    assert np.array_equal(np_(xq), oxq) and np.array_equal(np_(xd), oxd)
    assert np.array_equal(g_np.view(np.uint32), og.view(np.uint32))
    y_ref, bad = orc.moe_gemv_nvfp4(oc, os_, og, np_(ids),
                                    np_(gw) if gated else None, oxq if per_expert else oxq[0],
                                    oxd if per_expert else oxd[0], int(per_expert))
    assert bad == 1
    terms = np.stack([nvfp4_terms(orc, oc[e], os_[e], og[e],
                                  oxq[k:k + 1] if per_expert else oxq[:1],
                                  oxd[k:k + 1] if per_expert else oxd[:1])[0]
                      if e < E else np.zeros(N) for k, e in enumerate(ids.tolist())])
    if gated:
        assert_within(np_(y), y_ref, (np_(gw)[:, None] * terms).sum(axis=0), "nvfp4 moe gated")
    else:
        assert_within(np_(y), y_ref, terms, "nvfp4 moe")


def test_nvfp4_moe_gemv_tokens_matches_single_token(mem):
    E, N, K, top_k, T = 12, 160, 2048, 8, 5
    codes, scales, gexp = nvfp4_bank(mem, E, N, K, 620)
    ids = torch.stack([synth.routing(E, top_k, 621, t)[0] for t in range(T)])
    gw = torch.stack([synth.routing(E, top_k, 621, t)[1] for t in range(T)])
    x = synth.activations_bf16(T, K, 622)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    for gated in (False, True):
        g = gw.cuda() if gated else None
        y = mem.memra_nvfp4_moe_gemv_tokens(codes, scales, gexp, ids.cuda(), g, xq, xd, False)
        torch.cuda.synchronize()
        for t in range(T):
            one = mem.memra_nvfp4_moe_gemv(codes, scales, gexp, ids[t].cuda(),
                                           g[t] if gated else None, xq[t], xd[t], False)
            torch.cuda.synchronize()
            assert torch.equal(one.view(torch.int32), y[t].view(torch.int32)), (gated, t)


def test_nvfp4_degenerate_sizes(mem):
    """K = 0 zero-fills y; N = 0 or M = 0 launches nothing; an empty ingest leaves g."""
    y = torch.full((3, 5), 7.0, device="cuda")
    mem.memra_nvfp4_gemm_small_m(torch.zeros((5, 0), dtype=torch.uint8, device="cuda"),
                                 torch.zeros((5, 0), dtype=torch.uint8, device="cuda"), 1.0,
                                 torch.zeros((3, 0), dtype=torch.int8, device="cuda"),
                                 torch.zeros((3, 0), dtype=torch.float32, device="cuda"), y=y)
    torch.cuda.synchronize()
    assert not y.any()
    y0 = mem.memra_nvfp4_gemm_small_m(torch.zeros((0, 128), dtype=torch.uint8, device="cuda"),
                                      torch.zeros((0, 16), dtype=torch.uint8, device="cuda"), 1.0,
                                      torch.zeros((2, 256), dtype=torch.int8, device="cuda"),
                                      torch.zeros((2, 8), dtype=torch.float32, device="cuda"))
    assert y0.shape == (2, 0)
    g = torch.full((1,), 5.0, device="cuda")
    mem.memra_quantize_nvfp4(torch.zeros((0, 64), device="cuda"), g=g)
    torch.cuda.synchronize()
    assert float(g.item()) == 5.0
