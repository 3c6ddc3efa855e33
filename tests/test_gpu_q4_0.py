"""GPU parity for Q4_0 weights, through the C ABI.

The weight ingest must match the oracle bit for bit (packed codes and fp16 scales).
Products must match the oracle within |y - y_ref| <= 1e-4 * sum_b |d_w d_x s_b| + 1e-6,
and, since the library sums every product in one fp32 order, bit for bit the Q8_0
product of the same codes unpacked to int8 (c - 8).  Each side runs its own pipeline
from the same seeded fp32/bf16 inputs.
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


def check_q4_weights(orc, mem, w_cpu):
    wq4, wd = mem.memra_quantize_q4_0(w_cpu.cuda())
    torch.cuda.synchronize()
    oq4, od = orc.quantize_q4_0(np_(w_cpu))
    assert np.array_equal(np_(wq4), oq4)
    assert np.array_equal(wd_bits(wd), od)
    return wq4, wd, oq4, od


def unpack_torch(wq4):
    """int8 [N, K] codes minus 8 from packed [N, K/2] (byte j of a block: elements j, j+16)."""
    N, K2 = wq4.shape
    b = wq4.view(N, K2 // 16, 16).to(torch.int16)
    lo = (b & 0x0F) - 8
    hi = (b >> 4) - 8
    return torch.cat([lo, hi], dim=2).reshape(N, 2 * K2).to(torch.int8).contiguous()


@pytest.mark.parametrize("N,K,seed", [(37, 96, 1), (4096, 4096, 0), (3, 17408, 2)])
def test_quantize_q4_0_bit_exact(mem, orc, N, K, seed):
    check_q4_weights(orc, mem, synth.weights_fp32(N, K, seed, 500))


def test_quantize_q4_0_special_blocks(mem, orc):
    w = synth.weights_fp32(8, 256, 7, 501)
    w[0, 0:32] = 0.0                                   # zero block: d = +0, codes 8
    w[1, 0:32] = 0.0
    w[1, 3], w[1, 9] = 0.5, -0.5                       # tie, positive first: d < 0
    w[2, 0:32] = 0.0
    w[2, 3], w[2, 9] = -0.5, 0.5                       # tie, negative first: d > 0
    w[3, 32:64] = -0.0                                 # negative zeros
    w[4, 64:96] *= 1e-6                                # subnormal fp16 scales
    w[5, 96:128] *= 3e4                                # scales near the fp16 top
    w[6, 128:160] = 7.5 / 8.0                          # every value at the clamp point
    w[6, 128] = -1.0
    check_q4_weights(orc, mem, w)


@pytest.mark.parametrize("N,K,M", [(1003, 4096, 1), (777, 5120, 1), (300, 5120, 8),
                                   (64, 17408, 1), (130, 17408, 8), (12289, 4096, 2),
                                   (5120, 17408, 1), (513, 2048, 4), (1, 256, 3), (700, 5120, 16),
                                   (129, 17408, 11)])
def test_q4_0_gemm_parity(mem, orc, N, K, M):
    seed = N * 31 + K + M
    w = synth.weights_fp32(N, K, seed, 502)
    x = synth.activations_fp32(M, K, seed, 503, outlier_frac=0.001).to(torch.bfloat16)
    wq4, wd, oq4, od = check_q4_weights(orc, mem, w)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x))
    assert np.array_equal(np_(xq), oxq)
    y = Guarded((M, N), torch.float32)
    if M == 1:
        mem.memra_q4_0_gemv(wq4, wd, xq[0], xd[0], y=y.view[0])
    else:
        mem.memra_q4_0_gemm_small_m(wq4, wd, xq, xd, y=y.view)
    torch.cuda.synchronize()
    assert y.intact()
    y_ref = orc.gemm_q4_0(oq4, od, oxq, oxd)
    terms = abs_terms(orc.block_dots(orc.unpack_q4_0(oq4), oxq), od, oxd)
    assert_within(np_(y.view), y_ref, terms, "q4_0 N=%d K=%d M=%d" % (N, K, M))
    # One summation order for every product: the Q8_0 kernels on the unpacked codes
    # give the same bits, and each row equals the M = 1 result.
    y8 = mem.memra_q8_0_gemm_small_m(unpack_torch(wq4), wd, xq, xd)
    y1 = mem.memra_q4_0_gemv(wq4, wd, xq[M - 1], xd[M - 1])
    torch.cuda.synchronize()
    assert torch.equal(y.view.view(torch.int32), y8.view(torch.int32))
    assert torch.equal(y.view[M - 1].view(torch.int32), y1.view(torch.int32))


def test_q4_0_rejects_k_not_multiple_of_256(mem):
    wq4 = torch.zeros((4, 48), dtype=torch.uint8, device="cuda")
    wd = torch.zeros((4, 3), dtype=torch.float16, device="cuda")
    xq = torch.zeros((1, 96), dtype=torch.int8, device="cuda")
    xd = torch.zeros((1, 3), dtype=torch.float32, device="cuda")
    with pytest.raises(mem.MemraError) as e:
        mem.memra_q4_0_gemm_small_m(wq4, wd, xq, xd)
    assert e.value.status == 3


@pytest.mark.parametrize("gated,per_expert", [(False, False), (True, True), (True, False)])
def test_q4_0_moe_gemv_parity(mem, orc, gated, per_expert):
    """Routed experts on a Q4_0 bank: against the oracle's routed product of the unpacked
    codes, and bit for bit the Q8_0 routed product of the same codes."""
    E, N, K, top_k = 12, 200, 768, 8
    w = torch.stack([synth.weights_fp32(N, K, 61, e) for e in range(E)])
    wq4, wd, oq4, od = check_q4_weights(orc, mem, w.view(E * N, K))
    bank4, bankd = wq4.view(E, N, K // 2), wd.view(E, N, K // 32)
    ids = torch.tensor([3, 11, 0, 7, 3, 5, 9, 1], dtype=torch.int32)
    gw = torch.tensor([0.2, 0.15, 0.1, 0.1, 0.15, 0.1, 0.1, 0.1], dtype=torch.float32)
    x = synth.activations_bf16(top_k if per_expert else 1, K, 62)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x))
    assert np.array_equal(np_(xq), oxq)
    xq_in, xd_in = (xq, xd) if per_expert else (xq[0], xd[0])
    gw_in = gw.cuda() if gated else None
    y = mem.memra_q4_0_moe_gemv(bank4, bankd, ids.cuda(), gw_in, xq_in, xd_in, per_expert)
    bank8 = unpack_torch(wq4).view(E, N, K)
    y8 = mem.memra_q8_0_moe_gemv(bank8, bankd, ids.cuda(), gw_in, xq_in, xd_in, per_expert)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), y8.view(torch.int32))
    o8 = orc.unpack_q4_0(oq4).reshape(E, N, K)
    odb = od.reshape(E, N, K // 32)
    y_ref, bad = orc.moe_gemv(o8, odb, np_(ids), np_(gw) if gated else None, oxq, oxd,
                              1 if per_expert else 0)
    assert bad == 0
    terms = np.stack([abs_terms(orc.block_dots(o8[e], oxq[k:k + 1] if per_expert else oxq),
                                odb[e], oxd[k:k + 1] if per_expert else oxd)[0]
                      for k, e in enumerate(np_(ids))])
    if gated:
        assert_within(np_(y), y_ref, (np_(gw)[:, None] * terms).sum(axis=0), "q4_0 moe gated")
    else:
        assert_within(np_(y), y_ref, terms, "q4_0 moe")
