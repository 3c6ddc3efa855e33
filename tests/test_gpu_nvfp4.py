"""GPU parity for NVFP4 weights, through the C ABI.

The weight ingest must match the oracle bit for bit (codes, E4M3 scales and the tensor
scale).  Products must match the oracle within |y - y_ref| <= 1e-4 * sum |term| + 1e-6,
with one term per 16-element half-block, |(g/2) s d_x S|; each row must equal, bit for
bit, the M = 1 product of that row.  Each side runs its own pipeline from the same
seeded inputs.
"""
import json
import os

import numpy as np
import pytest
import torch

import synth
from _util import Guarded, assert_within, bf16_bits_np, np_

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


def nvfp4_terms(orc, oc, os_, og, oxq, oxd):
    N, K = oc.shape[0], oc.shape[1] * 2
    M = oxq.shape[0]
    c2 = orc.unpack_nvfp4(oc).astype(np.float64).reshape(N, K // 16, 16)
    S = np.einsum("nbi,mbi->mnb", c2, oxq.astype(np.float64).reshape(M, K // 16, 16))
    s = orc.e4m3_to_f32(os_).astype(np.float64)
    dx = np.repeat(oxd.astype(np.float64), 2, axis=1)
    return np.abs(0.5 * float(og) * s[None] * dx[:, None, :] * S).sum(axis=2)


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
    assert_within(np_(y.view), y_ref, nvfp4_terms(orc, oc, os_, og, oxq, oxd),
                  "nvfp4 N=%d K=%d M=%d" % (N, K, M))
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
