"""GPU parity for the GGUF block-array repack, through the C ABI.

The repack moves bytes only, so it must match the oracle bit for bit: random block
bytes (any fp16 bit pattern, any int8), ragged block counts, a block array that starts
on a 2-byte boundary only, and guard bands around both output planes.  A GGUF tensor
built from quantised weights must then give, through the products, the bits of the
same weights quantised on the device.
"""
import numpy as np
import pytest
import torch

import synth
from _util import Guarded, abs_terms, assert_within, bf16_bits_np, np_, wd_bits

pytestmark = pytest.mark.gpu

Q8_0_BLOCK = np.dtype([("d", "<u2"), ("qs", "i1", (32,))])
Q4_0_BLOCK = np.dtype([("d", "<u2"), ("qs", "u1", (16,))])


@pytest.fixture(scope="module")
def mem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_decode_quantize_gb300 as m
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    m.lib()
    return m


def _random_blocks(nbytes, seed, offset=0):
    """Seeded random bytes on the device, starting `offset` bytes into a fresh buffer."""
    raw = np.random.default_rng(seed).integers(0, 256, size=nbytes, dtype=np.uint8)
    buf = torch.empty(nbytes + offset, dtype=torch.uint8, device="cuda")
    dev = buf[offset:offset + nbytes]
    dev.copy_(torch.from_numpy(raw))
    return raw, dev


@pytest.mark.parametrize("N,K,offset", [(1, 32, 0), (7, 96, 2), (333, 5120, 0), (1000, 4096, 6),
                                        (5, 17408, 2)])
def test_repack_q8_0_bit_exact(mem, orc, N, K, offset):
    raw, dev = _random_blocks(N * (K // 32) * 34, 800 + N, offset)
    wq = Guarded((N, K), torch.int8)
    wd = Guarded((N, K // 32), torch.float16)
    mem.memra_repack_q8_0(dev, N, K, wq=wq.view, wd=wd.view)
    torch.cuda.synchronize()
    assert wq.intact() and wd.intact()
    oq, od = orc.repack_q8_0(raw, N, K)
    assert np.array_equal(np_(wq.view), oq)
    assert np.array_equal(wd_bits(wd.view), od)


@pytest.mark.parametrize("N,K,offset", [(1, 32, 0), (9, 64, 2), (257, 5120, 4), (64, 17408, 0)])
def test_repack_q4_0_bit_exact(mem, orc, N, K, offset):
    raw, dev = _random_blocks(N * (K // 32) * 18, 900 + N, offset)
    wq4 = Guarded((N, K // 2), torch.int8)  # uint8 plane viewed through int8 guards
    wd = Guarded((N, K // 32), torch.float16)
    mem.memra_repack_q4_0(dev, N, K, wq4=wq4.view.view(torch.uint8), wd=wd.view)
    torch.cuda.synchronize()
    assert wq4.intact() and wd.intact()
    oq4, od = orc.repack_q4_0(raw, N, K)
    assert np.array_equal(np_(wq4.view.view(torch.uint8)), oq4)
    assert np.array_equal(wd_bits(wd.view), od)


def test_repack_rejects_odd_block_address(mem):
    buf = torch.zeros(34 * 4 + 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(mem.MemraError) as e:
        mem.memra_repack_q8_0(buf[1:], 4, 32)
    assert e.value.status == 2


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_gguf_tensor_through_the_products(mem, orc, fmt):
    """Weights quantised by the oracle, laid out as a GGUF block array, repacked on the
    device: the product equals the oracle's, and bit for bit the product of the same
    weights quantised on the device."""
    N, K, M = 777, 5120, 3
    w = synth.weights_fp32(N, K, 71, 1)
    x = synth.activations_bf16(M, K, 71, 2)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x))
    if fmt == "q8_0":
        oq, od = orc.quantize_q8_0(w.numpy())
        aos = np.empty((N, K // 32), Q8_0_BLOCK)
        aos["qs"] = oq.reshape(N, K // 32, 32)
    else:
        oq, od = orc.quantize_q4_0(w.numpy())
        aos = np.empty((N, K // 32), Q4_0_BLOCK)
        aos["qs"] = oq.reshape(N, K // 32, 16)
    aos["d"] = od
    dev = torch.from_numpy(aos.view(np.uint8).reshape(-1).copy()).cuda()
    if fmt == "q8_0":
        wq, wd = mem.memra_repack_q8_0(dev, N, K)
        wq2, wd2 = mem.memra_quantize_q8_0(w.cuda())
        y = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd)
        y2 = mem.memra_q8_0_gemm_small_m(wq2, wd2, xq, xd)
        y_ref = orc.gemm(oq, od, oxq, oxd)
    else:
        wq, wd = mem.memra_repack_q4_0(dev, N, K)
        wq2, wd2 = mem.memra_quantize_q4_0(w.cuda())
        y = mem.memra_q4_0_gemm_small_m(wq, wd, xq, xd)
        y2 = mem.memra_q4_0_gemm_small_m(wq2, wd2, xq, xd)
        y_ref = orc.gemm_q4_0(oq, od, oxq, oxd)
    torch.cuda.synchronize()
    assert np.array_equal(np_(wq).view(np.uint8), oq.view(np.uint8))
    assert np.array_equal(wd_bits(wd), od)
    assert torch.equal(wq, wq2) and torch.equal(wd.view(torch.int16), wd2.view(torch.int16))
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    vals = oq if fmt == "q8_0" else orc.unpack_q4_0(oq)
    assert_within(np_(y), y_ref, abs_terms(orc.block_dots(vals, oxq), od, oxd), fmt + " gguf")
