"""The device-side failure path of the bulk-copy product kernel, driven without a fault.

Every wait of the kernel on its shared-memory barriers is bounded.  The test hook
memra_debug_set_wait_test shortens the bound and makes each CTA's producer stop after
one stage, leaving a stage that nothing completes: the consumers' and the producer's
waits run out, the kernel lets its issued copies land, writes NaN into its outputs,
sets status bit 2 (routed entry points) and returns.  The next call, with the hook off,
must give the normal results on the same context."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

LIMIT = 1 << 16   # SM cycles: tens of microseconds per wait


@pytest.fixture(scope="module")
def mem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_decode_quantize_gb300 as m
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    m.lib()
    return m


def test_dense_product_gives_up_and_recovers(mem):
    N, K = 8192, 4096   # 35.7 MB: the bulk-copy kernel, several stages per CTA
    w = synth.weights_fp32(N, K, 950, device="cuda")
    x = synth.activations_bf16(1, K, 951, device="cuda")
    wq, wd = mem.memra_quantize_q8_0(w)
    xq, xd = mem.memra_quantize_q8_1(x)
    ref = mem.memra_q8_0_gemv(wq, wd, xq[0], xd[0])
    torch.cuda.synchronize()
    assert bool(torch.isfinite(ref).all())
    try:
        mem.memra_debug_set_wait_test(LIMIT, 1)
        y = mem.memra_q8_0_gemv(wq, wd, xq[0], xd[0])
        torch.cuda.synchronize()                      # the kernel returned
    finally:
        mem.memra_debug_set_wait_test()
    assert bool(torch.isnan(y).all())                 # every CTA stalled and marked its rows
    again = mem.memra_q8_0_gemv(wq, wd, xq[0], xd[0])
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int32), ref.view(torch.int32))


def test_routed_product_reports_the_timeout(mem):
    E, N, K, top_k = 16, 4096, 2048, 8   # each CTA streams several stages of its experts
    wb = synth.weights_fp32(E * N, K, 952, device="cuda")
    bq, bd = mem.memra_quantize_q8_0(wb)
    bq, bd = bq.view(E, N, K), bd.view(E, N, K // 32)
    ids, gw = synth.routing(E, top_k, 953, device="cuda")
    x = synth.activations_bf16(1, K, 954, device="cuda")
    xq, xd = mem.memra_quantize_q8_1(x)
    ref = mem.memra_q8_0_moe_gemv(bq, bd, ids, None, xq[0], xd[0], False)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        mem.memra_debug_set_wait_test(LIMIT, 1)
        y = mem.memra_q8_0_moe_gemv(bq, bd, ids, None, xq[0], xd[0], False, dev_status=st)
        torch.cuda.synchronize()
    finally:
        mem.memra_debug_set_wait_test()
    assert int(st.item()) & 2
    assert bool(torch.isnan(y).any())
    st.zero_()
    again = mem.memra_q8_0_moe_gemv(bq, bd, ids, None, xq[0], xd[0], False, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(again.view(torch.int32), ref.view(torch.int32))


def test_hook_rejects_out_of_range_stall(mem):
    with pytest.raises(mem.MemraError) as e:
        mem.memra_debug_set_wait_test(LIMIT, 1 << 40)
    assert e.value.status == 1
    mem.memra_debug_set_wait_test()
