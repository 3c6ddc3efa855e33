"""The allocation-free routed FFN entry point, memra_q8_0_moe_ffn_noalloc.

Some callers cannot allocate device memory when they call the library: a runtime
confined to a fixed arena, a plug-in that is handed device pointers but no
allocator, a latency-bound decode loop.  This entry point gives them the routed FFN
layer with its gate|up workspace in an array inside the library.  Here it is called
through the C ABI twice in a row (different layers, so the shared array is
overwritten in between) and must match the workspace entry point each time.  The
file is collected last so that, on a failure, every other test has already run; it
also passes on its own in a fresh process."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

REL, ABS = 1e-4, 1e-6   # the parity tolerance used across the GPU tests


@pytest.fixture(scope="module")
def mem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_decode_quantize_gb300 as m
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    m.lib()
    return m


def bank(mem, E, N, K, *keys):
    w = synth.weights_fp32(E * N, K, *keys, device="cuda")
    q, d = mem.memra_quantize_q8_0(w)
    return q.view(E, N, K), d.view(E, N, K // 32)


def layer(mem, E, H, F, top_k, key):
    gq, gd = bank(mem, E, 2 * F, H, 500, key, 0)
    dq, dd = bank(mem, E, H, F, 500, key, 1)
    ids, gw = synth.routing(E, top_k, 500, key, 2, device="cuda")
    x = synth.activations_bf16(1, H, 500, key, 3, device="cuda")[0]
    return gq, gd, dq, dd, ids, gw, x


def test_noalloc_matches_workspace_entry_on_two_calls(mem):
    E, H, F, top_k = 32, 2048, 768, 8
    calls = [layer(mem, E, H, F, top_k, key) for key in (1, 2)]
    outs = []
    for gq, gd, dq, dd, ids, gw, x in calls:
        y = torch.full((H,), float("nan"), device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        mem.memra_q8_0_moe_ffn_noalloc(gq, gd, dq, dd, ids, gw, x, y, dev_status=st)
        outs.append((y, st))
    for (gq, gd, dq, dd, ids, gw, x), (y, st) in zip(calls, outs):
        ref = mem.memra_q8_0_moe_ffn(gq, gd, dq, dd, ids, gw, x)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.isfinite(y).all()
        err = (y.double() - ref.double()).abs()
        assert bool((err <= REL * ref.double().abs() + ABS).all())
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32))   # in fact bit-identical


def test_noalloc_at_the_size_limit(mem):
    """top_k * 2F exactly fills the array (the kernels write its last float): the result
    equals the workspace entry point's, bit for bit, on two calls in a row."""
    E, H, F, top_k = 8, 256, 4096, 8
    assert top_k * 2 * F == mem.MOE_NOALLOC_SCRATCH_FLOATS
    for key in (3, 4):
        gq, gd, dq, dd, ids, gw, x = layer(mem, E, H, F, top_k, key)
        y = torch.full((H,), float("nan"), device="cuda")
        mem.memra_q8_0_moe_ffn_noalloc(gq, gd, dq, dd, ids, gw, x, y)
        ws = torch.full((top_k, 2 * F), float("nan"), device="cuda")
        ref = mem.memra_q8_0_moe_ffn(gq, gd, dq, dd, ids, gw, x, workspace=ws)
        torch.cuda.synchronize()
        assert torch.isfinite(ws).all()          # every gate|up row was written
        assert torch.isfinite(y).all()
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), key


def test_noalloc_rejects_oversized_workspace(mem):
    E, H, F, top_k = 2, 64, 4128, 8     # top_k * 2F = 66048 > 65536 floats
    assert top_k * 2 * F > mem.MOE_NOALLOC_SCRATCH_FLOATS
    gq = torch.zeros((E, 2 * F, H), dtype=torch.int8, device="cuda")
    gd = torch.zeros((E, 2 * F, H // 32), dtype=torch.float16, device="cuda")
    dq = torch.zeros((E, H, F), dtype=torch.int8, device="cuda")
    dd = torch.zeros((E, H, F // 32), dtype=torch.float16, device="cuda")
    ids = torch.zeros(top_k, dtype=torch.int32, device="cuda")
    gw = torch.ones(top_k, device="cuda")
    x = torch.zeros(H, device="cuda")
    y = torch.full((H,), 3.0, device="cuda")
    with pytest.raises(mem.MemraError) as ei:
        mem.memra_q8_0_moe_ffn_noalloc(gq, gd, dq, dd, ids, gw, x, y)
    assert ei.value.status == 3
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
