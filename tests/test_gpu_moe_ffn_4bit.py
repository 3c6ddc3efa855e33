"""GPU checks of the routed FFN layer on Q4_0 and NVFP4 banks, through the C ABI.

The layer entry points must give, bit for bit, the format's own routed GEMVs run in
sequence (gate|up ungated on q8_1(x), SwiGLU + q8_1, down gated); the batched-token
entry points must give, bit for bit, the single-token layer on each token.  The routed
GEMVs themselves are checked against the oracle in test_gpu_q4_0.py and
test_gpu_nvfp4.py.
"""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

E, H, F, TOP_K = 16, 2048, 768, 8


@pytest.fixture(scope="module")
def mem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_decode_quantize_gb300 as m
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    m.lib()
    return m


def banks(mem, fmt, seed):
    """gate|up and down banks of `fmt`; NVFP4 experts are quantised one by one."""
    def bank(rows, K, key):
        if fmt == "q4_0":
            w = torch.stack([synth.weights_fp32(rows, K, seed, key, e) for e in range(E)])
            q, d = mem.memra_quantize_q4_0(w.view(E * rows, K).cuda())
            return q.view(E, rows, K // 2), d.view(E, rows, K // 32), None
        parts = [mem.memra_quantize_nvfp4(synth.weights_fp32(rows, K, seed, key, e).cuda())
                 for e in range(E)]
        return (torch.stack([p[0] for p in parts]), torch.stack([p[1] for p in parts]),
                torch.cat([p[2] for p in parts]))
    return bank(2 * F, H, 0), bank(H, F, 1)


def routed_gemv(mem, fmt, bank, ids, gw, xq, xd, per_expert):
    q, s, g = bank
    if fmt == "q4_0":
        return mem.memra_q4_0_moe_gemv(q, s, ids, gw, xq, xd, per_expert)
    return mem.memra_nvfp4_moe_gemv(q, s, g, ids, gw, xq, xd, per_expert)


def layer(mem, fmt, gu, dn, ids, gw, x, **kw):
    if fmt == "q4_0":
        return mem.memra_q4_0_moe_ffn(gu[0], gu[1], dn[0], dn[1], ids, gw, x, **kw)
    return mem.memra_nvfp4_moe_ffn(gu[0], gu[1], gu[2], dn[0], dn[1], dn[2], ids, gw, x, **kw)


@pytest.mark.parametrize("fmt", ["q4_0", "nvfp4"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_layer_equals_its_four_calls(mem, fmt, dtype):
    gu, dn = banks(mem, fmt, 800 if fmt == "q4_0" else 801)
    ids, gw = synth.routing(E, TOP_K, 802)
    ids, gw = ids.cuda(), gw.cuda()
    x = synth.normal((H,), 803).to(dtype).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = layer(mem, fmt, gu, dn, ids, gw, x, dev_status=st)
    xq, xd = mem.memra_quantize_q8_1(x[None])
    ygu = routed_gemv(mem, fmt, gu, ids, None, xq[0], xd[0], False)
    hq, hd = mem.memra_swiglu_quantize_q8_1(ygu)
    y4 = routed_gemv(mem, fmt, dn, ids, gw, hq, hd, True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y.view(torch.int32), y4.view(torch.int32))
    assert bool(torch.isfinite(y).all()) and bool(y.abs().sum() > 0)


@pytest.mark.parametrize("fmt", ["q4_0", "nvfp4"])
def test_batched_layer_equals_single_token_layer(mem, fmt):
    T = 3
    gu, dn = banks(mem, fmt, 810 if fmt == "q4_0" else 811)
    routes = [synth.routing(E, TOP_K, 812, t) for t in range(T)]
    ids = torch.stack([r[0] for r in routes]).cuda()
    gw = torch.stack([r[1] for r in routes]).cuda()
    x = synth.activations_bf16(T, H, 813).cuda()
    y = layer(mem, fmt, gu, dn, ids, gw, x)
    torch.cuda.synchronize()
    for t in range(T):
        one = layer(mem, fmt, gu, dn, ids[t], gw[t], x[t])
        torch.cuda.synchronize()
        assert torch.equal(one.view(torch.int32), y[t].view(torch.int32)), t


def test_nvfp4_layer_needs_the_expert_scales(mem):
    gu, dn = banks(mem, "nvfp4", 820)
    ids, gw = synth.routing(E, TOP_K, 821)
    ids, gw = ids.cuda(), gw.cuda()
    x = synth.normal((H,), 822).to(torch.bfloat16).cuda()
    lib = mem.lib()
    y = torch.empty((H,), device="cuda")
    ws = torch.empty((TOP_K * 2 * F,), device="cuda")
    st = lib.memra_nvfp4_moe_ffn(gu[0].data_ptr(), gu[1].data_ptr(), None, dn[0].data_ptr(),
                                 dn[1].data_ptr(), dn[2].data_ptr(), E, H, F, ids.data_ptr(),
                                 gw.data_ptr(), TOP_K, x.data_ptr(), 0, y.data_ptr(),
                                 ws.data_ptr(), None, None)
    assert st == 1                                   # no gate|up tensor scales
