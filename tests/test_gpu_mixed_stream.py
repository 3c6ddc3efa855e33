"""A chain of different entry points on one stream, each consuming the previous output.

Every kernel may let its successor launch early (programmatic dependent launch), and a
product streams weights before it waits for its predecessor.  This checks, across
kernel types, that no call reads an input before its producer has finished: the chain
run back to back (eagerly and as a replayed CUDA graph) must give the same bits as the
same calls with a device synchronise after each.
"""
import numpy as np
import pytest
import torch

import synth

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


Q8_0_BLOCK = np.dtype([("d", "<u2"), ("qs", "i1", (32,))])


@pytest.fixture(scope="module")
def chain(mem):
    H, F, E, top_k, T = 2048, 768, 16, 4, 3
    dev = "cuda"
    w1 = synth.weights_fp32(4096, H, 900, 1)
    wq1, wd1 = mem.memra_quantize_q8_0(w1.cuda())                      # Q8_0 4096 x 2048
    c2, s2, g2 = mem.memra_quantize_nvfp4(synth.weights_fp32(2560, 4096, 900, 2).cuda())
    g2 = float(g2.item())                                              # NVFP4 2560 x 4096
    q3, d3 = mem.memra_quantize_q4_0(synth.weights_fp32(H, 2560, 900, 3).cuda())  # Q4_0
    bank = torch.stack([synth.weights_fp32(F, H, 900, 4, e) for e in range(E)])
    bq, bd = mem.memra_quantize_q8_0(bank.view(E * F, H).cuda())
    bq, bd = bq.view(E, F, H), bd.view(E, F, H // 32)
    # a GGUF copy of w1, repacked on the device inside the chain
    oq, od = wq1.cpu().numpy(), wd1.cpu().view(torch.int16).numpy().view(np.uint16)
    aos = np.empty((4096, H // 32), Q8_0_BLOCK)
    aos["d"] = od
    aos["qs"] = oq.reshape(4096, H // 32, 32)
    gguf = torch.from_numpy(aos.view(np.uint8).reshape(-1).copy()).to(dev)
    ids = torch.stack([synth.routing(E, top_k, 901, t)[0] for t in range(T)]).to(dev)
    gw = torch.stack([synth.routing(E, top_k, 901, t)[1] for t in range(T)]).to(dev)
    x = synth.activations_bf16(T, H, 902).to(dev)
    return dict(wq1=wq1, wd1=wd1, c2=c2, s2=s2, g2=g2, q3=q3, d3=d3, bq=bq, bd=bd, gguf=gguf,
                ids=ids, gw=gw, x=x, H=H, T=T)


def run_chain(mem, c, sync):
    def step(v):
        if sync:
            torch.cuda.synchronize()
        return v
    wq, wd = step(mem.memra_repack_q8_0(c["gguf"], 4096, c["H"]))      # weights for step 2
    xq, xd = step(mem.memra_quantize_q8_1(c["x"]))                      # [T, 2048]
    y1 = step(mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd))              # [T, 4096] fp32
    x2q, x2d = step(mem.memra_quantize_q8_1(y1))
    y2 = step(mem.memra_nvfp4_gemm_small_m(c["c2"], c["s2"], c["g2"], x2q, x2d))  # [T, 2560]
    x3q, x3d = step(mem.memra_quantize_q8_1(y2))
    y3 = step(mem.memra_q4_0_gemm_small_m(c["q3"], c["d3"], x3q, x3d))  # [T, 2048]
    x4q, x4d = step(mem.memra_quantize_q8_1(y3))
    y4 = step(mem.memra_q8_0_moe_gemv_tokens(c["bq"], c["bd"], c["ids"], c["gw"], x4q, x4d,
                                             False))                    # [T, 768]
    return [y1, y2, y3, y4]


def bits(ts):
    torch.cuda.synchronize()
    return [t.clone().view(torch.int32) for t in ts]


def test_mixed_chain_back_to_back_equals_synchronised(mem, chain):
    ref = bits(run_chain(mem, chain, sync=True))
    for _ in range(3):
        got = bits(run_chain(mem, chain, sync=False))
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
    assert all(bool(torch.isfinite(t.view(torch.float32)).all()) for t in ref)


def test_mixed_chain_as_a_cuda_graph(mem, chain):
    ref = bits(run_chain(mem, chain, sync=True))
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        run_chain(mem, chain, sync=False)  # warm-up outside the graph
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        outs = run_chain(mem, chain, sync=False)
    for _ in range(3):
        g.replay()
        got = bits(outs)
        for a, b in zip(ref, got):
            assert torch.equal(a, b)
