"""memra_q8_0_gemv_chain: a decode step's chain of M = 1 products in one persistent
cooperative launch must give, for every step, exactly (bit for bit) what the
single-product fused entry point gives, and match the oracle."""
import numpy as np
import pytest
import torch

import synth
from _util import abs_terms, assert_within, bf16_bits_np, np_, wd_bits

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


def make_step(mem, N, K, key, dtype=torch.bfloat16):
    w = synth.weights_fp32(N, K, 600, key, device="cuda")
    wq, wd = mem.memra_quantize_q8_0(w)
    x = synth.activations_fp32(1, K, 601, key, outlier_frac=0.001, device="cuda")[0].to(dtype)
    y = torch.full((N,), float("nan"), device="cuda")
    return w, wq, wd, x, y


SHAPES = [(7168, 5120), (5120, 5120), (100, 17408), (0, 4096), (4097, 2048), (33, 256),
          (34816, 5120), (5120, 17408), (1, 768)]


def test_chain_matches_single_products_bitwise(mem):
    steps = [make_step(mem, N, K, i, torch.bfloat16 if i % 3 else torch.float32)
             for i, (N, K) in enumerate(SHAPES)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mem.memra_q8_0_gemv_chain([(wq, wd, x, y) for _, wq, wd, x, y in steps], dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for (N, K), (_, wq, wd, x, y) in zip(SHAPES, steps):
        ref = mem.memra_q8_0_quant_gemm(wq, wd, x[None])[0]
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), (N, K)


def test_chain_against_oracle_and_repeat(mem, orc):
    shapes = [(513, 5120), (97, 17408), (2048, 2048)]
    steps = [make_step(mem, N, K, 50 + i) for i, (N, K) in enumerate(shapes)]
    plan = mem.GemvChain([(wq, wd, x, y) for _, wq, wd, x, y in steps])
    plan.run()
    torch.cuda.synchronize()
    first = [y.clone() for *_, y in steps]
    for (w, wq, wd, x, y) in steps:
        oq, od = orc.quantize_q8_0(np_(w))
        assert np.array_equal(np_(wq), oq) and np.array_equal(wd_bits(wd), od)
        oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x.cpu())[None])
        assert_within(np_(y)[None], orc.gemm(oq, od, oxq, oxd),
                      abs_terms(orc.block_dots(oq, oxq), od, oxd), "chain step")
    for *_, y in steps:
        y.fill_(float("nan"))
    plan.run()                       # the sync words are re-zeroed by every call
    torch.cuda.synchronize()
    for a, (*_, y) in zip(first, steps):
        assert torch.equal(a.view(torch.int32), y.view(torch.int32))


def test_chain_in_a_cuda_graph(mem):
    steps = [make_step(mem, N, K, 80 + i) for i, (N, K) in enumerate([(3000, 5120), (512, 17408)])]
    plan = mem.GemvChain([(wq, wd, x, y) for _, wq, wd, x, y in steps])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.run()
    torch.cuda.synchronize()
    ref = [y.clone() for *_, y in steps]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run()
    for *_, y in steps:
        y.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, (*_, y) in zip(ref, steps):
        assert torch.equal(a.view(torch.int32), y.view(torch.int32))


DEP_SPEC = [(5120, 4096, None), (2048, 5120, 0), (0, 2048, 1), (17408, 2048, 1),
            (512, 17408, 3), (7168, 512, 4)]   # (N, K, step whose output is x)


def _dependent_chain(mem, key):
    """Steps whose activation is an earlier step's fp32 output (one step has no rows
    and feeds nothing), so each step must wait for every row of an earlier one."""
    ys, prods = [], []
    x0 = synth.activations_fp32(1, 4096, 602, key, device="cuda")[0].to(torch.bfloat16)
    for i, (N, K, src) in enumerate(DEP_SPEC):
        w = synth.weights_fp32(N, K, 603, key, i, device="cuda")
        wq, wd = mem.memra_quantize_q8_0(w)
        y = torch.full((N,), float("nan"), device="cuda")
        ys.append(y)
        prods.append((wq, wd, x0 if src is None else ys[src], y))
    return prods


def _sequential(mem, prods):
    """The same products one fused single-product call at a time, each fed with the
    previous calls' own outputs."""
    out = []
    for (wq, wd, x, _), (_, _, src) in zip(prods, DEP_SPEC):
        xin = x if src is None else out[src]
        out.append(mem.memra_q8_0_quant_gemm(wq, wd, xin[None])[0])
    return out


def test_chain_dependent_steps(mem):
    prods = _dependent_chain(mem, 90)
    ref = _sequential(mem, prods)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan = mem.GemvChain(prods, dev_status=st)
    for rep in range(3):
        for *_, y in prods:
            y.fill_(float("nan"))
        plan.run()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for i, ((*_, y), r) in enumerate(zip(prods, ref)):
            assert torch.equal(y.view(torch.int32), r.view(torch.int32)), (rep, i)


def test_chain_dependent_steps_graph_replays(mem):
    prods = _dependent_chain(mem, 91)
    ref = _sequential(mem, prods)
    plan = mem.GemvChain(prods)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run()
    for _ in range(5):
        for *_, y in prods:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for (*_, y), r in zip(prods, ref):
            assert torch.equal(y.view(torch.int32), r.view(torch.int32))


def test_chain_argument_errors(mem):
    bad = torch.zeros((64, 96), dtype=torch.int8, device="cuda")   # K = 96: not a multiple of 256
    with pytest.raises(mem.MemraError) as ei:
        mem.memra_q8_0_gemv_chain([(bad, torch.zeros((64, 3), dtype=torch.float16,
                                                      device="cuda"),
                                    torch.zeros(96, dtype=torch.bfloat16, device="cuda"),
                                    torch.zeros(64, device="cuda"))])
    assert ei.value.status == 1
