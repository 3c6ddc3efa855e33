"""GPU parity for routed experts over a batch of tokens, through the C ABI.

Each (token, slot) pair of a batched call is computed with the single-token
arithmetic, so token t's result must equal, bit for bit, the single-token call on
token t alone; and it must match the oracle (each token on its own) within the
library's tolerance.  Routings share experts across tokens on purpose: those pairs
stream the same expert rows at the same time.
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


def make_bank(mem, E, N, K, seed):
    w = torch.stack([synth.weights_fp32(N, K, seed, 700, e) for e in range(E)])
    wq, wd = mem.memra_quantize_q8_0(w.view(E * N, K).cuda())
    return wq.view(E, N, K), wd.view(E, N, K // 32)


def oracle_bank(orc, E, N, K, seed, wq=None, wd=None):
    """The same bank quantised by the oracle from the generator's fp32 (never from the
    GPU's planes); when the GPU's planes are given they must equal it bit for bit."""
    w = torch.stack([synth.weights_fp32(N, K, seed, 700, e) for e in range(E)])
    oq, od = orc.quantize_q8_0(np_(w).reshape(E * N, K))
    oq, od = oq.reshape(E, N, K), od.reshape(E, N, K // 32)
    if wq is not None:
        assert np.array_equal(np_(wq), oq) and np.array_equal(wd_bits(wd), od)
    return oq, od


def oracle_x(orc, x, xq=None, xd=None):
    """q8_1 of the generator's activation rows by the oracle; the GPU's quantisation, when
    given, must equal it bit for bit."""
    if x.dtype == torch.bfloat16:
        oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x.cpu()))
    else:
        oxq, oxd = orc.quantize_q8_1(np_(x))
    if xq is not None:
        assert np.array_equal(np_(xq).reshape(oxq.shape), oxq)
        assert np.array_equal(np_(xd).reshape(oxd.shape).view(np.uint32), oxd.view(np.uint32))
    return oxq, oxd


def batch_routing(E, T, top_k, seed):
    """Each token's top-k of its own seeded router; with E small the tokens share experts."""
    ids, gw = zip(*[synth.routing(E, top_k, seed, t) for t in range(T)])
    return torch.stack(ids), torch.stack(gw)


def unpack_torch(wq4):
    N, K2 = wq4.shape
    b = wq4.view(N, K2 // 16, 16).to(torch.int16)
    return torch.cat([(b & 0x0F) - 8, (b >> 4) - 8], dim=2).reshape(N, 2 * K2).to(torch.int8)


@pytest.mark.parametrize("T", [1, 3, 8, 16])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("per_expert", [False, True])
def test_moe_gemv_tokens_parity(mem, orc, T, gated, per_expert):
    E, N, K, top_k = 12, 200, 768, 8
    wq, wd = make_bank(mem, E, N, K, 40 + T)
    ids, gw = batch_routing(E, T, top_k, 41 + T)
    assert len(set(ids.flatten().tolist())) < ids.numel() or T == 1  # experts shared
    rows = T * top_k if per_expert else T
    x = synth.activations_bf16(rows, K, 42, T)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    if per_expert:
        xq, xd = xq.view(T, top_k, K), xd.view(T, top_k, K // 32)
    yshape = (T, N) if gated else (T, top_k, N)
    y = Guarded(yshape, torch.float32)
    ws = Guarded((T, top_k, N), torch.float32) if gated else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mem.memra_q8_0_moe_gemv_tokens(wq, wd, ids.cuda(), gw.cuda() if gated else None, xq, xd,
                                   per_expert, y=y.view,
                                   workspace=ws.view if gated else None, dev_status=st)
    torch.cuda.synchronize()
    assert y.intact() and (ws is None or ws.intact()) and int(st.item()) == 0
    # bit for bit the single-token call on each token
    for t in range(T):
        one = mem.memra_q8_0_moe_gemv(wq, wd, ids[t].cuda(), gw[t].cuda() if gated else None,
                                      xq[t], xd[t], per_expert)
        torch.cuda.synchronize()
        assert torch.equal(one.view(torch.int32), y.view[t].view(torch.int32)), t
    # and the oracle, each token on its own, on its own quantisation of the generator's
    # values (asserted equal to the GPU's first)
    oq, od = oracle_bank(orc, E, N, K, 40 + T, wq, wd)
    oxq, oxd = oracle_x(orc, x, xq, xd)
    if per_expert:
        oxq, oxd = oxq.reshape(T, top_k, K), oxd.reshape(T, top_k, K // 32)
    y_ref, bad = orc.moe_gemv_tokens(oq, od, np_(ids), np_(gw) if gated else None, oxq, oxd,
                                     int(per_expert))
    assert bad == 0
    for t in range(T):
        terms = np.stack([abs_terms(orc.block_dots(oq[e], oxq[t][k:k + 1] if per_expert
                                                   else oxq[t][None]),
                                    od[e], oxd[t][k:k + 1] if per_expert else oxd[t][None])[0]
                          for k, e in enumerate(np_(ids)[t])])
        if gated:
            assert_within(np_(y.view)[t], y_ref[t], (np_(gw)[t][:, None] * terms).sum(axis=0),
                          "tokens gated t=%d" % t)
        else:
            assert_within(np_(y.view)[t], y_ref[t], terms, "tokens t=%d" % t)


def test_moe_gemv_tokens_q4_0_matches_q8_0_of_unpacked(mem, orc):
    E, N, K, top_k, T = 10, 160, 1024, 8, 6
    w = torch.stack([synth.weights_fp32(N, K, 50, e) for e in range(E)])
    wq4, wd = mem.memra_quantize_q4_0(w.view(E * N, K).cuda())
    bank4, bankd = wq4.view(E, N, K // 2), wd.view(E, N, K // 32)
    bank8 = unpack_torch(wq4).view(E, N, K)
    ids, gw = batch_routing(E, T, top_k, 51)
    x = synth.activations_bf16(T, K, 52)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    for gated in (False, True):
        g = gw.cuda() if gated else None
        y4 = mem.memra_q4_0_moe_gemv_tokens(bank4, bankd, ids.cuda(), g, xq, xd, False)
        y8 = mem.memra_q8_0_moe_gemv_tokens(bank8, bankd, ids.cuda(), g, xq, xd, False)
        torch.cuda.synchronize()
        assert torch.equal(y4.view(torch.int32), y8.view(torch.int32)), gated
        for t in (0, T - 1):
            one = mem.memra_q4_0_moe_gemv(bank4, bankd, ids[t].cuda(), g[t] if gated else None,
                                          xq[t], xd[t], False)
            torch.cuda.synchronize()
            assert torch.equal(one.view(torch.int32), y4[t].view(torch.int32))


def test_moe_gemv_tokens_bad_ids(mem):
    E, N, K, top_k, T = 4, 64, 256, 3, 2
    wq, wd = make_bank(mem, E, N, K, 55)
    ids = torch.tensor([[1, 7, 2], [-1, 3, 3]], dtype=torch.int32)
    gw = torch.tensor([[0.5, 0.25, 0.25], [0.2, 0.4, 0.4]], dtype=torch.float32)
    x = synth.activations_bf16(T, K, 56)
    xq, xd = mem.memra_quantize_q8_1(x.cuda())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = mem.memra_q8_0_moe_gemv_tokens(wq, wd, ids.cuda(), None, xq, xd, False, dev_status=st)
    yg = mem.memra_q8_0_moe_gemv_tokens(wq, wd, ids.cuda(), gw.cuda(), xq, xd, False)
    torch.cuda.synchronize()
    assert int(st.item()) == 1
    assert not y[0, 1].any() and not y[1, 0].any()
    for t in range(T):
        one = mem.memra_q8_0_moe_gemv(wq, wd, ids[t].cuda(), gw[t].cuda(), xq[t], xd[t], False)
        torch.cuda.synchronize()
        assert torch.equal(one.view(torch.int32), yg[t].view(torch.int32))


def test_moe_gemv_tokens_limits(mem):
    E, N, K = 4, 32, 256
    wq, wd = make_bank(mem, E, N, K, 57)
    ids = torch.zeros((17, 8), dtype=torch.int32, device="cuda")  # 136 pairs > 128
    xq = torch.zeros((17, K), dtype=torch.int8, device="cuda")
    xd = torch.zeros((17, K // 32), dtype=torch.float32, device="cuda")
    with pytest.raises(mem.MemraError) as e:
        mem.memra_q8_0_moe_gemv_tokens(wq, wd, ids, None, xq, xd, False)
    assert e.value.status == 3
    y = mem.memra_q8_0_moe_gemv_tokens(wq, wd, ids[:16], None, xq[:16], xd[:16], False)
    torch.cuda.synchronize()
    assert y.shape == (16, 8, N)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T", [1, 5, 8])
def test_moe_ffn_tokens_matches_single_token_layer(mem, orc, dtype, T):
    E, H, F, top_k = 16, 2048, 768, 8
    gq, gd = make_bank(mem, E, 2 * F, H, 60)
    dq, dd = make_bank(mem, E, H, F, 61)
    ids, gw = batch_routing(E, T, top_k, 62 + T)
    x = synth.normal((T, H), 63, T).to(dtype).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty((T * top_k * (2 * F + H),), dtype=torch.float32, device="cuda")
    y = mem.memra_q8_0_moe_ffn_tokens(gq, gd, dq, dd, ids.cuda(), gw.cuda(), x, workspace=ws,
                                      dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for t in range(T):
        one = mem.memra_q8_0_moe_ffn(gq, gd, dq, dd, ids[t].cuda(), gw[t].cuda(), x[t])
        torch.cuda.synchronize()
        assert torch.equal(one.view(torch.int32), y[t].view(torch.int32)), t
    # the oracle's layer per token: quantisation of x is bit-exact, the rest within the
    # bound the single-token FFN test uses
    xo = bf16_bits_np(x.cpu()) if dtype == torch.bfloat16 else np_(x)
    xf = orc.bf16_bits_to_f32(xo) if dtype == torch.bfloat16 else xo
    ogq, ogd = oracle_bank(orc, E, 2 * F, H, 60, gq, gd)
    odq, odd = oracle_bank(orc, E, H, F, 61, dq, dd)
    y_ref, bad = orc.moe_ffn_tokens(xf, ogq, ogd, odq, odd, np_(ids), np_(gw))
    assert bad == 0
    err = np.abs(np_(y).astype(np.float64) - y_ref)
    assert np.all(err <= 0.02 * np.abs(y_ref).max(axis=1, keepdims=True) + 1e-5)


def test_moe_tokens_at_the_routed_workload_shapes(mem):
    """128 experts of gate|up 1536 x 2048 and down 2048 x 768, 8 tokens with their own
    routing: bit for bit the single-token layer on every token."""
    E, H, F, top_k, T = 128, 2048, 768, 8, 8
    gq, gd = make_bank(mem, E, 2 * F, H, 70)
    dq, dd = make_bank(mem, E, H, F, 71)
    ids, gw = batch_routing(E, T, top_k, 72)
    x = synth.activations_bf16(T, H, 73).cuda()
    y = mem.memra_q8_0_moe_ffn_tokens(gq, gd, dq, dd, ids.cuda(), gw.cuda(), x)
    torch.cuda.synchronize()
    for t in range(T):
        one = mem.memra_q8_0_moe_ffn(gq, gd, dq, dd, ids[t].cuda(), gw[t].cuda(), x[t])
        torch.cuda.synchronize()
        assert torch.equal(one.view(torch.int32), y[t].view(torch.int32)), t


def test_tokens_degenerate_sizes(mem):
    """K = 0: every sum is empty, so outputs are zero-filled; T = 0 or N = 0: nothing."""
    E, N, T, top_k = 3, 16, 2, 2
    ids = torch.zeros((T, top_k), dtype=torch.int32, device="cuda")
    gw = torch.full((T, top_k), 0.5, device="cuda")
    wq = torch.zeros((E, N, 0), dtype=torch.int8, device="cuda")
    wd = torch.zeros((E, N, 0), dtype=torch.float16, device="cuda")
    xq = torch.zeros((T, 0), dtype=torch.int8, device="cuda")
    xd = torch.zeros((T, 0), dtype=torch.float32, device="cuda")
    y = torch.full((T, top_k, N), 7.0, device="cuda")
    mem.memra_q8_0_moe_gemv_tokens(wq, wd, ids, None, xq, xd, False, y=y)
    yg = torch.full((T, N), 7.0, device="cuda")
    mem.memra_q8_0_moe_gemv_tokens(wq, wd, ids, gw, xq, xd, False, y=yg)
    torch.cuda.synchronize()
    assert not y.any() and not yg.any()
    lib = mem.lib()
    sentinel = torch.full((4,), 3.0, device="cuda")
    assert lib.memra_q8_0_moe_gemv_tokens(None, None, E, N, 64, None, None, 0, top_k, None, None,
                                          0, sentinel.data_ptr(), None, None, None) == 0
    assert lib.memra_q8_0_moe_gemv_tokens(None, None, E, 0, 64, None, None, T, top_k, None, None,
                                          0, sentinel.data_ptr(), None, None, None) == 0
    torch.cuda.synchronize()
    assert torch.all(sentinel == 3.0)
