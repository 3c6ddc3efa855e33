"""GPU checks of the routed FFN layer on Q4_0 and NVFP4 banks, through the C ABI.

The layer entry points must match the oracle's layer, built from its own quantisation
of the generator's fp32 weights and activations, stage by stage: the gate|up rows
within the product tolerance, then the output against the oracle's down projection of
its own SwiGLU rows within the bound that a one-step difference in the requantised
rows allows.  They must also give, bit for bit, the format's own routed GEMVs run in
sequence (gate|up ungated on q8_1(x), SwiGLU + q8_1, down gated), and the
batched-token entry points the single-token layer on each token.
"""
import numpy as np
import pytest
import torch

import synth
from _util import abs_terms, assert_within, bf16_bits_np, np_, nvfp4_terms, wd_bits

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


def oracle_banks(orc, fmt, seed):
    """The banks of `banks` quantised by the oracle from the generator's fp32, expert by
    expert: (planes [E, rows, ...], scales [E, rows, ...], tensor scales [E] or None)."""
    def bank(rows, K, key):
        parts = []
        for e in range(E):
            w = np_(synth.weights_fp32(rows, K, seed, key, e))
            parts.append(orc.quantize_q4_0(w) + (None,) if fmt == "q4_0" else
                         orc.quantize_nvfp4(w))
        g = None if fmt == "q4_0" else np.array([p[2] for p in parts], np.float32)
        return np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]), g
    return bank(2 * F, H, 0), bank(H, F, 1)


def assert_bank_equal(fmt, gpu, ob):
    assert np.array_equal(np_(gpu[0]), ob[0])
    if fmt == "q4_0":
        assert np.array_equal(wd_bits(gpu[1]), ob[1])
    else:
        assert np.array_equal(np_(gpu[1]), ob[1])
        assert np.array_equal(np_(gpu[2]).view(np.uint32), ob[2].view(np.uint32))


def oracle_product(orc, fmt, ob, e, xq, xd):
    """Expert e's product with q8_1 rows (y [M, N]) and its tolerance terms [M, N]."""
    if fmt == "q4_0":
        y = orc.gemm_q4_0(ob[0][e], ob[1][e], xq, xd)
        return y, abs_terms(orc.block_dots(orc.unpack_q4_0(ob[0][e]), xq), ob[1][e], xd)
    y = orc.gemm_nvfp4(ob[0][e], ob[1][e], ob[2][e], xq, xd)
    return y, nvfp4_terms(orc, ob[0][e], ob[1][e], ob[2][e], xq, xd)


def abs_weights(orc, fmt, ob, e):
    """|W| of expert e dequantised in fp64 [N, K]."""
    if fmt == "q4_0":
        v = orc.unpack_q4_0(ob[0][e]).astype(np.float64)
        d = np.repeat(ob[1][e].view(np.float16).astype(np.float64), 32, axis=1)
        return np.abs(v * d)
    v = orc.unpack_nvfp4(ob[0][e]).astype(np.float64)
    s = np.repeat(orc.e4m3_to_f32(ob[1][e]).astype(np.float64), 16, axis=1)
    return np.abs(0.5 * float(ob[2][e]) * s * v)


@pytest.mark.parametrize("fmt", ["q4_0", "nvfp4"])
@pytest.mark.parametrize("T", [1, 5])
def test_layer_matches_oracle(mem, orc, fmt, T):
    seed = 830 if fmt == "q4_0" else 831
    gu, dn = banks(mem, fmt, seed)
    gu_o, dn_o = oracle_banks(orc, fmt, seed)
    assert_bank_equal(fmt, gu, gu_o)
    assert_bank_equal(fmt, dn, dn_o)
    routes = [synth.routing(E, TOP_K, seed + 2, t) for t in range(T)]
    ids = torch.stack([r[0] for r in routes])
    gw = torch.stack([r[1] for r in routes])
    x = synth.activations_bf16(T, H, seed + 3, outlier_frac=0.001)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    if T == 1:
        ws = torch.empty((TOP_K * 2 * F,), device="cuda")
        y = layer(mem, fmt, gu, dn, ids[0].cuda(), gw[0].cuda(), x[0].cuda(), workspace=ws,
                  dev_status=st)[None]
    else:
        ws = torch.empty((T * TOP_K * (2 * F + H),), device="cuda")
        y = layer(mem, fmt, gu, dn, ids.cuda(), gw.cuda(), x.cuda(), workspace=ws,
                  dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ygu = np_(ws[:T * TOP_K * 2 * F]).reshape(T, TOP_K, 2 * F)
    y = np_(y)
    for t in range(T):
        xq, xd = orc.quantize_q8_1(bf16_bits_np(x[t:t + 1]))
        sel = np_(ids[t])
        g = np_(gw[t])
        # gate|up: every selected expert's rows within the product tolerance
        pr = [oracle_product(orc, fmt, gu_o, e, xq, xd) for e in sel]
        ygu_ref = np.stack([p[0][0] for p in pr])
        tol = 1e-4 * np.stack([p[1][0] for p in pr]) + 1e-6
        if T > 1:  # the batched layer keeps the gate|up rows
            assert_within(ygu[t], ygu_ref, np.stack([p[1][0] for p in pr]),
                          "%s gate|up t=%d" % (fmt, t))
        else:
            # the single-token layer keeps [silu(g) u | u]: the up rows within the
            # product tolerance, the SwiGLU rows within what the tolerances of g and u
            # allow (|silu'| <= 1.1) plus a few roundings
            assert_within(ygu[t][:, F:], ygu_ref[:, F:], np.stack([p[1][0] for p in pr])[:, F:],
                          "%s up t=%d" % (fmt, t))
            gr = ygu_ref[:, :F].astype(np.float64)
            ur = ygu_ref[:, F:].astype(np.float64)
            h_ref = orc.swiglu(ygu_ref).astype(np.float64)
            tg, tu = tol[:, :F], tol[:, F:]
            bound = (1.1 * tg * (np.abs(ur) + tu) + (np.abs(gr / (1 + np.exp(-gr))) + 1.1 * tg) * tu
                     + 1e-6 * np.abs(h_ref) + 1e-30)
            err = np.abs(ygu[t][:, :F].astype(np.float64) - h_ref)
            assert np.all(err <= bound), (fmt, "swiglu rows", float((err - bound).max()))
        # down from the oracle's own SwiGLU rows; gated sum in ascending k from 0
        hq, hd = orc.swiglu_quantize_q8_1(ygu_ref)
        y_ref = np.zeros(H, np.float32)
        bound = np.zeros(H)
        for k, e in enumerate(sel):
            yk = oracle_product(orc, fmt, dn_o, e, hq[k:k + 1], hd[k:k + 1])[0][0]
            y_ref = (y_ref + np.float32(g[k]) * yk).astype(np.float32)
            # the GPU requantises its own gate|up rows: each h may sit one step away
            bound += float(g[k]) * (abs_weights(orc, fmt, dn_o, e) @
                                    np.repeat(2.0 * hd[k].astype(np.float64), 32))
        err = np.abs(y[t].astype(np.float64) - y_ref)
        assert np.all(err <= bound + 1e-4 * np.abs(y_ref).max() + 1e-6), (fmt, t)
