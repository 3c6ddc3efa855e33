"""Parity at the workloads' full sizes, built and launched exactly as bench.py does.

Outputs the oracle can compute one by one are sampled (first and last rows plus
seeded random rows); properties that hold at any size are checked on everything.
The oracle gets the fp32 weights and bf16 activations from the input generator,
never a value the GPU produced."""
import numpy as np
import pytest
import torch

import bench
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


def sample_rows(N, n_random=48, seed=0):
    g = np.random.default_rng(seed)
    rows = set(range(min(8, N))) | set(range(max(0, N - 8), N))
    rows |= set(g.choice(N, size=min(n_random, N), replace=False).tolist())
    return np.array(sorted(rows))


def check_sampled(orc, w_dev, wq, wd, x_cpu, y, rows, what):
    """Oracle on the sampled rows of an fp32 weight tensor on the GPU."""
    w_rows = w_dev[torch.as_tensor(rows, device=w_dev.device)].cpu().numpy()
    oq, od = orc.quantize_q8_0(w_rows)
    idx = torch.as_tensor(rows, device=wq.device)
    assert np.array_equal(np_(wq[idx]), oq), what + ": weight quants"
    assert np.array_equal(wd_bits(wd[idx]), od), what + ": weight scales"
    oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x_cpu))
    y_ref = orc.gemm(oq, od, oxq, oxd)
    terms = abs_terms(orc.block_dots(oq, oxq), od, oxd)
    assert_within(np_(y)[:, rows], y_ref, terms, what)
    return oxq, oxd


def test_gemv_4096_full(mem, orc):
    c = synth.GEMV_4096
    w = synth.weights_fp32(c["N"], c["K"], c["seed"], device="cuda")
    wq, wd = mem.memra_quantize_q8_0(w)
    x = synth.activations_bf16(1, c["K"], c["seed"], 1, device="cuda")
    op = bench.Gemv(wq, wd, x, "gemv_4096")
    bench.run_gemv_op(mem, op)
    torch.cuda.synchronize()
    check_sampled(orc, w, wq, wd, x.cpu(), op.y, np.arange(c["N"]), "4096x4096 (all rows)")


@pytest.mark.parametrize("layer", [0, 63])
@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_dense27b_layer_sampled(mem, orc, layer, M):
    cfg = synth.DENSE27B
    wid = 1 if M == 1 else 2
    for t, (name, N, K) in enumerate(cfg["gemvs"]):
        w = synth.weights_fp32(N, K, wid, layer, t, device="cuda")
        wq, wd = mem.memra_quantize_q8_0(w)
        x = synth.activations_bf16(M, K, wid, layer, t, 1000 + M,
                                   outlier_frac=cfg["outlier_frac"],
                                   outlier_scale=cfg["outlier_scale"], device="cuda")
        op = bench.Gemv(wq, wd, x, name)
        bench.run_gemv_op(mem, op)
        torch.cuda.synchronize()
        # 0.1% outliers: exactly round(0.001 K) entries per row are scaled
        assert int((x.abs() > 8).sum(dim=1).max()) <= round(0.001 * K) + 8
        check_sampled(orc, w, wq, wd, x.cpu(), op.y, sample_rows(N, seed=layer * 10 + t),
                      "L%d %s M=%d" % (layer, name, M))
        del w, wq, wd, op
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layer", [0, 63])
def test_dense27b_q4_0_layer_sampled(mem, orc, layer):
    """The Q4_0 sweep as bench.py builds it: sampled rows against the oracle."""
    cfg = synth.DENSE27B
    for t, (name, N, K) in enumerate(cfg["gemvs"]):
        wq4, wd = bench.quantized_weights(mem, N, K, 5, layer, t, device="cuda", fmt="q4_0")
        x = synth.activations_bf16(1, K, 5, layer, t, 1001, outlier_frac=cfg["outlier_frac"],
                                   outlier_scale=cfg["outlier_scale"], device="cuda")
        op = bench.Gemv(wq4, wd, x, name)
        assert op.fmt == "q4_0" and op.weight_bytes == N * K // 2 + N * (K // 32) * 2
        bench.run_gemv_op(mem, op)
        torch.cuda.synchronize()
        rows = sample_rows(N, seed=500 + layer * 10 + t)
        w = synth.weights_fp32(N, K, 5, layer, t, device="cuda")
        w_rows = w[torch.as_tensor(rows, device="cuda")].cpu().numpy()
        oq4, od = orc.quantize_q4_0(w_rows)
        idx = torch.as_tensor(rows, device="cuda")
        assert np.array_equal(np_(wq4[idx]), oq4), name + ": packed codes"
        assert np.array_equal(wd_bits(wd[idx]), od), name + ": scales"
        oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x.cpu()))
        y_ref = orc.gemm_q4_0(oq4, od, oxq, oxd)
        terms = abs_terms(orc.block_dots(orc.unpack_q4_0(oq4), oxq), od, oxd)
        assert_within(np_(op.y)[:, rows], y_ref, terms, "q4_0 L%d %s" % (layer, name))
        del w, wq4, wd, op
    torch.cuda.empty_cache()


def test_dense27b_nvfp4_layer_sampled(mem, orc):
    """The NVFP4 sweep's layer 0 as bench.py builds it.  The tensor scale depends on the
    whole matrix, so the oracle quantises each full matrix (from the generator's fp32
    weights on the host) and the products are compared on sampled rows."""
    cfg = synth.DENSE27B
    layer = 0
    for t, (name, N, K) in enumerate(cfg["gemvs"]):
        codes, scales, g = bench.quantized_weights(mem, N, K, 6, layer, t, device="cuda",
                                                   fmt="nvfp4")
        x = synth.activations_bf16(1, K, 6, layer, t, 1001, outlier_frac=cfg["outlier_frac"],
                                   outlier_scale=cfg["outlier_scale"], device="cuda")
        op = bench.Gemv(codes, scales, x, name, fmt="nvfp4", g=g)
        assert op.weight_bytes == N * K // 2 + N * K // 16
        bench.run_gemv_op(mem, op)
        torch.cuda.synchronize()
        # the generator's values as bench.py draws them (on the device), read back whole
        w_host = synth.weights_fp32(N, K, 6, layer, t, device="cuda").cpu().numpy()
        oc, osc, og = orc.quantize_nvfp4(w_host)
        del w_host
        assert np.float32(g).view(np.uint32) == np.float32(og).view(np.uint32), name + ": g"
        rows = sample_rows(N, seed=600 + t)
        idx = torch.as_tensor(rows, device="cuda")
        assert np.array_equal(np_(codes[idx]), oc[rows]), name + ": codes"
        assert np.array_equal(np_(scales[idx]), osc[rows]), name + ": scales"
        oxq, oxd = orc.quantize_q8_1(bf16_bits_np(x.cpu()))
        y_ref = orc.gemm_nvfp4(oc[rows], osc[rows], og, oxq, oxd)
        c2 = orc.unpack_nvfp4(oc[rows]).astype(np.float64).reshape(len(rows), K // 16, 16)
        S = np.einsum("nbi,bi->nb", c2, oxq[0].astype(np.float64).reshape(K // 16, 16))
        terms = np.abs(0.5 * float(og) * orc.e4m3_to_f32(osc[rows]).astype(np.float64) *
                       np.repeat(oxd[0].astype(np.float64), 2)[None] * S).sum(axis=1)
        assert_within(np_(op.y)[:, rows], y_ref, terms[None], "nvfp4 L0 %s" % name)
        # and against the plain definition, summed element by element in fp64
        y64 = orc.nvfp4_dequant_gemm_f64(oc[rows], osc[rows], og, oxq, oxd)
        assert_within(np_(op.y)[:, rows], y64, terms[None], "nvfp4 L0 %s (fp64)" % name)
        del codes, scales, op, oc, osc
    torch.cuda.empty_cache()


def test_moe_layer_full_size(mem, orc):
    """One routed layer of the 128-expert MoE (hidden 2048, expert FFN 768, top-8)."""
    c = synth.MOE
    E, H, F, k = c["experts"], c["hidden"], c["ffn"], c["top_k"]
    layer = 5
    lay = bench.MoeLayer(mem, layer, torch.device("cuda"))
    lay.run(mem)
    torch.cuda.synchronize()
    assert int(lay.status.item()) == 0
    ids = np_(lay.ids)
    gw = np_(lay.gw)
    assert len(set(ids.tolist())) == k and abs(float(gw.sum()) - 1.0) < 1e-6
    wgu = synth.weights_fp32(E * 2 * F, H, 3, layer, 0, device="cuda").view(E, 2 * F, H)
    wdn = synth.weights_fp32(E * H, F, 3, layer, 1, device="cuda").view(E, H, F)
    sel = torch.as_tensor(ids.astype(np.int64), device="cuda")
    gq_o, gd_o = orc.quantize_q8_0(wgu[sel].reshape(-1, H).cpu().numpy())
    dq_o, dd_o = orc.quantize_q8_0(wdn[sel].reshape(-1, F).cpu().numpy())
    # the GPU's selected experts match the oracle's quantisation bit for bit
    assert np.array_equal(np_(lay.gq[sel]).reshape(-1, H), gq_o)
    assert np.array_equal(np_(lay.dq[sel]).reshape(-1, F), dq_o)
    gq_o = gq_o.reshape(k, 2 * F, H)
    gd_o = gd_o.reshape(k, 2 * F, H // 32)
    dq_o = dq_o.reshape(k, H, F)
    dd_o = dd_o.reshape(k, H, F // 32)
    local = np.arange(k, dtype=np.int32)   # the oracle's bank holds only the selected experts
    xq, xd = orc.quantize_q8_1(bf16_bits_np(lay.x.cpu()))
    ygu_ref, _ = orc.moe_gemv(gq_o, gd_o, local, None, xq, xd, 0)
    terms = np.stack([abs_terms(orc.block_dots(gq_o[i], xq), gd_o[i], xd)[0] for i in range(k)])
    assert_within(np_(lay.ygu), ygu_ref, terms, "moe gate/up")
    # stage-wise down projection from the oracle's own h
    hq, hd = orc.swiglu_quantize_q8_1(ygu_ref)
    y_ref, _ = orc.moe_gemv(dq_o, dd_o, local, gw, hq, hd, 1)
    y_full = orc.moe_ffn(np_(lay.x.float())[0], gq_o, gd_o, dq_o, dd_o, local, gw)[0]
    assert np.array_equal(y_ref, y_full)
    bound = np.zeros(H)
    for i in range(k):
        wabs = np.abs(dq_o[i].astype(np.float64) *
                      np.repeat(dd_o[i].view(np.float16).astype(np.float64), 32, axis=1))
        bound += float(gw[i]) * (wabs @ np.repeat(2.0 * hd[i].astype(np.float64), 32))
    err = np.abs(np_(lay.y).astype(np.float64) - y_ref)
    assert np.all(err <= bound + 1e-4 * np.abs(y_ref).max() + 1e-6)


@pytest.mark.parametrize("M", [1, 8])
def test_stress_shapes(mem, orc, M):
    s = synth.STRESS
    for t, (name, N, K) in enumerate(s["shapes"]):
        w = synth.weights_fp32(N, K, 4, t, device="cuda")
        zero_ids, scale_ids = synth.perturb_blocks(w, 4, t, zero_frac=s["zero_frac"],
                                                   scale_frac=s["scale_frac"], scale=s["scale"])
        wq, wd = mem.memra_quantize_q8_0(w)
        x = synth.activations_bf16(M, K, 4, t, 1000 + M, device="cuda")
        op = bench.Gemv(wq, wd, x, name)
        bench.run_gemv_op(mem, op)
        torch.cuda.synchronize()
        nblocks = N * (K // 32)
        # properties over the whole matrix: the zeroed blocks have d = 0 and q = 0
        flat_d = wd.view(-1)
        assert int((flat_d[zero_ids] == 0).sum()) == len(zero_ids) == round(0.01 * nblocks)
        assert int(wq.view(nblocks, 32)[zero_ids].abs().sum()) == 0
        assert bool(torch.all(flat_d[scale_ids].float() > 0))
        assert bool(torch.isfinite(op.y).all())
        rows = sample_rows(N, seed=100 + t)
        zrows = (zero_ids[:16] // (K // 32)).cpu().numpy()
        srows = (scale_ids[:16] // (K // 32)).cpu().numpy()
        rows = np.unique(np.concatenate([rows, zrows, srows]))
        check_sampled(orc, w, wq, wd, x.cpu(), op.y, rows, "%s M=%d" % (name, M))
        del w, wq, wd, op
        torch.cuda.empty_cache()
