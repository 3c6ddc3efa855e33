"""Pins for the CPU oracle: closed forms, invariants, brute force and library routines.

None of these checks recomputes the oracle's own formula: each compares it with
something fixed independently (numpy's IEEE binary16 conversion, int64 / fp64
brute force, libm's exp, exact special cases), chosen so that a dropped term, a
wrong sign, a wrong block index or a transposed operand fails at least one test.
"""

import numpy as np
import pytest

U32 = 2.0 ** -24  # fp32 unit roundoff


def rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------
# Scalar conversions against numpy (IEEE 754 binary16, round to nearest even).
# ----------------------------------------------------------------------------

def test_f16_to_f32_exhaustive(orc):
    codes = np.arange(65536, dtype=np.uint16)
    ours = orc.f16_bits_to_f32(codes)
    ref = codes.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_ties_and_random(orc):
    finite = np.arange(0x7C00, dtype=np.uint16)          # +0 .. max finite
    hv = finite.view(np.float16).astype(np.float64)
    mids = ((hv[:-1] + hv[1:]) / 2).astype(np.float32)  # exact ties between neighbours
    assert np.array_equal(mids.astype(np.float64), (hv[:-1] + hv[1:]) / 2)
    r = rng(1)
    rand_bits = r.integers(0, 2 ** 32, size=40000, dtype=np.uint64).astype(np.uint32)
    rand = rand_bits.view(np.float32)
    rand = rand[np.isfinite(rand)]
    logs = (r.uniform(-30, 17, size=20000)).astype(np.float64)
    scaled = (np.sign(r.standard_normal(20000)) * 2.0 ** logs).astype(np.float32)
    specials = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 70000.0, 2 ** -24, 2 ** -25,
                         1.5 * 2 ** -25, 2 ** -14, np.inf, -np.inf, 1e-30, 3.0e38],
                        dtype=np.float32)
    vals = np.concatenate([mids, -mids, hv.astype(np.float32), rand, scaled, specials])
    ours = orc.f32_to_f16_bits(vals)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_to_f32_matches_torch(orc):
    torch = pytest.importorskip("torch")
    codes = np.arange(0, 65536, 7, dtype=np.uint16)
    ours = orc.bf16_bits_to_f32(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ----------------------------------------------------------------------------
# Quantisers.
# ----------------------------------------------------------------------------

def _hand_block():
    # amax = 127 gives d = 1 exactly for both quantisers (127/127 is exact and 1.0 is
    # an fp16 number), so q is round-half-away of the value itself.
    v = np.zeros(32, np.float32)
    v[:10] = [127.0, 63.5, -63.5, 2.5, -2.5, 0.5, -0.5, 0.49, -126.6, 1.5]
    q = np.zeros(32, np.int8)
    q[:10] = [127, 64, -64, 3, -3, 1, -1, 0, -127, 2]
    return v, q


def test_quantizers_hand_worked_block(orc):
    v, q = _hand_block()
    wq, wd = orc.quantize_q8_0(v[None, :])
    assert wd[0, 0] == 0x3C00  # fp16 1.0
    assert np.array_equal(wq[0], q)
    xq, xd = orc.quantize_q8_1(v[None, :])
    assert xd[0, 0] == np.float32(1.0)
    assert np.array_equal(xq[0], q)
    # bf16 input: every value above is exactly representable in bf16 except 0.49 and -126.6
    torch = pytest.importorskip("torch")
    bits = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xq_b, xd_b = orc.quantize_q8_1(bits[None, :])
    assert xd_b[0, 0] == np.float32(1.0)
    assert np.array_equal(xq_b[0], q)


def test_zero_block_gives_zero_scale_and_quants(orc):
    w = np.zeros((2, 64), np.float32)
    w[1, 32:] = rng(2).standard_normal(32).astype(np.float32)
    wq, wd = orc.quantize_q8_0(w)
    assert wd[0, 0] == 0 and wd[0, 1] == 0 and wd[1, 0] == 0 and wd[1, 1] != 0
    assert not wq[0].any() and not wq[1, :32].any()
    xq, xd = orc.quantize_q8_1(w)
    assert xd[0, 0] == 0 and xd[1, 0] == 0 and xd[1, 1] > 0
    assert not xq[0].any() and not xq[1, :32].any()


@pytest.mark.parametrize("std", [0.02, 1.0, 300.0])
def test_weight_quant_invariants(orc, std):
    r = rng(3)
    w = (r.standard_normal((64, 256)) * std).astype(np.float32)
    wq, wd = orc.quantize_q8_0(w)
    d = wd.view(np.float16).astype(np.float64)
    assert wq.min() >= -127 and wq.max() <= 127
    deq = np.repeat(d, 32, axis=1) * wq
    err = np.abs(w.astype(np.float64) - deq)
    assert np.all(err <= np.repeat(d, 32, axis=1) / 2 * (1 + 1e-6))
    # the largest |w| in a block maps to +-127 (fp16 rounding of d moves amax/d by
    # at most 2^-11 * 127 < 0.5)
    blocks = np.abs(w).reshape(64, 8, 32)
    idx = blocks.argmax(axis=2)
    qb = np.abs(wq.reshape(64, 8, 32))
    assert np.all(np.take_along_axis(qb, idx[..., None], axis=2) == 127)
    # the scale is the fp16 value nearest amax/127 (checked with numpy's conversion)
    amax = blocks.max(axis=2).astype(np.float32)
    ref_d = (amax / np.float32(127.0)).astype(np.float16).view(np.uint16)
    assert np.array_equal(wd, ref_d)


def test_weight_quant_subnormal_scale_clamps(orc):
    # amax tiny enough that fp16(amax/127) is subnormal and rounds DOWN by a lot:
    # amax/127 = 1.4 * 2^-24 rounds to 2^-24, so amax/d = 177.8 -> clamped to 127.
    amax = np.float32(1.4 * 2 ** -24 * 127)
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = amax
    w[0, 1] = -amax / 2
    w[0, 2] = amax / 200
    wq, wd = orc.quantize_q8_0(w)
    assert wd[0, 0] == 1  # smallest subnormal
    assert wq[0, 0] == 127
    d = 2.0 ** -24
    assert wq[0, 1] == -round(float(amax) / 2 / d + 0.0)  # 88.9 -> -89
    assert wq[0, 2] == round(float(amax) / 200 / d)       # 0.889 -> 1


@pytest.mark.parametrize("std", [1.0, 1e-3, 1e4])
def test_activation_quant_invariants(orc, std):
    r = rng(4)
    x = (r.standard_normal((8, 512)) * std).astype(np.float32)
    x[0, :32] = 0.0
    xq, xd = orc.quantize_q8_1(x)
    assert xq.min() >= -127 and xq.max() <= 127
    amax = np.abs(x).reshape(8, 16, 32).max(axis=2)
    # d is the IEEE fp32 quotient amax / 127
    assert np.array_equal(xd, (amax / np.float32(127.0)).astype(np.float32))
    d = np.repeat(xd.astype(np.float64), 32, axis=1)
    err = np.abs(x.astype(np.float64) - d * xq)
    assert np.all(err <= d / 2 * (1 + 1e-6))
    idx = np.abs(x).reshape(8, 16, 32).argmax(axis=2)
    qb = np.abs(xq.reshape(8, 16, 32))
    hit = np.take_along_axis(qb, idx[..., None], axis=2)[..., 0]
    assert np.all(hit[amax > 0] == 127)


def test_quant_power_of_two_scaling(orc):
    r = rng(5)
    x = r.standard_normal((4, 128)).astype(np.float32)
    q1, d1 = orc.quantize_q8_1(x)
    for k in (-5, 1, 7):
        q2, d2 = orc.quantize_q8_1(x * np.float32(2.0 ** k))
        assert np.array_equal(q1, q2)
        assert np.array_equal(d2, d1 * np.float32(2.0 ** k))
    w = (r.standard_normal((4, 128)) * 0.02).astype(np.float32)
    wq1, wd1 = orc.quantize_q8_0(w)
    wq2, wd2 = orc.quantize_q8_0(w * np.float32(4.0))
    assert np.array_equal(wq1, wq2)
    assert np.array_equal(wd2.view(np.float16).astype(np.float32),
                          wd1.view(np.float16).astype(np.float32) * 4)


def test_quant_sign_symmetry(orc):
    r = rng(6)
    x = r.standard_normal((3, 96)).astype(np.float32)
    q1, d1 = orc.quantize_q8_1(x)
    q2, d2 = orc.quantize_q8_1(-x)
    assert np.array_equal(q2, -q1) and np.array_equal(d1, d2)


# ----------------------------------------------------------------------------
# Block dots and the GEMV / skinny GEMM.
# ----------------------------------------------------------------------------

def _rand_q(r, shape):
    return r.integers(-127, 128, size=shape).astype(np.int8)


def test_block_dots_int64_brute_force(orc):
    r = rng(7)
    N, K, M = 5, 160, 3
    wq = _rand_q(r, (N, K))
    xq = _rand_q(r, (M, K))
    s = orc.block_dots(wq, xq)
    ref = np.einsum("nbi,mbi->mnb", wq.reshape(N, K // 32, 32).astype(np.int64),
                    xq.reshape(M, K // 32, 32).astype(np.int64))
    assert np.array_equal(s.astype(np.int64), ref)
    # extreme block: every product 127*127 (or -127*-127)
    s2 = orc.block_dots(np.full((1, 32), -127, np.int8), np.full((1, 32), -127, np.int8))
    assert s2[0, 0, 0] == 32 * 127 * 127


def _case(seed, N, K, M, wstd=0.02):
    r = rng(seed)
    w = (r.standard_normal((N, K)) * wstd).astype(np.float32)
    x = r.standard_normal((M, K)).astype(np.float32)
    return w, x


def _abs_terms(orc, wq, wd, xq, xd):
    s = orc.block_dots(wq, xq).astype(np.float64)  # [M, N, nb]
    c = wd.view(np.float16).astype(np.float64)[None, :, :] * xd.astype(np.float64)[:, None, :]
    return np.abs(c * s).sum(axis=2)  # [M, N]


@pytest.mark.parametrize("N,K,M", [(7, 32, 1), (33, 544, 1), (16, 5120, 2), (9, 768, 8)])
def test_gemm_within_bound_of_fp64_brute_force(orc, N, K, M):
    w, x = _case(8 + K, N, K, M)
    wq, wd = orc.quantize_q8_0(w)
    xq, xd = orc.quantize_q8_1(x)
    y = orc.gemm(wq, wd, xq, xd)
    # independent fp64 brute force in numpy (dequantise, then matmul)
    Wd = wq.astype(np.float64) * np.repeat(wd.view(np.float16).astype(np.float64), 32, axis=1)
    Xd = xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 32, axis=1)
    y64 = Xd @ Wd.T
    # the C fp64 brute force agrees with numpy
    assert np.allclose(orc.dequant_gemm_f64(wq, wd, xq, xd), y64, rtol=1e-12, atol=1e-300)
    nb = K // 32
    gamma = (nb + 2) * U32 / (1 - (nb + 2) * U32)  # sequential-sum rounding bound
    bound = gamma * _abs_terms(orc, wq, wd, xq, xd)
    assert np.all(np.abs(y.astype(np.float64) - y64) <= bound + 1e-30)
    # and the stated parity tolerance holds a fortiori
    assert np.all(np.abs(y - y64) <= 1e-4 * _abs_terms(orc, wq, wd, xq, xd) + 1e-6)


def test_gemm_close_to_unquantized_product(orc):
    N, K, M = 24, 1024, 2
    w, x = _case(9, N, K, M)
    wq, wd = orc.quantize_q8_0(w)
    xq, xd = orc.quantize_q8_1(x)
    y = orc.gemm(wq, wd, xq, xd).astype(np.float64)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    dw = np.repeat(wd.view(np.float16).astype(np.float64), 32, axis=1)
    dx = np.repeat(xd.astype(np.float64), 32, axis=1)
    Wd = wq * dw
    Xd = xq * dx
    # |wx - w'x'| <= |w'| dx/2 + |x'| dw/2 + dw dx/4 elementwise
    qerr = (np.abs(Xd) @ (dw / 2).T + (dx / 2) @ np.abs(Wd).T + (dx / 2) @ (dw / 2).T)
    fperr = 1e-4 * _abs_terms(orc, wq, wd, xq, xd) + 1e-6
    assert np.all(np.abs(y - exact) <= qerr + fperr)


def test_gemm_one_hot_activation_exact(orc):
    r = rng(10)
    N, K = 6, 96
    w = (r.standard_normal((N, K)) * 0.02).astype(np.float32)
    wq, wd = orc.quantize_q8_0(w)
    for j in (0, 31, 32, 77, 95):
        x = np.zeros((1, K), np.float32)
        x[0, j] = 3.0
        xq, xd = orc.quantize_q8_1(x)
        assert xq[0, j] == 127 and np.count_nonzero(xq) == 1
        y = orc.gemm(wq, wd, xq, xd)[0]
        dw = wd[:, j // 32].view(np.float16).astype(np.float32)
        # single nonzero block sum s = 127 * q_w: y = fl(fl(d_w * d_x) * s)
        c = (dw * xd[0, j // 32]).astype(np.float32)
        expect = c * (np.int32(127) * wq[:, j].astype(np.int32)).astype(np.float32)
        assert np.array_equal(y, expect.astype(np.float32))


def test_gemm_power_of_two_linearity_exact(orc):
    w, x = _case(11, 12, 320, 2)
    wq, wd = orc.quantize_q8_0(w)
    xq, xd = orc.quantize_q8_1(x)
    y1 = orc.gemm(wq, wd, xq, xd)
    xq2, xd2 = orc.quantize_q8_1(x * np.float32(8.0))
    y2 = orc.gemm(wq, wd, xq2, xd2)
    assert np.array_equal(y2, y1 * np.float32(8.0))


def test_gemm_additivity_within_quantization_bound(orc):
    r = rng(12)
    N, K = 10, 256
    w = (r.standard_normal((N, K)) * 0.02).astype(np.float32)
    x1 = r.standard_normal((1, K)).astype(np.float32)
    x2 = r.standard_normal((1, K)).astype(np.float32)
    wq, wd = orc.quantize_q8_0(w)
    ys = []
    for x in (x1, x2, x1 + x2):
        xq, xd = orc.quantize_q8_1(x)
        ys.append(orc.gemm(wq, wd, xq, xd)[0].astype(np.float64))
    dw = np.repeat(wd.view(np.float16).astype(np.float64), 32, axis=1)
    Wd = wq * dw

    def qbound(x):
        _, xd = orc.quantize_q8_1(x)
        return np.abs(Wd) @ (np.repeat(xd.astype(np.float64), 32, axis=1)[0] / 2)

    tol = qbound(x1) + qbound(x2) + qbound(x1 + x2) + 1e-5
    assert np.all(np.abs(ys[2] - ys[0] - ys[1]) <= tol)


def test_gemm_row_permutation_exact(orc):
    w, x = _case(13, 20, 192, 1)
    wq, wd = orc.quantize_q8_0(w)
    xq, xd = orc.quantize_q8_1(x)
    y = orc.gemm(wq, wd, xq, xd)
    p = rng(14).permutation(20)
    yp = orc.gemm(wq[p], wd[p], xq, xd)
    assert np.array_equal(yp, y[:, p])


def test_gemm_zero_blocks(orc):
    w, x = _case(15, 8, 256, 1)
    w[3, :] = 0.0
    x[0, 64:96] = 0.0
    wq, wd = orc.quantize_q8_0(w)
    xq, xd = orc.quantize_q8_1(x)
    y = orc.gemm(wq, wd, xq, xd)
    assert y[0, 3] == 0.0
    keep = np.r_[0:64, 96:256]
    keep_b = np.r_[0:2, 3:8]
    y_cut = orc.gemm(wq[:, keep], wd[:, keep_b], xq[:, keep], xd[:, keep_b])
    assert np.array_equal(y, y_cut)


def test_gemm_rows_independent_of_m_and_threads(orc):
    w, x = _case(16, 40, 640, 8)
    wq, wd = orc.quantize_q8_0(w)
    xq, xd = orc.quantize_q8_1(x)
    y8 = orc.gemm(wq, wd, xq, xd)
    for m in range(8):
        y1 = orc.gemm(wq, wd, xq[m:m + 1], xd[m:m + 1])
        assert np.array_equal(y1[0], y8[m])
    assert np.array_equal(orc.gemm(wq, wd, xq, xd, threads=4), y8)


# ----------------------------------------------------------------------------
# exp, SwiGLU and the routed-expert GEMV.
# ----------------------------------------------------------------------------

def test_exp_cw_against_libm(orc):
    xs = np.concatenate([np.linspace(-87.0, 88.0, 20001, dtype=np.float32),
                         np.array([0.0, -0.0, 1e-8, -1e-8, 0.5, -0.5, 1.0], np.float32)])
    ours = orc.exp_cw(xs).astype(np.float64)
    ref = np.exp(xs.astype(np.float64))
    rel = np.abs(ours - ref) / ref
    assert rel.max() < 4 * U32 * 2  # within a few fp32 ulp
    assert orc.exp_cw(np.array([0.0], np.float32))[0] == 1.0
    # clamped outside [-87, 88]
    assert orc.exp_cw(np.array([200.0], np.float32))[0] == orc.exp_cw(np.array([88.0],
                                                                              np.float32))[0]


def test_swiglu_against_fp64(orc):
    r = rng(17)
    R, F = 3, 96
    gu = (r.standard_normal((R, 2 * F)) * 4).astype(np.float32)
    gu[0, :5] = [0.0, -30.0, 30.0, -90.0, 1e-3]
    h = orc.swiglu(gu).astype(np.float64)
    g = gu[:, :F].astype(np.float64)
    u = gu[:, F:].astype(np.float64)
    ref = g / (1 + np.exp(-g)) * u
    assert np.all(np.abs(h - ref) <= 1e-6 * np.abs(ref) + 1e-30 + 1e-36 * np.abs(u))
    # gate half really is the first half: silu(g)*u is not symmetric in (g, u)
    swapped = u / (1 + np.exp(-u)) * g
    assert not np.allclose(h, swapped)


def test_swiglu_quantize_is_quantize_of_swiglu(orc):
    r = rng(18)
    gu = r.standard_normal((4, 2 * 64)).astype(np.float32)
    hq, hd = orc.swiglu_quantize_q8_1(gu)
    q2, d2 = orc.quantize_q8_1(orc.swiglu(gu))
    assert np.array_equal(hq, q2) and np.array_equal(hd, d2)


def _bank(seed, E, N, K):
    r = rng(seed)
    w = (r.standard_normal((E, N, K)) * 0.02).astype(np.float32)
    wq = np.empty((E, N, K), np.int8)
    wd = np.empty((E, N, K // 32), np.uint16)
    return w, wq, wd


def test_moe_gemv_reduces_to_plain_gemv(orc):
    E, N, K = 5, 24, 128
    w, wq, wd = _bank(19, E, N, K)
    for e in range(E):
        wq[e], wd[e] = orc.quantize_q8_0(w[e])
    r = rng(20)
    x = r.standard_normal((3, K)).astype(np.float32)
    xq, xd = orc.quantize_q8_1(x)
    ids = np.array([4, 0, 2], np.int32)
    # ungated, per-expert activations: row k is the plain GEMV of expert ids[k]
    y, bad = orc.moe_gemv(wq, wd, ids, None, xq, xd, 1)
    assert bad == 0
    for k, e in enumerate(ids):
        assert np.array_equal(y[k], orc.gemm(wq[e], wd[e], xq[k:k + 1], xd[k:k + 1])[0])
    # ungated, shared activation
    y, _ = orc.moe_gemv(wq, wd, ids, None, xq[:1], xd[:1], 0)
    for k, e in enumerate(ids):
        assert np.array_equal(y[k], orc.gemm(wq[e], wd[e], xq[:1], xd[:1])[0])
    # top-1 with weight 1: the gated sum is that expert's GEMV exactly
    y1, _ = orc.moe_gemv(wq, wd, ids[:1], np.ones(1, np.float32), xq[:1], xd[:1], 0)
    assert np.array_equal(y1, orc.gemm(wq[4], wd[4], xq[:1], xd[:1])[0])


def test_moe_gemv_gated_sum_against_fp64(orc):
    E, N, K = 6, 16, 96
    w, wq, wd = _bank(21, E, N, K)
    for e in range(E):
        wq[e], wd[e] = orc.quantize_q8_0(w[e])
    r = rng(22)
    x = r.standard_normal((4, K)).astype(np.float32)
    xq, xd = orc.quantize_q8_1(x)
    ids = np.array([5, 1, 3, 1], np.int32)
    gw = np.array([0.4, 0.3, 0.2, 0.1], np.float32)
    y, bad = orc.moe_gemv(wq, wd, ids, gw, xq, xd, 1)
    assert bad == 0
    ref = np.zeros(N)
    tol = np.zeros(N)
    for k, e in enumerate(ids):
        ref += gw[k] * orc.dequant_gemm_f64(wq[e], wd[e], xq[k:k + 1], xd[k:k + 1])[0]
        tol += abs(gw[k]) * _abs_terms(orc, wq[e], wd[e], xq[k:k + 1], xd[k:k + 1])[0]
    assert np.all(np.abs(y - ref) <= 1e-4 * tol + 1e-6)


def test_moe_gemv_out_of_range_ids(orc):
    E, N, K = 3, 8, 64
    w, wq, wd = _bank(23, E, N, K)
    for e in range(E):
        wq[e], wd[e] = orc.quantize_q8_0(w[e])
    xq, xd = orc.quantize_q8_1(rng(24).standard_normal((1, K)).astype(np.float32))
    ids = np.array([1, 3, -1], np.int32)
    y, bad = orc.moe_gemv(wq, wd, ids, None, xq, xd, 0)
    assert bad == 2
    assert not y[1].any() and not y[2].any()
    assert np.array_equal(y[0], orc.gemm(wq[1], wd[1], xq, xd)[0])
    yg, bad = orc.moe_gemv(wq, wd, ids, np.array([1.0, 5.0, 7.0], np.float32), xq, xd, 0)
    assert bad == 2 and np.array_equal(yg, y[0])


def test_moe_ffn_single_expert_is_dense_ffn(orc):
    # E = 1, top_k = 1, weight 1: the layer is a dense SwiGLU FFN with Q8_0 weights.
    K, F, N_out = 64, 32, 64
    r = rng(25)
    wgu = (r.standard_normal((1, 2 * F, K)) * 0.05).astype(np.float32)
    wdn = (r.standard_normal((1, N_out, F)) * 0.05).astype(np.float32)
    gq, gd = orc.quantize_q8_0(wgu[0])
    dq, dd = orc.quantize_q8_0(wdn[0])
    x = r.standard_normal(K).astype(np.float32)
    y, bad = orc.moe_ffn(x, gq[None], gd[None], dq[None], dd[None], np.zeros(1, np.int32),
                         np.ones(1, np.float32))
    assert bad == 0
    xq, xd = orc.quantize_q8_1(x[None])
    hgu = orc.gemm(gq, gd, xq, xd)
    hq, hd = orc.swiglu_quantize_q8_1(hgu)
    ref = orc.gemm(dq, dd, hq, hd)[0]
    assert np.array_equal(y, ref)
    # and it tracks the unquantised fp64 FFN to within quantisation-level error
    xf = x.astype(np.float64)
    g_u = wgu[0].astype(np.float64) @ xf
    h = g_u[:F] / (1 + np.exp(-g_u[:F])) * g_u[F:]
    y64 = wdn[0].astype(np.float64) @ h
    assert np.max(np.abs(y - y64)) < 0.05 * np.max(np.abs(y64)) + 1e-6


# ----------------------------------------------------------------------------
# Q4_0 weights: packing, quantiser invariants and the product.
# ----------------------------------------------------------------------------

def _np_unpack_q4_0(q4):
    """Independent numpy unpack: byte j of a block -> element j (low nibble) and
    element j + 16 (high nibble); values q - 8."""
    N, K2 = q4.shape
    b = q4.reshape(N, K2 // 16, 16).astype(np.int16)
    lo = (b & 0x0F) - 8
    hi = (b >> 4) - 8
    return np.concatenate([lo, hi], axis=2).reshape(N, 2 * K2).astype(np.int8)


def test_q4_0_unpack_matches_hand_packing(orc):
    r = rng(40)
    codes = r.integers(0, 16, size=(5, 96))
    blocks = codes.reshape(5, 3, 32)
    packed = (blocks[:, :, :16] | (blocks[:, :, 16:] << 4)).astype(np.uint8).reshape(5, 48)
    assert np.array_equal(orc.unpack_q4_0(packed), (codes - 8).astype(np.int8))


@pytest.mark.parametrize("std", [0.02, 1.0, 300.0])
def test_q4_0_quant_invariants(orc, std):
    r = rng(41 + int(std))
    N, K = 40, 256
    w = (r.standard_normal((N, K)) * std).astype(np.float32)
    q4, d = orc.quantize_q4_0(w)
    v = _np_unpack_q4_0(q4).astype(np.int64)          # q - 8
    assert v.min() >= -8 and v.max() <= 7
    dv = d.view(np.float16).astype(np.float64)
    wb = w.astype(np.float64).reshape(N, K // 32, 32)
    vb = v.reshape(N, K // 32, 32)
    # the scale is numpy's fp16 of the first largest-magnitude element over -8
    first = np.argmax(np.abs(wb), axis=2)
    m = np.take_along_axis(wb, first[..., None], axis=2)[..., 0]
    assert np.array_equal(d.view(np.float16), (m / -8.0).astype(np.float32).astype(np.float16))
    # that element maps to -8
    assert np.all(np.take_along_axis(vb, first[..., None], axis=2) == -8)
    # round trip: within d/2 where the quotient is in range, within d where it clamps at +7
    ratio = wb / dv[..., None]
    err = np.abs(wb - dv[..., None] * vb)
    inside = ratio <= 7.5
    assert np.all(err[inside] <= np.abs(dv[..., None] * 0.5 + 0 * wb)[inside] * (1 + 2 ** -20))
    assert np.all(vb[~inside] == 7)
    assert np.all(err[~inside] <= np.abs(dv[..., None] + 0 * wb)[~inside] * (1 + 2 ** -9))


def test_q4_0_zero_block_and_sign_and_scaling(orc):
    r = rng(42)
    w = (r.standard_normal((3, 128)) * 0.5).astype(np.float32)
    w[1, 32:64] = 0.0
    w[2, 64:96] = -0.0
    q4, d = orc.quantize_q4_0(w)
    v = _np_unpack_q4_0(q4)
    assert int(d[1, 1]) == 0 and int(d[2, 2]) == 0          # +0 scale for zero blocks
    assert np.all(v[1, 32:64] == 0) and np.all(v[2, 64:96] == 0)
    # -w: the extreme flips sign, so the scale flips sign and every code is unchanged
    q4n, dn = orc.quantize_q4_0(-w)
    assert np.array_equal(q4n, q4)
    nz = d != 0
    assert np.array_equal(dn[nz], d[nz] ^ 0x8000)
    # 4w: same codes, scales exactly 4x
    q4s, ds = orc.quantize_q4_0(4 * w)
    assert np.array_equal(q4s, q4)
    assert np.array_equal(ds.view(np.float16).astype(np.float64),
                          4 * d.view(np.float16).astype(np.float64))


@pytest.mark.parametrize("N,K,M", [(7, 32, 1), (33, 544, 1), (16, 5120, 2), (9, 768, 8)])
def test_q4_0_gemm_within_bound_of_fp64_brute_force(orc, N, K, M):
    w, x = _case(50 + K, N, K, M)
    q4, wd = orc.quantize_q4_0(w)
    xq, xd = orc.quantize_q8_1(x)
    y = orc.gemm_q4_0(q4, wd, xq, xd)
    v = _np_unpack_q4_0(q4)
    Wd = v.astype(np.float64) * np.repeat(wd.view(np.float16).astype(np.float64), 32, axis=1)
    Xd = xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 32, axis=1)
    y64 = Xd @ Wd.T
    nb = K // 32
    s = np.einsum("mbi,nbi->mnb", xq.astype(np.int64).reshape(M, nb, 32),
                  v.astype(np.int64).reshape(N, nb, 32)).astype(np.float64)
    c = wd.view(np.float16).astype(np.float64)[None] * xd.astype(np.float64)[:, None, :]
    terms = np.abs(c * s).sum(axis=2)
    gamma = (nb + 2) * U32 / (1 - (nb + 2) * U32)
    assert np.all(np.abs(y.astype(np.float64) - y64) <= gamma * terms + 1e-30)
    # against the unquantised product: each weight is within |d|/2 (|d| where it clamps)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    dw = np.abs(np.repeat(wd.view(np.float16).astype(np.float64), 32, axis=1))
    dx = np.repeat(xd.astype(np.float64), 32, axis=1)
    qerr = np.abs(Xd) @ dw.T + (dx / 2) @ np.abs(Wd).T + (dx / 2) @ dw.T
    assert np.all(np.abs(y - exact) <= qerr + 1e-4 * terms + 1e-6)


# ----------------------------------------------------------------------------
# GGUF block arrays -> planes.  numpy's packed structured dtypes lay the blocks out
# independently of the oracle: fp16 scale little-endian, then the quants.
# ----------------------------------------------------------------------------

Q8_0_BLOCK = np.dtype([("d", "<u2"), ("qs", "i1", (32,))])
Q4_0_BLOCK = np.dtype([("d", "<u2"), ("qs", "u1", (16,))])


def test_gguf_block_dtypes_are_packed():
    assert Q8_0_BLOCK.itemsize == 34 and Q4_0_BLOCK.itemsize == 18


@pytest.mark.parametrize("N,K", [(1, 32), (7, 96), (33, 512)])
def test_repack_q8_0_round_trip(orc, N, K):
    r = rng(60 + N)
    w = (r.standard_normal((N, K)) * 0.02).astype(np.float32)
    wq, wd = orc.quantize_q8_0(w)
    aos = np.empty((N, K // 32), Q8_0_BLOCK)
    aos["d"] = wd
    aos["qs"] = wq.reshape(N, K // 32, 32)
    q2, d2 = orc.repack_q8_0(aos.view(np.uint8), N, K)
    assert np.array_equal(q2, wq) and np.array_equal(d2, wd)
    # The dequantised weights by the block definition (d * q, scale from the block's
    # first two bytes) equal those of the planes.
    raw = aos.view(np.uint8).reshape(N, K // 32, 34)
    d_blk = (raw[:, :, 0].astype(np.uint16) | (raw[:, :, 1].astype(np.uint16) << 8))
    deq_blk = d_blk.view(np.float16).astype(np.float64)[:, :, None] * \
        raw[:, :, 2:].view(np.int8).astype(np.float64)
    deq_pl = orc.f16_bits_to_f32(d2).astype(np.float64)[:, :, None] * \
        q2.reshape(N, K // 32, 32).astype(np.float64)
    assert np.array_equal(deq_blk, deq_pl)


@pytest.mark.parametrize("N,K", [(1, 32), (5, 256), (17, 1024)])
def test_repack_q4_0_round_trip(orc, N, K):
    r = rng(70 + N)
    w = (r.standard_normal((N, K)) * 0.02).astype(np.float32)
    q4, wd = orc.quantize_q4_0(w)
    aos = np.empty((N, K // 32), Q4_0_BLOCK)
    aos["d"] = wd
    aos["qs"] = q4.reshape(N, K // 32, 16)
    q2, d2 = orc.repack_q4_0(aos.view(np.uint8), N, K)
    assert np.array_equal(q2, q4) and np.array_equal(d2, wd)
    # Element j of a block is byte j's low nibble, element j + 16 its high nibble.
    raw = aos.view(np.uint8).reshape(N, K // 32, 18)[:, :, 2:].astype(np.int16)
    vals = np.concatenate([(raw & 15) - 8, (raw >> 4) - 8], axis=2).reshape(N, K)
    assert np.array_equal(orc.unpack_q4_0(q2), vals.astype(np.int8))


def test_repack_is_a_byte_permutation(orc):
    """Every input byte lands in exactly one output byte, unchanged: repack a block array
    whose bytes are all distinct positions' indices (mod 256, per byte plane)."""
    N, K = 3, 64
    nblk = N * K // 32
    raw = (np.arange(nblk * 34) % 251).astype(np.uint8)
    q, d = orc.repack_q8_0(raw, N, K)
    blk = raw.reshape(nblk, 34)
    assert np.array_equal(q.view(np.uint8).reshape(nblk, 32), blk[:, 2:])
    assert np.array_equal(d.reshape(nblk).view(np.uint8).reshape(nblk, 2), blk[:, :2])


# ----------------------------------------------------------------------------
# Routed experts for a batch of tokens: each token on its own.
# ----------------------------------------------------------------------------

def _quant_bank(orc, seed, E, N, K):
    w, wq, wd = _bank(seed, E, N, K)
    for e in range(E):
        wq[e], wd[e] = orc.quantize_q8_0(w[e])
    return wq, wd


def test_moe_gemv_tokens_single_token_and_shared_expert(orc):
    E, N, K, T, top_k = 6, 16, 96, 3, 2
    wq, wd = _quant_bank(orc, 30, E, N, K)
    x = rng(31).standard_normal((T, K)).astype(np.float32)
    xq, xd = orc.quantize_q8_1(x)
    # tokens 0 and 2 both route to expert 4, in different slots
    ids = np.array([[4, 1], [0, 5], [2, 4]], np.int32)
    gw = np.array([[0.7, 0.3], [0.5, 0.5], [0.25, 0.75]], np.float32)
    y, bad = orc.moe_gemv_tokens(wq, wd, ids, None, xq, xd, 0)
    assert bad == 0 and y.shape == (T, top_k, N)
    # pair (t, k) is expert ids[t, k] applied to token t's row, by the plain GEMV
    for t in range(T):
        for k in range(top_k):
            e = ids[t, k]
            assert np.array_equal(y[t, k], orc.gemm(wq[e], wd[e], xq[t:t + 1], xd[t:t + 1])[0])
    yg, _ = orc.moe_gemv_tokens(wq, wd, ids, gw, xq, xd, 0)
    # the gated row is the gated product of that token alone, with its own gates
    for t in range(T):
        one, _ = orc.moe_gemv(wq, wd, ids[t], gw[t], xq[t:t + 1], xd[t:t + 1], 0)
        assert np.array_equal(yg[t], one)
    # swapping two tokens swaps their rows
    perm = [2, 0, 1]
    yp, _ = orc.moe_gemv_tokens(wq, wd, ids[perm], gw[perm], xq[perm], xd[perm], 0)
    assert np.array_equal(yp, yg[perm])


def test_moe_gemv_tokens_per_pair_rows(orc):
    E, N, K, T, top_k = 4, 8, 64, 2, 3
    wq, wd = _quant_bank(orc, 32, E, N, K)
    x = rng(33).standard_normal((T, top_k, K)).astype(np.float32)
    xq, xd = orc.quantize_q8_1(x.reshape(T * top_k, K))
    xq, xd = xq.reshape(T, top_k, K), xd.reshape(T, top_k, K // 32)
    ids = np.array([[3, 0, 3], [1, 2, -1]], np.int32)
    y, bad = orc.moe_gemv_tokens(wq, wd, ids, None, xq, xd, 1)
    assert bad == 1 and not y[1, 2].any()
    assert np.array_equal(y[0, 2], orc.gemm(wq[3], wd[3], xq[0, 2:3], xd[0, 2:3])[0])
    assert np.array_equal(y[1, 0], orc.gemm(wq[1], wd[1], xq[1, 0:1], xd[1, 0:1])[0])


# ----------------------------------------------------------------------------
# NVFP4: the FP8 E4M3 and FP4 E2M1 conversions, the quantiser and the product.
# ----------------------------------------------------------------------------

def _torch_e4m3(values):
    import torch
    return torch.tensor(np.asarray(values, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_e4m3_decode_exhaustive_against_torch(orc):
    import torch
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(orc.e4m3_to_f32(codes), ref)


def test_e4m3_encode_against_torch(orc):
    """Every E4M3 value, every midpoint between neighbours (ties to even), one fp32 ulp
    either side of each midpoint, and random values, below the saturation point."""
    import torch
    pos = np.array(sorted(set(torch.tensor(np.arange(0, 127, dtype=np.uint8))
                               .view(torch.float8_e4m3fn).float().numpy().tolist())), np.float32)
    mids = ((pos[:-1].astype(np.float64) + pos[1:]) / 2).astype(np.float32)
    vals = np.concatenate([pos, mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(1000)),
                           np.exp(rng(80).uniform(np.log(1e-4), np.log(448), 20000))
                           .astype(np.float32)])
    vals = vals[vals <= 448]
    for v in (vals, -vals):
        assert np.array_equal(orc.f32_to_e4m3(v), _torch_e4m3(v))


def test_e4m3_saturates_at_448(orc):
    assert orc.f32_to_e4m3([464.0, 500.0, 1e30]).tolist() == [0x7E] * 3
    assert orc.f32_to_e4m3([-1e30]).tolist() == [0xFE]
    assert orc.f32_to_e4m3([0.0, -0.0]).tolist() == [0x00, 0x80]


def test_e2m1_table_ties_and_saturation(orc):
    # grid values map to their codes; midpoints go to the even mantissa; beyond 6 saturates
    table = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7,
             0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             0.2499: 0, 0.2501: 1, 5.0001: 7, 6.9: 7, 100.0: 7}
    v = np.array(list(table), np.float32)
    assert orc.f32_to_e2m1(v).tolist() == list(table.values())
    assert orc.f32_to_e2m1(-v[1:]).tolist() == [c | 8 for c in list(table.values())[1:]]
    assert orc.f32_to_e2m1([-0.0, -0.1]).tolist() == [8, 8]


def _np_unpack_nvfp4(codes):
    """Independent numpy unpack: byte j -> elements 2j (low nibble) and 2j + 1 (high)."""
    twice = np.array([0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12], np.int8)
    N, K2 = codes.shape
    out = np.empty((N, 2 * K2), np.int8)
    out[:, 0::2] = twice[codes & 15]
    out[:, 1::2] = twice[codes >> 4]
    return out


def test_nvfp4_unpack_matches_hand_packing(orc):
    codes = rng(81).integers(0, 256, size=(7, 48)).astype(np.uint8)
    assert np.array_equal(orc.unpack_nvfp4(codes), _np_unpack_nvfp4(codes))


@pytest.mark.parametrize("std", [0.02, 1.0, 300.0])
def test_nvfp4_quant_invariants(orc, std):
    r = rng(82 + int(std))
    N, K = 24, 256
    w = (r.standard_normal((N, K)) * std).astype(np.float32)
    w[3, 16:32] = 0.0                                       # one all-zero block
    codes, scales, g = orc.quantize_nvfp4(w)
    assert g == np.float32(np.abs(w).max()) / np.float32(2688)
    bmax = np.abs(w).reshape(N, K // 16, 16).max(axis=2)
    assert np.array_equal(scales, _torch_e4m3(bmax / (np.float32(6) * g)))
    s = orc.e4m3_to_f32(scales).astype(np.float64)
    assert scales[3, 1] == 0 and not _np_unpack_nvfp4(codes)[3, 16:32].any()
    v = _np_unpack_nvfp4(codes).astype(np.float64).reshape(N, K // 16, 16) / 2
    denom = (s * np.float64(g))[:, :, None]
    ratio = w.reshape(N, K // 16, 16) / np.where(denom == 0, 1, denom)
    # each code is the nearest E2M1 value of w / (s g) (half a grid step, within 6)
    step = np.where(np.abs(v) < 2, 0.5, np.where(np.abs(v) < 4, 1.0, 2.0))
    ok = (denom > 0) & (np.abs(ratio) <= 6)
    assert np.all(np.abs(ratio - v)[ok] <= step[ok] / 2 + 1e-6)
    # the block maximum maps to +-6 (the E4M3 scale is within 2^-4 of max / 6)
    amax_pos = np.abs(w).reshape(N, K // 16, 16).argmax(axis=2)
    top = np.take_along_axis(np.abs(v), amax_pos[:, :, None], axis=2)[:, :, 0]
    assert np.all(top[scales > 0] == 6.0)


def test_nvfp4_power_of_two_scaling_and_zero_tensor(orc):
    w = (rng(85).standard_normal((8, 128)) * 0.7).astype(np.float32)
    c1, s1, g1 = orc.quantize_nvfp4(w)
    c2, s2, g2 = orc.quantize_nvfp4(w * np.float32(64))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2) and g2 == g1 * 64
    c0, s0, g0 = orc.quantize_nvfp4(np.zeros((2, 64), np.float32))
    assert g0 == 0 and not c0.any() and not s0.any()


@pytest.mark.parametrize("N,K,M", [(17, 256, 1), (9, 1024, 3), (5, 96, 2)])
def test_nvfp4_gemm_within_bound_of_fp64_brute_force(orc, N, K, M):
    r = rng(86 + K)
    codes, scales, g = orc.quantize_nvfp4((r.standard_normal((N, K)) * 0.02).astype(np.float32))
    xq, xd = orc.quantize_q8_1(r.standard_normal((M, K)).astype(np.float32))
    y = orc.gemm_nvfp4(codes, scales, g, xq, xd)
    y64 = orc.nvfp4_dequant_gemm_f64(codes, scales, g, xq, xd)
    # sum of |term| over half-blocks, and the sequential fp32 bound (a few ulps per term)
    c2 = _np_unpack_nvfp4(codes).astype(np.float64)
    s = orc.e4m3_to_f32(scales).astype(np.float64)
    S = np.einsum("nbi,mbi->mnb", c2.reshape(N, K // 16, 16),
                  xq.astype(np.float64).reshape(M, K // 16, 16))
    terms = np.abs(0.5 * float(g) * s[None] * np.repeat(xd, 2, axis=1)[:, None, :] * S).sum(2)
    nb = K // 32
    assert np.all(np.abs(y - y64) <= (nb + 4) * 2.0 ** -23 * terms + 1e-30)


def test_nvfp4_gemm_one_hot_activation_exact(orc):
    # x one-hot at element j with q = 127, d_x = 1: y_n = fl(fl(g/2) * fl(fl(s d_x) * c2 127))
    N, K, j = 6, 64, 37
    codes, scales, g = orc.quantize_nvfp4((rng(87).standard_normal((N, K))).astype(np.float32))
    x = np.zeros((1, K), np.float32)
    x[0, j] = 127.0
    xq, xd = orc.quantize_q8_1(x)
    y = orc.gemm_nvfp4(codes, scales, g, xq, xd)[0]
    c2 = _np_unpack_nvfp4(codes)[:, j].astype(np.float32)
    s = orc.e4m3_to_f32(scales[:, j // 16])
    want = (np.float32(g) * np.float32(0.5)) * ((s * np.float32(1.0)) * (c2 * np.float32(127)))
    assert np.array_equal(y, want.astype(np.float32))


def test_moe_gemv_nvfp4_reduces_to_the_dense_product(orc):
    E, N, K = 4, 12, 256
    r = rng(88)
    banks = [orc.quantize_nvfp4((r.standard_normal((N, K)) * (0.01 * (e + 1))).astype(np.float32))
             for e in range(E)]
    codes = np.stack([b[0] for b in banks])
    scales = np.stack([b[1] for b in banks])
    gexp = np.array([b[2] for b in banks], np.float32)
    assert len(set(gexp.tolist())) == E                 # each expert its own tensor scale
    xq, xd = orc.quantize_q8_1(r.standard_normal((1, K)).astype(np.float32))
    ids = np.array([2, 0, 9, 3], np.int32)
    y, bad = orc.moe_gemv_nvfp4(codes, scales, gexp, ids, None, xq, xd, 0)
    assert bad == 1 and not y[2].any()
    for k, e in ((0, 2), (1, 0), (3, 3)):
        assert np.array_equal(y[k], orc.gemm_nvfp4(codes[e], scales[e], gexp[e], xq, xd)[0])
    y1, _ = orc.moe_gemv_nvfp4(codes, scales, gexp, ids[:1], np.ones(1, np.float32), xq, xd, 0)
    assert np.array_equal(y1, y[0])
    gw = np.array([0.5, 0.25, 0.75, 0.25], np.float32)
    yg, _ = orc.moe_gemv_nvfp4(codes, scales, gexp, ids, gw, xq, xd, 0)
    ref = sum(float(gw[k]) * orc.nvfp4_dequant_gemm_f64(codes[e], scales[e], gexp[e], xq, xd)[0]
              for k, e in ((0, 2), (1, 0), (3, 3)))
    assert np.allclose(yg, ref, rtol=1e-5, atol=1e-7 * np.abs(ref).max())


def test_e2m1_against_brute_force_nearest(orc):
    """E2M1 rounding by brute force: the nearest of the 8 grid magnitudes, a tie going to
    the neighbour with mantissa bit 0 (codes 0, 2, 4, 6), saturation at 6, sign bit kept."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = (grid[:-1] + grid[1:]) / 2
    r = rng(89)
    v = np.concatenate([r.uniform(-8, 8, 50000), grid, mids,
                        np.nextafter(mids.astype(np.float32), np.float32(0)),
                        np.nextafter(mids.astype(np.float32), np.float32(9)),
                        [6.5, 100.0, 1e30]]).astype(np.float32)

    def brute(x):
        a = min(abs(float(x)), 6.0)
        d = np.abs(grid - a)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
        return int(code) | (8 if np.signbit(x) else 0)

    want = np.array([brute(x) for x in v], np.uint8)
    assert np.array_equal(orc.f32_to_e2m1(v), want)
