"""CPU oracle for the Q8_0 decode hot path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and this
package never imports the product: the two share no code.

Thin numpy/ctypes wrappers around ``libmemra_oracle.so`` (``memra_oracle.cpp``).
Array conventions follow the library's planes: ``wq`` int8 [N, K], ``wd`` uint16
fp16 bits [N, K/32], ``xq`` int8 [M, K], ``xd`` float32 [M, K/32], ``y`` float32
[M, N].
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_f16.restype = ctypes.c_uint16
        L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_f32.restype = ctypes.c_float
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_exp_cw.argtypes = [ctypes.c_float]
        L.oracle_exp_cw.restype = ctypes.c_float
        L.oracle_quantize_q8_0.argtypes = [_ptr, _i64, _i64, _ptr, _ptr]
        L.oracle_quantize_q4_0.argtypes = [_ptr, _i64, _i64, _ptr, _ptr]
        L.oracle_unpack_q4_0.argtypes = [_ptr, _i64, _i64, _ptr]
        L.oracle_repack_q8_0.argtypes = [_ptr, _i64, _i64, _ptr, _ptr]
        L.oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
        L.oracle_f32_to_e4m3.restype = ctypes.c_uint8
        L.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_to_f32.restype = ctypes.c_float
        L.oracle_f32_to_e2m1.argtypes = [ctypes.c_float]
        L.oracle_f32_to_e2m1.restype = ctypes.c_uint8
        L.oracle_quantize_nvfp4.argtypes = [_ptr, _i64, _i64, _ptr, _ptr, _ptr]
        L.oracle_unpack_nvfp4.argtypes = [_ptr, _i64, _i64, _ptr]
        L.oracle_nvfp4_gemm.argtypes = [_ptr, _ptr, ctypes.c_float, _i64, _i64, _i64, _ptr, _ptr,
                                        _ptr, ctypes.c_int]
        L.oracle_nvfp4_dequant_gemm_f64.argtypes = [_ptr, _ptr, ctypes.c_float, _i64, _i64, _i64,
                                                    _ptr, _ptr, _ptr]
        L.oracle_repack_q4_0.argtypes = [_ptr, _i64, _i64, _ptr, _ptr]
        L.oracle_quantize_q8_1_f32.argtypes = [_ptr, _i64, _i64, _ptr, _ptr]
        L.oracle_quantize_q8_1_bf16.argtypes = [_ptr, _i64, _i64, _ptr, _ptr]
        L.oracle_block_dots.argtypes = [_ptr, _i64, _i64, _ptr, _i64, _ptr]
        L.oracle_q8_0_gemm.argtypes = [_ptr, _ptr, _i64, _i64, _i64, _ptr, _ptr, _ptr,
                                       ctypes.c_int]
        L.oracle_dequant_gemm_f64.argtypes = [_ptr, _ptr, _i64, _i64, _i64, _ptr, _ptr, _ptr]
        L.oracle_swiglu_f32.argtypes = [_ptr, _i64, _i64, _ptr]
        L.oracle_swiglu_quantize_q8_1.argtypes = [_ptr, _i64, _i64, _ptr, _ptr]
        L.oracle_q8_0_moe_gemv.argtypes = [_ptr, _ptr, _i64, _i64, _i64, _ptr, _ptr, _i64,
                                           _ptr, _ptr, ctypes.c_int, _ptr]
        L.oracle_q8_0_moe_gemv.restype = ctypes.c_int
        L.oracle_moe_ffn.argtypes = [_ptr, _i64, _ptr, _ptr, _ptr, _ptr, _i64, _i64, _i64,
                                     _ptr, _ptr, _i64, _ptr]
        L.oracle_moe_ffn.restype = ctypes.c_int
        L.oracle_openmp_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def f32_to_f16_bits(values):
    """fp32 -> IEEE binary16 bits, round to nearest even (element by element)."""
    v = np.asarray(values, dtype=np.float32).ravel()
    L = lib()
    out = np.array([L.oracle_f32_to_f16(float(x)) for x in v], dtype=np.uint16)
    return out.reshape(np.shape(values))


def f16_bits_to_f32(bits):
    b = np.asarray(bits, dtype=np.uint16).ravel()
    L = lib()
    out = np.array([L.oracle_f16_to_f32(int(x)) for x in b], dtype=np.float32)
    return out.reshape(np.shape(bits))


def bf16_bits_to_f32(bits):
    b = np.asarray(bits, dtype=np.uint16).ravel()
    L = lib()
    out = np.array([L.oracle_bf16_to_f32(int(x)) for x in b], dtype=np.float32)
    return out.reshape(np.shape(bits))


def exp_cw(values):
    v = np.asarray(values, dtype=np.float32).ravel()
    L = lib()
    out = np.array([L.oracle_exp_cw(float(x)) for x in v], dtype=np.float32)
    return out.reshape(np.shape(values))


def quantize_q8_0(w):
    """Weights fp32 [N, K] -> (wq int8 [N, K], wd fp16 bits uint16 [N, K/32])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 32 == 0
    q = np.empty((N, K), np.int8)
    d = np.empty((N, K // 32), np.uint16)
    lib().oracle_quantize_q8_0(_p(w), N, K, _p(q), _p(d))
    return q, d


def quantize_q4_0(w):
    """Weights fp32 [N, K] -> (q4 uint8 [N, K/2] packed codes, wd fp16 bits uint16 [N, K/32])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 32 == 0
    q4 = np.empty((N, K // 2), np.uint8)
    d = np.empty((N, K // 32), np.uint16)
    lib().oracle_quantize_q4_0(_p(w), N, K, _p(q4), _p(d))
    return q4, d


def unpack_q4_0(q4):
    """Packed Q4_0 codes uint8 [N, K/2] -> signed int8 values q - 8, [N, K]."""
    q4 = _c(q4, np.uint8)
    N, K2 = q4.shape
    wq = np.empty((N, 2 * K2), np.int8)
    lib().oracle_unpack_q4_0(_p(q4), N, 2 * K2, _p(wq))
    return wq


def repack_q8_0(blocks, N, K):
    """GGUF Q8_0 block bytes uint8 [N * K/32 * 34] -> (wq int8 [N, K], wd fp16 bits [N, K/32])."""
    blocks = _c(np.asarray(blocks).reshape(-1), np.uint8)
    assert K % 32 == 0 and blocks.size == N * (K // 32) * 34
    q = np.empty((N, K), np.int8)
    d = np.empty((N, K // 32), np.uint16)
    lib().oracle_repack_q8_0(_p(blocks), N, K, _p(q), _p(d))
    return q, d


def repack_q4_0(blocks, N, K):
    """GGUF Q4_0 block bytes uint8 [N * K/32 * 18] -> (q4 uint8 [N, K/2], wd fp16 bits [N, K/32])."""
    blocks = _c(np.asarray(blocks).reshape(-1), np.uint8)
    assert K % 32 == 0 and blocks.size == N * (K // 32) * 18
    q4 = np.empty((N, K // 2), np.uint8)
    d = np.empty((N, K // 32), np.uint16)
    lib().oracle_repack_q4_0(_p(blocks), N, K, _p(q4), _p(d))
    return q4, d


def f32_to_e4m3(values):
    v = np.asarray(values, np.float32)
    return np.array([lib().oracle_f32_to_e4m3(float(x)) for x in v.ravel()],
                    np.uint8).reshape(v.shape)


def e4m3_to_f32(bits):
    b = np.asarray(bits, np.uint8)
    return np.array([lib().oracle_e4m3_to_f32(int(x)) for x in b.ravel()],
                    np.float32).reshape(b.shape)


def f32_to_e2m1(values):
    v = np.asarray(values, np.float32)
    return np.array([lib().oracle_f32_to_e2m1(float(x)) for x in v.ravel()],
                    np.uint8).reshape(v.shape)


def quantize_nvfp4(w):
    """Weights fp32 [N, K] -> (codes uint8 [N, K/2], scales E4M3 bits uint8 [N, K/16], g)."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert K % 32 == 0
    codes = np.empty((N, K // 2), np.uint8)
    scales = np.empty((N, K // 16), np.uint8)
    g = np.zeros(1, np.float32)
    lib().oracle_quantize_nvfp4(_p(w), N, K, _p(codes), _p(scales), _p(g))
    return codes, scales, np.float32(g[0])


def unpack_nvfp4(codes):
    """NVFP4 codes uint8 [N, K/2] -> twice their E2M1 values, int8 [N, K]."""
    codes = _c(codes, np.uint8)
    N, K2 = codes.shape
    out = np.empty((N, 2 * K2), np.int8)
    lib().oracle_unpack_nvfp4(_p(codes), N, 2 * K2, _p(out))
    return out


def gemm_nvfp4(codes, scales, g, xq, xd, threads=1):
    """y[M, N] float32 = NVFP4 W (codes, E4M3 block scales, tensor scale g) times q8_1 x."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    xq = _c(xq, np.int8)
    xd = _c(xd, np.float32)
    N, K2 = codes.shape
    M = xq.shape[0]
    y = np.empty((M, N), np.float32)
    lib().oracle_nvfp4_gemm(_p(codes), _p(scales), float(g), N, 2 * K2, M, _p(xq), _p(xd),
                            _p(y), int(threads))
    return y


def nvfp4_dequant_gemm_f64(codes, scales, g, xq, xd):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    xq = _c(xq, np.int8)
    xd = _c(xd, np.float32)
    N, K2 = codes.shape
    M = xq.shape[0]
    y = np.empty((M, N), np.float64)
    lib().oracle_nvfp4_dequant_gemm_f64(_p(codes), _p(scales), float(g), N, 2 * K2, M, _p(xq),
                                        _p(xd), _p(y))
    return y


def gemm_q4_0(q4, wd, xq, xd, threads=1):
    """y[M, N] float32 = Q4_0 W times q8_1 x: the Q8_0 product of the unpacked codes."""
    return gemm(unpack_q4_0(q4), wd, xq, xd, threads=threads)


def quantize_q8_1(x):
    """Activations [M, K] (float32, or uint16 holding bf16 bits) -> (xq int8, xd float32)."""
    x = np.asarray(x)
    M, K = x.shape
    assert K % 32 == 0
    q = np.empty((M, K), np.int8)
    d = np.empty((M, K // 32), np.float32)
    if x.dtype == np.uint16:
        x = _c(x, np.uint16)
        lib().oracle_quantize_q8_1_bf16(_p(x), M, K, _p(q), _p(d))
    else:
        x = _c(x, np.float32)
        lib().oracle_quantize_q8_1_f32(_p(x), M, K, _p(q), _p(d))
    return q, d


def block_dots(wq, xq):
    """int32 s[M, N, K/32]."""
    wq = _c(wq, np.int8)
    xq = _c(xq, np.int8)
    N, K = wq.shape
    M = xq.shape[0]
    s = np.empty((M, N, K // 32), np.int32)
    lib().oracle_block_dots(_p(wq), N, K, _p(xq), M, _p(s))
    return s


def gemm(wq, wd, xq, xd, threads=1):
    """y[M, N] float32 = Q8_0 W times q8_1 x, per row sequential fp32 accumulation."""
    wq = _c(wq, np.int8)
    wd = _c(wd, np.uint16)
    xq = _c(xq, np.int8)
    xd = _c(xd, np.float32)
    N, K = wq.shape
    M = xq.shape[0]
    y = np.empty((M, N), np.float32)
    lib().oracle_q8_0_gemm(_p(wq), _p(wd), N, K, M, _p(xq), _p(xd), _p(y), int(threads))
    return y


def dequant_gemm_f64(wq, wd, xq, xd):
    wq = _c(wq, np.int8)
    wd = _c(wd, np.uint16)
    xq = _c(xq, np.int8)
    xd = _c(xd, np.float32)
    N, K = wq.shape
    M = xq.shape[0]
    y = np.empty((M, N), np.float64)
    lib().oracle_dequant_gemm_f64(_p(wq), _p(wd), N, K, M, _p(xq), _p(xd), _p(y))
    return y


def swiglu(gu):
    gu = _c(gu, np.float32)
    R, F2 = gu.shape
    F = F2 // 2
    h = np.empty((R, F), np.float32)
    lib().oracle_swiglu_f32(_p(gu), R, F, _p(h))
    return h


def swiglu_quantize_q8_1(gu):
    gu = _c(gu, np.float32)
    R, F2 = gu.shape
    F = F2 // 2
    assert F % 32 == 0
    hq = np.empty((R, F), np.int8)
    hd = np.empty((R, F // 32), np.float32)
    lib().oracle_swiglu_quantize_q8_1(_p(gu), R, F, _p(hq), _p(hd))
    return hq, hd


def moe_gemv(wq_bank, wd_bank, ids, gate_w, xq, xd, x_per_expert):
    """Returns (y, n_bad_ids). y is [top_k, N] without gate weights, [N] with."""
    wq_bank = _c(wq_bank, np.int8)
    wd_bank = _c(wd_bank, np.uint16)
    E, N, K = wq_bank.shape
    ids = _c(ids, np.int32)
    top_k = ids.shape[0]
    xq = _c(xq, np.int8)
    xd = _c(xd, np.float32)
    if gate_w is None:
        y = np.empty((top_k, N), np.float32)
        gp = None
    else:
        gate_w = _c(gate_w, np.float32)
        y = np.empty((N,), np.float32)
        gp = _p(gate_w)
    bad = lib().oracle_q8_0_moe_gemv(_p(wq_bank), _p(wd_bank), E, N, K, _p(ids), gp, top_k,
                                     _p(xq), _p(xd), int(x_per_expert), _p(y))
    return y, bad


def moe_ffn(x, gu_q, gu_d, dn_q, dn_d, ids, gate_w):
    """One routed MoE FFN layer for one token. x fp32 [K]; returns (y [N_out], n_bad)."""
    x = _c(x, np.float32)
    gu_q = _c(gu_q, np.int8)
    gu_d = _c(gu_d, np.uint16)
    dn_q = _c(dn_q, np.int8)
    dn_d = _c(dn_d, np.uint16)
    E, F2, K = gu_q.shape
    F = F2 // 2
    N_out = dn_q.shape[1]
    assert dn_q.shape == (E, N_out, F)
    ids = _c(ids, np.int32)
    gate_w = _c(gate_w, np.float32)
    y = np.empty((N_out,), np.float32)
    bad = lib().oracle_moe_ffn(_p(x), K, _p(gu_q), _p(gu_d), _p(dn_q), _p(dn_d), E, F, N_out,
                               _p(ids), _p(gate_w), ids.shape[0], _p(y))
    return y, bad


def moe_gemv_nvfp4(codes_bank, scales_bank, gexp, ids, gate_w, xq, xd, x_per_expert):
    """Routed experts on an NVFP4 bank, composed from gemm_nvfp4: slot k is expert ids[k]'s
    product with its own tensor scale gexp[ids[k]]; gated: y = sum over valid k, in
    ascending k, of gate_w[k] * y_k, from 0 with one fp32 rounding per multiply and add.
    Returns (y, n_bad)."""
    ids = np.asarray(ids)
    E, N = codes_bank.shape[0], codes_bank.shape[1]
    xq = np.asarray(xq)
    xd = np.asarray(xd)
    ys, bad = [], 0
    for k, e in enumerate(ids):
        if e < 0 or e >= E:
            bad += 1
            ys.append(np.zeros(N, np.float32))
            continue
        xk = (xq[k], xd[k]) if x_per_expert else (xq.reshape(-1), xd.reshape(-1))
        ys.append(gemm_nvfp4(codes_bank[e], scales_bank[e], gexp[e], xk[0][None],
                             xk[1][None])[0])
    if gate_w is None:
        return np.stack(ys), bad
    acc = np.zeros(N, np.float32)
    for k, e in enumerate(ids):
        if 0 <= e < E:
            acc = (acc + np.float32(gate_w[k]) * ys[k]).astype(np.float32)
    return acc, bad


def moe_gemv_tokens(wq_bank, wd_bank, ids, gate_w, xq, xd, x_per_expert):
    """Routed experts for a batch of tokens: each token's routed product on its own (the
    pages' batching changes which weights are read together, not what a token gets).
    ids [T, top_k], gate_w [T, top_k] or None; xq/xd [T, K] or [T, top_k, K].  Returns
    (y, n_bad): y [T, top_k, N] without gate weights, [T, N] with them."""
    ids = np.asarray(ids)
    ys, bad = [], 0
    for t in range(ids.shape[0]):
        y, b = moe_gemv(wq_bank, wd_bank, ids[t], None if gate_w is None else gate_w[t],
                        xq[t], xd[t], x_per_expert)
        ys.append(y)
        bad += b
    return np.stack(ys), bad


def moe_ffn_tokens(x, gu_q, gu_d, dn_q, dn_d, ids, gate_w):
    """The routed FFN layer for a batch of tokens, each on its own.  x fp32 [T, K],
    ids and gate_w [T, top_k]; returns (y [T, N_out], n_bad)."""
    ys, bad = [], 0
    for t in range(np.asarray(ids).shape[0]):
        y, b = moe_ffn(x[t], gu_q, gu_d, dn_q, dn_d, ids[t], gate_w[t])
        ys.append(y)
        bad += b
    return np.stack(ys), bad


def max_threads():
    return int(lib().oracle_openmp_max_threads())
