"""memra-gb300: Q8_0 decode GEMV / verify GEMM / routed-expert GEMV for GB300.

A thin Python binding over the C ABI in ``include/memra.h`` (``libmemra.so``).
The binding only marshals arguments: it checks tensor devices, dtypes, shapes and
contiguity, allocates outputs with torch when the caller passes none, and calls the
library on the current torch CUDA stream.  Every step of the computation runs in the
library's sm_103a kernels; there is no fallback.  If the library has not been built
(``block_quantized_decode_quantize_gb300.build.build()``) loading it raises.

Tensor conventions (all on one CUDA device, contiguous):
  wq  int8 [N, K]          Q8_0 quants            wd  float16 [N, K/32]  Q8_0 scales
  xq  int8 [M, K]          q8_1 quants            xd  float32 [M, K/32]  q8_1 scales
  y   float32 [M, N]       (the GEMV takes and returns 1-D x / y)
"""
import ctypes
import os

import torch

from . import build as _build

MEMRA_OK = 0
MEMRA_BF16 = 0
MEMRA_F32 = 1
MAX_M = 16
MAX_TOP_K = 64
MOE_NOALLOC_SCRATCH_FLOATS = 65536

_STATUS = {0: "MEMRA_OK", 1: "MEMRA_ERR_INVALID_ARG", 2: "MEMRA_ERR_ALIGNMENT",
           3: "MEMRA_ERR_UNSUPPORTED", 4: "MEMRA_ERR_CUDA"}


class MemraError(RuntimeError):
    def __init__(self, fn, status, cuda_error=0):
        self.status = status
        self.cuda_error = cuda_error
        msg = "%s returned %s" % (fn, _STATUS.get(status, status))
        if cuda_error:
            msg += " (cudaError %d)" % cuda_error
        super().__init__(msg)


_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32

_SIGS = {
    "memra_quantize_q8_0": [_p, _i64, _i64, _p, _p, _p],
    "memra_quantize_q8_1": [_p, _i32, _i64, _i64, _p, _p, _p],
    "memra_q8_0_gemv": [_p, _p, _i64, _i64, _p, _p, _p, _p],
    "memra_quantize_q4_0": [_p, _i64, _i64, _p, _p, _p],
    "memra_repack_q8_0": [_p, _i64, _i64, _p, _p, _p],
    "memra_quantize_nvfp4": [_p, _i64, _i64, _p, _p, _p, _p],
    "memra_read_stream": [_p, _i64, _p, _i32, _p],
    "memra_nvfp4_gemm_small_m": [_p, _p, ctypes.c_float, _i64, _i64, _i64, _p, _p, _p, _p],
    "memra_nvfp4_gemv": [_p, _p, ctypes.c_float, _i64, _i64, _p, _p, _p, _p],
    "memra_nvfp4_moe_gemv": [_p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _p, _i32, _p, _p,
                             _p],
    "memra_nvfp4_moe_gemv_tokens": [_p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _i64, _p, _p,
                                    _i32, _p, _p, _p, _p],
    "memra_repack_q4_0": [_p, _i64, _i64, _p, _p, _p],
    "memra_q4_0_gemv": [_p, _p, _i64, _i64, _p, _p, _p, _p],
    "memra_q4_0_gemm_small_m": [_p, _p, _i64, _i64, _i64, _p, _p, _p, _p],
    "memra_q4_0_moe_gemv": [_p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _p, _i32, _p, _p, _p],
    "memra_q8_0_gemm_small_m": [_p, _p, _i64, _i64, _i64, _p, _p, _p, _p],
    "memra_q8_0_gemm_small_m_mma": [_p, _p, _i64, _i64, _i64, _p, _p, _p, _p],
    "memra_q8_0_quant_gemm": [_p, _p, _i64, _i64, _i64, _p, _i32, _p, _p],
    "memra_q8_0_moe_gemv": [_p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _p, _i32, _p, _p, _p],
    "memra_q8_0_moe_gemv_tokens": [_p, _p, _i64, _i64, _i64, _p, _p, _i64, _i64, _p, _p, _i32,
                                   _p, _p, _p, _p],
    "memra_q4_0_moe_gemv_tokens": [_p, _p, _i64, _i64, _i64, _p, _p, _i64, _i64, _p, _p, _i32,
                                   _p, _p, _p, _p],
    "memra_q8_0_moe_ffn_tokens": [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _i64, _p, _i32,
                                  _p, _p, _p, _p],
    "memra_q4_0_moe_ffn": [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _i32, _p, _p, _p,
                           _p],
    "memra_nvfp4_moe_ffn": [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _i32, _p,
                            _p, _p, _p],
    "memra_q4_0_moe_ffn_tokens": [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _i64, _p, _i32,
                                  _p, _p, _p, _p],
    "memra_nvfp4_moe_ffn_tokens": [_p, _p, _p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _i64,
                                   _p, _i32, _p, _p, _p, _p],
    "memra_swiglu_quantize_q8_1": [_p, _i64, _i64, _p, _p, _p],
    "memra_q8_0_moe_ffn": [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _i32, _p, _p, _p,
                           _p],
    "memra_q8_0_moe_ffn_noalloc": [_p, _p, _p, _p, _i64, _i64, _i64, _p, _p, _i64, _p, _i32, _p,
                                   _p, _p],
    "memra_q8_0_block_dots": [_p, _i64, _i64, _p, _i64, _p, _p],
    "memra_debug_set_wait_test": [_i64, _i64],
}


def library_path():
    return _build.LIB


def lib():
    """The loaded C library (ctypes), with argument types set for every entry point."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError("libmemra.so is not built (expected at %s); run "
                               "block_quantized_decode_quantize_gb300.build.build()" % path)
        L = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.memra_status_string.argtypes = [ctypes.c_int]
        L.memra_status_string.restype = ctypes.c_char_p
        L.memra_last_cuda_error.restype = ctypes.c_int32
        L.memra_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(name, status):
    if status != MEMRA_OK:
        L = lib()
        raise MemraError(name, status, L.memra_last_cuda_error() if status == 4 else 0)


def _stream(t):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, name, dtype, device=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must have dtype %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))


def memra_quantize_q8_0(w, wq=None, wd=None):
    """fp32 weights [N, K] -> (wq int8 [N, K], wd float16 [N, K/32])."""
    _need(w, "w", torch.float32)
    N, K = w.shape
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.int8, device=w.device)
    if wd is None:
        wd = torch.empty((N, K // 32), dtype=torch.float16, device=w.device)
    _need(wq, "wq", torch.int8, w.device, (N, K))
    _need(wd, "wd", torch.float16, w.device, (N, K // 32))
    with torch.cuda.device(w.device):
        _check("memra_quantize_q8_0",
               lib().memra_quantize_q8_0(_ptr(w), N, K, _ptr(wq), _ptr(wd), _stream(w)))
    return wq, wd


def memra_quantize_q4_0(w, wq4=None, wd=None):
    """fp32 weights [N, K] -> (wq4 uint8 [N, K/2] packed 4-bit codes, wd float16 [N, K/32])."""
    _need(w, "w", torch.float32)
    N, K = w.shape
    if wq4 is None:
        wq4 = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    if wd is None:
        wd = torch.empty((N, K // 32), dtype=torch.float16, device=w.device)
    _need(wq4, "wq4", torch.uint8, w.device, (N, K // 2))
    _need(wd, "wd", torch.float16, w.device, (N, K // 32))
    with torch.cuda.device(w.device):
        _check("memra_quantize_q4_0",
               lib().memra_quantize_q4_0(_ptr(w), N, K, _ptr(wq4), _ptr(wd), _stream(w)))
    return wq4, wd


def _blocks(blocks, N, K, block_bytes):
    _need(blocks, "blocks", torch.uint8)
    if K % 32 != 0 or blocks.numel() != N * (K // 32) * block_bytes:
        raise ValueError("blocks must hold N * K/32 blocks of %d bytes (N=%d, K=%d), got %d bytes"
                         % (block_bytes, N, K, blocks.numel()))


def memra_repack_q8_0(blocks, N, K, wq=None, wd=None):
    """GGUF Q8_0 block bytes (uint8, N * K/32 * 34) -> (wq int8 [N, K], wd float16 [N, K/32])."""
    _blocks(blocks, N, K, 34)
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.int8, device=blocks.device)
    if wd is None:
        wd = torch.empty((N, K // 32), dtype=torch.float16, device=blocks.device)
    _need(wq, "wq", torch.int8, blocks.device, (N, K))
    _need(wd, "wd", torch.float16, blocks.device, (N, K // 32))
    with torch.cuda.device(blocks.device):
        _check("memra_repack_q8_0",
               lib().memra_repack_q8_0(_ptr(blocks), N, K, _ptr(wq), _ptr(wd), _stream(blocks)))
    return wq, wd


def memra_repack_q4_0(blocks, N, K, wq4=None, wd=None):
    """GGUF Q4_0 block bytes (uint8, N * K/32 * 18) -> (wq4 uint8 [N, K/2], wd float16 [N, K/32])."""
    _blocks(blocks, N, K, 18)
    if wq4 is None:
        wq4 = torch.empty((N, K // 2), dtype=torch.uint8, device=blocks.device)
    if wd is None:
        wd = torch.empty((N, K // 32), dtype=torch.float16, device=blocks.device)
    _need(wq4, "wq4", torch.uint8, blocks.device, (N, K // 2))
    _need(wd, "wd", torch.float16, blocks.device, (N, K // 32))
    with torch.cuda.device(blocks.device):
        _check("memra_repack_q4_0",
               lib().memra_repack_q4_0(_ptr(blocks), N, K, _ptr(wq4), _ptr(wd), _stream(blocks)))
    return wq4, wd


def memra_read_stream(buf, sink=None, ctas_per_sm=2):
    """Read every byte of the CUDA tensor `buf` once (diagnostic read stream); returns the
    per-CTA xor sink (uint32, zeroed here when not given)."""
    if not isinstance(buf, torch.Tensor) or not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    nbytes = buf.numel() * buf.element_size()
    if sink is None:
        sms = torch.cuda.get_device_properties(buf.device).multi_processor_count
        sink = torch.zeros((sms * ctas_per_sm,), dtype=torch.int32, device=buf.device)
    with torch.cuda.device(buf.device):
        _check("memra_read_stream",
               lib().memra_read_stream(_ptr(buf), nbytes, _ptr(sink), ctas_per_sm,
                                       _stream(buf)))
    return sink


def memra_quantize_q8_1(x, xq=None, xd=None):
    """Activations [M, K] (bf16 or fp32) -> (xq int8 [M, K], xd float32 [M, K/32])."""
    if x.dtype == torch.bfloat16:
        dt = MEMRA_BF16
    elif x.dtype == torch.float32:
        dt = MEMRA_F32
    else:
        raise TypeError("x must be bfloat16 or float32")
    _need(x, "x", x.dtype)
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if xd is None:
        xd = torch.empty((M, K // 32), dtype=torch.float32, device=x.device)
    _need(xq, "xq", torch.int8, x.device, (M, K))
    _need(xd, "xd", torch.float32, x.device, (M, K // 32))
    with torch.cuda.device(x.device):
        _check("memra_quantize_q8_1",
               lib().memra_quantize_q8_1(_ptr(x), dt, M, K, _ptr(xq), _ptr(xd), _stream(x)))
    return xq, xd


def memra_q8_0_gemm_small_m(wq, wd, xq, xd, y=None):
    """y [M, N] = W (Q8_0) x (q8_1) for M <= 16 activation rows (two weight passes above 8)."""
    _need(wq, "wq", torch.int8)
    N, K = wq.shape
    dev = wq.device
    _need(wd, "wd", torch.float16, dev, (N, K // 32))
    _need(xq, "xq", torch.int8, dev)
    M = xq.shape[0]
    _need(xq, "xq", torch.int8, dev, (M, K))
    _need(xd, "xd", torch.float32, dev, (M, K // 32))
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (M, N))
    with torch.cuda.device(dev):
        _check("memra_q8_0_gemm_small_m",
               lib().memra_q8_0_gemm_small_m(_ptr(wq), _ptr(wd), N, K, M, _ptr(xq), _ptr(xd),
                                             _ptr(y), _stream(wq)))
    return y


def memra_q8_0_gemm_small_m_mma(wq, wd, xq, xd, y=None):
    """memra_q8_0_gemm_small_m with the block sums on the tensor cores (bit-identical
    results; K a multiple of 1024 up to 5120, N >= 16)."""
    _need(wq, "wq", torch.int8)
    N, K = wq.shape
    dev = wq.device
    _need(wd, "wd", torch.float16, dev, (N, K // 32))
    _need(xq, "xq", torch.int8, dev)
    M = xq.shape[0]
    _need(xq, "xq", torch.int8, dev, (M, K))
    _need(xd, "xd", torch.float32, dev, (M, K // 32))
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (M, N))
    with torch.cuda.device(dev):
        _check("memra_q8_0_gemm_small_m_mma",
               lib().memra_q8_0_gemm_small_m_mma(_ptr(wq), _ptr(wd), N, K, M, _ptr(xq),
                                                 _ptr(xd), _ptr(y), _stream(wq)))
    return y


def memra_q8_0_quant_gemm(wq, wd, x, y=None):
    """y [M, N] = W (Q8_0) x, with x [M, K] (bf16 or fp32) quantised to q8_1 inside the
    kernel; bit-identical to memra_quantize_q8_1 followed by memra_q8_0_gemm_small_m."""
    _need(wq, "wq", torch.int8)
    N, K = wq.shape
    dev = wq.device
    _need(wd, "wd", torch.float16, dev, (N, K // 32))
    if x.dtype == torch.bfloat16:
        dt = MEMRA_BF16
    elif x.dtype == torch.float32:
        dt = MEMRA_F32
    else:
        raise TypeError("x must be bfloat16 or float32")
    _need(x, "x", x.dtype, dev)
    M = x.shape[0]
    _need(x, "x", x.dtype, dev, (M, K))
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (M, N))
    with torch.cuda.device(dev):
        _check("memra_q8_0_quant_gemm",
               lib().memra_q8_0_quant_gemm(_ptr(wq), _ptr(wd), N, K, M, _ptr(x), dt, _ptr(y),
                                           _stream(wq)))
    return y


def memra_q8_0_gemv(wq, wd, xq, xd, y=None):
    """y [N] = W (Q8_0) x (q8_1) for one activation row (xq [K], xd [K/32])."""
    _need(wq, "wq", torch.int8)
    N, K = wq.shape
    dev = wq.device
    _need(wd, "wd", torch.float16, dev, (N, K // 32))
    _need(xq, "xq", torch.int8, dev, (K,))
    _need(xd, "xd", torch.float32, dev, (K // 32,))
    if y is None:
        y = torch.empty((N,), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (N,))
    with torch.cuda.device(dev):
        _check("memra_q8_0_gemv",
               lib().memra_q8_0_gemv(_ptr(wq), _ptr(wd), N, K, _ptr(xq), _ptr(xd), _ptr(y),
                                     _stream(wq)))
    return y


def memra_q4_0_gemm_small_m(wq4, wd, xq, xd, y=None):
    """y [M, N] = W (Q4_0: wq4 uint8 [N, K/2], wd float16 [N, K/32]) x (q8_1), M <= 16."""
    _need(wq4, "wq4", torch.uint8)
    N, K2 = wq4.shape
    K = 2 * K2
    dev = wq4.device
    _need(wd, "wd", torch.float16, dev, (N, K // 32))
    _need(xq, "xq", torch.int8, dev)
    M = xq.shape[0]
    _need(xq, "xq", torch.int8, dev, (M, K))
    _need(xd, "xd", torch.float32, dev, (M, K // 32))
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (M, N))
    with torch.cuda.device(dev):
        _check("memra_q4_0_gemm_small_m",
               lib().memra_q4_0_gemm_small_m(_ptr(wq4), _ptr(wd), N, K, M, _ptr(xq), _ptr(xd),
                                             _ptr(y), _stream(wq4)))
    return y


def memra_quantize_nvfp4(w, codes=None, scales=None, g=None):
    """fp32 weights [N, K] -> (codes uint8 [N, K/2], scales uint8 E4M3 bits [N, K/16],
    g float32 [1] on the device: the tensor scale)."""
    _need(w, "w", torch.float32)
    N, K = w.shape
    if codes is None:
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // 16), dtype=torch.uint8, device=w.device)
    if g is None:
        g = torch.empty((1,), dtype=torch.float32, device=w.device)
    _need(codes, "codes", torch.uint8, w.device, (N, K // 2))
    _need(scales, "scales", torch.uint8, w.device, (N, K // 16))
    _need(g, "g", torch.float32, w.device, (1,))
    with torch.cuda.device(w.device):
        _check("memra_quantize_nvfp4",
               lib().memra_quantize_nvfp4(_ptr(w), N, K, _ptr(codes), _ptr(scales), _ptr(g),
                                          _stream(w)))
    return codes, scales, g


def memra_nvfp4_gemm_small_m(codes, scales, g, xq, xd, y=None):
    """y [M, N] = W (NVFP4: codes uint8 [N, K/2], scales uint8 E4M3 [N, K/16], tensor
    scale g, a Python float) x (q8_1), M <= 16."""
    _need(codes, "codes", torch.uint8)
    N, K2 = codes.shape
    K = 2 * K2
    dev = codes.device
    _need(scales, "scales", torch.uint8, dev, (N, K // 16))
    _need(xq, "xq", torch.int8, dev)
    M = xq.shape[0]
    _need(xq, "xq", torch.int8, dev, (M, K))
    _need(xd, "xd", torch.float32, dev, (M, K // 32))
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (M, N))
    with torch.cuda.device(dev):
        _check("memra_nvfp4_gemm_small_m",
               lib().memra_nvfp4_gemm_small_m(_ptr(codes), _ptr(scales), float(g), N, K, M,
                                              _ptr(xq), _ptr(xd), _ptr(y), _stream(codes)))
    return y


def memra_nvfp4_gemv(codes, scales, g, xq, xd, y=None):
    """y [N] = W (NVFP4) x (q8_1) for one activation row (xq [K], xd [K/32])."""
    _need(codes, "codes", torch.uint8)
    N, K2 = codes.shape
    K = 2 * K2
    dev = codes.device
    _need(scales, "scales", torch.uint8, dev, (N, K // 16))
    _need(xq, "xq", torch.int8, dev, (K,))
    _need(xd, "xd", torch.float32, dev, (K // 32,))
    if y is None:
        y = torch.empty((N,), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (N,))
    with torch.cuda.device(dev):
        _check("memra_nvfp4_gemv",
               lib().memra_nvfp4_gemv(_ptr(codes), _ptr(scales), float(g), N, K, _ptr(xq),
                                      _ptr(xd), _ptr(y), _stream(codes)))
    return y


def memra_q4_0_gemv(wq4, wd, xq, xd, y=None):
    """y [N] = W (Q4_0) x (q8_1) for one activation row (xq [K], xd [K/32])."""
    _need(wq4, "wq4", torch.uint8)
    N, K2 = wq4.shape
    K = 2 * K2
    dev = wq4.device
    _need(wd, "wd", torch.float16, dev, (N, K // 32))
    _need(xq, "xq", torch.int8, dev, (K,))
    _need(xd, "xd", torch.float32, dev, (K // 32,))
    if y is None:
        y = torch.empty((N,), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (N,))
    with torch.cuda.device(dev):
        _check("memra_q4_0_gemv",
               lib().memra_q4_0_gemv(_ptr(wq4), _ptr(wd), N, K, _ptr(xq), _ptr(xd), _ptr(y),
                                     _stream(wq4)))
    return y


def _moe_gemv(fn, wq_bank, qdtype, kmul, wd_bank, ids, gate_w, xq, xd, x_per_expert, y,
              dev_status):
    _need(wq_bank, "wq_bank", qdtype)
    E, N, Kq = wq_bank.shape
    K = Kq * kmul
    dev = wq_bank.device
    _need(wd_bank, "wd_bank", torch.float16, dev, (E, N, K // 32))
    _need(ids, "ids", torch.int32, dev)
    top_k = ids.shape[0]
    if gate_w is not None:
        _need(gate_w, "gate_w", torch.float32, dev, (top_k,))
    xpe = 1 if x_per_expert else 0
    if xpe:
        _need(xq, "xq", torch.int8, dev, (top_k, K))
        _need(xd, "xd", torch.float32, dev, (top_k, K // 32))
    else:
        _need(xq, "xq", torch.int8, dev, (K,))
        _need(xd, "xd", torch.float32, dev, (K // 32,))
    yshape = (N,) if gate_w is not None else (top_k, N)
    if y is None:
        y = torch.empty(yshape, dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, yshape)
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
    with torch.cuda.device(dev):
        _check(fn, getattr(lib(), fn)(_ptr(wq_bank), _ptr(wd_bank), E, N, K, _ptr(ids),
                                      _ptr(gate_w), top_k, _ptr(xq), _ptr(xd), xpe, _ptr(y),
                                      _ptr(dev_status), _stream(wq_bank)))
    return y


def memra_q8_0_moe_gemv(wq_bank, wd_bank, ids, gate_w, xq, xd, x_per_expert, y=None,
                        dev_status=None):
    """Routed-expert GEMV.  wq_bank int8 [E, N, K], wd_bank float16 [E, N, K/32],
    ids int32 [top_k], gate_w float32 [top_k] or None.  x_per_expert=False: xq [K],
    xd [K/32]; True: xq [top_k, K], xd [top_k, K/32].  Returns y [top_k, N] without
    gate weights, [N] with them."""
    return _moe_gemv("memra_q8_0_moe_gemv", wq_bank, torch.int8, 1, wd_bank, ids, gate_w, xq,
                     xd, x_per_expert, y, dev_status)


def memra_q4_0_moe_gemv(wq4_bank, wd_bank, ids, gate_w, xq, xd, x_per_expert, y=None,
                        dev_status=None):
    """memra_q8_0_moe_gemv on a Q4_0 bank: wq4_bank uint8 [E, N, K/2] (packed codes),
    wd_bank float16 [E, N, K/32]."""
    return _moe_gemv("memra_q4_0_moe_gemv", wq4_bank, torch.uint8, 2, wd_bank, ids, gate_w, xq,
                     xd, x_per_expert, y, dev_status)


def _moe_gemv_tokens(fn, wq_bank, qdtype, kmul, wd_bank, ids, gate_w, xq, xd, x_per_expert,
                     y, workspace, dev_status):
    _need(wq_bank, "wq_bank", qdtype)
    E, N, Kq = wq_bank.shape
    K = Kq * kmul
    dev = wq_bank.device
    _need(wd_bank, "wd_bank", torch.float16, dev, (E, N, K // 32))
    _need(ids, "ids", torch.int32, dev)
    T, top_k = ids.shape
    if gate_w is not None:
        _need(gate_w, "gate_w", torch.float32, dev, (T, top_k))
    xpe = 1 if x_per_expert else 0
    rows = (T, top_k) if xpe else (T,)
    _need(xq, "xq", torch.int8, dev, rows + (K,))
    _need(xd, "xd", torch.float32, dev, rows + (K // 32,))
    yshape = (T, N) if gate_w is not None else (T, top_k, N)
    if y is None:
        y = torch.empty(yshape, dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, yshape)
    if gate_w is not None:
        if workspace is None:
            workspace = torch.empty((T, top_k, N), dtype=torch.float32, device=dev)
        _need(workspace, "workspace", torch.float32, dev, (T, top_k, N))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
    with torch.cuda.device(dev):
        _check(fn, getattr(lib(), fn)(_ptr(wq_bank), _ptr(wd_bank), E, N, K, _ptr(ids),
                                      _ptr(gate_w), T, top_k, _ptr(xq), _ptr(xd), xpe, _ptr(y),
                                      _ptr(workspace), _ptr(dev_status), _stream(wq_bank)))
    return y


def memra_q8_0_moe_gemv_tokens(wq_bank, wd_bank, ids, gate_w, xq, xd, x_per_expert, y=None,
                               workspace=None, dev_status=None):
    """Routed experts for a batch of tokens.  ids int32 [T, top_k], gate_w float32
    [T, top_k] or None.  x_per_expert=False: xq [T, K], xd [T, K/32]; True: xq
    [T, top_k, K], xd [T, top_k, K/32].  Returns y [T, top_k, N] without gate weights,
    [T, N] with them (`workspace` float32 [T, top_k, N] then holds the per-pair rows)."""
    return _moe_gemv_tokens("memra_q8_0_moe_gemv_tokens", wq_bank, torch.int8, 1, wd_bank, ids,
                            gate_w, xq, xd, x_per_expert, y, workspace, dev_status)


def memra_q4_0_moe_gemv_tokens(wq4_bank, wd_bank, ids, gate_w, xq, xd, x_per_expert, y=None,
                               workspace=None, dev_status=None):
    """memra_q8_0_moe_gemv_tokens on a Q4_0 bank (wq4_bank uint8 [E, N, K/2])."""
    return _moe_gemv_tokens("memra_q4_0_moe_gemv_tokens", wq4_bank, torch.uint8, 2, wd_bank,
                            ids, gate_w, xq, xd, x_per_expert, y, workspace, dev_status)


def memra_q8_0_moe_ffn_tokens(gu_q, gu_d, dn_q, dn_d, ids, gate_w, x, y=None, workspace=None,
                              dev_status=None):
    """memra_q8_0_moe_ffn for a batch: ids int32 [T, top_k], gate_w float32 [T, top_k],
    x [T, H] (bf16 or fp32).  Returns y float32 [T, H].  `workspace` float32
    [T * top_k * (2F + H)] holds the pairs' gate|up rows, then their down rows."""
    _need(gu_q, "gu_q", torch.int8)
    E, F2, H = gu_q.shape
    F = F2 // 2
    dev = gu_q.device
    _need(gu_d, "gu_d", torch.float16, dev, (E, F2, H // 32))
    _need(dn_q, "dn_q", torch.int8, dev, (E, H, F))
    _need(dn_d, "dn_d", torch.float16, dev, (E, H, F // 32))
    _need(ids, "ids", torch.int32, dev)
    T, top_k = ids.shape
    _need(gate_w, "gate_w", torch.float32, dev, (T, top_k))
    if x.dtype == torch.bfloat16:
        dt = MEMRA_BF16
    elif x.dtype == torch.float32:
        dt = MEMRA_F32
    else:
        raise TypeError("x must be bfloat16 or float32")
    _need(x, "x", x.dtype, dev, (T, H))
    if y is None:
        y = torch.empty((T, H), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (T, H))
    ws = T * top_k * (F2 + H)
    if workspace is None:
        workspace = torch.empty((ws,), dtype=torch.float32, device=dev)
    _need(workspace, "workspace", torch.float32, dev, (ws,))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
    with torch.cuda.device(dev):
        _check("memra_q8_0_moe_ffn_tokens",
               lib().memra_q8_0_moe_ffn_tokens(_ptr(gu_q), _ptr(gu_d), _ptr(dn_q), _ptr(dn_d), E,
                                               H, F, _ptr(ids), _ptr(gate_w), T, top_k, _ptr(x),
                                               dt, _ptr(y), _ptr(workspace), _ptr(dev_status),
                                               _stream(gu_q)))
    return y


def memra_nvfp4_moe_gemv(codes_bank, scales_bank, gexp, ids, gate_w, xq, xd, x_per_expert,
                         y=None, dev_status=None):
    """Routed experts on an NVFP4 bank: codes_bank uint8 [E, N, K/2], scales_bank uint8
    E4M3 [E, N, K/16], gexp float32 [E] (each expert's tensor scale, on the device);
    the rest as memra_q8_0_moe_gemv."""
    _need(codes_bank, "codes_bank", torch.uint8)
    E, N, K2 = codes_bank.shape
    K = 2 * K2
    dev = codes_bank.device
    _need(scales_bank, "scales_bank", torch.uint8, dev, (E, N, K // 16))
    _need(gexp, "gexp", torch.float32, dev, (E,))
    _need(ids, "ids", torch.int32, dev)
    top_k = ids.shape[0]
    if gate_w is not None:
        _need(gate_w, "gate_w", torch.float32, dev, (top_k,))
    xpe = 1 if x_per_expert else 0
    rows = (top_k,) if xpe else ()
    _need(xq, "xq", torch.int8, dev, rows + (K,))
    _need(xd, "xd", torch.float32, dev, rows + (K // 32,))
    yshape = (N,) if gate_w is not None else (top_k, N)
    if y is None:
        y = torch.empty(yshape, dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, yshape)
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
    with torch.cuda.device(dev):
        _check("memra_nvfp4_moe_gemv",
               lib().memra_nvfp4_moe_gemv(_ptr(codes_bank), _ptr(scales_bank), _ptr(gexp), E, N,
                                          K, _ptr(ids), _ptr(gate_w), top_k, _ptr(xq), _ptr(xd),
                                          xpe, _ptr(y), _ptr(dev_status), _stream(codes_bank)))
    return y


def memra_nvfp4_moe_gemv_tokens(codes_bank, scales_bank, gexp, ids, gate_w, xq, xd,
                                x_per_expert, y=None, workspace=None, dev_status=None):
    """memra_q8_0_moe_gemv_tokens on an NVFP4 bank (layout as memra_nvfp4_moe_gemv)."""
    _need(codes_bank, "codes_bank", torch.uint8)
    E, N, K2 = codes_bank.shape
    K = 2 * K2
    dev = codes_bank.device
    _need(scales_bank, "scales_bank", torch.uint8, dev, (E, N, K // 16))
    _need(gexp, "gexp", torch.float32, dev, (E,))
    _need(ids, "ids", torch.int32, dev)
    T, top_k = ids.shape
    if gate_w is not None:
        _need(gate_w, "gate_w", torch.float32, dev, (T, top_k))
    xpe = 1 if x_per_expert else 0
    rows = (T, top_k) if xpe else (T,)
    _need(xq, "xq", torch.int8, dev, rows + (K,))
    _need(xd, "xd", torch.float32, dev, rows + (K // 32,))
    yshape = (T, N) if gate_w is not None else (T, top_k, N)
    if y is None:
        y = torch.empty(yshape, dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, yshape)
    if gate_w is not None:
        if workspace is None:
            workspace = torch.empty((T, top_k, N), dtype=torch.float32, device=dev)
        _need(workspace, "workspace", torch.float32, dev, (T, top_k, N))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
    with torch.cuda.device(dev):
        _check("memra_nvfp4_moe_gemv_tokens",
               lib().memra_nvfp4_moe_gemv_tokens(_ptr(codes_bank), _ptr(scales_bank), _ptr(gexp),
                                                 E, N, K, _ptr(ids), _ptr(gate_w), T, top_k,
                                                 _ptr(xq), _ptr(xd), xpe, _ptr(y),
                                                 _ptr(workspace), _ptr(dev_status),
                                                 _stream(codes_bank)))
    return y


def memra_q8_0_moe_ffn(gu_q, gu_d, dn_q, dn_d, ids, gate_w, x, y=None, workspace=None,
                       dev_status=None):
    """One routed-expert FFN layer: gu_q int8 [E, 2F, H], gu_d float16 [E, 2F, H/32],
    dn_q int8 [E, H, F], dn_d float16 [E, H, F/32], ids int32 [top_k], gate_w float32
    [top_k], x [H] (bf16 or fp32).  Returns y float32 [H].  `workspace` (float32
    [top_k, 2F]) receives the gate|up outputs; allocated here when not given."""
    _need(gu_q, "gu_q", torch.int8)
    E, F2, H = gu_q.shape
    F = F2 // 2
    dev = gu_q.device
    _need(gu_d, "gu_d", torch.float16, dev, (E, F2, H // 32))
    _need(dn_q, "dn_q", torch.int8, dev, (E, H, F))
    _need(dn_d, "dn_d", torch.float16, dev, (E, H, F // 32))
    _need(ids, "ids", torch.int32, dev)
    top_k = ids.shape[0]
    _need(gate_w, "gate_w", torch.float32, dev, (top_k,))
    if x.dtype == torch.bfloat16:
        dt = MEMRA_BF16
    elif x.dtype == torch.float32:
        dt = MEMRA_F32
    else:
        raise TypeError("x must be bfloat16 or float32")
    _need(x, "x", x.dtype, dev, (H,))
    if y is None:
        y = torch.empty((H,), dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, (H,))
    if workspace is None:
        workspace = torch.empty((top_k, F2), dtype=torch.float32, device=dev)
    _need(workspace, "workspace", torch.float32, dev, (top_k, F2))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
    with torch.cuda.device(dev):
        _check("memra_q8_0_moe_ffn",
               lib().memra_q8_0_moe_ffn(_ptr(gu_q), _ptr(gu_d), _ptr(dn_q), _ptr(dn_d), E, H, F,
                                        _ptr(ids), _ptr(gate_w), top_k, _ptr(x), dt, _ptr(y),
                                        _ptr(workspace), _ptr(dev_status), _stream(gu_q)))
    return y


def _moe_ffn_4bit(fmt, gu, gu_s, gu_g, dn, dn_s, dn_g, ids, gate_w, x, y, workspace,
                  dev_status):
    """Shared marshalling of the Q4_0 and NVFP4 routed FFN entry points (one token when
    ids is 1-D, a batch of tokens when it is [T, top_k])."""
    _need(gu, "gate|up bank", torch.uint8)
    E, F2, H2 = gu.shape
    H, F = 2 * H2, F2 // 2
    dev = gu.device
    sdt, sdiv = (torch.float16, 32) if fmt == "q4_0" else (torch.uint8, 16)
    _need(gu_s, "gate|up scales", sdt, dev, (E, F2, H // sdiv))
    _need(dn, "down bank", torch.uint8, dev, (E, H, F // 2))
    _need(dn_s, "down scales", sdt, dev, (E, H, F // sdiv))
    if fmt == "nvfp4":
        _need(gu_g, "gu_g", torch.float32, dev, (E,))
        _need(dn_g, "dn_g", torch.float32, dev, (E,))
    _need(ids, "ids", torch.int32, dev)
    tokens = ids.dim() == 2
    T, top_k = (ids.shape if tokens else (1, ids.shape[0]))
    _need(gate_w, "gate_w", torch.float32, dev, tuple(ids.shape))
    if x.dtype == torch.bfloat16:
        dt = MEMRA_BF16
    elif x.dtype == torch.float32:
        dt = MEMRA_F32
    else:
        raise TypeError("x must be bfloat16 or float32")
    yshape = (T, H) if tokens else (H,)
    _need(x, "x", x.dtype, dev, yshape)
    if y is None:
        y = torch.empty(yshape, dtype=torch.float32, device=dev)
    _need(y, "y", torch.float32, dev, yshape)
    ws = T * top_k * (F2 + H) if tokens else top_k * F2
    if workspace is None:
        workspace = torch.empty((ws,), dtype=torch.float32, device=dev)
    _need(workspace, "workspace", torch.float32, dev)
    if workspace.numel() != ws:
        raise ValueError("workspace must hold %d floats" % ws)
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
    L = lib()
    name = "memra_%s_moe_ffn%s" % (fmt, "_tokens" if tokens else "")
    banks = ([_ptr(gu), _ptr(gu_s), _ptr(dn), _ptr(dn_s)] if fmt == "q4_0" else
             [_ptr(gu), _ptr(gu_s), _ptr(gu_g), _ptr(dn), _ptr(dn_s), _ptr(dn_g)])
    sizes = [E, H, F, _ptr(ids), _ptr(gate_w)] + ([T, top_k] if tokens else [top_k])
    with torch.cuda.device(dev):
        _check(name, getattr(L, name)(*banks, *sizes, _ptr(x), dt, _ptr(y), _ptr(workspace),
                                      _ptr(dev_status), _stream(gu)))
    return y


def memra_q4_0_moe_ffn(gu_q4, gu_d, dn_q4, dn_d, ids, gate_w, x, y=None, workspace=None,
                       dev_status=None):
    """The routed FFN layer on Q4_0 banks (gu_q4 uint8 [E, 2F, H/2], gu_d float16
    [E, 2F, H/32], dn_q4 uint8 [E, H, F/2], dn_d float16 [E, H, F/32]).  ids [top_k] for
    one token (x [H]) or [T, top_k] for a batch (x [T, H], the batched entry point)."""
    return _moe_ffn_4bit("q4_0", gu_q4, gu_d, None, dn_q4, dn_d, None, ids, gate_w, x, y,
                         workspace, dev_status)


def memra_nvfp4_moe_ffn(gu_codes, gu_scales, gu_g, dn_codes, dn_scales, dn_g, ids, gate_w, x,
                        y=None, workspace=None, dev_status=None):
    """The routed FFN layer on NVFP4 banks (codes uint8 [E, rows, K/2], E4M3 scales uint8
    [E, rows, K/16], per-expert tensor scales float32 [E] for each bank).  ids [top_k]
    for one token or [T, top_k] for a batch."""
    return _moe_ffn_4bit("nvfp4", gu_codes, gu_scales, gu_g, dn_codes, dn_scales, dn_g, ids,
                         gate_w, x, y, workspace, dev_status)


def memra_q8_0_moe_ffn_noalloc(gu_q, gu_d, dn_q, dn_d, ids, gate_w, x, y, dev_status=None):
    """memra_q8_0_moe_ffn with the gate|up workspace inside the library: the C call
    allocates no device memory (the caller provides y).  For callers that cannot
    allocate at call time; top_k * 2F must not exceed MOE_NOALLOC_SCRATCH_FLOATS.
    The first call on a device should come before any stream capture; calls that
    overlap on the GPU share one scratch array and race."""
    _need(gu_q, "gu_q", torch.int8)
    E, F2, H = gu_q.shape
    F = F2 // 2
    dev = gu_q.device
    _need(gu_d, "gu_d", torch.float16, dev, (E, F2, H // 32))
    _need(dn_q, "dn_q", torch.int8, dev, (E, H, F))
    _need(dn_d, "dn_d", torch.float16, dev, (E, H, F // 32))
    _need(ids, "ids", torch.int32, dev)
    top_k = ids.shape[0]
    _need(gate_w, "gate_w", torch.float32, dev, (top_k,))
    if x.dtype == torch.bfloat16:
        dt = MEMRA_BF16
    elif x.dtype == torch.float32:
        dt = MEMRA_F32
    else:
        raise TypeError("x must be bfloat16 or float32")
    _need(x, "x", x.dtype, dev, (H,))
    _need(y, "y", torch.float32, dev, (H,))
    if dev_status is not None:
        _need(dev_status, "dev_status", torch.int32, dev, (1,))
    with torch.cuda.device(dev):
        _check("memra_q8_0_moe_ffn_noalloc",
               lib().memra_q8_0_moe_ffn_noalloc(_ptr(gu_q), _ptr(gu_d), _ptr(dn_q), _ptr(dn_d), E,
                                                H, F, _ptr(ids), _ptr(gate_w), top_k, _ptr(x),
                                                dt, _ptr(y), _ptr(dev_status), _stream(gu_q)))
    return y


def memra_swiglu_quantize_q8_1(gu, hq=None, hd=None):
    """gu float32 [R, 2F] (gate | up) -> (hq int8 [R, F], hd float32 [R, F/32])."""
    _need(gu, "gu", torch.float32)
    R, F2 = gu.shape
    F = F2 // 2
    if hq is None:
        hq = torch.empty((R, F), dtype=torch.int8, device=gu.device)
    if hd is None:
        hd = torch.empty((R, F // 32), dtype=torch.float32, device=gu.device)
    _need(hq, "hq", torch.int8, gu.device, (R, F))
    _need(hd, "hd", torch.float32, gu.device, (R, F // 32))
    with torch.cuda.device(gu.device):
        _check("memra_swiglu_quantize_q8_1",
               lib().memra_swiglu_quantize_q8_1(_ptr(gu), R, F, _ptr(hq), _ptr(hd),
                                                _stream(gu)))
    return hq, hd


def memra_q8_0_block_dots(wq, xq, s=None):
    """Exact int32 block sums s [M, N, K/32]."""
    _need(wq, "wq", torch.int8)
    N, K = wq.shape
    dev = wq.device
    _need(xq, "xq", torch.int8, dev)
    M = xq.shape[0]
    _need(xq, "xq", torch.int8, dev, (M, K))
    if s is None:
        s = torch.empty((M, N, K // 32), dtype=torch.int32, device=dev)
    _need(s, "s", torch.int32, dev, (M, N, K // 32))
    with torch.cuda.device(dev):
        _check("memra_q8_0_block_dots",
               lib().memra_q8_0_block_dots(_ptr(wq), N, K, _ptr(xq), M, _ptr(s), _stream(wq)))
    return s


def memra_debug_set_wait_test(wait_limit_cycles=0, stall_after_stages=-1):
    """Test hook: later product launches give up waiting after wait_limit_cycles SM
    cycles and, with stall_after_stages >= 0, stall after that many stages per CTA, so
    that their abort path runs (NaN outputs, status bit 2).  Defaults switch it off."""
    _check("memra_debug_set_wait_test",
           lib().memra_debug_set_wait_test(int(wait_limit_cycles), int(stall_after_stages)))


def version():
    return lib().memra_version().decode()
