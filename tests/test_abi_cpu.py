"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/memra.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "memra.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(memra_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    import block_quantized_decode_quantize_gb300 as m
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    return m.lib()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("memra_quantize_q8_1", "memra_q8_0_gemv", "memra_q8_0_gemm_small_m",
                     "memra_q8_0_moe_gemv"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert isinstance(getattr(L, name), ctypes._CFuncPtr)


def test_status_strings_and_version(L):
    assert L.memra_status_string(0) == b"MEMRA_OK"
    for s in range(1, 5):
        assert L.memra_status_string(s).startswith(b"MEMRA_ERR_")
    assert b"sm_103a" in L.memra_version()
    assert L.memra_last_cuda_error() == 0


# Fake device addresses: the checks below must reject the call before any of them is
# dereferenced or handed to CUDA.
A256 = 0x7f0000000000
BAD = A256 + 1


def test_gemv_argument_errors(L):
    f = L.memra_q8_0_gemm_small_m
    assert f(A256, A256, 64, 48, 1, A256, A256, A256, None) == 1      # K % 32 != 0
    assert f(A256, A256, -1, 64, 1, A256, A256, A256, None) == 1      # negative N
    assert f(A256, A256, 64, 64, 17, A256, A256, A256, None) == 3     # M > 16
    assert f(None, A256, 64, 64, 1, A256, A256, A256, None) == 1      # null weights
    assert f(A256 + 16, A256, 64, 64, 1, A256, A256, A256, None) == 2  # wq not 32-aligned
    assert f(A256, A256 + 1, 64, 64, 1, A256, A256, A256, None) == 2   # wd not 2-aligned
    assert f(A256, A256, 64, 64, 1, A256 + 8, A256, A256, None) == 2   # xq not 16-aligned
    assert f(A256, A256, 64, 64, 1, A256, A256, A256 + 2, None) == 2   # y not 4-aligned
    assert f(A256, A256, 64, 8 * 1024 * 1024, 1, A256, A256, A256, None) == 3  # x too big
    assert f(None, None, 0, 64, 1, None, None, None, None) == 0        # empty: no work
    assert L.memra_q8_0_gemv(A256, A256, 64, 33, A256, A256, A256, None) == 1


def test_fused_argument_errors(L):
    f = L.memra_q8_0_quant_gemm
    assert f(A256, A256, 64, 48, 1, A256, 0, A256, None) == 1       # K % 32
    assert f(A256, A256, 64, 64, 1, A256, 5, A256, None) == 1       # dtype
    assert f(A256, A256, 64, 64, 17, A256, 0, A256, None) == 3      # M > 16
    assert f(A256, A256, 64, 64, 1, A256 + 8, 0, A256, None) == 2   # x not 16-aligned
    assert f(A256 + 16, A256, 64, 64, 1, A256, 0, A256, None) == 2  # wq not 32-aligned
    assert f(None, None, 0, 64, 1, None, 0, None, None) == 0


def test_quantizer_argument_errors(L):
    assert L.memra_quantize_q8_1(A256, 0, 2, 40, A256, A256, None) == 1   # K % 32
    assert L.memra_quantize_q8_1(A256, 7, 2, 64, A256, A256, None) == 1   # bad dtype
    assert L.memra_quantize_q8_1(A256 + 4, 1, 2, 64, A256, A256, None) == 2
    assert L.memra_quantize_q8_1(None, 1, 0, 64, None, None, None) == 0
    assert L.memra_quantize_q8_0(A256, 4, 48, A256, A256, None) == 1
    assert L.memra_quantize_q8_0(A256, 4, 64, A256 + 8, A256, None) == 2
    assert L.memra_swiglu_quantize_q8_1(A256, 2, 48, A256, A256, None) == 1
    assert L.memra_swiglu_quantize_q8_1(A256 + 4, 2, 64, A256, A256, None) == 2


def test_q4_0_argument_errors(L):
    f = L.memra_q4_0_gemm_small_m
    assert f(A256, A256, 64, 48, 1, A256, A256, A256, None) == 1      # K % 32 != 0
    assert f(A256, A256, 64, 256, 17, A256, A256, A256, None) == 3    # M > 16
    assert f(A256, A256, 64, 96, 1, A256, A256, A256, None) == 3      # K % 256 != 0
    assert f(A256 + 8, A256, 64, 256, 1, A256, A256, A256, None) == 2  # wq4 not 16-aligned
    assert f(A256, A256 + 2, 64, 256, 1, A256, A256, A256, None) == 2  # wd not 16-aligned
    assert f(A256, A256, 64, 256, 1, A256, A256 + 4, A256, None) == 2  # xd not 16-aligned
    assert f(None, A256, 64, 256, 1, A256, A256, A256, None) == 1     # null weights
    assert f(None, None, 0, 256, 1, None, None, None, None) == 0       # empty: no work
    assert L.memra_q4_0_gemv(A256, A256, 64, 33, A256, A256, A256, None) == 1
    assert L.memra_quantize_q4_0(A256, 4, 48, A256, A256, None) == 1
    assert L.memra_quantize_q4_0(A256, 4, 64, A256 + 8, A256, None) == 2
    assert L.memra_quantize_q4_0(None, 0, 64, None, None, None) == 0


def test_repack_argument_errors(L):
    for f, _ in ((L.memra_repack_q8_0, 34), (L.memra_repack_q4_0, 18)):
        assert f(A256, 4, 48, A256, A256, None) == 1           # K % 32 != 0
        assert f(A256, -1, 64, A256, A256, None) == 1          # N < 0
        assert f(None, 4, 64, A256, A256, None) == 1           # null blocks
        assert f(A256, 4, 64, None, A256, None) == 1           # null quants
        assert f(A256 + 1, 4, 64, A256, A256, None) == 2       # blocks not 2-aligned
        assert f(A256, 4, 64, A256 + 8, A256, None) == 2       # quants not 16-aligned
        assert f(A256, 4, 64, A256, A256 + 1, None) == 2       # scales not 2-aligned
        assert f(A256, 1 << 62, 64, A256, A256, None) == 3     # bytes beyond int64
        assert f(None, 0, 64, None, None, None) == 0           # empty: no work
        assert f(None, 4, 0, None, None, None) == 0


def test_nvfp4_argument_errors(L):
    f = L.memra_nvfp4_gemm_small_m
    assert f(A256, A256, 1.0, 64, 48, 1, A256, A256, A256, None) == 1     # K % 32 != 0
    assert f(A256, A256, 1.0, 64, 256, 17, A256, A256, A256, None) == 3   # M > 16
    assert f(A256, A256, 1.0, 64, 96, 1, A256, A256, A256, None) == 3     # K % 256 != 0
    assert f(A256 + 8, A256, 1.0, 64, 256, 1, A256, A256, A256, None) == 2  # codes
    assert f(A256, A256 + 8, 1.0, 64, 256, 1, A256, A256, A256, None) == 2  # scales
    assert f(None, A256, 1.0, 64, 256, 1, A256, A256, A256, None) == 1
    assert f(None, None, 1.0, 0, 256, 1, None, None, None, None) == 0      # empty
    assert L.memra_nvfp4_gemv(A256, A256, 1.0, 64, 33, A256, A256, A256, None) == 1
    q = L.memra_quantize_nvfp4
    assert q(A256, 4, 48, A256, A256, A256, None) == 1                     # K % 32
    assert q(A256, 4, 64, A256, A256, None, None) == 1                     # no g
    assert q(A256 + 4, 4, 64, A256, A256, A256, None) == 2                 # w alignment
    assert q(A256, 4, 64, A256 + 4, A256, A256, None) == 2                 # codes alignment
    assert q(None, 0, 64, None, None, None, None) == 0


def test_moe_tokens_argument_errors(L):
    g = L.memra_q8_0_moe_gemv_tokens

    def call(E=4, N=16, K=64, gw=None, T=2, top_k=8, xpe=0, ws=None, y=A256):
        return g(A256, A256, E, N, K, A256, gw, T, top_k, A256, A256, xpe, y, ws, None, None)

    assert call(K=48) == 1                    # K % 32 != 0
    assert call(T=-1) == 1
    assert call(xpe=2) == 1
    assert call(top_k=65) == 3                # beyond MEMRA_MAX_TOP_K
    assert call(T=17, top_k=8) == 3           # 136 pairs > MEMRA_MAX_PAIRS
    assert call(T=200, top_k=1) == 3
    assert call(gw=A256, ws=None) == 1        # gated without a workspace
    assert call(y=None) == 1
    assert call(y=A256 + 2) == 2
    assert call(T=0) == 0 and call(N=0) == 0  # empty: no work
    f = L.memra_q8_0_moe_ffn_tokens

    def ffn(H=64, F=32, gw=A256, T=2, top_k=8, dt=0, ws=A256, x=A256):
        return f(A256, A256, A256, A256, 4, H, F, A256, gw, T, top_k, x, dt, A256, ws, None,
                 None)

    assert ffn(H=48) == 1 and ffn(F=48) == 1
    assert ffn(dt=7) == 1
    assert ffn(gw=None) == 1                  # the layer needs gate weights
    assert ffn(T=17) == 3
    assert ffn(ws=None) == 1 and ffn(x=None) == 1
    assert ffn(ws=A256 + 4) == 2 and ffn(x=A256 + 8) == 2
    assert ffn(T=0) == 0


def test_moe_argument_errors(L):
    f = L.memra_q8_0_moe_gemv
    args = dict(wq=A256, wd=A256, E=4, N=16, K=64, ids=A256, gw=None, top_k=2, xq=A256,
                xd=A256, xpe=0, y=A256, st=None)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return f(a["wq"], a["wd"], a["E"], a["N"], a["K"], a["ids"], a["gw"], a["top_k"],
                 a["xq"], a["xd"], a["xpe"], a["y"], a["st"], None)

    assert call(E=0) == 1
    assert call(top_k=0) == 1
    assert call(top_k=65) == 3
    assert call(xpe=2) == 1
    assert call(K=40) == 1
    assert call(ids=None) == 1
    assert call(wq=A256 + 16) == 2
    assert call(ids=A256 + 2) == 2
    assert call(N=0) == 0


def test_block_dots_argument_errors(L):
    assert L.memra_q8_0_block_dots(A256, 4, 40, A256, 1, A256, None) == 1
    assert L.memra_q8_0_block_dots(A256 + 16, 4, 64, A256, 1, A256, None) == 2
    assert L.memra_q8_0_block_dots(None, 0, 64, None, 1, None, None) == 0
