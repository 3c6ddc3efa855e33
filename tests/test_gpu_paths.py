"""The product kernels (shared-memory bulk-copy stream, register stream, and the
tensor-core kernel for several activation rows) implement one summation order, so they
must agree bit for bit.  Each child process pins the kernel choice with
MEMRA_GEMV_PATH (read once per process): the default selection, the register kernel
everywhere, the bulk-copy kernel wherever it applies (also for M > 1), and the
tensor-core kernel wherever it applies (also for M = 1).  The shapes include products
with many ring stages per CTA (12289 x 4096 ends in a one-row stage; 5120 x 17408 has
one-row stages), tensor-core tiles moved back over the previous tile (N = 17, 40, 1000
rows), a single 16-row tile (N = 16), and two-pass batches (M = 11, 16).  Q4_0 and NVFP4
products run on the bulk-copy kernel only; their children compare its stage geometries."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, torch
sys.path.insert(0, %(root)r)
import synth
import block_quantized_decode_quantize_gb300 as mem
out = {}
for (N, K, M) in [(1003, 4096, 1), (777, 5120, 1), (513, 2048, 4), (300, 5120, 8), (4100, 768, 1),
                  (64, 17408, 1), (12289, 4096, 1), (5120, 17408, 1), (12289, 4096, 2),
                  (1000, 1024, 3), (16, 1024, 8), (17, 2048, 5), (40, 3072, 7),
                  (5120, 5120, 16), (4096, 4096, 11), (2050, 17408, 8)]:
    w = synth.weights_fp32(N, K, 70, N, K, device="cuda")
    x = synth.activations_bf16(M, K, 71, N, K, M, outlier_frac=0.001, device="cuda")
    wq, wd = mem.memra_quantize_q8_0(w)
    xq, xd = mem.memra_quantize_q8_1(x)
    out["d%%d_%%d_%%d" %% (N, K, M)] = mem.memra_q8_0_gemm_small_m(wq, wd, xq, xd).cpu()
    out["f%%d_%%d_%%d" %% (N, K, M)] = mem.memra_q8_0_quant_gemm(wq, wd, x).cpu()
E, N, K, k = 10, 300, 768, 4
wb = synth.weights_fp32(E * N, K, 72, device="cuda")
bq, bd = mem.memra_quantize_q8_0(wb)
bq, bd = bq.view(E, N, K), bd.view(E, N, K // 32)
ids = torch.tensor([3, 9, 0, 3], dtype=torch.int32, device="cuda")
gw = torch.tensor([0.4, 0.3, 0.2, 0.1], device="cuda")
x = synth.activations_bf16(k, K, 73, device="cuda")
xq, xd = mem.memra_quantize_q8_1(x)
out["moe_u"] = mem.memra_q8_0_moe_gemv(bq, bd, ids, None, xq, xd, True).cpu()
out["moe_g"] = mem.memra_q8_0_moe_gemv(bq, bd, ids, gw, xq, xd, True).cpu()
out["moe_s"] = mem.memra_q8_0_moe_gemv(bq, bd, ids, gw, xq[0], xd[0], False).cpu()
# 4-bit dense products (bulk-copy kernel only): its stage geometries must agree.
for (N, K, M) in [(777, 5120, 1), (2050, 17408, 1), (3000, 5120, 1), (513, 2048, 4),
                  (300, 5120, 8), (1000, 4096, 2)]:
    w = synth.weights_fp32(N, K, 74, N, K, device="cuda")
    x = synth.activations_bf16(M, K, 75, N, K, M, outlier_frac=0.001, device="cuda")
    xq, xd = mem.memra_quantize_q8_1(x)
    c4, d4 = mem.memra_quantize_q4_0(w)
    out["q4_%%d_%%d_%%d" %% (N, K, M)] = mem.memra_q4_0_gemm_small_m(c4, d4, xq, xd).cpu()
    cn, sn, gn = mem.memra_quantize_nvfp4(w)
    out["nv_%%d_%%d_%%d" %% (N, K, M)] = mem.memra_nvfp4_gemm_small_m(cn, sn, float(gn.item()),
                                                                   xq, xd).cpu()
torch.cuda.synchronize()
torch.save(out, sys.argv[1])
"""


# Children: (name, environment).  Besides the kernel choice, the bulk-copy kernel's
# stage geometry (read once per process): small stages, so that every CTA wraps its
# ring many times and the tasks fall differently on the consumer warps, and no limit
# or a one-stage limit on the stages issued before the activation is staged.
VARIANTS = [
    ("reg", {"MEMRA_GEMV_PATH": "reg"}),
    ("tma", {"MEMRA_GEMV_PATH": "tma"}),
    ("mma", {"MEMRA_GEMV_PATH": "mma"}),
    ("tma_small_stages", {"MEMRA_GEMV_PATH": "tma", "MEMRA_TMA_STAGE_KB": "6",
                          "MEMRA_TMA_MULTI_STAGE_KB": "6", "MEMRA_TMA_ROUTED_STAGE_KB": "6"}),
    ("tma_prefill_all", {"MEMRA_GEMV_PATH": "tma", "MEMRA_TMA_PREFILL": "0",
                         "MEMRA_TMA_PREFILL_4BIT": "0"}),
    ("tma_prefill_1", {"MEMRA_GEMV_PATH": "tma", "MEMRA_TMA_PREFILL": "1",
                       "MEMRA_TMA_PREFILL_4BIT": "2"}),
]
_KNOBS = ("MEMRA_GEMV_PATH", "MEMRA_TMA_STAGE_KB", "MEMRA_TMA_MULTI_STAGE_KB",
          "MEMRA_TMA_ROUTED_STAGE_KB", "MEMRA_TMA_PREFILL", "MEMRA_TMA_PREFILL_4BIT")


def run_child(tmp_path, name, extra):
    path = str(tmp_path / ("out_%s.pt" % name))
    env = dict(os.environ)
    for k in _KNOBS:
        env.pop(k, None)
    env.update(extra)
    src = CHILD % {"root": ROOT}
    r = subprocess.run([sys.executable, "-c", src, path], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return torch.load(path)


def test_product_kernels_agree_bitwise(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_decode_quantize_gb300 import build
    build.build()
    a = run_child(tmp_path, "default", {})
    for name, extra in VARIANTS:
        b = run_child(tmp_path, name, extra)
        assert a.keys() == b.keys()
        for k in a:
            assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32)), (name, k)
