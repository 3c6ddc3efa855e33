"""Write the small regression fixtures under tests/golden/ from the CPU oracle.

The pages about memra print no worked Q8_0 example, so these fixtures are not the
pages' numbers: each is a small seeded case whose expected values come from the
oracle alone (this script imports nothing but the oracle, numpy and the input
generator).  They pin the oracle across machines and compilers (the same fixture
must reproduce on x86-64 and on aarch64) and give the GPU tests a stored case.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def f32_hex(a):
    return [format(int(v), "08x") for v in np.asarray(a, np.float32).view(np.uint32).ravel()]


def small_gemm_case():
    r = np.random.default_rng(20261202)
    N, K, M = 5, 96, 2
    w = (r.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[1, 32:64] = 0.0                      # one all-zero weight block
    x = r.standard_normal((M, K)).astype(np.float32)
    x[0, 7] *= 20.0                        # an outlier
    wq, wd = oracle.quantize_q8_0(w)
    xq, xd = oracle.quantize_q8_1(x)
    s = oracle.block_dots(wq, xq)
    y = oracle.gemm(wq, wd, xq, xd)
    return {
        "what": "Q8_0 weights x q8_1 activations, N=5 K=96 M=2, one zero weight block and "
                "one activation outlier",
        "source": "oracle regression fixture (tests/golden/make_golden.py); the pages print "
                  "no worked example",
        "N": N, "K": K, "M": M,
        "w_f32_hex": f32_hex(w), "x_f32_hex": f32_hex(x),
        "wq": wq.ravel().tolist(), "wd_f16_bits": wd.ravel().tolist(),
        "xq": xq.ravel().tolist(), "xd_f32_hex": f32_hex(xd),
        "block_sums": s.ravel().tolist(), "y_f32_hex": f32_hex(y),
    }


def main():
    case = small_gemm_case()
    with open(os.path.join(HERE, "q8_0_gemm_small.json"), "w") as f:
        json.dump(case, f, indent=0)
        f.write("\n")
    print("wrote q8_0_gemm_small.json")


if __name__ == "__main__":
    main()
