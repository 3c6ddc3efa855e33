"""The oracle against the stored fixtures under tests/golden/ (see make_golden.py)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def from_hex(h, shape):
    return np.array([int(v, 16) for v in h], np.uint32).view(np.float32).reshape(shape)


def test_hand_block(orc):
    g = load("q8_0_hand_block.json")
    w = np.array(g["w"], np.float32)[None]
    x = np.array(g["x"], np.float32)[None]
    wq, wd = orc.quantize_q8_0(w)
    xq, xd = orc.quantize_q8_1(x)
    assert wq.ravel().tolist() == g["wq"] and int(wd[0, 0]) == g["wd_f16_bits"]
    assert xq.ravel().tolist() == g["xq"] and float(xd[0, 0]) == g["xd"]
    assert int(orc.block_dots(wq, xq)[0, 0, 0]) == g["block_sum"]
    assert float(orc.gemm(wq, wd, xq, xd)[0, 0]) == g["y"]


def test_small_gemm_fixture(orc):
    g = load("q8_0_gemm_small.json")
    N, K, M = g["N"], g["K"], g["M"]
    w = from_hex(g["w_f32_hex"], (N, K))
    x = from_hex(g["x_f32_hex"], (M, K))
    wq, wd = orc.quantize_q8_0(w)
    xq, xd = orc.quantize_q8_1(x)
    assert wq.ravel().tolist() == g["wq"]
    assert wd.ravel().tolist() == g["wd_f16_bits"]
    assert xq.ravel().tolist() == g["xq"]
    assert np.array_equal(xd, from_hex(g["xd_f32_hex"], xd.shape))
    assert orc.block_dots(wq, xq).ravel().tolist() == g["block_sums"]
    y = orc.gemm(wq, wd, xq, xd)
    assert np.array_equal(y.view(np.uint32), from_hex(g["y_f32_hex"], (M, N)).view(np.uint32))


def test_q4_0_hand_block(orc):
    g = load("q4_0_hand_block.json")
    w = np.array(g["w"], np.float32)[None]
    q4, wd = orc.quantize_q4_0(w)
    assert q4.ravel().tolist() == g["packed"] and int(wd[0, 0]) == g["wd_f16_bits"]
    assert (orc.unpack_q4_0(q4).ravel() + 8).tolist() == g["codes"]
    x = np.array(g["x"], np.float32)[None]
    xq, xd = orc.quantize_q8_1(x)
    assert int(orc.block_dots(orc.unpack_q4_0(q4), xq)[0, 0, 0]) == g["block_sum"]
    assert float(orc.gemm_q4_0(q4, wd, xq, xd)[0, 0]) == g["y"]
    tq4, twd = orc.quantize_q4_0(np.array(g["tie_w"], np.float32)[None])
    assert (orc.unpack_q4_0(tq4).ravel() + 8).tolist() == g["tie_codes"]
    assert int(twd[0, 0]) == g["tie_wd_f16_bits"]


def test_gguf_q8_0_blocks_repack(orc):
    g = load("gguf_blocks.json")["q8_0"]
    N, K = g["N"], g["K"]
    blocks = np.frombuffer(bytes.fromhex(g["bytes_hex"]), np.uint8)
    wq, wd = orc.repack_q8_0(blocks, N, K)
    assert wq.ravel().tolist() == g["wq"]
    assert wd.ravel().tolist() == g["wd_f16_bits"]
    assert orc.f16_bits_to_f32(wd).ravel().tolist() == g["wd_values"]


def test_gguf_q4_0_blocks_repack(orc):
    g = load("gguf_blocks.json")["q4_0"]
    N, K = g["N"], g["K"]
    blocks = np.frombuffer(bytes.fromhex(g["bytes_hex"]), np.uint8)
    q4, wd = orc.repack_q4_0(blocks, N, K)
    assert q4.tolist() == g["q4"]
    assert wd.ravel().tolist() == g["wd_f16_bits"]
    assert orc.f16_bits_to_f32(wd).ravel().tolist() == g["wd_values"]
    # The repacked codes are the hand-quantised block's, and row 1 is all zeros.
    vals = orc.unpack_q4_0(q4)
    assert (vals[0].astype(int) + 8).tolist() == g["codes_row0"]
    assert not vals[1].any()


def test_nvfp4_hand_row(orc):
    g = load("nvfp4_hand_row.json")
    w = np.array(g["w"], np.float32)[None]
    codes, scales, gs = orc.quantize_nvfp4(w)
    assert float(gs) == g["g"]
    assert scales.ravel().tolist() == g["scales_e4m3_bits"]
    assert orc.e4m3_to_f32(scales).ravel().tolist() == g["scales_values"]
    c = np.array(g["codes"], np.uint8)
    # ModelOpt packing, by hand: element 2j in the low nibble of byte j, 2j+1 in the high.
    assert codes.ravel().tolist() == (c[0::2] | (c[1::2] << 4)).tolist()
    xq, xd = orc.quantize_q8_1(np.array(g["x"], np.float32)[None])
    assert xd.ravel().tolist() == [1.0, 1.0]
    assert float(orc.gemm_nvfp4(codes, scales, gs, xq, xd)[0, 0]) == g["y"]
    assert float(orc.nvfp4_dequant_gemm_f64(codes, scales, gs, xq, xd)[0, 0]) == g["y"]
