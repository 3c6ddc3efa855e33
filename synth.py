"""Seeded synthetic inputs for the Q8_0 decode workloads.

This module holds no quantisation or dot-product arithmetic: it only draws the
fp32 weights, bf16 activations and expert routings that both the CUDA library and
the CPU oracle are fed.  Every tensor is addressed by a tuple of integer keys
(workload, layer, tensor, ...) that is mixed into a torch generator seed, so any
tensor can be regenerated on its own and on either device.

Workloads (the shapes of the decode steps this library serves):

* ``gemv_4096``: one 4096 x 4096 Q8_0 GEMV, M = 1, seed 0.
* ``dense27b_sweep``: 64 decode layers of a dense ~27B model, M = 1: fused QKV
  5120 -> 7168, O 5120 -> 5120, gate+up 5120 -> 2 x 17408, down 17408 -> 5120;
  activations bf16 N(0, 1) with 0.1% of entries scaled x20.
* ``verify_small_m``: the same shapes with M in {2, 4, 8} activation rows.
* ``moe_top8``: 48 layers, 128 experts, hidden 2048, expert FFN 2048 -> 2 x 768 and
  768 -> 2048, top-8 routing from a seeded softmax.
* ``stress_large``: 151936 x 5120 (vocabulary head) and 5120 x 17408, M in {1, 8},
  with 1% of weight blocks zero and 1% scaled x50.

Weights are N(0, 0.02) fp32 before quantisation.
"""
import torch

WEIGHT_STD = 0.02

DENSE27B = {
    "hidden": 5120,
    "layers": 64,
    # (name, N, K) in execution order within one layer
    "gemvs": (("qkv", 7168, 5120), ("o", 5120, 5120), ("gate_up", 2 * 17408, 5120),
              ("down", 5120, 17408)),
    "outlier_frac": 0.001,
    "outlier_scale": 20.0,
}

MOE = {"experts": 128, "hidden": 2048, "ffn": 768, "top_k": 8, "layers": 48}

STRESS = {"shapes": (("lm_head", 151936, 5120), ("down", 5120, 17408)), "m": (1, 8),
          "zero_frac": 0.01, "scale_frac": 0.01, "scale": 50.0}

GEMV_4096 = {"N": 4096, "K": 4096, "seed": 0}

_MASK64 = (1 << 64) - 1


def _splitmix64(z):
    z = (z + 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def seed_of(*keys):
    """Mix integer keys into one 63-bit generator seed."""
    z = 0x243F6A8885A308D3
    for k in keys:
        z = _splitmix64(z ^ (int(k) & _MASK64))
    return z & ((1 << 63) - 1)


def generator(device, *keys):
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(*keys))
    return g


def normal(shape, *keys, std=1.0, device="cpu"):
    """fp32 N(0, std^2) samples, seeded by keys."""
    g = generator(device, *keys)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def weights_fp32(N, K, *keys, std=WEIGHT_STD, device="cpu"):
    return normal((N, K), *keys, std=std, device=device)


def perturb_blocks(w, *keys, zero_frac, scale_frac, scale):
    """In place: zero exactly round(zero_frac * blocks) 32-blocks of w [N, K] and scale
    exactly round(scale_frac * blocks) other blocks by `scale` (disjoint seeded sets).
    Returns (zero_block_ids, scaled_block_ids) as flat block indices n*(K/32)+b."""
    N, K = w.shape
    nb = N * (K // 32)
    n_zero = int(round(zero_frac * nb))
    n_scale = int(round(scale_frac * nb))
    g = generator(w.device, *keys, 0xB10C)
    perm = torch.randperm(nb, generator=g, device=w.device)
    zero_ids = perm[:n_zero]
    scale_ids = perm[n_zero:n_zero + n_scale]
    blocks = w.view(nb, 32)
    blocks[zero_ids] = 0.0
    blocks[scale_ids] *= scale
    return zero_ids, scale_ids


def activations_fp32(M, K, *keys, outlier_frac=0.0, outlier_scale=20.0, device="cpu"):
    """fp32 N(0, 1) [M, K]; in each row exactly round(outlier_frac*K) distinct seeded
    positions are multiplied by outlier_scale."""
    x = normal((M, K), *keys, device=device)
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        g = generator(device, *keys, 0x0071)
        for m in range(M):
            pos = torch.randperm(K, generator=g, device=device)[:n_out]
            x[m, pos] *= outlier_scale
    return x


def activations_bf16(M, K, *keys, outlier_frac=0.0, outlier_scale=20.0, device="cpu"):
    """bf16 activations (round-to-nearest-even from the fp32 draw)."""
    return activations_fp32(M, K, *keys, outlier_frac=outlier_frac,
                            outlier_scale=outlier_scale, device=device).to(torch.bfloat16)


def bf16_bits(t):
    """A bf16 tensor's raw 16-bit patterns as an int16 tensor (same device)."""
    return t.contiguous().view(torch.int16)


def routing(E, top_k, *keys, device="cpu"):
    """Top-k experts of a softmax over seeded N(0, 1) router logits.

    The softmax is taken in fp64, the k largest probabilities are selected (equal
    probabilities keep the lower expert id first) and renormalised to sum to one;
    the weights are returned in fp32.  Returns (ids int32 [top_k], weights fp32
    [top_k]) on `device`."""
    logits = normal((E,), *keys, device="cpu").to(torch.float64)
    p = torch.softmax(logits, dim=0)
    order = torch.sort(p, descending=True, stable=True).indices[:top_k]
    sel = p[order]
    w = (sel / sel.sum()).to(torch.float32)
    return order.to(torch.int32).to(device), w.to(device)


def dense27b_bytes_per_token():
    """Q8_0 weight bytes streamed per token by the dense sweep (34 bytes per 32 weights)."""
    per_layer = sum(N * K * 34 // 32 for _, N, K in DENSE27B["gemvs"])
    return per_layer * DENSE27B["layers"]


def q8_0_bytes(N, K):
    return N * K * 34 // 32


def ceil_div(a, b):
    return -(-a // b)

