#!/usr/bin/env python3
"""Benchmark of the Q8_0 decode hot path on GB300.

Default workload (one "step" = one decode token): a dense ~27B decode sweep, M = 1,
64 layers of distinct seeded weights, each layer = 4 x (q8_1 quantise of a bf16
activation, Q8_0 GEMV): fused QKV 5120->7168, O 5120->5120, gate+up 5120->34816,
down 17408->5120.  22.46 GB of Q8_0 weights stream from HBM per step (far above the
129 MB L2, so no flush is needed between steps).

Prints ONE JSON line.  ``value`` is weight-stream GB/s over the whole job (all
ranks); ``e2e`` repeats the measurement through the public API with the step's
activations copied in from pinned host memory and every output copied back;
``roofline`` is the GEMV kernel's achieved HBM bandwidth against the measured copy
peak; ``cpu_baseline`` is the CPU oracle on the host cores over a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl memra|reference]
                  [--workload dense27b_sweep|gemv_4096|verify_m2|verify_m4|verify_m8|
                              batch_m16|moe_top8|stress_lm_head|dense27b_sweep_q4_0|
                              dense27b_sweep_nvfp4|
                              moe_top8_q4_0|moe_top8_nvfp4|moe_top8_tokens8|moe_top8_tokens16]
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = ("Q8_0 decode GEMV weight-stream GB/s (% of GB300 HBM peak); "
          "µs per 27B layer sweep")
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOADS = ("dense27b_sweep", "gemv_4096", "verify_m2", "verify_m4", "verify_m8", "batch_m16",
             "moe_top8",
             "stress_lm_head", "dense27b_sweep_q4_0", "dense27b_sweep_nvfp4", "moe_top8_q4_0",
             "moe_top8_nvfp4", "moe_top8_tokens8", "moe_top8_tokens16")


# ----------------------------------------------------------------------------
# Workload construction (inputs from synth, weights quantised by the library).
# ----------------------------------------------------------------------------

class Gemv:
    """One product of a step: Q8_0 (wq int8 [N, K]), Q4_0 (wq uint8 [N, K/2]) or NVFP4
    (wq uint8 codes [N, K/2], wd E4M3 scales [N, K/16], tensor scale g) weights, its
    bf16 activation(s), q8_1 buffers, y."""

    def __init__(self, wq, wd, x, name, fmt=None, g=None):
        self.wq, self.wd, self.x, self.name, self.g = wq, wd, x, name, g
        self.fmt = fmt or ("q4_0" if wq.dtype == torch.uint8 else "q8_0")
        M, K = x.shape
        N = wq.shape[0]
        dev = wq.device
        self.xq = torch.empty((M, K), dtype=torch.int8, device=dev)
        self.xd = torch.empty((M, K // 32), dtype=torch.float32, device=dev)
        self.y = torch.empty((M, N), dtype=torch.float32, device=dev)

    @property
    def weight_bytes(self):
        return self.wq.numel() + self.wd.numel() * self.wd.element_size()  # quants + scales


def quantized_weights(mem, N, K, *keys, device, perturb=None, fmt="q8_0"):
    w = synth.weights_fp32(N, K, *keys, device=device)
    if perturb:
        synth.perturb_blocks(w, *keys, **perturb)
    if fmt == "q4_0":
        wq, wd = mem.memra_quantize_q4_0(w)
    elif fmt == "nvfp4":
        wq, wd, g = mem.memra_quantize_nvfp4(w)
        del w
        return wq, wd, float(g.item())
    else:
        wq, wd = mem.memra_quantize_q8_0(w)
    del w
    return wq, wd


def tokens_of(name):
    """Tokens one step decodes: a batch of sequences or of routed tokens, else 1."""
    if name.startswith("batch_m"):
        return rows_of(name)
    if "_tokens" in name:
        return int(name.rsplit("_tokens", 1)[1])
    return 1


def rows_of(name):
    """Activation rows of a dense-sweep workload: verify_mM and batch_mM have M, the
    plain sweeps 1."""
    for prefix in ("verify_m", "batch_m"):
        if name.startswith(prefix):
            return int(name[len(prefix):])
    return 1


def build_dense_sweep(mem, device, M=1, layers=None, workload_id=1, fmt="q8_0"):
    """The dense 27B-class sweep: per layer QKV, O, gate+up, down."""
    cfg = synth.DENSE27B
    L = cfg["layers"] if layers is None else layers
    ops = []
    for layer in range(L):
        for t, (name, N, K) in enumerate(cfg["gemvs"]):
            qw = quantized_weights(mem, N, K, workload_id, layer, t, device=device, fmt=fmt)
            x = synth.activations_bf16(M, K, workload_id, layer, t, 1000 + M,
                                       outlier_frac=cfg["outlier_frac"],
                                       outlier_scale=cfg["outlier_scale"], device=device)
            ops.append(Gemv(qw[0], qw[1], x, "L%d.%s" % (layer, name), fmt=fmt,
                            g=qw[2] if fmt == "nvfp4" else None))
    return ops


def sweep_rows_like(ops, M, workload_id=2):
    """The products of a built dense sweep (same weight tensors, no new weights) with M
    independent activation rows each, seeded like the verify workloads' activations."""
    cfg = synth.DENSE27B
    per_layer = len(cfg["gemvs"])
    out = []
    for i, op in enumerate(ops):
        layer, t = divmod(i, per_layer)
        K = op.x.shape[1]
        x = synth.activations_bf16(M, K, workload_id, layer, t, 1000 + M,
                                   outlier_frac=cfg["outlier_frac"],
                                   outlier_scale=cfg["outlier_scale"], device=op.wq.device)
        out.append(Gemv(op.wq, op.wd, x, op.name))
    return out


def build_gemv_4096(mem, device, copies=32):
    """One 4096x4096 GEMV (seed 0); `copies` distinct weight copies rotate so that the
    weights of consecutive calls are not L2 resident (32 x 17.8 MB >> 129 MB L2)."""
    c = synth.GEMV_4096
    wq, wd = quantized_weights(mem, c["N"], c["K"], c["seed"], device=device)
    x = synth.activations_bf16(1, c["K"], c["seed"], 1, device=device)
    ops = []
    for i in range(copies):
        ops.append(Gemv(wq.clone() if i else wq, wd.clone() if i else wd, x, "copy%d" % i))
    return ops


def build_stress(mem, device, M):
    s = synth.STRESS
    ops = []
    for t, (name, N, K) in enumerate(s["shapes"]):
        wq, wd = quantized_weights(mem, N, K, 4, t, device=device,
                                   perturb=dict(zero_frac=s["zero_frac"],
                                                scale_frac=s["scale_frac"], scale=s["scale"]))
        x = synth.activations_bf16(M, K, 4, t, 1000 + M, device=device)
        ops.append(Gemv(wq, wd, x, name))
    return ops


class MoeLayer:
    """One routed FFN layer for one token, or (tokens > 1) for a batch of tokens with
    their own routings through the batched entry points."""

    def __init__(self, mem, layer, device, fmt="q8_0", tokens=1):
        c = synth.MOE
        E, H, F, k = c["experts"], c["hidden"], c["ffn"], c["top_k"]
        self.fmt = fmt
        self.tokens = tokens
        kdiv = 1 if fmt == "q8_0" else 2  # quant bytes per weight: 1/2 for the 4-bit formats
        qg = quantized_weights(mem, E * 2 * F, H, 3, layer, 0, device=device, fmt=fmt)
        qd = quantized_weights(mem, E * H, F, 3, layer, 1, device=device, fmt=fmt)
        sdiv = 16 if fmt == "nvfp4" else 32  # scale entries per row: one per 16 or per 32
        self.gq, self.gd = qg[0].view(E, 2 * F, H // kdiv), qg[1].view(E, 2 * F, H // sdiv)
        self.dq, self.dd = qd[0].view(E, H, F // kdiv), qd[1].view(E, H, F // sdiv)
        if fmt == "nvfp4":
            # each bank quantised as one tensor: every expert carries the bank's scale
            self.ggu = torch.full((E,), qg[2], dtype=torch.float32, device=device)
            self.gdn = torch.full((E,), qd[2], dtype=torch.float32, device=device)
        if tokens > 1:
            if fmt != "q8_0":
                raise ValueError("the batched routed FFN takes Q8_0 banks")
            self._init_tokens(layer, device, E, H, F, k, tokens)
            return
        self.ids, self.gw = synth.routing(E, k, 3, layer, 2, device=device)
        self.x = synth.activations_bf16(1, H, 3, layer, 3, device=device)
        self.xq = torch.empty((1, H), dtype=torch.int8, device=device)
        self.xd = torch.empty((1, H // 32), dtype=torch.float32, device=device)
        self.ygu = torch.empty((k, 2 * F), dtype=torch.float32, device=device)
        self.hq = torch.empty((k, F), dtype=torch.int8, device=device)
        self.hd = torch.empty((k, F // 32), dtype=torch.float32, device=device)
        self.y = torch.empty((H,), dtype=torch.float32, device=device)
        self.status = torch.zeros((1,), dtype=torch.int32, device=device)
        # the selected experts' quant and scale planes, read once per token
        es = self.gd.element_size()
        self.weight_bytes = k * (self.gq[0].numel() + self.gd[0].numel() * es +
                                 self.dq[0].numel() + self.dd[0].numel() * es)

    def _init_tokens(self, layer, device, E, H, F, k, T):
        routes = [synth.routing(E, k, 3, layer, 2, t, device=device) for t in range(T)]
        self.ids = torch.stack([r[0] for r in routes]).contiguous()
        self.gw = torch.stack([r[1] for r in routes]).contiguous()
        self.x = synth.activations_bf16(T, H, 3, layer, 3, device=device)
        self.xq = torch.empty((T, H), dtype=torch.int8, device=device)
        self.xd = torch.empty((T, H // 32), dtype=torch.float32, device=device)
        P = T * k
        self.ws = torch.empty((P * (2 * F + H),), dtype=torch.float32, device=device)
        self.ygu = self.ws[:P * 2 * F].view(T, k, 2 * F)
        self.hq = torch.empty((T, k, F), dtype=torch.int8, device=device)
        self.hd = torch.empty((T, k, F // 32), dtype=torch.float32, device=device)
        self.ydn = self.ws[P * 2 * F:].view(T, k, H)
        self.y = torch.empty((T, H), dtype=torch.float32, device=device)
        self.status = torch.zeros((1,), dtype=torch.int32, device=device)
        # every distinct expert of the layer is read once per step
        distinct = len(set(self.ids.flatten().tolist()))
        self.pairs = P
        self.distinct = distinct
        self.weight_bytes = distinct * (self.gq[0].numel() + self.gd[0].numel() * 2 +
                                        self.dq[0].numel() + self.dd[0].numel() * 2)

    def gemv(self, mem, bank, *args, **kw):
        if self.fmt == "nvfp4":
            scales = args[0]
            gexp = self.ggu if bank is self.gq else self.gdn
            return mem.memra_nvfp4_moe_gemv(bank, scales, gexp, *args[1:], **kw)
        args = (bank,) + args
        if self.fmt == "q4_0":
            return mem.memra_q4_0_moe_gemv(*args, **kw)
        return mem.memra_q8_0_moe_gemv(*args, **kw)

    def run(self, mem, fused=False):
        if self.tokens > 1:
            self.run_tokens(mem, fused)
            return
        if fused:
            if self.fmt == "q4_0":
                mem.memra_q4_0_moe_ffn(self.gq, self.gd, self.dq, self.dd, self.ids, self.gw,
                                       self.x[0], y=self.y, workspace=self.ygu.view(-1),
                                       dev_status=self.status)
            elif self.fmt == "nvfp4":
                mem.memra_nvfp4_moe_ffn(self.gq, self.gd, self.ggu, self.dq, self.dd, self.gdn,
                                        self.ids, self.gw, self.x[0], y=self.y,
                                        workspace=self.ygu.view(-1), dev_status=self.status)
            else:
                mem.memra_q8_0_moe_ffn(self.gq, self.gd, self.dq, self.dd, self.ids, self.gw,
                                       self.x[0], y=self.y, workspace=self.ygu,
                                       dev_status=self.status)
            return
        mem.memra_quantize_q8_1(self.x, self.xq, self.xd)
        self.gemv(mem, self.gq, self.gd, self.ids, None, self.xq[0], self.xd[0], False,
                  y=self.ygu, dev_status=self.status)
        mem.memra_swiglu_quantize_q8_1(self.ygu, self.hq, self.hd)
        self.gemv(mem, self.dq, self.dd, self.ids, self.gw, self.hq, self.hd, True,
                  y=self.y, dev_status=self.status)

    def run_tokens(self, mem, fused):
        if fused:
            mem.memra_q8_0_moe_ffn_tokens(self.gq, self.gd, self.dq, self.dd, self.ids, self.gw,
                                          self.x, y=self.y, workspace=self.ws,
                                          dev_status=self.status)
            return
        T, k = self.ids.shape
        mem.memra_quantize_q8_1(self.x, self.xq, self.xd)
        self.gemv_tokens(mem, False)
        mem.memra_swiglu_quantize_q8_1(self.ygu.view(T * k, -1), self.hq.view(T * k, -1),
                                       self.hd.view(T * k, -1))
        self.gemv_tokens(mem, True)

    def gemv_tokens(self, mem, down):
        if down:
            mem.memra_q8_0_moe_gemv_tokens(self.dq, self.dd, self.ids, self.gw, self.hq, self.hd,
                                           True, y=self.y, workspace=self.ydn,
                                           dev_status=self.status)
        else:
            mem.memra_q8_0_moe_gemv_tokens(self.gq, self.gd, self.ids, None, self.xq, self.xd,
                                           False, y=self.ygu, dev_status=self.status)


def mma_suits(op):
    """Shapes the tensor-core entry point takes (K a multiple of 1024 up to 5120)."""
    N, K = op.wq.shape
    return op.fmt == "q8_0" and K % 1024 == 0 and K <= 5120 and N >= 16


def run_gemv_op(mem, op, quantize=True, fused=False, mma=False):
    """One product of a step: the fused entry point (quantisation in the kernel's
    prologue), or a q8_1 quantise launch followed by the GEMV / verify GEMM (with
    `mma`, the tensor-core entry point where the shape suits it)."""
    if fused:
        if op.fmt != "q8_0":
            raise ValueError("the fused quantise entry point takes Q8_0 weights")
        mem.memra_q8_0_quant_gemm(op.wq, op.wd, op.x, y=op.y)
        return
    if quantize:
        mem.memra_quantize_q8_1(op.x, op.xq, op.xd)
    if op.fmt == "nvfp4":
        if op.xq.shape[0] == 1:
            mem.memra_nvfp4_gemv(op.wq, op.wd, op.g, op.xq[0], op.xd[0], y=op.y[0])
        else:
            mem.memra_nvfp4_gemm_small_m(op.wq, op.wd, op.g, op.xq, op.xd, y=op.y)
        return
    if op.fmt == "q4_0":
        if op.xq.shape[0] == 1:
            mem.memra_q4_0_gemv(op.wq, op.wd, op.xq[0], op.xd[0], y=op.y[0])
        else:
            mem.memra_q4_0_gemm_small_m(op.wq, op.wd, op.xq, op.xd, y=op.y)
        return
    if mma and mma_suits(op):
        mem.memra_q8_0_gemm_small_m_mma(op.wq, op.wd, op.xq, op.xd, y=op.y)
    elif op.xq.shape[0] == 1:
        mem.memra_q8_0_gemv(op.wq, op.wd, op.xq[0], op.xd[0], y=op.y[0])
    else:
        mem.memra_q8_0_gemm_small_m(op.wq, op.wd, op.xq, op.xd, y=op.y)


class Workload:
    """A step = a fixed list of library calls; captured once into a CUDA graph."""

    def __init__(self, name, mem, device, layers=None, fused=False, ops=None, mma=False):
        self.name = name
        self.fused = fused
        self.mma = mma
        self.mem = mem
        self.device = device
        self.moe = None
        self.ops = []
        if ops is not None:
            self.ops = ops
        elif name == "dense27b_sweep":
            self.ops = build_dense_sweep(mem, device, M=1, layers=layers)
        elif name == "dense27b_sweep_nvfp4":
            self.ops = build_dense_sweep(mem, device, layers=layers, workload_id=6, fmt="nvfp4")
        elif name == "dense27b_sweep_q4_0":
            self.ops = build_dense_sweep(mem, device, M=1, layers=layers, workload_id=5,
                                         fmt="q4_0")
        elif name.startswith(("verify_m", "batch_m")):
            self.ops = build_dense_sweep(mem, device, M=rows_of(name),
                                         layers=layers, workload_id=2)
        elif name == "gemv_4096":
            self.ops = build_gemv_4096(mem, device)
        elif name == "stress_lm_head":
            self.ops = build_stress(mem, device, M=1) + build_stress(mem, device, M=8)
        elif name in ("moe_top8", "moe_top8_q4_0", "moe_top8_nvfp4", "moe_top8_tokens8",
                      "moe_top8_tokens16"):
            n = synth.MOE["layers"] if layers is None else layers
            fmt = ("q4_0" if name.endswith("q4_0") else
                   "nvfp4" if name.endswith("nvfp4") else "q8_0")
            tokens = tokens_of(name)
            self.moe = [MoeLayer(mem, layer, device, fmt=fmt, tokens=tokens)
                        for layer in range(n)]
        else:
            raise ValueError(name)
        self._pack_arenas()
        torch.cuda.synchronize(device)

    @property
    def weight_bytes(self):
        if self.moe is not None:
            return sum(m.weight_bytes for m in self.moe)
        return sum(op.weight_bytes for op in self.ops)

    @staticmethod
    def _arena(tensors, fill):
        """One contiguous buffer holding `tensors` (each view 16-byte aligned); returns the
        buffer and the views, filled from the tensors when `fill`."""
        step = 16 // tensors[0].element_size()
        sizes = [(t.numel() + step - 1) // step * step for t in tensors]
        arena = torch.empty(sum(sizes), dtype=tensors[0].dtype, device=tensors[0].device)
        views, off = [], 0
        for t, n in zip(tensors, sizes):
            v = arena[off:off + t.numel()].view(t.shape)
            if fill:
                v.copy_(t)
            views.append(v)
            off += n
        return arena, views

    def _pack_arenas(self):
        """Keep the step's activations in one contiguous bf16 buffer and its outputs in one
        fp32 buffer, as an engine's activation arena would, so that the end-to-end leg moves
        each with a single copy."""
        ins = self.inputs()
        self.in_arena, in_views = self._arena(ins, fill=True)
        new_in = {id(t): v for t, v in zip(ins, in_views)}
        self.out_arena, out_views = self._arena(self.outputs(), fill=False)
        if self.moe is not None:
            for m, x, y in zip(self.moe, in_views, out_views):
                m.x, m.y = x, y
        else:
            for op, y in zip(self.ops, out_views):
                op.x, op.y = new_in[id(op.x)], y

    @property
    def passes(self):
        """Product launches per dense product: batches above 8 rows take two passes."""
        if self.moe is not None:
            return 1
        return 2 if self.ops[0].xq.shape[0] > 8 else 1

    @property
    def launches_per_step(self):
        if self.moe is not None:
            if self.moe[0].tokens > 1:  # + the gated sum per token
                return (3 if self.fused else 5) * len(self.moe)
            return (2 if self.fused else 4) * len(self.moe)
        return (self.passes + (0 if self.fused else 1)) * len(self.ops)

    @property
    def gemv_launches_per_step(self):
        if self.moe is not None:
            return 2 * len(self.moe)
        return self.passes * len(self.ops)

    def step(self):
        if self.moe is not None:
            for m in self.moe:
                m.run(self.mem, fused=self.fused)
        else:
            for op in self.ops:
                run_gemv_op(self.mem, op, fused=self.fused, mma=self.mma)

    def gemv_only(self):
        """The step's weight-streaming kernels alone (activations already quantised)."""
        if self.moe is not None and self.fused:
            self.step()  # both launches of the fused layer stream weights
        elif self.moe is not None:
            for m in self.moe:
                if m.tokens > 1:
                    m.gemv_tokens(self.mem, False)
                    m.gemv_tokens(self.mem, True)
                    continue
                m.gemv(self.mem, m.gq, m.gd, m.ids, None, m.xq[0], m.xd[0], False,
                       y=m.ygu, dev_status=m.status)
                m.gemv(self.mem, m.dq, m.dd, m.ids, m.gw, m.hq, m.hd, True,
                       y=m.y, dev_status=m.status)
        else:
            for op in self.ops:
                run_gemv_op(self.mem, op, quantize=False, fused=self.fused, mma=self.mma)

    def inputs(self):
        if self.moe is not None:
            return [m.x for m in self.moe]
        seen, out = set(), []
        for op in self.ops:
            if id(op.x) not in seen:
                seen.add(id(op.x))
                out.append(op.x)
        return out

    def outputs(self):
        if self.moe is not None:
            return [m.y for m in self.moe]
        return [op.y for op in self.ops]

    def capture(self, fn):
        stream = torch.cuda.Stream(self.device)
        stream.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(stream):
            fn()  # warm-up outside the graph (sets kernel attributes)
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        torch.cuda.synchronize(self.device)
        return g


# ----------------------------------------------------------------------------
# Timing helpers.
# ----------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        self.lines = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            if not uuid.startswith("GPU-"):
                uuid = "GPU-" + uuid
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", uuid, "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [s.strip() for s in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
                power.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, world_size, device=None, backend_device="cpu"):
    """Max of a float over all ranks (identity for one rank)."""
    if world_size <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=backend_device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world_size):
    if world_size > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(kernel_source_hash):
    """DRAM bytes per launch of the GEMV kernel from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "gemv_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_sha256") == kernel_source_hash:
            return d
    except Exception:
        pass
    return None


def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("gemm.cu", "product.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "block_quantized_decode_quantize_gb300", "csrc",
                               name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def read_ceiling(mem, device, stream, nbytes=4 << 30, reps=8):
    """A plain read stream over `nbytes` of device memory (memra_read_stream), best over
    1-4 CTAs per SM: the ceiling the weight-streaming kernels approach."""
    buf = torch.ones((nbytes,), dtype=torch.uint8, device=device)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    best, per = 0.0, {}
    for c in (1, 2, 3, 4):
        sink = torch.zeros((sms * c,), dtype=torch.int32, device=device)
        with torch.cuda.stream(stream):
            for _ in range(2):
                mem.memra_read_stream(buf, sink, c)
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            start.record(stream)
            for _ in range(reps):
                mem.memra_read_stream(buf, sink, c)
            end.record(stream)
        end.synchronize()
        gbs = nbytes * reps / (start.elapsed_time(end) / 1e3) / 1e9
        per[str(c)] = round(gbs, 1)
        best = max(best, gbs)
    del buf
    return best, per


def time_graph(graph, reps, stream):
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            graph.replay()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1000.0


# ----------------------------------------------------------------------------
# CPU oracle sample (the reported CPU baseline and the reference arm).
# ----------------------------------------------------------------------------

class CpuOracleSample:
    """The CPU oracle (quantise x + GEMV, all host threads) on layer 0's four products
    of the dense sweep.  Weight ingest is done once, untimed, like the GPU's."""

    def __init__(self):
        import numpy as np

        import oracle
        self.oracle = oracle
        self.threads = os.cpu_count() or 1
        cfg = synth.DENSE27B
        self.items = []
        for t, (name, N, K) in enumerate(cfg["gemvs"]):
            w = synth.weights_fp32(N, K, 1, 0, t, device="cpu").numpy()
            wq, wd = oracle.quantize_q8_0(w)
            del w
            x = synth.activations_bf16(1, K, 1, 0, t, 1001, outlier_frac=cfg["outlier_frac"],
                                       outlier_scale=cfg["outlier_scale"])
            xb = x.view(torch.int16).numpy().view(np.uint16)
            self.items.append((name, wq, wd, xb, synth.q8_0_bytes(N, K)))
        self.done = 0

    def run_one(self, threads=None):
        """Run the next product; returns (seconds, weight bytes)."""
        name, wq, wd, xb, b = self.items[self.done % len(self.items)]
        t0 = time.perf_counter()
        xq, xd = self.oracle.quantize_q8_1(xb)
        self.oracle.gemm(wq, wd, xq, xd, threads=threads or self.threads)
        dt = time.perf_counter() - t0
        self.done += 1
        return dt, b

    def run_for(self, budget_s, threads=None):
        """Run products until `budget_s` seconds of oracle time; returns (GB/s, seconds,
        products)."""
        spent, nbytes, n = 0.0, 0, 0
        while spent < budget_s or n < len(self.items):
            dt, b = self.run_one(threads)
            spent += dt
            nbytes += b
            n += 1
        return nbytes / spent / 1e9, spent, n

    def describe(self, n):
        return ("%d Q8_0 products (q8_1 quantise of x + GEMV) cycling through layer 0's QKV, "
                "O, gate+up and down of the dense sweep; %d OpenMP threads"
                % (n, self.threads))


# ----------------------------------------------------------------------------
# Arms.
# ----------------------------------------------------------------------------

def workload_config(name, wl):
    cfg = {"workload": name}
    if name.startswith(("dense27b_sweep", "verify_m", "batch_m")):
        cfg.update({"layers": len(wl.ops) // 4, "hidden": synth.DENSE27B["hidden"],
                    "gemvs_per_layer": [[n, N, K] for n, N, K in synth.DENSE27B["gemvs"]],
                    "M": rows_of(name),
                    "activations": "bf16 N(0,1), 0.1% of entries x20"})
        if name.startswith("batch_m"):
            cfg["sequences"] = rows_of(name)
            cfg["passes_per_product"] = 2 if rows_of(name) > 8 else 1
    elif name == "gemv_4096":
        cfg.update({"N": 4096, "K": 4096, "M": 1, "weight_copies": len(wl.ops)})
    elif name.startswith("moe_top8"):
        cfg.update(dict(synth.MOE))
        if wl.moe[0].tokens > 1:
            cfg["tokens"] = wl.moe[0].tokens
            cfg["pairs_per_layer"] = wl.moe[0].pairs
            cfg["distinct_experts_per_layer"] = round(
                sum(m.distinct for m in wl.moe) / len(wl.moe), 2)
            cfg["weight_bytes_counted"] = "each distinct routed expert of a layer once"
    elif name == "stress_lm_head":
        cfg.update({"shapes": [[n, N, K] for n, N, K in synth.STRESS["shapes"]], "M": [1, 8]})
    cfg["weights"] = ("N(0,0.02) fp32 quantised to Q4_0 (32 4-bit codes + fp16 scale per block)"
                      if name.endswith("q4_0") else
                      "N(0,0.02) fp32 quantised to NVFP4 (E2M1 codes, E4M3 scale per 16, fp32 "
                      "tensor scale)" if name.endswith("nvfp4") else
                      "N(0,0.02) fp32 quantised to Q8_0 (32 int8 + fp16 scale per block)")
    cfg["weight_bytes_per_step"] = wl.weight_bytes
    cfg["l2"] = ("inputs larger than L2: %.2f GB of distinct weights per step vs 129 MB L2"
                 % (wl.weight_bytes / 1e9))
    return cfg


def time_step_and_products(wl, steps, warmup, stream):
    """Seconds for `steps` CUDA-graph replays of the whole step and of its product
    launches alone, after `warmup` replays of the step."""
    step_graph = wl.capture(wl.step)
    gemv_graph = wl.capture(wl.gemv_only)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step_graph.replay()
    torch.cuda.synchronize(wl.device)
    el = time_graph(step_graph, steps, stream)
    gel = time_graph(gemv_graph, steps, stream)
    return el, gel


def measure_configs(mem, device, main_wl, stream, peak, warmup):
    """Every other configuration of the benchmark on this GPU, each timed over a short
    region (CUDA-graph replays, CUDA events on the launching stream): the 4096 x 4096
    GEMV, the verify GEMMs at M = 2, 4, 8 on the dense sweep's own weights, the top-8
    MoE layer sweep, and the LM head + down stress shapes at M = 1 and 8."""
    legs = []
    legs.append(("cfg0_gemv_4096", lambda: Workload("gemv_4096", mem, device), 200,
                 "one call = q8_1 quantise + GEMV; 32 rotating weight copies (570 MB > L2)",
                 32))
    for M in (2, 4, 8):
        legs.append(("cfg2_verify_m%d" % M,
                     lambda M=M: Workload("verify_m%d" % M, mem, device,
                                          ops=sweep_rows_like(main_wl.ops, M)), 10,
                     "64-layer sweep, M = %d rows per product (the dense sweep's weights)" % M,
                     None))
    legs.append(("cfg3_moe_top8", lambda: Workload("moe_top8", mem, device, fused=True), 50,
                 "48 routed layers (memra_q8_0_moe_ffn), top-8 of 128 experts, one token",
                 None))
    for M in (1, 8):
        legs.append(("cfg4_lm_head_down_m%d" % M,
                     lambda M=M: Workload("stress_lm_head", mem, device,
                                          ops=build_stress(mem, device, M=M)), 50,
                     "LM head 151936x5120 + down 5120x17408, M = %d, 1%% zero and 1%% x50 blocks"
                     % M, None))
    out = {}
    for key, make, steps, what, calls in legs:
        wl = make()
        el, gel = time_step_and_products(wl, steps, warmup, stream)
        b = wl.weight_bytes
        us = el / steps * 1e6
        gbs = b * steps / el / 1e9
        d = {"what": what, "us_per_step": round(us, 2), "gb_s": round(gbs, 1),
             "frac_of_measured": round(gbs / peak, 4),
             "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
             "products_alone_gb_s": round(b * wl.passes * steps / gel / 1e9, 1),
             "weight_bytes_per_step": b, "steps": steps,
             "launches_per_step": wl.launches_per_step}
        if calls:
            d["us_per_call"] = round(us / calls, 3)
        if wl.moe is not None:
            d["tok_per_s"] = round(1e6 / us, 1)
        out[key] = d
        del wl
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()
    return out


def run_memra(args):
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import block_quantized_decode_quantize_gb300 as mem
    from block_quantized_decode_quantize_gb300 import build
    if rank == 0 or world == 1:
        build.build()
    barrier(world)
    mem.lib()

    # Dense products quantise with a separate launch unless --fused; the routed FFN
    # uses its two-kernel entry point unless --unfused.
    fused = ((not args.unfused) if args.workload.startswith("moe_top8") else args.fused)
    wl = Workload(args.workload, mem, device, layers=args.layers, fused=fused,
                  mma=args.mma)
    stream = torch.cuda.Stream(device)
    step_graph = wl.capture(wl.step)
    gemv_graph = wl.capture(wl.gemv_only)

    # Warm-up, then the timed region: K graph replays of the whole step.
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            step_graph.replay()
    torch.cuda.synchronize(device)
    barrier(world)
    torch.cuda.synchronize(device)
    clocks = ClockSampler(device)
    time.sleep(0.2)
    elapsed = time_graph(step_graph, args.steps, stream)
    torch.cuda.synchronize(device)
    clock_info = clocks.stop()
    barrier(world)
    elapsed_max = max_over_ranks(elapsed, world, backend_device=device)

    bytes_step = wl.weight_bytes
    value = world * bytes_step * args.steps / elapsed_max / 1e9
    ms_per_step = elapsed_max / args.steps * 1e3

    # Dominant kernel: the weight-streaming GEMV alone, same buffers and launch shapes.
    g_elapsed = time_graph(gemv_graph, args.steps, stream)
    n_gemv = wl.gemv_launches_per_step * args.steps
    gemv_avg_s = g_elapsed / n_gemv
    # Each launch streams its product's weights once (a two-pass batch streams them twice).
    bytes_per_launch = bytes_step * wl.passes / wl.gemv_launches_per_step
    achieved = bytes_per_launch / gemv_avg_s / 1e9
    peak, peak_kind = measured_peaks()
    prof = profile_traffic(kernel_source_hash())
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": (round(prof["dram_bytes_per_launch"] * bytes_per_launch /
                                  prof["weight_bytes_per_launch"])
                            if prof else None),
                "peak_kind": peak_kind + " copy bandwidth (MEASURED_PEAKS hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "kernel": "%s product kernel (%s, M=%s)" % (
                    {"q4_0": "Q4_0", "nvfp4": "NVFP4"}.get(
                        wl.ops[0].fmt if wl.ops else wl.moe[0].fmt, "Q8_0"),
                    "routed experts" if wl.moe is not None else
                    ("quantise fused" if wl.fused else "q8_1 input"),
                    1 if wl.moe is not None else "%d%s" % (
                        wl.ops[0].xq.shape[0],
                        " in 2 passes" if wl.passes == 2 else "")),
                "avg_launch_us": round(gemv_avg_s * 1e6, 3),
                "bytes_per_launch": int(bytes_per_launch),
                "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4)}

    # The read-only stream ceiling on this GPU (4 GiB, larger than L2), for context.
    ceiling, ceiling_per = (None, None) if args.no_read_ceiling else read_ceiling(mem, device,
                                                                                  stream)
    if ceiling:
        roofline["read_ceiling_gbs"] = round(ceiling, 1)
        roofline["frac_of_read_ceiling"] = round(achieved / ceiling, 4)

    # End to end through the public API: pinned host activations in, every output out.
    # The step's activations and outputs live in one arena each: one copy each way.
    ins = [wl.in_arena]
    outs = [wl.out_arena]
    h_in = [t.detach().cpu().pin_memory() for t in ins]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    e2e_steps = max(3, min(args.steps, 50))
    torch.cuda.synchronize(device)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            for d, h in zip(ins, h_in):
                d.copy_(h, non_blocking=True)
            step_graph.replay()
            for h, d in zip(h_out, outs):
                h.copy_(d, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, backend_device=device)
    e2e_value = world * bytes_step * e2e_steps / e2e_s / 1e9

    configs = None
    if args.workload == "dense27b_sweep" and args.layers is None and not args.no_configs:
        cs = ClockSampler(device)
        configs = measure_configs(mem, device, wl, stream, peak, args.warmup)
        configs["clocks"] = cs.stop()

    status_bad = 0
    if wl.moe is not None:
        status_bad = int(sum(int(m.status.item()) for m in wl.moe))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cs = CpuOracleSample()
        v, spent, n = cs.run_for(args.cpu_budget)
        v1, spent1, n1 = cs.run_for(min(4.0, args.cpu_budget), threads=1)
        cpu = {"value": round(v, 3), "unit": "GB/s", "cores": cs.threads, "kind": "oracle",
               "sample": cs.describe(n), "seconds": round(spent, 2),
               "single_thread": {"value": round(v1, 3), "unit": "GB/s", "products": n1,
                                 "seconds": round(spent1, 2)}}

    if rank == 0:
        cfg = workload_config(args.workload, wl)
        cfg["parallelism"] = "replicas x%d (no data-path collective)" % world
        if wl.moe is None:
            if wl.mma:
                cfg["products"] = ("memra_q8_0_gemm_small_m_mma (tensor cores) where K is a "
                                   "multiple of 1024 up to 5120, else memra_q8_0_gemm_small_m")
            cfg["activation_quantise"] = ("fused into the product's prologue "
                                          "(memra_q8_0_quant_gemm)" if wl.fused else
                                          "separate memra_quantize_q8_1 launch")
        else:
            if wl.moe[0].tokens > 1:
                cfg["layer_calls"] = ("memra_q8_0_moe_ffn_tokens (3 kernels)" if wl.fused else
                                      "quantize, moe_gemv_tokens, swiglu_quantize, "
                                      "moe_gemv_tokens (gated: + per-token sum)")
            else:
                cfg["layer_calls"] = ("memra_%s_moe_ffn (2 kernels)" % wl.moe[0].fmt
                                      if wl.fused else
                                      "quantize, moe_gemv, swiglu_quantize, moe_gemv")
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 (dp4a int32 block sums, fp32 scale-accumulate)",
            "data": "synthetic (seeded N(0,0.02) weights, bf16 N(0,1) activations)",
            "config": cfg,
            "us_per_step": round(ms_per_step * 1e3, 2),
            "tok_per_s": round(1e3 * tokens_of(args.workload) / ms_per_step, 2)
            if args.workload.startswith(
                ("moe_top8", "dense27b_sweep", "verify_m", "batch_m")) else None,
            "hbm_frac_of_measured": round(value / world / peak, 4),
            "hbm_frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "pinned H2D of the step's activation arena, CUDA-graph replay of "
                            "the step's C-ABI calls, D2H of the output arena, host sync per step",
                    "steps": e2e_steps},
            "gpu_launches": wl.launches_per_step * args.steps,
            "read_ceiling": {"value": round(ceiling, 1), "unit": "GB/s",
                             "kernel": "memra_read_stream (diagnostic)", "bytes": 4 << 30,
                             "by_ctas_per_sm": ceiling_per} if ceiling else None,
            "clocks": clock_info,
        }
        if configs is not None:
            line["configs"] = configs
        if status_bad:
            line["moe_status_flags"] = status_bad
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    world, rank, _ = dist_info()
    if rank != 0:
        return
    cs = CpuOracleSample()
    for _ in range(args.warmup):
        cs.run_one()
    spent, nbytes = 0.0, 0
    for _ in range(args.steps):
        dt, b = cs.run_one()
        spent += dt
        nbytes += b
    value = nbytes / spent / 1e9
    sample = ("each step one Q8_0 product (q8_1 quantise of x + GEMV) of layer 0 of the dense "
              "sweep, cycling QKV, O, gate+up, down; %d OpenMP threads" % cs.threads)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(spent / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "impl": "reference",
        "dtype": "int8 (int32 block sums, fp32 scale-accumulate)",
        "data": "synthetic (seeded N(0,0.02) weights, bf16 N(0,1) activations)",
        "config": {"workload": "dense27b_sweep", "layers_sampled": 1, "M": 1},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "kind": "oracle",
                         "cores": cs.threads, "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("memra", "reference"), default="memra")
    ap.add_argument("--workload", choices=WORKLOADS, default="dense27b_sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--fused", action="store_true",
                    help="dense workloads: quantise activations in the product's prologue "
                         "(memra_q8_0_quant_gemm) instead of a separate q8_1 launch")
    ap.add_argument("--mma", action="store_true",
                    help="dense workloads: the tensor-core entry point "
                         "(memra_q8_0_gemm_small_m_mma) for the products it takes")
    ap.add_argument("--unfused", action="store_true",
                    help="moe_top8 workloads: four calls per layer instead of the two-kernel "
                         "routed FFN entry point")
    ap.add_argument("--no-configs", action="store_true",
                    help="default workload: skip the short measurements of the other "
                         "configurations")
    ap.add_argument("--no-read-ceiling", action="store_true",
                    help="skip the 4 GiB read-stream ceiling (profiling captures)")
    ap.add_argument("--layers", type=int, default=None,
                    help="fewer layers than the workload's own (profiling captures only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_memra(args)


if __name__ == "__main__":
    main()
