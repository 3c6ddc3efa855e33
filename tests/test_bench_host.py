"""Host-side logic of bench.py: argument rules, rank aggregation over gloo (world
size 2 on CPU), workload byte counts, and the reference arm's JSON line (the CPU
oracle, which runs without a GPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

import bench
import synth


def test_dense_sweep_bytes_match_the_shapes():
    per_layer = (7168 * 5120 + 5120 * 5120 + 34816 * 5120 + 5120 * 17408) * 34 // 32
    assert synth.dense27b_bytes_per_token() == 64 * per_layer
    assert abs(synth.dense27b_bytes_per_token() / 1e9 - 22.46) < 0.01


def test_warmup_must_be_at_least_three():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2", "--steps", "1"])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, values, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(values[rank], world, backend_device="cpu")
        bench.barrier(world)
        out[rank] = m
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    values = [1.25, 3.5]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, values, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == 3.5 and out[1] == 3.5


def test_single_rank_aggregation_is_identity():
    assert bench.max_over_ranks(2.5, 1) == 2.5


def test_dist_info_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_info() == (1, 0, 0)


def test_workload_rows_and_tokens():
    assert bench.rows_of("dense27b_sweep") == 1
    assert bench.rows_of("verify_m8") == 8 and bench.rows_of("batch_m16") == 16
    assert bench.tokens_of("batch_m16") == 16 and bench.tokens_of("moe_top8_tokens8") == 8
    assert bench.tokens_of("moe_top8_tokens16") == 16
    assert bench.tokens_of("dense27b_sweep_nvfp4") == 1 and bench.tokens_of("verify_m4") == 1
    for name in ("batch_m16", "moe_top8_tokens8", "dense27b_sweep_nvfp4", "moe_top8_nvfp4"):
        assert name in bench.WORKLOADS


def test_unknown_workload_is_rejected():
    with pytest.raises(SystemExit):
        bench.main(["--workload", "no_such_workload"])


def test_verify_legs_share_the_sweep_weights():
    """The verify configurations reuse the dense sweep's weight tensors (no second copy)
    with M seeded activation rows per product."""
    ops = []
    for t, (name, N, K) in enumerate((("a", 8, 64), ("b", 4, 64), ("c", 16, 64), ("d", 4, 128))):
        wq = torch.zeros((N, K), dtype=torch.int8)
        wd = torch.zeros((N, K // 32), dtype=torch.float16)
        ops.append(bench.Gemv(wq, wd, torch.zeros((1, K), dtype=torch.bfloat16), name))
    rows = bench.sweep_rows_like(ops, 4)
    assert len(rows) == len(ops)
    for a, b in zip(ops, rows):
        assert b.wq.data_ptr() == a.wq.data_ptr() and b.wd.data_ptr() == a.wd.data_ptr()
        assert b.x.shape == (4, a.x.shape[1]) and b.y.shape == (4, a.wq.shape[0])
    again = bench.sweep_rows_like(ops, 4)
    assert all(torch.equal(p.x, q.x) for p, q in zip(rows, again))   # seeded


def test_reference_arm_prints_one_contract_line():
    """The reference arm times the oracle on the host cores and prints the JSON line the
    driver reads: the same metric and unit as the main arm, impl "reference", a CPU
    baseline describing the run and an e2e object with no host-device bytes."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], cwd=root, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"]["workload"] == "dense27b_sweep"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["value"] == d["value"] and cpu["unit"] == "GB/s"
    assert cpu["cores"] >= 1 and cpu["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == "GB/s"
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
