"""Host logic of bench.py without a GPU: the multi-rank reduction over gloo (world size 2),
the reference arm's rank rule, and the algorithmic byte / FLOP accounting."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch

    import bench

    r, w, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    slowest = bench.dist_max(1.5 * (r + 1), w)
    bench.dist_barrier(w)
    q.put((r, slowest))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 3.0), (1, 3.0)]


def test_reference_arm_only_rank0(monkeypatch):
    import bench

    class A:
        workload, steps, warmup = "b1_s2048", 1, 3

    assert bench.run_reference(A(), rank=1, world=2, local=1) is None


def test_reference_arm_line():
    """Rank 0 of the reference arm times the oracle on a bounded sample per step and reports that
    measured time (so K steps fit in the run's own clock), with the same config dict as the GPU
    arm and the full-step estimate beside it."""
    import bench
    from mla_latent_kv_absorb_gb300 import synth

    class A:
        workload, steps, warmup = "b1_s2048", 2, 1

    res = bench.run_reference(A(), rank=0, world=1, local=0)
    inp = synth.make_workload("b1_s2048")
    assert res["impl"] == "reference" and res["config"] == bench.bench_config(A(), inp, 1)
    assert res["metric"] == bench.METRIC and res["unit"] == bench.UNIT and res["higher_is_better"] is False
    cb = res["cpu_baseline"]
    assert cb["value"] == res["value"] > 0 and cb["kind"] == "oracle" and cb["cores"] >= 1
    assert cb["full_step_estimate_us"] >= res["value"]
    assert res["e2e"]["value"] == res["value"] and res["e2e"]["h2d_bytes_per_step"] == 0


def test_accounting_matches_roofline_table():
    import bench
    from mla_latent_kv_absorb_gb300 import synth

    class Fake:
        def __init__(self, kv_dtype, lens, q=1):
            self.kv_dtype, self.seq_lens, self.queries_per_seq = kv_dtype, np.asarray(lens, np.int32), q
            self.batch, self.num_tokens, self.rows = len(lens), int(sum(lens)), len(lens) * q

    acc = bench.workload_accounting(Fake("bf16", [65536] * 16))
    assert acc["kv_bytes"] == 1_207_959_552          # 16 x 1024 pages x 73,728 B
    assert abs(acc["step_flop"] / 1e9 - 292.6) < 0.5   # QK + PV + absorb + out-proj
    assert abs(acc["step_bytes"] / 1e6 - 1242.8) < 1.0
    acc = bench.workload_accounting(Fake("fp8_e4m3", [8192] * 128))
    assert acc["kv_bytes"] == 128 * 8192 * 644         # e4m3 latent + fp32 scale + bf16 k_R
    # four new tokens per sequence: the cache is read once, the attention FLOPs follow the rows
    acc = bench.workload_accounting(Fake("bf16", [8192] * 16, q=4))
    assert acc["kv_bytes"] == 16 * 8192 * 1152
    assert acc["scanned"] == 16 * (8189 + 8190 + 8191 + 8192)
    assert acc["decode_flop"] == acc["scanned"] * 128 * 2 * (576 + 512)


def test_warmup_floor():
    import bench

    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_kernel_hash_covers_included_sources():
    """A decode kernel's recorded traffic is keyed by a hash of its sources: every header its
    main file includes (transitively, within csrc/) must be part of that hash."""
    import re

    import bench

    for kernel, files in bench.KERNEL_SOURCES.items():
        todo, seen = [files[0]], set()
        while todo:
            rel = todo.pop()
            if rel in seen:
                continue
            seen.add(rel)
            text = open(os.path.join(ROOT, rel)).read()
            for inc in re.findall(r'#include\s+"([^"]+\.cuh)"', text):
                todo.append(os.path.join(os.path.dirname(rel), inc))
        assert seen <= set(files), (kernel, sorted(seen - set(files)))


def test_recorded_traffic_only_for_the_current_source(tmp_path, monkeypatch):
    import json

    import bench

    path = tmp_path / "traffic.json"
    rec = {"kernel": "decode_bf16_kernel", "workload": "b16_s65536", "tokens": 1000,
           "dram_bytes_per_launch": 2_000_000, "kernel_hash": bench.kernel_hash("decode_bf16_kernel")}
    path.write_text(json.dumps([rec]))
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(path))
    assert bench.recorded_traffic("decode_bf16_kernel", "b16_s65536", 1000) == 2_000_000
    assert bench.recorded_traffic("decode_bf16_kernel", "b16_s65536", 500) == 1_000_000  # scaled by tokens
    assert bench.recorded_traffic("decode_fp8_kernel", "b16_s65536", 1000) is None
    rec["kernel_hash"] = "0" * 16  # taken on another version of the kernel
    path.write_text(json.dumps([rec]))
    assert bench.recorded_traffic("decode_bf16_kernel", "b16_s65536", 1000) is None


def test_recorded_traffic_close_to_algorithmic_bytes():
    """Structural self-check on the committed ncu records: each decode kernel's measured DRAM
    traffic for one launch is within 5 % of the bytes the algorithm must move (every cached token
    once, the queries in, the latent outputs out): nothing is read twice."""
    import json

    import bench

    class Fake:
        def __init__(self, kv_dtype, lens):
            self.kv_dtype, self.seq_lens, self.queries_per_seq = kv_dtype, np.asarray(lens, np.int32), 1
            self.batch, self.num_tokens, self.rows = len(lens), int(sum(lens)), len(lens)

    shapes = {"b16_s65536": ("bf16", [65536] * 16), "b128_s8192_fp8": ("fp8_e4m3", [8192] * 128)}
    with open(bench.TRAFFIC_PATH) as f:
        records = json.load(f)
    assert {r["workload"] for r in records} == set(shapes)
    for r in records:
        dtype, lens = shapes[r["workload"]]
        algorithmic = bench.workload_accounting(Fake(dtype, lens))["decode_bytes"]
        ratio = r["dram_bytes_per_launch"] / algorithmic
        assert 0.95 <= ratio <= 1.05, (r["kernel"], ratio)
        assert r["dram_bytes_per_launch"] == r["dram_bytes_read"] + r["dram_bytes_write"]


def test_reference_arm_under_torchrun_two_ranks():
    """The reference arm launched the way the driver launches N > 1 (torchrun, two ranks on this
    host): rank 0 alone times the oracle and prints one JSON line, the other rank exits 0 without
    work."""
    import json
    import subprocess

    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus",
           "2", "--steps", "1", "--warmup", "3", "--workload", "b1_s2048"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
