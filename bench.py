#!/usr/bin/env python3
"""Benchmark of the MLA decode step on GB300: one JSON line on stdout (rank 0).

A step is one pass of the whole decode path over one batch: absorb W_UK into q, paged
split-KV decode, log-sum-exp merge of split partials, W_UV projection.  The default workload
is 16 sequences of 65,536 tokens (a 1.21 GB bf16 latent cache, shuffled 64-token pages),
the configuration the 70 %-of-roofline target is stated on.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

Timing: W warm-up steps, then exactly K timed steps between a barrier + synchronize on both
sides.  Each step is bracketed by CUDA events on the launch stream, with events between its
kernels so each kernel's duration is measured live; a 512 MB buffer is rewritten before every
step (outside the events) so L2 starts cold, and the 1.2 GB cache is itself larger than L2.
`value` is the mean device time per step (microseconds, lower is better); with N ranks every
rank runs its own replica of the workload and the slowest rank is reported.

`e2e` times the same step through the public API with host buffers (DecodeStep.run_host with
pinned tensors, i.e. the captured step of mla_step_graph_run): per step the block table and the
queries are copied host -> device, the kernels run and the output is copied back, with the
host waiting for it; wall clock around all of it.  The lengths do not change between steps, so
the split plan made (and copied) when the step was captured stays valid.

`--impl reference` times the CPU oracle (plain fp64 C, the definition of the result) on the
host cores, on a bounded sample of the same workload per step, scaled to a full step.
"""
from __future__ import annotations

import argparse
import ctypes
import ctypes.util
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_latent_kv_absorb_gb300 import synth  # noqa: E402

METRIC = "MLA decode us/step (KV TB/s & TFLOP/s as fraction of GB300 roofline)"
UNIT = "us/step"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "decode_traffic.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
KERNEL_SOURCES = {
    "decode_bf16_kernel": ["mla_latent_kv_absorb_gb300/csrc/decode.cuh", "mla_latent_kv_absorb_gb300/csrc/ptx.cuh"],
    "decode_fp8_kernel": ["mla_latent_kv_absorb_gb300/csrc/decode_fp8.cuh", "mla_latent_kv_absorb_gb300/csrc/decode.cuh",
                          "mla_latent_kv_absorb_gb300/csrc/ptx.cuh"],
}


# ----------------------------------------------------------------------------- distributed helpers

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def dist_barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def dist_max(value: float, world: int, device="cpu") -> float:
    """Max of a per-rank float over all ranks (the slowest rank sets the step time)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks (NVML, read only)

class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML in a thread (reads only)."""

    HW_SLOWDOWN, SW_POWER_CAP, HW_THERMAL, SW_THERMAL = 0x8, 0x4, 0x40, 0x20

    def __init__(self, index: int, period_s: float = 0.002):
        self.samples, self.reasons_seen = [], set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._period = period_s
        self._ok = False
        try:
            name = ctypes.util.find_library("nvidia-ml") or "libnvidia-ml.so.1"
            self.nvml = ctypes.CDLL(name)
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:  # 1 = SM
                self.max_mhz = int(mx.value)
            self._ok = True
        except OSError:
            pass

    def _read(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) == 0:
            self.samples.append(int(clk.value))
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(self.handle, ctypes.byref(rs)) == 0:
            v = int(rs.value)
            for bit, name in ((self.HW_SLOWDOWN, "hw_slowdown"), (self.SW_POWER_CAP, "sw_power_cap"),
                              (self.HW_THERMAL, "hw_thermal_slowdown"), (self.SW_THERMAL, "sw_thermal_slowdown")):
                if v & bit:
                    self.reasons_seen.add(name)

    def _loop(self):
        while not self._stop.is_set():
            self._read()
            time.sleep(self._period)

    def __enter__(self):
        if self._ok:
            self._t = threading.Thread(target=self._loop, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self._ok:
            self._stop.set()
            self._t.join()
            self._read()

    def summary(self):
        if not self._ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": "unavailable"}
        return {"sm_mhz": int(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons_seen), "samples": len(self.samples), "source": "nvml"}


# ----------------------------------------------------------------------------- accounting

def visible_tokens(seq_lens, q: int) -> int:
    """Cached tokens the step's queries attend to, summed over query rows: with q new tokens per
    sequence, token t of sequence b sees the first S_b - q + 1 + t."""
    lens = np.asarray(seq_lens, dtype=np.int64)
    return int((q * lens - q * (q - 1) // 2).sum())


def workload_accounting(inp):
    """Algorithmic bytes and FLOPs of one step (no partial-output traffic, no decompression).
    Every cached token is read once (the minimum, also when several query rows of a sequence
    attend to it); every (query row, visible token) pair costs the absorbed QK and PV FLOPs."""
    R, T = inp.rows, inp.num_tokens
    scanned = visible_tokens(inp.seq_lens, inp.queries_per_seq)
    row_bytes = 1152 if inp.kv_dtype == "bf16" else 512 + 4 + 128
    kv_bytes = T * row_bytes
    w_bytes = 2 * 128 * 128 * 512 * 2
    q_bytes = R * 128 * (128 + 64) * 2
    out_bytes = R * 128 * 128 * 2
    decode_bytes = kv_bytes + R * 128 * (512 + 64) * 2 + R * 128 * (512 * 2 + 4)
    attn_flop = scanned * 128 * 2 * (576 + 512)
    proj_flop = 2 * R * 128 * (2 * 128 * 512)
    return dict(tokens=T, scanned=scanned, kv_bytes=kv_bytes, step_bytes=kv_bytes + w_bytes + q_bytes + out_bytes,
                decode_bytes=decode_bytes, step_flop=attn_flop + proj_flop, decode_flop=attn_flop)


def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS)


def kernel_hash(kernel: str = "decode_bf16_kernel") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, tokens: int):
    """DRAM bytes per decode launch from the committed ncu record of this kernel, if it was taken
    on the current kernel source; scaled to this workload's tokens when captured on a smaller
    case of the same kernel."""
    try:
        with open(TRAFFIC_PATH) as f:
            records = json.load(f)
    except (OSError, ValueError):
        return None
    if isinstance(records, dict):
        records = [records]
    for t in records:
        if t.get("kernel") == kernel and t.get("kernel_hash") == kernel_hash(kernel):
            return t["dram_bytes_per_launch"] / t["tokens"] * tokens
    return None


def bench_config(args, inp, world):
    """The workload, identical in both arms' JSON lines."""
    cfg = {"workload": args.workload, "desc": synth.WORKLOADS[args.workload]["desc"],
           "global_batch": inp.batch * world, "seq_len": int(inp.seq_lens.max()),
           "tokens_per_replica": int(inp.num_tokens), "parallelism": f"replicas x{world}"}
    if inp.queries_per_seq > 1:
        cfg["queries_per_seq"] = inp.queries_per_seq
    return cfg


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "Hardware"):
        for line in text.splitlines():
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    parts = sorted({ln.split(":", 1)[1].strip() for ln in text.splitlines() if ln.startswith("CPU part")})
    return f"{os.uname().machine} (CPU part {', '.join(parts)})" if parts else os.uname().machine


# ----------------------------------------------------------------------------- the GPU arm

def run_ours(args, rank, world, local):
    from mla_latent_kv_absorb_gb300 import binding

    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    binding.lib()
    inp = synth.make_workload(args.workload, seed=synth.DEFAULT_SEED + rank, poison_tail=False)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, device)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt,
                              item_cost_pages=args.item_cost_pages, fused_absorb=args.absorb == "fused",
                              fused_tail=args.tail == "fused", queries_per_seq=inp.queries_per_seq, **kv)
    acc = workload_accounting(inp)
    peaks = load_peaks()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)

    # the kernels of one step, one by one (with the absorb as a kernel of its own, so that the decode
    # kernel's own duration gives the roofline)
    def k_absorb():
        binding.mla_absorb_q(q_c, step.w_uk, step.q_abs, stream)

    def k_decode():
        binding.mla_decode_paged(step.info, step.plan_dev, step.q_abs, q_r, kv_pool=step.kv_pool,
                                 block_table=step.block_table, o_lat=step.o_lat, lse=step.lse,
                                 dev_error=step.dev_error, workspace=step.workspace, kv_scale=step.kv_scale,
                                 kr_pool=step.kr_pool, softmax_scale=step.softmax_scale, stream=stream)

    def k_merge():
        binding.mla_combine_splits(step.info, step.plan_dev, step.workspace, step.o_lat, step.lse, stream)

    def k_proj():
        binding.mla_out_proj(step.o_lat, step.w_uv, step.out, stream)

    def k_tail():
        binding.mla_merge_out_proj(step.info, step.plan_dev, step.workspace, step.o_lat, step.lse, step.w_uv,
                                   step.out, step.dev_error, stream)

    parts = [("absorb", k_absorb), ("decode", k_decode)] + (
        [("merge_out_proj", k_tail)] if args.tail == "fused" else [("combine", k_merge), ("out_proj", k_proj)])

    def one_step(evs=None):
        if evs is None:
            return step.run(q_c, q_r, stream)
        for i, (_, fn) in enumerate(parts):
            evs[i].record(stream)
            fn()
        evs[len(parts)].record(stream)

    # the step as one CUDA graph (its kernels keep their programmatic dependencies)
    graph, graph_note = None, "not used (--no-graph)"
    if args.graph:
        try:
            graph = step.capture(q_c, q_r)
            graph_note = "captured"
        except Exception as e:  # noqa: BLE001 -- recorded in the JSON line; eager launches are timed instead
            graph_note = f"capture failed, eager launches timed: {e}"[:240]

    def whole_step():
        if graph is not None:
            graph.replay()
        else:
            one_step()

    # warm-up: at least W steps and at least --min-warmup-s seconds of work so clocks settle
    t0 = time.perf_counter()
    n = 0
    while n < args.warmup or time.perf_counter() - t0 < args.min_warmup_s:
        flush.fill_(n & 0xFF)
        whole_step()
        n += 1
        if n % 16 == 0:
            torch.cuda.synchronize(device)
    torch.cuda.synchronize(device)
    if step.device_error() != 0:
        raise RuntimeError(f"device error bits {step.device_error():#x} during warm-up")

    K = args.steps
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    eager_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)] for _ in range(K)]
    dist_barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clocks:
        # the metric: K whole steps (graph replays), nothing recorded between their kernels, so
        # each kernel may start under the previous one's tail (programmatic dependent launch)
        wall0 = time.perf_counter()
        for i in range(K):
            flush.fill_(i & 0xFF)
            step_ev[i][0].record(stream)
            whole_step()
            step_ev[i][1].record(stream)
        torch.cuda.synchronize(device)
        wall = time.perf_counter() - wall0
        dist_barrier(world)
        # the same steps launched eagerly, for comparison
        for i in range(K):
            flush.fill_(i & 0xFF)
            eager_ev[i][0].record(stream)
            one_step()
            eager_ev[i][1].record(stream)
        torch.cuda.synchronize(device)
        dist_barrier(world)
        # the breakdown: K more steps with an event between kernels (events serialise them); the
        # per-kernel times and the decode kernel's roofline come from here
        for i in range(K):
            flush.fill_(i & 0xFF)
            one_step(evs[i])
        torch.cuda.synchronize(device)
    dist_barrier(world)
    err = step.device_error()
    if err != 0:
        raise RuntimeError(f"device error bits {err:#x} in the timed region")

    if graph is not None and getattr(step, "graph_kernel_nodes", None) not in (None, step.launches_per_step):
        raise RuntimeError(f"the step graph holds {step.graph_kernel_nodes} kernels, expected {step.launches_per_step}")
    step_ms = [e[0].elapsed_time(e[1]) for e in step_ev]
    eager_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in eager_ev)
    k_ms = {name: [e[i].elapsed_time(e[i + 1]) for e in evs]
            for i, (name, _) in enumerate(parts)}
    ms = statistics.mean(step_ms)
    ms_max = dist_max(ms, world, device)
    decode_ms = statistics.mean(k_ms["decode"])

    # sampled parity against the oracle at full size (three heads of every sequence)
    parity = None
    if args.parity and rank == 0:
        parity = sampled_parity(inp, step.out)

    e2e = run_e2e(args, inp, step, binding, device, stream) if args.e2e else None

    bw = peaks.get("hbm_gbs")
    tf = peaks.get("bf16_tflops")
    achieved_gbs = acc["decode_bytes"] / (decode_ms * 1e-3) / 1e9
    achieved_tfs = acc["decode_flop"] / (decode_ms * 1e-3) / 1e12
    kernel_name = "decode_bf16_kernel" if inp.kv_dtype == "bf16" else "decode_fp8_kernel"
    traffic = recorded_traffic(kernel_name, args.workload, acc["tokens"])
    # the decode kernel's bound: whichever of its bytes and its (bf16 tensor-core) FLOPs takes
    # longer at the measured peaks
    if acc["decode_flop"] / (tf * 1e12) > acc["decode_bytes"] / (bw * 1e9):
        roofline = {"bound": "tensor", "kernel": kernel_name, "achieved": round(achieved_tfs, 1), "peak": tf,
                    "unit": "TFLOP/s", "frac": round(achieved_tfs / tf, 4),
                    "traffic": None if traffic is None else int(traffic),
                    "algorithmic_flop": acc["decode_flop"], "algorithmic_bytes": acc["decode_bytes"],
                    "peak_source": peaks.get("source"), "hbm_frac": round(achieved_gbs / bw, 4)}
    else:
        roofline = {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved_gbs, 1), "peak": bw,
                    "unit": "GB/s", "frac": round(achieved_gbs / bw, 4),
                    "traffic": None if traffic is None else int(traffic),
                    "algorithmic_bytes": acc["decode_bytes"], "peak_source": peaks.get("source"),
                    "tensor_frac": round(achieved_tfs / tf, 4)}
    # the same fractions against GB300's nominal figures: HBM3e 8 TB/s, dense BF16 2.25 PFLOP/s
    # (without 2:4 sparsity)
    nom_bw, nom_tf = 8000.0, 2250.0
    nominal = {"hbm_gbs": nom_bw, "bf16_tflops": nom_tf, "source": "GB300 nominal (HBM3e 8 TB/s, dense BF16)",
               "decode_hbm_frac": round(achieved_gbs / nom_bw, 4), "decode_tensor_frac": round(achieved_tfs / nom_tf, 4),
               "step_frac": round(max(acc["step_bytes"] / (nom_bw * 1e9), acc["step_flop"] / (nom_tf * 1e12)) * 1e6
                                  / (ms_max * 1e3), 4)}
    step_roof_us = max(acc["step_bytes"] / (bw * 1e9), acc["step_flop"] / (tf * 1e12)) * 1e6
    decode_roof_us = max(acc["decode_bytes"] / (bw * 1e9), acc["decode_flop"] / (tf * 1e12)) * 1e6
    res = {
        "metric": METRIC,
        "value": round(ms_max * 1e3, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if inp.kv_dtype == "bf16" else "fp8_e4m3+bf16",
        "data": "synthetic (seeded N(0,1) cache/queries, N(0,1/512) weights)",
        "config": bench_config(args, inp, world),
        "setup": {"l2": "512 MB buffer rewritten before every timed step; cache (1.2 GB) > L2",
                   "timing": "value: K replays of the step's CUDA graph, each between two events; "
                             "step_us_eager: K eager launches of the same step; kernels_us and roofline: a third "
                             "pass of K steps with the absorb as a kernel of its own and an event between kernels",
                   "graph": graph_note,
                   "plan": {"clusters": step.info.num_clusters, "items": step.info.num_items,
                            "combine_seqs": step.info.num_combine, "max_splits": step.info.max_splits,
                            "item_cost_pages": args.item_cost_pages},
                   "absorb": args.absorb, "tail": args.tail},
        "step_us_eager": round(eager_ms * 1e3, 2),
        "kernels_us": {k: round(statistics.mean(v) * 1e3, 2) for k, v in k_ms.items()},
        "kv_tbps": round(acc["kv_bytes"] / (ms_max * 1e-3) / 1e12, 3),
        "step_tflops": round(acc["step_flop"] / (ms_max * 1e-3) / 1e12, 1),
        "decode_tflops": round(acc["decode_flop"] / (decode_ms * 1e-3) / 1e12, 1),
        "roofline": roofline,
        "step_roofline_frac": round(step_roof_us / (ms_max * 1e3), 4),
        "decode_roofline_frac": round(decode_roof_us / (decode_ms * 1e3), 4),
        "clocks": clocks.summary(),
        "wall_s_timed": round(wall, 4),
        "gpu_launches": K * (step.graph_kernel_nodes if graph is not None and
                             getattr(step, "graph_kernel_nodes", None) else step.launches_per_step),
        "gpu_launches_source": ("kernel nodes of the captured step graph"
                                if graph is not None and getattr(step, "graph_kernel_nodes", None)
                                else "launches per step as issued"),
        "roofline_nominal": nominal,
        "e2e": e2e,
        "parity": parity,
    }
    if rank == 0 and args.cpu_baseline and world >= 1:
        res["cpu_baseline"] = cpu_baseline(inp)
    return res


def sampled_parity(inp, out_dev):
    import oracle
    from mla_latent_kv_absorb_gb300 import binding

    heads = [0, 77, 127]
    if inp.queries_per_seq > 1:
        inp = oracle.query_row_inputs(inp, inp.queries_per_seq)  # one decode query per row
    q_abs = oracle.absorb_q(inp.q_c, inp.w_uk)
    o, _ = oracle.latent_attention(inp, q_abs, softmax_scale=binding.SOFTMAX_SCALE, heads=heads)
    full = np.zeros((inp.batch, 128, 512))
    full[:, heads, :] = o
    ref = oracle.out_proj(full, inp.w_uv)[:, heads, :]
    got = out_dev[:, heads, :].double().cpu().numpy()
    d = got - ref
    tol = {"max_abs": 2e-2, "rel_l2": 1e-2} if inp.kv_dtype == "bf16" else {"max_abs": 5e-2, "rel_l2": 5e-2}
    max_abs, rel = float(np.abs(d).max()), float(np.linalg.norm(d) / np.linalg.norm(ref))
    return {"heads": heads, "max_abs": max_abs, "rel_l2": rel, "tol": tol,
            "ok": bool(np.isfinite(got).all() and max_abs <= tol["max_abs"] and rel <= tol["rel_l2"])}


def run_e2e(args, inp, step, binding, device, stream):
    """Through the public API with pinned host buffers (DecodeStep.run_host): the first call plans
    and captures the step (mla_step_graph_create, warm-up); every timed call launches it
    (mla_step_graph_run), which copies block table and queries from the pinned tensors, runs the
    kernels, copies the output back and waits for it."""
    q_c_h = inp.q_c.pin_memory()
    q_r_h = inp.q_r.pin_memory()
    bt_h = torch.from_numpy(np.ascontiguousarray(inp.block_table)).pin_memory()
    out_h = torch.empty(tuple(step.out.shape), dtype=step.out.dtype).pin_memory()
    times = []
    for i in range(args.warmup + args.steps):
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        step.run_host(q_c_h, q_r_h, block_table=bt_h, seq_lens=inp.seq_lens, out=out_h, stream=stream)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    h2d = bt_h.numel() * 4 + q_c_h.numel() * 2 + q_r_h.numel() * 2
    d2h = out_h.numel() * 2
    return {"value": round(statistics.mean(times) * 1e6, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "path": "captured" if step._host_graph is not None else "one call per step",
            "plan_bytes_at_capture": int(step.info.plan_bytes)}


# ----------------------------------------------------------------------------- the CPU oracle

def _one_sequence(inp, tokens=None):
    q = inp.queries_per_seq
    keep = min(q, 16)  # a long chunk is sampled by its last 16 query rows (same visible lengths)
    sub = synth.DecodeInputs(seq_lens=inp.seq_lens[:1].copy(), block_table=inp.block_table[:1].copy(),
                             num_pool_pages=inp.num_pool_pages, q_c=inp.q_c[q - keep:q], q_r=inp.q_r[q - keep:q],
                             w_uk=inp.w_uk, w_uv=inp.w_uv, kv_dtype=inp.kv_dtype, pool=inp.pool, c8=inp.c8,
                             kv_scale=inp.kv_scale, kr=inp.kr, queries_per_seq=keep)
    q = keep
    if tokens is not None:
        sub.seq_lens[0] = max(q, min(int(sub.seq_lens[0]), tokens))
    return sub


def _rows_note(sub) -> str:
    return f", {sub.queries_per_seq} query rows" if sub.queries_per_seq > 1 else ""


def _query_rows(sub):
    """The sample as ordinary decode queries (one per query row) for the oracle."""
    import oracle
    return oracle.query_row_inputs(sub, sub.queries_per_seq) if sub.queries_per_seq > 1 else sub


def cpu_baseline(inp, tokens=None):
    """The CPU oracle on the host cores, on a bounded sample of the workload, scaled to a full
    step (the oracle's work is linear in tokens x heads): the naive oracle (decompress k and v
    per head) on sequence 0 x 16 heads, and the absorbed oracle on sequence 0 x all heads."""
    import oracle
    from mla_latent_kv_absorb_gb300.binding import SOFTMAX_SCALE

    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    heads = list(range(0, 128, 8))
    sub = _one_sequence(inp, tokens)
    S0 = int(sub.seq_lens[0])
    rows = _query_rows(sub)
    seen = visible_tokens(sub.seq_lens, sub.queries_per_seq)
    t0 = time.perf_counter()
    oracle.decode_naive(rows, softmax_scale=SOFTMAX_SCALE, heads=heads)
    dt_naive = time.perf_counter() - t0
    t0 = time.perf_counter()
    q_abs = oracle.absorb_q(rows.q_c, rows.w_uk)
    o, _ = oracle.latent_attention(rows, q_abs, softmax_scale=SOFTMAX_SCALE)
    oracle.out_proj(o, rows.w_uv)
    dt_abs = time.perf_counter() - t0
    total_seen = visible_tokens(inp.seq_lens, inp.queries_per_seq)
    scale_naive = (total_seen * 128) / (seen * len(heads))
    scale_abs = total_seen / seen
    return {"value": round(dt_naive * scale_naive * 1e6, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"naive fp64 oracle, sequence 0 ({S0} tokens{_rows_note(sub)}) x heads 0,8,..,120; "
                      f"{dt_naive:.2f} s measured, "
                      f"scaled x{scale_naive:.0f} to the full step",
            "absorbed": {"value": round(dt_abs * scale_abs * 1e6, 1), "unit": UNIT,
                         "sample": f"absorbed fp64 oracle (absorb, latent attention, W_UV) on sequence 0 "
                                   f"({S0} tokens{_rows_note(sub)}) x all heads; {dt_abs:.2f} s measured, "
                                   f"scaled x{scale_abs:.0f}"}}


def run_reference(args, rank, world, local):
    """The CPU oracle as the reference arm, rank 0 only.  Each step runs the naive oracle on a
    bounded sample of the workload (sequence 0, 8,192 tokens, 16 of the 128 heads); the line's
    value is the measured time of that step, and the full-step time it implies is given beside it."""
    if rank != 0:
        return None
    import oracle
    from mla_latent_kv_absorb_gb300.binding import SOFTMAX_SCALE

    inp = synth.make_workload(args.workload, poison_tail=False)
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    heads = list(range(0, 128, 8))
    sub = _one_sequence(inp, 8192)
    rows = _query_rows(sub)
    per_step = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.decode_naive(rows, softmax_scale=SOFTMAX_SCALE, heads=heads)
        if i >= args.warmup:
            per_step.append(time.perf_counter() - t0)
    v = statistics.mean(per_step) * 1e6
    scale = (visible_tokens(inp.seq_lens, inp.queries_per_seq) * 128) / (
        visible_tokens(sub.seq_lens, sub.queries_per_seq) * len(heads))
    sample = (f"naive fp64 oracle per step on sequence 0 ({int(sub.seq_lens[0])} tokens{_rows_note(sub)}) "
              f"x heads 0,8,..,120 "
              f"(1/{scale:.0f} of the workload)")
    cb = {"value": round(v, 1), "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
          "sample": sample, "full_step_estimate_us": round(v * scale, 1)}
    return {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (the same seeded workload)",
            "config": bench_config(args, inp, world), "cpu_baseline": cb,
            "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- prefill chunk

def prefill_accounting(S: int, T: int, row_bytes: int):
    """Algorithmic FLOPs and bytes of one decompressed prefill chunk: key and value
    decompression of all S tokens for 128 heads, causal attention of the T new tokens (head
    dim 192 for scores, 128 for values); bytes = the cache rows, both weights, queries, output."""
    seen = visible_tokens([S], T)
    flop = 2 * (2 * S * 512 * 128 * 128) + seen * 128 * 2 * (192 + 128)
    nbytes = S * row_bytes + 2 * (128 * 128 * 512 * 2) + T * 128 * 192 * 2 + T * 128 * 128 * 2
    return dict(flop=flop, bytes=nbytes, seen=seen)


def run_prefill(args, rank, world, local):
    """A chunk of new tokens at the end of one sequence through the decompressed form
    (mla_prefill_decompressed: gather, key and value decompression, causal attention)."""
    from mla_latent_kv_absorb_gb300 import binding

    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    binding.lib()
    inp = synth.make_workload(args.workload, seed=synth.DEFAULT_SEED + rank, poison_tail=False)
    S, T = int(inp.seq_lens[0]), inp.queries_per_seq
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, device)
    pool = kv.pop("kv_pool")
    ws = torch.empty(int(binding.lib().mla_prefill_workspace_bytes(S)), dtype=torch.uint8, device=device)
    out = torch.empty(T, 128, 128, dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)

    def step(qc=q_c, qr=q_r):
        binding.mla_prefill_decompressed(kv_pool=pool, block_table_row=bt[0], seq_len=S, q_c=qc, q_r=qr, w_uk=w_uk,
                                         w_uv=w_uv, out=out, dev_error=err, workspace=ws, stream=stream, **kv)

    t0, n = time.perf_counter(), 0
    while n < args.warmup or time.perf_counter() - t0 < args.min_warmup_s:
        flush.fill_(n & 0xFF)
        step()
        n += 1
    torch.cuda.synchronize(device)
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    dist_barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clocks:
        for i in range(K):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize(device)
    dist_barrier(world)
    if binding.mla_read_device_error(err) != 0:
        raise RuntimeError("device error in the timed region")
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms_max = dist_max(ms, world, device)
    row_bytes = 1152 if inp.kv_dtype == "bf16" else (644 if inp.kv_dtype == "fp8_e4m3" else 420)
    acc = prefill_accounting(S, T, row_bytes)
    peaks = load_peaks()
    tf, bw = peaks.get("bf16_tflops"), peaks.get("hbm_gbs")
    achieved_tf = acc["flop"] / (ms_max * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "whole chunk (gather, 2 decompression GEMMs, attention)",
                "achieved": round(achieved_tf, 1), "peak": tf, "unit": "TFLOP/s", "frac": round(achieved_tf / tf, 4),
                "traffic": None, "algorithmic_flop": acc["flop"], "algorithmic_bytes": acc["bytes"],
                "peak_source": peaks.get("source"),
                "hbm_frac": round(acc["bytes"] / (ms_max * 1e-3) / 1e9 / bw, 4)}
    if acc["bytes"] / (bw * 1e9) > acc["flop"] / (tf * 1e12):
        roofline["bound"] = "hbm"

    # sampled parity: query rows first, middle, last x three heads against the oracle
    parity = None
    if args.parity and rank == 0:
        import dataclasses

        import oracle
        rows = oracle.query_row_inputs(inp, T)
        idx = np.array([0, T // 2, T - 1])
        sub = dataclasses.replace(rows, seq_lens=rows.seq_lens[idx].copy(),
                                  block_table=np.ascontiguousarray(rows.block_table[idx]),
                                  q_c=rows.q_c[idx], q_r=rows.q_r[idx], queries_per_seq=1)
        heads = [0, 77, 127]
        ref = oracle.decode_naive(sub, softmax_scale=binding.SOFTMAX_SCALE, heads=heads)
        got = out[torch.from_numpy(idx).to(device)][:, heads, :].double().cpu().numpy()
        d = got - ref
        tol = {"max_abs": 2e-2, "rel_l2": 1e-2}
        max_abs, rel = float(np.abs(d).max()), float(np.linalg.norm(d) / np.linalg.norm(ref))
        parity = {"rows": idx.tolist(), "heads": heads, "max_abs": max_abs, "rel_l2": rel, "tol": tol,
                  "ok": bool(np.isfinite(got).all() and max_abs <= tol["max_abs"] and rel <= tol["rel_l2"])}

    # e2e: queries from pinned host memory, the chunk, the output back, wall clock
    e2e = None
    if args.e2e:
        q_c_h, q_r_h = inp.q_c.pin_memory(), inp.q_r.pin_memory()
        out_h = torch.empty(T, 128, 128, dtype=torch.bfloat16).pin_memory()
        times = []
        for i in range(args.warmup + K):
            torch.cuda.synchronize(device)
            t0 = time.perf_counter()
            q_c.copy_(q_c_h, non_blocking=True)
            q_r.copy_(q_r_h, non_blocking=True)
            step()
            out_h.copy_(out, non_blocking=True)
            torch.cuda.synchronize(device)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        e2e = {"value": round(statistics.mean(times) * 1e6, 2), "unit": UNIT,
               "h2d_bytes_per_step": int(q_c_h.numel() * 2 + q_r_h.numel() * 2),
               "d2h_bytes_per_step": int(out_h.numel() * 2)}

    cb = None
    if args.cpu_baseline and rank == 0:
        import oracle
        cores = len(os.sched_getaffinity(0))
        oracle.set_threads(cores)
        sub = _one_sequence(inp)
        heads = list(range(0, 128, 8))
        t0 = time.perf_counter()
        oracle.decode_naive(_query_rows(sub), softmax_scale=binding.SOFTMAX_SCALE, heads=heads)
        dt = time.perf_counter() - t0
        scale = (acc["seen"] * 128) / (visible_tokens(sub.seq_lens, sub.queries_per_seq) * len(heads))
        cb = {"value": round(dt * scale * 1e6, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
              "cpu_model": cpu_model(),
              "sample": f"naive fp64 oracle on the chunk's last {sub.queries_per_seq} query rows x heads 0,8,..,120; "
                        f"{dt:.2f} s measured, scaled x{scale:.0f} to the chunk"}

    return {"metric": "MLA prefill chunk us/chunk (decompressed form), TFLOP/s as fraction of GB300 roofline",
            "value": round(ms_max * 1e3, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(ms_max, 5), "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) cache/queries, N(0,1/512) weights)",
            "config": bench_config(args, inp, world),
            "setup": {"l2": "512 MB buffer rewritten before every timed chunk",
                      "timing": "CUDA events around each mla_prefill_decompressed call"},
            "chunk_tflops": round(achieved_tf, 1), "roofline": roofline, "clocks": clocks.summary(),
            "gpu_launches": 4 * K, "gpu_launches_source": "gather, two decompression GEMMs, attention per chunk",
            "e2e": e2e, "parity": parity, "cpu_baseline": cb}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default="b16_s65536")
    ap.add_argument("--min-warmup-s", type=float, default=0.5,
                    help="keep warming up for at least this long (0: exactly --warmup steps, for profilers)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-parity", dest="parity", action="store_false")
    ap.add_argument("--item-cost-pages", type=int, default=0,
                    help="planner: charge in pages per extra item of a CTA pair (0: the library's default of 7; "
                         "negative: equal page runs)")
    ap.add_argument("--absorb", choices=["fused", "separate"], default="separate",
                    help="absorb as the decode kernel's prologue, or as a kernel of its own before it")
    ap.add_argument("--tail", choices=["fused", "separate"], default="separate",
                    help="split merge and W_UV projection in one kernel, or as two kernels")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time eager launches for the value instead of replays of the step's CUDA graph")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, rank, world, local)
    elif synth.WORKLOADS[args.workload].get("prefill"):
        res = run_prefill(args, rank, world, local)
    else:
        res = run_ours(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
