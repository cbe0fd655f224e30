"""GPU parity: every kernel of the decode step, through the C ABI, against the CPU oracle.

All inputs come from the seeded generator; every expected value comes from ``oracle/``.
Tails of last pages are NaN-poisoned, so a kernel that reads past S_b fails.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
from parity_util import SCALE, TOL_BF16, assert_close, bf16_round  # noqa: E402

from mla_latent_kv_absorb_gb300 import binding, synth  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _sync_err(step_or_err):
    torch.cuda.synchronize()
    bits = binding.mla_read_device_error(step_or_err)
    assert bits == 0, f"device error bits {bits:#x}"


# ------------------------------------------------------------------------------------ absorb

@pytest.mark.parametrize("batch", [1, 16, 17, 128, 130, 256, 257])
def test_absorb_q(batch):
    inp = synth.make_inputs([1] * batch, seed=100 + batch)
    q_abs = torch.empty(batch, 128, 512, dtype=torch.bfloat16, device=DEV)
    binding.mla_absorb_q(inp.q_c.to(DEV), inp.w_uk.to(DEV), q_abs)
    torch.cuda.synchronize()
    ref = oracle.absorb_q(inp.q_c, inp.w_uk)
    assert_close(q_abs, ref, TOL_BF16, f"q_abs B={batch}")


# ------------------------------------------------------------------------------------ out-proj

@pytest.mark.parametrize("batch", [1, 16, 33, 129, 256, 300])
def test_out_proj(batch):
    inp = synth.make_inputs([1] * batch, seed=200 + batch)
    g = torch.Generator().manual_seed(batch)
    o_lat = (torch.randn(batch, 128, 512, generator=g) * 0.05).to(torch.bfloat16)
    out = torch.empty(batch, 128, 128, dtype=torch.bfloat16, device=DEV)
    binding.mla_out_proj(o_lat.to(DEV), inp.w_uv.to(DEV), out)
    torch.cuda.synchronize()
    ref = oracle.out_proj(o_lat.double().numpy(), inp.w_uv)
    assert_close(out, ref, TOL_BF16, f"out B={batch}")


# ------------------------------------------------------------------------------------ decode kernel alone

def _decode_only(inp, *, min_pages=0, max_clusters=0, item_cost=0):
    """Run mla_decode_paged (+ merge) on bf16-rounded oracle q_abs; return (o_lat, lse, info, q_abs_bf16)."""
    q_abs_bf16 = bf16_round(oracle.absorb_q(inp.q_c, inp.w_uk))
    _, q_r, _, _, kv, bt = binding.inputs_to_device(inp, DEV)
    plan, info = binding.mla_plan_splits(inp.seq_lens, binding.num_sms(), min_pages_per_split=min_pages,
                                         max_clusters=max_clusters, item_cost_pages=item_cost)
    plan_dev = torch.from_numpy(plan).to(DEV)
    B = inp.batch
    o_lat = torch.full((B, 128, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, 128), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(info.workspace_bytes // 4, 4), dtype=torch.float32, device=DEV)
    binding.mla_decode_paged(info, plan_dev, q_abs_bf16.to(DEV), q_r, block_table=bt, o_lat=o_lat, lse=lse,
                             dev_error=err, workspace=ws, **kv)
    binding.mla_combine_splits(info, plan_dev, ws, o_lat, lse)
    _sync_err(err)
    return o_lat, lse, info, q_abs_bf16


def _check_latent(inp, o_lat, lse, q_abs_bf16, heads=None):
    ref_o, ref_l = oracle.latent_attention(inp, q_abs_bf16.double().numpy(), softmax_scale=SCALE, heads=heads)
    hs = slice(None) if heads is None else list(heads)
    assert_close(o_lat[:, hs] if heads is None else o_lat[:, hs, :], ref_o, TOL_BF16, "o_lat")
    assert_close(lse[:, hs] if heads is None else lse[:, hs], ref_l, TOL_BF16, "lse")


@pytest.mark.parametrize("lens", [[1], [64], [65], [700], [100, 37, 64 * 5], [129, 1, 2000, 63]])
def test_decode_single_item(lens):
    """One item per sequence (no merge): the decode kernel's own o_lat and lse."""
    inp = synth.make_inputs(lens, seed=300 + len(lens), poison_tail=True)
    o_lat, lse, info, q = _decode_only(inp, min_pages=10 ** 6)
    assert info.num_combine == 0
    _check_latent(inp, o_lat, lse, q)


@pytest.mark.parametrize("lens,min_pages", [([4000], 1), ([64 * 40 + 5, 1, 9000], 2), ([3000] * 8, 4),
                                            ([100] * 200, 1)])
def test_decode_split_and_merge(lens, min_pages):
    """Sequences cut into several items: partials + the log-sum-exp merge kernel."""
    inp = synth.make_inputs(lens, seed=400 + len(lens), poison_tail=True)
    o_lat, lse, info, q = _decode_only(inp, min_pages=min_pages)
    assert info.num_combine > 0 or len(lens) > 76
    _check_latent(inp, o_lat, lse, q)


def test_decode_few_clusters_many_items():
    """Two CTA pairs walk many items each (item boundaries inside the pipelines)."""
    lens = [70, 1, 640, 129, 3, 64, 2000, 65]
    inp = synth.make_inputs(lens, seed=501, poison_tail=True)
    o_lat, lse, info, q = _decode_only(inp, min_pages=1, max_clusters=2)
    assert info.num_clusters == 2 and info.num_items >= len(lens)
    _check_latent(inp, o_lat, lse, q)


@pytest.mark.parametrize("item_cost", [7, 50])
def test_decode_cost_balanced_plan(item_cost):
    """Plans cut with a per-item charge (pairs holding several items get fewer pages, and the
    packing may leave pairs unused) decode to the oracle's result as equal-run plans do."""
    lens = [64 * 40 + 5, 1, 9000, 300, 64 * 20, 4000]
    inp = synth.make_inputs(lens, seed=503 + item_cost, poison_tail=True)
    o_lat, lse, info, q = _decode_only(inp, min_pages=2, item_cost=item_cost)
    assert info.num_combine > 0
    _check_latent(inp, o_lat, lse, q)


def test_decode_large_scores_rescale():
    """Scores whose running max climbs page after page (cache rows scaled from 0.1 up to 1.0
    and queries scaled by 6): the lazy-rescale path of the online softmax runs several times.
    Cache values stay O(1) so the absolute tolerance keeps its meaning."""
    inp = synth.make_inputs([64 * 30 + 7, 900], seed=502, poison_tail=True)
    g = torch.Generator().manual_seed(5)
    inp.q_c = (inp.q_c.float() * 6.0).to(torch.bfloat16)
    inp.q_r = (torch.randn(2, 128, 64, generator=g) * 6.0).to(torch.bfloat16)
    pool = inp.pool.float()
    for b in range(2):
        n = (int(inp.seq_lens[b]) + 63) // 64
        for j in range(n):
            pool[int(inp.block_table[b, j])] *= 0.1 + 0.9 * j / max(n - 1, 1)
    inp.pool = pool.to(torch.bfloat16)
    o_lat, lse, info, q = _decode_only(inp, min_pages=10 ** 6)
    _check_latent(inp, o_lat, lse, q)


# ------------------------------------------------------------------------------------ end to end

def _run_step(inp, **kw):
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, **kv, **kw)
    out = step.run(q_c, q_r)
    torch.cuda.synchronize()
    assert step.device_error() == 0
    return out, step


def test_end_to_end_b1_s2048_naive():
    """B=1, S=2048, identity block table: the whole step against the naive (decompressed) oracle."""
    inp = synth.make_workload("b1_s2048", poison_tail=True)
    out, step = _run_step(inp)
    ref = oracle.decode_naive(inp, softmax_scale=SCALE)
    assert_close(out, ref, TOL_BF16, "out vs naive oracle")


def test_end_to_end_b16_s4096():
    """B=16, S=4096, shuffled pool: absorbed oracle on all heads, naive oracle on three heads."""
    inp = synth.make_workload("b16_s4096", poison_tail=True)
    out, step = _run_step(inp)
    _, _, _, ref = oracle.decode_absorbed(inp, softmax_scale=SCALE)
    assert_close(out, ref, TOL_BF16, "out vs absorbed oracle")
    heads = [0, 61, 127]
    ref_n = oracle.decode_naive(inp, softmax_scale=SCALE, heads=heads)
    assert_close(out[:, heads, :], ref_n, TOL_BF16, "out vs naive oracle (3 heads)")


def test_end_to_end_ragged_b64():
    """B=64 ragged lengths in [128, 32768] (seed 42): split planning and merge at full size;
    the oracle computes every 8th head."""
    inp = synth.make_workload("b64_ragged", poison_tail=True)
    out, step = _run_step(inp)
    assert step.info.num_combine > 0
    heads = list(range(0, 128, 8))
    q_abs = oracle.absorb_q(inp.q_c, inp.w_uk)
    o, _ = oracle.latent_attention(inp, q_abs, softmax_scale=SCALE, heads=heads)
    full = np.zeros((inp.batch, 128, 512))
    full[:, heads, :] = o
    ref = oracle.out_proj(full, inp.w_uv)[:, heads, :]
    assert_close(out[:, heads, :], ref, TOL_BF16, "out (every 8th head)")


def test_end_to_end_b16_s65536_sampled():
    """B=16, S=65536 (1.2 GB cache): the launch configuration the bench times; the oracle
    computes three heads of every sequence."""
    inp = synth.make_workload("b16_s65536", poison_tail=False)
    out, step = _run_step(inp)
    assert step.info.num_clusters == binding.num_sms() // 2
    heads = [0, 77, 127]
    q_abs = oracle.absorb_q(inp.q_c, inp.w_uk)
    o, _ = oracle.latent_attention(inp, q_abs, softmax_scale=SCALE, heads=heads)
    full = np.zeros((inp.batch, 128, 512))
    full[:, heads, :] = o
    ref = oracle.out_proj(full, inp.w_uv)[:, heads, :]
    assert_close(out[:, heads, :], ref, TOL_BF16, "out (3 heads)")


def test_end_to_end_one_sequence_of_a_million_tokens():
    """The longest case: one sequence of 1,048,575 tokens (16,384 pages, the last one short by a
    token, NaN-poisoned past its end), so every CTA pair scans a piece of it and the merge
    combines more partials than one warp has lanes; the oracle computes three heads."""
    inp = synth.make_inputs([1048575], seed=77, poison_tail=True)
    out, step = _run_step(inp)
    assert step.info.num_combine == 1 and step.info.max_splits == binding.num_sms() // 2 > 32
    heads = [0, 64, 127]
    q_abs = oracle.absorb_q(inp.q_c, inp.w_uk)
    o, _ = oracle.latent_attention(inp, q_abs, softmax_scale=SCALE, heads=heads)
    full = np.zeros((inp.batch, 128, 512))
    full[:, heads, :] = o
    ref = oracle.out_proj(full, inp.w_uv)[:, heads, :]
    assert_close(out[:, heads, :], ref, TOL_BF16, "out (3 heads, 1M tokens)")


def test_step_is_deterministic():
    inp = synth.make_inputs([5000, 300, 64], seed=7, poison_tail=True)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
    a = step.run(q_c, q_r).clone()
    b = step.run(q_c, q_r).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_run_host_matches_device_run():
    """DecodeStep.run_host (host tensors in, one staged upload, re-plan) gives the same bits as
    run() on device tensors, twice in a row."""
    inp = synth.make_inputs([3000, 700, 64 * 9 + 1], seed=11, poison_tail=True)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
    ref = step.run(q_c, q_r).clone()
    torch.cuda.synchronize()
    bt_h = torch.from_numpy(np.ascontiguousarray(inp.block_table))
    for _ in range(2):
        out = step.run_host(inp.q_c, inp.q_r, block_table=bt_h, seq_lens=inp.seq_lens)
        assert step.device_error() == 0
        assert torch.equal(out, ref.cpu())


def test_run_host_new_lengths_and_fp8():
    """run_host re-plans when the lengths change (same batch, same buffers) and gives the bits of
    a DecodeStep built for the new lengths; the same holds for an FP8 cache."""
    for kv_dtype in ("bf16", "fp8_e4m3"):
        inp = synth.make_inputs([3000, 700, 64 * 9 + 1], seed=12, poison_tail=False, kv_dtype=kv_dtype)
        q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
        step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
        short = np.array([1800, 65, 64 * 9 + 1], dtype=np.int32)
        fresh = binding.DecodeStep(short, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
        ref = fresh.run(q_c, q_r).clone()
        torch.cuda.synchronize()
        out = step.run_host(inp.q_c.pin_memory(), inp.q_r.pin_memory(), seq_lens=short)
        assert step.device_error() == 0
        assert torch.equal(out, ref.cpu()), kv_dtype


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_graph_replay_matches_eager(kv_dtype):
    """DecodeStep.capture: replaying the step's CUDA graph gives the bits of an eager step on
    the same queries, also for queries copied into the captured tensors afterwards."""
    inp = synth.make_inputs([3000, 700, 64 * 9 + 1], seed=13, poison_tail=True, kv_dtype=kv_dtype)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
    assert step.info.num_combine > 0
    graph = step.capture(q_c, q_r)
    g = torch.Generator().manual_seed(5)
    for _ in range(2):
        new_c = torch.randn(tuple(q_c.shape), generator=g).to(torch.bfloat16).to(DEV)
        new_r = torch.randn(tuple(q_r.shape), generator=g).to(torch.bfloat16).to(DEV)
        q_c.copy_(new_c)
        q_r.copy_(new_r)
        graph.replay()
        got = step.out.clone()
        ref = step.run(new_c, new_r).clone()
        torch.cuda.synchronize()
        assert step.device_error() == 0
        assert torch.equal(got, ref)


@pytest.mark.parametrize("fused_absorb,fused_tail,kernels", [(False, False, 4), (True, False, 3), (False, True, 3),
                                                             (True, True, 2)])
def test_step_graph_kernel_count(fused_absorb, fused_tail, kernels):
    """The captured bf16 step holds exactly the kernels the configuration launches: absorb,
    decode, merge, projection, or fewer with the fused calls (counted from the graph's nodes
    through the driver; skipped where torch cannot keep the captured graph for inspection); every
    configuration gives the same output bits."""
    inp = synth.make_inputs([3000, 700], seed=14)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2,
                              fused_absorb=fused_absorb, fused_tail=fused_tail, **kv)
    assert step.info.num_combine > 0
    ref = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
    want = ref.run(q_c, q_r).clone()
    graph = step.capture(q_c, q_r)
    graph.replay()
    torch.cuda.synchronize()
    assert step.device_error() == 0 and torch.equal(step.out, want)
    assert step.launches_per_step == kernels
    if step.graph_kernel_nodes is None:
        pytest.skip("this torch build does not keep the captured graph")
    assert step.graph_kernel_nodes == kernels
