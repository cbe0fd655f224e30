"""GPU parity of the absorb run as the decode kernel's prologue (mla_absorb_decode_paged).

Each case runs the fused call and the two separate calls (mla_absorb_q, then mla_decode_paged)
on the same seeded inputs: q_abs, o_lat, lse and the split partials must agree bit for bit
(the prologue issues the absorb's MMAs in the same order), the job counter must be back at zero
after every call, and the result must match the oracle within the bf16 tolerance.
"""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
from parity_util import SCALE, TOL_BF16, assert_close, bf16_round  # noqa: E402

from mla_latent_kv_absorb_gb300 import binding, synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _buffers(B, info):
    return dict(o_lat=torch.full((B, 128, 512), float("nan"), dtype=torch.bfloat16, device=DEV),
                lse=torch.full((B, 128), float("nan"), dtype=torch.float32, device=DEV),
                dev_error=torch.zeros(1, dtype=torch.int32, device=DEV),
                workspace=torch.zeros(max(info.workspace_bytes // 4, 4), dtype=torch.float32, device=DEV))


def _run_both(inp, min_pages, repeats=1):
    q_c, q_r, w_uk, _, kv, bt = binding.inputs_to_device(inp, DEV)
    plan, info = binding.mla_plan_splits(inp.seq_lens, binding.num_sms(), min_pages_per_split=min_pages)
    plan_dev = torch.from_numpy(plan).to(DEV)
    B = inp.batch
    # separate kernels
    ref = _buffers(B, info)
    q_abs_ref = torch.empty(B, 128, 512, dtype=torch.bfloat16, device=DEV)
    binding.mla_absorb_q(q_c, w_uk, q_abs_ref)
    binding.mla_decode_paged(info, plan_dev, q_abs_ref, q_r, block_table=bt, **ref, **kv)
    # fused, `repeats` calls in a row on the same counter
    sync = torch.zeros(2, dtype=torch.int32, device=DEV)
    outs = []
    for _ in range(repeats):
        got = _buffers(B, info)
        q_abs = torch.full((B, 128, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
        binding.mla_absorb_decode_paged(info, plan_dev, q_c, w_uk, q_abs, sync, q_r, block_table=bt, **got, **kv)
        torch.cuda.synchronize()
        assert binding.mla_read_device_error(got["dev_error"]) == 0
        assert torch.equal(sync.cpu(), torch.zeros(2, dtype=torch.int32)), "job counter not reset"
        outs.append((q_abs, got))
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(ref["dev_error"]) == 0
    return info, q_abs_ref, ref, outs


@pytest.mark.parametrize("lens,min_pages", [
    ([700, 65], 10 ** 6),                  # two pairs in the plan: the other pairs only run absorb jobs
    ([3000, 700, 64 * 9 + 1], 2),          # split sequences
    ([300] * 130, 2),                      # 130 sequences: two row tiles, 256 absorb jobs
    ([4096] * 16, 0),                      # the B=16, S=4096 shape, default plan
])
def test_fused_absorb_matches_separate_kernels(lens, min_pages):
    inp = synth.make_inputs(lens, seed=800 + len(lens), poison_tail=True)
    info, q_abs_ref, ref, outs = _run_both(inp, min_pages)
    q_abs, got = outs[0]
    assert torch.equal(q_abs, q_abs_ref), "q_abs differs from mla_absorb_q"
    assert torch.equal(got["o_lat"].isnan(), ref["o_lat"].isnan())
    single = ~ref["o_lat"].isnan().any(dim=2).any(dim=1)  # sequences written by the decode itself
    assert torch.equal(got["o_lat"][single], ref["o_lat"][single]) and torch.equal(got["lse"][single], ref["lse"][single])
    n = int(info.num_partials)
    if n:
        assert torch.equal(got["workspace"][: n * (128 * 512 + 128)], ref["workspace"][: n * (128 * 512 + 128)])
    # and against the oracle, after the merge
    q_abs_oracle = oracle.absorb_q(inp.q_c, inp.w_uk)
    assert_close(q_abs, q_abs_oracle, TOL_BF16, "q_abs")
    if info.num_combine:
        plan, _ = binding.mla_plan_splits(inp.seq_lens, binding.num_sms(), min_pages_per_split=min_pages)
        plan_dev = torch.from_numpy(plan).to(DEV)
        binding.mla_combine_splits(info, plan_dev, got["workspace"], got["o_lat"], got["lse"])
        torch.cuda.synchronize()
    heads = list(range(0, 128, 16)) if inp.num_tokens > 20000 else None
    ref_o, ref_l = oracle.latent_attention(inp, bf16_round(q_abs_oracle).double().numpy(), softmax_scale=SCALE,
                                           heads=heads)
    hs = list(range(128)) if heads is None else heads
    assert_close(got["o_lat"][:, hs, :], ref_o, TOL_BF16, "o_lat")
    assert_close(got["lse"][:, hs], ref_l, TOL_BF16, "lse")


def test_fused_absorb_three_calls_in_a_row():
    """The counter the score CTAs wait on is zeroed by each call, so calls in a row agree."""
    inp = synth.make_inputs([2000, 64 * 5 + 3, 129], seed=811, poison_tail=True)
    _, q_abs_ref, ref, outs = _run_both(inp, 2, repeats=3)
    for q_abs, got in outs:
        assert torch.equal(q_abs, q_abs_ref)
        assert torch.equal(got["workspace"], outs[0][1]["workspace"])


def test_fused_absorb_fp8_cache_runs_two_kernels():
    """With the e4m3 cache the absorb runs as its own kernel inside the call: same results as the
    separate calls, counter untouched."""
    inp = synth.make_inputs([1500, 64 * 3 + 1], seed=812, poison_tail=True, kv_dtype="fp8_e4m3")
    _, q_abs_ref, ref, outs = _run_both(inp, 2)
    q_abs, got = outs[0]
    assert torch.equal(q_abs, q_abs_ref)
    assert torch.equal(got["workspace"], ref["workspace"])
