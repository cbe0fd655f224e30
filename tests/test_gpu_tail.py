"""GPU parity of the fused step tail, mla_merge_out_proj (split merge and W_UV projection in one
kernel), through the C ABI.

Each case decodes a seeded workload, then runs the tail two ways on copies of the same decode
output: the separate merge and projection kernels, and the fused kernel.  The fused result
must equal the separate one bit for bit (same merge arithmetic per element, same MMA order),
and both must match the oracle (merged latent output projected through W_UV) within the bf16
tolerance.
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


def _decode(inp, min_pages):
    q_abs = bf16_round(oracle.absorb_q(inp.q_c, inp.w_uk))
    _, q_r, _, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    plan, info = binding.mla_plan_splits(inp.seq_lens, binding.num_sms(), min_pages_per_split=min_pages)
    plan_dev = torch.from_numpy(plan).to(DEV)
    B = inp.batch
    o_lat = torch.full((B, 128, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, 128), float("nan"), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(info.workspace_bytes // 4, 4), dtype=torch.float32, device=DEV)
    binding.mla_decode_paged(info, plan_dev, q_abs.to(DEV), q_r, block_table=bt, o_lat=o_lat, lse=lse,
                             dev_error=err, workspace=ws, **kv)
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(err) == 0
    return info, plan_dev, ws, o_lat, lse, w_uv, q_abs


@pytest.mark.parametrize("lens,min_pages", [
    ([4000], 1),                          # one sequence cut into many items
    ([64 * 40 + 5, 1, 9000, 63], 2),      # split and single-item sequences mixed
    ([300] * 130, 2),                     # two 128-row tiles of sequences
    ([65536], 1),                         # more than 32 partials for one sequence
    ([700, 65], 10 ** 6),                 # nothing to merge: the projection alone
])
def test_merge_out_proj_matches_separate_kernels_and_oracle(lens, min_pages):
    inp = synth.make_inputs(lens, seed=700 + len(lens), poison_tail=True)
    info, plan_dev, ws, o_lat, lse, w_uv, q_abs = _decode(inp, min_pages)
    B = inp.batch
    if min_pages == 1 and lens == [65536]:
        assert info.max_splits > 32
    # separate kernels
    o_a, l_a = o_lat.clone(), lse.clone()
    out_a = torch.empty(B, 128, 128, dtype=torch.bfloat16, device=DEV)
    binding.mla_combine_splits(info, plan_dev, ws, o_a, l_a)
    binding.mla_out_proj(o_a, w_uv, out_a)
    # fused kernel
    o_b, l_b = o_lat.clone(), lse.clone()
    out_b = torch.full((B, 128, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.mla_merge_out_proj(info, plan_dev, ws, o_b, l_b, w_uv, out_b, err)
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(err) == 0
    assert torch.equal(o_b, o_a) and torch.equal(l_b, l_a), "merged rows differ from the merge kernel's"
    assert torch.equal(out_b, out_a), "fused projection differs from the separate kernels"
    # against the oracle: latent attention, then W_UV
    heads = list(range(0, 128, 16)) if inp.num_tokens > 20000 else None
    ref_o, _ = oracle.latent_attention(inp, q_abs.double().numpy(), softmax_scale=SCALE, heads=heads)
    hs = list(range(128)) if heads is None else heads
    full = np.zeros((B, 128, 512))
    full[:, hs, :] = ref_o
    ref = oracle.out_proj(full, inp.w_uv)[:, hs, :]
    assert_close(out_b[:, hs, :], ref, TOL_BF16, "out (fused tail)")


def test_merge_out_proj_twice_in_a_row_is_stable():
    """A second fused call on merged rows it already wrote leaves them unchanged (it re-merges
    from the partials, not from o_lat)."""
    inp = synth.make_inputs([3000, 64 * 9 + 1], seed=711, poison_tail=True)
    info, plan_dev, ws, o_lat, lse, w_uv, _ = _decode(inp, 2)
    assert info.num_combine > 0
    out1 = torch.empty(inp.batch, 128, 128, dtype=torch.bfloat16, device=DEV)
    out2 = torch.empty_like(out1)
    binding.mla_merge_out_proj(info, plan_dev, ws, o_lat, lse, w_uv, out1)
    o1 = o_lat.clone()
    binding.mla_merge_out_proj(info, plan_dev, ws, o_lat, lse, w_uv, out2)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(o1, o_lat)
