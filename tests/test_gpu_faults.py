"""Failure detection on the GPU without faulting it: a bad block-table entry and a wait that
runs out are reported through the device error word and the context stays usable."""
import os
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from mla_latent_kv_absorb_gb300 import binding, synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_wait_timeout_sets_error_bit():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.mla_debug_wait_timeout(err, 50_000_000)  # 50 ms on a barrier nothing completes
    bits = binding.mla_read_device_error(err)
    assert bits & binding.MLA_DEVERR_TIMEOUT
    # the context still works
    x = torch.ones(1024, device=DEV)
    assert float(x.sum()) == 1024.0


def test_bad_block_table_entry_is_reported():
    inp = synth.make_inputs([300, 200], seed=9)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    bt[1, 1] = inp.num_pool_pages + 5   # outside the pool
    bt[0, 0] = -3
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, **kv)
    step.run(q_c, q_r)
    bits = step.device_error()
    assert bits & binding.MLA_DEVERR_BAD_PAGE
    assert not bits & binding.MLA_DEVERR_TIMEOUT
    x = torch.ones(1024, device=DEV)
    assert float(x.sum()) == 1024.0


def test_short_block_table_row_is_reported():
    """A table of exactly batch x max_pages entries whose rows are too short for the lengths:
    the kernel reads no entry past a row (the last sequence would otherwise read past the
    allocation), reports MLA_DEVERR_BAD_PAGE, and the context stays usable."""
    inp = synth.make_inputs([200, 300], seed=10)          # 4 and 5 pages
    q_c, q_r, w_uk, w_uv, kv, bt_full = binding.inputs_to_device(inp, DEV)
    bt = bt_full[:, :4].contiguous()                      # sequence 1 needs 5 entries
    assert bt.numel() == 2 * 4
    plan, info = binding.mla_plan_splits(inp.seq_lens, binding.num_sms())
    plan_dev = torch.from_numpy(plan).to(DEV)
    q_abs = torch.empty(2, 128, 512, dtype=torch.bfloat16, device=DEV)
    binding.mla_absorb_q(q_c, w_uk, q_abs)
    o_lat = torch.empty(2, 128, 512, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(2, 128, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(info.workspace_bytes // 4, 4), dtype=torch.float32, device=DEV)
    binding.mla_decode_paged(info, plan_dev, q_abs, q_r, block_table=bt, o_lat=o_lat, lse=lse, dev_error=err,
                             workspace=ws, **kv)
    bits = binding.mla_read_device_error(err)
    assert bits & binding.MLA_DEVERR_BAD_PAGE
    assert not bits & binding.MLA_DEVERR_TIMEOUT
    x = torch.ones(1024, device=DEV)
    assert float(x.sum()) == 1024.0
    # the host-side entry points refuse such a table before launching anything
    with pytest.raises(ValueError):
        binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, **kv)
