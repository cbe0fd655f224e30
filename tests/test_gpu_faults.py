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
