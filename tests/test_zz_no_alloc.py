"""mla_decode_paged_static_ws: decode plus split merge on the library's fixed scratch array.

Compared, bit for bit, with mla_decode_paged + mla_combine_splits on a caller workspace, over
two calls in a row on different plans (the second call finds the first call's partials in the
array).  Named to be collected last, so it also runs after every other GPU test.
"""
import ctypes
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
from parity_util import bf16_round  # noqa: E402

from mla_latent_kv_absorb_gb300 import binding, build, synth  # noqa: E402

DEV = "cuda:0"


def test_static_ws_rejects_oversized_plan():
    """Host-side check, no GPU needed: a plan with more partials than the array holds."""
    build.build_library()
    L = binding.lib()
    lens = [64 * 64] * 200
    _, info = binding.mla_plan_splits(lens, 152, min_pages_per_split=1, item_cost_pages=-1)  # equal page runs
    assert info.num_partials > binding.MLA_STATIC_WS_MAX_PARTIALS
    p = ctypes.c_void_p
    st = L.mla_decode_paged_static_ws(ctypes.byref(info), p(0x20000), p(0x10000), p(0x30000), binding.MLA_KV_BF16,
                                      p(0x40000), None, None, 100, p(0x60000), 80, ctypes.c_float(0.07),
                                      p(0x70000), p(0x80000), p(0x50000), None)
    assert st == binding.MLA_ERR_WORKSPACE
    assert "static workspace holds at most 128" in L.mla_last_error_string().decode()


def _case(lens, seed, min_pages, kv_dtype="bf16"):
    inp = synth.make_inputs(lens, seed=seed, poison_tail=True, kv_dtype=kv_dtype)
    q_abs = bf16_round(oracle.absorb_q(inp.q_c, inp.w_uk)).to(DEV)
    _, q_r, _, _, kv, bt = binding.inputs_to_device(inp, DEV)
    plan, info = binding.mla_plan_splits(inp.seq_lens, binding.num_sms(), min_pages_per_split=min_pages)
    args = dict(info=info, plan_dev=torch.from_numpy(plan).to(DEV), q_abs=q_abs, q_r=q_r, block_table=bt, **kv)
    return inp.batch, args


def _outputs(B):
    return (torch.full((B, 128, 512), float("nan"), dtype=torch.bfloat16, device=DEV),
            torch.full((B, 128), float("nan"), dtype=torch.float32, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV))


def _reference(B, a):
    o, l, err = _outputs(B)
    ws = torch.empty(max(a["info"].workspace_bytes // 4, 4), dtype=torch.float32, device=DEV)
    binding.mla_decode_paged(a["info"], a["plan_dev"], a["q_abs"], a["q_r"], kv_pool=a["kv_pool"],
                             block_table=a["block_table"], o_lat=o, lse=l, dev_error=err, workspace=ws,
                             kv_scale=a.get("kv_scale"), kr_pool=a.get("kr_pool"))
    binding.mla_combine_splits(a["info"], a["plan_dev"], ws, o, l)
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(err) == 0
    return o, l


def _static(a, o, l, err):
    binding.mla_decode_paged_static_ws(a["info"], a["plan_dev"], a["q_abs"], a["q_r"], kv_pool=a["kv_pool"],
                                       block_table=a["block_table"], o_lat=o, lse=l, dev_error=err,
                                       kv_scale=a.get("kv_scale"), kr_pool=a.get("kr_pool"))


@pytest.mark.gpu
def test_static_ws_matches_workspace_entry_point():
    Ba, a = _case([3000, 700, 64 * 40 + 5, 1], seed=901, min_pages=2)
    Bb, b = _case([9000, 129, 64 * 7], seed=902, min_pages=1)
    assert a["info"].num_combine > 0 and b["info"].num_combine > 0
    assert a["info"].num_partials <= binding.MLA_STATIC_WS_MAX_PARTIALS
    assert b["info"].num_partials <= binding.MLA_STATIC_WS_MAX_PARTIALS
    ref_a, ref_b = _reference(Ba, a), _reference(Bb, b)

    # two calls in a row on one stream (the first one on this device also does the set-up)
    oa, la, ea = _outputs(Ba)
    ob, lb, eb = _outputs(Bb)
    _static(a, oa, la, ea)
    _static(b, ob, lb, eb)
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(ea) == 0 and binding.mla_read_device_error(eb) == 0
    assert torch.equal(oa, ref_a[0]) and torch.equal(la, ref_a[1])
    assert torch.equal(ob, ref_b[0]) and torch.equal(lb, ref_b[1])

    # again, in the other order, with the device's free memory unchanged across the calls
    oa2, la2, ea2 = _outputs(Ba)
    ob2, lb2, eb2 = _outputs(Bb)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    _static(b, ob2, lb2, eb2)
    _static(a, oa2, la2, ea2)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0
    assert torch.equal(oa2, ref_a[0]) and torch.equal(la2, ref_a[1])
    assert torch.equal(ob2, ref_b[0]) and torch.equal(lb2, ref_b[1])


@pytest.mark.gpu
def test_static_ws_single_item_plan():
    """A plan without split partials never touches the array."""
    B, a = _case([700, 65], seed=903, min_pages=10 ** 6)
    assert a["info"].workspace_bytes == 0
    ref = _reference(B, a)
    o, l, err = _outputs(B)
    _static(a, o, l, err)
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(err) == 0
    assert torch.equal(o, ref[0]) and torch.equal(l, ref[1])


@pytest.mark.gpu
def test_static_ws_matches_workspace_entry_point_fp8():
    """The e4m3 cache through the fixed array: split partials, two calls in a row."""
    Ba, a = _case([2000, 64 * 30 + 17, 300], seed=904, min_pages=2, kv_dtype="fp8_e4m3")
    Bb, b = _case([5000, 64], seed=905, min_pages=1, kv_dtype="fp8_e4m3")
    assert a["info"].num_combine > 0 and b["info"].num_combine > 0
    ref_a, ref_b = _reference(Ba, a), _reference(Bb, b)
    oa, la, ea = _outputs(Ba)
    ob, lb, eb = _outputs(Bb)
    _static(a, oa, la, ea)
    _static(b, ob, lb, eb)
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(ea) == 0 and binding.mla_read_device_error(eb) == 0
    assert torch.equal(oa, ref_a[0]) and torch.equal(la, ref_a[1])
    assert torch.equal(ob, ref_b[0]) and torch.equal(lb, ref_b[1])
