"""GPU parity of several new tokens per sequence in one decode step (plan option
queries_per_seq = q): query row b*q + t is new token t of sequence b and sees the first
S_b - q + 1 + t cached tokens.  The whole step (absorb, decode with splits, merge, projection)
is compared with the oracle's prefix decodes of the same rows, for the bf16 and FP8 caches,
and the host-buffer paths must give the device path's bits.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
from parity_util import SCALE, TOL_BF16, TOL_FP8, assert_close, bf16_round  # noqa: E402

from mla_latent_kv_absorb_gb300 import binding, synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _mq_inputs(lens, q, seed, kv_dtype="bf16"):
    inp = synth.make_inputs(lens, seed=seed, poison_tail=True, kv_dtype=kv_dtype)
    g = torch.Generator().manual_seed(seed + 1)
    rows = len(lens) * q
    inp.q_c = torch.randn(rows, 128, 128, generator=g).to(torch.bfloat16)
    inp.q_r = torch.randn(rows, 128, 64, generator=g).to(torch.bfloat16)
    return inp


@pytest.mark.parametrize("q,kv_dtype", [(2, "bf16"), (4, "bf16"), (7, "bf16"), (3, "fp8_e4m3")])
def test_multi_query_step_matches_oracle(q, kv_dtype):
    lens = [3000, 700, 64 * 9 + q, q, 129]  # S_b = q: the first new token sees one cached token
    inp = _mq_inputs(lens, q, seed=900 + q, kv_dtype=kv_dtype)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2,
                              queries_per_seq=q, **kv)
    assert step.info.batch == len(lens) * q and step.info.queries_per_seq == q and step.info.num_combine > 0
    out = step.run(q_c, q_r).clone()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    tol = TOL_BF16 if kv_dtype == "bf16" else TOL_FP8
    rows = oracle.query_row_inputs(inp, q)
    q_abs = bf16_round(oracle.absorb_q(inp.q_c, inp.w_uk))
    assert_close(step.q_abs, q_abs, TOL_BF16, "q_abs")
    o_ref, l_ref = oracle.latent_attention(rows, q_abs.double().numpy(), softmax_scale=SCALE)
    assert_close(step.o_lat, o_ref, tol, f"o_lat q={q}")
    assert_close(step.lse, l_ref, tol, f"lse q={q}")
    want = oracle.out_proj(bf16_round(o_ref).double().numpy(), inp.w_uv)
    assert_close(out, want, tol, f"out q={q}")
    # the decompressed definition on a few heads of every row
    heads = [3, 100]
    naive = oracle.decode_naive(rows, softmax_scale=SCALE, heads=heads)
    assert_close(out[:, heads, :], naive, tol, f"out vs naive q={q}")


def test_multi_query_host_paths_match_device_path():
    q = 3
    inp = _mq_inputs([2000, 64 * 5 + 3, 300], q, seed=950)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    mk = lambda: binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2,
                                    queries_per_seq=q, **kv)
    dev_step, one_call, graphed = mk(), mk(), mk()
    want = dev_step.run(q_c, q_r).cpu()
    bt_h = torch.from_numpy(np.ascontiguousarray(inp.block_table))
    got1 = one_call.run_host(inp.q_c, inp.q_r, block_table=bt_h)
    out_p = torch.empty(inp.batch * q, 128, 128, dtype=torch.bfloat16).pin_memory()
    got2 = graphed.run_host(inp.q_c.pin_memory(), inp.q_r.pin_memory(), block_table=bt_h.pin_memory(), out=out_p)
    assert graphed._host_graph is not None
    assert one_call.device_error() == 0 and graphed.device_error() == 0
    assert torch.equal(got1, want) and torch.equal(got2, want)


@pytest.mark.parametrize("fused_absorb,fused_tail", [(True, False), (False, True), (True, True)])
def test_multi_query_through_the_fused_calls(fused_absorb, fused_tail):
    """The fused absorb (decode prologue) and the fused merge + projection take the same query
    rows: bit-identical to the separate kernels."""
    q = 3
    inp = _mq_inputs([2500, 64 * 7 + 3, 700], q, seed=960)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    mk = lambda **f: binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2,
                                        queries_per_seq=q, **kv, **f)
    want = mk().run(q_c, q_r).clone()
    step = mk(fused_absorb=fused_absorb, fused_tail=fused_tail)
    got = step.run(q_c, q_r).clone()
    torch.cuda.synchronize()
    assert step.device_error() == 0 and step.info.num_combine > 0
    assert torch.equal(got, want)


def test_multi_query_static_workspace_matches():
    """The no-allocation decode entry point takes the query rows too (same plan, same bits)."""
    q = 2
    inp = _mq_inputs([3000, 900], q, seed=970)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2,
                              queries_per_seq=q, **kv)
    step.run(q_c, q_r)
    torch.cuda.synchronize()
    assert step.info.num_partials <= binding.MLA_STATIC_WS_MAX_PARTIALS
    o2 = torch.empty_like(step.o_lat)
    l2 = torch.empty_like(step.lse)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.mla_decode_paged_static_ws(step.info, step.plan_dev, step.q_abs, q_r, kv_pool=kv["kv_pool"],
                                       block_table=bt, o_lat=o2, lse=l2, dev_error=err)
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(err) == 0
    assert torch.equal(o2, step.o_lat) and torch.equal(l2, step.lse)
