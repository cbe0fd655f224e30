"""GPU tests of the captured step from host memory (mla_step_graph_create / _run, used by
DecodeStep.run_host when every host tensor is pinned).

The graph path must give the bits of the one-call path (mla_decode_step_host, taken by
run_host for pageable tensors) for the same inputs, also after new queries are written into the
same pinned tensors, after a change of lengths (a new graph) and for the FP8 cache; and one case
is checked against the oracle directly.
"""
import ctypes
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


def _steps(inp):
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    mk = lambda: binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
    return mk(), mk()


def _pinned(t):
    return t.clone().pin_memory()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_graph_path_matches_one_call_path(kv_dtype):
    inp = synth.make_inputs([3000, 700, 64 * 9 + 1, 129], seed=31, poison_tail=True, kv_dtype=kv_dtype)
    one_call, graphed = _steps(inp)
    bt_h = torch.from_numpy(np.ascontiguousarray(inp.block_table))
    q_c_p, q_r_p, bt_p = _pinned(inp.q_c), _pinned(inp.q_r), _pinned(bt_h)
    out_p = torch.empty(inp.batch, 128, 128, dtype=torch.bfloat16).pin_memory()
    g = torch.Generator().manual_seed(5)
    for i in range(3):
        if i:
            # the next step's queries, written into the same pinned tensors
            q_c_p.copy_(torch.randn(tuple(q_c_p.shape), generator=g).to(torch.bfloat16))
            q_r_p.copy_(torch.randn(tuple(q_r_p.shape), generator=g).to(torch.bfloat16))
        want = one_call.run_host(q_c_p.clone(), q_r_p.clone(), block_table=bt_h.clone()).clone()
        got = graphed.run_host(q_c_p, q_r_p, block_table=bt_p, out=out_p)
        assert got is out_p
        assert graphed._host_graph is not None and one_call._host_graph is None
        if i == 0:
            handle = graphed._host_graph[0].value
        assert graphed._host_graph[0].value == handle, "the graph was captured again"
        assert one_call.device_error() == 0 and graphed.device_error() == 0
        assert torch.equal(got, want), (kv_dtype, i)
    assert graphed.info.num_combine > 0


def test_graph_path_new_lengths_and_oracle():
    """New lengths make a new graph; its result is the one of a step built for those lengths
    and matches the oracle."""
    inp = synth.make_inputs([3000, 700, 64 * 9 + 1], seed=32, poison_tail=False)
    step, _ = _steps(inp)
    q_c_p, q_r_p = _pinned(inp.q_c), _pinned(inp.q_r)
    out_p = torch.empty(inp.batch, 128, 128, dtype=torch.bfloat16).pin_memory()
    step.run_host(q_c_p, q_r_p, out=out_p)
    first = step._host_graph[0].value
    short = np.array([1800, 65, 64 * 9 + 1], dtype=np.int32)
    got = step.run_host(q_c_p, q_r_p, seq_lens=short, out=out_p).clone()
    assert step._host_graph[0].value != first
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    fresh = binding.DecodeStep(short, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
    ref = fresh.run(q_c, q_r).cpu()
    assert step.device_error() == 0 and torch.equal(got, ref)
    # the oracle on the new lengths
    inp.seq_lens = short
    q_abs = bf16_round(oracle.absorb_q(inp.q_c, inp.w_uk))
    o_ref, _ = oracle.latent_attention(inp, q_abs.double().numpy(), softmax_scale=SCALE)
    want = oracle.out_proj(bf16_round(o_ref).double().numpy(), inp.w_uv)
    assert_close(got, want, TOL_BF16, "out (captured step)")


def test_graph_runs_on_another_stream_and_rejects_pageable_buffers():
    inp = synth.make_inputs([2000, 300], seed=33, poison_tail=False)
    step, ref_step = _steps(inp)
    q_c_p, q_r_p = _pinned(inp.q_c), _pinned(inp.q_r)
    out_p = torch.empty(inp.batch, 128, 128, dtype=torch.bfloat16).pin_memory()
    want = ref_step.run_host(inp.q_c, inp.q_r).clone()
    side = torch.cuda.Stream(DEV)
    step.run_host(q_c_p, q_r_p, out=out_p, stream=side)
    got = step.run_host(q_c_p, q_r_p, out=out_p, stream=side)
    assert torch.equal(got, want)
    # pageable out: the library refuses to capture copies from it
    L = binding.lib()
    h = ctypes.c_void_p()
    bufs = binding.StepBuffers(binding._addr(step._q_c_dev), binding._addr(step._q_r_dev), binding._addr(step.q_abs),
                               binding._addr(step.block_table), binding._addr(step._d_stage),
                               binding._addr(step.workspace),
                               0 if step.workspace is None else step.workspace.numel() * 4,
                               binding._addr(step.o_lat), binding._addr(step.lse), binding._addr(step.out),
                               binding._addr(step.dev_error), binding._addr(step._h_stage), step._h_stage.numel() * 4)
    opts = binding.PlanOptions(2, 0, 0, 0, 0)
    info = binding.PlanInfo()
    pageable_out = torch.empty(inp.batch, 128, 128, dtype=torch.bfloat16)
    st = L.mla_step_graph_create(inp.seq_lens.ctypes.data_as(ctypes.c_void_p), inp.batch, binding.num_sms(),
                                 ctypes.byref(opts), binding._ptr(q_c_p), binding._ptr(q_r_p), None,
                                 int(step.block_table.shape[1]), binding._ptr(step.w_uk), binding._ptr(step.w_uv),
                                 binding.MLA_KV_BF16, binding._ptr(step.kv_pool), None, None,
                                 int(step.kv_pool.shape[0]), ctypes.c_float(step.softmax_scale), ctypes.byref(bufs),
                                 binding._ptr(pageable_out), ctypes.byref(info), None, ctypes.byref(h))
    assert st == binding.MLA_ERR_INVALID_ARG and h.value is None
