"""GPU parity of a prefill chunk: the last T tokens of a sequence attended causally over the
whole sequence (query t sees the first S - T + 1 + t tokens).  Chunks of at least 256 tokens
take the decompressed form (gather, per-head decompression of keys and values, causal
attention kernel), shorter ones the absorbed decode with T query rows; both are compared with
the oracle's prefix decodes of the same rows, for bf16 and quantised caches.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
import oracle_pins as pins  # noqa: E402
from parity_util import SCALE, TOL_BF16, TOL_FP8, assert_close, bf16_round  # noqa: E402

from mla_latent_kv_absorb_gb300 import binding, synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _chunk_inputs(S, T, seed, kv_dtype="bf16"):
    inp = synth.make_inputs([S], seed=seed, poison_tail=True, kv_dtype=kv_dtype)
    g = torch.Generator().manual_seed(seed + 1)
    inp.q_c = torch.randn(T, 128, 128, generator=g).to(torch.bfloat16)
    inp.q_r = torch.randn(T, 128, 64, generator=g).to(torch.bfloat16)
    return inp


def _oracle_out(inp, T):
    rows = oracle.query_row_inputs(inp, T)
    q_abs = bf16_round(oracle.absorb_q(inp.q_c, inp.w_uk)).double().numpy()
    o_lat, _ = oracle.latent_attention(rows, q_abs, softmax_scale=SCALE)
    return oracle.out_proj(o_lat, inp.w_uv), rows


def _run(inp, T, threshold=binding.PREFILL_THRESHOLD):
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    kv = dict(kv)
    pool = kv.pop("kv_pool")
    out, err = binding.prefill_chunk(int(inp.seq_lens[0]), q_c, q_r, w_uk=w_uk, w_uv=w_uv, kv_pool=pool,
                                     block_table_row=bt[0], threshold=threshold, **kv)
    torch.cuda.synchronize()
    assert binding.mla_read_device_error(err) == 0
    return out.cpu()


@pytest.mark.parametrize("S,T", [(640, 260), (300, 300), (1000, 256), (777, 384)])
def test_decompressed_chunk_matches_oracle(S, T):
    inp = _chunk_inputs(S, T, seed=1000 + S + T)
    got = _run(inp, T)
    want, rows = _oracle_out(inp, T)
    assert_close(got, want, TOL_BF16, f"prefill S={S} T={T}")
    # the decompressed definition itself on two heads
    heads = [7, 90]
    naive = oracle.decode_naive(rows, softmax_scale=SCALE, heads=heads)
    assert_close(got[:, heads, :], naive, TOL_BF16, "prefill vs naive")


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "nvfp4"])
def test_decompressed_chunk_quantised_cache(kv_dtype):
    """The gather dequantises the FP8 or NVFP4 cache into the bf16 rows the decompression reads."""
    S, T = 520, 270
    if kv_dtype == "nvfp4":
        inp = pins.nvfp4_inputs((S,), seed=1101, poison=True)  # rows written by the oracle's quantiser
        g = torch.Generator().manual_seed(1102)
        inp.q_c = torch.randn(T, 128, 128, generator=g).to(torch.bfloat16)
        inp.q_r = torch.randn(T, 128, 64, generator=g).to(torch.bfloat16)
    else:
        inp = _chunk_inputs(S, T, seed=1100, kv_dtype=kv_dtype)
    got = _run(inp, T)
    want, _ = _oracle_out(inp, T)
    assert_close(got, want, TOL_FP8, f"prefill {kv_dtype}")


@pytest.mark.parametrize("T", [1, 37, 255])
def test_short_chunks_take_the_absorbed_path(T):
    S = 700
    inp = _chunk_inputs(S, T, seed=1200 + T)
    got = _run(inp, T)
    want, _ = _oracle_out(inp, T)
    assert_close(got, want, TOL_BF16, f"absorbed chunk T={T}")


def test_both_forms_agree_across_the_threshold():
    """The same 300-token chunk through both forms (threshold moved): the results agree within
    the bf16 tolerance of each other."""
    S, T = 900, 300
    inp = _chunk_inputs(S, T, seed=1300)
    dec = _run(inp, T)
    absd = _run(inp, T, threshold=T + 1)
    assert_close(dec, absd.double().numpy(), TOL_BF16, "decompressed vs absorbed")
