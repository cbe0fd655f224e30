"""GPU parity of the cache-append kernels (mla_append_kv) against the oracle, byte for byte.

The append is integer and byte work (a copy, or an e4m3 quantisation whose every rounding is
fixed by the rule), so the bar is exact equality of the whole pool: written slots, scales and
untouched slots alike.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
from oracle_pins import _quant_rows  # noqa: E402

from mla_latent_kv_absorb_gb300 import binding, synth  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
PAGES = 8


def _u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _tokens(n: int, seed: int):
    """bf16 c_KV [n, 512] and k_R [n, 64]: N(0,1) rows scaled by 2^U(-12, 8), the quantiser's
    special rows (outliers, subnormal codes, exact ties, signed zeros) first."""
    g = torch.Generator().manual_seed(seed)
    scales = torch.exp2(torch.empty(n).uniform_(-12.0, 8.0, generator=g))
    c = (torch.randn(n, 512, generator=g) * scales[:, None]).to(torch.bfloat16)
    special = _quant_rows()
    k = min(n, special.shape[0])
    c[:k] = special[:k]
    r = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    return c, r


def _slots(n: int, seed: int) -> np.ndarray:
    """n distinct slots of the pool in random order; two of them negative (padding) when n > 8."""
    s = np.random.default_rng(seed).permutation(PAGES * 64)[:n].astype(np.int32)
    if n > 8:
        s[5], s[n - 2] = -1, -7
    return s


def _append(c, r, slots, **kv):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.mla_append_kv(c.to(DEV), r.to(DEV), torch.from_numpy(slots).to(DEV), dev_error=err, **kv)
    torch.cuda.synchronize()
    return binding.mla_read_device_error(err)


@pytest.mark.parametrize("n", [1, 13, 300])
def test_append_bf16_matches_oracle(n):
    c, r = _tokens(n, seed=n)
    slots = _slots(n, seed=n)
    pool0 = torch.randn(PAGES, 64, 576, generator=torch.Generator().manual_seed(99)).to(torch.bfloat16)
    ref = {"pool": _u16(pool0).copy()}
    assert oracle.append_kv(c, r, slots, ref) == 0
    pool = pool0.to(DEV)
    assert _append(c, r, slots, kv_pool=pool) == 0
    assert np.array_equal(_u16(pool.cpu()), ref["pool"])


@pytest.mark.parametrize("n", [1, 13, 300])
def test_append_fp8_matches_oracle(n):
    c, r = _tokens(n, seed=100 + n)
    slots = _slots(n, seed=100 + n)
    g = torch.Generator().manual_seed(98)
    c8_0 = torch.randint(0, 256, (PAGES, 64, 512), generator=g, dtype=torch.uint8)
    sc0 = torch.rand(PAGES, 64, generator=g)
    kr0 = torch.randn(PAGES, 64, 64, generator=g).to(torch.bfloat16)
    ref = {"c8": c8_0.numpy().copy(), "scale": sc0.numpy().copy(), "kr": _u16(kr0).copy()}
    assert oracle.append_kv(c, r, slots, ref) == 0
    c8, sc, kr = c8_0.to(DEV), sc0.to(DEV), kr0.to(DEV)
    assert _append(c, r, slots, kv_pool=c8, kv_scale=sc, kr_pool=kr) == 0
    got_c8 = c8.cpu().numpy()
    bad = np.argwhere(got_c8 != ref["c8"])
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}"
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), ref["scale"].view(np.uint32))
    assert np.array_equal(_u16(kr.cpu()), ref["kr"])


def test_append_slot_past_pool_is_reported_and_skipped():
    c, r = _tokens(4, seed=7)
    slots = np.array([0, PAGES * 64, 3, PAGES * 64 + 100], np.int32)
    for fp8 in (False, True):
        if fp8:
            c8_0 = torch.zeros(PAGES, 64, 512, dtype=torch.uint8)
            sc0 = torch.zeros(PAGES, 64)
            kr0 = torch.zeros(PAGES, 64, 64, dtype=torch.bfloat16)
            ref = {"c8": c8_0.numpy().copy(), "scale": sc0.numpy().copy(), "kr": _u16(kr0).copy()}
            dev = dict(kv_pool=c8_0.to(DEV), kv_scale=sc0.to(DEV), kr_pool=kr0.to(DEV))
        else:
            pool0 = torch.zeros(PAGES, 64, 576, dtype=torch.bfloat16)
            ref = {"pool": _u16(pool0).copy()}
            dev = dict(kv_pool=pool0.to(DEV))
        assert oracle.append_kv(c, r, slots, ref) == -1
        assert _append(c, r, slots, **dev) == 16  # MLA_DEVERR_BAD_SLOT, and nothing else
        if fp8:
            assert np.array_equal(dev["kv_pool"].cpu().numpy(), ref["c8"])
            assert np.array_equal(dev["kv_scale"].cpu().numpy().view(np.uint32), ref["scale"].view(np.uint32))
            assert np.array_equal(_u16(dev["kr_pool"].cpu()), ref["kr"])
        else:
            assert np.array_equal(_u16(dev["kv_pool"].cpu()), ref["pool"])


def test_append_then_decode_step():
    """Knock the last token of every sequence out of a bf16 cache (NaN rows), append it back
    through the kernel: the pool is the original bit for bit and the decode step gives the
    original step's bits."""
    inp = synth.make_inputs([300, 64, 129], seed=31, poison_tail=False)
    q_c, q_r, w_uk, w_uv, kv, bt = binding.inputs_to_device(inp, DEV)
    step = binding.DecodeStep(inp.seq_lens, w_uk=w_uk, w_uv=w_uv, block_table=bt, min_pages_per_split=2, **kv)
    ref = step.run(q_c, q_r).clone()
    torch.cuda.synchronize()
    slots = np.array([int(inp.block_table[b, (int(S) - 1) // 64]) * 64 + (int(S) - 1) % 64
                      for b, S in enumerate(inp.seq_lens)], np.int32)
    rows = inp.pool.reshape(-1, 576)[torch.from_numpy(slots).long()].clone()
    pool = kv["kv_pool"]
    pool.view(-1, 576)[torch.from_numpy(slots).long().to(DEV)] = float("nan")
    assert _append(rows[:, :512].contiguous(), rows[:, 512:].contiguous(), slots, kv_pool=pool) == 0
    assert torch.equal(pool.cpu().view(torch.int16), inp.pool.view(torch.int16))
    out = step.run(q_c, q_r).clone()
    torch.cuda.synchronize()
    assert step.device_error() == 0
    assert torch.equal(out, ref)


def _nvfp4_tokens(n: int, seed: int):
    """Like _tokens, plus NVFP4 cases: rows with zero blocks, a block far below the token's
    maximum (its scale rounds to a subnormal e4m3 or to zero), and a lone outlier."""
    c, r = _tokens(n, seed)
    if n >= 8:
        g = torch.Generator().manual_seed(seed + 1)
        x = torch.randn(4, 512, generator=g)
        x[0, 32:64] = 0.0                          # two zero blocks
        x[1, 0] = 1e4                              # one outlier: the other blocks' scales shrink
        x[2, 16:32] *= 1e-9                        # a block whose scale rounds to zero
        x[3, :16] = -0.0
        c[-4:] = x.to(torch.bfloat16)
    return c, r


@pytest.mark.parametrize("n", [1, 13, 300])
def test_append_nvfp4_matches_oracle(n):
    c, r = _nvfp4_tokens(n, seed=200 + n)
    slots = _slots(n, seed=200 + n)
    g = torch.Generator().manual_seed(97)
    rows0 = torch.randint(0, 256, (PAGES, 64, binding.NVFP4_ROW), generator=g, dtype=torch.uint8)
    sc0 = torch.rand(PAGES, 64, generator=g)
    kr0 = torch.randn(PAGES, 64, 64, generator=g).to(torch.bfloat16)
    ref = {"c4": rows0.numpy().copy(), "scale": sc0.numpy().copy(), "kr": _u16(kr0).copy()}
    assert oracle.append_kv(c, r, slots, ref) == 0
    rows, sc, kr = rows0.to(DEV), sc0.to(DEV), kr0.to(DEV)
    assert _append(c, r, slots, kv_pool=rows, kv_scale=sc, kr_pool=kr) == 0
    got = rows.cpu().numpy()
    bad = np.argwhere(got != ref["c4"])
    assert bad.size == 0, f"{len(bad)} bytes differ, first at {bad[:3].tolist()}"
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), ref["scale"].view(np.uint32))
    assert np.array_equal(_u16(kr.cpu()), ref["kr"])


def test_nvfp4_cache_is_rejected_by_the_decode():
    """No decode kernel reads the NVFP4 cache yet: the decode call says so on the host."""
    inp = synth.make_inputs([100], seed=5)
    q_abs = torch.zeros(1, 128, 512, dtype=torch.bfloat16, device=DEV)
    plan, info = binding.mla_plan_splits(inp.seq_lens, binding.num_sms())
    rows = torch.zeros(inp.num_pool_pages, 64, binding.NVFP4_ROW, dtype=torch.uint8, device=DEV)
    with pytest.raises(binding.MlaError) as e:
        binding.mla_decode_paged(info, torch.from_numpy(plan).to(DEV), q_abs, inp.q_r.to(DEV), kv_pool=rows,
                                 kv_scale=torch.ones(inp.num_pool_pages, 64, device=DEV),
                                 kr_pool=torch.zeros(inp.num_pool_pages, 64, 64, dtype=torch.bfloat16, device=DEV),
                                 block_table=torch.from_numpy(inp.block_table).to(DEV),
                                 o_lat=torch.empty(1, 128, 512, dtype=torch.bfloat16, device=DEV),
                                 lse=torch.empty(1, 128, device=DEV), dev_error=torch.zeros(1, dtype=torch.int32,
                                                                                            device=DEV))
    assert e.value.status == binding.MLA_ERR_UNSUPPORTED
