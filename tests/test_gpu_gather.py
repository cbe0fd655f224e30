"""GPU parity of the paged-cache gather (mla_gather_kv) against the oracle, bit for bit.

Every row is integer work (a copy) or one fp32 product rounded to bf16, fixed by the stated rule,
so the bar is equality of the whole output for bf16, FP8 and NVFP4 caches.
"""
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle  # noqa: E402
from oracle_pins import nvfp4_inputs  # noqa: E402

from mla_latent_kv_absorb_gb300 import binding, synth  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gather(inp):
    kv = {}
    if inp.kv_dtype == "bf16":
        kv["kv_pool"] = inp.pool.to(DEV)
    else:
        kv["kv_pool"], kv["kv_scale"], kv["kr_pool"] = inp.c8.to(DEV), inp.kv_scale.to(DEV), inp.kr.to(DEV)
    sl = torch.from_numpy(np.ascontiguousarray(inp.seq_lens, np.int32))
    cu = torch.zeros(inp.batch + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(sl, 0)
    out = torch.full((int(cu[-1]), 576), float("nan"), dtype=torch.bfloat16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.mla_gather_kv(block_table=torch.from_numpy(np.ascontiguousarray(inp.block_table)).to(DEV),
                          seq_lens=sl.to(DEV), cu_seqlens=cu.to(DEV), out=out, dev_error=err, **kv)
    torch.cuda.synchronize()
    return out.cpu().view(torch.int16).numpy().view(np.uint16), binding.mla_read_device_error(err)


@pytest.mark.parametrize("kind", ["bf16", "fp8_e4m3", "nvfp4"])
@pytest.mark.parametrize("lens", [[1, 64, 65], [700, 3, 2000, 129]])
def test_gather_matches_oracle(kind, lens):
    if kind == "nvfp4":
        inp = nvfp4_inputs(tuple(lens), seed=40 + len(lens))
    else:
        inp = synth.make_inputs(lens, seed=40 + len(lens), kv_dtype=kind, poison_tail=True)
    got, bits = _gather(inp)
    assert bits == 0
    ref, _ = oracle.gather_kv(inp)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{kind}: {len(bad)} values differ, first at {bad[:3].tolist()}"


def test_gather_bad_page_is_reported():
    inp = synth.make_inputs([130, 70], seed=44)
    inp.block_table = inp.block_table.copy()
    inp.block_table[1, 0] = inp.num_pool_pages + 3
    got, bits = _gather(inp)
    assert bits & binding.MLA_DEVERR_BAD_PAGE
    vals = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.isfinite(vals[:130]).all()                  # sequence 0 is complete
    assert np.isnan(vals[130:130 + 64]).all()             # the bad page's rows are not written
    assert np.isfinite(vals[130 + 64:]).all()             # the rest of sequence 1 is
    x = torch.ones(16, device=DEV)                        # the context still works
    assert float(x.sum()) == 16.0
