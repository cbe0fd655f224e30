"""Seeded synthetic decode inputs, shared by the tests, the bench and the oracle checks.

This module only draws random numbers and lays them out the way a paged latent cache is
stored. It holds none of the attention arithmetic, so the CUDA path and the CPU oracle can
both take their inputs from here without sharing any of the method.

Recipe (one ``torch.Generator('cpu')`` seeded once, drawn in this fixed order):

1. ragged context lengths, when asked for: integers uniform on [lo, hi] inclusive;
2. ``q_c``  [B, 128, 128] ~ N(0, 1);
3. ``q_R``  [B, 128, 64]  ~ N(0, 1) (already rotated: no RoPE is applied on the path);
4. ``W_UK`` [128, 128, 512] ~ N(0, 1/512), layout (heads, d_hc, d_c);
5. ``W_UV`` [128, 128, 512] ~ N(0, 1/512), same layout;
6. the pool's ``c_KV`` rows [N_pg, 64, 512] ~ N(0, 1), drawn 1024 pages at a time;
7. the pool's ``k_R`` rows  [N_pg, 64, 64]  ~ N(0, 1), drawn 1024 pages at a time;
8. the page permutation (``randperm(N_pg)``) when the block table is shuffled.

Every draw is fp32 ``randn``, scaled, then rounded to bf16 (round to nearest even).
The pool holds exactly ``N_pg = sum_b ceil(S_b / 64)`` pages. Logical page ``j`` of
sequence ``b`` lives in physical page ``perm[offset_b + j]`` (identity when unshuffled).
Slots past ``S_b`` in a sequence's last page are NaN when ``poison_tail`` is set, so that
a reader that fails to mask them shows it; otherwise they keep their random values.

FP8 cache: per token, over the 512 ``c_KV`` dims only, ``sigma = absmax / 448`` (1 if the
row is all zero) in fp32 and ``c8 = e4m3(c / sigma)`` through torch's ``float8_e4m3fn``
cast (round to nearest even). ``k_R`` stays bf16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

NUM_HEADS = 128
D_HC = 128
D_C = 512
D_R = 64
D_ROW = D_C + D_R
PAGE = 64
DEFAULT_SEED = 42
_DRAW_PAGES = 1024  # pages per randn call when filling the pool


@dataclasses.dataclass
class DecodeInputs:
    """One decode batch: queries, weights, paged cache and block table (all host/CPU)."""

    seq_lens: np.ndarray          # int32 [B]
    block_table: np.ndarray       # int32 [B, max_pages]
    num_pool_pages: int
    q_c: torch.Tensor             # bf16 [B, 128, 128]
    q_r: torch.Tensor             # bf16 [B, 128, 64]
    w_uk: torch.Tensor            # bf16 [128, 128, 512]
    w_uv: torch.Tensor            # bf16 [128, 128, 512]
    kv_dtype: str                 # "bf16", "fp8_e4m3" or "nvfp4" (c8 then holds [N_pg, 64, 288] NVFP4 rows)
    pool: Optional[torch.Tensor] = None      # bf16 [N_pg, 64, 576]   (bf16 cache)
    c8: Optional[torch.Tensor] = None        # uint8 [N_pg, 64, 512]  (fp8 cache: e4m3 codes)
    kv_scale: Optional[torch.Tensor] = None  # fp32 [N_pg, 64]        (fp8 cache)
    kr: Optional[torch.Tensor] = None        # bf16 [N_pg, 64, 64]    (fp8 cache)
    seed: int = DEFAULT_SEED
    queries_per_seq: int = 1      # q_c / q_r hold batch * queries_per_seq rows (row b*q + t: token t of b)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def rows(self) -> int:
        return self.batch * self.queries_per_seq

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def num_tokens(self) -> int:
        return int(self.seq_lens.sum())


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def ragged_lengths(batch: int, lo: int, hi: int, gen: torch.Generator) -> np.ndarray:
    """Context lengths uniform on the integers [lo, hi]."""
    return torch.randint(lo, hi + 1, (batch,), generator=gen, dtype=torch.int64).numpy().astype(np.int32)


def make_inputs(
    seq_lens,
    *,
    seed: int = DEFAULT_SEED,
    shuffle_pages: bool = True,
    kv_dtype: str = "bf16",
    poison_tail: bool = False,
    ragged: Optional[tuple] = None,
    batch: Optional[int] = None,
    queries_per_seq: int = 1,
) -> DecodeInputs:
    """Draw one decode batch.

    ``seq_lens``: list of context lengths, or ``None`` with ``ragged=(lo, hi)`` and
    ``batch`` to draw them (first, from the same generator).  ``queries_per_seq`` = q > 1 draws
    q query rows per sequence (several new tokens decoded at once; the lengths count them).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    if seq_lens is None:
        assert ragged is not None and batch is not None
        lens = ragged_lengths(batch, ragged[0], ragged[1], gen)
    else:
        lens = np.asarray(seq_lens, dtype=np.int32)
    if lens.ndim != 1 or lens.size == 0 or (lens < 1).any():
        raise ValueError("seq_lens must be a non-empty list of positive lengths")
    B = int(lens.size)
    pages_per_seq = (lens.astype(np.int64) + PAGE - 1) // PAGE
    n_pages = int(pages_per_seq.sum())
    max_pages = int(pages_per_seq.max())

    if queries_per_seq < 1 or (lens < queries_per_seq).any():
        raise ValueError("queries_per_seq must be >= 1 and at most every length")
    rows = B * queries_per_seq
    q_c = _bf16(torch.randn(rows, NUM_HEADS, D_HC, generator=gen))
    q_r = _bf16(torch.randn(rows, NUM_HEADS, D_R, generator=gen))
    wstd = 1.0 / math.sqrt(D_C)
    w_uk = _bf16(torch.randn(NUM_HEADS, D_HC, D_C, generator=gen) * wstd)
    w_uv = _bf16(torch.randn(NUM_HEADS, D_HC, D_C, generator=gen) * wstd)

    c_chunks = []
    for p0 in range(0, n_pages, _DRAW_PAGES):
        n = min(_DRAW_PAGES, n_pages - p0)
        c_chunks.append(torch.randn(n, PAGE, D_C, generator=gen))
    r_chunks = []
    for p0 in range(0, n_pages, _DRAW_PAGES):
        n = min(_DRAW_PAGES, n_pages - p0)
        r_chunks.append(torch.randn(n, PAGE, D_R, generator=gen))
    ckv = torch.cat(c_chunks) if len(c_chunks) > 1 else c_chunks[0]
    kr = torch.cat(r_chunks) if len(r_chunks) > 1 else r_chunks[0]
    del c_chunks, r_chunks

    if shuffle_pages:
        perm = torch.randperm(n_pages, generator=gen).numpy().astype(np.int32)
    else:
        perm = np.arange(n_pages, dtype=np.int32)

    offsets = np.concatenate([[0], np.cumsum(pages_per_seq)[:-1]]).astype(np.int64)
    block_table = np.full((B, max_pages), -1, dtype=np.int32)
    for b in range(B):
        block_table[b, : pages_per_seq[b]] = perm[offsets[b] : offsets[b] + pages_per_seq[b]]

    # Pool rows are drawn in physical order; the logical→physical map is the block table.
    tail_mask = None
    if poison_tail:
        tail_mask = np.zeros((n_pages, PAGE), dtype=bool)
        for b in range(B):
            last = int(block_table[b, pages_per_seq[b] - 1])
            used = int(lens[b]) - PAGE * (int(pages_per_seq[b]) - 1)
            tail_mask[last, used:] = True
        tail_mask = torch.from_numpy(tail_mask)

    inp = DecodeInputs(
        seq_lens=lens, block_table=block_table, num_pool_pages=n_pages,
        q_c=q_c, q_r=q_r, w_uk=w_uk, w_uv=w_uv, kv_dtype=kv_dtype, seed=seed, queries_per_seq=queries_per_seq,
    )
    if kv_dtype == "bf16":
        pool = torch.empty(n_pages, PAGE, D_ROW, dtype=torch.bfloat16)
        pool[:, :, :D_C] = _bf16(ckv)
        pool[:, :, D_C:] = _bf16(kr)
        if tail_mask is not None:
            pool[tail_mask] = float("nan")
        inp.pool = pool
    elif kv_dtype == "fp8_e4m3":
        absmax = ckv.abs().amax(dim=-1)
        sigma = torch.where(absmax > 0, absmax / 448.0, torch.ones_like(absmax)).to(torch.float32)
        codes = (ckv / sigma.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
        krb = _bf16(kr)
        if tail_mask is not None:
            codes[tail_mask] = 0x7F          # e4m3 NaN
            sigma[tail_mask] = float("nan")
            krb[tail_mask] = float("nan")
        inp.c8, inp.kv_scale, inp.kr = codes.contiguous(), sigma.contiguous(), krb.contiguous()
    else:
        raise ValueError(f"unknown kv_dtype {kv_dtype!r}")
    return inp


# The five decode workloads, by what they are. Each entry: a short name, the builder
# keyword arguments, and a one-line description.
WORKLOADS = {
    "b1_s2048": dict(seq_lens=[2048], shuffle_pages=False,
                     desc="B=1, S=2048, identity block table, bf16 cache"),
    "b16_s4096": dict(seq_lens=[4096] * 16, shuffle_pages=True,
                      desc="B=16, S=4096 each, shuffled shared page pool, bf16 cache"),
    "b16_s65536": dict(seq_lens=[65536] * 16, shuffle_pages=True,
                       desc="B=16, S=65536 each (64K context, 1.21 GB bf16 cache), shuffled pages, split-KV"),
    "b64_ragged": dict(seq_lens=None, ragged=(128, 32768), batch=64, shuffle_pages=True,
                       desc="B=64, S uniform on [128, 32768] from the seed, shuffled pages, bf16 cache"),
    "b128_s8192_fp8": dict(seq_lens=[8192] * 128, shuffle_pages=True, kv_dtype="fp8_e4m3",
                           desc="B=128, S=8192 each, c_KV e4m3 + fp32 per-token absmax scale, k_R bf16"),
    "b16_s8192_q4": dict(seq_lens=[8192] * 16, shuffle_pages=True, queries_per_seq=4,
                         desc="B=16, S=8192 each, 4 new tokens per sequence decoded at once (causal among them), "
                              "bf16 cache"),
    "prefill_s4096_t1024": dict(seq_lens=[4096], shuffle_pages=True, queries_per_seq=1024, prefill=True,
                                desc="prefill chunk: the last 1,024 tokens of one 4,096-token sequence, causal, "
                                     "decompressed form, bf16 cache"),
    "prefill_s16384_t4096": dict(seq_lens=[16384], shuffle_pages=True, queries_per_seq=4096, prefill=True,
                                 desc="prefill chunk: the last 4,096 tokens of one 16,384-token sequence, causal, "
                                      "decompressed form, bf16 cache"),
}


def make_workload(name: str, *, seed: int = DEFAULT_SEED, poison_tail: bool = False) -> DecodeInputs:
    kw = dict(WORKLOADS[name])
    kw.pop("desc")
    kw.pop("prefill", None)
    return make_inputs(kw.pop("seq_lens"), seed=seed, poison_tail=poison_tail, **kw)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor → its uint16 bit patterns (numpy), for C readers."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
