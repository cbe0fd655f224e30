"""Pins for the CPU oracle: facts fixed by the pages or by mathematics, not by the oracle.

Each ``check_*`` raises AssertionError when the oracle disagrees.  They are plain functions
so that ``test_oracle_pins.py`` can run them against the real oracle and
``test_oracle_mutants.py`` can run them against deliberately broken builds of it.
"""
from __future__ import annotations

import dataclasses
import json
import math
import os

import numpy as np
import torch

import oracle
from mla_latent_kv_absorb_gb300 import synth

SCALE = 1.0 / math.sqrt(synth.D_HC + synth.D_R)
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _cache_rows_f64(inp, b: int) -> tuple:
    """(c [S, 512], k_R [S, 64]) of sequence b in logical order, widened to float64."""
    S = int(inp.seq_lens[b])
    rows_c, rows_r = [], []
    for t in range(S):
        page, slot = int(inp.block_table[b, t // 64]), t % 64
        if inp.kv_dtype == "bf16":
            row = inp.pool[page, slot].to(torch.float64).numpy()
            rows_c.append(row[:512])
            rows_r.append(row[512:])
        else:
            codes = inp.c8[page, slot].numpy()
            deq = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
            rows_c.append(deq * float(inp.kv_scale[page, slot]))
            rows_r.append(inp.kr[page, slot].to(torch.float64).numpy())
    return np.stack(rows_c), np.stack(rows_r)


def _rel(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def tiny_inputs(seq_lens=(1, 65, 130), seed=7, kv_dtype="bf16", poison=True):
    return synth.make_inputs(list(seq_lens), seed=seed, shuffle_pages=True, kv_dtype=kv_dtype,
                             poison_tail=poison)


# ----------------------------------------------------------------------------- element decoding

def check_e4m3_all_codes():
    """All 256 e4m3 codes decode to what torch's float8_e4m3fn (a library routine) gives."""
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan_ours, nan_ref = np.isnan(ours), np.isnan(ref)
    assert (nan_ours == nan_ref).all(), "NaN codes differ"
    assert nan_ref.sum() == 2 and nan_ref[0x7F] and nan_ref[0xFF]
    assert np.array_equal(ours[~nan_ours], ref[~nan_ref]), "e4m3 values differ"
    # values fixed by the format itself
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0          # largest finite
    assert ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6    # smallest subnormal / normal
    assert ours[0x38] == 1.0 and ours[0x00] == 0.0


# ----------------------------------------------------------------------------- naive path closed forms

def check_single_token_is_projected_value(kv_dtype="bf16"):
    """S = 1: the only weight is 1, so out[b,h] = W_UV[h] c_0 exactly (up to fp64 rounding).
    For the fp8 cache c_0 is the stored code decoded by torch (a library routine) times the
    token's scale."""
    inp = synth.make_inputs([1, 1], seed=3, shuffle_pages=True, poison_tail=True, kv_dtype=kv_dtype)
    heads = [0, 5, 127]
    out = oracle.decode_naive(inp, softmax_scale=SCALE, heads=heads)
    wv = _f64(inp.w_uv)
    for b in range(2):
        c, _ = _cache_rows_f64(inp, b)
        for i, h in enumerate(heads):
            ref = wv[h] @ c[0]
            assert np.allclose(out[b, i], ref, rtol=1e-12, atol=1e-13), f"S=1 closed form b={b} h={h}"


def check_single_token_is_projected_value_fp8():
    check_single_token_is_projected_value("fp8_e4m3")


def check_zero_query_gives_mean_value(kv_dtype="bf16"):
    """q_c = q_R = 0: every score is 0, weights are 1/S, out = W_UV[h] mean_t c_t."""
    inp = synth.make_inputs([70, 3], seed=4, shuffle_pages=True, poison_tail=True, kv_dtype=kv_dtype)
    inp.q_c = torch.zeros_like(inp.q_c)
    inp.q_r = torch.zeros_like(inp.q_r)
    heads = [1, 64]
    out = oracle.decode_naive(inp, softmax_scale=SCALE, heads=heads)
    wv = _f64(inp.w_uv)
    for b in range(2):
        c, _ = _cache_rows_f64(inp, b)
        for i, h in enumerate(heads):
            ref = wv[h] @ c.mean(axis=0)
            assert np.allclose(out[b, i], ref, rtol=1e-11, atol=1e-13), f"uniform weights b={b} h={h}"


def check_zero_query_gives_mean_value_fp8():
    check_zero_query_gives_mean_value("fp8_e4m3")


def _constructed(seq_len=5, seed=11):
    """Inputs whose scores are known in closed form.

    W_UK[h] is zero except W_UK[h, d0, c0] = w (d0 != c0 so a swapped d/c index reads a zero);
    q_c[b,h] = alpha e_d0, q_R[b,h] = gamma e_r0, cache row t has c[c0] = beta_t, k_R[r0] = delta_t
    and random values elsewhere in c (which only the value path sees).  Then
    s_t = (alpha w beta_t + gamma delta_t) / sqrt(192) and v_t = W_UV[h] c_t.
    """
    g = torch.Generator().manual_seed(seed)
    inp = synth.make_inputs([seq_len], seed=seed, shuffle_pages=False, poison_tail=True)
    d0, c0, r0 = 3, 200, 17
    w, alpha, gamma = 0.5, 2.0, -1.5
    w_uk = torch.zeros(128, 128, 512)
    w_uk[:, d0, c0] = w
    inp.w_uk = w_uk.to(torch.bfloat16)
    q_c = torch.zeros(1, 128, 128)
    q_c[0, :, d0] = alpha
    inp.q_c = q_c.to(torch.bfloat16)
    q_r = torch.zeros(1, 128, 64)
    q_r[0, :, r0] = gamma
    inp.q_r = q_r.to(torch.bfloat16)
    beta = torch.tensor([4.0, -2.0, 1.0, 3.5, 0.25, -3.0, 2.0, 0.5])[:seq_len]
    delta = torch.tensor([1.0, 2.0, -4.0, 0.5, 3.0, 1.0, -1.0, 2.5])[:seq_len]
    pool = inp.pool.clone()
    for t in range(seq_len):
        page = int(inp.block_table[0, t // 64])
        row = torch.randn(576, generator=g)
        row[512:] = 0.0
        row[c0] = beta[t]
        row[512 + r0] = delta[t]
        pool[page, t % 64] = row.to(torch.bfloat16)
    inp.pool = pool
    s = (alpha * w * beta.double() + gamma * delta.double()) / math.sqrt(192.0)
    return inp, s.numpy()


def check_constructed_scores():
    """Scores built to be known: pins the scale 1/sqrt(d_hc + d_R), the W_UK index order, the
    sign and presence of the RoPE term and the softmax itself."""
    inp, s = _constructed()
    heads = [0, 77]
    out, probs = oracle.decode_naive(inp, softmax_scale=SCALE, heads=heads, want_probs=True)
    S = len(s)
    e = np.exp(s - s.max())
    p_ref = e / e.sum()
    c, _ = _cache_rows_f64(inp, 0)
    wv = _f64(inp.w_uv)
    for i, h in enumerate(heads):
        assert np.allclose(probs[0, i, :S], p_ref, rtol=1e-12, atol=1e-15), "attention weights"
        assert np.all(probs[0, i, S:] == 0.0)
        ref = wv[h] @ (p_ref @ c)
        assert np.allclose(out[0, i], ref, rtol=1e-11, atol=1e-13), "weighted value"


def check_softmax_rows_sum_to_one():
    inp = tiny_inputs((1, 65, 130), seed=5)
    _, probs = oracle.decode_naive(inp, softmax_scale=SCALE, heads=[0, 9, 100], want_probs=True)
    for b, S in enumerate(inp.seq_lens):
        row = probs[b, :, :S]
        assert np.all(row >= 0.0)
        assert np.allclose(row.sum(axis=-1), 1.0, rtol=0, atol=1e-12), "softmax row sum"
        assert np.all(probs[b, :, S:] == 0.0), "weights past S_b"


# ----------------------------------------------------------------------------- absorption identity

def check_absorbed_equals_naive(kv_dtype="bf16"):
    """Page 1 section 4: q_c . (W_UK c) = (W_UK^T q_c) . c, and likewise on the value side, so
    the absorbed path (absorb -> latent attention -> W_UV) equals the naive path up to fp64
    rounding."""
    inp = tiny_inputs((1, 65, 130), seed=6, kv_dtype=kv_dtype)
    heads = list(range(0, 128, 9))
    naive = oracle.decode_naive(inp, softmax_scale=SCALE, heads=heads)
    _, _, _, out = oracle.decode_absorbed(inp, softmax_scale=SCALE)
    got = out[:, heads, :]
    assert _rel(got, naive) < 1e-12, f"absorbed vs naive rel {_rel(got, naive):.3e}"
    assert np.max(np.abs(got - naive)) < 1e-12


def check_absorbed_equals_naive_fp8():
    check_absorbed_equals_naive("fp8_e4m3")


def check_absorb_q_rows():
    """q_abs[b,h] = q_c[b,h] @ W_UK[h] as a matrix-vector product (library routine)."""
    inp = tiny_inputs((3, 3), seed=8)
    q_abs = oracle.absorb_q(inp.q_c, inp.w_uk)
    qc, wk = _f64(inp.q_c), _f64(inp.w_uk)
    for b in range(2):
        for h in (0, 31, 127):
            assert np.allclose(q_abs[b, h], qc[b, h] @ wk[h], rtol=1e-12, atol=1e-14)


def check_out_proj_rows():
    """out[b,h] = W_UV[h] @ o_lat[b,h] as a matrix-vector product (library routine)."""
    inp = tiny_inputs((3, 3), seed=9)
    o = np.random.default_rng(0).standard_normal((2, 128, 512))
    out = oracle.out_proj(o, inp.w_uv)
    wv = _f64(inp.w_uv)
    for b in range(2):
        for h in (0, 64, 127):
            assert np.allclose(out[b, h], wv[h] @ o[b, h], rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------- invariances

def check_page_permutation_invariance():
    """Moving pages to other physical slots (block table updated) changes nothing, bit for bit."""
    a = synth.make_inputs([100, 200], seed=12, shuffle_pages=False, poison_tail=True)
    b = synth.make_inputs([100, 200], seed=12, shuffle_pages=False, poison_tail=True)
    perm = np.random.default_rng(1).permutation(a.num_pool_pages)
    pool = torch.empty_like(a.pool)
    pool[torch.from_numpy(perm)] = a.pool
    b.pool = pool
    b.block_table = np.where(a.block_table >= 0, perm[np.maximum(a.block_table, 0)], -1).astype(np.int32)
    heads = [2, 50]
    na, nb = (oracle.decode_naive(x, softmax_scale=SCALE, heads=heads) for x in (a, b))
    assert np.array_equal(na, nb), "naive path depends on physical placement"
    qa = oracle.absorb_q(a.q_c, a.w_uk)
    oa, la = oracle.latent_attention(a, qa, softmax_scale=SCALE)
    ob, lb = oracle.latent_attention(b, qa, softmax_scale=SCALE)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb), "latent path depends on physical placement"


def check_nan_tail_ignored():
    """Slots past S_b (NaN-poisoned) have no effect: same output as with finite tails."""
    clean = synth.make_inputs([70, 129], seed=13, shuffle_pages=True, poison_tail=False)
    dirty = synth.make_inputs([70, 129], seed=13, shuffle_pages=True, poison_tail=True)
    assert torch.isnan(dirty.pool).any()
    nc = oracle.decode_naive(clean, softmax_scale=SCALE, heads=[0, 127])
    nd = oracle.decode_naive(dirty, softmax_scale=SCALE, heads=[0, 127])
    assert np.isfinite(nd).all() and np.array_equal(nc, nd)


def check_split_combine_invariance(kv_dtype="bf16"):
    """Any partition of a sequence's pages, merged by log-sum-exp, equals the unsplit result."""
    inp = synth.make_inputs([64 * 7 + 5, 64 * 3], seed=14, kv_dtype=kv_dtype, poison_tail=True)
    q = oracle.absorb_q(inp.q_c, inp.w_uk)
    full_o, full_l = oracle.latent_attention(inp, q, softmax_scale=SCALE)
    pages = (inp.seq_lens + 63) // 64
    rng = np.random.default_rng(2)
    for trial in range(3):
        cuts = [sorted(set([0, int(p)] + list(rng.integers(1, max(int(p), 2), size=3)))) for p in pages]
        n = max(len(c) - 1 for c in cuts)
        lse_parts = np.full((n, inp.batch * 128), -np.inf)
        o_parts = np.zeros((n, inp.batch * 128, 512))
        for j in range(n):
            pb = [c[j] if j < len(c) - 1 else c[-1] for c in cuts]
            pe = [c[j + 1] if j < len(c) - 1 else c[-1] for c in cuts]
            o, l = oracle.latent_attention(inp, q, softmax_scale=SCALE, page_begin=pb, page_end=pe)
            lse_parts[j] = l.reshape(-1)
            o_parts[j] = o.reshape(-1, 512)
        lse, o = oracle.lse_combine(lse_parts, o_parts)
        assert np.allclose(lse, full_l.reshape(-1), rtol=0, atol=1e-12), "split lse"
        assert _rel(o, full_o.reshape(-1, 512)) < 1e-12, "split o_lat"


def check_lse_combine_closed_forms():
    rng = np.random.default_rng(3)
    o = rng.standard_normal((4, 512))
    lse = np.array([0.3, -2.0, 5.0, 1.0])
    # two equal parts: lse + ln 2, output unchanged
    l2, o2 = oracle.lse_combine(np.stack([lse, lse]), np.stack([o, o]))
    assert np.allclose(l2, lse + math.log(2.0), atol=1e-15) and np.allclose(o2, o, atol=1e-15)
    # an empty part (lse = -inf) carries no weight
    l3, o3 = oracle.lse_combine(np.stack([lse, np.full(4, -np.inf)]), np.stack([o, 7 * o]))
    assert np.allclose(l3, lse, atol=0) and np.allclose(o3, o, atol=1e-15)
    # weights exp(lse_j - lse) for two different parts
    la, lb = np.zeros(4), np.full(4, math.log(3.0))
    l4, o4 = oracle.lse_combine(np.stack([la, lb]), np.stack([o, -o]))
    assert np.allclose(l4, math.log(4.0), atol=1e-15)
    assert np.allclose(o4, 0.25 * o - 0.75 * o, atol=1e-15)


def check_latent_attention_rows():
    """Latent attention of one row equals softmax(q . C^T * scale) @ C written with numpy."""
    inp = tiny_inputs((130,), seed=15)
    q = oracle.absorb_q(inp.q_c, inp.w_uk)
    o, l = oracle.latent_attention(inp, q, softmax_scale=SCALE, heads=[0, 99])
    c, r = _cache_rows_f64(inp, 0)
    qr = _f64(inp.q_r)
    for i, h in enumerate((0, 99)):
        s = (c @ q[0, h] + r @ qr[0, h]) * SCALE
        m = s.max()
        ref_l = m + math.log(np.exp(s - m).sum())
        assert abs(l[0, i] - ref_l) < 1e-12
        assert _rel(o[0, i], np.exp(s - ref_l) @ c) < 1e-12


# ----------------------------------------------------------------------------- printed figures

def check_cache_geometry_golden():
    """Cache figures printed on the pages, recomputed from the oracle's dimensions."""
    g = json.load(open(os.path.join(GOLDEN, "cache_geometry.json")))
    row = oracle.D_C + oracle.D_R
    assert row == g["row_elements"]["value"]
    row_bytes = row * 2
    assert row_bytes / 1024 == g["row_bytes_bf16_kib"]["value"]
    mha = oracle.NUM_HEADS * oracle.D_HC * 2 * 2
    assert mha / 1024 == g["mha_row_bytes_kib"]["value"]
    assert round(100 * (1 - row_bytes / mha), 2) == g["compression_percent"]["value"]
    assert oracle.PAGE == g["page_tokens"]["value"]
    page_bytes = oracle.PAGE * row_bytes
    assert page_bytes == 73728 and round(page_bytes / 1024) == g["page_bytes_kib_approx"]["value"]
    assert 16 * row_bytes / 1024 == g["page16_bytes_kib"]["value"]
    m = g["mha_cache_tib_64k_b16"]
    assert round(m["context_tokens"] * m["batch"] * m["layers"] * mha / 2 ** 40, 2) == m["value"]
    k = g["h100_kernel_smem_bytes"]
    smem = (k["tile_s"] * oracle.D_C + k["tile_s"] * oracle.D_R) * 2 * k["stages"]
    assert smem == k["value"] and round(smem / 1024) == k["approx_kib"]
    r = g["ridge_flop_per_byte_h100"]
    assert round(r["tflops"] / r["tbps"]) == r["value"]
    k3 = g["mla_kib_per_token_24_layers"]
    assert round(k3["layers"] * row_bytes / 1024, 1) == k3["value"]
    assert abs(g["softmax_scale"]["value"] - 1 / math.sqrt(oracle.D_HC + oracle.D_R)) < 1e-16


# ------------------------------------------------------------------ cache append (write side)

def _e4m3_values(codes: np.ndarray) -> np.ndarray:
    """Values of e4m3 codes through torch's float8_e4m3fn (independent of the oracle's decoder)."""
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def _torch_quantize(c: torch.Tensor):
    """Per-row FP8 cache quantisation through torch: sigma = absmax / 448 in float32 (1 for an
    all-zero row), codes = float8_e4m3fn cast of c / sigma."""
    c = c.to(torch.float32)
    amax = c.abs().amax(dim=-1)
    sigma = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (c / sigma.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.numpy(), sigma.numpy()


def check_e4m3_encode_round_trip():
    """Every finite e4m3 code (both signs, -0 included) encodes back to itself."""
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    got = oracle.e4m3_encode(_e4m3_values(codes).astype(np.float32))
    assert np.array_equal(got, codes), np.nonzero(got != codes)


def check_e4m3_encode_ties_and_neighbours():
    """A value halfway between two adjacent codes goes to the one with the even mantissa field;
    one float step below or above the midpoint goes to the nearer code; magnitudes from 448 up
    give 448; both signs."""
    v = _e4m3_values(np.arange(0x7F))
    lo = np.arange(0x7E)
    hi = lo + 1
    mid64 = (v[lo] + v[hi]) / 2
    mid = mid64.astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), mid64)  # midpoints are exact in float32
    even = np.where(lo % 2 == 0, lo, hi)
    below = np.nextafter(mid, np.float32(0))
    above = np.nextafter(mid, np.float32(np.inf))
    for sgn, sbit in ((1.0, 0x00), (-1.0, 0x80)):
        s32 = np.float32(sgn)
        assert np.array_equal(oracle.e4m3_encode(s32 * mid), (even | sbit).astype(np.uint8))
        assert np.array_equal(oracle.e4m3_encode(s32 * below), (lo | sbit).astype(np.uint8))
        assert np.array_equal(oracle.e4m3_encode(s32 * above), (hi | sbit).astype(np.uint8))
        big = s32 * np.array([448.0, 455.0, 463.99, 464.0, 1e4, 3e38], np.float32)
        assert np.array_equal(oracle.e4m3_encode(big), np.full(big.size, 0x7E | sbit, np.uint8))


def check_e4m3_encode_against_torch():
    """Every finite bf16 value below 464 in magnitude and 200,000 random float32 values spread
    log-uniformly over the e4m3 range (subnormals included) encode as torch's float8_e4m3fn
    cast (round to nearest, ties to even) does."""
    x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 464)]
    g = np.random.default_rng(5)
    mag = np.exp2(g.uniform(-12.0, np.log2(460.0), 200_000)).astype(np.float32)
    sgn = np.where(g.random(mag.size) < 0.5, np.float32(-1), np.float32(1))
    x = np.concatenate([x, mag * sgn])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def _quant_rows() -> torch.Tensor:
    """bf16 latent rows covering the quantiser's cases: N(0,1) at three scales, a negative
    outlier, many values landing among the e4m3 subnormals, exact ties once scaled, and an
    all-zero row holding negative zeros."""
    g = torch.Generator().manual_seed(21)
    rows = [torch.randn(512, generator=g) * s for s in (1.0, 1e-3, 37.0)]
    r = torch.randn(512, generator=g)
    r[17] = -5e3
    rows.append(r)
    r = torch.randn(512, generator=g) * 1e-3
    r[3] = 1.0
    rows.append(r)
    ties = torch.tensor([1.0625, 1.1875, -2.0 ** -10, 3 * 2.0 ** -10, 0.5 + 1 / 32, -(0.75 + 1 / 32)])
    r = ties.repeat(86)[:512].clone()
    r[0] = 448.0  # sigma = 1, so c / sigma = c exactly
    rows.append(r)
    r = torch.zeros(512)
    r[::3] = -0.0
    rows.append(r)
    return torch.stack(rows).to(torch.bfloat16)


def check_quantize_token_rule():
    """Each row's largest magnitude maps to +-448 (code 0x7E / 0xFE); every code is within half
    an e4m3 step of c / sigma; an all-zero row gets sigma 1 and (signed) zero codes; and the
    whole token equals torch's pipeline (absmax / 448 in float32, float8_e4m3fn cast)."""
    rows = _quant_rows()
    ref_codes, ref_sigma = _torch_quantize(rows)
    for i in range(rows.shape[0]):
        codes, sigma = oracle.quantize_token(rows[i])
        assert np.array_equal(codes, ref_codes[i]), (i, np.nonzero(codes != ref_codes[i])[0][:5])
        assert sigma.tobytes() == np.float32(ref_sigma[i]).tobytes(), (i, sigma, ref_sigma[i])
        c = rows[i].to(torch.float32).numpy()
        if not np.any(c != 0):
            assert sigma == np.float32(1.0)
            assert np.array_equal(codes, np.where(np.signbit(c), 0x80, 0x00).astype(np.uint8))
            continue
        k = int(np.argmax(np.abs(c)))
        assert codes[k] == (0xFE if c[k] < 0 else 0x7E)
        q = (c / sigma).astype(np.float64)
        e = np.floor(np.log2(np.maximum(np.abs(q), 2.0 ** -6)))
        assert np.all(np.abs(_e4m3_values(codes) - q) <= np.exp2(e - 4)), i


def check_append_rebuilds_cache():
    """Appending every token of a synthetic bf16 cache (read from its pages in logical order)
    into an empty pool rebuilds the cache bit for bit and leaves unused slots alone; into an
    empty FP8 cache it gives torch's quantisation of the same rows and k_R unchanged.  Negative
    slots are skipped; a slot past the pool is skipped and reported."""
    inp = tiny_inputs(seq_lens=(1, 65, 130), seed=9, poison=False)
    pool = inp.pool.contiguous().view(torch.int16).numpy().view(np.uint16)
    N = inp.num_pool_pages
    slots, rows = [], []
    for b in range(inp.batch):
        for t in range(int(inp.seq_lens[b])):
            page, row = int(inp.block_table[b, t // 64]), t % 64
            slots.append(page * 64 + row)
            rows.append(pool[page, row])
    slots = np.array(slots, np.int32)
    rows = np.stack(rows)
    c_kv, k_r = np.ascontiguousarray(rows[:, :512]), np.ascontiguousarray(rows[:, 512:])
    empty = np.full((N, 64, 576), 0xFFFF, np.uint16)
    assert oracle.append_kv(c_kv, k_r, slots, {"pool": empty}) == 0
    used = np.zeros(N * 64, bool)
    used[slots] = True
    flat_new, flat_old = empty.reshape(N * 64, 576), pool.reshape(N * 64, 576)
    assert np.array_equal(flat_new[used], flat_old[used])
    assert np.all(flat_new[~used] == 0xFFFF)

    fp8 = {"c8": np.full((N, 64, 512), 0x7F, np.uint8), "scale": np.full((N, 64), np.nan, np.float32),
           "kr": np.full((N, 64, 64), 0xFFFF, np.uint16)}
    assert oracle.append_kv(c_kv, k_r, slots, fp8) == 0
    ref_codes, ref_sigma = _torch_quantize(torch.from_numpy(c_kv.view(np.int16)).view(torch.bfloat16))
    assert np.array_equal(fp8["c8"].reshape(N * 64, 512)[slots], ref_codes)
    assert np.array_equal(fp8["scale"].reshape(N * 64)[slots].view(np.uint32), ref_sigma.view(np.uint32))
    assert np.array_equal(fp8["kr"].reshape(N * 64, 64)[slots], k_r)
    assert np.all(fp8["c8"].reshape(N * 64, 512)[~used] == 0x7F)

    cache = {"pool": np.full((N, 64, 576), 0xFFFF, np.uint16)}
    assert oracle.append_kv(c_kv[:3], k_r[:3], np.array([-1, N * 64, 5], np.int32), cache) == -1
    flat = cache["pool"].reshape(N * 64, 576)
    assert np.array_equal(flat[5], rows[2])
    assert np.all(np.delete(flat, 5, axis=0) == 0xFFFF)


ALL_CHECKS = [
    check_e4m3_all_codes,
    check_single_token_is_projected_value,
    check_single_token_is_projected_value_fp8,
    check_zero_query_gives_mean_value,
    check_zero_query_gives_mean_value_fp8,
    check_constructed_scores,
    check_softmax_rows_sum_to_one,
    check_absorbed_equals_naive,
    check_absorbed_equals_naive_fp8,
    check_absorb_q_rows,
    check_out_proj_rows,
    check_page_permutation_invariance,
    check_nan_tail_ignored,
    check_split_combine_invariance,
    check_lse_combine_closed_forms,
    check_latent_attention_rows,
    check_cache_geometry_golden,
    check_e4m3_encode_round_trip,
    check_e4m3_encode_ties_and_neighbours,
    check_e4m3_encode_against_torch,
    check_quantize_token_rule,
    check_append_rebuilds_cache,
]


# ----------------------------------------------------------------------------- NVFP4 cache (e2m1 + e4m3 block scales)

# e2m1 values straight from the format (sign, 2 exponent bits with bias 1, 1 mantissa bit;
# exponent field 0 subnormal): codes 0..7 and their negatives 8..15.
E2M1_TABLE = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def check_e2m1_values():
    """The sixteen e2m1 codes decode to the format's values, -0 included."""
    got = oracle.e2m1_value(np.arange(16, dtype=np.uint8))
    assert np.array_equal(got, E2M1_TABLE)
    assert np.signbit(got[8]) and not np.signbit(got[0])


def _nearest_ok(codes: np.ndarray, x: np.ndarray) -> np.ndarray:
    """For each x, is the code's value at least as near as every e2m1 value (after clamping the
    magnitude to 6)?"""
    vals = E2M1_TABLE[codes & 0xF]
    xc = np.clip(x.astype(np.float64), -6.0, 6.0)
    best = np.min(np.abs(xc[:, None] - E2M1_TABLE[None, :8] * np.where(xc < 0, -1.0, 1.0)[:, None]), axis=1)
    return np.abs(vals - xc) <= best + 0.0


def check_e2m1_encode_rule():
    """Every code round-trips (both signs, -0 -> 0x8); midpoints go to the even mantissa field;
    one float32 step either side goes to the nearer value; magnitudes >= 6 give 6; and 100,000
    random values get a nearest code."""
    for c in range(16):
        assert int(oracle.e2m1_encode(np.array([E2M1_TABLE[c]], np.float32))[0]) == c, c
    mids = {0.25: 0x0, 0.75: 0x2, 1.25: 0x2, 1.75: 0x4, 2.5: 0x4, 3.5: 0x6, 5.0: 0x6}
    for m, code in mids.items():
        assert int(oracle.e2m1_encode(np.array([m], np.float32))[0]) == code, m
        assert int(oracle.e2m1_encode(np.array([-m], np.float32))[0]) == (code | 0x8), -m
        up, down = np.nextafter(np.float32(m), np.float32(10)), np.nextafter(np.float32(m), np.float32(-10))
        hi_code = int(np.searchsorted(E2M1_TABLE[:8], m))
        assert int(oracle.e2m1_encode(np.array([up], np.float32))[0]) == hi_code, m
        assert int(oracle.e2m1_encode(np.array([down], np.float32))[0]) == hi_code - 1, m
    big = np.array([6.0, 6.5, 7.0, 1e30, -6.0, -1e30], np.float32)
    assert np.array_equal(oracle.e2m1_encode(big), np.array([7, 7, 7, 7, 15, 15], np.uint8))
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(100000) * 3).astype(np.float32)
    codes = oracle.e2m1_encode(x)
    assert _nearest_ok(codes, x).all()
    assert np.array_equal(codes >= 8, np.signbit(x))


def _bf16_rows(rows: np.ndarray) -> np.ndarray:
    """float32 rows rounded to bf16, as uint16 bit patterns."""
    return torch.from_numpy(np.ascontiguousarray(rows, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def _nvfp4_deq(row: np.ndarray, sigma: float) -> np.ndarray:
    """Values of one NVFP4 row through the format table and torch's e4m3 (library), not the oracle."""
    codes = np.empty(512, np.uint8)
    codes[0::2] = row[:256] & 0xF
    codes[1::2] = row[:256] >> 4
    scales = _e4m3_values(row[256:288])
    return E2M1_TABLE[codes] * np.repeat(scales, 16) * float(sigma)


def check_nvfp4_quantize_rule():
    """sigma = absmax / 2688 (float32; 1 for a zero row); block scale = e4m3 nearest to
    ((block absmax / sigma) / 6) (torch's e4m3 cast); the token's largest value maps to code 6 in a
    block of scale 448; every code is the nearest e2m1 to x / (sigma S_b) (float32); value 2j sits
    in the low nibble of byte j; zero rows and zero blocks give zero codes and scales."""
    rng = np.random.default_rng(11)
    rows = [rng.standard_normal(512) * s for s in (1.0, 0.01, 300.0)]
    r = rng.standard_normal(512)
    r[64:96] = 0.0  # two zero blocks
    rows.append(r)
    rows.append(np.zeros(512))
    one = np.zeros(512)
    one[0] = 2.0
    rows.append(one)
    two = np.zeros(512)
    two[1] = -3.0
    rows.append(two)
    bits = _bf16_rows(np.stack(rows))
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    for i in range(bits.shape[0]):
        row, sigma = oracle.quantize_token_nvfp4(bits[i])
        c = vals[i]
        amax = np.float32(np.abs(c).max())
        want_sigma = np.float32(amax / np.float32(2688.0)) if amax > 0 else np.float32(1.0)
        assert sigma == want_sigma, i
        bmax = np.abs(c).reshape(32, 16).max(axis=1).astype(np.float32)
        t = ((bmax / sigma).astype(np.float32) / np.float32(6.0)).astype(np.float32)
        want_scales = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(row[256:288], want_scales), i
        S = _e4m3_values(row[256:288])
        codes = np.empty(512, np.uint8)
        codes[0::2] = row[:256] & 0xF
        codes[1::2] = row[:256] >> 4
        den = (sigma * np.repeat(S, 16).astype(np.float32)).astype(np.float32)
        live = den > 0
        q = np.where(live, c / np.where(live, den, 1), 0).astype(np.float32)
        assert _nearest_ok(codes[live], q[live]).all(), i
        assert np.all(E2M1_TABLE[codes[~live]] == 0), i
        if amax > 0:
            k = int(np.argmax(np.abs(c)))
            assert S[k // 16] == 448.0 and abs(E2M1_TABLE[codes[k]]) == 6.0, i
    row, sigma = oracle.quantize_token_nvfp4(bits[4])
    assert sigma == 1.0 and not row.any()
    row, _ = oracle.quantize_token_nvfp4(bits[5])
    assert row[0] == 0x07 and not row[1:256].any()        # value 0 in the low nibble
    row, _ = oracle.quantize_token_nvfp4(bits[6])
    assert row[0] == 0xF0 and not row[1:256].any()        # value 1 (negative) in the high nibble


def nvfp4_inputs(seq_lens=(1, 65, 130), seed=7, poison=True):
    """A synthetic decode batch whose cache is NVFP4: the bf16 cache's rows appended, through the
    oracle's quantiser, into the same page layout (k_R kept in bf16)."""
    inp = tiny_inputs(seq_lens, seed=seed, poison=poison)
    pool = inp.pool.contiguous().view(torch.int16).numpy().view(np.uint16)
    N = inp.num_pool_pages
    flat = pool.reshape(N * 64, 576)
    slots = np.arange(N * 64, dtype=np.int32)
    c_kv = np.ascontiguousarray(np.nan_to_num(flat[:, :512].view(np.int16)).view(np.uint16))
    finite = np.isfinite(torch.from_numpy(flat[:, :512].view(np.int16)).view(torch.bfloat16).float().numpy()).all(1)
    slots = np.where(finite, slots, -1).astype(np.int32)
    cache = {"c4": np.zeros((N, 64, 288), np.uint8), "scale": np.ones((N, 64), np.float32),
             "kr": np.ascontiguousarray(pool[:, :, 512:])}
    assert oracle.append_kv(c_kv, np.ascontiguousarray(flat[:, 512:]), slots, cache) == 0
    if poison:  # slots that were poisoned stay poisoned: NaN scales and k_R
        cache["scale"].reshape(-1)[~finite] = np.nan
    inp.kv_dtype = "nvfp4"
    inp.c8 = torch.from_numpy(cache["c4"])
    inp.kv_scale = torch.from_numpy(cache["scale"])
    inp.kr = torch.from_numpy(cache["kr"].view(np.int16)).view(torch.bfloat16)
    inp.pool = None
    return inp


def _nvfp4_rows_f64(inp, b: int) -> tuple:
    S = int(inp.seq_lens[b])
    cs, rs = [], []
    for t in range(S):
        page, slot = int(inp.block_table[b, t // 64]), t % 64
        cs.append(_nvfp4_deq(inp.c8[page, slot].numpy(), float(inp.kv_scale[page, slot])))
        rs.append(inp.kr[page, slot].to(torch.float64).numpy())
    return np.stack(cs), np.stack(rs)


def check_nvfp4_cache_closed_forms():
    """With an NVFP4 cache (values through the format table and torch's e4m3): S = 1 gives
    W_UV[h] c_0, zero queries give W_UV[h] mean(c), and the absorbed path equals the naive one."""
    inp = nvfp4_inputs((1, 1), seed=21)
    heads = [0, 7, 127]
    out = oracle.decode_naive(inp, softmax_scale=SCALE, heads=heads)
    wv = _f64(inp.w_uv)
    for b in range(2):
        c, _ = _nvfp4_rows_f64(inp, b)
        for i, h in enumerate(heads):
            assert np.allclose(out[b, i], wv[h] @ c[0], rtol=1e-12, atol=1e-13), (b, h)
    inp = nvfp4_inputs((70, 3), seed=22)
    inp.q_c = torch.zeros_like(inp.q_c)
    inp.q_r = torch.zeros_like(inp.q_r)
    out = oracle.decode_naive(inp, softmax_scale=SCALE, heads=heads)
    wv = _f64(inp.w_uv)
    for b in range(2):
        c, _ = _nvfp4_rows_f64(inp, b)
        for i, h in enumerate(heads):
            assert np.allclose(out[b, i], wv[h] @ c.mean(axis=0), rtol=1e-11, atol=1e-13), (b, h)
    inp = nvfp4_inputs((1, 65, 130), seed=23)
    hs = list(range(0, 128, 9))
    naive = oracle.decode_naive(inp, softmax_scale=SCALE, heads=hs)
    _, _, _, absorbed = oracle.decode_absorbed(inp, softmax_scale=SCALE)
    assert _rel(absorbed[:, hs, :], naive) < 1e-12


ALL_CHECKS += [check_e2m1_values, check_e2m1_encode_rule, check_nvfp4_quantize_rule, check_nvfp4_cache_closed_forms]


def _bf16_bits_of_f32(x: np.ndarray) -> np.ndarray:
    """bf16 nearest to float32 values (torch's conversion: ties to even), as uint16 bits."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def check_gather_kv():
    """The gathered rows, in logical order: the stored bits of a bf16 cache; for FP8,
    bf16(float32(e4m3 value) * sigma); for NVFP4, bf16(float32(e2m1 value * e4m3 block scale) *
    sigma), each value formed with torch's e4m3 decoding and conversions (library routines) and
    numpy float32 products; k_R copied; row offsets the cumulative lengths."""
    for kind in ("bf16", "fp8_e4m3", "nvfp4"):
        inp = nvfp4_inputs((3, 64, 130), seed=31) if kind == "nvfp4" else tiny_inputs((3, 64, 130), seed=31,
                                                                                       kv_dtype=kind)
        out, cu = oracle.gather_kv(inp)
        assert list(cu) == [0, 3, 67, 197]
        for b in range(inp.batch):
            for t in range(int(inp.seq_lens[b])):
                page, slot = int(inp.block_table[b, t // 64]), t % 64
                got = out[cu[b] + t]
                if kind == "bf16":
                    want = inp.pool[page, slot].contiguous().view(torch.int16).numpy().view(np.uint16)
                    assert np.array_equal(got, want), (kind, b, t)
                    continue
                sigma = np.float32(inp.kv_scale[page, slot])
                if kind == "fp8_e4m3":
                    vals = _e4m3_values(inp.c8[page, slot].numpy()).astype(np.float32)
                else:
                    row = inp.c8[page, slot].numpy()
                    codes = np.empty(512, np.uint8)
                    codes[0::2] = row[:256] & 0xF
                    codes[1::2] = row[:256] >> 4
                    vals = (E2M1_TABLE[codes].astype(np.float32) *
                            np.repeat(_e4m3_values(row[256:288]).astype(np.float32), 16)).astype(np.float32)
                want = _bf16_bits_of_f32((vals * sigma).astype(np.float32))
                assert np.array_equal(got[:512], want), (kind, b, t)
                assert np.array_equal(got[512:], inp.kr[page, slot].contiguous().view(torch.int16).numpy().view(
                    np.uint16)), (kind, b, t)


ALL_CHECKS += [check_gather_kv]


# ----------------------------------------------------------------------------- several new tokens per sequence

def mq_inputs(seq_lens=(5, 70, 131), q=3, seed=41):
    """A tiny bf16 cache with q query rows per sequence (row b*q + t: new token t of sequence b)."""
    inp = tiny_inputs(seq_lens, seed=seed, poison=True)
    g = torch.Generator().manual_seed(seed + 1)
    rows = inp.batch * q
    inp.q_c = torch.randn(rows, synth.NUM_HEADS, synth.D_HC, generator=g).to(torch.bfloat16)
    inp.q_r = torch.randn(rows, synth.NUM_HEADS, synth.D_R, generator=g).to(torch.bfloat16)
    return inp


def check_multi_query_single_token_is_decode():
    """q = 1: the query rows are the sequences themselves, and the step is the ordinary decode."""
    inp = tiny_inputs((5, 70, 131), seed=42)
    rows = oracle.query_row_inputs(inp, 1)
    assert np.array_equal(rows.seq_lens, inp.seq_lens) and np.array_equal(rows.block_table, inp.block_table)
    heads = np.array([0, 77])
    assert np.array_equal(oracle.decode_naive(rows, softmax_scale=SCALE, heads=heads),
                          oracle.decode_naive(inp, softmax_scale=SCALE, heads=heads))


def check_multi_query_rows_are_prefix_decodes():
    """Query row b*q + t is an ordinary decode of sequence b cut to its first S_b - q + 1 + t
    tokens, with that row's query: built here by slicing the inputs by hand, one sequence at a
    time.  Pins the row order, the causal lengths and the block-table row of each query."""
    q = 3
    inp = mq_inputs(q=q)
    heads = np.array([0, 77])
    got = oracle.decode_naive(oracle.query_row_inputs(inp, q), softmax_scale=SCALE, heads=heads)
    for b in range(inp.batch):
        for t in range(q):
            r = b * q + t
            one = dataclasses.replace(inp, seq_lens=np.array([int(inp.seq_lens[b]) - q + 1 + t], np.int32),
                                      block_table=np.ascontiguousarray(inp.block_table[b:b + 1]),
                                      q_c=inp.q_c[r:r + 1], q_r=inp.q_r[r:r + 1])
            want = oracle.decode_naive(one, softmax_scale=SCALE, heads=heads)
            assert np.array_equal(got[r], want[0]), (b, t)


def check_multi_query_is_causal():
    """A new token does not see the new tokens after it: changing the cache row of new token
    t' leaves the outputs of tokens t < t' bit for bit and changes those of t >= t'."""
    q = 3
    inp = mq_inputs(q=q)
    heads = np.array([5])
    base = oracle.decode_naive(oracle.query_row_inputs(inp, q), softmax_scale=SCALE, heads=heads)
    g = torch.Generator().manual_seed(3)
    for b in range(inp.batch):
        for tp in range(q):
            pos = int(inp.seq_lens[b]) - q + tp  # the cache position of new token tp
            page, slot = int(inp.block_table[b, pos // 64]), pos % 64
            mod = dataclasses.replace(inp, pool=inp.pool.clone())
            mod.pool[page, slot] = (4 * torch.randn(576, generator=g)).to(torch.bfloat16)
            out = oracle.decode_naive(oracle.query_row_inputs(mod, q), softmax_scale=SCALE, heads=heads)
            for t in range(q):
                same = np.array_equal(out[b * q + t], base[b * q + t])
                assert same == (t < tp), (b, tp, t)
            others = [r for r in range(inp.batch * q) if r // q != b]
            assert np.array_equal(out[others], base[others])


ALL_CHECKS += [check_multi_query_single_token_is_decode, check_multi_query_rows_are_prefix_decodes,
               check_multi_query_is_causal]
