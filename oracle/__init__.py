"""CPU oracle for MLA latent-KV decode -- TEST INFRASTRUCTURE ONLY.

A plain, slow fp64 statement of what the decode step computes (``mla_oracle.c``), loaded
through ctypes.  Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
use it.  The CUDA library never imports, links or calls anything here, and the two share no
code: the only common module is the seeded input generator, which holds no attention math.

Parity status of each function (what pins it, see ``tests/test_oracle_pins.py``):
  e4m3 decode         -- all 256 codes against torch's float8_e4m3fn, plus printed values.
  decode_naive        -- closed forms (S = 1, uniform weights, constructed scores), softmax
                         rows summing to 1, permutation/NaN-tail invariance.
  absorb_q, latent_attention, out_proj
                      -- the absorption identity against decode_naive (page 1 section 4),
                         single-row closed forms.
  lse_combine         -- split-partition invariance against an unsplit latent_attention and
                         equal-weight closed form.
  e4m3_encode, quantize_token, append_kv
                      -- every finite code round-trips, midpoints go to the even code, a sweep
                         against torch's float8_e4m3fn cast, the half-step error bound, the
                         all-zero row; appending every token of a synthetic cache rebuilds it.
  e2m1_value, e2m1_encode, quantize_token_nvfp4 (and the NVFP4 cache in every decode function)
                      -- the sixteen e2m1 values of the format; round trips, midpoints to the
                         even code, saturation; the token's largest value maps to code 6 under
                         block scale 448; every code nearest to its scaled value; zero rows and
                         zero blocks; S = 1 and q = 0 closed forms and absorbed = naive on an
                         NVFP4 cache built by append_kv.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libmla_oracle.so")

NUM_HEADS, D_HC, D_C, D_R, D_ROW, PAGE = 128, 128, 512, 64, 576, 64
NV_ROW = D_C // 2 + D_C // 16  # NVFP4 row of one token: packed e2m1 codes, then e4m3 block scales

_lib = None


def build(force: bool = False, src: Optional[str] = None, out: Optional[str] = None) -> str:
    """Compile the oracle with gcc (OpenMP if the toolchain has it). Returns the .so path."""
    src = src or _SRC
    out = out or _LIB_PATH
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-fno-fast-math", "-ffp-contract=off", src, "-o", out, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    return out


def _load(path: str):
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    L.oracle_e4m3_value.restype = f64
    L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_decode.argtypes = [P, i64, P]
    L.oracle_set_threads.argtypes = [i32]
    L.oracle_max_threads.restype = i32
    L.oracle_decode_naive.restype = i32
    L.oracle_decode_naive.argtypes = [i32, P, P, i32, i32, i32, P, P, P, P, P, P, P, P, f64, i32, P, P, P]
    L.oracle_absorb_q.argtypes = [i32, P, P, P]
    L.oracle_latent_attention.restype = i32
    L.oracle_latent_attention.argtypes = [i32, P, P, P, P, i32, P, P, i32, i32, P, P, P, P, f64, i32, P, P, P]
    L.oracle_out_proj.argtypes = [i32, P, P, P]
    L.oracle_lse_combine.argtypes = [i32, i32, P, P, P, P]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_encode_many.argtypes = [P, i64, P]
    L.oracle_quantize_token.restype = ctypes.c_float
    L.oracle_quantize_token.argtypes = [P, P]
    L.oracle_e2m1_value.restype = f64
    L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
    L.oracle_e2m1_encode.restype = ctypes.c_uint8
    L.oracle_e2m1_encode.argtypes = [ctypes.c_float]
    L.oracle_e2m1_encode_many.argtypes = [P, i64, P]
    L.oracle_quantize_token_nvfp4.restype = ctypes.c_float
    L.oracle_quantize_token_nvfp4.argtypes = [P, P]
    L.oracle_gather_kv.restype = i32
    L.oracle_gather_kv.argtypes = [i32, P, P, i32, P, i32, i32, P, P, P, P, P]
    L.oracle_append_kv.restype = i32
    L.oracle_append_kv.argtypes = [i32, P, P, P, i32, i32, P, P, P, P]
    L.oracle_query_rows.restype = ctypes.c_int
    L.oracle_query_rows.argtypes = [i32, i32, P, P, P]
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _load(build())
    return _lib


def _use_library(path: Optional[str]) -> None:
    """Swap in another build of the oracle (the mutation tests load broken copies)."""
    global _lib
    _lib = None if path is None else _load(path)


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(t) -> np.ndarray:
    """bf16 torch tensor (or uint16 array) → contiguous uint16 bit patterns."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _arr(t, dtype) -> np.ndarray:
    if t is None:
        return None
    if not isinstance(t, np.ndarray):
        t = t.contiguous().numpy()
    return np.ascontiguousarray(t, dtype=dtype)


class _Cache:
    """The paged cache of a ``synth.DecodeInputs`` as C arrays."""

    def __init__(self, inp):
        self.kv_fp8 = {"bf16": 0, "fp8_e4m3": 1, "nvfp4": 2}[inp.kv_dtype]
        self.num_pages = int(inp.num_pool_pages)
        self.pool = _u16(inp.pool) if inp.pool is not None else None
        self.c8 = _arr(inp.c8, np.uint8) if inp.c8 is not None else None
        self.scale = _arr(inp.kv_scale, np.float32) if inp.kv_scale is not None else None
        self.kr = _u16(inp.kr) if inp.kr is not None else None

    def args(self):
        return [self.kv_fp8, self.num_pages, _p(self.pool), _p(self.c8), _p(self.scale), _p(self.kr)]


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib().oracle_e4m3_decode(_p(codes), codes.size, _p(out))
    return out


def _heads(heads: Optional[Sequence[int]]) -> np.ndarray:
    h = np.arange(NUM_HEADS, dtype=np.int32) if heads is None else np.asarray(heads, dtype=np.int32)
    assert h.ndim == 1 and h.size > 0 and (h >= 0).all() and (h < NUM_HEADS).all()
    return np.ascontiguousarray(h)


def decode_naive(inp, *, softmax_scale: float, heads=None, want_probs: bool = False):
    """Decompressed-path decode. Returns out [B, n_heads, 128] (and probs if asked)."""
    hs = _heads(heads)
    B = inp.batch
    out = np.empty((B, hs.size, D_HC), dtype=np.float64)
    probs = np.empty((B, hs.size, inp.max_pages * PAGE), dtype=np.float64) if want_probs else None
    sl = _arr(inp.seq_lens, np.int32)
    bt = _arr(inp.block_table, np.int32)
    qc, qr, wk, wv = _u16(inp.q_c), _u16(inp.q_r), _u16(inp.w_uk), _u16(inp.w_uv)
    rc = lib().oracle_decode_naive(B, _p(sl), _p(bt), inp.max_pages, *_Cache(inp).args(),
                                   _p(qc), _p(qr), _p(wk), _p(wv), float(softmax_scale),
                                   hs.size, _p(hs), _p(out), _p(probs))
    if rc != 0:
        raise ValueError("block table entry out of range")
    return (out, probs) if want_probs else out


def absorb_q(q_c, w_uk) -> np.ndarray:
    """q_abs [B, 128, 512] in float64."""
    qc, wk = _u16(q_c), _u16(w_uk)
    B = qc.shape[0]
    out = np.empty((B, NUM_HEADS, D_C), dtype=np.float64)
    lib().oracle_absorb_q(B, _p(qc), _p(wk), _p(out))
    return out


def latent_attention(inp, q_lat: np.ndarray, *, softmax_scale: float, heads=None,
                     page_begin=None, page_end=None):
    """Latent-space attention over a page range of each sequence. Returns (o_lat, lse)."""
    hs = _heads(heads)
    B = inp.batch
    q_lat = np.ascontiguousarray(q_lat, dtype=np.float64)
    assert q_lat.shape == (B, NUM_HEADS, D_C)
    pages = (inp.seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    pb = np.zeros(B, np.int32) if page_begin is None else np.asarray(page_begin, np.int32)
    pe = pages.astype(np.int32) if page_end is None else np.asarray(page_end, np.int32)
    o = np.empty((B, hs.size, D_C), dtype=np.float64)
    lse = np.empty((B, hs.size), dtype=np.float64)
    sl = _arr(inp.seq_lens, np.int32)
    bt = _arr(inp.block_table, np.int32)
    qr = _u16(inp.q_r)
    rc = lib().oracle_latent_attention(B, _p(q_lat), _p(qr), _p(sl), _p(bt), inp.max_pages,
                                       _p(np.ascontiguousarray(pb)), _p(np.ascontiguousarray(pe)),
                                       *_Cache(inp).args(), float(softmax_scale), hs.size, _p(hs),
                                       _p(o), _p(lse))
    if rc != 0:
        raise ValueError("block table entry out of range")
    return o, lse


def out_proj(o_lat: np.ndarray, w_uv) -> np.ndarray:
    """out [B, 128, 128] from o_lat [B, 128, 512] (float64) and W_UV (bf16)."""
    o_lat = np.ascontiguousarray(o_lat, dtype=np.float64)
    B = o_lat.shape[0]
    assert o_lat.shape == (B, NUM_HEADS, D_C)
    wv = _u16(w_uv)
    out = np.empty((B, NUM_HEADS, D_HC), dtype=np.float64)
    lib().oracle_out_proj(B, _p(o_lat), _p(wv), _p(out))
    return out


def lse_combine(lse_parts: np.ndarray, o_parts: np.ndarray):
    """Merge n partial results: lse_parts [n, rows], o_parts [n, rows, 512]."""
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    n, rows = lse_parts.shape
    assert o_parts.shape == (n, rows, D_C)
    lse = np.empty(rows, dtype=np.float64)
    o = np.empty((rows, D_C), dtype=np.float64)
    lib().oracle_lse_combine(rows, n, _p(lse_parts), _p(o_parts), _p(lse), _p(o))
    return lse, o


def decode_absorbed(inp, *, softmax_scale: float):
    """Absorbed path end to end in fp64: (q_abs, o_lat, lse, out)."""
    q_abs = absorb_q(inp.q_c, inp.w_uk)
    o_lat, lse = latent_attention(inp, q_abs, softmax_scale=softmax_scale)
    out = out_proj(o_lat, inp.w_uv)
    return q_abs, o_lat, lse, out


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 codes (uint8) of float32 values, ties to even, clamped to +-448."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_many(_p(x), x.size, _p(out))
    return out


def e2m1_value(codes) -> np.ndarray:
    """Values of e2m1 codes (the low 4 bits of each uint8)."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    return np.array([lib().oracle_e2m1_value(int(c)) for c in codes.reshape(-1)], dtype=np.float64).reshape(codes.shape)


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """Nearest e2m1 codes (uint8, low 4 bits) of float32 values, ties to even, clamped to +-6."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e2m1_encode_many(_p(x), x.size, _p(out))
    return out


def quantize_token_nvfp4(c) -> tuple:
    """One token's 512 bf16 latent values -> (NVFP4 row uint8 [288]: 256 bytes of packed e2m1
    codes then 32 e4m3 block scales, sigma float32)."""
    c = _u16(c).reshape(-1)
    assert c.size == D_C
    row = np.zeros(NV_ROW, dtype=np.uint8)
    sigma = lib().oracle_quantize_token_nvfp4(_p(c), _p(row))
    return row, np.float32(sigma)


def quantize_token(c) -> tuple:
    """One token's 512 bf16 latent values -> (codes uint8 [512], sigma float32)."""
    c = _u16(c).reshape(-1)
    assert c.size == D_C
    codes = np.empty(D_C, dtype=np.uint8)
    sigma = lib().oracle_quantize_token(_p(c), _p(codes))
    return codes, np.float32(sigma)


def gather_kv(inp) -> tuple:
    """Every sequence's cache rows, in logical order, as one contiguous bf16 array (uint16 bits)
    [total tokens, 576], with the row offsets cu_seqlens [B + 1]: the stored bits of a bf16 cache;
    for FP8 and NVFP4 caches each latent value formed in fp32 (code times scales, one rounding)
    and rounded to bf16."""
    sl = _arr(inp.seq_lens, np.int32)
    cu = np.zeros(inp.batch + 1, np.int32)
    cu[1:] = np.cumsum(sl)
    out = np.zeros((int(cu[-1]), D_ROW), np.uint16)
    bt = _arr(inp.block_table, np.int32)
    rc = lib().oracle_gather_kv(inp.batch, _p(sl), _p(bt), inp.max_pages, _p(cu), *_Cache(inp).args(), _p(out))
    if rc != 0:
        raise ValueError("block table entry out of range")
    return out, cu


def append_kv(c_kv, k_r, slots, cache: dict) -> int:
    """Write tokens into a paged cache held as numpy arrays, in place.

    c_kv bf16 [n, 512], k_r bf16 [n, 64], slots int32 [n] (page * 64 + row; negative = skip).
    cache: {"pool": uint16 [N, 64, 576]} for a bf16 cache, {"c8": uint8 [N, 64, 512],
    "scale": float32 [N, 64], "kr": uint16 [N, 64, 64]} for FP8, or {"c4": uint8 [N, 64, 288],
    "scale", "kr"} for NVFP4.  Returns 0, or -1 when a slot was past the pool (that token
    skipped)."""
    ck, kr = _u16(c_kv), _u16(k_r)
    sl = np.ascontiguousarray(slots, dtype=np.int32)
    n = sl.size
    assert ck.shape == (n, D_C) and kr.shape == (n, D_R)
    mode = 2 if "c4" in cache else (1 if "c8" in cache else 0)
    codes = cache.get("c4") if mode == 2 else cache.get("c8")
    arrays = [cache.get("pool"), codes, cache.get("scale"), cache.get("kr")]
    for a in arrays:
        assert a is None or (isinstance(a, np.ndarray) and a.flags.c_contiguous)
    num_pages = (codes if mode else cache["pool"]).shape[0]
    return int(lib().oracle_append_kv(n, _p(ck), _p(kr), _p(sl), mode, num_pages, *[_p(a) for a in arrays]))


def query_rows(seq_lens, q: int):
    """Several new tokens per sequence (oracle_query_rows): (row_len, row_table) for the
    B * q query rows, row b*q + t being new token t of sequence b."""
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    B = int(sl.size)
    row_len = np.empty(B * q, dtype=np.int32)
    row_table = np.empty(B * q, dtype=np.int32)
    if lib().oracle_query_rows(B, int(q), _p(sl), _p(row_len), _p(row_table)) != 0:
        raise ValueError("every sequence needs at least q tokens (and q >= 1)")
    return row_len, row_table


def query_row_inputs(inp, q: int):
    """The inputs of a q-tokens-per-sequence step as B * q ordinary decode queries: inp.q_c and
    inp.q_r already hold B * q rows; each query row gets its visible length and its sequence's
    block-table row.  Every oracle function then applies unchanged."""
    row_len, row_table = query_rows(inp.seq_lens, q)
    if int(inp.q_c.shape[0]) != row_len.size or int(inp.q_r.shape[0]) != row_len.size:
        raise ValueError("q_c and q_r need B * q rows")
    return dataclasses.replace(inp, seq_lens=row_len,
                               block_table=np.ascontiguousarray(np.asarray(inp.block_table)[row_table]))
