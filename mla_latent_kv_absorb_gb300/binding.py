"""ctypes binding of libmla_gb300.so: the C ABI of include/mla.h under the same names.

Argument marshalling only: torch tensors supply device memory and streams, every step of the
decode runs in the library's CUDA kernels.  If the library has not been built this module
raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import numpy as np
import torch

from . import D_C, D_HC, D_R, D_ROW, NUM_HEADS, PAGE

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla_gb300.so")

# mla_status
MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_ALIGNMENT, MLA_ERR_UNSUPPORTED = 0, 1, 2, 3
MLA_ERR_WORKSPACE, MLA_ERR_CUDA, MLA_ERR_DEVICE_FAULT = 4, 5, 6
# mla_kv_dtype
MLA_KV_BF16, MLA_KV_FP8_E4M3, MLA_KV_NVFP4 = 0, 1, 2
NVFP4_ROW = D_C // 2 + D_C // 16  # bytes of one token's NVFP4 row: packed e2m1 codes, then e4m3 block scales
# device error bits
MLA_DEVERR_BAD_PAGE, MLA_DEVERR_TIMEOUT, MLA_DEVERR_SMEM_ALIGN, MLA_DEVERR_BAD_PLAN = 1, 2, 4, 8

SOFTMAX_SCALE = 1.0 / math.sqrt(D_HC + D_R)


class MlaError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


class PlanOptions(ctypes.Structure):
    _fields_ = [("min_pages_per_split", ctypes.c_int32), ("max_clusters", ctypes.c_int32),
                ("wait_timeout_ns", ctypes.c_int64), ("item_cost_pages", ctypes.c_int32),
                ("queries_per_seq", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_clusters", ctypes.c_int32), ("num_items", ctypes.c_int32),
                ("num_partials", ctypes.c_int32), ("num_combine", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("total_pages", ctypes.c_int32), ("queries_per_seq", ctypes.c_int32), ("plan_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("wait_timeout_ns", ctypes.c_int64)]


EXPORTS = ("mla_status_string", "mla_last_error_string", "mla_plan_bytes_max", "mla_plan_splits", "mla_absorb_q", "mla_decode_paged",
           "mla_combine_splits", "mla_out_proj", "mla_read_device_error", "mla_debug_wait_timeout",
           "mla_decode_paged_static_ws", "mla_decode_step_host", "mla_append_kv", "mla_merge_out_proj",
           "mla_absorb_decode_paged", "mla_gather_kv", "mla_step_graph_create", "mla_step_graph_run",
           "mla_step_graph_destroy", "mla_prefill_workspace_bytes", "mla_prefill_decompressed")

# capacity of the library's fixed split-partial array (mla_decode_paged_static_ws)
MLA_STATIC_WS_MAX_PARTIALS = 128

_lib = None


class StepBuffers(ctypes.Structure):
    """mla_step_buffers: the device buffers of mla_decode_step_host, plus its pinned plan staging."""
    _fields_ = [("q_c", ctypes.c_void_p), ("q_r", ctypes.c_void_p), ("q_abs", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("plan", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("o_lat", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("dev_error", ctypes.c_void_p), ("plan_host", ctypes.c_void_p),
                ("plan_capacity", ctypes.c_size_t)]


def lib() -> ctypes.CDLL:
    """Open libmla_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() or "
                           "python -m mla_latent_kv_absorb_gb300.build")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz, u32p = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_status_string.argtypes = [ctypes.c_int]
    L.mla_last_error_string.restype = ctypes.c_char_p
    L.mla_last_error_string.argtypes = []
    L.mla_plan_bytes_max.restype = sz
    L.mla_plan_bytes_max.argtypes = [i32, i32]
    L.mla_plan_splits.restype = ctypes.c_int
    L.mla_plan_splits.argtypes = [P, i32, i32, ctypes.POINTER(PlanOptions), P, sz, ctypes.POINTER(PlanInfo)]
    L.mla_absorb_q.restype = ctypes.c_int
    L.mla_absorb_q.argtypes = [P, P, P, i32, P]
    L.mla_decode_paged.restype = ctypes.c_int
    L.mla_decode_paged.argtypes = [ctypes.POINTER(PlanInfo), P, P, P, ctypes.c_int, P, P, P, i32, P, i32,
                                   ctypes.c_float, P, sz, P, P, u32p, P]
    L.mla_decode_paged_static_ws.restype = ctypes.c_int
    L.mla_decode_paged_static_ws.argtypes = [ctypes.POINTER(PlanInfo), P, P, P, ctypes.c_int, P, P, P, i32, P, i32,
                                             ctypes.c_float, P, P, u32p, P]
    L.mla_combine_splits.restype = ctypes.c_int
    L.mla_combine_splits.argtypes = [ctypes.POINTER(PlanInfo), P, P, sz, P, P, P]
    L.mla_out_proj.restype = ctypes.c_int
    L.mla_out_proj.argtypes = [P, P, P, i32, P]
    L.mla_absorb_decode_paged.restype = ctypes.c_int
    L.mla_absorb_decode_paged.argtypes = [ctypes.POINTER(PlanInfo), P, P, P, P, P, P, ctypes.c_int, P, P, P, i32, P,
                                          i32, ctypes.c_float, P, sz, P, P, P, P]
    L.mla_gather_kv.restype = ctypes.c_int
    L.mla_gather_kv.argtypes = [ctypes.c_int, P, P, P, i32, P, i32, P, P, i32, P, P, P]
    L.mla_merge_out_proj.restype = ctypes.c_int
    L.mla_merge_out_proj.argtypes = [ctypes.POINTER(PlanInfo), P, P, sz, P, P, P, P, P, P]
    L.mla_decode_step_host.restype = ctypes.c_int
    L.mla_decode_step_host.argtypes = [P, i32, i32, ctypes.POINTER(PlanOptions), P, P, P, i32, P, P, ctypes.c_int, P,
                                       P, P, i32, ctypes.c_float, ctypes.POINTER(StepBuffers), P,
                                       ctypes.POINTER(PlanInfo), P]
    step_args = [P, i32, i32, ctypes.POINTER(PlanOptions), P, P, P, i32, P, P, ctypes.c_int, P, P, P, i32,
                 ctypes.c_float, ctypes.POINTER(StepBuffers), P, ctypes.POINTER(PlanInfo), P]
    L.mla_step_graph_create.restype = ctypes.c_int
    L.mla_step_graph_create.argtypes = step_args + [ctypes.POINTER(ctypes.c_void_p)]
    L.mla_step_graph_run.restype = ctypes.c_int
    L.mla_step_graph_run.argtypes = [P, i32, P]
    L.mla_step_graph_destroy.restype = ctypes.c_int
    L.mla_step_graph_destroy.argtypes = [P]
    L.mla_prefill_workspace_bytes.restype = sz
    L.mla_prefill_workspace_bytes.argtypes = [i32]
    L.mla_prefill_decompressed.restype = ctypes.c_int
    L.mla_prefill_decompressed.argtypes = [ctypes.c_int, P, P, P, i32, P, i32, i32, i32, P, P, P, P, ctypes.c_float,
                                           P, sz, P, u32p, P]
    L.mla_append_kv.restype = ctypes.c_int
    L.mla_append_kv.argtypes = [i32, P, P, P, ctypes.c_int, i32, P, P, P, u32p, P]
    L.mla_read_device_error.restype = ctypes.c_int
    L.mla_read_device_error.argtypes = [u32p, ctypes.POINTER(ctypes.c_uint32), P]
    L.mla_debug_wait_timeout.restype = ctypes.c_int
    L.mla_debug_wait_timeout.argtypes = [u32p, i64, P]
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().mla_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != MLA_OK:
        msg = status_string(status)
        if status == MLA_ERR_CUDA or (status == MLA_ERR_WORKSPACE and fn == "mla_decode_paged_static_ws"):
            msg += ": " + lib().mla_last_error_string().decode()
        raise MlaError(fn, status, msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _addr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _need(t: torch.Tensor, name: str, dtype, shape=None, device=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if device and not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


# --------------------------------------------------------------------------- C ABI, same names

def mla_plan_splits(seq_lens, num_sms: int, *, min_pages_per_split: int = 0, max_clusters: int = 0,
                    wait_timeout_ns: int = 0, item_cost_pages: int = 0, queries_per_seq: int = 0):
    """Host planning. Returns (plan image as an int32 numpy array, PlanInfo).  With
    queries_per_seq = q > 1 the plan covers len(seq_lens) * q query rows (token t of sequence b
    is row b * q + t and sees the first S_b - q + 1 + t cached tokens)."""
    lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    B = int(lens.size)
    cap = int(lib().mla_plan_bytes_max(B * max(1, int(queries_per_seq)), int(num_sms)))
    if cap == 0:
        raise MlaError("mla_plan_splits", MLA_ERR_INVALID_ARG, "bad batch or SM count")
    buf = np.zeros(cap // 4, dtype=np.int32)
    opts = PlanOptions(int(min_pages_per_split), int(max_clusters), int(wait_timeout_ns), int(item_cost_pages),
                       int(queries_per_seq))
    info = PlanInfo()
    st = lib().mla_plan_splits(lens.ctypes.data_as(ctypes.c_void_p), B, int(num_sms), ctypes.byref(opts),
                               buf.ctypes.data_as(ctypes.c_void_p), cap, ctypes.byref(info))
    _check("mla_plan_splits", st)
    return buf[: info.plan_bytes // 4].copy(), info


def mla_absorb_q(q_c: torch.Tensor, w_uk: torch.Tensor, q_abs: torch.Tensor, stream=None) -> None:
    B = q_c.shape[0]
    _need(q_c, "q_c", torch.bfloat16, (B, NUM_HEADS, D_HC))
    _need(w_uk, "w_uk", torch.bfloat16, (NUM_HEADS, D_HC, D_C))
    _need(q_abs, "q_abs", torch.bfloat16, (B, NUM_HEADS, D_C))
    _check("mla_absorb_q", lib().mla_absorb_q(_ptr(q_c), _ptr(w_uk), _ptr(q_abs), B, _stream(stream)))


def mla_out_proj(o_lat: torch.Tensor, w_uv: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    B = o_lat.shape[0]
    _need(o_lat, "o_lat", torch.bfloat16, (B, NUM_HEADS, D_C))
    _need(w_uv, "w_uv", torch.bfloat16, (NUM_HEADS, D_HC, D_C))
    _need(out, "out", torch.bfloat16, (B, NUM_HEADS, D_HC))
    _check("mla_out_proj", lib().mla_out_proj(_ptr(o_lat), _ptr(w_uv), _ptr(out), B, _stream(stream)))


def mla_decode_paged(info: PlanInfo, plan_dev: torch.Tensor, q_abs: torch.Tensor, q_r: torch.Tensor, *,
                     kv_pool: torch.Tensor, block_table: torch.Tensor, o_lat: torch.Tensor, lse: torch.Tensor,
                     dev_error: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                     kv_scale: Optional[torch.Tensor] = None, kr_pool: Optional[torch.Tensor] = None,
                     softmax_scale: float = SOFTMAX_SCALE, stream=None) -> None:
    B = q_abs.shape[0]
    _need(plan_dev, "plan_dev", torch.int32)
    _need(q_abs, "q_abs", torch.bfloat16, (B, NUM_HEADS, D_C))
    _need(q_r, "q_r", torch.bfloat16, (B, NUM_HEADS, D_R))
    _need(block_table, "block_table", torch.int32)
    _need(o_lat, "o_lat", torch.bfloat16, (B, NUM_HEADS, D_C))
    _need(lse, "lse", torch.float32, (B, NUM_HEADS))
    _need(dev_error, "dev_error", torch.int32, (1,))
    if block_table.dim() != 2 or block_table.shape[0] * max(1, int(info.queries_per_seq)) != B:
        raise ValueError("block_table must be [sequences, max_pages] (query rows / queries_per_seq)")
    dtype = _kv_dtype(kv_pool, kv_scale, kr_pool)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().mla_decode_paged(ctypes.byref(info), _ptr(plan_dev), _ptr(q_abs), _ptr(q_r), dtype, _ptr(kv_pool),
                                _ptr(kv_scale), _ptr(kr_pool), int(kv_pool.shape[0]), _ptr(block_table),
                                int(block_table.shape[1]), float(softmax_scale), _ptr(workspace), ws_bytes,
                                _ptr(o_lat), _ptr(lse), _ptr(dev_error), _stream(stream))
    _check("mla_decode_paged", st)


def mla_absorb_decode_paged(info: PlanInfo, plan_dev: torch.Tensor, q_c: torch.Tensor, w_uk: torch.Tensor,
                            q_abs: torch.Tensor, absorb_sync: torch.Tensor, q_r: torch.Tensor, *,
                            kv_pool: torch.Tensor, block_table: torch.Tensor, o_lat: torch.Tensor, lse: torch.Tensor,
                            dev_error: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                            kv_scale: Optional[torch.Tensor] = None, kr_pool: Optional[torch.Tensor] = None,
                            softmax_scale: float = SOFTMAX_SCALE, stream=None) -> None:
    """Absorb and decode in one launch (the absorb as the decode kernel's prologue); q_abs is
    written.  absorb_sync: int32 [2] on the device, zero before the first call (left zero by
    every call that reports no device error)."""
    B = q_c.shape[0]
    _need(plan_dev, "plan_dev", torch.int32)
    _need(q_c, "q_c", torch.bfloat16, (B, NUM_HEADS, D_HC))
    _need(w_uk, "w_uk", torch.bfloat16, (NUM_HEADS, D_HC, D_C))
    _need(q_abs, "q_abs", torch.bfloat16, (B, NUM_HEADS, D_C))
    _need(absorb_sync, "absorb_sync", torch.int32, (2,))
    _need(q_r, "q_r", torch.bfloat16, (B, NUM_HEADS, D_R))
    _need(block_table, "block_table", torch.int32)
    _need(o_lat, "o_lat", torch.bfloat16, (B, NUM_HEADS, D_C))
    _need(lse, "lse", torch.float32, (B, NUM_HEADS))
    _need(dev_error, "dev_error", torch.int32, (1,))
    if block_table.dim() != 2 or block_table.shape[0] * max(1, int(info.queries_per_seq)) != B:
        raise ValueError("block_table must be [sequences, max_pages] (query rows / queries_per_seq)")
    dtype = _kv_dtype(kv_pool, kv_scale, kr_pool)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().mla_absorb_decode_paged(ctypes.byref(info), _ptr(plan_dev), _ptr(q_c), _ptr(w_uk), _ptr(q_abs),
                                       _ptr(absorb_sync), _ptr(q_r), dtype, _ptr(kv_pool), _ptr(kv_scale),
                                       _ptr(kr_pool), int(kv_pool.shape[0]), _ptr(block_table),
                                       int(block_table.shape[1]), float(softmax_scale), _ptr(workspace), ws_bytes,
                                       _ptr(o_lat), _ptr(lse), _ptr(dev_error), _stream(stream))
    _check("mla_absorb_decode_paged", st)


def mla_decode_paged_static_ws(info: PlanInfo, plan_dev: torch.Tensor, q_abs: torch.Tensor, q_r: torch.Tensor, *,
                               kv_pool: torch.Tensor, block_table: torch.Tensor, o_lat: torch.Tensor,
                               lse: torch.Tensor, dev_error: torch.Tensor, kv_scale: Optional[torch.Tensor] = None,
                               kr_pool: Optional[torch.Tensor] = None, softmax_scale: float = SOFTMAX_SCALE,
                               stream=None) -> None:
    """Decode plus split merge with the library's fixed scratch array: allocates nothing.
    Calls that may overlap on one device race on that array (see include/mla.h)."""
    B = q_abs.shape[0]
    _need(plan_dev, "plan_dev", torch.int32)
    _need(q_abs, "q_abs", torch.bfloat16, (B, NUM_HEADS, D_C))
    _need(q_r, "q_r", torch.bfloat16, (B, NUM_HEADS, D_R))
    _need(block_table, "block_table", torch.int32)
    _need(o_lat, "o_lat", torch.bfloat16, (B, NUM_HEADS, D_C))
    _need(lse, "lse", torch.float32, (B, NUM_HEADS))
    _need(dev_error, "dev_error", torch.int32, (1,))
    if block_table.dim() != 2 or block_table.shape[0] * max(1, int(info.queries_per_seq)) != B:
        raise ValueError("block_table must be [sequences, max_pages] (query rows / queries_per_seq)")
    dtype = _kv_dtype(kv_pool, kv_scale, kr_pool)
    st = lib().mla_decode_paged_static_ws(ctypes.byref(info), _ptr(plan_dev), _ptr(q_abs), _ptr(q_r), dtype,
                                          _ptr(kv_pool), _ptr(kv_scale), _ptr(kr_pool), int(kv_pool.shape[0]),
                                          _ptr(block_table), int(block_table.shape[1]), float(softmax_scale),
                                          _ptr(o_lat), _ptr(lse), _ptr(dev_error), _stream(stream))
    _check("mla_decode_paged_static_ws", st)


def _kv_dtype(kv_pool, kv_scale, kr_pool) -> int:
    if kv_scale is None:
        _need(kv_pool, "kv_pool", torch.bfloat16)
        if kv_pool.dim() != 3 or tuple(kv_pool.shape[1:]) != (PAGE, D_ROW):
            raise ValueError("bf16 kv_pool must be [pages, 64, 576]")
        return MLA_KV_BF16
    _need(kv_pool, "kv_pool (e4m3 codes or NVFP4 rows)", torch.uint8)
    if kv_pool.dim() == 3 and tuple(kv_pool.shape[1:]) == (PAGE, NVFP4_ROW):
        _need(kv_scale, "kv_scale", torch.float32, (kv_pool.shape[0], PAGE))
        _need(kr_pool, "kr_pool", torch.bfloat16, (kv_pool.shape[0], PAGE, D_R))
        return MLA_KV_NVFP4
    if kv_pool.dim() != 3 or tuple(kv_pool.shape[1:]) != (PAGE, D_C):
        raise ValueError("fp8 kv_pool must be [pages, 64, 512] (NVFP4: [pages, 64, 288])")
    _need(kv_scale, "kv_scale", torch.float32, (kv_pool.shape[0], PAGE))
    _need(kr_pool, "kr_pool", torch.bfloat16, (kv_pool.shape[0], PAGE, D_R))
    return MLA_KV_FP8_E4M3


def mla_combine_splits(info: PlanInfo, plan_dev: torch.Tensor, workspace: Optional[torch.Tensor],
                       o_lat: torch.Tensor, lse: torch.Tensor, stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().mla_combine_splits(ctypes.byref(info), _ptr(plan_dev), _ptr(workspace), ws_bytes, _ptr(o_lat),
                                  _ptr(lse), _stream(stream))
    _check("mla_combine_splits", st)


def mla_merge_out_proj(info: PlanInfo, plan_dev: torch.Tensor, workspace: Optional[torch.Tensor],
                       o_lat: torch.Tensor, lse: torch.Tensor, w_uv: torch.Tensor, out: torch.Tensor,
                       dev_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """Split merge and W_UV projection in one launch (merged rows as mla_combine_splits writes
    them, out as mla_out_proj computes it)."""
    B = int(info.batch)
    _need(o_lat, "o_lat", torch.bfloat16, (B, NUM_HEADS, D_C))
    _need(lse, "lse", torch.float32, (B, NUM_HEADS))
    _need(w_uv, "w_uv", torch.bfloat16, (NUM_HEADS, D_HC, D_C))
    _need(out, "out", torch.bfloat16, (B, NUM_HEADS, D_HC))
    if dev_error is not None:
        _need(dev_error, "dev_error", torch.int32, (1,))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().mla_merge_out_proj(ctypes.byref(info), _ptr(plan_dev), _ptr(workspace), ws_bytes, _ptr(o_lat),
                                  _ptr(lse), _ptr(w_uv), _ptr(out), _ptr(dev_error), _stream(stream))
    _check("mla_merge_out_proj", st)


def mla_append_kv(c_kv: torch.Tensor, k_r: torch.Tensor, slots: torch.Tensor, *, kv_pool: torch.Tensor,
                  dev_error: torch.Tensor, kv_scale: Optional[torch.Tensor] = None,
                  kr_pool: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write new tokens into the paged cache: token i to slot slots[i] (page * 64 + row; negative
    = skip).  bf16 cache: kv_pool [pages, 64, 576].  FP8 cache (kv_scale given): c_KV quantised
    per token into kv_pool [pages, 64, 512] (e4m3 codes) and kv_scale [pages, 64], k_R into
    kr_pool [pages, 64, 64]."""
    if not isinstance(slots, torch.Tensor) or slots.dim() != 1:
        raise ValueError("slots must be a 1-d tensor")
    n = int(slots.shape[0])
    _need(slots, "slots", torch.int32, (n,))
    _need(c_kv, "c_kv", torch.bfloat16, (n, D_C))
    _need(k_r, "k_r", torch.bfloat16, (n, D_R))
    _need(dev_error, "dev_error", torch.int32, (1,))
    dtype = _kv_dtype(kv_pool, kv_scale, kr_pool)
    st = lib().mla_append_kv(n, _ptr(c_kv), _ptr(k_r), _ptr(slots), dtype, int(kv_pool.shape[0]), _ptr(kv_pool),
                             _ptr(kv_scale), _ptr(kr_pool), _ptr(dev_error), _stream(stream))
    _check("mla_append_kv", st)


def mla_gather_kv(*, kv_pool: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                  cu_seqlens: torch.Tensor, out: torch.Tensor, dev_error: torch.Tensor,
                  kv_scale: Optional[torch.Tensor] = None, kr_pool: Optional[torch.Tensor] = None,
                  stream=None) -> None:
    """Every sequence's cache rows in logical order into out [total, 576] (bf16), dequantised
    from an FP8 or NVFP4 cache; cu_seqlens [B + 1] gives each sequence's first row."""
    dtype = _kv_dtype(kv_pool, kv_scale, kr_pool)
    _need(block_table, "block_table", torch.int32)
    B = int(seq_lens.shape[0])
    _need(seq_lens, "seq_lens", torch.int32, (B,))
    _need(cu_seqlens, "cu_seqlens", torch.int32, (B + 1,))
    _need(out, "out", torch.bfloat16)
    _need(dev_error, "dev_error", torch.int32, (1,))
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch, max_pages]")
    if out.dim() != 2 or out.shape[1] != D_ROW:
        raise ValueError("out must be [total tokens, 576]")
    st = lib().mla_gather_kv(dtype, _ptr(kv_pool), _ptr(kv_scale), _ptr(kr_pool), int(kv_pool.shape[0]),
                             _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens), _ptr(cu_seqlens), B,
                             _ptr(out), _ptr(dev_error), _stream(stream))
    _check("mla_gather_kv", st)


# Chunks of at least this many new tokens take the decompressed form, shorter ones the absorbed
# decode (page 1 section 3, kPrefillThresh in mla_config.h; section 6 measures the switch).
PREFILL_THRESHOLD = 256


def mla_prefill_decompressed(*, kv_pool: torch.Tensor, block_table_row: torch.Tensor, seq_len: int,
                             q_c: torch.Tensor, q_r: torch.Tensor, w_uk: torch.Tensor, w_uv: torch.Tensor,
                             out: torch.Tensor, dev_error: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                             kv_scale: Optional[torch.Tensor] = None, kr_pool: Optional[torch.Tensor] = None,
                             softmax_scale: float = SOFTMAX_SCALE, stream=None) -> None:
    """The last T = q_c.shape[0] tokens of one sequence of seq_len cached tokens, attended
    causally in the decompressed form: out [T, 128, 128].  workspace: at least
    mla_prefill_workspace_bytes(seq_len) bytes (allocated here when None)."""
    T = int(q_c.shape[0])
    _need(q_c, "q_c", torch.bfloat16, (T, NUM_HEADS, D_HC))
    _need(q_r, "q_r", torch.bfloat16, (T, NUM_HEADS, D_R))
    _need(out, "out", torch.bfloat16, (T, NUM_HEADS, D_HC))
    _need(block_table_row, "block_table_row", torch.int32)
    _need(dev_error, "dev_error", torch.int32, (1,))
    need = int(lib().mla_prefill_workspace_bytes(int(seq_len)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_c.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    dtype = _kv_dtype(kv_pool, kv_scale, kr_pool)
    st = lib().mla_prefill_decompressed(dtype, _ptr(kv_pool), _ptr(kv_scale), _ptr(kr_pool), int(kv_pool.shape[0]),
                                        _ptr(block_table_row), int(block_table_row.numel()), int(seq_len), T,
                                        _ptr(q_c), _ptr(q_r), _ptr(w_uk), _ptr(w_uv), float(softmax_scale),
                                        _ptr(workspace), ws_bytes, _ptr(out), _ptr(dev_error), _stream(stream))
    _check("mla_prefill_decompressed", st)


def prefill_chunk(seq_len: int, q_c: torch.Tensor, q_r: torch.Tensor, *, w_uk: torch.Tensor, w_uv: torch.Tensor,
                  kv_pool: torch.Tensor, block_table_row: torch.Tensor, kv_scale: Optional[torch.Tensor] = None,
                  kr_pool: Optional[torch.Tensor] = None, threshold: int = PREFILL_THRESHOLD,
                  softmax_scale: float = SOFTMAX_SCALE, stream=None):
    """A chunk of T = q_c.shape[0] new tokens at the end of one sequence of seq_len cached
    tokens (the chunk's cache rows included): chunks shorter than `threshold` run the absorbed
    decode with T query rows (DecodeStep, queries_per_seq = T), longer ones the decompressed
    form (mla_prefill_decompressed).  Returns (out [T, 128, 128], device error word)."""
    T = int(q_c.shape[0])
    bt = block_table_row.reshape(1, -1)
    if T < threshold:
        step = DecodeStep(np.array([seq_len], np.int32), w_uk=w_uk, w_uv=w_uv, kv_pool=kv_pool, block_table=bt,
                          kv_scale=kv_scale, kr_pool=kr_pool, device=q_c.device, queries_per_seq=T,
                          softmax_scale=softmax_scale)
        return step.run(q_c, q_r, stream), step.dev_error
    out = torch.empty(T, NUM_HEADS, D_HC, dtype=torch.bfloat16, device=q_c.device)
    err = torch.zeros(1, dtype=torch.int32, device=q_c.device)
    mla_prefill_decompressed(kv_pool=kv_pool, block_table_row=bt[0], seq_len=seq_len, q_c=q_c, q_r=q_r, w_uk=w_uk,
                             w_uv=w_uv, out=out, dev_error=err, kv_scale=kv_scale, kr_pool=kr_pool,
                             softmax_scale=softmax_scale, stream=stream)
    return out, err


def mla_read_device_error(dev_error: torch.Tensor, stream=None) -> int:
    """Device error bits (0 = none); waits for the stream."""
    bits = ctypes.c_uint32(0)
    st = lib().mla_read_device_error(_ptr(dev_error), ctypes.byref(bits), _stream(stream))
    if st not in (MLA_OK, MLA_ERR_DEVICE_FAULT):
        _check("mla_read_device_error", st)
    return int(bits.value)


def mla_debug_wait_timeout(dev_error: torch.Tensor, timeout_ns: int, stream=None) -> None:
    _check("mla_debug_wait_timeout", lib().mla_debug_wait_timeout(_ptr(dev_error), int(timeout_ns), _stream(stream)))


# --------------------------------------------------------------------------- one decode step

def _check_table_rows(seq_lens, block_table) -> None:
    """Every page of every sequence needs an entry in its block-table row."""
    if block_table is None or block_table.dim() != 2:
        return
    pages = (np.asarray(seq_lens, dtype=np.int64) + PAGE - 1) // PAGE
    if pages.size and int(pages.max()) > int(block_table.shape[1]):
        raise ValueError(f"block_table rows hold {int(block_table.shape[1])} pages, a sequence needs "
                         f"{int(pages.max())}")


def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device if device is not None else torch.cuda.current_device()).multi_processor_count


class DecodeStep:
    """Device buffers and plan for one batch shape; ``run`` enqueues the step's kernels.

    absorb (q_c -> q_abs) -> paged decode (-> o_lat, lse, split partials) -> split merge -> W_UV
    projection (-> out), each a kernel of its own, chained by programmatic dependent launch (the
    measured fastest order at every workload of the benchmark).  fused_absorb runs the absorb as
    the bf16 decode kernel's prologue (mla_absorb_decode_paged); fused_tail runs merge and
    projection as one kernel (mla_merge_out_proj).  All buffers are allocated here, by torch, once.
    """

    def __init__(self, seq_lens, *, w_uk: torch.Tensor, w_uv: torch.Tensor, kv_pool: torch.Tensor,
                 block_table: torch.Tensor, kv_scale: Optional[torch.Tensor] = None,
                 kr_pool: Optional[torch.Tensor] = None, device=None, min_pages_per_split: int = 0,
                 max_clusters: int = 0, wait_timeout_ns: int = 0, item_cost_pages: int = 0,
                 softmax_scale: float = SOFTMAX_SCALE, fused_absorb: bool = False, fused_tail: bool = False,
                 queries_per_seq: int = 1):
        self.device = torch.device(device if device is not None else "cuda")
        self.seq_lens = np.asarray(seq_lens, dtype=np.int32)
        self.num_seqs = int(self.seq_lens.size)
        self.queries_per_seq = max(1, int(queries_per_seq))
        # query rows: token t of sequence b is row b * q + t (q_c, q_r, q_abs, o_lat, lse, out)
        self.batch = self.num_seqs * self.queries_per_seq
        self._plan_opts = dict(min_pages_per_split=min_pages_per_split, max_clusters=max_clusters,
                               wait_timeout_ns=wait_timeout_ns, item_cost_pages=item_cost_pages,
                               queries_per_seq=self.queries_per_seq)
        self._num_sms = num_sms(self.device)
        self.plan_host, self.info = mla_plan_splits(self.seq_lens, self._num_sms, **self._plan_opts)
        self.plan_dev = torch.from_numpy(self.plan_host).to(self.device)
        self.w_uk, self.w_uv = w_uk, w_uv
        self.kv_pool, self.kv_scale, self.kr_pool = kv_pool, kv_scale, kr_pool
        self.block_table = block_table
        _check_table_rows(self.seq_lens, block_table)
        self.softmax_scale = softmax_scale
        self.fused_absorb, self.fused_tail = bool(fused_absorb), bool(fused_tail)
        B = self.batch
        ws = int(self.info.workspace_bytes)
        self.workspace = torch.empty(max(ws // 4, 4), dtype=torch.float32, device=self.device) if ws else None
        self.q_abs = torch.empty(B, NUM_HEADS, D_C, dtype=torch.bfloat16, device=self.device)
        self.o_lat = torch.empty(B, NUM_HEADS, D_C, dtype=torch.bfloat16, device=self.device)
        self.lse = torch.empty(B, NUM_HEADS, dtype=torch.float32, device=self.device)
        self.out = torch.empty(B, NUM_HEADS, D_HC, dtype=torch.bfloat16, device=self.device)
        self.dev_error = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.absorb_sync = torch.zeros(2, dtype=torch.int32, device=self.device)  # absorb-in-decode job counter
        self._h_stage = self._d_stage = None  # pinned host / device staging of run_host
        self._host_graph = None  # (mla_step_graph handle, key of the buffers and lengths it was made for)

    def run(self, q_c: torch.Tensor, q_r: torch.Tensor, stream=None) -> torch.Tensor:
        kv = dict(kv_pool=self.kv_pool, block_table=self.block_table, o_lat=self.o_lat, lse=self.lse,
                  dev_error=self.dev_error, workspace=self.workspace, kv_scale=self.kv_scale, kr_pool=self.kr_pool,
                  softmax_scale=self.softmax_scale, stream=stream)
        if self.fused_absorb:
            mla_absorb_decode_paged(self.info, self.plan_dev, q_c, self.w_uk, self.q_abs, self.absorb_sync, q_r, **kv)
        else:
            mla_absorb_q(q_c, self.w_uk, self.q_abs, stream)
            mla_decode_paged(self.info, self.plan_dev, self.q_abs, q_r, **kv)
        if self.fused_tail:
            mla_merge_out_proj(self.info, self.plan_dev, self.workspace, self.o_lat, self.lse, self.w_uv, self.out,
                               self.dev_error, stream)
        else:
            mla_combine_splits(self.info, self.plan_dev, self.workspace, self.o_lat, self.lse, stream)
            mla_out_proj(self.o_lat, self.w_uv, self.out, stream)
        return self.out

    @staticmethod
    def _host_key(q_c, q_r, block_table, lens, out):
        bt = None if block_table is None else (block_table.data_ptr(), tuple(block_table.shape), block_table.dtype)
        return (lens.tobytes(), q_c.data_ptr(), q_c.numel(), q_c.dtype, q_r.data_ptr(), q_r.numel(), q_r.dtype, bt,
                out.data_ptr(), out.numel(), out.dtype)

    def _drop_host_graph(self) -> None:
        if self._host_graph is not None:
            handle, self._host_graph = self._host_graph[0], None
            lib().mla_step_graph_destroy(handle)

    def __del__(self):
        try:
            self._drop_host_graph()
        except Exception:
            pass

    def run_host(self, q_c: torch.Tensor, q_r: torch.Tensor, *, block_table: Optional[torch.Tensor] = None,
                 seq_lens=None, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """One decode step from host (CPU) tensors, end to end: plan on the host for ``seq_lens``
        (the lengths given at construction when None; same batch size), copy the block table (a
        CPU int32 [batch, max_pages] tensor, when given; otherwise the device table given at
        construction is used) and the queries to the device, run the four kernels, and copy the
        result into ``out`` (a CPU bf16 [batch, 128, 128] tensor, pinned and allocated once if not
        given).  Returns ``out`` once the stream is done.

        When ``out``, the queries and the table are all pinned, the step is captured once as a
        CUDA graph (``mla_step_graph_create``: the plan is copied to the device at capture) and
        later calls with the same tensors and lengths only launch it (``mla_step_graph_run``),
        so a serving loop that writes each step's queries into the same pinned tensors pays for
        the copies and kernels only.  Otherwise each call is one ``mla_decode_step_host``."""
        lens = self.seq_lens if seq_lens is None else np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
        if self._host_graph is not None and out is not None:
            if self._host_key(q_c, q_r, block_table, lens, out) == self._host_graph[1]:
                _check("mla_step_graph_run", lib().mla_step_graph_run(self._host_graph[0], 1, _stream(stream)))
                return out
        B = self.batch
        _need(q_c, "q_c", torch.bfloat16, (B, NUM_HEADS, D_HC), device=False)
        _need(q_r, "q_r", torch.bfloat16, (B, NUM_HEADS, D_R), device=False)
        if lens.size != self.num_seqs:
            raise ValueError("run_host: seq_lens must keep the number of sequences")
        if block_table is not None:
            _need(block_table, "block_table", torch.int32, device=False)
            if block_table.dim() != 2 or block_table.shape[0] != self.num_seqs:
                raise ValueError("block_table must be [sequences, max_pages]")
        if not np.array_equal(lens, self.seq_lens) or self._h_stage is None:
            # new lengths: size the workspace for their plan (the library plans again itself)
            self._drop_host_graph()
            self.seq_lens = lens.copy()
            _, info = mla_plan_splits(lens, self._num_sms, **self._plan_opts)
            ws = int(info.workspace_bytes)
            if ws and (self.workspace is None or self.workspace.numel() * 4 < ws):
                self.workspace = torch.empty(ws // 4, dtype=torch.float32, device=self.device)
            if self._h_stage is None:
                cap = int(lib().mla_plan_bytes_max(B, self._num_sms))
                self._h_stage = torch.empty(cap // 4, dtype=torch.int32).pin_memory()
                self._d_stage = torch.empty(cap // 4, dtype=torch.int32, device=self.device)
                self._q_c_dev = torch.empty(B, NUM_HEADS, D_HC, dtype=torch.bfloat16, device=self.device)
                self._q_r_dev = torch.empty(B, NUM_HEADS, D_R, dtype=torch.bfloat16, device=self.device)
        if block_table is not None and (getattr(self, "_bt_dev", None) is None or
                                        tuple(self._bt_dev.shape) != tuple(block_table.shape)):
            self._drop_host_graph()
            self._bt_dev = torch.empty(tuple(block_table.shape), dtype=torch.int32, device=self.device)
        bt_dev = self._bt_dev if block_table is not None else self.block_table
        _check_table_rows(lens, bt_dev)
        use_graph = out is not None and q_c.is_pinned() and q_r.is_pinned() and out.is_pinned() and \
            (block_table is None or block_table.is_pinned())
        if out is None:
            out = torch.empty(B, NUM_HEADS, D_HC, dtype=torch.bfloat16).pin_memory()
        _need(out, "out", torch.bfloat16, (B, NUM_HEADS, D_HC), device=False)
        dtype = MLA_KV_BF16 if self.kv_scale is None else MLA_KV_FP8_E4M3
        bufs = StepBuffers(_addr(self._q_c_dev), _addr(self._q_r_dev), _addr(self.q_abs), _addr(bt_dev),
                           _addr(self._d_stage), _addr(self.workspace),
                           0 if self.workspace is None else self.workspace.numel() * 4, _addr(self.o_lat),
                           _addr(self.lse), _addr(self.out), _addr(self.dev_error), _addr(self._h_stage),
                           self._h_stage.numel() * 4)
        opts = PlanOptions(int(self._plan_opts["min_pages_per_split"]), int(self._plan_opts["max_clusters"]),
                           int(self._plan_opts["wait_timeout_ns"]), int(self._plan_opts["item_cost_pages"]),
                           self.queries_per_seq)
        info = PlanInfo()
        args = (lens.ctypes.data_as(ctypes.c_void_p), self.num_seqs, self._num_sms, ctypes.byref(opts), _ptr(q_c), _ptr(q_r),
                _ptr(block_table), int(bt_dev.shape[1]), _ptr(self.w_uk), _ptr(self.w_uv), dtype, _ptr(self.kv_pool),
                _ptr(self.kv_scale), _ptr(self.kr_pool), int(self.kv_pool.shape[0]), float(self.softmax_scale),
                ctypes.byref(bufs), _ptr(out), ctypes.byref(info), _stream(stream))
        if use_graph:
            self._drop_host_graph()
            handle = ctypes.c_void_p()
            _check("mla_step_graph_create", lib().mla_step_graph_create(*args, ctypes.byref(handle)))
            self._host_graph = (handle, self._host_key(q_c, q_r, block_table, lens, out))
            self.info = info
            _check("mla_step_graph_run", lib().mla_step_graph_run(handle, 1, _stream(stream)))
            return out
        _check("mla_decode_step_host", lib().mla_decode_step_host(*args))
        self.info = info
        return out

    def capture(self, q_c: torch.Tensor, q_r: torch.Tensor) -> "torch.cuda.CUDAGraph":
        """Capture one step into a CUDA graph and return it.

        The graph holds the step's kernels with their programmatic dependencies, reading
        ``q_c`` / ``q_r`` and writing ``self.out`` at their current addresses: copy the next
        step's queries into those tensors and call ``replay()`` (it runs on the current stream).
        The lengths, block table and cache are those of this object and stay fixed in the graph
        (a new plan needs a new capture).  One step runs eagerly first so that one-time set-up
        stays out of the capture."""
        self.run(q_c, q_r)
        torch.cuda.synchronize(self.device)
        try:  # keep the captured graph so that its nodes can be counted
            graph, kept = torch.cuda.CUDAGraph(keep_graph=True), True
        except TypeError:
            graph, kept = torch.cuda.CUDAGraph(), False
        with torch.cuda.graph(graph):
            self.run(q_c, q_r)
        self.graph_kernel_nodes = None
        if kept:
            try:
                self.graph_kernel_nodes = graph_kernel_nodes(graph.raw_cuda_graph())
            except (OSError, AttributeError, RuntimeError):
                self.graph_kernel_nodes = None
            graph.instantiate()
        return graph

    def device_error(self, stream=None) -> int:
        return mla_read_device_error(self.dev_error, stream)

    @property
    def launches_per_step(self) -> int:
        # the absorb runs inside the bf16 decode kernel when fused (a kernel of its own with the e4m3
        # cache); the merge is skipped when no sequence is split
        n = 1 if (self.fused_absorb and self.kv_scale is None) else 2
        if self.fused_tail:
            return n + 1
        return n + 1 + (1 if self.info.num_combine > 0 else 0)


def graph_kernel_nodes(raw_graph: int) -> int:
    """Number of kernel nodes in a CUDA graph (driver API, read only)."""
    cu = ctypes.CDLL("libcuda.so.1")
    n = ctypes.c_size_t(0)
    if cu.cuGraphGetNodes(ctypes.c_void_p(raw_graph), None, ctypes.byref(n)) != 0:
        raise RuntimeError("cuGraphGetNodes failed")
    nodes = (ctypes.c_void_p * n.value)()
    if n.value and cu.cuGraphGetNodes(ctypes.c_void_p(raw_graph), nodes, ctypes.byref(n)) != 0:
        raise RuntimeError("cuGraphGetNodes failed")
    kernels = 0
    for i in range(n.value):
        t = ctypes.c_int(-1)
        if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) != 0:
            raise RuntimeError("cuGraphNodeGetType failed")
        kernels += int(t.value == 0)  # CU_GRAPH_NODE_TYPE_KERNEL
    return kernels


def inputs_to_device(inp, device="cuda"):
    """Move a synth.DecodeInputs to the device: (q_c, q_r, w_uk, w_uv, kv dict, block_table)."""
    dev = torch.device(device)
    kv = {}
    if inp.kv_dtype == "bf16":
        kv["kv_pool"] = inp.pool.to(dev)
    else:
        kv["kv_pool"] = inp.c8.to(dev)
        kv["kv_scale"] = inp.kv_scale.to(dev)
        kv["kr_pool"] = inp.kr.to(dev)
    bt = torch.from_numpy(np.ascontiguousarray(inp.block_table)).to(dev)
    return inp.q_c.to(dev), inp.q_r.to(dev), inp.w_uk.to(dev), inp.w_uv.to(dev), kv, bt
