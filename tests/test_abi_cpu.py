"""The C ABI library without a GPU: it loads, exports what include/mla.h declares, and its
host-side checks reject bad arguments before anything is launched.

Every call below fails host validation by construction (null, misaligned or inconsistent
arguments), so none of them reaches a kernel launch even where a GPU is present.
"""
import ctypes
import os
import re
import sys

import numpy as np
import pytest

from mla_latent_kv_absorb_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build_library()
    return binding.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("mla_plan_splits", "mla_absorb_q", "mla_decode_paged", "mla_combine_splits", "mla_out_proj"):
        assert n in names
    assert set(names) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), f"{name} not exported"


def test_status_strings(L):
    for s in range(7):
        assert binding.status_string(s) not in ("", "unknown status")
    assert binding.status_string(99) == "unknown status"


def _p(v):
    return ctypes.c_void_p(v)


def test_absorb_and_out_proj_reject_bad_args(L):
    assert L.mla_absorb_q(None, _p(4096), _p(8192), 1, None) == binding.MLA_ERR_INVALID_ARG
    assert L.mla_absorb_q(_p(4096), _p(8192), _p(12288), 0, None) == binding.MLA_ERR_INVALID_ARG
    assert L.mla_absorb_q(_p(4097), _p(8192), _p(12288), 1, None) == binding.MLA_ERR_ALIGNMENT
    assert L.mla_out_proj(_p(4096), None, _p(8192), 1, None) == binding.MLA_ERR_INVALID_ARG
    assert L.mla_out_proj(_p(4096), _p(8200), _p(12288), 1, None) == binding.MLA_ERR_ALIGNMENT


def _info(**kw):
    lens = kw.pop("lens", [100, 5000])
    plan, info = binding.mla_plan_splits(lens, 152, min_pages_per_split=2)
    for k, v in kw.items():
        setattr(info, k, v)
    return plan, info


def _decode(L, info, *, ws=None, ws_bytes=0, q_abs=0x10000, dtype=binding.MLA_KV_BF16, scale=0.07,
            kv_scale=None, kr=None, dev_error=0x50000):
    return L.mla_decode_paged(ctypes.byref(info), _p(0x20000), _p(q_abs), _p(0x30000), dtype, _p(0x40000),
                              _p(kv_scale) if kv_scale else None, _p(kr) if kr else None, 100, _p(0x60000), 80,
                              ctypes.c_float(scale), _p(ws) if ws else None, ws_bytes, _p(0x70000), _p(0x80000),
                              _p(dev_error) if dev_error else None, None)


def test_decode_rejects_bad_args(L):
    _, info = _info()
    assert info.workspace_bytes > 0
    # inconsistent plan header
    _, bad = _info(num_clusters=0)
    assert _decode(L, bad, ws=0x90000, ws_bytes=info.workspace_bytes) == binding.MLA_ERR_INVALID_ARG
    # missing pointers / bad scale / bad dtype
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes, q_abs=0) == binding.MLA_ERR_INVALID_ARG
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes, dev_error=0) == binding.MLA_ERR_INVALID_ARG
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes, scale=0.0) == binding.MLA_ERR_INVALID_ARG
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes, scale=float("nan")) == binding.MLA_ERR_INVALID_ARG
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes, dtype=7) == binding.MLA_ERR_INVALID_ARG
    # fp8 without its scale / k_R pools
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes,
                   dtype=binding.MLA_KV_FP8_E4M3) == binding.MLA_ERR_INVALID_ARG
    # fp8 with a misaligned k_R pool or scale array
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes, dtype=binding.MLA_KV_FP8_E4M3,
                   kv_scale=0xA0000, kr=0xB0008) == binding.MLA_ERR_ALIGNMENT
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes, dtype=binding.MLA_KV_FP8_E4M3,
                   kv_scale=0xA0002, kr=0xB0000) == binding.MLA_ERR_ALIGNMENT
    # misaligned query
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes, q_abs=0x10008) == binding.MLA_ERR_ALIGNMENT
    # workspace missing or too small
    assert _decode(L, info, ws=None, ws_bytes=0) == binding.MLA_ERR_WORKSPACE
    assert _decode(L, info, ws=0x90000, ws_bytes=info.workspace_bytes - 1) == binding.MLA_ERR_WORKSPACE


def test_combine_rejects_bad_args(L):
    plan, info = _info()
    assert info.num_combine > 0
    assert L.mla_combine_splits(ctypes.byref(info), _p(0x20000), None, 0, _p(0x70000), _p(0x80000),
                                None) == binding.MLA_ERR_WORKSPACE
    assert L.mla_combine_splits(ctypes.byref(info), None, _p(0x90000), info.workspace_bytes, _p(0x70000),
                                _p(0x80000), None) == binding.MLA_ERR_INVALID_ARG
    assert L.mla_combine_splits(ctypes.byref(info), _p(0x20000), _p(0x90004), info.workspace_bytes, _p(0x70000),
                                _p(0x80000), None) == binding.MLA_ERR_ALIGNMENT


def test_absorb_decode_rejects_bad_args(L):
    """The fused absorb + decode checks its extra buffers, then the decode's own arguments."""
    plan, info = _info()
    p = _p
    def call(q_c=0x100000, w_uk=0x200000, q_abs=0x300000, sync=0x400000, ws_bytes=None, bt=0x60000):
        wb = info.workspace_bytes if ws_bytes is None else ws_bytes
        return L.mla_absorb_decode_paged(ctypes.byref(info), p(0x20000), p(q_c), p(w_uk), p(q_abs), p(sync),
                                         p(0x30000), binding.MLA_KV_BF16, p(0x40000), None, None, 100, p(bt), 80,
                                         ctypes.c_float(0.07), p(0x90000), wb, p(0x70000), p(0x80000), p(0x50000),
                                         None)
    assert call(q_c=0) == binding.MLA_ERR_INVALID_ARG
    assert call(sync=0) == binding.MLA_ERR_INVALID_ARG
    assert call(sync=0x400004) == binding.MLA_ERR_ALIGNMENT
    assert call(w_uk=0x200008) == binding.MLA_ERR_ALIGNMENT
    assert call(ws_bytes=info.workspace_bytes - 1) == binding.MLA_ERR_WORKSPACE
    assert call(bt=0) == binding.MLA_ERR_INVALID_ARG


def test_merge_out_proj_rejects_bad_args(L):
    """The fused merge + projection checks its plan, buffers, workspace and alignment on the host."""
    plan, info = _info()
    assert info.num_combine > 0
    def call(plan_p=0x20000, ws=0x90000, ws_bytes=None, o=0x70000, l=0x80000, w=0xA0000, out=0xB0000, err=None):
        wb = info.workspace_bytes if ws_bytes is None else ws_bytes
        return L.mla_merge_out_proj(ctypes.byref(info), _p(plan_p), _p(ws), wb, _p(o), _p(l), _p(w), _p(out),
                                    _p(err), None)
    assert call(plan_p=0) == binding.MLA_ERR_INVALID_ARG
    assert call(w=0) == binding.MLA_ERR_INVALID_ARG
    assert call(out=0) == binding.MLA_ERR_INVALID_ARG
    assert call(ws=0, ws_bytes=0) == binding.MLA_ERR_WORKSPACE
    assert call(ws_bytes=info.workspace_bytes - 1) == binding.MLA_ERR_WORKSPACE
    assert call(w=0xA0008) == binding.MLA_ERR_ALIGNMENT
    assert call(l=0x80002) == binding.MLA_ERR_ALIGNMENT
    assert call(err=0x50002) == binding.MLA_ERR_ALIGNMENT


def test_debug_and_error_reader_reject_bad_args(L):
    assert L.mla_debug_wait_timeout(None, 10 ** 8, None) == binding.MLA_ERR_INVALID_ARG
    assert L.mla_debug_wait_timeout(_p(0x50000), 10, None) == binding.MLA_ERR_INVALID_ARG
    assert L.mla_read_device_error(None, None, None) == binding.MLA_ERR_INVALID_ARG


def test_plan_rejects_bad_args(L):
    with pytest.raises(binding.MlaError):
        binding.mla_plan_splits([10, 0, 5], 152)            # S = 0
    with pytest.raises(binding.MlaError):
        binding.mla_plan_splits([10], 1)                    # fewer than 2 SMs
    with pytest.raises(binding.MlaError):
        binding.mla_plan_splits([10], 152, min_pages_per_split=-1)
    lens = np.array([100], dtype=np.int32)
    info = binding.PlanInfo()
    buf = np.zeros(4, dtype=np.int32)  # too small
    st = L.mla_plan_splits(lens.ctypes.data_as(ctypes.c_void_p), 1, 152, None, buf.ctypes.data_as(ctypes.c_void_p),
                           buf.nbytes, ctypes.byref(info))
    assert st == binding.MLA_ERR_WORKSPACE


def _step_host(L, bufs, *, lens=(100, 5000), q=0x1000, out=0x2000, opts=None):
    arr = np.asarray(lens, dtype=np.int32)
    o = opts if opts is not None else binding.PlanOptions(2, 0, 0)
    info = binding.PlanInfo()
    return L.mla_decode_step_host(arr.ctypes.data_as(ctypes.c_void_p), len(lens), 152, ctypes.byref(o), _p(q),
                                  _p(q + 0x100), None, 80, _p(0x3000), _p(0x4000), binding.MLA_KV_BF16, _p(0x5000),
                                  None, None, 100, ctypes.c_float(0.07),
                                  ctypes.byref(bufs) if bufs is not None else None, _p(out), ctypes.byref(info),
                                  None), info


def test_step_host_rejects_bad_args(L):
    """The host-step entry point plans on the host and checks its buffers before any copy or
    launch: missing buffers are invalid arguments; a workspace smaller than the plan needs is a
    workspace error (with the plan header still returned)."""
    cap = int(L.mla_plan_bytes_max(2, 152))
    plan_host = np.zeros(cap // 4, dtype=np.int32)
    bufs = binding.StepBuffers(0x10000, 0x11000, 0x12000, 0x13000, 0x14000, 0x15000, 64, 0x16000, 0x17000,
                               0x18000, 0x19000, plan_host.ctypes.data, cap)
    st, _ = _step_host(L, None)
    assert st == binding.MLA_ERR_INVALID_ARG
    st, _ = _step_host(L, bufs, out=0)
    assert st == binding.MLA_ERR_INVALID_ARG
    no_plan = binding.StepBuffers(0x10000, 0x11000, 0x12000, 0x13000, 0x14000, 0x15000, 64, 0x16000, 0x17000,
                                  0x18000, 0x19000, 0, cap)
    st, _ = _step_host(L, no_plan)
    assert st == binding.MLA_ERR_INVALID_ARG
    st, info = _step_host(L, bufs)  # 5000 tokens over two pairs or more: split, so a workspace is due
    assert st == binding.MLA_ERR_WORKSPACE
    assert info.workspace_bytes > 64 and info.batch == 2
    small_cap = binding.StepBuffers(0x10000, 0x11000, 0x12000, 0x13000, 0x14000, 0x15000, 1 << 30, 0x16000,
                                    0x17000, 0x18000, 0x19000, plan_host.ctypes.data, 16)
    st, _ = _step_host(L, small_cap)
    assert st != binding.MLA_OK  # the plan does not fit its staging buffer
    st, _ = _step_host(L, bufs, lens=(100, 64 * 80 + 1))  # 81 pages, rows of 80 entries
    assert st == binding.MLA_ERR_INVALID_ARG


def test_step_graph_rejects_bad_args(L):
    """The captured-step entry points check their arguments before any copy or capture: a missing
    handle pointer or buffers are invalid arguments, the workspace rule is the one of
    mla_decode_step_host, host buffers that are not page-locked are refused, and destroying NULL
    is a no-op."""
    cap = int(L.mla_plan_bytes_max(2, 152))
    plan_host = np.zeros(cap // 4, dtype=np.int32)
    lens = np.asarray((100, 5000), dtype=np.int32)
    q_c = np.zeros(2 * 128 * 128, dtype=np.uint16)
    q_r = np.zeros(2 * 128 * 64, dtype=np.uint16)
    out = np.zeros(2 * 128 * 128, dtype=np.uint16)
    opts = binding.PlanOptions(2, 0, 0)

    def create(bufs, handle, *, out_ptr=out.ctypes.data):
        info = binding.PlanInfo()
        st = L.mla_step_graph_create(lens.ctypes.data_as(ctypes.c_void_p), 2, 152, ctypes.byref(opts),
                                     _p(q_c.ctypes.data), _p(q_r.ctypes.data), None, 80, _p(0x3000), _p(0x4000),
                                     binding.MLA_KV_BF16, _p(0x5000), None, None, 100, ctypes.c_float(0.07),
                                     ctypes.byref(bufs) if bufs is not None else None, _p(out_ptr),
                                     ctypes.byref(info), None, handle)
        return st, info

    bufs = binding.StepBuffers(0x10000, 0x11000, 0x12000, 0x13000, 0x14000, 0x15000, 1 << 30, 0x16000, 0x17000,
                               0x18000, 0x19000, plan_host.ctypes.data, cap)
    small_ws = binding.StepBuffers(0x10000, 0x11000, 0x12000, 0x13000, 0x14000, 0x15000, 64, 0x16000, 0x17000,
                                   0x18000, 0x19000, plan_host.ctypes.data, cap)
    h = ctypes.c_void_p(0xdead)
    st, _ = create(bufs, None)
    assert st == binding.MLA_ERR_INVALID_ARG
    st, _ = create(None, ctypes.byref(h))
    assert st == binding.MLA_ERR_INVALID_ARG and h.value is None  # the handle is cleared on failure
    st, _ = create(bufs, ctypes.byref(h), out_ptr=0)
    assert st == binding.MLA_ERR_INVALID_ARG
    st, info = create(small_ws, ctypes.byref(h))
    assert st == binding.MLA_ERR_WORKSPACE and info.workspace_bytes > 64
    st, info = create(bufs, ctypes.byref(h))  # plain numpy memory is not page-locked
    assert st == binding.MLA_ERR_INVALID_ARG and info.batch == 2 and h.value is None
    assert L.mla_step_graph_run(None, 1, None) == binding.MLA_ERR_INVALID_ARG
    assert L.mla_step_graph_destroy(None) == binding.MLA_OK


def test_prefill_rejects_bad_args(L):
    """The decompressed prefill checks its arguments before any launch."""
    F = L.mla_prefill_decompressed
    ws = int(L.mla_prefill_workspace_bytes(1000))
    assert ws >= 1000 * (1152 + 2 * 32768) and L.mla_prefill_workspace_bytes(0) == 0

    def call(*, seq=1000, chunk=300, q=0x10000, ws_bytes=ws, bt=0x4000, dtype=binding.MLA_KV_BF16, pages=16):
        return F(dtype, _p(0x1000), None, None, 100, _p(bt), pages, seq, chunk, _p(q), _p(0x20000), _p(0x30000),
                 _p(0x40000), ctypes.c_float(0.07), _p(0x50000), ws_bytes, _p(0x60000), _p(0x70000), None)

    assert call(q=0) == binding.MLA_ERR_INVALID_ARG
    assert call(chunk=1001) == binding.MLA_ERR_INVALID_ARG          # more new tokens than the sequence
    assert call(chunk=0) == binding.MLA_ERR_INVALID_ARG
    assert call(pages=15) == binding.MLA_ERR_INVALID_ARG            # 1000 tokens need 16 pages
    assert call(dtype=binding.MLA_KV_FP8_E4M3) == binding.MLA_ERR_INVALID_ARG  # no scales / k_R pool
    assert call(q=0x10008) == binding.MLA_ERR_ALIGNMENT
    assert call(bt=0x4002) == binding.MLA_ERR_ALIGNMENT
    assert call(ws_bytes=ws - 1) == binding.MLA_ERR_WORKSPACE


def test_decode_step_rejects_short_table_rows():
    """The binding checks that each sequence's pages fit its block-table row (no GPU needed:
    the check runs before anything is allocated on the device)."""
    import torch

    bt = torch.zeros(2, 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="block_table rows"):
        binding._check_table_rows(np.array([200, 300], dtype=np.int32), bt)
    binding._check_table_rows(np.array([200, 256], dtype=np.int32), bt)


def test_append_rejects_bad_args(L):
    A = L.mla_append_kv
    bf16, fp8 = binding.MLA_KV_BF16, binding.MLA_KV_FP8_E4M3
    ok = dict(c=_p(0x10000), r=_p(0x20000), s=_p(0x30000), pool=_p(0x40000), scale=_p(0x50000),
              kr=_p(0x60000), err=_p(0x70000))

    def call(n=4, dtype=bf16, pages=8, **kw):
        a = {**ok, **kw}
        return A(n, a["c"], a["r"], a["s"], dtype, pages, a["pool"], a["scale"], a["kr"], a["err"], None)

    assert call(n=0) == binding.MLA_OK                       # nothing to write: no launch
    assert call(n=-1) == binding.MLA_ERR_INVALID_ARG
    assert call(pages=0) == binding.MLA_ERR_INVALID_ARG
    assert call(dtype=7) == binding.MLA_ERR_INVALID_ARG
    assert call(c=None) == binding.MLA_ERR_INVALID_ARG
    assert call(s=None) == binding.MLA_ERR_INVALID_ARG
    assert call(err=None) == binding.MLA_ERR_INVALID_ARG
    assert call(dtype=fp8, scale=None) == binding.MLA_ERR_INVALID_ARG
    assert call(dtype=fp8, kr=None) == binding.MLA_ERR_INVALID_ARG
    assert call(c=_p(0x10008)) == binding.MLA_ERR_ALIGNMENT
    assert call(pool=_p(0x40004)) == binding.MLA_ERR_ALIGNMENT
    assert call(s=_p(0x30002)) == binding.MLA_ERR_ALIGNMENT
    assert call(dtype=fp8, kr=_p(0x60008)) == binding.MLA_ERR_ALIGNMENT
    assert call(dtype=fp8, scale=_p(0x50002)) == binding.MLA_ERR_ALIGNMENT
    nv = binding.MLA_KV_NVFP4
    assert call(dtype=nv, scale=None) == binding.MLA_ERR_INVALID_ARG
    assert call(dtype=nv, kr=None) == binding.MLA_ERR_INVALID_ARG
    assert call(dtype=nv, pool=_p(0x40008)) == binding.MLA_ERR_ALIGNMENT
    assert call(dtype=nv, kr=_p(0x60008)) == binding.MLA_ERR_ALIGNMENT


def test_gather_rejects_bad_args(L):
    G = L.mla_gather_kv
    ok = dict(pool=_p(0x40000), scale=_p(0x50000), kr=_p(0x60000), bt=_p(0x10000), sl=_p(0x20000),
              cu=_p(0x30000), out=_p(0x70000), err=_p(0x80000))

    def call(dtype=binding.MLA_KV_BF16, pages=8, maxp=4, batch=2, **kw):
        a = {**ok, **kw}
        return G(dtype, a["pool"], a["scale"], a["kr"], pages, a["bt"], maxp, a["sl"], a["cu"], batch, a["out"],
                 a["err"], None)

    assert call(dtype=9) == binding.MLA_ERR_INVALID_ARG
    assert call(batch=0) == binding.MLA_ERR_INVALID_ARG
    assert call(pages=0) == binding.MLA_ERR_INVALID_ARG
    assert call(out=None) == binding.MLA_ERR_INVALID_ARG
    assert call(dtype=binding.MLA_KV_NVFP4, scale=None) == binding.MLA_ERR_INVALID_ARG
    assert call(dtype=binding.MLA_KV_FP8_E4M3, kr=None) == binding.MLA_ERR_INVALID_ARG
    assert call(pool=_p(0x40008)) == binding.MLA_ERR_ALIGNMENT
    assert call(out=_p(0x70008)) == binding.MLA_ERR_ALIGNMENT
    assert call(cu=_p(0x30002)) == binding.MLA_ERR_ALIGNMENT
    assert call(batch=70000) == binding.MLA_ERR_UNSUPPORTED


def test_decode_rejects_nvfp4_cache(L):
    """The NVFP4 cache is written by mla_append_kv; the decode entry points report it unsupported."""
    plan, info = _info()
    p = _p
    st = L.mla_decode_paged(ctypes.byref(info), p(0x20000), p(0x10000), p(0x30000), binding.MLA_KV_NVFP4,
                            p(0x40000), p(0x50000), p(0x60000), 100, p(0x60000), 80, ctypes.c_float(0.07),
                            p(0x90000), info.workspace_bytes, p(0x70000), p(0x80000), p(0x50000), None)
    assert st == binding.MLA_ERR_UNSUPPORTED


def test_append_binding_checks_tensors():
    """The Python binding refuses host tensors, wrong dtypes and shapes before any call."""
    import torch

    c = torch.zeros(4, 512, dtype=torch.bfloat16)
    r = torch.zeros(4, 64, dtype=torch.bfloat16)
    s = torch.zeros(4, dtype=torch.int32)
    pool = torch.zeros(2, 64, 576, dtype=torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="1-d"):
        binding.mla_append_kv(c, r, s.view(2, 2), kv_pool=pool, dev_error=err)
    with pytest.raises(ValueError, match="CUDA"):
        binding.mla_append_kv(c, r, s, kv_pool=pool, dev_error=err)
    with pytest.raises(TypeError):
        binding.mla_append_kv(c, r, s.long(), kv_pool=pool, dev_error=err)


def test_nvtx_ranges_switch_on_without_changing_results():
    """With MLA_NVTX=1 every entry point opens and closes an NVTX range; the argument checks and
    their statuses are the same (run in a fresh process, since the switch is read once)."""
    import subprocess
    code = ("import ctypes, sys; sys.path.insert(0, %r); from mla_latent_kv_absorb_gb300 import binding; "
            "L = binding.lib(); p = ctypes.c_void_p; "
            "assert L.mla_absorb_q(None, p(4096), p(8192), 1, None) == binding.MLA_ERR_INVALID_ARG; "
            "assert L.mla_out_proj(p(4096), p(8200), p(12288), 1, None) == binding.MLA_ERR_ALIGNMENT; "
            "assert L.mla_append_kv(-1, None, None, None, 0, 1, None, None, None, None, None) != 0; "
            "print('ok')") % ROOT
    env = dict(os.environ, MLA_NVTX="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr
