"""The C-ABI library builds, loads and exports every declared entry point;
host-side validation rejects bad arguments before anything is launched.
No test here touches a GPU (fake, never-dereferenced device pointers are
only passed to calls that must fail validation first)."""
import ctypes
import os
import re

import pytest

from radixattention_prefix_shared_gb300 import binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "sgl_attn.h")

FAKE = ctypes.c_void_p(0x100000)     # aligned, never dereferenced
MISALIGNED = ctypes.c_void_p(0x100008)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sgl_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sgl_store_kv", "sgl_extend_attention", "sgl_decode_attention"):
        assert n in names


def test_library_exports_every_declared_symbol(cuda_lib):
    for name in declared_functions():
        assert hasattr(cuda_lib, name), f"{name} declared in sgl_attn.h but not exported"


def test_status_strings_and_version(cuda_lib):
    for code, name in B.STATUS.items():
        assert cuda_lib.sgl_status_string(code).decode() == name
    assert cuda_lib.sgl_status_string(99).decode() == "SGL_ERR_UNKNOWN"
    assert re.match(r"^\d+\.\d+\.\d+$", cuda_lib.sgl_version().decode())


def test_dims_struct_layout_matches_header():
    # int32 x3, int64 (8-aligned), float -> 32 bytes with padding
    assert ctypes.sizeof(B.sgl_attn_dims) == 32
    assert B.sgl_attn_dims.pool_size.offset == 16 and B.sgl_attn_dims.sm_scale.offset == 24


def _dims(**kw):
    d = dict(num_q_heads=4, num_kv_heads=2, head_dim=128, pool_size=1024, sm_scale=0.0)
    d.update(kw)
    return B.make_dims(**d)


def test_store_kv_validation(cuda_lib):
    f = cuda_lib.sgl_store_kv
    d = _dims()
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, None, None) == 1                        # dims NULL
    assert f(FAKE, FAKE, FAKE, -1, FAKE, FAKE, ctypes.byref(d), None) == 1            # n < 0
    assert f(None, None, None, 0, None, None, ctypes.byref(d), None) == 0             # n == 0: no-op
    assert f(None, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), None) == 1             # null k_new
    assert f(MISALIGNED, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), None) == 1       # misaligned
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(_dims(head_dim=96)), None) == 2
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(_dims(num_q_heads=3)), None) == 1
    assert f(FAKE, FAKE, FAKE, 2048, FAKE, FAKE, ctypes.byref(d), None) == 1          # n > pool
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(_dims(sm_scale=-1.0)), None) == 1


def _extend(cuda_lib, d, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, pk=FAKE, pv=FAKE, rtt=FAKE, rows=4, stride=64, rpi=FAKE,
             pl=FAKE, el=FAKE, batch=2, total=10, max_e=6, max_p=30, out=FAKE, ws=FAKE, wsb=256)
    a.update(kw)
    return cuda_lib.sgl_extend_attention(a["q"], a["k"], a["v"], a["pk"], a["pv"], a["rtt"], a["rows"],
                                         a["stride"], a["rpi"], a["pl"], a["el"], a["batch"], a["total"],
                                         a["max_e"], a["max_p"], a["out"], a["ws"], a["wsb"],
                                         ctypes.byref(d), None)


def test_extend_validation(cuda_lib):
    d = _dims()
    assert _extend(cuda_lib, d, batch=0) == 0
    assert _extend(cuda_lib, d, total=0) == 0
    assert _extend(cuda_lib, d, batch=-1) == 1
    assert _extend(cuda_lib, d, q=None) == 1
    assert _extend(cuda_lib, d, out=MISALIGNED) == 1
    assert _extend(cuda_lib, d, stride=0) == 1
    assert _extend(cuda_lib, d, max_e=11) == 1          # max_extend above total_extend
    assert _extend(cuda_lib, d, ws=None) == 3
    assert _extend(cuda_lib, d, wsb=16) == 3
    assert _extend(cuda_lib, _dims(head_dim=32)) == 2


def test_decode_validation_and_workspace_size(cuda_lib):
    d = _dims(num_q_heads=16, num_kv_heads=8)
    need = B.decode_workspace_bytes(248, 32768, d)
    # partial accumulators dominate: 8 KV heads come in groups of 4, so a call
    # may take 512-key items (e4m3 span units): 64 per 32,768-key request
    assert need > 248 * 64 * 8 * 2 * 128 * 4
    # KV heads not in groups of 4: items of 1,024 keys at the least
    d6 = _dims(num_q_heads=12, num_kv_heads=6)
    need6 = B.decode_workspace_bytes(248, 32768, d6)
    assert 248 * 32 * 6 * 2 * 128 * 4 < need6 < 248 * 64 * 6 * 2 * 128 * 4
    f = cuda_lib.sgl_decode_attention

    def call(**kw):
        a = dict(q=FAKE, pk=FAKE, pv=FAKE, rtt=FAKE, rows=4, stride=64, rpi=FAKE, sl=FAKE, batch=2,
                 max_s=64, out=FAKE, ws=FAKE, wsb=need)
        a.update(kw)
        return f(a["q"], a["pk"], a["pv"], a["rtt"], a["rows"], a["stride"], a["rpi"], a["sl"],
                 a["batch"], a["max_s"], a["out"], a["ws"], a["wsb"], ctypes.byref(d), None)
    assert call(batch=0) == 0
    assert call(max_s=0) == 1
    assert call(sl=None) == 1
    assert call(ws=None) == 3
    assert call(wsb=B.decode_workspace_bytes(2, 64, d) - 1) == 3
    # query heads per KV head: up to 128
    d129 = _dims(num_q_heads=258, num_kv_heads=2)
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 64, FAKE, FAKE, 2, 64, FAKE, FAKE,
             B.decode_workspace_bytes(2, 64, d129), ctypes.byref(d129), None) == 2
    # groups above 16 run as KV-head copies: the scratch is the same size per query head
    assert B.decode_workspace_bytes(2, 64, _dims(num_q_heads=64, num_kv_heads=2)) >= \
        B.decode_workspace_bytes(2, 64, _dims(num_q_heads=32, num_kv_heads=2))
    assert B.extend_workspace_bytes(8, 16384, d) >= 16


def test_cascade_validation_and_workspace_size(cuda_lib):
    d = _dims(num_q_heads=16, num_kv_heads=4)
    need = B.cascade_decode_workspace_bytes(8, 512, 3, d)
    # status bytes in front, plus per-request group states
    assert need >= B.decode_workspace_bytes(8, 512, d) + 256 + 8 * 3 * 16 * 128 * 4
    f = cuda_lib.sgl_cascade_decode_attention

    def call(**kw):
        a = dict(q=FAKE, pk=FAKE, pv=FAKE, rtt=FAKE, rows=8, stride=512, rpi=FAKE, sl=FAKE, batch=8,
                 max_s=512, gs=FAKE, gl=FAKE, gd=FAKE, mo=FAKE, mem=FAKE, n_groups=2, max_m=4,
                 max_d=3, out=FAKE, ws=FAKE, wsb=need)
        a.update(kw)
        return f(a["q"], a["pk"], a["pv"], a["rtt"], a["rows"], a["stride"], a["rpi"], a["sl"],
                 a["batch"], a["max_s"], a["gs"], a["gl"], a["gd"], a["mo"], a["mem"], a["n_groups"],
                 a["max_m"], a["max_d"], a["out"], a["ws"], a["wsb"], ctypes.byref(d), None)
    assert call(batch=0) == 0
    assert call(n_groups=-1) == 1
    assert call(gs=None) == 1
    assert call(mem=None) == 1
    assert call(max_d=0) == 1
    assert call(max_m=0) == 1
    assert call(n_groups=70000) == 2
    assert call(ws=None) == 3
    assert call(wsb=need - 1) == 3
    assert call(q=MISALIGNED) == 1
    # no groups: group arrays may be null
    assert call(n_groups=0, gs=None, gl=None, gd=None, mo=None, mem=None, max_d=0, max_m=0,
                ws=None) == 3
    c = cuda_lib.sgl_check_cascade_groups
    assert cuda_lib.sgl_check_cascade_scratch_bytes(8, 3) == 96
    assert c(FAKE, 8, 512, FAKE, FAKE, 8, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 3, FAKE, 95, FAKE, None) == 3
    assert c(FAKE, 8, 512, FAKE, FAKE, 8, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, 3, None, 0, FAKE, None) == 0
    assert c(FAKE, 8, 512, FAKE, FAKE, 8, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 4, 3, FAKE, 96, None, None) == 1


def test_fp8_validation(cuda_lib):
    d = _dims()
    f = cuda_lib.sgl_store_kv_fp8
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, 1.0, 0.0, ctypes.byref(d), None) == 1      # v_scale 0
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, float("nan"), 1.0, ctypes.byref(d), None) == 1
    assert f(FAKE, FAKE, FAKE, 4, FAKE, FAKE, float("inf"), 1.0, ctypes.byref(d), None) == 1
    assert f(None, None, None, 0, None, None, 1.0, 1.0, ctypes.byref(d), None) == 0
    assert f(MISALIGNED, FAKE, FAKE, 4, FAKE, FAKE, 1.0, 1.0, ctypes.byref(d), None) == 1
    g = cuda_lib.sgl_decode_attention_fp8
    need = B.decode_workspace_bytes(2, 64, d)
    assert g(FAKE, FAKE, FAKE, -1.0, 1.0, FAKE, 4, 64, FAKE, FAKE, 2, 64, FAKE, FAKE, need,
             ctypes.byref(d), None) == 1
    assert g(FAKE, FAKE, FAKE, 1.0, 1.0, FAKE, 4, 64, FAKE, FAKE, 2, 64, FAKE, None, need,
             ctypes.byref(d), None) == 3
    assert g(FAKE, FAKE, FAKE, 1.0, 1.0, FAKE, 4, 64, FAKE, FAKE, 0, 64, FAKE, FAKE, need,
             ctypes.byref(d), None) == 0


def test_fp8_extend_and_cascade_validation(cuda_lib):
    """The e4m3 extend takes no k_new / v_new (the suffix is read from the
    pool) and rejects bad scales; the e4m3 cascade validates like the bf16 one."""
    d = _dims()
    x = cuda_lib.sgl_extend_attention_fp8

    def ext(**kw):
        a = dict(q=FAKE, pk=FAKE, pv=FAKE, ks=1.0, vs=1.0, rtt=FAKE, rows=4, stride=64, rpi=FAKE,
                 pl=FAKE, el=FAKE, batch=2, total=10, max_e=6, max_p=30, out=FAKE, ws=FAKE, wsb=256)
        a.update(kw)
        return x(a["q"], a["pk"], a["pv"], a["ks"], a["vs"], a["rtt"], a["rows"], a["stride"], a["rpi"],
                 a["pl"], a["el"], a["batch"], a["total"], a["max_e"], a["max_p"], a["out"], a["ws"],
                 a["wsb"], ctypes.byref(d), None)
    assert ext(ks=0.0) == 1 and ext(vs=float("nan")) == 1 and ext(ks=float("inf")) == 1
    assert ext(batch=0) == 0
    assert ext(q=None) == 1 and ext(pk=MISALIGNED) == 1 and ext(out=MISALIGNED) == 1
    assert ext(max_e=11) == 1
    assert ext(ws=None) == 3 and ext(wsb=16) == 3
    dd = _dims(head_dim=96)
    assert x(FAKE, FAKE, FAKE, 1.0, 1.0, FAKE, 4, 64, FAKE, FAKE, FAKE, 2, 10, 6, 30, FAKE, FAKE, 256,
             ctypes.byref(dd), None) == 2
    c = cuda_lib.sgl_cascade_decode_attention_fp8
    dc = _dims(num_q_heads=16, num_kv_heads=4)
    need = B.cascade_decode_workspace_bytes(8, 512, 3, dc)

    def casc(**kw):
        a = dict(ks=1.0, vs=1.0, q=FAKE, gs=FAKE, n_groups=2, max_d=3, ws=FAKE, wsb=need)
        a.update(kw)
        return c(a["q"], FAKE, FAKE, a["ks"], a["vs"], FAKE, 8, 512, FAKE, FAKE, 8, 512, a["gs"], FAKE, FAKE,
                 FAKE, FAKE, a["n_groups"], 4, a["max_d"], FAKE, a["ws"], a["wsb"], ctypes.byref(dc), None)
    assert casc(ks=-1.0) == 1 and casc(vs=0.0) == 1
    assert casc(gs=None) == 1 and casc(max_d=0) == 1 and casc(q=MISALIGNED) == 1
    assert casc(ws=None) == 3 and casc(wsb=need - 1) == 3
    ch = cuda_lib.sgl_check_extend_fp8_indices
    assert ch(FAKE, 0, 64, FAKE, FAKE, FAKE, 2, 10, 6, 30, 1024, FAKE, None) == 1
    assert ch(FAKE, 4, 64, FAKE, FAKE, FAKE, 0, 0, 0, 0, 1024, FAKE, None) == 0


def test_check_calls_validate_on_host(cuda_lib):
    assert cuda_lib.sgl_check_store_kv_indices(FAKE, 4, 1024, FAKE, 16, None, None) == 1
    assert cuda_lib.sgl_check_store_kv_indices(FAKE, 4, 1024, FAKE, 16, FAKE, None) == 3  # bitmap small
    assert cuda_lib.sgl_check_store_kv_indices(FAKE, 0, 1024, None, 0, FAKE, None) == 0
    assert cuda_lib.sgl_check_decode_indices(FAKE, 0, 64, FAKE, FAKE, 2, 64, 1024, FAKE, None) == 1
    assert cuda_lib.sgl_check_extend_indices(FAKE, 4, 64, FAKE, FAKE, FAKE, 0, 0, 0, 0, 1024, FAKE, None) == 0


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle, and its binding has no
    non-CUDA code path."""
    pkg = os.path.dirname(B.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                src = open(os.path.join(root, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f


def test_wait_limit_setter_returns_the_previous_limit():
    """sgl_set_device_wait_limit_ns is host state only: it returns the limit
    it replaces, and 0 restores the 2 s default."""
    from radixattention_prefix_shared_gb300 import binding as B
    lib = B.lib()
    default = 2_000_000_000
    assert lib.sgl_set_device_wait_limit_ns(12345) == default
    assert lib.sgl_set_device_wait_limit_ns(0) == 12345
    assert lib.sgl_set_device_wait_limit_ns(0) == default


def test_mixed_validation(cuda_lib):
    """sgl_mixed_attention checks both batches' arguments (the extend's, then
    the decode's) and its SM split before anything is launched."""
    d = _dims(num_q_heads=16, num_kv_heads=8)
    need = B.decode_workspace_bytes(2, 64, d)
    f = cuda_lib.sgl_mixed_attention

    def call(dims=d, **kw):
        a = dict(qe=FAKE, k=FAKE, v=FAKE, erpi=FAKE, pl=FAKE, el=FAKE, eb=2, total=10, max_e=6, max_p=30,
                 oe=FAKE, ews=FAKE, ewsb=256, qd=FAKE, drpi=FAKE, sl=FAKE, db=2, max_s=64, od=FAKE,
                 dws=FAKE, dwsb=need, pk=FAKE, pv=FAKE, rtt=FAKE, rows=4, stride=64, sms=-1)
        a.update(kw)
        return f(a["qe"], a["k"], a["v"], a["erpi"], a["pl"], a["el"], a["eb"], a["total"], a["max_e"],
                 a["max_p"], a["oe"], a["ews"], a["ewsb"], a["qd"], a["drpi"], a["sl"], a["db"], a["max_s"],
                 a["od"], a["dws"], a["dwsb"], a["pk"], a["pv"], a["rtt"], a["rows"], a["stride"], a["sms"],
                 ctypes.byref(dims) if dims is not None else None, None)
    assert call(eb=0, db=0, sms=0) == 0                  # both batches empty: nothing to launch
    assert call() == 1                                   # extend_sms < 0
    assert call(dims=None) == 1
    assert call(qe=None) == 1                            # extend argument
    assert call(max_e=11) == 1                           # max_extend above total_extend
    assert call(ews=None) == 3                           # extend workspace
    assert call(sl=None) == 1                            # decode argument
    assert call(max_s=0) == 1
    assert call(dwsb=need - 1) == 3                      # decode workspace
    assert call(dims=_dims(head_dim=32)) == 2
