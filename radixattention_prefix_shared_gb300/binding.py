"""Thin ctypes binding of libsgl_attn.so (names follow the C ABI).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (PyTorch provides device memory and streams);
bf16 tensors are ``torch.bfloat16``, indices ``torch.int32``.  A call that
the library rejects raises ``SglError``.  If the library is missing it is
built from source with nvcc; if that is impossible the import fails loudly --
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_i32, c_i64, c_f32, c_size, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

STATUS = {0: "SGL_OK", 1: "SGL_ERR_INVALID_ARG", 2: "SGL_ERR_UNSUPPORTED", 3: "SGL_ERR_WORKSPACE",
          4: "SGL_ERR_CUDA", 5: "SGL_ERR_INDEX"}


class SglError(RuntimeError):
    def __init__(self, func: str, code: int):
        super().__init__(f"{func} failed: {STATUS.get(code, code)}")
        self.code = code


class sgl_attn_dims(ctypes.Structure):
    _fields_ = [("num_q_heads", c_i32), ("num_kv_heads", c_i32), ("head_dim", c_i32),
                ("pool_size", c_i64), ("sm_scale", c_f32)]


_P = ctypes.POINTER
_SIGS = {
    "sgl_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "sgl_version": (ctypes.c_char_p, []),
    "sgl_set_device_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "sgl_store_kv": (ctypes.c_int, [c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, _P(sgl_attn_dims), c_vp]),
    "sgl_extend_attention": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_vp, c_vp,
                                            c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_size,
                                            _P(sgl_attn_dims), c_vp]),
    "sgl_decode_attention": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_i32,
                                            c_i32, c_vp, c_vp, c_size, _P(sgl_attn_dims), c_vp]),
    "sgl_decode_attention_noalloc": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_i32,
                                                    c_i32, c_vp, _P(sgl_attn_dims), c_vp]),
    "sgl_mixed_attention": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32,
                                           c_vp, c_vp, c_size, c_vp, c_vp, c_vp, c_i32, c_i32, c_vp, c_vp,
                                           c_size, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, _P(sgl_attn_dims),
                                           c_vp]),
    "sgl_extend_workspace_bytes": (c_size, [c_i32, c_i32, _P(sgl_attn_dims)]),
    "sgl_decode_workspace_bytes": (c_size, [c_i32, c_i32, _P(sgl_attn_dims)]),
    "sgl_check_store_kv_indices": (ctypes.c_int, [c_vp, c_i32, c_i64, c_vp, c_size, c_vp, c_vp]),
    "sgl_check_extend_indices": (ctypes.c_int, [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32,
                                                c_i32, c_i64, c_vp, c_vp]),
    "sgl_check_decode_indices": (ctypes.c_int, [c_vp, c_i32, c_i32, c_vp, c_vp, c_i32, c_i32, c_i64,
                                                c_vp, c_vp]),
    "sgl_cascade_decode_attention": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_vp, c_vp,
                                                    c_i32, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32,
                                                    c_i32, c_i32, c_vp, c_vp, c_size, _P(sgl_attn_dims),
                                                    c_vp]),
    "sgl_cascade_decode_workspace_bytes": (c_size, [c_i32, c_i32, c_i32, _P(sgl_attn_dims)]),
    "sgl_radix_create": (c_vp, []),
    "sgl_radix_destroy": (None, [c_vp]),
    "sgl_radix_match_prefix": (c_i32, [c_vp, c_vp, c_i32, c_vp, c_i32, _P(c_i64)]),
    "sgl_radix_insert": (c_i32, [c_vp, c_vp, c_vp, c_i32]),
    "sgl_radix_inc_lock_ref": (ctypes.c_int, [c_vp, c_i64]),
    "sgl_radix_dec_lock_ref": (ctypes.c_int, [c_vp, c_i64]),
    "sgl_radix_evict": (c_i32, [c_vp, c_i32, c_vp, c_i32]),
    "sgl_radix_evictable_tokens": (c_i64, [c_vp]),
    "sgl_radix_protected_tokens": (c_i64, [c_vp]),
    "sgl_radix_groups": (c_i32, [c_vp, c_vp, c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, _P(c_i32)]),
    "sgl_store_kv_fp8": (ctypes.c_int, [c_vp, c_vp, c_vp, c_i32, c_vp, c_vp, c_f32, c_f32,
                                        _P(sgl_attn_dims), c_vp]),
    "sgl_decode_attention_fp8": (ctypes.c_int, [c_vp, c_vp, c_vp, c_f32, c_f32, c_vp, c_i32, c_i32, c_vp,
                                                c_vp, c_i32, c_i32, c_vp, c_vp, c_size, _P(sgl_attn_dims),
                                                c_vp]),
    "sgl_extend_attention_fp8": (ctypes.c_int, [c_vp, c_vp, c_vp, c_f32, c_f32, c_vp, c_i32, c_i32, c_vp,
                                                c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_vp, c_size,
                                                _P(sgl_attn_dims), c_vp]),
    "sgl_cascade_decode_attention_fp8": (ctypes.c_int, [c_vp, c_vp, c_vp, c_f32, c_f32, c_vp, c_i32, c_i32,
                                                        c_vp, c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_vp,
                                                        c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_size,
                                                        _P(sgl_attn_dims), c_vp]),
    "sgl_check_extend_fp8_indices": (ctypes.c_int, [c_vp, c_i32, c_i32, c_vp, c_vp, c_vp, c_i32, c_i32,
                                                    c_i32, c_i32, c_i64, c_vp, c_vp]),
    "sgl_check_cascade_scratch_bytes": (c_size, [c_i32, c_i32]),
    "sgl_check_cascade_groups": (ctypes.c_int, [c_vp, c_i32, c_i32, c_vp, c_vp, c_i32, c_vp, c_vp, c_vp,
                                                c_vp, c_vp, c_i32, c_i32, c_i32, c_vp, c_size, c_vp,
                                                c_vp]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the C-ABI library."""
    global _lib
    if _lib is None:
        path = _build.LIB_PATH
        if not os.path.exists(path) or os.environ.get("SGL_ATTN_REBUILD"):
            path = _build.build()
        cdll = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            f = getattr(cdll, name)
            f.restype = res
            f.argtypes = args
        _lib = cdll
    return _lib


def lib_path() -> str:
    return _build.LIB_PATH


def _check(name: str, code: int) -> None:
    if code != 0:
        raise SglError(name, code)


def make_dims(num_q_heads, num_kv_heads, head_dim, pool_size, sm_scale=0.0) -> sgl_attn_dims:
    return sgl_attn_dims(int(num_q_heads), int(num_kv_heads), int(head_dim), int(pool_size), float(sm_scale))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dims_for(q_or_new, pool_k, sm_scale):
    return make_dims(q_or_new.shape[1] if q_or_new is not None else pool_k.shape[1],
                     pool_k.shape[1], pool_k.shape[2], pool_k.shape[0], sm_scale)


# ----------------------------------------------------------------- calls

def sgl_store_kv(k_new, v_new, slots, pool_k, pool_v, stream=None):
    """pool_k[slots[i]] = k_new[i]; pool_v[slots[i]] = v_new[i]."""
    d = make_dims(pool_k.shape[1], pool_k.shape[1], pool_k.shape[2], pool_k.shape[0])
    _check("sgl_store_kv", lib().sgl_store_kv(_ptr(k_new), _ptr(v_new), _ptr(slots), int(slots.shape[0]),
                                              _ptr(pool_k), _ptr(pool_v), ctypes.byref(d), _stream(stream)))


def extend_workspace_bytes(batch, total_extend, dims: sgl_attn_dims) -> int:
    return int(lib().sgl_extend_workspace_bytes(int(batch), int(total_extend), ctypes.byref(dims)))


def decode_workspace_bytes(batch, max_seq_len, dims: sgl_attn_dims) -> int:
    return int(lib().sgl_decode_workspace_bytes(int(batch), int(max_seq_len), ctypes.byref(dims)))


def new_workspace(nbytes: int, device):
    """A zero-filled device byte buffer (16-byte aligned by the allocator)."""
    import torch
    return torch.zeros(max(16, int(nbytes)), dtype=torch.uint8, device=device)


def sgl_extend_attention(q, k_new, v_new, pool_k, pool_v, req_to_token, req_pool_idx, prefix_lens,
                         extend_lens, out=None, *, max_extend, max_prefix=0, total_extend=None,
                         workspace=None, sm_scale=0.0, stream=None):
    """Attention of the suffix tokens over cached prefix + causal suffix.

    ``max_extend``/``max_prefix``/``total_extend`` are host-side values (the
    library never reads device memory on the host)."""
    import torch
    T = int(q.shape[0]) if total_extend is None else int(total_extend)
    d = _dims_for(q, pool_k, sm_scale)
    if out is None:
        out = torch.empty_like(q)
    B = int(req_pool_idx.shape[0])
    if workspace is None:
        workspace = new_workspace(extend_workspace_bytes(B, T, d), q.device)
    _check("sgl_extend_attention", lib().sgl_extend_attention(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(pool_k), _ptr(pool_v), _ptr(req_to_token),
        int(req_to_token.shape[0]), int(req_to_token.shape[1]), _ptr(req_pool_idx), _ptr(prefix_lens),
        _ptr(extend_lens), B, T, int(max_extend), int(max_prefix), _ptr(out), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), ctypes.byref(d), _stream(stream)))
    return out


def sgl_mixed_attention(q_ext, k_new, v_new, ext_req_pool_idx, prefix_lens, extend_lens, q_dec,
                        dec_req_pool_idx, seq_lens, pool_k, pool_v, req_to_token, out_ext=None, out_dec=None, *,
                        max_extend, max_prefix=0, max_seq_len, total_extend=None, ext_workspace=None,
                        dec_workspace=None, extend_sms=0, sm_scale=0.0, stream=None):
    """An extend batch and a decode batch over the same pools in one launch
    (outputs equal to sgl_extend_attention's and sgl_decode_attention's)."""
    import torch
    T = int(q_ext.shape[0]) if total_extend is None else int(total_extend)
    d = _dims_for(q_ext, pool_k, sm_scale)
    Be, Bd = int(ext_req_pool_idx.shape[0]), int(q_dec.shape[0])
    if out_ext is None:
        out_ext = torch.empty_like(q_ext)
    if out_dec is None:
        out_dec = torch.empty_like(q_dec)
    if ext_workspace is None:
        ext_workspace = new_workspace(extend_workspace_bytes(Be, T, d), q_ext.device)
    if dec_workspace is None:
        dec_workspace = new_workspace(decode_workspace_bytes(Bd, max_seq_len, d), q_dec.device)
    _check("sgl_mixed_attention", lib().sgl_mixed_attention(
        _ptr(q_ext), _ptr(k_new), _ptr(v_new), _ptr(ext_req_pool_idx), _ptr(prefix_lens), _ptr(extend_lens),
        Be, T, int(max_extend), int(max_prefix), _ptr(out_ext), _ptr(ext_workspace),
        int(ext_workspace.numel() * ext_workspace.element_size()), _ptr(q_dec), _ptr(dec_req_pool_idx),
        _ptr(seq_lens), Bd, int(max_seq_len), _ptr(out_dec), _ptr(dec_workspace),
        int(dec_workspace.numel() * dec_workspace.element_size()), _ptr(pool_k), _ptr(pool_v),
        _ptr(req_to_token), int(req_to_token.shape[0]), int(req_to_token.shape[1]), int(extend_sms),
        ctypes.byref(d), _stream(stream)))
    return out_ext, out_dec


def sgl_decode_attention(q, pool_k, pool_v, req_to_token, req_pool_idx, seq_lens, out=None, *,
                         max_seq_len, workspace=None, sm_scale=0.0, stream=None):
    """One query per request over all ``seq_len`` keys of its row."""
    import torch
    d = _dims_for(q, pool_k, sm_scale)
    if out is None:
        out = torch.empty_like(q)
    B = int(q.shape[0])
    if workspace is None:
        workspace = new_workspace(decode_workspace_bytes(B, max_seq_len, d), q.device)
    _check("sgl_decode_attention", lib().sgl_decode_attention(
        _ptr(q), _ptr(pool_k), _ptr(pool_v), _ptr(req_to_token), int(req_to_token.shape[0]),
        int(req_to_token.shape[1]), _ptr(req_pool_idx), _ptr(seq_lens), B, int(max_seq_len), _ptr(out),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()), ctypes.byref(d),
        _stream(stream)))
    return out


def sgl_check_store_kv_indices(slots, pool_size, d_error, bitmap=None, stream=None):
    import torch
    need = ((int(pool_size) + 31) // 32 * 4 + 15) // 16 * 16
    if bitmap is None:
        bitmap = torch.empty(need, dtype=torch.uint8, device=slots.device)
    _check("sgl_check_store_kv_indices", lib().sgl_check_store_kv_indices(
        _ptr(slots), int(slots.shape[0]), int(pool_size), _ptr(bitmap),
        int(bitmap.numel()), _ptr(d_error), _stream(stream)))


def sgl_check_extend_indices(req_to_token, req_pool_idx, prefix_lens, extend_lens, *, total_extend,
                             max_extend, max_prefix, pool_size, d_error, stream=None, fp8=False):
    """``fp8``: the e4m3 extend's check (suffix positions' slots too)."""
    name = "sgl_check_extend_fp8_indices" if fp8 else "sgl_check_extend_indices"
    _check(name, getattr(lib(), name)(
        _ptr(req_to_token), int(req_to_token.shape[0]), int(req_to_token.shape[1]), _ptr(req_pool_idx),
        _ptr(prefix_lens), _ptr(extend_lens), int(req_pool_idx.shape[0]), int(total_extend),
        int(max_extend), int(max_prefix), int(pool_size), _ptr(d_error), _stream(stream)))


def sgl_check_decode_indices(req_to_token, req_pool_idx, seq_lens, *, max_seq_len, pool_size, d_error,
                             stream=None):
    _check("sgl_check_decode_indices", lib().sgl_check_decode_indices(
        _ptr(req_to_token), int(req_to_token.shape[0]), int(req_to_token.shape[1]), _ptr(req_pool_idx),
        _ptr(seq_lens), int(req_pool_idx.shape[0]), int(max_seq_len), int(pool_size), _ptr(d_error),
        _stream(stream)))


# ----------------------------------------------------------------- cascade

def cascade_decode_workspace_bytes(batch, max_seq_len, max_depth, dims: sgl_attn_dims) -> int:
    return int(lib().sgl_cascade_decode_workspace_bytes(int(batch), int(max_seq_len), int(max_depth),
                                                        ctypes.byref(dims)))


def sgl_cascade_decode_attention(q, pool_k, pool_v, req_to_token, req_pool_idx, seq_lens,
                                 group_start, group_len, group_depth, group_member_off, group_members,
                                 out=None, *, max_seq_len, max_group_members, max_depth,
                                 workspace=None, sm_scale=0.0, stream=None, kv_scales=None):
    """Decode attention with shared-prefix groups read once per group.

    ``group_*`` are int32 device tensors (CSR members); ``max_seq_len``,
    ``max_group_members`` and ``max_depth`` are host values.  A new workspace
    is zero-filled; a reused one must keep its first 256 bytes zero.
    ``kv_scales=(k_scale, v_scale)`` selects the e4m3-pool entry point."""
    import torch
    d = _dims_for(q, pool_k, sm_scale)
    if out is None:
        out = torch.empty_like(q)
    B = int(q.shape[0])
    G = int(group_start.shape[0])
    if workspace is None:
        workspace = new_workspace(cascade_decode_workspace_bytes(B, max_seq_len, max_depth, d), q.device)
    if kv_scales is None:
        name, head = "sgl_cascade_decode_attention", (_ptr(q), _ptr(pool_k), _ptr(pool_v))
    else:
        name = "sgl_cascade_decode_attention_fp8"
        head = (_ptr(q), _ptr(pool_k), _ptr(pool_v), float(kv_scales[0]), float(kv_scales[1]))
    _check(name, getattr(lib(), name)(
        *head, _ptr(req_to_token), int(req_to_token.shape[0]),
        int(req_to_token.shape[1]), _ptr(req_pool_idx), _ptr(seq_lens), B, int(max_seq_len),
        _ptr(group_start), _ptr(group_len), _ptr(group_depth), _ptr(group_member_off), _ptr(group_members),
        G, int(max_group_members), int(max_depth), _ptr(out), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), ctypes.byref(d), _stream(stream)))
    return out


def sgl_check_cascade_groups(req_to_token, req_pool_idx, seq_lens, group_start, group_len, group_depth,
                             group_member_off, group_members, *, max_group_members, max_depth, d_error,
                             scratch=None, stream=None):
    import torch
    B = int(req_pool_idx.shape[0])
    need = int(lib().sgl_check_cascade_scratch_bytes(B, int(max_depth)))
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=req_to_token.device)
    _check("sgl_check_cascade_groups", lib().sgl_check_cascade_groups(
        _ptr(req_to_token), int(req_to_token.shape[0]), int(req_to_token.shape[1]), _ptr(req_pool_idx),
        _ptr(seq_lens), B, _ptr(group_start), _ptr(group_len), _ptr(group_depth), _ptr(group_member_off),
        _ptr(group_members), int(group_start.shape[0]), int(max_group_members), int(max_depth),
        _ptr(scratch), int(scratch.numel()), _ptr(d_error), _stream(stream)))


# ----------------------------------------------------------------- FP8 pool

def sgl_store_kv_fp8(k_new, v_new, slots, pool_k, pool_v, k_scale, v_scale, stream=None):
    """pool[slots[i]] = e4m3(new[i] / scale) for K and V (pools: torch.uint8 [S, Hkv, D])."""
    d = make_dims(pool_k.shape[1], pool_k.shape[1], pool_k.shape[2], pool_k.shape[0])
    _check("sgl_store_kv_fp8", lib().sgl_store_kv_fp8(
        _ptr(k_new), _ptr(v_new), _ptr(slots), int(slots.shape[0]), _ptr(pool_k), _ptr(pool_v),
        float(k_scale), float(v_scale), ctypes.byref(d), _stream(stream)))


def sgl_decode_attention_fp8(q, pool_k, pool_v, k_scale, v_scale, req_to_token, req_pool_idx, seq_lens,
                             out=None, *, max_seq_len, workspace=None, sm_scale=0.0, stream=None):
    """Decode attention over an e4m3 pool (values are code * scale)."""
    import torch
    d = _dims_for(q, pool_k, sm_scale)
    if out is None:
        out = torch.empty_like(q)
    B = int(q.shape[0])
    if workspace is None:
        workspace = new_workspace(decode_workspace_bytes(B, max_seq_len, d), q.device)
    _check("sgl_decode_attention_fp8", lib().sgl_decode_attention_fp8(
        _ptr(q), _ptr(pool_k), _ptr(pool_v), float(k_scale), float(v_scale), _ptr(req_to_token),
        int(req_to_token.shape[0]), int(req_to_token.shape[1]), _ptr(req_pool_idx), _ptr(seq_lens), B,
        int(max_seq_len), _ptr(out), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        ctypes.byref(d), _stream(stream)))
    return out


def sgl_extend_attention_fp8(q, pool_k, pool_v, k_scale, v_scale, req_to_token, req_pool_idx, prefix_lens,
                             extend_lens, out=None, *, max_extend, max_prefix=0, total_extend=None,
                             workspace=None, sm_scale=0.0, stream=None):
    """Extend attention over an e4m3 pool: prefix AND suffix keys are read
    from the pool through ``req_to_token`` (the suffix stored first)."""
    import torch
    T = int(q.shape[0]) if total_extend is None else int(total_extend)
    d = _dims_for(q, pool_k, sm_scale)
    if out is None:
        out = torch.empty_like(q)
    B = int(req_pool_idx.shape[0])
    if workspace is None:
        workspace = new_workspace(extend_workspace_bytes(B, T, d), q.device)
    _check("sgl_extend_attention_fp8", lib().sgl_extend_attention_fp8(
        _ptr(q), _ptr(pool_k), _ptr(pool_v), float(k_scale), float(v_scale), _ptr(req_to_token),
        int(req_to_token.shape[0]), int(req_to_token.shape[1]), _ptr(req_pool_idx), _ptr(prefix_lens),
        _ptr(extend_lens), B, T, int(max_extend), int(max_prefix), _ptr(out), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), ctypes.byref(d), _stream(stream)))
    return out


# ----------------------------------------------------------------- radix tree

class RadixTree:
    """The library's radix tree of cached token runs (host side, C++).

    Token ids and slots are int sequences; node handles are ints."""

    def __init__(self):
        self._t = lib().sgl_radix_create()
        if not self._t:
            raise MemoryError("sgl_radix_create failed")

    def __del__(self):
        if getattr(self, "_t", None):
            lib().sgl_radix_destroy(self._t)
            self._t = None

    @staticmethod
    def _arr(xs):
        import numpy as np
        return np.ascontiguousarray(np.asarray(xs, dtype=np.int32))

    def match_prefix(self, tokens):
        """(matched length, slots along the path, last node handle)."""
        toks = self._arr(tokens)
        out = self._arr([0] * max(1, toks.size))
        node = c_i64(0)
        m = lib().sgl_radix_match_prefix(self._t, toks.ctypes.data, int(toks.size), out.ctypes.data,
                                         int(out.size), ctypes.byref(node))
        if m < 0:
            raise SglError("sgl_radix_match_prefix", 1)
        return int(m), out[:m].tolist(), int(node.value)

    def insert(self, tokens, slots):
        toks, sl = self._arr(tokens), self._arr(slots)
        if toks.size != sl.size:
            raise ValueError("one slot per token")
        m = lib().sgl_radix_insert(self._t, toks.ctypes.data, sl.ctypes.data, int(toks.size))
        if m < 0:
            raise SglError("sgl_radix_insert", 1)
        return int(m)

    def inc_lock_ref(self, node):
        _check("sgl_radix_inc_lock_ref", lib().sgl_radix_inc_lock_ref(self._t, int(node)))

    def dec_lock_ref(self, node):
        _check("sgl_radix_dec_lock_ref", lib().sgl_radix_dec_lock_ref(self._t, int(node)))

    def evict(self, num_tokens):
        cap = int(self.evictable_tokens) + 1
        out = self._arr([0] * cap)
        n = lib().sgl_radix_evict(self._t, int(num_tokens), out.ctypes.data, cap)
        if n < 0:
            raise SglError("sgl_radix_evict", 1)
        return out[:n].tolist()

    @property
    def evictable_tokens(self):
        return int(lib().sgl_radix_evictable_tokens(self._t))

    @property
    def protected_tokens(self):
        return int(lib().sgl_radix_protected_tokens(self._t))

    def groups(self, nodes):
        """Shared-prefix groups of a batch: (start, len, depth, member_off, members) int32 arrays."""
        import numpy as np
        hs = np.ascontiguousarray(np.asarray(nodes, dtype=np.int64))
        nm = c_i32(0)
        ng = lib().sgl_radix_groups(self._t, hs.ctypes.data, int(hs.size), None, None, None, None, None,
                                    0, 0, ctypes.byref(nm))
        if ng < 0:
            raise SglError("sgl_radix_groups", 1)
        start, length, depth = (np.zeros(ng, np.int32) for _ in range(3))
        off, mem = np.zeros(ng + 1, np.int32), np.zeros(max(1, nm.value), np.int32)
        ng2 = lib().sgl_radix_groups(self._t, hs.ctypes.data, int(hs.size), start.ctypes.data,
                                     length.ctypes.data, depth.ctypes.data, off.ctypes.data, mem.ctypes.data,
                                     ng, int(mem.size), ctypes.byref(nm))
        assert ng2 == ng
        return start, length, depth, off, mem[: nm.value]
