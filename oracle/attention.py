"""fp64 reference definitions (test infrastructure only; see package docstring).

Readings taken where the pages leave a step open:
  * GQA head map: query head ``h`` reads KV head ``h // (Hq // Hkv)``
    (contiguous groups; "Inside SGLang", Step 3 says two query heads share each
    KV head but not which two).
  * Causal alignment in EXTEND: suffix query ``i`` of a request with prefix
    length ``p`` sits at absolute position ``p + i`` and sees keys ``0 .. p+i``
    (all of the prefix, suffix keys up to itself) -- i.e. the last rows of full
    causal attention over prefix+suffix.
  * Decode: ``seq_len`` includes the new token, whose K/V store_kv wrote first;
    the query sees keys ``0 .. seq_len-1``, all read through req_to_token.
  * Scale: ``1/sqrt(head_dim)`` unless given.
"""
from __future__ import annotations

import math

import numpy as np


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def default_scale(head_dim: int) -> float:
    """Softmax scale 1/sqrt(head_dim) ("Inside SGLang", Step 3: 0.0884 at 128)."""
    return 1.0 / math.sqrt(head_dim)


# ---------------------------------------------------------------- store_kv

def store_kv(pool_k, pool_v, k_new, v_new, slots):
    """Index assignment ``pool[slots[i]] = new[i]`` on copies of the pools.

    Bit patterns are copied unchanged (uint16 in, uint16 out)."""
    pk = np.array(pool_k, copy=True)
    pv = np.array(pool_v, copy=True)
    slots = np.asarray(slots, dtype=np.int64)
    for i, s in enumerate(slots):
        pk[s] = k_new[i]
        pv[s] = v_new[i]
    return pk, pv


def store_kv_range(pool_k, pool_v, k_new, v_new, start: int):
    """The contiguous-range form: ``pool[start:start+n] = new``."""
    pk = np.array(pool_k, copy=True)
    pv = np.array(pool_v, copy=True)
    n = len(k_new)
    pk[start: start + n] = k_new
    pv[start: start + n] = v_new
    return pk, pv


# ---------------------------------------------------------------- gathers

def request_kv(pool_k, pool_v, req_to_token, row: int, n: int):
    """Walk ``req_to_token[row, 0:n]`` and read those slots' K and V rows.

    Returns float64 arrays [n, Hkv, D]."""
    slots = np.asarray(req_to_token[int(row), : int(n)], dtype=np.int64)
    return bf16_bits_to_f64(pool_k[slots]), bf16_bits_to_f64(pool_v[slots])


def _kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    return h // (num_q_heads // num_kv_heads)


def _visible_keys(prefix_len: int, i: int) -> int:
    """Number of keys suffix query ``i`` sees (positions 0 .. prefix_len+i)."""
    return prefix_len + i + 1


def _softmax_attend(qv: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * K @ q) @ V for one query vector; K, V [n, D]."""
    s = scale * (K @ qv)
    m = np.max(s)
    w = np.exp(s - m)
    return (w @ V) / np.sum(w)


# ---------------------------------------------------------------- extend

def extend_attention(q, k_new, v_new, pool_k, pool_v, req_to_token, req_pool_idx,
                     prefix_lens, extend_lens, num_kv_heads: int, sm_scale=None,
                     tokens=None) -> np.ndarray:
    """EXTEND attention, float64.

    q [T, Hq, D], k_new/v_new [T, Hkv, D] hold the suffix tokens of all
    requests back to back (request r's rows start at the exclusive prefix sum
    of extend_lens).  The prefix K/V of request r is read from the pool through
    ``req_to_token[req_pool_idx[r], 0:prefix_lens[r]]``.  Returns [T, Hq, D]
    (or only the rows listed in ``tokens``, in that order).
    """
    q = np.asarray(q)
    T, Hq, D = q.shape
    scale = default_scale(D) if sm_scale is None else float(sm_scale)
    prefix_lens = np.asarray(prefix_lens, dtype=np.int64)
    extend_lens = np.asarray(extend_lens, dtype=np.int64)
    offs = np.concatenate([[0], np.cumsum(extend_lens)])
    want = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = np.zeros((want.size, Hq, D), np.float64)
    req_of = np.searchsorted(offs, want, side="right") - 1
    for r in np.unique(req_of):
        p, e, o = int(prefix_lens[r]), int(extend_lens[r]), int(offs[r])
        Kp, Vp = request_kv(pool_k, pool_v, req_to_token, req_pool_idx[r], p)
        Ks = bf16_bits_to_f64(k_new[o: o + e])
        Vs = bf16_bits_to_f64(v_new[o: o + e])
        K = np.concatenate([Kp, Ks], axis=0)          # [p+e, Hkv, D]
        V = np.concatenate([Vp, Vs], axis=0)
        for n in np.nonzero(req_of == r)[0]:
            i = int(want[n]) - o
            L = _visible_keys(p, i)
            qi = bf16_bits_to_f64(q[o + i])               # [Hq, D]
            for h in range(Hq):
                kh = _kv_head_of(h, Hq, num_kv_heads)
                out[n, h] = _softmax_attend(qi[h], K[:L, kh], V[:L, kh], scale)
    return out


# ---------------------------------------------------------------- decode

def decode_attention(q, pool_k, pool_v, req_to_token, req_pool_idx, seq_lens,
                     num_kv_heads: int, sm_scale=None, requests=None) -> np.ndarray:
    """DECODE attention, float64: one query per request over all ``seq_len``
    keys of its row (the new token's K/V already stored).  q [B, Hq, D];
    returns [B, Hq, D] (or only the requests listed)."""
    q = np.asarray(q)
    B, Hq, D = q.shape
    scale = default_scale(D) if sm_scale is None else float(sm_scale)
    want = np.arange(B) if requests is None else np.asarray(requests, dtype=np.int64)
    out = np.zeros((want.size, Hq, D), np.float64)
    for n, r in enumerate(want):
        K, V = request_kv(pool_k, pool_v, req_to_token, req_pool_idx[r], seq_lens[r])
        qr = bf16_bits_to_f64(q[r])
        for h in range(Hq):
            kh = _kv_head_of(h, Hq, num_kv_heads)
            out[n, h] = _softmax_attend(qr[h], K[:, kh], V[:, kh], scale)
    return out
