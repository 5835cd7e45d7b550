"""FP8 (e4m3) KV pool: encoding, store and decode, float64 (test infrastructure
only; see the package docstring).

"Inside SGLang", Step 6 (Decide how much memory becomes KV cache): with
``--kv-cache-dtype fp8_e4m3`` each token's K and V cost half the bytes; the
attention backend reads FP8 directly, and K and V carry scales from the
checkpoint (1.0 when missing).

Readings taken where the page leaves a step open:
  * the format is e4m3 "fn": 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
    bits, subnormals, no infinities, codes 0x7f / 0xff are NaN, largest
    finite value 448;
  * one scale per tensor (K and V separately); a stored code c stands for
    ``decode(c) * scale``;
  * every key and value an attention over an e4m3 pool reads comes from the
    pool: an EXTEND's suffix rows are stored (quantised) before it runs and
    read back through ``req_to_token`` like its prefix, so extend, decode and
    cascade decode all see the same dequantised values for a position;
  * quantising takes the float32 quotient ``x / scale`` (IEEE division,
    round to nearest even) and rounds it to e4m3 to nearest, ties to even,
    saturating to +-448 (finite inputs never become NaN).
"""
from __future__ import annotations

import numpy as np

from .attention import (_cascade_decode, _kv_head_of, _softmax_attend, _visible_keys, bf16_bits_to_f64,
                        default_scale)

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 codes (uint8) -> exact float64 values (NaN codes -> NaN)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def _round_half_even(x: np.ndarray) -> np.ndarray:
    f = np.floor(x)
    r = x - f
    up = (r > 0.5) | ((r == 0.5) & (np.fmod(f, 2.0) != 0))
    return f + up


def e4m3_encode(x_f32) -> np.ndarray:
    """Finite float32 values -> e4m3 codes, nearest (ties to even), saturating."""
    x = np.asarray(x_f32, dtype=np.float32).astype(np.float64)   # exact
    neg = np.signbit(x)
    a = np.abs(x)
    code = np.zeros(a.shape, np.int64)
    # subnormal range: multiples of 2^-9 below 2^-6 (q = 8 is the smallest normal)
    sub = a < 2.0 ** -6
    code[sub] = _round_half_even(a[sub] * 2.0 ** 9).astype(np.int64)
    nrm = ~sub
    mant, ex = np.frexp(a[nrm])                  # a = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1                                   # a = (2 mant) * 2^e, 2 mant in [1, 2)
    q = _round_half_even((2.0 * mant - 1.0) * 8.0).astype(np.int64)
    carry = q == 8
    e = e + carry
    q = np.where(carry, 0, q)
    code[nrm] = ((e + 7) << 3) | q
    code = np.minimum(code, 0x7E)                # saturate at 448
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def quantize(bits_bf16, scale: float) -> np.ndarray:
    """bf16 values (bit patterns) -> e4m3 codes of ``x / scale`` (float32 quotient)."""
    x = bf16_bits_to_f64(bits_bf16).astype(np.float32)
    return e4m3_encode(x / np.float32(scale))


def store_kv_fp8(pool_k, pool_v, k_new, v_new, slots, k_scale: float, v_scale: float):
    """``pool[slots[i]] = quantize(new[i])`` on copies of the uint8 pools."""
    pk = np.array(pool_k, copy=True)
    pv = np.array(pool_v, copy=True)
    slots = np.asarray(slots, dtype=np.int64)
    qk, qv = quantize(k_new, k_scale), quantize(v_new, v_scale)
    for i, s in enumerate(slots):
        pk[s] = qk[i]
        pv[s] = qv[i]
    return pk, pv


def decode_attention_fp8(q, pool_k, pool_v, k_scale: float, v_scale: float, req_to_token,
                         req_pool_idx, seq_lens, num_kv_heads: int, sm_scale=None,
                         requests=None) -> np.ndarray:
    """DECODE attention over an e4m3 pool, float64: the keys and values of a
    request are its rows read through ``req_to_token``, dequantised
    (``decode(code) * scale``); then the same softmax attention as
    ``decode_attention``."""
    q = np.asarray(q)
    B, Hq, D = q.shape
    scale = default_scale(D) if sm_scale is None else float(sm_scale)
    want = np.arange(B) if requests is None else np.asarray(requests, dtype=np.int64)
    out = np.zeros((want.size, Hq, D), np.float64)
    for n, r in enumerate(want):
        slots = np.asarray(req_to_token[int(req_pool_idx[r]), : int(seq_lens[r])], dtype=np.int64)
        K = e4m3_decode(pool_k[slots]) * float(k_scale)
        V = e4m3_decode(pool_v[slots]) * float(v_scale)
        qr = bf16_bits_to_f64(q[r])
        for h in range(Hq):
            kh = _kv_head_of(h, Hq, num_kv_heads)
            out[n, h] = _softmax_attend(qr[h], K[:, kh], V[:, kh], scale)
    return out


def _dequant(codes, scale: float) -> np.ndarray:
    return e4m3_decode(codes) * float(scale)


def extend_attention_fp8(q, pool_k, pool_v, k_scale: float, v_scale: float, req_to_token,
                         req_pool_idx, prefix_lens, extend_lens, num_kv_heads: int, sm_scale=None,
                         tokens=None) -> np.ndarray:
    """EXTEND attention over an e4m3 pool, float64.

    q [T, Hq, D] holds the suffix queries of all requests back to back
    (request r's rows start at the exclusive prefix sum of extend_lens).
    Request r's keys and values are its row ``req_to_token[req_pool_idx[r],
    0 : p + e]`` -- cached prefix and freshly stored suffix alike --
    dequantised; suffix query i (position p + i) attends to keys 0 .. p + i,
    as in ``extend_attention``.  Returns [T, Hq, D] (or the listed rows)."""
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
        slots = np.asarray(req_to_token[int(req_pool_idx[r]), : p + e], dtype=np.int64)
        K = _dequant(pool_k[slots], k_scale)         # [p+e, Hkv, D]
        V = _dequant(pool_v[slots], v_scale)
        for n in np.nonzero(req_of == r)[0]:
            i = int(want[n]) - o
            L = _visible_keys(p, i)
            qi = bf16_bits_to_f64(q[o + i])
            for h in range(Hq):
                kh = _kv_head_of(h, Hq, num_kv_heads)
                out[n, h] = _softmax_attend(qi[h], K[:L, kh], V[:L, kh], scale)
    return out


def cascade_decode_attention_fp8(q, pool_k, pool_v, k_scale: float, v_scale: float, req_to_token,
                                 req_pool_idx, seq_lens, group_start, group_len, group_depth,
                                 member_off, members, num_kv_heads: int, sm_scale=None,
                                 requests=None) -> np.ndarray:
    """``cascade_decode_attention`` over an e4m3 pool: each group's keys (read
    once, from its first member's row) and each request's private tail are
    dequantised (``decode(code) * scale``) before the softmax states are
    formed and merged."""
    return _cascade_decode(q, lambda slots: (_dequant(pool_k[slots], k_scale), _dequant(pool_v[slots], v_scale)),
                           req_to_token, req_pool_idx, seq_lens, group_start, group_len, group_depth,
                           member_off, members, num_kv_heads, sm_scale, requests)
