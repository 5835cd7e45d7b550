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


# ---------------------------------------------------------------- cascade

def partial_state(qv: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Softmax state of one query over a subset of its keys, float64:
    ``(m, l, acc)`` with ``m`` the largest score, ``l = sum_j exp(s_j - m)``
    and ``acc = sum_j exp(s_j - m) V_j``.  An empty subset gives
    ``(-inf, 0, 0)``."""
    if K.shape[0] == 0:
        return -math.inf, 0.0, np.zeros(V.shape[1], np.float64)
    s = scale * (K @ qv)
    m = float(np.max(s))
    w = np.exp(s - m)
    return m, float(np.sum(w)), w @ V


def merge_states(states) -> np.ndarray:
    """Softmax over the union of disjoint key subsets from their states:
    with ``M = max m_i``, ``out = sum_i e^(m_i - M) acc_i / sum_i e^(m_i - M) l_i``.
    This is the exact regrouping of the sums in the softmax definition
    ("Inside SGLang", Step 3: Look inside the forward pass), the same algebra
    a split-KV decode uses to join its chunks."""
    M = max(m for m, _, _ in states)
    num = sum(math.exp(m - M) * acc for m, _, acc in states if m != -math.inf)
    den = sum(math.exp(m - M) * l for m, l, _ in states if m != -math.inf)
    return num / den


def cascade_decode_attention(q, pool_k, pool_v, req_to_token, req_pool_idx, seq_lens,
                             group_start, group_len, group_depth, member_off, members,
                             num_kv_heads: int, sm_scale=None, requests=None) -> np.ndarray:
    """DECODE attention computed group by group, float64.

    A group is a run of positions ``[group_start[j], group_start[j] +
    group_len[j])`` shared by the requests ``members[member_off[j] :
    member_off[j+1]]``; its keys are read once, from the row of its first
    member, and every member's queries attend to them.  Request ``r``'s groups,
    taken by ``group_depth``, cover positions ``[0, shared_len_r)`` back to back;
    its own keys ``[shared_len_r, seq_lens[r])`` are the private tail.  The
    output merges the states of the groups and the tail (``merge_states``).
    Requests that share a prefix hold identical slot numbers there ("Inside
    SGLang", Step 3: Paged KV and the kernels that read it), so when every
    member's row agrees with its group's first member over the group's range,
    this equals ``decode_attention``.  Returns [B, Hq, D] (or the listed
    requests)."""
    return _cascade_decode(q, lambda slots: (bf16_bits_to_f64(pool_k[slots]), bf16_bits_to_f64(pool_v[slots])),
                           req_to_token, req_pool_idx, seq_lens, group_start, group_len, group_depth,
                           member_off, members, num_kv_heads, sm_scale, requests)


def _cascade_decode(q, read_kv, req_to_token, req_pool_idx, seq_lens, group_start, group_len,
                    group_depth, member_off, members, num_kv_heads, sm_scale, requests):
    """``cascade_decode_attention`` with the pool read through
    ``read_kv(slots) -> (K, V)`` (float64 rows) so that the e4m3 pool's
    variant shares the grouping."""
    q = np.asarray(q)
    B, Hq, D = q.shape
    scale = default_scale(D) if sm_scale is None else float(sm_scale)
    group_start = np.asarray(group_start, np.int64)
    group_len = np.asarray(group_len, np.int64)
    group_depth = np.asarray(group_depth, np.int64)
    member_off = np.asarray(member_off, np.int64)
    members = np.asarray(members, np.int64)
    # each request's groups, in depth order
    mine = [[] for _ in range(B)]
    for j in range(group_start.size):
        for r in members[member_off[j]: member_off[j + 1]]:
            mine[int(r)].append((int(group_depth[j]), j))
    want = np.arange(B) if requests is None else np.asarray(requests, dtype=np.int64)
    out = np.zeros((want.size, Hq, D), np.float64)
    for n, r in enumerate(want):
        r = int(r)
        qr = bf16_bits_to_f64(q[r])
        pieces = []      # (K, V) of each group, then of the tail
        shared = 0
        for _, j in sorted(mine[r]):
            first = int(members[member_off[j]])
            a, e = int(group_start[j]), int(group_start[j] + group_len[j])
            pieces.append(read_kv(np.asarray(req_to_token[int(req_pool_idx[first]), a:e], np.int64)))
            shared = e
        pieces.append(read_kv(np.asarray(req_to_token[int(req_pool_idx[r]), shared:int(seq_lens[r])], np.int64)))
        for h in range(Hq):
            kh = _kv_head_of(h, Hq, num_kv_heads)
            out[n, h] = merge_states([partial_state(qr[h], K[:, kh], V[:, kh], scale)
                                      for K, V in pieces])
    return out
