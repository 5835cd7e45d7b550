"""Algorithmic work of each step, for throughput and roofline accounting.

Only the work the method needs is counted: masked key/query pairs, padding,
re-reads and scratch traffic are never credited.

* KV bytes per token = KV heads x (key + value width) x layers x bytes per
  value ("Inside SGLang", Step 6: Decide how much memory becomes KV cache;
  114,688 B for Qwen3-0.6B: 8 heads, width 128, 28 layers, 16-bit).
* Decode reads every earlier token's K and V ("Inside SGLang", Step 3,
  Prefill and decode have different shapes: about 3.76 GB per step per
  request at 32,768 tokens for that model).
"""
from __future__ import annotations

import numpy as np


def kv_bytes_per_token(num_kv_heads: int, head_dim: int, layers: int = 1, elem_bytes: int = 2) -> int:
    return int(num_kv_heads) * 2 * int(head_dim) * int(layers) * int(elem_bytes)


def decode_bytes(seq_lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 kv_elem_bytes: int = 2) -> int:
    """K+V rows of every key (2-byte bf16 or 1-byte e4m3 values), the int32
    slot index of every key, q in, out (bf16)."""
    seq = np.asarray(seq_lens, dtype=np.int64)
    n_keys = int(seq.sum())
    B = int(seq.size)
    return (n_keys * kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes=kv_elem_bytes)
            + 4 * n_keys + 2 * 2 * B * num_q_heads * head_dim)


def decode_unique_bytes(req_to_token, req_pool_idx, seq_lens, num_q_heads, num_kv_heads, head_dim,
                        kv_elem_bytes: int = 2) -> int:
    """Like ``decode_bytes`` but counting each distinct slot once (shared
    prefixes read once)."""
    rows = [np.asarray(req_to_token[int(r), : int(s)]) for r, s in zip(req_pool_idx, seq_lens)]
    uniq = np.unique(np.concatenate(rows)).size if rows else 0
    seq = np.asarray(seq_lens, dtype=np.int64)
    return (uniq * kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes=kv_elem_bytes) + 4 * int(seq.sum())
            + 2 * 2 * int(seq.size) * num_q_heads * head_dim)


def cascade_decode_bytes(group_len, shared_lens, seq_lens, num_q_heads, num_kv_heads, head_dim,
                         kv_elem_bytes: int = 2) -> int:
    """Like ``decode_bytes`` with every shared group's keys read once: the K+V
    rows (2-byte bf16 or 1-byte e4m3 values) and slot ids of each group's keys
    and of each request's private tail ``[shared_len, seq_len)``, plus q in
    and out (bf16)."""
    seq = np.asarray(seq_lens, dtype=np.int64)
    tail = np.maximum(seq - np.asarray(shared_lens, dtype=np.int64), 0)
    n_keys = int(np.sum(np.asarray(group_len, dtype=np.int64))) + int(tail.sum())
    return (n_keys * (kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes=kv_elem_bytes) + 4)
            + 2 * 2 * int(seq.size) * num_q_heads * head_dim)


def extend_pairs(prefix_lens, extend_lens) -> int:
    """Unmasked (query, key) pairs per query head: suffix query i of a request
    with prefix p sees p + i + 1 keys, so the request adds e*p + e(e+1)/2."""
    p = np.asarray(prefix_lens, dtype=np.int64)
    e = np.asarray(extend_lens, dtype=np.int64)
    return int(np.sum(e * p + e * (e + 1) // 2))


def extend_flops(prefix_lens, extend_lens, num_q_heads: int, head_dim: int) -> int:
    """2 flops per multiply-add for q.k and for p.v over every unmasked pair."""
    return 4 * int(head_dim) * int(num_q_heads) * extend_pairs(prefix_lens, extend_lens)


def extend_bytes(prefix_lens, extend_lens, num_q_heads, num_kv_heads, head_dim) -> int:
    """Minimum HBM traffic of one extend call: prefix K/V rows and their slot
    indices, suffix q/k/v in, out."""
    p = int(np.sum(prefix_lens))
    T = int(np.sum(extend_lens))
    kv = kv_bytes_per_token(num_kv_heads, head_dim)
    return p * kv + 4 * p + T * kv + 2 * 2 * T * num_q_heads * head_dim


def store_kv_bytes(n: int, num_kv_heads: int, head_dim: int, kv_elem_bytes: int = 2) -> int:
    """Read n new bf16 K and V rows, write them to their slots (bf16, or e4m3
    codes), read n slot ids."""
    return (n * kv_bytes_per_token(num_kv_heads, head_dim)
            + n * kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes=kv_elem_bytes) + 4 * int(n))
