"""Small seeded layouts for tests (inputs only; built with the workload module)."""
from __future__ import annotations

import math

import numpy as np

from radixattention_prefix_shared_gb300 import workloads as W


def extend_case(seed, *, Hq, Hkv, D, prefix_lens, extend_lens, shares=(), std=1.0,
                pool_size=None, scale=None, decode_after=False):
    """An extend batch over a seeded permutation of a small pool.

    ``shares`` holds (a, b, n): request b's first n prefix slots are request
    a's first n.  With ``decode_after`` one decode step follows (seq_len =
    prefix + extend + 1 per request)."""
    g = np.random.default_rng(seed)
    total = sum(prefix_lens) + sum(extend_lens) + len(extend_lens)
    S = pool_size or max(64, 2 * total + 32)
    perm = g.permutation(S).astype(np.int32)
    pos = 0
    prefix = []
    for p in prefix_lens:
        prefix.append(perm[pos: pos + p].copy())
        pos += p
    for a, b, n in shares:
        prefix[b][:n] = prefix[a][:n]
    live = np.concatenate(prefix + [np.zeros(0, np.int32)])
    _, first = np.unique(live, return_index=True)
    live = live[np.sort(first)]
    n_ext = sum(extend_lens)
    ext_slots = perm[pos: pos + n_ext]
    dec_slots = perm[pos + n_ext: pos + n_ext + len(extend_lens)]
    sc = scale if scale is not None else 1.0 / math.sqrt(D)
    dims = W.Dims(Hq, Hkv, D, S, sc)
    stride = max([p + e + 1 for p, e in zip(prefix_lens, extend_lens)] + [1])
    w = W.build_workload("case", dims, seed, extend_prefix=prefix, extend_lens=list(extend_lens),
                         std=std, live_slots=live, slot_source=ext_slots, reserve=dec_slots,
                         rtt_rows=len(extend_lens) + 3, rtt_stride=stride)
    if decode_after:
        rows = w.extend.req_pool_idx
        seq = np.asarray(prefix_lens) + np.asarray(extend_lens) + 1
        for i in range(len(prefix_lens)):
            w.req_to_token[rows[i], seq[i] - 1] = dec_slots[i]
        w.decode = [W._decode_batch(seed, 0, len(prefix_lens), dims, dec_slots, rows, seq, std)]
    return w


def decode_case(seed, *, Hq, Hkv, D, seq_lens, std=1.0, pool_size=None, shares=(), scale=None):
    """A decode batch; request j's row holds seq_lens[j]-1 cached slots and the
    new token's slot last.  ``shares`` as in ``extend_case``."""
    g = np.random.default_rng(seed)
    S = pool_size or max(64, 2 * sum(seq_lens) + 32)
    perm = g.permutation(S).astype(np.int32)
    pos = 0
    ctx = []
    for s in seq_lens:
        ctx.append(perm[pos: pos + s - 1].copy())
        pos += s - 1
    for a, b, n in shares:
        ctx[b][:n] = ctx[a][:n]
    sc = scale if scale is not None else 1.0 / math.sqrt(D)
    dims = W.Dims(Hq, Hkv, D, S, sc)
    live = np.concatenate(ctx + [np.zeros(0, np.int32)])
    _, first = np.unique(live, return_index=True)
    live = live[np.sort(first)]
    return W.build_workload("case", dims, seed, decode_ctx=ctx, std=std, live_slots=live,
                            slot_source=perm[pos:], rtt_rows=len(seq_lens) + 2,
                            rtt_stride=max(seq_lens) + 3)
