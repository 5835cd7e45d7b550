"""Seeded synthetic inputs for slot-indexed (page size 1) attention.

This module draws values and lays out KV-pool slots. It holds none of the
attention arithmetic: both the CUDA path (tests, bench) and the CPU oracle's
tests take their inputs from here, and neither side's computation lives here.

Slot layouts follow the pages' model of the KV cache:
  * "Inside SGLang", Step 3 (Paged KV and the kernels that read it): a pool of
    one slot per token, a table ``req_to_token`` mapping each request position
    to a slot, and prefix sharing as identical slot numbers in two rows.
  * "SGLang" notes, RadixAttention / Eviction: nodes hold runs of tokens and
    their pool slots; only unlocked nodes are evicted, leaf first, in LRU order.
  * "Origins: the paper and the first commit", Batching and Memory: EXTEND
    computes only the suffix after a cached prefix, ``seq_len = prefix + extend``,
    and the allocator hands out distinct free slots.

Values: every tensor is drawn as float32 ``N(0, std^2)`` from numpy PCG64 and
rounded to bfloat16 (round to nearest even); arrays hold the bf16 bit patterns
as ``uint16``.  Large value sets are drawn in chunks of ``CHUNK_ROWS`` rows,
each chunk from its own seed ``(seed, stream, chunk)``, so that any row range
can be regenerated on its own (the oracle checks sampled outputs of the large
workloads without holding every row in host memory).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

CHUNK_ROWS = 1024
BF16_NAN = np.uint16(0x7FC0)

# stream ids: one independent random stream per purpose
_S_LAYOUT, _S_LIVE_K, _S_LIVE_V = 1, 2, 3
_S_EXT_Q, _S_EXT_K, _S_EXT_V = 11, 12, 13
_S_DEC_Q, _S_DEC_K, _S_DEC_V = 21, 22, 23


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest even); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _normal_chunk(seed: int, stream: int, chunk: int, n: int, std: float) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, chunk])))
    x = g.standard_normal(n, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x)


class RowSource:
    """``n_rows`` rows of shape ``row_shape`` of bf16 N(0, std^2) values.

    Chunk ``c`` (rows ``[c*CHUNK_ROWS, (c+1)*CHUNK_ROWS)``) is drawn from seed
    ``(seed, stream, c)`` alone, so ``rows(a, b)`` regenerates only the chunks
    it touches and always returns the same bits.
    """

    def __init__(self, seed: int, stream: int, n_rows: int, row_shape, std: float):
        self.seed, self.stream = int(seed), int(stream)
        self.n_rows = int(n_rows)
        self.row_shape = tuple(int(s) for s in row_shape)
        self.row_elems = int(np.prod(self.row_shape))
        self.std = float(std)
        self._cache: dict[int, np.ndarray] = {}

    def _chunk(self, c: int) -> np.ndarray:
        rows = min(CHUNK_ROWS, self.n_rows - c * CHUNK_ROWS)
        full = _normal_chunk(self.seed, self.stream, c, CHUNK_ROWS * self.row_elems, self.std)
        return full[: rows * self.row_elems].reshape((rows,) + self.row_shape)

    def rows(self, start: int, stop: int) -> np.ndarray:
        start, stop = max(0, int(start)), min(self.n_rows, int(stop))
        out = np.empty((max(0, stop - start),) + self.row_shape, np.uint16)
        if stop <= start:
            return out
        c0, c1 = start // CHUNK_ROWS, (stop - 1) // CHUNK_ROWS
        chunks = list(range(c0, c1 + 1))

        def fill(c):
            blk = self._chunk(c)
            a = max(start, c * CHUNK_ROWS)
            b = min(stop, c * CHUNK_ROWS + blk.shape[0])
            out[a - start: b - start] = blk[a - c * CHUNK_ROWS: b - c * CHUNK_ROWS]

        if len(chunks) > 2:
            with ThreadPoolExecutor(_threads()) as ex:
                list(ex.map(fill, chunks))
        else:
            for c in chunks:
                fill(c)
        return out

    def take(self, idx: np.ndarray) -> np.ndarray:
        """Rows at arbitrary indices (chunks are cached across calls)."""
        idx = np.asarray(idx, dtype=np.int64).reshape(-1)
        out = np.empty((idx.size,) + self.row_shape, np.uint16)
        if idx.size == 0:
            return out
        chunk_of = idx // CHUNK_ROWS
        for c in np.unique(chunk_of):
            c = int(c)
            if c not in self._cache:
                if len(self._cache) > 64:
                    self._cache.clear()
                self._cache[c] = self._chunk(c)
            sel = np.nonzero(chunk_of == c)[0]
            out[sel] = self._cache[c][idx[sel] - c * CHUNK_ROWS]
        return out

    def all(self) -> np.ndarray:
        return self.rows(0, self.n_rows)


def normal_bf16(seed: int, stream: int, shape, std: float) -> np.ndarray:
    """A whole array of bf16 N(0, std^2) values (rows along axis 0)."""
    shape = tuple(int(s) for s in shape)
    return RowSource(seed, stream, shape[0], shape[1:], std).all()


@dataclass
class Dims:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    pool_size: int
    sm_scale: float


@dataclass
class ExtendBatch:
    """One EXTEND call: suffix tokens of ``B`` requests, back to back."""
    q: np.ndarray              # uint16 [T, Hq, D]
    k_new: np.ndarray          # uint16 [T, Hkv, D]
    v_new: np.ndarray          # uint16 [T, Hkv, D]
    slots: np.ndarray          # int32 [T]  pool slots assigned to the suffix tokens
    req_pool_idx: np.ndarray   # int32 [B]
    prefix_lens: np.ndarray    # int32 [B]
    extend_lens: np.ndarray    # int32 [B]

    @property
    def total_extend(self) -> int:
        return int(self.extend_lens.sum())


@dataclass
class DecodeBatch:
    """One DECODE call: one new token per request, written by store_kv first."""
    q: np.ndarray              # uint16 [B, Hq, D]
    k_new: np.ndarray          # uint16 [B, Hkv, D]
    v_new: np.ndarray          # uint16 [B, Hkv, D]
    slots: np.ndarray          # int32 [B]  slot of the new token (= row[seq_len-1])
    req_pool_idx: np.ndarray   # int32 [B]
    seq_lens: np.ndarray       # int32 [B]  includes the new token


@dataclass
class Workload:
    name: str
    dims: Dims
    req_to_token: np.ndarray            # int32 [R, stride]
    live_slots: np.ndarray              # int32 [n_live] slots cached before the step
    live_k: RowSource                   # rows aligned with live_slots, [Hkv, D] each
    live_v: RowSource
    extend: ExtendBatch | None = None
    decode: list = field(default_factory=list)   # list[DecodeBatch], run in order
    recipe: dict = field(default_factory=dict)

    # ----- host views of the pool (for the oracle's tests) -----
    def pool_view(self, decode_steps: int = 0, with_extend: bool = True) -> "PoolView":
        """The pool after store_kv of the extend suffix (if any) and of the first
        ``decode_steps`` decode batches; unused slots read as NaN."""
        return PoolView(self, decode_steps, with_extend)

    def dense_pools(self, decode_steps: int = 0, with_extend: bool = True):
        """Materialised [S, Hkv, D] uint16 pools (small workloads only)."""
        d = self.dims
        if d.pool_size * d.num_kv_heads * d.head_dim > (1 << 27):
            raise ValueError("pool too large to materialise on the host")
        pk = np.full((d.pool_size, d.num_kv_heads, d.head_dim), BF16_NAN, np.uint16)
        pv = pk.copy()
        pk[self.live_slots] = self.live_k.all()
        pv[self.live_slots] = self.live_v.all()
        if with_extend and self.extend is not None:
            pk[self.extend.slots] = self.extend.k_new
            pv[self.extend.slots] = self.extend.v_new
        for s in range(decode_steps):
            b = self.decode[s]
            pk[b.slots] = b.k_new
            pv[b.slots] = b.v_new
        return pk, pv


@dataclass
class CascadeGroups:
    """Runs of positions shared by several requests of one decode batch.

    Group ``j`` covers positions ``[group_start[j], group_start[j] +
    group_len[j])`` of every member's row; its members are
    ``members[member_off[j]:member_off[j+1]]`` (indices into the decode batch)
    and ``group_depth[j]`` is its rank among each member's groups, which cover
    ``[0, shared_len)`` back to back.  In a radix tree these are the nodes with
    two or more running requests below them.
    """
    group_start: np.ndarray    # int32 [G]
    group_len: np.ndarray      # int32 [G]
    group_depth: np.ndarray    # int32 [G]
    member_off: np.ndarray     # int32 [G+1]
    members: np.ndarray        # int32 [nnz]

    @property
    def n_groups(self) -> int:
        return int(self.group_start.size)

    @property
    def max_members(self) -> int:
        return int(np.diff(self.member_off).max()) if self.n_groups else 0

    @property
    def max_depth(self) -> int:
        """Number of depth levels (largest depth + 1; 0 without groups)."""
        return int(self.group_depth.max()) + 1 if self.n_groups else 0

    def shared_lens(self, batch: int) -> np.ndarray:
        """Per request: the end of its deepest group (0 if it is in none)."""
        out = np.zeros(batch, np.int64)
        for j in range(self.n_groups):
            m = self.members[self.member_off[j]: self.member_off[j + 1]]
            out[m] = np.maximum(out[m], int(self.group_start[j]) + int(self.group_len[j]))
        return out


def shared_prefix_groups(req_to_token: np.ndarray, req_pool_idx, seq_lens,
                         min_members: int = 2) -> CascadeGroups:
    """The shared-prefix groups of a decode batch, read off its rows.

    Requests whose rows hold the same slot at a position share that token
    ("Inside SGLang", Step 3: Paged KV and the kernels that read it -- shared
    prefixes are identical leading slot numbers).  Starting at position 0, the
    requests are split by their slot; a set of at least ``min_members``
    requests forms a group that runs while all of them agree (and none has
    ended), then the set splits again at the first disagreement: a compressed
    trie over the slot sequences, i.e. the radix tree's nodes restricted to the
    running requests.  Groups are listed by (depth, start, first member).
    """
    rtt = np.asarray(req_to_token)
    rows = np.asarray(req_pool_idx, np.int64)
    lens = np.asarray(seq_lens, np.int64)
    found = []
    work = [(np.nonzero(lens > 0)[0], 0, 0)]
    while work:
        mem, pos, depth = work.pop()
        if mem.size < min_members:
            continue
        at = rtt[rows[mem], pos]
        for v in np.unique(at):
            sub = mem[at == v]
            if sub.size < min_members:
                continue
            lim = int(lens[sub].min())
            block = rtt[rows[sub], pos:lim]
            agree = np.all(block == block[0], axis=0)
            stop = np.nonzero(~agree)[0]
            end = pos + (int(stop[0]) if stop.size else lim - pos)
            found.append((depth, pos, end - pos, np.sort(sub)))
            rest = sub[lens[sub] > end]
            work.append((rest, end, depth + 1))
    found.sort(key=lambda f: (f[0], f[1], int(f[3][0])))
    off = np.zeros(len(found) + 1, np.int32)
    off[1:] = np.cumsum([f[3].size for f in found])
    cat = np.concatenate([f[3] for f in found]) if found else np.zeros(0)
    return CascadeGroups(group_start=np.asarray([f[1] for f in found], np.int32),
                         group_len=np.asarray([f[2] for f in found], np.int32),
                         group_depth=np.asarray([f[0] for f in found], np.int32),
                         member_off=off, members=cat.astype(np.int32))


class PoolView:
    """Read-only ``pool[slots]`` access that regenerates rows on demand."""

    def __init__(self, w: Workload, decode_steps: int, with_extend: bool):
        self.w = w
        d = w.dims
        self.shape = (d.pool_size, d.num_kv_heads, d.head_dim)
        self._live = np.full(d.pool_size, -1, np.int64)
        self._live[w.live_slots] = np.arange(w.live_slots.size)
        # new-token map: slot -> (source id, row)
        self._src = np.full(d.pool_size, -1, np.int32)
        self._row = np.full(d.pool_size, -1, np.int64)
        self._new = []
        if with_extend and w.extend is not None:
            self._add(w.extend.slots, w.extend.k_new, w.extend.v_new)
        for s in range(decode_steps):
            b = w.decode[s]
            self._add(b.slots, b.k_new, b.v_new)

    def _add(self, slots, k, v):
        sid = len(self._new)
        self._new.append((k, v))
        self._src[slots] = sid
        self._row[slots] = np.arange(slots.size)

    def rows(self, slots, which: str) -> np.ndarray:
        slots = np.asarray(slots, dtype=np.int64).reshape(-1)
        out = np.full((slots.size,) + self.shape[1:], BF16_NAN, np.uint16)
        src = self._src[slots]
        live = self._live[slots]
        m_live = (src < 0) & (live >= 0)
        if m_live.any():
            rs = self.w.live_k if which == "k" else self.w.live_v
            out[m_live] = rs.take(live[m_live])
        for sid, (k, v) in enumerate(self._new):
            m = src == sid
            if m.any():
                out[m] = (k if which == "k" else v)[self._row[slots[m]]]
        return out

    @property
    def k(self):
        return _PoolSide(self, "k")

    @property
    def v(self):
        return _PoolSide(self, "v")


class _PoolSide:
    def __init__(self, view: PoolView, which: str):
        self.view, self.which = view, which
        self.shape = view.shape

    def __getitem__(self, slots):
        slots = np.asarray(slots)
        return self.view.rows(slots, self.which).reshape(slots.shape + self.shape[1:])


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def _fill_rtt_tails(rtt: np.ndarray, lens: np.ndarray, rows: np.ndarray,
                    unused: np.ndarray, g: np.random.Generator) -> None:
    """Entries past each row's length point at unused (NaN-poisoned) slots,
    always inside the pool, so a kernel that reads past a length returns NaN
    instead of touching memory outside the pool."""
    if unused.size == 0:
        raise ValueError("no unused slot left to poison req_to_token tails")
    fill = unused[g.integers(0, unused.size, size=rtt.size)].astype(np.int32).reshape(rtt.shape)
    used = np.zeros(rtt.shape, bool)
    for r, n in zip(rows, lens):
        used[r, :n] = True
    rtt[~used] = fill[~used]


def _unused_slots(pool_size: int, *used) -> np.ndarray:
    mask = np.ones(pool_size, bool)
    for u in used:
        mask[np.asarray(u, dtype=np.int64)] = False
    return np.nonzero(mask)[0].astype(np.int32)


def _decode_batch(seed, stream_base, B, dims, slots, rpi, seq_lens, std) -> DecodeBatch:
    H, Hk, D = dims.num_q_heads, dims.num_kv_heads, dims.head_dim
    return DecodeBatch(
        q=normal_bf16(seed, _S_DEC_Q + stream_base, (B, H, D), std),
        k_new=normal_bf16(seed, _S_DEC_K + stream_base, (B, Hk, D), std),
        v_new=normal_bf16(seed, _S_DEC_V + stream_base, (B, Hk, D), std),
        slots=np.asarray(slots, np.int32), req_pool_idx=np.asarray(rpi, np.int32),
        seq_lens=np.asarray(seq_lens, np.int32))


def _extend_batch(seed, dims, slots, rpi, prefix_lens, extend_lens, std) -> ExtendBatch:
    H, Hk, D = dims.num_q_heads, dims.num_kv_heads, dims.head_dim
    T = int(np.sum(extend_lens))
    return ExtendBatch(
        q=normal_bf16(seed, _S_EXT_Q, (T, H, D), std),
        k_new=normal_bf16(seed, _S_EXT_K, (T, Hk, D), std),
        v_new=normal_bf16(seed, _S_EXT_V, (T, Hk, D), std),
        slots=np.asarray(slots, np.int32), req_pool_idx=np.asarray(rpi, np.int32),
        prefix_lens=np.asarray(prefix_lens, np.int32),
        extend_lens=np.asarray(extend_lens, np.int32))


# --------------------------------------------------------------------------
# generic builder: explicit per-request contexts
# --------------------------------------------------------------------------

def build_workload(name: str, dims: Dims, seed: int, *,
                   extend_prefix: list | None = None, extend_lens=None,
                   decode_ctx: list | None = None, std: float = 1.0,
                   rtt_rows: int | None = None, rtt_stride: int | None = None,
                   live_slots=None, slot_source: np.ndarray | None = None,
                   reserve=None, recipe: dict | None = None) -> Workload:
    """Lay out one extend batch and/or one decode batch from explicit contexts.

    ``extend_prefix[i]`` is the array of cached slots of extend request i;
    ``decode_ctx[j]`` is the array of cached slots before decode request j's
    new token.  New-token slots come, in order, from ``slot_source`` (default:
    a seeded permutation of the unused slots).  ``live_slots`` (default: the
    union of all cached slots, in first-use order) get values.  Slots in
    ``reserve`` (new tokens of later steps) are never used as poison targets.
    """
    g = _rng(seed, _S_LAYOUT)
    S = dims.pool_size
    extend_prefix = [np.asarray(p, np.int32) for p in (extend_prefix or [])]
    decode_ctx = [np.asarray(c, np.int32) for c in (decode_ctx or [])]
    if live_slots is None:
        cat = np.concatenate(extend_prefix + decode_ctx + [np.zeros(0, np.int32)])
        _, first = np.unique(cat, return_index=True)
        live_slots = cat[np.sort(first)]
    live_slots = np.asarray(live_slots, np.int32)
    Be, Bd = len(extend_prefix), len(decode_ctx)
    ext_lens = np.asarray(extend_lens if extend_lens is not None else [], np.int32)
    assert ext_lens.size == Be
    n_new = int(ext_lens.sum()) + Bd
    if slot_source is None:
        free = _unused_slots(S, live_slots)
        slot_source = free[g.permutation(free.size)]
    new_slots = np.asarray(slot_source[:n_new], np.int32)
    assert new_slots.size == n_new, "pool too small for the new tokens"
    R = rtt_rows if rtt_rows is not None else Be + Bd
    lens = [p.size + int(e) for p, e in zip(extend_prefix, ext_lens)] + [c.size + 1 for c in decode_ctx]
    stride = rtt_stride if rtt_stride is not None else max(lens + [1])
    assert R >= Be + Bd and stride >= max(lens + [1])
    rows = g.permutation(R)[: Be + Bd].astype(np.int32)
    rtt = np.zeros((R, stride), np.int32)
    pos = 0
    ext_slots = []
    for i, (p, e) in enumerate(zip(extend_prefix, ext_lens)):
        s = new_slots[pos: pos + int(e)]
        pos += int(e)
        ext_slots.append(s)
        rtt[rows[i], : p.size] = p
        rtt[rows[i], p.size: p.size + int(e)] = s
    dec_slots = new_slots[pos: pos + Bd]
    for j, c in enumerate(decode_ctx):
        rtt[rows[Be + j], : c.size] = c
        rtt[rows[Be + j], c.size] = dec_slots[j]
    unused = _unused_slots(S, live_slots, new_slots,
                           np.zeros(0, np.int32) if reserve is None else reserve)
    _fill_rtt_tails(rtt, lens, rows, unused, g)
    H, Hk, D = dims.num_q_heads, dims.num_kv_heads, dims.head_dim
    w = Workload(name=name, dims=dims, req_to_token=rtt, live_slots=live_slots,
                 live_k=RowSource(seed, _S_LIVE_K, live_slots.size, (Hk, D), std),
                 live_v=RowSource(seed, _S_LIVE_V, live_slots.size, (Hk, D), std),
                 recipe=dict(recipe or {}))
    if Be:
        w.extend = _extend_batch(seed, dims, np.concatenate(ext_slots) if ext_slots else np.zeros(0, np.int32),
                                 rows[:Be], [p.size for p in extend_prefix], ext_lens, std)
    if Bd:
        w.decode = [_decode_batch(seed, 0, Bd, dims, dec_slots, rows[Be:],
                                  [c.size + 1 for c in decode_ctx], std)]
    return w


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

def tiny(seed: int = 1001) -> Workload:
    """Tiny extend+decode correctness case.

    2 query heads / 2 KV heads, head_dim 64, a 512-slot pool; four requests with
    prefix lengths {0,16,33,64} and extend lengths {8,1,31,17}, then one decode
    step each.  Requests 1 and 2 share the slots of their first 16 prefix
    tokens.  Every token takes the next slot of one seeded permutation of the
    pool.  q/k/v ~ N(0,1)/8, softmax scale 1/8.
    """
    dims = Dims(2, 2, 64, 512, 1.0 / 8.0)
    g = _rng(seed, _S_LAYOUT + 100)
    perm = g.permutation(dims.pool_size).astype(np.int32)
    P, E = [0, 16, 33, 64], [8, 1, 31, 17]
    pos = 0
    prefix = []
    for i, p in enumerate(P):
        if i == 2:
            own = perm[pos: pos + p - 16]
            pos += p - 16
            prefix.append(np.concatenate([prefix[1][:16], own]))
        else:
            prefix.append(perm[pos: pos + p])
            pos += p
    # suffix slots, then the decode slots, continue along the same permutation
    n_ext = sum(E)
    ext_slots = perm[pos: pos + n_ext]
    dec_slots = perm[pos + n_ext: pos + n_ext + len(P)]
    live = np.concatenate(prefix)
    _, first = np.unique(live, return_index=True)
    live = live[np.sort(first)]
    w = build_workload("tiny", dims, seed, extend_prefix=prefix, extend_lens=E,
                       std=1.0 / 8.0, rtt_rows=8, rtt_stride=128, live_slots=live,
                       slot_source=ext_slots, reserve=dec_slots,
                       recipe=dict(prefix_lens=P, extend_lens=E, shared="requests 1,2 share 16 prefix slots"))
    # the decode step continues each extend request by one token
    ext = w.extend
    rows = ext.req_pool_idx
    seq = np.asarray(P) + np.asarray(E) + 1
    for i in range(len(P)):
        w.req_to_token[rows[i], seq[i] - 1] = dec_slots[i]
    w.decode = [_decode_batch(seed, 0, len(P), dims, dec_slots, rows, seq, 1.0 / 8.0)]
    return w


def _page_runs(g: np.random.Generator, pool_size: int, page_size: int, lens) -> list:
    """Slots of requests that own whole pages: pages of ``page_size``
    consecutive slots are taken from one seeded permutation of the pool's
    pages, ceil(n / page_size) per request, and request j's positions fill its
    pages in order (the tail of its last page stays free)."""
    pages = g.permutation(pool_size // page_size).astype(np.int64)
    out, pos = [], 0
    for n in lens:
        k = -(-int(n) // page_size)
        mine = pages[pos: pos + k]
        pos += k
        assert mine.size == k, "pool too small"
        out.append((mine[:, None] * page_size + np.arange(page_size)).reshape(-1)[: int(n)].astype(np.int32))
    return out


def decode_llama7b(seed: int = 1002, batch: int = 64, pool_size: int = 1 << 20,
                   seq_range=(512, 4096), page_size: int = 1) -> Workload:
    """Plain paged decode, Llama-7B-like heads (32 q / 32 kv, head_dim 128).

    seq_lens ~ U[512, 4096] (integers, inclusive) including the new token; every
    token's slot is drawn without replacement from one seeded permutation of
    the pool (fully fragmented); the new token's slot is the last of its row.
    With ``page_size`` > 1 every request owns whole pages of that many
    consecutive slots instead (``_page_runs``), its new token in them.
    """
    dims = Dims(32, 32, 128, pool_size, 1.0 / math.sqrt(128))
    g = _rng(seed, _S_LAYOUT + 100)
    seq = g.integers(seq_range[0], seq_range[1] + 1, size=batch).astype(np.int32)
    recipe = dict(batch=batch, seq_range=list(seq_range), pool=pool_size, page_size=page_size)
    if page_size > 1:
        rows = _page_runs(g, pool_size, page_size, seq)
        return build_workload("decode_llama7b", dims, seed, decode_ctx=[r[:-1] for r in rows], std=1.0,
                              rtt_stride=int(seq_range[1]),
                              slot_source=np.array([r[-1] for r in rows], np.int32), recipe=recipe)
    perm = g.permutation(pool_size).astype(np.int32)
    ctx, pos = [], 0
    for s in seq:
        ctx.append(perm[pos: pos + s - 1])
        pos += s - 1
    return build_workload("decode_llama7b", dims, seed, decode_ctx=ctx, std=1.0,
                          rtt_stride=int(seq_range[1]), slot_source=perm[pos:], recipe=recipe)


def shared_prompt_extend(seed: int = 1003, batch: int = 64, prefix: int = 4096,
                         extend: int = 256, pool_size: int = 1 << 21,
                         heads=(32, 8), page_size: int = 1) -> Workload:
    """Shared system prompt: every request's row starts with the same prefix
    slots, then extends by ``extend`` private causal tokens (GQA 32/8, d 128).
    With ``page_size`` > 1 (dividing ``prefix``) the prefix and each request's
    suffix own whole pages of that many consecutive slots (``_page_runs``)."""
    dims = Dims(heads[0], heads[1], 128, pool_size, 1.0 / math.sqrt(128))
    g = _rng(seed, _S_LAYOUT + 100)
    recipe = dict(batch=batch, prefix=prefix, extend=extend, pool=pool_size, page_size=page_size)
    if page_size > 1:
        assert prefix % page_size == 0, "the shared prefix must fill whole pages"
        runs = _page_runs(g, pool_size, page_size, [prefix] + [extend] * batch)
        shared = runs[0]
        return build_workload("shared_prompt_extend", dims, seed,
                              extend_prefix=[shared] * batch, extend_lens=[extend] * batch,
                              std=1.0, slot_source=np.concatenate(runs[1:]), live_slots=shared,
                              recipe=recipe)
    perm = g.permutation(pool_size).astype(np.int32)
    shared = perm[:prefix]
    return build_workload("shared_prompt_extend", dims, seed,
                          extend_prefix=[shared] * batch, extend_lens=[extend] * batch,
                          std=1.0, slot_source=perm[prefix:], live_slots=shared, recipe=recipe)


def tree_of_thought_decode(seed: int = 1004, depth: int = 4, fanout: int = 4,
                           segment: int = 512, steps: int = 17,
                           pool_size: int = 1 << 20) -> Workload:
    """Tree-of-thought branching decode (GQA 32/8, head_dim 128).

    A tree of ``depth`` levels below an implicit empty root, ``fanout``
    children per node and ``segment`` tokens per node; every leaf is one decode
    request whose row is its ancestors' segment slots (shared by all
    descendants) followed by its own.  ``steps`` decode batches run back to
    back (one step, then a 16-step loop), each appending one token per leaf.
    Segment and new-token slots come from one seeded permutation of the pool.
    """
    dims = Dims(32, 8, 128, pool_size, 1.0 / math.sqrt(128))
    g = _rng(seed, _S_LAYOUT + 100)
    perm = g.permutation(pool_size).astype(np.int32)
    level_sizes = [fanout ** (l + 1) for l in range(depth)]
    n_seg = sum(level_sizes)
    leaves = level_sizes[-1]
    seg_base = np.cumsum([0] + level_sizes)[:-1]
    seg_slots = perm[: n_seg * segment].reshape(n_seg, segment)
    ctx_len = depth * segment
    ctx = []
    for leaf in range(leaves):
        segs = [int(seg_base[l] + leaf // (fanout ** (depth - 1 - l))) for l in range(depth)]
        ctx.append(np.concatenate([seg_slots[s] for s in segs]))
    new = perm[n_seg * segment: n_seg * segment + steps * leaves].reshape(steps, leaves)
    stride = ctx_len + steps
    w = build_workload("tree_of_thought_decode", dims, seed, decode_ctx=ctx, std=1.0,
                       rtt_stride=stride, live_slots=seg_slots.reshape(-1),
                       slot_source=new[0], reserve=new.reshape(-1),
                       recipe=dict(depth=depth, fanout=fanout, segment=segment, steps=steps,
                                   leaves=leaves, segments=n_seg, pool=pool_size))
    rows = w.decode[0].req_pool_idx
    batches = [w.decode[0]]
    for s in range(1, steps):
        seq = np.full(leaves, ctx_len + s + 1, np.int32)
        w.req_to_token[rows, ctx_len + s] = new[s]
        batches.append(_decode_batch(seed, 100 * s, leaves, dims, new[s], rows, seq, 1.0))
    w.decode = batches
    # tails past the last step still point at poisoned slots (filled above for
    # the step-0 lengths; positions ctx_len+1.. were overwritten step by step)
    return w


def random_tree_decode(seed: int = 1006, dims: Dims | None = None, fanouts=(3, 3, 2),
                       seg_len=(1, 300), own_len=(0, 40), n_solo: int = 2,
                       pool_size: int = 1 << 16, std: float = 1.0) -> Workload:
    """Decode over a random prefix tree with ragged node lengths.

    Below an implicit root, level ``l`` nodes have ``fanouts[l]`` children;
    every node holds U[seg_len] tokens, each leaf is one decode request whose
    row is its ancestors' tokens, then its own U[own_len] private tokens, then
    the new one.  ``n_solo`` more requests share nothing.  The batch order is
    shuffled, so no group's members are contiguous.  Slots come from one
    seeded permutation of the pool.
    """
    dims = dims or Dims(16, 4, 128, pool_size, 1.0 / math.sqrt(128))
    assert dims.pool_size == pool_size
    g = _rng(seed, _S_LAYOUT + 100)
    perm = g.permutation(pool_size).astype(np.int32)
    pos = 0

    def take(n):
        nonlocal pos
        out = perm[pos: pos + n]
        pos += n
        assert out.size == n, "pool too small"
        return out

    level = [np.zeros(0, np.int32)]
    for f in fanouts:
        level = [np.concatenate([ctx, take(int(g.integers(seg_len[0], seg_len[1] + 1)))])
                 for ctx in level for _ in range(f)]
    ctx = [np.concatenate([c, take(int(g.integers(own_len[0], own_len[1] + 1)))]) for c in level]
    ctx += [take(int(g.integers(seg_len[0], 2 * seg_len[1] + 1))) for _ in range(n_solo)]
    ctx = [ctx[i] for i in g.permutation(len(ctx))]
    live = np.concatenate(ctx)
    _, first = np.unique(live, return_index=True)
    live = live[np.sort(first)]
    return build_workload("random_tree_decode", dims, seed, decode_ctx=ctx, std=std,
                          live_slots=live, slot_source=perm[pos:],
                          recipe=dict(fanouts=list(fanouts), seg_len=list(seg_len),
                                      own_len=list(own_len), n_solo=n_solo, pool=pool_size))


def tree_groups(w: Workload, step: int = 0) -> CascadeGroups:
    """Shared-prefix groups of decode step ``step`` of a tree workload."""
    b = w.decode[step]
    return shared_prefix_groups(w.req_to_token, b.req_pool_idx, b.seq_lens)


def _eviction_layout(g: np.random.Generator, pool_size: int, live_lens: np.ndarray,
                     evict_frac: float, chunk: int = 2048, concurrency: int = 16):
    """Place live and filler sequences in a pool, then evict unlocked leaves.

    Sequences (live ones locked, fillers not) are allocated from a sequential
    free list in arrival order: each starts at a random time, prefills its
    prompt in ``chunk``-token steps and then decodes one token per step, so the
    slots of concurrent sequences interleave.  Fillers are added until the pool
    is full; arrival times are uniform over a window in which ``concurrency``
    sequences are in flight on average.  Eviction then frees unlocked nodes leaf first in LRU order: a
    filler's tail is its leaf, its last access is its finishing time, and
    removing a tail leaves the parent as the next leaf with the same access
    time, so fillers are freed whole, oldest first, until ``evict_frac`` of the
    pool is free (the last one partly, from its tail).  The freed slots are
    shuffled into the free list.  Returns (slots of each live sequence,
    shuffled free list).
    """
    n_live = int(live_lens.sum())
    assert n_live <= pool_size
    fill_lens = []
    room = pool_size - n_live
    while room > 0:
        L = int(round(math.exp(g.uniform(math.log(1024), math.log(32768)))))
        L = min(L, room)
        fill_lens.append(L)
        room -= L
    lens = np.concatenate([live_lens, np.asarray(fill_lens, np.int64)]).astype(np.int64)
    nseq = lens.size
    prompt = np.maximum(1, np.round(lens * g.uniform(0.5, 1.0, size=nseq))).astype(np.int64)
    prompt = np.minimum(prompt, lens)
    n_chunks = (prompt + chunk - 1) // chunk
    # arrivals are uniform over a window sized so that on average
    # ``concurrency`` sequences are being allocated at once
    duration = n_chunks + (lens - prompt)
    horizon = max(1, int(duration.sum() // concurrency))
    start = g.integers(0, horizon, size=nseq)
    # per-token (time, seq, position) keys
    seq_id = np.repeat(np.arange(nseq), lens)
    first = np.cumsum(lens) - lens
    pos = np.arange(lens.sum()) - np.repeat(first, lens)
    in_prompt = pos < prompt[seq_id]
    t = np.where(in_prompt, start[seq_id] + pos // chunk,
                 start[seq_id] + n_chunks[seq_id] + (pos - prompt[seq_id]))
    order = np.lexsort((pos, seq_id, t))
    slot_of_token = np.empty(lens.sum(), np.int64)
    slot_of_token[order] = np.arange(lens.sum())
    finish = start + n_chunks + (lens - prompt)
    # evict fillers oldest-finish first, each from its tail
    n_live_seq = live_lens.size
    target = int(round(evict_frac * pool_size))
    fill_ids = np.arange(n_live_seq, nseq)
    fill_ids = fill_ids[np.argsort(finish[fill_ids], kind="stable")]
    freed = []
    got = 0
    for s in fill_ids:
        if got >= target:
            break
        take = min(int(lens[s]), target - got)
        a = first[s] + lens[s] - take
        freed.append(slot_of_token[a: first[s] + lens[s]])
        got += take
    assert got == target, "not enough unlocked filler to evict"
    freed = np.concatenate(freed)
    free_list = freed[g.permutation(freed.size)].astype(np.int32)
    live_slots = [slot_of_token[first[i]: first[i] + lens[i]].astype(np.int32) for i in range(n_live_seq)]
    return live_slots, free_list, dict(fillers=len(fill_lens), evicted=target)


def chunked_prefill_mix(seed: int = 1005, n_chunks: int = 8, chunk: int = 2048,
                        prefix_max: int = 16384, n_decode: int = 248,
                        decode_range=(1024, 32768), pool_size: int = 1 << 22,
                        evict_frac: float = 0.3, heads=(16, 8)) -> Workload:
    """Chunked-prefill mixed batch, Qwen3-0.6B-like GQA (16 q / 8 kv, d 128).

    ``n_chunks`` extend requests of ``chunk`` new tokens with cached prefixes
    ~ U[0, prefix_max]; ``n_decode`` decode requests with seq_lens
    log-uniform in ``decode_range`` (round(exp(U(ln a, ln b))), including the
    new token).  Slots come from ``_eviction_layout`` (30% of the pool evicted
    leaf first, LRU); new tokens take slots from the shuffled free list.
    """
    dims = Dims(heads[0], heads[1], 128, pool_size, 1.0 / math.sqrt(128))
    g = _rng(seed, _S_LAYOUT + 100)
    prefix = g.integers(0, prefix_max + 1, size=n_chunks).astype(np.int64)
    lo, hi = math.log(decode_range[0]), math.log(decode_range[1])
    seq = np.round(np.exp(g.uniform(lo, hi, size=n_decode))).astype(np.int64)
    seq = np.clip(seq, decode_range[0], decode_range[1])
    live_lens = np.concatenate([prefix, seq - 1])
    live, free_list, stats = _eviction_layout(g, pool_size, live_lens, evict_frac)
    stride = int(max(prefix_max + chunk, decode_range[1]))
    return build_workload("chunked_prefill_mix", dims, seed,
                          extend_prefix=live[:n_chunks], extend_lens=[chunk] * n_chunks,
                          decode_ctx=live[n_chunks:], std=1.0, rtt_stride=stride,
                          slot_source=free_list,
                          recipe=dict(n_chunks=n_chunks, chunk=chunk, prefix_max=prefix_max,
                                      n_decode=n_decode, decode_range=list(decode_range),
                                      pool=pool_size, evict_frac=evict_frac, **stats))


CONFIGS = {
    1: tiny,
    2: decode_llama7b,
    3: shared_prompt_extend,
    4: tree_of_thought_decode,
    5: chunked_prefill_mix,
}


def make(config: int, **kw) -> Workload:
    return CONFIGS[config](**kw)


# --------------------------------------------------------------------------
# device upload (setup only; uses torch for memory, not for the path)
# --------------------------------------------------------------------------

def to_device(w: Workload, device="cuda", poison: bool = True, rows_per_copy: int = 1 << 16):
    """Allocate the pools on ``device`` (NaN everywhere when ``poison``), write
    the cached tokens' rows, and upload every index/value array.  Returns a
    dict of torch tensors; bf16 arrays become torch.bfloat16."""
    import torch

    d = w.dims
    shape = (d.pool_size, d.num_kv_heads, d.head_dim)
    fill = torch.tensor([int(BF16_NAN) if poison else 0], dtype=torch.int16).view(torch.bfloat16)
    pk = torch.empty(shape, dtype=torch.bfloat16, device=device)
    pv = torch.empty(shape, dtype=torch.bfloat16, device=device)
    pk.fill_(fill.item())
    pv.fill_(fill.item())
    slots_all = torch.from_numpy(w.live_slots.astype(np.int64))
    for a in range(0, w.live_slots.size, rows_per_copy):
        b = min(a + rows_per_copy, w.live_slots.size)
        idx = slots_all[a:b].to(device)
        pk.index_copy_(0, idx, bf16_tensor(w.live_k.rows(a, b), device))
        pv.index_copy_(0, idx, bf16_tensor(w.live_v.rows(a, b), device))
    out = dict(pool_k=pk, pool_v=pv, req_to_token=int_tensor(w.req_to_token, device))
    if w.extend is not None:
        e = w.extend
        out["extend"] = dict(q=bf16_tensor(e.q, device), k_new=bf16_tensor(e.k_new, device),
                             v_new=bf16_tensor(e.v_new, device), slots=int_tensor(e.slots, device),
                             req_pool_idx=int_tensor(e.req_pool_idx, device),
                             prefix_lens=int_tensor(e.prefix_lens, device),
                             extend_lens=int_tensor(e.extend_lens, device))
    out["decode"] = [dict(q=bf16_tensor(b.q, device), k_new=bf16_tensor(b.k_new, device),
                          v_new=bf16_tensor(b.v_new, device), slots=int_tensor(b.slots, device),
                          req_pool_idx=int_tensor(b.req_pool_idx, device),
                          seq_lens=int_tensor(b.seq_lens, device)) for b in w.decode]
    return out


def bf16_tensor(bits: np.ndarray, device="cpu"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if str(device) != "cpu" else t


def int_tensor(a: np.ndarray, device="cpu"):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))
    return t.to(device) if str(device) != "cpu" else t


def bf16_bits(t) -> np.ndarray:
    """torch bf16 tensor -> numpy uint16 bits (copied to host)."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
