"""The C++ radix tree (C ABI, host only) against the radix-tree oracle.

Random operation sequences -- inserts of sequences that often share a prefix,
lookups, locks of a lookup's last node, unlocks, evictions -- run on both; every
result must match exactly (matched lengths, slot lists, what insert reports as
cached, the order of evicted slots, evictable / locked token counts, the
shared-prefix groups of a batch).
"""
import numpy as np
import pytest

import oracle
from oracle.radix import RadixTree as Oracle
from radixattention_prefix_shared_gb300 import binding as B
from radixattention_prefix_shared_gb300 import workloads as W


def _seq(rng, stems, vocab):
    if stems and rng.random() < 0.75:
        base = stems[int(rng.integers(len(stems)))]
        cut = int(rng.integers(0, len(base) + 1))
        return base[:cut] + [int(x) for x in rng.integers(0, vocab, size=int(rng.integers(0, 10)))]
    return [int(x) for x in rng.integers(0, vocab, size=int(rng.integers(1, 16)))]


@pytest.mark.parametrize("seed,vocab", [(0, 3), (1, 5), (2, 8), (3, 4), (4, 2)])
def test_random_operations_match_the_oracle(seed, vocab):
    rng = np.random.default_rng(seed)
    c, o = B.RadixTree(), Oracle()
    stems, nxt, locks = [], 0, []          # locks: (c handle, oracle node)
    for step in range(600):
        op = rng.random()
        s = _seq(rng, stems, vocab)
        if op < 0.35:
            slots = list(range(nxt, nxt + len(s)))
            nxt += len(s)
            assert c.insert(s, slots) == o.insert(s, slots), step
            stems.append(s)
        elif op < 0.6:
            mc, sc, hc = c.match_prefix(s)
            mo, so, no = o.match_prefix(s)
            assert (mc, sc) == (mo, so), step
            if mc and rng.random() < 0.5:
                c.inc_lock_ref(hc)
                o.inc_lock_ref(no)
                locks.append((hc, no))
        elif op < 0.72 and locks:
            hc, no = locks.pop(int(rng.integers(len(locks))))
            c.dec_lock_ref(hc)
            o.dec_lock_ref(no)
        else:
            k = int(rng.integers(1, 25))
            assert c.evict(k) == o.evict(k), step
        assert (c.evictable_tokens, c.protected_tokens) == (o.evictable, o.protected), step
        if step % 50 == 49 and stems:
            # groups of a batch of lookups
            batch = [stems[int(i)] for i in rng.integers(0, len(stems), size=12)]
            hs = [c.match_prefix(x)[2] for x in batch]
            ns = [o.match_prefix(x)[2] for x in batch]
            start, length, depth, off, mem = c.groups(hs)
            want = o.groups(ns)
            got = [(int(depth[j]), int(start[j]), int(length[j]), mem[off[j]:off[j + 1]].tolist())
                   for j in range(start.size)]
            assert got == want, step


def test_stale_handles_and_unbalanced_unlocks_are_refused():
    c = B.RadixTree()
    c.insert([1, 2, 3], [10, 11, 12])
    _, _, h = c.match_prefix([1, 2, 3])
    with pytest.raises(B.SglError):
        c.dec_lock_ref(h)                               # never locked
    assert c.evict(10) == [10, 11, 12]
    with pytest.raises(B.SglError):
        c.inc_lock_ref(h)                               # its node was evicted
    c.insert([4, 5], [20, 21])                          # may reuse the node's storage
    with pytest.raises(B.SglError):
        c.inc_lock_ref(h)
    assert c.evictable_tokens == 2 and c.protected_tokens == 0


def test_a_tree_built_batch_feeds_cascade_decode():
    """Lay out a decode batch the way a serving loop does -- look each prompt
    up in the tree, reuse the cached slots, take fresh slots for the rest,
    insert -- and hand the tree's groups to the cascade oracle, which must
    equal plain decode."""
    rng = np.random.default_rng(11)
    tree = B.RadixTree()
    dims = W.Dims(4, 2, 16, 4096, 0.25)
    free = list(rng.permutation(dims.pool_size).astype(int))
    system = [int(x) for x in rng.integers(0, 50, size=40)]
    prompts = []
    for _ in range(3):
        branch = system + [int(x) for x in rng.integers(0, 50, size=int(rng.integers(5, 30)))]
        for _ in range(int(rng.integers(2, 5))):
            prompts.append(branch + [int(x) for x in rng.integers(0, 50, size=int(rng.integers(0, 20)))])
    prompts.append([int(x) for x in rng.integers(0, 50, size=25)])
    rows = np.zeros((len(prompts), 128), np.int32)
    seq = []
    for r, p in enumerate(prompts):
        m, slots, _ = tree.match_prefix(p)
        new = [free.pop() for _ in range(len(p) - m + 1)]        # rest of the prompt + the decode token
        row = slots + new
        assert tree.insert(p, row[: len(p)]) == m
        rows[r, : len(row)] = row
        seq.append(len(row))
    nodes = [tree.match_prefix(p)[2] for p in prompts]
    start, length, depth, off, mem = tree.groups(nodes)
    assert start.size > 0 and depth.max() >= 1
    cg = W.CascadeGroups(start, length, depth, off, mem)
    # the groups are exactly what the rows share
    ref = W.shared_prefix_groups(rows, np.arange(len(prompts)), np.asarray(seq) - 1)
    for a, b in zip((cg.group_start, cg.group_len, cg.group_depth, cg.member_off, cg.members),
                    (ref.group_start, ref.group_len, ref.group_depth, ref.member_off, ref.members)):
        assert np.array_equal(a, b)
    live = np.unique(rows[rows > 0])
    k = W.f32_to_bf16_bits(rng.standard_normal((dims.pool_size, 2, 16)).astype(np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal((dims.pool_size, 2, 16)).astype(np.float32))
    q = W.f32_to_bf16_bits(rng.standard_normal((len(prompts), 4, 16)).astype(np.float32))
    rpi, sl = np.arange(len(prompts)), np.asarray(seq)
    plain = oracle.decode_attention(q, k, v, rows, rpi, sl, 2, 0.25)
    casc = oracle.cascade_decode_attention(q, k, v, rows, rpi, sl, cg.group_start, cg.group_len, cg.group_depth,
                                           cg.member_off, cg.members, 2, 0.25)
    assert live.size > 0 and np.max(np.abs(plain - casc)) < 1e-12


def test_tree_tokens_give_the_batch_hit_rate():
    """The paper's notation: hit rate = 1 - C / prompt tokens with C the summed
    edge lengths of the batch's radix tree -- brute force: C is the number of
    distinct token prefixes of the batch."""
    import bench
    rng = np.random.default_rng(13)
    stems, rows = [], []
    for _ in range(60):
        s = _seq(rng, stems, 4)
        stems.append(s)
        rows.append(np.asarray(s, np.int32))
    got = bench.prefix_sharing(rows)
    distinct = {tuple(r[: i + 1].tolist()) for r in rows for i in range(len(r))}
    total = sum(len(r) for r in rows)
    assert got["tree_tokens"] == len(distinct) and got["prompt_tokens"] == total
    assert abs(got["within_batch_hit_rate"] - (1 - len(distinct) / total)) < 1e-4
    # a tree workload (depth 3, fan-out 2, 16-token segments): 2 + 4 + 8 segments, each
    # cached once, plus one new token per leaf
    w = W.tree_of_thought_decode(depth=3, fanout=2, segment=16, steps=1, pool_size=1 << 12)
    sh = bench.sharing_of(w)["decode"]
    assert sh["tree_tokens"] == (2 + 4 + 8) * 16 + 8 and sh["prompt_tokens"] == 8 * (3 * 16 + 1)


def test_bench_groups_come_from_the_radix_tree():
    """The bench's cascade groups (the library's radix tree, step by step)
    equal the groups read off the rows, at every decode step of a tree
    workload, and a batch with no shared prefix has none."""
    import bench
    w = W.tree_of_thought_decode(depth=3, fanout=3, segment=20, steps=4, pool_size=1 << 14)
    got = bench.radix_tree_groups(w)
    assert len(got) == len(w.decode)
    for s, cg in enumerate(got):
        ref = W.tree_groups(w, s)
        assert cg.n_groups == ref.n_groups > 0
        for a, b in zip((cg.group_start, cg.group_len, cg.group_depth, cg.member_off, cg.members),
                        (ref.group_start, ref.group_len, ref.group_depth, ref.member_off, ref.members)):
            assert np.array_equal(a, b), s
    plain = W.decode_llama7b(pool_size=1 << 19)
    assert all(g.n_groups == 0 for g in bench.radix_tree_groups(plain))
