"""Pins of the radix-tree oracle against things other than itself.

  * brute force: a plain dictionary of every cached token prefix (first
    inserted slot wins) gives the matched length and slots of any lookup, and
    what insert reports as already cached;
  * the pages' eviction rules as scenarios ("Inside SGLang", Step 4: only
    unlocked leaves, least recently used first, a parent that becomes a leaf is
    next, a shared stem lasts longest; "SGLang" notes, Eviction; a split keeps
    the lock of the node it was cut from);
  * invariants: evictable + locked tokens = tokens in the tree; evict never
    frees a locked token; every freed slot leaves the brute-force model;
  * groups: for every pair of requests, the deepest group holding both ends
    where their token sequences diverge.
"""
import numpy as np
import pytest

from oracle.radix import RadixTree


class Model:
    """Brute force: {token prefix: slot of its last token}."""

    def __init__(self):
        self.d = {}

    def match(self, toks):
        n, slots = 0, []
        while n < len(toks) and tuple(toks[: n + 1]) in self.d:
            slots.append(self.d[tuple(toks[: n + 1])])
            n += 1
        return n, slots

    def insert(self, toks, slots):
        n, _ = self.match(toks)
        for i in range(n, len(toks)):
            self.d[tuple(toks[: i + 1])] = slots[i]
        return n


def _seq(rng, stems, vocab=6):
    """A token sequence that often shares a prefix with an earlier one."""
    if stems and rng.random() < 0.7:
        base = stems[int(rng.integers(len(stems)))]
        cut = int(rng.integers(0, len(base) + 1))
        return base[:cut] + [int(x) for x in rng.integers(0, vocab, size=int(rng.integers(0, 8)))]
    return [int(x) for x in rng.integers(0, vocab, size=int(rng.integers(1, 12)))]


@pytest.mark.parametrize("seed", range(6))
def test_match_and_insert_equal_brute_force(seed):
    rng = np.random.default_rng(seed)
    t, m, stems, nxt = RadixTree(), Model(), [], 1000
    for _ in range(300):
        s = _seq(rng, stems)
        if rng.random() < 0.5:
            slots = list(range(nxt, nxt + len(s)))
            nxt += len(s)
            assert t.insert(s, slots) == m.insert(s, slots)
            stems.append(s)
        else:
            n, slots, _ = t.match_prefix(s)
            assert (n, slots) == m.match(s)
        assert t.total_tokens() == len(m.d)


def test_eviction_follows_the_pages_rules():
    t = RadixTree()
    stem = list(range(100, 120))
    t.insert(stem + [1, 2, 3], list(range(0, 23)))          # branch A
    t.insert(stem + [4, 5], [0] * 20 + [50, 51])             # branch B (stem slots are duplicates)
    t.insert([9, 9], [60, 61])                               # an unrelated leaf C
    t.match_prefix(stem + [1, 2, 3])                         # touch A: B and C are older
    # least recently used leaf first: B (inserted first), then C
    assert t.evict(1) == [50, 51]
    assert t.evict(1) == [60, 61]
    # the stem outlives its branches: A goes next, then the stem itself
    assert t.evict(1) == [20, 21, 22]
    assert t.evict(1) == list(range(0, 20))
    assert t.total_tokens() == 0 and t.evict(5) == []


def test_a_split_tail_keeps_its_access_time():
    """A match ending inside a node passes only the cut-off prefix: the tail
    keeps the older time and is evicted before a leaf touched later."""
    t = RadixTree()
    t.insert([1, 2, 3], [10, 11, 12])
    t.insert([5], [50])
    t.match_prefix([1])
    assert t.evict(1) == [11, 12]
    assert t.evict(1) == [50]


def test_locked_paths_survive_and_split_keeps_the_lock():
    t = RadixTree()
    a = list(range(10))
    t.insert(a, list(range(10)))
    _, _, node = t.match_prefix(a)
    t.inc_lock_ref(node)
    # B shares 5 tokens: A's node is cut at 5; both halves must stay locked
    b = a[:5] + [77, 78]
    assert t.insert(b, list(range(200, 207))) == 5
    assert t.protected == 10 and t.evictable == 2
    assert sorted(t.evict(100)) == [205, 206]
    assert t.match_prefix(a)[0] == 10
    t.dec_lock_ref(node)
    assert t.protected == 0 and t.evictable == 10
    assert sorted(t.evict(100)) == list(range(10))


@pytest.mark.parametrize("seed", range(4))
def test_random_lock_evict_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    t, m, stems, nxt, locks = RadixTree(), Model(), [], 0, []
    for _ in range(400):
        op = rng.random()
        s = _seq(rng, stems)
        if op < 0.4:
            slots = list(range(nxt, nxt + len(s)))
            nxt += len(s)
            t.insert(s, slots)
            m.insert(s, slots)
            stems.append(s)
        elif op < 0.6:
            n, _, node = t.match_prefix(s)
            if n:
                t.inc_lock_ref(node)
                locks.append((s[:n], node))
        elif op < 0.7 and locks:
            _, node = locks.pop(int(rng.integers(len(locks))))
            t.dec_lock_ref(node)
        else:
            freed = t.evict(int(rng.integers(1, 20)))
            gone = {k for k, v in m.d.items() if v in set(freed)}
            assert len(gone) == len(freed)
            for k in gone:
                del m.d[k]
            for toks, _ in locks:                # locked paths are intact
                assert t.match_prefix(toks)[0] == len(toks)
        assert t.evictable + t.protected == t.total_tokens() == len(m.d)
        assert t.evictable >= 0 and t.protected >= 0


def test_groups_end_where_requests_diverge():
    rng = np.random.default_rng(7)
    t, stems, nxt = RadixTree(), [], 0
    reqs = []
    for _ in range(40):
        s = _seq(rng, stems, vocab=3)
        t.insert(s, list(range(nxt, nxt + len(s))))
        nxt += len(s)
        stems.append(s)
    for s in stems[:25]:
        n, _, node = t.match_prefix(s)
        reqs.append((s[:n], node))
    groups = t.groups([node for _, node in reqs])
    ends = {}
    for depth, start, length, ms in groups:
        assert length >= 1 and len(ms) >= 2
        for x in ms:
            for y in ms:
                ends[(x, y)] = max(ends.get((x, y), 0), start + length)
    for x, (sx, _) in enumerate(reqs):
        for y, (sy, _) in enumerate(reqs):
            if x != y:
                n = min(len(sx), len(sy))
                common = next((i for i in range(n) if sx[i] != sy[i]), n)
                assert ends.get((x, y), 0) == common


def _split_without_lock(self, child, k):
    parent = child.parent
    new = self._new_node(child.key[:k], child.value[:k], parent, child.last_access)
    parent.children[child.key[0]] = new
    child.key, child.value = child.key[k:], child.value[k:]
    child.parent = new
    new.children[child.key[0]] = child
    return new


def _touch_without_time(self, node):
    node.last_access = node.seq          # creation order instead of access order


@pytest.mark.parametrize("slip", ["split drops the lock", "eviction ignores access times"])
def test_pins_catch_planted_slips(slip, monkeypatch):
    import oracle.radix as R
    if slip == "split drops the lock":
        monkeypatch.setattr(R.RadixTree, "_split", _split_without_lock)
        case = test_locked_paths_survive_and_split_keeps_the_lock
    else:
        monkeypatch.setattr(R.RadixTree, "_touch", _touch_without_time)
        case = test_eviction_follows_the_pages_rules
    with pytest.raises(AssertionError):
        case()
