"""Pins of the cascade (shared-prefix-once) decode oracle and of the
shared-prefix groups the workloads derive from req_to_token rows.

Cascade decode reads the keys that several requests share once per group and
merges per-group softmax states with each request's private tail.  Nothing
here is compared with itself:
  * invariant: cascade == plain decode (oracle.decode_attention, pinned in
    test_oracle.py against full causal attention recomputed by torch) when
    the groups describe slots the members really share -- shared prefixes are
    identical slot numbers ("Inside SGLang", Step 3: Paged KV and the kernels
    that read it);
  * closed forms and brute force for the state merge (math.exp loops);
  * brute force for the groups: for every pair of requests, the end of the
    deepest group holding both equals the length of their common slot prefix;
  * planted slips in the merge and in the tail boundary are caught.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import attention as OA
from radixattention_prefix_shared_gb300 import workloads as W


def _small_tree(seed=5, **kw):
    dims = W.Dims(4, 2, 16, 1 << 14, 0.25)
    return W.random_tree_decode(seed=seed, dims=dims, pool_size=1 << 14, **kw)


def _run_both(w, cg, step=0):
    b = w.decode[step]
    pk, pv = w.dense_pools(decode_steps=step + 1)
    plain = oracle.decode_attention(b.q, pk, pv, w.req_to_token, b.req_pool_idx, b.seq_lens,
                                    w.dims.num_kv_heads, w.dims.sm_scale)
    casc = oracle.cascade_decode_attention(b.q, pk, pv, w.req_to_token, b.req_pool_idx, b.seq_lens,
                                           cg.group_start, cg.group_len, cg.group_depth,
                                           cg.member_off, cg.members, w.dims.num_kv_heads,
                                           w.dims.sm_scale)
    return plain, casc


# ------------------------------------------------------------ merge algebra

def test_merge_of_two_single_keys_closed_form():
    v1, v2 = np.array([1.0, -2.0]), np.array([0.5, 4.0])
    s1, s2 = 0.3, -1.7
    st = [OA.partial_state(np.array([1.0]), np.array([[s1]]), v1[None], 1.0),
          OA.partial_state(np.array([1.0]), np.array([[s2]]), v2[None], 1.0)]
    want = (math.exp(s1) * v1 + math.exp(s2) * v2) / (math.exp(s1) + math.exp(s2))
    assert np.allclose(OA.merge_states(st), want, rtol=0, atol=1e-15)
    # an empty subset contributes nothing, and the order of the states is free
    empty = OA.partial_state(np.array([1.0]), np.zeros((0, 1)), np.zeros((0, 2)), 1.0)
    assert empty[0] == -math.inf and empty[1] == 0.0
    assert np.allclose(OA.merge_states([empty, st[1], st[0]]), want, rtol=0, atol=1e-15)


def test_merge_survives_far_apart_maxima():
    # exp(1000) overflows float64: the merge must work relative to the max
    v = np.eye(3)
    st = [OA.partial_state(np.array([1.0]), np.array([[1000.0]]), v[:1], 1.0),
          OA.partial_state(np.array([1.0]), np.array([[0.0], [-5.0]]), v[1:], 1.0)]
    assert np.allclose(OA.merge_states(st), v[0], rtol=0, atol=1e-300)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_merge_of_random_split_equals_brute_force(seed):
    rng = np.random.default_rng(seed)
    n, d = int(rng.integers(2, 9)), int(rng.integers(1, 4))
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    scale = 0.7
    cut = np.sort(rng.choice(np.arange(1, n), size=int(rng.integers(1, n)), replace=False))
    parts = np.split(np.arange(n), cut)
    got = OA.merge_states([OA.partial_state(q, K[p], V[p], scale) for p in parts])
    w = [math.exp(scale * sum(q[t] * K[j, t] for t in range(d))) for j in range(n)]
    want = [sum(w[j] * V[j, t] for j in range(n)) / sum(w) for t in range(d)]
    assert max(abs(a - b) for a, b in zip(got, want)) < 1e-12


# ------------------------------------------------------------ groups

def test_groups_of_the_tree_workload_are_its_shared_nodes():
    w = W.tree_of_thought_decode(depth=3, fanout=3, segment=40, steps=2, pool_size=1 << 14)
    cg = W.tree_groups(w)
    # levels 0 and 1 are shared (3 and 9 nodes); leaf segments are private
    assert cg.n_groups == 3 + 9 and set(cg.group_len.tolist()) == {40}
    assert np.bincount(cg.group_depth).tolist() == [3, 9]
    assert sorted(np.diff(cg.member_off).tolist()) == [3] * 9 + [9] * 3
    assert np.array_equal(cg.shared_lens(27), np.full(27, 80))
    for j in range(cg.n_groups):
        m = cg.members[cg.member_off[j]: cg.member_off[j + 1]]
        d = int(cg.group_depth[j])
        # leaf l sits under level-d node l // 3^(2-d)
        assert len({int(x) // 3 ** (2 - d) for x in m}) == 1 and cg.group_start[j] == 40 * d


@pytest.mark.parametrize("seed", [5, 6, 7])
def test_deepest_common_group_ends_at_common_prefix(seed):
    w = _small_tree(seed)
    b = w.decode[0]
    cg = W.tree_groups(w)
    B = b.seq_lens.size
    rows = [w.req_to_token[b.req_pool_idx[r], : b.seq_lens[r]] for r in range(B)]
    ends = {}
    for j in range(cg.n_groups):
        m = [int(x) for x in cg.members[cg.member_off[j]: cg.member_off[j + 1]]]
        e = int(cg.group_start[j] + cg.group_len[j])
        for x in m:
            for y in m:
                ends[(x, y)] = max(ends.get((x, y), 0), e)
    for x in range(B):
        for y in range(B):
            if x == y:
                continue
            n = min(rows[x].size, rows[y].size)
            common = next((i for i in range(n) if rows[x][i] != rows[y][i]), n)
            assert ends.get((x, y), 0) == common, (x, y)


@pytest.mark.parametrize("seed", [5, 8])
def test_groups_tile_each_request_and_are_shared(seed):
    w = _small_tree(seed)
    b = w.decode[0]
    cg = W.tree_groups(w)
    mine = {}
    for j in range(cg.n_groups):
        m = cg.members[cg.member_off[j]: cg.member_off[j + 1]]
        assert m.size >= 2 and np.all(np.diff(m) > 0)
        a, e = int(cg.group_start[j]), int(cg.group_start[j] + cg.group_len[j])
        ref = w.req_to_token[b.req_pool_idx[m[0]], a:e]
        for r in m:
            assert np.array_equal(w.req_to_token[b.req_pool_idx[r], a:e], ref)
            mine.setdefault(int(r), []).append((int(cg.group_depth[j]), a, e))
    for r, gs in mine.items():
        gs.sort()
        assert [d for d, _, _ in gs] == list(range(len(gs)))
        assert gs[0][1] == 0 and all(gs[i][2] == gs[i + 1][1] for i in range(len(gs) - 1))
        assert gs[-1][2] <= b.seq_lens[r]


# ------------------------------------------------------------ cascade

@pytest.mark.parametrize("seed", [5, 6])
def test_cascade_equals_plain_decode(seed):
    w = _small_tree(seed)
    cg = W.tree_groups(w)
    assert cg.n_groups > 0 and cg.max_depth >= 2
    plain, casc = _run_both(w, cg)
    assert np.max(np.abs(plain - casc)) < 1e-12


def test_cascade_on_tree_steps():
    w = W.tree_of_thought_decode(depth=3, fanout=2, segment=33, steps=3, pool_size=1 << 13)
    for step in range(3):
        plain, casc = _run_both(w, W.tree_groups(w, step), step)
        assert np.max(np.abs(plain - casc)) < 1e-12


def test_cascade_reads_group_keys_from_the_first_member():
    w = _small_tree(9)
    b = w.decode[0]
    cg = W.tree_groups(w)
    j = int(np.argmax(np.diff(cg.member_off)))
    m = cg.members[cg.member_off[j]: cg.member_off[j + 1]]
    a = int(cg.group_start[j])
    victim = int(m[-1])
    # break the sharing: the victim's first group position points elsewhere
    other = w.live_slots[~np.isin(w.live_slots, w.req_to_token[b.req_pool_idx[victim]])][0]
    broken = W.Workload(**{**w.__dict__, "req_to_token": w.req_to_token.copy()})
    broken.req_to_token[b.req_pool_idx[victim], a] = other
    pk, pv = w.dense_pools(decode_steps=1)
    args = (cg.group_start, cg.group_len, cg.group_depth, cg.member_off, cg.members,
            w.dims.num_kv_heads, w.dims.sm_scale)
    got = oracle.cascade_decode_attention(b.q, pk, pv, broken.req_to_token, b.req_pool_idx,
                                          b.seq_lens, *args, requests=[victim])
    plain_broken = oracle.decode_attention(b.q, pk, pv, broken.req_to_token, b.req_pool_idx,
                                           b.seq_lens, w.dims.num_kv_heads, w.dims.sm_scale,
                                           requests=[victim])
    plain_shared = oracle.decode_attention(b.q, pk, pv, w.req_to_token, b.req_pool_idx,
                                           b.seq_lens, w.dims.num_kv_heads, w.dims.sm_scale,
                                           requests=[victim])
    assert np.max(np.abs(got - plain_shared)) < 1e-12
    assert np.max(np.abs(got - plain_broken)) > 1e-6


CASCADE_MUTANTS = {
    "merge without max rescale": lambda states: (
        sum(acc for _, _, acc in states) / sum(l for _, l, _ in states)),
    "merge keeps only the largest state": lambda states: (
        (lambda s: s[2] / s[1])(max(states, key=lambda t: t[0]))),
}


@pytest.mark.parametrize("name", list(CASCADE_MUTANTS))
def test_cascade_pins_catch_planted_slips(name, monkeypatch):
    w = _small_tree(6)
    cg = W.tree_groups(w)
    plain, _ = _run_both(w, cg)
    monkeypatch.setattr(OA, "merge_states", CASCADE_MUTANTS[name])
    _, casc = _run_both(w, cg)
    assert np.max(np.abs(plain - casc)) > 1e-6, f"planted slip '{name}' not caught"


def test_cascade_pin_catches_uncovered_keys():
    """Groups one position too short leave keys that no state covers."""
    w = _small_tree(7)
    cg = W.tree_groups(w)
    plain, _ = _run_both(w, cg)
    cg2 = W.CascadeGroups(cg.group_start, cg.group_len - 1 * (cg.group_len > 1), cg.group_depth,
                          cg.member_off, cg.members)
    _, casc = _run_both(w, cg2)
    assert np.max(np.abs(plain - casc)) > 1e-6
