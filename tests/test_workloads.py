"""Properties of the seeded slot layouts (host only)."""
import numpy as np
import pytest

from radixattention_prefix_shared_gb300 import workloads as W


def _rows(w, rows, lens):
    return [w.req_to_token[r, :n] for r, n in zip(rows, lens)]


def _check_common(w):
    S = w.dims.pool_size
    assert w.req_to_token.dtype == np.int32
    assert w.req_to_token.min() >= 0 and w.req_to_token.max() < S
    assert np.unique(w.live_slots).size == w.live_slots.size
    new = []
    if w.extend is not None:
        new.append(w.extend.slots)
    new += [b.slots for b in w.decode]
    new = np.concatenate(new)
    assert np.unique(new).size == new.size, "new-token slots must be distinct"
    assert np.intersect1d(new, w.live_slots).size == 0, "new tokens must take free slots"


def test_tiny_layout():
    w = W.tiny()
    _check_common(w)
    e, d = w.extend, w.decode[0]
    assert list(e.prefix_lens) == [0, 16, 33, 64] and list(e.extend_lens) == [8, 1, 31, 17]
    assert list(d.seq_lens) == [9, 18, 65, 82]
    assert e.q.shape == (57, 2, 64) and d.q.shape == (4, 2, 64)
    r1, r2 = w.req_to_token[e.req_pool_idx[1]], w.req_to_token[e.req_pool_idx[2]]
    assert np.array_equal(r1[:16], r2[:16])
    assert np.intersect1d(r1[:16], r2[16:33]).size == 0
    # the suffix slots sit in the rows after the prefix, the decode slot last
    off = 0
    for r in range(4):
        row = w.req_to_token[e.req_pool_idx[r]]
        p, n = e.prefix_lens[r], e.extend_lens[r]
        assert np.array_equal(row[p: p + n], e.slots[off: off + n])
        assert row[p + n] == d.slots[r]
        off += n
    # tails past seq_len point at slots nobody writes (NaN in the pool)
    used = set(np.concatenate([w.live_slots, e.slots, d.slots]).tolist())
    for r in range(4):
        tail = w.req_to_token[e.req_pool_idx[r], d.seq_lens[r]:]
        assert not (set(tail.tolist()) & used)
    # q/k/v ~ N(0,1)/8
    x = (e.q.astype(np.uint32) << 16).view(np.float32)
    assert abs(x.std() - 0.125) < 0.01


def test_row_source_regenerates_any_range():
    rs = W.RowSource(5, 9, 3000, (2, 8), 1.0)
    full = rs.all()
    assert np.array_equal(rs.rows(1000, 2500), full[1000:2500])
    idx = np.array([2999, 0, 1024, 1023, 7])
    assert np.array_equal(rs.take(idx), full[idx])
    assert np.array_equal(W.RowSource(5, 9, 3000, (2, 8), 1.0).rows(17, 18), full[17:18])


def test_decode_layout_small():
    w = W.decode_llama7b(batch=8, pool_size=1 << 15)
    _check_common(w)
    b = w.decode[0]
    assert b.seq_lens.min() >= 512 and b.seq_lens.max() <= 4096
    rows = _rows(w, b.req_pool_idx, b.seq_lens)
    allslots = np.concatenate(rows)
    assert np.unique(allslots).size == allslots.size        # no sharing
    assert all(r[-1] == s for r, s in zip(rows, b.slots))


def test_shared_prompt_layout_small():
    w = W.shared_prompt_extend(batch=4, prefix=300, extend=40, pool_size=1 << 12)
    _check_common(w)
    e = w.extend
    rows = [w.req_to_token[r] for r in e.req_pool_idx]
    for r in rows[1:]:
        assert np.array_equal(r[:300], rows[0][:300])
    assert e.total_extend == 160


def test_tree_layout_small():
    w = W.tree_of_thought_decode(depth=3, fanout=2, segment=4, steps=3, pool_size=512)
    _check_common(w)
    assert len(w.decode) == 3
    b0 = w.decode[0]
    leaves = b0.req_pool_idx.size
    assert leaves == 8
    rows = [w.req_to_token[r] for r in b0.req_pool_idx]
    # siblings share their parent's segments, cousins only the root-level one
    assert np.array_equal(rows[0][:8], rows[1][:8]) and not np.array_equal(rows[0][8:12], rows[1][8:12])
    assert np.array_equal(rows[0][:4], rows[3][:4]) and not np.array_equal(rows[0][4:8], rows[3][4:8])
    for s, b in enumerate(w.decode):
        assert (b.seq_lens == 12 + s + 1).all()
        for i, r in enumerate(b.req_pool_idx):
            assert w.req_to_token[r, 12 + s] == b.slots[i]


def test_chunked_prefill_layout_small():
    S = 1 << 17
    w = W.chunked_prefill_mix(n_chunks=3, chunk=256, prefix_max=4096, n_decode=12,
                              decode_range=(64, 8192), pool_size=S)
    _check_common(w)
    rec = w.recipe
    assert rec["evicted"] == round(0.3 * S)
    e, d = w.extend, w.decode[0]
    assert (e.extend_lens == 256).all() and (e.prefix_lens <= 4096).all()
    assert d.seq_lens.min() >= 64 and d.seq_lens.max() <= 8192
    # live contexts are spread over the pool (interleaved allocation)
    row = w.req_to_token[d.req_pool_idx[np.argmax(d.seq_lens)], : d.seq_lens.max() - 1]
    runs = np.count_nonzero(np.diff(row) != 1) + 1
    assert runs > 1
    # new tokens come from slots freed by the eviction
    assert np.intersect1d(e.slots, w.live_slots).size == 0


def test_same_seed_same_bits():
    a, b = W.tiny(), W.tiny()
    assert np.array_equal(a.req_to_token, b.req_to_token)
    assert np.array_equal(a.extend.q, b.extend.q)
    assert np.array_equal(a.live_k.all(), b.live_k.all())


@pytest.mark.parametrize("page", [16, 64])
def test_paged_layouts_own_whole_pages(page):
    """With a page size, every request's positions fill whole pages of
    consecutive slots (page-aligned), no page is shared between two requests
    except the shared prompt's, and the new tokens sit inside their pages."""
    w = W.decode_llama7b(batch=8, pool_size=1 << 16, seq_range=(100, 700), page_size=page)
    d = w.decode[0]
    owner = {}
    for r in range(d.seq_lens.size):
        row = w.req_to_token[d.req_pool_idx[r], : d.seq_lens[r]].astype(np.int64)
        assert row[-1] == d.slots[r]
        for k in range(0, row.size, page):
            run = row[k: k + page]
            assert run[0] % page == 0 and np.array_equal(run, run[0] + np.arange(run.size))
            assert owner.setdefault(run[0] // page, r) == r
    sp = W.shared_prompt_extend(batch=4, prefix=256, extend=40, pool_size=1 << 14, page_size=page)
    e = sp.extend
    assert e.slots.size == 4 * 40 and np.unique(e.slots).size == e.slots.size
    assert np.all(e.slots.reshape(4, 40)[:, 0] % page == 0)
    shared = sp.req_to_token[e.req_pool_idx[0], :256].astype(np.int64)
    assert np.all(shared.reshape(-1, page)[:, 0] % page == 0)
    assert all(np.array_equal(sp.req_to_token[r, :256], shared) for r in e.req_pool_idx)


def test_parity_sampler_covers_every_tile_edge():
    """The full-size extend sample holds both ends of every Q tile of the
    chosen requests, and the decode sample keeps the extremes."""
    from _sampling import extreme_prefix_requests, sample_requests, tile_edge_tokens
    e = W.chunked_prefill_mix(pool_size=1 << 19, n_decode=4).extend
    reqs = extreme_prefix_requests(e)
    assert len(reqs) == 2
    assert e.prefix_lens[reqs].max() == e.prefix_lens.max() and e.prefix_lens[reqs].min() == e.prefix_lens.min()
    toks = tile_edge_tokens(e, reqs, 2)
    assert toks.size == len(reqs) * 2 * (2048 // 64)
    offs = np.concatenate([[0], np.cumsum(e.extend_lens)])
    for r in reqs:
        mine = toks[(toks >= offs[r]) & (toks < offs[r + 1])] - offs[r]
        assert mine[0] == 0 and mine[-1] == e.extend_lens[r] - 1
        assert set(mine[::2] % 64) == {0} and set(mine[1::2] % 64) == {63}
    # a ragged last tile ends at the request's last token
    class _E:
        extend_lens = np.array([70, 5])
        prefix_lens = np.array([0, 9])
    assert tile_edge_tokens(_E, [0, 1], 4).tolist() == [0, 31, 32, 63, 64, 69, 70, 74]
    assert sample_requests(np.arange(10), 20, 0) == list(range(10))
    s = sample_requests(np.array([5, 1, 9, 3, 7, 2]), 2, 1)
    assert 2 in s and 1 in s
