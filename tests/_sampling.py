"""Which rows the full-size parity tests compare with the oracle (host
only; no torch)."""
import numpy as np

TILE_ROWS = 128  # rows of an extend Q tile: tokens x query heads of one KV head


def sample_requests(seq, k, seed):
    """k requests at random plus the longest and the shortest (all if k >= B)."""
    seq = np.asarray(seq)
    if k >= seq.size:
        return list(range(seq.size))
    rng = np.random.default_rng(seed)
    pick = {int(np.argmax(seq)), int(np.argmin(seq))}
    pick |= set(int(x) for x in rng.choice(seq.size, size=k, replace=False))
    return sorted(pick)


def tile_edge_tokens(e, requests, g):
    """Row indices (into the extend batch) of the first and the last token of
    every Q tile of the listed requests: a tile holds 128 / g tokens."""
    tpt = TILE_ROWS // g
    offs = np.concatenate([[0], np.cumsum(e.extend_lens)])
    toks = set()
    for r in requests:
        n = int(e.extend_lens[r])
        for a in range(0, n, tpt):
            toks |= {int(offs[r] + a), int(offs[r] + min(a + tpt, n) - 1)}
    return np.array(sorted(toks))


def extreme_prefix_requests(e):
    """The requests with the longest and the shortest prefix (among those
    with suffix tokens)."""
    live = np.nonzero(np.asarray(e.extend_lens) > 0)[0]
    p = np.asarray(e.prefix_lens)[live]
    return sorted({int(live[np.argmax(p)]), int(live[np.argmin(p)])})
