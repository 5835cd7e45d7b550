"""Pins of the fp64 oracle against things other than itself.

Each pin below would fail for a plausible slip in the oracle: the mutation
tests at the end plant such slips (in the oracle, on the CPU) and check that
a pin catches every one.

  * library special case: EXTEND rows == the last rows of full causal
    attention recomputed from scratch by torch's scaled_dot_product_attention
    (float64, CPU) over prefix+suffix -- "Origins: the paper and the first
    commit", Batching (EXTEND computes only the suffix; seq_len = prefix +
    extend) with "Inside SGLang", Step 3 (mask above the diagonal);
  * closed forms: q = 0 gives the mean of the visible V rows; one key gives
    its V row exactly; a dominant key gives its V row; constant V rows give
    that constant;
  * invariants: decode == extend with one new token; relabelling slots by a
    permutation changes nothing; requests sharing prefix slots == requests
    with private copies ("Inside SGLang", Step 3: sharing is identical slot
    numbers, no copy);
  * brute force: pure-Python loops with math.exp on tiny sizes;
  * printed numbers: the 1/sqrt(128) scale and the KV byte figures.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as OA
from radixattention_prefix_shared_gb300 import workloads as W
from radixattention_prefix_shared_gb300 import workmodel as WM

from _cases import decode_case, extend_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")


# ------------------------------------------------------------------ helpers

def _bits_to_torch64(bits):
    """bf16 bits -> float64 through torch's own bfloat16 dtype (a second,
    independent conversion route)."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double()


def _oracle_extend(w, **kw):
    e = w.extend
    pk, pv = w.dense_pools(with_extend=False)
    return oracle.extend_attention(e.q, e.k_new, e.v_new, pk, pv, w.req_to_token, e.req_pool_idx,
                                   e.prefix_lens, e.extend_lens, w.dims.num_kv_heads,
                                   w.dims.sm_scale, **kw)


def _sdpa_extend(w):
    """Full causal attention over prefix+suffix per request, last rows kept."""
    e = w.extend
    pk, pv = w.dense_pools(with_extend=False)
    Hq, Hkv, D = w.dims.num_q_heads, w.dims.num_kv_heads, w.dims.head_dim
    out = []
    off = 0
    for r in range(e.extend_lens.size):
        p, n = int(e.prefix_lens[r]), int(e.extend_lens[r])
        slots = w.req_to_token[e.req_pool_idx[r], :p]
        K = torch.cat([_bits_to_torch64(pk[slots]), _bits_to_torch64(e.k_new[off: off + n])])
        V = torch.cat([_bits_to_torch64(pv[slots]), _bits_to_torch64(e.v_new[off: off + n])])
        Q = torch.cat([torch.zeros(p, Hq, D, dtype=torch.float64), _bits_to_torch64(e.q[off: off + n])])
        o = torch.nn.functional.scaled_dot_product_attention(
            Q.transpose(0, 1)[None], K.transpose(0, 1)[None], V.transpose(0, 1)[None],
            is_causal=True, scale=w.dims.sm_scale, enable_gqa=(Hq != Hkv))
        out.append(o[0].transpose(0, 1)[p:].numpy())
        off += n
    return np.concatenate(out) if out else np.zeros((0, Hq, D))


def _oracle_decode(w, step=0, **kw):
    b = w.decode[step]
    pk, pv = w.dense_pools(decode_steps=step + 1)
    return oracle.decode_attention(b.q, pk, pv, w.req_to_token, b.req_pool_idx, b.seq_lens,
                                   w.dims.num_kv_heads, w.dims.sm_scale, **kw)


EXTEND_SHAPES = [
    dict(Hq=2, Hkv=2, D=16, prefix_lens=[0, 5, 17], extend_lens=[4, 1, 9]),
    dict(Hq=4, Hkv=2, D=8, prefix_lens=[3, 0, 12, 7], extend_lens=[6, 3, 2, 1]),
    dict(Hq=8, Hkv=2, D=32, prefix_lens=[40, 1], extend_lens=[13, 30]),
    dict(Hq=6, Hkv=3, D=64, prefix_lens=[0, 64, 33, 16], extend_lens=[8, 1, 31, 17]),
]


# ------------------------------------------------------------ library pin

@pytest.mark.parametrize("shape", EXTEND_SHAPES)
def test_extend_equals_full_causal_recompute(shape):
    w = extend_case(7, **shape)
    got = _oracle_extend(w)
    ref = _sdpa_extend(w)
    assert got.shape == ref.shape
    assert np.max(np.abs(got - ref)) < 1e-12


def test_tiny_workload_extend_equals_full_causal_recompute():
    w = W.tiny()
    assert np.max(np.abs(_oracle_extend(w) - _sdpa_extend(w))) < 1e-12


# ------------------------------------------------------------ closed forms

def _zero_q(w):
    w.extend.q[:] = 0
    for b in w.decode:
        b.q[:] = 0
    return w


def test_zero_query_gives_mean_of_visible_values():
    w = _zero_q(extend_case(3, Hq=4, Hkv=2, D=16, prefix_lens=[5, 0, 9], extend_lens=[3, 4, 2],
                            decode_after=True))
    got = _oracle_extend(w)
    e = w.extend
    pk, pv = w.dense_pools(with_extend=False)
    off = 0
    for r in range(3):
        p, n = int(e.prefix_lens[r]), int(e.extend_lens[r])
        Vrows = np.concatenate([pv[w.req_to_token[e.req_pool_idx[r], :p]], e.v_new[off: off + n]])
        Vf = OA.bf16_bits_to_f64(Vrows)
        for i in range(n):
            for h in range(4):
                want = Vf[: p + i + 1, h // 2].mean(axis=0)
                assert np.max(np.abs(got[off + i, h] - want)) < 1e-14
        off += n
    # decode: mean over all seq_len rows of the request
    d = _oracle_decode(w)
    b = w.decode[0]
    pk, pv = w.dense_pools(decode_steps=1)
    for r in range(3):
        Vf = OA.bf16_bits_to_f64(pv[w.req_to_token[b.req_pool_idx[r], : b.seq_lens[r]]])
        for h in range(4):
            assert np.max(np.abs(d[r, h] - Vf[:, h // 2].mean(axis=0))) < 1e-14


def test_single_key_gives_its_value_row_exactly():
    w = decode_case(5, Hq=4, Hkv=4, D=32, seq_lens=[1, 1, 1])
    d = _oracle_decode(w)
    b = w.decode[0]
    assert np.array_equal(d, OA.bf16_bits_to_f64(b.v_new))
    # extend with prefix 0: suffix query 0 sees only its own key
    w2 = extend_case(6, Hq=2, Hkv=1, D=16, prefix_lens=[0, 0], extend_lens=[3, 1])
    got = _oracle_extend(w2)
    V = OA.bf16_bits_to_f64(w2.extend.v_new)
    assert np.array_equal(got[0], np.repeat(V[0], 2, axis=0))
    assert np.array_equal(got[3], np.repeat(V[3], 2, axis=0))


def test_dominant_key_selects_its_value_row():
    w = decode_case(8, Hq=2, Hkv=1, D=16, seq_lens=[6])
    b = w.decode[0]
    one = W.f32_to_bf16_bits(np.ones(16, np.float32))
    b.q[0, :] = one
    # every cached key 0 except position 3, which is 8*ones: score 8*16/4 = 32
    pk, pv = w.dense_pools(decode_steps=1)
    row = w.req_to_token[b.req_pool_idx[0]]
    pk[row[:5]] = 0
    pk[row[3]] = W.f32_to_bf16_bits(np.full((1, 16), 8.0, np.float32))
    pk[row[5]] = 0
    d = oracle.decode_attention(b.q, pk, pv, w.req_to_token, b.req_pool_idx, b.seq_lens, 1)
    want = OA.bf16_bits_to_f64(pv[row[3], 0])
    assert np.max(np.abs(d[0, 0] - want)) < 1e-12 * (1 + np.abs(want).max())
    assert np.max(np.abs(d[0, 1] - want)) < 1e-12 * (1 + np.abs(want).max())


def test_constant_values_give_that_constant():
    w = extend_case(9, Hq=4, Hkv=4, D=8, prefix_lens=[7, 2], extend_lens=[5, 3])
    c = W.f32_to_bf16_bits(np.float32([0.3125]))[0]
    w.extend.v_new[:] = c
    pk, pv = w.dense_pools(with_extend=False)
    pv[:] = c
    e = w.extend
    got = oracle.extend_attention(e.q, e.k_new, e.v_new, pk, pv, w.req_to_token, e.req_pool_idx,
                                  e.prefix_lens, e.extend_lens, 4)
    assert np.max(np.abs(got - 0.3125)) < 1e-15


# ------------------------------------------------------------ invariants

def test_decode_equals_extend_with_one_new_token():
    w = decode_case(11, Hq=8, Hkv=2, D=32, seq_lens=[1, 7, 40, 129])
    b = w.decode[0]
    pk, pv = w.dense_pools(decode_steps=1)
    d = oracle.decode_attention(b.q, pk, pv, w.req_to_token, b.req_pool_idx, b.seq_lens, 2)
    # same request as EXTEND: prefix = seq_len-1 cached slots, one suffix token
    # whose k/v are the decode token's
    pk0, pv0 = w.dense_pools(decode_steps=0)
    x = oracle.extend_attention(b.q, b.k_new, b.v_new, pk0, pv0, w.req_to_token, b.req_pool_idx,
                                b.seq_lens - 1, np.ones_like(b.seq_lens), 2)
    assert np.max(np.abs(d - x)) < 1e-14


def _relabel(w, pk, pv, g):
    perm = g.permutation(w.dims.pool_size)
    pk2 = np.empty_like(pk)
    pv2 = np.empty_like(pv)
    pk2[perm] = pk
    pv2[perm] = pv
    return perm[w.req_to_token].astype(np.int32), pk2, pv2


def test_slot_permutation_changes_nothing():
    w = extend_case(12, Hq=4, Hkv=2, D=16, prefix_lens=[9, 30, 0], extend_lens=[4, 7, 5],
                    shares=[(0, 1, 9)], decode_after=True)
    e = w.extend
    pk, pv = w.dense_pools(with_extend=False)
    base = _oracle_extend(w)
    rtt2, pk2, pv2 = _relabel(w, pk, pv, np.random.default_rng(0))
    got = oracle.extend_attention(e.q, e.k_new, e.v_new, pk2, pv2, rtt2, e.req_pool_idx,
                                  e.prefix_lens, e.extend_lens, 2)
    assert np.array_equal(base, got)
    b = w.decode[0]
    pk, pv = w.dense_pools(decode_steps=1)
    base = oracle.decode_attention(b.q, pk, pv, w.req_to_token, b.req_pool_idx, b.seq_lens, 2)
    rtt2, pk2, pv2 = _relabel(w, pk, pv, np.random.default_rng(1))
    got = oracle.decode_attention(b.q, pk2, pv2, rtt2, b.req_pool_idx, b.seq_lens, 2)
    assert np.array_equal(base, got)


def test_shared_prefix_equals_private_copies():
    w = extend_case(13, Hq=4, Hkv=1, D=16, prefix_lens=[20, 20, 11], extend_lens=[3, 6, 2],
                    shares=[(0, 1, 16), (0, 2, 11)])
    e = w.extend
    pk, pv = w.dense_pools(with_extend=False)
    shared = _oracle_extend(w)
    # give requests 1 and 2 private copies of the shared slots
    rtt = w.req_to_token.copy()
    used = set(np.concatenate([w.live_slots, e.slots]).tolist())
    free = [s for s in range(w.dims.pool_size) if s not in used]
    for r, n in ((1, 16), (2, 11)):
        row = e.req_pool_idx[r]
        for j in range(n):
            s_new = free.pop()
            pk[s_new] = pk[rtt[row, j]]
            pv[s_new] = pv[rtt[row, j]]
            rtt[row, j] = s_new
    assert len(np.intersect1d(rtt[e.req_pool_idx[1], :16], rtt[e.req_pool_idx[0], :16])) == 0
    private = oracle.extend_attention(e.q, e.k_new, e.v_new, pk, pv, rtt, e.req_pool_idx,
                                      e.prefix_lens, e.extend_lens, 1)
    assert np.array_equal(shared, private)


def test_sampled_rows_match_full_output():
    w = extend_case(14, Hq=4, Hkv=2, D=16, prefix_lens=[9, 0, 21], extend_lens=[4, 7, 5])
    full = _oracle_extend(w)
    toks = np.array([15, 0, 4, 10, 3])
    assert np.array_equal(_oracle_extend(w, tokens=toks), full[toks])
    full_d = _oracle_decode(extend_case(14, Hq=4, Hkv=2, D=16, prefix_lens=[9, 0, 21],
                                        extend_lens=[4, 7, 5], decode_after=True))
    wd = extend_case(14, Hq=4, Hkv=2, D=16, prefix_lens=[9, 0, 21], extend_lens=[4, 7, 5],
                     decode_after=True)
    assert np.array_equal(_oracle_decode(wd, requests=[2, 0]), full_d[[2, 0]])


# ------------------------------------------------------------ brute force

def _brute_attention(qvec, keys, vals, scale):
    scores = [scale * sum(a * b for a, b in zip(qvec, k)) for k in keys]
    m = max(scores)
    ws = [math.exp(s - m) for s in scores]
    tot = sum(ws)
    return [sum(w_ * v[d] for w_, v in zip(ws, vals)) / tot for d in range(len(vals[0]))]


def _f(bits):
    return [float(x) for x in OA.bf16_bits_to_f64(bits).reshape(-1)]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_tiny_extend_and_decode(seed):
    rng = np.random.default_rng(seed)
    Hkv = int(rng.integers(1, 3))
    Hq = Hkv * int(rng.integers(1, 3))
    D = int(rng.integers(1, 5))
    P = [int(x) for x in rng.integers(0, 4, size=3)]
    E = [int(x) for x in rng.integers(1, 3, size=3)]
    w = extend_case(100 + seed, Hq=Hq, Hkv=Hkv, D=D, prefix_lens=P, extend_lens=E, decode_after=True)
    e = w.extend
    pk, pv = w.dense_pools(with_extend=False)
    got = _oracle_extend(w)
    scale = w.dims.sm_scale
    t = 0
    for r in range(3):
        row = w.req_to_token[e.req_pool_idx[r]]
        for i in range(E[r]):
            for h in range(Hq):
                kh = h // (Hq // Hkv)
                keys, vals = [], []
                for j in range(P[r]):
                    keys.append(_f(pk[row[j], kh]))
                    vals.append(_f(pv[row[j], kh]))
                o = t - i
                for j in range(i + 1):
                    keys.append(_f(e.k_new[o + j, kh]))
                    vals.append(_f(e.v_new[o + j, kh]))
                want = _brute_attention(_f(e.q[t, h]), keys, vals, scale)
                assert max(abs(a - b) for a, b in zip(got[t, h], want)) < 1e-12
            t += 1
    b = w.decode[0]
    pk, pv = w.dense_pools(decode_steps=1)
    d = _oracle_decode(w)
    for r in range(3):
        row = w.req_to_token[b.req_pool_idx[r]]
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            keys = [_f(pk[row[j], kh]) for j in range(b.seq_lens[r])]
            vals = [_f(pv[row[j], kh]) for j in range(b.seq_lens[r])]
            want = _brute_attention(_f(b.q[r, h]), keys, vals, scale)
            assert max(abs(a - c) for a, c in zip(d[r, h], want)) < 1e-12


# ------------------------------------------------------------ store_kv

def test_store_kv_is_an_index_assignment():
    rng = np.random.default_rng(3)
    S, Hkv, D, n = 40, 2, 8, 9
    pk = rng.integers(0, 1 << 16, size=(S, Hkv, D), dtype=np.uint16)
    pv = rng.integers(0, 1 << 16, size=(S, Hkv, D), dtype=np.uint16)
    k = rng.integers(0, 1 << 16, size=(n, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(n, Hkv, D), dtype=np.uint16)
    slots = rng.permutation(S)[:n]
    nk, nv = oracle.store_kv(pk, pv, k, v, slots)
    for s in range(S):
        hit = np.nonzero(slots == s)[0]
        if hit.size:
            assert np.array_equal(nk[s], k[hit[0]]) and np.array_equal(nv[s], v[hit[0]])
        else:
            assert np.array_equal(nk[s], pk[s]) and np.array_equal(nv[s], pv[s])
    # the contiguous-range form equals the indexed form on a range of slots
    a, b = oracle.store_kv_range(pk, pv, k, v, 17)
    c, d = oracle.store_kv(pk, pv, k, v, np.arange(17, 17 + n))
    assert np.array_equal(a, c) and np.array_equal(b, d)
    # bit patterns (NaN payloads included) are copied unchanged
    k[0, 0, 0] = 0x7FC1
    nk, _ = oracle.store_kv(pk, pv, k, v, slots)
    assert nk[slots[0], 0, 0] == 0x7FC1


# ------------------------------------------------------------ printed numbers

def test_printed_scale_and_byte_figures():
    g = json.load(open(GOLDEN))
    sc = g["softmax_scale_head_dim_128"]
    assert round(OA.default_scale(128), sc["decimals"]) == sc["value"]
    for key in ("kv_bytes_per_token_qwen3_0_6b", "kv_bytes_per_token_llama_3_1_8b"):
        m = g[key]["model"]
        assert WM.kv_bytes_per_token(m["kv_heads"], m["head_dim"], m["layers"], m["elem_bytes"]) == g[key]["value"]
    d = g["decode_kv_read_32768_tokens_gb"]
    m = g["kv_bytes_per_token_qwen3_0_6b"]["model"]
    per_tok = WM.kv_bytes_per_token(m["kv_heads"], m["head_dim"], m["layers"])
    assert round(per_tok * d["tokens"] / 1e9, d["decimals"]) == d["value"]


def test_extend_pair_count_by_enumeration():
    P, E = [0, 5, 130], [3, 1, 77]
    pairs = 0
    for p, e in zip(P, E):
        for i in range(e):
            pairs += sum(1 for j in range(p + e) if j <= p + i)
    assert WM.extend_pairs(P, E) == pairs
    assert WM.extend_flops(P, E, 2, 8) == 4 * 8 * 2 * pairs


# ------------------------------------------------------------ planted slips

MUTANTS = {
    "gqa map h % Hkv": ("_kv_head_of", lambda h, hq, hk: h % hk),
    "top-left causal alignment": ("_visible_keys", lambda p, i: i + 1),
    "query misses its own key": ("_visible_keys", lambda p, i: max(1, p + i)),
    "scale dropped": ("default_scale", lambda d: 1.0),
    "prefix K rows misaligned with V rows": ("request_kv", None),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_slips(name, monkeypatch):
    attr, fn = MUTANTS[name]
    if attr == "request_kv":
        orig = OA.request_kv

        def fn(pk, pv, rtt, row, n):
            K, V = orig(pk, pv, rtt, row, n)
            return (np.concatenate([K[1:], K[:1]]) if n > 1 else K), V
    shape = dict(Hq=4, Hkv=2, D=16, prefix_lens=[0, 5, 17], extend_lens=[4, 3, 9])
    w = extend_case(21, **shape)
    ref = _sdpa_extend(w)
    monkeypatch.setattr(OA, attr, fn)
    e = w.extend
    pk, pv = w.dense_pools(with_extend=False)
    got = OA.extend_attention(e.q, e.k_new, e.v_new, pk, pv, w.req_to_token, e.req_pool_idx,
                              e.prefix_lens, e.extend_lens, 2, None if attr == "default_scale" else w.dims.sm_scale)
    assert np.max(np.abs(got - ref)) > 1e-3, f"planted slip '{name}' not caught"
