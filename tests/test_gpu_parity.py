"""GPU path vs the fp64 oracle, through the C ABI.

Bar: store_kv and every gather bit-exact; attention outputs within max-abs
2e-2 and mean-abs 2e-3 of the oracle (bf16 storage, fp32 accumulation).
Unused pool slots hold NaN and req_to_token entries past each length point at
such slots, so a read of any wrong slot shows up as NaN in the output.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from oracle.attention import bf16_bits_to_f64  # noqa: E402
from radixattention_prefix_shared_gb300 import binding as B  # noqa: E402
from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _cases import decode_case, extend_case  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

from _gpu import DEV, MAX_ABS, MEAN_ABS, Run, assert_close, oracle_decode, oracle_extend  # noqa: E402


# ------------------------------------------------------------------ store_kv

@pytest.mark.parametrize("Hkv,D,n", [(2, 64, 57), (8, 128, 1000), (32, 128, 64), (1, 64, 1)])
def test_store_kv_bit_exact(Hkv, D, n):
    rng = np.random.default_rng(n)
    S = 4 * n + 16
    pk = rng.integers(0, 1 << 16, size=(S, Hkv, D), dtype=np.uint16)   # any bits, NaNs included
    pv = rng.integers(0, 1 << 16, size=(S, Hkv, D), dtype=np.uint16)
    k = rng.integers(0, 1 << 16, size=(n, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(n, Hkv, D), dtype=np.uint16)
    slots = rng.permutation(S)[:n].astype(np.int32)
    want_k, want_v = oracle.store_kv(pk, pv, k, v, slots)
    tk, tv = W.bf16_tensor(pk, DEV), W.bf16_tensor(pv, DEV)
    B.sgl_store_kv(W.bf16_tensor(k, DEV), W.bf16_tensor(v, DEV), W.int_tensor(slots, DEV), tk, tv)
    torch.cuda.synchronize()
    assert np.array_equal(W.bf16_bits(tk), want_k)
    assert np.array_equal(W.bf16_bits(tv), want_v)


# ------------------------------------------------------------------ tiny workload

def test_tiny_workload_extend_then_decode():
    w = W.tiny()
    run = Run(w)
    got = run.extend()
    assert_close(got, oracle_extend(w), "tiny extend")
    # the suffix K/V landed in the pool bit-exactly
    pk, pv = w.dense_pools(with_extend=True)
    assert np.array_equal(W.bf16_bits(run.t["pool_k"]), pk)
    assert np.array_equal(W.bf16_bits(run.t["pool_v"]), pv)
    got = run.decode(0)
    assert_close(got, oracle_decode(w, 0), "tiny decode")


# ------------------------------------------------------------------ extend shapes

EXTEND_SHAPES = [
    # (Hq, Hkv, D, prefix_lens, extend_lens)
    (2, 2, 64, [0, 16, 33, 64], [8, 1, 31, 17]),
    (4, 4, 128, [0, 127, 128, 129], [1, 128, 129, 300]),
    (8, 2, 128, [300, 5, 0], [64, 65, 200]),
    (32, 8, 128, [250], [130]),
    (16, 8, 128, [1, 513], [257, 33]),
    (16, 2, 64, [40, 0, 700], [9, 100, 31]),
    (8, 1, 128, [129], [40]),
    (6, 2, 128, [70, 3], [50, 90]),          # g = 3: 42 tokens per tile, 2 padding rows
    (16, 1, 128, [100, 0], [40, 17]),        # g = 16: 8 tokens per tile
    (32, 1, 64, [64, 7], [33, 20]),          # g = 32: 4 tokens per tile
]


@pytest.mark.parametrize("shape", EXTEND_SHAPES, ids=lambda s: f"{s[0]}q{s[1]}kv{s[2]}d")
def test_extend_matches_oracle(shape):
    Hq, Hkv, D, P, E = shape
    w = extend_case(sum(P) + sum(E), Hq=Hq, Hkv=Hkv, D=D, prefix_lens=P, extend_lens=E,
                    shares=[(0, len(P) - 1, min(P[0], P[-1]))] if len(P) > 1 else ())
    got = Run(w).extend()
    assert_close(got, oracle_extend(w), f"extend {shape}")


def test_extend_with_empty_requests_and_scale():
    w = extend_case(77, Hq=4, Hkv=2, D=128, prefix_lens=[10, 0, 50], extend_lens=[0, 20, 5], scale=0.05)
    got = Run(w).extend()
    assert_close(got, oracle_extend(w), "empty request rows")


# ------------------------------------------------------------------ decode shapes

DECODE_SHAPES = [
    (2, 2, 64, [1, 2, 31, 32, 33, 100]),
    (32, 32, 128, [512, 513, 1025, 1]),
    (32, 8, 128, [2049, 700, 3000]),
    (16, 8, 128, [1024, 4097, 5]),
    (8, 1, 128, [600, 1]),
    (16, 2, 64, [530, 64]),
    (4, 1, 64, [1500]),
    (4, 2, 64, [700, 3, 1025]),
    # group sizes without a CUDA-core build: tensor-core rows (3, 5, 6, 7; 16 uses rows 8..15)
    (6, 2, 128, [700, 1, 33]),
    (10, 2, 128, [1500, 17]),
    (12, 2, 64, [300, 2049]),
    (28, 4, 128, [1025, 64]),
    (32, 2, 128, [900, 1, 4100]),
    (16, 1, 64, [513]),
    # group sizes 9..15: rows 8..15 partly filled
    (18, 2, 128, [700, 33]),
    (24, 2, 64, [1500, 1]),
    (30, 2, 128, [513, 2049]),
    (13, 1, 128, [800]),
    # groups above 16: KV-head copies of <= 16 query heads
    (32, 1, 128, [900, 33]),                 # 2 x 16
    (48, 2, 128, [700, 2]),                  # 2 x 12 per KV head
    (34, 2, 64, [500, 1]),                   # 17 = 17 x 1 (prime)
    # KV heads in groups of 4 (e4m3 pools gather a slot's 4 rows as one span;
    # items of 512 keys): one, three and two groups, every span group size
    (8, 4, 64, [1, 511, 512, 513, 1300]),
    (24, 12, 128, [2049, 64, 1]),
    (48, 12, 64, [777, 3]),
    (8, 8, 128, [1024, 255]),
]


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: f"{s[0]}q{s[1]}kv{s[2]}d")
def test_decode_matches_oracle(shape):
    Hq, Hkv, D, S = shape
    w = decode_case(sum(S), Hq=Hq, Hkv=Hkv, D=D, seq_lens=S)
    got = Run(w).decode()
    assert_close(got, oracle_decode(w), f"decode {shape}")


def test_decode_long_context():
    """128 K-token and 70 K-token rows: 128 and 69 splits of at most 1,024 keys
    merged by the combine; a 3-key row beside them."""
    w = decode_case(77, Hq=8, Hkv=2, D=128, seq_lens=[131072, 70001, 3])
    got = Run(w).decode()
    assert_close(got, oracle_decode(w, pool=w.pool_view(decode_steps=1)), "decode 128K context")


def test_extend_long_prefix_sampled():
    """A 64 K-token cached prefix (512 key blocks before the suffix), sampled rows."""
    w = extend_case(78, Hq=8, Hkv=2, D=128, prefix_lens=[65536, 1000], extend_lens=[300, 129])
    got = Run(w).extend()
    toks = [0, 1, 150, 299, 300, 428]
    assert_close(got[toks], oracle_extend(w, tokens=toks, pool=w.pool_view(with_extend=False)),
                 "extend 64K prefix")


def test_single_key_outputs_are_bit_exact():
    w = decode_case(5, Hq=8, Hkv=2, D=128, seq_lens=[1, 1, 1])
    got = Run(w).decode()
    want = np.repeat(w.decode[0].v_new, 4, axis=1)          # each query head reads its KV head
    assert np.array_equal(got, want)
    w2 = extend_case(6, Hq=4, Hkv=4, D=64, prefix_lens=[0, 0], extend_lens=[3, 1])
    got = Run(w2).extend()
    assert np.array_equal(got[0], w2.extend.v_new[0])
    assert np.array_equal(got[3], w2.extend.v_new[3])


# ------------------------------------------------------------------ invariants

def _relabelled(w, seed):
    """Same logical workload, every slot moved by a permutation of the pool."""
    import copy
    w2 = copy.deepcopy(w)
    perm = np.random.default_rng(seed).permutation(w.dims.pool_size).astype(np.int32)
    w2.req_to_token = perm[w.req_to_token]
    w2.live_slots = perm[w.live_slots]
    if w.extend is not None:
        w2.extend.slots = perm[w.extend.slots]
    for b in w2.decode:
        b.slots = perm[b.slots]
    return w2


def test_slot_permutation_gives_bit_identical_outputs():
    w = extend_case(31, Hq=16, Hkv=8, D=128, prefix_lens=[300, 129, 0], extend_lens=[70, 129, 5],
                    decode_after=True)
    r1, r2 = Run(w), Run(_relabelled(w, 9))
    assert np.array_equal(r1.extend(), r2.extend())
    assert np.array_equal(r1.decode(), r2.decode())


def test_shared_prefix_equals_private_copies_bit_identical():
    w = extend_case(32, Hq=8, Hkv=2, D=128, prefix_lens=[400, 400, 200], extend_lens=[33, 60, 1],
                    shares=[(0, 1, 400), (0, 2, 200)], decode_after=True)
    r_shared = Run(w)
    e_shared, d_shared = r_shared.extend(), r_shared.decode()
    # private copies: give requests 1 and 2 their own slots holding the same rows
    import copy
    w2 = copy.deepcopy(w)
    used = np.concatenate([w.live_slots, w.extend.slots, w.decode[0].slots])
    free = np.setdiff1d(np.arange(w.dims.pool_size), used)
    rows = w.extend.req_pool_idx
    extra_slots, src_slots = [], []
    k = 0
    for r, n in ((1, 400), (2, 200)):
        old = w2.req_to_token[rows[r], :n].copy()
        new = free[k:k + n]
        k += n
        w2.req_to_token[rows[r], :n] = new
        extra_slots.append(new)
        src_slots.append(old)
    r_priv = Run(w2)
    pk, pv = r_priv.t["pool_k"], r_priv.t["pool_v"]
    for new, old in zip(extra_slots, src_slots):
        ni, oi = torch.from_numpy(new.astype(np.int64)).to(DEV), torch.from_numpy(old.astype(np.int64)).to(DEV)
        pk[ni] = pk[oi]
        pv[ni] = pv[oi]
    torch.cuda.synchronize()
    assert np.array_equal(e_shared, r_priv.extend())
    assert np.array_equal(d_shared, r_priv.decode())


def test_decode_equals_extend_with_one_token():
    w = decode_case(41, Hq=16, Hkv=8, D=128, seq_lens=[1, 300, 1030])
    run = Run(w)
    d = bf16_bits_to_f64(run.decode())
    b, t = w.decode[0], run.t["decode"][0]
    x = B.sgl_extend_attention(t["q"], t["k_new"], t["v_new"], run.t["pool_k"], run.t["pool_v"],
                               run.t["req_to_token"], t["req_pool_idx"], t["seq_lens"] - 1,
                               torch.ones_like(t["seq_lens"]), max_extend=1,
                               max_prefix=int(b.seq_lens.max()) - 1, workspace=run.ws_ext)
    torch.cuda.synchronize()
    x = bf16_bits_to_f64(W.bf16_bits(x))
    assert np.abs(d - x).max() <= 2 * MAX_ABS / 4


# ------------------------------------------------------------------ checked mode

def test_checked_mode_reports_bad_indices():
    w = extend_case(51, Hq=4, Hkv=2, D=64, prefix_lens=[20, 7], extend_lens=[5, 9], decode_after=True)
    t = W.to_device(w, DEV)
    e, te = w.extend, t["extend"]
    err = torch.zeros(4, dtype=torch.int32, device=DEV)
    S = w.dims.pool_size
    kw = dict(total_extend=e.total_extend, max_extend=9, max_prefix=20, pool_size=S, d_error=err)
    B.sgl_check_extend_indices(t["req_to_token"], te["req_pool_idx"], te["prefix_lens"], te["extend_lens"], **kw)
    B.sgl_check_store_kv_indices(te["slots"], S, err)
    b, tb = w.decode[0], t["decode"][0]
    B.sgl_check_decode_indices(t["req_to_token"], tb["req_pool_idx"], tb["seq_lens"],
                               max_seq_len=int(b.seq_lens.max()), pool_size=S, d_error=err)
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0, 0, 0]
    # an out-of-range slot inside a prefix
    rtt = t["req_to_token"].clone()
    rtt[int(e.req_pool_idx[0]), 3] = S + 5
    B.sgl_check_extend_indices(rtt, te["req_pool_idx"], te["prefix_lens"], te["extend_lens"], **kw)
    torch.cuda.synchronize()
    assert err.tolist() == [1, 0, 3, S + 5]
    # duplicate slots in one store
    err.zero_()
    dup = te["slots"].clone()
    dup[4] = dup[1]
    B.sgl_check_store_kv_indices(dup, S, err)
    torch.cuda.synchronize()
    assert err[0].item() == 6 and err[3].item() == int(dup[1].item())
    # a request row outside req_to_token, and a wrong total
    err.zero_()
    bad = te["req_pool_idx"].clone()
    bad[1] = w.req_to_token.shape[0]
    B.sgl_check_extend_indices(t["req_to_token"], bad, te["prefix_lens"], te["extend_lens"], **kw)
    torch.cuda.synchronize()
    assert err[0].item() == 2 and err[1].item() == 1
    err.zero_()
    kw["total_extend"] = e.total_extend + 1
    B.sgl_check_extend_indices(t["req_to_token"], te["req_pool_idx"], te["prefix_lens"], te["extend_lens"], **kw)
    torch.cuda.synchronize()
    assert err[0].item() == 5
    # decode: seq_len 0
    err.zero_()
    sl = tb["seq_lens"].clone()
    sl[0] = 0
    B.sgl_check_decode_indices(t["req_to_token"], tb["req_pool_idx"], sl, max_seq_len=100, pool_size=S, d_error=err)
    torch.cuda.synchronize()
    assert err[0].item() == 3


def test_zero_sized_calls_are_noops():
    z = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device=DEV)
    pool = torch.zeros(16, 2, 64, dtype=torch.bfloat16, device=DEV)
    B.sgl_store_kv(z, z, torch.zeros(0, dtype=torch.int32, device=DEV), pool, pool)
    i0 = torch.zeros(0, dtype=torch.int32, device=DEV)
    rtt = torch.zeros(1, 4, dtype=torch.int32, device=DEV)
    B.sgl_decode_attention(torch.zeros(0, 2, 64, dtype=torch.bfloat16, device=DEV), pool, pool, rtt, i0, i0,
                           max_seq_len=1)
    B.sgl_extend_attention(z, z, z, pool, pool, rtt, i0, i0, i0, max_extend=0)
    torch.cuda.synchronize()


def test_repeated_launches_are_bit_identical():
    """The kernels are deterministic: repeated launches over the same inputs
    (many K/V ring reuses per CTA) give identical bits, and they match the
    oracle -- any read of a shared-memory stage before its copies landed would
    show up as a run-to-run difference."""
    w = extend_case(61, Hq=16, Hkv=8, D=128, prefix_lens=[3000, 1700, 40], extend_lens=[300, 129, 700],
                    decode_after=True)
    run = Run(w)
    first = run.extend()
    assert_close(first, oracle_extend(w), "repeated extend")
    e, te = w.extend, run.t["extend"]
    for _ in range(12):
        out = B.sgl_extend_attention(te["q"], te["k_new"], te["v_new"], run.t["pool_k"], run.t["pool_v"],
                                     run.t["req_to_token"], te["req_pool_idx"], te["prefix_lens"],
                                     te["extend_lens"], max_extend=int(e.extend_lens.max()),
                                     max_prefix=int(e.prefix_lens.max()), workspace=run.ws_ext)
        torch.cuda.synchronize()
        assert np.array_equal(W.bf16_bits(out), first)
    d0 = run.decode()
    b, tb = w.decode[0], run.t["decode"][0]
    for _ in range(4):
        out = B.sgl_decode_attention(tb["q"], run.t["pool_k"], run.t["pool_v"], run.t["req_to_token"],
                                     tb["req_pool_idx"], tb["seq_lens"], max_seq_len=int(b.seq_lens.max()))
        torch.cuda.synchronize()
        assert np.array_equal(W.bf16_bits(out), d0)
