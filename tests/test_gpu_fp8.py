"""FP8 (e4m3) KV pool through the C ABI against the fp64 oracle.

"Inside SGLang", Step 6 (Decide how much memory becomes KV cache): with
--kv-cache-dtype fp8_e4m3 each token's K and V take half the bytes and the
attention kernels read FP8 directly, with one scale per tensor.  The store is
an integer decision (a quantised code) and must match the oracle's encoder
bit for bit; decode, extend (suffix read back from the pool) and cascade
decode over the codes are checked against the oracle over the dequantised
rows.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import fp8 as F  # noqa: E402
from radixattention_prefix_shared_gb300 import binding as B  # noqa: E402
from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _cases import decode_case, extend_case  # noqa: E402
from _gpu import DEV, REL_MAX_OF_RMS, assert_close  # noqa: E402
from _sampling import extreme_prefix_requests, sample_requests, tile_edge_tokens  # noqa: E402
from test_gpu_cascade import TREES, groups_on_device  # noqa: E402
from test_gpu_parity import DECODE_SHAPES, EXTEND_SHAPES  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def fp8_pools(w, steps, k_scale, v_scale, rows_per_call=1 << 16):
    """Device e4m3 pools holding every cached row and the first `steps`
    decode batches' new rows, written by sgl_store_kv_fp8."""
    d = w.dims
    pk = torch.zeros((d.pool_size, d.num_kv_heads, d.head_dim), dtype=torch.uint8, device=DEV)
    pv = torch.zeros_like(pk)
    n = w.live_slots.size
    for a in range(0, n, rows_per_call):
        b = min(n, a + rows_per_call)
        B.sgl_store_kv_fp8(W.bf16_tensor(w.live_k.rows(a, b), DEV), W.bf16_tensor(w.live_v.rows(a, b), DEV),
                           W.int_tensor(w.live_slots[a:b], DEV), pk, pv, k_scale, v_scale)
    for s in range(steps):
        bt = w.decode[s]
        B.sgl_store_kv_fp8(W.bf16_tensor(bt.k_new, DEV), W.bf16_tensor(bt.v_new, DEV),
                           W.int_tensor(bt.slots, DEV), pk, pv, k_scale, v_scale)
    return pk, pv


def decode_fp8(w, pk, pv, k_scale, v_scale, step=0):
    b = w.decode[step]
    out = B.sgl_decode_attention_fp8(W.bf16_tensor(b.q, DEV), pk, pv, k_scale, v_scale,
                                     W.int_tensor(w.req_to_token, DEV), W.int_tensor(b.req_pool_idx, DEV),
                                     W.int_tensor(b.seq_lens, DEV), max_seq_len=int(b.seq_lens.max()),
                                     sm_scale=w.dims.sm_scale)
    torch.cuda.synchronize()
    return W.bf16_bits(out)


def oracle_fp8(w, k_scale, v_scale, step=0, requests=None):
    """The oracle's decode over rows quantised by the oracle's own encoder."""
    b = w.decode[step]
    view = w.pool_view(decode_steps=step + 1)
    if requests is None:
        requests = np.arange(b.seq_lens.size)
    slots = np.unique(np.concatenate([w.req_to_token[b.req_pool_idx[r], : b.seq_lens[r]] for r in requests]))
    S = w.dims.pool_size
    pk = np.zeros((S, w.dims.num_kv_heads, w.dims.head_dim), np.uint8)
    pv = np.zeros_like(pk)
    pk[slots] = F.quantize(view.k[slots], k_scale)
    pv[slots] = F.quantize(view.v[slots], v_scale)
    return F.decode_attention_fp8(b.q, pk, pv, k_scale, v_scale, w.req_to_token, b.req_pool_idx, b.seq_lens,
                                  w.dims.num_kv_heads, w.dims.sm_scale, requests=requests)


@pytest.mark.parametrize("Hkv,D,scale", [(2, 64, 1.0), (8, 128, 1.0 / 64), (32, 128, 0.0173)])
def test_store_kv_fp8_bit_exact(Hkv, D, scale):
    rng = np.random.default_rng(Hkv + D)
    n, S = 777, 4096
    # values across the range: big ones saturate, tiny ones are subnormal codes
    mag = np.exp2(rng.uniform(-16, 10, size=(n, Hkv, D))) * rng.choice([-1.0, 1.0], size=(n, Hkv, D))
    k = W.f32_to_bf16_bits(mag.astype(np.float32))
    v = W.f32_to_bf16_bits((rng.standard_normal((n, Hkv, D)) * 3).astype(np.float32))
    slots = rng.permutation(S)[:n].astype(np.int32)
    pk = torch.zeros((S, Hkv, D), dtype=torch.uint8, device=DEV)
    pv = torch.zeros_like(pk)
    B.sgl_store_kv_fp8(W.bf16_tensor(k, DEV), W.bf16_tensor(v, DEV), W.int_tensor(slots, DEV), pk, pv,
                       scale, 2 * scale)
    torch.cuda.synchronize()
    gk, gv = pk.cpu().numpy(), pv.cpu().numpy()
    assert np.array_equal(gk[slots], F.quantize(k, scale))
    assert np.array_equal(gv[slots], F.quantize(v, 2 * scale))
    untouched = np.setdiff1d(np.arange(S), slots)
    assert not gk[untouched].any() and not gv[untouched].any()


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: f"{s[0]}q{s[1]}kv{s[2]}d")
def test_decode_fp8_matches_oracle(shape):
    Hq, Hkv, D, S = shape
    w = decode_case(sum(S) + 7, Hq=Hq, Hkv=Hkv, D=D, seq_lens=S)
    ks, vs = 1.0 / 32, 0.0173
    pk, pv = fp8_pools(w, 1, ks, vs)
    assert_close(decode_fp8(w, pk, pv, ks, vs), oracle_fp8(w, ks, vs), f"decode fp8 {shape}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (8, 2)])
def test_decode_fp8_wide_scores(hq, hkv):
    """Scores spread over tens of natural-log units (unit-variance q and k, a
    large softmax scale): with one, two or four query heads per KV head the K
    codes meet the query as three e4m3 terms in the tensor core, whose
    rounding the large scores would magnify, and P meets the V codes as two
    e4m3 terms, most of them tiny -- the output must still match."""
    w = decode_case(61 + hq, Hq=hq, Hkv=hkv, D=128, seq_lens=[900, 333, 2000, 1], scale=0.8)
    ks, vs = 1.0 / 32, 1.0 / 32
    pk, pv = fp8_pools(w, 1, ks, vs)
    assert_close(decode_fp8(w, pk, pv, ks, vs), oracle_fp8(w, ks, vs), f"decode fp8 wide scores {hq}/{hkv}")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8)])
def test_decode_fp8_query_range(hq, hkv):
    """Queries whose dims span six orders of magnitude (a few dims 300x,
    half of them 1/1000x): each head's query is scaled by a power of two into
    e4m3's range before its three terms are taken."""
    w = decode_case(71 + hq, Hq=hq, Hkv=hkv, D=128, seq_lens=[700, 64, 1500])
    b = w.decode[0]
    q = (b.q.astype(np.uint32) << 16).view(np.float32).copy()
    q[..., :4] *= 300.0
    q[..., 64:] *= 1e-3
    q[1] *= 1e-20                    # one request's queries far below e4m3's range
    b.q[...] = W.f32_to_bf16_bits(q)
    ks, vs = 1.0 / 32, 1.0 / 32
    pk, pv = fp8_pools(w, 1, ks, vs)
    assert_close(decode_fp8(w, pk, pv, ks, vs), oracle_fp8(w, ks, vs), f"decode fp8 query range {hq}/{hkv}")


def test_decode_fp8_single_key_bit_exact():
    w = decode_case(9, Hq=8, Hkv=2, D=128, seq_lens=[1, 1, 1])
    ks, vs = 1.0 / 16, 1.0 / 8         # powers of two: code * scale is exact in bf16
    pk, pv = fp8_pools(w, 1, ks, vs)
    got = decode_fp8(w, pk, pv, ks, vs)
    v = F.e4m3_decode(F.quantize(w.decode[0].v_new, vs)) * vs
    want = W.f32_to_bf16_bits(np.repeat(v, 4, axis=1).astype(np.float32))
    assert np.array_equal(got, want)


def test_decode_fp8_full_size_sampled():
    """The Llama-7B-like decode workload at full size over an e4m3 pool."""
    w = W.decode_llama7b()
    ks, vs = 1.0 / 64, 1.0 / 64
    pk, pv = fp8_pools(w, 1, ks, vs)
    got = decode_fp8(w, pk, pv, ks, vs)
    x = (got.astype(np.uint32) << 16).view(np.float32)
    assert np.isfinite(x).all()
    seq = w.decode[0].seq_lens
    reqs = sample_requests(seq, 16, 41)
    assert_close(got[reqs], oracle_fp8(w, ks, vs, requests=reqs), "decode_llama7b fp8", rel_max=REL_MAX_OF_RMS)


# ------------------------------------------------------------------ extend

def extend_pools(w, k_scale, v_scale):
    """e4m3 pools with every cached row and the extend batch's suffix rows
    (stored with sgl_store_kv_fp8 before the attention, as a serving step does)."""
    pk, pv = fp8_pools(w, 0, k_scale, v_scale)
    e = w.extend
    B.sgl_store_kv_fp8(W.bf16_tensor(e.k_new, DEV), W.bf16_tensor(e.v_new, DEV), W.int_tensor(e.slots, DEV),
                       pk, pv, k_scale, v_scale)
    return pk, pv


def extend_fp8(w, pk, pv, k_scale, v_scale):
    e = w.extend
    ws = B.new_workspace(256, DEV)
    out = B.sgl_extend_attention_fp8(W.bf16_tensor(e.q, DEV), pk, pv, k_scale, v_scale,
                                     W.int_tensor(w.req_to_token, DEV), W.int_tensor(e.req_pool_idx, DEV),
                                     W.int_tensor(e.prefix_lens, DEV), W.int_tensor(e.extend_lens, DEV),
                                     max_extend=int(e.extend_lens.max()), max_prefix=int(e.prefix_lens.max()),
                                     workspace=ws, sm_scale=w.dims.sm_scale)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0, "extend kernel reported a timeout"
    return W.bf16_bits(out)


def oracle_extend_fp8(w, k_scale, v_scale, tokens=None):
    """The oracle's FP8 extend over the rows the listed tokens read, quantised
    by the oracle's own encoder."""
    e = w.extend
    view = w.pool_view()
    offs = np.concatenate([[0], np.cumsum(e.extend_lens)])
    T = int(offs[-1])
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    reqs = np.unique(np.searchsorted(offs, toks, side="right") - 1)
    slots = np.unique(np.concatenate([w.req_to_token[e.req_pool_idx[r], : e.prefix_lens[r] + e.extend_lens[r]]
                                      for r in reqs]))
    S = w.dims.pool_size
    pk = np.zeros((S, w.dims.num_kv_heads, w.dims.head_dim), np.uint8)
    pv = np.zeros_like(pk)
    pk[slots] = F.quantize(view.k[slots], k_scale)
    pv[slots] = F.quantize(view.v[slots], v_scale)
    return F.extend_attention_fp8(e.q, pk, pv, k_scale, v_scale, w.req_to_token, e.req_pool_idx, e.prefix_lens,
                                  e.extend_lens, w.dims.num_kv_heads, w.dims.sm_scale, tokens=tokens)


@pytest.mark.parametrize("shape", EXTEND_SHAPES, ids=lambda s: f"{s[0]}q{s[1]}kv{s[2]}d")
def test_extend_fp8_matches_oracle(shape):
    Hq, Hkv, D, P, E = shape
    w = extend_case(sum(P) + sum(E) + 3, Hq=Hq, Hkv=Hkv, D=D, prefix_lens=P, extend_lens=E,
                    shares=[(0, len(P) - 1, min(P[0], P[-1]))] if len(P) > 1 else ())
    ks, vs = 1.0 / 32, 0.0173
    pk, pv = extend_pools(w, ks, vs)
    assert_close(extend_fp8(w, pk, pv, ks, vs), oracle_extend_fp8(w, ks, vs), f"extend fp8 {shape}")


def test_extend_fp8_wide_scores_move_the_reference():
    """Scores spread over tens of log2 units: later blocks exceed the lazy
    reference by more than the f16 P bound (2^15), so the rescale path runs;
    empty requests and a custom scale ride along."""
    # unit-variance values with a large softmax scale: scores spread with a
    # standard deviation of ~9 (the output stays at unit scale, where the
    # absolute tolerance applies)
    w = extend_case(91, Hq=8, Hkv=2, D=128, prefix_lens=[900, 0, 333], extend_lens=[200, 0, 150], scale=0.8)
    ks, vs = 1.0 / 32, 1.0 / 32
    pk, pv = extend_pools(w, ks, vs)
    assert_close(extend_fp8(w, pk, pv, ks, vs), oracle_extend_fp8(w, ks, vs), "extend fp8 wide scores")


def test_extend_fp8_single_key_bit_exact():
    """One key per query (no prefix, first suffix token): the output is that
    key's value, code * scale, exact in bf16 for power-of-two scales."""
    w = extend_case(5, Hq=4, Hkv=1, D=64, prefix_lens=[0, 0], extend_lens=[1, 1])
    ks, vs = 1.0 / 8, 1.0 / 4
    pk, pv = extend_pools(w, ks, vs)
    got = extend_fp8(w, pk, pv, ks, vs)
    v = F.e4m3_decode(F.quantize(w.extend.v_new, vs)) * vs
    assert np.array_equal(got, W.f32_to_bf16_bits(np.repeat(v, 4, axis=1).astype(np.float32)))


def test_extend_fp8_checked_mode_covers_the_suffix():
    """A bad slot at a suffix position: only the e4m3 extend reads it, and
    only its index check reports it."""
    w = extend_case(8, Hq=4, Hkv=2, D=64, prefix_lens=[10, 20], extend_lens=[5, 7])
    e = w.extend
    rtt = w.req_to_token.copy()
    rtt[e.req_pool_idx[1], 20 + 3] = w.dims.pool_size + 5
    args = (W.int_tensor(rtt, DEV), W.int_tensor(e.req_pool_idx, DEV), W.int_tensor(e.prefix_lens, DEV),
            W.int_tensor(e.extend_lens, DEV))
    kw = dict(total_extend=int(e.extend_lens.sum()), max_extend=7, max_prefix=20, pool_size=w.dims.pool_size)
    for fp8, want in ((False, [0, 0, 0, 0]), (True, [1, 1, 23, w.dims.pool_size + 5])):
        err = torch.zeros(4, dtype=torch.int32, device=DEV)
        B.sgl_check_extend_indices(*args, d_error=err, fp8=fp8, **kw)
        torch.cuda.synchronize()
        assert err.cpu().tolist() == want, fp8


def test_shared_prompt_extend_fp8_full_sampled():
    """The shared-system-prompt extend workload at full size over an e4m3 pool."""
    w = W.shared_prompt_extend()
    ks, vs = 1.0 / 64, 1.0 / 64
    pk, pv = extend_pools(w, ks, vs)
    got = extend_fp8(w, pk, pv, ks, vs)
    x = (got.astype(np.uint32) << 16).view(np.float32)
    assert np.isfinite(x).all()
    offs = np.concatenate([[0], np.cumsum(w.extend.extend_lens)])
    rng = np.random.default_rng(12)
    toks = np.unique(np.concatenate([[0, offs[-1] - 1, offs[5], offs[6] - 1],
                                     rng.integers(0, offs[-1], size=8)]))
    assert_close(got[toks], oracle_extend_fp8(w, ks, vs, tokens=toks), "shared_prompt_extend fp8",
                 rel_max=REL_MAX_OF_RMS)


def test_chunked_prefill_mix_fp8_full_sampled():
    """The chunked-prefill mix at full size over an e4m3 pool, as the bench
    runs it: every cached row, the chunks' suffix rows and the decode tokens'
    rows stored quantised, then the extend (suffix read back from the pool)
    and the decode.  Extend: both ends of every Q tile of the requests with
    the longest and the shortest prefix; decode: 40 requests and the
    extremes."""
    w = W.chunked_prefill_mix()
    ks, vs = 1.0 / 64, 1.0 / 64
    pk, pv = fp8_pools(w, 1, ks, vs)
    e = w.extend
    B.sgl_store_kv_fp8(W.bf16_tensor(e.k_new, DEV), W.bf16_tensor(e.v_new, DEV), W.int_tensor(e.slots, DEV),
                       pk, pv, ks, vs)
    ext = extend_fp8(w, pk, pv, ks, vs)
    dec = decode_fp8(w, pk, pv, ks, vs)
    for bits, what in ((ext, "extend"), (dec, "decode")):
        x = (bits.astype(np.uint32) << 16).view(np.float32)
        assert np.isfinite(x).all(), what
    toks = tile_edge_tokens(e, extreme_prefix_requests(e), w.dims.num_q_heads // w.dims.num_kv_heads)
    assert_close(ext[toks], oracle_extend_fp8(w, ks, vs, tokens=toks), "chunked extend fp8",
                 rel_max=REL_MAX_OF_RMS)
    reqs = sample_requests(w.decode[0].seq_lens, 40, 7)
    assert_close(dec[reqs], oracle_fp8(w, ks, vs, requests=reqs), "chunked decode fp8", rel_max=REL_MAX_OF_RMS)


# ------------------------------------------------------------------ cascade

@pytest.mark.parametrize("tree", TREES, ids=lambda t: f"{t[0]}q{t[1]}kv{t[2]}d-{'x'.join(map(str, t[3]))}")
def test_cascade_fp8_matches_oracle(tree):
    Hq, Hkv, D, fan, seg, own = tree
    dims = W.Dims(Hq, Hkv, D, 1 << 17, 1.0 / np.sqrt(D))
    w = W.random_tree_decode(seed=40 + Hq + D, dims=dims, fanouts=fan, seg_len=seg, own_len=own,
                             pool_size=1 << 17)
    cg = W.tree_groups(w)
    assert cg.n_groups > 0
    ks, vs = 1.0 / 32, 0.0173
    pk, pv = fp8_pools(w, 1, ks, vs)
    b = w.decode[0]
    md = max(cg.max_depth, 1)
    out = B.sgl_cascade_decode_attention(W.bf16_tensor(b.q, DEV), pk, pv, W.int_tensor(w.req_to_token, DEV),
                                         W.int_tensor(b.req_pool_idx, DEV), W.int_tensor(b.seq_lens, DEV),
                                         *groups_on_device(cg), max_seq_len=int(b.seq_lens.max()),
                                         max_group_members=max(cg.max_members, 1), max_depth=md,
                                         sm_scale=dims.sm_scale, kv_scales=(ks, vs))
    torch.cuda.synchronize()
    got = W.bf16_bits(out)
    # the cascade oracle equals the FP8 decode oracle on shared slots (pinned on the CPU)
    assert_close(got, oracle_fp8(w, ks, vs), f"cascade fp8 {tree}")


def test_tree_of_thought_cascade_fp8_full_sampled():
    """The tree-of-thought workload's first step at full size through the
    e4m3 cascade."""
    w = W.tree_of_thought_decode()
    cg = W.tree_groups(w)
    ks, vs = 1.0 / 64, 1.0 / 64
    pk, pv = fp8_pools(w, 1, ks, vs)
    b = w.decode[0]
    out = B.sgl_cascade_decode_attention(W.bf16_tensor(b.q, DEV), pk, pv, W.int_tensor(w.req_to_token, DEV),
                                         W.int_tensor(b.req_pool_idx, DEV), W.int_tensor(b.seq_lens, DEV),
                                         *groups_on_device(cg), max_seq_len=int(b.seq_lens.max()),
                                         max_group_members=cg.max_members, max_depth=cg.max_depth,
                                         sm_scale=w.dims.sm_scale, kv_scales=(ks, vs))
    torch.cuda.synchronize()
    got = W.bf16_bits(out)
    x = (got.astype(np.uint32) << 16).view(np.float32)
    assert np.isfinite(x).all()
    reqs = sample_requests(b.seq_lens, 32, 8)
    assert_close(got[reqs], oracle_fp8(w, ks, vs, requests=reqs), "tree cascade fp8", rel_max=REL_MAX_OF_RMS)
