"""Pins of the FP8 (e4m3) KV oracle against things other than itself.

  * library routine: torch's float8_e4m3fn dtype decodes every code and
    rounds float32 values to nearest (ties to even) -- the oracle's encoder
    and decoder must agree with it wherever the value is in range (|x| <= 464,
    the rounding boundary above 448; torch overflows to NaN beyond it, where
    the reading here saturates to 448 like the GPU's satfinite conversion);
  * closed forms: ties, the smallest subnormal, saturation;
  * invariant: decode over an e4m3 pool equals the (pinned) bf16 decode over
    the same values held in bf16, which holds every e4m3 value exactly
    ("Inside SGLang", Step 6: --kv-cache-dtype fp8_e4m3 halves the bytes of
    each token; K and V carry one scale each);
  * the same invariant for extend (against the pinned bf16 extend, whose
    suffix keys are the rows stored at the suffix slots) and for cascade
    decode (against the pinned bf16 cascade and the FP8 decode);
  * cross-function: the last suffix row of an FP8 extend equals an FP8
    decode of the same query over the same row.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as F
from radixattention_prefix_shared_gb300 import workloads as W

from _cases import decode_case, extend_case


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def _torch_encode(x_f32):
    return torch.from_numpy(np.asarray(x_f32, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_every_code_decodes_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    a, b = F.e4m3_decode(codes), _torch_decode(codes)
    assert np.array_equal(np.isnan(a), np.isnan(b)) and np.isnan(a).sum() == 2
    assert np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])
    assert F.e4m3_decode([0x7E])[0] == 448.0 and F.e4m3_decode([0x01])[0] == 2.0 ** -9


@pytest.mark.parametrize("seed", [0, 1])
def test_encoding_rounds_like_torch(seed):
    rng = np.random.default_rng(seed)
    # magnitudes across the whole range, subnormals included, both signs
    mag = np.exp2(rng.uniform(-12, np.log2(464), size=200000))
    x = (mag * rng.choice([-1.0, 1.0], size=mag.size)).astype(np.float32)
    # exact ties: midpoints between neighbouring finite codes
    vals = F.e4m3_decode(np.arange(0x7E, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, np.float32([0.0, -0.0, 464.0, -464.0])])
    assert np.array_equal(F.e4m3_encode(x), _torch_encode(x))


def test_ties_subnormals_and_saturation_closed_forms():
    enc = lambda v: int(F.e4m3_encode(np.float32([v]))[0])  # noqa: E731
    assert enc(1.0) == 0x38
    assert enc(1.0625) == 0x38 and enc(1.1875) == 0x3A      # ties to the even mantissa
    assert enc(2.0 ** -10) == 0x00 and enc(3 * 2.0 ** -10) == 0x02
    assert enc(2.0 ** -6) == 0x08                            # smallest normal
    assert enc(460.0) == 0x7E and enc(1e6) == 0x7E and enc(-1e6) == 0xFE
    assert all(int(F.e4m3_encode(F.e4m3_decode([c]).astype(np.float32))[0]) == c
               for c in range(256) if (c & 0x7F) != 0x7F)


def test_quantize_is_the_float32_quotient_rounded():
    rng = np.random.default_rng(3)
    bits = W.f32_to_bf16_bits(rng.standard_normal(4096).astype(np.float32) * 3)
    for s in (1.0, 1.0 / 64, 0.0173):
        x = torch.from_numpy(oracle.bf16_bits_to_f64(bits).astype(np.float32))
        qt = x / torch.tensor(s, dtype=torch.float32)
        want = qt.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = F.quantize(bits, s)
        inr = qt.abs().numpy() <= 464.0
        assert np.array_equal(got[inr], want[inr])
        # beyond the range torch gives NaN; the reading here saturates to +-448
        assert np.all(got[~inr] == np.where(qt.numpy()[~inr] < 0, 0xFE, 0x7E))
        assert s == 1.0 or (~inr).any()


def test_store_fp8_is_an_index_assignment():
    rng = np.random.default_rng(4)
    S, Hkv, D, n = 30, 2, 8, 7
    pk = rng.integers(0, 256, size=(S, Hkv, D), dtype=np.uint8)
    pv = pk.copy()
    k = W.f32_to_bf16_bits(rng.standard_normal((n, Hkv, D)).astype(np.float32))
    v = W.f32_to_bf16_bits(rng.standard_normal((n, Hkv, D)).astype(np.float32))
    slots = rng.permutation(S)[:n]
    nk, nv = F.store_kv_fp8(pk, pv, k, v, slots, 0.5, 0.25)
    for s in range(S):
        hit = np.nonzero(slots == s)[0]
        if hit.size:
            assert np.array_equal(nk[s], F.quantize(k[hit[0]], 0.5))
            assert np.array_equal(nv[s], F.quantize(v[hit[0]], 0.25))
        else:
            assert np.array_equal(nk[s], pk[s]) and np.array_equal(nv[s], pv[s])


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.25, 2.0)])
def test_fp8_decode_equals_bf16_decode_on_the_same_values(k_scale, v_scale):
    w = decode_case(61, Hq=4, Hkv=2, D=16, seq_lens=[1, 7, 40])
    b = w.decode[0]
    pk, pv = w.dense_pools(decode_steps=1)
    pk[pk == W.BF16_NAN] = 0      # unused (poisoned) slots: any finite value
    pv[pv == W.BF16_NAN] = 0
    qk, qv = F.quantize(pk, k_scale), F.quantize(pv, v_scale)
    # the dequantised values held exactly in bf16 (power-of-two scales keep them exact)
    bk = W.f32_to_bf16_bits((F.e4m3_decode(qk) * k_scale).astype(np.float32))
    bv = W.f32_to_bf16_bits((F.e4m3_decode(qv) * v_scale).astype(np.float32))
    assert np.array_equal(oracle.bf16_bits_to_f64(bk), F.e4m3_decode(qk) * k_scale)
    got = F.decode_attention_fp8(b.q, qk, qv, k_scale, v_scale, w.req_to_token, b.req_pool_idx, b.seq_lens,
                                 2, w.dims.sm_scale)
    want = oracle.decode_attention(b.q, bk, bv, w.req_to_token, b.req_pool_idx, b.seq_lens, 2, w.dims.sm_scale)
    assert np.max(np.abs(got - want)) < 1e-12


@pytest.mark.parametrize("slip", ["ties away from zero", "truncation"])
def test_pins_catch_planted_encoder_slips(slip, monkeypatch):
    rng = np.random.default_rng(5)
    x = (np.exp2(rng.uniform(-10, 8, size=20000)) * rng.choice([-1, 1], size=20000)).astype(np.float32)
    x = np.concatenate([x, np.float32([1.0625, 3 * 2.0 ** -10])])
    want = _torch_encode(x)
    assert np.array_equal(F.e4m3_encode(x), want)
    bad = (lambda v: np.floor(v + 0.5)) if slip == "ties away from zero" else np.floor
    monkeypatch.setattr(F, "_round_half_even", bad)
    assert not np.array_equal(F.e4m3_encode(x), want), f"planted slip '{slip}' not caught"


def _exact_pools(w, decode_steps, k_scale, v_scale):
    """e4m3 pools of a small workload and the same values held exactly in bf16
    (power-of-two scales keep code * scale exact)."""
    pk, pv = w.dense_pools(decode_steps=decode_steps)
    pk[pk == W.BF16_NAN] = 0
    pv[pv == W.BF16_NAN] = 0
    qk, qv = F.quantize(pk, k_scale), F.quantize(pv, v_scale)
    bk = W.f32_to_bf16_bits((F.e4m3_decode(qk) * k_scale).astype(np.float32))
    bv = W.f32_to_bf16_bits((F.e4m3_decode(qv) * v_scale).astype(np.float32))
    if np.log2(k_scale) % 1 == 0 and np.log2(v_scale) % 1 == 0:
        assert np.array_equal(oracle.bf16_bits_to_f64(bv), F.e4m3_decode(qv) * v_scale)
    return qk, qv, bk, bv


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.25, 2.0)])
def test_fp8_extend_equals_bf16_extend_on_the_same_values(k_scale, v_scale):
    w = extend_case(62, Hq=4, Hkv=2, D=16, prefix_lens=[0, 5, 33, 17], extend_lens=[3, 1, 20, 9],
                    shares=((2, 3, 11),))
    e = w.extend
    qk, qv, bk, bv = _exact_pools(w, 0, k_scale, v_scale)
    got = F.extend_attention_fp8(e.q, qk, qv, k_scale, v_scale, w.req_to_token, e.req_pool_idx,
                                 e.prefix_lens, e.extend_lens, 2, w.dims.sm_scale)
    # the bf16 extend takes the suffix keys from k_new / v_new: here the rows
    # stored at the suffix slots
    want = oracle.extend_attention(e.q, bk[e.slots], bv[e.slots], bk, bv, w.req_to_token, e.req_pool_idx,
                                   e.prefix_lens, e.extend_lens, 2, w.dims.sm_scale)
    assert np.max(np.abs(got - want)) < 1e-12
    some = [0, 4, 23, 32]
    sub = F.extend_attention_fp8(e.q, qk, qv, k_scale, v_scale, w.req_to_token, e.req_pool_idx,
                                 e.prefix_lens, e.extend_lens, 2, w.dims.sm_scale, tokens=some)
    assert np.array_equal(sub, got[some])


def test_fp8_extend_last_row_is_an_fp8_decode():
    w = extend_case(63, Hq=6, Hkv=2, D=16, prefix_lens=[7, 0, 40], extend_lens=[5, 12, 1])
    e = w.extend
    ks, vs = 0.0173, 0.031
    qk, qv, _, _ = _exact_pools(w, 0, ks, vs)
    ext = F.extend_attention_fp8(e.q, qk, qv, ks, vs, w.req_to_token, e.req_pool_idx, e.prefix_lens,
                                 e.extend_lens, 2, w.dims.sm_scale)
    last = np.cumsum(e.extend_lens) - 1
    dec = F.decode_attention_fp8(e.q[last], qk, qv, ks, vs, w.req_to_token, e.req_pool_idx,
                                 e.prefix_lens + e.extend_lens, 2, w.dims.sm_scale)
    assert np.max(np.abs(ext[last] - dec)) < 1e-12
    # an earlier row sees fewer keys: it differs from the decode over the whole row
    assert np.max(np.abs(ext[last - 1][2] - dec[2])) > 1e-3


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.5, 0.125)])
def test_fp8_cascade_equals_bf16_cascade_and_fp8_decode(k_scale, v_scale):
    dims = W.Dims(4, 2, 16, 1 << 14, 0.25)
    w = W.random_tree_decode(seed=21, dims=dims, pool_size=1 << 14, fanouts=(2, 3), seg_len=(1, 40))
    cg = W.tree_groups(w)
    b = w.decode[0]
    qk, qv, bk, bv = _exact_pools(w, 1, k_scale, v_scale)
    args = (w.req_to_token, b.req_pool_idx, b.seq_lens, cg.group_start, cg.group_len, cg.group_depth,
            cg.member_off, cg.members, 2, dims.sm_scale)
    got = F.cascade_decode_attention_fp8(b.q, qk, qv, k_scale, v_scale, *args)
    assert np.max(np.abs(got - oracle.cascade_decode_attention(b.q, bk, bv, *args))) < 1e-12
    dec = F.decode_attention_fp8(b.q, qk, qv, k_scale, v_scale, w.req_to_token, b.req_pool_idx, b.seq_lens,
                                 2, dims.sm_scale)
    assert cg.n_groups > 0 and np.max(np.abs(got - dec)) < 1e-12


@pytest.mark.parametrize("slip", ["suffix read one position late", "V scale dropped"])
def test_pins_catch_planted_extend_slips(slip, monkeypatch):
    if slip == "V scale dropped":
        monkeypatch.setattr(F, "_dequant", lambda codes, scale: F.e4m3_decode(codes) * (scale if scale != 2.0 else 1.0))
        case = lambda: test_fp8_extend_equals_bf16_extend_on_the_same_values(0.25, 2.0)  # noqa: E731
    else:
        real = F.extend_attention_fp8

        def sloppy(q, pool_k, pool_v, ks, vs, rtt, rpi, pl, el, hkv, sc=None, tokens=None):
            # the suffix read from the row one position late
            rtt = np.array(rtt, copy=True)
            for r, p, e in zip(rpi, pl, el):
                rtt[r, p: p + e] = rtt[r, p + 1: p + e + 1]
            return real(q, pool_k, pool_v, ks, vs, rtt, rpi, pl, el, hkv, sc, tokens)
        monkeypatch.setattr(F, "extend_attention_fp8", sloppy)
        case = test_fp8_extend_last_row_is_an_fp8_decode
    with pytest.raises(AssertionError):
        case()
