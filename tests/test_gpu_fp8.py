"""FP8 (e4m3) KV pool through the C ABI against the fp64 oracle.

"Inside SGLang", Step 6 (Decide how much memory becomes KV cache): with
--kv-cache-dtype fp8_e4m3 each token's K and V take half the bytes and the
attention kernels read FP8 directly, with one scale per tensor.  The store is
an integer decision (a quantised code) and must match the oracle's encoder
bit for bit; decode over the codes is checked against the oracle's decode
over the dequantised rows.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import fp8 as F  # noqa: E402
from radixattention_prefix_shared_gb300 import binding as B  # noqa: E402
from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _cases import decode_case  # noqa: E402
from _gpu import DEV, assert_close  # noqa: E402
from test_gpu_parity import DECODE_SHAPES  # noqa: E402

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
    reqs = sorted({int(np.argmax(seq)), int(np.argmin(seq)), 3, 17, 40})
    assert_close(got[reqs], oracle_fp8(w, ks, vs, requests=reqs), "decode_llama7b fp8")
