"""The five workloads at full size, launched as bench.py launches them.

Outputs are checked against the oracle on rows it computes one by one:
every request of the Llama-7B-like decode; at least 32 decode requests of the
other batches, always with the longest and the shortest; for extend, the
first and the last token of every 128-row Q tile of the requests with the
longest and the shortest prefix (and of three shared-prompt requests), so
every Q tile and both ends of it are read.  Besides the absolute bounds,
every sample pins its largest error to a fraction of its own output RMS.
store_kv is checked bit-exactly on sampled slots; the NaN-poisoned unused
slots make any stray read visible in every output row.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _gpu import DEV, REL_MAX_OF_RMS, Run, assert_close, oracle_decode, oracle_extend  # noqa: E402
from _sampling import extreme_prefix_requests, sample_requests, tile_edge_tokens  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _check_all_finite(bits, what):
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.isfinite(x).all(), f"{what}: non-finite values (stray read of a poisoned slot?)"


def _check_store(run, batch, n=256, seed=0):
    rng = np.random.default_rng(seed)
    idx = rng.choice(batch.slots.size, size=min(n, batch.slots.size), replace=False)
    sl = torch.from_numpy(batch.slots[idx].astype(np.int64)).to(DEV)
    assert np.array_equal(W.bf16_bits(run.t["pool_k"][sl]), batch.k_new[idx])
    assert np.array_equal(W.bf16_bits(run.t["pool_v"][sl]), batch.v_new[idx])


def test_decode_llama7b_full():
    """Every request of the batch."""
    w = W.decode_llama7b()
    run = Run(w)
    got = run.decode()
    _check_all_finite(got, "decode")
    _check_store(run, w.decode[0])
    want = oracle_decode(w, 0, pool=w.pool_view(decode_steps=1))
    assert_close(got, want, "decode_llama7b (all 64 requests)", rel_max=REL_MAX_OF_RMS)


def test_decode_llama7b_paged_full():
    """The Llama-7B-like decode with requests owning whole pages of 64 slots."""
    w = W.decode_llama7b(page_size=64)
    got = Run(w).decode()
    _check_all_finite(got, "decode paged")
    reqs = sample_requests(w.decode[0].seq_lens, 16, 3)
    want = oracle_decode(w, 0, requests=reqs, pool=w.pool_view(decode_steps=1))
    assert_close(got[reqs], want, "decode_llama7b page 64", rel_max=REL_MAX_OF_RMS)


def test_shared_prompt_extend_full():
    w = W.shared_prompt_extend()
    run = Run(w)
    got = run.extend()
    _check_all_finite(got, "extend")
    _check_store(run, w.extend)
    toks = tile_edge_tokens(w.extend, [0, 37, 63], w.dims.num_q_heads // w.dims.num_kv_heads)
    want = oracle_extend(w, tokens=toks, pool=w.pool_view(with_extend=False))
    assert_close(got[toks], want, "shared_prompt_extend (tile edges of 3 requests)", rel_max=REL_MAX_OF_RMS)


def test_tree_of_thought_decode_full():
    w = W.tree_of_thought_decode()
    run = Run(w)
    outs = [run.decode(s) for s in range(len(w.decode))]
    for s in (0, 8, len(w.decode) - 1):
        _check_all_finite(outs[s], f"decode step {s}")
        reqs = sample_requests(w.decode[s].seq_lens, 32, 10 + s)
        want = oracle_decode(w, s, requests=reqs, pool=w.pool_view(decode_steps=s + 1))
        assert_close(outs[s][reqs], want, f"tree decode step {s}", rel_max=REL_MAX_OF_RMS)
    _check_store(run, w.decode[-1])


def test_tree_of_thought_cascade_full():
    """The tree workload through cascade decode, with the shared levels read
    once per group; sampled leaves against the oracle's plain decode."""
    from test_gpu_cascade import cascade
    w = W.tree_of_thought_decode()
    run = Run(w)
    cg = W.tree_groups(w)
    assert cg.n_groups == 84 and cg.max_members == 64
    outs = [cascade(run, W.tree_groups(w, s), step=s) for s in range(len(w.decode))]
    for s in (0, 8, len(w.decode) - 1):
        _check_all_finite(outs[s], f"cascade step {s}")
        reqs = sample_requests(w.decode[s].seq_lens, 32, 20 + s)
        want = oracle_decode(w, s, requests=reqs, pool=w.pool_view(decode_steps=s + 1))
        assert_close(outs[s][reqs], want, f"tree cascade step {s}", rel_max=REL_MAX_OF_RMS)


def test_chunked_prefill_mix_full():
    w = W.chunked_prefill_mix()
    run = Run(w)
    ext = run.extend()
    dec = run.decode()
    _check_all_finite(ext, "extend")
    _check_all_finite(dec, "decode")
    _check_store(run, w.extend)
    _check_store(run, w.decode[0])
    pool = w.pool_view(decode_steps=1)
    reqs_e = extreme_prefix_requests(w.extend)
    toks = tile_edge_tokens(w.extend, reqs_e, w.dims.num_q_heads // w.dims.num_kv_heads)
    assert_close(ext[toks], oracle_extend(w, tokens=toks, pool=pool),
                 f"chunked extend (tile edges of requests {reqs_e})", rel_max=REL_MAX_OF_RMS)
    reqs = sample_requests(w.decode[0].seq_lens, 40, 6)
    assert len(reqs) >= 32
    assert_close(dec[reqs], oracle_decode(w, 0, requests=reqs, pool=pool),
                 f"chunked decode ({len(reqs)} requests)", rel_max=REL_MAX_OF_RMS)
