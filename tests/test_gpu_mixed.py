"""sgl_mixed_attention: the extend batch and the decode batch of one step in
one launch, through the C ABI.

The single launch runs the extend kernel's pipeline and the split-KV decode
loop side by side on the SMs (an SM whose side runs out takes the other
side's work), so its outputs must be the separate calls' outputs bit for bit,
whatever the split of the SMs -- and those are pinned to the oracle.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from radixattention_prefix_shared_gb300 import binding as B  # noqa: E402
from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _cases import extend_case  # noqa: E402
from _gpu import DEV, REL_MAX_OF_RMS, Run, assert_close, oracle_decode, oracle_extend  # noqa: E402
from _sampling import extreme_prefix_requests, sample_requests, tile_edge_tokens  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _store_step(run):
    t = run.t
    te, tb = t["extend"], t["decode"][0]
    B.sgl_store_kv(te["k_new"], te["v_new"], te["slots"], t["pool_k"], t["pool_v"])
    B.sgl_store_kv(tb["k_new"], tb["v_new"], tb["slots"], t["pool_k"], t["pool_v"])


def _limits(w):
    e, b = w.extend, w.decode[0]
    return dict(max_extend=int(e.extend_lens.max()) if e.extend_lens.size else 0,
                max_prefix=int(e.prefix_lens.max()) if e.prefix_lens.size else 0,
                max_seq_len=int(b.seq_lens.max()) if b.seq_lens.size else 1)


def mixed(run, extend_sms=0, ext_ws=None):
    """One mixed call over the step (its new rows stored first)."""
    w, t = run.w, run.t
    te, tb = t["extend"], t["decode"][0]
    lim = _limits(w)
    oe, od = B.sgl_mixed_attention(te["q"], te["k_new"], te["v_new"], te["req_pool_idx"], te["prefix_lens"],
                                   te["extend_lens"], tb["q"], tb["req_pool_idx"], tb["seq_lens"], t["pool_k"],
                                   t["pool_v"], t["req_to_token"], extend_sms=extend_sms, ext_workspace=ext_ws,
                                   sm_scale=w.dims.sm_scale, **lim)
    torch.cuda.synchronize()
    return W.bf16_bits(oe), W.bf16_bits(od)


def separate(run):
    """The same step as two calls: extend, then decode."""
    w, t = run.w, run.t
    te, tb = t["extend"], t["decode"][0]
    lim = _limits(w)
    oe = B.sgl_extend_attention(te["q"], te["k_new"], te["v_new"], t["pool_k"], t["pool_v"], t["req_to_token"],
                                te["req_pool_idx"], te["prefix_lens"], te["extend_lens"],
                                max_extend=lim["max_extend"], max_prefix=lim["max_prefix"],
                                sm_scale=w.dims.sm_scale)
    od = B.sgl_decode_attention(tb["q"], t["pool_k"], t["pool_v"], t["req_to_token"], tb["req_pool_idx"],
                                tb["seq_lens"], max_seq_len=lim["max_seq_len"], sm_scale=w.dims.sm_scale)
    torch.cuda.synchronize()
    return W.bf16_bits(oe), W.bf16_bits(od)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.fixture(scope="module")
def chunked_small():
    """The chunked-prefill mix's step shape (8 x 2,048-token chunks, GQA
    16/8, head dim 128) with 24 decode requests over a 2^19-slot pool."""
    w = W.chunked_prefill_mix(pool_size=1 << 19, n_decode=24)
    run = Run(w)
    _store_step(run)
    return w, run, separate(run)


@pytest.mark.parametrize("split", ["auto", "one", "half", "all_but_one"])
def test_mixed_equals_separate_calls(chunked_small, split):
    w, run, (ref_e, ref_d) = chunked_small
    n = _sms()
    extend_sms = {"auto": 0, "one": 1, "half": n // 2, "all_but_one": n - 1}[split]
    ws = B.new_workspace(256, DEV)
    got_e, got_d = mixed(run, extend_sms, ws)
    assert int(ws[:4].view(torch.int32).item()) == 0, "extend role reported a timeout"
    assert np.array_equal(got_e, ref_e), "extend rows differ from sgl_extend_attention's"
    assert np.array_equal(got_d, ref_d), "decode rows differ from sgl_decode_attention's"


def test_mixed_matches_oracle(chunked_small):
    w, run, _ = chunked_small
    got_e, got_d = mixed(run, 0)
    pool = w.pool_view(decode_steps=1)
    toks = tile_edge_tokens(w.extend, extreme_prefix_requests(w.extend), 2)
    assert_close(got_e[toks], oracle_extend(w, tokens=toks, pool=pool), "mixed extend", rel_max=REL_MAX_OF_RMS)
    reqs = sample_requests(w.decode[0].seq_lens, 24, 5)
    assert_close(got_d[reqs], oracle_decode(w, 0, requests=reqs, pool=pool), "mixed decode", rel_max=REL_MAX_OF_RMS)


def test_mixed_tiny_head_dim_64():
    """One query head per KV head at head dim 64; the decode step's keys
    include the extend's suffix rows (stored before the call)."""
    w = W.tiny()
    run = Run(w)
    _store_step(run)
    ref_e, ref_d = separate(run)
    for extend_sms in (0, 3, _sms() - 1):
        got_e, got_d = mixed(run, extend_sms)
        assert np.array_equal(got_e, ref_e) and np.array_equal(got_d, ref_d), extend_sms
    assert_close(got_e, oracle_extend(w, pool=w.pool_view(decode_steps=1)), "mixed tiny extend")
    assert_close(got_d, oracle_decode(w, 0, pool=w.pool_view(decode_steps=1)), "mixed tiny decode")


def test_mixed_other_group_sizes_run_the_two_kernels():
    """Four query heads per KV head (not built into the single launch): the
    call still returns the two calls' outputs."""
    w = extend_case(33, Hq=32, Hkv=8, D=128, prefix_lens=[300, 0, 700], extend_lens=[64, 200, 9],
                    decode_after=True)
    run = Run(w)
    _store_step(run)
    ref_e, ref_d = separate(run)
    got_e, got_d = mixed(run, 40)
    assert np.array_equal(got_e, ref_e) and np.array_equal(got_d, ref_d)
    assert_close(got_d, oracle_decode(w, 0, pool=w.pool_view(decode_steps=1)), "mixed g=4 decode")


def test_mixed_with_one_side_empty(chunked_small):
    w, run, (ref_e, ref_d) = chunked_small
    t = run.t
    te, tb = t["extend"], t["decode"][0]
    lim = _limits(w)
    empty_i = torch.zeros(0, dtype=torch.int32, device=DEV)
    q0 = torch.empty((0,) + tuple(tb["q"].shape[1:]), dtype=tb["q"].dtype, device=DEV)
    # no decode requests: the extend alone
    oe, _ = B.sgl_mixed_attention(te["q"], te["k_new"], te["v_new"], te["req_pool_idx"], te["prefix_lens"],
                                  te["extend_lens"], q0, empty_i, empty_i, t["pool_k"], t["pool_v"],
                                  t["req_to_token"], sm_scale=w.dims.sm_scale, **lim)
    # no extend batch: the decode alone
    qe0 = torch.empty((0,) + tuple(te["q"].shape[1:]), dtype=te["q"].dtype, device=DEV)
    ke0 = torch.empty((0,) + tuple(te["k_new"].shape[1:]), dtype=te["k_new"].dtype, device=DEV)
    _, od = B.sgl_mixed_attention(qe0, ke0, ke0, empty_i, empty_i, empty_i, tb["q"], tb["req_pool_idx"],
                                  tb["seq_lens"], t["pool_k"], t["pool_v"], t["req_to_token"],
                                  sm_scale=w.dims.sm_scale, total_extend=0, **lim)
    torch.cuda.synchronize()
    assert np.array_equal(W.bf16_bits(oe), ref_e)
    assert np.array_equal(W.bf16_bits(od), ref_d)
