"""Failure detection on the GPU: the extend and cascade-group kernels' bounded
waits give up, report it, and leave the device usable.

Every wait of these kernels on a stage barrier (a copy landed, S computed, P
written, a ring slot freed) is bounded.  A normal call's waits last
microseconds, so setting the limit to a nanosecond with
sgl_set_device_wait_limit_ns makes them give up on purpose -- no fault, no
flag that nothing sets, only the short limit.  The kernel must then record
0x5701 in its workspace's status word, let its own copies and tensor-core work
finish, free its tensor memory and return; the next call with the default
limit must give correct results on the same device.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from radixattention_prefix_shared_gb300 import binding as B  # noqa: E402
from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _cases import extend_case  # noqa: E402
from _gpu import DEV, Run, assert_close, oracle_decode, oracle_extend  # noqa: E402
from test_gpu_cascade import groups_on_device  # noqa: E402
from test_gpu_fp8 import extend_pools, oracle_extend_fp8  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

TIMEOUT_CODE = 0x5701


class short_waits:
    """Every bounded wait of launches made inside the block gives up after ~1 ns."""

    def __enter__(self):
        self.prev = B.lib().sgl_set_device_wait_limit_ns(1)
        return self

    def __exit__(self, *exc):
        torch.cuda.synchronize()
        B.lib().sgl_set_device_wait_limit_ns(0)   # the default again


def _status(ws):
    return int(ws[:4].view(torch.int32).item())


def _extend(run, ws):
    e, te = run.w.extend, run.t["extend"]
    return B.sgl_extend_attention(te["q"], te["k_new"], te["v_new"], run.t["pool_k"], run.t["pool_v"],
                                  run.t["req_to_token"], te["req_pool_idx"], te["prefix_lens"],
                                  te["extend_lens"], max_extend=int(e.extend_lens.max()),
                                  max_prefix=int(e.prefix_lens.max()), workspace=ws,
                                  sm_scale=run.w.dims.sm_scale)


def _cascade(run, cg, ws):
    w = run.w
    b, tb = w.decode[0], run.t["decode"][0]
    return B.sgl_cascade_decode_attention(tb["q"], run.t["pool_k"], run.t["pool_v"], run.t["req_to_token"],
                                          tb["req_pool_idx"], tb["seq_lens"], *groups_on_device(cg),
                                          max_seq_len=int(b.seq_lens.max()),
                                          max_group_members=max(cg.max_members, 1),
                                          max_depth=max(cg.max_depth, 1), workspace=ws,
                                          sm_scale=w.dims.sm_scale)


def _device_answers():
    x = torch.arange(1 << 20, device=DEV, dtype=torch.float32)
    assert float(x.sum().item()) == float((1 << 20) * ((1 << 20) - 1) / 2)


def test_extend_gives_up_then_recovers():
    w = extend_case(91, Hq=16, Hkv=8, D=128, prefix_lens=[1, 513, 2000], extend_lens=[257, 33, 300])
    run = Run(w)
    te = run.t["extend"]
    B.sgl_store_kv(te["k_new"], te["v_new"], te["slots"], run.t["pool_k"], run.t["pool_v"])
    ws = B.new_workspace(256, DEV)
    with short_waits():
        _extend(run, ws)
    assert _status(ws) == TIMEOUT_CODE
    _device_answers()
    # the same call with the default limit, on the same device, is correct
    ws2 = B.new_workspace(256, DEV)
    out = _extend(run, ws2)
    torch.cuda.synchronize()
    assert _status(ws2) == 0
    assert_close(W.bf16_bits(out), oracle_extend(w), "extend after a timed-out call")


def test_extend_fp8_gives_up_then_recovers():
    w = extend_case(92, Hq=8, Hkv=2, D=128, prefix_lens=[300, 5, 900], extend_lens=[64, 65, 200])
    ks, vs = 1.0 / 32, 1.0 / 32
    pk, pv = extend_pools(w, ks, vs)
    e, d = w.extend, w.dims
    args = (W.bf16_tensor(e.q, DEV), pk, pv, ks, vs, W.int_tensor(w.req_to_token, DEV),
            W.int_tensor(e.req_pool_idx, DEV), W.int_tensor(e.prefix_lens, DEV), W.int_tensor(e.extend_lens, DEV))
    kw = dict(max_extend=int(e.extend_lens.max()), max_prefix=int(e.prefix_lens.max()), sm_scale=d.sm_scale)
    ws = B.new_workspace(256, DEV)
    with short_waits():
        B.sgl_extend_attention_fp8(*args, workspace=ws, **kw)
    assert _status(ws) == TIMEOUT_CODE
    _device_answers()
    ws2 = B.new_workspace(256, DEV)
    out = B.sgl_extend_attention_fp8(*args, workspace=ws2, **kw)
    torch.cuda.synchronize()
    assert _status(ws2) == 0
    assert_close(W.bf16_bits(out), oracle_extend_fp8(w, ks, vs), "fp8 extend after a timed-out call")


def test_cascade_group_pass_gives_up_then_recovers():
    dims = W.Dims(16, 4, 128, 1 << 17, 1.0 / np.sqrt(128))
    w = W.random_tree_decode(seed=93, dims=dims, fanouts=(3, 3, 2), seg_len=(100, 300), own_len=(0, 40),
                             pool_size=1 << 17)
    cg = W.tree_groups(w)
    assert cg.n_groups > 0
    run = Run(w)
    b, tb = w.decode[0], run.t["decode"][0]
    B.sgl_store_kv(tb["k_new"], tb["v_new"], tb["slots"], run.t["pool_k"], run.t["pool_v"])
    d = B.make_dims(dims.num_q_heads, dims.num_kv_heads, dims.head_dim, dims.pool_size)
    nbytes = B.cascade_decode_workspace_bytes(b.q.shape[0], int(b.seq_lens.max()), max(cg.max_depth, 1), d)
    ws = B.new_workspace(nbytes, DEV)
    with short_waits():
        _cascade(run, cg, ws)
    assert _status(ws) == TIMEOUT_CODE
    _device_answers()
    ws2 = B.new_workspace(nbytes, DEV)
    out = _cascade(run, cg, ws2)
    torch.cuda.synchronize()
    assert _status(ws2) == 0
    assert_close(W.bf16_bits(out), oracle_decode(w, 0), "cascade after a timed-out call")


def test_mixed_launch_gives_up_then_recovers():
    """The single mixed launch: its extend tiles' waits give up (the CTA that
    ran one takes no more work), the decode work still completes, and the next
    call with the default limit equals the separate calls."""
    from test_gpu_mixed import _store_step, mixed, separate
    w = W.chunked_prefill_mix(pool_size=1 << 19, n_decode=24)
    run = Run(w)
    _store_step(run)
    ref_e, ref_d = separate(run)
    ws = B.new_workspace(256, DEV)
    with short_waits():
        mixed(run, 60, ws)
    assert _status(ws) == TIMEOUT_CODE
    _device_answers()
    ws2 = B.new_workspace(256, DEV)
    got_e, got_d = mixed(run, 60, ws2)
    assert _status(ws2) == 0
    assert np.array_equal(got_e, ref_e) and np.array_equal(got_d, ref_d)
