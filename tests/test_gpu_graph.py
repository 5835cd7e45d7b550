"""The entry points inside CUDA graphs.

Decode steps are launched many times with the same shapes, so a serving loop
records them once as a CUDA graph and replays them ("Inside SGLang", Step 3:
Paged KV and the kernels that read it -- decode graphs captured per batch
size and replayed with one call).  Every call issues only kernel launches on
its stream once its kernels are set up on the device, so a captured step
replays exactly what eager launches compute; a replay reads the buffers as
they are at replay time.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from radixattention_prefix_shared_gb300 import binding as B  # noqa: E402
from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _gpu import DEV, assert_close, oracle_decode  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


class Step:
    """store_kv + extend + decode (+ cascade decode) of one workload with fixed buffers."""

    def __init__(self, w, groups=None):
        self.w, self.t = w, W.to_device(w, DEV)
        d = w.dims
        self.dims = B.make_dims(d.num_q_heads, d.num_kv_heads, d.head_dim, d.pool_size)
        self.ws_e = B.new_workspace(256, DEV)
        b = w.decode[0]
        self.ws_d = B.new_workspace(B.decode_workspace_bytes(b.q.shape[0], int(b.seq_lens.max()), self.dims), DEV)
        self.out_d = torch.empty_like(self.t["decode"][0]["q"])
        self.out_e = torch.empty_like(self.t["extend"]["q"]) if w.extend is not None else None
        self.groups = groups
        if groups is not None:
            self.g_dev = [W.int_tensor(a, DEV) for a in (groups.group_start, groups.group_len, groups.group_depth,
                                                         groups.member_off, groups.members)]
            self.ws_c = B.new_workspace(B.cascade_decode_workspace_bytes(
                b.q.shape[0], int(b.seq_lens.max()), max(groups.max_depth, 1), self.dims), DEV)
            self.out_c = torch.empty_like(self.out_d)

    def run(self):
        w, t = self.w, self.t
        if w.extend is not None:
            e, te = w.extend, t["extend"]
            B.sgl_store_kv(te["k_new"], te["v_new"], te["slots"], t["pool_k"], t["pool_v"])
            B.sgl_extend_attention(te["q"], te["k_new"], te["v_new"], t["pool_k"], t["pool_v"], t["req_to_token"],
                                   te["req_pool_idx"], te["prefix_lens"], te["extend_lens"], self.out_e,
                                   max_extend=int(e.extend_lens.max()), max_prefix=int(e.prefix_lens.max()),
                                   workspace=self.ws_e, sm_scale=w.dims.sm_scale)
        b, tb = w.decode[0], t["decode"][0]
        B.sgl_store_kv(tb["k_new"], tb["v_new"], tb["slots"], t["pool_k"], t["pool_v"])
        B.sgl_decode_attention(tb["q"], t["pool_k"], t["pool_v"], t["req_to_token"], tb["req_pool_idx"],
                               tb["seq_lens"], self.out_d, max_seq_len=int(b.seq_lens.max()),
                               workspace=self.ws_d, sm_scale=w.dims.sm_scale)
        if self.groups is not None:
            g = self.groups
            B.sgl_cascade_decode_attention(tb["q"], t["pool_k"], t["pool_v"], t["req_to_token"],
                                           tb["req_pool_idx"], tb["seq_lens"], *self.g_dev, self.out_c,
                                           max_seq_len=int(b.seq_lens.max()),
                                           max_group_members=max(g.max_members, 1),
                                           max_depth=max(g.max_depth, 1), workspace=self.ws_c,
                                           sm_scale=w.dims.sm_scale)

    def outputs(self):
        outs = [self.out_d] + ([self.out_e] if self.out_e is not None else [])
        outs += [self.out_c] if self.groups is not None else []
        return [W.bf16_bits(o) for o in outs]


def _capture(step):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step.run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step.run()
    torch.cuda.synchronize()
    return g


def test_replayed_step_equals_eager_launches():
    w = W.chunked_prefill_mix(pool_size=1 << 18, n_decode=12, n_chunks=2, chunk=300, prefix_max=3000)
    step = Step(w)
    step.run()
    torch.cuda.synchronize()
    eager = step.outputs()
    for o in (step.out_d, step.out_e):
        o.zero_()
    g = _capture(step)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(step.outputs(), eager):
        assert np.array_equal(a, b)
    assert_close(step.outputs()[0], oracle_decode(w, 0, pool=w.pool_view(decode_steps=1)), "graph decode")


def test_replay_reads_the_buffers_at_replay_time():
    dims = W.Dims(16, 4, 128, 1 << 16, 1.0 / np.sqrt(128))
    w = W.random_tree_decode(seed=77, dims=dims, pool_size=1 << 16)
    step = Step(w, groups=W.tree_groups(w))
    g = _capture(step)
    g.replay()
    torch.cuda.synchronize()
    first = step.outputs()
    # new queries in place: the replay must use them
    tb = step.t["decode"][0]
    q2 = W.normal_bf16(99, 1, tuple(tb["q"].shape), 1.0)
    tb["q"].copy_(W.bf16_tensor(q2, DEV))
    g.replay()
    torch.cuda.synchronize()
    second = step.outputs()
    assert not np.array_equal(second[0], first[0])
    step.run()
    torch.cuda.synchronize()
    for a, b in zip(step.outputs(), second):
        assert np.array_equal(a, b)
    w.decode[0].q = q2
    want = oracle_decode(w)
    assert_close(second[0], want, "graph replay decode, new q")
    assert_close(second[1], want, "graph replay cascade, new q")
