"""Cascade decode (shared prefixes read once per group) through the C ABI,
against the fp64 oracle's plain decode.

The cascade must give the decode result whenever the groups describe slots
the members really share ("Inside SGLang", Step 3: Paged KV and the kernels
that read it -- shared prefixes are identical slot numbers), so the oracle
here is oracle.decode_attention itself; oracle.cascade_decode_attention is
pinned to it on the CPU.  Trees are random with ragged node lengths, members
are scattered through the batch, and one group is wide enough to need
several CTAs of members.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from radixattention_prefix_shared_gb300 import binding as B  # noqa: E402
from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _gpu import DEV, Run, assert_close, oracle_decode  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def groups_on_device(cg):
    return [W.int_tensor(a, DEV) for a in (cg.group_start, cg.group_len, cg.group_depth,
                                           cg.member_off, cg.members)]


def cascade(run, cg, step=0, workspace=None, store=True):
    w = run.w
    b, tb = w.decode[step], run.t["decode"][step]
    if store:
        B.sgl_store_kv(tb["k_new"], tb["v_new"], tb["slots"], run.t["pool_k"], run.t["pool_v"])
    md = max(cg.max_depth, 1)
    if workspace is None:
        d = B.make_dims(w.dims.num_q_heads, w.dims.num_kv_heads, w.dims.head_dim, w.dims.pool_size)
        workspace = B.new_workspace(B.cascade_decode_workspace_bytes(b.q.shape[0], int(b.seq_lens.max()), md, d), DEV)
    out = B.sgl_cascade_decode_attention(tb["q"], run.t["pool_k"], run.t["pool_v"], run.t["req_to_token"],
                                         tb["req_pool_idx"], tb["seq_lens"], *groups_on_device(cg),
                                         max_seq_len=int(b.seq_lens.max()),
                                         max_group_members=max(cg.max_members, 1), max_depth=md,
                                         workspace=workspace, sm_scale=w.dims.sm_scale)
    torch.cuda.synchronize()
    assert int(workspace[:4].view(torch.int32).item()) == 0, "group pass reported a timeout"
    return W.bf16_bits(out)


TREES = [
    # (Hq, Hkv, D, fanouts, seg_len, own_len)
    (16, 4, 128, (3, 3, 2), (1, 300), (0, 40)),
    (8, 8, 64, (2, 3), (50, 700), (0, 600)),
    (32, 4, 128, (3, 2), (1, 200), (0, 3)),
    (16, 8, 128, (1, 150), (100, 700), (0, 600)),   # one group of 150 members
    (4, 2, 64, (2, 2, 2), (120, 140), (0, 1)),      # g = 2, D = 64
    (12, 2, 128, (2, 3), (40, 300), (0, 50)),        # g = 6
    (32, 2, 128, (3, 2), (10, 200), (1, 30)),        # g = 16
    (24, 2, 128, (2, 3), (20, 150), (0, 20)),        # g = 12
    (32, 1, 128, (2, 3), (20, 150), (0, 20)),        # g = 32: two KV-head copies in decode
]


@pytest.mark.parametrize("tree", TREES, ids=lambda t: f"{t[0]}q{t[1]}kv{t[2]}d-{'x'.join(map(str, t[3]))}")
def test_cascade_matches_oracle(tree):
    Hq, Hkv, D, fan, seg, own = tree
    dims = W.Dims(Hq, Hkv, D, 1 << 17, 1.0 / np.sqrt(D))
    w = W.random_tree_decode(seed=300 + Hq + D, dims=dims, fanouts=fan, seg_len=seg, own_len=own,
                             pool_size=1 << 17)
    cg = W.tree_groups(w)
    assert cg.n_groups > 0
    got = cascade(Run(w), cg)
    assert_close(got, oracle_decode(w), f"cascade {tree}")


def test_cascade_equals_plain_decode_and_without_groups_is_bit_identical():
    dims = W.Dims(16, 4, 128, 1 << 16, 1.0 / np.sqrt(128))
    w = W.random_tree_decode(seed=41, dims=dims, pool_size=1 << 16)
    run = Run(w)
    plain = run.decode()
    casc = cascade(run, W.tree_groups(w), store=False)
    a = (plain.astype(np.uint32) << 16).view(np.float32)
    c = (casc.astype(np.uint32) << 16).view(np.float32)
    assert np.abs(a - c).max() <= 1e-2
    # no groups: every key is tail, the kernels' arithmetic is plain decode's
    none = W.CascadeGroups(*(np.zeros(0, np.int32),) * 3, np.zeros(1, np.int32), np.zeros(0, np.int32))
    assert np.array_equal(cascade(run, none, store=False), plain)


def test_cascade_on_tree_steps_reuses_workspace():
    w = W.tree_of_thought_decode(depth=3, fanout=3, segment=200, steps=3, pool_size=1 << 16)
    run = Run(w)
    cg = W.tree_groups(w)
    d = B.make_dims(32, 8, 128, w.dims.pool_size)
    ws = B.new_workspace(B.cascade_decode_workspace_bytes(27, 603, cg.max_depth, d), DEV)
    for s in range(3):
        assert_close(cascade(run, W.tree_groups(w, s), step=s, workspace=ws), oracle_decode(w, s),
                     f"tree step {s}")


def test_cascade_repeated_launches_bit_identical():
    dims = W.Dims(16, 4, 128, 1 << 16, 1.0 / np.sqrt(128))
    w = W.random_tree_decode(seed=43, dims=dims, pool_size=1 << 16)
    run = Run(w)
    cg = W.tree_groups(w)
    a = cascade(run, cg)
    for _ in range(3):
        assert np.array_equal(cascade(run, cg, store=False), a)


def test_cascade_checked_mode():
    dims = W.Dims(8, 4, 64, 1 << 14, 0.125)
    w = W.random_tree_decode(seed=44, dims=dims, fanouts=(2, 3, 2), seg_len=(5, 40), own_len=(1, 9),
                             pool_size=1 << 14)
    t = W.to_device(w, DEV)
    b, tb = w.decode[0], t["decode"][0]
    cg = W.tree_groups(w)
    err = torch.zeros(4, dtype=torch.int32, device=DEV)

    def check(groups, rtt=None, max_members=None, seq_lens=None):
        err.zero_()
        B.sgl_check_cascade_groups(t["req_to_token"] if rtt is None else rtt, tb["req_pool_idx"],
                                   tb["seq_lens"] if seq_lens is None else seq_lens,
                                   *groups_on_device(groups),
                                   max_group_members=max_members or groups.max_members,
                                   max_depth=cg.max_depth, d_error=err)
        torch.cuda.synchronize()
        return err.tolist()

    assert check(cg) == [0, 0, 0, 0]
    j = int(np.nonzero(cg.group_depth == 1)[0][0])
    m0 = int(cg.members[cg.member_off[j]])
    # kind 7: a member outside the batch; a member count above the host max
    bad = W.CascadeGroups(cg.group_start, cg.group_len, cg.group_depth, cg.member_off, cg.members.copy())
    bad.members[cg.member_off[j]] = b.seq_lens.size
    assert check(bad)[0] == 7
    assert check(cg, max_members=1)[0] == 7
    # kind 8: a member whose seq_len ends inside one of its groups
    sl = tb["seq_lens"].clone()
    sl[m0] = int(cg.group_start[j] + cg.group_len[j]) - 1
    e = check(cg, seq_lens=sl)
    assert e[0] == 8 and e[2] == m0
    # kind 9: a member whose slot differs inside the group
    rtt = t["req_to_token"].clone()
    victim = int(cg.members[cg.member_off[j + 1] - 1])
    row, pos = int(b.req_pool_idx[victim]), int(cg.group_start[j])
    rtt[row, pos] = (int(w.req_to_token[row, pos]) + 1) % w.dims.pool_size
    e = check(cg, rtt=rtt)
    assert e[0] == 9 and e[1] == j and e[3] == victim
    # kind 10: a gap between a request's groups (depth-1 group starts late)
    bad = W.CascadeGroups(cg.group_start.copy(), cg.group_len.copy(), cg.group_depth, cg.member_off, cg.members)
    bad.group_start[j] += 1
    bad.group_len[j] -= 1
    assert bad.group_len[j] >= 1
    assert check(bad)[0] == 10
    # kind 10: two groups at one depth
    bad = W.CascadeGroups(cg.group_start, cg.group_len, cg.group_depth.copy(), cg.member_off, cg.members)
    bad.group_depth[j] = 0
    assert check(bad)[0] == 10
