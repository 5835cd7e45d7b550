"""Algorithmic-work accounting (the numerators of every roofline figure),
checked by enumerating the bytes each step must move on tiny inputs, and the
bench's rule that ncu traffic is reported only for the kernel source it was
taken on."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from radixattention_prefix_shared_gb300 import workmodel as WM  # noqa: E402


def _enumerated_decode_bytes(seq_lens, hq, hkv, d, elem):
    total = 0
    for s in seq_lens:
        for _ in range(s):                       # every key of the request
            total += hkv * d * elem              # its K row (all KV heads)
            total += hkv * d * elem              # its V row
            total += 4                           # its int32 slot id
        total += hq * d * 2                      # the bf16 query
        total += hq * d * 2                      # the bf16 output
    return total


@pytest.mark.parametrize("elem", [2, 1])
def test_decode_bytes_by_enumeration(elem):
    seq = [1, 7, 33]
    assert WM.decode_bytes(seq, 4, 2, 8, elem) == _enumerated_decode_bytes(seq, 4, 2, 8, elem)


@pytest.mark.parametrize("elem", [2, 1])
def test_cascade_bytes_read_each_group_once(elem):
    # three requests share positions [0, 4) (one group), requests 0 and 1 also
    # share [4, 6) (a second group); the rest of each row is private
    seq = [9, 6, 5]
    shared = [6, 6, 4]
    groups = [4, 2]
    hq, hkv, d = 4, 2, 8
    total = 0
    for s, sh in zip(seq, shared):
        for _ in range(sh, s):                   # every private tail key
            total += 2 * hkv * d * elem + 4      # K + V rows, slot id
        total += 2 * hq * d * 2                  # bf16 query in, output out
    for n in groups:
        for _ in range(n):                       # every group key, once
            total += 2 * hkv * d * elem + 4
    assert WM.cascade_decode_bytes(groups, shared, seq, hq, hkv, d, elem) == total
    # with no sharing it is plain decode
    assert (WM.cascade_decode_bytes([], [0, 0, 0], seq, hq, hkv, d, elem)
            == WM.decode_bytes(seq, hq, hkv, d, elem))


@pytest.mark.parametrize("elem", [2, 1])
def test_decode_unique_bytes_counts_shared_slots_once(elem):
    rtt = np.array([[3, 4, 5, 9], [3, 4, 6, 0], [7, 8, 0, 0]], dtype=np.int32)
    seq = [4, 3, 2]
    hq, hkv, d = 2, 1, 4
    uniq = len({3, 4, 5, 9, 6, 7, 8})
    want = uniq * 2 * hkv * d * elem + 4 * sum(seq) + len(seq) * 2 * hq * d * 2
    assert WM.decode_unique_bytes(rtt, [0, 1, 2], seq, hq, hkv, d, elem) == want


def test_bench_counts_e4m3_cascade_bytes_at_one_byte_a_value():
    """The bench's read-once decode bytes over an e4m3 pool use one byte per
    K/V value, like its plain-decode bytes."""
    import bench
    from radixattention_prefix_shared_gb300 import workloads as W
    w = W.tree_of_thought_decode(pool_size=1 << 18, steps=1)
    groups = [W.tree_groups(w, 0)]
    b16, b8 = bench.work_of(w, groups, 2), bench.work_of(w, groups, 1)
    qo = 2 * 2 * w.decode[0].q.shape[0] * w.dims.num_q_heads * w.dims.head_dim
    n_keys = (b16["decode_read_once_bytes"] - qo) // (2 * w.dims.num_kv_heads * w.dims.head_dim * 2 + 4)
    assert b8["decode_read_once_bytes"] == n_keys * (2 * w.dims.num_kv_heads * w.dims.head_dim + 4) + qo
    assert b8["decode_read_once_bytes"] < b16["decode_read_once_bytes"]


@pytest.mark.parametrize("elem", [2, 1])
def test_store_kv_bytes_by_enumeration(elem):
    n, hkv, d = 5, 3, 16
    per_token = 0
    per_token += 2 * hkv * d * 2                 # read the new bf16 K and V rows
    per_token += 2 * hkv * d * elem              # write them (bf16 or e4m3 codes)
    per_token += 4                               # read the slot id
    assert WM.store_kv_bytes(n, hkv, d, elem) == n * per_token


def test_extend_bytes_by_enumeration():
    P, E = [0, 5, 130], [3, 1, 77]
    hq, hkv, d = 4, 2, 8
    kv = 2 * hkv * d * 2
    want = sum(P) * (kv + 4) + sum(E) * kv + 2 * sum(E) * hq * d * 2
    assert WM.extend_bytes(P, E, hq, hkv, d) == want


def test_traffic_reported_only_for_the_captured_source(monkeypatch):
    import bench
    entry = None
    for wl in ("chunked_prefill_mix", "shared_prompt_extend"):
        entry = bench.measured_traffic("extend", wl)
        if entry is not None:
            break
    if entry is None:
        pytest.skip("no extend capture matches the current source")
    assert entry > 0
    # a source that changed since the capture reports no traffic
    monkeypatch.setattr(bench, "kernel_source_hash", lambda name: "0" * 16)
    assert bench.measured_traffic("extend", wl) is None
    # nor does a workload that was never captured
    monkeypatch.undo()
    assert bench.measured_traffic("extend", "no_such_workload") is None
