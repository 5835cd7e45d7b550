"""Shared helpers of the GPU tests: run a workload's steps through the C ABI
and compare with the oracle."""
import numpy as np
import torch

import oracle
from oracle.attention import bf16_bits_to_f64
from radixattention_prefix_shared_gb300 import binding as B
from radixattention_prefix_shared_gb300 import workloads as W

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
DEV = "cuda:0"


# ------------------------------------------------------------------ helpers

# Full-size samples also pin the largest error against the size of the
# outputs: at N(0,1) inputs an output row averages hundreds to thousands of V
# rows, so its RMS is only ~0.03-0.04 and the absolute bound above is most of
# it.  Rounding the output to bf16 alone costs up to 2^-9 of a value, and the
# fp32 sums add far less; 5% of the sample's RMS leaves room for that while a
# dropped or doubled key block (an error of the order of the output itself)
# fails.
REL_MAX_OF_RMS = 0.05


def assert_close(got_bits, want, what="", rel_max=None):
    got = bf16_bits_to_f64(got_bits)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output (a poisoned slot was read?)"
    err = np.abs(got - want)
    rms = float(np.sqrt(np.mean(want ** 2)))
    print(f"\n[parity] {what}: max abs {err.max():.3e} mean abs {err.mean():.3e} output rms {rms:.3e}")
    assert err.max() <= MAX_ABS, f"{what}: max abs err {err.max():.3g}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3g}"
    if rel_max is not None:
        assert err.max() <= rel_max * rms, f"{what}: max abs err {err.max():.3g} > {rel_max} x rms {rms:.3g}"
    return err.max(), err.mean()


class Run:
    """Upload a workload and run its steps through the C ABI."""

    def __init__(self, w, poison=True):
        self.w = w
        self.t = W.to_device(w, DEV, poison=poison)
        self.ws_ext = B.new_workspace(256, DEV)

    def extend(self):
        e, te = self.w.extend, self.t["extend"]
        B.sgl_store_kv(te["k_new"], te["v_new"], te["slots"], self.t["pool_k"], self.t["pool_v"])
        out = B.sgl_extend_attention(te["q"], te["k_new"], te["v_new"], self.t["pool_k"], self.t["pool_v"],
                                     self.t["req_to_token"], te["req_pool_idx"], te["prefix_lens"],
                                     te["extend_lens"], max_extend=int(e.extend_lens.max()),
                                     max_prefix=int(e.prefix_lens.max()), workspace=self.ws_ext,
                                     sm_scale=self.w.dims.sm_scale)
        torch.cuda.synchronize()
        assert int(self.ws_ext[:4].view(torch.int32).item()) == 0, "extend kernel reported a timeout"
        return W.bf16_bits(out)

    def decode(self, step=0):
        b, tb = self.w.decode[step], self.t["decode"][step]
        B.sgl_store_kv(tb["k_new"], tb["v_new"], tb["slots"], self.t["pool_k"], self.t["pool_v"])
        out = B.sgl_decode_attention(tb["q"], self.t["pool_k"], self.t["pool_v"], self.t["req_to_token"],
                                     tb["req_pool_idx"], tb["seq_lens"], max_seq_len=int(b.seq_lens.max()),
                                     sm_scale=self.w.dims.sm_scale)
        torch.cuda.synchronize()
        return W.bf16_bits(out)


def oracle_extend(w, tokens=None, pool=None):
    e = w.extend
    if pool is None:
        pk, pv = w.dense_pools(with_extend=False)
    else:
        pk, pv = pool.k, pool.v
    return oracle.extend_attention(e.q, e.k_new, e.v_new, pk, pv, w.req_to_token, e.req_pool_idx,
                                   e.prefix_lens, e.extend_lens, w.dims.num_kv_heads, w.dims.sm_scale,
                                   tokens=tokens)


def oracle_decode(w, step=0, requests=None, pool=None):
    b = w.decode[step]
    if pool is None:
        pk, pv = w.dense_pools(decode_steps=step + 1)
    else:
        pk, pv = pool.k, pool.v
    return oracle.decode_attention(b.q, pk, pv, w.req_to_token, b.req_pool_idx, b.seq_lens,
                                   w.dims.num_kv_heads, w.dims.sm_scale, requests=requests)


