"""sgl_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory.

Runtimes whose memory planner fixes every device buffer at start-up, and
plugin-style hosts that hand a kernel only its inputs and outputs, may not
call cudaMalloc when attention runs, so they cannot pass the decode
workspace.  The no-alloc entry point takes its split-KV scratch from a fixed
array inside the library instead.  These tests call it through the C ABI and
check that it returns what sgl_decode_attention returns, on two calls in a
row (the second call finds the first call's data in the shared array), and
that work too large for the array is refused before anything is launched.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle.attention import bf16_bits_to_f64  # noqa: E402
from radixattention_prefix_shared_gb300 import binding as B  # noqa: E402
from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402

from _cases import decode_case  # noqa: E402

DEV = "cuda:0"
MAX_ABS, MEAN_ABS = 2e-2, 2e-3
SCRATCH_BYTES = 32 * 1024 * 1024  # SGL_DECODE_NOALLOC_SCRATCH_BYTES


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, q, pool_k, pool_v, rtt, rpi, seq, max_seq, out):
    d = B.make_dims(q.shape[1], pool_k.shape[1], pool_k.shape[2], pool_k.shape[0])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sgl_decode_attention_noalloc(_p(q), _p(pool_k), _p(pool_v), _p(rtt), rtt.shape[0],
                                            rtt.shape[1], _p(rpi), _p(seq), q.shape[0], int(max_seq),
                                            _p(out), ctypes.byref(d), stream)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = B.lib()
    cases = [decode_case(71, Hq=16, Hkv=8, D=128, seq_lens=[3000, 1, 700, 2049, 513]),
             decode_case(72, Hq=32, Hkv=32, D=128, seq_lens=[1500, 64, 4097])]
    runs = []
    for w in cases:
        t = W.to_device(w, DEV)
        b, tb = w.decode[0], t["decode"][0]
        B.sgl_store_kv(tb["k_new"], tb["v_new"], tb["slots"], t["pool_k"], t["pool_v"])
        d = B.make_dims(w.dims.num_q_heads, w.dims.num_kv_heads, w.dims.head_dim, w.dims.pool_size)
        assert B.decode_workspace_bytes(b.q.shape[0], int(b.seq_lens.max()), d) <= SCRATCH_BYTES
        ref = B.sgl_decode_attention(tb["q"], t["pool_k"], t["pool_v"], t["req_to_token"], tb["req_pool_idx"],
                                     tb["seq_lens"], max_seq_len=int(b.seq_lens.max()))
        runs.append((t, tb, int(b.seq_lens.max()), ref))
    torch.cuda.synchronize()
    outs = []
    for t, tb, max_seq, _ in runs:           # two calls in a row on the shared scratch
        out = torch.full_like(tb["q"], float("nan"))
        assert _noalloc(lib, tb["q"], t["pool_k"], t["pool_v"], t["req_to_token"], tb["req_pool_idx"],
                        tb["seq_lens"], max_seq, out) == 0
        outs.append(out)
    torch.cuda.synchronize()
    for (_, _, _, ref), out in zip(runs, outs):
        got = bf16_bits_to_f64(W.bf16_bits(out))
        want = bf16_bits_to_f64(W.bf16_bits(ref))
        assert np.isfinite(got).all()
        err = np.abs(got - want)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())
        # the same kernels on the same inputs: the results are bit-identical
        assert np.array_equal(W.bf16_bits(out), W.bf16_bits(ref))


def test_noalloc_refuses_work_larger_than_its_scratch():
    lib = B.lib()
    d = B.make_dims(16, 8, 128, 1 << 22)
    need = B.decode_workspace_bytes(248, 32768, d)
    assert need > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x100000)       # never dereferenced: refused on the host first
    code = lib.sgl_decode_attention_noalloc(fake, fake, fake, fake, 256, 32768, fake, fake, 248, 32768,
                                            fake, ctypes.byref(d), None)
    assert code == 3  # SGL_ERR_WORKSPACE


@pytest.mark.parametrize("hq,hkv,d", [(16, 8, 256), (256, 1, 128)])
def test_noalloc_reports_unbuilt_shapes_like_the_workspace_entry_point(hq, hkv, d):
    """A shape the kernels are not built for (head_dim 256; 256 query heads on
    one KV head) is SGL_ERR_UNSUPPORTED from both entry points, even when its
    scratch would also exceed the fixed array."""
    lib = B.lib()
    dims = B.make_dims(hq, hkv, d, 1 << 22)
    fake = ctypes.c_void_p(0x100000)       # never dereferenced: refused on the host first
    ws = lib.sgl_decode_attention(fake, fake, fake, fake, 256, 32768, fake, fake, 248, 32768, fake,
                                  fake, 1 << 40, ctypes.byref(dims), None)
    na = lib.sgl_decode_attention_noalloc(fake, fake, fake, fake, 256, 32768, fake, fake, 248, 32768,
                                          fake, ctypes.byref(dims), None)
    assert ws == na == 2  # SGL_ERR_UNSUPPORTED
