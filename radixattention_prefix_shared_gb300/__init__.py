"""GB300-native slot-indexed attention over a page-size-1 KV pool.

The compute path is the C-ABI library ``libsgl_attn.so`` (hand-written CUDA
for sm_103a, sources in ``csrc/``); ``binding`` is a thin ctypes layer with the
same names (``sgl_store_kv``, ``sgl_extend_attention``, ``sgl_decode_attention``).
``workloads`` draws seeded synthetic inputs and ``workmodel`` counts the
algorithmic bytes and flops used for roofline accounting.
"""
__all__ = ["binding", "workloads", "workmodel"]
