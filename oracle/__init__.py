"""CPU oracle for slot-indexed attention over a page-size-1 KV pool.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may.  It shares no code with the
CUDA library (no kernels, headers, helpers, tables or pre/post-processing);
its inputs are plain numpy arrays (bf16 as uint16 bit patterns, int32 indices).

What it computes, and where the pages fix it:
  * store_kv: ``key_buffer[out_cache_loc] = cache_k`` (and V), an index
    assignment of new rows into pool slots -- "Origins: the paper and the
    first commit", Execution: RadixAttention and two sets of kernels.
  * extend / decode attention: plain softmax attention (scores q.k, scale
    1/sqrt(head_dim), keys later than the query masked, softmax, times V) --
    "Inside SGLang", Step 3: Look inside the forward pass -- with the keys and
    values of a request read through ``req_to_token`` (same page, Paged KV and
    the kernels that read it), the prefix from the pool and only the suffix
    computed (EXTEND) -- "Origins", Batching: Req, Batch and the three forward
    modes; Execution (extend_attention_fwd reads k and v from the pool through
    req_to_token).
  * cascade decode: the same decode output assembled from per-group softmax
    states (keys shared by several requests, read once per group) and each
    request's private tail, merged exactly; shared prefixes are identical
    slot numbers in the rows ("Inside SGLang", Step 3: Paged KV and the
    kernels that read it).
  * FP8 KV pool (``oracle.fp8``): e4m3 codes with one scale per tensor,
    quantised from the float32 quotient x / scale; decode, extend (suffix
    rows read back from the pool like the prefix) and cascade decode over
    the dequantised rows -- "Inside SGLang", Step 6 (Decide how much memory
    becomes KV cache: --kv-cache-dtype fp8_e4m3, scales from the checkpoint).
  * radix tree (``oracle.radix``): token runs with their KV slots, match
    with node splitting, insert, lock counts on the path to the root,
    leaf-first LRU eviction -- "Inside SGLang", Step 4 and the "SGLang"
    notes (RadixAttention, Eviction).
All arithmetic is float64.  Every function is pinned by ``tests/test_oracle.py``
against closed forms, a library routine (full causal attention recomputed from
scratch), invariants and brute force; see that file for the list.
"""
from .attention import (  # noqa: F401
    bf16_bits_to_f64,
    default_scale,
    store_kv,
    store_kv_range,
    request_kv,
    extend_attention,
    decode_attention,
    partial_state,
    merge_states,
    cascade_decode_attention,
)
from . import fp8  # noqa: F401
from . import radix  # noqa: F401
