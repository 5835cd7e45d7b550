"""Throughput of the slot-indexed attention hot path on GB300.

One step = one pass of the whole path over one batch: store_kv of every new
token, extend attention over the chunked-prefill requests, decode attention
over the decode requests (the chunked-prefill mix workload: 8 extend chunks of
2,048 tokens after cached prefixes of up to 16,384 tokens, plus 248 decode
requests with contexts of 1,024..32,768 tokens, Qwen3-0.6B-like GQA 16/8,
head dim 128, pool of 4,194,304 slots after a 30% leaf-first LRU eviction).

Prints ONE JSON line (rank 0).  `value` is query tokens (extend + decode) per
second of device time with inputs resident in HBM; `e2e` is the same metric
with the step's inputs copied from pinned host memory and its outputs read
back inside the timed region.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from radixattention_prefix_shared_gb300 import workloads as W  # noqa: E402
from radixattention_prefix_shared_gb300 import workmodel as WM  # noqa: E402

METRIC = "extend+decode attention tokens/s; HBM GB/s and TC util vs GB300 peak"
WORKLOAD_NAMES = {1: "tiny", 2: "decode_llama7b", 3: "shared_prompt_extend",
                  4: "tree_of_thought_decode", 5: "chunked_prefill_mix"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
FP8_SCALE = 1.0 / 64  # per-tensor K and V scale of an e4m3 pool: N(0,1) rows stay inside +-448


# ----------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


def kernel_source_hash(name: str) -> str:
    """Hash of a kernel's sources: common.cuh, the launcher file and, where
    there is one, the device header beside it (decode.cu -> decode_dev.cuh)."""
    import hashlib
    csrc = os.path.join(ROOT, "radixattention_prefix_shared_gb300", "csrc")
    files = ["common.cuh", name]
    dev = name[:-3] + "_dev.cuh" if name.endswith(".cu") else None
    if dev is not None and os.path.exists(os.path.join(csrc, dev)):
        files.append(dev)
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel source as it is now (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        e = d[workload][kernel]
        if e.get("source_hash") != kernel_source_hash(e["source_file"]):
            return None
        return int(e["bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, group=None, device=None) -> float:
    """Largest value of x over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ----------------------------------------------------------------- GPU arm

class Step:
    """Device buffers of one workload and the launches of one step."""

    def __init__(self, w: W.Workload, device, cascade: str = "off", kv: str = "bf16",
                 overlap: bool = False):
        import torch
        from radixattention_prefix_shared_gb300 import binding as B
        self.B, self.torch, self.w, self.dev = B, torch, w, device
        self.overlap = overlap
        self.side = torch.cuda.Stream(device=device) if overlap else None
        t = W.to_device(w, device)
        self.t = t
        self.fp8 = kv == "fp8"
        if self.fp8:
            # the cached rows pass through the quantising store once (setup);
            # one scale per tensor, as a checkpoint provides
            self.k_scale = self.v_scale = FP8_SCALE
            pk8 = torch.zeros(t["pool_k"].shape, dtype=torch.uint8, device=device)
            pv8 = torch.zeros_like(pk8)
            live = torch.from_numpy(w.live_slots.astype(np.int64)).to(device)
            for a in range(0, live.numel(), 1 << 16):
                idx = live[a: a + (1 << 16)]
                B.sgl_store_kv_fp8(t["pool_k"][idx].contiguous(), t["pool_v"][idx].contiguous(),
                                   idx.to(torch.int32), pk8, pv8, self.k_scale, self.v_scale)
            torch.cuda.synchronize()
            t["pool_k"], t["pool_v"] = pk8, pv8
        d = w.dims
        self.Hq, self.Hkv, self.D = d.num_q_heads, d.num_kv_heads, d.head_dim
        # one store_kv over every new token: the extend and first-decode k/v
        # are views of one contiguous buffer
        parts_k, parts_v, parts_s = [], [], []
        if w.extend is not None:
            parts_k.append(t["extend"]["k_new"]); parts_v.append(t["extend"]["v_new"])
            parts_s.append(t["extend"]["slots"])
        if w.decode:
            parts_k.append(t["decode"][0]["k_new"]); parts_v.append(t["decode"][0]["v_new"])
            parts_s.append(t["decode"][0]["slots"])
        self.k_all = torch.cat(parts_k).contiguous()
        self.v_all = torch.cat(parts_v).contiguous()
        self.s_all = torch.cat(parts_s).contiguous()
        n_ext = 0
        if w.extend is not None:
            n_ext = w.extend.total_extend
            t["extend"]["k_new"] = self.k_all[:n_ext]
            t["extend"]["v_new"] = self.v_all[:n_ext]
        if w.decode:
            t["decode"][0]["k_new"] = self.k_all[n_ext:]
            t["decode"][0]["v_new"] = self.v_all[n_ext:]
        self.ws_ext = B.new_workspace(256, device)
        self.out_ext = torch.empty_like(t["extend"]["q"]) if w.extend is not None else None
        # cascade decode: the shared-prefix groups of every decode step, from
        # the library's radix tree as a serving loop's host side keeps it;
        # "auto" uses them when the batch shares prefixes
        self.groups = []
        if cascade != "off" and w.decode:
            self.groups = radix_tree_groups(w)
            if cascade == "auto" and not any(g.n_groups for g in self.groups):
                self.groups = []
        self.cascade = bool(self.groups)
        self.groups_dev = [[W.int_tensor(a, device) for a in (g.group_start, g.group_len, g.group_depth,
                                                              g.member_off, g.members)]
                           for g in self.groups]
        self.out_dec, self.ws_dec = [], []
        for s, (b, tb) in enumerate(zip(w.decode, t["decode"])):
            self.out_dec.append(torch.empty_like(tb["q"]))
            dims = B.make_dims(self.Hq, self.Hkv, self.D, d.pool_size)
            if self.cascade:
                nb = B.cascade_decode_workspace_bytes(b.q.shape[0], int(b.seq_lens.max()),
                                                      max(self.groups[s].max_depth, 1), dims)
            else:
                nb = B.decode_workspace_bytes(b.q.shape[0], int(b.seq_lens.max()), dims)
            self.ws_dec.append(B.new_workspace(nb, device))
        self.tokens = (w.extend.total_extend if w.extend is not None else 0) + sum(b.q.shape[0] for b in w.decode)
        self.launches = 0

    def run(self, ev=None):
        """One step; records events [start, after store, after extend, after decode].

        With `overlap` (and no events) the extend and the decode batches, which
        touch different requests, run on two streams and join before the step
        ends: the decode CTAs take the SMs the extend's last wave leaves idle.
        The decode follows the store; over a bf16 pool the extend does not
        need it and starts beside it."""
        B, t, w = self.B, self.t, self.w
        torch = self.torch
        launches = 0
        fork = self.overlap and ev is None and w.extend is not None and bool(w.decode)
        if fork:
            # over a bf16 pool the extend reads its suffix from k_new / v_new
            # and its prefix from rows stored by earlier steps, so it does not
            # wait for this step's store; the decode (which reads its own new
            # row from the pool) and the e4m3 extend (which reads its suffix
            # back from the pool) do
            main = torch.cuda.current_stream()
            self.side.wait_stream(main)
            self.store(self.k_all, self.v_all, self.s_all)
            launches += 1
            if self.fp8:
                self.side.wait_stream(main)
            with torch.cuda.stream(self.side):
                launches += self.run_extend()
            launches += self.run_decode()
            main.wait_stream(self.side)
            self.launches = launches
            return
        if ev is not None:
            ev[0].record()
        self.store(self.k_all, self.v_all, self.s_all)
        launches += 1
        if ev is not None:
            ev[1].record()
        launches += self.run_extend()
        if ev is not None:
            ev[2].record()
        launches += self.run_decode()
        if ev is not None:
            ev[3].record()
        self.launches = launches

    def run_extend(self):
        B, t, w = self.B, self.t, self.w
        launches = 0
        if w.extend is not None and self.fp8:
            # the suffix rows were stored (quantised) with the step's store and
            # are read back from the pool like the prefix
            e, te = w.extend, t["extend"]
            B.sgl_extend_attention_fp8(te["q"], t["pool_k"], t["pool_v"], self.k_scale, self.v_scale,
                                       t["req_to_token"], te["req_pool_idx"], te["prefix_lens"],
                                       te["extend_lens"], self.out_ext, max_extend=int(e.extend_lens.max()),
                                       max_prefix=int(e.prefix_lens.max()), workspace=self.ws_ext)
            launches += 1
        elif w.extend is not None:
            e, te = w.extend, t["extend"]
            B.sgl_extend_attention(te["q"], te["k_new"], te["v_new"], t["pool_k"], t["pool_v"],
                                   t["req_to_token"], te["req_pool_idx"], te["prefix_lens"],
                                   te["extend_lens"], self.out_ext, max_extend=int(e.extend_lens.max()),
                                   max_prefix=int(e.prefix_lens.max()), workspace=self.ws_ext)
            launches += 1
        return launches

    def run_decode(self):
        B, t, w = self.B, self.t, self.w
        launches = 0
        for s, (b, tb) in enumerate(zip(w.decode, t["decode"])):
            if s > 0:
                self.store(tb["k_new"], tb["v_new"], tb["slots"])
                launches += 1
            if self.cascade:
                g = self.groups[s]
                B.sgl_cascade_decode_attention(tb["q"], t["pool_k"], t["pool_v"], t["req_to_token"],
                                               tb["req_pool_idx"], tb["seq_lens"], *self.groups_dev[s],
                                               self.out_dec[s], max_seq_len=int(b.seq_lens.max()),
                                               max_group_members=max(g.max_members, 1),
                                               max_depth=max(g.max_depth, 1), workspace=self.ws_dec[s],
                                               kv_scales=(self.k_scale, self.v_scale) if self.fp8 else None)
                launches += 4 if g.n_groups else 3   # plan, groups, split, combine
            elif self.fp8:
                B.sgl_decode_attention_fp8(tb["q"], t["pool_k"], t["pool_v"], self.k_scale, self.v_scale,
                                           t["req_to_token"], tb["req_pool_idx"], tb["seq_lens"],
                                           self.out_dec[s], max_seq_len=int(b.seq_lens.max()),
                                           workspace=self.ws_dec[s])
                launches += 3                        # plan, split, combine
            else:
                B.sgl_decode_attention(tb["q"], t["pool_k"], t["pool_v"], t["req_to_token"],
                                       tb["req_pool_idx"], tb["seq_lens"], self.out_dec[s],
                                       max_seq_len=int(b.seq_lens.max()), workspace=self.ws_dec[s])
                launches += 3                        # plan, split, combine
        return launches

    def store(self, k, v, slots):
        t = self.t
        if self.fp8:
            self.B.sgl_store_kv_fp8(k, v, slots, t["pool_k"], t["pool_v"], self.k_scale, self.v_scale)
        else:
            self.B.sgl_store_kv(k, v, slots, t["pool_k"], t["pool_v"])

    def twin(self):
        """A second set of per-step input/output buffers over the same pools
        and req_to_token (for double-buffered host transfers)."""
        import copy
        import torch
        o = copy.copy(self)
        o.t = dict(self.t)
        if self.w.extend is not None:
            o.t["extend"] = {k: v.clone() for k, v in self.t["extend"].items()}
        o.t["decode"] = [{k: v.clone() for k, v in tb.items()} for tb in self.t["decode"]]
        o.k_all, o.v_all, o.s_all = self.k_all.clone(), self.v_all.clone(), self.s_all.clone()
        n_ext = 0
        if self.w.extend is not None:
            n_ext = self.w.extend.total_extend
            o.t["extend"]["k_new"] = o.k_all[:n_ext]
            o.t["extend"]["v_new"] = o.v_all[:n_ext]
        if self.w.decode:
            o.t["decode"][0]["k_new"] = o.k_all[n_ext:]
            o.t["decode"][0]["v_new"] = o.v_all[n_ext:]
        o.ws_ext = self.B.new_workspace(256, self.dev)
        o.out_ext = torch.empty_like(self.out_ext) if self.out_ext is not None else None
        o.out_dec = [torch.empty_like(x) for x in self.out_dec]
        o.ws_dec = [torch.zeros_like(x) for x in self.ws_dec]
        o.groups_dev = [[x.clone() for x in g] for g in self.groups_dev]
        return o

    # inputs that arrive from the host every step, and the results read back
    def host_io(self):
        import torch
        ins, outs = [self.k_all, self.v_all, self.s_all], []
        if self.w.extend is not None:
            te = self.t["extend"]
            ins += [te["q"], te["req_pool_idx"], te["prefix_lens"], te["extend_lens"]]
            outs.append(self.out_ext)
        for s, tb in enumerate(self.t["decode"]):
            ins += [tb["q"], tb["req_pool_idx"], tb["seq_lens"]]
            if self.cascade:
                ins += self.groups_dev[s]
            if s > 0:
                ins += [tb["k_new"], tb["v_new"], tb["slots"]]
            outs.append(self.out_dec[s])
        pin_in = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x) for x in ins]
        pin_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in outs]
        return list(zip(pin_in, ins)), list(zip(outs, pin_out))


# reduced instances of the workloads for profiler captures (a few GB on the
# device, inputs still larger than L2); same kernels, same per-request shapes
SMALL = {2: dict(pool_size=1 << 18), 3: dict(pool_size=1 << 17),
         4: dict(pool_size=1 << 18), 5: dict(pool_size=1 << 19, n_decode=24)}


PAGED = (2, 3)  # workloads that lay their slots out in whole pages when asked


def small_kwargs(args):
    kw = dict(SMALL.get(args.config, {})) if getattr(args, "small", False) else {}
    if getattr(args, "page_size", 1) > 1:
        kw["page_size"] = args.page_size
    return kw


def prefix_sharing(rows):
    """Batch cache hit rate ("Origins: the paper and the first commit", the
    paper's notation table: hit rate = 1 - C / prompt tokens, C = the summed
    edge lengths of the batch's radix tree), from the library's radix tree with
    every row's slots inserted as its tokens."""
    from radixattention_prefix_shared_gb300 import binding as B
    tree = B.RadixTree()
    total = 0
    for row in rows:
        tree.insert(row, row)
        total += len(row)
    unique = tree.evictable_tokens
    return {"prompt_tokens": int(total), "tree_tokens": int(unique),
            "within_batch_hit_rate": round(1.0 - unique / total, 4) if total else 0.0}


def sharing_of(w: W.Workload):
    out = {}
    if w.extend is not None:
        e = w.extend
        out["extend"] = prefix_sharing([w.req_to_token[r, : p + n] for r, p, n in
                                        zip(e.req_pool_idx, e.prefix_lens, e.extend_lens)])
        # tokens whose KV the step reads from the cache instead of computing
        out["extend"]["cached_prefix_fraction"] = round(
            float(e.prefix_lens.sum()) / max(1.0, float(e.prefix_lens.sum() + e.extend_lens.sum())), 4)
    if w.decode:
        b = w.decode[0]
        out["decode"] = prefix_sharing([w.req_to_token[r, :n] for r, n in zip(b.req_pool_idx, b.seq_lens)])
    return out


def radix_tree_groups(w: W.Workload):
    """The shared-prefix groups of every decode step of ``w`` from the
    library's radix tree ("Inside SGLang", Step 4: match_prefix and insert):
    each step inserts every request's row up to its new token (slot ids stand
    in for token ids: requests that share a prefix share its slots), looks
    the row up for the node it ends on, and asks the tree for the groups of
    those nodes (sgl_radix_groups)."""
    from radixattention_prefix_shared_gb300 import binding as B
    tree = B.RadixTree()
    out = []
    for b in w.decode:
        nodes = []
        for r, n in zip(b.req_pool_idx, b.seq_lens):
            row = w.req_to_token[int(r), : int(n)]
            tree.insert(row, row)
            nodes.append(tree.match_prefix(row)[2])
        out.append(W.CascadeGroups(*tree.groups(nodes)))
    return out


def work_of(w: W.Workload, groups=(), kv_elem_bytes=2):
    d = w.dims
    flops = 0
    ext_bytes = 0
    if w.extend is not None:
        e = w.extend
        flops = WM.extend_flops(e.prefix_lens, e.extend_lens, d.num_q_heads, d.head_dim)
        ext_bytes = WM.extend_bytes(e.prefix_lens, e.extend_lens, d.num_q_heads, d.num_kv_heads, d.head_dim)
    dec_bytes = sum(WM.decode_bytes(b.seq_lens, d.num_q_heads, d.num_kv_heads, d.head_dim, kv_elem_bytes)
                    for b in w.decode)
    # with cascade groups each shared group's keys are read once per step
    dec_unique = sum(WM.cascade_decode_bytes(g.group_len, g.shared_lens(b.q.shape[0]), b.seq_lens,
                                             d.num_q_heads, d.num_kv_heads, d.head_dim, kv_elem_bytes)
                     for g, b in zip(groups, w.decode)) if groups else dec_bytes
    n_new = (w.extend.total_extend if w.extend is not None else 0) + sum(b.q.shape[0] for b in w.decode)
    st_bytes = WM.store_kv_bytes(n_new, d.num_kv_heads, d.head_dim, kv_elem_bytes)
    return dict(extend_flops=flops, extend_bytes=ext_bytes, decode_bytes=dec_bytes,
                decode_read_once_bytes=dec_unique, store_bytes=st_bytes)


def capture_step(step):
    """One step recorded as a CUDA graph (every launch of the step, replayed
    with one call, as a serving loop replays its decode step)."""
    import torch
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


def gpu_arm(args):
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.make(args.config, seed=1000 + args.config + 7919 * rank, **small_kwargs(args))
    step = Step(w, dev, args.cascade, args.kv, overlap=args.overlap == "on")
    work = work_of(w, step.groups, 1 if step.fp8 else 2)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # 2x L2
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        step.run()
        flush.zero_()
    torch.cuda.synchronize()

    graph = capture_step(step) if args.graph == "on" else None
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    gevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    launches = 0
    with ClockSampler(local) as clocks:
        wall0 = time.perf_counter()
        if graph is not None:
            # the headline: the step replayed as one CUDA graph
            for k in range(args.steps):
                gevs[k][0].record()
                graph.replay()
                gevs[k][1].record()
                launches += step.launches
                flush.zero_()                   # outside the events: L2 cold for every step
        # per-kernel breakdown: the same step launched eagerly between events
        for k in range(args.steps):
            step.run(evs[k])
            launches += step.launches
            flush.zero_()
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier()
    t_eager = [evs[k][0].elapsed_time(evs[k][3]) for k in range(args.steps)]
    t_step = [gevs[k][0].elapsed_time(gevs[k][1]) for k in range(args.steps)] if graph is not None else t_eager
    t_store = [evs[k][0].elapsed_time(evs[k][1]) for k in range(args.steps)]
    t_ext = [evs[k][1].elapsed_time(evs[k][2]) for k in range(args.steps)]
    t_dec = [evs[k][2].elapsed_time(evs[k][3]) for k in range(args.steps)]
    total_ms = max_over_ranks(sum(t_step), device=dev)
    ms_per_step = total_ms / args.steps
    value = world * step.tokens * args.steps / (total_ms / 1e3)

    # End to end: every step copies its inputs in from pinned host memory and
    # reads its results back.  As in a serving loop the transfers overlap the
    # neighbouring steps' kernels: two buffer sets alternate, inputs travel on
    # an H2D stream, results on a D2H stream, and events order buffer reuse.
    bufs = [step, step.twin()]
    io = [b.host_io() for b in bufs]
    graphs = [graph, capture_step(bufs[1])] if graph is not None else None
    h2d_bytes = sum(x.numel() * x.element_size() for x, _ in io[0][0])
    d2h_bytes = sum(x.numel() * x.element_size() for x, _ in io[0][1])
    e_steps = max(4, min(args.steps, 40))
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    compute = torch.cuda.current_stream()

    def e2e_loop(n):
        done = [torch.cuda.Event() for _ in range(n)]
        got = [torch.cuda.Event() for _ in range(n)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(h2d_s)
        for k in range(n):
            b, (h2d, d2h) = bufs[k % 2], io[k % 2]
            inp = torch.cuda.Event()
            with torch.cuda.stream(h2d_s):
                if k >= 2:
                    h2d_s.wait_event(done[k - 2])      # step k-2 no longer reads this set
                for src, dst in h2d:
                    dst.copy_(src, non_blocking=True)
                inp.record(h2d_s)
            compute.wait_event(inp)
            if k >= 2:
                compute.wait_event(got[k - 2])         # step k-2's results are out
            if graphs is not None:
                graphs[k % 2].replay()
            else:
                b.run()
            done[k].record(compute)
            flush.zero_()
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[k])
                for src, dst in d2h:
                    dst.copy_(src, non_blocking=True)
                got[k].record(d2h_s)
        d2h_s.wait_event(got[n - 1])
        end.record(d2h_s)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    e2e_loop(3)
    barrier()
    torch.cuda.synchronize()
    e_ms = max_over_ranks(e2e_loop(e_steps) / e_steps, device=dev)
    e2e_value = world * step.tokens / (e_ms / 1e3)

    pk = peaks()
    ms_ext = statistics.mean(t_ext)
    ms_dec = statistics.mean(t_dec)
    ms_store = statistics.mean(t_store)
    kernels = {}
    if work["extend_flops"]:
        tf = work["extend_flops"] / (ms_ext / 1e3) / 1e12
        kernels["extend"] = {"ms": round(ms_ext, 4), "tflops": round(tf, 2),
                             "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                             "algorithmic_tflop": round(work["extend_flops"] / 1e12, 4)}
    if work["decode_bytes"]:
        # the roofline counts the bytes the path must read: every key once per
        # request (plain decode), or once per shared group (cascade)
        alg = work["decode_read_once_bytes"] if step.cascade else work["decode_bytes"]
        gbs = alg / (ms_dec / 1e3) / 1e9
        kernels["decode"] = {"ms": round(ms_dec, 4), "gbs": round(gbs, 1),
                             "frac_of_hbm_peak": round(gbs / pk["hbm_gbs"], 4),
                             "algorithmic_gb": round(alg / 1e9, 4),
                             "path": "cascade" if step.cascade else "plain"}
        if step.cascade:
            kernels["decode"]["logical_gb"] = round(work["decode_bytes"] / 1e9, 4)
            kernels["decode"]["logical_gbs"] = round(work["decode_bytes"] / (ms_dec / 1e3) / 1e9, 1)
    gbs_st = work["store_bytes"] / (ms_store / 1e3) / 1e9
    kernels["store_kv"] = {"ms": round(ms_store, 4), "gbs": round(gbs_st, 1),
                           "algorithmic_gb": round(work["store_bytes"] / 1e9, 4)}
    # traffic is looked up per workload and pool type (an e4m3 pool's kernels
    # move other bytes)
    wl = WORKLOAD_NAMES[args.config]
    tkey = wl + ("_fp8" if step.fp8 else "")
    if "decode" in kernels and (ms_dec >= ms_ext or "extend" not in kernels):
        ach = kernels["decode"]["gbs"]
        roof = {"kernel": "cascade decode (plan + groups + split + combine)" if step.cascade
                else "decode (plan + split + combine)", "bound": "hbm", "achieved": ach,
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
                "traffic": measured_traffic("decode", tkey), "peak_source": pk["source"]}
    else:
        ach = kernels["extend"]["tflops"]
        roof = {"kernel": "extend", "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(ach / pk["bf16_tflops"], 4),
                "traffic": measured_traffic("extend", tkey), "peak_source": pk["source"]}
    d = w.dims
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if step.fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": wl + ("(small)" if args.small else ""), "num_q_heads": d.num_q_heads, "num_kv_heads": d.num_kv_heads,
                   "head_dim": d.head_dim, "pool_slots": d.pool_size,
                   "extend_tokens": int(w.extend.total_extend) if w.extend is not None else 0,
                   "decode_requests": int(sum(b.q.shape[0] for b in w.decode)),
                   "query_tokens_per_step": int(step.tokens), "parallelism": f"replicas{world}",
                   "decode_path": ("cascade" if step.cascade else "plain") if w.decode else None,
                   "launch": "cuda_graph" if graph is not None else "eager",
                   "extend_decode_overlap": step.overlap,
                   "kv_cache_dtype": "fp8_e4m3" if step.fp8 else "bf16",
                   "page_size": int(w.recipe.get("page_size", 1)),
                   "prefix_sharing": sharing_of(w),
                   "l2": "flushed between steps (256 MiB write)"},
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d_bytes),
                "d2h_bytes_per_step": int(d2h_bytes), "ms_per_step": round(e_ms, 4),
                "transfers": "each step's inputs H2D from pinned memory and results D2H, overlapped with "
                             "the neighbouring steps' kernels (two buffer sets, H2D and D2H streams)"},
        "gpu_launches": int(launches),
        "roofline": roof,
        "kernels": kernels,
        "eager_ms_per_step": round(statistics.mean(t_eager), 4),
        "clocks": clocks.summary(),
        "wall_s_timed": round(wall, 3),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------------------- CPU oracle

_ORACLE_CACHE: dict = {}

def oracle_sample(config: int, seed: int, budget_s: float, min_tokens: int = 4, max_tokens: int = 100000):
    """Time the fp64 oracle on query tokens drawn uniformly from one step of
    the workload until ``budget_s`` of CPU time has been spent."""
    import oracle
    if config not in _ORACLE_CACHE:
        w0 = W.make(config)
        views = [w0.pool_view(decode_steps=s + 1) for s in range(len(w0.decode))] or [w0.pool_view()]
        _ORACLE_CACHE[config] = (w0, views)
    w, views = _ORACLE_CACHE[config]
    pool = views[-1]
    rng = np.random.default_rng(seed)
    n_ext = w.extend.total_extend if w.extend is not None else 0
    n_dec = [b.q.shape[0] for b in w.decode]
    total = n_ext + sum(n_dec)
    order = rng.permutation(total)
    done, spent = 0, 0.0
    t0 = time.perf_counter()
    for q_idx in order[:max_tokens]:
        a = time.perf_counter()
        if q_idx < n_ext:
            e = w.extend
            oracle.extend_attention(e.q, e.k_new, e.v_new, pool.k, pool.v, w.req_to_token, e.req_pool_idx,
                                    e.prefix_lens, e.extend_lens, w.dims.num_kv_heads, w.dims.sm_scale,
                                    tokens=[int(q_idx)])
        else:
            j = int(q_idx - n_ext)
            s = 0
            while j >= n_dec[s]:
                j -= n_dec[s]
                s += 1
            b = w.decode[s]
            pool_s = views[s]
            oracle.decode_attention(b.q, pool_s.k, pool_s.v, w.req_to_token, b.req_pool_idx, b.seq_lens,
                                    w.dims.num_kv_heads, w.dims.sm_scale, requests=[j])
        spent += time.perf_counter() - a
        done += 1
        if spent >= budget_s and done >= min_tokens:
            break
    return done, spent, time.perf_counter() - t0


def cpu_baseline(config: int, budget_s: float = 15.0):
    """Run the oracle single-threaded in a fresh process (spawned: no GPU
    context is inherited) and report its tokens/s on the sample."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = (f"import sys, json; sys.path.insert(0, {ROOT!r}); import bench; "
            f"d, s, w = bench.oracle_sample({config}, 0, {budget_s}); "
            f"print(json.dumps({{'tokens': d, 'seconds': s}}))")
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=budget_s * 10 + 600)
        res = json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as exc:  # pragma: no cover
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle", "error": str(exc)[:200]}
    return {"value": round(res["tokens"] / res["seconds"], 4), "unit": "tokens/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{res['tokens']} query tokens drawn uniformly from one step of "
                      f"{WORKLOAD_NAMES[config]} (fp64 NumPy, 1 thread, {res['seconds']:.1f} s)"}


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle  # noqa: F401
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for k in range(args.warmup):
        oracle_sample(args.config, 100 + k, per_step / 2, min_tokens=1, max_tokens=2)
    toks, secs = 0, 0.0
    for k in range(args.steps):
        d, s, _ = oracle_sample(args.config, k, per_step, min_tokens=1)
        toks += d
        secs += s
    value = toks / secs
    cores = 1 if os.environ.get("OPENBLAS_NUM_THREADS") == "1" else len(os.sched_getaffinity(0))
    line = {"metric": METRIC, "impl": "reference", "value": round(value, 4), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / args.steps, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAMES[args.config], "parallelism": "cpu"},
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{toks} query tokens over {args.steps} steps, drawn uniformly from "
                                       f"one step of {WORKLOAD_NAMES[args.config]}"},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, choices=sorted(WORKLOAD_NAMES))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="KV pool element type (fp8: e4m3 codes with per-tensor scales)")
    ap.add_argument("--overlap", choices=["on", "off"], default="on",
                    help="run the extend and the decode batches of a step on two streams")
    ap.add_argument("--graph", choices=["on", "off"], default="on",
                    help="time the step replayed as one CUDA graph (per-kernel times stay eager)")
    ap.add_argument("--cascade", choices=["auto", "on", "off"], default="auto",
                    help="decode through shared-prefix groups (auto: when the batch shares prefixes)")
    ap.add_argument("--small", action="store_true",
                    help="reduced pool / batch of the workload, for profiler captures")
    ap.add_argument("--page-size", type=int, default=1,
                    help="requests own whole pages of this many consecutive slots (configs 2 and 3)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.page_size < 1 or (args.page_size > 1 and args.config not in PAGED):
        ap.error(f"--page-size > 1 is built for configs {PAGED}")
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
