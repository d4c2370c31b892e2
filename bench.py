#!/usr/bin/env python3
"""Benchmark: paged decode steps on GB300.

One step = the whole hot path for one layer: the host block manager makes every sequence's
append slot writable (allocating or copy-on-write), the changed block table is uploaded, the
copy-on-write pairs are copied, every sequence's new K/V token is appended, and decode
attention runs over the paged cache.  Positions advance one token per step through a window
of WINDOW steps and then wrap (the later passes re-append the same slots), so every timed step
is a real decode step while per-step inputs stay bounded.

Prints ONE JSON line (rank 0).  ``value`` is achieved HBM GB/s of the attention's algorithmic
bytes (KV attended + q + out + block-table entries used + context_lens) over the whole step
time, with every input resident in HBM; ``e2e`` is the same metric with each step's q/k/v
copied from pinned host memory and the output copied back inside the timed region;
``roofline`` is the decode-attention call alone, timed with CUDA events on its stream.

  python bench.py [--gpus N --steps K --warmup W --config 8b --partition 0]
  python bench.py --impl reference   # the CPU oracle on a bounded sample of the same workload
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WINDOW = 64
E2E_RING = 4          # e2e: device input/output slots in flight (copies of step k overlap steps k-3 .. k-1)
WARM_SECONDS = 0.25   # warm-up runs at least this long (and at least --warmup steps) right before timing
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per decode_kernel launch, from one
# ncu capture of each workload's attention call.  Reported only while the kernel sources hash to
# the version the counters were taken on; null otherwise.
NCU_TRAFFIC = {
    "sources_sha256_16": "44ffaa3d3391f948",
    "8b": 552_095_488, "70b": 543_195_904, "long_quant": 1_076_637_952, "long_quant_tok": 1_093_696_768,
    "prefix_cow": 282_179_072, "int4_8b": 190_577_920, "swa": 1_081_974_272, "tiny": 283_904,
}
KERNEL_SOURCES = ["paged_kv_cache_table_gb300/csrc/decode_attention.cu",
                  "paged_kv_cache_table_gb300/csrc/pa_device.cuh",
                  "paged_kv_cache_table_gb300/csrc/pa_internal.h"]
METRIC = "paged decode attn: achieved HBM GB/s (% of GB300 peak); decode tokens/s/layer"
L2_BYTES = 129 * 1024 * 1024
MODEL_LAYERS = {"8b": 32, "70b": 80}  # decoder layers of the models whose attention shapes these are


def _bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_sources_hash() -> str:
    """First 16 hex digits of the sha256 of the kernel sources with comments and whitespace removed
    (so that documentation edits keep the counters; any code change drops them)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update("".join(src.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    if kernel_sources_hash() != NCU_TRAFFIC["sources_sha256_16"]:
        return None
    return NCU_TRAFFIC.get(workload)


def seq_bytes(w, ctx_s: int) -> int:
    """Algorithmic bytes one sequence contributes to a decode-attention call: its attended K
    and V (sink positions counted at bf16; under a sliding window only the window's positions),
    its q and out rows, the block-table entries it uses and its context length."""
    ctx_s = int(ctx_s)
    lo = max(0, ctx_s - w.window) if w.window else 0
    n_sink = max(0, min(ctx_s, w.num_sink) - lo)
    kv = (ctx_s - lo - n_sink) * w.H_kv * (w.k_row_bytes() + w.kv_row_bytes()) + n_sink * w.H_kv * w.D * 2 * 2
    return kv + 2 * w.H_q * w.D * 2 + (-(-ctx_s // 16) - lo // 16) * 4 + 4


def attention_bytes(w, ctx: np.ndarray) -> int:
    """Algorithmic bytes of one decode-attention call (what must cross HBM at least once)."""
    # per-KV-head fp32 scales read by the call (per-token K scales are in the K row bytes)
    scales = {"e4m3": 2 * w.H_kv * 4, "e4m3_tok": w.H_kv * 4}.get(w.k_dtype, 0)
    return sum(seq_bytes(w, c) for c in np.asarray(ctx)) + scales


# ----------------------------------------------------------------------------------
# distributed helpers (one process per GPU; replicas, no collective on the data path)
# ----------------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max_sum(elapsed_s: float, units: float, backend_device=None):
    """Max of the elapsed times and sum of the units over all ranks (identity at world 1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return elapsed_s, units
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=backend_device)
    u = torch.tensor([units], dtype=torch.float64, device=backend_device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        busy = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------
class DecodeBench:
    """One layer's paged cache and the per-step inputs of a WINDOW-step cycle, on one GPU."""

    def __init__(self, name, device, partition=0, horizon=None, shared=False):
        import torch
        from paged_kv_cache_table_gb300 import native as N
        from paged_kv_cache_table_gb300.workloads import make_workload
        self.torch, self.N = torch, N
        self.dev = device
        self.partition = partition
        w = make_workload(name, steps=WINDOW, **({"horizon": horizon} if horizon else {}))
        self.w = w
        n_slots = w.num_blocks * 16
        if w.k_dtype == "bf16":
            self.k = torch.empty((n_slots, w.H_kv, w.D), dtype=torch.bfloat16, device=device)
            self.v = torch.empty_like(self.k)
        else:  # 8-bit codes (per-token K: then the scales), or int4 codes followed by the group parameters
            self.k = torch.empty(n_slots * w.H_kv * w.k_row_bytes(), dtype=torch.uint8, device=device)
            self.v = torch.empty(n_slots * w.H_kv * w.kv_row_bytes(), dtype=torch.uint8, device=device)
        self.k_scales = None if w.k_scales is None else w.k_scales.to(device)
        self.v_scales = None if w.v_scales is None else w.v_scales.to(device)
        self.k_sink = self.v_sink = None
        if w.num_sink:
            self.k_sink = torch.empty((w.B, w.num_sink, w.H_kv, w.D), dtype=torch.bfloat16, device=device)
            self.v_sink = torch.empty_like(self.k_sink)
        self.desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks, w.k_dtype, w.v_dtype,
                                self.k_scales, self.v_scales, self.k_sink, self.v_sink, w.num_sink,
                                sliding_window=w.window)
        self.tables = w.tables.copy()
        self.tables_dev = torch.from_numpy(self.tables).to(device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.bm = N.BlockManager(w.num_blocks)
        blocks, counts = np.unique(w.tables[w.tables >= 0], return_counts=True)
        owner = 1 if w.prefix else 0  # a cached prefix holds its own reference to its blocks
        for b, c in zip(blocks, counts):
            self.bm.claim(int(b))
            for _ in range(int(c) - 1 + owner):
                self.bm.incref(int(b))
        # cached tokens, appended in bounded chunks
        chunk = 1 << 17
        for a in range(0, len(w.fill_seq), chunk):
            b = min(len(w.fill_seq), a + chunk)
            N.pa_kv_append_tokens(self.desc, self.k, self.v, w.fill_k[a:b].to(device), w.fill_v[a:b].to(device),
                                  b - a, torch.from_numpy(w.fill_seq[a:b]).to(device),
                                  torch.from_numpy(w.fill_pos[a:b]).to(device), self.tables_dev, self.err)
        if w.prefix:
            self._fork_and_fill_suffixes()
        torch.cuda.synchronize()
        # per-step inputs, resident
        self.q = w.q.to(device)
        self.k_new = w.k_new.to(device)
        self.v_new = w.v_new.to(device)
        self.pos = [w.positions(i) for i in range(WINDOW)]
        self.ctx = [w.context_lens(i) for i in range(WINDOW)]
        self.pos_dev = torch.from_numpy(np.stack(self.pos)).to(device)
        self.ctx_dev = torch.from_numpy(np.stack(self.ctx)).to(device)
        self.max_ctx = int(max(c.max() for c in self.ctx))
        self.ws_bytes = N.pa_decode_workspace_size(self.desc, self.max_ctx, partition)
        # shared: the prefix's whole blocks attended once for all sequences (pa_decode_attention_shared)
        self.shared = bool(shared and w.prefix)
        if self.shared:
            self.shared_len = w.prefix - w.prefix % 16
            self.shared_seqs = torch.arange(w.B, dtype=torch.int32, device=device)
            self.ws_bytes = N.pa_decode_shared_workspace_size(self.desc, self.max_ctx, partition, self.shared_len)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.out = torch.empty((w.B, w.H_q, w.D), dtype=torch.bfloat16, device=device)
        self.step_bytes = [attention_bytes(w, c) for c in self.ctx]
        # pinned staging for table uploads (one slot per step of a cycle) and e2e buffers
        self.tab_ring = [torch.empty(self.tables.shape, dtype=torch.int32).pin_memory() for _ in range(WINDOW)]
        self.pair_ring = [torch.empty((w.B, 2), dtype=torch.int32).pin_memory() for _ in range(WINDOW)]
        self.pairs_dev = torch.empty((w.B, 2), dtype=torch.int32, device=device)
        # e2e: each step's q, k_new, v_new packed into one pinned row (one upload per step),
        # two device copies of that row and of the output, drained by a copy stream
        nq, nk = w.B * w.H_q * w.D, w.B * w.H_kv * w.D
        self.in_elems = nq + 2 * nk
        h_in = torch.empty((WINDOW, self.in_elems), dtype=torch.bfloat16)
        h_in[:, :nq] = w.q.reshape(WINDOW, nq)
        h_in[:, nq:nq + nk] = w.k_new.reshape(WINDOW, nk)
        h_in[:, nq + nk:] = w.v_new.reshape(WINDOW, nk)
        self.h_in = [r for r in h_in.pin_memory()]
        self.h_out = [r for r in torch.empty((WINDOW, w.B, w.H_q, w.D), dtype=torch.bfloat16).pin_memory()]
        self.d_in = [torch.empty(self.in_elems, dtype=torch.bfloat16, device=device) for _ in range(E2E_RING)]
        self.d_views = [(d[:nq].view(w.B, w.H_q, w.D), d[nq:nq + nk].view(w.B, w.H_kv, w.D),
                         d[nq + nk:].view(w.B, w.H_kv, w.D)) for d in self.d_in]
        self.d_out = [torch.empty_like(self.out) for _ in range(E2E_RING)]
        self.host_s = 0.0
        self.warm_steps = 0
        self._touch_pinned()
        # raw device pointers for the per-step calls (the binding takes ints as pointers)
        P = lambda t: t.data_ptr()
        self.ptr = dict(k=P(self.k), v=P(self.v), tab=P(self.tables_dev), ws=P(self.ws), err=P(self.err),
                        out=P(self.out))
        self.ptr_step = [(P(self.q[j]), P(self.k_new[j]), P(self.v_new[j]), P(self.pos_dev[j]), P(self.ctx_dev[j]))
                         for j in range(WINDOW)]
        self.ptr_e2e = [tuple(P(t) for t in v) + (P(o),) for v, o in zip(self.d_views, self.d_out)]
        self.launches_per_step = 3  # append + attention + merge (plus a copy kernel on CoW steps)
        self.cow_launches = 0

    def _touch_pinned(self):
        """Move every pinned staging slot through a copy once during set-up: the first copy from or
        to a pinned page costs far more than the later ones (measured, a first pass through the
        ring slots made the GPU wait on the host), and the timed steps should see the steady
        state a serving loop reaches after its first steps."""
        torch = self.torch
        scratch_tab = torch.empty(self.tables.shape, dtype=torch.int32, device=self.dev)
        scratch_pairs = torch.empty_like(self.pairs_dev)
        for j in range(WINDOW):
            self.tab_ring[j].numpy()[...] = self.tables
            scratch_tab.copy_(self.tab_ring[j], non_blocking=True)
            scratch_pairs.copy_(self.pair_ring[j], non_blocking=True)
            self.d_in[j % E2E_RING].copy_(self.h_in[j], non_blocking=True)
            self.h_out[j].copy_(self.d_out[j % E2E_RING], non_blocking=True)
        torch.cuda.synchronize()

    def warm(self, warmup, stream):
        """Untimed steps right before a timed region: at least `warmup` of them and at least
        WARM_SECONDS of wall time, so that the timed steps start from steady clocks and a full
        queue of work rather than from a GPU that has been idle.  Returns the next step index."""
        i = 0
        t0 = time.perf_counter()
        while i < warmup or time.perf_counter() - t0 < WARM_SECONDS:
            self.step(i, stream)
            i += 1
            if i % 64 == 0:
                self.torch.cuda.synchronize()
        self.torch.cuda.synchronize()
        self.warm_steps = i
        return i

    def _fork_and_fill_suffixes(self):
        """Prefix workload set-up: every sequence writes its private suffix after the shared
        prefix.  The first suffix token lands in the shared, partly filled prefix block, so the
        block manager copy-on-writes it for every sequence (the fork); the later tokens open
        private blocks.  Afterwards the timed steps append at prefix + suffix length."""
        torch, N, w, dev = self.torch, self.N, self.w, self.dev
        lens = w.suffix_len.astype(np.int64)
        self.fork_pairs = 0
        for p in range(w.prefix, w.prefix + int(lens.max())):
            pos = np.where(p < w.prefix + lens, p, -1).astype(np.int32)
            pairs, changed = self.bm.prepare_step(self.tables, pos)
            if changed:
                self.tables_dev.copy_(torch.from_numpy(self.tables))
            if len(pairs):
                N.pa_block_copy(self.desc, self.k, self.v, torch.from_numpy(pairs).to(dev), len(pairs), self.err)
                self.fork_pairs += len(pairs)
        seq = np.repeat(np.arange(w.B, dtype=np.int32), lens)
        pos = np.concatenate([np.arange(w.prefix, w.prefix + n, dtype=np.int32) for n in lens])
        N.pa_kv_append_tokens(self.desc, self.k, self.v, w.suffix_k.to(dev), w.suffix_v.to(dev), len(seq),
                              torch.from_numpy(seq).to(dev), torch.from_numpy(pos).to(dev), self.tables_dev,
                              self.err)
        w.ctx_old = (w.prefix + lens).astype(np.int32)
        # bytes the attention reads once from DRAM: the shared prefix blocks count once
        self.shared_tokens = w.prefix - (w.prefix % 16)

    def unique_bytes(self, ctx):
        """Prefix workload: algorithmic bytes with the shared full prefix blocks counted once."""
        w = self.w
        per_tok = w.H_kv * w.D * w.kv_elem_bytes() * 2
        return attention_bytes(w, ctx) - (w.B - 1) * self.shared_tokens * per_tok

    def step(self, i, stream, ev=None, buf=None):
        """One decode step on `stream`.  `buf` selects a double-buffered e2e input/output slot
        (default: the resident inputs of this step); `ev` = events around the attention call."""
        N, w, P = self.N, self.w, self.ptr
        j = i % WINDOW
        pairs, changed = self.bm.prepare_step(self.tables, self.pos[j])
        if changed:
            self.tab_ring[j].numpy()[...] = self.tables
            self.tables_dev.copy_(self.tab_ring[j], non_blocking=True)
        if len(pairs):
            self.pair_ring[j].numpy()[:len(pairs)] = pairs
            self.pairs_dev[:len(pairs)].copy_(self.pair_ring[j][:len(pairs)], non_blocking=True)
            N.pa_block_copy(self.desc, self.k, self.v, self.pairs_dev, len(pairs), self.err, stream)
            self.cow_launches += 1
        q, kn, vn, pos, ctx = self.ptr_step[j]
        out = P["out"]
        if buf is not None:
            q, kn, vn, out = self.ptr_e2e[buf]
        if self.shared:
            N.pa_kv_append(self.desc, P["k"], P["v"], kn, vn, P["tab"], pos, P["err"], stream)
            if ev is not None:
                ev[0].record()
            N.pa_decode_attention_shared(self.desc, out, q, P["k"], P["v"], P["tab"], ctx, self.max_ctx, w.scale,
                                         self.partition, self.shared_seqs.data_ptr(), w.B, self.shared_len, P["ws"],
                                         self.ws_bytes, P["err"], stream)
            if ev is not None:
                ev[1].record()
            return
        if ev is None:
            # the step as one call: the append overlaps the attention's streaming of other blocks
            N.pa_decode_step(self.desc, out, q, P["k"], P["v"], kn, vn, P["tab"], pos, ctx, self.max_ctx, w.scale,
                             self.partition, P["ws"], self.ws_bytes, P["err"], stream)
            return
        N.pa_kv_append(self.desc, P["k"], P["v"], kn, vn, P["tab"], pos, P["err"], stream)
        ev[0].record()
        N.pa_decode_attention(self.desc, out, q, P["k"], P["v"], P["tab"], ctx, self.max_ctx, w.scale,
                              self.partition, P["ws"], self.ws_bytes, P["err"], stream)
        ev[1].record()

    def run(self, steps, warmup, per_call_events=False):
        """Device-resident steps.  Returns (elapsed_s, attention_ms_per_call or None, bytes)."""
        torch = self.torch
        sid = torch.cuda.current_stream().cuda_stream
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)] if per_call_events else None
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        first = self.warm(warmup, sid)
        barrier(self.dev)
        torch.cuda.synchronize()
        self.first_step = first
        self.cow_launches = 0
        t0.record()
        nbytes = 0
        h0 = time.perf_counter()
        for k in range(steps):
            i = first + k
            self.step(i, sid, ev=None if evs is None else evs[k])
            nbytes += self.step_bytes[i % WINDOW]
        self.host_s = time.perf_counter() - h0
        t1.record()
        torch.cuda.synchronize()
        barrier(self.dev)
        elapsed = t0.elapsed_time(t1) / 1e3
        att = None if evs is None else [a.elapsed_time(b) for a, b in evs]
        return elapsed, att, nbytes

    def run_e2e(self, steps, warmup):
        """Steps fed from pinned host memory: a copy stream uploads step k's q/k/v into one of
        E2E_RING device slots and downloads the output of the step that last used that slot,
        while the compute stream runs the steps before k; every copy of every timed step is
        inside the timed region, and the region ends when the last output is back in host
        memory."""
        torch = self.torch
        comp = torch.cuda.current_stream()
        copy = torch.cuda.Stream()
        R = E2E_RING
        in_ready = [torch.cuda.Event() for _ in range(R)]
        done = [torch.cuda.Event() for _ in range(R)]
        pending = {}

        def issue(k, i):
            b = k % R
            j = i % WINDOW
            with torch.cuda.stream(copy):
                if b in pending:
                    copy.wait_event(done[b])  # the step that used slot b consumed its input, wrote out[b]
                    self.h_out[pending.pop(b)].copy_(self.d_out[b], non_blocking=True)
                self.d_in[b].copy_(self.h_in[j], non_blocking=True)
                in_ready[b].record(copy)
            comp.wait_event(in_ready[b])
            self.step(i, comp.cuda_stream, buf=b)
            done[b].record(comp)
            pending[b] = j

        def drain():
            with torch.cuda.stream(copy):
                for b in sorted(pending):
                    copy.wait_event(done[b])
                    self.h_out[pending[b]].copy_(self.d_out[b], non_blocking=True)
            pending.clear()

        # warm-up through the same pipeline, then the timed steps
        k, t_w = 0, time.perf_counter()
        while k < warmup or time.perf_counter() - t_w < WARM_SECONDS:
            issue(k, k)
            k += 1
            if k % 64 == 0:
                drain()
                torch.cuda.synchronize()
        drain()
        torch.cuda.synchronize()
        first = k
        barrier(self.dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(comp)
        copy.wait_event(t0)
        nbytes = 0
        h0 = time.perf_counter()
        for k in range(steps):
            issue(k, first + k)
            nbytes += self.step_bytes[(first + k) % WINDOW]
        drain()
        self.host_s = time.perf_counter() - h0
        comp.wait_stream(copy)
        t1.record(comp)
        torch.cuda.synchronize()
        barrier(self.dev)
        return t0.elapsed_time(t1) / 1e3, nbytes


class SlidingBench(DecodeBench):
    """Sliding-window decode: positions keep advancing (no wrap-around), every step makes the
    append slot writable, appends, attends over the window and then releases the blocks behind
    it (pa_bm_slide_window), so the pool holds O(window) blocks per sequence however long the
    sequences grow.  The table goes up whenever a step changed it (an allocation or a release);
    q/k/v reuse a WINDOW-step ring of inputs."""

    def __init__(self, name, device, horizon):
        super().__init__(name, device, 0, horizon=horizon)
        torch, w = self.torch, self.w
        self.horizon = horizon
        self.t = 0
        self.dirty = False
        self.pos_all = [(w.ctx_old + t).astype(np.int32) for t in range(horizon)]
        self.ctx_all = [(w.ctx_old + t + 1).astype(np.int32) for t in range(horizon)]
        self.pos_all_dev = torch.from_numpy(np.stack(self.pos_all)).to(device)
        self.ctx_all_dev = torch.from_numpy(np.stack(self.ctx_all)).to(device)
        self.max_ctx = int(self.ctx_all[-1].max())
        self.ws_bytes = self.N.pa_decode_workspace_size(self.desc, self.max_ctx, 0)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.ptr["ws"] = self.ws.data_ptr()
        self.tab_ev = [None] * WINDOW
        self.uploads = 0
        self.held_blocks_max = 0

    def bytes_at(self, t):
        return attention_bytes(self.w, self.ctx_all[t])

    def step(self, i, stream, ev=None, buf=None):
        torch, N, w, P = self.torch, self.N, self.w, self.ptr
        t = self.t
        if t >= self.horizon:
            raise RuntimeError("sliding bench ran past its horizon")
        self.t += 1
        j = t % WINDOW
        pairs, changed = self.bm.prepare_step(self.tables, self.pos_all[t])
        if len(pairs):
            raise RuntimeError("unexpected copy-on-write in the sliding-window workload")
        if changed or self.dirty:
            if self.tab_ev[j] is not None:
                self.tab_ev[j].synchronize()  # the copy that last read this pinned slot is done
            self.tab_ring[j].numpy()[...] = self.tables
            self.tables_dev.copy_(self.tab_ring[j], non_blocking=True)
            self.tab_ev[j] = torch.cuda.Event()
            self.tab_ev[j].record()
            self.uploads += 1
        q, kn, vn = self.ptr_step[j][:3]
        pos = self.pos_all_dev[t].data_ptr()
        ctx = self.ctx_all_dev[t].data_ptr()
        if ev is None:
            N.pa_decode_step(self.desc, P["out"], q, P["k"], P["v"], kn, vn, P["tab"], pos, ctx, self.max_ctx,
                             w.scale, 0, P["ws"], self.ws_bytes, P["err"], stream)
        else:
            N.pa_kv_append(self.desc, P["k"], P["v"], kn, vn, P["tab"], pos, P["err"], stream)
            ev[0].record()
            N.pa_decode_attention(self.desc, P["out"], q, P["k"], P["v"], P["tab"], ctx, self.max_ctx, w.scale,
                                  0, P["ws"], self.ws_bytes, P["err"], stream)
            ev[1].record()
        released, _ = self.bm.slide_window(self.tables, self.ctx_all[t], w.window)
        self.dirty = released > 0
        self.held_blocks_max = max(self.held_blocks_max, w.num_blocks - self.bm.num_free())

    def run(self, steps, warmup, per_call_events=False):
        torch = self.torch
        sid = torch.cuda.current_stream().cuda_stream
        for i in range(warmup):
            self.step(i, sid)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)] if per_call_events else None
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        first = self.t
        t0.record()
        for k in range(steps):
            self.step(k, sid, ev=None if evs is None else evs[k])
        t1.record()
        torch.cuda.synchronize()
        nbytes = sum(self.bytes_at(t) for t in range(first, first + steps))
        att = None if evs is None else [a.elapsed_time(b) for a, b in evs]
        return t0.elapsed_time(t1) / 1e3, att, nbytes


class PrefillBench:
    """Chunked-prefill row: each step appends every sequence's chunk of new K/V tokens and runs
    causal prefill attention of the chunk's queries over the paged cache.  kind "fp8": the cache
    holds E4M3 K / INT8 V with per-head scales from the data's absmax (decoded block by block)."""

    def __init__(self, device, kind="bf16"):
        import torch
        from paged_kv_cache_table_gb300 import native as N
        from paged_kv_cache_table_gb300.workloads import make_prefill_workload
        self.torch, self.N = torch, N
        w = make_prefill_workload()
        self.w = w
        shape = (w.num_blocks * 16, w.H_kv, w.D)
        if kind == "bf16":
            self.k = torch.empty(shape, dtype=torch.bfloat16, device=device)
            self.v = torch.empty(shape, dtype=torch.bfloat16, device=device)
            self.desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks)
        else:
            self.k = torch.empty(shape, dtype=torch.uint8, device=device)
            self.v = torch.empty(shape, dtype=torch.uint8, device=device)
            kk, vv = torch.cat([w.fill_k, w.new_k]).float().abs(), torch.cat([w.fill_v, w.new_v]).float().abs()
            self.k_scales = (kk.amax(dim=(0, 2)) / 448.0).to(device)
            self.v_scales = (vv.amax(dim=(0, 2)) / 127.0).to(device)
            self.desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks, "e4m3", "int8",
                                    self.k_scales, self.v_scales)
        self.tables = torch.from_numpy(w.tables).to(device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        N.pa_kv_append_tokens(self.desc, self.k, self.v, w.fill_k.to(device), w.fill_v.to(device), len(w.fill_seq),
                              torch.from_numpy(w.fill_seq).to(device), torch.from_numpy(w.fill_pos).to(device),
                              self.tables, self.err)
        self.new_k, self.new_v = w.new_k.to(device), w.new_v.to(device)
        self.new_seq = torch.from_numpy(w.new_seq).to(device)
        self.new_pos = torch.from_numpy(w.new_pos).to(device)
        self.q = w.q.to(device)
        self.q_start = torch.from_numpy(w.q_start()).to(device)
        self.ctx = torch.from_numpy(w.context_lens()).to(device)
        self.out = torch.empty_like(self.q)
        self.max_q = int(w.chunk.max())
        ctx, n = w.context_lens().astype(np.int64), w.chunk.astype(np.int64)
        # causal (query, key) pairs: the query at position p reads p + 1 keys
        pairs = sum(int(((c - m + 1) + c) * m // 2) for c, m in zip(ctx, n))
        self.flops = 4 * w.D * w.H_q * pairs
        self.tokens = int(n.sum())

    def step(self, stream):
        N, w = self.N, self.w
        N.pa_prefill_step(self.desc, self.out, self.q, self.k, self.v, self.new_k, self.new_v, self.tokens,
                          self.new_seq, self.new_pos, self.tables, self.q_start, self.ctx, self.max_q, w.scale,
                          self.err, stream)

    def run(self, steps, warmup):
        torch = self.torch
        sid = torch.cuda.current_stream().cuda_stream
        for _ in range(warmup):
            self.step(sid)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            self.step(sid)
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / 1e3 / steps

    def run_attention(self, steps, warmup, ws=False):
        """Seconds per prefill-attention call alone (the cache already holds the chunk), timed with
        CUDA events on the stream the kernel is launched on.  ws: through pa_prefill_attention_ws
        (each attended block decoded once into a workspace, then the bf16 tensor-core path)."""
        torch, N, w = self.torch, self.N, self.w
        sid = torch.cuda.current_stream().cuda_stream
        max_ctx = int(w.max_blocks * 16)
        nbytes = N.pa_prefill_workspace_size(self.desc, max_ctx) if ws else 0
        wsbuf = torch.empty(max(1, nbytes), dtype=torch.uint8, device=self.out.device) if ws else None

        def call():
            if ws:
                N.pa_prefill_attention_ws(self.desc, self.out, self.q, self.k, self.v, self.tables, self.q_start,
                                          self.ctx, self.max_q, max_ctx, w.scale, wsbuf, nbytes, self.err, sid)
            else:
                N.pa_prefill_attention(self.desc, self.out, self.q, self.k, self.v, self.tables, self.q_start,
                                       self.ctx, self.max_q, w.scale, self.err, sid)
        for _ in range(warmup):
            call()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            call()
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / 1e3 / steps


def prefix_cache_row(device, warmup):
    """Prefix-cache row: host cost of a lookup (hash chain + match + release through the binding)
    against a cache of 64 distinct 2048-token prompts (8192 entries), and the prefill-attention
    time of 8 requests that hit (128 new tokens over a 2048-token cached prefix) against the same
    requests missing (all 2176 tokens prefilled)."""
    import torch
    from paged_kv_cache_table_gb300 import native as N
    from paged_kv_cache_table_gb300.workloads import make_prefill_workload
    rng = np.random.default_rng(20268)
    n_prompts, plen, qlen = 64, 2048, 128
    bm = N.BlockManager(n_prompts * plen // 16 + 1024)
    pc = N.PrefixCache(bm)
    prompts = [rng.integers(0, 128000, plen).astype(np.int32) for _ in range(n_prompts)]
    width = (plen + qlen) // 16 + 1
    for pr in prompts:
        d = N.block_hashes(pr)
        row = np.full(width, -1, dtype=np.int32)
        for i in range(len(d)):
            row[i] = bm.alloc()
        pc.insert(d, row, len(d))
        bm.release(row, width)
    reqs = [np.concatenate([prompts[i % n_prompts], rng.integers(0, 128000, qlen).astype(np.int32)])
            for i in range(512)]
    hits = 0
    t0 = time.perf_counter()
    for r in reqs:
        d = N.block_hashes(r)
        row = np.full(width, -1, dtype=np.int32)
        hits += pc.match(d, (len(r) - 1) // 16, row)
        bm.release(row, width)
    host_us = (time.perf_counter() - t0) / len(reqs) * 1e6
    t0 = time.perf_counter()
    for r in reqs[:128]:
        N.block_hashes(r)
    hash_us = (time.perf_counter() - t0) / 128 * 1e6
    entries = len(pc)
    pc.close()
    del bm

    def prefill_ms(cached, chunk):
        w = make_prefill_workload(B=8, cached_list=[cached] * 8, chunk_list=[chunk] * 8, seed=20269)
        shape = (w.num_blocks * 16, w.H_kv, w.D)
        k = torch.empty(shape, dtype=torch.bfloat16, device=device)
        v = torch.empty(shape, dtype=torch.bfloat16, device=device)
        desc = N.make_desc(w.B, w.H_q, w.H_kv, w.D, w.num_blocks, w.max_blocks)
        tab = torch.from_numpy(w.tables).to(device)
        err = torch.zeros(1, dtype=torch.int32, device=device)
        allk = torch.cat([w.fill_k, w.new_k]) if len(w.fill_seq) else w.new_k
        allv = torch.cat([w.fill_v, w.new_v]) if len(w.fill_seq) else w.new_v
        seq = np.concatenate([w.fill_seq, w.new_seq]).astype(np.int32)
        pos = np.concatenate([w.fill_pos, w.new_pos]).astype(np.int32)
        N.pa_kv_append_tokens(desc, k, v, allk.to(device), allv.to(device), len(seq),
                              torch.from_numpy(seq).to(device), torch.from_numpy(pos).to(device), tab, err)
        q = w.q.to(device)
        out = torch.empty_like(q)
        qs = torch.from_numpy(w.q_start()).to(device)
        ctx = torch.from_numpy(w.context_lens()).to(device)
        for _ in range(max(3, warmup)):
            N.pa_prefill_attention(desc, out, q, k, v, tab, qs, ctx, chunk, w.scale, err)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        e0.record()
        for _ in range(reps):
            N.pa_prefill_attention(desc, out, q, k, v, tab, qs, ctx, chunk, w.scale, err)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps, int(err.item())

    hit_ms, e_hit = prefill_ms(plen, qlen)
    miss_ms, e_miss = prefill_ms(0, plen + qlen)
    return {"workload": f"cache of {n_prompts} x {plen}-token prompts ({entries} entries); requests = a cached "
                        f"prompt + {qlen} new tokens; prefill of 8 such requests, 32/8 heads, d 128",
            "host_us_per_lookup": round(host_us, 2), "host_us_per_hash_chain": round(hash_us, 2),
            "blocks_hit_per_request": round(hits / len(reqs), 2),
            "prefill_attention_ms_hit": round(hit_ms, 4), "prefill_attention_ms_miss": round(miss_ms, 4),
            "prefill_attention_speedup": round(miss_ms / hit_ms, 2), "err_flag": e_hit | e_miss}


def cpu_model() -> str:
    """The host CPU's name as /proc/cpuinfo gives it (model name on x86, implementer/part on Arm)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown"
    for line in info.splitlines():
        if line.lower().startswith("model name"):
            return line.split(":", 1)[1].strip()
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = (x.strip() for x in line.split(":", 1))
            fields.setdefault(k, v)
    if "CPU implementer" in fields:
        return f"arm implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return "unknown"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_throughput(name, workers, steps=None, warmup=0, budget_s=None):
    """The oracle, as it stands, on this host's cores: `workers` spawned processes (one thread each)
    split the workload's sequences between them (sequence s goes to worker s % workers) and run
    whole decode steps of their sequences (copy-on-write decision, append, gather through the
    table, attention of every query head), all at once.

    steps given: `warmup` untimed steps, then `steps` timed steps of every sequence (the same
    work per step as one GPU step).  budget_s given: sequence-steps, round-robin over the
    worker's sequences, for about budget_s seconds (a bounded sample).
    Returns bytes, seconds (the slowest worker's), sequence-steps and the sample's description."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    start = ctx.Event()
    q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(name, w, workers, steps, warmup, budget_s, start, q))
             for w in range(workers)]
    for p in procs:
        p.start()
    for _ in range(workers):
        msg = q.get(timeout=900)
        if msg != "ready":
            raise RuntimeError(f"oracle worker failed: {msg}")
    start.set()
    res = [q.get(timeout=1800) for _ in range(workers)]
    for p in procs:
        p.join(timeout=120)
    bad = [r for r in res if "error" in r]
    if bad:
        raise RuntimeError(f"oracle worker failed: {bad[0]['error']}")
    return {"bytes": sum(r["bytes"] for r in res), "seconds": max(r["seconds"] for r in res),
            "seq_steps": sum(r["seq_steps"] for r in res), "workers": workers}


def _oracle_worker(name, worker, workers, steps, warmup, budget_s, start, q):
    try:
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
        import torch
        torch.set_num_threads(1)
        import oracle as O
        from paged_kv_cache_table_gb300.workloads import bf16_bits, make_workload
        n_steps = WINDOW if steps is None else min(WINDOW, steps + warmup)
        w = make_workload(name, steps=n_steps)
        if w.prefix:
            raise ValueError("the oracle baseline covers workloads without a shared prefix")
        mine = [s for s in range(w.B) if s % workers == worker]
        ks = None if w.k_scales is None else w.k_scales.numpy()
        vs = None if w.v_scales is None else w.v_scales.numpy()
        cache = O.PagedKVCache(w.num_blocks, w.H_kv, w.D, k_dtype=w.k_dtype, v_dtype=w.v_dtype, k_scales=ks,
                               v_scales=vs, num_seqs=w.B, num_sink=w.num_sink)
        pool = O.BlockPool(w.num_blocks)
        for b in np.unique(w.tables[w.tables >= 0]):
            pool.claim(int(b))
        tables = w.tables.astype(np.int64).copy()
        kb_all, vb_all = bf16_bits(w.fill_k), bf16_bits(w.fill_v)
        for i in np.nonzero(np.isin(w.fill_seq, mine))[0]:
            s = int(w.fill_seq[i])
            cache.append(s, tables[s], int(w.fill_pos[i]), kb_all[i], vb_all[i])
        qs = [O.bf16_bits_to_f64(bf16_bits(w.q[j])) for j in range(n_steps)]
        kn = [bf16_bits(w.k_new[j]) for j in range(n_steps)]
        vn = [bf16_bits(w.v_new[j]) for j in range(n_steps)]

        def seq_step(i, s):
            j = i % n_steps
            pos, ctx = int(w.ctx_old[s]) + j, int(w.ctx_old[s]) + j + 1
            act = pool.prepare_append(tables[s], pos)
            if act[0] == "copy":
                cache.block_copy(act[1], act[2])
            cache.append(s, tables[s], pos, kn[j][s], vn[j][s])
            K, V = cache.gather(s, tables[s], ctx, O.window_start(ctx, w.window))
            O.decode_attention(qs[j][s], K, V, w.scale)
            return seq_bytes(w, ctx)

        q.put("ready")
        start.wait()
        nbytes, n, secs = 0, 0, 0.0
        if steps is not None:
            for i in range(warmup):
                for s in mine:
                    seq_step(i, s)
            t0 = time.perf_counter()
            for i in range(warmup, warmup + steps):
                for s in mine:
                    nbytes += seq_step(i, s)
                    n += 1
            secs = time.perf_counter() - t0
        else:
            t0 = time.perf_counter()
            while mine and secs < budget_s:
                nbytes += seq_step(n // len(mine), mine[n % len(mine)])
                n += 1
                secs = time.perf_counter() - t0
        q.put({"bytes": nbytes, "seconds": secs, "seq_steps": n})
    except Exception as e:  # reported to the parent, which raises
        q.put({"error": repr(e)})


def cpu_baseline(name, budget_s):
    """The oracle timed on all host cores and on one, each on a bounded sample of the workload."""
    cores = host_cores()
    workers = min(cores, 64)
    allc = oracle_throughput(name, workers, budget_s=budget_s)
    one = oracle_throughput(name, 1, budget_s=budget_s)
    desc = "sequence-steps (copy-on-write decision, append, gather, attention of every query head) of the {} workload, " \
           "round-robin over its sequences, fp64 numpy oracle, {}"
    return {"value": round(allc["bytes"] / allc["seconds"] / 1e9, 6), "unit": "GB/s", "cores": workers,
            "kind": "oracle",
            "sample": f"{allc['seq_steps']} " + desc.format(name, f"{workers} processes x 1 thread, ~{budget_s:.0f} s"),
            "single_thread": {"value": round(one["bytes"] / one["seconds"] / 1e9, 6), "unit": "GB/s", "cores": 1,
                              "sample": f"{one['seq_steps']} " + desc.format(name, f"1 thread, ~{budget_s:.0f} s")},
            "nproc": os.cpu_count(), "cpu_model": cpu_model()}


def run_reference(args):
    """The reference arm: the oracle, as it stands, on every host core, running whole decode steps
    of the same workload as the GPU arm (every sequence of --config per step)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    workers = min(host_cores(), 64)
    r = oracle_throughput(args.config, workers, steps=args.steps, warmup=args.warmup)
    value = r["bytes"] / r["seconds"] / 1e9
    sample = (f"{args.steps} whole decode steps ({r['seq_steps']} sequence-steps) of the {args.config} workload after "
              f"{args.warmup} untimed ones, fp64 numpy oracle, {workers} processes x 1 thread")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * r["seconds"] / max(1, args.steps), 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.config, "oracle": "CPU fp64 numpy", "same_steps_as_gpu_arm": True},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": workers, "kind": "oracle",
                             "sample": sample, "nproc": os.cpu_count(), "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_native(args):
    import torch
    import torch.distributed as dist
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=device)
    from paged_kv_cache_table_gb300.build import build
    if rank == 0:
        build()
    barrier(device)
    peak, peak_kind = _peaks()

    b = DecodeBench(args.config, device, args.partition)
    w = b.w
    # device-resident steps (value), clocks sampled meanwhile
    with ClockSampler(local) as cs:
        elapsed, _, nbytes = b.run(args.steps, args.warmup)
    clocks = cs.summary()
    host_ms = 1e3 * b.host_s / args.steps
    cow_launches = b.cow_launches
    warm_steps = b.warm_steps
    # the same steps with CUDA events around every attention call (roofline of the kernel)
    # (at least 200 calls: with a short --steps the mean would carry the first calls' ramp)
    n_calls = max(args.steps, 200)
    _, att_ms, nbytes_ev = b.run(n_calls, args.warmup, per_call_events=True)
    el_max, bytes_all = reduce_max_sum(elapsed, nbytes, device)
    value = bytes_all / el_max / 1e9
    ms_per_step = 1e3 * el_max / args.steps
    tok_s_layer = ws * w.B * args.steps / el_max
    att_mean_ms = float(np.mean(att_ms))
    att_pct = {k: round(float(np.percentile(att_ms, q)), 5) for k, q in (("p10", 10), ("median", 50), ("p90", 90))}
    att_bytes = nbytes_ev / n_calls
    achieved = att_bytes / (att_mean_ms / 1e3) / 1e9
    # end-to-end through the same API with host buffers
    el_e2e, nbytes_e2e = b.run_e2e(args.steps, args.warmup)
    host_ms_e2e = 1e3 * b.host_s / args.steps
    el_e2e, bytes_e2e = reduce_max_sum(el_e2e, nbytes_e2e, device)
    h2d = (w.B * w.H_q * w.D + 2 * w.B * w.H_kv * w.D) * 2
    d2h = w.B * w.H_q * w.D * 2
    err = int(b.err.item())

    def measure_decode(name):
        nb = DecodeBench(name, device, args.partition)
        n2 = max(50, args.steps // 4)
        e2, _, by2 = nb.run(n2, args.warmup)
        _, a2, by_ev = nb.run(n2, args.warmup, per_call_events=True)
        a_ms = float(np.mean(a2))
        ab = by_ev / len(a2)
        if nb.w.prefix:
            ub = float(np.mean([nb.unique_bytes(nb.ctx[(nb.first_step + k) % WINDOW]) for k in range(len(a2))]))
            extra_prefix = {"unique_bytes_per_call": int(ub),
                            "attention_gbs_unique": round(ub / (a_ms / 1e3) / 1e9, 1),
                            "fork_copy_pairs": nb.fork_pairs}
            sb = DecodeBench(name, device, args.partition, shared=True)
            e3, _, _ = sb.run(n2, args.warmup)
            _, a3, _ = sb.run(n2, args.warmup, per_call_events=True)
            s_ms = float(np.mean(a3))
            ub3 = float(np.mean([sb.unique_bytes(sb.ctx[(sb.first_step + k) % WINDOW]) for k in range(len(a3))]))
            extra_prefix["shared_prefix"] = {
                "path": f"pa_decode_attention_shared over the {sb.shared_len} shared positions of all {sb.w.B} "
                        "sequences (prefix kernel + decode of the private positions + merge), after pa_kv_append",
                "attention_ms_per_call": round(s_ms, 5),
                "attention_gbs_unique": round(ub3 / (s_ms / 1e3) / 1e9, 1),
                "attention_frac_unique": round(ub3 / (s_ms / 1e3) / 1e9 / peak, 4),
                "ms_per_step": round(1e3 * e3 / len(a3), 4),
                "tokens_per_s_per_layer": round(sb.w.B * len(a3) / e3, 1),
                "err_flag": int(sb.err.item())}
            del sb
        else:
            extra_prefix = {}
        r = {**extra_prefix, "value": round(by2 / e2 / 1e9, 1), "unit": "GB/s",
             "algorithmic_bytes_per_call": int(ab), "ncu_traffic_per_call": ncu_traffic(name),
             "attention_gbs": round(ab / (a_ms / 1e3) / 1e9, 1),
             "attention_frac": round(ab / (a_ms / 1e3) / 1e9 / peak, 4),
             "attention_ms_per_call": round(a_ms, 5),
             "ms_per_step": round(1e3 * e2 / len(a2), 4),
             "tokens_per_s_per_layer": round(nb.w.B * len(a2) / e2, 1),
             "err_flag": int(nb.err.item())}
        layers = MODEL_LAYERS.get(name)
        if layers:  # the whole model's attention, one such layer after another
            r[f"tokens_per_s_model_{layers}_layers"] = round(nb.w.B * len(a2) / e2 / layers, 1)
        del nb
        torch.cuda.empty_cache()
        return r

    extra = {}
    if args.also and args.also != "none" and rank == 0:
        for name in args.also.split(","):
            extra[name] = measure_decode(name)

    next_rows = {}
    if rank == 0 and not args.no_next:
        pb = PrefillBench(device)
        sec = pb.run(max(20, args.steps // 50), args.warmup)
        a_sec = pb.run_attention(max(50, args.steps // 20), args.warmup)
        bf16_peak = _bf16_peak()
        next_rows["chunked_prefill"] = {
            "workload": f"{pb.w.B} sequences, cached U[0..3584], chunk {pb.max_q} tokens, "
                        f"{pb.w.H_q}/{pb.w.H_kv} heads, d {pb.w.D}, bf16",
            "ms_per_step": round(sec * 1e3, 4), "tflops": round(pb.flops / sec / 1e12, 1),
            "frac_of_bf16_peak": round(pb.flops / sec / 1e12 / bf16_peak, 4),
            "attention_ms_per_call": round(a_sec * 1e3, 4),
            "attention_tflops": round(pb.flops / a_sec / 1e12, 1),
            "attention_frac_of_bf16_peak": round(pb.flops / a_sec / 1e12 / bf16_peak, 4),
            "prefill_tokens_per_s_per_layer": round(pb.tokens / sec, 1), "err_flag": int(pb.err.item())}
        del pb
        torch.cuda.empty_cache()
        pq = PrefillBench(device, kind="fp8")
        pq.run(1, 0)  # one step appends the chunk's K/V codes
        x_sec = pq.run_attention(max(50, args.steps // 4), args.warmup, ws=True)
        q_sec = pq.run_attention(max(50, args.steps // 20), args.warmup)
        next_rows["chunked_prefill_fp8_cache"] = {
            "workload": "the chunked-prefill workload over an E4M3 K / INT8 V cache (per-head scales)",
            "path": "pa_prefill_attention_ws: each attended block decoded once into the workspace as bf16, then "
                    "the tcgen05 kernel",
            "attention_ms_per_call": round(x_sec * 1e3, 4), "attention_tflops": round(pq.flops / x_sec / 1e12, 1),
            "attention_frac_of_bf16_peak": round(pq.flops / x_sec / 1e12 / bf16_peak, 4),
            "no_workspace": {"path": "pa_prefill_attention: blocks decoded per 16-token query tile into shared "
                                     "memory, warp-level tensor-core products",
                             "attention_ms_per_call": round(q_sec * 1e3, 4),
                             "attention_tflops": round(pq.flops / q_sec / 1e12, 1)},
            "err_flag": int(pq.err.item())}
        del pq
        torch.cuda.empty_cache()
        n_sw = max(100, args.steps // 4)
        sb = SlidingBench("swa", device, horizon=2 * (n_sw + args.warmup))
        e_sw, _, by_sw = sb.run(n_sw, args.warmup)
        _, a_sw, _ = sb.run(n_sw, args.warmup, per_call_events=True)
        first = sb.t - n_sw
        ab_sw = float(np.mean([sb.bytes_at(t) for t in range(first, sb.t)]))
        a_ms = float(np.mean(a_sw))
        sw = sb.w
        next_rows["sliding_window_decode"] = {
            "workload": f"swa: B={sw.B}, H_q={sw.H_q}, H_kv={sw.H_kv}, d={sw.D}, window {sw.window}, cached ctx "
                        f"U[{int(sw.ctx_old.min())}..{int(sw.ctx_old.max())}], positions advancing, blocks "
                        f"released behind the window every step",
            "value": round(by_sw / e_sw / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(1e3 * e_sw / n_sw, 4),
            "tokens_per_s_per_layer": round(sw.B * n_sw / e_sw, 1),
            "attention_gbs": round(ab_sw / (a_ms / 1e3) / 1e9, 1),
            "attention_frac": round(ab_sw / (a_ms / 1e3) / 1e9 / peak, 4),
            "attention_ms_per_call": round(a_ms, 5),
            "table_uploads": sb.uploads, "table_bytes": int(sb.tables.nbytes),
            "held_blocks_max": sb.held_blocks_max, "pool_blocks": sw.num_blocks,
            "err_flag": int(sb.err.item())}
        del sb
        torch.cuda.empty_cache()
        next_rows["prefix_cache"] = prefix_cache_row(device, args.warmup)
        torch.cuda.empty_cache()
        next_rows["int4_kv_decode"] = {
            "workload": "int4_8b: the 8b shape with K and V as INT4 codes + bf16 scale + zero point per "
                        "32 dims (80 bytes per token-head row)", **measure_decode("int4_8b")}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        cpu = cpu_baseline(args.config, args.cpu_seconds)

    if rank == 0:
        kv_bytes = int(sum(b.step_bytes) / WINDOW)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "warmup_steps_run": warm_steps,
            "warmup_note": f"untimed steps right before timing: at least --warmup and at least {WARM_SECONDS} s",
            "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.k_dtype == "bf16" else "fp8e4m3/int8",
            "data": "synthetic",
            "config": {"workload": f"{args.config}: B={w.B}, H_q={w.H_q}, H_kv={w.H_kv}, d={w.D}, block 16, "
                                   f"cached ctx U[{int(w.ctx_old.min())}..{int(w.ctx_old.max())}] + <=64 "
                                   f"decoded, 1 layer per step",
                       "partition_size": args.partition, "parallelism": f"replicas x{ws}",
                       "l2": f"inputs larger than L2 ({kv_bytes / 1e6:.0f} MB attended per step vs "
                             f"{L2_BYTES / 1e6:.0f} MB L2)"},
            "tokens_per_s_per_layer": round(tok_s_layer, 1),
            f"tokens_per_s_model_{MODEL_LAYERS.get(args.config, 32)}_layers":
                round(tok_s_layer / MODEL_LAYERS.get(args.config, 32), 1),
            "pct_of_hbm_peak": round(100 * value / peak, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": args.traffic if args.traffic is not None else ncu_traffic(args.config),
                         "traffic_note": "ncu DRAM bytes per decode_kernel launch; achieved covers the "
                                         "whole call (decode_kernel + merge_kernel)",
                         "kernel": "pa_decode_attention (decode_kernel + merge_kernel)",
                         "peak_kind": peak_kind, "ms_per_call": round(att_mean_ms, 5),
                         "ms_per_call_percentiles": att_pct, "calls_timed": n_calls,
                         "algorithmic_bytes_per_call": int(att_bytes)},
            "e2e": {"value": round(bytes_e2e / el_e2e / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(1e3 * el_e2e / args.steps, 5),
                    "host_ms_per_step": round(host_ms_e2e, 5)},
            "host_ms_per_step": round(host_ms, 5),
            "gpu_launches": args.steps * b.launches_per_step + cow_launches,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "err_flag": err,
        }
        if extra:
            line["also"] = extra
        if next_rows:
            line["next_rows"] = next_rows
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="8b")
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--also", default="tiny,70b,prefix_cow,long_quant,long_quant_tok",
                    help="more decode workloads reported under 'also' (comma list, or 'none')")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the rows beyond decode (chunked prefill)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="length of each CPU oracle sample (all cores, then one)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per attention call of the current kernel sources (null when unknown)")
    ap.add_argument("--attention-only", action="store_true",
                    help="with --config: one decode step, then --warmup + --steps decode-attention calls on the "
                         "same inputs, one JSON line; for profiling the decode kernel")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="with --attention-only on a workload with a shared prefix: the calls attend the prefix "
                         "once for all sequences (pa_decode_attention_shared)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the chunked-prefill row (append + prefill attention steps) and print it; "
                         "for profiling that kernel")
    ap.add_argument("--prefill-ws", action="store_true",
                    help="with --prefill-only: time the attention call through pa_prefill_attention_ws")
    ap.add_argument("--prefill-kind", default="bf16", choices=["bf16", "fp8"],
                    help="with --prefill-only: the cache the chunk attends over (fp8: E4M3 K / INT8 V)")
    args = ap.parse_args(argv)
    ws, _, _ = dist_env()
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU: start the N replicas under torch.distributed.run
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(29500 + os.getpid() % 1000),
               os.path.abspath(__file__)] + list(sys.argv[1:] if argv is None else argv)
        return subprocess.call(cmd)
    if ws != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but {ws} processes were launched (WORLD_SIZE)")
    if args.impl == "reference":
        return run_reference(args)
    if args.prefill_only:
        return run_prefill_only(args)
    if args.attention_only:
        return run_attention_only(args)
    return run_native(args)


def run_attention_only(args):
    """One decode step on --config (append + attention), then --warmup + --steps attention calls on the
    step's inputs; prints the mean call time.  --shared-prefix (a workload with a shared prefix): the
    calls go through pa_decode_attention_shared."""
    import torch
    from paged_kv_cache_table_gb300 import native as N
    b = DecodeBench(args.config, torch.device("cuda", 0), args.partition, shared=args.shared_prefix)
    if args.shared_prefix and not b.shared:
        raise SystemExit(f"--shared-prefix: workload {args.config} has no shared prefix")
    s = torch.cuda.current_stream().cuda_stream
    b.step(0, s)

    def call():
        if b.shared:
            N.pa_decode_attention_shared(b.desc, b.out, b.q[0], b.k, b.v, b.tables_dev, b.ctx_dev[0], b.max_ctx,
                                         b.w.scale, args.partition, b.shared_seqs, b.w.B, b.shared_len, b.ws,
                                         b.ws_bytes, b.err, s)
            return
        N.pa_decode_attention(b.desc, b.out, b.q[0], b.k, b.v, b.tables_dev, b.ctx_dev[0], b.max_ctx, b.w.scale,
                              args.partition, b.ws, b.ws_bytes, b.err, s)
    for _ in range(max(0, args.warmup)):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(max(1, args.steps)):
        call()
    t1.record()
    torch.cuda.synchronize()
    print(json.dumps({"row": "decode_attention_shared" if b.shared else "decode_attention", "config": args.config,
                      "steps": args.steps, "warmup": args.warmup,
                      "ms_per_call": round(t0.elapsed_time(t1) / max(1, args.steps), 5),
                      "err_flag": int(b.err.item())}))
    return 0 if int(b.err.item()) == 0 else 1


def run_prefill_only(args):
    """--steps chunked-prefill steps after --warmup, then one JSON line with the step time."""
    import torch
    device = torch.device("cuda", 0)
    pb = PrefillBench(device, kind=args.prefill_kind)
    if args.prefill_ws:  # the attention call alone, through the workspace path, after one step's append
        pb.run(1, 0)
        sec = pb.run_attention(max(1, args.steps), max(0, args.warmup), ws=True)
    else:
        sec = pb.run(max(1, args.steps), max(0, args.warmup))
    print(json.dumps({"row": "chunked_prefill", "cache": args.prefill_kind, "workspace_path": bool(args.prefill_ws),
                      "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 4),
                      "tflops": round(pb.flops / sec / 1e12, 1), "err_flag": int(pb.err.item())}))
    return 0 if int(pb.err.item()) == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
