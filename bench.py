"""Benchmark of the paged-KV hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole path over one batch of synthetic input:
copy_blocks (Copy-on-Write pairs, if any) -> reshape_and_cache (this step's
new tokens) -> chunked prefill (if any) -> decode partial -> log-sum-exp merge,
all on one stream with inputs resident in HBM.  The default workload is the
long-context split-K decode (batch 8, 64/8 heads, D=128, bs=16, contexts
U{32768..131072}, 512-token partitions merged by log-sum-exp), the largest
decode workload that the measurement runs on one GPU; the others (the
Llama-8B-style GQA decode, shared prefix, mixed prefill + decode, verify)
are selectable with --workload.

Reported (one JSON line from rank 0):
* value: algorithmic bytes of the step (KV + Q + O + block tables + lengths +
  this step's cache writes) / step time, GB/s, summed over ranks (replicas);
  decode_tokens_per_s alongside;
* roofline: the dominant kernel (decode partial) timed with CUDA events on its
  stream inside the timed region, against the measured HBM copy bandwidth;
* cpu_baseline: the float64 CPU oracle on a bounded sample of the same
  workload on this host (rank 0 only);
* e2e: the same metric through the public API with host buffers: pinned host
  -> device copies of the step's inputs and a device -> host read of its
  outputs inside the timed region, three steps in flight; the kernels of a
  one-stream step are the library calls marshalled once (ops.recording) and
  issued again each step, those of a two-stream step one CUDA graph.
``--impl reference`` times the CPU oracle itself as the reference arm.
``--kv-layout contiguous|vmm`` (decode-only workloads) runs the same step on
the competing design of "vAttention 完全拆解": one contiguous
[slots][max_len][kv_heads][head_dim] K and V per layer (plain device memory,
or a virtual range whose 2 MiB pages are mapped on demand), no Block Table;
the contexts are the paged step's, copied in before timing.
Multi-GPU: independent replicas (the path needs no collective); N>1 runs under
torch.distributed.run with one rank per GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention: achieved KV GB/s vs GB300 HBM peak; decode tokens/s"
DEFAULT_WORKLOAD = "long_context_splitk_decode"
E2E_SETS = 3  # staging buffer sets, i.e. end-to-end steps in flight
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int, device) -> float:
    """The largest x over all ranks (x itself on one rank): the slowest replica sets the time."""
    if ws == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: float, steps: int, seconds: float, ws: int) -> float:
    """Weak scaling: every rank moves the same bytes per step; all ranks' bytes over the max time."""
    return ws * bytes_per_rank_step * steps / seconds / 1e9


def measured_tensor_peak():
    """Dense bf16 TFLOP/s: the measured burst figure (a kernel timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_traffic(profile_name: str, source_file: str, block_size: int = 16):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source.

    The summaries were taken on the workloads' own 16-token blocks; another
    block size is another launch, whose traffic they do not give (None)."""
    if block_size != 16:
        return None
    path = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h:
        return None
    cur = hashlib.sha256(open(os.path.join(ROOT, source_file), "rb").read()).hexdigest()
    if not cur.startswith(h.group(1)):
        return None  # the kernel changed since the counters were taken
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workload set-up
class Step:
    """Device buffers and host copies of one workload step; runs it through the C ABI."""

    def __init__(self, wl: W.Workload, device: torch.device, value_seed: int, overlap_streams: bool = True,
                 shared_prefix: bool = True, kv_layout: str = "paged", verify_impl: str = "mma",
                 verify_ctas: int = 0):
        from paged_kv_cache_76_gb300 import ops
        from paged_kv_cache_76_gb300.allocator import BlockAllocator
        self.ops = ops
        self._rec = None  # a plan being recorded (record_plan)
        self.wl = wl
        self.dev = device
        self.verify_impl = verify_impl
        self.verify_ctas = verify_ctas
        a = BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
        a.run(wl.setup_ops)
        slots, pairs = a.run(wl.step_ops)
        self.alloc = a
        vals = W.make_values(wl, device=device, seed=value_seed)
        self.vals = vals
        self.k_cache, self.v_cache = vals["k_cache"], vals["v_cache"]
        self.pre_k = None
        self.h = {}   # pinned host copies of every per-step input
        self.d = {}   # device copies
        self.h["k_new"] = vals["k_new"].cpu().pin_memory()
        self.h["v_new"] = vals["v_new"].cpu().pin_memory()
        self.h["slots"] = torch.tensor(slots, dtype=torch.int32).pin_memory()
        self.h["pairs"] = torch.tensor(pairs, dtype=torch.int32).reshape(-1, 2).pin_memory()
        self.n_pairs = len(pairs)
        self.dec = bool(wl.decode_seqs)
        self.pre = bool(wl.prefill)
        self.layout = kv_layout
        if kv_layout != "paged" and (self.pre or self.n_pairs or wl.q_len != 1 or not self.dec):
            raise ValueError("--kv-layout contiguous|vmm takes a decode-only workload")
        if self.dec:
            maxblk = max(len(a.block_table(s)) for s in wl.decode_seqs)
            t, l = a.build_tables(wl.decode_seqs, maxblk)
            self.dec_lens = l.astype(np.int64)
            self.dec_tables_np = t
            self.h["dec_tables"] = torch.from_numpy(t).pin_memory()
            self.h["dec_lens"] = torch.from_numpy(l).pin_memory()
            self.h["q_decode"] = vals["q_decode"].cpu().pin_memory()
            self.split = ops.decode_split_tokens(maxblk, wl.block_size, wl.split_tokens)
            n = ops.decode_workspace_size(len(wl.decode_seqs), wl.q_heads, wl.head_dim, maxblk, wl.block_size,
                                          self.split)
            # a prefix every decode request shares (e.g. a common system prompt)
            # goes through pa_decode_shared_prefix: read once for all queries
            self.prefix_len = 0
            if wl.q_len > 1:  # speculative verify: k+1 queries per request
                self.split = ops.verify_split_tokens(maxblk, wl.block_size, wl.q_len, wl.split_tokens)
                n = ops.verify_workspace_size(len(wl.decode_seqs), wl.q_len, wl.q_heads, wl.head_dim, maxblk,
                                              wl.block_size, self.split)
            if shared_prefix and wl.q_len == 1 and wl.block_size >= 8 and len(wl.decode_seqs) >= 8:
                nshared = a.common_prefix(wl.decode_seqs)
                if nshared >= 8:
                    self.prefix_len = nshared * wl.block_size
                    self.h["prefix_blocks"] = torch.tensor(t[0, :nshared], dtype=torch.int32).pin_memory()
                    # the suffix partition: the workload's, else the call's automatic choice
                    self.split = ops.decode_shared_prefix_split_tokens(maxblk, wl.block_size, self.prefix_len,
                                                                       wl.split_tokens)
                    n = ops.decode_shared_prefix_workspace_size(len(wl.decode_seqs), wl.q_heads, wl.head_dim, maxblk,
                                                                wl.block_size, self.prefix_len, self.split)
            if kv_layout != "paged":
                shared_prefix = False
                self.prefix_len = 0
                n = self._contiguous_setup(a, device)
            self.workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=device) if n else None
        if self.pre:
            seqs = [s for s, _, _ in wl.prefill]
            maxblk = max(len(a.block_table(s)) for s in seqs)
            t, l = a.build_tables(seqs, maxblk)
            self.pre_lens = l.astype(np.int64)
            self.pre_tables_np = t
            self.chunks = [c for _, c, _ in wl.prefill]
            self.h["pre_tables"] = torch.from_numpy(t).pin_memory()
            self.h["pre_lens"] = torch.from_numpy(l).pin_memory()
            self.h["q_start"] = torch.tensor(np.concatenate([[0], np.cumsum(self.chunks)]),
                                             dtype=torch.int32).pin_memory()
            self.h["q_prefill"] = vals["q_prefill"].cpu().pin_memory()
            self.max_q_len = max(self.chunks)
        # One pinned staging buffer for every per-step input and one for the
        # outputs, so an end-to-end step is a single host->device copy, the
        # kernels, and a single device->host copy.
        def layout(tensors):
            offs, off = {}, 0
            for k, v in tensors.items():
                offs[k] = off
                off += (v.numel() * v.element_size() + 255) // 256 * 256
            return offs, max(off, 256)

        def views(buf, offs, like):
            return {k: buf[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                    for k, v in like.items()}

        offs, nbytes = layout(self.h)
        self.h_stage = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        self.d_stage = torch.empty(nbytes, dtype=torch.uint8, device=device)
        hv = views(self.h_stage, offs, self.h)
        for k, v in self.h.items():
            hv[k].copy_(v)
        self.h = hv
        self.d = views(self.d_stage, offs, self.h)
        self.d_stage.copy_(self.h_stage)
        outs = {}
        if self.dec:
            outs["dec"] = self.h["q_decode"]
        if self.pre:
            outs["pre"] = self.h["q_prefill"]
        ooffs, obytes = layout(outs)
        self.d_out = torch.empty(obytes, dtype=torch.uint8, device=device)
        self.h_outbuf = torch.empty(obytes, dtype=torch.uint8).pin_memory()
        self.out_used = sum(v.numel() * v.element_size() for v in outs.values())
        dv = views(self.d_out, ooffs, outs)
        hv = views(self.h_outbuf, ooffs, outs)
        self.side = None
        self.prefill_ctas = 0
        if self.pre and self.dec and overlap_streams:
            # prefill (tensor-bound) on a second stream at the highest priority,
            # so that its CTAs take their SMs first; decode (HBM-bound) fills the rest
            self.side = torch.cuda.Stream(device, priority=torch.cuda.Stream.priority_range()[1])
            self.ev_fork, self.ev_join = torch.cuda.Event(), torch.cuda.Event()
        self.prefix_side = None
        if self.dec and self.prefix_len and overlap_streams:
            # the shared prefix's tensor-core pass on a second stream, forked at
            # the start of the step: it reads only q and blocks this step does
            # not write, and runs beside the HBM-bound suffix decode
            self.prefix_side = torch.cuda.Stream(device, priority=torch.cuda.Stream.priority_range()[1])
            self.ev_pfork = torch.cuda.Event()
        # more sets of staging buffers: the end-to-end loop keeps E2E_SETS steps
        # in flight (the host launches step i+E2E_SETS-1 before it reads step
        # i's result), so host-side jitter does not starve the GPU
        self._sets = [dict(h_stage=self.h_stage, d_stage=self.d_stage, d=self.d, d_out=self.d_out,
                           h_outbuf=self.h_outbuf, out_dec=dv.get("dec"), out_pre=dv.get("pre"))]
        for _ in range(E2E_SETS - 1):
            h2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
            h2.copy_(self.h_stage)
            d2 = torch.empty(nbytes, dtype=torch.uint8, device=device)
            d2.copy_(h2)
            o2 = torch.empty(obytes, dtype=torch.uint8, device=device)
            dv2 = views(o2, ooffs, outs)
            self._sets.append(dict(h_stage=h2, d_stage=d2, d=views(d2, offs, self.h), d_out=o2,
                                   h_outbuf=torch.empty(obytes, dtype=torch.uint8).pin_memory(),
                                   out_dec=dv2.get("dec"), out_pre=dv2.get("pre")))
        self.out_dec = dv.get("dec")
        self.out_pre = dv.get("pre")
        self.h_out_dec = hv.get("dec")
        self.h_out_pre = hv.get("pre")

    def _contiguous_setup(self, a, device):
        """Contiguous per-slot K/V holding the paged step's contexts (request r in slot r)."""
        from paged_kv_cache_76_gb300 import vattention as va
        wl = self.wl
        S = len(wl.decode_seqs)
        row = wl.kv_heads * wl.head_dim * 2
        lens = self.dec_lens.astype(np.int64)
        self.vkv = None
        if self.layout == "vmm":
            G = va.VirtualKV.granularity()
            unit = int(np.lcm(16, G // math.gcd(G, row)))
            L = int(-(-int(lens.max()) // unit) * unit)
            t0 = time.perf_counter()
            self.vkv = va.VirtualKV(S, L, 1, wl.kv_heads, wl.head_dim, wl.torch_dtype, page_bytes=G)
            for _ in range(S):
                self.vkv.alloc_slot()
            self.vkv.step(lens.astype(np.int32))
            torch.cuda.synchronize()
            self.vmm_setup_s = time.perf_counter() - t0
            self.ck, self.cv = self.vkv.tensor(0, False), self.vkv.tensor(0, True)
        else:
            L = int(-(-int(lens.max()) // 16) * 16)
            self.ck = torch.empty(S, L, wl.kv_heads, wl.head_dim, dtype=wl.torch_dtype, device=device)
            self.cv = torch.empty_like(self.ck)
        self.max_len = L
        # history: every token but this step's new one, copied block by block
        # (rows inside each slot's mapped range only)
        bs = wl.block_size
        for r, s in enumerate(wl.decode_seqs):
            hist = int(lens[r]) - 1
            t = self.dec_tables_np[r]
            for j in range(-(-hist // bs)):
                n = min(bs, hist - j * bs)
                self.ck[r, j * bs:j * bs + n] = self.k_cache[int(t[j]), :n]
                self.cv[r, j * bs:j * bs + n] = self.v_cache[int(t[j]), :n]
        torch.cuda.synchronize()
        del self.h["dec_tables"]  # no Block Table on this layout
        self.h["slot_ids"] = torch.arange(S, dtype=torch.int32).pin_memory()
        self.h["positions"] = torch.from_numpy((lens - 1).astype(np.int32)).pin_memory()
        return self.ops.decode_workspace_size(S, wl.q_heads, wl.head_dim, L // 16, 16, wl.split_tokens)

    def _run_contiguous(self, stream, ev):
        from paged_kv_cache_76_gb300 import vattention as va
        o, d, wl = self.ops, self.d, self.wl
        if self.vkv is not None:
            self.vkv.reshape_and_cache(0, d["k_new"], d["v_new"], d["slot_ids"], d["positions"], stream=stream)
        else:
            va.reshape_and_cache_slots(d["k_new"], d["v_new"], d["slot_ids"], d["positions"], self.ck, self.cv,
                                       stream=stream)
        if ev is not None:
            ev[0].record(stream)
        if self.vkv is not None:
            self.vkv.decode(0, d["q_decode"], d["slot_ids"], d["dec_lens"], wl.scale, out=self.out_dec,
                            split_tokens=wl.split_tokens, workspace=self.workspace, stream=stream)
        else:
            va.decode_contiguous(d["q_decode"], self.ck, self.cv, d["slot_ids"], d["dec_lens"], wl.scale,
                                 out=self.out_dec, split_tokens=wl.split_tokens, workspace=self.workspace,
                                 stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def _do(self, fn):
        """A stream/event operation of the step: run it, or add it to the plan being recorded."""
        if self._rec is not None:
            self._rec.add(fn)
        else:
            fn()

    def record_plan(self, stream):
        """The step's launches and stream/event operations, marshalled once (ops.recording)."""
        with self.ops.recording() as rec:
            self._rec = rec
            try:
                self.run(stream)
            finally:
                self._rec = None
        return rec

    # -- one step through the C ABI; ev = (start, end) events around the decode partial kernel
    def run(self, stream, ev=None):
        o, d, wl = self.ops, self.d, self.wl
        if self.layout != "paged":
            return self._run_contiguous(stream, ev)
        if self.prefix_side is not None:
            self._do(lambda: self.ev_pfork.record(stream))
            self._do(lambda: self.prefix_side.wait_event(self.ev_pfork))
        if self.n_pairs:
            o.copy_blocks(self.k_cache, self.v_cache, d["pairs"], stream=stream)
        o.reshape_and_cache(d["k_new"], d["v_new"], d["slots"], self.k_cache, self.v_cache, stream=stream)
        overlap = self.pre and self.dec and self.side is not None
        if overlap:
            # prefill (tensor-bound) on a second stream, concurrent with decode (HBM-bound);
            # both only read the cache this step's reshape_and_cache wrote
            self._do(lambda: self.ev_fork.record(stream))
            self._do(lambda: self.side.wait_event(self.ev_fork))
            o.chunked_prefill(d["q_prefill"], d["q_start"], d["pre_lens"], self.k_cache, self.v_cache,
                              d["pre_tables"], wl.scale, self.max_q_len, out=self.out_pre, stream=self.side,
                              max_ctas=self.prefill_ctas)
            self._do(lambda: self.ev_join.record(self.side))
        elif self.pre:
            if ev is not None and not self.dec:
                ev[0].record(stream)
            o.chunked_prefill(d["q_prefill"], d["q_start"], d["pre_lens"], self.k_cache, self.v_cache,
                              d["pre_tables"], wl.scale, self.max_q_len, out=self.out_pre, stream=stream)
            if ev is not None and not self.dec:
                ev[1].record(stream)
        if self.dec and self.prefix_len:
            if ev is not None:
                ev[0].record(stream)
            o.decode_shared_prefix(d["q_decode"], self.k_cache, self.v_cache, d["prefix_blocks"], self.prefix_len,
                                   d["dec_tables"], d["dec_lens"], wl.scale, out=self.out_dec, split_tokens=self.split,
                                   workspace=self.workspace, stream=stream, prefix_stream=self.prefix_side)
            if ev is not None:
                ev[1].record(stream)
        elif self.dec and wl.q_len > 1:
            if ev is not None:
                ev[0].record(stream)
            if self.verify_impl == "tc":
                o.verify_decode_tc(d["q_decode"], self.k_cache, self.v_cache, d["dec_tables"], d["dec_lens"],
                                   wl.scale, out=self.out_dec, max_ctas=self.verify_ctas, stream=stream)
            else:
                o.verify_decode(d["q_decode"], self.k_cache, self.v_cache, d["dec_tables"], d["dec_lens"], wl.scale,
                                out=self.out_dec, split_tokens=self.split, workspace=self.workspace, stream=stream)
            if ev is not None:
                ev[1].record(stream)
        elif self.dec:
            if ev is not None:
                ev[0].record(stream)
            o.decode_partial(d["q_decode"], self.k_cache, self.v_cache, d["dec_tables"], d["dec_lens"], wl.scale,
                             self.out_dec, split_tokens=self.split, workspace=self.workspace, stream=stream)
            if ev is not None:
                ev[1].record(stream)
            o.lse_merge(self.workspace, d["dec_lens"], d["q_decode"], d["dec_tables"], wl.block_size, self.out_dec,
                        split_tokens=self.split, stream=stream)
        if overlap:
            self._do(lambda: stream.wait_event(self.ev_join))

    def calibrate_prefill_ctas(self, stream, sms: int, reps: int = 3) -> int:
        """SMs to leave to the prefill when it runs beside decode.

        Decode is bound by HBM and keeps its speed on fewer SMs, so the prefill
        gets about as many SMs as it needs to finish with the decode: time each
        part alone (uncapped, `reps` runs, after one untimed run) and give the
        prefill 1.4 x SMs x t_prefill / t_decode CTAs, within [SMs/8, SMs/2]
        (the step time is flat from ~56 to ~64 CTAs on the mixed workload and
        rises steeply below; the margin keeps the cap on the flat side).
        """
        o, d, wl = self.ops, self.d, self.wl
        def timed(fn):
            fn()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps
        def pre():
            o.chunked_prefill(d["q_prefill"], d["q_start"], d["pre_lens"], self.k_cache, self.v_cache,
                              d["pre_tables"], wl.scale, self.max_q_len, out=self.out_pre, stream=stream)
        def dec():
            saved, self.pre = self.pre, False
            try:
                self.run(stream)
            finally:
                self.pre = saved
        t_pre, t_dec = timed(pre), timed(dec)
        cap = int(round(1.4 * sms * t_pre / max(t_dec, 1e-6)))
        self.prefill_ctas = max(max(1, sms // 8), min(sms // 2, cap))
        return self.prefill_ctas

    def select(self, k: int):
        """Use staging buffer set k (0 .. E2E_SETS-1) for the following steps."""
        for name, val in self._sets[k].items():
            setattr(self, name, val)

    def run_e2e(self, stream):
        """Host buffers in, host buffers out: one copy each way inside the step."""
        self.d_stage.copy_(self.h_stage, non_blocking=True)
        self.run(stream)
        self.h_outbuf.copy_(self.d_out, non_blocking=True)

    def e2e_bytes(self):
        return int(self.h_stage.numel()), int(self.h_outbuf.numel())

    # -- algorithmic bytes
    def bytes_breakdown(self):
        return step_bytes(self.wl, self.dec_lens if self.dec else None, self.dec_tables_np if self.dec else None,
                          self.pre_lens if self.pre else None, self.chunks if self.pre else None,
                          int(self.h["slots"].numel()), self.n_pairs, self.layout)


def step_bytes(wl: W.Workload, dec_lens, dec_tables, pre_lens, chunks, new_tokens: int, n_pairs: int,
               layout: str = "paged"):
    """Algorithmic bytes (and prefill flops) of one step, per part.

    decode: per request of context L, K and V of its L tokens, its q_len query
    and output rows, one int32 table entry per logical block and its int32
    length (a slot id instead of the table on the contiguous layout);
    decode_unique: the same with every (physical block, offset) cache row the
    batch reads counted once (a shared prefix is read once);
    reshape_and_cache: read k, v and write them, plus the slot, per new token;
    copy_blocks: read and write one block of K and of V, plus the pair;
    prefill: the chunk's K/V history, its query and output rows, table and
    bounds; prefill_flops: 4 * Hq * D per visible (query, key) pair.
    """
    e = 2
    tok = wl.kv_heads * wl.head_dim * e          # one token's K (or V), all KV heads
    qrow = wl.q_heads * wl.head_dim * e
    bs = wl.block_size
    out = {}
    if dec_lens is not None:
        L = np.asarray(dec_lens, dtype=np.int64)
        table = 4 * np.ceil(L / bs) if layout == "paged" else 4
        out["decode"] = int(np.sum(2 * L * tok + 2 * qrow * wl.q_len + table + 4))
        used = {}
        for r, Lr in enumerate(L):
            for j in range(int(math.ceil(Lr / bs))):
                b = int(dec_tables[r, j])
                used[b] = max(used.get(b, 0), min(bs, int(Lr) - j * bs))
        out["decode_unique"] = int(sum(used.values()) * 2 * tok +
                                   np.sum(2 * qrow * wl.q_len + 4 * np.ceil(L / bs) + 4))
    out["reshape_and_cache"] = new_tokens * (4 * tok + 4)
    out["copy_blocks"] = n_pairs * (4 * bs * tok + 8)
    if pre_lens is not None:
        L = np.asarray(pre_lens, dtype=np.int64)
        ch = np.asarray(chunks)
        out["prefill"] = int(np.sum(2 * L * tok + 2 * ch * qrow + 4 * np.ceil(L / bs) + 8))
        vis = sum(sum(int(L[i]) - int(ch[i]) + q + 1 for q in range(int(ch[i]))) for i in range(len(ch)))
        out["prefill_flops"] = 4 * vis * wl.q_heads * wl.head_dim
    return out


# ----------------------------------------------------------------------------- the CPU oracle on a sample
class HostStep:
    """The same workload step on the host alone, for the CPU oracle legs.

    Block tables and slots come from the oracle's own allocator replaying the
    workload's scripts; values are drawn on the host per (request, KV head)
    unit from a seeded generator (the oracle's cost does not depend on them).
    Nothing here touches the GPU or the CUDA library.
    """

    def __init__(self, wl: W.Workload, value_seed: int):
        from oracle.block_pool import SequenceManager
        self.wl = wl
        self.seed = value_seed
        a = SequenceManager(wl.num_blocks, wl.block_size, wl.free_order)
        a.run(wl.setup_ops)
        slots, _ = a.run(wl.step_ops)
        self.slots = np.asarray(slots, dtype=np.int64)
        self.dec = bool(wl.decode_seqs)
        self.pre = bool(wl.prefill)

        def tables(seqs):
            t = [a.block_table(s) for s in seqs]
            width = max(1, max(len(x) for x in t))
            arr = np.full((len(seqs), width), -1, dtype=np.int64)
            for i, x in enumerate(t):
                arr[i, :len(x)] = x
            return arr, np.asarray([a.num_tokens[s] for s in seqs], dtype=np.int64)

        if self.dec:
            self.dec_tables_np, self.dec_lens = tables(wl.decode_seqs)
        if self.pre:
            self.pre_tables_np, self.pre_lens = tables([s for s, _, _ in wl.prefill])
            self.chunks = [c for _, c, _ in wl.prefill]

    def _draw(self, rng, shape):
        if self.wl.value_dist == "uniform":
            a = rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
        else:
            a = rng.standard_normal(size=shape, dtype=np.float32)
        return torch.from_numpy(a).to(self.wl.torch_dtype).double().numpy()  # exact upcasts of the input type

    def unit_inputs(self, unit):
        """Host float64 inputs of one unit: its request's blocks for one KV head (not timed)."""
        kind, r, g = unit
        wl = self.wl
        bs, G, D = wl.block_size, wl.q_heads // wl.kv_heads, wl.head_dim
        rng = np.random.Generator(np.random.PCG64([self.seed, 0 if kind == "decode" else 1, r, g]))
        if kind == "decode":
            table, L = self.dec_tables_np[r], int(self.dec_lens[r])
            q = self._draw(rng, (wl.q_len, G, D))  # decode: [1, G, D]; verify: [q_len, G, D]
        else:
            table, L = self.pre_tables_np[r], int(self.pre_lens[r])
            q = self._draw(rng, (self.chunks[r], G, D))
        nblk = int(math.ceil(L / bs))
        kc = self._draw(rng, (nblk, bs, 1, D))
        vc = self._draw(rng, (nblk, bs, 1, D))
        # this step's new tokens that land in these blocks (remapped to the sub-pool)
        pos = {int(b): i for i, b in enumerate(table[:nblk])}
        sub = [pos[int(s) // bs] * bs + int(s) % bs for s in self.slots if s >= 0 and int(s) // bs in pos]
        kn = self._draw(rng, (len(sub), 1, D))
        vn = self._draw(rng, (len(sub), 1, D))
        return dict(q=q, kc=kc, vc=vc, kn=kn, vn=vn, slots=np.asarray(sub, np.int64),
                    table=np.arange(nblk)[None], L=L, chunk=(q.shape[0] if kind == "prefill" else 1))

    def units(self):
        """(kind, request index, kv head) units of the step, in a fixed order."""
        wl = self.wl
        units = []
        if self.dec:
            units += [("decode", r, g) for r in range(len(wl.decode_seqs)) for g in range(wl.kv_heads)]
        if self.pre:
            units += [("prefill", r, g) for r in range(len(wl.prefill)) for g in range(wl.kv_heads)]
        return units

    def unit_bytes(self, unit):
        """The unit's share of the step's algorithmic bytes (its KV head's share of table and length)."""
        kind, r, g = unit
        wl = self.wl
        e, D, G, bs = 2, wl.head_dim, wl.q_heads // wl.kv_heads, wl.block_size
        if kind == "decode":
            L = int(self.dec_lens[r])
            return 2 * L * D * e + 2 * G * D * e * wl.q_len + (4 * math.ceil(L / bs) + 4) / wl.kv_heads
        L = int(self.pre_lens[r])
        c = self.chunks[r]
        return 2 * L * D * e + 2 * c * G * D * e + (4 * math.ceil(L / bs) + 8) / wl.kv_heads


def run_oracle_units(hs: HostStep, units, budget_s: float):
    """Time the oracle (as it stands) on units until the budget is spent."""
    from oracle import paged_attention as opa
    wl = hs.wl
    done_bytes, t_oracle, done = 0.0, 0.0, []
    cpu0 = time.process_time()
    cpu_inputs = 0.0
    for u in units:
        c0 = time.process_time()
        x = hs.unit_inputs(u)
        cpu_inputs += time.process_time() - c0
        t0 = time.perf_counter()
        kc, vc = opa.reshape_and_cache(x["kn"], x["vn"], x["slots"], x["kc"], x["vc"])
        if u[0] == "decode" and wl.q_len > 1:
            opa.verify_decode(x["q"][None], kc, vc, x["table"], [x["L"]], wl.scale)
        elif u[0] == "decode":
            opa.decode(x["q"], kc, vc, x["table"], [x["L"]], wl.scale)
        else:
            opa.chunked_prefill(x["q"], [0, x["chunk"]], [x["L"]], kc, vc, x["table"], wl.scale)
        t_oracle += time.perf_counter() - t0
        done_bytes += hs.unit_bytes(u)
        done.append(u)
        if t_oracle >= budget_s:
            break
    cpu = time.process_time() - cpu0 - cpu_inputs
    return done_bytes, t_oracle, done, cpu


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--split", type=int, default=None, help="decode partition size (default: the workload's)")
    ap.add_argument("--block-size", type=int, default=None, choices=[4, 8, 16, 32],
                    help="tokens per block for the decode workloads built from one context draw "
                         "(llama8b_gqa_decode, long_context_splitk_decode, spec_verify_decode); default 16")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--jsonl", default=None, help="also append the result line to this file")
    ap.add_argument("--e2e-launch", default="auto", choices=["auto", "graph", "eager"],
                    help="kernels of each end-to-end step: eager launches marshalled once (ops.recording), or a "
                         "CUDA graph per buffer set; auto = eager for one-stream steps, graph for steps that fork "
                         "a second stream")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--serial", action="store_true", help="run prefill and decode on one stream, one after the other")
    ap.add_argument("--kv-layout", default="paged", choices=["paged", "contiguous", "vmm"],
                    help="decode-only workloads: paged blocks (default), or one contiguous K/V per request slot in "
                         "plain memory or in on-demand-mapped virtual memory (the vAttention comparison)")
    ap.add_argument("--verify-impl", default="auto", choices=["auto", "mma", "tc"],
                    help="verify workloads: the warp-MMA partition kernel with its merge (pa_verify_decode), the "
                         "tcgen05 one-tile kernel (pa_verify_decode_tc), or auto: tcgen05 when a unit has more than "
                         "16 (query, group head) columns and blocks of >= 8 tokens (measured faster there)")
    ap.add_argument("--verify-ctas", type=int, default=0,
                    help="--verify-impl tc: CTAs of the kernel (0: one per (request, KV head) unit)")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="decode a shared prefix per request instead of once for the batch")
    ap.add_argument("--prefill-ctas", type=int, default=None,
                    help="CTAs for a prefill running beside decode (0: one per work unit; default: calibrated)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    ws, rank, local = dist_env()
    if args.block_size is not None and args.block_size != 16:
        if args.workload not in ("llama8b_gqa_decode", "long_context_splitk_decode", "spec_verify_decode"):
            ap.error("--block-size applies to llama8b_gqa_decode, long_context_splitk_decode, spec_verify_decode")
        wl = W.WORKLOADS[args.workload](block_size=args.block_size)
    else:
        wl = W.WORKLOADS[args.workload]()
    if args.split is not None:
        wl.split_tokens = args.split
    if args.impl == "reference":
        # the CPU oracle on rank 0 alone, on the host: no GPU, no CUDA library
        if rank == 0:
            reference_arm(args, wl, ws)
        return

    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(device)
    from paged_kv_cache_76_gb300 import _lib
    _lib.lib()  # fails loudly if the CUDA library is missing

    if args.verify_impl == "auto":
        cols = wl.q_len * (wl.q_heads // wl.kv_heads)
        args.verify_impl = "tc" if wl.q_len > 1 and cols > 16 and wl.block_size >= 8 else "mma"
    step = Step(wl, device, value_seed=1000 * rank, overlap_streams=not args.serial,
                shared_prefix=not args.no_shared_prefix, kv_layout=args.kv_layout, verify_impl=args.verify_impl,
                verify_ctas=args.verify_ctas)
    peak, peak_kind = measured_peaks()

    stream = torch.cuda.Stream(device)
    if step.side is not None:
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        if args.prefill_ctas is not None:
            step.prefill_ctas = args.prefill_ctas
        else:
            step.calibrate_prefill_ctas(stream, sms)
    nb = step.bytes_breakdown()
    total_bytes = sum(v for k, v in nb.items() if k not in ("decode_unique", "prefill_flops"))
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step.run(stream)
    stream.synchronize()
    from paged_kv_cache_76_gb300 import ops
    if ops.get_device_error(stream) != 0:
        raise RuntimeError("device error recorded during warm-up")

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = None
    if total_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    clocks = ClockSampler(torch.cuda.current_device() if ws == 1 else local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = ops.launch_count()
    if flush is None:
        # inputs larger than L2: the K steps back to back in one event pair
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for i in range(args.steps):
                step.run(stream)
            t_end.record(stream)
    else:
        # a step that fits in L2: each step in its own event pair, with a
        # write of a buffer twice the L2 between steps (outside the pairs)
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(i & 0xFF)
                pairs[i][0].record(stream)
                step.run(stream)
                pairs[i][1].record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    launches = ops.launch_count() - launches0
    clk = clocks.stop()
    if ws > 1:
        torch.distributed.barrier()
    ms = t_start.elapsed_time(t_end) if flush is None else sum(a.elapsed_time(b) for a, b in pairs)
    if ops.get_device_error(stream) != 0:
        raise RuntimeError("device error recorded during the timed region")
    ms = reduce_max(ms, ws, device)
    ms_per_step = ms / args.steps

    # Dominant kernel: the same K steps again, each decode-partial launch
    # bracketed by CUDA events on its stream.  (Kept out of the region above:
    # an event between two kernels ends their programmatic-launch overlap.)
    dec_ms = None
    if step.dec or step.pre:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                if flush is not None:
                    flush.fill_(i & 0xFF)
                step.run(stream, evs[i])
        stream.synchronize()
        launch_ms = np.array([a.elapsed_time(b) for a, b in evs])
        dec_ms = float(np.mean(launch_ms))
        launch_pct = {"launch_ms_p50": round(float(np.percentile(launch_ms, 50)), 5),
                      "launch_ms_p99": round(float(np.percentile(launch_ms, 99)), 5)}

    # e2e: host buffers through the public API.  Every step copies its inputs
    # from pinned host memory (one buffer), runs the kernels (a CUDA graph per
    # staging-buffer set) and copies its outputs back, and the host reads
    # them.  The copies run on two copy streams, so step i+1's inputs go up
    # and step i-1's outputs come down while step i computes; E2E_SETS buffer
    # sets rotate, each reused only after the host has read its outputs.
    e2e_val = None
    h2d, d2h = step.e2e_bytes()
    e2e_mode = ("H2D copy stream -> kernels (CUDA graph) -> D2H copy stream per step; copies overlap the "
                "neighbouring steps' kernels; the host reads every step's outputs")
    graphs = None
    plans = None
    e2e_launch = args.e2e_launch
    if e2e_launch == "auto":
        # measured on GB300: recorded eager launches beat a graph replay by 2-5 us per step when the
        # step runs on one stream (the 8B-style step: 95.2 against 100.5 us); a step that forks a
        # second stream issues more host calls than the GPU takes to run it (shared prefix: 86-90 us
        # eager against 71.4 us as a graph)
        e2e_launch = "graph" if (step.side is not None or step.prefix_side is not None) else "eager"
    if e2e_launch == "eager":
        e2e_mode = e2e_mode.replace("kernels (CUDA graph)", "kernels (eager launches, marshalled once)")
    nsets = len(step._sets)
    with torch.cuda.stream(stream):
        for k in list(range(nsets)) + [0]:
            step.select(k)
            step.run_e2e(stream)
    stream.synchronize()
    eager_out = step.h_outbuf.clone()  # the eager step's outputs, for checking a replay
    try:
        if e2e_launch == "eager":
            raise StopIteration
        graphs = []
        for k in range(nsets):
            step.select(k)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step.run(stream)
            graphs.append(g)
        for k in range(nsets):
            step.select(k)
            step.d_out.zero_()
            with torch.cuda.stream(stream):
                graphs[k].replay()  # replays on the current stream
            stream.synchronize()
            step.h_outbuf.copy_(step.d_out)
            if ops.get_device_error(stream) != 0:
                raise RuntimeError("device error in graph replay")
            if not torch.equal(step.h_outbuf[:step.out_used], eager_out[:step.out_used]):
                raise RuntimeError("graph replay output differs from the eager step")
    except StopIteration:
        graphs = None
    except Exception as exc:  # capture not possible here: eager launches instead
        graphs = None
        e2e_mode = f"eager kernel launches, copies on two copy streams (graph capture not used: {exc})"
    if graphs is None:
        # eager: each set's launches marshalled once (ops.recording), issued as they are every step
        plans = []
        for k in range(nsets):
            step.select(k)
            plans.append(step.record_plan(stream))
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = {n: [torch.cuda.Event() for _ in range(nsets)] for n in ("up", "kern", "down")}
    checksum = 0
    sets = step._sets
    host_out = [b["h_outbuf"].numpy() for b in sets]  # the pinned output buffers, read by the host
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        k = i % nsets
        b = sets[k]
        if i >= nsets:
            up.wait_event(ev["kern"][k])  # step i-nsets's kernels are done with this input buffer
        with torch.cuda.stream(up):
            b["d_stage"].copy_(b["h_stage"], non_blocking=True)
        ev["up"][k].record(up)
        stream.wait_event(ev["up"][k])
        if i >= nsets:
            stream.wait_event(ev["down"][k])  # step i-nsets's outputs have left this output buffer
        step.select(k)
        with torch.cuda.stream(stream):
            if graphs is not None:
                graphs[k].replay()
            else:
                plans[k]()
        ev["kern"][k].record(stream)
        down.wait_event(ev["kern"][k])
        with torch.cuda.stream(down):
            b["h_outbuf"].copy_(b["d_out"], non_blocking=True)
        ev["down"][k].record(down)
        if i >= nsets - 1:  # step i-nsets+1's outputs, in pinned host memory; its set is reused next
            kk = (i + 1) % nsets
            ev["down"][kk].synchronize()
            checksum += int(host_out[kk][:64].sum())
    for i in range(max(0, args.e2e_steps - nsets + 1), args.e2e_steps):  # the last steps' outputs
        kk = i % nsets
        ev["down"][kk].synchronize()
        checksum += int(host_out[kk][:64].sum())
    e2e_s = time.perf_counter() - t0
    step.select(0)
    e2e_s = reduce_max(e2e_s, ws, device)
    e2e_val = whole_job_gbs(total_bytes, args.e2e_steps, e2e_s, ws)

    value = whole_job_gbs(total_bytes, args.steps, ms * 1e-3, ws)
    n_dec = len(wl.decode_seqs)
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded; N(0,1) or U[-1,1] per workload)",
        "decode_tokens_per_s": round(ws * n_dec / (ms_per_step * 1e-3), 1) if n_dec else None,
        "config": {
            "workload": wl.name,
            "batch": n_dec,
            "q_heads": wl.q_heads, "kv_heads": wl.kv_heads, "head_dim": wl.head_dim,
            "block_size": wl.block_size, "num_blocks": wl.num_blocks,
            "allocator": {"waste_slots": step.alloc.stats()["waste_slots"],
                          "table_entries": int(np.sum(np.ceil(step.dec_lens / wl.block_size))) if n_dec else 0},
            "context_lens": [int(min(step.dec_lens)), int(max(step.dec_lens))] if n_dec else None,
            "mean_context": float(np.mean(step.dec_lens)) if n_dec else None,
            "split_tokens": step.split if n_dec else None,
            "queries_per_request": wl.q_len,
            "verify_impl": step.verify_impl if wl.q_len > 1 else None,
            "kv_layout": step.layout,
            "prefill_chunks": step.chunks if step.pre else None,
            "copy_pairs": step.n_pairs,
            "bytes_per_step": nb,
            "l2": (f"inputs larger than L2: {total_bytes / 1e6:.0f} MB moved per step vs {L2_BYTES / 1e6:.0f} MB L2"
                   if flush is None else
                   f"L2 flushed between steps ({2 * L2_BYTES / 1e6:.0f} MB written outside each step's event pair; "
                   f"{total_bytes / 1e6:.1f} MB moved per step)"),
            "parallelism": f"replicas x{ws}",
            "streams": (f"prefill on a second, highest-priority stream over {step.prefill_ctas or 'all'} CTAs, "
                        f"concurrent with decode" if step.side is not None else
                        "shared-prefix pass on a second, highest-priority stream, concurrent with the suffix decode"
                        if step.prefix_side is not None else "one"),
        },
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if step.layout != "paged":
        res["config"]["max_len"] = step.max_len
        if step.vkv is not None:
            vs = step.vkv.stats()
            res["config"]["vmm"] = {"page_bytes": vs["page_bytes"], "pages_mapped": vs["pages_mapped"],
                                    "bytes_committed": vs["bytes_committed"], "bytes_used": vs["bytes_used"],
                                    "step_failures": vs["step_failures"], "bytes_reserved": vs["bytes_reserved"],
                                    "map_calls": vs["map_calls"],
                                    "map_us_per_page": round(vs["total_map_ns"] / max(1, vs["map_calls"]) / 1e3, 2),
                                    "setup_s": round(step.vmm_setup_s, 3)}
    if step.dec and step.prefix_len:
        ub = nb["decode_unique"]
        # DRAM traffic of the call's dominant kernel, the suffix decode pass
        straffic = kernel_traffic(f"decode_partial_{wl.name}.md", "paged_kv_cache_76_gb300/csrc/decode.cu",
                                  wl.block_size)
        flops = 4 * len(wl.decode_seqs) * wl.q_heads * wl.head_dim * step.prefix_len
        res["roofline"] = {
            "kernel": "pa_decode_shared_prefix (tcgen05 prefix pass + suffix decode + merge)",
            "bound": "hbm",
            "achieved": round(ub / (dec_ms * 1e-3) / 1e9, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(ub / (dec_ms * 1e-3) / 1e9 / peak, 4),
            "traffic": straffic,
            "traffic_kernel": "decode_partial_kernel (suffix pass)",
            "algorithmic_bytes_per_launch": ub,
            "logical_bytes_per_launch": nb["decode"],
            "achieved_logical": round(nb["decode"] / (dec_ms * 1e-3) / 1e9, 1),
            "prefix_tokens": step.prefix_len,
            "prefix_tflops": round(flops / (dec_ms * 1e-3) / 1e12, 1),
            "avg_launch_ms": round(dec_ms, 5),
            **launch_pct,
            "timing": "CUDA events around each of K pa_decode_shared_prefix calls (3 kernels) on the bench "
                      "stream, in a second pass of the same K steps",
        }
    elif step.dec:
        dec_bytes = nb["decode"]
        achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
        prof = (f"decode_partial_{wl.name}.md" if step.layout == "paged" else
                f"decode_contiguous_{step.layout}_{wl.name}.md")
        verify = wl.q_len > 1
        traffic = (kernel_traffic(f"attn_tile_{wl.name}.md", "paged_kv_cache_76_gb300/csrc/attn_tile.cu",
                                  wl.block_size) if verify and step.verify_impl == "tc" else
                   kernel_traffic(prof, "paged_kv_cache_76_gb300/csrc/decode.cu", wl.block_size))
        res["roofline"] = {
            "kernel": ("attn_tile_kernel, causal over each request's k+1 queries (pa_verify_decode_tc)"
                       if verify and step.verify_impl == "tc" else
                       "decode_partial_kernel with q_len=k+1 + lse_merge (pa_verify_decode)" if verify
                       else "decode_partial_kernel" if step.layout == "paged" else
                       f"decode_partial_kernel, contiguous mode + lse_merge ({step.layout} memory)"),
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": dec_bytes,
            "avg_launch_ms": round(dec_ms, 5),
            **launch_pct,
            "timing": ("CUDA events around each of K pa_verify_decode_tc calls on the bench stream, in a second "
                       "pass of the same K steps" if verify and step.verify_impl == "tc" else
                       f"CUDA events around each of K pa_verify_decode calls (partial + merge kernels) on the "
                       f"bench stream, in a second pass of the same K steps" if verify else
                       "CUDA events around each of K contiguous decode calls (partial + merge kernels) on the "
                       "bench stream, in a second pass of the same K steps" if step.layout != "paged" else
                       "CUDA events around each of K decode_partial launches on the bench stream, "
                       "in a second pass of the same K steps"),
        }
        if verify:
            res["roofline"]["q_len"] = wl.q_len
        if "decode_unique" in nb and nb["decode_unique"] < dec_bytes:
            res["roofline"]["unique_bytes_per_launch"] = nb["decode_unique"]
            res["roofline"]["achieved_unique"] = round(nb["decode_unique"] / (dec_ms * 1e-3) / 1e9, 1)
            res["roofline"]["frac_unique"] = round(nb["decode_unique"] / (dec_ms * 1e-3) / 1e9 / peak, 4)
    elif step.pre:
        # prefill alone: the tcgen05 kernel is tensor-bound; causal QK^T + PV
        # flops of the visible (query, key) pairs against the measured bf16 peak
        tpeak, tkind = measured_tensor_peak()
        fl = nb["prefill_flops"]
        ptraffic = kernel_traffic(f"attn_tc_{wl.name}.md", "paged_kv_cache_76_gb300/csrc/attn_tc.cu", wl.block_size) \
            if wl.block_size >= 8 else None
        res["roofline"] = {
            "kernel": "attn_tc_kernel" if wl.block_size >= 8 else "chunked_prefill_kernel",
            "bound": "tensor",
            "achieved": round(fl / (dec_ms * 1e-3) / 1e12, 1),
            "peak": tpeak,
            "peak_kind": tkind,
            "unit": "TFLOP/s",
            "frac": round(fl / (dec_ms * 1e-3) / 1e12 / tpeak, 4),
            "traffic": ptraffic,
            "algorithmic_flops_per_launch": fl,
            "avg_launch_ms": round(dec_ms, 5),
            **launch_pct,
            "timing": "CUDA events around each of K chunked-prefill launches on the bench stream, in a second "
                      "pass of the same K steps",
        }
    res["e2e"] = {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                  "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps, "mode": e2e_mode,
                  "ms_per_step": round(e2e_s / args.e2e_steps * 1e3, 4)}
    if rank == 0 and not args.no_cpu_baseline:
        hs = HostStep(wl, value_seed=1000 * rank)
        units = hs.units()
        b, t_or, done, cpu = run_oracle_units(hs, units, args.cpu_budget)
        res["cpu_baseline"] = {
            "value": round(b / t_or / 1e9, 6), "unit": "GB/s",
            "cores": max(1, int(round(cpu / max(t_or, 1e-9)))),
            "kind": "oracle",
            "sample": f"{len(done)} of {len(units)} (request, kv-head) units of {wl.name}, "
                      f"first {len(done)} in order; {t_or:.1f} s of float64 NumPy oracle",
            "host_cores_available": len(os.sched_getaffinity(0)),
        }
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))
        if args.jsonl:
            with open(args.jsonl, "a") as f:
                f.write(json.dumps(res) + "\n")


def reference_arm(args, wl: W.Workload, ws: int):
    """The reference arm: the float64 CPU oracle, a bounded sample per step.

    Tables, slots and values come from HostStep (the oracle's allocator and
    host-drawn values); nothing here loads the CUDA library.
    """
    hs = HostStep(wl, value_seed=0)
    units = hs.units()
    per_step = max(1, len(units) // 64)
    # steps = per_step units each, rotating through the workload
    k = 0
    t_warm = time.perf_counter()
    for _ in range(args.warmup):  # at least 3 warm-up steps, then at most ~30 s of them
        run_oracle_units(hs, [units[(k + i) % len(units)] for i in range(per_step)], 1e9)
        k += per_step
        if k >= 3 * per_step and time.perf_counter() - t_warm > 30:
            break
    tot_b, tot_t, cpu_t, n_units, n_steps = 0.0, 0.0, 0.0, 0, 0
    for _ in range(args.steps):
        us = [units[(k + i) % len(units)] for i in range(per_step)]
        b, t, done, cpu = run_oracle_units(hs, us, 1e9)
        tot_b += b
        tot_t += t
        cpu_t += cpu
        n_units += len(done)
        n_steps += 1
        k += per_step
        if tot_t > 100:  # a bounded sample: the whole arm ends within a few minutes
            break
    val = tot_b / tot_t / 1e9  # rank 0 alone runs the oracle
    res = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(val, 6),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": n_steps,
        "warmup": args.warmup,
        "ms_per_step": round(tot_t / max(1, n_steps) * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "units_per_step": per_step,
                   "note": "each step is a bounded sample of the workload: per_step (request, kv-head) units"},
        "cpu_baseline": {"value": round(val, 6), "unit": "GB/s", "kind": "oracle",
                         "cores": max(1, int(round(cpu_t / max(tot_t, 1e-9)))),
                         "sample": f"{n_units} (request, kv-head) units of {wl.name}"},
        "e2e": {"value": round(val, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res))


if __name__ == "__main__":
    main()
