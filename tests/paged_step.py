"""Run one workload step on each side, independently.

* ``oracle_step``: the oracle's Python allocator replays the workload script,
  then the float64 oracle applies copy_blocks, reshape_and_cache, chunked
  prefill and decode to the pre-step pool.
* ``device_step``: the C++ allocator (through the C ABI) replays the same
  script, then the CUDA kernels run the same step on the GPU.

They share only the workload description and the seeded input tensors.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from oracle import paged_attention as opa
from oracle.block_pool import SequenceManager

TOL_MAX = 1e-2    # max-abs error vs the float64 oracle
TOL_MEAN = 1e-3   # mean-abs error vs the float64 oracle
# The output is stored once in the input type (round to nearest even): half
# an ulp, at most 2^-8 |x| in bf16 (8 significant bits) and 2^-11 |x| in fp16.
# It matters only where a row's softmax is nearly one-hot and the output is a
# V row of magnitude ~4 (inputs built for that: assert_close(..., rounding=True));
# averages over many keys stay far below 1e-2 with it or without it.
OUT_ROUNDING = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11, torch.float32: 0.0}


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def raw16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy()


def padded(tables, width):
    out = np.full((len(tables), max(width, 1)), -1, dtype=np.int64)
    for i, t in enumerate(tables):
        out[i, :len(t)] = t
    return out


def oracle_step(wl: W.Workload, vals: dict, decode_rows=None, prefill_rows=None, compact=False):
    """Float64 reference of one step.

    ``decode_rows`` / ``prefill_rows`` restrict the attention work to sampled
    outputs.  ``compact`` copies only the physical blocks those outputs read
    into a small pool (blocks renumbered, slots and copy pairs remapped, other
    tokens' writes dropped); the oracle's output does not depend on physical
    block ids (pinned by the relabelling test of the oracle), so this is the
    same computation on a smaller pool.
    """
    m = SequenceManager(wl.num_blocks, wl.block_size, wl.free_order)
    m.run(wl.setup_ops)
    slots, pairs = m.run(wl.step_ops)
    bs = wl.block_size
    dec_seqs = wl.decode_seqs if decode_rows is None else [wl.decode_seqs[i] for i in decode_rows]
    dec_idx = list(range(len(wl.decode_seqs))) if decode_rows is None else list(decode_rows)
    pre_seqs = [s for s, _, _ in wl.prefill]
    remap = None
    if compact:
        need = set()
        for s in list(dec_seqs) + pre_seqs:
            need |= set(m.block_table(s))
        pairs = [(a, b) for a, b in pairs if b in need]
        need |= {a for a, _ in pairs}
        ids = sorted(need)
        remap = {b: i for i, b in enumerate(ids)}
        idx = torch.as_tensor(ids, dtype=torch.long, device=vals["k_cache"].device)
        kc, vc = to_f64(vals["k_cache"][idx]), to_f64(vals["v_cache"][idx])
        slots = [remap[x // bs] * bs + x % bs if x // bs in remap else -1 for x in slots]
        pairs = [(remap[a], remap[b]) for a, b in pairs]
    else:
        kc, vc = to_f64(vals["k_cache"]), to_f64(vals["v_cache"])
    tab = (lambda s: [remap[b] for b in m.block_table(s)]) if remap else m.block_table
    if pairs:
        kc, vc = opa.copy_blocks(kc, vc, pairs)
    kc, vc = opa.reshape_and_cache(to_f64(vals["k_new"]), to_f64(vals["v_new"]), slots, kc, vc)
    res = {"slots": slots, "pairs": pairs, "k_cache": kc, "v_cache": vc, "manager": m}
    if wl.decode_seqs:
        tabs = [tab(s) for s in dec_seqs]
        lens = [m.num_tokens[s] for s in dec_seqs]
        q = to_f64(vals["q_decode"])[dec_idx]
        attend = opa.decode if wl.q_len == 1 else opa.verify_decode
        res["decode"] = attend(q, kc, vc, padded(tabs, max(map(len, tabs))), lens, wl.scale)
        res["decode_lens"] = lens
    if wl.prefill:
        tabs = [tab(s) for s in pre_seqs]
        lens = [m.num_tokens[s] for s in pre_seqs]
        q_start = np.concatenate([[0], np.cumsum([c for _, c, _ in wl.prefill])])
        q = to_f64(vals["q_prefill"])
        res["prefill"] = opa.chunked_prefill(q, q_start, lens, kc, vc, padded(tabs, max(map(len, tabs))),
                                             wl.scale, rows=prefill_rows)
        res["prefill_lens"] = lens
    return res


class DeviceStep:
    """Device-side state of one workload step (allocator tables, buffers)."""

    def __init__(self, wl: W.Workload, vals: dict, device="cuda", split_tokens=None):
        from paged_kv_cache_76_gb300.allocator import BlockAllocator
        self.wl = wl
        self.dev = torch.device(device)
        a = BlockAllocator(wl.num_blocks, wl.block_size, wl.free_order)
        a.run(wl.setup_ops)
        slots, pairs = a.run(wl.step_ops)
        self.alloc = a
        self.slots_host = np.asarray(slots, dtype=np.int32)
        self.pairs_host = np.asarray(pairs, dtype=np.int32).reshape(-1, 2)
        self.split_tokens = wl.split_tokens if split_tokens is None else split_tokens
        d = self.dev
        # private copies: the step writes the pool, the caller's tensors stay the pre-step input
        self.k_cache = vals["k_cache"].to(d, copy=True).contiguous()
        self.v_cache = vals["v_cache"].to(d, copy=True).contiguous()
        self.k_new = vals["k_new"].to(d).contiguous()
        self.v_new = vals["v_new"].to(d).contiguous()
        self.slots = torch.from_numpy(self.slots_host).to(d)
        self.pairs = torch.from_numpy(self.pairs_host).to(d)
        if wl.decode_seqs:
            maxblk = max(len(a.block_table(s)) for s in wl.decode_seqs)
            t, l = a.build_tables(wl.decode_seqs, maxblk)
            self.dec_tables_host, self.dec_lens_host = t, l
            self.dec_tables = torch.from_numpy(t).to(d)
            self.dec_lens = torch.from_numpy(l).to(d)
            self.q_decode = vals["q_decode"].to(d).contiguous()
            self.out_decode = torch.empty_like(self.q_decode)
            from paged_kv_cache_76_gb300 import ops
            if wl.q_len == 1:
                self.workspace = ops.make_workspace(self.q_decode, self.dec_tables, wl.block_size, self.split_tokens)
            else:
                n = ops.verify_workspace_size(len(wl.decode_seqs), wl.q_len, wl.q_heads, wl.head_dim, maxblk,
                                              wl.block_size, self.split_tokens)
                self.workspace = torch.empty(n, dtype=torch.uint8, device=d) if n else None
        if wl.prefill:
            seqs = [s for s, _, _ in wl.prefill]
            maxblk = max(len(a.block_table(s)) for s in seqs)
            t, l = a.build_tables(seqs, maxblk)
            self.pre_tables_host, self.pre_lens_host = t, l
            self.pre_tables = torch.from_numpy(t).to(d)
            self.pre_lens = torch.from_numpy(l).to(d)
            qs = np.concatenate([[0], np.cumsum([c for _, c, _ in wl.prefill])]).astype(np.int32)
            self.q_start = torch.from_numpy(qs).to(d)
            self.max_q_len = max(c for _, c, _ in wl.prefill)
            self.q_prefill = vals["q_prefill"].to(d).contiguous()
            self.out_prefill = torch.empty_like(self.q_prefill)

    def run(self, stream=None):
        """copy_blocks -> reshape_and_cache -> chunked prefill -> decode, one stream."""
        from paged_kv_cache_76_gb300 import ops
        wl = self.wl
        if self.pairs.shape[0]:
            ops.copy_blocks(self.k_cache, self.v_cache, self.pairs, stream=stream)
        ops.reshape_and_cache(self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache, stream=stream)
        if wl.prefill:
            ops.chunked_prefill(self.q_prefill, self.q_start, self.pre_lens, self.k_cache, self.v_cache,
                                self.pre_tables, wl.scale, self.max_q_len, out=self.out_prefill, stream=stream)
        if wl.decode_seqs:
            attend = ops.decode if wl.q_len == 1 else ops.verify_decode
            attend(self.q_decode, self.k_cache, self.v_cache, self.dec_tables, self.dec_lens, wl.scale,
                   out=self.out_decode, split_tokens=self.split_tokens, workspace=self.workspace, stream=stream)


def assert_close(got: torch.Tensor, ref: np.ndarray, what="", rounding=False):
    """max-abs <= TOL_MAX and mean-abs <= TOL_MEAN against the oracle; with
    ``rounding``, the max-abs bound also admits the output's own rounding."""
    g = to_f64(got)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - ref)
    excess = err - (OUT_ROUNDING[got.dtype] * np.abs(ref) if rounding else 0.0)
    assert excess.max() <= TOL_MAX, f"{what}: max-abs {err.max():.3g} (beyond the allowed rounding " \
                                    f"{excess.max():.3g}) > {TOL_MAX}"
    assert err.mean() <= TOL_MEAN, f"{what}: mean-abs {err.mean():.3g} > {TOL_MEAN}"
    return float(err.max()), float(err.mean())
