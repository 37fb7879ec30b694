"""Python handle over the vAttention-style contiguous virtual KV manager
(``pa_vkv_*`` and ``pa_decode_contiguous`` in include/pa.h): argument
marshalling only; the mapping, the bookkeeping and the kernels are the
library's."""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import _lib
from ._lib import PA_ERR_NO_FREE_BLOCKS, PAError, check
from .ops import _keep, _launch

__all__ = ["VirtualKV", "NoPages", "decode_contiguous", "reshape_and_cache_slots"]


class NoPages(PAError):
    """The page budget cannot cover the step; nothing changed."""


def _chk(st, what):
    if st == PA_ERR_NO_FREE_BLOCKS:
        raise NoPages(st, what)
    return check(st, what)


def _stream(stream=None):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _dev(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t.data_ptr()


def _i32(t, name):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return _dev(t, name)


def _rows(ref, *named):
    """Each (name, tensor, rows) is on ref's device with `rows` leading entries:
    the C calls read them by pointer, past their end otherwise."""
    for name, t, rows in named:
        if t.device != ref.device:
            raise ValueError(f"{name} is on {t.device}, not {ref.device}")
        if t.dim() == 0 or t.shape[0] != rows:
            raise ValueError(f"{name} has shape {tuple(t.shape)}: {rows} rows expected")


def _check_contiguous_kv(k_cache, v_cache, dtype, head_dim):
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("caches are [num_slots, max_len, kv_heads, head_dim], K and V alike")
    if k_cache.dtype != dtype or v_cache.dtype != dtype or k_cache.shape[3] != head_dim:
        raise ValueError("the caches must have the data's dtype and head_dim")
    if v_cache.device != k_cache.device:
        raise ValueError("k_cache and v_cache must be on one device")


def _code(dt):
    if dt == torch.bfloat16:
        return _lib.PA_BF16
    if dt == torch.float16:
        return _lib.PA_FP16
    raise TypeError(f"unsupported dtype {dt}")


class _CudaArray:
    """A device range exposed through the CUDA array interface (no copy)."""

    def __init__(self, ptr, shape, typestr, owner):
        self.__cuda_array_interface__ = {"data": (ptr, False), "shape": tuple(shape), "typestr": typestr,
                                         "version": 3, "strides": None}
        self._owner = owner


class VirtualKV:
    """Contiguous virtual K/V tensors [num_slots][max_len][kv_heads][head_dim] per layer."""

    def __init__(self, num_slots, max_len, num_layers, kv_heads, head_dim, dtype=torch.bfloat16, page_bytes=0,
                 max_pages=1 << 40, dry_run=False):
        self._L = _lib.lib()
        self.num_slots, self.max_len, self.num_layers = int(num_slots), int(max_len), int(num_layers)
        self.kv_heads, self.head_dim, self.dtype = int(kv_heads), int(head_dim), dtype
        h = C.c_void_p()
        _chk(self._L.pa_vkv_create(self.num_slots, self.max_len, self.num_layers, self.kv_heads, self.head_dim,
                                   _code(dtype), int(page_bytes), int(max_pages),
                                   _lib.PA_VKV_DRY_RUN if dry_run else 0, C.byref(h)), "pa_vkv_create")
        self._h = h
        self.dry_run = dry_run

    def close(self):
        if getattr(self, "_h", None):
            self._L.pa_vkv_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def granularity() -> int:
        g = C.c_size_t(0)
        check(_lib.lib().pa_vkv_granularity(C.byref(g)), "pa_vkv_granularity")
        return int(g.value)

    def alloc_slot(self) -> int:
        s = C.c_int(-1)
        _chk(self._L.pa_vkv_alloc_slot(self._h, C.byref(s)), "pa_vkv_alloc_slot")
        return int(s.value)

    def free_slot(self, slot: int):
        _chk(self._L.pa_vkv_free_slot(self._h, int(slot)), "pa_vkv_free_slot")

    def step(self, lens, stream=None):
        a = np.ascontiguousarray(lens, dtype=np.int32)
        if a.shape != (self.num_slots,):
            raise ValueError("one length per slot")
        st = None if self.dry_run else _stream(stream)
        _chk(self._L.pa_vkv_step(self._h, a.ctypes.data_as(C.POINTER(C.c_int32)), st), "pa_vkv_step")

    def slot_pages(self, slot: int) -> int:
        return _chk(self._L.pa_vkv_slot_pages(self._h, int(slot)), "pa_vkv_slot_pages")

    def slot_tokens(self) -> np.ndarray:
        out = np.empty(self.num_slots, dtype=np.int32)
        _chk(self._L.pa_vkv_slot_tokens(self._h, out.ctypes.data_as(C.POINTER(C.c_int32)), None),
             "pa_vkv_slot_tokens")
        return out

    def stats(self) -> dict:
        s = _lib.VkvStats()
        _chk(self._L.pa_vkv_get_stats(self._h, C.byref(s)), "pa_vkv_get_stats")
        return {n: int(getattr(s, n)) for n, _ in s._fields_}

    def tensor(self, layer: int, is_v: bool) -> torch.Tensor:
        """Layer ``layer``'s K or V as a torch view of the virtual range (rows
        past a slot's mapped pages must not be touched)."""
        p = C.c_void_p()
        _chk(self._L.pa_vkv_tensor(self._h, int(layer), int(bool(is_v)), C.byref(p)), "pa_vkv_tensor")
        if not p.value:
            raise ValueError("no memory in dry-run mode")
        shape = (self.num_slots, self.max_len, self.kv_heads, self.head_dim)
        # the array interface has no bf16: expose 16-bit integers and view them
        t = torch.as_tensor(_CudaArray(p.value, shape, "<i2", self), device="cuda")
        return t.view(self.dtype)

    def decode(self, layer, q, slot_ids, context_lens, scale, out=None, split_tokens=0, workspace=None,
               stream=None):
        B, hq, d = q.shape
        if out is None:
            out = torch.empty_like(q)
        if d != self.head_dim or q.dtype != self.dtype or out.dtype != q.dtype or out.shape != q.shape:
            raise ValueError("q and out are [num_seqs, q_heads, head_dim] of the KV's head_dim and dtype")
        _rows(q, ("slot_ids", slot_ids, B), ("context_lens", context_lens, B), ("out", out, B))
        if workspace is None:
            n = int(self._L.pa_decode_workspace_size(B, hq, d, self.max_len // 16, 16, int(split_tokens)))
            workspace = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
        ws, wb = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
        _keep(out, workspace)
        _launch("pa_vkv_decode", self._h, int(layer), _dev(q, "q"), _i32(slot_ids, "slot_ids"),
                _i32(context_lens, "context_lens"), B, hq, float(scale), int(split_tokens), ws, wb, _dev(out, "out"),
                _stream(stream))
        return out

    def reshape_and_cache(self, layer, k, v, slot_ids, positions, stream=None):
        if k.shape != v.shape or k.dim() != 3 or tuple(k.shape[1:]) != (self.kv_heads, self.head_dim) or \
                k.dtype != self.dtype or v.dtype != self.dtype:
            raise ValueError("k and v are [num_tokens, kv_heads, head_dim] of the KV's dtype")
        n = int(k.shape[0])
        _rows(k, ("v", v, n), ("slot_ids", slot_ids, n), ("positions", positions, n))
        _launch("pa_vkv_reshape_and_cache", self._h, int(layer), _dev(k, "k"), _dev(v, "v"),
                _i32(slot_ids, "slot_ids"), _i32(positions, "positions"), int(k.shape[0]), _stream(stream))


def decode_contiguous(q, k_cache, v_cache, slot_ids, context_lens, scale, slot_tokens=None, out=None,
                      split_tokens=0, workspace=None, stream=None):
    """pa_decode_contiguous over plain [num_slots][max_len][kv_heads][head_dim] tensors."""
    ns, L, hkv, d = k_cache.shape
    B, hq, dq = q.shape
    if out is None:
        out = torch.empty_like(q)
    _check_contiguous_kv(k_cache, v_cache, q.dtype, dq)
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must have q's shape and dtype")
    _rows(q, ("context_lens", context_lens, B), ("out", out, B), ("k_cache", k_cache, ns))
    if slot_ids is not None:
        _rows(q, ("slot_ids", slot_ids, B))
    if slot_tokens is not None:
        _rows(q, ("slot_tokens", slot_tokens, ns))
    lib = _lib.lib()
    if workspace is None:
        n = int(lib.pa_decode_workspace_size(B, hq, d, L // 16, 16, int(split_tokens)))
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    ws, wb = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    _keep(out, workspace)
    _launch(
        "pa_decode_contiguous",
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ns, L,
        _i32(slot_ids, "slot_ids") if slot_ids is not None else None,
        _i32(slot_tokens, "slot_tokens") if slot_tokens is not None else None, _i32(context_lens, "context_lens"),
        B, hq, hkv, d, float(scale), int(split_tokens), ws, wb, _dev(out, "out"), _code(q.dtype), _stream(stream))
    return out


def reshape_and_cache_slots(k, v, slot_ids, positions, k_cache, v_cache, slot_tokens=None, stream=None):
    ns, L, hkv, d = k_cache.shape
    _check_contiguous_kv(k_cache, v_cache, k.dtype, d)
    if k.shape != v.shape or k.dim() != 3 or tuple(k.shape[1:]) != (hkv, d) or v.dtype != k.dtype:
        raise ValueError("k and v are [num_tokens, kv_heads, head_dim] of the cache")
    n = int(k.shape[0])
    _rows(k, ("v", v, n), ("slot_ids", slot_ids, n), ("positions", positions, n), ("k_cache", k_cache, ns))
    if slot_tokens is not None:
        _rows(k, ("slot_tokens", slot_tokens, ns))
    _launch(
        "pa_reshape_and_cache_slots",
        _dev(k, "k"), _dev(v, "v"), _i32(slot_ids, "slot_ids"), _i32(positions, "positions"), int(k.shape[0]),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), ns, L,
        _i32(slot_tokens, "slot_tokens") if slot_tokens is not None else None, hkv, d, _code(k.dtype),
        _stream(stream))
