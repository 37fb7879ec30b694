"""Torch-tensor binding of the paged-KV C ABI (argument marshalling only).

Every function passes ``data_ptr()`` values, sizes and the current CUDA
stream to the function of the same name in ``include/pa.h``; all work runs in
the library's kernels.  Tensors must be contiguous CUDA tensors of the
documented shapes; int32 index tensors live on the same device.
"""
from __future__ import annotations

import math
import threading

import torch

from . import _lib
from ._lib import PA_BF16, PA_FP16, check

__all__ = [
    "reshape_and_cache",
    "copy_blocks",
    "swap_blocks",
    "decode",
    "decode_partial",
    "lse_merge",
    "decode_split_tokens",
    "decode_workspace_size",
    "chunked_prefill",
    "decode_shared_prefix",
    "decode_shared_prefix_workspace_size",
    "decode_shared_prefix_split_tokens",
    "verify_decode",
    "verify_split_tokens",
    "verify_workspace_size",
    "get_device_error",
    "selftest_wait_timeout",
    "launch_count",
    "dtype_code",
    "recording",
    "Recording",
]


def dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return PA_BF16
    if dt == torch.float16:
        return PA_FP16
    raise TypeError(f"unsupported dtype {dt}: use torch.bfloat16 or torch.float16")


class Recording:
    """Library launches marshalled once, to be issued again as they are.

    Inside ``with recording() as rec:`` the launching functions of this module
    check and marshal their arguments but launch nothing: each appends a
    callable to ``rec.steps`` that issues the same C call with the same
    pointers, sizes and streams.  ``rec.add(fn)`` appends any other step (an
    event record or wait) in order.  ``rec()`` runs the steps in order: the
    same launches for a fraction of the host time of the marshalling (the
    tensors must stay alive and in place).  A recording belongs to the thread
    that opened it; other threads launch as usual meanwhile.
    """

    def __init__(self):
        self.steps = []
        self.keep = []  # tensors a recorded launch writes or reads that the caller did not pass in

    def add(self, fn):
        self.steps.append(fn)

    def __call__(self):
        for fn in self.steps:
            fn()


_tls = threading.local()  # .rec: the open recording of this thread, if any


class recording:
    """Context manager: see :class:`Recording`."""

    def __enter__(self) -> Recording:
        if getattr(_tls, "rec", None) is not None:
            raise RuntimeError("recordings do not nest")
        _tls.rec = Recording()
        return _tls.rec

    def __exit__(self, *exc):
        _tls.rec = None
        return False


def _keep(*tensors) -> None:
    """Inside a recording, keep tensors allocated by the call alive with the recording."""
    rec = getattr(_tls, "rec", None)
    if rec is not None:
        rec.keep.extend(t for t in tensors if t is not None)


def _launch(name: str, *args) -> None:
    """Issue (or, inside a recording, record) the C call `name`(*args)."""
    fn = getattr(_lib.lib(), name)
    rec = getattr(_tls, "rec", None)
    if rec is not None:
        rec.add(lambda: check(fn(*args), name))
        return
    check(fn(*args), name)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return _dev(t, name)


def _cache_dims(k_cache: torch.Tensor):
    if k_cache.dim() != 4:
        raise ValueError("caches are [num_blocks, block_size, kv_heads, head_dim]")
    return k_cache.shape


# The C calls take raw pointers and sizes; these checks are what keeps a
# mismatched tensor from being read as the wrong type, past its end, or from
# another GPU's memory.
def _check_caches(k_cache, v_cache):
    _cache_dims(k_cache)
    if v_cache.shape != k_cache.shape or v_cache.dtype != k_cache.dtype or v_cache.device != k_cache.device:
        raise ValueError("k_cache and v_cache must agree in shape, dtype and device")


def _check_index(ref, name: str, t, rows: int, cols: int = None, table: bool = False):
    """An index tensor on ref's device with `rows` leading entries; 2-D with
    `cols` columns if given, 2-D if `table`."""
    if t.device != ref.device:
        raise ValueError(f"{name} is on {t.device}, not {ref.device}")
    two_d = table or cols is not None
    if t.dim() == 0 or t.shape[0] != rows or (two_d and t.dim() != 2) or (cols is not None and t.shape[1] != cols):
        raise ValueError(f"{name} has shape {tuple(t.shape)}: {rows} rows{' x ' + str(cols) if cols else ''} expected")


def _check_attention(q, k_cache, v_cache, out):
    """q, both caches and out share one dtype and device; out has q's shape."""
    _check_caches(k_cache, v_cache)
    if k_cache.dtype != q.dtype or out.dtype != q.dtype:
        raise TypeError(f"q ({q.dtype}), the caches ({k_cache.dtype}) and out ({out.dtype}) must share a dtype")
    if k_cache.device != q.device or out.device != q.device:
        raise ValueError("q, the caches and out must be on one device")
    if out.shape != q.shape:
        raise ValueError(f"out has shape {tuple(out.shape)}, q {tuple(q.shape)}")


def launch_count() -> int:
    return int(_lib.lib().pa_launch_count())


def reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, stream=None):
    nb, bs, hkv, d = _cache_dims(k_cache)
    _check_caches(k_cache, v_cache)
    if k.shape != v.shape or k.dim() != 3 or k.shape[1:] != (hkv, d):
        raise ValueError("k and v are [num_tokens, kv_heads, head_dim] of the cache")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype or k.device != k_cache.device or v.device != k.device:
        raise ValueError("k and v must have the cache's dtype and device")
    _check_index(k, "slot_mapping", slot_mapping, int(k.shape[0]))
    _launch(
        "pa_reshape_and_cache",
        _dev(k, "k"), _dev(v, "v"), _i32(slot_mapping, "slot_mapping"), int(k.shape[0]),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), nb, bs, hkv, d, dtype_code(k_cache.dtype),
        _stream(stream))


def copy_blocks(k_cache, v_cache, pairs, stream=None):
    """``pairs``: int32 [n, 2] (src, dst) on the cache's device."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    _check_caches(k_cache, v_cache)
    _check_index(k_cache, "pairs", pairs, int(pairs.shape[0]) if pairs.dim() else -1, 2)
    _launch(
        "pa_copy_blocks",
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _i32(pairs, "pairs"), int(pairs.shape[0]),
        nb, bs, hkv, d, dtype_code(k_cache.dtype), _stream(stream))


def _dev_or_pinned(t: torch.Tensor, name: str):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    return t.data_ptr()


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs, stream=None):
    """Copy blocks between two pools of the cache layout, either of which may
    live in pinned host memory (``pin_memory=True``); ``pairs``: int32 [n, 2]
    (src, dst), on the device or pinned.  Asynchronous on ``stream``."""
    if src_v.shape != src_k.shape or dst_v.shape != dst_k.shape or src_k.shape[1:] != dst_k.shape[1:] \
            or src_k.dtype != dst_k.dtype or src_v.dtype != src_k.dtype or dst_v.dtype != dst_k.dtype:
        raise ValueError("the pools must agree in block shape and dtype")
    if pairs.dtype != torch.int32:
        raise TypeError("pairs must be int32")
    ns, bs, hkv, d = _cache_dims(src_k)
    nd = dst_k.shape[0]
    _launch(
        "pa_swap_blocks",
        _dev_or_pinned(src_k, "src_k"), _dev_or_pinned(src_v, "src_v"), _dev_or_pinned(dst_k, "dst_k"),
        _dev_or_pinned(dst_v, "dst_v"), _dev_or_pinned(pairs, "pairs"), int(pairs.shape[0]), ns, nd, bs, hkv, d,
        dtype_code(src_k.dtype), _stream(stream))


def decode_split_tokens(max_blocks_per_seq: int, block_size: int, split_tokens: int = 0) -> int:
    return check(_lib.lib().pa_decode_split_tokens(max_blocks_per_seq, block_size, split_tokens),
                 "pa_decode_split_tokens")


def decode_workspace_size(num_seqs, q_heads, head_dim, max_blocks_per_seq, block_size, split_tokens=0) -> int:
    return int(_lib.lib().pa_decode_workspace_size(num_seqs, q_heads, head_dim, max_blocks_per_seq,
                                                   block_size, split_tokens))


def _check_decode(q, k_cache, v_cache, block_tables, context_lens, out):
    nb, bs, hkv, d = _cache_dims(k_cache)
    if q.dim() != 3 or q.shape[2] != d:
        raise ValueError("q is [num_seqs, q_heads, head_dim] of the cache's head_dim")
    _check_attention(q, k_cache, v_cache, out)
    _check_index(q, "block_tables", block_tables, int(q.shape[0]), table=True)
    _check_index(q, "context_lens", context_lens, int(q.shape[0]))


def _decode_args(q, k_cache, v_cache, block_tables, context_lens, scale, out, split_tokens, workspace):
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, dq = q.shape
    _check_decode(q, k_cache, v_cache, block_tables, context_lens, out)
    maxblk = int(block_tables.shape[1])
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) \
        if workspace is not None else (None, 0)
    return (_dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _i32(block_tables, "block_tables"),
            maxblk, _i32(context_lens, "context_lens"), B, hq, hkv, d, bs, nb, float(scale), int(split_tokens),
            ws_ptr, ws_bytes, _dev(out, "out"), dtype_code(q.dtype))


def make_workspace(q, block_tables, block_size, split_tokens=0):
    """Allocate (with torch) the scratch that :func:`decode` needs, or None."""
    B, hq, d = q.shape
    n = decode_workspace_size(B, hq, d, int(block_tables.shape[1]), block_size, split_tokens)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, split_tokens=0, workspace=None,
           stream=None):
    if out is None:
        out = torch.empty_like(q)
    _check_decode(q, k_cache, v_cache, block_tables, context_lens, out)
    if workspace is None:
        workspace = make_workspace(q, block_tables, k_cache.shape[1], split_tokens)
    args = _decode_args(q, k_cache, v_cache, block_tables, context_lens, scale, out, split_tokens, workspace)
    _keep(out, workspace)
    _launch("pa_decode", *args, _stream(stream))
    return out


def decode_partial(q, k_cache, v_cache, block_tables, context_lens, scale, out, split_tokens=0, workspace=None,
                   stream=None):
    args = _decode_args(q, k_cache, v_cache, block_tables, context_lens, scale, out, split_tokens, workspace)
    _launch("pa_decode_partial", *args, _stream(stream))


def lse_merge(workspace, context_lens, q, block_tables, block_size, out, split_tokens=0, stream=None):
    B, hq, d = q.shape
    if out.shape != q.shape or out.device != q.device:
        raise ValueError("out must have q's shape and device")
    _check_index(q, "context_lens", context_lens, B)
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) \
        if workspace is not None else (None, 0)
    _launch("pa_lse_merge", ws_ptr, ws_bytes, _i32(context_lens, "context_lens"), B, hq, d,
            int(block_tables.shape[1]), block_size, int(split_tokens), _dev(out, "out"), dtype_code(out.dtype),
            _stream(stream))


def verify_split_tokens(max_blocks_per_seq: int, block_size: int, q_len: int, split_tokens: int = 0) -> int:
    return check(_lib.lib().pa_verify_split_tokens(max_blocks_per_seq, block_size, q_len, split_tokens),
                 "pa_verify_split_tokens")


def verify_workspace_size(num_seqs, q_len, q_heads, head_dim, max_blocks_per_seq, block_size, split_tokens=0) -> int:
    return int(_lib.lib().pa_verify_workspace_size(num_seqs, q_len, q_heads, head_dim, max_blocks_per_seq,
                                                   block_size, split_tokens))


def verify_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, split_tokens=0, workspace=None,
                  stream=None):
    """pa_verify_decode: ``q`` is [num_seqs, k+1, q_heads, head_dim]; query i of
    request r sees its first ``context_lens[r] - k + i`` tokens."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    if q.dim() != 4:
        raise ValueError("q is [num_seqs, q_len, q_heads, head_dim]")
    B, ql, hq, dq = q.shape
    if out is None:
        out = torch.empty_like(q)
    if dq != d:
        raise ValueError("head_dim mismatch")
    _check_attention(q, k_cache, v_cache, out)
    _check_index(q, "block_tables", block_tables, B, table=True)
    _check_index(q, "context_lens", context_lens, B)
    maxblk = int(block_tables.shape[1])
    if workspace is None:
        n = verify_workspace_size(B, ql, hq, d, maxblk, bs, split_tokens)
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel() * workspace.element_size()) \
        if workspace is not None else (None, 0)
    _keep(out, workspace)
    _launch(
        "pa_verify_decode",
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _i32(block_tables, "block_tables"), maxblk,
        _i32(context_lens, "context_lens"), B, ql, hq, hkv, d, bs, nb, float(scale), int(split_tokens), ws_ptr,
        ws_bytes, _dev(out, "out"), dtype_code(q.dtype), _stream(stream))
    return out


def decode_shared_prefix_workspace_size(num_seqs, q_heads, head_dim, max_blocks_per_seq, block_size, prefix_len,
                                        split_tokens=0) -> int:
    return int(_lib.lib().pa_decode_shared_prefix_workspace_size(num_seqs, q_heads, head_dim, max_blocks_per_seq,
                                                                 block_size, prefix_len, split_tokens))


def decode_shared_prefix_split_tokens(max_blocks_per_seq, block_size, prefix_len, split_tokens=0) -> int:
    """Suffix partition size pa_decode_shared_prefix uses (0: its automatic choice)."""
    return check(_lib.lib().pa_decode_shared_prefix_split_tokens(int(max_blocks_per_seq), int(block_size),
                                                                 int(prefix_len), int(split_tokens)),
                 "pa_decode_shared_prefix_split_tokens")


def decode_shared_prefix(q, k_cache, v_cache, prefix_blocks, prefix_len, block_tables, context_lens, scale, out=None,
                         split_tokens=0, workspace=None, stream=None, prefix_stream=None):
    """pa_decode_shared_prefix: decode whose requests share ``prefix_blocks`` (int32, device).

    ``prefix_stream`` (a torch.cuda.Stream): run the prefix pass there,
    concurrently with the suffix pass; the caller orders it after the writes
    of ``q``, the prefix's K/V and the previous use of ``workspace``."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, hq, dq = q.shape
    if dq != d:
        raise ValueError("head_dim mismatch")
    if out is None:
        out = torch.empty_like(q)
    _check_attention(q, k_cache, v_cache, out)
    _check_index(q, "block_tables", block_tables, B, table=True)
    _check_index(q, "context_lens", context_lens, B)
    if prefix_blocks.device != q.device or prefix_blocks.numel() < int(prefix_len) // bs:
        raise ValueError("prefix_blocks must hold prefix_len / block_size block ids on q's device")
    maxblk = int(block_tables.shape[1])
    if workspace is None:
        n = decode_shared_prefix_workspace_size(B, hq, d, maxblk, bs, int(prefix_len), split_tokens)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    _keep(out, workspace)
    _launch(
        "pa_decode_shared_prefix",
        _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _i32(prefix_blocks, "prefix_blocks"),
        int(prefix_len), _i32(block_tables, "block_tables"), maxblk, _i32(context_lens, "context_lens"), B, hq, hkv,
        d, bs, nb, float(scale), int(split_tokens), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _dev(out, "out"),
        dtype_code(q.dtype), _stream(stream), prefix_stream.cuda_stream if prefix_stream is not None else None)
    return out


def verify_decode_tc(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, max_ctas=0, stream=None):
    """pa_verify_decode_tc: ``q`` is [num_seqs, k+1, q_heads, head_dim]; the
    verify attention on the tcgen05 kernel (no workspace)."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    B, ql, hq, dq = q.shape
    if dq != d:
        raise ValueError("head_dim mismatch")
    if out is None:
        out = torch.empty_like(q)
    _check_attention(q, k_cache, v_cache, out)
    _check_index(q, "block_tables", block_tables, B, table=True)
    _check_index(q, "context_lens", context_lens, B)
    _keep(out)
    _launch("pa_verify_decode_tc", _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
            _i32(block_tables, "block_tables"), int(block_tables.shape[1]), _i32(context_lens, "context_lens"), B,
            ql, hq, hkv, d, bs, nb, float(scale), int(max_ctas), _dev(out, "out"), dtype_code(q.dtype),
            _stream(stream))
    return out


def chunked_prefill(q, q_start, context_lens, k_cache, v_cache, block_tables, scale, max_q_len, out=None,
                    stream=None, max_ctas=0):
    """pa_chunked_prefill; ``max_ctas`` > 0 caps the CTAs (SMs) the tensor-core path uses."""
    nb, bs, hkv, d = _cache_dims(k_cache)
    T, hq, dq = q.shape
    if dq != d:
        raise ValueError("head_dim mismatch")
    R = int(context_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    _check_attention(q, k_cache, v_cache, out)
    _check_index(q, "context_lens", context_lens, R)
    _check_index(q, "q_start", q_start, R + 1)
    _check_index(q, "block_tables", block_tables, R, table=True)
    _keep(out)
    _launch(
        "pa_chunked_prefill",
        _dev(q, "q"), _i32(q_start, "q_start"), _i32(context_lens, "context_lens"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"), _i32(block_tables, "block_tables"), int(block_tables.shape[1]), R, T,
        int(max_q_len), int(max_ctas), hq, hkv, d, bs, nb, float(scale), _dev(out, "out"), dtype_code(q.dtype),
        _stream(stream))
    return out


def selftest_wait_timeout(wait_ms: int = 50, stream=None) -> None:
    """Launch the library's bounded-wait self-test (pa_selftest_wait_timeout):
    afterwards the error word holds PA_DEVERR_TIMEOUT."""
    check(_lib.lib().pa_selftest_wait_timeout(int(wait_ms), _stream(stream)), "pa_selftest_wait_timeout")


def get_device_error(stream=None) -> int:
    """Read and clear the device error word (synchronises the stream)."""
    import ctypes as C
    code = C.c_int32(0)
    st = _lib.lib().pa_get_device_error(C.byref(code), _stream(stream))
    if st not in (_lib.PA_OK, _lib.PA_ERR_DEVICE_CHECK):
        check(st, "pa_get_device_error")
    return int(code.value)


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
