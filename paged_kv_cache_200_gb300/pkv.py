"""Thin ctypes binding of ``libpkv.so`` (declared in ``include/pkv.h``).

Argument marshalling only: every computation runs in the library's CUDA
kernels.  Torch tensors supply device pointers, the current CUDA stream and
workspace memory.  There is no CPU fallback: if the library is missing the
first call raises.

Functions mirror the C entry points:

* ``kv_cache_write(k, v, k_cache, v_cache, slot_mapping, ...)``
* ``paged_attn_decode(q, k_cache, v_cache, cache_seqlens, block_table, scale, ...)``
* ``paged_attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_len_q, max_len_k, ...)``
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "pkv.h")

PKV_BF16 = 0
PKV_FP8_E4M3 = 2
PKV_INT8 = 3

DEVERR_SLOT = 1
DEVERR_BLOCK = 2
DEVERR_LENGTH = 4
DEVERR_TIMEOUT = 8

_c_void_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_abi_version": (ctypes.c_int, []),
    "pkv_kv_cache_write": (ctypes.c_int, [
        _c_void_p, _i64, _c_void_p, _i64, _i32, _i32, _i32, _c_void_p, _c_void_p, _i32, _i64,
        _c_void_p, _f32, _f32, _c_void_p, _c_void_p]),
    "pkv_copy_blocks": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i32, _c_void_p, _i32, _c_void_p, _c_void_p]),
    "pkv_paged_attn_decode_workspace": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "pkv_set_nvtx": (None, [_i32]),
    "pkv_paged_attn_decode": (ctypes.c_int, [
        _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _c_void_p, _i32, _i32, _i32, _i32, _i32,
        _i32, _i32, _i32, _f32, _f32, _f32, _c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p, _c_void_p]),
    "pkv_paged_attn_decode_with_kvcache": (ctypes.c_int, [
        _c_void_p, _c_void_p, _i64, _c_void_p, _i64, _c_void_p, _c_void_p, _i32, _c_void_p, _c_void_p, _i32, _i32,
        _i32, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _f32, _f32, _f32, _c_void_p, _c_void_p, _c_void_p, _sz,
        _c_void_p, _c_void_p]),
    "pkv_paged_attn_decode_noalloc": (ctypes.c_int, [
        _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _c_void_p, _i32, _i32, _i32, _i32, _i32,
        _i32, _i32, _i32, _f32, _f32, _f32, _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "pkv_paged_attn_decode_noalloc_max_scratch": (_sz, []),
    "pkv_paged_attn_varlen_workspace": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pkv_paged_attn_varlen": (ctypes.c_int, [
        _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _c_void_p, _i32, _i32, _i32, _i32, _i32,
        _c_void_p, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _i32, _f32, _f32, _c_void_p, _c_void_p,
        _c_void_p, _sz, _c_void_p, _c_void_p]),
}

_lib = None


class PkvError(RuntimeError):
    """A libpkv call returned a non-zero status."""

    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def declared_functions(header: str = HEADER):
    """Names of the functions ``include/pkv.h`` declares."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def lib(path: str = LIB_PATH):
    """Load the library (once) and declare argument types."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with paged_kv_cache_200_gb300.build.build()")
        handle = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            if hasattr(handle, name):
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
        _lib = handle
    return _lib


def set_nvtx(on: bool = True):
    """Turn the library's NVTX ranges (one per compute call, named after the C entry point) on or off."""
    lib().pkv_set_nvtx(1 if on else 0)


def _check(status: int):
    if status != 0:
        raise PkvError(status, lib().pkv_status_string(status).decode())


def _ptr(t):
    # (the argument types are c_void_p: a plain int or None converts directly)
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    """The cudaStream_t (as an int) of ``stream``, default: the current device's current stream (the
    library launches on the current device)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:  # the same handle as current_stream().cuda_stream, without building a Stream
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _cache_dtype(cache: torch.Tensor) -> int:
    if cache.dtype == _BF16:
        return PKV_BF16
    if cache.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return PKV_FP8_E4M3
    if cache.dtype == torch.int8:
        return PKV_INT8
    raise TypeError(f"unsupported cache dtype {cache.dtype}")


_BF16 = torch.bfloat16
_I32 = torch.int32
_fns = {}


def _fn(name):
    """The library function (bound once, with its argument types)."""
    f = _fns.get(name)
    if f is None:
        f = getattr(lib(), name)
        _fns[name] = f
    return f


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")


_workspaces = {}


def workspace(nbytes: int, device, stream=None) -> torch.Tensor:
    """A cached scratch buffer of at least ``nbytes`` (grows, never shrinks), one per
    (device, stream).

    Calls on one stream run in order, so they can share a buffer; calls on two
    streams may overlap on the GPU and get separate buffers (the varlen call also
    keeps its work counter in there).  A caller that passes ``workspace_buf``
    itself must not share one buffer between calls that can overlap.
    """
    dev = torch.device(device)
    index = dev.index if dev.index is not None else torch.cuda.current_device()
    if stream is None:
        stream = torch.cuda.current_stream(index)
    key = (index, int(stream.cuda_stream))
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=dev)
        _workspaces[key] = buf
    return buf


# ---------------------------------------------------------------------------
# KV-cache write
# ---------------------------------------------------------------------------


def kv_cache_write(k, v, k_cache, v_cache, slot_mapping, k_inv_scale: float = 1.0, v_inv_scale: float = 1.0,
                   err_flag=None, stream=None):
    """Scatter each token's K/V row into the caches at ``slot_mapping[t]`` (negative = skip).

    ``k``, ``v``: ``[T, Hkv, D]`` bf16 with the inner two dims contiguous (any
    row stride).  Caches: ``[..., Hkv, D]`` contiguous: bf16, uint8 E4M3 codes
    or int8 codes.  FP8 stores ``e4m3(x * inv_scale)``; INT8 stores
    ``clamp(rint(x * inv_scale), -127, 127)`` with NaN stored as 0.
    """
    # One combined check on the common path (this runs once per layer and
    # step); the detailed checks below only name what is wrong.
    T, Hkv, D = k.shape
    ks, vs = k.stride(), v.stride()
    if not (k.is_cuda and v.is_cuda and k_cache.is_cuda and v_cache.is_cuda and slot_mapping.is_cuda
            and (err_flag is None or err_flag.is_cuda) and k.dtype == _BF16 and v.dtype == _BF16
            and v.shape == k.shape and ks[2] == 1 and vs[2] == 1 and ks[1] == D and vs[1] == D
            and k_cache.is_contiguous() and v_cache.is_contiguous() and v_cache.shape == k_cache.shape
            and k_cache.shape[-2:] == (Hkv, D) and slot_mapping.dtype == _I32 and slot_mapping.numel() == T):
        _require_cuda(k, v, k_cache, v_cache, slot_mapping, err_flag)
        if v.shape != k.shape or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
            raise ValueError("k and v must be bf16 tensors of the same shape [T, Hkv, D]")
        if ks[2] != 1 or vs[2] != 1 or ks[1] != D or vs[1] != D:
            raise ValueError("k/v inner dims [Hkv, D] must be contiguous")
        if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
            raise ValueError("caches must be contiguous")
        if k_cache.shape[-2:] != (Hkv, D) or v_cache.shape != k_cache.shape:
            raise ValueError("caches must end in [Hkv, D] and match each other")
        raise ValueError("slot_mapping must be int32 with one entry per token")
    num_slots = k_cache.numel() // (Hkv * D)
    st = _fn("pkv_kv_cache_write")(k.data_ptr(), ks[0], v.data_ptr(), vs[0], T, Hkv, D, k_cache.data_ptr(),
                                   v_cache.data_ptr(), _cache_dtype(k_cache), num_slots, slot_mapping.data_ptr(),
                                   k_inv_scale, v_inv_scale, _ptr(err_flag), _stream(stream))
    if st:
        _check(st)


# ---------------------------------------------------------------------------
# copy-on-write of shared blocks
# ---------------------------------------------------------------------------


def copy_blocks(k_cache, v_cache, block_pairs, err_flag=None, stream=None):
    """Block ``dst`` of each cache becomes a copy of block ``src``, for each row of ``block_pairs``.

    Caches: ``[num_blocks, block_size, Hkv, D]`` contiguous (bf16, E4M3 or
    INT8 codes; the bytes are copied as they are); ``v_cache`` may be ``None``.  ``block_pairs``: int32 ``[n, 2]``
    ``(src, dst)`` on the device; no dst may also be a src of the same call.
    """
    _require_cuda(k_cache, block_pairs, *([] if v_cache is None else [v_cache]))
    if not k_cache.is_contiguous() or (v_cache is not None and
                                       (not v_cache.is_contiguous() or v_cache.shape != k_cache.shape
                                        or v_cache.dtype != k_cache.dtype)):
        raise ValueError("caches must be contiguous and match each other")
    if block_pairs.dtype != torch.int32 or block_pairs.dim() != 2 or block_pairs.shape[1] != 2 or \
            not block_pairs.is_contiguous():
        raise ValueError("block_pairs must be a contiguous int32 [n, 2] tensor")
    num_blocks = k_cache.shape[0]
    block_bytes = k_cache[0].numel() * k_cache.element_size()
    st = lib().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), block_bytes, num_blocks, _ptr(block_pairs),
                               block_pairs.shape[0], _ptr(err_flag), _stream(stream))
    _check(st)


# ---------------------------------------------------------------------------
# paged decode attention
# ---------------------------------------------------------------------------


def paged_attn_decode(q, k_cache, v_cache, cache_seqlens, block_table, scale: float, max_seqlen_k: int = None,
                      k_scale: float = 1.0, v_scale: float = 1.0, out=None, lse=None, return_lse=False,
                      err_flag=None, workspace_buf=None, stream=None):
    """Decode attention over a paged cache; returns ``out [B, Hq, D]`` (and ``lse [B, Hq]``).

    ``k_cache``/``v_cache``: ``[num_blocks, block_size, Hkv, D]``.
    ``cache_seqlens``: int32 ``[B]`` tokens to attend; ``block_table``: int32
    ``[B, max_blocks_per_seq]``.  ``max_seqlen_k`` is a host upper bound of the
    lengths (default: the block table's capacity; no device sync is made).
    """
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    # one combined check on the common path (once per layer and step); the
    # detailed checks below only name what is wrong
    if not (q.is_cuda and k_cache.is_cuda and v_cache.is_cuda and cache_seqlens.is_cuda and block_table.is_cuda
            and (out is None or out.is_cuda) and (lse is None or lse.is_cuda)
            and (err_flag is None or err_flag.is_cuda) and (workspace_buf is None or workspace_buf.is_cuda)
            and D2 == D and v_cache.shape == k_cache.shape and q.dtype == _BF16 and q.is_contiguous()
            and k_cache.is_contiguous() and v_cache.is_contiguous() and block_table.is_contiguous()
            and cache_seqlens.dtype == _I32 and block_table.dtype == _I32):
        _require_cuda(q, k_cache, v_cache, cache_seqlens, block_table, out, lse, err_flag, workspace_buf)
        if D2 != D or v_cache.shape != k_cache.shape:
            raise ValueError("cache shape mismatch")
        if q.dtype != torch.bfloat16 or not q.is_contiguous():
            raise ValueError("q must be contiguous bf16 [B, Hq, D]")
        if not (k_cache.is_contiguous() and v_cache.is_contiguous() and block_table.is_contiguous()):
            raise ValueError("caches and block_table must be contiguous")
        raise ValueError("cache_seqlens and block_table must be int32")
    MB = block_table.shape[1]
    if max_seqlen_k is None:
        max_seqlen_k = MB * bs
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    ws = workspace_buf
    if ws is None:  # (a caller-provided buffer skips the size query; the call checks it)
        need = _fn("pkv_paged_attn_decode_workspace")(B, Hq, Hkv, D, max(int(max_seqlen_k), 1))
        ws = workspace(need, q.device, stream) if need else None
    st = _fn("pkv_paged_attn_decode")(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), _cache_dtype(k_cache),
                                      cache_seqlens.data_ptr(), block_table.data_ptr(), MB, B, Hq, Hkv, D, bs, NB,
                                      int(max_seqlen_k), scale, k_scale, v_scale, out.data_ptr(), _ptr(lse),
                                      _ptr(ws), 0 if ws is None else ws.numel(), _ptr(err_flag),
                                      _stream(stream))
    if st:
        _check(st)
    return (out, lse) if (return_lse or lse is not None) else out


def paged_attn_decode_with_kvcache(q, k_new, v_new, k_cache, v_cache, cache_seqlens, block_table, scale: float,
                                   max_seqlen_k: int = None, k_scale: float = 1.0, v_scale: float = 1.0,
                                   k_inv_scale: float = 1.0, v_inv_scale: float = 1.0, out=None, lse=None,
                                   return_lse=False, err_flag=None, workspace_buf=None, stream=None):
    """Append each sequence's new K/V row to its cache, then decode, in one launch.

    ``cache_seqlens``: int32 ``[B]`` tokens cached BEFORE this step; the new row
    ``k_new[b]``/``v_new[b]`` (bf16 ``[B, Hkv, D]``, inner dims contiguous) goes
    to position ``cache_seqlens[b]`` and ``cache_seqlens[b] + 1`` positions are
    attended.  ``max_seqlen_k``: host bound of ``cache_seqlens + 1`` (default:
    the block table's capacity).  FP8 caches store ``e4m3(x * inv_scale)``.
    """
    _require_cuda(q, k_new, v_new, k_cache, v_cache, cache_seqlens, block_table)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape mismatch")
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise ValueError("q must be contiguous bf16 [B, Hq, D]")
    if k_new.shape != (B, Hkv, D) or v_new.shape != (B, Hkv, D) or k_new.dtype != torch.bfloat16 or \
            v_new.dtype != torch.bfloat16:
        raise ValueError("k_new and v_new must be bf16 [B, Hkv, D]")
    if k_new.stride(-1) != 1 or v_new.stride(-1) != 1 or k_new.stride(1) != D or v_new.stride(1) != D:
        raise ValueError("k_new/v_new inner dims [Hkv, D] must be contiguous")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous() and block_table.is_contiguous()):
        raise ValueError("caches and block_table must be contiguous")
    if cache_seqlens.dtype != torch.int32 or block_table.dtype != torch.int32:
        raise ValueError("cache_seqlens and block_table must be int32")
    MB = block_table.shape[1]
    if max_seqlen_k is None:
        max_seqlen_k = MB * bs
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    L = lib()
    ws = workspace_buf
    if ws is None:  # (a caller-provided buffer skips the size query; the call checks it)
        need = L.pkv_paged_attn_decode_workspace(B, Hq, Hkv, D, max(int(max_seqlen_k), 1))
        ws = workspace(need, q.device, stream) if need else None
    st = L.pkv_paged_attn_decode_with_kvcache(
        _ptr(q), _ptr(k_new), k_new.stride(0), _ptr(v_new), v_new.stride(0), _ptr(k_cache), _ptr(v_cache),
        _cache_dtype(k_cache), _ptr(cache_seqlens), _ptr(block_table), MB, B, Hq, Hkv, D, bs, NB, int(max_seqlen_k),
        float(scale), float(k_scale), float(v_scale), float(k_inv_scale), float(v_inv_scale), _ptr(out), _ptr(lse),
        _ptr(ws), 0 if ws is None else ws.numel(), _ptr(err_flag), _stream(stream))
    _check(st)
    return (out, lse) if (return_lse or lse is not None) else out


def paged_attn_decode_noalloc(q, k_cache, v_cache, cache_seqlens, block_table, scale: float,
                              max_seqlen_k: int = None, k_scale: float = 1.0, v_scale: float = 1.0, out=None,
                              lse=None, err_flag=None, stream=None):
    """``paged_attn_decode`` for callers that cannot allocate: partials go to the library's fixed scratch.

    Same arguments and result as ``paged_attn_decode`` (``out`` must be given by
    callers that must not allocate; ``lse`` is optional).  Raises ``PkvError``
    (PKV_ERR_WORKSPACE) when the request needs more scratch than the fixed 32 MiB.
    Calls that overlap on the GPU share the scratch and must not be issued.
    """
    _require_cuda(q, k_cache, v_cache, cache_seqlens, block_table)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    MB = block_table.shape[1]
    if max_seqlen_k is None:
        max_seqlen_k = MB * bs
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    st = lib().pkv_paged_attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _cache_dtype(k_cache),
                                             _ptr(cache_seqlens), _ptr(block_table), MB, B, Hq, Hkv, D, bs, NB,
                                             int(max_seqlen_k), float(scale), float(k_scale), float(v_scale),
                                             _ptr(out), _ptr(lse), _ptr(err_flag), _stream(stream))
    _check(st)
    return out


# ---------------------------------------------------------------------------
# varlen (prefill) attention
# ---------------------------------------------------------------------------


def paged_attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_len_q: int, max_len_k: int, block_table=None,
                      scale: float = None, causal: bool = True, out=None, lse=None, return_lse=False,
                      err_flag=None, workspace_buf=None, stream=None, gather_k_tokens: int = 0,
                      k_scale: float = 1.0, v_scale: float = 1.0):
    """Causal varlen attention; returns ``out [total_q, Hq, D]`` (and ``lse [Hq, total_q]``).

    Without ``block_table``: ``k``/``v`` are packed ``[total_k, Hkv, D]``.  With it:
    ``k``/``v`` are the paged caches ``[num_blocks, block_size, Hkv, D]`` and
    ``block_table`` is int32 ``[B, max_blocks_per_seq]``.  ``max_len_q`` /
    ``max_len_k`` are host upper bounds of the lengths (no device sync is made).
    Paged mode: ``gather_k_tokens`` (a host bound on the summed keys of the
    sequences the prefill tiles serve) lets the library gather their K/V into
    a packed bf16 buffer first, which blocks under 64 tokens and one-byte
    caches (uint8 E4M3 or int8 codes, value = code * k_scale / v_scale) use.
    Without it a one-byte cache with head dim 128 is read page by page and
    widened to f16 in shared memory (the query taken as f16 too); head dim 64
    needs it unless no sequence has more than 8 queries (then every query row
    runs on the decode kernels).  Without ``workspace_buf`` the scratch comes
    from a buffer cached per (device, stream).
    """
    _require_cuda(q, k, v, cu_seqlens_q, cu_seqlens_k, block_table)
    T, Hq, D = q.shape
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise ValueError("q must be contiguous bf16 [total_q, Hq, D]")
    if not (k.is_contiguous() and v.is_contiguous()) or k.shape != v.shape:
        raise ValueError("k and v must be contiguous and of the same shape")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("cu_seqlens must be int32")
    B = cu_seqlens_q.numel() - 1
    if block_table is None:
        total_k, Hkv, _ = k.shape
        MB, bs, NB = 0, 0, 0
    else:
        NB, bs, Hkv, _ = k.shape
        total_k = int(gather_k_tokens)
        if block_table.dtype != torch.int32 or not block_table.is_contiguous():
            raise ValueError("block_table must be contiguous int32")
        MB = block_table.shape[1]
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    L = lib()
    paged = 1 if block_table is not None else 0
    ws = workspace_buf
    if ws is None:  # (a caller-provided buffer skips the size query; the call checks it)
        need = L.pkv_paged_attn_varlen_workspace(B, T, total_k, Hq, Hkv, D, int(max_len_q), int(max_len_k), paged,
                                                 _cache_dtype(k), bs)
        ws = workspace(need, q.device, stream) if need else None
    st = L.pkv_paged_attn_varlen(_ptr(q), _ptr(k), _ptr(v), _cache_dtype(k), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), B, T, total_k, int(max_len_q), int(max_len_k),
                                 _ptr(block_table), MB, bs, NB, Hq, Hkv, D, float(scale), 1 if causal else 0,
                                 float(k_scale), float(v_scale), _ptr(out), _ptr(lse), _ptr(ws),
                                 0 if ws is None else ws.numel(),
                                 _ptr(err_flag), _stream(stream))
    _check(st)
    return (out, lse) if (return_lse or lse is not None) else out
