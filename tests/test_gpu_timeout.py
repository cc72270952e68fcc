"""A bounded wait inside a kernel runs out, is reported, and leaves the GPU usable.

Every mbarrier wait in the decode and prefill kernels gives up after a
deadline; the kernel then sets PKV_DEVERR_TIMEOUT in the caller's error flag,
waits (again with a deadline) for the copies and MMAs it issued, frees its
tensor memory and returns.  These tests run that exit for real without faulting
the GPU: a test-only build of the library (1 ms deadline, never the product
library) has host-set hooks that withhold one TMA copy, so that the wait on it
cannot complete.  Each call must return normally with the timeout bit set, and
the next call on the same context, with the hook cleared, must match the oracle.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_200_gb300 import workloads as W
from _helpers import BF16_ATOL, BF16_RTOL, FP8_ATOL, FP8_RTOL, assert_close, bits, f64

pytestmark = pytest.mark.gpu

DEVERR_TIMEOUT = 8


@pytest.fixture(scope="module")
def tlib():
    from paged_kv_cache_200_gb300 import build as B
    from paged_kv_cache_200_gb300 import pkv

    lib = ctypes.CDLL(B.build_test_library())
    for name, (res, args) in pkv._SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    lib.pkv_test_decode_skip_group.argtypes = [ctypes.c_int]
    lib.pkv_test_prefill_skip_k.argtypes = [ctypes.c_int]
    yield lib
    lib.pkv_test_decode_skip_group(-1)
    lib.pkv_test_prefill_skip_k(-1)


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _decode(lib, wl, err):
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    kc, vc = wl.k_cache.view(shape4), wl.v_cache.view(shape4)
    out = torch.empty_like(wl.q)
    lse = torch.empty((wl.batch, wl.num_heads), dtype=torch.float32, device="cuda")
    need = lib.pkv_paged_attn_decode_workspace(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.max_seqlen)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    st = lib.pkv_paged_attn_decode(_p(wl.q), _p(kc), _p(vc), 0, _p(wl.cache_seqlens), _p(wl.block_table),
                                   wl.block_table.shape[1], wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                   wl.block_size, wl.num_blocks, wl.max_seqlen, wl.scale, 1.0, 1.0, _p(out), _p(lse),
                                   _p(ws), ws.numel(), _p(err), _stream())
    return st, out, lse


def test_decode_wait_runs_out_then_the_next_call_is_correct(tlib):
    # one sequence of 3000 cached tokens, 8 q / 2 kv heads: the first CTA's warp 0 streams several groups
    wl = W.make_decode([3000], 8, 2, 128, 16, seed=301, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tlib.pkv_test_decode_skip_group(1)  # warp 0 of the first CTA never receives its second group
    st, _, _ = _decode(tlib, wl, err)
    torch.cuda.synchronize()  # the kernel returned: no trap, no hang
    assert st == 0
    assert int(err.item()) & DEVERR_TIMEOUT

    tlib.pkv_test_decode_skip_group(-1)
    err.zero_()
    st, out, lse = _decode(tlib, wl, err)
    torch.cuda.synchronize()
    assert st == 0 and int(err.item()) == 0
    ref, ref_lse = O.paged_attn_decode(bits(wl.q), bits(wl.k_cache), bits(wl.v_cache), wl.cache_seqlens.cpu().numpy(),
                                       wl.block_table.cpu().numpy(), wl.block_size, wl.scale)
    assert_close(f64(out), ref, BF16_ATOL, BF16_RTOL, "decode after a timeout")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, "decode lse after a timeout")


def _varlen(lib, wl, err):
    out = torch.empty_like(wl.q)
    lse = torch.empty((wl.num_heads, wl.total_q), dtype=torch.float32, device="cuda")
    total_k = int(wl.k_lens.sum())
    need = lib.pkv_paged_attn_varlen_workspace(wl.batch, wl.total_q, total_k, wl.num_heads, wl.num_kv_heads,
                                               wl.head_dim, wl.max_len_q, wl.max_len_k, 0, 0, 0)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    st = lib.pkv_paged_attn_varlen(_p(wl.q), _p(wl.k), _p(wl.v), 0, _p(wl.cu_seqlens_q), _p(wl.cu_seqlens_k),
                                   wl.batch, wl.total_q, total_k, wl.max_len_q, wl.max_len_k, _p(None), 0, 0, 0,
                                   wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.scale, 1, 1.0, 1.0, _p(out),
                                   _p(lse), _p(ws), ws.numel(), _p(err), _stream())
    return st, out, lse


def test_prefill_wait_runs_out_then_the_next_call_is_correct(tlib):
    # 4 sequences of 1024 tokens, 16 q heads: 256 work items, so every CTA (the first one too) gets one
    wl = W.make_varlen_packed([1024] * 4, [1024] * 4, 16, 4, 128, seed=302, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tlib.pkv_test_prefill_skip_k(0)  # the first CTA never receives its first K tile
    st, _, _ = _varlen(tlib, wl, err)
    torch.cuda.synchronize()  # the persistent kernel returned: its roles gave up, drained and freed TMEM
    assert st == 0
    assert int(err.item()) & DEVERR_TIMEOUT

    tlib.pkv_test_prefill_skip_k(-1)
    err.zero_()
    st, out, lse = _varlen(tlib, wl, err)
    torch.cuda.synchronize()
    assert st == 0 and int(err.item()) == 0
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(wl.k), bits(wl.v), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True)
    assert_close(f64(out), ref, BF16_ATOL, BF16_RTOL, "prefill after a timeout")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, "prefill lse after a timeout")


def _varlen_paged_fp8(lib, wl, kc, vc, err):
    out = torch.empty_like(wl.q)
    lse = torch.empty((wl.num_heads, wl.total_q), dtype=torch.float32, device="cuda")
    need = lib.pkv_paged_attn_varlen_workspace(wl.batch, wl.total_q, 0, wl.num_heads, wl.num_kv_heads, wl.head_dim,
                                               wl.max_len_q, wl.max_len_k, 1, 2, wl.block_size)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    st = lib.pkv_paged_attn_varlen(_p(wl.q), _p(kc), _p(vc), 2, _p(wl.cu_seqlens_q), _p(wl.cu_seqlens_k),
                                   wl.batch, wl.total_q, 0, wl.max_len_q, wl.max_len_k, _p(wl.block_table),
                                   wl.block_table.shape[1], wl.block_size, wl.num_blocks, wl.num_heads,
                                   wl.num_kv_heads, wl.head_dim, wl.scale, 1, wl.extra["k_scale"],
                                   wl.extra["v_scale"], _p(out), _p(lse), _p(ws), ws.numel(), _p(err), _stream())
    return st, out, lse


def test_one_byte_tile_loop_wait_runs_out_then_the_next_call_is_correct(tlib):
    """FP8 pages read by the prefill tile loop (no gather bound): the widening warp's wait for the
    withheld K tile runs out, the call returns with the timeout bit, and the next call is correct."""
    wl = W.to_fp8_cache(W.make_varlen_paged([1024] * 4, [0] * 4, 16, 4, 128, 16, seed=303, device="cuda"))
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    tlib.pkv_kv_cache_write(_p(wl.k_new), wl.k_new.stride(0), _p(wl.v_new), wl.v_new.stride(0), wl.k_new.shape[0],
                            wl.num_kv_heads, wl.head_dim, _p(kc), _p(vc), 2, wl.num_blocks * wl.block_size,
                            _p(wl.slot_mapping), wl.extra["k_inv_scale"], wl.extra["v_inv_scale"], _p(None),
                            _stream())
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tlib.pkv_test_prefill_skip_k(0)  # the first CTA never receives its first K tile
    st, _, _ = _varlen_paged_fp8(tlib, wl, kc, vc, err)
    torch.cuda.synchronize()  # the kernel returned: its roles gave up, drained and freed TMEM
    assert st == 0
    assert int(err.item()) & DEVERR_TIMEOUT

    tlib.pkv_test_prefill_skip_k(-1)
    err.zero_()
    st, out, lse = _varlen_paged_fp8(tlib, wl, kc, vc, err)
    torch.cuda.synchronize()
    assert st == 0 and int(err.item()) == 0
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=wl.block_size,
                                       kv_dtype="fp8_e4m3", k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
    assert_close(f64(out), ref, FP8_ATOL, FP8_RTOL, "fp8 tile-loop prefill after a timeout")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, "fp8 tile-loop prefill lse after a timeout")

