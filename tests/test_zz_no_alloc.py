"""The decode entry point that allocates nothing, against the workspace entry point and the oracle.

Some callers cannot allocate device memory: an engine that has reserved all of
it for its own pool, or a loop that must not take cudaMalloc's implicit device
synchronisation.  For them the library offers a decode call whose split-KV
partials live in a fixed device array inside the library.  These tests call it
directly through the C ABI on several calls in a row (bf16, FP8 and INT8 caches,
and a later call whose split plan is longer than the earlier ones, so stale
partials left in the shared array must never be read) and check that

* its output and lse are bit for bit those of the regular entry point, which
  runs the same kernels on the same split plan with a caller workspace;
* both are within the parity tolerance of the fp64 oracle;
* a request too large for the fixed array (if the device's split plan can ask for one) is
  refused before anything runs.

This file is collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_200_gb300 import workloads as W
from _helpers import BF16_ATOL, BF16_RTOL, FP8_ATOL, FP8_RTOL, assert_close, bits, built_library, f64

pytestmark = pytest.mark.gpu

_DTYPE_CODE = {"bf16": 0, "fp8_e4m3": 2, "int8": 3}


def _c_noalloc(lib, wl, out, lse):
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    kc, vc = wl.k_cache.view(shape4), wl.v_cache.view(shape4)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.pkv_paged_attn_decode_noalloc(
        p(wl.q), p(kc), p(vc), _DTYPE_CODE[wl.cache_dtype], p(wl.cache_seqlens), p(wl.block_table),
        wl.block_table.shape[1], wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
        wl.num_blocks, wl.max_seqlen, wl.scale, wl.k_scale, wl.v_scale, p(out), p(lse), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _partials_per_row(lib, wl):
    """Workspace bytes of the call's split plan per (sequence, query head): grows with its split count."""
    need = lib.pkv_paged_attn_decode_workspace(wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.max_seqlen)
    return need / (wl.batch * wl.num_heads)


def test_noalloc_decode_is_the_workspace_decode_on_consecutive_calls():
    pkv = built_library()
    lib = pkv.lib()
    cases = [
        W.make_decode([3000, 17, 9000, 512], 32, 8, 128, 16, seed=101, device="cuda"),            # several splits
        W.make_decode([40, 2500, 700], 16, 4, 64, 32, seed=102, device="cuda", cache_dtype="fp8_e4m3"),
        W.make_decode([5000, 600, 3100], 32, 8, 128, 16, seed=103, device="cuda", cache_dtype="int8"),
        # few sequences, one long: more splits per (sequence, head) than every call above
        W.make_decode([30000, 100], 32, 8, 128, 16, seed=104, device="cuda"),
        W.make_decode([3000, 17, 9000, 512], 32, 8, 128, 16, seed=101, device="cuda"),            # the first again
    ]
    assert _partials_per_row(lib, cases[3]) > max(_partials_per_row(lib, c) for c in cases[:3])
    for wl in cases:
        shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
        ref, ref_lse = pkv.paged_attn_decode(wl.q, wl.k_cache.view(shape4), wl.v_cache.view(shape4),
                                             wl.cache_seqlens, wl.block_table, wl.scale,
                                             max_seqlen_k=wl.max_seqlen, k_scale=wl.k_scale, v_scale=wl.v_scale,
                                             return_lse=True)
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _c_noalloc(lib, wl, out, lse) == 0
        torch.cuda.synchronize()
        # same kernels, same split plan: identical bits
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"{wl.cache_dtype}: out differs"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), f"{wl.cache_dtype}: lse differs"
        # and both match the oracle
        oref, oref_lse = O.paged_attn_decode(bits(wl.q), bits(wl.k_cache), bits(wl.v_cache),
                                             wl.cache_seqlens.cpu().numpy(), wl.block_table.cpu().numpy(),
                                             wl.block_size, wl.scale, wl.cache_dtype, wl.k_scale, wl.v_scale)
        atol, rtol = (FP8_ATOL, FP8_RTOL) if wl.cache_dtype != "bf16" else (BF16_ATOL, BF16_RTOL)
        assert_close(f64(out), oref, atol, rtol, f"noalloc {wl.cache_dtype} out")
        assert_close(f64(lse), oref_lse, 1e-3, 1e-3, f"noalloc {wl.cache_dtype} lse")


def test_noalloc_refuses_only_requests_beyond_its_fixed_scratch():
    """A request whose split-KV partials exceed the fixed array is refused before anything runs.

    The partials are bounded by the split plan (at most about group x 8 waves x the resident CTAs of
    the device rows of head_dim floats), so on a device of this size the sweep may find no request
    that exceeds the array: then every swept request fits it and none is refused for its size."""
    pkv = built_library()
    lib = pkv.lib()
    limit = lib.pkv_paged_attn_decode_noalloc_max_scratch()
    assert limit == 32 << 20
    over, biggest = None, 0
    for Hkv in (1, 8):
        for g in (1, 2, 4, 8):
            for D in (64, 128):
                for B in (1, 2, 4, 8, 16, 18, 19, 32, 64, 128, 256, 1024, 4096):
                    for L in (513, 4096, 16385, 100000, 131073, 1 << 20, 1 << 24):
                        w = lib.pkv_paged_attn_decode_workspace(B, Hkv * g, Hkv, D, L)
                        biggest = max(biggest, w)
                        if w > limit and over is None:
                            over = (B, Hkv * g, Hkv, D, L)
    if over is None:
        assert 0 < biggest <= limit
        return
    B, Hq, Hkv, D, L = over
    nul = ctypes.c_void_p(0)
    st = lib.pkv_paged_attn_decode_noalloc(nul, nul, nul, 0, nul, nul, 32768, B, Hq, Hkv, D, 32, 1 << 20, L, 0.1,
                                           1.0, 1.0, nul, nul, nul, nul)
    assert st == 3  # PKV_ERR_WORKSPACE, refused before any launch
