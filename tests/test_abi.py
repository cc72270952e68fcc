"""The C-ABI library builds, loads, and exports every function include/pkv.h declares.

No kernel runs here: only calls that the library rejects on the host before
touching the GPU are made.
"""

import ctypes
import shutil

import pytest

from _helpers import built_library

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not __import__("os").path.exists(
    "/usr/local/cuda/bin/nvcc"), reason="nvcc not available")


def test_every_declared_symbol_is_exported():
    pkv = built_library()
    names = pkv.declared_functions()
    assert "pkv_kv_cache_write" in names and "pkv_paged_attn_decode" in names
    lib = pkv.lib()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding declares a signature for every exported entry point
    assert set(names) <= set(pkv._SIGNATURES), set(names) - set(pkv._SIGNATURES)


def test_status_strings_and_version():
    pkv = built_library()
    lib = pkv.lib()
    assert lib.pkv_abi_version() >= 1
    for code in range(5):
        assert lib.pkv_status_string(code).startswith(b"PKV_")


def test_host_side_argument_validation():
    pkv = built_library()
    lib = pkv.lib()
    nul = ctypes.c_void_p(0)
    # negative token count / bad head dims are rejected before any launch
    assert lib.pkv_kv_cache_write(nul, 128, nul, 128, -1, 1, 128, nul, nul, 0, 16, nul, 1.0, 1.0, nul, nul) == 1
    assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 4, 1, 128, nul, nul, 7, 16, nul, 1.0, 1.0, nul, nul) == 2
    assert lib.pkv_kv_cache_write(nul, 12, nul, 12, 4, 1, 12, nul, nul, 0, 16, nul, 1.0, 1.0, nul, nul) == 2
    # zero tokens: nothing to do
    assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 0, 1, 128, nul, nul, 0, 16, nul, 1.0, 1.0, nul, nul) == 0
    # null pointers with work to do
    assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 4, 1, 128, nul, nul, 0, 16, nul, 1.0, 1.0, nul, nul) == 1
    # decode: head_dim 96 unsupported, group of 16 unsupported, block size 8 unsupported
    args = lambda H, Hkv, D, bs: (nul, nul, nul, 0, nul, nul, 4, 1, H, Hkv, D, bs, 8, 64, 0.1, 1.0, 1.0,
                                  nul, nul, nul, 0, nul, nul)
    assert lib.pkv_paged_attn_decode(*args(8, 2, 96, 16)) == 2
    assert lib.pkv_paged_attn_decode(*args(32, 2, 128, 16)) == 2
    assert lib.pkv_paged_attn_decode(*args(8, 2, 128, 8)) == 2
    assert lib.pkv_paged_attn_decode(*args(8, 3, 128, 16)) == 1


def test_dtype_codes_outside_bf16_fp8_int8_are_unsupported():
    """float16 is not built: code 1 (and any other unknown code) is refused by every entry point that
    takes a dtype, with PKV_ERR_UNSUPPORTED, before any launch."""
    pkv = built_library()
    lib = pkv.lib()
    nul = ctypes.c_void_p(0)
    row = ctypes.c_void_p(4096)  # non-null, aligned new-row pointers (never dereferenced: refused first)
    for dt in (1, 4, -1):
        assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 4, 1, 128, nul, nul, dt, 16, nul, 1.0, 1.0, nul, nul) == 2
        assert lib.pkv_paged_attn_decode(nul, nul, nul, dt, nul, nul, 4, 1, 8, 2, 128, 16, 8, 64, 0.1, 1.0, 1.0,
                                         nul, nul, nul, 0, nul, nul) == 2
        assert lib.pkv_paged_attn_decode_with_kvcache(nul, row, 1024, row, 1024, nul, nul, dt, nul, nul, 4, 1, 8,
                                                      2, 128, 16, 8, 64, 0.1, 1.0, 1.0, 1.0, 1.0, nul, nul, nul,
                                                      0, nul, nul) == 2
        assert lib.pkv_paged_attn_varlen(nul, nul, nul, dt, nul, nul, 4, 16, 0, 4, 64, nul, 8, 16, 64, 8, 2, 128,
                                         0.1, 1, 1.0, 1.0, nul, nul, nul, 0, nul, nul) == 2


def test_one_byte_caches_need_valid_inverse_scales():
    """An FP8 or INT8 cache write (and the append of decode-with-append) refuses a zero, negative,
    infinite or NaN inverse scale before any launch; a bf16 cache ignores the scales."""
    pkv = built_library()
    lib = pkv.lib()
    nul = ctypes.c_void_p(0)
    bad = (0.0, -1.0, float("inf"), float("nan"))
    for dt in (2, 3):  # PKV_FP8_E4M3, PKV_INT8
        for x in bad:
            for ki, vi in ((x, 1.0), (1.0, x)):
                assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 4, 1, 128, nul, nul, dt, 16, nul, ki, vi, nul,
                                              nul) == 1
                assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 0, 1, 128, nul, nul, dt, 16, nul, ki, vi, nul,
                                              nul) == 1
    # valid scales and zero tokens: nothing to do; bf16: the scales are not used
    for dt in (2, 3):
        assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 0, 1, 128, nul, nul, dt, 16, nul, 0.5, 2.0, nul, nul) == 0
    assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 0, 1, 128, nul, nul, 0, 16, nul, 0.0, float("nan"), nul,
                                  nul) == 0

    # decode with append: an empty batch with valid scales is a no-op, with a bad one it is refused
    def append(dt, ki, vi):
        return lib.pkv_paged_attn_decode_with_kvcache(nul, nul, 1024, nul, 1024, nul, nul, dt, nul, nul, 4, 0, 8, 2,
                                                      128, 16, 8, 64, 0.1, 1.0, 1.0, ki, vi, nul, nul, nul, 0, nul,
                                                      nul)

    for dt in (2, 3):
        assert append(dt, 0.5, 0.25) == 0
        for x in bad:
            assert append(dt, x, 1.0) == 1
            assert append(dt, 1.0, x) == 1
    assert append(0, 0.0, float("nan")) == 0  # bf16 cache: the scales are not used


def test_one_byte_varlen_modes():
    """A one-byte (FP8 / INT8) cache in a varlen call: packed K/V is refused; in paged mode it is
    accepted with a gather bound, without one when the tile loop can widen the pages itself (head
    dim 128) or when every query row goes to the decode kernels, and refused otherwise (head dim
    64 with prefill tiles and no gather bound).  Accepted calls then fail on their null pointers,
    status 1, before any launch."""
    pkv = built_library()
    lib = pkv.lib()
    nul = ctypes.c_void_p(0)
    tbl = ctypes.c_void_p(4096)  # a non-null block table pointer (never dereferenced: refused first)

    def varlen(dt, table, max_len_q, total_k=0, D=128):
        return lib.pkv_paged_attn_varlen(nul, nul, nul, dt, nul, nul, 4, 16, total_k, max_len_q, 64, table, 8, 16,
                                         64, 8, 2, D, 0.1, 1, 0.5, 0.5, nul, nul, nul, 0, nul, nul)

    for dt in (2, 3):
        assert varlen(dt, nul, 4) == 2            # packed K/V in one-byte codes
        assert varlen(dt, tbl, 40) == 1           # prefill tiles widen the pages (d128): accepted
        assert varlen(dt, tbl, 40, D=64) == 2     # d64 prefill tiles need the gather bound
        assert varlen(dt, tbl, 40, 4096, D=64) == 1
        assert varlen(dt, tbl, 4, D=64) == 1      # all rows routed: accepted (then: null pointers)
        assert varlen(dt, tbl, 40, 4096) == 1     # with a gather bound: accepted (then: null pointers)


def test_copy_blocks_host_validation():
    pkv = built_library()
    lib = pkv.lib()
    nul = ctypes.c_void_p(0)
    # negative pair count, block bytes not a multiple of 16, empty pool: rejected before any launch
    assert lib.pkv_copy_blocks(nul, nul, 4096, 8, nul, -1, nul, nul) == 1
    assert lib.pkv_copy_blocks(nul, nul, 4100, 8, nul, 1, nul, nul) == 1
    assert lib.pkv_copy_blocks(nul, nul, 4096, 0, nul, 1, nul, nul) == 1
    # no pairs: nothing to do; pairs without a cache: rejected
    assert lib.pkv_copy_blocks(nul, nul, 4096, 8, nul, 0, nul, nul) == 0
    assert lib.pkv_copy_blocks(nul, nul, 4096, 8, nul, 3, nul, nul) == 1


def test_empty_calls_do_nothing_and_invalid_sizes_are_rejected():
    """Degenerate calls return before any launch: an empty batch is a no-op, while a bad
    size is rejected even when there is nothing to compute."""
    pkv = built_library()
    lib = pkv.lib()
    nul = ctypes.c_void_p(0)

    def decode(batch, Hq=8, Hkv=2, D=128, bs=16, scale=0.1):
        return lib.pkv_paged_attn_decode(nul, nul, nul, 0, nul, nul, 4, batch, Hq, Hkv, D, bs, 8, 64, scale, 1.0,
                                         1.0, nul, nul, nul, 0, nul, nul)

    assert decode(0) == 0                 # empty batch: nothing to do
    assert decode(-1) == 1                # negative batch
    assert decode(0, scale=0.0) == 1      # an invalid scale is rejected even with nothing to do
    assert decode(3, scale=0.0) == 1
    assert decode(3) == 1                 # null pointers with work to do

    def varlen(batch, total_q, max_len_q, Hq=8, Hkv=2, D=128, causal=1):
        return lib.pkv_paged_attn_varlen(nul, nul, nul, 0, nul, nul, batch, total_q, 0, max_len_q, 0, nul, 0, 0, 0,
                                         Hq, Hkv, D, 0.1, causal, 1.0, 1.0, nul, nul, nul, 0, nul, nul)

    assert varlen(0, 0, 0) == 0           # empty batch
    assert varlen(4, 0, 0) == 0           # no queries
    assert varlen(4, 10, 4) == 1          # null pointers with work to do
    assert varlen(4, 10, 4, D=96) == 2    # unsupported head dim
    assert varlen(4, 10, 4, causal=0) == 2  # only causal attention is provided
    assert varlen(4, 10, 4, Hq=6, Hkv=4) == 1  # heads not a multiple of the kv heads

    def append(batch):
        return lib.pkv_paged_attn_decode_with_kvcache(nul, nul, 1024, nul, 1024, nul, nul, 0, nul, nul, 4, batch, 8,
                                                      2, 128, 16, 8, 64, 0.1, 1.0, 1.0, 1.0, 1.0, nul, nul, nul, 0,
                                                      nul, nul)

    assert append(0) == 0
    assert append(2) == 1


def _split_plan(batch, num_kv_heads, max_len, sms, resident):
    """The decode split plan as the library states it: positions per CTA (a multiple of 64,
    at least 512, at most the whole sequence).  Few (sequence, kv head) units: the split
    count with the fewest waves x (split + 96); otherwise about 16 CTAs per SM."""
    whole = (max_len + 63) // 64 * 64

    def clamp(c):
        return min(max((c + 63) // 64 * 64, 512), whole)

    if whole <= 512:
        return whole
    units = batch * num_kv_heads
    if units < sms:
        slots = sms * resident
        best, best_c = None, whole
        for n in range(1, 8 * slots // units + 2):
            c = clamp(-(-max_len // n))
            waves = -(-units * -(-max_len // c) // slots)
            cost = waves * (c + 96)
            if best is None or cost < best:
                best, best_c = cost, c
            if c == 512:
                break
        return best_c
    return clamp(-(-max_len * units // (sms * 16)))


@pytest.mark.parametrize("shape", [(8, 64, 8, 128, 131073), (64, 32, 8, 128, 16385), (1, 8, 8, 128, 32768),
                                   (3, 4, 2, 64, 71), (2, 16, 2, 64, 600000)])
def test_decode_workspace_follows_the_split_plan(shape):
    """The workspace query sizes the larger of the bf16 (2 CTAs per SM) and one-byte (4 per SM) plans."""
    import torch

    pkv = built_library()
    lib = pkv.lib()
    B, Hq, Hkv, D, L = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148

    def ws(res):
        c = _split_plan(B, Hkv, L, sms, res)
        splits = -(-L // c)
        if splits <= 1:
            return 0
        rows = B * Hq * splits
        return rows * D * 4 + (rows * 4 + 255) // 256 * 256

    assert lib.pkv_paged_attn_decode_workspace(B, Hq, Hkv, D, L) == max(ws(2), ws(4))


def test_split_plan_ends_long_contexts_on_whole_waves():
    """8 x 128K tokens: 19 splits of 6912 positions, 1216 CTAs = 4 waves of 2 CTAs per SM on 152 SMs."""
    c = _split_plan(8, 8, 131073, 152, 2)
    assert c == 6912 and -(-131073 // c) == 19
    assert (8 * 8 * 19) % (152 * 2) == 0


def test_nvtx_ranges_switch_on_and_off_around_calls():
    """Tracing on, calls that return before any launch (nothing to do, or refused), tracing off:
    the ranges open and close without a tool attached."""
    pkv = built_library()
    lib = pkv.lib()
    nul = ctypes.c_void_p(0)
    pkv.set_nvtx(True)
    try:
        assert lib.pkv_kv_cache_write(nul, 128, nul, 128, 0, 1, 128, nul, nul, 0, 16, nul, 1.0, 1.0, nul, nul) == 0
        assert lib.pkv_kv_cache_write(nul, 128, nul, 128, -1, 1, 128, nul, nul, 0, 16, nul, 1.0, 1.0, nul, nul) == 1
        assert lib.pkv_copy_blocks(nul, nul, 16, 1, nul, 0, nul, nul) == 0
        assert lib.pkv_paged_attn_decode(nul, nul, nul, 0, nul, nul, 4, 1, 8, 3, 128, 16, 8, 64, 0.1, 1.0, 1.0,
                                         nul, nul, nul, 0, nul, nul) == 1
        assert lib.pkv_paged_attn_varlen(nul, nul, nul, 1, nul, nul, 4, 16, 0, 4, 64, nul, 8, 16, 64, 8, 2, 128,
                                         0.1, 1, 1.0, 1.0, nul, nul, nul, 0, nul, nul) == 2
    finally:
        pkv.set_nvtx(False)
