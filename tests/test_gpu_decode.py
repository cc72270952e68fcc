"""Paged decode attention on the GPU vs the fp64 oracle.

Small cases compare every output; the full-size workloads (64 sequences of
1K..16K tokens; 8 sequences of 131072 tokens, bf16 and FP8) compare sampled
sequences computed by the oracle one by one, in the launch configuration the
benchmark times.
"""

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_200_gb300 import workloads as W
from _helpers import BF16_ATOL, BF16_RTOL, FP8_ATOL, FP8_RTOL, assert_close, bits, built_library, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    return built_library()


def _cache4(wl, t):
    return t.view(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)


def _gpu_step(pkv, wl, write=True, max_seqlen_k=None, return_lse=True):
    """Write the new tokens (optional) then decode; returns (out, lse, k_cache, v_cache)."""
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    if write:
        pkv.kv_cache_write(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping, k_inv_scale=wl.k_inv_scale,
                           v_inv_scale=wl.v_inv_scale)
    out, lse = pkv.paged_attn_decode(wl.q, _cache4(wl, kc), _cache4(wl, vc), wl.cache_seqlens, wl.block_table,
                                     wl.scale, max_seqlen_k=max_seqlen_k or wl.max_seqlen, k_scale=wl.k_scale,
                                     v_scale=wl.v_scale, return_lse=True)
    torch.cuda.synchronize()
    return out, lse, kc, vc


def _oracle(wl, kc_bits, vc_bits, seqs=None):
    return O.paged_attn_decode(bits(wl.q), kc_bits, vc_bits, wl.cache_seqlens.cpu().numpy(),
                               wl.block_table.cpu().numpy(), wl.block_size, wl.scale, wl.cache_dtype,
                               wl.k_scale, wl.v_scale, seqs=seqs)


def _tol(wl):
    return (FP8_ATOL, FP8_RTOL) if wl.cache_dtype in ("fp8_e4m3", "int8") else (BF16_ATOL, BF16_RTOL)


def _check(wl, out, lse, ref, ref_lse, seqs=None):
    atol, rtol = _tol(wl)
    got = f64(out)
    gl = f64(lse)
    if seqs is not None:
        got, gl, ref, ref_lse = got[seqs], gl[seqs], ref[seqs], ref_lse[seqs]
    err = assert_close(got, ref, atol, rtol, f"{wl.name} out")
    assert_close(gl, ref_lse, 1e-3, 1e-3, f"{wl.name} lse")
    return err


def test_decode_worked_example(pkv):
    """The docs' decode example: write at the derived slots, attend lengths 31/33/71."""
    wl = W.decode_example(device="cuda")
    out, lse, kc, vc = _gpu_step(pkv, wl)
    rk, rv = O.kv_cache_write(bits(wl.k_new), bits(wl.v_new), bits(wl.k_cache), bits(wl.v_cache),
                              wl.slot_mapping.cpu().numpy())
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    ref, ref_lse = _oracle(wl, rk, rv)
    _check(wl, out, lse, ref, ref_lse)


CASES = [
    # (lens_before, Hq, Hkv, D, bs, cache_dtype)
    ([0, 14, 15, 16, 30, 31, 32, 33, 63, 100], 8, 8, 128, 16, "bf16"),
    ([5, 200, 1500, 47, 3000], 32, 8, 128, 16, "bf16"),
    ([5, 200, 1500, 47, 3000], 64, 8, 128, 32, "bf16"),
    ([1, 31, 700, 2049], 4, 2, 64, 32, "bf16"),
    ([9, 600, 1300], 3, 1, 64, 16, "bf16"),
    ([17, 555, 2500, 4100], 16, 2, 128, 64, "bf16"),
    ([5, 200, 1500, 47, 3000], 32, 8, 128, 16, "fp8_e4m3"),
    ([5, 200, 1500, 47, 3000], 64, 8, 128, 32, "fp8_e4m3"),
    ([1, 31, 700, 2049], 4, 2, 64, 32, "fp8_e4m3"),
    ([0, 3, 63, 1000], 8, 1, 64, 16, "fp8_e4m3"),
    ([5, 200, 1500, 47, 3000], 32, 8, 128, 16, "int8"),
    ([1, 31, 700, 2049], 4, 2, 64, 32, "int8"),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[1]}q{c[2]}kv_d{c[3]}_bs{c[4]}_{c[5]}_{i}" for i, c in enumerate(CASES)])
def test_decode_small_cases(pkv, case):
    lens, Hq, Hkv, D, bs, dt = case
    wl = W.make_decode(lens, Hq, Hkv, D, bs, seed=sum(lens) + Hq, device="cuda", cache_dtype=dt, extra_blocks=5)
    out, lse, kc, vc = _gpu_step(pkv, wl)
    rk, rv = O.kv_cache_write(bits(wl.k_new), bits(wl.v_new), bits(wl.k_cache), bits(wl.v_cache),
                              wl.slot_mapping.cpu().numpy(), cache_dtype=wl.cache_dtype,
                              k_inv_scale=np.float32(wl.k_inv_scale), v_inv_scale=np.float32(wl.v_inv_scale))
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    ref, ref_lse = _oracle(wl, rk, rv)
    _check(wl, out, lse, ref, ref_lse)


def test_decode_split_count_does_not_change_result(pkv):
    """The same inputs with different host bounds (hence split sizes) agree within rounding."""
    wl = W.make_decode([4000, 7000, 123], 32, 8, 128, 16, seed=3, device="cuda")
    a, la, _, _ = _gpu_step(pkv, wl, max_seqlen_k=wl.max_seqlen)
    b, lb, _, _ = _gpu_step(pkv, wl, max_seqlen_k=wl.max_seqlen * 40)
    assert_close(f64(a), f64(b), 1e-2, 1e-2, "splits")
    assert_close(f64(la), f64(lb), 1e-4, 1e-4, "splits lse")


def test_decode_nan_poisoned_unused_slots(pkv):
    """Slots no sequence attends hold NaN: outputs must not change."""
    wl = W.make_decode([7, 40, 300], 16, 4, 128, 16, seed=11, device="cuda", extra_blocks=4)
    out0, lse0, kc, vc = _gpu_step(pkv, wl)
    table = wl.block_table.cpu().numpy()
    used = np.zeros(wl.num_blocks * wl.block_size, dtype=bool)
    for b, L in enumerate(wl.cache_seqlens.cpu().numpy()):
        for p in range(L):
            used[O.slot_of(table[b], p, wl.block_size)] = True
    unused = torch.from_numpy(np.flatnonzero(~used)).cuda()
    kc[unused] = float("nan")
    vc[unused] = float("nan")
    out1, lse1 = pkv.paged_attn_decode(wl.q, _cache4(wl, kc), _cache4(wl, vc), wl.cache_seqlens, wl.block_table,
                                       wl.scale, max_seqlen_k=wl.max_seqlen, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_decode_block_permutation_invariance(pkv):
    wl = W.make_decode([100, 333, 1025], 32, 8, 128, 16, seed=13, device="cuda", extra_blocks=3)
    out0, _, kc, vc = _gpu_step(pkv, wl)
    nb, bs = wl.num_blocks, wl.block_size
    perm = torch.from_numpy(np.random.default_rng(0).permutation(nb)).cuda()
    kc2 = torch.empty_like(kc).view(nb, bs, -1)
    vc2 = torch.empty_like(vc).view(nb, bs, -1)
    kc2[perm] = kc.view(nb, bs, -1)
    vc2[perm] = vc.view(nb, bs, -1)
    bt = wl.block_table.long()
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int()
    out1 = pkv.paged_attn_decode(wl.q, kc2.view(nb, bs, wl.num_kv_heads, -1), vc2.view(nb, bs, wl.num_kv_heads, -1),
                                 wl.cache_seqlens, bt2, wl.scale, max_seqlen_k=wl.max_seqlen)
    torch.cuda.synchronize()
    assert torch.equal(out0, out1)


def test_decode_bad_block_id_is_flagged_not_dereferenced(pkv):
    wl = W.make_decode([40, 40], 8, 2, 64, 16, seed=17, device="cuda")
    bt = wl.block_table.clone()
    bt[1, 1] = 1 << 28  # far outside the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.paged_attn_decode(wl.q, _cache4(wl, wl.k_cache), _cache4(wl, wl.v_cache), wl.cache_seqlens, bt,
                                wl.scale, max_seqlen_k=wl.max_seqlen, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_BLOCK
    assert torch.isfinite(out.float()).all()
    # sequence 0 is untouched by the bad entry
    ref, _ = _oracle(wl, bits(wl.k_cache), bits(wl.v_cache), seqs=[0])
    assert_close(f64(out)[0], ref[0], BF16_ATOL, BF16_RTOL, "seq 0")


def test_decode_length_beyond_block_table_is_flagged(pkv):
    wl = W.make_decode([40, 20], 8, 2, 64, 16, seed=19, device="cuda")
    lens = wl.cache_seqlens.clone()
    lens[1] = 10_000  # more than the table holds
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_attn_decode(wl.q, _cache4(wl, wl.k_cache), _cache4(wl, wl.v_cache), lens, wl.block_table, wl.scale,
                          max_seqlen_k=wl.max_seqlen, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_LENGTH


def test_fp8_subnormal_codes_are_exact(pkv):
    """K and V made of E4M3 subnormal codes only: the widening must keep them (no flush to zero)."""
    B, Hq, Hkv, D, bs = 2, 8, 1, 64, 16
    L = 48
    wl = W.make_decode([L - 1] * B, Hq, Hkv, D, bs, seed=23, device="cuda", cache_dtype="fp8_e4m3")
    g = torch.Generator(device="cuda").manual_seed(1)
    mag = torch.randint(1, 8, wl.k_cache.shape, device="cuda", dtype=torch.uint8, generator=g)
    sign = torch.randint(0, 2, wl.k_cache.shape, device="cuda", dtype=torch.uint8, generator=g) << 7
    kc = (mag | sign).contiguous()
    vc = torch.roll(kc, 1, dims=0).contiguous()
    out, lse = pkv.paged_attn_decode(wl.q, _cache4(wl, kc), _cache4(wl, vc), wl.cache_seqlens, wl.block_table,
                                     wl.scale, max_seqlen_k=wl.max_seqlen, k_scale=64.0, v_scale=64.0,
                                     return_lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = O.paged_attn_decode(bits(wl.q), bits(kc), bits(vc), wl.cache_seqlens.cpu().numpy(),
                                       wl.block_table.cpu().numpy(), bs, wl.scale, "fp8_e4m3", 64.0, 64.0)
    # values are ~0.1..0.9 after scaling: a flush would leave zeros
    assert_close(f64(out), ref, 1e-2, 2e-2, "subnormal V")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, "subnormal K")


# ---------------------------------------------------------------------------
# full-size workloads, sampled sequences
# ---------------------------------------------------------------------------


def _full_size(pkv, wl, seqs):
    out, lse, kc, vc = _gpu_step(pkv, wl)
    # the new tokens were written bit-exactly where the scheduler put them
    slots = wl.slot_mapping.long()
    if wl.cache_dtype == "bf16":
        assert torch.equal(kc[slots], wl.k_new) and torch.equal(vc[slots], wl.v_new)
        kb, vb = kc, vc
    else:
        quant = O.quantize_to_e4m3 if wl.cache_dtype == "fp8_e4m3" else O.quantize_to_int8
        assert np.array_equal(bits(kc[slots]), quant(bits(wl.k_new), np.float32(wl.k_inv_scale)))
        assert np.array_equal(bits(vc[slots]), quant(bits(wl.v_new), np.float32(wl.v_inv_scale)))
        kb, vb = kc, vc
    # copy only the sampled sequences' blocks to the host for the oracle
    table = wl.block_table.cpu().numpy()
    lens = wl.cache_seqlens.cpu().numpy()
    sub_blocks = sorted({int(x) for s in seqs for x in table[s][:-(-lens[s] // wl.block_size)]})
    remap = {blk: i for i, blk in enumerate(sub_blocks)}
    idx = torch.tensor(sub_blocks, device="cuda")
    kc4, vc4 = _cache4(wl, kb), _cache4(wl, vb)
    k_sub = bits(kc4[idx]).reshape(-1, wl.num_kv_heads, wl.head_dim)
    v_sub = bits(vc4[idx]).reshape(-1, wl.num_kv_heads, wl.head_dim)
    table_sub = np.full_like(table, -1)
    for s in seqs:
        n = -(-lens[s] // wl.block_size)
        table_sub[s, :n] = [remap[int(x)] for x in table[s][:n]]
    ref, ref_lse = O.paged_attn_decode(bits(wl.q), k_sub, v_sub, lens, table_sub, wl.block_size, wl.scale,
                                       wl.cache_dtype, wl.k_scale, wl.v_scale, seqs=seqs)
    err = _check(wl, out, lse, ref, ref_lse, seqs=seqs)
    assert torch.isfinite(out.float()).all()
    return err


def test_decode_batch64_full_size_sampled(pkv):
    wl = W.decode_batch(device="cuda")
    lens = wl.lens_before
    seqs = [int(np.argmin(lens)), int(np.argmax(lens)), 7, 33]
    _full_size(pkv, wl, seqs)


@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3", "int8"])
def test_long_decode_full_size_sampled(pkv, dt):
    wl = W.long_decode(device="cuda", cache_dtype=dt)
    _full_size(pkv, wl, [0, 5])


def test_nvtx_tracing_changes_no_result(pkv):
    """With NVTX ranges on, the write, decode and varlen calls give the same bits as with them off."""
    wl = W.decode_example(device="cuda")
    vw = W.make_varlen_packed([200, 1, 131], [200, 7, 300], 8, 2, 128, seed=77, device="cuda")

    def run():
        out, lse, kc, vc = _gpu_step(pkv, wl)
        vo, vl = pkv.paged_attn_varlen(vw.q, vw.k, vw.v, vw.cu_seqlens_q, vw.cu_seqlens_k, vw.max_len_q,
                                       vw.max_len_k, scale=vw.scale, return_lse=True)
        torch.cuda.synchronize()
        return out, lse, kc, vc, vo, vl

    plain = run()
    pkv.set_nvtx(True)
    try:
        traced = run()
    finally:
        pkv.set_nvtx(False)
    for a, b in zip(plain, traced):  # byte for byte (lse is float32)
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))
    rk, rv = O.kv_cache_write(bits(wl.k_new), bits(wl.v_new), bits(wl.k_cache), bits(wl.v_cache),
                              wl.slot_mapping.cpu().numpy())
    assert np.array_equal(bits(traced[2]), rk) and np.array_equal(bits(traced[3]), rv)
    ref, ref_lse = _oracle(wl, rk, rv)
    _check(wl, traced[0], traced[1], ref, ref_lse)
