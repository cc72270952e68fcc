"""Decode with the step's append in one launch, on the GPU, against the oracle.

Sources: "ページド・アテンション" (transformers docs), "デコードパス": the example's
cache_seqlens count the tokens cached before the step, and the new token takes
the next position; "効率的な KV キャッシュ管理と Attention 計算" (itan.pw),
"Attention モジュールの実装": the step's K/V are written, then attended.
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


def _fused(pkv, wl, err=None):
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    before = (wl.cache_seqlens - 1).contiguous()
    out, lse = pkv.paged_attn_decode_with_kvcache(
        wl.q, wl.k_new, wl.v_new, _cache4(wl, kc), _cache4(wl, vc), before, wl.block_table, wl.scale,
        max_seqlen_k=wl.max_seqlen, k_scale=wl.k_scale, v_scale=wl.v_scale, k_inv_scale=wl.k_inv_scale,
        v_inv_scale=wl.v_inv_scale, return_lse=True, err_flag=err)
    torch.cuda.synchronize()
    return out, lse, kc, vc


def _separate(pkv, wl):
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    pkv.kv_cache_write(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping, k_inv_scale=wl.k_inv_scale,
                       v_inv_scale=wl.v_inv_scale)
    out, lse = pkv.paged_attn_decode(wl.q, _cache4(wl, kc), _cache4(wl, vc), wl.cache_seqlens, wl.block_table,
                                     wl.scale, max_seqlen_k=wl.max_seqlen, k_scale=wl.k_scale, v_scale=wl.v_scale,
                                     return_lse=True)
    torch.cuda.synchronize()
    return out, lse, kc, vc


def _oracle(wl, seqs=None):
    return O.paged_attn_decode_with_kvcache(
        bits(wl.q), bits(wl.k_new), bits(wl.v_new), bits(wl.k_cache), bits(wl.v_cache), wl.lens_before,
        wl.block_table.cpu().numpy(), wl.block_size, wl.scale, wl.cache_dtype, wl.k_scale, wl.v_scale,
        wl.k_inv_scale, wl.v_inv_scale, seqs=seqs)


def test_with_kvcache_worked_example(pkv):
    wl = W.decode_example(device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, kc, vc = _fused(pkv, wl, err)
    ref, ref_lse, rk, rv = _oracle(wl)
    assert int(err.item()) == 0
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)  # rows 94, 32, 198 and nothing else
    assert_close(f64(out), ref, BF16_ATOL, BF16_RTOL, "out")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, "lse")


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs,dt", [
    ([0, 15, 16, 31, 32, 100, 1500], 32, 8, 128, 16, "bf16"),
    ([1, 63, 64, 700, 2049], 4, 2, 64, 32, "fp8_e4m3"),
    ([0, 5, 3000], 64, 8, 128, 32, "fp8_e4m3"),
    ([9, 600, 1300], 3, 1, 64, 16, "bf16"),
    ([0, 77, 2100], 16, 4, 128, 16, "int8"),
])
def test_with_kvcache_small_cases(pkv, lens, Hq, Hkv, D, bs, dt):
    wl = W.make_decode(lens, Hq, Hkv, D, bs, seed=31 + len(lens), device="cuda", cache_dtype=dt)
    out, lse, kc, vc = _fused(pkv, wl)
    ref, ref_lse, rk, rv = _oracle(wl)
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)
    atol, rtol = (FP8_ATOL, FP8_RTOL) if dt in ("fp8_e4m3", "int8") else (BF16_ATOL, BF16_RTOL)
    assert_close(f64(out), ref, atol, rtol, "out")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, "lse")


def test_empty_cache_attends_only_the_new_token(pkv):
    wl = W.make_decode([0, 0, 0], 8, 2, 128, 16, seed=5, device="cuda")
    out, _, _, _ = _fused(pkv, wl)
    vn = wl.v_new.float().repeat_interleave(4, dim=1)
    assert torch.equal(out.float(), vn)


def test_bad_block_at_the_new_position_is_flagged_and_not_written(pkv):
    wl = W.make_decode([20, 40], 8, 2, 128, 16, seed=6, device="cuda", extra_blocks=2)
    table = wl.block_table.clone()
    table[1, 40 // 16] = wl.num_blocks + 3  # the block the new token of sequence 1 needs
    wl.block_table = table
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, _, kc, vc = _fused(pkv, wl, err)
    assert int(err.item()) & 2
    # sequence 0 was appended; no other slot changed
    s0 = int(wl.slot_mapping[0].item())
    changed = (kc != wl.k_cache).reshape(kc.shape[0], -1).any(dim=1).nonzero().flatten().tolist()
    assert changed == [s0] or changed == []  # equal values would not show as a change
    assert torch.equal(kc[s0], wl.k_new[0]) and torch.equal(vc[s0], wl.v_new[0])


@pytest.mark.parametrize("which", ["decode_batch", "long_bf16", "long_fp8"])
def test_fused_equals_write_then_decode_at_full_size(pkv, which):
    """The benchmark's workloads: one launch gives the same caches and outputs as two."""
    if which == "decode_batch":
        wl = W.decode_batch(device="cuda")
    else:
        wl = W.long_decode(device="cuda", cache_dtype="bf16" if which == "long_bf16" else "fp8_e4m3")
    out, lse, kc, vc = _fused(pkv, wl)
    out2, lse2, kc2, vc2 = _separate(pkv, wl)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # and two sampled sequences against the oracle
    seqs = [0, wl.batch - 1]
    table = wl.block_table.cpu().numpy()
    blocks = sorted({int(x) for s in seqs for x in table[s][:-(-int(wl.lens_before[s] + 1) // wl.block_size)]})
    remap = {blk: i for i, blk in enumerate(blocks)}
    idx = torch.tensor(blocks, device="cuda")
    sh = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    ks = bits(kc.view(sh)[idx]).reshape(-1, wl.num_kv_heads, wl.head_dim)
    vs = bits(vc.view(sh)[idx]).reshape(-1, wl.num_kv_heads, wl.head_dim)
    ts = np.full_like(table, -1)
    for s in seqs:
        n = -(-int(wl.lens_before[s] + 1) // wl.block_size)
        ts[s, :n] = [remap[int(x)] for x in table[s][:n]]
    ref, ref_lse = O.paged_attn_decode(bits(wl.q), ks, vs, wl.cache_seqlens.cpu().numpy(), ts, wl.block_size,
                                       wl.scale, wl.cache_dtype, wl.k_scale, wl.v_scale, seqs=seqs)
    atol, rtol = (FP8_ATOL, FP8_RTOL) if wl.cache_dtype == "fp8_e4m3" else (BF16_ATOL, BF16_RTOL)
    assert_close(f64(out)[seqs], ref[seqs], atol, rtol, "out")
