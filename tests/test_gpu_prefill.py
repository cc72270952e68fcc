"""Causal varlen prefill (tcgen05 kernel) on the GPU vs the fp64 oracle.

Small cases compare every output row; the full-size workloads (8 sequences of
128..2048 tokens, packed and paged; the mixed chunked-prefill batch) compare
sampled sequences in the launch configuration the benchmark uses.
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


def _packed(pkv, wl, max_len_k=None):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = pkv.paged_attn_varlen(wl.q, wl.k, wl.v, wl.cu_seqlens_q, wl.cu_seqlens_k, wl.max_len_q,
                                     max_len_k or wl.max_len_k, scale=wl.scale, return_lse=True, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    return out, lse


def _check_rows(out, lse, ref, ref_lse, rows=None, what=""):
    got, gl = f64(out), f64(lse)
    if rows is not None:
        got, ref, gl, ref_lse = got[rows], ref[rows], gl[:, rows], ref_lse[:, rows]
    assert_close(got, ref, BF16_ATOL, BF16_RTOL, what + " out")
    assert_close(gl, ref_lse, 1e-3, 1e-3, what + " lse")


PACKED = [
    # (q_lens, k_lens, Hq, Hkv, D)
    ([128], [128], 4, 4, 128),
    ([1, 2, 127, 128, 129, 300], [1, 2, 127, 128, 129, 300], 8, 2, 128),
    ([100, 37, 260], [400, 37, 900], 8, 1, 128),              # queries are the last positions
    ([10, 3, 1], [0, 1, 7], 4, 2, 64),                         # the docs' varlen example (empty rows)
    ([256, 513], [256, 513], 16, 2, 64),
    ([700, 5, 1000], [700, 5, 1000], 32, 8, 128),
    ([33, 200], [33, 200], 8, 8, 64),
    ([50], [50], 2, 1, 128),                                   # one pair of heads, one tile
    ([10, 3, 1], [0, 1, 7], 4, 2, 128),                        # empty rows, paired heads
    ([300, 129], [300, 500], 6, 2, 128),                       # odd group: single-CTA path
    # 40 sequences of 1..400 queries over 0..300 more keys: many units of every tile count
    (list(np.random.default_rng(5).integers(1, 401, 40)),
     list(np.random.default_rng(5).integers(1, 401, 40) + np.random.default_rng(6).integers(0, 301, 40)), 8, 2, 64),
]


@pytest.mark.parametrize("case", PACKED, ids=[f"{len(c[0])}seq_{c[2]}q{c[3]}kv_d{c[4]}_{i}" for i, c in enumerate(PACKED)])
def test_varlen_packed_small(pkv, case):
    q_lens, k_lens, Hq, Hkv, D = case
    wl = W.make_varlen_packed(q_lens, k_lens, Hq, Hkv, D, seed=sum(q_lens) + 7 * Hq + D, device="cuda")
    out, lse = _packed(pkv, wl)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(wl.k), bits(wl.v), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True)
    _check_rows(out, lse, ref, ref_lse, what=str(case))


def _write_new_tokens(pkv, wl):
    kc, vc = wl.k_cache.clone(), wl.v_cache.clone()
    pkv.kv_cache_write(wl.k_new, wl.v_new, kc, vc, wl.slot_mapping, k_inv_scale=wl.extra.get("k_inv_scale", 1.0),
                       v_inv_scale=wl.extra.get("v_inv_scale", 1.0))
    return kc, vc


def _paged(pkv, wl, kc, vc, gather=False, max_len_k=None):
    """Paged varlen; gather=True gives the library the bound that lets it gather K/V into a packed buffer."""
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = pkv.paged_attn_varlen(wl.q, kc.view(shape4), vc.view(shape4), wl.cu_seqlens_q, wl.cu_seqlens_k,
                                     wl.max_len_q, max_len_k or wl.max_len_k, block_table=wl.block_table, scale=wl.scale,
                                     return_lse=True, err_flag=err, gather_k_tokens=W.gather_tokens(wl) if gather else 0,
                                     k_scale=wl.extra.get("k_scale", 1.0), v_scale=wl.extra.get("v_scale", 1.0))
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    return out, lse


PAGED = [
    # (q_lens, prefix_lens, Hq, Hkv, D, bs)
    ([128, 50, 300], [0, 0, 0], 8, 2, 128, 16),
    ([64, 129, 7], [500, 31, 1000], 8, 2, 128, 32),
    ([200, 1, 1, 64], [0, 700, 33, 900], 32, 8, 128, 16),
    ([90, 260], [130, 0], 4, 1, 64, 64),
    ([300, 17], [40, 257], 8, 4, 128, 128),
    ([150, 150], [600, 5], 8, 2, 128, 256),
    ([100, 333], [77, 0], 8, 2, 64, 16),
    ([250, 3], [200, 600], 16, 4, 128, 64),
]


@pytest.mark.parametrize("gather", [False, True], ids=["direct", "gathered"])
@pytest.mark.parametrize("case", PAGED, ids=[f"bs{c[5]}_{c[2]}q{c[3]}kv_d{c[4]}_{i}" for i, c in enumerate(PAGED)])
def test_varlen_paged_small(pkv, case, gather):
    q_lens, prefix, Hq, Hkv, D, bs = case
    wl = W.make_varlen_paged(q_lens, prefix, Hq, Hkv, D, bs, seed=sum(q_lens) + sum(prefix) + bs, device="cuda",
                             extra_blocks=3)
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=gather)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=bs)
    _check_rows(out, lse, ref, ref_lse, what=str(case))


def test_varlen_paged_equals_packed(pkv):
    """The same keys read through a permuted pool or packed give the same result."""
    wl = W.make_varlen_paged([300, 77, 500], [0, 0, 0], 16, 4, 128, 16, seed=41, device="cuda")
    kc, vc = _write_new_tokens(pkv, wl)
    out_p, _ = _paged(pkv, wl, kc, vc)
    out_k = pkv.paged_attn_varlen(wl.q, wl.k_new, wl.v_new, wl.cu_seqlens_q, wl.cu_seqlens_q, wl.max_len_q,
                                  wl.max_len_q, scale=wl.scale)
    torch.cuda.synchronize()
    assert_close(f64(out_p), f64(out_k), 1e-2, 1e-2, "paged vs packed")


def test_varlen_paged_nan_poisoned_unused_slots(pkv):
    wl = W.make_varlen_paged([100, 45], [60, 200], 8, 2, 128, 32, seed=43, device="cuda", extra_blocks=4)
    kc, vc = _write_new_tokens(pkv, wl)
    out0, lse0 = _paged(pkv, wl, kc, vc)
    table = wl.block_table.cpu().numpy()
    used = np.zeros(wl.num_blocks * wl.block_size, dtype=bool)
    for b, L in enumerate(wl.k_lens):
        for p in range(int(L)):
            used[O.slot_of(table[b], p, wl.block_size)] = True
    unused = torch.from_numpy(np.flatnonzero(~used)).cuda()
    kc[unused] = float("nan")
    vc[unused] = float("nan")
    out1, lse1 = _paged(pkv, wl, kc, vc)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_varlen_chunked_equals_whole(pkv):
    """Prefix reuse: the last chunk's queries over prefix+chunk keys equal the same rows of one prefill."""
    L, split = 700, 450
    whole = W.make_varlen_packed([L], [L], 8, 2, 128, seed=45, device="cuda")
    out_w, _ = _packed(pkv, whole)
    part = pkv.paged_attn_varlen(whole.q[split:].contiguous(), whole.k, whole.v,
                                 torch.tensor([0, L - split], dtype=torch.int32, device="cuda"),
                                 torch.tensor([0, L], dtype=torch.int32, device="cuda"), L - split, L,
                                 scale=whole.scale)
    torch.cuda.synchronize()
    assert_close(f64(part), f64(out_w[split:]), 1e-2, 1e-2, "chunked")


def test_varlen_bad_block_is_flagged(pkv):
    wl = W.make_varlen_paged([64, 64], [100, 100], 8, 2, 128, 16, seed=47, device="cuda")
    kc, vc = _write_new_tokens(pkv, wl)
    bt = wl.block_table.clone()
    bt[0, 2] = 1 << 29
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    out = pkv.paged_attn_varlen(wl.q, kc.view(shape4), vc.view(shape4), wl.cu_seqlens_q, wl.cu_seqlens_k,
                                wl.max_len_q, wl.max_len_k, block_table=bt, scale=wl.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_BLOCK
    ref, _ = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                 wl.cu_seqlens_k.cpu().numpy(), wl.scale, True, block_table=wl.block_table.cpu().numpy(),
                                 block_size=16, seqs=[1])
    rows = np.arange(64, 128)
    assert_close(f64(out)[rows], ref[rows], BF16_ATOL, BF16_RTOL, "sequence 1")


# ---------------------------------------------------------------------------
# full-size workloads, sampled sequences
# ---------------------------------------------------------------------------


def _sub_pool(wl, kc, vc, seqs):
    """Host copies of only the blocks the sampled sequences use, with a remapped table."""
    table = wl.block_table.cpu().numpy()
    nb = [-(-int(L) // wl.block_size) for L in wl.k_lens]
    blocks = sorted({int(x) for s in seqs for x in table[s][:nb[s]]})
    remap = {blk: i for i, blk in enumerate(blocks)}
    idx = torch.tensor(blocks, device="cuda")
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    ks = bits(kc.view(shape4)[idx]).reshape(-1, wl.num_kv_heads, wl.head_dim)
    vs = bits(vc.view(shape4)[idx]).reshape(-1, wl.num_kv_heads, wl.head_dim)
    tsub = np.full_like(table, -1)
    for s in seqs:
        tsub[s, :nb[s]] = [remap[int(x)] for x in table[s][:nb[s]]]
    return ks, vs, tsub


def _rows_of(wl, seqs):
    cu = wl.cu_seqlens_q.cpu().numpy()
    return np.concatenate([np.arange(cu[s], cu[s + 1]) for s in seqs])


def test_varlen_prefill_full_size_packed(pkv):
    wl = W.varlen_prefill(device="cuda")
    out, lse = _packed(pkv, wl)
    seqs = [int(np.argmax(wl.q_lens)), int(np.argmin(wl.q_lens))]
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(wl.k), bits(wl.v), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True, seqs=seqs)
    _check_rows(out, lse, ref, ref_lse, rows=_rows_of(wl, seqs), what="prefill packed")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("gather", [False, True], ids=["direct", "gathered"])
def test_varlen_prefill_full_size_paged(pkv, gather):
    wl = W.varlen_prefill(device="cuda", paged=True)
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=gather)
    seqs = [int(np.argmax(wl.q_lens)), 3]
    ks, vs, tsub = _sub_pool(wl, kc, vc, seqs)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), ks, vs, wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True, block_table=tsub,
                                       block_size=wl.block_size, seqs=seqs)
    _check_rows(out, lse, ref, ref_lse, rows=_rows_of(wl, seqs), what="prefill paged")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("gather", [False, True], ids=["direct", "gathered"])
def test_mixed_chunked_full_size(pkv, gather):
    """Four 512-query chunks over 0/2K/4K/8K prefixes (two sharing blocks) + 60 decode rows, one call."""
    wl = W.mixed_chunked(device="cuda")
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=gather)
    seqs = [0, 1, 2, 3, 4, 30, 63]
    ks, vs, tsub = _sub_pool(wl, kc, vc, seqs)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), ks, vs, wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True, block_table=tsub,
                                       block_size=wl.block_size, seqs=seqs)
    _check_rows(out, lse, ref, ref_lse, rows=_rows_of(wl, seqs), what="mixed")
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("gather", [False, True], ids=["direct", "gathered"])
def test_mixed_light_chunk_heavy_decode(pkv, gather):
    """One 200-query chunk beside 100 long decode rows: the call gives the prefill few CTAs (the routed
    rows' decode kernels take the other SMs from the start); every output row is still exact."""
    rng = np.random.default_rng(21)
    dec = rng.integers(4096, 8192, size=100, endpoint=True)
    wl = W.make_varlen_paged(np.r_[200, np.ones(100, dtype=np.int64)], np.r_[100, dec], 32, 8, 128, 16, seed=22,
                             device="cuda")
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=gather)
    seqs = [0, 1, 50, 100]
    ks, vs, tsub = _sub_pool(wl, kc, vc, seqs)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), ks, vs, wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True, block_table=tsub,
                                       block_size=wl.block_size, seqs=seqs)
    _check_rows(out, lse, ref, ref_lse, rows=_rows_of(wl, seqs), what="light chunk")


MIXED_MATRIX = [(hq, hkv, d, dt, g) for hq, hkv in ((8, 2), (6, 2)) for d in (64, 128)
                for dt in ("bf16", "fp8_e4m3", "int8") for g in (False, True)
                if not (dt != "bf16" and d == 64 and not g)]  # one-byte d64 pages need the gather bound


@pytest.mark.parametrize("case", MIXED_MATRIX,
                         ids=[f"{c[0]}q{c[1]}kv_d{c[2]}_{c[3]}_{'gathered' if c[4] else 'direct'}" for c in MIXED_MATRIX])
def test_mixed_batch_matrix(pkv, case):
    """Three chunks over prefixes beside 25 routed decode rows, in one call, for even and odd GQA
    groups (head pairs / tile pairs), head dim 64 and 128, bf16 / FP8 / INT8 caches, pages read
    directly or gathered: every output row against the oracle.  The call splits the SMs between
    the prefill tiles and the decode rows by its own model of the two loads."""
    Hq, Hkv, D, dt, gather = case
    rng = np.random.default_rng(Hq + D)
    dec = rng.integers(100, 1200, size=25, endpoint=True)
    wl = W.make_varlen_paged(np.r_[300, 130, 77, np.ones(25, dtype=np.int64)], np.r_[0, 450, 900, dec], Hq, Hkv, D,
                             16, seed=Hq * 7 + D, device="cuda", extra_blocks=2)
    if dt != "bf16":
        wl = W.to_fp8_cache(wl, dt)
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=gather)
    kw = dict(kv_dtype=dt, k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"]) if dt != "bf16" else {}
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=16, **kw)
    atol, rtol = (BF16_ATOL, BF16_RTOL) if dt == "bf16" else (FP8_ATOL, FP8_RTOL)
    assert_close(f64(out), ref, atol, rtol, f"mixed {case}")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, f"mixed lse {case}")


# ---------------------------------------------------------------------------
# FP8 E4M3 cache in prefill (K/V gathered and widened, scales folded)
# ---------------------------------------------------------------------------


FP8_PAGED = [
    # (q_lens, prefix_lens, Hq, Hkv, D, bs)
    ([128, 50, 300], [0, 0, 0], 8, 2, 128, 16),
    ([200, 1, 1, 64], [0, 700, 33, 900], 32, 8, 128, 16),
    ([90, 260], [130, 0], 4, 1, 64, 64),
    ([150, 150], [600, 5], 8, 2, 128, 256),
]


@pytest.mark.parametrize("case", FP8_PAGED, ids=[f"bs{c[5]}_{c[2]}q{c[3]}kv_d{c[4]}_{i}" for i, c in
                                                 enumerate(FP8_PAGED)])
def test_varlen_paged_fp8(pkv, case):
    q_lens, prefix, Hq, Hkv, D, bs = case
    wl = W.to_fp8_cache(W.make_varlen_paged(q_lens, prefix, Hq, Hkv, D, bs, seed=sum(q_lens) + 7, device="cuda",
                                            extra_blocks=2))
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=True)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=bs,
                                       kv_dtype="fp8_e4m3", k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
    assert_close(f64(out), ref, FP8_ATOL, FP8_RTOL, f"fp8 {case}")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, f"fp8 lse {case}")


# One-byte pages read by the tile loop itself (no gather bound): head dim 128 only.
CODED_DIRECT = [c for c in FP8_PAGED if c[4] == 128] + [
    ([1, 2, 127, 128, 129, 300], [0, 5, 0, 700, 1, 2], 8, 1, 128, 32),   # ragged tails, odd group
    ([260], [0], 64, 8, 128, 128),                                       # one page per tile
]


@pytest.mark.parametrize("dt", ["fp8_e4m3", "int8"])
@pytest.mark.parametrize("case", CODED_DIRECT, ids=[f"bs{c[5]}_{c[2]}q{c[3]}kv_{i}" for i, c in
                                                    enumerate(CODED_DIRECT)])
def test_varlen_paged_one_byte_direct(pkv, case, dt):
    """FP8 / INT8 pages widened to f16 in shared memory by the tile loop, against the oracle
    over the same codes; and equal, within the same tolerance, to the gathered path."""
    q_lens, prefix, Hq, Hkv, D, bs = case
    wl = W.to_fp8_cache(W.make_varlen_paged(q_lens, prefix, Hq, Hkv, D, bs, seed=sum(q_lens) + 11, device="cuda",
                                            extra_blocks=2), dt)
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=False)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=bs,
                                       kv_dtype=dt, k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
    assert_close(f64(out), ref, FP8_ATOL, FP8_RTOL, f"{dt} direct {case}")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, f"{dt} direct lse {case}")
    out_g, _ = _paged(pkv, wl, kc, vc, gather=True)
    assert_close(f64(out), f64(out_g), FP8_ATOL, FP8_RTOL, f"{dt} direct vs gathered {case}")


@pytest.mark.parametrize("dt", ["fp8_e4m3", "int8"])
def test_varlen_prefill_full_size_paged_one_byte_direct(pkv, dt):
    wl = W.to_fp8_cache(W.varlen_prefill(device="cuda", paged=True), dt)
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=False)
    seqs = [int(np.argmax(wl.q_lens)), 3]
    ks, vs, tsub = _sub_pool(wl, kc, vc, seqs)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), ks, vs, wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True, block_table=tsub,
                                       block_size=wl.block_size, seqs=seqs, kv_dtype=dt,
                                       k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
    rows = _rows_of(wl, seqs)
    assert_close(f64(out)[rows], ref[rows], FP8_ATOL, FP8_RTOL, f"prefill paged {dt} direct")


def test_varlen_prefill_full_size_paged_fp8(pkv):
    wl = W.to_fp8_cache(W.varlen_prefill(device="cuda", paged=True))
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=True)
    seqs = [int(np.argmax(wl.q_lens)), 3]
    ks, vs, tsub = _sub_pool(wl, kc, vc, seqs)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), ks, vs, wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True, block_table=tsub,
                                       block_size=wl.block_size, seqs=seqs, kv_dtype="fp8_e4m3",
                                       k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
    rows = _rows_of(wl, seqs)
    assert_close(f64(out)[rows], ref[rows], FP8_ATOL, FP8_RTOL, "prefill paged fp8")


def test_gather_bound_too_small_is_flagged(pkv):
    """Keys past the caller's gather bound are not gathered; the call flags it and faults nothing."""
    wl = W.make_varlen_paged([300, 200], [100, 0], 8, 2, 128, 16, seed=99, device="cuda")
    kc, vc = _write_new_tokens(pkv, wl)
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_attn_varlen(wl.q, kc.view(shape4), vc.view(shape4), wl.cu_seqlens_q, wl.cu_seqlens_k, wl.max_len_q,
                          wl.max_len_k, block_table=wl.block_table, scale=wl.scale, err_flag=err,
                          gather_k_tokens=W.gather_tokens(wl) - 100)
    torch.cuda.synchronize()
    assert int(err.item()) & 4  # PKV_DEVERR_LENGTH


@pytest.mark.parametrize("batch", [1100, 2300])
def test_packed_batch_larger_than_the_prep_cta(pkv, batch):
    """1100 or 2300 packed sequences of 1..40 queries (more than the prep kernel's 1024 threads:
    the unit list over two or three sequences per thread): every row against the oracle."""
    rng = np.random.default_rng(31)
    lq = rng.integers(1, 41, size=batch)
    lk = lq + rng.integers(0, 30, size=batch)
    wl = W.make_varlen_packed(list(lq), list(lk), 8, 2, 64, seed=32, device="cuda")
    out, lse = _packed(pkv, wl)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(wl.k), bits(wl.v), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True)
    _check_rows(out, lse, ref, ref_lse, what=f"{batch} packed sequences")


@pytest.mark.parametrize("n_dec", [1300, 2400])
@pytest.mark.parametrize("gather", [False, True], ids=["direct", "gathered"])
def test_mixed_batch_larger_than_the_prep_cta(pkv, gather, n_dec):
    """Three chunks among 1300 or 2400 decode rows (more than the prep kernel's 1024 threads:
    routing, packed offsets carried across two or three chunks of sequences, the unit list and
    the SM split over them): every row against the oracle."""
    rng = np.random.default_rng(33)
    q_lens = np.ones(n_dec + 3, dtype=np.int64)
    prefix = rng.integers(8, 96, size=n_dec + 3)
    pos = rng.choice(n_dec + 3, size=3, replace=False)  # the chunks sit among the decode rows
    q_lens[pos] = [150, 64, 200]
    prefix[pos] = [0, 300, 129]
    wl = W.make_varlen_paged(q_lens, prefix, 8, 2, 128, 16, seed=34, device="cuda")
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=gather)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=16)
    _check_rows(out, lse, ref, ref_lse, what=f"{n_dec + 3}-sequence mixed batch ({'gathered' if gather else 'direct'})")


@pytest.mark.parametrize("gather", [False, True], ids=["direct", "gathered"])
def test_keys_past_the_block_table_are_flagged(pkv, gather):
    """A sequence that claims more keys than its block-table row holds is flagged
    (PKV_DEVERR_LENGTH); no key past the table is read, and the other sequence is exact."""
    wl = W.make_varlen_paged([64, 40], [100, 30], 8, 2, 128, 16, seed=97, device="cuda")
    kc, vc = _write_new_tokens(pkv, wl)
    cap0 = wl.block_table.shape[1] * wl.block_size
    cu_k = torch.tensor([0, cap0 + 14, cap0 + 14 + 70], dtype=torch.int32, device="cuda")
    shape4 = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pkv.paged_attn_varlen(wl.q, kc.view(shape4), vc.view(shape4), wl.cu_seqlens_q, cu_k, wl.max_len_q,
                                cap0 + 14, block_table=wl.block_table, scale=wl.scale, err_flag=err,
                                gather_k_tokens=cap0 + 14 + 70 if gather else 0)
    torch.cuda.synchronize()
    assert int(err.item()) & 4  # PKV_DEVERR_LENGTH
    ref, _ = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                 wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                 block_table=wl.block_table.cpu().numpy(), block_size=16, seqs=[1])
    rows = np.arange(64, 104)
    assert_close(f64(out)[rows], ref[rows], BF16_ATOL, BF16_RTOL, "sequence 1")


def test_more_queries_than_max_len_q_is_flagged(pkv):
    """A sequence with more queries than the caller's max_len_q is flagged (PKV_DEVERR_LENGTH); the tiles
    that the bound covers (those with the most keys, counted from the sequence's end) are still exact."""
    wl = W.make_varlen_packed([300, 100], [300, 100], 8, 2, 128, seed=98, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(wl.q)
    pkv.paged_attn_varlen(wl.q, wl.k, wl.v, wl.cu_seqlens_q, wl.cu_seqlens_k, 128, wl.max_len_k, scale=wl.scale,
                          out=out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 4  # PKV_DEVERR_LENGTH
    ref, _ = O.paged_attn_varlen(bits(wl.q), bits(wl.k), bits(wl.v), wl.cu_seqlens_q.cpu().numpy(),
                                 wl.cu_seqlens_k.cpu().numpy(), wl.scale, True)
    rows = np.r_[256:300, 300:400]  # the last query tile of each sequence
    assert_close(f64(out)[rows], ref[rows], BF16_ATOL, BF16_RTOL, "last tiles")


# ---------------------------------------------------------------------------
# several new tokens per sequence (speculative verification): each query row of
# a sequence with up to 8 queries goes to the decode kernels
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("chunk", [False, True], ids=["verify_only", "with_chunk"])
@pytest.mark.parametrize("dt", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("gather", [False, True], ids=["direct", "gathered"])
def test_multi_query_decode_rows(pkv, dt, gather, chunk):
    """1..8 new tokens per sequence: every query row goes to the decode kernels when no
    sequence has more than 8 queries; with a longer chunk in the batch only the
    single-query rows do, and the rest run on the prefill tiles."""
    rng = np.random.default_rng(61)
    q_lens = rng.integers(1, 9, size=12)            # 1..8 new tokens
    if chunk:
        q_lens[3] = 40                              # and one longer chunk (prefill tiles)
    prefix = rng.integers(0, 3000, size=12)
    prefix[5] = 0                                   # a sequence that is only its new tokens
    wl = W.make_varlen_paged(q_lens, prefix, 32, 8, 128, 16, seed=62, device="cuda")
    if dt != "bf16":
        wl = W.to_fp8_cache(wl)
    kc, vc = _write_new_tokens(pkv, wl)
    # (a one-byte cache without a gather bound: the longer chunk's tiles widen the pages themselves)
    out, lse = _paged(pkv, wl, kc, vc, gather=gather)
    kw = {} if dt == "bf16" else dict(kv_dtype="fp8_e4m3", k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=16, **kw)
    atol, rtol = (BF16_ATOL, BF16_RTOL) if dt == "bf16" else (FP8_ATOL, FP8_RTOL)
    assert_close(f64(out), ref, atol, rtol, f"multi-query {dt}")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, f"multi-query lse {dt}")


@pytest.mark.parametrize("case", FP8_PAGED[:3], ids=[f"bs{c[5]}_{c[2]}q{c[3]}kv_d{c[4]}_{i}" for i, c in
                                                     enumerate(FP8_PAGED[:3])])
def test_varlen_paged_int8(pkv, case):
    q_lens, prefix, Hq, Hkv, D, bs = case
    wl = W.to_fp8_cache(W.make_varlen_paged(q_lens, prefix, Hq, Hkv, D, bs, seed=sum(q_lens) + 9, device="cuda",
                                            extra_blocks=2), "int8")
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=True)
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=bs,
                                       kv_dtype="int8", k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
    assert_close(f64(out), ref, FP8_ATOL, FP8_RTOL, f"int8 {case}")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, f"int8 lse {case}")


# (max queries, Hq, Hkv, D, block size, cache type): every sequence's (query, head) rows
# fit one decode pass (queries x group <= 16), so each sequence's K/V is read once
ONE_PASS = [
    (4, 32, 8, 128, 16, "bf16"),      # 16 rows: two 8-row blocks
    (2, 64, 8, 128, 32, "bf16"),      # group 8: 16 rows
    (4, 8, 4, 64, 16, "bf16"),        # group 2: 8 rows, one block, d64
    (4, 32, 8, 128, 16, "fp8_e4m3"),
    (4, 32, 8, 128, 16, "int8"),
    (3, 16, 4, 128, 32, "bf16"),      # 12 rows: the second block half used
]


@pytest.mark.parametrize("case", ONE_PASS, ids=[f"q{c[0]}_{c[1]}q{c[2]}kv_d{c[3]}_bs{c[4]}_{c[5]}" for c in ONE_PASS])
def test_multi_query_one_pass(pkv, case):
    """Speculative verification with few queries: one decode CTA per (split, kv head, sequence)
    computes every query row of the sequence, each over its own bottom-right causal prefix."""
    max_q, Hq, Hkv, D, bs, dt = case
    rng = np.random.default_rng(71 + max_q + Hq)
    q_lens = rng.integers(1, max_q + 1, size=10)
    q_lens[0] = max_q
    prefix = rng.integers(0, 3000, size=10)
    prefix[2] = 0                                   # only its new tokens
    prefix[4] = 5000                                # several splits
    wl = W.make_varlen_paged(q_lens, prefix, Hq, Hkv, D, bs, seed=72 + max_q, device="cuda")
    if dt != "bf16":
        wl = W.to_fp8_cache(wl, dt)
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=False)
    kw = {} if dt == "bf16" else dict(kv_dtype=dt, k_scale=wl.extra["k_scale"], v_scale=wl.extra["v_scale"])
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=bs, **kw)
    atol, rtol = (BF16_ATOL, BF16_RTOL) if dt == "bf16" else (FP8_ATOL, FP8_RTOL)
    assert_close(f64(out), ref, atol, rtol, f"one-pass multi-query {case}")
    assert_close(f64(lse), ref_lse, 1e-3, 1e-3, f"one-pass multi-query lse {case}")


# From this host key bound on, head dim 128 bf16 calls run the prefill kernel whose
# softmax warps all work on one tile at a time (two threads per row).
LONG_BOUND = 4096
PACKED_128 = [c for c in PACKED if c[4] == 128] + [([256, 40], [5000, 40], 8, 2, 128)]


@pytest.mark.parametrize("case", PACKED_128, ids=[f"{len(c[0])}seq_{c[2]}q{c[3]}kv_{i}" for i, c in
                                                  enumerate(PACKED_128)])
def test_varlen_packed_long_key_bound(pkv, case):
    """The packed cases again with a key bound of LONG_BOUND (the one-tile softmax), against the oracle."""
    q_lens, k_lens, Hq, Hkv, D = case
    wl = W.make_varlen_packed(q_lens, k_lens, Hq, Hkv, D, seed=sum(q_lens) + 7 * Hq + D, device="cuda")
    out, lse = _packed(pkv, wl, max_len_k=max(wl.max_len_k, LONG_BOUND))
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(wl.k), bits(wl.v), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True)
    _check_rows(out, lse, ref, ref_lse, what=str(case))


PAGED_128 = [c for c in PAGED if c[4] == 128]


@pytest.mark.parametrize("gather", [False, True], ids=["direct", "gathered"])
@pytest.mark.parametrize("case", PAGED_128, ids=[f"bs{c[5]}_{c[2]}q{c[3]}kv_{i}" for i, c in enumerate(PAGED_128)])
def test_varlen_paged_long_key_bound(pkv, case, gather):
    """The paged cases (routed single-query rows included) with a key bound of LONG_BOUND."""
    q_lens, prefix, Hq, Hkv, D, bs = case
    wl = W.make_varlen_paged(q_lens, prefix, Hq, Hkv, D, bs, seed=sum(q_lens) + sum(prefix) + bs, device="cuda",
                             extra_blocks=3)
    kc, vc = _write_new_tokens(pkv, wl)
    out, lse = _paged(pkv, wl, kc, vc, gather=gather, max_len_k=max(wl.max_len_k, LONG_BOUND))
    ref, ref_lse = O.paged_attn_varlen(bits(wl.q), bits(kc), bits(vc), wl.cu_seqlens_q.cpu().numpy(),
                                       wl.cu_seqlens_k.cpu().numpy(), wl.scale, True,
                                       block_table=wl.block_table.cpu().numpy(), block_size=bs)
    _check_rows(out, lse, ref, ref_lse, what=str(case))
