"""Pins for the CPU oracle: worked examples, closed forms, brute force, invariants.

Each test ties the oracle to something other than itself: numbers printed on
the pages (``tests/golden``), the OCP E4M3 definition, an independent
pure-Python recomputation on tiny inputs, or mathematical invariants.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(x):
    """fp32 -> bf16 bits, round to nearest even (test-side helper, finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def _rand_bf16(rng, shape, scale=1.0):
    return _bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))


# ---------------------------------------------------------------------------
# worked examples
# ---------------------------------------------------------------------------


def test_varlen_worked_example_indexing():
    g = _golden("varlen_example.json")
    cu_q = O.cu_seqlens_from_lens(g["q_lens"])
    cu_k = O.cu_seqlens_from_lens(g["k_lens"])
    assert cu_q.tolist() == g["cu_seq_lens_q"]
    assert cu_k.tolist() == g["cu_seq_lens_k"]
    assert max(g["q_lens"]) == g["max_length_q"] and max(g["k_lens"]) == g["max_length_k"]
    assert cu_q[-1] == g["q_total_tokens"] and cu_k[-1] == g["k_total_tokens"]
    assert O.request_index(cu_q).tolist() == g["q_request_index"]
    assert O.request_index(cu_k).tolist() == g["k_request_index"]


def test_decode_worked_example_blocks_and_slots():
    g = _golden("decode_example.json")
    bs = g["block_size"]
    table = np.array(g["block_table"])
    for b, L in enumerate(g["cache_seqlens"]):
        held = [int(x) for x in table[b] if x >= 0]
        assert held == g["cached_in_blocks"][b]
        # every cached position resolves into one of the blocks the row lists
        used = {O.slot_of(table[b], p, bs) // bs for p in range(L)}
        assert used <= set(held)
        # the row already holds the block the new token (position L) goes to
        assert O.blocks_needed(L + 1, bs) == len(held)
        # "needs a second block" <=> L+1 tokens need more blocks than L tokens
        assert (O.blocks_needed(L + 1, bs) > O.blocks_needed(L, bs)) == g["new_token_needs_another_block"][b]
        assert L // bs == g["new_token_logical_block"][b]
        assert table[b][L // bs] == g["new_token_physical_block"][b]
        assert O.slot_of(table[b], L, bs) == g["derived_new_token_slots"][b]
    # blocks of sequence 2 are not contiguous (3, 5, 6)
    assert np.any(np.diff(g["cached_in_blocks"][2]) != 1)
    with pytest.raises(ValueError):
        O.slot_of(table[0], 40, bs)  # logical block 1 of seq 0 is unallocated (-1)


def test_kv_size_closed_forms():
    g = _golden("kv_size.json")
    for c in g["cases"]:
        n = O.kv_bytes(c["layers"], c["kv_heads"], c["head_dim"], c["tokens"], c["requests"], c["bytes"])
        if "expect_bytes" in c:
            assert n == c["expect_bytes"], c["what"]
        else:
            assert abs(n / 2 ** 30 - c["expect_gib_approx"]) < 0.05 * c["expect_gib_approx"], c["what"]
        # FP8 / INT8 halves every case exactly
        assert O.kv_bytes(c["layers"], c["kv_heads"], c["head_dim"], c["tokens"], c["requests"], 1) * 2 == n
    # GQA (8 KV heads) is 4x smaller than 32 KV heads
    assert O.kv_bytes(32, 32, 128, 1, 1, 2) == 4 * O.kv_bytes(32, 8, 128, 1, 1, 2)


# ---------------------------------------------------------------------------
# FP8 E4M3 (OCP 8-bit floating point specification)
# ---------------------------------------------------------------------------

_SPECIALS = [
    (0.0, 0x00), (-0.0, 0x80), (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (-448.0, 0xFE),
    (2.0 ** -6, 0x08),          # smallest normal
    (2.0 ** -9, 0x01),          # smallest subnormal
    (7 * 2.0 ** -9, 0x07),      # largest subnormal
    (2.0 ** -10, 0x00),         # half the smallest subnormal: tie, rounds to even (zero)
    (3 * 2.0 ** -10, 0x02),     # 1.5 subnormal steps: tie between codes 1 and 2 -> even 2
    (1.0625, 0x38),             # tie between 1.0 (M=0) and 1.125 (M=1) -> M=0
    (1.1875, 0x3A),             # tie between 1.125 (M=1) and 1.25 (M=2) -> M=2
    (240.0, 0x77),              # 1.875 * 2^7
    (464.0, 0x7E),              # above the largest finite: saturates
    (1e30, 0x7E), (-1e30, 0xFE), (np.inf, 0x7E), (-np.inf, 0xFE),
]


@pytest.mark.parametrize("x,code", _SPECIALS)
def test_e4m3_special_values(x, code):
    assert int(O.e4m3_encode_rne_satfinite(np.float32(x))) == code


def test_e4m3_decode_table():
    codes = np.arange(256, dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    finite = np.delete(np.arange(256), [0x7F, 0xFF])
    v = vals[finite]
    assert np.all(np.isfinite(v))
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6
    assert vals[0x38] == 1.0 and vals[0xB8] == -1.0
    # positive codes 0..126 are strictly increasing
    assert np.all(np.diff(vals[:0x7F]) > 0)
    # encode(decode(c)) == c for every non-NaN code
    assert np.array_equal(O.e4m3_encode_rne_satfinite(v.astype(np.float32)), finite.astype(np.uint8))


def test_e4m3_encoder_matches_exhaustive_nearest():
    """Brute force: nearest of the finite codes, ties to the even code, clamp beyond 448."""
    rng = np.random.default_rng(7)
    codes = np.arange(0, 0x7F)  # non-negative finite codes, value increasing with code
    table = O.e4m3_decode(codes.astype(np.uint8))
    xs = np.concatenate([
        rng.standard_normal(3000) * 50, rng.standard_normal(2000) * 0.01,
        (table[:-1] + table[1:]) / 2,              # exact midpoints (ties)
        rng.uniform(-460, 460, 2000)]).astype(np.float32)
    got = O.e4m3_encode_rne_satfinite(xs)
    for x, c in zip(xs.astype(np.float64), got):
        a = min(abs(x), 448.0)
        d = np.abs(table - a)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        want = int(want) | (0x80 if np.signbit(x) else 0)
        assert int(c) == want, (x, int(c), want)


def test_quantize_single_f32_multiply():
    rng = np.random.default_rng(3)
    x = _rand_bf16(rng, 4096)
    inv = np.float32(81.4)
    got = O.quantize_to_e4m3(x, inv)
    xf = O.bf16_bits_to_f64(x).astype(np.float32)
    prod = (xf * inv).astype(np.float32)
    assert np.array_equal(got, O.e4m3_encode_rne_satfinite(prod))
    # the dequantised value is within half a step of x (relative 2^-4 for normals)
    deq = O.e4m3_decode(got) / np.float64(inv)
    xs = O.bf16_bits_to_f64(x)
    big = np.abs(xs * inv) >= 2 ** -6
    assert np.all(np.abs(deq[big] - xs[big]) <= np.abs(xs[big]) * 2 ** -4 + 1e-12)


# ---------------------------------------------------------------------------
# KV-cache write
# ---------------------------------------------------------------------------


def test_write_round_trip_through_block_table():
    rng = np.random.default_rng(11)
    Hkv, D, bs = 2, 8, 4
    lens = [5, 1, 9, 4]
    nblk = [-(-n // bs) for n in lens]
    nb = sum(nblk) + 2
    perm = rng.permutation(nb)
    table = np.full((len(lens), max(nblk)), -1, dtype=np.int64)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n]
        off += n
    streams = [_rand_bf16(rng, (L, Hkv, D)) for L in lens]
    k = np.concatenate(streams)
    v = np.concatenate([s[:, ::-1, :] for s in streams])
    slots = np.concatenate([[table[b][p // bs] * bs + p % bs for p in range(L)] for b, L in enumerate(lens)])
    kc0 = _rand_bf16(rng, (nb * bs, Hkv, D))
    vc0 = _rand_bf16(rng, (nb * bs, Hkv, D))
    kc, vc = O.kv_cache_write(k, v, kc0, vc0, slots)
    for b, L in enumerate(lens):
        assert np.array_equal(O.gather_paged_rows(kc, table[b], L, bs), streams[b])
        assert np.array_equal(O.gather_paged_rows(vc, table[b], L, bs), streams[b][:, ::-1, :])
    untouched = np.setdiff1d(np.arange(nb * bs), slots)
    assert np.array_equal(kc[untouched], kc0[untouched])
    assert np.array_equal(vc[untouched], vc0[untouched])
    # inputs are not modified
    assert not np.array_equal(kc, kc0)


def test_write_negative_slot_is_padding():
    rng = np.random.default_rng(12)
    k = _rand_bf16(rng, (3, 1, 8))
    kc0 = _rand_bf16(rng, (6, 1, 8))
    kc, _ = O.kv_cache_write(k, k, kc0, kc0, [4, -1, 0])
    assert np.array_equal(kc[4], k[0]) and np.array_equal(kc[0], k[2])
    assert np.array_equal(kc[[1, 2, 3, 5]], kc0[[1, 2, 3, 5]])


def test_write_fp8_codes():
    rng = np.random.default_rng(13)
    k = _rand_bf16(rng, (4, 2, 8))
    kc0 = np.zeros((8, 2, 8), dtype=np.uint8)
    kc, vc = O.kv_cache_write(k, k, kc0, kc0, [7, 2, 5, 0], cache_dtype="fp8_e4m3",
                              k_inv_scale=np.float32(100.0), v_inv_scale=np.float32(0.5))
    for t, s in enumerate([7, 2, 5, 0]):
        assert np.array_equal(kc[s], O.quantize_to_e4m3(k[t], np.float32(100.0)))
        assert np.array_equal(vc[s], O.quantize_to_e4m3(k[t], np.float32(0.5)))


# ---------------------------------------------------------------------------
# attention: an independent pure-Python recomputation on tiny inputs
# ---------------------------------------------------------------------------


def _brute_attention(qrow, keys, vals, scale):
    """Direct softmax-weighted mean over a list of key/value vectors (plain Python)."""
    if not keys:
        return [0.0] * len(qrow), -math.inf
    logits = [scale * sum(a * b for a, b in zip(qrow, kk)) for kk in keys]
    mx = max(logits)
    ws = [math.exp(x - mx) for x in logits]
    z = sum(ws)
    out = [sum(w * vv[d] for w, vv in zip(ws, vals)) / z for d in range(len(qrow))]
    return out, mx + math.log(z)


def _tiny_paged_case(rng, lens, Hq, Hkv, D, bs, extra=3):
    """Per-sequence contiguous K/V streams scattered into a permuted pool."""
    nblk = [max(1, -(-n // bs)) for n in lens]
    nb = sum(nblk) + extra
    perm = rng.permutation(nb)
    table = np.full((len(lens), max(nblk) + 1), -1, dtype=np.int64)
    off = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[off:off + n]
        off += n
    kc = _rand_bf16(rng, (nb * bs, Hkv, D))
    vc = _rand_bf16(rng, (nb * bs, Hkv, D))
    ks, vs = [], []
    for b, L in enumerate(lens):
        kk = _rand_bf16(rng, (L, Hkv, D))
        vv = _rand_bf16(rng, (L, Hkv, D))
        for p in range(L):
            s = table[b][p // bs] * bs + p % bs
            kc[s] = kk[p]
            vc[s] = vv[p]
        ks.append(kk)
        vs.append(vv)
    return table, kc, vc, ks, vs


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 2), (3, 1)])
def test_decode_oracle_vs_brute_force(Hq, Hkv):
    rng = np.random.default_rng(100 + Hq * 10 + Hkv)
    D, bs = 8, 4
    lens = [1, 3, 4, 5, 9, 13]
    table, kc, vc, ks, vs = _tiny_paged_case(rng, lens, Hq, Hkv, D, bs)
    q = _rand_bf16(rng, (len(lens), Hq, D))
    scale = 0.37
    out, lse = O.paged_attn_decode(q, kc, vc, np.array(lens), table, bs, scale)
    G = Hq // Hkv
    for b, L in enumerate(lens):
        for h in range(Hq):
            keys = O.bf16_bits_to_f64(ks[b][:, h // G, :]).tolist()
            vals = O.bf16_bits_to_f64(vs[b][:, h // G, :]).tolist()
            want, wl = _brute_attention(O.bf16_bits_to_f64(q[b, h]).tolist(), keys, vals, scale)
            assert np.allclose(out[b, h], want, rtol=1e-12, atol=1e-12)
            assert abs(lse[b, h] - wl) < 1e-12


@pytest.mark.parametrize("paged", [False, True])
def test_varlen_oracle_vs_brute_force(paged):
    rng = np.random.default_rng(200 + paged)
    Hq, Hkv, D, bs = 4, 2, 8, 4
    q_lens = [3, 1, 5, 4, 2]
    k_lens = [3, 6, 5, 9, 0]
    G = Hq // Hkv
    q = _rand_bf16(rng, (sum(q_lens), Hq, D))
    cu_q = O.cu_seqlens_from_lens(q_lens)
    cu_k = O.cu_seqlens_from_lens(k_lens)
    if paged:
        table, kc, vc, ks, vs = _tiny_paged_case(rng, k_lens, Hq, Hkv, D, bs)
        out, lse = O.paged_attn_varlen(q, kc, vc, cu_q, cu_k, 0.5, True, block_table=table, block_size=bs)
    else:
        ks = [_rand_bf16(rng, (L, Hkv, D)) for L in k_lens]
        vs = [_rand_bf16(rng, (L, Hkv, D)) for L in k_lens]
        out, lse = O.paged_attn_varlen(q, np.concatenate(ks), np.concatenate(vs), cu_q, cu_k, 0.5, True)
    for b in range(len(q_lens)):
        Lq, Lk = q_lens[b], k_lens[b]
        for i in range(Lq):
            row = cu_q[b] + i
            n_vis = max(0, min(Lk, i + Lk - Lq + 1))  # bottom-right: keys 0 .. i+Lk-Lq
            for h in range(Hq):
                keys = O.bf16_bits_to_f64(ks[b][:n_vis, h // G, :]).tolist()
                vals = O.bf16_bits_to_f64(vs[b][:n_vis, h // G, :]).tolist()
                want, wl = _brute_attention(O.bf16_bits_to_f64(q[row, h]).tolist(), keys, vals, 0.5)
                assert np.allclose(out[row, h], want, rtol=1e-12, atol=1e-12)
                assert (lse[h, row] == wl) if n_vis == 0 else abs(lse[h, row] - wl) < 1e-12


# ---------------------------------------------------------------------------
# closed-form special cases and invariants
# ---------------------------------------------------------------------------


def test_single_key_returns_its_value():
    rng = np.random.default_rng(21)
    table, kc, vc, ks, vs = _tiny_paged_case(rng, [1, 1], 4, 2, 8, 4)
    q = _rand_bf16(rng, (2, 4, 8))
    out, lse = O.paged_attn_decode(q, kc, vc, np.array([1, 1]), table, 4, 0.3)
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b, h], O.bf16_bits_to_f64(vs[b][0, h // 2]))
            s = 0.3 * float(O.bf16_bits_to_f64(q[b, h]) @ O.bf16_bits_to_f64(ks[b][0, h // 2]))
            assert abs(lse[b, h] - s) < 1e-12


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(22)
    L, Hkv, D = 7, 1, 8
    k = np.repeat(_rand_bf16(rng, (1, Hkv, D)), L, axis=0)
    v = _rand_bf16(rng, (L, Hkv, D))
    q = _rand_bf16(rng, (1, 2, D))
    out, lse = O.paged_attn_varlen(q, k, v, [0, 1], [0, L], 0.9, causal=True)
    vm = O.bf16_bits_to_f64(v)[:, 0, :].mean(axis=0)
    assert np.allclose(out[0, 0], vm, atol=1e-14) and np.allclose(out[0, 1], vm, atol=1e-14)
    s = 0.9 * float(O.bf16_bits_to_f64(q[0, 0]) @ O.bf16_bits_to_f64(k[0, 0]))
    assert abs(lse[0, 0] - (s + math.log(L))) < 1e-12


def test_dominant_logit_selects_its_value():
    rng = np.random.default_rng(23)
    L, D = 6, 8
    k = np.zeros((L, 1, D), dtype=np.uint16)
    k[3, 0, 0] = _bf16_bits(np.float32(64.0))   # only key 3 aligns with q
    v = _rand_bf16(rng, (L, 1, D))
    q = np.zeros((1, 1, D), dtype=np.uint16)
    q[0, 0, 0] = _bf16_bits(np.float32(64.0))
    out, _ = O.paged_attn_varlen(q, k, v, [0, 1], [0, L], 1.0, causal=True)
    assert np.allclose(out[0, 0], O.bf16_bits_to_f64(v[3, 0]), atol=1e-300)


def test_gqa_equals_mha_with_replicated_kv_heads():
    rng = np.random.default_rng(24)
    Hq, Hkv, D = 8, 2, 8
    lens = [4, 7]
    k = _rand_bf16(rng, (sum(lens), Hkv, D))
    v = _rand_bf16(rng, (sum(lens), Hkv, D))
    q = _rand_bf16(rng, (sum(lens), Hq, D))
    cu = O.cu_seqlens_from_lens(lens)
    out_gqa, lse_gqa = O.paged_attn_varlen(q, k, v, cu, cu, 0.4)
    rep = np.repeat(k, Hq // Hkv, axis=1)      # kv head h//G becomes head h
    repv = np.repeat(v, Hq // Hkv, axis=1)
    out_mha, lse_mha = O.paged_attn_varlen(q, rep, repv, cu, cu, 0.4)
    assert np.array_equal(out_gqa, out_mha) and np.array_equal(lse_gqa, lse_mha)


def test_block_permutation_invariance_bitwise():
    rng = np.random.default_rng(25)
    lens = [5, 17, 9]
    table, kc, vc, _, _ = _tiny_paged_case(rng, lens, 4, 2, 8, 4)
    q = _rand_bf16(rng, (3, 4, 8))
    out0, lse0 = O.paged_attn_decode(q, kc, vc, np.array(lens), table, 4, 0.3)
    nb = kc.shape[0] // 4
    perm = rng.permutation(nb)               # block i moves to perm[i]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    for i in range(nb):
        kc2[perm[i] * 4:(perm[i] + 1) * 4] = kc[i * 4:(i + 1) * 4]
        vc2[perm[i] * 4:(perm[i] + 1) * 4] = vc[i * 4:(i + 1) * 4]
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    out1, lse1 = O.paged_attn_decode(q, kc2, vc2, np.array(lens), table2, 4, 0.3)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_decode_equals_varlen_with_one_query():
    rng = np.random.default_rng(26)
    lens = [3, 8, 12]
    table, kc, vc, _, _ = _tiny_paged_case(rng, lens, 4, 2, 8, 4)
    q = _rand_bf16(rng, (3, 4, 8))
    dec, dlse = O.paged_attn_decode(q, kc, vc, np.array(lens), table, 4, 0.3)
    var, vlse = O.paged_attn_varlen(q, kc, vc, [0, 1, 2, 3], O.cu_seqlens_from_lens(lens), 0.3,
                                    block_table=table, block_size=4)
    assert np.array_equal(dec, var) and np.array_equal(dlse, vlse.T)


def test_each_query_of_a_multi_query_sequence_is_a_decode_over_its_prefix():
    """Speculative verification (several new tokens per sequence): under bottom-right
    alignment, query i of a sequence with Lq queries and Lk keys is a one-query decode over
    the first i + Lk - Lq + 1 keys.  This is the identity the decode kernels rely on when
    they serve such rows one by one."""
    rng = np.random.default_rng(31)
    lk = [9, 14, 6]
    lq = [3, 4, 1]
    table, kc, vc, _, _ = _tiny_paged_case(rng, lk, 4, 2, 8, 4)
    total_q = sum(lq)
    q = _rand_bf16(rng, (total_q, 4, 8))
    var, vlse = O.paged_attn_varlen(q, kc, vc, O.cu_seqlens_from_lens(lq), O.cu_seqlens_from_lens(lk), 0.3,
                                    block_table=table, block_size=4)
    row = 0
    for b in range(len(lk)):
        for i in range(lq[b]):
            keys = i + lk[b] - lq[b] + 1
            one = np.full(len(lk), 0)
            one[b] = keys
            dec, dlse = O.paged_attn_decode(q[row:row + 1].repeat(len(lk), axis=0), kc, vc, one, table, 4, 0.3,
                                            seqs=[b])
            # same terms, summed over a masked longer row on the varlen side: fp64 rounding only
            assert np.allclose(dec[b], var[row], rtol=1e-12, atol=1e-13), (b, i)
            assert np.allclose(dlse[b], vlse[:, row], rtol=1e-12, atol=1e-13), (b, i)
            row += 1


def test_chunked_prefill_equals_whole_prefill():
    """Prefix reuse: queries of a later chunk over prefix+chunk keys = the same rows of the whole prefill."""
    rng = np.random.default_rng(27)
    L, Hq, Hkv, D = 13, 4, 2, 8
    q = _rand_bf16(rng, (L, Hq, D))
    k = _rand_bf16(rng, (L, Hkv, D))
    v = _rand_bf16(rng, (L, Hkv, D))
    whole, wlse = O.paged_attn_varlen(q, k, v, [0, L], [0, L], 0.3)
    for split in (1, 5, 12):
        part, plse = O.paged_attn_varlen(q[split:], k, v, [0, L - split], [0, L], 0.3)
        assert np.allclose(part, whole[split:], rtol=0, atol=1e-13)
        assert np.allclose(plse, wlse[:, split:], rtol=0, atol=1e-13)


def test_varlen_example_semantics_bottom_right():
    """The docs' varlen example under bottom-right alignment (a reading, see module docs).

    r0 has no keys (rows are zero); r1's first two queries see no key, its last
    sees the one key; r2's single query sees all seven keys.
    """
    rng = np.random.default_rng(28)
    g = _golden("varlen_example.json")
    q = _rand_bf16(rng, (14, 2, 8))
    k = _rand_bf16(rng, (8, 1, 8))
    v = _rand_bf16(rng, (8, 1, 8))
    out, lse = O.paged_attn_varlen(q, k, v, g["cu_seq_lens_q"], g["cu_seq_lens_k"], 0.35)
    assert np.all(out[:12] == 0) and np.all(np.isneginf(lse[:, :12]))
    assert np.array_equal(out[12, 0], O.bf16_bits_to_f64(v[0, 0]))
    kf, vf = O.bf16_bits_to_f64(k[1:, 0]), O.bf16_bits_to_f64(v[1:, 0])
    s = 0.35 * kf @ O.bf16_bits_to_f64(q[13, 1])
    w = np.exp(s - s.max())
    assert np.allclose(out[13, 1], w @ vf / w.sum(), atol=1e-14)


def test_fp8_attention_uses_dequantised_values():
    rng = np.random.default_rng(29)
    lens = [6, 3]
    table, kc, vc, _, _ = _tiny_paged_case(rng, lens, 2, 1, 8, 4)
    kq = O.quantize_to_e4m3(kc, np.float32(30.0))
    vq = O.quantize_to_e4m3(vc, np.float32(20.0))
    q = _rand_bf16(rng, (2, 2, 8))
    ks, vs = 1 / 30.0, 1 / 20.0
    out, _ = O.paged_attn_decode(q, kq, vq, np.array(lens), table, 4, 0.3, "fp8_e4m3", ks, vs)
    # same as bf16-free attention over decode(code) * scale given as explicit fp64 arrays
    kd = O.e4m3_decode(kq) * np.float64(np.float32(ks))
    vd = O.e4m3_decode(vq) * np.float64(np.float32(vs))
    for b, L in enumerate(lens):
        kr = np.stack([kd[table[b][p // 4] * 4 + p % 4] for p in range(L)])
        vr = np.stack([vd[table[b][p // 4] * 4 + p % 4] for p in range(L)])
        o, _ = O.attention_rows(O.bf16_bits_to_f64(q[b])[None], kr, vr, 0.3, True)
        assert np.array_equal(out[b], o[0])


def test_int8_attention_uses_dequantised_values():
    """INT8 cache (A18): attention runs on code * scale, each code an exact integer in [-127, 127]."""
    rng = np.random.default_rng(30)
    lens = [5, 7]
    table, kc, vc, _, _ = _tiny_paged_case(rng, lens, 2, 1, 8, 4)
    kq = O.quantize_to_int8(kc, np.float32(40.0))
    vq = O.quantize_to_int8(vc, np.float32(25.0))
    q = _rand_bf16(rng, (2, 2, 8))
    ks, vs = 1 / 40.0, 1 / 25.0
    out, _ = O.paged_attn_decode(q, kq, vq, np.array(lens), table, 4, 0.3, "int8", ks, vs)
    kd = kq.astype(np.float64) * np.float64(np.float32(ks))
    vd = vq.astype(np.float64) * np.float64(np.float32(vs))
    for b, L in enumerate(lens):
        kr = np.stack([kd[table[b][p // 4] * 4 + p % 4] for p in range(L)])
        vr = np.stack([vd[table[b][p // 4] * 4 + p % 4] for p in range(L)])
        o, _ = O.attention_rows(O.bf16_bits_to_f64(q[b])[None], kr, vr, 0.3, True)
        assert np.array_equal(out[b], o[0])


# ---------------------------------------------------------------------------
# copy-on-write of shared blocks ([CH15] "PagedAttention：メモリを「ページ」で貸し出す")
# ---------------------------------------------------------------------------


def _pool(nb, bs, hkv, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, 1 << 16, size=(nb * bs, hkv, d), dtype=np.uint64).astype(np.uint16),
            rng.integers(0, 1 << 16, size=(nb * bs, hkv, d), dtype=np.uint64).astype(np.uint16))


def test_copy_on_write_fork_keeps_the_shared_prefix():
    # sequence A holds 70 tokens in blocks [3, 0, 6] (block size 32); B forks
    # from A sharing blocks 3 and 0 and gets a private copy of the partly
    # filled block 6 in block 5 before either writes token 70
    bs = 32
    kc, vc = _pool(8, bs, 2, 16, 11)
    kc2, vc2 = O.copy_blocks(kc, vc, [[6, 5]], bs)
    for cache, new in ((kc, kc2), (vc, vc2)):
        a_rows = O.gather_paged_rows(cache, [3, 0, 6], 70, bs)
        b_rows = O.gather_paged_rows(new, [3, 0, 5], 70, bs)
        assert np.array_equal(a_rows, b_rows)
    # B's next token goes to its private block; A's rows do not change
    k_new = np.full((1, 2, 16), 0x3F80, dtype=np.uint16)
    slot_b = O.slot_of([3, 0, 5], 70, bs)
    kc3, vc3 = O.kv_cache_write(k_new, k_new, kc2, vc2, [slot_b])
    assert np.array_equal(O.gather_paged_rows(kc3, [3, 0, 6], 71, bs), O.gather_paged_rows(kc, [3, 0, 6], 71, bs))
    assert np.array_equal(O.gather_paged_rows(kc3, [3, 0, 5], 71, bs)[70], k_new[0])


def test_copy_blocks_touches_only_destinations_bitwise():
    bs = 16
    kc, vc = _pool(10, bs, 2, 8, 12)
    kc[5 * bs, 0, 0] = 0x7FC1  # a NaN payload is copied as bits
    pairs = [[5, 1], [2, 9], [7, 7]]
    kc2, vc2 = O.copy_blocks(kc, vc, pairs, bs)
    for cache, new in ((kc, kc2), (vc, vc2)):
        for blk in range(10):
            rows = slice(blk * bs, (blk + 1) * bs)
            src = {1: 5, 9: 2}.get(blk, blk)
            assert np.array_equal(new[rows], cache[src * bs:(src + 1) * bs])
    assert kc2[1 * bs, 0, 0] == 0x7FC1


def test_copy_blocks_reads_the_cache_as_before_the_call():
    bs = 4
    kc, vc = _pool(4, bs, 1, 4, 13)
    kc2, _ = O.copy_blocks(kc, vc, [[0, 1], [1, 2]], bs)
    assert np.array_equal(kc2[2 * bs:3 * bs], kc[1 * bs:2 * bs])   # old block 1, not block 0
    assert np.array_equal(kc2[1 * bs:2 * bs], kc[0:bs])
    with pytest.raises(IndexError):
        O.copy_blocks(kc, vc, [[0, 4]], bs)


# ---------------------------------------------------------------------------
# decode with the step's append ([PA] "デコードパス" example: lengths before the step)
# ---------------------------------------------------------------------------


def test_decode_with_append_on_the_worked_example():
    g = _golden("decode_example.json")
    bs, table = g["block_size"], np.array(g["block_table"])
    rng = np.random.default_rng(21)
    Hq, Hkv, D = 4, 2, 8
    nb = 8
    kc = _rand_bf16(rng, (nb * bs, Hkv, D))
    vc = _rand_bf16(rng, (nb * bs, Hkv, D))
    q = _rand_bf16(rng, (3, Hq, D))
    k_new = _rand_bf16(rng, (3, Hkv, D))
    v_new = _rand_bf16(rng, (3, Hkv, D))
    out, lse, kc2, vc2 = O.paged_attn_decode_with_kvcache(q, k_new, v_new, kc, vc, g["cache_seqlens"], table, bs,
                                                          0.25)
    # the new rows land in the slots the page's example implies; nothing else changes
    slots = g["derived_new_token_slots"]
    for b, s in enumerate(slots):
        assert np.array_equal(kc2[s], k_new[b]) and np.array_equal(vc2[s], v_new[b])
    other = np.setdiff1d(np.arange(nb * bs), slots)
    assert np.array_equal(kc2[other], kc[other]) and np.array_equal(vc2[other], vc[other])
    # each sequence attends its cached tokens followed by the new one (plain-Python recomputation)
    for b, L in enumerate(g["cache_seqlens"]):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            keys = [O.bf16_bits_to_f64(kc[O.slot_of(table[b], p, bs), kvh]).tolist() for p in range(L)]
            vals = [O.bf16_bits_to_f64(vc[O.slot_of(table[b], p, bs), kvh]).tolist() for p in range(L)]
            keys.append(O.bf16_bits_to_f64(k_new[b, kvh]).tolist())
            vals.append(O.bf16_bits_to_f64(v_new[b, kvh]).tolist())
            ref, ref_lse = _brute_attention(O.bf16_bits_to_f64(q[b, h]).tolist(), keys, vals, 0.25)
            assert np.allclose(out[b, h], ref, rtol=1e-12, atol=1e-12)
            assert math.isclose(lse[b, h], ref_lse, rel_tol=1e-12, abs_tol=1e-12)


def test_decode_with_append_on_an_empty_cache_returns_the_new_value():
    rng = np.random.default_rng(22)
    kc = _rand_bf16(rng, (4 * 16, 1, 8))
    vc = _rand_bf16(rng, (4 * 16, 1, 8))
    q = _rand_bf16(rng, (1, 2, 8))
    kn = _rand_bf16(rng, (1, 1, 8))
    vn = _rand_bf16(rng, (1, 1, 8))
    out, _, _, _ = O.paged_attn_decode_with_kvcache(q, kn, vn, kc, vc, [0], np.array([[2, -1]]), 16, 0.5)
    assert np.array_equal(out[0, 0], O.bf16_bits_to_f64(vn[0, 0]))
    assert np.array_equal(out[0, 1], O.bf16_bits_to_f64(vn[0, 0]))


# ---------------------------------------------------------------------------
# INT8 KV codes ([CH15] KV size: INT8 halves the cache; symmetric per-tensor reading)
# ---------------------------------------------------------------------------


def test_int8_quantiser_rounding_and_saturation():
    vals = np.array([0.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, 127.0, 127.5, 300.0, -300.0, 3.25, -3.75],
                    dtype=np.float32)
    # every value above is exact in bf16; ties go to the even code, 127.5 saturates
    codes = O.quantize_to_int8(_bf16_bits(vals), 1.0)
    assert codes.tolist() == [0, 0, 2, 2, 0, -2, -2, 126, 127, 127, 127, -127, 3, -4]
    inf = _bf16_bits(np.array([np.inf, -np.inf], dtype=np.float32))
    assert O.quantize_to_int8(inf, 1.0).tolist() == [127, -127]


def test_int8_codes_round_trip_and_dequantise():
    codes = np.arange(-127, 128, dtype=np.int8)
    vals = O.cache_values_f64(codes, "int8", 0.25)
    assert np.array_equal(vals, codes.astype(np.float64) * 0.25)
    # re-quantising the exact bf16 images of the values gives the codes back
    back = O.quantize_to_int8(_bf16_bits(codes.astype(np.float32)), 1.0)
    assert np.array_equal(back, codes)
    # the scale is applied by one float32 multiply before the rounding
    x = _bf16_bits(np.array([10.0], dtype=np.float32))
    assert O.quantize_to_int8(x, np.float32(1.0 / 3.0)).tolist() == [3]
