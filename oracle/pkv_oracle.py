"""Plain fp64 CPU oracle for the paged KV-cache hot path (test infrastructure).

This module is test infrastructure.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline leg may call it; the CUDA library never does,
and nothing here calls the CUDA library.  It shares no code, table or helper
with the GPU path.

Sources (web pages, cited by title and section):

* [KVM]  "効率的な KV キャッシュ管理と Attention 計算" (itan.pw, "Efficient KV cache
  management and attention"), sections "Triton カーネルによる KV キャッシュ書き込み"
  (KV-cache write), "Python 層からのカーネル呼び出し" (wrapper and its stride
  checks) and "Attention モジュールの実装" (layer: write first, then varlen or
  decode attention).
* [PA]   "ページド・アテンション" (transformers docs, "Paged attention"), sections
  "Varlen パス" (cu_seq_lens indexing and its worked example) and "デコードパス"
  (block_table / cache_seqlens and its worked example).
* [CH15] "KV cache / batching / paged attention" (1s.xyz, chapter 15), sections
  "KVキャッシュはどれくらいメモリを食う？" (KV-size product), "KVを小さくするモデル側の
  工夫：MQA・GQA・MLA" (GQA), "PagedAttention：メモリを「ページ」で貸し出す"
  (non-contiguous blocks), "プレフィックスキャッシュとchunked prefill" and
  "FlashAttention：注意計算そのものを速く" (tiling gives exactly the plain result).

Readings where the pages are silent (each one is listed with its reason in the
design notes of the repository):

* A slot is a flat row of the cache viewed as ``[num_blocks*block_size, Hkv, D]``:
  ``slot = block_table[b][p // bs] * bs + p % bs``.
* A negative slot in ``slot_mapping`` marks a padding token and is not written.
* ``cache_seqlens`` counts the tokens to attend, i.e. after the new token was
  written (the layer writes first, then calls decode attention with
  ``current_lens``).
* q head ``h`` reads kv head ``h // (Hq // Hkv)``.
* Causal masking is aligned bottom-right: query ``i`` of a sequence with ``Lq``
  queries and ``Lk`` keys sees key ``j`` iff ``j <= i + Lk - Lq``.
* A query row that sees no key outputs zeros and has ``lse = -inf``.
* FP8 is OCP E4M3 (bias 7, no infinities, S.1111.111 is NaN, largest finite 448),
  quantised as ``e4m3_rne_satfinite(f32(x) * f32(inv_scale))``, dequantised as
  ``decode(code) * scale``.

Everything that is floating point is evaluated in fp64 with NumPy.  The only
fp32 step is the FP8 quantiser's single multiply, whose precision decides an
integer code and so follows the fp32 arithmetic that the format's users apply.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0  # largest finite OCP E4M3 magnitude: 1.75 * 2**8

# ---------------------------------------------------------------------------
# scalar formats
# ---------------------------------------------------------------------------


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) exactly to fp64.

    A bfloat16 is the upper half of an IEEE binary32, so placing the 16 bits at
    the top of a 32-bit word gives the same number as a float32, which fp64
    represents exactly.
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """Value of each OCP E4M3 code, in fp64 (NaN for S.1111.111).

    E4M3 has 1 sign, 4 exponent (bias 7) and 3 mantissa bits.  Exponent field 0
    holds subnormals ``M * 2**-9``; fields 1..15 hold ``(1 + M/8) * 2**(E-7)``,
    except ``E=15, M=7`` which is NaN.  There are no infinities.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (8 + m).astype(np.float64) * np.ldexp(1.0, e - 10)  # (1+M/8)*2^(E-7)
    subnormal = m.astype(np.float64) * 2.0 ** -9
    mag = np.where(e == 0, subnormal, normal)
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e4m3_encode_rne_satfinite(x) -> np.ndarray:
    """Encode float32 values as OCP E4M3 codes, round-to-nearest-even, saturating.

    Magnitudes above the largest finite value (448, and infinities) become 448
    with the input's sign; NaN becomes the NaN code.  Otherwise the value is
    rounded to the nearest representable E4M3 value, ties to the even code.

    Written from the format's definition: within the binade ``[2**e, 2**(e+1))``
    (``e >= -6``) the representable step is ``2**(e-3)``; below ``2**-6`` the
    subnormal step is ``2**-9``.  Rounding ``|x| / step`` to the nearest even
    integer and multiplying back is exact in fp64 for every float32 input.
    """
    x32 = np.asarray(x, dtype=np.float32)
    neg = np.signbit(x32)
    a = np.abs(x32.astype(np.float64))
    isnan = np.isnan(a)
    a = np.where(isnan, 0.0, a)
    a = np.minimum(a, E4M3_MAX)
    _, fe = np.frexp(a)  # a = f * 2**fe, f in [0.5, 1)
    e = np.maximum(fe - 1, -6)  # binade exponent, clamped into the subnormal range
    step = np.ldexp(1.0, e - 3)
    val = np.rint(a / step) * step  # np.rint rounds half to even
    # re-derive the fields from the rounded value (it may have moved up a binade)
    _, ve = np.frexp(val)
    ve = ve - 1
    is_sub = val < 2.0 ** -6
    mant_sub = np.rint(val / 2.0 ** -9).astype(np.int64)
    e_field = np.where(is_sub, 0, ve + 7)
    mant_norm = np.rint(val / np.ldexp(1.0, ve - 3)).astype(np.int64) - 8
    m_field = np.where(is_sub, mant_sub, mant_norm)
    code = (e_field.astype(np.int64) << 3) | m_field
    code = np.where(isnan, 0x7F, code)
    code = np.where(neg, code | 0x80, code)
    return code.astype(np.uint8)


def quantize_to_e4m3(x_bf16_bits, inv_scale) -> np.ndarray:
    """FP8 KV quantisation: ``e4m3_rne_satfinite(f32(x) * f32(inv_scale))``.

    [CH15] "KVキャッシュはどれくらいメモリを食う？" states that an FP8 cache halves the
    KV size; the pages do not fix the scheme, so the per-tensor scale reading
    above applies.  The product is one IEEE float32 multiply (round to nearest
    even), the code one rounding of that product.
    """
    x32 = (np.asarray(x_bf16_bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    prod = (x32 * np.float32(inv_scale)).astype(np.float32)
    return e4m3_encode_rne_satfinite(prod)


INT8_MAX = 127


def quantize_to_int8(x_bf16_bits, inv_scale) -> np.ndarray:
    """INT8 KV quantisation: ``clamp(round_half_even(f32(x) * f32(inv_scale)), -127, 127)``.

    [CH15] "KVキャッシュはどれくらいメモリを食う？" states that an INT8 cache, like FP8,
    halves the KV size, and fixes nothing else.  Reading: symmetric codes with a
    per-tensor scale (absmax / 127), one float32 multiply, round half to even,
    saturation at +-127 (-128 unused so that the range is symmetric).  A NaN
    input gives code 0.
    """
    x32 = (np.asarray(x_bf16_bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    prod = (x32 * np.float32(inv_scale)).astype(np.float32).astype(np.float64)
    prod = np.where(np.isnan(prod), 0.0, prod)
    return np.clip(np.rint(prod), -INT8_MAX, INT8_MAX).astype(np.int8)


def cache_values_f64(cache, cache_dtype: str, scale: float = 1.0) -> np.ndarray:
    """Values held by a cache (or K/V tensor) as fp64: bf16 bits, or E4M3 / INT8 codes * scale."""
    if cache_dtype == "bf16":
        return bf16_bits_to_f64(cache)
    if cache_dtype == "fp8_e4m3":
        return e4m3_decode(cache) * np.float64(np.float32(scale))
    if cache_dtype == "int8":
        return np.asarray(cache, dtype=np.int8).astype(np.float64) * np.float64(np.float32(scale))
    raise ValueError(f"unknown cache dtype {cache_dtype!r}")


# ---------------------------------------------------------------------------
# indexing ([PA] "Varlen パス" / "デコードパス", [KVM] KV-cache write)
# ---------------------------------------------------------------------------


def cu_seqlens_from_lens(lens) -> np.ndarray:
    """Cumulative sequence lengths ``[0, l0, l0+l1, ...]`` ([PA] "Varlen パス", example)."""
    lens = np.asarray(lens, dtype=np.int64)
    out = np.zeros(len(lens) + 1, dtype=np.int64)
    for i, n in enumerate(lens):
        out[i + 1] = out[i] + int(n)
    return out


def request_index(cu_seqlens) -> np.ndarray:
    """For each packed token, the sequence it belongs to ([PA] "Varlen パス", example).

    Token ``t`` belongs to sequence ``b`` iff ``cu[b] <= t < cu[b+1]``.
    """
    cu = [int(c) for c in cu_seqlens]
    idx = []
    for b in range(len(cu) - 1):
        idx.extend([b] * (cu[b + 1] - cu[b]))
    return np.asarray(idx, dtype=np.int64)


def blocks_needed(length: int, block_size: int) -> int:
    """Blocks a sequence of ``length`` tokens occupies ([PA] "デコードパス", example)."""
    return -(-int(length) // int(block_size))


def slot_of(block_table_row, pos: int, block_size: int) -> int:
    """Flat cache row of logical position ``pos`` of one sequence.

    Row ``b`` of ``block_table`` lists the physical blocks of sequence ``b`` in
    logical order; ``-1`` marks an unallocated entry ([PA] "デコードパス", cache
    behaviour and example).  Position ``pos`` lies in logical block
    ``pos // bs`` at offset ``pos % bs``.
    """
    blk = int(block_table_row[pos // block_size])
    if blk < 0:
        raise ValueError(f"position {pos} lies in an unallocated block")
    return blk * block_size + pos % block_size


def gather_paged_rows(cache, block_table_row, length: int, block_size: int) -> np.ndarray:
    """Rows ``0..length-1`` of one sequence, read through its block table, in logical order."""
    rows = [cache[slot_of(block_table_row, p, block_size)] for p in range(int(length))]
    if not rows:
        return np.zeros((0,) + tuple(cache.shape[1:]), dtype=cache.dtype)
    return np.stack(rows)


# ---------------------------------------------------------------------------
# KV-cache write ([KVM] "Triton カーネルによる KV キャッシュ書き込み")
# ---------------------------------------------------------------------------


def kv_cache_write(k, v, k_cache, v_cache, slot_mapping, cache_dtype: str = "bf16",
                   k_inv_scale: float = 1.0, v_inv_scale: float = 1.0):
    """Scatter each new token's K and V rows into the cache at its slot.

    ``k``, ``v``: bf16 bits ``[T, Hkv, D]``.  ``k_cache``, ``v_cache``:
    ``[num_slots, Hkv, D]`` (bf16 bits or E4M3 codes).  For every token ``t``
    in order, row ``slot_mapping[t]`` of each cache becomes token ``t``'s row
    ([KVM]: one program per token loads the ``Hkv*D`` contiguous elements and
    stores them at ``slot * Hkv*D``).  Negative slots are padding and are not
    written.  Returns new arrays; the inputs are not modified.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    T = len(slots)
    if k.shape[0] != T or v.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    for t in range(T):
        s = int(slots[t])
        if s < 0:
            continue
        if s >= kc.shape[0]:
            raise IndexError(f"slot {s} outside the cache of {kc.shape[0]} slots")
        if cache_dtype == "bf16":
            kc[s] = k[t]
            vc[s] = v[t]
        elif cache_dtype == "fp8_e4m3":
            kc[s] = quantize_to_e4m3(k[t], k_inv_scale)
            vc[s] = quantize_to_e4m3(v[t], v_inv_scale)
        elif cache_dtype == "int8":
            kc[s] = quantize_to_int8(k[t], k_inv_scale)
            vc[s] = quantize_to_int8(v[t], v_inv_scale)
        else:
            raise ValueError(cache_dtype)
    return kc, vc


def copy_blocks(k_cache, v_cache, block_pairs, block_size: int):
    """Copy-on-write of shared blocks: block ``dst`` of each cache becomes a copy of block ``src``.

    [CH15] "PagedAttention：メモリを「ページ」で貸し出す": answers generated from
    one prompt share the blocks of the common part, and a shared block is
    copied only when it has to be written.  ``k_cache``/``v_cache``:
    ``[num_slots, Hkv, D]`` (any element type; the copy is of the stored
    values, bit for bit).  ``block_pairs``: ``[n, 2]`` rows ``(src, dst)``.
    Every copy reads the caches as they were before the call.  Returns new
    arrays; the inputs are not modified.
    """
    kc0 = np.asarray(k_cache)
    vc0 = np.asarray(v_cache)
    kc = np.array(kc0, copy=True)
    vc = np.array(vc0, copy=True)
    nb = kc0.shape[0] // block_size
    for src, dst in np.asarray(block_pairs, dtype=np.int64).reshape(-1, 2):
        if not (0 <= src < nb and 0 <= dst < nb):
            raise IndexError(f"block pair ({src}, {dst}) outside the pool of {nb} blocks")
        rows_s = slice(int(src) * block_size, (int(src) + 1) * block_size)
        rows_d = slice(int(dst) * block_size, (int(dst) + 1) * block_size)
        kc[rows_d] = kc0[rows_s]
        vc[rows_d] = vc0[rows_s]
    return kc, vc


# ---------------------------------------------------------------------------
# attention (plain definition; [CH15] FlashAttention section: the tiled result
# equals ordinary attention, so the oracle is ordinary attention)
# ---------------------------------------------------------------------------


def attention_rows(q, k, v, scale: float, causal: bool):
    """Softmax attention of one sequence with GQA, in fp64.

    ``q``: ``[Lq, Hq, D]``; ``k``, ``v``: ``[Lk, Hkv, D]`` (fp64 values).
    Logit ``s_ij = scale * <q_i, k_j>``; weights ``exp(s_ij - max_j s_ij)``
    over the visible keys; output ``sum_j w_ij v_j / sum_j w_ij``;
    ``lse_i = max_j s_ij + log(sum_j w_ij)``.  With ``causal`` query ``i`` sees
    key ``j`` iff ``j <= i + Lk - Lq``.  Rows that see no key give zeros and
    ``lse = -inf``.  Returns ``(out [Lq, Hq, D], lse [Lq, Hq])``.
    """
    Lq, Hq, D = q.shape
    Lk, Hkv = k.shape[0], k.shape[1]
    if Hq % Hkv:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    group = Hq // Hkv
    out = np.zeros((Lq, Hq, D), dtype=np.float64)
    lse = np.full((Lq, Hq), -np.inf, dtype=np.float64)
    if Lq == 0 or Lk == 0:
        return out, lse
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    visible = (j <= i + (Lk - Lq)) if causal else np.ones((Lq, Lk), dtype=bool)
    has_key = visible.any(axis=1)
    for h in range(Hq):
        g = h // group
        s = scale * (q[:, h, :] @ k[:, g, :].T)
        s = np.where(visible, s, -np.inf)
        m = np.where(has_key, s.max(axis=1), 0.0)
        w = np.where(visible, np.exp(s - m[:, None]), 0.0)
        den = w.sum(axis=1)
        o = w @ v[:, g, :]
        out[has_key, h, :] = o[has_key] / den[has_key, None]
        lse[has_key, h] = m[has_key] + np.log(den[has_key])
    return out, lse


def paged_attn_decode(q, k_cache, v_cache, cache_seqlens, block_table, block_size: int,
                      scale: float, cache_dtype: str = "bf16", k_scale: float = 1.0,
                      v_scale: float = 1.0, seqs=None):
    """Decode attention: one query token per sequence over its paged cache.

    [PA] "デコードパス": each sequence has exactly one query token; its keys are
    the first ``cache_seqlens[b]`` positions, found through row ``b`` of
    ``block_table``.  [KVM] "Attention モジュールの実装" calls this with
    ``causal=True`` after writing the new token, so all ``cache_seqlens[b]``
    positions are visible.

    ``q``: bf16 bits ``[B, Hq, D]``; caches ``[num_slots, Hkv, D]``.
    ``seqs`` optionally restricts the work to some sequences (others are NaN).
    Returns ``(out [B, Hq, D], lse [B, Hq])`` in fp64.
    """
    qf = bf16_bits_to_f64(q)
    B, Hq, D = qf.shape
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    for b in (range(B) if seqs is None else seqs):
        L = int(cache_seqlens[b])
        kr = cache_values_f64(gather_paged_rows(k_cache, block_table[b], L, block_size), cache_dtype, k_scale)
        vr = cache_values_f64(gather_paged_rows(v_cache, block_table[b], L, block_size), cache_dtype, v_scale)
        o, l_ = attention_rows(qf[b][None], kr, vr, scale, causal=True)
        out[b] = o[0]
        lse[b] = l_[0]
    return out, lse


def paged_attn_decode_with_kvcache(q, k_new, v_new, k_cache, v_cache, cache_seqlens_before, block_table,
                                   block_size: int, scale: float, cache_dtype: str = "bf16", k_scale: float = 1.0,
                                   v_scale: float = 1.0, k_inv_scale: float = 1.0, v_inv_scale: float = 1.0,
                                   seqs=None):
    """Append each sequence's new token to its cache, then decode ([PA] "デコードパス"; [KVM] layer).

    The [PA] example counts cached tokens before the step: sequence ``b``'s new
    token takes position ``cache_seqlens_before[b]``, i.e. the slot its block
    table gives for that position ("fits in the held block" or "needs the next
    block").  [KVM]: the layer writes the step's K/V first and then attends.
    So: ``kv_cache_write`` at those slots, then ``paged_attn_decode`` over
    ``cache_seqlens_before + 1`` positions.  Returns ``(out, lse, k_cache, v_cache)``.
    """
    lens = np.asarray(cache_seqlens_before, dtype=np.int64)
    slots = [slot_of(block_table[b], int(lens[b]), block_size) for b in range(len(lens))]
    kc, vc = kv_cache_write(k_new, v_new, k_cache, v_cache, slots, cache_dtype, k_inv_scale, v_inv_scale)
    out, lse = paged_attn_decode(q, kc, vc, lens + 1, block_table, block_size, scale, cache_dtype, k_scale,
                                 v_scale, seqs=seqs)
    return out, lse, kc, vc


def paged_attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool = True,
                      block_table=None, block_size: int | None = None, kv_dtype: str = "bf16",
                      k_scale: float = 1.0, v_scale: float = 1.0, seqs=None):
    """Variable-length (packed) attention, causal by default, GQA.

    [PA] "Varlen パス": queries of sequence ``b`` are packed rows
    ``cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1`` of ``q``; its keys number
    ``cu_seqlens_k[b+1] - cu_seqlens_k[b]``.  Without a block table the keys
    are the packed rows ``cu_seqlens_k[b] ..`` of ``k``/``v`` ([PA] example).
    With a block table ([KVM] "Attention モジュールの実装": prefill with prefix
    sharing passes the caches and ``block_tables``) ``k``/``v`` are the caches
    and key ``j`` of sequence ``b`` is read at ``slot_of(block_table[b], j)``.

    Returns ``(out [sum Lq, Hq, D], lse [Hq, sum Lq])`` in fp64; ``seqs``
    optionally restricts the work to some sequences (other rows are NaN).
    """
    qf = bf16_bits_to_f64(q)
    T, Hq, D = qf.shape
    cu_q = [int(c) for c in cu_seqlens_q]
    cu_k = [int(c) for c in cu_seqlens_k]
    B = len(cu_q) - 1
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((Hq, T), np.nan)
    for b in (range(B) if seqs is None else seqs):
        q0, q1 = cu_q[b], cu_q[b + 1]
        Lk = cu_k[b + 1] - cu_k[b]
        if block_table is None:
            kr = k[cu_k[b]:cu_k[b + 1]]
            vr = v[cu_k[b]:cu_k[b + 1]]
        else:
            kr = gather_paged_rows(k, block_table[b], Lk, block_size)
            vr = gather_paged_rows(v, block_table[b], Lk, block_size)
        kf = cache_values_f64(kr, kv_dtype, k_scale)
        vf = cache_values_f64(vr, kv_dtype, v_scale)
        o, l_ = attention_rows(qf[q0:q1], kf, vf, scale, causal)
        out[q0:q1] = o
        lse[:, q0:q1] = l_.T
    return out, lse


# ---------------------------------------------------------------------------
# KV size ([CH15] "KVキャッシュはどれくらいメモリを食う？")
# ---------------------------------------------------------------------------


def kv_bytes(layers: int, kv_heads: int, head_dim: int, tokens: int, requests: int,
             bytes_per_elt: int) -> int:
    """KV-cache bytes: 2 (K and V) x layers x KV heads x head dim x tokens x requests x bytes."""
    return 2 * layers * kv_heads * head_dim * tokens * requests * bytes_per_elt
