"""Seeded synthetic inputs for the paged KV-cache path.

This module only draws inputs: sequence lengths, block pools, block tables,
the scheduler's slot mapping and cumulative lengths, and N(0,1) bf16 values.
It holds no attention arithmetic.  The one piece of quantisation here lays
down the pre-existing history of a one-byte cache (``fp8_codes_via_torch``,
``int8_codes_via_torch``) with torch's own conversions, as input preparation:
the oracle dequantises whatever codes it is given, and the rows the library
writes are checked against the oracle's own quantiser.  Both the CUDA path and
the CPU oracle receive the same tensors from here.

Lengths and block permutations come from ``numpy.random.default_rng(seed)``
(integers uniform, inclusive bounds).  Values are drawn as float32 N(0,1) by a
``torch.Generator`` seeded with ``seed`` on the requested device and rounded
to bf16, so every consumer sees identical bits.

The five workload shapes follow the source pages:

* ``decode_example``: the paged-attention docs' decode example (3 sequences,
  cache lengths 30/32/70, block size 32, the printed block table).
* ``varlen_prefill``: a Qwen3-like layer (32 q / 8 kv heads, d128), 8 sequences
  of 128..2048 tokens, written into a 16-token-block permuted pool.
* ``decode_batch``: 64 sequences, Llama-3.1-8B attention shape, cache lengths
  1024..16384, block size 16.
* ``mixed_chunked``: four 512-token prefill chunks over prefixes of
  0/2K/4K/8K tokens (the 2K prefix is the leading part of the 4K one, sharing
  its blocks) plus 60 decode sequences of 512..8192 cached tokens.
* ``long_decode``: 8 sequences of 131072 cached tokens, Llama-3.1-70B
  attention shape (64 q / 8 kv heads), block size 32, bf16 or FP8 cache.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

FP8_MAX = 448.0


def bf16_randn(shape, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) drawn in float32 and rounded (nearest-even) to bf16."""
    return torch.randn(tuple(shape), generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _as_i32(a, device) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device=device)


def per_tensor_fp8_scales(x: torch.Tensor):
    """(scale, inv_scale) as float32: scale = absmax(x) / 448, inv_scale = 1 / scale."""
    amax = np.float32(x.detach().abs().max().float().cpu().item())
    scale = np.float32(amax / np.float32(FP8_MAX))
    if scale == 0:
        scale = np.float32(1.0)
    inv = np.float32(np.float32(1.0) / scale)
    return float(scale), float(inv)


def per_tensor_int8_scales(x: torch.Tensor):
    """(scale, inv_scale) as float32: scale = absmax(x) / 127, inv_scale = 1 / scale."""
    amax = np.float32(x.detach().abs().max().float().cpu().item())
    scale = np.float32(amax / np.float32(127.0))
    if scale == 0:
        scale = np.float32(1.0)
    inv = np.float32(np.float32(1.0) / scale)
    return float(scale), float(inv)


def int8_codes_via_torch(x: torch.Tensor, inv_scale: float) -> torch.Tensor:
    """INT8 codes of ``x * inv_scale`` (torch's round half to even, clamped to +-127; input preparation only)."""
    y = x.float() * torch.tensor(inv_scale, dtype=torch.float32, device=x.device)
    return torch.round(y).clamp_(-127, 127).to(torch.int8)


def fp8_codes_via_torch(x: torch.Tensor, inv_scale: float) -> torch.Tensor:
    """E4M3 codes of ``x * inv_scale`` using torch's float8 cast (input preparation only).

    Used to lay down a pre-existing FP8 history in a cache.  The products stay
    within +-448 by construction of the scale, so the cast never overflows.
    """
    y = x.float() * torch.tensor(inv_scale, dtype=torch.float32, device=x.device)
    y = y.clamp_(-FP8_MAX, FP8_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def allocate_blocks(nblocks_per_seq, rng, extra_blocks: int = 0, shared=None):
    """Random physical block ids for each sequence (a permuted pool).

    ``nblocks_per_seq[b]`` blocks are given to sequence ``b``.  ``shared`` is a
    list of ``(dst, src, n)``: the first ``n`` blocks of ``dst`` are the first
    ``n`` blocks of ``src`` (a shared prefix); ``dst`` draws only the rest.
    Returns ``(block_table [B, max_blocks] int32 with -1 padding, num_blocks)``.
    """
    nblk = [int(n) for n in nblocks_per_seq]
    own = list(nblk)
    share_map = {}
    for dst, src, n in (shared or []):
        own[dst] -= n
        share_map[dst] = (src, n)
    pool = sum(own) + int(extra_blocks)
    perm = rng.permutation(pool)
    B = len(nblk)
    mb = max(max(nblk) if nblk else 1, 1)
    table = np.full((B, mb), -1, dtype=np.int32)
    off = 0
    rows = {}
    for b in range(B):
        rows[b] = list(perm[off:off + own[b]])
        off += own[b]
    for b in range(B):
        if b in share_map:
            src, n = share_map[b]
            ids = list(rows[src][:n]) + rows[b]
        else:
            ids = rows[b]
        table[b, :len(ids)] = ids
    return table, pool


def slots_for_positions(block_table_row, positions, block_size: int) -> np.ndarray:
    """The scheduler's slot for each position: physical block * block_size + offset."""
    pos = np.asarray(positions, dtype=np.int64)
    blk = np.asarray(block_table_row, dtype=np.int64)[pos // block_size]
    return (blk * block_size + pos % block_size).astype(np.int32)


@dataclass
class DecodeWorkload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    lens_before: np.ndarray          # cached tokens before the new one
    cache_seqlens: torch.Tensor      # int32 [B], tokens to attend (after the write)
    block_table: torch.Tensor        # int32 [B, max_blocks]
    slot_mapping: torch.Tensor       # int32 [B], where each new token goes
    q: torch.Tensor                  # bf16 [B, Hq, D]
    k_new: torch.Tensor              # bf16 [B, Hkv, D]
    v_new: torch.Tensor
    k_cache: torch.Tensor            # bf16 or uint8 (E4M3) [num_slots, Hkv, D]
    v_cache: torch.Tensor
    cache_dtype: str = "bf16"
    k_scale: float = 1.0
    v_scale: float = 1.0
    k_inv_scale: float = 1.0
    v_inv_scale: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def max_seqlen(self):
        return int(np.max(self.lens_before)) + 1 if len(self.lens_before) else 0


def make_decode(lens_before, num_heads, num_kv_heads, head_dim, block_size, seed, device="cpu",
                cache_dtype="bf16", extra_blocks=0, name="decode", block_table=None,
                slot_mapping=None, num_blocks=None, scale=None) -> DecodeWorkload:
    """A decode batch: each sequence has ``lens_before[b]`` cached tokens and gets one new one."""
    rng = np.random.default_rng(seed)
    lens_before = np.asarray(lens_before, dtype=np.int64)
    B = len(lens_before)
    total = lens_before + 1
    if block_table is None:
        nblk = [-(-int(n) // block_size) for n in total]
        table, nb = allocate_blocks(nblk, rng, extra_blocks)
    else:
        table = np.asarray(block_table, dtype=np.int32)
        nb = int(num_blocks)
    if slot_mapping is None:
        slots = np.array([slots_for_positions(table[b], [lens_before[b]], block_size)[0] for b in range(B)],
                         dtype=np.int32)
    else:
        slots = np.asarray(slot_mapping, dtype=np.int32)
    g = _generator(seed, device)
    q = bf16_randn((B, num_heads, head_dim), g, device)
    k_new = bf16_randn((B, num_kv_heads, head_dim), g, device)
    v_new = bf16_randn((B, num_kv_heads, head_dim), g, device)
    ns = nb * block_size
    k_hist = bf16_randn((ns, num_kv_heads, head_dim), g, device)
    v_hist = bf16_randn((ns, num_kv_heads, head_dim), g, device)
    wl = DecodeWorkload(
        name=name, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=block_size, num_blocks=nb,
        scale=float(scale if scale is not None else 1.0 / np.sqrt(head_dim)),
        lens_before=lens_before, cache_seqlens=_as_i32(total, device), block_table=_as_i32(table, device),
        slot_mapping=_as_i32(slots, device), q=q, k_new=k_new, v_new=v_new,
        k_cache=k_hist, v_cache=v_hist, cache_dtype="bf16")
    if cache_dtype in ("fp8_e4m3", "int8"):
        scales = per_tensor_fp8_scales if cache_dtype == "fp8_e4m3" else per_tensor_int8_scales
        codes = fp8_codes_via_torch if cache_dtype == "fp8_e4m3" else int8_codes_via_torch
        ks, kinv = scales(torch.cat([k_hist.reshape(-1), k_new.reshape(-1)]))
        vs, vinv = scales(torch.cat([v_hist.reshape(-1), v_new.reshape(-1)]))
        wl.k_cache = codes(k_hist, kinv)
        wl.v_cache = codes(v_hist, vinv)
        del k_hist, v_hist
        wl.cache_dtype = cache_dtype
        wl.k_scale, wl.k_inv_scale, wl.v_scale, wl.v_inv_scale = ks, kinv, vs, vinv
    return wl


# The paged-attention docs' decode example: block size 32, at most 4 blocks per
# sequence, 3 sequences with 30 / 32 / 70 cached tokens and this block table.
EXAMPLE_BLOCK_TABLE = [[2, -1, -1, -1], [0, 1, -1, -1], [3, 5, 6, -1]]
EXAMPLE_CACHE_SEQLENS = [30, 32, 70]
EXAMPLE_NUM_BLOCKS = 8
# Slot mapping printed with the example workload, kept as a write-only case:
# its third entry (134 = block 4, offset 6) is a block that no sequence owns.
EXAMPLE_LITERAL_SLOTS = [94, 32, 134]


def decode_example(seed=1001, device="cpu", slot_mapping=None) -> DecodeWorkload:
    """3 sequences, 4 q / 2 kv heads, d64, block size 32, 8 blocks, the docs' block table."""
    return make_decode(EXAMPLE_CACHE_SEQLENS, 4, 2, 64, 32, seed, device, name="decode_example",
                       block_table=EXAMPLE_BLOCK_TABLE, num_blocks=EXAMPLE_NUM_BLOCKS,
                       slot_mapping=slot_mapping, scale=1.0 / 8.0)


def decode_batch(seed=1003, device="cpu", batch=64, lo=1024, hi=16384) -> DecodeWorkload:
    """64 sequences, Llama-3.1-8B attention shape (32 q / 8 kv heads, d128), block size 16."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi, size=batch, endpoint=True)
    return make_decode(lens, 32, 8, 128, 16, seed + 7919, device, name="decode_batch64")


def long_decode(seed=1005, device="cpu", cache_dtype="bf16", batch=8, length=131072) -> DecodeWorkload:
    """8 sequences of 131072 cached tokens, 64 q / 8 kv heads, d128, block size 32."""
    return make_decode([length] * batch, 64, 8, 128, 32, seed, device, cache_dtype=cache_dtype,
                       name=f"long_decode_{cache_dtype}")


@dataclass
class VarlenWorkload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    q_lens: np.ndarray
    k_lens: np.ndarray
    cu_seqlens_q: torch.Tensor       # int32 [B+1]
    cu_seqlens_k: torch.Tensor       # int32 [B+1]
    q: torch.Tensor                  # bf16 [sum Lq, Hq, D]
    k: torch.Tensor                  # packed bf16 [sum Lk, Hkv, D] (packed mode) or None
    v: torch.Tensor
    # paged mode
    block_size: int = 0
    num_blocks: int = 0
    block_table: torch.Tensor = None   # int32 [B, max_blocks]
    k_cache: torch.Tensor = None       # [num_slots, Hkv, D], history already present
    v_cache: torch.Tensor = None
    k_new: torch.Tensor = None         # bf16 [sum Lq, Hkv, D], the new tokens' K/V
    v_new: torch.Tensor = None
    slot_mapping: torch.Tensor = None  # int32 [sum Lq]
    extra: dict = field(default_factory=dict)

    @property
    def batch(self):
        return len(self.q_lens)

    @property
    def max_len_q(self):
        return int(np.max(self.q_lens)) if len(self.q_lens) else 0

    @property
    def max_len_k(self):
        return int(np.max(self.k_lens)) if len(self.k_lens) else 0

    @property
    def total_q(self):
        return int(np.sum(self.q_lens))


def _prefix_sums(lens):
    out = np.zeros(len(lens) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(lens, dtype=np.int64))
    return out


def make_varlen_packed(q_lens, k_lens, num_heads, num_kv_heads, head_dim, seed, device="cpu",
                       name="varlen_packed", scale=None) -> VarlenWorkload:
    """Packed Q [sum Lq] and K/V [sum Lk] with cumulative lengths (no cache)."""
    q_lens = np.asarray(q_lens, dtype=np.int64)
    k_lens = np.asarray(k_lens, dtype=np.int64)
    g = _generator(seed, device)
    q = bf16_randn((int(q_lens.sum()), num_heads, head_dim), g, device)
    k = bf16_randn((int(k_lens.sum()), num_kv_heads, head_dim), g, device)
    v = bf16_randn((int(k_lens.sum()), num_kv_heads, head_dim), g, device)
    return VarlenWorkload(
        name=name, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        scale=float(scale if scale is not None else 1.0 / np.sqrt(head_dim)),
        q_lens=q_lens, k_lens=k_lens, cu_seqlens_q=_as_i32(_prefix_sums(q_lens), device),
        cu_seqlens_k=_as_i32(_prefix_sums(k_lens), device), q=q, k=k, v=v)


def make_varlen_paged(q_lens, prefix_lens, num_heads, num_kv_heads, head_dim, block_size, seed,
                      device="cpu", shared=None, extra_blocks=0, name="varlen_paged",
                      scale=None, history=True) -> VarlenWorkload:
    """Prefill chunks of ``q_lens`` new tokens over ``prefix_lens`` cached tokens, paged.

    The history (every slot of the pool) holds N(0,1) values; the new tokens'
    K/V are separate tensors with a slot mapping that places token ``i`` of
    sequence ``b`` at logical position ``prefix_lens[b] + i``.  Keys per
    sequence: ``prefix + q_len``.  ``shared``: ``(dst, src, nblocks)`` triples
    for shared leading prefix blocks.
    """
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    prefix_lens = np.asarray(prefix_lens, dtype=np.int64)
    k_lens = prefix_lens + q_lens
    nblk = [-(-int(n) // block_size) for n in k_lens]
    table, nb = allocate_blocks(nblk, rng, extra_blocks, shared)
    slots = np.concatenate([
        slots_for_positions(table[b], np.arange(prefix_lens[b], k_lens[b]), block_size)
        for b in range(len(q_lens))]) if len(q_lens) else np.zeros(0, np.int32)
    g = _generator(seed, device)
    T = int(q_lens.sum())
    q = bf16_randn((T, num_heads, head_dim), g, device)
    k_new = bf16_randn((T, num_kv_heads, head_dim), g, device)
    v_new = bf16_randn((T, num_kv_heads, head_dim), g, device)
    ns = nb * block_size
    if history:
        k_cache = bf16_randn((ns, num_kv_heads, head_dim), g, device)
        v_cache = bf16_randn((ns, num_kv_heads, head_dim), g, device)
    else:  # metadata only (host-side checks)
        k_cache = v_cache = None
    return VarlenWorkload(
        name=name, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        scale=float(scale if scale is not None else 1.0 / np.sqrt(head_dim)),
        q_lens=q_lens, k_lens=k_lens, cu_seqlens_q=_as_i32(_prefix_sums(q_lens), device),
        cu_seqlens_k=_as_i32(_prefix_sums(k_lens), device), q=q, k=None, v=None,
        block_size=block_size, num_blocks=nb, block_table=_as_i32(table, device),
        k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new,
        slot_mapping=_as_i32(slots, device), extra={"prefix_lens": prefix_lens})


def gather_tokens(wl: VarlenWorkload) -> int:
    """Summed key counts of the sequences with more than one query (the prefill gather bound)."""
    return int(np.sum(wl.k_lens[wl.q_lens > 1]))


def to_fp8_cache(wl: VarlenWorkload, cache_dtype: str = "fp8_e4m3") -> VarlenWorkload:
    """The same paged workload with a coded cache (FP8 E4M3, or INT8 with cache_dtype="int8"):
    per-tensor absmax/448 (absmax/127) scales over the history and the new tokens, history
    codes laid down with torch casts."""
    scales = per_tensor_fp8_scales if cache_dtype == "fp8_e4m3" else per_tensor_int8_scales
    codes = fp8_codes_via_torch if cache_dtype == "fp8_e4m3" else int8_codes_via_torch
    ks, kinv = scales(torch.cat([wl.k_cache.reshape(-1), wl.k_new.reshape(-1)]))
    vs, vinv = scales(torch.cat([wl.v_cache.reshape(-1), wl.v_new.reshape(-1)]))
    out = VarlenWorkload(**{f: getattr(wl, f) for f in wl.__dataclass_fields__})
    out.k_cache = codes(wl.k_cache, kinv)
    out.v_cache = codes(wl.v_cache, vinv)
    out.extra = dict(wl.extra, cache_dtype=cache_dtype, k_scale=ks, v_scale=vs, k_inv_scale=kinv, v_inv_scale=vinv)
    out.name = wl.name + "_" + cache_dtype
    return out


def varlen_prefill(seed=1002, device="cpu", paged=False, batch=8, lo=128, hi=2048) -> VarlenWorkload:
    """8 sequences with q_len = k_len uniform in [128, 2048]; 32 q / 8 kv heads, d128.

    Packed mode draws packed K/V; paged mode draws the same shapes as new
    tokens to be written into a 16-token-block permuted pool.
    """
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi, size=batch, endpoint=True)
    if paged:
        return make_varlen_paged(lens, np.zeros_like(lens), 32, 8, 128, 16, seed + 7919, device,
                                 name="varlen_prefill_paged")
    return make_varlen_packed(lens, lens, 32, 8, 128, seed + 7919, device, name="varlen_prefill")


def mixed_chunked(seed=1004, device="cpu", n_decode=60, history=True) -> VarlenWorkload:
    """4 chunks of 512 queries over prefixes 0/2K/4K/8K, then 60 decode rows.

    The 2K-prefix chunk's 128 prefix blocks are the first 128 blocks of the
    4K-prefix chunk (a shared leading prefix).  Decode rows have 512..8192
    cached tokens and one query each.
    """
    rng = np.random.default_rng(seed)
    dec = rng.integers(512, 8192, size=n_decode, endpoint=True)
    q_lens = np.concatenate([[512, 512, 512, 512], np.ones(n_decode, dtype=np.int64)])
    prefix = np.concatenate([[0, 2048, 4096, 8192], dec])
    shared = [(1, 2, 2048 // 16)]
    return make_varlen_paged(q_lens, prefix, 32, 8, 128, 16, seed + 7919, device, shared=shared,
                             name="mixed_chunked", history=history)
