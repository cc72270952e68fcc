"""Host-side checks of the seeded input generators against the oracle's indexing."""

import numpy as np

import oracle as O
from paged_kv_cache_200_gb300 import workloads as W


def test_decode_example_metadata():
    wl = W.decode_example()
    assert wl.block_table.tolist() == W.EXAMPLE_BLOCK_TABLE
    assert wl.cache_seqlens.tolist() == [31, 33, 71]          # attended after the write
    assert wl.slot_mapping.tolist() == [94, 32, 198]
    assert wl.k_cache.shape == (8 * 32, 2, 64) and wl.q.shape == (3, 4, 64)
    assert wl.scale == 1.0 / 8.0


def test_generated_slots_follow_block_table():
    wl = W.make_decode([5, 16, 31, 40], 8, 2, 64, 16, seed=5, extra_blocks=3)
    table = wl.block_table.numpy()
    for b, L in enumerate(wl.lens_before):
        assert wl.slot_mapping[b].item() == O.slot_of(table[b], int(L), 16)
        assert O.blocks_needed(L + 1, 16) == int((table[b] >= 0).sum())
    ids = table[table >= 0]
    assert len(np.unique(ids)) == len(ids) and ids.max() < wl.num_blocks


def test_varlen_generators():
    wl = W.varlen_prefill()
    assert np.all((wl.q_lens >= 128) & (wl.q_lens <= 2048)) and len(wl.q_lens) == 8
    assert wl.cu_seqlens_q.tolist() == O.cu_seqlens_from_lens(wl.q_lens).tolist()
    assert wl.q.shape == (int(wl.q_lens.sum()), 32, 128)
    pw = W.varlen_prefill(paged=True)
    assert np.array_equal(pw.q_lens, wl.q_lens)
    table = pw.block_table.numpy()
    cu = pw.cu_seqlens_q.numpy()
    for b in range(8):
        sl = pw.slot_mapping.numpy()[cu[b]:cu[b + 1]]
        assert sl.tolist() == [O.slot_of(table[b], p, 16) for p in range(int(pw.q_lens[b]))]


def test_mixed_chunked_shared_prefix_layout():
    wl = W.mixed_chunked(history=False)
    table = wl.block_table.numpy()
    assert wl.q_lens[:4].tolist() == [512] * 4 and np.all(wl.q_lens[4:] == 1)
    assert wl.k_lens[:4].tolist() == [512, 2048 + 512, 4096 + 512, 8192 + 512]
    assert np.all((wl.k_lens[4:] >= 513) & (wl.k_lens[4:] <= 8193))
    # the 2K-prefix chunk's prefix blocks are the 4K-prefix chunk's leading blocks
    assert np.array_equal(table[1, :128], table[2, :128])
    # every other block id appears once
    ids = np.concatenate([table[b][table[b] >= 0] for b in range(len(table)) if b != 1] + [table[1, 128:][table[1, 128:] >= 0]])
    assert len(np.unique(ids)) == len(ids) == wl.num_blocks
    # new tokens of the chunks go to private blocks
    cu = wl.cu_seqlens_q.numpy()
    shared_slots = set()
    for p in range(2048):
        shared_slots.add(O.slot_of(table[2], p, 16))
    assert not (set(wl.slot_mapping.numpy()[cu[1]:cu[2]].tolist()) & shared_slots)


def test_fp8_scales_from_absmax():
    wl = W.make_decode([20, 7], 4, 2, 64, 16, seed=9, cache_dtype="fp8_e4m3")
    assert wl.k_cache.dtype.itemsize == 1 and wl.cache_dtype == "fp8_e4m3"
    assert np.float32(wl.k_inv_scale) == np.float32(np.float32(1.0) / np.float32(wl.k_scale))
    vals = O.e4m3_decode(wl.k_cache.numpy())
    assert np.nanmax(np.abs(vals)) <= 448.0
