"""Copy-on-write of shared blocks on the GPU against the oracle (bit-exact).

Source: "KV cache / batching / paged attention" (1s.xyz, chapter 15), section
"PagedAttention：メモリを「ページ」で貸し出す": blocks of a common prompt are
shared and copied only when one answer must write into them.
"""

import numpy as np
import pytest
import torch

import oracle as O
from _helpers import bits, built_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    return built_library()


def _pairs(rng, nb, n):
    """n (src, dst) pairs: distinct destinations, none of them a source."""
    perm = rng.permutation(nb)
    dst = perm[:n]
    src = rng.choice(perm[n:], size=n, replace=True)
    return np.stack([src, dst], axis=1).astype(np.int32)


@pytest.mark.parametrize("dtype,bs,hkv,d,n", [(torch.bfloat16, 16, 8, 128, 37), (torch.uint8, 32, 2, 64, 5),
                                              (torch.bfloat16, 64, 4, 128, 1), (torch.bfloat16, 16, 1, 64, 200)])
def test_copy_blocks_matches_oracle(pkv, dtype, bs, hkv, d, n):
    rng = np.random.default_rng(n)
    nb = 2 * n + 9
    g = torch.Generator(device="cuda").manual_seed(n)
    if dtype == torch.uint8:
        kc = torch.randint(0, 256, (nb, bs, hkv, d), generator=g, device="cuda", dtype=torch.int32).to(torch.uint8)
        vc = torch.randint(0, 256, (nb, bs, hkv, d), generator=g, device="cuda", dtype=torch.int32).to(torch.uint8)
    else:
        kc = torch.randn((nb, bs, hkv, d), generator=g, device="cuda").to(dtype)
        vc = torch.randn((nb, bs, hkv, d), generator=g, device="cuda").to(dtype)
        kc.view(torch.int16)[0, 0, 0, :4] = 0x7FC1  # a NaN payload is copied as bits
    pairs = _pairs(rng, nb, n)
    k_ref, v_ref = O.copy_blocks(bits(kc).reshape(nb * bs, hkv, d), bits(vc).reshape(nb * bs, hkv, d), pairs, bs)
    pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc).reshape(nb * bs, hkv, d), k_ref)
    assert np.array_equal(bits(vc).reshape(nb * bs, hkv, d), v_ref)


def test_copy_blocks_k_only_empty_and_bad_ids(pkv):
    nb, bs = 12, 16
    kc = torch.randn((nb, bs, 2, 64), device="cuda").to(torch.bfloat16)
    before = kc.clone()
    pkv.copy_blocks(kc, None, torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(kc, before)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pairs = np.array([[3, 7], [2, nb], [-1, 5], [4, 9]], dtype=np.int32)
    pkv.copy_blocks(kc, None, torch.from_numpy(pairs).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 2  # PKV_DEVERR_BLOCK
    k_ref, _ = O.copy_blocks(bits(before).reshape(nb * bs, 2, 64), bits(before).reshape(nb * bs, 2, 64),
                             pairs[[0, 3]], bs)
    assert np.array_equal(bits(kc).reshape(nb * bs, 2, 64), k_ref)  # the bad pairs were skipped


def test_fork_then_decode_gives_the_same_attention(pkv):
    # sequence 1 forks from sequence 0 (72 tokens, blocks of 32): it shares the
    # two full blocks and gets a copy of the partly filled third one; decode
    # over both tables then attends the same tokens
    bs, hkv, hq, d = 32, 2, 4, 64
    nb = 8
    g = torch.Generator(device="cuda").manual_seed(3)
    kc = torch.randn((nb, bs, hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn((nb, bs, hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    pkv.copy_blocks(kc, vc, torch.tensor([[6, 1]], dtype=torch.int32, device="cuda"))
    table = torch.tensor([[3, 0, 6], [3, 0, 1]], dtype=torch.int32, device="cuda")
    q = torch.randn((1, hq, d), generator=g, device="cuda").to(torch.bfloat16).repeat(2, 1, 1)
    lens = torch.tensor([72, 72], dtype=torch.int32, device="cuda")
    out = pkv.paged_attn_decode(q, kc, vc, lens, table, d ** -0.5, max_seqlen_k=72)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1])


def test_copy_blocks_full_pool(pkv):
    # the 64-sequence decode pool (16-token blocks, 8 x 128 bf16: 32 KB per block), 4096 pairs
    from paged_kv_cache_200_gb300 import workloads as W
    wl = W.decode_batch(device="cuda")
    sh = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
    kc, vc = wl.k_cache.view(sh), wl.v_cache.view(sh)
    rng = np.random.default_rng(7)
    pairs = _pairs(rng, wl.num_blocks, 4096)
    k0, v0 = kc.clone(), vc.clone()
    pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    src = torch.from_numpy(pairs[:, 0].astype(np.int64)).cuda()
    dst = torch.from_numpy(pairs[:, 1].astype(np.int64)).cuda()
    assert torch.equal(kc[dst].view(torch.int16), k0[src].view(torch.int16))
    assert torch.equal(vc[dst].view(torch.int16), v0[src].view(torch.int16))
    untouched = torch.ones(wl.num_blocks, dtype=torch.bool, device="cuda")
    untouched[dst] = False
    assert torch.equal(kc[untouched].view(torch.int16), k0[untouched].view(torch.int16))
    assert torch.equal(vc[untouched].view(torch.int16), v0[untouched].view(torch.int16))
