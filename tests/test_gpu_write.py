"""KV-cache write on the GPU vs the oracle: bit-exact, whole caches compared."""

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_200_gb300 import workloads as W
from _helpers import bits, built_library

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    return built_library()


def _run_write(pkv, k, v, kc, vc, slots, **kw):
    kc2, vc2 = kc.clone(), vc.clone()
    pkv.kv_cache_write(k, v, kc2, vc2, slots, **kw)
    torch.cuda.synchronize()
    return kc2, vc2


def test_decode_example_write_derived_slots(pkv):
    wl = W.decode_example(device="cuda")
    kc, vc = _run_write(pkv, wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    rk, rv = O.kv_cache_write(bits(wl.k_new), bits(wl.v_new), bits(wl.k_cache), bits(wl.v_cache),
                              wl.slot_mapping.cpu().numpy())
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)


def test_decode_example_write_literal_slots(pkv):
    """The literal slot list printed with the workload ([94, 32, 134]), write only."""
    wl = W.decode_example(device="cuda", slot_mapping=W.EXAMPLE_LITERAL_SLOTS)
    kc, vc = _run_write(pkv, wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    rk, rv = O.kv_cache_write(bits(wl.k_new), bits(wl.v_new), bits(wl.k_cache), bits(wl.v_cache),
                              np.array(W.EXAMPLE_LITERAL_SLOTS))
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)


@pytest.mark.parametrize("Hkv,D", [(1, 64), (2, 64), (8, 128), (4, 128), (1, 8)])
def test_write_random_slots_with_padding(pkv, Hkv, D):
    g = torch.Generator(device="cuda").manual_seed(Hkv * 1000 + D)
    T, NS = 777, 1500
    k = torch.randn(T, Hkv, D, device="cuda", generator=g).bfloat16()
    v = torch.randn(T, Hkv, D, device="cuda", generator=g).bfloat16()
    kc = torch.randn(NS, Hkv, D, device="cuda", generator=g).bfloat16()
    vc = torch.randn(NS, Hkv, D, device="cuda", generator=g).bfloat16()
    rng = np.random.default_rng(D)
    slots = rng.permutation(NS)[:T].astype(np.int32)
    slots[rng.random(T) < 0.1] = -1
    s_t = torch.from_numpy(slots).cuda()
    k2, v2 = _run_write(pkv, k, v, kc, vc, s_t)
    rk, rv = O.kv_cache_write(bits(k), bits(v), bits(kc), bits(vc), slots)
    assert np.array_equal(bits(k2), rk) and np.array_equal(bits(v2), rv)


def test_write_from_fused_qkv_views(pkv):
    """K and V as strided views of a fused [T, (Hq+2Hkv)*D] projection output."""
    T, Hq, Hkv, D = 333, 32, 8, 128
    g = torch.Generator(device="cuda").manual_seed(5)
    qkv = torch.randn(T, (Hq + 2 * Hkv) * D, device="cuda", generator=g).bfloat16()
    k = qkv[:, Hq * D:(Hq + Hkv) * D].view(T, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].view(T, Hkv, D)
    assert k.stride(0) == (Hq + 2 * Hkv) * D
    NS = 400
    kc = torch.zeros(NS, Hkv, D, device="cuda", dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    slots = np.random.default_rng(1).permutation(NS)[:T].astype(np.int32)
    k2, v2 = _run_write(pkv, k, v, kc, vc, torch.from_numpy(slots).cuda())
    rk, rv = O.kv_cache_write(bits(k), bits(v), bits(kc), bits(vc), slots)
    assert np.array_equal(bits(k2), rk) and np.array_equal(bits(v2), rv)


@pytest.mark.parametrize("inv", [1.0, 37.25, 81.4, 1000.0])
def test_write_fp8_bit_exact(pkv, inv):
    T, Hkv, D, NS = 500, 8, 128, 640
    g = torch.Generator(device="cuda").manual_seed(int(inv))
    k = (torch.randn(T, Hkv, D, device="cuda", generator=g) * 3).bfloat16()
    v = torch.randn(T, Hkv, D, device="cuda", generator=g).bfloat16()
    kc = torch.randint(0, 255, (NS, Hkv, D), device="cuda", dtype=torch.uint8, generator=g)
    vc = kc.clone()
    slots = np.random.default_rng(2).permutation(NS)[:T].astype(np.int32)
    k_inv, v_inv = np.float32(inv), np.float32(inv / 3)
    k2, v2 = _run_write(pkv, k, v, kc, vc, torch.from_numpy(slots).cuda(), k_inv_scale=float(k_inv),
                        v_inv_scale=float(v_inv))
    rk, rv = O.kv_cache_write(bits(k), bits(v), bits(kc), bits(vc), slots, cache_dtype="fp8_e4m3",
                              k_inv_scale=k_inv, v_inv_scale=v_inv)
    assert np.array_equal(bits(k2), rk) and np.array_equal(bits(v2), rv)


def test_write_fp8_special_values(pkv):
    """Saturation, ties and subnormals go through the hardware conversion exactly as the oracle."""
    vals = np.array([0.0, -0.0, 1.0, 448.0, 464.0, 1e5, -1e5, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10,
                     1.0625, 1.1875, 240.0, -240.0, 0.3, -17.0] * 8, dtype=np.float32)
    x = torch.from_numpy(vals).bfloat16().cuda().view(16, 1, 8)
    kc = torch.zeros(16, 1, 8, dtype=torch.uint8, device="cuda")
    slots = torch.arange(16, dtype=torch.int32, device="cuda")
    k2, _ = _run_write(pkv, x, x, kc, kc, slots, k_inv_scale=1.0, v_inv_scale=1.0)
    rk, _ = O.kv_cache_write(bits(x), bits(x), bits(kc), bits(kc), np.arange(16), cache_dtype="fp8_e4m3",
                             k_inv_scale=np.float32(1.0), v_inv_scale=np.float32(1.0))
    assert np.array_equal(bits(k2), rk)


def test_write_out_of_range_slot_is_flagged_and_skipped(pkv):
    T, Hkv, D, NS = 4, 2, 64, 10
    k = torch.ones(T, Hkv, D, device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros(NS, Hkv, D, device="cuda", dtype=torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.tensor([1, 10, 3, 1 << 30], dtype=torch.int32, device="cuda")
    k2, _ = _run_write(pkv, k, k, kc, kc, slots, err_flag=err)
    assert int(err.item()) & pkv.DEVERR_SLOT
    got = bits(k2)
    assert np.all(got[[0, 2, 4, 5, 6, 7, 8, 9]] == 0) and np.all(got[[1, 3]] == bits(k)[0])


def test_varlen_prefill_write_full_size(pkv):
    """The prefill workload's ~8.7K tokens into a 16-token-block permuted pool."""
    wl = W.varlen_prefill(device="cuda", paged=True)
    kc, vc = _run_write(pkv, wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, wl.slot_mapping)
    slots = wl.slot_mapping.cpu().numpy()
    # oracle on the written rows + untouched rows unchanged
    rk, rv = O.kv_cache_write(bits(wl.k_new), bits(wl.v_new), bits(wl.k_cache), bits(wl.v_cache), slots)
    assert np.array_equal(bits(kc), rk) and np.array_equal(bits(vc), rv)


def test_zero_tokens_is_a_noop(pkv):
    k = torch.empty(0, 2, 64, device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros(8, 2, 64, device="cuda", dtype=torch.bfloat16)
    pkv.kv_cache_write(k, k, kc, kc, torch.empty(0, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(kc).item() == 0


@pytest.mark.parametrize("inv", [1.0, 21.5, 1000.0])
def test_write_int8_bit_exact(pkv, inv):
    T, Hkv, D, NS = 500, 8, 128, 640
    g = torch.Generator(device="cuda").manual_seed(int(inv) + 5)
    k = (torch.randn(T, Hkv, D, device="cuda", generator=g) * 3).bfloat16()
    v = torch.randn(T, Hkv, D, device="cuda", generator=g).bfloat16()
    kc = torch.randint(-127, 128, (NS, Hkv, D), device="cuda", dtype=torch.int8, generator=g)
    vc = kc.clone()
    slots = np.random.default_rng(3).permutation(NS)[:T].astype(np.int32)
    k_inv, v_inv = np.float32(inv), np.float32(inv / 3)
    k2, v2 = _run_write(pkv, k, v, kc, vc, torch.from_numpy(slots).cuda(), k_inv_scale=float(k_inv),
                        v_inv_scale=float(v_inv))
    rk, rv = O.kv_cache_write(bits(k), bits(v), bits(kc), bits(vc), slots, cache_dtype="int8",
                              k_inv_scale=k_inv, v_inv_scale=v_inv)
    assert np.array_equal(bits(k2), rk) and np.array_equal(bits(v2), rv)


def test_write_int8_special_values(pkv):
    """Ties to even, saturation at +-127 and infinities, as the oracle."""
    vals = np.array([0.0, -0.0, 0.5, 1.5, 2.5, -2.5, 126.5, 127.5, 300.0, -300.0, np.inf, -np.inf, 3.25, -3.75,
                     64.0, -1.0] * 8, dtype=np.float32)
    x = torch.from_numpy(vals).bfloat16().cuda().view(16, 1, 8)
    kc = torch.zeros(16, 1, 8, dtype=torch.int8, device="cuda")
    slots = torch.arange(16, dtype=torch.int32, device="cuda")
    k2, _ = _run_write(pkv, x, x, kc, kc, slots, k_inv_scale=1.0, v_inv_scale=1.0)
    rk, _ = O.kv_cache_write(bits(x), bits(x), bits(kc), bits(kc), np.arange(16), cache_dtype="int8",
                             k_inv_scale=np.float32(1.0), v_inv_scale=np.float32(1.0))
    assert np.array_equal(bits(k2), rk)
