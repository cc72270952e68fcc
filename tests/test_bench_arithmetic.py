"""The roofline arithmetic bench.py reports, pinned to closed forms (no GPU).

The decode roofline counts the attended K/V rows plus Q and O; the prefill
roofline counts 4*D*Hq FLOPs per visible causal (query, key) pair.  These are
checked against the sizes the workloads are defined by and against brute force.
"""

import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _brute_pairs(lq, lk):
    # query i (0-based) of a sequence with lq queries and lk keys sees key j iff j <= i + lk - lq
    return sum(1 for i in range(lq) for j in range(lk) if j <= i + lk - lq)


@pytest.mark.parametrize("L", [1, 2, 127, 128, 129, 1000])
def test_causal_pairs_square_is_triangular(L):
    assert bench.causal_pairs([L], [L]) == L * (L + 1) // 2


@pytest.mark.parametrize("lq,lk", [(3, 10), (10, 3), (1, 7), (7, 0), (0, 5), (512, 512 + 2048)])
def test_causal_pairs_bottom_right_matches_brute_force(lq, lk):
    assert bench.causal_pairs([lq], [lk]) == _brute_pairs(lq, lk)


def test_causal_pairs_prefix_closed_form():
    # a chunk of Lq queries over a prefix of P cached keys: Lq*P + Lq(Lq+1)/2 pairs
    for lq, p in [(512, 0), (512, 2048), (512, 4096), (512, 8192)]:
        assert bench.causal_pairs([lq], [lq + p]) == lq * p + lq * (lq + 1) // 2


def test_decode_bytes_of_the_worked_example():
    # 3 sequences attending 31 + 33 + 71 = 135 positions, 2 kv heads of d64, bf16 K and V,
    # plus Q and O of 3 x 4 heads x 64 bf16
    wl = SimpleNamespace(cache_dtype="bf16", lens_before=np.array([30, 32, 70]), num_kv_heads=2, head_dim=64,
                         batch=3, num_heads=4)
    assert bench.decode_bytes(wl) == 135 * 2 * 64 * 2 * 2 + 2 * 3 * 4 * 64 * 2
    assert bench.write_bytes(wl) == 3 * 2 * 64 * (2 + 2) * 2


@pytest.mark.parametrize("dt,elt", [("bf16", 2), ("fp8_e4m3", 1), ("int8", 1)])
def test_decode_bytes_of_the_long_context_workload(dt, elt):
    # 8 sequences x (131072 + 1) positions x 8 kv heads x 128 x elt bytes, K and V
    wl = SimpleNamespace(cache_dtype=dt, lens_before=np.full(8, 131072), num_kv_heads=8, head_dim=128,
                         batch=8, num_heads=64)
    kv = 8 * 131073 * 8 * 128 * elt * 2
    assert bench.decode_bytes(wl) == kv + 2 * 8 * 64 * 128 * 2
    if dt == "bf16":
        assert abs(kv / 1e9 - 4.295) < 1e-3


def test_job_throughput_units():
    # 2.296 GB per step at 0.3529 ms is 6506 GB/s
    assert bench.job_throughput_gbs(2_295_832_576, 0.3529, 1) == pytest.approx(6505.6, rel=1e-4)
