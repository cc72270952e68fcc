"""The Python binding fails loudly instead of falling back to the CPU (no GPU needed).

Every entry point refuses host tensors before calling the library, and a
missing library file is an error, not a silent substitute.
"""

import os

import pytest
import torch

from paged_kv_cache_200_gb300 import pkv


def _cpu_case():
    B, Hq, Hkv, D, bs, nb = 2, 4, 2, 64, 16, 4
    return dict(
        q=torch.zeros(B, Hq, D, dtype=torch.bfloat16),
        k_new=torch.zeros(B, Hkv, D, dtype=torch.bfloat16),
        v_new=torch.zeros(B, Hkv, D, dtype=torch.bfloat16),
        k_cache=torch.zeros(nb, bs, Hkv, D, dtype=torch.bfloat16),
        v_cache=torch.zeros(nb, bs, Hkv, D, dtype=torch.bfloat16),
        lens=torch.tensor([5, 7], dtype=torch.int32),
        table=torch.tensor([[0, -1], [1, -1]], dtype=torch.int32),
        slots=torch.tensor([4, 16 + 6], dtype=torch.int32),
        cu=torch.tensor([0, 1, 2], dtype=torch.int32),
        pairs=torch.tensor([[0, 2]], dtype=torch.int32),
    )


@pytest.mark.parametrize("call", ["write", "decode", "decode_with_kvcache", "decode_noalloc", "varlen", "copy"])
def test_host_tensors_are_refused(call):
    c = _cpu_case()
    with pytest.raises(ValueError, match="CUDA"):
        if call == "write":
            pkv.kv_cache_write(c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], c["slots"])
        elif call == "decode":
            pkv.paged_attn_decode(c["q"], c["k_cache"], c["v_cache"], c["lens"], c["table"], 0.125, max_seqlen_k=8)
        elif call == "decode_with_kvcache":
            pkv.paged_attn_decode_with_kvcache(c["q"], c["k_new"], c["v_new"], c["k_cache"], c["v_cache"], c["lens"],
                                               c["table"], 0.125, max_seqlen_k=8)
        elif call == "decode_noalloc":
            pkv.paged_attn_decode_noalloc(c["q"], c["k_cache"], c["v_cache"], c["lens"], c["table"], 0.125,
                                          max_seqlen_k=8)
        elif call == "varlen":
            pkv.paged_attn_varlen(c["q"].view(-1, 2, 64)[:2], c["k_cache"], c["v_cache"], c["cu"], c["cu"], 1, 8,
                                  block_table=c["table"], scale=0.125)
        else:
            pkv.copy_blocks(c["k_cache"], c["v_cache"], c["pairs"])


def test_missing_library_is_an_error(tmp_path):
    saved = pkv._lib
    try:
        pkv._lib = None
        with pytest.raises(RuntimeError, match="missing"):
            pkv.lib(os.path.join(str(tmp_path), "libpkv.so"))
    finally:
        pkv._lib = saved
