"""Test infrastructure: the plain CPU oracle for the paged KV-cache hot path.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never calls it, and it never calls the product path.

Everything here is fp64 NumPy, written straight from the definitions on the
source pages (cited per function in ``pkv_oracle``).  No tiling, no online
softmax, no blocking: a reader can check each function against the pages.
"""

from .pkv_oracle import (  # noqa: F401
    E4M3_MAX,
    INT8_MAX,
    attention_rows,
    bf16_bits_to_f64,
    cache_values_f64,
    blocks_needed,
    copy_blocks,
    cu_seqlens_from_lens,
    e4m3_decode,
    e4m3_encode_rne_satfinite,
    gather_paged_rows,
    kv_bytes,
    kv_cache_write,
    paged_attn_decode,
    paged_attn_decode_with_kvcache,
    paged_attn_varlen,
    quantize_to_e4m3,
    quantize_to_int8,
    request_index,
    slot_of,
)
