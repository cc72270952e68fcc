"""Test helpers: tensor <-> oracle array conversion, tolerance checks, library loading."""

import numpy as np
import torch

# bf16 attention: |err| <= 2e-2 + 2e-2*|ref|.  One-byte KV caches (FP8 E4M3, and INT8 on the
# same bound): |err| <= 6e-2, absolute only, against the oracle on the dequantised cache.
BF16_ATOL = 2e-2
BF16_RTOL = 2e-2
FP8_ATOL = 6e-2
FP8_RTOL = 0.0


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns; uint8 / int8 tensor -> numpy uint8 / int8."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.uint8, torch.int8):
        return t.numpy()
    raise TypeError(t.dtype)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def assert_close(got, ref, atol, rtol, what=""):
    """|got - ref| <= atol + rtol*|ref| element-wise (NaN in ref = not computed, skipped)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    mask = ~np.isnan(ref)
    both_inf = np.isinf(ref) & (got == ref)
    with np.errstate(invalid="ignore"):  # inf - inf where got and ref are opposite infinities: flagged below
        err = np.where(mask & ~both_inf, np.abs(got - ref), 0.0)
    bound = atol + rtol * np.abs(np.where(np.isfinite(ref), ref, 0.0))
    bad = mask & ~both_inf & ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {mask.sum()} elements out of tolerance; max err "
                             f"{err.max():.3e}; first at {idx.tolist()}: got {got[tuple(idx[0])]} ref "
                             f"{ref[tuple(idx[0])]}")
    return float(err.max()) if err.size else 0.0


def built_library():
    """Build (if stale) and load libpkv; returns the pkv binding module."""
    from paged_kv_cache_200_gb300 import build as B
    B.build()
    from paged_kv_cache_200_gb300 import pkv
    pkv.lib()
    return pkv
