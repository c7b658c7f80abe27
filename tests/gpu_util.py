"""Helpers for the GPU parity tests: host copies, exact widening and the
element-wise tolerance check.

Tolerance: an output element passes iff |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|
(max abs error 2e-3, max rel error 1e-2, combined in allclose form because a
bf16 output alone is rounded by up to 2^-9 relative; NaN always fails).
"""
import numpy as np
import torch

import oracle

ATOL = 2e-3
RTOL = 1e-2
ORACLE_DTYPE = {"f16": oracle.F16, "bf16": oracle.BF16}


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 host copy of an fp16/bf16 tensor's bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def check_close(got: torch.Tensor, ref: np.ndarray, what: str):
    g = f64(got)
    diff = np.abs(g - ref)
    bad = ~(diff <= ATOL + RTOL * np.abs(ref))
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside |d| <= {ATOL} + {RTOL}|ref|; "
            f"max abs {np.nanmax(diff):.3e}; first bad at {tuple(idx)}: got {g[tuple(idx)]!r} ref {ref[tuple(idx)]!r}")
    rel = diff / np.maximum(np.abs(ref), 1e-30)
    return float(diff.max(initial=0.0)), float(np.median(rel))


def oracle_write(case, layer: int):
    """Oracle pools after this step's KV write (uint16 bit arrays)."""
    kh, vh = bits(case.k_cache[layer]), bits(case.v_cache[layer])
    skipped = oracle.kv_cache_write(kh, vh, bits(case.k_new[layer]), bits(case.v_new[layer]),
                                    case.slot_mapping.cpu().numpy())
    assert skipped == 0
    return kh, vh
