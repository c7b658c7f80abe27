"""Helpers for the GPU parity tests: host copies, exact widening and the
element-wise tolerance check.

Tolerance: an output element passes iff |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|
(max abs error 2e-3, max rel error 1e-2, combined in allclose form because a
bf16 output alone is rounded by up to 2^-9 relative; NaN always fails).
Every check also reports the two errors separately: the max abs error over
all elements, and the max rel error over the elements with |oracle| >= 0.2
(below that the relative error of an output near zero says nothing).  An
element with |oracle| < 0.2 whose abs error exceeds 2e-3 passes only through
the relative term; such elements are counted as "flagged" and reported in the
run's summary (tests/conftest.py).
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


REL_FLOOR = 0.2

# totals over every check of the session, printed in the pytest summary
STATS = {"checks": 0, "elements": 0, "max_abs": 0.0, "max_rel": 0.0, "flagged": 0, "worst_flagged": None}


def check_close(got: torch.Tensor, ref: np.ndarray, what: str):
    """Assert the tolerance element by element; return (max abs error, max rel
    error over |ref| >= 0.2, number of flagged elements)."""
    g = f64(got)
    diff = np.abs(g - ref)
    bad = ~(diff <= ATOL + RTOL * np.abs(ref))
    if bad.any():
        idx = tuple(int(i) for i in np.argwhere(bad)[0])
        finite = diff[~np.isnan(diff)]
        worst = float(finite.max()) if finite.size else float("nan")
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside |d| <= {ATOL} + {RTOL}|ref|; "
            f"max abs {worst:.3e}; first bad at {idx}: got {float(g[idx])!r} ref {float(ref[idx])!r}")
    big = np.abs(ref) >= REL_FLOOR
    max_abs = float(diff.max(initial=0.0))
    max_rel = float((diff[big] / np.abs(ref[big])).max(initial=0.0))
    flagged = (~big) & (diff > ATOL)
    n_flag = int(flagged.sum())
    STATS["checks"] += 1
    STATS["elements"] += int(diff.size)
    STATS["max_abs"] = max(STATS["max_abs"], max_abs)
    STATS["max_rel"] = max(STATS["max_rel"], max_rel)
    if n_flag:
        STATS["flagged"] += n_flag
        worst = float(diff[flagged].max())
        if STATS["worst_flagged"] is None or worst > STATS["worst_flagged"][0]:
            STATS["worst_flagged"] = (worst, what)
    return max_abs, max_rel, n_flag


def oracle_write(case, layer: int):
    """Oracle pools after this step's KV write (uint16 bit arrays)."""
    kh, vh = bits(case.k_cache[layer]), bits(case.v_cache[layer])
    skipped = oracle.kv_cache_write(kh, vh, bits(case.k_new[layer]), bits(case.v_new[layer]),
                                    case.slot_mapping.cpu().numpy())
    assert skipped == 0
    return kh, vh
