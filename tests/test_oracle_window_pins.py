"""Pins for the oracle's sliding window ("Модуль 04: KV-кэш и арифметика
памяти", section 4: a ring buffer of capacity W keeps the last W tokens and the
mask stays on absolute positions; section 5.2: window attention).  A query at
position p sees keys max(0, p - W + 1) .. p.  Each check ties the oracle to
something other than itself:

* special cases: a window at least as long as the context is plain attention;
  a window of one key returns the query token's own value;
* the page's ring example: capacity 8 after 12 writes holds positions 4..11, so
  with equal keys the output is the mean of those rows;
* torch's scaled-dot-product attention with an explicit band mask on a
  contiguous copy, for decode and for chunked prefill;
* blocks wholly before the window may be freed (-1) or hold NaN: nothing
  changes;
* planted mistakes: mutated copies of the oracle must fail this battery.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

D = 128
BS = 16


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _case(lens, hkv, seed, nan_old=0, dtype=torch.bfloat16):
    """Per-sequence contiguous K/V scattered page by page into a NaN pool at
    permuted blocks; returns pool bits, tables and the contiguous copies."""
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    pages = [-(-n // BS) for n in lens]
    nb = sum(pages) + 2
    perm = list(rng.permutation(nb))
    kpool = torch.full((nb, BS, hkv, D), float("nan"), dtype=dtype)
    vpool = torch.full((nb, BS, hkv, D), float("nan"), dtype=dtype)
    bt = np.full((len(lens), max(pages)), -1, np.int32)
    seqs = []
    for s, n in enumerate(lens):
        k = torch.randn((n, hkv, D), generator=gen).to(dtype)
        v = torch.randn((n, hkv, D), generator=gen).to(dtype)
        seqs.append((k, v))
        for p in range(pages[s]):
            b = perm.pop()
            rows = slice(p * BS, min(n, (p + 1) * BS))
            kpool[b, :rows.stop - rows.start] = k[rows]
            vpool[b, :rows.stop - rows.start] = v[rows]
            bt[s, p] = b
    return kpool, vpool, bt, seqs


def _band_sdpa(q, k, v, scale, qpos, window):
    """q [Lq, Hq, D] at positions qpos, k/v [Lk, Hkv, D] at positions 0..Lk-1."""
    lk = k.shape[0]
    kpos = np.arange(lk)
    mask = (kpos[None, :] <= qpos[:, None]) & (kpos[None, :] > qpos[:, None] - window)
    qq = q.to(torch.float64).permute(1, 0, 2)[None]
    kk = k.to(torch.float64).permute(1, 0, 2)[None]
    vv = v.to(torch.float64).permute(1, 0, 2)[None]
    out = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=torch.from_numpy(mask)[None, None], scale=scale,
                                         enable_gqa=True)
    return out[0].permute(1, 0, 2).numpy()


def _decode_vs_band(hq, hkv, lens, window, seed):
    kpool, vpool, bt, seqs = _case(lens, hkv, seed)
    gen = torch.Generator().manual_seed(seed + 1)
    q = torch.randn((len(lens), hq, D), generator=gen).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(D)
    out = oracle.paged_attn_decode_window(_bits(q), _bits(kpool), _bits(vpool), bt, np.asarray(lens, np.int32),
                                          scale, window, oracle.BF16)
    worst = 0.0
    for s, (k, v) in enumerate(seqs):
        ref = _band_sdpa(q[s:s + 1], k, v, scale, np.asarray([lens[s] - 1]), window)[0]
        worst = max(worst, float(np.abs(out[s] - ref).max()))
    return worst


@pytest.mark.parametrize("window", [1, 5, 16, 17, 100, 1000])
def test_decode_window_matches_band_masked_sdpa(window):
    assert _decode_vs_band(8, 2, [1, 15, 16, 17, 40, 300], window, seed=window) < 1e-12


def _prefill_vs_band(hq, hkv, chunks, window, seed):
    lens = [s + n for s, n in chunks]
    kpool, vpool, bt, seqs = _case(lens, hkv, seed)
    gen = torch.Generator().manual_seed(seed + 2)
    rows = sum(n for _, n in chunks)
    q = torch.randn((rows, hq, D), generator=gen).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(D)
    cs = np.asarray([s for s, _ in chunks], np.int32)
    cl = np.asarray([n for _, n in chunks], np.int32)
    out = oracle.paged_attn_prefill_window(_bits(q), _bits(kpool), _bits(vpool), cs, cl, bt,
                                           np.asarray(lens, np.int32), scale, window, oracle.BF16)
    worst, r0 = 0.0, 0
    for c, (start, n) in enumerate(chunks):
        k, v = seqs[c]
        ref = _band_sdpa(q[r0:r0 + n], k, v, scale, start + np.arange(n), window)
        worst = max(worst, float(np.abs(out[r0:r0 + n] - ref).max()))
        r0 += n
    return worst


@pytest.mark.parametrize("window", [1, 7, 64, 200])
def test_prefill_window_matches_band_masked_sdpa(window):
    assert _prefill_vs_band(4, 2, [(0, 40), (50, 30), (300, 17)], window, seed=window + 3) < 1e-12


def test_window_as_long_as_the_context_is_plain_attention():
    lens = [17, 100, 250]
    kpool, vpool, bt, _ = _case(lens, 2, seed=9)
    q = torch.randn((3, 8, D), generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    args = (_bits(q), _bits(kpool), _bits(vpool), bt, np.asarray(lens, np.int32), 0.088)
    full = oracle.paged_attn_decode(*args, oracle.BF16)
    assert np.array_equal(oracle.paged_attn_decode_window(*args, 250, oracle.BF16), full)
    assert np.array_equal(oracle.paged_attn_decode_window(*args, 10 ** 6, oracle.BF16), full)


def test_window_of_one_returns_the_token_value():
    lens = [1, 33, 64]
    kpool, vpool, bt, seqs = _case(lens, 2, seed=4)
    q = torch.randn((3, 4, D), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    out = oracle.paged_attn_decode_window(_bits(q), _bits(kpool), _bits(vpool), bt, np.asarray(lens, np.int32),
                                          0.088, 1, oracle.BF16)
    for s, (_, v) in enumerate(seqs):
        last = v[-1].to(torch.float64).numpy()                     # [Hkv, D]
        assert np.array_equal(out[s], np.repeat(last, 2, axis=0))   # 2 query heads per KV head


def test_ring_example_of_the_page_positions_4_to_11():
    # capacity 8, 12 tokens written: the last 8 positions 4..11 are visible; with
    # equal keys every visible value weighs the same, and value row j is j
    n, window = 12, 8
    kpool = torch.zeros((1, BS, 1, D), dtype=torch.bfloat16)
    vpool = torch.zeros((1, BS, 1, D), dtype=torch.bfloat16)
    for j in range(n):
        vpool[0, j] = float(j)
    bt = np.zeros((1, 1), np.int32)
    q = torch.ones((1, 1, D), dtype=torch.bfloat16)
    out = oracle.paged_attn_decode_window(_bits(q), _bits(kpool), _bits(vpool), bt, np.asarray([n], np.int32),
                                          0.088, window, oracle.BF16)
    assert np.allclose(out, np.mean(np.arange(4, 12)), rtol=0, atol=1e-12)


def test_blocks_before_the_window_are_never_read():
    lens = [200, 90]
    kpool, vpool, bt, _ = _case(lens, 2, seed=12)
    q = torch.randn((2, 4, D), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    window = 40
    args = lambda table: (_bits(q), _bits(kpool), _bits(vpool), table, np.asarray(lens, np.int32), 0.088, window,
                          oracle.BF16)
    ref = oracle.paged_attn_decode_window(*args(bt))
    freed = bt.copy()
    for s, n in enumerate(lens):
        first_page = max(0, n - window) // BS
        for p in range(first_page):
            kpool[bt[s, p]] = float("nan")       # stale data in the freed blocks
            freed[s, p] = -1                     # and the table no longer points at them
    assert np.array_equal(oracle.paged_attn_decode_window(*args(freed)), ref)


# ---- planted mistakes ----------------------------------------------------------------

def _battery():
    failed = []
    for name, fn in [("one-key", test_window_of_one_returns_the_token_value),
                     ("ring", test_ring_example_of_the_page_positions_4_to_11),
                     ("never-read", test_blocks_before_the_window_are_never_read)]:
        try:
            fn()
        except Exception:
            failed.append(name)
    try:
        if not _decode_vs_band(4, 2, [17, 40], 16, seed=8) < 1e-12:
            failed.append("decode-band")
        if not _prefill_vs_band(4, 2, [(0, 20), (30, 9)], 7, seed=9) < 1e-12:
            failed.append("prefill-band")
    except Exception:
        failed.append("band(raised)")
    return failed


MUTATIONS = {
    "window-one-too-wide": ("const int32_t lo = (P->window > 0 && p - P->window + 1 > 0) ? p - P->window + 1 : 0;",
                            "const int32_t lo = (P->window > 0 && p - P->window > 0) ? p - P->window : 0;"),
    "gather-ignores-window": ("const int32_t glo = (P->window > 0 && pos0 - P->window + 1 > 0) ? pos0 - P->window + 1 : 0;",
                              "const int32_t glo = 0;"),
}


def test_window_battery_passes_on_the_real_oracle():
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_window_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "liboracle_mut.so"))
    with oracle.use_library(lib):
        failed = _battery()
    assert failed, f"planted mistake '{name}' was not caught by any pin"
