"""Pins for the oracle's int8 KV pool ("Модуль 04: KV-кэш и арифметика памяти",
section 5, ``KV8Cache``: int8 codes with one fp32 scale per (token, KV head),
``scale = max|x| / 127 + 1e-8``, ``code = clip(rint(x / scale), -127, 127)``,
read back as ``code * scale``).  Each check ties the oracle to something other
than its own formula:

* closed forms: integer rows in [-127, 127] that reach ±127 quantise to
  themselves with scale exactly 1; an all-zero row gets scale 1e-8 and zero
  codes; a constant row maps to ±127;
* properties of round-to-nearest: every element comes back within half a scale,
  codes stay in [-127, 127];
* the paged layout: rows written to permuted slots land at their blocks,
  offsets and heads, scales at [block][head][offset];
* decode over the int8 pool against torch's scaled-dot-product attention on the
  dequantised keys and values laid out contiguously;
* the page's byte formula for an int8 cache (``cache_footprint``: one byte per
  element plus two fp32 scales per token and head);
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


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _pool(num_blocks, hkv):
    return (np.zeros((num_blocks, BS, hkv, D), np.int8), np.zeros((num_blocks, BS, hkv, D), np.int8),
            np.zeros((num_blocks, hkv, BS), np.float32), np.zeros((num_blocks, hkv, BS), np.float32))


def _write(rows_k, rows_v, slots, num_blocks, hkv, dtype=oracle.F16):
    k8, v8, ks, vs = _pool(num_blocks, hkv)
    tdt = torch.float16 if dtype == oracle.F16 else torch.bfloat16
    kb = _bits(torch.as_tensor(rows_k, dtype=torch.float32).to(tdt))
    vb = _bits(torch.as_tensor(rows_v, dtype=torch.float32).to(tdt))
    skipped = oracle.kv_cache_write_q8(k8, v8, ks, vs, kb, vb, dtype, np.asarray(slots, np.int64))
    return k8, v8, ks, vs, skipped


# ---- quantising write ------------------------------------------------------------

def test_integer_rows_reaching_127_quantise_to_themselves():
    rng = np.random.default_rng(1)
    rows = rng.integers(-127, 128, size=(5, 2, D)).astype(np.float32)
    rows[..., 7] = 127.0       # every (token, head) row reaches the top of the range
    rows[1, 0, 9] = -127.0
    k8, v8, ks, vs, skipped = _write(rows, -rows, [3, 20, 21, 40, 63], 4, 2)
    assert skipped == 0
    for t, slot in enumerate([3, 20, 21, 40, 63]):
        b, o = divmod(slot, BS)
        for h in range(2):
            # 127 / 127 = 1 exactly and 1 + 1e-8 rounds back to 1 in fp32
            assert ks[b, h, o] == np.float32(1.0) and vs[b, h, o] == np.float32(1.0)
            assert np.array_equal(k8[b, o, h].astype(np.float32), rows[t, h])
            assert np.array_equal(v8[b, o, h].astype(np.float32), -rows[t, h])


def test_zero_row_gets_the_epsilon_scale_and_zero_codes():
    k8, v8, ks, vs, _ = _write(np.zeros((1, 1, D)), np.zeros((1, 1, D)), [5], 1, 1)
    assert ks[0, 0, 5] == np.float32(1e-8) and vs[0, 0, 5] == np.float32(1e-8)
    assert not k8.any() and not v8.any()


def test_constant_row_maps_to_plus_or_minus_127():
    for c in (0.75, -3.5, 1000.0):
        k8, v8, ks, vs, _ = _write(np.full((1, 1, D), c), np.full((1, 1, D), -c), [0], 1, 1)
        assert np.all(k8[0, 0, 0] == np.sign(c) * 127) and np.all(v8[0, 0, 0] == -np.sign(c) * 127)


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_round_trip_within_half_a_scale(dtype):
    gen = torch.Generator().manual_seed(7)
    tdt = torch.float16 if dtype == oracle.F16 else torch.bfloat16
    k = (torch.randn((64, 4, D), generator=gen) * 3).to(tdt)
    v = torch.randn((64, 4, D), generator=gen).to(tdt)
    k8, v8, ks, vs = _pool(4, 4)
    oracle.kv_cache_write_q8(k8, v8, ks, vs, _bits(k), _bits(v), dtype, np.arange(64))
    for codes, scales, src in ((k8, ks, k), (v8, vs, v)):
        x = src.to(torch.float64).numpy().reshape(4, BS, 4, D)
        s = scales.astype(np.float64).transpose(0, 2, 1)[..., None]        # [block, offset, head, 1]
        err = np.abs(x - codes.astype(np.float64) * s)
        assert np.all(err <= 0.5 * s * (1 + 2 ** -20) + 1e-12)
        assert codes.min() >= -127 and codes.max() <= 127
        top = np.abs(x).argmax(axis=-1)                                   # the largest element of each row
        assert np.all(np.abs(np.take_along_axis(codes, top[..., None], -1)) == 127)


def test_paged_layout_of_codes_and_scales_and_skipped_slots():
    # distinct integer rows (which quantise to themselves, scale 1) at permuted slots
    rng = np.random.default_rng(3)
    slots = rng.permutation(6 * BS)[:10]
    rows = np.zeros((12, 2, D), np.float32)
    for t in range(12):
        rows[t] = ((np.arange(2 * D).reshape(2, D) + 11 * t) % 255) - 127
        rows[t, :, 0] = 127
    all_slots = list(slots) + [-1, 6 * BS]                                 # two out of range
    k8, v8, ks, vs, skipped = _write(rows, rows, all_slots, 6, 2)
    assert skipped == 2
    for t, slot in enumerate(slots):
        b, o = divmod(int(slot), BS)
        assert np.array_equal(k8[b, o].astype(np.float32), rows[t])
        assert np.all(ks[b, :, o] == 1.0)
    untouched = np.ones((6, BS), bool)
    for slot in slots:
        untouched[divmod(int(slot), BS)] = False
    assert not k8[untouched].any() and np.all(ks.transpose(0, 2, 1)[untouched] == 0.0)


# ---- decode over the int8 pool -----------------------------------------------------

def _decode_q8_vs_sdpa(hq, hkv, lens, seed, dtype=oracle.BF16):
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    tdt = torch.float16 if dtype == oracle.F16 else torch.bfloat16
    pages = [-(-n // BS) for n in lens]
    nb = sum(pages) + 3
    perm = rng.permutation(nb)
    bt = np.full((len(lens), max(pages)), -1, np.int32)
    slots, ks_src, vs_src, pos = [], [], [], []
    i = 0
    for s, n in enumerate(lens):
        for p in range(pages[s]):
            bt[s, p] = perm[i]
            i += 1
        for j in range(n):
            slots.append(int(bt[s, j // BS]) * BS + j % BS)
    k = (torch.randn((len(slots), hkv, D), generator=gen) * 2).to(tdt)
    v = torch.randn((len(slots), hkv, D), generator=gen).to(tdt)
    k8, v8, ks, vs = _pool(nb, hkv)
    assert oracle.kv_cache_write_q8(k8, v8, ks, vs, _bits(k), _bits(v), dtype, np.asarray(slots)) == 0
    q = torch.randn((len(lens), hq, D), generator=gen).to(tdt)
    scale = 1.0 / np.sqrt(D)
    out = oracle.paged_attn_decode_q8(_bits(q), k8, v8, ks, vs, bt, np.asarray(lens, np.int32), scale, dtype)
    worst, t0 = 0.0, 0
    for s, n in enumerate(lens):
        idx = np.asarray(slots[t0:t0 + n])
        t0 += n
        b, o = idx // BS, idx % BS
        # the test's own contiguous dequantisation of the codes the oracle stored
        kd = k8[b, o].astype(np.float32) * ks[b, :, o][..., None]
        vd = v8[b, o].astype(np.float32) * vs[b, :, o][..., None]
        qq = q[s].to(torch.float64)[None, :, None, :]                               # [1, Hq, 1, D]
        kk = torch.from_numpy(kd.astype(np.float64)).permute(1, 0, 2)[None]         # [1, Hkv, n, D]
        vv = torch.from_numpy(vd.astype(np.float64)).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(qq, kk, vv, scale=scale, enable_gqa=True)[0, :, 0].numpy()
        worst = max(worst, float(np.abs(out[s] - ref).max()))
    return worst


@pytest.mark.parametrize("hq,hkv", [(2, 2), (8, 2), (16, 8)])
def test_decode_over_int8_pool_matches_sdpa_on_dequantised_kv(hq, hkv):
    assert _decode_q8_vs_sdpa(hq, hkv, [1, 15, 16, 17, 70], seed=hq * 7 + hkv) < 1e-12


def _prefill_q8_vs_sdpa(hq, hkv, chunks, seed, dtype=oracle.BF16):
    """Chunked prefill over an int8 pool against causal SDPA on the test's own
    contiguous dequantisation; also returns whether each chunk's last row equals
    the int8 decode of the same sequence bit for bit."""
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    tdt = torch.float16 if dtype == oracle.F16 else torch.bfloat16
    lens = [st + n for st, n in chunks]
    pages = [-(-n // BS) for n in lens]
    nb = sum(pages) + 2
    perm = rng.permutation(nb)
    bt = np.full((len(lens), max(pages)), -1, np.int32)
    slots, i = [], 0
    for s, n in enumerate(lens):
        for p in range(pages[s]):
            bt[s, p] = perm[i]
            i += 1
        slots.append([int(bt[s, j // BS]) * BS + j % BS for j in range(n)])
    flat = [x for row in slots for x in row]
    k = (torch.randn((len(flat), hkv, D), generator=gen) * 2).to(tdt)
    v = torch.randn((len(flat), hkv, D), generator=gen).to(tdt)
    k8, v8, ks, vs = _pool(nb, hkv)
    assert oracle.kv_cache_write_q8(k8, v8, ks, vs, _bits(k), _bits(v), dtype, np.asarray(flat)) == 0
    rows = sum(n for _, n in chunks)
    q = torch.randn((rows, hq, D), generator=gen).to(tdt)
    scale = 1.0 / np.sqrt(D)
    cs = np.asarray([st for st, _ in chunks], np.int32)
    cl = np.asarray([n for _, n in chunks], np.int32)
    ctx = np.asarray(lens, np.int32)
    out = oracle.paged_attn_prefill_q8(_bits(q), k8, v8, ks, vs, cs, cl, bt, ctx, scale, dtype)
    worst, r0, same = 0.0, 0, True
    for c, (st, n) in enumerate(chunks):
        idx = np.asarray(slots[c])
        b, o = idx // BS, idx % BS
        kd = k8[b, o].astype(np.float32) * ks[b, :, o][..., None]
        vd = v8[b, o].astype(np.float32) * vs[b, :, o][..., None]
        qq = q[r0:r0 + n].to(torch.float64).permute(1, 0, 2)[None]                  # [1, Hq, n, D]
        kk = torch.from_numpy(kd.astype(np.float64)).permute(1, 0, 2)[None]        # [1, Hkv, L, D]
        vv = torch.from_numpy(vd.astype(np.float64)).permute(1, 0, 2)[None]
        mask = torch.from_numpy(np.arange(st + n)[None, :] <= (st + np.arange(n))[:, None])
        ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale, enable_gqa=True)
        worst = max(worst, float(np.abs(out[r0:r0 + n] - ref[0].permute(1, 0, 2).numpy()).max()))
        last = oracle.paged_attn_decode_q8(_bits(q[r0 + n - 1:r0 + n]), k8, v8, ks, vs, bt[c:c + 1], ctx[c:c + 1],
                                           scale, dtype)
        same = same and np.array_equal(last[0], out[r0 + n - 1])
        r0 += n
    return worst, same


@pytest.mark.parametrize("hq,hkv", [(2, 2), (8, 2), (16, 8)])
def test_prefill_over_int8_pool_matches_sdpa_and_decode(hq, hkv):
    worst, same = _prefill_q8_vs_sdpa(hq, hkv, [(0, 20), (17, 33), (100, 9)], seed=hq + 5 * hkv)
    assert worst < 1e-12 and same


def test_int8_cache_bytes_follow_the_pages_footprint_formula():
    # cache_footprint: kv_bytes(L, Hkv, d, cap, 1) + L * cap * Hkv * 2 * 4 (two fp32 scales per token and head)
    L, hkv, tokens = 28, 8, 512 * BS
    k8, v8, ks, vs = _pool(512, hkv)
    per_layer = k8.nbytes + v8.nbytes + ks.nbytes + vs.nbytes
    assert L * per_layer == oracle.kv_bytes(L, hkv, D, tokens, 1) + L * tokens * hkv * 2 * 4
    assert L * per_layer // tokens == 59136          # Qwen3-0.6B geometry: 57 344 B of codes + 1 792 B of scales


# ---- planted mistakes ----------------------------------------------------------------

def _battery():
    failed = []
    for name, fn in [("integer-rows", test_integer_rows_reaching_127_quantise_to_themselves),
                     ("zero-row", test_zero_row_gets_the_epsilon_scale_and_zero_codes),
                     ("round-trip", lambda: test_round_trip_within_half_a_scale(oracle.F16)),
                     ("layout", test_paged_layout_of_codes_and_scales_and_skipped_slots)]:
        try:
            fn()
        except Exception:
            failed.append(name)
    try:
        if not _decode_q8_vs_sdpa(4, 2, [1, 17, 33], seed=5) < 1e-12:
            failed.append("decode-sdpa")
    except Exception:
        failed.append("decode-sdpa(raised)")
    try:
        worst, same = _prefill_q8_vs_sdpa(4, 2, [(0, 9), (20, 12)], seed=6)
        if not (worst < 1e-12 and same):
            failed.append("prefill-sdpa")
    except Exception:
        failed.append("prefill-sdpa(raised)")
    return failed


MUTATIONS = {
    "epsilon-dropped": ("scale = scale + 1e-8f;", "scale = scale + 0.0f;"),
    "floor-not-rint": ("float c = rintf((float)widen(src[x], dtype) / scale);",
                       "float c = floorf((float)widen(src[x], dtype) / scale);"),
    "scale-token-major": ("scl[(block * num_kv_heads + h) * block_size + offset] = scale;",
                          "scl[(block * block_size + offset) * num_kv_heads + h] = scale;"),
    "read-uses-k-scale-for-v": ("const float ks = k_scale[sidx], vs = v_scale[sidx];",
                                "const float ks = k_scale[sidx], vs = k_scale[sidx];"),
    "range-divisor-128": ("float scale = amax / 127.0f;", "float scale = amax / 128.0f;"),
    "read-offset-shifted": ("const int32_t offset = j % block_size;", "const int32_t offset = (j + 1) % block_size;"),
}


def test_q8_battery_passes_on_the_real_oracle():
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_q8_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "liboracle_mut.so"))
    with oracle.use_library(lib):
        failed = _battery()
    assert failed, f"planted mistake '{name}' was not caught by any pin"
