"""Pins for the oracle's fp8 (E4M3) KV pool: the int8 pool's layout and
per-(token, KV head) scales ("Модуль 04: KV-кэш и арифметика памяти", section
5: KV8Cache's absmax scaling; section 5.4: FP8 KV as the production default),
with E4M3 codes, scale = max|x| / 448 + 1e-8 and code = e4m3(x / scale).
Each check ties the oracle to something other than itself:

* the E4M3 codec against torch's float8_e4m3fn on every pattern, on every
  midpoint between neighbouring values (ties to even) and on random values;
* closed forms: a row whose largest magnitude is 448 has scale 1 and codes
  equal to the E4M3 rounding of the row; an all-zero row gets scale 1e-8;
* the round trip stays within half an E4M3 step of every element;
* the paged layout of codes and scales;
* decode over the fp8 pool against torch's scaled-dot-product attention on
  the test's own dequantisation of the stored codes;
* chunked prefill over the fp8 pool against causal SDPA on the same
  dequantisation, and each chunk's last row against the fp8 decode of its
  sequence, bit for bit;
* planted mistakes in mutated copies of the oracle fail this battery.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

D, BS = 128, 16
E4M3 = torch.float8_e4m3fn


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _pool(nb, hkv):
    return (np.zeros((nb, BS, hkv, D), np.uint8), np.zeros((nb, BS, hkv, D), np.uint8),
            np.zeros((nb, hkv, BS), np.float32), np.zeros((nb, hkv, BS), np.float32))


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(E4M3).to(torch.float64).numpy()


def _codec():
    codes = np.arange(256, dtype=np.uint8)
    tv = _torch_decode(codes)
    ov = np.array([oracle.e4m3_to_f64(c) for c in codes])
    ok = ~np.isnan(tv)
    assert np.array_equal(tv[ok], ov[ok]) and np.array_equal(np.isnan(tv), np.isnan(ov))
    vals = np.unique(tv[ok])
    rng = np.random.default_rng(0)
    for x in (vals, (vals[:-1] + vals[1:]) / 2, rng.uniform(-448, 448, 4000), rng.uniform(-1, 1, 4000) * 2e-3):
        x32 = x.astype(np.float32)
        want = torch.from_numpy(x32).to(E4M3).view(torch.uint8).numpy()
        got = np.array([oracle.f64_to_e4m3(float(v)) for v in x32], np.uint8)
        keep = ~((x32 == 0) & np.signbit(x32))
        assert np.array_equal(got[keep], want[keep])


def test_e4m3_codec_matches_torch_on_patterns_midpoints_and_random_values():
    _codec()


def _closed_forms():
    rng = np.random.default_rng(1)
    reps = np.unique(_torch_decode(np.arange(0, 0x7f)))           # the non-negative finite E4M3 values
    rows = rng.choice(reps, size=(3, 2, D)) * rng.choice([-1.0, 1.0], size=(3, 2, D))
    rows[..., 5] = 448.0                                            # every row reaches 448: scale 1
    k8, v8, ks, vs = _pool(4, 2)
    kb = _bits(torch.from_numpy(rows).to(torch.bfloat16))
    zero = _bits(torch.zeros((3, 2, D), dtype=torch.bfloat16))
    assert oracle.kv_cache_write_f8(k8, v8, ks, vs, kb, zero, oracle.BF16, np.array([1, 17, 40])) == 0
    for t, slot in enumerate([1, 17, 40]):
        b, o = divmod(slot, BS)
        assert np.all(ks[b, :, o] == np.float32(1.0))
        assert np.all(vs[b, :, o] == np.float32(1e-8)) and not v8[b, o].any()
        assert np.array_equal(_torch_decode(k8[b, o]), rows[t])     # representable values come back exactly


def test_closed_forms_of_the_write():
    _closed_forms()


@pytest.mark.parametrize("dtype", [oracle.F16, oracle.BF16])
def test_round_trip_within_half_an_e4m3_step(dtype):
    g = torch.Generator().manual_seed(2)
    x = (torch.randn((6, 4, D), generator=g) * torch.exp(torch.randn((6, 4, 1), generator=g) * 3))
    x = x.to(torch.float16 if dtype == oracle.F16 else torch.bfloat16)
    k8, v8, ks, vs = _pool(2, 4)
    assert oracle.kv_cache_write_f8(k8, v8, ks, vs, _bits(x), _bits(x), dtype, np.arange(6)) == 0
    xv = x.to(torch.float64).numpy()
    for t in range(6):
        b, o = divmod(t, BS)
        deq = _torch_decode(k8[b, o]) * ks[b, :, o][:, None].astype(np.float64)
        y = np.abs(xv[t]) / ks[b, :, o][:, None]                   # magnitude in code units
        step = np.where(y >= 2.0 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(y, 1e-30))) - 3), 2.0 ** -9)
        assert np.all(np.abs(deq - xv[t]) <= 0.5 * step * ks[b, :, o][:, None] * (1 + 1e-6) + 1e-12)


def _decode_vs_sdpa(hq, hkv, lens, seed):
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    pages = [-(-n // BS) for n in lens]
    nb = sum(pages) + 2
    perm = rng.permutation(nb)
    bt = np.full((len(lens), max(pages)), -1, np.int32)
    slots, i = [], 0
    for s, n in enumerate(lens):
        for p in range(pages[s]):
            bt[s, p] = perm[i]
            i += 1
        slots += [int(bt[s, j // BS]) * BS + j % BS for j in range(n)]
    k = (torch.randn((len(slots), hkv, D), generator=gen) * 2).to(torch.bfloat16)
    v = torch.randn((len(slots), hkv, D), generator=gen).to(torch.bfloat16)
    k8, v8, ks, vs = _pool(nb, hkv)
    assert oracle.kv_cache_write_f8(k8, v8, ks, vs, _bits(k), _bits(v), oracle.BF16, np.asarray(slots)) == 0
    q = torch.randn((len(lens), hq, D), generator=gen).to(torch.bfloat16)
    scale = 1.0 / np.sqrt(D)
    out = oracle.paged_attn_decode_f8(_bits(q), k8, v8, ks, vs, bt, np.asarray(lens, np.int32), scale, oracle.BF16)
    worst, t0 = 0.0, 0
    for s, n in enumerate(lens):
        idx = np.asarray(slots[t0:t0 + n])
        t0 += n
        b, o = idx // BS, idx % BS
        kd = (_torch_decode(k8[b, o]).astype(np.float32) * ks[b, :, o][..., None]).astype(np.float64)
        vd = (_torch_decode(v8[b, o]).astype(np.float32) * vs[b, :, o][..., None]).astype(np.float64)
        qq = q[s].to(torch.float64)[None, :, None, :]
        kk = torch.from_numpy(kd).permute(1, 0, 2)[None]
        vv = torch.from_numpy(vd).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(qq, kk, vv, scale=scale, enable_gqa=True)[0, :, 0].numpy()
        worst = max(worst, float(np.abs(out[s] - ref).max()))
    return worst


@pytest.mark.parametrize("hq,hkv", [(2, 2), (8, 2), (16, 8)])
def test_decode_over_fp8_pool_matches_sdpa_on_dequantised_kv(hq, hkv):
    assert _decode_vs_sdpa(hq, hkv, [1, 15, 16, 17, 70], seed=hq + hkv) < 1e-12


def _prefill_vs_sdpa(hq, hkv, chunks, seed, dtype=oracle.BF16):
    """Chunked prefill over an fp8 pool against causal SDPA on the test's own
    dequantisation (torch's E4M3 decoding times the stored scales); also
    returns whether each chunk's last row equals the fp8 decode of the same
    sequence bit for bit."""
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
    assert oracle.kv_cache_write_f8(k8, v8, ks, vs, _bits(k), _bits(v), dtype, np.asarray(flat)) == 0
    rows = sum(n for _, n in chunks)
    q = torch.randn((rows, hq, D), generator=gen).to(tdt)
    scale = 1.0 / np.sqrt(D)
    cs = np.asarray([st for st, _ in chunks], np.int32)
    cl = np.asarray([n for _, n in chunks], np.int32)
    ctx = np.asarray(lens, np.int32)
    out = oracle.paged_attn_prefill_f8(_bits(q), k8, v8, ks, vs, cs, cl, bt, ctx, scale, dtype)
    worst, r0, same = 0.0, 0, True
    for c, (st, n) in enumerate(chunks):
        idx = np.asarray(slots[c])
        b, o = idx // BS, idx % BS
        kd = (_torch_decode(k8[b, o]).astype(np.float32) * ks[b, :, o][..., None]).astype(np.float64)
        vd = (_torch_decode(v8[b, o]).astype(np.float32) * vs[b, :, o][..., None]).astype(np.float64)
        qq = q[r0:r0 + n].to(torch.float64).permute(1, 0, 2)[None]                  # [1, Hq, n, D]
        kk = torch.from_numpy(kd).permute(1, 0, 2)[None]                            # [1, Hkv, L, D]
        vv = torch.from_numpy(vd).permute(1, 0, 2)[None]
        mask = torch.from_numpy(np.arange(st + n)[None, :] <= (st + np.arange(n))[:, None])
        ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale, enable_gqa=True)
        worst = max(worst, float(np.abs(out[r0:r0 + n] - ref[0].permute(1, 0, 2).numpy()).max()))
        last = oracle.paged_attn_decode_f8(_bits(q[r0 + n - 1:r0 + n]), k8, v8, ks, vs, bt[c:c + 1], ctx[c:c + 1],
                                           scale, dtype)
        same = same and np.array_equal(last[0], out[r0 + n - 1])
        r0 += n
    return worst, same


@pytest.mark.parametrize("hq,hkv", [(2, 2), (8, 2), (16, 8)])
def test_prefill_over_fp8_pool_matches_sdpa_and_decode(hq, hkv):
    worst, same = _prefill_vs_sdpa(hq, hkv, [(0, 20), (17, 33), (100, 9)], seed=hq + 3 * hkv)
    assert worst < 1e-12 and same


# ---- planted mistakes ----------------------------------------------------------------

def _battery():
    failed = []
    for name, fn in [("codec", _codec), ("closed-forms", _closed_forms),
                     ("round-trip", lambda: test_round_trip_within_half_an_e4m3_step(oracle.F16))]:
        try:
            fn()
        except Exception:
            failed.append(name)
    try:
        if not _decode_vs_sdpa(4, 2, [1, 17, 33], seed=5) < 1e-12:
            failed.append("decode-sdpa")
    except Exception:
        failed.append("decode-sdpa(raised)")
    try:
        worst, same = _prefill_vs_sdpa(4, 2, [(0, 9), (20, 7)], seed=6)
        if not (worst < 1e-12 and same):
            failed.append("prefill-sdpa")
    except Exception:
        failed.append("prefill-sdpa(raised)")
    return failed


MUTATIONS = {
    "scale-uses-int8-range": ("        float scale = amax / 448.0f;\n", "        float scale = amax / 127.0f;\n"),
    "decoder-bias": ("    mag = ldexp((double)(8 + f), e - 10);", "    mag = ldexp((double)(8 + f), e - 11);"),
    "ties-away-from-zero": ("  double r = nearbyint(a / quantum) * quantum;", "  double r = round(a / quantum) * quantum;"),
    "int-codes-in-the-read": (
        "      const float kc = fp8 ? (float)oracle_e4m3_to_f64((uint8_t)k_cache[base + x]) : (float)k_cache[base + x];",
        "      const float kc = (float)k_cache[base + x];"),
}


def test_f8_battery_passes_on_the_real_oracle():
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_f8_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "liboracle_mut.so"))
    with oracle.use_library(lib):
        failed = _battery()
    assert failed, f"planted mistake '{name}' was not caught by any pin"
