"""Pins for the fp64 oracle: each check ties it to something other than itself.

* the 16-bit decoders against numpy's / torch's own conversions, on every pattern;
* the paged store against the worked examples of "Модуль 12: Финальный проект:
  мини-движок инференса", task 12.1 ("Вход и выход") and the layout in the
  qwen_serve/paged.py docstring;
* decode and chunked-prefill attention against torch's
  ``scaled_dot_product_attention`` (fp64, ``enable_gqa``) on a contiguous copy
  of K/V that the test scatters into pages by whole-block copies;
* closed-form special cases (one key, zero query, equal keys, constant V per
  KV head, one dominant key);
* invariants the pages state: pages may sit anywhere, shared prefix pages are
  stored once, chunked prefill equals unchunked, decode equals the last row of
  a causal prefill;
* the KV byte counts the pages print (tests/golden/kv_closed_forms.txt);
* planted mistakes: mutated copies of the oracle must fail the battery.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D = 128
BS = 16
DT = {"f16": (torch.float16, oracle.F16), "bf16": (torch.bfloat16, oracle.BF16)}


# ---- helpers (test-side; none of them computes attention) ---------------------

def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _paged_from_contiguous(seqs, num_blocks, hkv, dtype, rng, shared_pages=0):
    """Scatter per-sequence contiguous K/V [n, Hkv, D] into a NaN-filled pool by
    whole 16-row page copies at randomly permuted block ids.  Sequences may
    share their first ``shared_pages`` pages (taken from sequence 0)."""
    tdt = DT[dtype][0]
    kpool = torch.full((num_blocks, BS, hkv, D), float("nan"), dtype=tdt)
    vpool = torch.full((num_blocks, BS, hkv, D), float("nan"), dtype=tdt)
    perm = list(rng.permutation(num_blocks))
    width = max(-(-k.shape[0] // BS) for k, _ in seqs)
    bt = np.full((len(seqs), width), -1, np.int32)
    shared_ids = []
    for s, (k, v) in enumerate(seqs):
        n = k.shape[0]
        pages = -(-n // BS)
        kp = torch.full((pages * BS, hkv, D), float("nan"), dtype=tdt)
        vp = torch.full((pages * BS, hkv, D), float("nan"), dtype=tdt)
        kp[:n], vp[:n] = k, v
        kp, vp = kp.view(pages, BS, hkv, D), vp.view(pages, BS, hkv, D)
        for p in range(pages):
            if p < shared_pages and s > 0:
                bt[s, p] = shared_ids[p]
                continue
            b = perm.pop()
            kpool[b], vpool[b] = kp[p], vp[p]
            bt[s, p] = b
            if s == 0 and p < shared_pages:
                shared_ids.append(b)
    return kpool, vpool, bt


def _sdpa(q, k, v, scale, causal=False):
    """torch reference on contiguous tensors: q [Lq, Hq, D], k/v [Lk, Hkv, D]."""
    qq = q.to(torch.float64).permute(1, 0, 2).unsqueeze(0)
    kk = k.to(torch.float64).permute(1, 0, 2).unsqueeze(0)
    vv = v.to(torch.float64).permute(1, 0, 2).unsqueeze(0)
    out = F.scaled_dot_product_attention(qq, kk, vv, scale=scale, is_causal=causal, enable_gqa=True)
    return out.squeeze(0).permute(1, 0, 2).numpy()


def _maxdiff(a, b) -> float:
    """Largest absolute difference; NaN anywhere counts as an infinite difference."""
    d = np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))
    return float("inf") if np.isnan(d).any() else float(d.max(initial=0.0))


def _randn(gen, shape, dtype):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(DT[dtype][0])


# ---- 16-bit decoders ----------------------------------------------------------

def test_f16_decoder_matches_numpy_on_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(pats, oracle.F16)
    ref = pats.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_bf16_decoder_matches_torch_on_every_pattern():
    pats = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = pats.view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.widen(pats.numpy().view(np.uint16), oracle.BF16)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


# ---- paged store: worked examples ----------------------------------------------

def _golden_examples():
    out = {}
    with open(os.path.join(GOLDEN, "paged_worked_examples.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = (x.strip() for x in line.split("="))
                out[k] = int(v)
    return out


def test_write_then_read_worked_example():
    ex = _golden_examples()
    gen = torch.Generator().manual_seed(7)
    hkv = 8
    kpool = np.random.default_rng(0).integers(0, 65536, (64, BS, hkv, D), dtype=np.uint16)
    vpool = kpool[::-1].copy()
    before_k, before_v = kpool.copy(), vpool.copy()
    k_new, v_new = _randn(gen, (2, hkv, D), "f16"), _randn(gen, (2, hkv, D), "f16")
    # blocks [0, 1], positions 0 and 1 -> block 0, offsets 0 and 1 -> flat slots 0, 1
    assert oracle.kv_cache_write(kpool, vpool, k_new, v_new, np.array([0, 1])) == 0
    for h in range(hkv):
        kr, vr = oracle.gather_head(kpool, vpool, oracle.F16, [0, 1], h, 2)
        assert kr.shape[0] == ex["write_then_read_rows"]
        assert np.array_equal(kr, k_new[:, h].to(torch.float64).numpy())
        assert np.array_equal(vr, v_new[:, h].to(torch.float64).numpy())
    changed = np.any(kpool != before_k, axis=(2, 3))
    assert changed.sum() == 2 and changed[0, 0] and changed[0, 1]
    assert np.array_equal(np.any(vpool != before_v, axis=(2, 3)), changed)
    kr, _ = oracle.gather_head(kpool, vpool, oracle.F16, [0, 1], 0, 17)
    assert kr.shape == (ex["read_rows_for_length_17"], D)


def test_write_follows_pool_layout_with_permuted_table():
    """Block b is the outer index of a layer's pool and the in-block slot the
    next one; logical position j of a sequence with table [5, 2] is block
    table[j // 16], slot j % 16."""
    gen = torch.Generator().manual_seed(8)
    hkv = 8
    kpool = np.zeros((64, BS, hkv, D), np.uint16)
    vpool = np.zeros((64, BS, hkv, D), np.uint16)
    k_new, v_new = _randn(gen, (3, hkv, D), "bf16"), _randn(gen, (3, hkv, D), "bf16")
    slots = np.array([5 * 16 + 15, 2 * 16 + 0, 2 * 16 + 1])      # positions 15, 16, 17
    oracle.kv_cache_write(kpool, vpool, k_new, v_new, slots)
    kb, vb = _bits(k_new), _bits(v_new)
    for i, (b, o) in enumerate([(5, 15), (2, 0), (2, 1)]):
        assert np.array_equal(kpool[b, o], kb[i]) and np.array_equal(vpool[b, o], vb[i])
    assert np.count_nonzero(np.any(kpool != 0, axis=(2, 3))) == 3
    for h in range(hkv):
        kr, _ = oracle.gather_head(kpool, vpool, oracle.BF16, [5, 2], h, 18)
        assert np.array_equal(kr[15:18], k_new[:, h].to(torch.float64).numpy())


def test_write_repeated_slot_keeps_last_and_skips_out_of_range():
    gen = torch.Generator().manual_seed(9)
    kpool = np.zeros((4, BS, 2, D), np.uint16)
    vpool = np.zeros((4, BS, 2, D), np.uint16)
    k_new, v_new = _randn(gen, (4, 2, D), "f16"), _randn(gen, (4, 2, D), "f16")
    skipped = oracle.kv_cache_write(kpool, vpool, k_new, v_new, np.array([3, 3, 64, -1]))
    assert skipped == 2
    assert np.array_equal(kpool[0, 3], _bits(k_new)[1])
    assert np.count_nonzero(np.any(kpool != 0, axis=(2, 3))) == 1


def test_block_placement_uses_exactly_ceil_len_over_16_blocks():
    ex = _golden_examples()
    assert workloads.cdiv(20, ex["block_size"]) == ex["blocks_for_20_tokens"]
    rng = np.random.default_rng(12)
    lens = [int(x) for x in rng.integers(1, 513, 32)]
    bt, nb = workloads._place(rng, lens, 0, None, 0.25)
    used = bt[bt >= 0]
    assert len(used) == len(set(used.tolist())) == sum(-(-n // ex["block_size"]) for n in lens)
    assert used.max() < nb


# ---- attention against torch SDPA on contiguous K/V ------------------------------

def _decode_vs_sdpa(dtype, hq, hkv, lens, seed):
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    seqs = [(_randn(gen, (n, hkv, D), dtype), _randn(gen, (n, hkv, D), dtype)) for n in lens]
    kpool, vpool, bt = _paged_from_contiguous(seqs, sum(-(-n // BS) for n in lens) + 3, hkv, dtype, rng)
    q = _randn(gen, (len(lens), hq, D), dtype)
    scale = 1.0 / math.sqrt(D)
    got = oracle.paged_attn_decode(q, kpool, vpool, bt, lens, scale, DT[dtype][1])
    err = 0.0
    for s, (k, v) in enumerate(seqs):
        ref = _sdpa(q[s:s + 1], k, v, scale)[0]
        err = max(err, _maxdiff(got[s], ref))
    return err


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (8, 2), (16, 8)])
def test_decode_matches_torch_sdpa(dtype, hq, hkv):
    assert _decode_vs_sdpa(dtype, hq, hkv, [1, 15, 16, 17, 33], seed=hq * 10 + hkv) < 1e-12


def _prefill_vs_sdpa(dtype, hq, hkv, chunks, seed):
    """One sequence of total length L; the chunks (start, n) tile [0, L).  The
    reference is one causal pass over the whole sequence (top-left aligned
    square mask), whose rows start..start+n-1 are the chunk's rows."""
    gen = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    L = chunks[-1][0] + chunks[-1][1]
    k, v = _randn(gen, (L, hkv, D), dtype), _randn(gen, (L, hkv, D), dtype)
    kpool, vpool, bt = _paged_from_contiguous([(k, v)], -(-L // BS) + 2, hkv, dtype, rng)
    q_all = _randn(gen, (L, hq, D), dtype)
    scale = 1.0 / math.sqrt(D)
    ref = _sdpa(q_all, k, v, scale, causal=True)
    # chunks of one sequence, each with the same block-table row
    starts = [s for s, _ in chunks]
    lens = [n for _, n in chunks]
    got = oracle.paged_attn_prefill(q_all, kpool, vpool, starts, lens, np.repeat(bt, len(chunks), 0),
                                    [s + n for s, n in chunks], scale, DT[dtype][1])
    return _maxdiff(got, ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2), (8, 2)])
def test_chunked_prefill_matches_torch_causal_sdpa(dtype, hq, hkv):
    chunks = [(0, 17), (17, 16), (33, 1), (34, 30)]
    assert _prefill_vs_sdpa(dtype, hq, hkv, chunks, seed=hq + hkv) < 1e-12


# ---- closed forms -------------------------------------------------------------

def _single(dtype, hq, hkv, k, v, q, n, seed=0):
    rng = np.random.default_rng(seed)
    kpool, vpool, bt = _paged_from_contiguous([(k, v)], -(-n // BS) + 2, hkv, dtype, rng)
    return oracle.paged_attn_decode(q.unsqueeze(0), kpool, vpool, bt, [n], 1 / math.sqrt(D), DT[dtype][1])[0]


def test_one_key_returns_its_value_exactly():
    gen = torch.Generator().manual_seed(1)
    k, v, q = _randn(gen, (1, 2, D), "f16"), _randn(gen, (1, 2, D), "f16"), _randn(gen, (4, D), "f16")
    out = _single("f16", 4, 2, k, v, q, 1)
    for g in range(4):
        assert np.array_equal(out[g], v[0, g // 2].to(torch.float64).numpy())


def test_zero_query_averages_values():
    gen = torch.Generator().manual_seed(2)
    n = 37
    k, v = _randn(gen, (n, 2, D), "bf16"), _randn(gen, (n, 2, D), "bf16")
    out = _single("bf16", 4, 2, k, v, torch.zeros(4, D, dtype=torch.bfloat16), n)
    mean = v.to(torch.float64).mean(0).numpy()
    for g in range(4):
        assert _maxdiff(out[g], mean[g // 2]) < 1e-14


def test_equal_keys_average_values():
    gen = torch.Generator().manual_seed(3)
    n = 40
    k = _randn(gen, (1, 2, D), "f16").expand(n, 2, D).contiguous()
    v = _randn(gen, (n, 2, D), "f16")
    out = _single("f16", 4, 2, k, v, _randn(gen, (4, D), "f16"), n)
    mean = v.to(torch.float64).mean(0).numpy()
    for g in range(4):
        assert _maxdiff(out[g], mean[g // 2]) < 1e-14


def test_constant_values_per_kv_head_fix_the_gqa_map():
    """Query head g must read KV head g // (Hq/Hkv): with V of KV head h equal
    to h+1 everywhere, query heads hG .. hG+G-1 output h+1."""
    gen = torch.Generator().manual_seed(4)
    hq, hkv, n = 8, 4, 50
    k = _randn(gen, (n, hkv, D), "f16")
    v = torch.arange(1, hkv + 1, dtype=torch.float16).view(1, hkv, 1).expand(n, hkv, D).contiguous()
    out = _single("f16", hq, hkv, k, v, _randn(gen, (hq, D), "f16"), n)
    for g in range(hq):
        assert _maxdiff(out[g], np.full(D, g // (hq // hkv) + 1.0)) < 1e-13


def test_dominant_key_selects_its_value():
    gen = torch.Generator().manual_seed(5)
    n, j = 33, 20
    q = _randn(gen, (2, D), "f16")
    k = (_randn(gen, (n, 1, D), "f16") * 0.01).to(torch.float16)
    k[j, 0] = (q[0] * 4).to(torch.float16)      # score ~ 4|q|^2 / sqrt(128) >> others
    v = _randn(gen, (n, 1, D), "f16")
    out = _single("f16", 2, 1, k, v, q, n)
    assert _maxdiff(out[0], v[j, 0].to(torch.float64).numpy()) < 1e-6


# ---- invariants -----------------------------------------------------------------

def test_physical_block_permutation_changes_nothing():
    gen = torch.Generator().manual_seed(6)
    lens = [5, 16, 40, 70]
    seqs = [(_randn(gen, (n, 2, D), "bf16"), _randn(gen, (n, 2, D), "bf16")) for n in lens]
    q = _randn(gen, (4, 4, D), "bf16")
    outs = []
    for seed in (1, 2, 3):
        kp, vp, bt = _paged_from_contiguous(seqs, 40, 2, "bf16", np.random.default_rng(seed))
        outs.append(oracle.paged_attn_decode(q, kp, vp, bt, lens, 0.1, oracle.BF16))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_shared_prefix_pages_equal_private_copies():
    gen = torch.Generator().manual_seed(7)
    prefix_k, prefix_v = _randn(gen, (48, 2, D), "bf16"), _randn(gen, (48, 2, D), "bf16")
    seqs = []
    for n in (3, 20, 33):
        sk, sv = _randn(gen, (n, 2, D), "bf16"), _randn(gen, (n, 2, D), "bf16")
        seqs.append((torch.cat([prefix_k, sk]), torch.cat([prefix_v, sv])))
    lens = [s[0].shape[0] for s in seqs]
    q = _randn(gen, (3, 4, D), "bf16")
    kp, vp, bt = _paged_from_contiguous(seqs, 40, 2, "bf16", np.random.default_rng(1), shared_pages=3)
    assert (bt[:, :3] == bt[0, :3]).all()
    shared = oracle.paged_attn_decode(q, kp, vp, bt, lens, 0.1, oracle.BF16)
    kp2, vp2, bt2 = _paged_from_contiguous(seqs, 40, 2, "bf16", np.random.default_rng(1))
    assert len(set(bt2[:, :3].ravel().tolist())) == 9
    private = oracle.paged_attn_decode(q, kp2, vp2, bt2, lens, 0.1, oracle.BF16)
    assert np.array_equal(shared, private)


def test_chunked_equals_unchunked_and_decode_equals_last_prefill_row():
    gen = torch.Generator().manual_seed(8)
    L, hq, hkv = 70, 4, 2
    k, v = _randn(gen, (L, hkv, D), "f16"), _randn(gen, (L, hkv, D), "f16")
    kp, vp, bt = _paged_from_contiguous([(k, v)], 8, hkv, "f16", np.random.default_rng(2))
    q = _randn(gen, (L, hq, D), "f16")
    one = oracle.paged_attn_prefill(q, kp, vp, [0], [L], bt, [L], 0.09, oracle.F16)
    chunks = [(0, 16), (16, 1), (17, 40), (57, 13)]
    many = oracle.paged_attn_prefill(q, kp, vp, [s for s, _ in chunks], [n for _, n in chunks],
                                     np.repeat(bt, 4, 0), [s + n for s, n in chunks], 0.09, oracle.F16)
    assert np.array_equal(one, many)
    for pos in (0, 15, 16, 69):
        dec = oracle.paged_attn_decode(q[pos:pos + 1], kp, vp, bt, [pos + 1], 0.09, oracle.F16)
        assert np.array_equal(dec[0], one[pos])


def test_oracle_rejects_inconsistent_inputs():
    kp = np.zeros((4, BS, 1, D), np.uint16)
    q = np.zeros((1, 1, D), np.uint16)
    with pytest.raises(ValueError):
        oracle.paged_attn_decode(q, kp, kp, np.array([[0]]), [0], 1.0, oracle.F16)     # empty context
    with pytest.raises(ValueError):
        oracle.paged_attn_decode(q, kp, kp, np.array([[0]]), [17], 1.0, oracle.F16)    # past the table
    with pytest.raises(ValueError):
        oracle.paged_attn_decode(q, kp, kp, np.array([[9]]), [3], 1.0, oracle.F16)     # block id out of pool
    with pytest.raises(ValueError):
        oracle.paged_attn_prefill(q, kp, kp, [0], [1], np.array([[0]]), [2], 1.0, oracle.F16)


# ---- KV closed forms printed on the pages ---------------------------------------

def _closed_forms():
    rows = []
    with open(os.path.join(GOLDEN, "kv_closed_forms.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(tuple(int(x) for x in line.split()))
    return rows


@pytest.mark.parametrize("row", _closed_forms())
def test_kv_byte_closed_forms(row):
    *args, expected = row
    assert oracle.kv_bytes(*args) == expected
    assert workloads.kv_bytes(*args) == expected


def test_prefill_flop_count_of_the_mixed_step():
    # 3 chunks of 512 on prefixes 0, 512, 1536 with 16 query heads, head_dim 128
    assert workloads.prefill_flops([(0, 512), (512, 512), (1536, 512)], 16) == 11_817_451_520


def test_prefill_flop_count_under_a_window():
    chunks = [(0, 512), (512, 512), (1536, 512)]
    full = workloads.prefill_flops(chunks, 16)
    assert workloads.prefill_flops(chunks, 16, window=2048) == full    # no row sees more than 2048 keys
    # W = 512: every row of the last two chunks sees 512 keys; row i of the first sees i + 1
    pairs = 512 * 513 // 2 + 2 * 512 * 512
    assert workloads.prefill_flops(chunks, 16, window=512) == 4 * 128 * 16 * pairs
    assert workloads.prefill_flops([(5, 3)], 1, window=1) == 4 * 128 * 3


# ---- planted mistakes: the battery must catch each -------------------------------

def _battery():
    """Returns the names of the pins that fail on the currently loaded oracle."""
    failed = []
    try:
        if _decode_vs_sdpa("f16", 4, 2, [1, 17, 33], seed=3) > 1e-12:
            failed.append("decode-sdpa")
    except Exception:
        failed.append("decode-sdpa(raised)")
    try:
        if _prefill_vs_sdpa("bf16", 4, 2, [(0, 17), (17, 20)], seed=4) > 1e-12:
            failed.append("prefill-sdpa")
    except Exception:
        failed.append("prefill-sdpa(raised)")
    for name, fn in [("one-key", test_one_key_returns_its_value_exactly),
                     ("gqa-map", test_constant_values_per_kv_head_fix_the_gqa_map),
                     ("write-layout", test_write_follows_pool_layout_with_permuted_table),
                     ("f16-decoder", test_f16_decoder_matches_numpy_on_every_pattern),
                     ("bf16-decoder", test_bf16_decoder_matches_torch_on_every_pattern)]:
        try:
            fn()
        except Exception:
            failed.append(name)
    return failed


MUTATIONS = {
    "gqa-map-interleaved": ("for (int32_t qh = h * G; qh < (h + 1) * G; ++qh)",
                            "for (int32_t qh = h; qh < P->num_q_heads; qh += P->num_kv_heads)"),
    "causal-excludes-self": ("p - lo + 1, d, P->scale, s,", "p - lo + (i == 0), d, P->scale, s,"),
    "scale-dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "values-from-keys": ("out[x] += p * vv[(int64_t)j * d + x];", "out[x] += p * kk[(int64_t)j * d + x];"),
    "slot-offset-shifted": ("int32_t entry = j / block_size, offset = j % block_size;",
                            "int32_t entry = j / block_size, offset = (j + 1) % block_size;"),
    "table-entry-by-offset": ("int32_t entry = j / block_size, offset = j % block_size;",
                              "int32_t entry = j % block_size, offset = j / block_size;"),
    "f16-exponent-bias": ("mag = ldexp((double)(1024 + f), e - 25);", "mag = ldexp((double)(1024 + f), e - 24);"),
    "bf16-fraction-width": ("mag = ldexp((double)(128 + f), e - 134);", "mag = ldexp((double)(128 + f), e - 133);"),
    "write-block-stride": ("int64_t dst = (block * block_size + offset) * row;",
                           "int64_t dst = (offset * num_blocks + block) * row;"),
    "normaliser-dropped": ("double p = s[j] / z;", "double p = s[j];"),
}


def test_battery_passes_on_the_real_oracle():
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "liboracle_mut.so"))
    with oracle.use_library(lib):
        failed = _battery()
    assert failed, f"planted mistake '{name}' was not caught by any pin"
