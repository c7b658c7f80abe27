"""Pins for the oracle's q/k RMSNorm + rotary embedding + KV write ("Модуль 12:
Финальный проект: мини-движок инференса", qwen_serve/model.py: rms_norm,
_rope_tables, _rotate_half, apply_rope, Qwen3Model.forward; "Модуль 04: KV-кэш
и арифметика памяти", section 4: the key is rotated to its absolute position
before it is stored).  Each check ties the oracle to something other than
itself:

* its 16-bit rounding against torch's fp32 -> bf16/fp16 conversion on every
  16-bit pattern and on every midpoint between neighbours (ties to even);
* closed forms of RMSNorm: rows of +-2^k give sign * weight exactly, a row of
  2^-10 shows the eps term, unit weights give mean square ~1;
* closed forms of the rotation with crafted table rows: cos 1 / sin 0 is the
  identity, cos 0 / sin 1 is rotate_half exactly (sign and NeoX pairing);
* numpy complex multiplication (z_i + i z_{i+64}) e^{i theta} on the page's
  tables at random positions;
* the write: v bits unchanged, the rotated k in the slot, other slots
  untouched, bad positions and slots skipped;
* planted mistakes in mutated copies of the oracle fail this battery.
"""
import os

import numpy as np
import pytest
import torch

import oracle

D, BS = 128, 16
TDT = {oracle.BF16: torch.bfloat16, oracle.F16: torch.float16}


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _val(b, dt):
    return torch.from_numpy(np.asarray(b, np.uint16).view(np.int16)).view(TDT[dt]).to(torch.float64).numpy()


def _tables(max_pos, theta=1e6, dt=oracle.BF16):
    # the page's NeoX tables: frequencies theta^(-2i/d) in fp32, duplicated halves, cast to the 16-bit type
    inv = 1.0 / (theta ** (torch.arange(0, D, 2, dtype=torch.float32) / D))
    f = torch.outer(torch.arange(max_pos, dtype=torch.float32), inv)
    c, s = torch.cos(f), torch.sin(f)
    return _bits(torch.cat([c, c], -1).to(TDT[dt])), _bits(torch.cat([s, s], -1).to(TDT[dt]))


def _run(q, k, v, wq, wk, cos, sin, pos, slots, nb=8, hkv=None, dt=oracle.BF16, eps=1e-6):
    hkv = hkv or k.shape[1]
    kc = np.zeros((nb, BS, hkv, D), np.uint16)
    vc = np.zeros((nb, BS, hkv, D), np.uint16)
    out, skipped = oracle.qk_norm_rope_kv_write(q, k, v, wq, wk, eps, cos, sin, pos, slots, kc, vc, dt)
    return out, kc, vc, skipped


def _rand(shape, seed, dt=oracle.BF16, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return _bits((torch.randn(shape, generator=g) * scale).to(TDT[dt]))


@pytest.mark.parametrize("dt", [oracle.BF16, oracle.F16])
def test_rounding_matches_torch_on_every_pattern_and_midpoint(dt):
    pats = np.arange(1 << 16, dtype=np.uint16)
    vals = _val(pats, dt)
    ok = np.isfinite(vals)
    vals, pats = vals[ok], pats[ok]
    order = np.argsort(vals, kind="stable")
    vs = vals[order]
    mids = (vs[:-1] + vs[1:]) / 2            # exact in fp32 for neighbours of a 16-bit format
    for x in (vs, mids):
        x32 = x.astype(np.float32)
        assert np.array_equal(x32.astype(np.float64), x)
        want = _bits(torch.from_numpy(x32).to(TDT[dt]))
        got = np.array([oracle.f64_to_16(float(v), dt) for v in x], np.uint16)
        neg_zero = (x == 0) & np.signbit(x)
        assert np.array_equal(got[~neg_zero], want[~neg_zero])


def _norm_closed_forms():
    # rows of +-2^k: mean square 4^k, inv = 2^-k (eps below the fp32 resolution) -> y = +-1, out = +-w
    rng = np.random.default_rng(0)
    signs = rng.choice([-1.0, 1.0], size=(3, 1, D))
    powers = np.array([1.0, 4.0, 0.25]).reshape(3, 1, 1)
    q = _bits(torch.from_numpy(signs * powers).to(torch.bfloat16))
    wq = _rand((D,), 1)
    wk = _bits(torch.ones(D).to(torch.bfloat16))
    cos, sin = _bits(torch.ones(1, D).to(torch.bfloat16)), _bits(torch.zeros(1, D).to(torch.bfloat16))
    k = q[:, :1].copy()
    out, kc, _, _ = _run(q, k, k, wq, wk, cos, sin, [0, 0, 0], [0, 1, 2])
    want = _bits(torch.from_numpy(signs * _val(wq, oracle.BF16)).to(torch.bfloat16))
    assert np.array_equal(out, want)
    assert np.array_equal(kc[0, :3, 0], _bits(torch.from_numpy(signs[:, 0]).to(torch.bfloat16)))


def test_rms_norm_of_powers_of_two_is_sign_times_weight():
    _norm_closed_forms()


def _eps_form():
    # a row of 2^-10: var = 2^-20 is comparable to eps = 1e-6, so y = 2^-10 / sqrt(2^-20 + 1e-6)
    q = _bits(torch.full((1, 1, D), 2.0 ** -10).to(torch.bfloat16))
    w = _bits(torch.ones(D).to(torch.bfloat16))
    cos, sin = _bits(torch.ones(1, D).to(torch.bfloat16)), _bits(torch.zeros(1, D).to(torch.bfloat16))
    out, _, _, _ = _run(q, q, q, w, w, cos, sin, [0], [0])
    y = np.float32(2.0 ** -10) * np.float32(1.0 / np.sqrt(np.float64(np.float32(2.0 ** -20) + np.float32(1e-6))))
    want = _bits(torch.full((1, 1, D), float(y)).to(torch.bfloat16))
    assert np.array_equal(out, want)
    assert _val(out, oracle.BF16).max() < 0.8           # far from the eps-free value 1.0


def test_rms_norm_eps_term():
    _eps_form()


@pytest.mark.parametrize("dt", [oracle.BF16, oracle.F16])
def test_unit_weight_rows_have_unit_mean_square(dt):
    q = _rand((64, 4, D), 2, dt, scale=3.0)
    w = _bits(torch.ones(D).to(TDT[dt]))
    cos, sin = _tables(4, dt=dt)
    out, _, _, _ = _run(q, q[:, :2], q[:, :2], w, w, cos, sin, np.zeros(64, np.int32), np.arange(64), dt=dt)
    ms = (_val(out, dt) ** 2).mean(-1)
    assert np.abs(ms - 1).max() < 2e-2


def _rotation_forms():
    z = _rand((2, 1, D), 3)
    w = _bits(torch.ones(D).to(torch.bfloat16))
    # table row 0: cos 1, sin 0 (identity); row 1: cos 0, sin 1 (rotate_half exactly)
    cos = _bits(torch.stack([torch.ones(D), torch.zeros(D)]).to(torch.bfloat16))
    sin = _bits(torch.stack([torch.zeros(D), torch.ones(D)]).to(torch.bfloat16))
    normed, _, _, _ = _run(z, z, z, w, w, cos, sin, [0, 0], [0, 1])
    out, _, _, _ = _run(z, z, z, w, w, cos, sin, [0, 1], [0, 1])
    assert np.array_equal(out[0], normed[0])
    n1 = normed[1, 0]
    want = np.concatenate([n1[64:] ^ np.uint16(0x8000), n1[:64]])     # (-z[64:], z[:64])
    assert np.array_equal(out[1, 0], want)


def test_rotation_closed_forms_fix_sign_and_pairing():
    _rotation_forms()


def _complex_form(dt=oracle.BF16):
    rng = np.random.default_rng(4)
    max_pos = 40000
    cos, sin = _tables(max_pos, dt=dt)
    pos = rng.integers(0, max_pos, size=32).astype(np.int32)
    z = _rand((32, 2, D), 5, dt)
    w = _bits(torch.ones(D).to(TDT[dt]))
    ident_c = _bits(torch.ones(1, D).to(TDT[dt]))
    ident_s = _bits(torch.zeros(1, D).to(TDT[dt]))
    normed, _, _, _ = _run(z, z, z, w, w, ident_c, ident_s, np.zeros(32, np.int32), np.arange(32), nb=2, dt=dt)
    out, _, _, _ = _run(z, z, z, w, w, cos, sin, pos, np.arange(32), nb=2, dt=dt)
    n = _val(normed, dt)
    c = _val(cos, dt)[pos][:, None, :64]
    s = _val(sin, dt)[pos][:, None, :64]
    zc = (n[..., :64] + 1j * n[..., 64:]) * (c + 1j * s)       # rotation by the table's angle
    got = _val(out, dt)
    err = np.abs(np.concatenate([zc.real, zc.imag], -1) - got)
    scale = np.abs(n[..., :64]) + np.abs(n[..., 64:])
    tol = 2.0 ** (-6 if dt == oracle.BF16 else -9) * np.concatenate([scale, scale], -1) + 1e-6
    assert (err <= tol).all()


@pytest.mark.parametrize("dt", [oracle.BF16, oracle.F16])
def test_rotation_matches_complex_multiplication(dt):
    _complex_form(dt)


def _write_form():
    T, hq, hkv = 5, 4, 2
    q, k, v = _rand((T, hq, D), 6), _rand((T, hkv, D), 7), _rand((T, hkv, D), 8)
    wq, wk = _rand((D,), 9), _rand((D,), 10)
    cos, sin = _tables(100)
    pos = np.array([3, 99, 0, 100, 7], np.int32)      # position 100 is outside the 100-row tables
    slots = np.array([17, 4, 8 * BS, 5, 0], np.int64)  # slot 128 is outside an 8-block pool
    out, kc, vc, skipped = _run(q, k, v, wq, wk, cos, sin, pos, slots)
    assert skipped == 2
    for t in (0, 1, 4):
        b, o = divmod(int(slots[t]), BS)
        assert np.array_equal(vc[b, o], v[t])
        one, _, _, _ = _run(k[t:t + 1], k[t:t + 1], v[t:t + 1], wk, wk, cos, sin, pos[t:t + 1], [0])
        assert np.array_equal(kc[b, o], one[0])          # k rotated like a query head with k's weight
    written = {int(s) for s in slots[[0, 1, 4]]}
    for s in range(8 * BS):
        if s not in written:
            assert not kc.reshape(-1, hkv, D)[s].any() and not vc.reshape(-1, hkv, D)[s].any()
    assert not out[2].any() and not out[3].any()


def test_write_stores_rotated_k_and_raw_v_and_skips_bad_tokens():
    _write_form()


def _gqa_weights_form():
    # the query heads take the q weight and the KV heads the k weight
    q = _bits(torch.ones(1, 2, D).to(torch.bfloat16))
    wq = _bits(torch.full((D,), 2.0).to(torch.bfloat16))
    wk = _bits(torch.full((D,), 3.0).to(torch.bfloat16))
    cos, sin = _bits(torch.ones(1, D).to(torch.bfloat16)), _bits(torch.zeros(1, D).to(torch.bfloat16))
    out, kc, _, _ = _run(q, q[:, :1], q[:, :1], wq, wk, cos, sin, [0], [0])
    assert (_val(out, oracle.BF16) == 2.0).all() and (_val(kc[0, 0], oracle.BF16) == 3.0).all()


def test_query_and_key_heads_take_their_own_weights():
    _gqa_weights_form()


# ---- planted mistakes ----------------------------------------------------------------

def _battery():
    failed = []
    for name, fn in [("powers", _norm_closed_forms), ("eps", _eps_form), ("rotation", _rotation_forms),
                     ("complex", _complex_form), ("write", _write_form), ("weights", _gqa_weights_form)]:
        try:
            fn()
        except Exception:
            failed.append(name)
    return failed


MUTATIONS = {
    "eps-dropped": ("  const float s = var + eps;\n", "  const float s = var;\n"),
    "rotate-half-sign": ("    const double rot = i < h ? -widen(z[i + h], dtype) : widen(z[i - h], dtype);",
                         "    const double rot = i < h ? widen(z[i + h], dtype) : -widen(z[i - h], dtype);"),
    "interleaved-pairs": ("    const double rot = i < h ? -widen(z[i + h], dtype) : widen(z[i - h], dtype);",
                          "    const double rot = (i % 2 == 0) ? -widen(z[i + 1], dtype) : widen(z[i - 1], dtype);"),
    "position-off-by-one": ("    const uint16_t *cos_row = cos_table + (int64_t)pos * head_dim;",
                            "    const uint16_t *cos_row = cos_table + (int64_t)(pos + 1 < max_position ? pos + 1 : pos) * head_dim;"),
    "k-takes-q-weight": ("      rms_norm_row(k + src, k_weight, eps, head_dim, dtype, normed);",
                         "      rms_norm_row(k + src, q_weight, eps, head_dim, dtype, normed);"),
    "v-not-written": ("      for (int32_t x = 0; x < head_dim; ++x) v_cache[dst + x] = v[src + x];\n", ""),
    "weight-not-applied": ("    out[i] = narrow(widen(yb, dtype) * widen(weight[i], dtype), dtype);",
                           "    out[i] = yb;"),
}


def test_rope_battery_passes_on_the_real_oracle():
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_rope_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "liboracle_mut.so"))
    with oracle.use_library(lib):
        failed = _battery()
    assert failed, f"planted mistake '{name}' was not caught by any pin"
