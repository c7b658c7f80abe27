"""GPU parity of the q/k RMSNorm + rotary embedding fused into the KV write
("Модуль 12: Финальный проект: мини-движок инференса", qwen_serve/model.py:
rms_norm, apply_rope, Qwen3Model.forward; "Модуль 04: KV-кэш и арифметика
памяти", section 4: rotate the key before storing it), through the C-ABI:
bit-exact against the oracle (q_out and both pools, which follow the page's
rounding points), in place, with bad tokens, and followed by a decode over the
rotated cache."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
from gpu_util import ORACLE_DTYPE, bits, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
BS, D = 16, 128
TDT = {"bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.get_device_error()
    yield
    st, detail = pa.get_device_error()
    assert st == 0, f"unexpected device error {pa.STATUS.get(st, st)} at index {detail}"


def _tables(max_pos, dtype, theta=1e6):
    # NeoX rotary tables: frequencies theta^(-2i/d) in fp32, duplicated halves, cast to the model dtype
    inv = 1.0 / (theta ** (torch.arange(0, D, 2, dtype=torch.float32) / D))
    f = torch.outer(torch.arange(max_pos, dtype=torch.float32), inv)
    c, s = torch.cos(f), torch.sin(f)
    return torch.cat([c, c], -1).to(TDT[dtype]).to(DEV), torch.cat([s, s], -1).to(TDT[dtype]).to(DEV)


def _case(T, hq, hkv, dtype, seed, nb=None, max_pos=32768):
    g = torch.Generator(device=DEV).manual_seed(seed)
    dt = TDT[dtype]
    mag = lambda shape: torch.exp(torch.randn(shape[:-1] + (1,), generator=g, device=DEV) * 2)
    q = (torch.randn((T, hq, D), generator=g, device=DEV) * mag((T, hq, D))).to(dt)
    k = (torch.randn((T, hkv, D), generator=g, device=DEV) * mag((T, hkv, D))).to(dt)
    v = torch.randn((T, hkv, D), generator=g, device=DEV).to(dt)
    wq = (1 + 0.3 * torch.randn(D, generator=g, device=DEV)).to(dt)
    wk = (1 + 0.3 * torch.randn(D, generator=g, device=DEV)).to(dt)
    nb = nb or (T + BS - 1) // BS + 3
    rng = np.random.default_rng(seed)
    slots = torch.from_numpy(rng.permutation(nb * BS)[:T].astype(np.int64)).to(DEV)
    pos = torch.from_numpy(rng.integers(0, max_pos, size=T).astype(np.int32)).to(DEV)
    kc = torch.full((nb, BS, hkv, D), float("nan"), device=DEV).to(dt)
    vc = torch.full((nb, BS, hkv, D), float("nan"), device=DEV).to(dt)
    cos, sin = _tables(max_pos, dtype)
    return dict(q=q, k=k, v=v, wq=wq, wk=wk, cos=cos, sin=sin, pos=pos, slots=slots, kc=kc, vc=vc, dtype=dtype)


def _oracle(c, eps):
    kh, vh = bits(c["kc"]), bits(c["vc"])
    out, skipped = oracle.qk_norm_rope_kv_write(bits(c["q"]), bits(c["k"]), bits(c["v"]), bits(c["wq"]),
                                                bits(c["wk"]), eps, bits(c["cos"]), bits(c["sin"]),
                                                c["pos"].cpu().numpy(), c["slots"].cpu().numpy(), kh, vh,
                                                ORACLE_DTYPE[c["dtype"]])
    return out, kh, vh, skipped


def _gpu(c, eps, q_out=None):
    out = pa.qk_norm_rope_kv_write(c["q"], c["k"], c["v"], c["wq"], c["wk"], eps, c["cos"], c["sin"], c["pos"],
                                   c["slots"], c["kc"], c["vc"], q_out=q_out)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T", [1, 7, 300, 2048])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (8, 8), (16, 2)])
def test_fused_write_is_bit_exact(T, dtype, hq, hkv):
    c = _case(T, hq, hkv, dtype, seed=T + hq + (dtype == "f16"))
    ref_q, ref_k, ref_v, skipped = _oracle(c, 1e-6)
    out = _gpu(c, 1e-6)
    assert skipped == 0
    assert np.array_equal(bits(out), ref_q), "q_out"
    assert np.array_equal(bits(c["kc"]), ref_k), "k pool"
    assert np.array_equal(bits(c["vc"]), ref_v), "v pool"


def test_in_place_and_a_large_eps():
    c = _case(64, 16, 8, "bf16", seed=3)
    ref_q, ref_k, _, _ = _oracle(c, 0.5)
    out = _gpu(c, 0.5, q_out=c["q"])
    assert out.data_ptr() == c["q"].data_ptr()
    assert np.array_equal(bits(out), ref_q) and np.array_equal(bits(c["kc"]), ref_k)


def test_bad_position_and_slot_are_reported_and_skipped():
    c = _case(6, 16, 8, "bf16", seed=4, nb=2, max_pos=64)
    c["pos"][2] = 64                     # outside the 64-row tables
    c["slots"][4] = 2 * BS               # outside the 2-block pool
    c["q"] = c["q"].contiguous()
    q_out = torch.zeros_like(c["q"])
    ref_q, ref_k, ref_v, skipped = _oracle(c, 1e-6)
    _gpu(c, 1e-6, q_out=q_out)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail in (2, 4) and skipped == 2
    assert np.array_equal(bits(q_out), ref_q)
    assert np.array_equal(bits(c["kc"]), ref_k) and np.array_equal(bits(c["vc"]), ref_v)


def test_decode_over_the_rotated_cache():
    # decode queries = the normed, rotated q of each sequence's newest token
    hq, hkv, dtype = 16, 8, "bf16"
    lens = [5, 40, 77]
    T = sum(lens)
    c = _case(T, hq, hkv, dtype, seed=8, nb=16)
    bt = np.full((len(lens), 8), -1, np.int32)
    slots, pos, r = [], [], 0
    blocks = np.random.default_rng(8).permutation(16)
    for s, n in enumerate(lens):
        pages = -(-n // BS)
        bt[s, :pages] = blocks[r:r + pages]
        r += pages
        for j in range(n):
            slots.append(int(bt[s, j // BS]) * BS + j % BS)
            pos.append(j)
    c["slots"] = torch.tensor(slots, dtype=torch.int64, device=DEV)
    c["pos"] = torch.tensor(pos, dtype=torch.int32, device=DEV)
    ref_q, ref_k, ref_v, _ = _oracle(c, 1e-6)
    out = _gpu(c, 1e-6)
    assert np.array_equal(bits(out), ref_q)
    last = np.cumsum(lens) - 1
    qd = out[torch.from_numpy(last).to(DEV)].contiguous()
    ctx = np.asarray(lens, np.int32)
    got = pa.paged_attn_decode(qd, c["kc"], c["vc"], torch.from_numpy(bt).to(DEV), torch.from_numpy(ctx).to(DEV),
                               1 / np.sqrt(D))
    torch.cuda.synchronize()
    ref = oracle.paged_attn_decode(ref_q[last], ref_k, ref_v, bt, ctx, 1 / np.sqrt(D), oracle.BF16)
    check_close(got, ref, "decode over the rotated cache")
