"""GPU parity of the decode with PA_DECODE_EARLY_PAGES (pa_paged_attn_decode_ex):
the one-launch decode fetches every page but a sequence's last one before the
preceding kernel has finished.  The preceding kernel here is a KV write that
rewrites every row of every sequence's last page with fresh values, the most
a caller keeping the promise may write.  A last page fetched too early would
show stale rows.  Results must match the oracle on the pool after the write,
and the plain decode bit for bit (the arithmetic is the same)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
import workloads
from gpu_util import ORACLE_DTYPE, bits, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
BS = 16


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.get_device_error()
    yield
    st, detail = pa.get_device_error()
    assert st == 0, f"unexpected device error {pa.STATUS.get(st, st)} at index {detail}"


def _last_page_rows(case):
    """Flat slots of every cached row of each sequence's last page (up to 16 per sequence)."""
    bt = case.block_tables.cpu().numpy()
    out = []
    for s, n in enumerate(case.context_lens.cpu().numpy()):
        j = np.arange((int(n) - 1) // BS * BS, int(n))
        out.append(bt[s, j // BS].astype(np.int64) * BS + j % BS)
    return np.concatenate(out)


def _write_then_decode(case, early, append=False, layer=0, seed=0):
    """A fresh copy of the pools; a write of fresh rows into every last page,
    then the decode on the same stream right behind it."""
    kc, vc = case.k_cache[layer].clone(), case.v_cache[layer].clone()
    slots = torch.from_numpy(_last_page_rows(case)).to(DEV)
    gen = torch.Generator(device=DEV).manual_seed(100 + seed)
    rows = lambda: torch.randn((slots.numel(), case.hkv, 128), generator=gen, device=DEV).to(kc.dtype)
    kr, vr = rows(), rows()
    torch.cuda.synchronize()
    pa.kv_cache_write(kr, vr, slots, kc, vc)
    if append:
        out = pa.paged_attn_decode_append(case.q[layer], case.k_new[layer], case.v_new[layer], kc, vc,
                                          case.block_tables, case.context_lens, case.scale,
                                          max_context_len=case.max_context_len, early_pages=early)
    else:
        out = pa.paged_attn_decode(case.q[layer], kc, vc, case.block_tables, case.context_lens, case.scale,
                                   max_context_len=case.max_context_len, early_pages=early)
    torch.cuda.synchronize()
    return out, kc, vc


def _check(case, out, kc, vc, what):
    ref = oracle.paged_attn_decode(bits(case.q[0]), bits(kc), bits(vc), case.block_tables.cpu().numpy(),
                                   case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    check_close(out, ref, what)


@pytest.mark.parametrize("hq,hkv,dtype", [(16, 8, "f16"), (32, 8, "bf16"), (8, 8, "bf16"), (16, 2, "f16")])
def test_early_pages_after_a_last_page_write(hq, hkv, dtype):
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 64, 100, 250, 511, 512, 700, 1024, 1023]
    case = workloads.build_case(f"early-{hq}x{hkv}-{dtype}", dtype, hq, hkv, seed=hq + hkv, device=DEV,
                                decode_lens=lens)
    assert pa.decode_kernel_launches(len(lens), hkv, case.max_context_len) == 1
    out, kc, vc = _write_then_decode(case, True)
    _check(case, out, kc, vc, case.name)
    plain, _, _ = _write_then_decode(case, False)
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))


def test_early_pages_on_the_qwen3_0_6b_step_every_layer():
    case = workloads.qwen3_0_6b_decode(device=DEV, n_layers=3)
    for layer in range(3):
        out, kc, vc = _write_then_decode(case, True, layer=layer, seed=layer)
        ref = oracle.paged_attn_decode(bits(case.q[layer]), bits(kc), bits(vc), case.block_tables.cpu().numpy(),
                                       case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
        check_close(out, ref, f"{case.name} layer {layer}")


def test_early_pages_with_the_fused_append():
    case = workloads.build_case("early-append", "f16", 16, 8, seed=31, device=DEV,
                                decode_lens=[3, 16, 17, 200, 513, 1000])
    out, kc, vc = _write_then_decode(case, True, append=True)
    # the append wrote each new token at ctx - 1 over the fresh rows
    kh, vh = bits(kc), bits(vc)
    assert oracle.kv_cache_write(kh, vh, bits(case.k_new[0]), bits(case.v_new[0]),
                                 case.slot_mapping.cpu().numpy()) == 0
    assert np.array_equal(kh, bits(kc)) and np.array_equal(vh, bits(vc))
    _check(case, out, kc, vc, case.name)


def test_early_pages_on_the_split_path():
    lens = [4096] * 40
    case = workloads.build_case("early-split", "bf16", 32, 8, seed=33, device=DEV, decode_lens=lens)
    assert pa.decode_kernel_launches(len(lens), 8, case.max_context_len) == 2
    out, kc, vc = _write_then_decode(case, True)
    _check(case, out, kc, vc, case.name)


def test_early_pages_reports_bad_lengths_and_block_ids():
    case = workloads.build_case("early-bad", "f16", 16, 8, seed=34, device=DEV, decode_lens=[40, 300, 77])
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    ctx = case.context_lens.clone()
    ctx[1] = 0
    bt = case.block_tables.clone()
    bt[2, 1] = case.num_blocks + 5
    out = torch.zeros_like(case.q[0])
    pa.paged_attn_decode(case.q[0], kc, vc, bt, ctx, case.scale, out=out, max_context_len=300, early_pages=True)
    torch.cuda.synchronize()
    st, _ = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"]
    assert torch.count_nonzero(out[1]) == 0
    ref = oracle.paged_attn_decode(bits(case.q[0]), bits(kc), bits(vc), case.block_tables.cpu().numpy(),
                                   case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    check_close(out[:1], ref[:1], "the valid sequence")


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("hq,hkv,dtype", [(16, 8, "f16"), (32, 8, "bf16"), (16, 2, "bf16")])
def test_early_pages_on_8bit_pools_after_a_last_page_write(fp8, hq, hkv, dtype):
    # every token quantised into an 8-bit pool; then the quantising write of
    # fresh rows into every last page directly ahead of the decode
    lens = [1, 2, 15, 16, 17, 33, 250, 512, 700, 1023]
    case = workloads.build_case(f"early8-{fp8}-{hq}x{hkv}", dtype, hq, hkv, seed=hq + 5 * hkv + fp8, device=DEV,
                                decode_lens=lens)
    bt = case.block_tables.cpu().numpy()
    allslots = np.concatenate([bt[s, np.arange(n) // BS].astype(np.int64) * BS + np.arange(n) % BS
                               for s, n in enumerate(case.context_lens.cpu().numpy())])
    sl = torch.from_numpy(allslots).to(DEV)
    kc, vc = case.k_cache[0], case.v_cache[0]
    krows = kc.view(-1, hkv, 128)[sl].contiguous()
    vrows = vc.view(-1, hkv, 128)[sl].contiguous()
    last = torch.from_numpy(_last_page_rows(case)).to(DEV)
    gen = torch.Generator(device=DEV).manual_seed(7)
    fresh = lambda: torch.randn((last.numel(), hkv, 128), generator=gen, device=DEV).to(kc.dtype)
    kf, vf = fresh(), fresh()
    alloc, write, decode = ((pa.alloc_pool_f8, pa.kv_cache_write_f8, pa.paged_attn_decode_f8) if fp8 else
                            (pa.alloc_pool_q8, pa.kv_cache_write_q8, pa.paged_attn_decode_q8))
    outs = []
    for early in (True, False):
        pool = alloc(case.num_blocks, hkv, DEV)
        write(krows, vrows, sl, *pool)
        torch.cuda.synchronize()
        write(kf, vf, last, *pool)
        outs.append(decode(case.q[0], *pool, case.block_tables, case.context_lens, case.scale,
                           max_context_len=case.max_context_len, early_pages=early))
        torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    host = tuple(t.cpu().numpy() for t in pool)
    ref = (oracle.paged_attn_decode_f8 if fp8 else oracle.paged_attn_decode_q8)(
        bits(case.q[0]), *host, bt, case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    check_close(outs[0], ref, case.name)
