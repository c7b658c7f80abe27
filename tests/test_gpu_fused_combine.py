"""GPU parity of the decode as one kernel over all SMs
(pa_paged_attn_decode_ex with PA_DECODE_ZEROED_WORKSPACE): pages are dealt
evenly to every warp the GPU holds and the last piece of each split
(sequence, KV head) to finish merges the pieces, counting arrivals in the
caller's zero-filled workspace.  Every result is checked against the fp64
oracle, and after every call the workspace's counters must be zero again
(the next call relies on it); calls in a row on one workspace, with other
lengths, check that no state leaks from one call into the next."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
import workloads
from gpu_util import ORACLE_DTYPE, bits, check_close, oracle_write

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.get_device_error()
    yield
    st, detail = pa.get_device_error()
    assert st == 0, f"unexpected device error {pa.STATUS.get(st, st)} at index {detail}"


def _counters_are_zero(ws, num_seqs, hkv):
    # the counters are the workspace's last block: one int32 per (sequence, KV head), 256-byte aligned
    n = (num_seqs * hkv * 4 + 255) // 256 * 256
    return int(torch.count_nonzero(ws[-n:].view(torch.int32))) == 0


def _oracle(case, q, kc, vc, ctx, bt=None):
    bt = case.block_tables if bt is None else bt
    return oracle.paged_attn_decode(bits(q), bits(kc), bits(vc), bt.cpu().numpy(), ctx.cpu().numpy(), case.scale,
                                    ORACLE_DTYPE[case.dtype])


def _written(case, layer=0):
    kc, vc = case.k_cache[layer].clone(), case.v_cache[layer].clone()
    pa.kv_cache_write(case.k_new[layer], case.v_new[layer], case.slot_mapping, kc, vc)
    kh, vh = oracle_write(case, layer)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh)
    return kc, vc


@pytest.mark.parametrize("cfg", [1, 2, 4, 5])
def test_one_launch_decode_on_the_workloads_twice(cfg):
    case = workloads.BY_INDEX[cfg](device=DEV)
    kc, vc = _written(case)
    S = case.q[0].shape[0]
    ws = pa.alloc_decode_workspace(S, case.hq, case.hkv, case.max_context_len, DEV)
    out = pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, case.context_lens, case.scale, workspace=ws,
                               max_context_len=case.max_context_len, zeroed_workspace=True)
    torch.cuda.synchronize()
    assert _counters_are_zero(ws, S, case.hkv)
    check_close(out, _oracle(case, case.q[0], kc, vc, case.context_lens), f"{case.name}, call 1")
    # the same workspace again: other queries, shorter lengths (so other split points)
    g = torch.Generator(device=DEV).manual_seed(7 + cfg)
    q2 = torch.randn(case.q[0].shape, generator=g, device=DEV).to(case.q[0].dtype)
    cut = torch.from_numpy(np.random.default_rng(cfg).integers(1, 30, size=S).astype(np.int32)).to(DEV)
    ctx2 = torch.clamp(case.context_lens - cut, min=1)
    out2 = pa.paged_attn_decode(q2, kc, vc, case.block_tables, ctx2, case.scale, workspace=ws,
                                max_context_len=case.max_context_len, zeroed_workspace=True)
    torch.cuda.synchronize()
    assert _counters_are_zero(ws, S, case.hkv)
    check_close(out2, _oracle(case, q2, kc, vc, ctx2), f"{case.name}, call 2")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (8, 8), (16, 2), (64, 8)])
def test_one_launch_decode_ragged_lengths(dtype, hq, hkv):
    lens = [1, 15, 16, 17, 33, 100, 250, 513, 1000, 2047, 4096, 31, 7]
    case = workloads.build_case(f"fused-ragged-{hq}-{hkv}", dtype, hq, hkv, seed=41, device=DEV, decode_lens=lens)
    kc, vc = _written(case)
    ws = pa.alloc_decode_workspace(len(lens), hq, hkv, case.max_context_len, DEV)
    out = pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, case.context_lens, case.scale, workspace=ws,
                               max_context_len=case.max_context_len, zeroed_workspace=True)
    torch.cuda.synchronize()
    assert _counters_are_zero(ws, len(lens), hkv)
    check_close(out, _oracle(case, case.q[0], kc, vc, case.context_lens), case.name)


def test_one_launch_decode_many_calls_in_a_row():
    # 12 calls on one workspace, lengths changing every call; each checked
    case = workloads.qwen3_0_6b_decode(device=DEV, n_layers=1)
    kc, vc = _written(case)
    S = case.q[0].shape[0]
    ws = pa.alloc_decode_workspace(S, case.hq, case.hkv, case.max_context_len, DEV)
    rng = np.random.default_rng(12)
    for i in range(12):
        ctx = torch.from_numpy(rng.integers(1, case.context_lens.cpu().numpy() + 1).astype(np.int32)).to(DEV)
        out = pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, ctx, case.scale, workspace=ws,
                                   max_context_len=case.max_context_len, zeroed_workspace=True, early_pages=True)
        torch.cuda.synchronize()
        assert _counters_are_zero(ws, S, case.hkv), f"call {i}"
        check_close(out, _oracle(case, case.q[0], kc, vc, ctx), f"call {i}")


@pytest.mark.parametrize("append", [False, True])
def test_one_launch_decode_with_early_pages_after_a_last_page_write(append):
    # the write just ahead rewrites every row of every last page; those pages
    # are fetched after the wait, the others before it
    case = workloads.build_case("fused-early", "bf16", 32, 8, seed=43, device=DEV,
                                decode_lens=[40, 300, 77, 1024, 16, 17, 2000, 513])
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    bt = case.block_tables.cpu().numpy()
    slots = []
    for s, n in enumerate(case.context_lens.cpu().numpy()):
        j = np.arange((int(n) - 1) // 16 * 16, int(n) - (1 if append else 0))
        slots.append(bt[s, j // 16].astype(np.int64) * 16 + j % 16)
    slots = torch.from_numpy(np.concatenate(slots)).to(DEV)
    g = torch.Generator(device=DEV).manual_seed(44)
    kr = torch.randn((slots.numel(), 8, 128), generator=g, device=DEV).to(kc.dtype)
    vr = torch.randn((slots.numel(), 8, 128), generator=g, device=DEV).to(kc.dtype)
    ws = pa.alloc_decode_workspace(8, 32, 8, case.max_context_len, DEV)
    torch.cuda.synchronize()
    pa.kv_cache_write(kr, vr, slots, kc, vc)
    if append:
        out = pa.paged_attn_decode_append(case.q[0], case.k_new[0], case.v_new[0], kc, vc, case.block_tables,
                                          case.context_lens, case.scale, workspace=ws,
                                          max_context_len=case.max_context_len, early_pages=True,
                                          zeroed_workspace=True)
    else:
        out = pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, case.context_lens, case.scale,
                                   workspace=ws, max_context_len=case.max_context_len, early_pages=True,
                                   zeroed_workspace=True)
    torch.cuda.synchronize()
    assert _counters_are_zero(ws, 8, 8)
    # the pool as the decode saw it: the rewritten last pages (and, with append, the new rows)
    check_close(out, _oracle(case, case.q[0], kc, vc, case.context_lens), case.name)


@pytest.mark.parametrize("fp8", [False, True])
def test_one_launch_decode_on_8bit_pools(fp8):
    case = workloads.qwen3_8b_decode(device=DEV)
    kc, vc = _written(case)
    bt_h, ctx_h = case.block_tables.cpu().numpy(), case.context_lens.cpu().numpy()
    slots = np.concatenate([bt_h[s, np.arange(n) // 16].astype(np.int64) * 16 + np.arange(n) % 16
                            for s, n in enumerate(ctx_h)])
    sl = torch.from_numpy(slots).to(DEV)
    rows_k, rows_v = kc.view(-1, 8, 128)[sl].contiguous(), vc.view(-1, 8, 128)[sl].contiguous()
    pool = (pa.alloc_pool_f8 if fp8 else pa.alloc_pool_q8)(case.num_blocks, 8, DEV)
    (pa.kv_cache_write_f8 if fp8 else pa.kv_cache_write_q8)(rows_k, rows_v, sl, *pool)
    ws = pa.alloc_decode_workspace(64, 32, 8, case.max_context_len, DEV)
    dec = pa.paged_attn_decode_f8 if fp8 else pa.paged_attn_decode_q8
    out = dec(case.q[0], *pool, case.block_tables, case.context_lens, case.scale, workspace=ws,
              max_context_len=case.max_context_len, zeroed_workspace=True)
    plain = dec(case.q[0], *pool, case.block_tables, case.context_lens, case.scale,
                max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    assert _counters_are_zero(ws, 64, 8)
    host = [t.cpu().numpy() for t in pool]
    ref = (oracle.paged_attn_decode_f8 if fp8 else oracle.paged_attn_decode_q8)(
        bits(case.q[0]), *host, bt_h, ctx_h, case.scale, ORACLE_DTYPE[case.dtype])
    check_close(out, ref, "one launch")
    check_close(plain, ref, "split + combine")


def test_one_launch_decode_reports_bad_lengths_and_block_ids():
    case = workloads.build_case("fused-bad", "f16", 16, 8, seed=45, device=DEV, decode_lens=[40, 300, 77, 900])
    kc, vc = _written(case)
    ctx = case.context_lens.clone()
    ctx[1] = 0
    bt = case.block_tables.clone()
    bt[2, 1] = case.num_blocks + 5
    out = torch.zeros_like(case.q[0])
    ws = pa.alloc_decode_workspace(4, 16, 8, 900, DEV)
    pa.paged_attn_decode(case.q[0], kc, vc, bt, ctx, case.scale, out=out, workspace=ws, max_context_len=900,
                         zeroed_workspace=True)
    torch.cuda.synchronize()
    st, _ = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"]
    assert torch.count_nonzero(out[1]) == 0
    assert _counters_are_zero(ws, 4, 8)
    ref = _oracle(case, case.q[0], kc, vc, case.context_lens)
    check_close(out[0], ref[0], "sequence before the bad ones")
    check_close(out[3], ref[3], "sequence after the bad ones")
