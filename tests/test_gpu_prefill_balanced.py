"""GPU parity of the balanced chunked prefill (pa_paged_attn_prefill_chunk_ex):
one CTA per SM, each taking an equal share of all (query tile, key tile)
pairs; query tiles cut between CTAs are merged by the piece that arrives last,
counting arrivals in the caller's zero-filled workspace.  Every output is
checked against the fp64 oracle, and after every call the workspace's
counters must be zero again (the next call relies on it).  The cases cover the
mixed-step chunks, ragged chunks at every head ratio and both dtypes, long
prefixes (tiles cut into many pieces), sliding windows, many chunks, chunk
metadata errors, the fallback past 256 chunks, and calls in a row on one
workspace."""
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


def _counters_are_zero(ws, case, mcl):
    g = case.hq // case.hkv
    tq = 128 // g
    n = case.chunk_starts.numel() * case.hkv * ((mcl + tq - 1) // tq)
    return int(torch.count_nonzero(ws[:4 * n].view(torch.int32))) == 0


def _written(case):
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    kh, vh = oracle_write(case, 0)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh)
    return kc, vc


def _oracle(case, kc, vc, q=None, window=0):
    args = (bits(case.q_chunks[0] if q is None else q), bits(kc), bits(vc), case.chunk_starts.cpu().numpy(),
            case.chunk_lens.cpu().numpy(), case.chunk_block_tables.cpu().numpy(),
            case.chunk_context_lens.cpu().numpy(), case.scale)
    if window:
        return oracle.paged_attn_prefill_window(*args, window, ORACLE_DTYPE[case.dtype])
    return oracle.paged_attn_prefill(*args, ORACLE_DTYPE[case.dtype])


def _balanced(case, kc, vc, ws, mcl, q=None, window=0, out=None):
    out = pa.paged_attn_prefill_chunk_window(case.q_chunks[0] if q is None else q, case.chunk_starts,
                                             case.chunk_lens, kc, vc, case.chunk_block_tables,
                                             case.chunk_context_lens, case.scale, window, out=out,
                                             max_chunk_len=mcl, workspace=ws)
    torch.cuda.synchronize()
    return out


def _check(case, what, window=0, calls=1, mcl=None):
    kc, vc = _written(case)
    mcl = mcl or max(n for _, n in case.meta["chunks"])
    ws = pa.alloc_prefill_workspace(case.chunk_starts.numel(), case.hq, case.hkv, mcl, DEV)
    for i in range(calls):
        q = case.q_chunks[0]
        if i:  # other queries on the same workspace
            g = torch.Generator(device=DEV).manual_seed(300 + i)
            q = torch.randn(q.shape, generator=g, device=DEV).to(q.dtype)
        out = _balanced(case, kc, vc, ws, mcl, q=q, window=window)
        assert _counters_are_zero(ws, case, mcl), f"{what}: counters left set after call {i + 1}"
        check_close(out, _oracle(case, kc, vc, q=q, window=window), f"{what}, call {i + 1}")


def test_balanced_prefill_of_the_mixed_step_three_calls():
    _check(workloads.qwen3_0_6b_mixed_step(device=DEV), "mixed-step chunks", calls=3)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (16, 2), (64, 8)])
def test_balanced_prefill_ragged_chunks(dtype, hq, hkv):
    chunks = [(0, 1), (0, 15), (16, 16), (1, 17), (100, 63), (7, 64), (0, 65), (1000, 127), (5, 128),
              (129, 129), (0, 511), (1536, 512)]
    case = workloads.build_case(f"balanced-ragged-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=hq + 3 * hkv,
                                device=DEV, chunks=chunks)
    _check(case, case.name)


def test_balanced_prefill_long_prefixes_cut_into_many_pieces():
    # three query tiles over 6000- to 9000-token prefixes: each tile is cut among several CTAs
    case = workloads.build_case("balanced-long", "bf16", 32, 8, seed=51, device=DEV,
                                chunks=[(9000, 64), (6000, 33), (7777, 512)])
    _check(case, "long prefixes", calls=2)


@pytest.mark.parametrize("window", [1, 64, 200, 512, 1024])
def test_balanced_prefill_sliding_window(window):
    case = workloads.build_case(f"balanced-window-{window}", "bf16", 16, 8, seed=52, device=DEV,
                                chunks=[(0, 512), (512, 512), (1536, 512), (3000, 77)])
    _check(case, f"window {window}", window=window)


@pytest.mark.parametrize("start,hq", [(1000, 16), (300, 32), (4000, 8)])
def test_balanced_prefill_with_fewer_positions_than_sms(start, hq):
    # one short chunk over a long prefix: fewer work positions than SMs, so
    # every CTA takes at most one key tile and each query tile is cut into
    # one piece per key tile, all merged by the last to arrive
    case = workloads.build_case(f"balanced-few-{start}-{hq}", "bf16", hq, 8, seed=57, device=DEV,
                                chunks=[(start, 40)])
    _check(case, f"one 40-token chunk after {start}", calls=2)


def test_balanced_prefill_many_small_chunks():
    rng = np.random.default_rng(53)
    chunks = [(int(rng.integers(0, 900)), int(rng.integers(1, 40))) for _ in range(200)]
    case = workloads.build_case("balanced-many", "f16", 16, 8, seed=53, device=DEV, chunks=chunks)
    _check(case, "200 chunks", mcl=40)


def test_balanced_prefill_past_256_chunks_falls_back_to_the_plain_launch():
    rng = np.random.default_rng(54)
    chunks = [(int(rng.integers(0, 900)), int(rng.integers(1, 8))) for _ in range(300)]
    case = workloads.build_case("balanced-300", "f16", 16, 8, seed=54, device=DEV, chunks=chunks)
    _check(case, "300 chunks", mcl=8)


def test_balanced_prefill_equals_the_plain_launch_up_to_rounding():
    case = workloads.qwen3_0_6b_mixed_step(device=DEV)
    kc, vc = _written(case)
    ws = pa.alloc_prefill_workspace(3, case.hq, case.hkv, 512, DEV)
    bal = _balanced(case, kc, vc, ws, 512)
    plain = pa.paged_attn_prefill_chunk(case.q_chunks[0], case.chunk_starts, case.chunk_lens, kc, vc,
                                        case.chunk_block_tables, case.chunk_context_lens, case.scale,
                                        max_chunk_len=512)
    torch.cuda.synchronize()
    assert (bal.float() - plain.float()).abs().max().item() < 4e-3


def test_balanced_prefill_reports_bad_chunks_and_leaves_them_untouched():
    case = workloads.build_case("balanced-bad", "bf16", 16, 8, seed=55, device=DEV,
                                chunks=[(0, 40), (64, 30), (2000, 300)])
    kc, vc = _written(case)
    ctx = case.chunk_context_lens.clone()
    ctx[1] += 1                                      # context must be start + len
    out = torch.zeros_like(case.q_chunks[0])
    ws = pa.alloc_prefill_workspace(3, 16, 8, 300, DEV)
    pa.paged_attn_prefill_chunk(case.q_chunks[0], case.chunk_starts, case.chunk_lens, kc, vc,
                                case.chunk_block_tables, ctx, case.scale, out=out, max_chunk_len=300, workspace=ws)
    torch.cuda.synchronize()
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    assert torch.count_nonzero(out[40:70]) == 0
    assert _counters_are_zero(ws, case, 300)
    ref = _oracle(case, kc, vc)
    check_close(out[:40], ref[:40], "chunk before the bad one")
    check_close(out[70:], ref[70:], "chunk after the bad one")


def test_balanced_prefill_requires_its_workspace():
    case = workloads.build_case("balanced-nows", "bf16", 16, 8, seed=56, device=DEV, chunks=[(0, 40)])
    lib = pa.load_library()
    pool = pa.make_pool(case.k_cache[0], case.v_cache[0])
    import ctypes
    st = lib.pa_paged_attn_prefill_chunk_ex(
        case.q_chunks[0].data_ptr(), case.chunk_starts.data_ptr(), case.chunk_lens.data_ptr(), ctypes.byref(pool),
        case.chunk_block_tables.data_ptr(), case.chunk_block_tables.shape[1], case.chunk_context_lens.data_ptr(),
        1, 16, 40, 40, ctypes.c_float(case.scale), 0, case.q_chunks[0].data_ptr(), None, 0, None)
    assert st == pa.STATUS_CODE["PA_ERR_WORKSPACE"]
