"""GPU parity of sliding-window attention ("Модуль 04: KV-кэш и арифметика
памяти", section 4: the last W tokens stay visible and the mask compares
absolute positions; section 5.2: window attention) through the C-ABI: decode
on both decode paths and chunked prefill against the oracle's window
functions, windows from one key to longer than the context, and blocks
wholly before the window freed (-1 in the table) or holding NaN."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
import workloads
from gpu_util import ORACLE_DTYPE, bits, check_close, oracle_write

pytestmark = pytest.mark.gpu
DEV = "cuda"
BS = 16
LENS = [1, 2, 15, 16, 17, 31, 33, 64, 65, 250, 1000, 1023, 4097]
CHUNKS = [(0, 1), (0, 15), (16, 16), (1, 17), (100, 63), (7, 64), (0, 65), (1000, 127), (5, 128),
          (129, 129), (0, 511), (1536, 512)]


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.get_device_error()
    yield
    st, detail = pa.get_device_error()
    assert st == 0, f"unexpected device error {pa.STATUS.get(st, st)} at index {detail}"


def _written(case):
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    torch.cuda.synchronize()
    kh, vh = oracle_write(case, 0)
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh)
    return kc, vc


def _free_before(bt, kc, vc, first_key):
    """A copy of the block table with every block wholly before first_key[s]
    freed (-1), those blocks filled with NaN in the pools."""
    freed = bt.clone()
    host = bt.cpu().numpy()
    for s, lo in enumerate(first_key):
        for pg in range(int(lo) // BS):
            b = int(host[s, pg])
            kc[b] = float("nan")
            vc[b] = float("nan")
            freed[s, pg] = -1
    return freed


def _decode_case(name, dtype, hq, hkv, seed, lens=LENS):
    return workloads.build_case(name, dtype, hq, hkv, seed=seed, device=DEV, decode_lens=lens)


def _decode_check(case, kc, vc, window, bt=None, bound=None, what=""):
    bt_dev = case.block_tables if bt is None else bt
    out = pa.paged_attn_decode_window(case.q[0], kc, vc, bt_dev, case.context_lens, case.scale, window,
                                      max_context_len=bound or case.meta["max_context_len"])
    torch.cuda.synchronize()
    ref = oracle.paged_attn_decode_window(bits(case.q[0]), bits(kc), bits(vc), case.block_tables.cpu().numpy(),
                                          case.context_lens.cpu().numpy(), case.scale, window,
                                          ORACLE_DTYPE[case.dtype])
    check_close(out, ref, what or f"{case.name}, window {window}")
    return out


@pytest.mark.parametrize("window", [1, 5, 16, 100, 128, 200, 1000])
@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 16, 8), ("f16", 32, 8), ("bf16", 8, 8), ("f16", 16, 2)])
def test_decode_window_ragged(window, dtype, hq, hkv):
    case = _decode_case(f"win-decode-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=window + hq)
    kc, vc = _written(case)
    _decode_check(case, kc, vc, window)


@pytest.mark.parametrize("window", [7, 100, 600])
def test_decode_window_on_both_paths(window):
    lens = [700, 1024]
    case = _decode_case("win-paths", "bf16", 16, 8, seed=91 + window, lens=lens)
    kc, vc = _written(case)
    wide = torch.full((2, 1024), -1, dtype=torch.int32, device=DEV)
    wide[:, :case.block_tables.shape[1]] = case.block_tables
    assert pa.decode_kernel_launches(2, 8, max(lens)) == 1 and pa.decode_kernel_launches(2, 8, 16384) == 2
    for bound in (max(lens), 16384):
        _decode_check(case, kc, vc, window, bt=wide, bound=bound, what=f"window {window}, bound {bound}")


@pytest.mark.parametrize("bound", [None, 16384])
def test_decode_never_reads_blocks_before_the_window(bound):
    window = 40
    case = _decode_case("win-freed", "bf16", 16, 8, seed=5)
    kc, vc = _written(case)
    wide = torch.full((len(LENS), 1024), -1, dtype=torch.int32, device=DEV)
    wide[:, :case.block_tables.shape[1]] = case.block_tables
    ref = _decode_check(case, kc, vc, window, bt=wide, bound=bound).clone()
    first = [max(0, n - window) for n in LENS]
    freed = _free_before(wide, kc, vc, first)
    out = pa.paged_attn_decode_window(case.q[0], kc, vc, freed, case.context_lens, case.scale, window,
                                      max_context_len=bound or max(LENS))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_decode_window_as_long_as_the_context_is_the_plain_call():
    case = _decode_case("win-full", "f16", 16, 8, seed=6)
    kc, vc = _written(case)
    plain = pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, case.context_lens, case.scale)
    for window in (0, max(LENS), 10 ** 6):
        got = pa.paged_attn_decode_window(case.q[0], kc, vc, case.block_tables, case.context_lens, case.scale,
                                          window)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), plain.view(torch.int16)), window


def _prefill(case, kc, vc, window, bt=None):
    out = pa.paged_attn_prefill_chunk_window(case.q_chunks[0], case.chunk_starts, case.chunk_lens, kc, vc,
                                             case.chunk_block_tables if bt is None else bt,
                                             case.chunk_context_lens, case.scale, window,
                                             max_chunk_len=max(n for _, n in case.meta["chunks"]))
    torch.cuda.synchronize()
    return out


def _prefill_ref(case, kc, vc, window):
    return oracle.paged_attn_prefill_window(bits(case.q_chunks[0]), bits(kc), bits(vc),
                                            case.chunk_starts.cpu().numpy(), case.chunk_lens.cpu().numpy(),
                                            case.chunk_block_tables.cpu().numpy(),
                                            case.chunk_context_lens.cpu().numpy(), case.scale, window,
                                            ORACLE_DTYPE[case.dtype])


@pytest.mark.parametrize("window", [1, 7, 64, 127, 128, 129, 200, 1000])
@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 16, 8), ("f16", 32, 8), ("bf16", 8, 8), ("f16", 16, 2)])
def test_prefill_window_ragged(window, dtype, hq, hkv):
    case = workloads.build_case(f"win-prefill-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=window + 3 * hq,
                                device=DEV, chunks=CHUNKS)
    kc, vc = _written(case)
    check_close(_prefill(case, kc, vc, window), _prefill_ref(case, kc, vc, window),
                f"{case.name}, window {window}")


@pytest.mark.parametrize("window", [3, 100, 300])
def test_prefill_never_reads_blocks_before_the_window(window):
    case = workloads.build_case("win-prefill-freed", "bf16", 16, 8, seed=17, device=DEV, chunks=CHUNKS)
    kc, vc = _written(case)
    ref = _prefill(case, kc, vc, window).clone()
    # blocks wholly before the first query's window of each chunk
    first = [max(0, s - window + 1) for s, _ in CHUNKS]
    freed = _free_before(case.chunk_block_tables, kc, vc, first)
    out = _prefill(case, kc, vc, window, bt=freed)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_prefill_window_as_long_as_the_context_is_the_plain_call():
    case = workloads.build_case("win-prefill-full", "bf16", 32, 8, seed=18, device=DEV, chunks=CHUNKS)
    kc, vc = _written(case)
    plain = pa.paged_attn_prefill_chunk(case.q_chunks[0], case.chunk_starts, case.chunk_lens, kc, vc,
                                        case.chunk_block_tables, case.chunk_context_lens, case.scale,
                                        max_chunk_len=512)
    for window in (0, 2048, 10 ** 6):
        got = _prefill(case, kc, vc, window)
        assert torch.equal(got.view(torch.int16), plain.view(torch.int16)), window


def test_decode_window_on_the_qwen3_8b_workload():
    # the full Qwen3-8B decode (64 x 4096, bf16, exactly full pool) under a 1024-key window, as the bench runs it
    case = workloads.qwen3_8b_decode(device=DEV)
    kc, vc = _written(case)
    assert pa.decode_kernel_launches(64, 8, 4096, 1024) == 2
    _decode_check(case, kc, vc, 1024)


def test_prefill_window_on_the_mixed_step_chunks():
    case = workloads.qwen3_0_6b_mixed_step(device=DEV)
    kc, vc = _written(case)
    check_close(_prefill(case, kc, vc, 512), _prefill_ref(case, kc, vc, 512), "mixed-step chunks, window 512")
