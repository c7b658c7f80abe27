"""Edge cases at the limits of the C-ABI: the largest batch a decode call
accepts (16384 sequences), single-KV-head pools (multi-query attention, head
ratios 1 to 8), many tiny prefill chunks in one call, and a chunk of the
maximum length 512 on a long prefix — each against the oracle."""
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


def _decode(case):
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    out = pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, case.context_lens, case.scale,
                               max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    kh, vh = oracle_write(case, 0)
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh)
    ref = oracle.paged_attn_decode(bits(case.q[0]), kh, vh, case.block_tables.cpu().numpy(),
                                   case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    check_close(out, ref, case.name)


def test_decode_of_the_largest_batch():
    rng = np.random.default_rng(3)
    lens = [int(x) for x in rng.integers(1, 40, size=16384)]
    _decode(workloads.build_case("max-batch", "bf16", 16, 8, seed=3, device=DEV, decode_lens=lens))


@pytest.mark.parametrize("hq", [1, 2, 4, 8])
def test_decode_with_a_single_kv_head(hq):
    lens = [1, 16, 17, 300, 2000, 5000]
    _decode(workloads.build_case(f"mqa-{hq}", "f16", hq, 1, seed=hq, device=DEV, decode_lens=lens))


def _prefill(case, mcl):
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    out = pa.paged_attn_prefill_chunk(case.q_chunks[0], case.chunk_starts, case.chunk_lens, kc, vc,
                                      case.chunk_block_tables, case.chunk_context_lens, case.scale,
                                      max_chunk_len=mcl)
    torch.cuda.synchronize()
    ref = oracle.paged_attn_prefill(bits(case.q_chunks[0]), bits(kc), bits(vc), case.chunk_starts.cpu().numpy(),
                                    case.chunk_lens.cpu().numpy(), case.chunk_block_tables.cpu().numpy(),
                                    case.chunk_context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    check_close(out, ref, case.name)


def test_prefill_of_many_tiny_chunks():
    rng = np.random.default_rng(4)
    chunks = [(int(s), int(n)) for s, n in zip(rng.integers(0, 300, size=120), rng.integers(1, 8, size=120))]
    _prefill(workloads.build_case("tiny-chunks", "bf16", 16, 8, seed=4, device=DEV, chunks=chunks), 7)


@pytest.mark.parametrize("hq,hkv", [(8, 1), (32, 8)])
def test_prefill_of_a_maximum_chunk_on_a_long_prefix(hq, hkv):
    case = workloads.build_case(f"max-chunk-{hq}x{hkv}", "bf16", hq, hkv, seed=5 + hq, device=DEV,
                                chunks=[(7777, 512)])
    _prefill(case, 512)
