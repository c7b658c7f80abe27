"""GPU parity of the KV write fused into the decode (pa_paged_attn_decode_append):
the same result as pa_kv_cache_write of each sequence's new token followed by
pa_paged_attn_decode ("Модуль 12: Финальный проект: мини-движок инференса",
qwen_serve/paged.py PagedKVCache.write then qwen_serve/model.py attention) —
pools bit-exact against the oracle's write, outputs bit-identical to the two
separate calls and within tolerance of the oracle, on both decode paths."""
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


def _both(case, bound=None, bt=None):
    bt = case.block_tables if bt is None else bt
    mcl = bound or case.max_context_len
    # fused
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    fused = pa.paged_attn_decode_append(case.q[0], case.k_new[0], case.v_new[0], kc, vc, bt, case.context_lens,
                                        case.scale, max_context_len=mcl)
    # separate
    kc2, vc2 = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc2, vc2)
    sep = pa.paged_attn_decode(case.q[0], kc2, vc2, bt, case.context_lens, case.scale, max_context_len=mcl)
    torch.cuda.synchronize()
    return fused, kc, vc, sep


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (16, 2), (64, 8)])
def test_append_matches_write_then_decode(dtype, hq, hkv):
    lens = [1, 2, 15, 16, 17, 31, 33, 64, 65, 250, 1000, 1023, 4097]
    case = workloads.build_case(f"append-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=hq + hkv, device=DEV,
                                decode_lens=lens)
    fused, kc, vc, sep = _both(case)
    kh, vh = oracle_write(case, 0)
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh), "pool after the fused write"
    assert torch.equal(fused.view(torch.int16), sep.view(torch.int16)), "fused differs from write + decode"
    ref = oracle.paged_attn_decode(bits(case.q[0]), kh, vh, case.block_tables.cpu().numpy(),
                                   case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[dtype])
    check_close(fused, ref, case.name)


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8)])
def test_append_on_both_decode_paths(hq, hkv):
    lens = [700, 1024, 3]
    case = workloads.build_case("append-paths", "bf16", hq, hkv, seed=5 + hq, device=DEV, decode_lens=lens)
    wide = torch.full((3, 1024), -1, dtype=torch.int32, device=DEV)
    wide[:, :case.block_tables.shape[1]] = case.block_tables
    assert pa.decode_kernel_launches(3, hkv, max(lens)) == 1 and pa.decode_kernel_launches(3, hkv, 16384) == 2
    kh, vh = oracle_write(case, 0)
    for bound in (max(lens), 16384):
        fused, kc, vc, sep = _both(case, bound=bound, bt=wide)
        assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh), f"pool, bound {bound}"
        assert torch.equal(fused.view(torch.int16), sep.view(torch.int16)), f"bound {bound}"


def test_append_of_the_qwen3_0_6b_step_and_the_8b_decode():
    for case in (workloads.qwen3_0_6b_decode(device=DEV, n_layers=1), workloads.qwen3_8b_decode(device=DEV)):
        fused, kc, vc, sep = _both(case)
        assert torch.equal(fused.view(torch.int16), sep.view(torch.int16)), case.name
        kh, vh = oracle_write(case, 0)
        assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh), case.name
        del kc, vc


def test_append_skips_a_sequence_with_a_bad_length():
    case = workloads.build_case("append-bad", "f16", 16, 8, seed=9, device=DEV, decode_lens=[40, 70])
    ctx = case.context_lens.clone()
    ctx[1] = 0
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    before = bits(kc)
    pa.paged_attn_decode_append(case.q[0], case.k_new[0], case.v_new[0], kc, vc, case.block_tables, ctx,
                                case.scale, max_context_len=70)
    torch.cuda.synchronize()
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    slots = case.slot_mapping.cpu().numpy()
    after = bits(kc).reshape(-1, 8, 128)
    assert np.array_equal(after[slots[0]], bits(case.k_new[0])[0])            # sequence 0 written
    assert np.array_equal(after[slots[1]], before.reshape(-1, 8, 128)[slots[1]])   # sequence 1 untouched
