"""GPU parity of the int8 KV pool ("Модуль 04: KV-кэш и арифметика памяти",
section 5, KV8Cache: int8 codes with one fp32 scale per token and KV head)
through the C-ABI: the quantising write is bit-exact against the oracle (codes
and scales), and decode over the int8 pool matches the oracle's decode on the
dequantised values within the attention tolerance, on both decode paths."""
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


def _token_slots(case):
    """Flat slots of every position [0, ctx) of every decode sequence."""
    bt = case.block_tables.cpu().numpy()
    out = []
    for s, n in enumerate(case.context_lens.cpu().numpy()):
        j = np.arange(int(n))
        out.append(bt[s, j // BS].astype(np.int64) * BS + j % BS)
    return np.concatenate(out)


def _quantised_pools(case, layer=0):
    """Every token of the step (cached and new) quantised into an int8 pool on
    the GPU and, from the same rows, by the oracle."""
    kc, vc = case.k_cache[layer].clone(), case.v_cache[layer].clone()
    pa.kv_cache_write(case.k_new[layer], case.v_new[layer], case.slot_mapping, kc, vc)
    slots = _token_slots(case)
    sl = torch.from_numpy(slots).to(DEV)
    krows = kc.view(-1, case.hkv, 128)[sl].contiguous()
    vrows = vc.view(-1, case.hkv, 128)[sl].contiguous()
    gpu = pa.alloc_pool_q8(case.num_blocks, case.hkv, DEV)
    pa.kv_cache_write_q8(krows, vrows, sl, *gpu)
    host = (np.zeros((case.num_blocks, BS, case.hkv, 128), np.int8),
            np.zeros((case.num_blocks, BS, case.hkv, 128), np.int8),
            np.zeros((case.num_blocks, case.hkv, BS), np.float32),
            np.zeros((case.num_blocks, case.hkv, BS), np.float32))
    assert oracle.kv_cache_write_q8(*host, bits(krows), bits(vrows), ORACLE_DTYPE[case.dtype], slots) == 0
    torch.cuda.synchronize()
    return gpu, host


def _check_write(gpu, host, what):
    for g, h, name in zip(gpu, host, ("k codes", "v codes", "k scales", "v scales")):
        gn = g.cpu().numpy()
        if gn.dtype == np.float32:
            assert np.array_equal(gn.view(np.uint32), h.view(np.uint32)), f"{what}: {name} not bit-exact"
        else:
            assert np.array_equal(gn, h), f"{what}: {name} not bit-exact"


def _decode_and_check(case, gpu, host, bound=None, bt=None, what=""):
    bt_dev = case.block_tables if bt is None else bt
    out = pa.paged_attn_decode_q8(case.q[0], *gpu, bt_dev, case.context_lens, case.scale,
                                  max_context_len=bound or case.max_context_len)
    torch.cuda.synchronize()
    ref = oracle.paged_attn_decode_q8(bits(case.q[0]), *host, case.block_tables.cpu().numpy(),
                                      case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    return check_close(out, ref, what or case.name)


def test_q8_tiny_workload():
    case = workloads.tiny_decode(device=DEV)
    gpu, host = _quantised_pools(case)
    _check_write(gpu, host, case.name)
    _decode_and_check(case, gpu, host)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (16, 2)])
def test_q8_ragged_lengths(dtype, hq, hkv):
    lens = [1, 2, 15, 16, 17, 31, 33, 64, 65, 250, 1000, 1023, 4097]
    case = workloads.build_case(f"q8-ragged-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=hq * 31 + hkv,
                                device=DEV, decode_lens=lens)
    gpu, host = _quantised_pools(case)
    _check_write(gpu, host, case.name)
    _decode_and_check(case, gpu, host)


@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 16, 8), ("f16", 32, 8)])
def test_q8_one_launch_and_split_paths(dtype, hq, hkv):
    lens = [700, 1024]
    case = workloads.build_case(f"q8-paths-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=41 + hq, device=DEV,
                                decode_lens=lens)
    gpu, host = _quantised_pools(case)
    wide = torch.full((2, 1024), -1, dtype=torch.int32, device=DEV)
    wide[:, :case.block_tables.shape[1]] = case.block_tables
    assert pa.decode_kernel_launches(2, hkv, max(lens)) == 1
    assert pa.decode_kernel_launches(2, hkv, 16384) == 2
    for bound in (max(lens), 16384):
        _decode_and_check(case, gpu, host, bound=bound, bt=wide, what=f"{case.name}, bound {bound}")


def test_q8_qwen3_8b_geometry():
    case = workloads.qwen3_8b_decode(device=DEV)
    gpu, host = _quantised_pools(case)
    _check_write(gpu, host, case.name)
    _decode_and_check(case, gpu, host)


def test_q8_large_magnitudes_and_zero_rows():
    # rows far from N(0, 1): large and tiny magnitudes, exact zeros
    case = workloads.build_case("q8-magnitudes", "bf16", 16, 8, seed=77, device=DEV, decode_lens=[40, 300])
    gen = torch.Generator(device=DEV).manual_seed(5)
    for pool in (case.k_cache[0], case.v_cache[0]):
        scale = torch.exp(torch.randn(pool.shape[:3], generator=gen, device=DEV) * 4)[..., None]
        pool.copy_((pool.float() * scale).to(pool.dtype))
        pool[:, 3] = 0          # slot 3 of every block: an all-zero row
    gpu, host = _quantised_pools(case)
    _check_write(gpu, host, case.name)
    _decode_and_check(case, gpu, host)


def test_q8_write_bad_slot_is_reported_and_skipped():
    k = torch.randn((3, 8, 128), device=DEV).to(torch.float16)
    gpu = pa.alloc_pool_q8(4, 8, DEV)
    slots = torch.tensor([5, 4 * BS, 17], dtype=torch.int64, device=DEV)
    pa.kv_cache_write_q8(k, k, slots, *gpu)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    host = (np.zeros((4, BS, 8, 128), np.int8), np.zeros((4, BS, 8, 128), np.int8),
            np.zeros((4, 8, BS), np.float32), np.zeros((4, 8, BS), np.float32))
    assert oracle.kv_cache_write_q8(*host, bits(k), bits(k), oracle.F16, slots.cpu().numpy()) == 1
    _check_write(gpu, host, "bad slot")
