"""GPU parity of the fp8 KV pool ("Модуль 04: KV-кэш и арифметика памяти",
sections 5.1 and 5.4: K and V stored as FP8 E4M3 with one fp32 scale per token
and KV head) through the C-ABI: the quantising write is bit-exact against the
oracle (codes and scales), and decode over the fp8 pool matches the oracle's
decode on the dequantised values within the attention tolerance, on both
decode paths."""
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


def _host_pool(nb, hkv):
    return (np.zeros((nb, BS, hkv, 128), np.uint8), np.zeros((nb, BS, hkv, 128), np.uint8),
            np.zeros((nb, hkv, BS), np.float32), np.zeros((nb, hkv, BS), np.float32))


def _quantised_pools(case, layer=0):
    """Every token of the step (cached and new) quantised into an fp8 pool on
    the GPU and, from the same rows, by the oracle."""
    kc, vc = case.k_cache[layer].clone(), case.v_cache[layer].clone()
    pa.kv_cache_write(case.k_new[layer], case.v_new[layer], case.slot_mapping, kc, vc)
    slots = _token_slots(case)
    sl = torch.from_numpy(slots).to(DEV)
    krows = kc.view(-1, case.hkv, 128)[sl].contiguous()
    vrows = vc.view(-1, case.hkv, 128)[sl].contiguous()
    gpu = pa.alloc_pool_f8(case.num_blocks, case.hkv, DEV)
    pa.kv_cache_write_f8(krows, vrows, sl, *gpu)
    host = _host_pool(case.num_blocks, case.hkv)
    assert oracle.kv_cache_write_f8(*host, bits(krows), bits(vrows), ORACLE_DTYPE[case.dtype], slots) == 0
    torch.cuda.synchronize()
    return gpu, host


def _check_write(gpu, host, what):
    for g, h, name in zip(gpu, host, ("k codes", "v codes", "k scales", "v scales")):
        gn = g.cpu().numpy()
        if gn.dtype == np.float32:
            assert np.array_equal(gn.view(np.uint32), h.view(np.uint32)), f"{what}: {name} not bit-exact"
        else:
            bad = np.flatnonzero(gn != h)
            assert bad.size == 0, f"{what}: {name} differ at {bad.size} places, first {bad[:4]}"


def _decode_and_check(case, gpu, host, bound=None, bt=None, what=""):
    bt_dev = case.block_tables if bt is None else bt
    out = pa.paged_attn_decode_f8(case.q[0], *gpu, bt_dev, case.context_lens, case.scale,
                                  max_context_len=bound or case.max_context_len)
    torch.cuda.synchronize()
    ref = oracle.paged_attn_decode_f8(bits(case.q[0]), *host, case.block_tables.cpu().numpy(),
                                      case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    return check_close(out, ref, what or case.name)


def test_f8_tiny_workload():
    case = workloads.tiny_decode(device=DEV)
    gpu, host = _quantised_pools(case)
    _check_write(gpu, host, case.name)
    _decode_and_check(case, gpu, host)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (16, 2)])
def test_f8_ragged_lengths(dtype, hq, hkv):
    lens = [1, 2, 15, 16, 17, 31, 33, 64, 65, 250, 1000, 1023, 4097]
    case = workloads.build_case(f"f8-ragged-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=hq * 37 + hkv,
                                device=DEV, decode_lens=lens)
    gpu, host = _quantised_pools(case)
    _check_write(gpu, host, case.name)
    _decode_and_check(case, gpu, host)


@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 16, 8), ("f16", 32, 8), ("bf16", 64, 8)])
def test_f8_one_launch_and_split_paths(dtype, hq, hkv):
    lens = [700, 1024]
    case = workloads.build_case(f"f8-paths-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=43 + hq, device=DEV,
                                decode_lens=lens)
    gpu, host = _quantised_pools(case)
    wide = torch.full((2, 1024), -1, dtype=torch.int32, device=DEV)
    wide[:, :case.block_tables.shape[1]] = case.block_tables
    assert pa.decode_kernel_launches(2, hkv, max(lens)) == 1
    assert pa.decode_kernel_launches(2, hkv, 16384) == 2
    for bound in (max(lens), 16384):
        _decode_and_check(case, gpu, host, bound=bound, bt=wide, what=f"{case.name}, bound {bound}")


def test_f8_qwen3_8b_geometry():
    case = workloads.qwen3_8b_decode(device=DEV)
    gpu, host = _quantised_pools(case)
    _check_write(gpu, host, case.name)
    _decode_and_check(case, gpu, host)


def test_f8_large_magnitudes_subnormal_codes_and_zero_rows():
    # elements shrunk by up to e^-5|z| (many quotients land in E4M3's subnormal
    # range, below 2^-6), whole rows scaled by e^(2z) (scales far from 1), zero
    # rows, and one large element that sets its row's scale
    case = workloads.build_case("f8-magnitudes", "bf16", 16, 8, seed=79, device=DEV, decode_lens=[40, 300])
    gen = torch.Generator(device=DEV).manual_seed(6)
    for pool in (case.k_cache[0], case.v_cache[0]):
        shrink = torch.exp(-5 * torch.randn(pool.shape, generator=gen, device=DEV).abs())
        rows = torch.exp(2 * torch.randn(pool.shape[:3], generator=gen, device=DEV))[..., None]
        pool.copy_((pool.float() * shrink * rows).to(pool.dtype))
        pool[:, 3] = 0          # slot 3 of every block: an all-zero row
        pool[:, 5, :, 0] = 64   # slot 5: one element well above the rest of its row
    gpu, host = _quantised_pools(case)
    _check_write(gpu, host, case.name)
    codes = gpu[0].cpu().numpy()
    assert np.count_nonzero(((codes & 0x78) == 0) & ((codes & 7) != 0)) > 1000, "expected subnormal codes"
    _decode_and_check(case, gpu, host)


def test_f8_codes_are_never_nan():
    case = workloads.build_case("f8-nan-free", "f16", 32, 8, seed=80, device=DEV, decode_lens=[513, 77])
    gpu, host = _quantised_pools(case)
    for codes in gpu[:2]:
        c = codes.cpu().numpy()
        assert not np.any((c & 0x7f) == 0x7f)


def test_f8_write_bad_slot_is_reported_and_skipped():
    k = torch.randn((3, 8, 128), device=DEV).to(torch.float16)
    gpu = pa.alloc_pool_f8(4, 8, DEV)
    slots = torch.tensor([5, 4 * BS, 17], dtype=torch.int64, device=DEV)
    pa.kv_cache_write_f8(k, k, slots, *gpu)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    host = _host_pool(4, 8)
    assert oracle.kv_cache_write_f8(*host, bits(k), bits(k), oracle.F16, slots.cpu().numpy()) == 1
    _check_write(gpu, host, "bad slot")


def test_f8_rejects_an_int8_pool():
    gpu = pa.alloc_pool_q8(4, 8, DEV)
    k = torch.zeros((1, 8, 128), device=DEV, dtype=torch.float16)
    with pytest.raises(TypeError):
        pa.kv_cache_write_f8(k, k, torch.zeros(1, dtype=torch.int64, device=DEV), *gpu)
