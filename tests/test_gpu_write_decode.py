"""GPU parity of kv_cache_write (bit-exact) and paged decode (within tolerance)
against the fp64 oracle, through the C-ABI, on the five workloads and on
ragged edge cases."""
import math

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


def gpu_write(case, layer):
    kc, vc = case.k_cache[layer].clone(), case.v_cache[layer].clone()
    pa.kv_cache_write(case.k_new[layer], case.v_new[layer], case.slot_mapping, kc, vc)
    return kc, vc


def decode_and_check(case, layer=0, what=""):
    kc, vc = gpu_write(case, layer)
    kh, vh = oracle_write(case, layer)
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh), f"{what}: write not bit-exact"
    out = pa.paged_attn_decode(case.q[layer], kc, vc, case.block_tables, case.context_lens, case.scale,
                               max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    ref = oracle.paged_attn_decode(bits(case.q[layer]), kh, vh, case.block_tables.cpu().numpy(),
                                   case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    return check_close(out, ref, what or case.name), out, (kc, vc)


# ---- kv_cache_write ----------------------------------------------------------------

@pytest.mark.parametrize("cfg", [1, 3])
def test_write_bit_exact_whole_pool(cfg):
    case = workloads.BY_INDEX[cfg](device=DEV)
    kc, vc = gpu_write(case, 0)
    torch.cuda.synchronize()
    kh, vh = oracle_write(case, 0)
    assert np.array_equal(bits(kc), kh)
    assert np.array_equal(bits(vc), vh)


def test_write_all_layers_of_the_decode_step():
    case = workloads.qwen3_0_6b_decode(device=DEV)
    for layer in (0, 13, 27):
        kc, vc = gpu_write(case, layer)
        kh, vh = oracle_write(case, layer)
        assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh)


def test_write_empty_and_bad_slot():
    case = workloads.tiny_decode(device=DEV)
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    before = bits(kc)
    empty = torch.empty(0, 8, 128, dtype=kc.dtype, device=DEV)
    pa.kv_cache_write(empty, empty, torch.empty(0, dtype=torch.int64, device=DEV), kc, vc)
    torch.cuda.synchronize()
    assert np.array_equal(bits(kc), before)
    slots = case.slot_mapping.clone()
    slots[2] = 64 * 16            # one past the pool
    pa.kv_cache_write(case.k_new[0], case.v_new[0], slots, kc, vc)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 2
    kh, vh = bits(case.k_cache[0]), bits(case.v_cache[0])
    keep = [0, 1, 3]
    oracle.kv_cache_write(kh, vh, bits(case.k_new[0])[keep], bits(case.v_new[0])[keep],
                          case.slot_mapping.cpu().numpy()[keep])
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh)


# ---- decode: the five workloads ------------------------------------------------------

def test_decode_tiny_workload():
    decode_and_check(workloads.tiny_decode(device=DEV))


def test_decode_qwen3_0_6b_step_layers():
    case = workloads.qwen3_0_6b_decode(device=DEV)
    for layer in (0, 27):
        decode_and_check(case, layer, f"{case.name} layer {layer}")


def test_decode_part_of_mixed_step():
    decode_and_check(workloads.qwen3_0_6b_mixed_step(device=DEV))


def test_decode_qwen3_8b_full():
    decode_and_check(workloads.qwen3_8b_decode(device=DEV))


def test_decode_prefix_shared_long_tail():
    decode_and_check(workloads.prefix_shared_tail(device=DEV))


# ---- decode: ragged edges, head ratios, dtypes ------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (16, 2)])
def test_decode_ragged_lengths(dtype, hq, hkv):
    lens = [1, 2, 15, 16, 17, 31, 33, 64, 65, 250, 1000, 1023, 4097]
    case = workloads.build_case(f"ragged-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=hq * 100 + hkv,
                                device=DEV, decode_lens=lens)
    decode_and_check(case)


def test_decode_single_key_returns_its_value_bits():
    case = workloads.build_case("ctx1", "bf16", 32, 8, seed=21, device=DEV, decode_lens=[1] * 5)
    _, out, (kc, vc) = decode_and_check(case)
    bt = case.block_tables[:, 0].long()
    v0 = vc[bt, 0]                                   # [S, Hkv, 128]
    ref = v0.repeat_interleave(4, dim=1)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_decode_one_sequence_per_many_workers_and_many_per_worker():
    # one very long sequence (many fragments) and many tiny ones (many items per warp)
    decode_and_check(workloads.build_case("long1", "bf16", 32, 8, seed=22, device=DEV, decode_lens=[32768]))
    decode_and_check(workloads.build_case("tiny4096", "f16", 16, 8, seed=23, device=DEV,
                                          decode_lens=list(np.random.default_rng(0).integers(1, 40, 4096))))


def test_decode_block_permutation_is_bitwise_invariant():
    a = workloads.build_case("perm-a", "bf16", 16, 8, seed=31, device=DEV, decode_lens=[100, 700, 33, 2000])
    kc, vc = gpu_write(a, 0)
    out_a = pa.paged_attn_decode(a.q[0], kc, vc, a.block_tables, a.context_lens, a.scale,
                                 max_context_len=a.max_context_len)
    # move every block to a new physical id
    perm = torch.randperm(a.num_blocks, generator=torch.Generator().manual_seed(5)).to(DEV)
    kc2, vc2 = torch.empty_like(kc), torch.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = torch.where(a.block_tables >= 0, perm[a.block_tables.long().clamp(min=0)].int(), a.block_tables)
    out_b = pa.paged_attn_decode(a.q[0], kc2, vc2, bt2.contiguous(), a.context_lens, a.scale,
                                 max_context_len=a.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))


def test_decode_shared_prefix_equals_private_copies():
    a = workloads.prefix_shared_tail(device=DEV)
    kc, vc = gpu_write(a, 0)
    out_shared = pa.paged_attn_decode(a.q[0], kc, vc, a.block_tables, a.context_lens, a.scale,
                                      max_context_len=a.max_context_len)
    # give every sequence a private copy of the 13 shared prefix blocks
    S = a.block_tables.shape[0]
    extra = 13 * (S - 1)
    kc2 = torch.cat([kc, torch.empty((extra,) + tuple(kc.shape[1:]), dtype=kc.dtype, device=DEV)])
    vc2 = torch.cat([vc, torch.empty((extra,) + tuple(vc.shape[1:]), dtype=vc.dtype, device=DEV)])
    bt2 = a.block_tables.clone()
    nxt = a.num_blocks
    for s in range(1, S):
        for j in range(13):
            kc2[nxt], vc2[nxt] = kc[a.block_tables[s, j]], vc[a.block_tables[s, j]]
            bt2[s, j] = nxt
            nxt += 1
    assert len(set(bt2[:, :13].flatten().tolist())) == 13 * S
    out_private = pa.paged_attn_decode(a.q[0], kc2, vc2, bt2, a.context_lens, a.scale,
                                       max_context_len=a.max_context_len)
    torch.cuda.synchronize()
    assert torch.equal(out_shared.view(torch.int16), out_private.view(torch.int16))
    assert torch.equal(kc[a.block_tables[0, :13].long()].view(torch.int16),
                       kc2[a.block_tables[0, :13].long()].view(torch.int16))


def test_decode_launch_size_changes_only_rounding():
    case = workloads.build_case("split", "bf16", 32, 8, seed=41, device=DEV, decode_lens=[3000, 17, 900, 4500])
    kc, vc = gpu_write(case, 0)
    outs = []
    for mcl in (case.max_context_len, case.block_tables.shape[1] * 16, 4500):
        outs.append(pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, case.context_lens, case.scale,
                                         max_context_len=mcl).float())
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 4e-3


# ---- decode: data errors are reported, never faulted -----------------------------------------

def test_decode_bad_block_id_and_bad_length_are_reported():
    case = workloads.build_case("bad", "f16", 16, 8, seed=51, device=DEV, decode_lens=[40, 50, 60])
    kc, vc = gpu_write(case, 0)
    bt = case.block_tables.clone()
    bt[1, 2] = case.num_blocks + 1000            # outside the pool
    out = torch.zeros_like(case.q[0])
    pa.paged_attn_decode(case.q[0], kc, vc, bt, case.context_lens, case.scale, out=out,
                         max_context_len=case.max_context_len)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    ref = oracle.paged_attn_decode(bits(case.q[0]), bits(kc), bits(vc), case.block_tables.cpu().numpy(),
                                   case.context_lens.cpu().numpy(), case.scale, oracle.F16)
    check_close(out[0], ref[0], "sequence before the bad one")
    check_close(out[2], ref[2], "sequence after the bad one")

    ctx = case.context_lens.clone()
    ctx[2] = 0
    out = torch.zeros_like(case.q[0])
    pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, ctx, case.scale, out=out,
                         max_context_len=case.max_context_len)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 2
    assert torch.count_nonzero(out[2]) == 0           # untouched
    check_close(out[:2], ref[:2], "valid sequences")


def test_decode_empty_batch_is_a_no_op():
    case = workloads.tiny_decode(device=DEV)
    q = case.q[0][:0]
    out = pa.paged_attn_decode(q, case.k_cache[0], case.v_cache[0], case.block_tables[:0],
                               case.context_lens[:0], case.scale, max_context_len=16)
    torch.cuda.synchronize()
    assert out.shape[0] == 0


def test_decode_workspace_reused_across_batch_sizes():
    # one workspace sized for the largest call serves smaller and larger batches in turn
    big = workloads.qwen3_8b_decode(device=DEV)
    kc, vc = big.k_cache[0].clone(), big.v_cache[0].clone()
    pa.kv_cache_write(big.k_new[0], big.v_new[0], big.slot_mapping, kc, vc)
    ref = oracle.paged_attn_decode(bits(big.q[0]), bits(kc), bits(vc), big.block_tables.cpu().numpy(),
                                   big.context_lens.cpu().numpy(), big.scale, oracle.BF16)
    ws = pa.alloc_decode_workspace(64, 32, 8, 4096, DEV)
    for n in (64, 5, 64, 17):
        out = pa.paged_attn_decode(big.q[0][:n].contiguous(), kc, vc,
                                   big.block_tables[:n].contiguous(), big.context_lens[:n].contiguous(),
                                   big.scale, workspace=ws, max_context_len=4096)
        torch.cuda.synchronize()
        check_close(out, ref[:n], f"{n} sequences on a reused workspace")


@pytest.mark.parametrize("dtype,hq,hkv", [("bf16", 16, 8), ("f16", 32, 8), ("bf16", 8, 8), ("bf16", 64, 8)])
def test_decode_one_cta_per_item_and_split_paths_agree(dtype, hq, hkv):
    # two sequences, 2 x Hkv items: the exact length bound selects one CTA per
    # item; a loose bound (16K tokens, too many pages for one SM) selects the
    # split kernels.  Both must match the oracle on the same inputs.
    lens = [700, 1024]
    case = workloads.build_case(f"paths-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=31 + hq, device=DEV,
                                decode_lens=lens)
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    ref = oracle.paged_attn_decode(bits(case.q[0]), bits(kc), bits(vc), case.block_tables.cpu().numpy(),
                                   case.context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[case.dtype])
    wide = torch.full((2, 1024), -1, dtype=torch.int32, device=DEV)      # room for a 16K-token bound
    wide[:, :case.block_tables.shape[1]] = case.block_tables
    assert pa.decode_kernel_launches(2, hkv, max(lens)) == 1
    assert pa.decode_kernel_launches(2, hkv, 16384) == 2
    for bound in (max(lens), 16384):
        out = pa.paged_attn_decode(case.q[0], kc, vc, wide, case.context_lens, case.scale, max_context_len=bound)
        torch.cuda.synchronize()
        check_close(out, ref, f"{case.name}, length bound {bound}")
