"""GPU parity of the causal chunked-prefill kernel (tcgen05 tensor cores)
against the fp64 oracle, through the C-ABI: the mixed-step workload, ragged
chunk lengths and starts, every supported head ratio, both dtypes, chunked
versus unchunked, decode versus the last prefill row, and data errors."""
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


def run_prefill(case, layer=0, max_chunk_len=None):
    kc, vc = case.k_cache[layer].clone(), case.v_cache[layer].clone()
    pa.kv_cache_write(case.k_new[layer], case.v_new[layer], case.slot_mapping, kc, vc)
    mcl = max_chunk_len or max(n for _, n in case.meta["chunks"])
    out = pa.paged_attn_prefill_chunk(case.q_chunks[layer], case.chunk_starts, case.chunk_lens, kc, vc,
                                      case.chunk_block_tables, case.chunk_context_lens, case.scale,
                                      max_chunk_len=mcl)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_prefill(case, kc, vc, layer=0):
    return oracle.paged_attn_prefill(bits(case.q_chunks[layer]), bits(kc), bits(vc),
                                     case.chunk_starts.cpu().numpy(), case.chunk_lens.cpu().numpy(),
                                     case.chunk_block_tables.cpu().numpy(), case.chunk_context_lens.cpu().numpy(),
                                     case.scale, ORACLE_DTYPE[case.dtype])


def prefill_and_check(case, what=None, max_chunk_len=None):
    out, kc, vc = run_prefill(case, max_chunk_len=max_chunk_len)
    kh, vh = oracle_write(case, 0)
    assert np.array_equal(bits(kc), kh) and np.array_equal(bits(vc), vh)
    ref = oracle_prefill(case, kc, vc)
    return check_close(out, ref, what or case.name), out


def test_prefill_small_two_chunks():
    prefill_and_check(workloads.build_case("two-chunks", "bf16", 16, 8, seed=11, device=DEV,
                                           chunks=[(0, 100), (40, 37)]))


def test_prefill_of_the_mixed_step():
    case = workloads.qwen3_0_6b_mixed_step(device=DEV)
    prefill_and_check(case, "mixed-step prefill chunks")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (16, 2)])
def test_prefill_ragged_chunks(dtype, hq, hkv):
    chunks = [(0, 1), (0, 15), (16, 16), (1, 17), (100, 63), (7, 64), (0, 65), (1000, 127), (5, 128),
              (129, 129), (0, 511), (1536, 512)]
    case = workloads.build_case(f"ragged-prefill-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=hq + 7 * hkv,
                                device=DEV, chunks=chunks)
    prefill_and_check(case)


def test_prefill_max_chunk_len_larger_than_needed():
    case = workloads.build_case("mcl", "bf16", 32, 8, seed=12, device=DEV, chunks=[(300, 40), (0, 9)])
    prefill_and_check(case, max_chunk_len=512)


def test_chunked_equals_unchunked_on_gpu():
    one = workloads.build_case("whole", "bf16", 16, 8, seed=13, device=DEV, chunks=[(0, 512)], num_blocks=64)
    # same data: the whole 512-token chunk at once versus the same positions as 3 chunks
    out_one, kc, vc = run_prefill(one)
    cuts = [(0, 100), (100, 300), (300, 512)]
    q = one.q_chunks[0]
    bt = one.chunk_block_tables.repeat(3, 1).contiguous()
    outs = []
    for s, e in cuts:
        outs.append(pa.paged_attn_prefill_chunk(
            q[s:e].contiguous(), torch.tensor([s], dtype=torch.int32, device=DEV),
            torch.tensor([e - s], dtype=torch.int32, device=DEV), kc, vc, bt[:1],
            torch.tensor([e], dtype=torch.int32, device=DEV), one.scale, max_chunk_len=e - s))
    torch.cuda.synchronize()
    many = torch.cat(outs)
    assert (many.float() - out_one.float()).abs().max().item() < 4e-3


def test_decode_equals_last_row_of_prefill():
    case = workloads.build_case("dec-vs-pre", "bf16", 32, 8, seed=14, device=DEV, chunks=[(200, 77)])
    out, kc, vc = run_prefill(case)
    last = case.q_chunks[0][-1:].contiguous()
    dec = pa.paged_attn_decode(last, kc, vc, case.chunk_block_tables, case.chunk_context_lens, case.scale,
                               max_context_len=277)
    torch.cuda.synchronize()
    assert (dec.float() - out[-1:].float()).abs().max().item() < 4e-3


def test_prefill_inconsistent_chunk_is_reported_and_untouched():
    case = workloads.build_case("badchunk", "bf16", 16, 8, seed=15, device=DEV, chunks=[(0, 40), (64, 30)])
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    ctx = case.chunk_context_lens.clone()
    ctx[1] += 1                                      # context must be start + len
    out = torch.zeros_like(case.q_chunks[0])
    pa.paged_attn_prefill_chunk(case.q_chunks[0], case.chunk_starts, case.chunk_lens, kc, vc,
                                case.chunk_block_tables, ctx, case.scale, out=out, max_chunk_len=40)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    assert torch.count_nonzero(out[40:]) == 0
    ref = oracle_prefill(case, kc, vc)
    check_close(out[:40], ref[:40], "valid chunk")


def test_prefill_long_prefixes():
    # few query tiles, each reading many key tiles (6000- and 3000-token prefixes)
    case = workloads.build_case("long-prefix", "bf16", 32, 8, seed=16, device=DEV, chunks=[(6000, 64), (3000, 33)])
    prefill_and_check(case, "long prefixes")


def test_prefill_is_deterministic():
    case = workloads.build_case("repeat", "bf16", 16, 8, seed=21, device=DEV, chunks=[(700, 300), (0, 200)])
    out1, kc, vc = run_prefill(case)
    out2 = pa.paged_attn_prefill_chunk(case.q_chunks[0], case.chunk_starts, case.chunk_lens, kc, vc,
                                       case.chunk_block_tables, case.chunk_context_lens, case.scale,
                                       max_chunk_len=300)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_prefill_many_small_chunks():
    rng = np.random.default_rng(17)
    chunks = [(int(rng.integers(0, 900)), int(rng.integers(1, 8))) for _ in range(300)]
    case = workloads.build_case("many-chunks", "f16", 16, 8, seed=17, device=DEV, chunks=chunks)
    prefill_and_check(case, "300 chunks", max_chunk_len=8)


def test_prefill_single_short_chunk():
    case = workloads.build_case("tiny", "bf16", 8, 8, seed=18, device=DEV, chunks=[(0, 3)])
    prefill_and_check(case, "one 3-token chunk")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (64, 8)])
@pytest.mark.parametrize("seed", [41, 42, 43])
def test_prefill_rows_just_past_the_second_term_threshold(hq, hkv, seed):
    # Query tiles whose first row sees 128 keys or more take P in one term of
    # the input dtype (bf16 here, the coarser one); the rounding errors of P
    # then average over at least 128 probabilities.  Rows with 128 .. ~700
    # visible keys, and tiles straddling the threshold, must stay inside the
    # tolerance as well as the rows that get the second term.
    case = workloads.build_case(f"threshold-{hq}x{hkv}-{seed}", "bf16", hq, hkv, seed=seed, device=DEV,
                                chunks=[(0, 400), (100, 200), (126, 64), (127, 1), (128, 40)])
    prefill_and_check(case)
