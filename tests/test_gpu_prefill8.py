"""GPU parity of the chunked prefill over 8-bit pools
(pa_paged_attn_prefill_chunk_q8; "Модуль 04: KV-кэш и арифметика памяти",
section 5, KV8Cache, and section 5.4, FP8 KV): every token of each chunk's
context is quantised into an int8 or E4M3 pool by the library's write and,
from the same 16-bit rows, by the oracle's write (checked bit-exact); the
prefill over the device pool is then compared element by element with the
oracle's prefill over its own pool.  Cases: the mixed-step chunks, ragged
chunks at every head ratio and both query dtypes, unused slots holding E4M3
NaN codes, long prefixes, bad chunk metadata and bad block ids."""
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


def _chunk_slots(case):
    """Flat slots of every position [0, ctx) of every chunk (each once)."""
    bt = case.chunk_block_tables.cpu().numpy()
    out = []
    for c, n in enumerate(case.chunk_context_lens.cpu().numpy()):
        j = np.arange(int(n))
        out.append(bt[c, j // BS].astype(np.int64) * BS + j % BS)
    return np.unique(np.concatenate(out))


def _pools(case, fp8, nan_codes=False):
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    slots = _chunk_slots(case)
    sl = torch.from_numpy(slots).to(DEV)
    krows = kc.view(-1, case.hkv, 128)[sl].contiguous()
    vrows = vc.view(-1, case.hkv, 128)[sl].contiguous()
    gpu = (pa.alloc_pool_f8 if fp8 else pa.alloc_pool_q8)(case.num_blocks, case.hkv, DEV)
    code_t = np.uint8 if fp8 else np.int8
    host = (np.zeros((case.num_blocks, BS, case.hkv, 128), code_t),
            np.zeros((case.num_blocks, BS, case.hkv, 128), code_t),
            np.zeros((case.num_blocks, case.hkv, BS), np.float32),
            np.zeros((case.num_blocks, case.hkv, BS), np.float32))
    if nan_codes:  # every slot the write leaves alone holds an E4M3 NaN
        for t in gpu[:2]:
            t.fill_(0x7F)
        for a in host[:2]:
            a.fill(0x7F)
    (pa.kv_cache_write_f8 if fp8 else pa.kv_cache_write_q8)(krows, vrows, sl, *gpu)
    write = oracle.kv_cache_write_f8 if fp8 else oracle.kv_cache_write_q8
    assert write(*host, bits(krows), bits(vrows), ORACLE_DTYPE[case.dtype], slots) == 0
    torch.cuda.synchronize()
    for g, h, name in zip(gpu, host, ("k codes", "v codes", "k scales", "v scales")):
        gn = g.cpu().numpy()
        same = np.array_equal(gn.view(np.uint32), h.view(np.uint32)) if gn.dtype == np.float32 else \
            np.array_equal(gn.view(np.uint8), h.view(np.uint8))
        assert same, f"{case.name}: {name} of the write not bit-exact"
    return gpu, host


def _prefill(case, gpu, fp8, mcl, bt=None, ctx=None, out=None):
    fn = pa.paged_attn_prefill_chunk_f8 if fp8 else pa.paged_attn_prefill_chunk_q8
    out = fn(case.q_chunks[0], case.chunk_starts, case.chunk_lens, *gpu,
             case.chunk_block_tables if bt is None else bt,
             case.chunk_context_lens if ctx is None else ctx, case.scale, out=out, max_chunk_len=mcl)
    torch.cuda.synchronize()
    return out


def _oracle(case, host, fp8):
    fn = oracle.paged_attn_prefill_f8 if fp8 else oracle.paged_attn_prefill_q8
    return fn(bits(case.q_chunks[0]), *host, case.chunk_starts.cpu().numpy(), case.chunk_lens.cpu().numpy(),
              case.chunk_block_tables.cpu().numpy(), case.chunk_context_lens.cpu().numpy(), case.scale,
              ORACLE_DTYPE[case.dtype])


def _check(case, fp8, what, nan_codes=False):
    gpu, host = _pools(case, fp8, nan_codes)
    mcl = max(n for _, n in case.meta["chunks"])
    out = _prefill(case, gpu, fp8, mcl)
    check_close(out, _oracle(case, host, fp8), what)


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill8_of_the_mixed_step(fp8):
    case = workloads.qwen3_0_6b_mixed_step(device=DEV)
    _check(case, fp8, f"mixed-step chunks, {'E4M3' if fp8 else 'int8'} pool")


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (16, 2), (64, 8)])
def test_prefill8_ragged_chunks(fp8, dtype, hq, hkv):
    chunks = [(0, 1), (0, 15), (16, 16), (1, 17), (100, 63), (7, 64), (0, 65), (1000, 127), (5, 128),
              (129, 129), (0, 511), (1536, 512)]
    case = workloads.build_case(f"prefill8-ragged-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=hq + 3 * hkv + 7,
                                device=DEV, chunks=chunks)
    _check(case, fp8, f"{case.name}, {'E4M3' if fp8 else 'int8'}")


def test_prefill8_slots_past_the_sequence_hold_e4m3_nans():
    # pages end mid-page: the unused value rows of the last pages hold NaN codes
    case = workloads.build_case("prefill8-nan", "bf16", 16, 8, seed=61, device=DEV,
                                chunks=[(3, 20), (40, 33), (500, 129)])
    _check(case, True, "NaN codes past each sequence", nan_codes=True)


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill8_long_prefixes(fp8):
    case = workloads.build_case("prefill8-long", "bf16", 32, 8, seed=62, device=DEV,
                                chunks=[(9000, 64), (6000, 33), (7777, 512)])
    _check(case, fp8, f"long prefixes, {'E4M3' if fp8 else 'int8'}")


@pytest.mark.parametrize("fp8", [False, True])
def test_prefill8_reports_bad_chunks_and_block_ids(fp8):
    case = workloads.build_case("prefill8-bad", "f16", 16, 8, seed=63, device=DEV,
                                chunks=[(0, 40), (64, 30), (2000, 300)])
    gpu, host = _pools(case, fp8)
    ref = _oracle(case, host, fp8)
    ctx = case.chunk_context_lens.clone()
    ctx[1] += 1                                       # context must be start + len
    out = torch.zeros_like(case.q_chunks[0])
    _prefill(case, gpu, fp8, 300, ctx=ctx, out=out)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    assert torch.count_nonzero(out[40:70]) == 0       # the bad chunk is left unwritten
    check_close(out[:40], ref[:40], "chunk before the bad one")
    check_close(out[70:], ref[70:], "chunk after the bad one")
    # a block id outside the pool in chunk 2's table: reported, its page skipped, nothing else touched
    bt = case.chunk_block_tables.clone()
    bt[2, 5] = case.num_blocks + 3
    out2 = _prefill(case, gpu, fp8, 300, bt=bt)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 2
    check_close(out2[:70], ref[:70], "chunks whose tables are intact")
    assert torch.isfinite(out2[70:].float()).all()
