"""GPU parity of the persistent mixed step (pa_mixed_step; page "Модуль 04:
KV-кэш и арифметика памяти", section 3.4: a step that prefills chunks while
running sequences decode): one launch does the chunks'
prefill (after the write of the chunks' new tokens) beside the sequences'
decode (which writes each sequence's new token as it reads its page).
Against the oracle: the pools bit-exact
after the write, both outputs element by element within tolerance; the
launch's counters are zero again after every call, and repeated calls on one
workspace (whose item counters must then be zero again too) give the same
outputs bit for bit.  Cases: the mixed step as the
bench runs it, ragged mixes at four head ratios and both dtypes, a step with
only decode, only prefill or only the write, repeated calls, and bad slots,
chunk metadata and context lengths (reported; the rest of the step intact)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
import workloads
from gpu_util import ORACLE_DTYPE, bits, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.get_device_error()
    yield
    st, detail = pa.get_device_error()
    assert st == 0, f"unexpected device error {pa.STATUS.get(st, st)} at index {detail}"


def _run(case, ws=None, chunks=True, decode=True, **over):
    """One pa_mixed_step call over layer 0 of the case (pool modified in place):
    the case's new tokens are the chunks' (first) and one per decoding
    sequence (after them, in sequence order)."""
    kc, vc = case.k_cache[0], case.v_cache[0]
    tc = sum(n for _, n in case.meta["chunks"])
    if ws is None:
        ws = pa.alloc_mixed_step_workspace(case.context_lens.numel() if decode else 0, case.hq, case.hkv, DEV)
    args = dict(k_chunks=case.k_new[0][:tc], v_chunks=case.v_new[0][:tc], chunk_slots=case.slot_mapping[:tc])
    if chunks:
        args.update(q_chunks=case.q_chunks[0], chunk_starts=case.chunk_starts, chunk_lens=case.chunk_lens,
                    chunk_block_tables=case.chunk_block_tables, chunk_context_lens=case.chunk_context_lens)
    if decode:
        args.update(q=case.q[0], k_dec=case.k_new[0][tc:], v_dec=case.v_new[0][tc:], block_tables=case.block_tables,
                    context_lens=case.context_lens)
    args.update(over)
    mcl = max(n for _, n in case.meta["chunks"]) if chunks else 512
    oc, od = pa.mixed_step(kc, vc, case.scale, ws, max_chunk_len=mcl, **args)
    torch.cuda.synchronize()
    return oc, od, ws


def _oracle(case, kh, vh, chunks=True, decode=True):
    d = ORACLE_DTYPE[case.dtype]
    assert oracle.kv_cache_write(kh, vh, bits(case.k_new[0]), bits(case.v_new[0]), case.slot_mapping.cpu().numpy()) == 0
    refp = oracle.paged_attn_prefill(bits(case.q_chunks[0]), kh, vh, case.chunk_starts.cpu().numpy(),
                                     case.chunk_lens.cpu().numpy(), case.chunk_block_tables.cpu().numpy(),
                                     case.chunk_context_lens.cpu().numpy(), case.scale, d) if chunks else None
    refd = oracle.paged_attn_decode(bits(case.q[0]), kh, vh, case.block_tables.cpu().numpy(),
                                    case.context_lens.cpu().numpy(), case.scale, d) if decode else None
    return refp, refd


def _check(case, what, chunks=True, decode=True):
    kh, vh = bits(case.k_cache[0]), bits(case.v_cache[0])
    oc, od, ws = _run(case, chunks=chunks, decode=decode)
    refp, refd = _oracle(case, kh, vh, chunks, decode)
    assert np.array_equal(bits(case.k_cache[0]), kh) and np.array_equal(bits(case.v_cache[0]), vh), \
        f"{what}: pools after the write"
    if chunks:
        check_close(oc, refp, f"{what}: prefill")
    if decode:
        check_close(od, refd, f"{what}: decode")
    assert int(torch.count_nonzero(ws[:16])) == 0, f"{what}: the launch's counters not zero again"


def test_mixed_step_as_benchmarked():
    case = workloads.qwen3_0_6b_mixed_step(device=DEV)   # 3 x 512 chunks on prefixes 0/512/1536 + 512 decodes
    _check(case, "mixed step")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 8), (32, 8), (64, 8)])
def test_mixed_step_ragged(dtype, hq, hkv):
    rng = np.random.default_rng(hq + hkv)
    chunks = [(0, 1), (17, 63), (100, 129), (0, 512), (1000, 300)]
    lens = [int(x) for x in rng.integers(1, 3000, size=40)] + [1, 16, 17, 4096]
    case = workloads.build_case(f"mixed-{dtype}-{hq}x{hkv}", dtype, hq, hkv, seed=hq * 3 + hkv, device=DEV,
                                chunks=chunks, decode_lens=lens)
    _check(case, case.name)


def test_mixed_step_decode_without_append():
    # the sequences' new tokens already in the pool (k_dec = v_dec = None)
    case = workloads.build_case("mixed-noapp", "bf16", 16, 8, seed=86, device=DEV, chunks=[(32, 100)],
                                decode_lens=[9, 260, 1500])
    kh, vh = bits(case.k_cache[0]), bits(case.v_cache[0])
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_cache[0], case.v_cache[0])
    oc, od, ws = _run(case, k_dec=None, v_dec=None)
    refp, refd = _oracle(case, kh, vh)
    check_close(oc, refp, "no append: prefill")
    check_close(od, refd, "no append: decode")


def test_mixed_step_decode_only_and_prefill_only():
    case = workloads.build_case("mixed-dec", "bf16", 16, 8, seed=81, device=DEV, decode_lens=[5, 700, 2048, 33])
    _check(case, "decode only", chunks=False)
    case = workloads.build_case("mixed-pre", "bf16", 16, 8, seed=82, device=DEV, chunks=[(64, 200), (0, 512)])
    _check(case, "prefill only", decode=False)


def test_mixed_step_write_only():
    # rows written through slots alone (no chunk reads them in this call)
    case = workloads.build_case("mixed-write", "f16", 16, 8, seed=83, device=DEV, decode_lens=[40, 90])
    kh, vh = bits(case.k_cache[0]), bits(case.v_cache[0])
    ws = pa.alloc_mixed_step_workspace(0, case.hq, case.hkv, DEV)
    pa.mixed_step(case.k_cache[0], case.v_cache[0], case.scale, ws, k_chunks=case.k_new[0], v_chunks=case.v_new[0],
                  chunk_slots=case.slot_mapping)
    torch.cuda.synchronize()
    assert oracle.kv_cache_write(kh, vh, bits(case.k_new[0]), bits(case.v_new[0]), case.slot_mapping.cpu().numpy()) == 0
    assert np.array_equal(bits(case.k_cache[0]), kh) and np.array_equal(bits(case.v_cache[0]), vh)
    assert int(torch.count_nonzero(ws[:16])) == 0


def test_mixed_step_repeated_calls_reuse_the_workspace():
    # the write is idempotent, so three calls on one workspace must give the
    # first call's outputs bit for bit (the launch's counters are zero again)
    case = workloads.build_case("mixed-rep", "bf16", 32, 8, seed=84, device=DEV, chunks=[(300, 400), (0, 77)],
                                decode_lens=[int(x) for x in np.random.default_rng(5).integers(1, 2000, 300)])
    kh, vh = bits(case.k_cache[0]), bits(case.v_cache[0])
    oc, od, ws = _run(case)
    oc, od = oc.clone(), od.clone()
    for _ in range(2):
        oc2, od2, _ = _run(case, ws=ws)
        assert torch.equal(oc2, oc) and torch.equal(od2, od)
    refp, refd = _oracle(case, kh, vh)
    check_close(oc, refp, "repeated: prefill")
    check_close(od, refd, "repeated: decode")


def test_mixed_step_reports_bad_inputs():
    case = workloads.build_case("mixed-bad", "bf16", 16, 8, seed=85, device=DEV, chunks=[(0, 40), (64, 30)],
                                decode_lens=[50, 300, 77])
    kh, vh = bits(case.k_cache[0]), bits(case.v_cache[0])
    refp, refd = _oracle(case, kh.copy(), vh.copy())
    # a context length past the block table: that sequence is reported and left unwritten
    ctx = case.context_lens.clone()
    ctx[1] = case.block_tables.shape[1] * 16 + 1
    out = torch.zeros_like(case.q[0])
    oc, od, ws = _run(case, context_lens=ctx, out=out)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    assert torch.count_nonzero(od[1]) == 0
    check_close(od[0], refd[0], "decode beside a bad sequence")
    check_close(od[2], refd[2], "decode beside a bad sequence")
    check_close(oc, refp, "prefill beside a bad sequence")
    assert int(torch.count_nonzero(ws[:16])) == 0
    # bad chunk metadata: the chunk is reported and left unwritten
    cctx = case.chunk_context_lens.clone()
    cctx[1] += 1
    outc = torch.zeros_like(case.q_chunks[0])
    oc, od, ws = _run(case, chunk_context_lens=cctx, out_chunks=outc)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    assert torch.count_nonzero(oc[40:]) == 0
    check_close(oc[:40], refp[:40], "chunk before the bad one")
    check_close(od, refd, "decode beside a bad chunk")
    # a slot outside the pool: that token's write is reported and skipped
    slots = case.slot_mapping.clone()
    slots[5] = case.num_blocks * 16 + 7
    kc0, vc0 = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.mixed_step(case.k_cache[0], case.v_cache[0], case.scale, pa.alloc_mixed_step_workspace(0, case.hq, case.hkv, DEV),
                  k_chunks=case.k_new[0], v_chunks=case.v_new[0], chunk_slots=slots)
    torch.cuda.synchronize()
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 5
    ok = torch.ones(slots.numel(), dtype=torch.bool, device=DEV)
    ok[5] = False
    flat = lambda t: t.view(-1, case.hkv, 128)
    assert torch.equal(flat(case.k_cache[0])[slots[ok]], case.k_new[0][ok])
    assert torch.equal(flat(case.v_cache[0])[slots[ok]], case.v_new[0][ok])
    del kc0, vc0
