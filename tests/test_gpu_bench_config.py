"""Parity in the launch configuration the benchmark times: the bench's own step
objects, captured as one CUDA graph of the whole step (every layer's calls,
programmatic dependent launch between them) and replayed several times, then
checked against the oracle: pools bit-exact after the writes, every layer's
decode output (or each distinct pool's last one) and the mixed step's prefill
output within tolerance."""
import numpy as np
import pytest
import torch

import bench
import oracle
from gpu_util import ORACLE_DTYPE, bits, check_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def _clean_error_word():
    import paged_kv_gqa_cache_gb300 as pa
    pa.get_device_error()
    yield
    st, detail = pa.get_device_error()
    assert st == 0, f"unexpected device error {pa.STATUS.get(st, st)} at index {detail}"


def _replay(step_fn, times=3):
    stream = torch.cuda.Stream(device=DEV)
    g = bench.graph_of(step_fn, 1, stream)
    bench.time_replays(g, times, stream)
    torch.cuda.synchronize()


def _check_decode_step(step, layers_to_check):
    c = step.case
    before = [(bits(c.k_cache[i]), bits(c.v_cache[i])) for i in layers_to_check]
    _replay(step.run)
    bt, ctx = c.block_tables.cpu().numpy(), c.context_lens.cpu().numpy()
    for (kh, vh), i in zip(before, layers_to_check):
        assert oracle.kv_cache_write(kh, vh, bits(c.k_new[i]), bits(c.v_new[i]), c.slot_mapping.cpu().numpy()) == 0
        assert np.array_equal(bits(c.k_cache[i]), kh) and np.array_equal(bits(c.v_cache[i]), vh), f"pool {i}"
        ref = oracle.paged_attn_decode(bits(c.q[i]), kh, vh, bt, ctx, c.scale, ORACLE_DTYPE[c.dtype])
        check_close(step.out[i], ref, f"{step.desc[:40]}, pool {i}")


@pytest.mark.parametrize("fused", [True, False])   # the bench's default: one launch over all SMs
@pytest.mark.parametrize("early", [True, False])   # the bench's default passes PA_DECODE_EARLY_PAGES
def test_qwen3_0_6b_decode_step_as_benchmarked(early, fused):
    step = bench.DecodeStep(DEV, workload=2, early_pages=early, fused=fused)     # 28 layers, 28 distinct pools
    _check_decode_step(step, range(step.case.n_layers))


@pytest.mark.parametrize("early", [True, False])
def test_qwen3_0_6b_decode_step_with_the_fused_append(early):
    step = bench.DecodeStep(DEV, workload=2, append=True, early_pages=early)
    _check_decode_step(step, range(step.case.n_layers))


@pytest.mark.parametrize("fused", [True, False])
def test_qwen3_8b_decode_as_benchmarked(fused):
    step = bench.DecodeStep(DEV, workload=4, pools=4, early_pages=True, fused=fused)  # 36 layers, 4 pools of 1 GiB
    _check_decode_step(step, range(step.case.n_layers))


def test_prefix_shared_tail_as_benchmarked():
    step = bench.DecodeStep(DEV, workload=5, early_pages=True, fused=True)      # 8 calls cycling 4 pools
    _check_decode_step(step, range(step.case.n_layers))


def test_mixed_step_as_benchmarked():
    step = bench.MixedStep(DEV, overlap=True, fused=True)   # 28 layers, 2 pools, prefill beside decode
    c = step.case
    before = [(bits(c.k_cache[i]), bits(c.v_cache[i])) for i in range(2)]
    _replay(step.run)
    for i, (kh, vh) in enumerate(before):
        assert oracle.kv_cache_write(kh, vh, bits(c.k_new[i]), bits(c.v_new[i]), c.slot_mapping.cpu().numpy()) == 0
        assert np.array_equal(bits(c.k_cache[i]), kh) and np.array_equal(bits(c.v_cache[i]), vh)
        refp = oracle.paged_attn_prefill(bits(c.q_chunks[i]), kh, vh, c.chunk_starts.cpu().numpy(),
                                         c.chunk_lens.cpu().numpy(), c.chunk_block_tables.cpu().numpy(),
                                         c.chunk_context_lens.cpu().numpy(), c.scale, oracle.BF16)
        check_close(step.out_p[i], refp, f"mixed step prefill, pool {i}")
        refd = oracle.paged_attn_decode(bits(c.q[i]), kh, vh, c.block_tables.cpu().numpy(),
                                        c.context_lens.cpu().numpy(), c.scale, oracle.BF16)
        check_close(step.out_d[i], refd, f"mixed step decode, pool {i}")


def test_persistent_mixed_step_as_benchmarked():
    step = bench.MixedStep(DEV, persistent=True)   # 28 layers, 2 pools, one pa_mixed_step launch per layer
    c = step.case
    before = [(bits(c.k_cache[i]), bits(c.v_cache[i])) for i in range(2)]
    _replay(step.run)
    for i, (kh, vh) in enumerate(before):
        assert oracle.kv_cache_write(kh, vh, bits(c.k_new[i]), bits(c.v_new[i]), c.slot_mapping.cpu().numpy()) == 0
        assert np.array_equal(bits(c.k_cache[i]), kh) and np.array_equal(bits(c.v_cache[i]), vh)
        refp = oracle.paged_attn_prefill(bits(c.q_chunks[i]), kh, vh, c.chunk_starts.cpu().numpy(),
                                         c.chunk_lens.cpu().numpy(), c.chunk_block_tables.cpu().numpy(),
                                         c.chunk_context_lens.cpu().numpy(), c.scale, oracle.BF16)
        check_close(step.out_p[i], refp, f"persistent mixed step prefill, pool {i}")
        refd = oracle.paged_attn_decode(bits(c.q[i]), kh, vh, c.block_tables.cpu().numpy(),
                                        c.context_lens.cpu().numpy(), c.scale, oracle.BF16)
        check_close(step.out_d[i], refd, f"persistent mixed step decode, pool {i}")
    assert int(step.mws[:16].count_nonzero()) == 0   # the launch's counters


def _same_pool(gpu, host, what):
    for g, h, name in zip(gpu, host, ("k codes", "v codes", "k scales", "v scales")):
        gn = g.cpu().numpy()
        ok = np.array_equal(gn.view(np.uint32), h.view(np.uint32)) if gn.dtype == np.float32 else \
            np.array_equal(gn.view(np.uint8), h.view(np.uint8))
        assert ok, f"{what}: {name} differ from the oracle's"


@pytest.mark.parametrize("fp8", [False, True])
def test_mixed_step_over_8bit_pools_as_benchmarked(fp8):
    step = bench.MixedStepQ8(DEV, fp8=fp8, overlap=True)   # 8-bit write, prefill and decode per layer
    c = step.case
    BS = 16
    slots = []
    for bt, ctx in ((c.block_tables, c.context_lens), (c.chunk_block_tables, c.chunk_context_lens)):
        b = bt.cpu().numpy()
        for s_, n in enumerate(ctx.cpu().numpy()):
            j = np.arange(int(n))
            slots.append(b[s_, j // BS].astype(np.int64) * BS + j % BS)
    slots = np.unique(np.concatenate(slots))
    write = oracle.kv_cache_write_f8 if fp8 else oracle.kv_cache_write_q8
    code_t = np.uint8 if fp8 else np.int8
    hosts = []
    for i in range(2):   # the oracle's own pools, quantised from the same 16-bit rows
        h = (np.zeros((c.num_blocks, BS, c.hkv, 128), code_t), np.zeros((c.num_blocks, BS, c.hkv, 128), code_t),
             np.zeros((c.num_blocks, c.hkv, BS), np.float32), np.zeros((c.num_blocks, c.hkv, BS), np.float32))
        rows = lambda t: bits(t[i]).reshape(-1, c.hkv, 128)[slots]
        assert write(*h, rows(c.k_cache), rows(c.v_cache), oracle.BF16, slots) == 0
        _same_pool(step.q8[i], h, f"pool {i} before the step")
        hosts.append(h)
    _replay(step.run)
    pre = oracle.paged_attn_prefill_f8 if fp8 else oracle.paged_attn_prefill_q8
    dec = oracle.paged_attn_decode_f8 if fp8 else oracle.paged_attn_decode_q8
    for i, h in enumerate(hosts):
        assert write(*h, bits(c.k_new[i]), bits(c.v_new[i]), oracle.BF16, c.slot_mapping.cpu().numpy()) == 0
        _same_pool(step.q8[i], h, f"pool {i} after the step")
        refp = pre(bits(c.q_chunks[i]), *h, c.chunk_starts.cpu().numpy(), c.chunk_lens.cpu().numpy(),
                   c.chunk_block_tables.cpu().numpy(), c.chunk_context_lens.cpu().numpy(), c.scale, oracle.BF16)
        check_close(step.out_p[i], refp, f"8-bit mixed step prefill, pool {i}")
        refd = dec(bits(c.q[i]), *h, c.block_tables.cpu().numpy(), c.context_lens.cpu().numpy(), c.scale,
                   oracle.BF16)
        check_close(step.out_d[i], refd, f"8-bit mixed step decode, pool {i}")


@pytest.mark.parametrize("append", [False, True])
def test_end_to_end_path_returns_the_right_outputs_to_the_host(append):
    # the e2e leg: inputs copied from pinned host memory each step, the library
    # calls reading the copies (metadata included), outputs copied back
    step = bench.DecodeStep(DEV, workload=2, append=append, early_pages=True, fused=True)
    c = step.case
    before = [(bits(c.k_cache[i]), bits(c.v_cache[i])) for i in range(c.n_layers)]
    stream = torch.cuda.Stream(device=DEV)
    bench.e2e_measure(step, 3, 3, stream)
    bt, ctx = c.block_tables.cpu().numpy(), c.context_lens.cpu().numpy()
    for l in (0, 13, step.L - 1):
        kh, vh = before[l % c.n_layers]
        assert oracle.kv_cache_write(kh, vh, bits(c.k_new[l]), bits(c.v_new[l]), c.slot_mapping.cpu().numpy()) == 0
        ref = oracle.paged_attn_decode(bits(c.q[l]), kh, vh, bt, ctx, c.scale, ORACLE_DTYPE[c.dtype])
        check_close(step.e2e_outputs[l], ref, f"e2e layer {l}")


def test_mixed_step_end_to_end_path_returns_the_right_outputs_to_the_host():
    # the mixed step's e2e leg: every layer's inputs and the step's metadata
    # copied from pinned host memory, both outputs of every layer copied back
    step = bench.MixedStep(DEV, overlap=True, fused=True)
    c = step.case
    before = [(bits(c.k_cache[i]), bits(c.v_cache[i])) for i in range(2)]
    stream = torch.cuda.Stream(device=DEV)
    bench.e2e_measure_mixed(step, 1, 0, stream)     # the warm-up call and one timed step
    for l in (0, step.L - 1):
        kh, vh = before[l % 2]
        assert oracle.kv_cache_write(kh, vh, bits(c.k_new[l % 2]), bits(c.v_new[l % 2]),
                                     c.slot_mapping.cpu().numpy()) == 0
        out_d, out_p = step.e2e_outputs[l]
        refp = oracle.paged_attn_prefill(bits(c.q_chunks[l % 2]), kh, vh, c.chunk_starts.cpu().numpy(),
                                         c.chunk_lens.cpu().numpy(), c.chunk_block_tables.cpu().numpy(),
                                         c.chunk_context_lens.cpu().numpy(), c.scale, oracle.BF16)
        check_close(out_p, refp, f"mixed e2e prefill, layer {l}")
        refd = oracle.paged_attn_decode(bits(c.q[l % 2]), kh, vh, c.block_tables.cpu().numpy(),
                                        c.context_lens.cpu().numpy(), c.scale, oracle.BF16)
        check_close(out_d, refd, f"mixed e2e decode, layer {l}")
