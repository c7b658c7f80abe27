"""Failure detection and out-of-bounds checks on the GPU, without any fault:

* the library's bounded wait gives up on a barrier that nothing completes,
  records PA_ERR_TIMEOUT, and the context stays usable (a decode right after
  still matches the oracle);
* canary regions around every output buffer and every pool stay intact
  through the write, decode (both paths), fused append, prefill, int8 write
  and decode, fused norm + RoPE write and block copy, including calls that
  carry out-of-range block ids and slots (which must be reported and skipped).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
import workloads
from gpu_util import ORACLE_DTYPE, bits, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 8192          # elements of canary before and after each buffer (16 KB for 16-bit data)
CANARY16 = 0x7BCD     # a finite 16-bit pattern no kernel writes by accident


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.get_device_error()
    yield
    pa.get_device_error()


class Guarded:
    """A tensor of `shape` inside a larger allocation whose head and tail hold canaries."""

    def __init__(self, src: torch.Tensor):
        n = src.numel()
        self.big = torch.empty(n + 2 * GUARD, dtype=src.dtype, device=DEV)
        raw = self.big.view(torch.int16) if src.element_size() == 2 else self.big.view(torch.int8)
        raw.fill_(CANARY16 if src.element_size() == 2 else 0x5A)
        if src.element_size() == 4:
            self.big.view(torch.int32).fill_(0x3F7BCD5A)
        self.t = self.big[GUARD:GUARD + n].view(src.shape)
        self.t.copy_(src)
        self.head = self.big[:GUARD].clone()
        self.tail = self.big[GUARD + n:].clone()

    def intact(self) -> bool:
        n = self.t.numel()
        eq = lambda a, b: torch.equal(a.view(torch.uint8), b.view(torch.uint8))
        return eq(self.big[:GUARD], self.head) and eq(self.big[GUARD + n:], self.tail)


def _check_all(bufs, what):
    torch.cuda.synchronize()
    for name, g in bufs.items():
        assert g.intact(), f"{what}: canary around {name} was overwritten"


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    pa.selftest_bounded_wait(20000)   # 20 ms
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_TIMEOUT"] and detail == -1
    c = workloads.tiny_decode(device=DEV)
    kc, vc = c.k_cache[0].clone(), c.v_cache[0].clone()
    pa.kv_cache_write(c.k_new[0], c.v_new[0], c.slot_mapping, kc, vc)
    out = pa.paged_attn_decode(c.q[0], kc, vc, c.block_tables, c.context_lens, c.scale)
    torch.cuda.synchronize()
    assert pa.get_device_error()[0] == 0
    ref = oracle.paged_attn_decode(bits(c.q[0]), bits(kc), bits(vc), c.block_tables.cpu().numpy(),
                                   c.context_lens.cpu().numpy(), c.scale, oracle.F16)
    check_close(out, ref, "decode after the timeout self-test")


@pytest.mark.parametrize("bound", [None, 16384])
def test_canaries_survive_write_decode_and_append(bound):
    c = workloads.build_case("canary-decode", "bf16", 32, 8, seed=3, device=DEV, decode_lens=[1, 17, 300, 1000])
    bt = torch.full((4, 1024), -1, dtype=torch.int32, device=DEV)
    bt[:, :c.block_tables.shape[1]] = c.block_tables
    bt[3, 5] = c.num_blocks + 7                      # an out-of-range block id inside sequence 3's context
    g = {"k_cache": Guarded(c.k_cache[0]), "v_cache": Guarded(c.v_cache[0]),
         "out": Guarded(torch.zeros_like(c.q[0])), "out2": Guarded(torch.zeros_like(c.q[0]))}
    slots = c.slot_mapping.clone()
    slots[1] = c.num_blocks * 16                      # one slot past the pool
    pa.kv_cache_write(c.k_new[0], c.v_new[0], slots, g["k_cache"].t, g["v_cache"].t)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    mcl = bound or 1000
    pa.paged_attn_decode(c.q[0], g["k_cache"].t, g["v_cache"].t, bt, c.context_lens, c.scale, out=g["out"].t,
                         max_context_len=mcl)
    assert pa.get_device_error()[0] == pa.STATUS_CODE["PA_ERR_RANGE"]
    pa.paged_attn_decode_append(c.q[0], c.k_new[0], c.v_new[0], g["k_cache"].t, g["v_cache"].t, bt,
                                c.context_lens, c.scale, out=g["out2"].t, max_context_len=mcl)
    assert pa.get_device_error()[0] == pa.STATUS_CODE["PA_ERR_RANGE"]
    _check_all(g, f"decode, bound {bound}")


def test_canaries_survive_prefill_with_a_bad_block():
    c = workloads.build_case("canary-prefill", "bf16", 16, 8, seed=4, device=DEV,
                             chunks=[(0, 100), (200, 77), (1000, 512)])
    g = {"k_cache": Guarded(c.k_cache[0]), "v_cache": Guarded(c.v_cache[0]),
         "out": Guarded(torch.zeros_like(c.q_chunks[0]))}
    pa.kv_cache_write(c.k_new[0], c.v_new[0], c.slot_mapping, g["k_cache"].t, g["v_cache"].t)
    bt = c.chunk_block_tables.clone()
    bt[2, 3] = -5                                     # a bad block id in the last chunk's prefix
    pa.paged_attn_prefill_chunk(c.q_chunks[0], c.chunk_starts, c.chunk_lens, g["k_cache"].t, g["v_cache"].t, bt,
                                c.chunk_context_lens, c.scale, out=g["out"].t, max_chunk_len=512)
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 2
    pa.paged_attn_prefill_chunk_window(c.q_chunks[0], c.chunk_starts, c.chunk_lens, g["k_cache"].t,
                                       g["v_cache"].t, c.chunk_block_tables, c.chunk_context_lens, c.scale, 100,
                                       out=g["out"].t, max_chunk_len=512)
    assert pa.get_device_error()[0] == 0
    _check_all(g, "prefill")


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_canaries_survive_int8_write_and_decode(kind):
    c = workloads.build_case("canary-q8", "f16", 16, 8, seed=5, device=DEV, decode_lens=[5, 64, 700])
    f8 = kind == "fp8"
    pool = (pa.alloc_pool_f8 if f8 else pa.alloc_pool_q8)(c.num_blocks, 8, DEV)
    g = {n: Guarded(t) for n, t in zip(("k_codes", "v_codes", "k_scale", "v_scale"), pool)}
    g["out"] = Guarded(torch.zeros_like(c.q[0]))
    slots = c.slot_mapping.clone()
    slots[0] = -1
    (pa.kv_cache_write_f8 if f8 else pa.kv_cache_write_q8)(c.k_new[0], c.v_new[0], slots, g["k_codes"].t,
                                                          g["v_codes"].t, g["k_scale"].t, g["v_scale"].t)
    assert pa.get_device_error() == (pa.STATUS_CODE["PA_ERR_RANGE"], 0)
    for bound in (700, 16384):
        bt = torch.full((3, 1024), -1, dtype=torch.int32, device=DEV)
        bt[:, :c.block_tables.shape[1]] = c.block_tables
        (pa.paged_attn_decode_f8 if f8 else pa.paged_attn_decode_q8)(
            c.q[0], g["k_codes"].t, g["v_codes"].t, g["k_scale"].t, g["v_scale"].t, bt, c.context_lens, c.scale,
            out=g["out"].t, max_context_len=bound)
        assert pa.get_device_error()[0] == 0
    _check_all(g, kind)


def test_canaries_survive_rope_write_and_block_copy():
    T, hq, hkv, nb = 40, 16, 8, 8
    gen = torch.Generator(device=DEV).manual_seed(6)
    mk = lambda *shape: torch.randn(shape, generator=gen, device=DEV).to(torch.bfloat16)
    q, k, v = mk(T, hq, 128), mk(T, hkv, 128), mk(T, hkv, 128)
    w = torch.ones(128, device=DEV, dtype=torch.bfloat16)
    cos, sin = torch.ones(64, 128, device=DEV, dtype=torch.bfloat16), torch.zeros(64, 128, device=DEV,
                                                                                  dtype=torch.bfloat16)
    pos = torch.arange(T, dtype=torch.int32, device=DEV)
    pos[7] = 64                                       # past the 64-row tables
    slots = torch.arange(T, dtype=torch.int64, device=DEV) * 3 % (nb * 16)
    slots[9] = nb * 16                                # past the pool
    g = {"k_cache": Guarded(torch.zeros(nb, 16, hkv, 128, device=DEV, dtype=torch.bfloat16)),
         "v_cache": Guarded(torch.zeros(nb, 16, hkv, 128, device=DEV, dtype=torch.bfloat16)),
         "q_out": Guarded(torch.zeros_like(q))}
    pa.qk_norm_rope_kv_write(q, k, v, w, w, 1e-6, cos, sin, pos, slots, g["k_cache"].t, g["v_cache"].t,
                             q_out=g["q_out"].t)
    assert pa.get_device_error()[0] == pa.STATUS_CODE["PA_ERR_RANGE"]
    pairs = torch.tensor([[0, 5], [1, 8], [2, 6]], dtype=torch.int32, device=DEV)   # block 8 is past the pool
    pa.kv_block_copy([(g["k_cache"].t, g["v_cache"].t)], pairs)
    assert pa.get_device_error() == (pa.STATUS_CODE["PA_ERR_RANGE"], 1)
    _check_all(g, "rope write and block copy")
