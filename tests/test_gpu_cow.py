"""GPU parity of the copy-on-write block copy ("Модуль 12: Финальный проект:
мини-движок инференса", qwen_serve/paged.py, SequenceCache._cow_copy) through
the C-ABI — bit-exact against the oracle's copy — and of the allocator-driven
step: block tables, slots and lengths from the library's host allocator, a
fork whose first write copies the shared tail block on the device, then KV
write and decode against the oracle fed the same tables."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
from gpu_util import bits, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
BS, D = 16, 128


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.get_device_error()
    yield
    st, detail = pa.get_device_error()
    assert st == 0, f"unexpected device error {pa.STATUS.get(st, st)} at index {detail}"


def _layers(n, nb, hkv, dtype=torch.float16, seed=0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    mk = lambda: torch.randn((nb, BS, hkv, D), generator=g, device=DEV).to(dtype)
    return [(mk(), mk()) for _ in range(n)]


def _host(pools):
    return [bits(k) for k, _ in pools], [bits(v) for _, v in pools]


@pytest.mark.parametrize("layers,nb,hkv,dtype", [(28, 64, 8, torch.float16), (3, 40, 2, torch.bfloat16),
                                                 (70, 12, 1, torch.float16)])
def test_block_copy_is_bit_exact(layers, nb, hkv, dtype):
    pools = _layers(layers, nb, hkv, dtype, seed=layers)
    hk, hv = _host(pools)
    rng = np.random.default_rng(layers)
    perm = rng.permutation(nb)
    n = min(10, nb // 2)
    pairs = np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int32)   # distinct dst, none a src
    pa.kv_block_copy(pools, torch.from_numpy(pairs).to(DEV))
    torch.cuda.synchronize()
    assert oracle.kv_block_copy(hk, hv, pairs) == 0
    for l, (k, v) in enumerate(pools):
        assert np.array_equal(bits(k), hk[l]) and np.array_equal(bits(v), hv[l]), f"layer {l}"


def test_block_copy_bad_pair_is_reported_and_skipped():
    pools = _layers(2, 8, 2, seed=9)
    hk, hv = _host(pools)
    pairs = np.array([[1, 2], [3, 8], [4, 5]], np.int32)
    pa.kv_block_copy(pools, torch.from_numpy(pairs).to(DEV))
    st, detail = pa.get_device_error()
    assert st == pa.STATUS_CODE["PA_ERR_RANGE"] and detail == 1
    assert oracle.kv_block_copy(hk, hv, pairs) == 1
    for l, (k, v) in enumerate(pools):
        assert np.array_equal(bits(k), hk[l]) and np.array_equal(bits(v), hv[l])


def _write(pools, host, slots, seed):
    """The same new K/V rows into the device pools (library) and the host pools (oracle)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    hkv = pools[0][0].shape[2]
    sl = torch.tensor(slots, dtype=torch.int64, device=DEV)
    for l, (k_cache, v_cache) in enumerate(pools):
        k = torch.randn((len(slots), hkv, D), generator=g, device=DEV).to(k_cache.dtype)
        v = torch.randn((len(slots), hkv, D), generator=g, device=DEV).to(k_cache.dtype)
        pa.kv_cache_write(k, v, sl, k_cache, v_cache)
        assert oracle.kv_cache_write(host[0][l], host[1][l], bits(k), bits(v), np.asarray(slots, np.int64)) == 0


def _copies(alloc, pools, host):
    pairs = np.asarray(alloc.take_copies(), np.int32).reshape(-1, 2)
    if len(pairs):
        pa.kv_block_copy(pools, torch.from_numpy(pairs).to(DEV))
        assert oracle.kv_block_copy(host[0], host[1], pairs) == 0
    return len(pairs)


def test_allocator_driven_fork_write_and_decode():
    layers, nb, hkv, hq = 2, 48, 8, 16
    pools = _layers(layers, nb, hkv, seed=21)
    host = _host(pools)
    alloc = pa.BlockAllocator(nb)
    a = alloc.sequence()
    _write(pools, host, a.reserve(37), seed=1)        # a's prompt: 37 tokens
    a.commit(37)
    b = alloc.sequence()
    b.fork_from(a)                                     # shares a's 3 blocks
    c = alloc.sequence()
    c.adopt_prefix(a.blocks[:2])                       # shares a's 2 full blocks
    _write(pools, host, c.reserve(5), seed=2)
    c.commit(5)
    assert _copies(alloc, pools, host) == 0
    # one decode step for a, b and c: b's token lands in the shared tail block -> copy first
    a_tail = [h[a.blocks[2]].copy() for h in host[0]]   # a's positions 32..36 before b writes
    slots = {}
    for name, s in (("a", a), ("b", b), ("c", c)):
        slots[name] = s.reserve(1)
    assert _copies(alloc, pools, host) == 1 and alloc.stats()["n_cow"] == 1
    assert b.blocks[:2] == a.blocks[:2] and b.blocks[2] != a.blocks[2]
    _write(pools, host, slots["a"] + slots["b"] + slots["c"], seed=3)
    for l, (k, v) in enumerate(pools):
        assert np.array_equal(bits(k), host[0][l]) and np.array_equal(bits(v), host[1][l]), f"pool, layer {l}"

    bt, _, _, ctx = pa.build_step_tables([a, b, c], 8)
    assert list(ctx) == [38, 38, 38]
    q = torch.randn((3, hq, D), device=DEV).to(torch.float16)
    bt_d, ctx_d = torch.from_numpy(bt).to(DEV), torch.from_numpy(ctx).to(DEV)
    scale = 1.0 / np.sqrt(D)
    for l, (k, v) in enumerate(pools):
        out = pa.paged_attn_decode(q, k, v, bt_d, ctx_d, scale)
        torch.cuda.synchronize()
        ref = oracle.paged_attn_decode(bits(q), host[0][l], host[1][l], bt, ctx, scale, oracle.F16)
        check_close(out, ref, f"allocator-driven decode, layer {l}")
    # a kept its own tail: b's copy and b's write left a's positions 32..36 untouched
    for l, (k, _) in enumerate(pools):
        assert np.array_equal(bits(k[a.blocks[2]])[:5], a_tail[l][:5])
    for s in (a, b, c):
        s.commit(1)
    alloc.close()
