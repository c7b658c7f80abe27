"""The seeded input recipe (workloads/), on the CPU: each of the five
workloads has the sizes, length mix and dtype it is stated to have, its block
tables hand out every physical block to at most one sequence (the prefix-shared
workload's 13 shared blocks excepted) with -1 past each sequence's pages, the
step's new-token slots are the chunk tokens first and then one per decoding
sequence at position ctx - 1, all distinct and inside the pool, and (in parity
mode) exactly the slots that hold no cached token are NaN."""
import math

import numpy as np
import pytest
import torch

import workloads

BS = 16


@pytest.fixture
def light_pools(monkeypatch):
    """Build the large workloads without their pools (the structure is what is
    checked); record the cached-slot mask each build would have NaN-filled around."""
    seen = {}

    def fake(gen, num_blocks, hkv, dtype, device, n_layers, valid_slots, nan_fill):
        seen["valid"] = valid_slots.clone()
        return [None] * n_layers, [None] * n_layers

    monkeypatch.setattr(workloads, "_pools", fake)
    return seen


def _rows(case):
    """(block-table row, context length, new-token positions) per sequence, chunks first."""
    out = []
    if case.chunk_starts is not None:
        for c in range(case.chunk_starts.numel()):
            s, n = int(case.chunk_starts[c]), int(case.chunk_lens[c])
            assert int(case.chunk_context_lens[c]) == s + n
            out.append((case.chunk_block_tables[c].numpy(), s + n, range(s, s + n)))
    if case.context_lens is not None:
        for j in range(case.context_lens.numel()):
            ctx = int(case.context_lens[j])
            out.append((case.block_tables[j].numpy(), ctx, range(ctx - 1, ctx)))
    return out


def _check_structure(case, shared_blocks=0):
    rows = _rows(case)
    owner = {}
    for i, (bt, ctx, _) in enumerate(rows):
        pages = math.ceil(ctx / BS)
        assert bt.dtype == np.int32
        assert (bt[:pages] >= 0).all() and (bt[:pages] < case.num_blocks).all()
        assert (bt[pages:] == -1).all(), "table entries past a sequence's pages are -1"
        for p, b in enumerate(bt[:pages]):
            if p < shared_blocks:
                assert b == rows[0][0][p], "the shared prefix is the same physical blocks in every row"
                continue
            assert int(b) not in owner, f"block {b} handed out twice"
            owner[int(b)] = i
    if shared_blocks:
        assert not set(owner) & {int(b) for b in rows[0][0][:shared_blocks]}
    # the step's new slots: chunk tokens, then one per decoding sequence
    expect = [int(bt[p // BS]) * BS + p % BS for bt, _, new in rows for p in new]
    slots = case.slot_mapping.numpy()
    assert case.slot_mapping.dtype == torch.int64
    assert slots.tolist() == expect
    assert len(set(expect)) == len(expect)
    assert all(0 <= s < case.num_blocks * BS for s in expect)
    # cached tokens: every position before the step's new ones
    cached = np.zeros(case.num_blocks * BS, bool)
    for bt, ctx, new in rows:
        for p in range(new.start):
            cached[int(bt[p // BS]) * BS + p % BS] = True
    assert not cached[slots].any()
    return cached


def test_tiny_decode():
    case = workloads.tiny_decode()
    assert (case.dtype, case.hq, case.hkv, case.num_blocks) == ("f16", 16, 8, 64)
    assert case.context_lens.tolist() == [17, 33, 100, 250]
    assert case.k_cache[0].dtype == torch.float16 and case.k_cache[0].shape == (64, BS, 8, 128)
    cached = _check_structure(case)
    # parity mode: NaN exactly where no token is cached (the new slots included)
    for pool in (case.k_cache[0], case.v_cache[0]):
        nan = torch.isnan(pool.view(64 * BS, -1)).all(dim=1).numpy()
        fin = torch.isfinite(pool.view(64 * BS, -1)).all(dim=1).numpy()
        assert (nan == ~cached).all() and (fin == cached).all()
    assert case.q[0].shape == (4, 16, 128) and case.k_new[0].shape == (4, 8, 128)


def test_qwen3_0_6b_decode_step():
    case = workloads.qwen3_0_6b_decode(n_layers=2)
    assert (case.dtype, case.hq, case.hkv, case.num_blocks, case.n_layers) == ("f16", 16, 8, 512, 2)
    lens = case.context_lens.tolist()
    assert len(lens) == 8 and all(512 <= n <= 1024 for n in lens)
    cached = _check_structure(case)
    for layer in range(2):
        nan = torch.isnan(case.k_cache[layer].view(512 * BS, -1)).all(dim=1).numpy()
        assert (nan == ~cached).all()
    assert not torch.equal(case.k_cache[0], case.k_cache[1]), "each layer has its own values"


def test_qwen3_0_6b_mixed_step(light_pools):
    case = workloads.qwen3_0_6b_mixed_step()
    assert (case.dtype, case.hq, case.hkv) == ("bf16", 16, 8)
    assert list(zip(case.chunk_starts.tolist(), case.chunk_lens.tolist())) == [(0, 512), (512, 512), (1536, 512)]
    lens = case.context_lens.tolist()
    assert len(lens) == 512 and min(lens) >= 16 and max(lens) <= 1024
    assert case.slot_mapping.numel() == 2048, "the step's token budget: 3 x 512 chunk tokens + 512 decodes"
    assert case.q_chunks[0].shape == (1536, 16, 128) and case.q[0].shape == (512, 16, 128)
    need = sum(math.ceil(n / BS) for n in lens) + sum(math.ceil((s + n) / BS) for s, n in case.meta["chunks"])
    assert case.num_blocks == math.ceil(need * 1.25), "pool = needed blocks + 25 % free"
    cached = _check_structure(case)
    assert (light_pools["valid"].numpy() == cached).all()


def test_qwen3_8b_decode_fills_its_pool_exactly(light_pools):
    case = workloads.qwen3_8b_decode()
    assert (case.dtype, case.hq, case.hkv, case.num_blocks) == ("bf16", 32, 8, 16384)
    assert case.context_lens.tolist() == [4096] * 64
    _check_structure(case)
    used = np.sort(case.block_tables.numpy().ravel())
    assert (used == np.arange(16384)).all(), "64 x 256 pages are a permutation of the whole pool"
    assert workloads.decode_kv_bytes(case.context_lens.tolist(), 8) == 1 << 30


def test_prefix_shared_tail(light_pools):
    case = workloads.prefix_shared_tail()
    assert (case.dtype, case.hq, case.hkv) == ("bf16", 32, 8)
    lens = case.context_lens.tolist()
    assert len(lens) == 32 and all(208 + 16 <= n <= 208 + 32768 for n in lens)
    # log-uniform suffixes: a long tail, not a narrow band
    suffix = np.array(lens) - 208
    assert suffix.max() / suffix.min() > 100
    assert case.meta["shared_prefix_blocks"] == 13
    cached = _check_structure(case, shared_blocks=13)
    assert (light_pools["valid"].numpy() == cached).all()


def test_by_index_names_the_five_workloads():
    assert sorted(workloads.BY_INDEX) == [1, 2, 3, 4, 5]
    assert workloads.BY_INDEX[4] is workloads.qwen3_8b_decode


def test_cases_are_reproducible_from_their_seed():
    a, b = workloads.tiny_decode(), workloads.tiny_decode()
    assert torch.equal(a.q[0], b.q[0]) and torch.equal(a.slot_mapping, b.slot_mapping)
    assert torch.equal(torch.nan_to_num(a.k_cache[0]), torch.nan_to_num(b.k_cache[0]))
