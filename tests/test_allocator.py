"""Host-side block allocator and block-table builder of the library (page
"Модуль 12: Финальный проект: мини-движок инференса", task 12.1 and
qwen_serve/paged.py: BlockAllocator, SequenceCache), through the C-ABI; no
GPU involved.  The worked examples and acceptance item 5 of task 12.1 are
checked as printed there; copy-on-write follows that task's rule (fork shares
every block, the first write into a shared partly filled block copies it)."""
import numpy as np
import pytest

import paged_kv_gqa_cache_gb300 as pa

BS = 16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_gqa_cache_gb300 import _build
    _build.build()


def _err(fn, code):
    with pytest.raises(pa.PagedAttnError) as e:
        fn()
    assert e.value.status == pa.STATUS_CODE[code]


def test_allocator_worked_example():
    # allocate(3) on a 64-block pool -> [0, 1, 2], 61 free, refcount[0] == 1;
    # release(0) -> refcount 0, back in the free list; retain(1); release(1) -> alive, refcount 1
    a = pa.BlockAllocator(64)
    assert a.allocate(3) == [0, 1, 2]
    assert a.stats()["free"] == 61 and a.refcount(0) == 1
    a.release(0)
    assert a.refcount(0) == 0 and a.stats()["free"] == 62
    a.retain(1)
    a.release(1)
    assert a.refcount(1) == 1


def test_free_list_is_first_in_first_out():
    a = pa.BlockAllocator(4)
    assert a.allocate(4) == [0, 1, 2, 3]
    a.release(2)
    a.release(0)
    assert a.allocate(2) == [2, 0]


def test_sequence_reserve_worked_example():
    # reserve(20) on an empty table -> blocks [0, 1], in-block offsets 0..15 then 0..3,
    # length still 0; after commit(20) length 20 and blocks unchanged
    a = pa.BlockAllocator(64)
    s = a.sequence()
    slots = s.reserve(20)
    assert s.blocks == [0, 1] and s.length == 0
    assert [x // BS for x in slots] == [0] * 16 + [1] * 4
    assert [x % BS for x in slots] == list(range(16)) + list(range(4))
    s.commit(20)
    assert s.length == 20 and s.blocks == [0, 1] and s.reserved == 0


def test_no_fragmentation_acceptance_mix():
    # 32 sequences of random length 1..512: occupied blocks are exactly
    # sum ceil(len / 16), used + free == total throughout, and after every
    # release free == total and used == 0
    rng = np.random.default_rng(5)
    a = pa.BlockAllocator(1100)
    seqs, lens = [], rng.integers(1, 512, size=32, endpoint=True)
    for n in lens:
        s = a.sequence()
        left = int(n)
        while left:
            step = int(min(left, rng.integers(1, 64)))
            s.reserve(step)
            s.commit(step)
            left -= step
            st = a.stats()
            assert st["used"] + st["free"] == st["total"]
        seqs.append(s)
    assert a.stats()["used"] == sum(-(-int(n) // BS) for n in lens)
    for s in seqs:
        s.release()
        st = a.stats()
        assert st["used"] + st["free"] == st["total"]
    assert a.stats()["free"] == 1100 and a.stats()["used"] == 0


def test_fork_shares_every_block_and_copies_on_first_write():
    a = pa.BlockAllocator(64)
    s1 = a.sequence()
    s1.reserve(20)
    s1.commit(20)
    s2 = a.sequence()
    s2.fork_from(s1)
    assert s2.blocks == s1.blocks and s2.length == 20
    assert all(a.refcount(b) == 2 for b in s1.blocks)
    assert a.stats()["shared"] == 2
    slots = s2.reserve(1)          # position 20 lands in the shared, partly filled block 1
    assert s2.blocks[0] == s1.blocks[0] and s2.blocks[1] != s1.blocks[1]
    assert a.stats()["n_cow"] == 1
    assert a.take_copies() == [(s1.blocks[1], s2.blocks[1])]
    assert a.take_copies() == []
    assert slots == [s2.blocks[1] * BS + 4]
    assert a.refcount(s1.blocks[1]) == 1 and a.refcount(s2.blocks[1]) == 1 and a.refcount(s1.blocks[0]) == 2


def test_fork_of_a_full_tail_needs_no_copy():
    a = pa.BlockAllocator(64)
    s1 = a.sequence()
    s1.reserve(32)
    s1.commit(32)
    s2 = a.sequence()
    s2.fork_from(s1)
    s2.reserve(1)
    assert a.stats()["n_cow"] == 0 and s2.blocks[:2] == s1.blocks and len(s2.blocks) == 3


def test_the_source_copies_too_if_it_writes_first():
    a = pa.BlockAllocator(64)
    s1 = a.sequence()
    s1.reserve(5)
    s1.commit(5)
    s2 = a.sequence()
    s2.fork_from(s1)
    old = s1.blocks[0]
    s1.reserve(1)
    assert s1.blocks[0] != old and s2.blocks == [old] and a.take_copies() == [(old, s1.blocks[0])]


def test_adopt_prefix_never_copies():
    a = pa.BlockAllocator(64)
    owner = a.sequence()
    owner.reserve(40)
    owner.commit(40)
    s = a.sequence()
    s.adopt_prefix(owner.blocks[:2])   # two full blocks
    assert s.length == 32 and a.refcount(owner.blocks[0]) == 2
    s.reserve(3)
    assert a.stats()["n_cow"] == 0 and len(s.blocks) == 3 and s.blocks[:2] == owner.blocks[:2]


def test_out_of_blocks_changes_nothing():
    a = pa.BlockAllocator(4)
    s = a.sequence()
    s.reserve(40)                      # 3 blocks
    before = a.stats()
    _err(lambda: s.reserve(30), "PA_ERR_NO_BLOCKS")   # needs 2 more, 1 free
    assert a.stats() == before and s.reserved == 40 and len(s.blocks) == 3
    _err(lambda: a.allocate(2), "PA_ERR_NO_BLOCKS")
    assert a.stats() == before


def test_misuse_is_refused():
    a = pa.BlockAllocator(8)
    _err(lambda: a.release(3), "PA_ERR_STATE")        # a free block
    _err(lambda: a.retain(3), "PA_ERR_STATE")
    _err(lambda: a.release(8), "PA_ERR_RANGE")
    s = a.sequence()
    s.reserve(4)
    _err(lambda: s.commit(5), "PA_ERR_STATE")          # beyond the reservation
    t = a.sequence()
    _err(lambda: t.fork_from(s), "PA_ERR_STATE")        # s has reserved, uncommitted tokens
    s.commit(4)
    _err(lambda: s.adopt_prefix([0]), "PA_ERR_STATE")   # not empty
    _err(lambda: t.adopt_prefix([5]), "PA_ERR_STATE")   # a free block
    t.fork_from(s)
    _err(lambda: t.fork_from(s), "PA_ERR_STATE")        # not empty


def test_step_tables_for_decode_and_prefill():
    a = pa.BlockAllocator(64)
    d = a.sequence()
    d.reserve(37)
    d.commit(37)
    d.reserve(1)                       # a decode step: one new token
    p = a.sequence()
    p.reserve(100)                     # a prefill chunk of 100 on an empty prefix
    bt, starts, lens, ctx = pa.build_step_tables([d, p], 8)
    assert bt.shape == (2, 8) and bt.dtype == np.int32
    assert list(bt[0]) == d.blocks + [-1] * (8 - len(d.blocks))
    assert list(bt[1]) == p.blocks + [-1] * (8 - len(p.blocks))
    assert list(starts) == [37, 0] and list(lens) == [1, 100] and list(ctx) == [38, 100]
    _err(lambda: pa.build_step_tables([d, p], 6), "PA_ERR_SHAPE")   # p holds 7 blocks
