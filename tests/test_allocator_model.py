"""Randomised check of the native block allocator and sequence tables against a
small Python model of the rules they implement (page "Модуль 12: Финальный
проект: мини-движок инференса", task 12.1 and qwen_serve/paged.py:
BlockAllocator with a first-in first-out free list and reference counts,
all-or-nothing allocation; SequenceCache reserve / commit; fork sharing every
block; the first write into a shared, partly filled block copies it; a prefix
adopted by reference).  Every operation, including refused ones, must give the
same status, slots, block lists, lengths, reference counts, statistics and
recorded copies on both sides.  No GPU involved."""
from collections import deque

import numpy as np
import pytest

import paged_kv_gqa_cache_gb300 as pa

BS = 16
OK, NO_BLOCKS, STATE = 0, pa.STATUS_CODE["PA_ERR_NO_BLOCKS"], pa.STATUS_CODE["PA_ERR_STATE"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_gqa_cache_gb300 import _build
    _build.build()


class Refused(Exception):
    def __init__(self, status):
        self.status = status


class ModelPool:
    def __init__(self, n):
        self.free = deque(range(n))
        self.ref = [0] * n
        self.copies = []
        self.n_allocated = 0
        self.n_cow = 0

    def _take(self):
        b = self.free.popleft()
        self.ref[b] += 1
        self.n_allocated += 1
        return b

    def _drop(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def allocate(self, n):
        if n > len(self.free):
            raise Refused(NO_BLOCKS)
        return [self._take() for _ in range(n)]

    def retain(self, b):
        if self.ref[b] == 0:
            raise Refused(STATE)
        self.ref[b] += 1

    def release(self, b):
        if self.ref[b] <= 0:
            raise Refused(STATE)
        self._drop(b)

    def stats(self):
        return dict(total=len(self.ref), free=len(self.free), used=sum(r > 0 for r in self.ref),
                    shared=sum(r > 1 for r in self.ref), n_allocated=self.n_allocated, n_cow=self.n_cow)

    def take_copies(self):
        out, self.copies = self.copies, []
        return out


class ModelSeq:
    def __init__(self, pool):
        self.pool, self.blocks, self.length, self.reserved = pool, [], 0, 0

    def empty(self):
        return not self.blocks and self.length == 0 and self.reserved == 0

    def reserve(self, n):
        p = self.pool
        pos = self.length + self.reserved
        need, have = -(-(pos + n) // BS), len(self.blocks)
        bi = pos // BS
        cow = bi < have and p.ref[self.blocks[bi]] > 1      # the block written into is shared
        if max(need - have, 0) + cow > len(p.free):
            raise Refused(NO_BLOCKS)
        if cow:
            src, dst = self.blocks[bi], p._take()
            p.copies.append((src, dst))
            p._drop(src)
            self.blocks[bi] = dst
            p.n_cow += 1
        self.blocks += [p._take() for _ in range(have, need)]
        self.reserved += n
        return [self.blocks[q // BS] * BS + q % BS for q in range(pos, pos + n)]

    def commit(self, n):
        if n > self.reserved:
            raise Refused(STATE)
        self.length += n
        self.reserved -= n

    def fork_from(self, other):
        if not self.empty() or other.reserved:
            raise Refused(STATE)
        for b in other.blocks:
            self.pool.ref[b] += 1
        self.blocks, self.length = list(other.blocks), other.length

    def adopt_prefix(self, blocks):
        if not self.empty() or any(self.pool.ref[b] == 0 for b in blocks):
            raise Refused(STATE)
        for b in blocks:
            self.pool.ref[b] += 1
        self.blocks, self.length = list(blocks), BS * len(blocks)

    def release(self):
        for b in self.blocks:
            self.pool._drop(b)
        self.blocks, self.length, self.reserved = [], 0, 0


def both(model_fn, native_fn):
    """Runs an operation on both sides; returns its result, or the refusal, after checking they agree."""
    try:
        want = ("ok", model_fn())
    except Refused as e:
        want = ("refused", e.status)
    try:
        got = ("ok", native_fn())
    except pa.PagedAttnError as e:
        got = ("refused", e.status)
    assert got == want
    return want


def check_state(mp, np_, mseqs, nseqs, loose):
    n = len(mp.ref)
    assert [np_.refcount(b) for b in range(n)] == mp.ref
    assert np_.stats() == mp.stats()
    for ms, ns in zip(mseqs, nseqs):
        assert (ns.blocks, ns.length, ns.reserved) == (ms.blocks, ms.length, ms.reserved)
        assert len(set(ms.blocks)) == len(ms.blocks)
    # every reference is held by a sequence or by the loose list, and free ids have none
    held = [0] * n
    for ms in mseqs:
        for b in ms.blocks:
            held[b] += 1
    for b in loose:
        held[b] += 1
    assert held == mp.ref
    assert all(mp.ref[b] == 0 for b in mp.free) and len(set(mp.free)) == len(mp.free)


def check_step_tables(mseqs, nseqs, max_blocks):
    """pa_build_step_tables against the model: tables padded with -1, starts =
    committed lengths, lens = reserved tokens, contexts = their sums; a sequence
    holding more blocks than max_blocks refuses the whole call."""
    if any(len(m.blocks) > max_blocks for m in mseqs):
        with pytest.raises(pa.PagedAttnError) as e:
            pa.build_step_tables(nseqs, max_blocks)
        assert e.value.status == pa.STATUS_CODE["PA_ERR_SHAPE"]
        return
    bt, starts, lens, ctx = pa.build_step_tables(nseqs, max_blocks)
    for k, m in enumerate(mseqs):
        assert list(bt[k]) == m.blocks + [-1] * (max_blocks - len(m.blocks))
        assert (starts[k], lens[k], ctx[k]) == (m.length, m.reserved, m.length + m.reserved)


def _run(seed):
    """One random run of 500 operations; returns the model pool and the refusals seen."""
    rng = np.random.default_rng(seed)
    refusals = []
    nblocks = int(rng.choice([9, 17, 40]))
    mp, np_ = ModelPool(nblocks), pa.BlockAllocator(nblocks)
    mseqs, nseqs, loose = [], [], []
    for step in range(500):
        op = rng.choice(["new", "reserve", "commit", "fork", "adopt", "release_seq", "allocate", "retain",
                         "release", "copies"], p=[.08, .27, .2, .1, .06, .07, .07, .05, .05, .05])
        i = int(rng.integers(len(mseqs))) if mseqs else None
        res = None
        if op == "new" and len(mseqs) < 8:
            mseqs.append(ModelSeq(mp))
            nseqs.append(np_.sequence())
        elif op == "reserve" and mseqs:
            n = int(rng.choice([1, 1, 1, 3, 15, 16, 17, 40]))
            res = both(lambda: mseqs[i].reserve(n), lambda: nseqs[i].reserve(n))
        elif op == "commit" and mseqs:
            r = mseqs[i].reserved
            # mostly everything reserved (a finished step), sometimes part, sometimes one too many (refused)
            n = r if rng.random() < 0.6 else int(rng.integers(0, r + 2))
            res = both(lambda: mseqs[i].commit(n), lambda: nseqs[i].commit(n))
        elif op in ("fork", "adopt") and len(mseqs) >= 2:
            # mostly an empty target and a source with nothing reserved (the valid case); else any pair
            empties = [k for k, m in enumerate(mseqs) if m.empty()]
            sources = [k for k, m in enumerate(mseqs) if m.blocks and not m.reserved]
            if rng.random() < 0.8 and empties and sources:
                i, j = int(rng.choice(empties)), int(rng.choice(sources))
            else:
                j = int(rng.integers(len(mseqs)))
            if j != i and op == "fork":
                res = both(lambda: mseqs[i].fork_from(mseqs[j]), lambda: nseqs[i].fork_from(nseqs[j]))
            elif j != i:
                full = mseqs[j].blocks[:mseqs[j].length // BS]
                k = int(rng.integers(0, len(full) + 1))
                res = both(lambda: mseqs[i].adopt_prefix(full[:k]), lambda: nseqs[i].adopt_prefix(full[:k]))
        elif op == "release_seq" and mseqs:
            both(mseqs[i].release, nseqs[i].release)
        elif op == "allocate":
            n = int(rng.integers(0, 4))
            res = both(lambda: mp.allocate(n), lambda: np_.allocate(n))
            if res[0] == "ok":
                loose += res[1]
        elif op == "retain" and loose:
            b = loose[int(rng.integers(len(loose)))]
            both(lambda: mp.retain(b), lambda: np_.retain(b))
            loose.append(b)
        elif op == "release" and loose:
            b = loose.pop(int(rng.integers(len(loose))))
            both(lambda: mp.release(b), lambda: np_.release(b))
        elif op == "copies":
            both(mp.take_copies, np_.take_copies)
        if res is not None and res[0] == "refused":
            refusals.append((op, res[1]))
        check_state(mp, np_, mseqs, nseqs, loose)
        if nseqs and step % 25 == 0:
            check_step_tables(mseqs, nseqs, int(rng.choice([2, 4, 64])))
    # a block that nothing holds any more cannot be retained or released
    free_ids = list(mp.free)
    if free_ids:
        b = free_ids[0]
        both(lambda: mp.retain(b), lambda: np_.retain(b))
        both(lambda: mp.release(b), lambda: np_.release(b))
    for ms, ns in zip(mseqs, nseqs):
        both(ms.release, ns.release)
    for b in loose:
        both(lambda: mp.release(b), lambda: np_.release(b))
    check_state(mp, np_, mseqs, nseqs, [])
    assert np_.stats()["free"] == nblocks
    return mp, refusals


@pytest.mark.parametrize("seed", range(12))
def test_random_operations_match_the_model(seed):
    _run(seed)


def test_the_random_runs_reach_copy_on_write_and_every_refusal():
    runs = [_run(seed) for seed in range(12)]
    assert sum(mp.n_cow for mp, _ in runs) >= 30
    seen = {r for _, refusals in runs for r in refusals}
    for want in [("reserve", NO_BLOCKS), ("commit", STATE), ("fork", STATE), ("adopt", STATE)]:
        assert want in seen, f"no {want} in the random runs"
