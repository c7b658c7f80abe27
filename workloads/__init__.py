"""Seeded synthetic inputs for paged-KV GQA attention.

Shared by the tests, the smoke check and the benchmark.  This module holds
none of the attention arithmetic: it draws values, lengths and block
placements, and composes the caller-side inputs (block tables and slot
mappings) the way an engine's block manager would.

Recipe (stated once, used everywhere):

* q, K, V values ~ N(0, 1) drawn in fp32 by ``torch.Generator(device)``
  seeded with ``1000 + seed``, then cast to fp16/bf16 (round to nearest even).
* Lengths and block placement come from ``numpy.random.default_rng(seed)``.
  Physical blocks are handed out from a random permutation of the pool, so a
  sequence's pages sit anywhere in memory ("Phase 10: LLMs from Scratch —
  Inference Optimization", paged-attention section: pages may live anywhere).
* Block-table entries past a sequence's last page are -1 (never read).
* In parity mode every pool slot that holds no token yet is NaN, so a kernel
  that reads past a sequence's length, or into another sequence's page,
  produces NaN; the slots of this step's new tokens are NaN until written.

Geometry follows the pages: Qwen3-0.6B (28 layers, 16 query heads, 8 KV heads,
head_dim 128) and Qwen3-8B (36 layers, 32 / 8 heads, head_dim 128), 16-token
blocks ("Модуль 12: Финальный проект: мини-движок инференса", opening section
and "Память"; "Модуль 04: KV-кэш и арифметика памяти", section 2.1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

BLOCK = 16
HEAD_DIM = 128

QWEN3_0_6B = dict(name="Qwen3-0.6B", n_layers=28, hq=16, hkv=8)
QWEN3_8B = dict(name="Qwen3-8B", n_layers=36, hq=32, hkv=8)

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


def cdiv(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class Case:
    """One step's inputs for one or more layers sharing one block table.

    Decode part: ``q`` [S, Hq, d] for sequences with ``context_lens`` (the new
    token is at position ctx-1).  Prefill part: ``q_chunks`` [sum(n), Hq, d]
    for chunks (``chunk_starts``, ``chunk_lens``) with their own block-table
    rows.  New tokens of the step: ``k_new``/``v_new`` [T, Hkv, d] and
    ``slot_mapping`` [T] (chunk tokens first, then one per decode sequence).
    ``k_cache``/``v_cache`` are lists (one pool per layer) of
    [num_blocks, 16, Hkv, d] tensors.
    """
    name: str
    dtype: str
    hq: int
    hkv: int
    num_blocks: int
    scale: float
    k_cache: List[torch.Tensor]
    v_cache: List[torch.Tensor]
    k_new: List[torch.Tensor]
    v_new: List[torch.Tensor]
    slot_mapping: torch.Tensor
    # decode sequences
    q: Optional[List[torch.Tensor]] = None
    block_tables: Optional[torch.Tensor] = None
    context_lens: Optional[torch.Tensor] = None
    # prefill chunks
    q_chunks: Optional[List[torch.Tensor]] = None
    chunk_starts: Optional[torch.Tensor] = None
    chunk_lens: Optional[torch.Tensor] = None
    chunk_block_tables: Optional[torch.Tensor] = None
    chunk_context_lens: Optional[torch.Tensor] = None
    meta: Dict = field(default_factory=dict)

    @property
    def n_layers(self) -> int:
        return len(self.k_cache)

    @property
    def max_context_len(self) -> int:
        return int(self.meta.get("max_context_len", 0))


def _place(rng: np.random.Generator, lens: Sequence[int], num_blocks: int,
           shared: Optional[List[int]] = None, extra_free: float = 0.0):
    """Hand out physical blocks: one block-table row per sequence.

    ``shared`` lists physical blocks that open every row (a shared prefix of
    full blocks).  Returns (block_tables int32 [S, max_pages] padded with -1,
    pool size).
    """
    shared = shared or []
    pages = [cdiv(n, BLOCK) for n in lens]
    private = [p - len(shared) for p in pages]
    assert all(p >= 0 for p in private)
    need = sum(private) + len(shared)
    if num_blocks <= 0:
        num_blocks = int(math.ceil(need * (1.0 + extra_free)))
    assert need <= num_blocks, f"pool of {num_blocks} blocks cannot hold {need}"
    perm = rng.permutation(num_blocks)
    shared_ids = perm[:len(shared)] if shared else np.zeros(0, np.int64)
    cursor = len(shared)
    width = max(pages) if pages else 1
    bt = np.full((len(lens), max(width, 1)), -1, np.int32)
    for s, p in enumerate(private):
        row = list(shared_ids) + list(perm[cursor:cursor + p])
        cursor += p
        bt[s, :len(row)] = row
    return bt, num_blocks


def _slots(bt_row: np.ndarray, lo: int, hi: int) -> np.ndarray:
    """Flat physical slots (block * 16 + offset) of logical positions [lo, hi) of a sequence."""
    pos = np.arange(lo, hi, dtype=np.int64)
    return bt_row[pos // BLOCK].astype(np.int64) * BLOCK + pos % BLOCK


def _values(gen: torch.Generator, shape, dtype: str, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(DTYPES[dtype])


def _pools(gen, num_blocks, hkv, dtype, device, n_layers, valid_slots: Optional[torch.Tensor],
           nan_fill: bool):
    ks, vs = [], []
    for _ in range(n_layers):
        k = _values(gen, (num_blocks, BLOCK, hkv, HEAD_DIM), dtype, device)
        v = _values(gen, (num_blocks, BLOCK, hkv, HEAD_DIM), dtype, device)
        if nan_fill:
            bad = ~valid_slots.view(num_blocks, BLOCK)
            k[bad] = float("nan")
            v[bad] = float("nan")
        ks.append(k)
        vs.append(v)
    return ks, vs


def build_case(name: str, dtype: str, hq: int, hkv: int, *, seed: int, device="cpu",
               decode_lens: Sequence[int] = (), chunks: Sequence[tuple] = (),
               num_blocks: int = 0, extra_free: float = 0.25, shared_prefix_blocks: int = 0,
               n_layers: int = 1, nan_fill: bool = True, fixed_bt: Optional[np.ndarray] = None) -> Case:
    """Assemble a step: decode sequences (lengths include the new token) and
    prefill chunks ``(start, n)`` (n new tokens after ``start`` cached ones)."""
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device=device)
    gen.manual_seed(1000 + seed)
    dev = torch.device(device)

    chunk_ctx = [s + n for s, n in chunks]
    all_lens = list(chunk_ctx) + list(decode_lens)
    if fixed_bt is not None:
        bt_all = fixed_bt.astype(np.int32)
        assert num_blocks > 0
    else:
        shared = list(range(shared_prefix_blocks)) if shared_prefix_blocks else None
        bt_all, num_blocks = _place(rng, all_lens, num_blocks, shared, extra_free)
    nc = len(chunks)

    # slots that hold an already-cached token (positions before this step's new ones)
    valid = np.zeros(num_blocks * BLOCK, dtype=bool)
    new_slots: List[np.ndarray] = []
    for i, (start, n) in enumerate(chunks):
        valid[_slots(bt_all[i], 0, start)] = True
        new_slots.append(_slots(bt_all[i], start, start + n))
    for j, ctx in enumerate(decode_lens):
        valid[_slots(bt_all[nc + j], 0, ctx - 1)] = True
        new_slots.append(_slots(bt_all[nc + j], ctx - 1, ctx))
    new_slots_all = np.concatenate(new_slots) if new_slots else np.zeros(0, np.int64)
    T = int(new_slots_all.shape[0])
    valid = torch.from_numpy(valid)

    k_cache, v_cache = _pools(gen, num_blocks, hkv, dtype, dev, n_layers, valid.to(dev), nan_fill)
    k_new = [_values(gen, (T, hkv, HEAD_DIM), dtype, dev) for _ in range(n_layers)]
    v_new = [_values(gen, (T, hkv, HEAD_DIM), dtype, dev) for _ in range(n_layers)]
    case = Case(name=name, dtype=dtype, hq=hq, hkv=hkv, num_blocks=num_blocks,
                scale=1.0 / math.sqrt(HEAD_DIM), k_cache=k_cache, v_cache=v_cache,
                k_new=k_new, v_new=v_new,
                slot_mapping=torch.from_numpy(new_slots_all).to(dev))
    if decode_lens:
        case.q = [_values(gen, (len(decode_lens), hq, HEAD_DIM), dtype, dev) for _ in range(n_layers)]
        case.block_tables = torch.from_numpy(np.ascontiguousarray(bt_all[nc:])).to(dev)
        case.context_lens = torch.tensor(list(decode_lens), dtype=torch.int32, device=dev)
    if chunks:
        rows = sum(n for _, n in chunks)
        case.q_chunks = [_values(gen, (rows, hq, HEAD_DIM), dtype, dev) for _ in range(n_layers)]
        case.chunk_starts = torch.tensor([s for s, _ in chunks], dtype=torch.int32, device=dev)
        case.chunk_lens = torch.tensor([n for _, n in chunks], dtype=torch.int32, device=dev)
        case.chunk_block_tables = torch.from_numpy(np.ascontiguousarray(bt_all[:nc])).to(dev)
        case.chunk_context_lens = torch.tensor(chunk_ctx, dtype=torch.int32, device=dev)
    case.meta.update(max_context_len=max(all_lens) if all_lens else 0,
                     decode_lens=list(decode_lens), chunks=list(chunks),
                     shared_prefix_blocks=shared_prefix_blocks, seed=seed)
    return case


# ---- the five workloads -------------------------------------------------------

def tiny_decode(device="cpu", nan_fill=True) -> Case:
    """Tiny decode, one layer, Qwen3-0.6B attention geometry, fp16: 4 sequences of
    context {17, 33, 100, 250} in a 64-block pool, plus the write of their 4 new tokens."""
    lens = [17, 33, 100, 250]
    rng = np.random.default_rng(1)
    perm = rng.permutation(64)
    pages = [cdiv(n, BLOCK) for n in lens]                 # 2, 3, 7, 16 = 28 blocks
    bt = np.full((4, max(pages)), -1, np.int32)
    cur = 0
    for s, p in enumerate(pages):
        bt[s, :p] = perm[cur:cur + p]
        cur += p
    return build_case("tiny-decode", "f16", 16, 8, seed=1, device=device, decode_lens=lens,
                      num_blocks=64, fixed_bt=bt, nan_fill=nan_fill)


def qwen3_0_6b_decode_lens(seed: int = 2) -> List[int]:
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(512, 1024, size=8, endpoint=True)]


def qwen3_0_6b_decode(device="cpu", n_layers=28, nan_fill=True) -> Case:
    """Qwen3-0.6B decode step: 8 sequences of context U[512, 1024], fp16, one
    512-block pool per layer (28 layers), block table shared by all layers."""
    return build_case("qwen3-0.6b-decode", "f16", 16, 8, seed=2, device=device,
                      decode_lens=qwen3_0_6b_decode_lens(), num_blocks=512, n_layers=n_layers,
                      nan_fill=nan_fill)


def qwen3_0_6b_mixed_step(device="cpu", n_layers=1, nan_fill=True) -> Case:
    """Qwen3-0.6B mixed chunked-prefill step (budget 2048), bf16: chunks of 512
    new tokens on cached prefixes of 0, 512 and 1536 tokens, plus 512 decode
    sequences of context U[16, 1024]; pool = needed blocks + 25 % free."""
    rng = np.random.default_rng(3)
    lens = [int(x) for x in rng.integers(16, 1024, size=512, endpoint=True)]
    return build_case("qwen3-0.6b-mixed-step", "bf16", 16, 8, seed=3, device=device,
                      decode_lens=lens, chunks=[(0, 512), (512, 512), (1536, 512)],
                      n_layers=n_layers, nan_fill=nan_fill)


def qwen3_8b_decode(device="cpu", n_layers=1, nan_fill=True) -> Case:
    """Qwen3-8B decode, bf16: 64 sequences x 4096 context in an exactly-full
    16384-block pool per layer."""
    return build_case("qwen3-8b-decode", "bf16", 32, 8, seed=4, device=device,
                      decode_lens=[4096] * 64, num_blocks=16384, n_layers=n_layers,
                      nan_fill=nan_fill)


def prefix_shared_tail_lens(seed: int = 5) -> List[int]:
    rng = np.random.default_rng(seed)
    suffix = np.floor(np.exp(rng.uniform(math.log(16), math.log(32768), size=32))).astype(int)
    return [208 + int(s) for s in suffix]


def prefix_shared_tail(device="cpu", n_layers=1, nan_fill=True) -> Case:
    """Prefix-shared long-tail decode, Qwen3-8B geometry, bf16: 32 sequences whose
    first 13 blocks (208 tokens) are the same physical blocks, then private
    suffixes log-uniform in [16, 32768] tokens; pool = needed + 25 %."""
    return build_case("qwen3-8b-prefix-shared-tail", "bf16", 32, 8, seed=5, device=device,
                      decode_lens=prefix_shared_tail_lens(), shared_prefix_blocks=13, n_layers=n_layers,
                      nan_fill=nan_fill)


# the workloads by their index (1 tiny decode .. 5 prefix-shared tail), as bench.py --workload takes them
BY_INDEX = {1: tiny_decode, 2: qwen3_0_6b_decode, 3: qwen3_0_6b_mixed_step, 4: qwen3_8b_decode,
            5: prefix_shared_tail}


# ---- byte / flop accounting used by the benchmark -------------------------------

def kv_bytes(n_layers: int, n_kv_heads: int, head_dim: int, tokens: int, bytes_per_elem: int) -> int:
    """KV bytes = 2 (K and V) x layers x KV heads x head_dim x tokens x bytes/elem
    ("Модуль 04: KV-кэш и арифметика памяти", section 2.1)."""
    return 2 * n_layers * n_kv_heads * head_dim * tokens * bytes_per_elem


def decode_kv_bytes(context_lens: Sequence[int], hkv: int, elt: int = 2, unique_tokens: Optional[int] = None) -> int:
    """Algorithmic KV bytes one decode call must read: every visible key and
    value row once (per layer).  ``unique_tokens`` counts shared prefix pages once."""
    tokens = sum(context_lens) if unique_tokens is None else unique_tokens
    return kv_bytes(1, hkv, HEAD_DIM, tokens, elt)


def prefill_flops(chunks: Sequence[tuple], hq: int, head_dim: int = HEAD_DIM, window: int = 0) -> int:
    """Algorithmic FLOPs of causal chunk attention: 2 matmuls (QK^T and PV) x
    2 flops per multiply-add x head_dim x query heads x visible (query, key)
    pairs (with a sliding window of W keys the query at position p sees
    min(p + 1, W) keys)."""
    if window > 0:
        pairs = sum(min(s + i + 1, window) for s, n in chunks for i in range(n))
    else:
        pairs = sum(n * s + n * (n + 1) // 2 for s, n in chunks)
    return 4 * head_dim * hq * pairs
