"""fp64 CPU oracle for paged-KV GQA attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (``paged_kv_gqa_cache_gb300``)
never does; the two share no code.  The arithmetic lives in ``oracle.c`` (plain
C, fp64, no fast-math); this module only compiles it with gcc and marshals
numpy arrays.

Sources are cited by page title and section:

* "Модуль 12: Финальный проект: мини-движок инференса", qwen_serve/paged.py
  (PagedKVCache docstring, write, read) and qwen_serve/model.py
  (Qwen3Model.forward attention loop) — layout, slot addressing, GQA map,
  causal mask on absolute positions.
* "Модуль 04: KV-кэш и арифметика памяти", section 1 (output formula),
  section 2.1 (KV byte formula), kv_cache.py ``attend`` (GQA by repeat),
  section 5 (``KV8Cache``: int8 codes with one fp32 scale per token and head).
* "Phase 10: LLMs from Scratch — Inference Optimization", step 2 (causal SDPA).

Every function here is pinned by ``tests/test_oracle_pins.py`` against things
other than itself: library decoders of the 16-bit formats, torch's
scaled-dot-product attention on a contiguous copy built by block-level
reshapes, closed-form special cases, invariants the pages state, and the
pages' printed KV byte counts (``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None
_luts: dict = {}

F16, BF16 = 0, 1


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile oracle.c into a shared library with gcc (portable flags only)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-Wall", "-o", tmp, src, "-lm", "-lpthread"])
        os.replace(tmp, out)
    return out


def open_library(path: str):
    """Load a compiled oracle and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = f64
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = f64
    lib.oracle_kv_cache_write.argtypes = [P, P, i64, i32, i32, i32, P, P, P, i64]
    lib.oracle_kv_cache_write.restype = i64
    lib.oracle_f64_to_16.argtypes = [f64, ctypes.c_int]
    lib.oracle_f64_to_16.restype = ctypes.c_uint16
    lib.oracle_qk_norm_rope_kv_write.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, i32, P, P, i64, i32, i32,
                                                 P, P, P, i64, i32, i32, i32]
    lib.oracle_qk_norm_rope_kv_write.restype = i64
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f64.restype = f64
    lib.oracle_f64_to_e4m3.argtypes = [f64]
    lib.oracle_f64_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_kv_cache_write_f8.argtypes = [P, P, P, P, i64, i32, i32, i32, P, P, i32, P, i64]
    lib.oracle_kv_cache_write_f8.restype = i64
    lib.oracle_paged_attn_decode_f8.argtypes = [P, i32, P, P, P, P, i64, i32, i32, i32, P, i32, P,
                                                i32, i32, f64, P, i32]
    lib.oracle_paged_attn_decode_f8.restype = ctypes.c_int
    lib.oracle_kv_block_copy.argtypes = [P, P, i64, i32, i32, i32, P, i64]
    lib.oracle_kv_block_copy.restype = i64
    lib.oracle_gather_head.argtypes = [P, P, ctypes.c_int, i64, i32, i32, i32, P, i32, i32, P, P]
    lib.oracle_gather_head.restype = ctypes.c_int
    lib.oracle_paged_attn_decode.argtypes = [P, i32, P, P, i64, i32, i32, i32, P, i32, P,
                                             i32, i32, f64, P, i32]
    lib.oracle_paged_attn_decode.restype = ctypes.c_int
    lib.oracle_paged_attn_prefill.argtypes = [P, i32, P, P, i64, i32, i32, i32, P, P, P,
                                              i32, P, i32, i32, f64, P, i32]
    lib.oracle_paged_attn_prefill.restype = ctypes.c_int
    lib.oracle_paged_attn_decode_window.argtypes = [P, i32, P, P, i64, i32, i32, i32, P, i32, P,
                                                    i32, i32, f64, i32, P, i32]
    lib.oracle_paged_attn_decode_window.restype = ctypes.c_int
    lib.oracle_paged_attn_prefill_window.argtypes = [P, i32, P, P, i64, i32, i32, i32, P, P, P,
                                                     i32, P, i32, i32, f64, i32, P, i32]
    lib.oracle_paged_attn_prefill_window.restype = ctypes.c_int
    lib.oracle_paged_attn_prefill_q8.argtypes = [P, i32, P, P, P, P, i64, i32, i32, i32, P, P, P, i32, P, i32, i32,
                                                 f64, P, i32]
    lib.oracle_paged_attn_prefill_q8.restype = ctypes.c_int
    lib.oracle_paged_attn_prefill_f8.argtypes = lib.oracle_paged_attn_prefill_q8.argtypes
    lib.oracle_paged_attn_prefill_f8.restype = ctypes.c_int
    lib.oracle_kv_cache_write_q8.argtypes = [P, P, P, P, i64, i32, i32, i32, P, P, i32, P, i64]
    lib.oracle_kv_cache_write_q8.restype = i64
    lib.oracle_gather_head_q8.argtypes = [P, P, P, P, i64, i32, i32, i32, P, i32, i32, P, P]
    lib.oracle_gather_head_q8.restype = ctypes.c_int
    lib.oracle_paged_attn_decode_q8.argtypes = [P, i32, P, P, P, P, i64, i32, i32, i32, P, i32, P,
                                                i32, i32, f64, P, i32]
    lib.oracle_paged_attn_decode_q8.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


class use_library:
    """Context manager: route this module's calls to another compiled oracle
    (the pin tests use it to show that a planted mistake is caught)."""

    def __init__(self, path: str):
        self.lib = open_library(path)

    def __enter__(self):
        global _lib
        _load()
        self.saved, _lib = _lib, self.lib
        _luts.clear()
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        _luts.clear()
        return False


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits(a) -> np.ndarray:
    """16-bit patterns of an fp16/bf16 array (numpy uint16/float16, or torch CPU tensor)."""
    if hasattr(a, "detach"):  # torch tensor: reinterpret its bytes, never convert values
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(a)
    if a.dtype.itemsize != 2:
        raise TypeError(f"expected a 16-bit array, got {a.dtype}")
    return a.view(np.uint16)


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


def widen(bits, dtype: int) -> np.ndarray:
    """Exact fp64 values of an array of 16-bit patterns (elementwise, via the C decoder)."""
    b = _bits(bits)
    if dtype not in _luts:
        fn = _load().oracle_bf16_to_f64 if dtype == BF16 else _load().oracle_f16_to_f64
        _luts[dtype] = np.fromiter((fn(x) for x in range(65536)), dtype=np.float64, count=65536)
    return _luts[dtype][b.reshape(-1)].reshape(b.shape)


def kv_cache_write(k_cache, v_cache, k, v, slot_mapping) -> int:
    """In-place write of new K/V rows into their slots (pool arrays as uint16 bits).

    k_cache, v_cache: uint16 [num_blocks, block_size, Hkv, d] (modified in place).
    k, v: [T, Hkv, d] 16-bit; slot_mapping: int64 [T].  Returns #skipped slots.
    """
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    nb, bs, hkv, d = k_cache.shape
    kb, vb = _bits(k), _bits(v)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return int(_load().oracle_kv_cache_write(_ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d,
                                             _ptr(kb), _ptr(vb), _ptr(sm), sm.shape[0]))


def f64_to_16(x: float, dtype: int) -> int:
    """The 16-bit pattern nearest to x (ties to even)."""
    return int(_load().oracle_f64_to_16(float(x), dtype))


def qk_norm_rope_kv_write(q, k, v, q_weight, k_weight, eps: float, cos_table, sin_table, positions,
                          slot_mapping, k_cache, v_cache, dtype: int):
    """q/k RMSNorm and rotary embedding at absolute positions, then the KV write
    ("Модуль 12", qwen_serve/model.py rms_norm / apply_rope / Qwen3Model.forward;
    "Модуль 04" section 4: rotate before storing), at the page's rounding points.

    q [T, Hq, d], k, v [T, Hkv, d], weights [d], tables [max_position, d]: 16-bit
    bit patterns.  k_cache, v_cache (uint16 pools) are modified in place.
    Returns (q_out bits [T, Hq, d], number of skipped tokens)."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    wq, wk, cs, sn = _bits(q_weight), _bits(k_weight), _bits(cos_table), _bits(sin_table)
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    T, hq, d = qb.shape
    nb, bs, hkv, dk = k_cache.shape
    assert dk == d and kb.shape == (T, hkv, d) and vb.shape == (T, hkv, d) and cs.shape[1] == d
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    out = np.zeros_like(qb)
    skipped = _load().oracle_qk_norm_rope_kv_write(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(wq), _ptr(wk), eps, _ptr(cs), _ptr(sn), cs.shape[0], _ptr(pos),
        _ptr(sm), T, hq, dtype, _ptr(out), _ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d)
    return out, int(skipped)


def kv_block_copy(k_pools, v_pools, pairs) -> int:
    """Copy-on-write block copy ("Модуль 12", qwen_serve/paged.py,
    SequenceCache._cow_copy): in every layer's pool (uint16 bit arrays
    [num_blocks, block_size, Hkv, d], modified in place) block dst receives
    block src, for each (src, dst) row of ``pairs`` in order.  Returns the
    number of pairs skipped (a block id outside the pool)."""
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    skipped = 0
    for k_cache, v_cache in zip(k_pools, v_pools):
        assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous and k_cache.shape == v_cache.shape
        nb, bs, hkv, d = k_cache.shape
        skipped = int(_load().oracle_kv_block_copy(_ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d, _ptr(pr),
                                                   pr.shape[0]))
    return skipped


def gather_head(k_cache, v_cache, dtype: int, block_table_row, kv_head: int, upto: int):
    """fp64 K/V rows of positions [0, upto) for one KV head (the page's ``read``)."""
    kc, vc = _bits(k_cache), _bits(v_cache)
    nb, bs, hkv, d = kc.shape
    bt = np.ascontiguousarray(block_table_row, dtype=np.int32)
    ko = np.zeros((upto, d), np.float64)
    vo = np.zeros((upto, d), np.float64)
    rc = _load().oracle_gather_head(_ptr(kc), _ptr(vc), dtype, nb, bs, hkv, d, _ptr(bt),
                                    kv_head, upto, _ptr(ko), _ptr(vo))
    if rc != 0:
        raise IndexError("block id outside the pool")
    return ko, vo


def paged_attn_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                      dtype: int, num_threads: int = 0) -> np.ndarray:
    """fp64 decode attention: q [S, Hq, d] → out [S, Hq, d]."""
    qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
    nb, bs, hkv, d = kc.shape
    s, hq, dq = qb.shape
    assert dq == d
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    assert bt.shape[0] == s and ctx.shape == (s,)
    out = np.zeros((s, hq, d), np.float64)
    rc = _load().oracle_paged_attn_decode(_ptr(qb), dtype, _ptr(kc), _ptr(vc), nb, bs, hkv, d,
                                          _ptr(bt), bt.shape[1], _ptr(ctx), s, hq, float(scale),
                                          _ptr(out), num_threads)
    if rc != 0:
        raise ValueError(f"oracle decode rejected its inputs (code {rc})")
    return out


def paged_attn_prefill(q, k_cache, v_cache, chunk_starts, chunk_lens, block_tables,
                       context_lens, scale: float, dtype: int, num_threads: int = 0) -> np.ndarray:
    """fp64 causal chunked-prefill attention: q [sum(chunk_lens), Hq, d] → out, same shape."""
    qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
    nb, bs, hkv, d = kc.shape
    rows, hq, dq = qb.shape
    assert dq == d
    cs = np.ascontiguousarray(chunk_starts, dtype=np.int32)
    cl = np.ascontiguousarray(chunk_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    assert int(cl.sum()) == rows and bt.shape[0] == cs.shape[0] == ctx.shape[0]
    out = np.zeros((rows, hq, d), np.float64)
    rc = _load().oracle_paged_attn_prefill(_ptr(qb), dtype, _ptr(kc), _ptr(vc), nb, bs, hkv, d,
                                           _ptr(cs), _ptr(cl), _ptr(bt), bt.shape[1], _ptr(ctx),
                                           cs.shape[0], hq, float(scale), _ptr(out), num_threads)
    if rc != 0:
        raise ValueError(f"oracle prefill rejected its inputs (code {rc})")
    return out


def paged_attn_decode_window(q, k_cache, v_cache, block_tables, context_lens, scale: float, window: int,
                             dtype: int, num_threads: int = 0) -> np.ndarray:
    """fp64 decode attention with a sliding window of ``window`` keys ("Модуль 04:
    KV-кэш и арифметика памяти", sections 4 and 5.2): sequence s sees positions
    max(0, ctx - window) .. ctx - 1; blocks wholly before them are never read."""
    qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
    nb, bs, hkv, d = kc.shape
    s, hq, dq = qb.shape
    assert dq == d
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((s, hq, d), np.float64)
    rc = _load().oracle_paged_attn_decode_window(_ptr(qb), dtype, _ptr(kc), _ptr(vc), nb, bs, hkv, d,
                                                 _ptr(bt), bt.shape[1], _ptr(ctx), s, hq, float(scale),
                                                 int(window), _ptr(out), num_threads)
    if rc != 0:
        raise ValueError(f"oracle decode rejected its inputs (code {rc})")
    return out


def paged_attn_prefill_window(q, k_cache, v_cache, chunk_starts, chunk_lens, block_tables, context_lens,
                              scale: float, window: int, dtype: int, num_threads: int = 0) -> np.ndarray:
    """fp64 causal chunked prefill with a sliding window: the row at position p
    sees keys max(0, p - window + 1) .. p (window 0: no window)."""
    qb, kc, vc = _bits(q), _bits(k_cache), _bits(v_cache)
    nb, bs, hkv, d = kc.shape
    rows, hq, dq = qb.shape
    cs = np.ascontiguousarray(chunk_starts, dtype=np.int32)
    cl = np.ascontiguousarray(chunk_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((rows, hq, d), np.float64)
    rc = _load().oracle_paged_attn_prefill_window(_ptr(qb), dtype, _ptr(kc), _ptr(vc), nb, bs, hkv, d,
                                                  _ptr(cs), _ptr(cl), _ptr(bt), bt.shape[1], _ptr(ctx),
                                                  cs.shape[0], hq, float(scale), int(window), _ptr(out),
                                                  num_threads)
    if rc != 0:
        raise ValueError(f"oracle prefill rejected its inputs (code {rc})")
    return out


def e4m3_to_f64(code: int) -> float:
    return float(_load().oracle_e4m3_to_f64(int(code) & 0xff))


def f64_to_e4m3(x: float) -> int:
    """The E4M3 pattern nearest to x (ties to even, saturating at 448)."""
    return int(_load().oracle_f64_to_e4m3(float(x)))


def kv_cache_write_f8(k_codes, v_codes, k_scale, v_scale, k, v, dtype: int, slot_mapping) -> int:
    """In-place write into an fp8 (E4M3) pool: scale = max|x| / 448 + 1e-8 per
    (token, KV head), code = e4m3(x / scale).  Codes uint8 [nb, 16, Hkv, d],
    scales fp32 [nb, Hkv, 16] (modified in place).  Returns #skipped slots."""
    for a, t in ((k_codes, np.uint8), (v_codes, np.uint8), (k_scale, np.float32), (v_scale, np.float32)):
        assert a.dtype == t and a.flags.c_contiguous
    nb, bs, hkv, d = k_codes.shape
    kb, vb = _bits(k), _bits(v)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return int(_load().oracle_kv_cache_write_f8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), nb, bs,
                                                hkv, d, _ptr(kb), _ptr(vb), dtype, _ptr(sm), sm.shape[0]))


def paged_attn_decode_f8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale: float,
                         dtype: int, num_threads: int = 0) -> np.ndarray:
    """fp64 decode over an fp8 (E4M3) pool: keys and values are e4m3 * scale."""
    qb = _bits(q)
    kc, vc = np.ascontiguousarray(k_codes, np.uint8), np.ascontiguousarray(v_codes, np.uint8)
    ks, vs = np.ascontiguousarray(k_scale, np.float32), np.ascontiguousarray(v_scale, np.float32)
    nb, bs, hkv, d = kc.shape
    s, hq, dq = qb.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((s, hq, d), np.float64)
    rc = _load().oracle_paged_attn_decode_f8(_ptr(qb), dtype, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb, bs, hkv,
                                             d, _ptr(bt), bt.shape[1], _ptr(ctx), s, hq, float(scale), _ptr(out),
                                             num_threads)
    if rc != 0:
        raise ValueError(f"oracle decode rejected its inputs (code {rc})")
    return out


def paged_attn_prefill_q8(q, k_codes, v_codes, k_scale, v_scale, chunk_starts, chunk_lens, block_tables,
                          context_lens, scale: float, dtype: int, num_threads: int = 0) -> np.ndarray:
    """fp64 causal chunked prefill over an int8 pool ("Модуль 04", section 5:
    keys and values are the dequantised fp32 numbers code * scale)."""
    qb = _bits(q)
    kc, vc = np.ascontiguousarray(k_codes, np.int8), np.ascontiguousarray(v_codes, np.int8)
    ks, vs = np.ascontiguousarray(k_scale, np.float32), np.ascontiguousarray(v_scale, np.float32)
    nb, bs, hkv, d = kc.shape
    rows, hq, dq = qb.shape
    cs = np.ascontiguousarray(chunk_starts, dtype=np.int32)
    cl = np.ascontiguousarray(chunk_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((rows, hq, d), np.float64)
    rc = _load().oracle_paged_attn_prefill_q8(_ptr(qb), dtype, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb, bs, hkv,
                                              d, _ptr(cs), _ptr(cl), _ptr(bt), bt.shape[1], _ptr(ctx), cs.shape[0],
                                              hq, float(scale), _ptr(out), num_threads)
    if rc != 0:
        raise ValueError(f"oracle prefill rejected its inputs (code {rc})")
    return out


def paged_attn_prefill_f8(q, k_codes, v_codes, k_scale, v_scale, chunk_starts, chunk_lens, block_tables,
                          context_lens, scale: float, dtype: int, num_threads: int = 0) -> np.ndarray:
    """fp64 causal chunked prefill over an fp8 (E4M3) pool: keys and values are
    e4m3 * scale, as in ``paged_attn_decode_f8``."""
    qb = _bits(q)
    kc, vc = np.ascontiguousarray(k_codes, np.uint8), np.ascontiguousarray(v_codes, np.uint8)
    ks, vs = np.ascontiguousarray(k_scale, np.float32), np.ascontiguousarray(v_scale, np.float32)
    nb, bs, hkv, d = kc.shape
    rows, hq, dq = qb.shape
    cs = np.ascontiguousarray(chunk_starts, dtype=np.int32)
    cl = np.ascontiguousarray(chunk_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((rows, hq, d), np.float64)
    rc = _load().oracle_paged_attn_prefill_f8(_ptr(qb), dtype, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb, bs, hkv,
                                              d, _ptr(cs), _ptr(cl), _ptr(bt), bt.shape[1], _ptr(ctx), cs.shape[0],
                                              hq, float(scale), _ptr(out), num_threads)
    if rc != 0:
        raise ValueError(f"oracle prefill rejected its inputs (code {rc})")
    return out


def kv_cache_write_q8(k_codes, v_codes, k_scale, v_scale, k, v, dtype: int, slot_mapping) -> int:
    """In-place quantising write into an int8 pool ("Модуль 04: KV-кэш и
    арифметика памяти", section 5, ``KV8Cache.write``).

    k_codes, v_codes: int8 [num_blocks, block_size, Hkv, d]; k_scale, v_scale:
    float32 [num_blocks, Hkv, block_size] (modified in place).  k, v: [T, Hkv, d]
    16-bit patterns of ``dtype``; slot_mapping: int64 [T].  Returns #skipped slots.
    """
    for a in (k_codes, v_codes):
        assert a.dtype == np.int8 and a.flags.c_contiguous
    for a in (k_scale, v_scale):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    nb, bs, hkv, d = k_codes.shape
    assert k_scale.shape == (nb, hkv, bs)
    kb, vb = _bits(k), _bits(v)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return int(_load().oracle_kv_cache_write_q8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale),
                                                nb, bs, hkv, d, _ptr(kb), _ptr(vb), dtype, _ptr(sm),
                                                sm.shape[0]))


def gather_head_q8(k_codes, v_codes, k_scale, v_scale, block_table_row, kv_head: int, upto: int):
    """Dequantised fp32 K/V rows (as fp64) of positions [0, upto) for one KV head."""
    nb, bs, hkv, d = k_codes.shape
    bt = np.ascontiguousarray(block_table_row, dtype=np.int32)
    ko = np.zeros((upto, d), np.float64)
    vo = np.zeros((upto, d), np.float64)
    rc = _load().oracle_gather_head_q8(_ptr(k_codes), _ptr(v_codes), _ptr(k_scale), _ptr(v_scale), nb, bs,
                                       hkv, d, _ptr(bt), kv_head, upto, _ptr(ko), _ptr(vo))
    if rc != 0:
        raise IndexError("block id outside the pool")
    return ko, vo


def paged_attn_decode_q8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale: float,
                         dtype: int, num_threads: int = 0) -> np.ndarray:
    """fp64 decode attention over an int8 pool: q [S, Hq, d] 16-bit → out [S, Hq, d]."""
    qb = _bits(q)
    nb, bs, hkv, d = k_codes.shape
    s, hq, dq = qb.shape
    assert dq == d and k_scale.shape == (nb, hkv, bs)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    assert bt.shape[0] == s and ctx.shape == (s,)
    out = np.zeros((s, hq, d), np.float64)
    kc, vc = np.ascontiguousarray(k_codes), np.ascontiguousarray(v_codes)
    ks, vs = np.ascontiguousarray(k_scale, dtype=np.float32), np.ascontiguousarray(v_scale, dtype=np.float32)
    rc = _load().oracle_paged_attn_decode_q8(_ptr(qb), dtype, _ptr(kc), _ptr(vc), _ptr(ks), _ptr(vs), nb, bs,
                                             hkv, d, _ptr(bt), bt.shape[1], _ptr(ctx), s, hq, float(scale),
                                             _ptr(out), num_threads)
    if rc != 0:
        raise ValueError(f"oracle decode rejected its inputs (code {rc})")
    return out


def kv_bytes(n_layers: int, n_kv_heads: int, head_dim: int, tokens: int, bytes_per_elem: int) -> int:
    """KV-cache bytes: K and V, per layer, per KV head, per dim, per token
    ("Модуль 04: KV-кэш и арифметика памяти", section 2.1)."""
    return 2 * n_layers * n_kv_heads * head_dim * tokens * bytes_per_elem
