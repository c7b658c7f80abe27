"""Python binding of libpagedattn (GQA attention over a paged KV cache, GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libpagedattn.so`` (built in-tree by ``_build.build()``).  Tensors
must be CUDA tensors; calls are enqueued on ``torch.cuda.current_stream()``.
There is no fallback: if the shared library is missing this module raises.

Calls (see include/pagedattn.h for the full contract):

* ``kv_cache_write(k, v, slot_mapping, k_cache, v_cache)``
* ``paged_attn_decode(q, k_cache, v_cache, block_tables, context_lens, scale, ...)``
* ``paged_attn_prefill_chunk(q, chunk_starts, chunk_lens, k_cache, v_cache,
  block_tables, context_lens, scale, ...)``
* ``kv_cache_write_q8`` / ``paged_attn_decode_q8`` on an int8 pool
  (``alloc_pool_q8``: codes plus one fp32 scale per token and KV head)
* ``kv_cache_write_f8`` / ``paged_attn_decode_f8`` on an fp8 pool
  (``alloc_pool_f8``: the same layout with E4M3 codes held as uint8)
* ``paged_attn_decode_window`` / ``paged_attn_prefill_chunk_window``: sliding window
* ``qk_norm_rope_kv_write``: q/k RMSNorm + rotary embedding fused into the KV write
* ``kv_block_copy(pools, pairs)``: copy-on-write block copy over every layer
* ``BlockAllocator`` / ``Sequence`` / ``build_step_tables``: the host-side block
  allocator and block-table builder (native code in the same library; no GPU)
* ``get_device_error()``
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedattn.so")

PA_F16, PA_BF16 = 0, 1
PA_OK = 0
STATUS = {0: "PA_OK", -1: "PA_ERR_NULL", -2: "PA_ERR_SHAPE", -3: "PA_ERR_DTYPE", -4: "PA_ERR_UNSUPPORTED",
          -5: "PA_ERR_WORKSPACE", -6: "PA_ERR_CUDA", -7: "PA_ERR_RANGE", -8: "PA_ERR_TIMEOUT",
          -9: "PA_ERR_ALIGN", -10: "PA_ERR_NO_BLOCKS", -11: "PA_ERR_STATE"}
STATUS_CODE = {v: k for k, v in STATUS.items()}
EXPORTS = ("pa_kv_cache_write", "pa_decode_workspace_bytes", "pa_paged_attn_decode",
           "pa_paged_attn_prefill_chunk", "pa_get_device_error", "pa_status_string",
           "pa_last_cuda_error", "pa_abi_version", "pa_paged_attn_decode_noalloc",
           "pa_decode_kernel_launches", "pa_kv_cache_write_q8", "pa_paged_attn_decode_q8",
           "pa_kv_cache_write_f8", "pa_paged_attn_decode_f8",
           "pa_paged_attn_decode_window", "pa_paged_attn_prefill_chunk_window", "pa_kv_block_copy",
           "pa_qk_norm_rope_kv_write", "pa_paged_attn_decode_append", "pa_selftest_bounded_wait",
           "pa_paged_attn_decode_ex", "pa_paged_attn_decode_q8_ex", "pa_prefill_workspace_bytes",
           "pa_paged_attn_prefill_chunk_ex", "pa_paged_attn_prefill_chunk_q8", "pa_mixed_step",
           "pa_mixed_step_workspace_bytes",
           "pa_allocator_create", "pa_allocator_destroy", "pa_allocator_allocate", "pa_allocator_retain",
           "pa_allocator_release", "pa_allocator_refcount", "pa_allocator_stats_get", "pa_allocator_take_copies",
           "pa_sequence_create", "pa_sequence_destroy", "pa_sequence_reserve", "pa_sequence_commit",
           "pa_sequence_adopt_prefix", "pa_sequence_fork", "pa_sequence_release", "pa_sequence_length",
           "pa_sequence_reserved", "pa_sequence_num_blocks", "pa_sequence_blocks", "pa_build_step_tables")


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({_status_string(status)})")


class KVPool(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


class KVPoolQ8(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class AllocatorStats(ctypes.Structure):
    _fields_ = [("total", ctypes.c_int32), ("free", ctypes.c_int32), ("used", ctypes.c_int32),
                ("shared", ctypes.c_int32), ("n_allocated", ctypes.c_int64), ("n_cow", ctypes.c_int64)]


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Load libpagedattn.so and declare the C signatures.  Works without a GPU
    (nothing is called); raises OSError if the library has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise OSError(f"libpagedattn.so not built at {path}; run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        pool_p = ctypes.POINTER(KVPool)
        q8_p = ctypes.POINTER(KVPoolQ8)
        lib.pa_kv_cache_write_q8.argtypes = [P, P, i32, P, i32, q8_p, P]
        lib.pa_kv_cache_write_q8.restype = i32
        lib.pa_paged_attn_decode_q8.argtypes = [P, i32, q8_p, P, i32, P, i32, i32, i32, ctypes.c_float, P, P,
                                                ctypes.c_size_t, P]
        lib.pa_paged_attn_decode_q8.restype = i32
        lib.pa_kv_cache_write_f8.argtypes = lib.pa_kv_cache_write_q8.argtypes
        lib.pa_kv_cache_write_f8.restype = i32
        lib.pa_paged_attn_decode_f8.argtypes = lib.pa_paged_attn_decode_q8.argtypes
        lib.pa_paged_attn_decode_f8.restype = i32
        lib.pa_paged_attn_decode_q8_ex.argtypes = [P, i32, q8_p, i32, P, i32, P, i32, i32, i32, ctypes.c_float,
                                                   ctypes.c_uint32, P, P, ctypes.c_size_t, P]
        lib.pa_paged_attn_decode_q8_ex.restype = i32
        lib.pa_kv_cache_write.argtypes = [P, P, P, i32, pool_p, P]
        lib.pa_kv_cache_write.restype = i32
        lib.pa_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.pa_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.pa_decode_kernel_launches.argtypes = [i32, i32, i32]
        lib.pa_decode_kernel_launches.restype = i32
        lib.pa_paged_attn_decode.argtypes = [P, pool_p, P, i32, P, i32, i32, i32, ctypes.c_float, P, P,
                                             ctypes.c_size_t, P]
        lib.pa_paged_attn_decode.restype = i32
        lib.pa_paged_attn_decode_window.argtypes = [P, pool_p, P, i32, P, i32, i32, i32, ctypes.c_float, i32, P,
                                                    P, ctypes.c_size_t, P]
        lib.pa_paged_attn_decode_window.restype = i32
        lib.pa_paged_attn_decode_append.argtypes = [P, P, P, pool_p, P, i32, P, i32, i32, i32, ctypes.c_float, P,
                                                    P, ctypes.c_size_t, P]
        lib.pa_paged_attn_decode_append.restype = i32
        lib.pa_paged_attn_decode_ex.argtypes = [P, pool_p, P, i32, P, i32, i32, i32, ctypes.c_float, i32, P, P,
                                                ctypes.c_uint32, P, P, ctypes.c_size_t, P]
        lib.pa_paged_attn_decode_ex.restype = i32
        lib.pa_paged_attn_decode_noalloc.argtypes = [P, pool_p, P, i32, P, i32, i32, i32, ctypes.c_float, P, P]
        lib.pa_paged_attn_decode_noalloc.restype = i32
        lib.pa_paged_attn_prefill_chunk.argtypes = [P, P, P, pool_p, P, i32, P, i32, i32, i32, i32,
                                                    ctypes.c_float, P, P]
        lib.pa_paged_attn_prefill_chunk.restype = i32
        lib.pa_paged_attn_prefill_chunk_window.argtypes = [P, P, P, pool_p, P, i32, P, i32, i32, i32, i32,
                                                           ctypes.c_float, i32, P, P]
        lib.pa_paged_attn_prefill_chunk_window.restype = i32
        lib.pa_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.pa_prefill_workspace_bytes.restype = ctypes.c_size_t
        lib.pa_paged_attn_prefill_chunk_ex.argtypes = [P, P, P, pool_p, P, i32, P, i32, i32, i32, i32,
                                                       ctypes.c_float, i32, P, P, ctypes.c_size_t, P]
        lib.pa_paged_attn_prefill_chunk_ex.restype = i32
        lib.pa_paged_attn_prefill_chunk_q8.argtypes = [P, i32, P, P, q8_p, i32, P, i32, P, i32, i32, i32, i32,
                                                       ctypes.c_float, P, P]
        lib.pa_paged_attn_prefill_chunk_q8.restype = i32
        lib.pa_qk_norm_rope_kv_write.argtypes = [P, P, P, P, P, ctypes.c_float, P, P, i32, P, P, i32, i32, P,
                                                 pool_p, P]
        lib.pa_qk_norm_rope_kv_write.restype = i32
        lib.pa_selftest_bounded_wait.argtypes = [ctypes.c_uint32, P]
        lib.pa_selftest_bounded_wait.restype = i32
        lib.pa_kv_block_copy.argtypes = [pool_p, i32, P, i32, P]
        lib.pa_kv_block_copy.restype = i32
        ip = ctypes.POINTER(i32)
        for name, args, res in (
                ("pa_allocator_create", [i32, ctypes.POINTER(P)], i32), ("pa_allocator_destroy", [P], None),
                ("pa_allocator_allocate", [P, i32, ip], i32), ("pa_allocator_retain", [P, i32], i32),
                ("pa_allocator_release", [P, i32], i32), ("pa_allocator_refcount", [P, i32], i32),
                ("pa_allocator_stats_get", [P, ctypes.POINTER(AllocatorStats)], i32),
                ("pa_allocator_take_copies", [P, ip, i32, ip], i32),
                ("pa_sequence_create", [P, ctypes.POINTER(P)], i32), ("pa_sequence_destroy", [P], None),
                ("pa_sequence_reserve", [P, i32, ctypes.POINTER(i64)], i32),
                ("pa_sequence_commit", [P, i32], i32), ("pa_sequence_adopt_prefix", [P, ip, i32], i32),
                ("pa_sequence_fork", [P, P], i32), ("pa_sequence_release", [P], i32),
                ("pa_sequence_length", [P], i32), ("pa_sequence_reserved", [P], i32),
                ("pa_sequence_num_blocks", [P], i32), ("pa_sequence_blocks", [P, ip, i32], i32),
                ("pa_build_step_tables", [ctypes.POINTER(P), i32, i32, ip, ip, ip, ip], i32)):
            fn = getattr(lib, name)
            fn.argtypes, fn.restype = args, res
        lib.pa_mixed_step_workspace_bytes.argtypes = [i32, i32, i32]
        lib.pa_mixed_step_workspace_bytes.restype = ctypes.c_size_t
        lib.pa_mixed_step.argtypes = [pool_p, i32, ctypes.c_float, P, P, P, i32,
                                      P, P, P, P, i32, P, i32, i32, i32, P,
                                      P, P, P, P, i32, P, i32, P, P, ctypes.c_size_t, P]
        lib.pa_mixed_step.restype = i32
        lib.pa_get_device_error.argtypes = [P, ctypes.POINTER(i32)]
        lib.pa_get_device_error.restype = i32
        lib.pa_status_string.argtypes = [i32]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_last_cuda_error.argtypes = []
        lib.pa_last_cuda_error.restype = i32
        lib.pa_abi_version.argtypes = []
        lib.pa_abi_version.restype = i32
        _lib = lib
        return lib


def _status_string(status: int) -> str:
    try:
        return load_library().pa_status_string(status).decode()
    except OSError:
        return "library not loaded"


def _check(status: int, what: str):
    if status != PA_OK:
        raise PagedAttnError(status, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


def _need(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def make_pool(k_cache: torch.Tensor, v_cache: torch.Tensor) -> KVPool:
    """Descriptor of one layer's pool: k_cache, v_cache [num_blocks, 16, Hkv, 128]."""
    _need(k_cache, "k_cache")
    _need(v_cache, "v_cache", k_cache.dtype)
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache must both be [num_blocks, block_size, num_kv_heads, head_dim]")
    nb, bs, hkv, d = k_cache.shape
    return KVPool(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, hkv, d, _dtype_code(k_cache))


def kv_cache_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, stream=None) -> None:
    """Write new K/V rows [T, Hkv, 128] into flat slots ``slot_mapping`` (int64 [T])."""
    pool = make_pool(k_cache, v_cache)
    _need(k, "k", k_cache.dtype)
    _need(v, "v", k_cache.dtype)
    _need(slot_mapping, "slot_mapping", torch.int64)
    T = slot_mapping.numel()
    if k.shape != (T, pool.num_kv_heads, pool.head_dim) or v.shape != k.shape:
        raise ValueError(f"k, v must be [{T}, {pool.num_kv_heads}, {pool.head_dim}]")
    lib = load_library()
    _check(lib.pa_kv_cache_write(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                                 ctypes.byref(pool), _stream(stream)), "pa_kv_cache_write")


def alloc_pool_q8(num_blocks: int, num_kv_heads: int, device=None):
    """An int8 pool ("Модуль 04: KV-кэш и арифметика памяти", section 5): K and V
    codes int8 [num_blocks, 16, Hkv, 128] and fp32 scales [num_blocks, Hkv, 16]."""
    dev = device or "cuda"
    codes = lambda: torch.zeros((num_blocks, 16, num_kv_heads, 128), dtype=torch.int8, device=dev)
    scales = lambda: torch.zeros((num_blocks, num_kv_heads, 16), dtype=torch.float32, device=dev)
    return codes(), codes(), scales(), scales()


def alloc_pool_f8(num_blocks: int, num_kv_heads: int, device=None):
    """An fp8 pool: the int8 pool's layout with E4M3 codes stored as uint8."""
    k, v, ks, vs = alloc_pool_q8(num_blocks, num_kv_heads, device)
    return k.view(torch.uint8), v.view(torch.uint8), ks, vs


def make_pool_q8(k_codes, v_codes, k_scale, v_scale, code_dtype=torch.int8) -> KVPoolQ8:
    _need(k_codes, "k_codes", code_dtype)
    _need(v_codes, "v_codes", code_dtype)
    _need(k_scale, "k_scale", torch.float32)
    _need(v_scale, "v_scale", torch.float32)
    if k_codes.dim() != 4 or k_codes.shape != v_codes.shape:
        raise ValueError("k_codes and v_codes must both be [num_blocks, block_size, num_kv_heads, head_dim]")
    nb, bs, hkv, d = k_codes.shape
    if k_scale.shape != (nb, hkv, bs) or v_scale.shape != k_scale.shape:
        raise ValueError(f"k_scale and v_scale must be [{nb}, {hkv}, {bs}]")
    return KVPoolQ8(k_codes.data_ptr(), v_codes.data_ptr(), k_scale.data_ptr(), v_scale.data_ptr(), nb, bs, hkv, d)


def kv_cache_write_q8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_codes: torch.Tensor,
                      v_codes: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor, stream=None,
                      _fp8: bool = False) -> None:
    """Quantise new K/V rows [T, Hkv, 128] (fp16 / bf16) into flat slots of an int8 pool."""
    pool = make_pool_q8(k_codes, v_codes, k_scale, v_scale, torch.uint8 if _fp8 else torch.int8)
    _need(k, "k")
    _need(v, "v", k.dtype)
    _need(slot_mapping, "slot_mapping", torch.int64)
    T = slot_mapping.numel()
    if k.shape != (T, pool.num_kv_heads, pool.head_dim) or v.shape != k.shape:
        raise ValueError(f"k, v must be [{T}, {pool.num_kv_heads}, {pool.head_dim}]")
    lib = load_library()
    fn, name = (lib.pa_kv_cache_write_f8, "pa_kv_cache_write_f8") if _fp8 else \
        (lib.pa_kv_cache_write_q8, "pa_kv_cache_write_q8")
    _check(fn(k.data_ptr(), v.data_ptr(), _dtype_code(k), slot_mapping.data_ptr(), T, ctypes.byref(pool),
              _stream(stream)), name)


def paged_attn_decode_q8(q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor, k_scale: torch.Tensor,
                         v_scale: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                         scale: float, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                         max_context_len: Optional[int] = None, stream=None, _fp8: bool = False,
                         early_pages: bool = False, zeroed_workspace: bool = False) -> torch.Tensor:
    """Decode attention over an int8 pool: q [S, Hq, 128] (fp16 / bf16) → out, same dtype.
    ``early_pages`` and ``zeroed_workspace`` as for :func:`paged_attn_decode`."""
    pool = make_pool_q8(k_codes, v_codes, k_scale, v_scale, torch.uint8 if _fp8 else torch.int8)
    _need(q, "q")
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    S, hq, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks], context_lens [S]")
    mb = block_tables.shape[1]
    mcl = int(max_context_len) if max_context_len is not None else mb * pool.block_size
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype)
    if workspace is None:
        workspace = alloc_decode_workspace(S, hq, pool.num_kv_heads, mcl, q.device)
    _need(workspace, "workspace")
    lib = load_library()
    wsb = workspace.numel() * workspace.element_size()
    flags = (DECODE_EARLY_PAGES if early_pages else 0) | (DECODE_ZEROED_WORKSPACE if zeroed_workspace else 0)
    if flags:
        _check(lib.pa_paged_attn_decode_q8_ex(q.data_ptr(), _dtype_code(q), ctypes.byref(pool), 1 if _fp8 else 0,
                                              block_tables.data_ptr(), mb, context_lens.data_ptr(), S, hq, mcl,
                                              float(scale), flags, out.data_ptr(), workspace.data_ptr(),
                                              wsb, _stream(stream)), "pa_paged_attn_decode_q8_ex")
        return out
    fn, name = (lib.pa_paged_attn_decode_f8, "pa_paged_attn_decode_f8") if _fp8 else \
        (lib.pa_paged_attn_decode_q8, "pa_paged_attn_decode_q8")
    _check(fn(q.data_ptr(), _dtype_code(q), ctypes.byref(pool), block_tables.data_ptr(), mb, context_lens.data_ptr(),
              S, hq, mcl, float(scale), out.data_ptr(), workspace.data_ptr(), wsb, _stream(stream)), name)
    return out


def kv_cache_write_f8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_codes: torch.Tensor,
                      v_codes: torch.Tensor, k_scale: torch.Tensor, v_scale: torch.Tensor, stream=None) -> None:
    """Quantise new K/V rows [T, Hkv, 128] (fp16 / bf16) into flat slots of an fp8 (E4M3) pool."""
    kv_cache_write_q8(k, v, slot_mapping, k_codes, v_codes, k_scale, v_scale, stream, _fp8=True)


def paged_attn_decode_f8(q: torch.Tensor, k_codes: torch.Tensor, v_codes: torch.Tensor, k_scale: torch.Tensor,
                         v_scale: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                         scale: float, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                         max_context_len: Optional[int] = None, stream=None,
                         early_pages: bool = False, zeroed_workspace: bool = False) -> torch.Tensor:
    """Decode attention over an fp8 (E4M3) pool: q [S, Hq, 128] (fp16 / bf16) → out, same dtype."""
    return paged_attn_decode_q8(q, k_codes, v_codes, k_scale, v_scale, block_tables, context_lens, scale, out,
                                workspace, max_context_len, stream, _fp8=True, early_pages=early_pages,
                                zeroed_workspace=zeroed_workspace)


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, max_context_len: int) -> int:
    return int(load_library().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, max_context_len))


def decode_kernel_launches(num_seqs: int, num_kv_heads: int, max_context_len: int, window: int = 0) -> int:
    """Kernels one decode call with these sizes launches on the current device
    (1: one cluster per sequence and KV head; 2: split-K then combine).  A
    window call plans like a plain call bounded by the window's pages (see
    pa_paged_attn_decode_window)."""
    if window > 0:
        max_context_len = min(max_context_len, 16 * ((window - 1) // 16 + 2))
    return int(load_library().pa_decode_kernel_launches(num_seqs, num_kv_heads, max_context_len))


def alloc_decode_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, max_context_len: int,
                           device=None) -> torch.Tensor:
    """A decode workspace, zero-filled (so it may also serve calls with
    ``zeroed_workspace=True``, which leave it zeroed)."""
    n = decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, max_context_len)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def paged_attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                      out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      max_context_len: Optional[int] = None, stream=None,
                      early_pages: bool = False, zeroed_workspace: bool = False) -> torch.Tensor:
    """Decode attention: q [S, Hq, 128] → out [S, Hq, 128] (pool dtype).

    ``max_context_len`` is a host-side bound on ``context_lens`` (no device
    sync is made to find it); it defaults to the block table's capacity.
    ``early_pages``: the caller promises that the work enqueued just before
    this call writes no page of a sequence but its last visible one (a
    decode step's KV write), so the pages may be fetched before it ends
    (``pa_paged_attn_decode_ex`` with ``PA_DECODE_EARLY_PAGES``).
    ``zeroed_workspace``: the caller promises that ``workspace`` was
    zero-filled (as :func:`alloc_decode_workspace` does) and only used by
    calls that did not time out since; the decode then runs as one kernel over
    all SMs that merges split sequences itself
    (``PA_DECODE_ZEROED_WORKSPACE``)."""
    return _decode(q, k_cache, v_cache, block_tables, context_lens, scale, 0, out, workspace, max_context_len,
                   stream, flags=_flags(early_pages, zeroed_workspace))


def paged_attn_decode_window(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float, window: int,
                             out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                             max_context_len: Optional[int] = None, stream=None,
                             zeroed_workspace: bool = False) -> torch.Tensor:
    """Decode attention over the last ``window`` keys of each sequence (window
    0: all of them); otherwise as :func:`paged_attn_decode`."""
    return _decode(q, k_cache, v_cache, block_tables, context_lens, scale, int(window), out, workspace,
                   max_context_len, stream, flags=_flags(False, zeroed_workspace))


def paged_attn_decode_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                             v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                             scale: float, out: Optional[torch.Tensor] = None,
                             workspace: Optional[torch.Tensor] = None, max_context_len: Optional[int] = None,
                             stream=None, early_pages: bool = False, zeroed_workspace: bool = False) -> torch.Tensor:
    """Write each sequence's new token (k_new, v_new [S, Hkv, 128]) at position
    context_lens[s] - 1 of its block table and decode, in one call; otherwise
    as :func:`paged_attn_decode`."""
    _need(k_new, "k_new", k_cache.dtype)
    _need(v_new, "v_new", k_cache.dtype)
    if k_new.shape != (q.shape[0], k_cache.shape[2], q.shape[2]) or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be [S, Hkv, 128]")
    return _decode(q, k_cache, v_cache, block_tables, context_lens, scale, 0, out, workspace, max_context_len,
                   stream, append=(k_new, v_new), flags=_flags(early_pages, zeroed_workspace))


DECODE_EARLY_PAGES = 1
DECODE_ZEROED_WORKSPACE = 2


def _flags(early_pages: bool, zeroed_workspace: bool) -> int:
    return (DECODE_EARLY_PAGES if early_pages else 0) | (DECODE_ZEROED_WORKSPACE if zeroed_workspace else 0)


def _decode(q, k_cache, v_cache, block_tables, context_lens, scale, window, out, workspace, max_context_len,
            stream, append=None, flags=0):
    pool = make_pool(k_cache, v_cache)
    _need(q, "q", k_cache.dtype)
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    S, hq, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks], context_lens [S]")
    mb = block_tables.shape[1]
    mcl = int(max_context_len) if max_context_len is not None else mb * pool.block_size
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype)
    if workspace is None:
        workspace = alloc_decode_workspace(S, hq, pool.num_kv_heads, mcl, q.device)
    _need(workspace, "workspace")
    lib = load_library()
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream))
    if flags:
        kn, vn = (append[0].data_ptr(), append[1].data_ptr()) if append is not None else (None, None)
        _check(lib.pa_paged_attn_decode_ex(q.data_ptr(), ctypes.byref(pool), block_tables.data_ptr(), mb,
                                           context_lens.data_ptr(), S, hq, mcl, float(scale), window, kn, vn,
                                           flags, out.data_ptr(), *ws), "pa_paged_attn_decode_ex")
    elif append is not None:
        _check(lib.pa_paged_attn_decode_append(q.data_ptr(), append[0].data_ptr(), append[1].data_ptr(),
                                               ctypes.byref(pool), block_tables.data_ptr(), mb,
                                               context_lens.data_ptr(), S, hq, mcl, float(scale), out.data_ptr(),
                                               *ws), "pa_paged_attn_decode_append")
    elif window:
        _check(lib.pa_paged_attn_decode_window(q.data_ptr(), ctypes.byref(pool), block_tables.data_ptr(), mb,
                                               context_lens.data_ptr(), S, hq, mcl, float(scale), window,
                                               out.data_ptr(), *ws), "pa_paged_attn_decode_window")
    else:
        _check(lib.pa_paged_attn_decode(q.data_ptr(), ctypes.byref(pool), block_tables.data_ptr(), mb,
                                        context_lens.data_ptr(), S, hq, mcl, float(scale), out.data_ptr(), *ws),
               "pa_paged_attn_decode")
    return out


def paged_attn_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                              block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                              out: Optional[torch.Tensor] = None, max_context_len: Optional[int] = None,
                              stream=None) -> torch.Tensor:
    """Decode attention for callers that cannot allocate device memory or pass
    a workspace: the library's fixed scratch array stands in for it (see
    include/pagedattn.h for its size limit and the set-up on first use).
    ``out`` should be preallocated by such callers."""
    pool = make_pool(k_cache, v_cache)
    _need(q, "q", k_cache.dtype)
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    S, hq, d = q.shape
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks], context_lens [S]")
    mb = block_tables.shape[1]
    mcl = int(max_context_len) if max_context_len is not None else mb * pool.block_size
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype)
    _check(load_library().pa_paged_attn_decode_noalloc(
        q.data_ptr(), ctypes.byref(pool), block_tables.data_ptr(), mb, context_lens.data_ptr(), S, hq, mcl,
        float(scale), out.data_ptr(), _stream(stream)), "pa_paged_attn_decode_noalloc")
    return out


def paged_attn_prefill_chunk(q: torch.Tensor, chunk_starts: torch.Tensor, chunk_lens: torch.Tensor,
                             k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                             context_lens: torch.Tensor, scale: float, out: Optional[torch.Tensor] = None,
                             max_chunk_len: int = 512, stream=None,
                             workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Causal chunked-prefill attention: q [sum(chunk_lens), Hq, 128] → out (pool dtype).

    With ``workspace`` (from :func:`alloc_prefill_workspace`: zero-filled, and
    kept zero by every call) the call runs as one launch balanced over the
    SMs (``pa_paged_attn_prefill_chunk_ex``)."""
    return _prefill(q, chunk_starts, chunk_lens, k_cache, v_cache, block_tables, context_lens, scale, 0, out,
                    max_chunk_len, stream, workspace)


def paged_attn_prefill_chunk_window(q: torch.Tensor, chunk_starts: torch.Tensor, chunk_lens: torch.Tensor,
                                    k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                                    context_lens: torch.Tensor, scale: float, window: int,
                                    out: Optional[torch.Tensor] = None, max_chunk_len: int = 512,
                                    stream=None, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Chunked prefill where the query at position p sees keys p - window + 1 .. p
    (window 0: all earlier keys); otherwise as :func:`paged_attn_prefill_chunk`."""
    return _prefill(q, chunk_starts, chunk_lens, k_cache, v_cache, block_tables, context_lens, scale, int(window),
                    out, max_chunk_len, stream, workspace)


def prefill_workspace_bytes(num_chunks: int, num_q_heads: int, num_kv_heads: int, max_chunk_len: int) -> int:
    return int(load_library().pa_prefill_workspace_bytes(num_chunks, num_q_heads, num_kv_heads, max_chunk_len))


def alloc_prefill_workspace(num_chunks: int, num_q_heads: int, num_kv_heads: int, max_chunk_len: int,
                            device=None) -> torch.Tensor:
    """A zero-filled workspace for the balanced prefill on the current device."""
    n = prefill_workspace_bytes(num_chunks, num_q_heads, num_kv_heads, max_chunk_len)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def _prefill(q, chunk_starts, chunk_lens, k_cache, v_cache, block_tables, context_lens, scale, window, out,
             max_chunk_len, stream, workspace=None):
    pool = make_pool(k_cache, v_cache)
    _need(q, "q", k_cache.dtype)
    for name, t in (("chunk_starts", chunk_starts), ("chunk_lens", chunk_lens),
                    ("block_tables", block_tables), ("context_lens", context_lens)):
        _need(t, name, torch.int32)
    C = chunk_starts.numel()
    if chunk_lens.numel() != C or context_lens.numel() != C or block_tables.dim() != 2 \
            or block_tables.shape[0] != C:
        raise ValueError("chunk metadata must have one entry (block-table row) per chunk")
    rows, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype)
    lib = load_library()
    args = (q.data_ptr(), chunk_starts.data_ptr(), chunk_lens.data_ptr(), ctypes.byref(pool),
            block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), C, hq, rows,
            int(max_chunk_len), float(scale))
    if workspace is not None:
        _need(workspace, "workspace")
        _check(lib.pa_paged_attn_prefill_chunk_ex(*args, window, out.data_ptr(), workspace.data_ptr(),
                                                  workspace.numel() * workspace.element_size(), _stream(stream)),
               "pa_paged_attn_prefill_chunk_ex")
    elif window:
        _check(lib.pa_paged_attn_prefill_chunk_window(*args, window, out.data_ptr(), _stream(stream)),
               "pa_paged_attn_prefill_chunk_window")
    else:
        _check(lib.pa_paged_attn_prefill_chunk(*args, out.data_ptr(), _stream(stream)),
               "pa_paged_attn_prefill_chunk")
    return out


def paged_attn_prefill_chunk_q8(q: torch.Tensor, chunk_starts: torch.Tensor, chunk_lens: torch.Tensor,
                                k_codes: torch.Tensor, v_codes: torch.Tensor, k_scale: torch.Tensor,
                                v_scale: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                scale: float, out: Optional[torch.Tensor] = None, max_chunk_len: int = 512,
                                stream=None, _fp8: bool = False) -> torch.Tensor:
    """Causal chunked-prefill attention over an int8 pool (``pa_paged_attn_prefill_chunk_q8``):
    q [sum(chunk_lens), Hq, 128] (fp16 / bf16) → out, same dtype."""
    pool = make_pool_q8(k_codes, v_codes, k_scale, v_scale, torch.uint8 if _fp8 else torch.int8)
    _need(q, "q")
    for name, t in (("chunk_starts", chunk_starts), ("chunk_lens", chunk_lens),
                    ("block_tables", block_tables), ("context_lens", context_lens)):
        _need(t, name, torch.int32)
    C = chunk_starts.numel()
    if chunk_lens.numel() != C or context_lens.numel() != C or block_tables.dim() != 2 \
            or block_tables.shape[0] != C:
        raise ValueError("chunk metadata must have one entry (block-table row) per chunk")
    rows, hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", q.dtype)
    _check(load_library().pa_paged_attn_prefill_chunk_q8(
        q.data_ptr(), _dtype_code(q), chunk_starts.data_ptr(), chunk_lens.data_ptr(), ctypes.byref(pool),
        1 if _fp8 else 0, block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), C, hq, rows,
        int(max_chunk_len), float(scale), out.data_ptr(), _stream(stream)), "pa_paged_attn_prefill_chunk_q8")
    return out


def paged_attn_prefill_chunk_f8(q: torch.Tensor, chunk_starts: torch.Tensor, chunk_lens: torch.Tensor,
                                k_codes: torch.Tensor, v_codes: torch.Tensor, k_scale: torch.Tensor,
                                v_scale: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                                scale: float, out: Optional[torch.Tensor] = None, max_chunk_len: int = 512,
                                stream=None) -> torch.Tensor:
    """Causal chunked-prefill attention over an fp8 (E4M3) pool; as :func:`paged_attn_prefill_chunk_q8`."""
    return paged_attn_prefill_chunk_q8(q, chunk_starts, chunk_lens, k_codes, v_codes, k_scale, v_scale,
                                       block_tables, context_lens, scale, out, max_chunk_len, stream, _fp8=True)


def mixed_step_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int) -> int:
    return int(load_library().pa_mixed_step_workspace_bytes(num_seqs, num_q_heads, num_kv_heads))


def alloc_mixed_step_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for :func:`mixed_step` (every call leaves it zero again)."""
    n = mixed_step_workspace_bytes(num_seqs, num_q_heads, num_kv_heads)
    if n == 0:
        raise ValueError("unsupported sizes for the mixed step")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def mixed_step(k_cache: torch.Tensor, v_cache: torch.Tensor, scale: float, workspace: torch.Tensor,
               k_chunks: Optional[torch.Tensor] = None, v_chunks: Optional[torch.Tensor] = None,
               chunk_slots: Optional[torch.Tensor] = None, q_chunks: Optional[torch.Tensor] = None,
               chunk_starts: Optional[torch.Tensor] = None, chunk_lens: Optional[torch.Tensor] = None,
               chunk_block_tables: Optional[torch.Tensor] = None, chunk_context_lens: Optional[torch.Tensor] = None,
               q: Optional[torch.Tensor] = None, k_dec: Optional[torch.Tensor] = None,
               v_dec: Optional[torch.Tensor] = None, block_tables: Optional[torch.Tensor] = None,
               context_lens: Optional[torch.Tensor] = None, out_chunks: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, max_chunk_len: int = 512, stream=None):
    """A whole mixed step in one persistent launch (``pa_mixed_step``): the
    write of the chunks' new tokens k_chunks / v_chunks [Tc, Hkv, 128] through
    chunk_slots, then the chunked prefill of q_chunks, beside the decode of q
    with each sequence's new token k_dec / v_dec [S, Hkv, 128] (None: already in
    the pool) written at position context_lens - 1.  Either part may be None.
    Returns (out_chunks, out)."""
    pool = make_pool(k_cache, v_cache)
    hkv = k_cache.shape[2]
    _need(workspace, "workspace")
    T = 0 if chunk_slots is None else chunk_slots.numel()
    if T:
        _need(chunk_slots, "chunk_slots", torch.int64)
        _need(k_chunks, "k_chunks", k_cache.dtype)
        _need(v_chunks, "v_chunks", k_cache.dtype)
    if q_chunks is not None:
        _need(chunk_starts, "chunk_starts", torch.int32)
    C = 0 if q_chunks is None else chunk_starts.numel()
    S = 0 if q is None else q.shape[0]
    hq = q_chunks.shape[1] if C else (q.shape[1] if S else hkv)
    if C:
        _need(q_chunks, "q_chunks", k_cache.dtype)
        for name, t in (("chunk_starts", chunk_starts), ("chunk_lens", chunk_lens),
                        ("chunk_block_tables", chunk_block_tables), ("chunk_context_lens", chunk_context_lens)):
            _need(t, name, torch.int32)
        if out_chunks is None:
            out_chunks = torch.empty_like(q_chunks)
        _need(out_chunks, "out_chunks", q_chunks.dtype)
    if S:
        _need(q, "q", k_cache.dtype)
        _need(block_tables, "block_tables", torch.int32)
        _need(context_lens, "context_lens", torch.int32)
        if (k_dec is None) != (v_dec is None):
            raise ValueError("k_dec and v_dec go together")
        if k_dec is not None:
            _need(k_dec, "k_dec", k_cache.dtype)
            _need(v_dec, "v_dec", k_cache.dtype)
        if out is None:
            out = torch.empty_like(q)
        _need(out, "out", q.dtype)
    ptr = lambda t, on: t.data_ptr() if (on and t is not None) else None
    _check(load_library().pa_mixed_step(
        ctypes.byref(pool), hq, float(scale), ptr(k_chunks, T), ptr(v_chunks, T), ptr(chunk_slots, T), T,
        ptr(q_chunks, C), ptr(chunk_starts, C), ptr(chunk_lens, C), ptr(chunk_block_tables, C),
        chunk_block_tables.shape[1] if C else 0, ptr(chunk_context_lens, C), C, q_chunks.shape[0] if C else 0,
        int(max_chunk_len), ptr(out_chunks, C),
        ptr(q, S), ptr(k_dec, S), ptr(v_dec, S), ptr(block_tables, S), block_tables.shape[1] if S else 0,
        ptr(context_lens, S), S, ptr(out, S),
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(stream)),
        "pa_mixed_step")
    return out_chunks, out


def selftest_bounded_wait(limit_us: int = 20000, stream=None) -> None:
    """Launch the library's bounded-wait self-test (a wait that must give up
    after ``limit_us`` and record PA_ERR_TIMEOUT); read it with get_device_error()."""
    _check(load_library().pa_selftest_bounded_wait(int(limit_us), _stream(stream)), "pa_selftest_bounded_wait")


def get_device_error(stream=None) -> Tuple[int, int]:
    """Synchronise the stream and return (status, detail) of the device error
    word, clearing it."""
    detail = ctypes.c_int32(0)
    st = load_library().pa_get_device_error(_stream(stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def raise_device_error(stream=None) -> None:
    st, detail = get_device_error(stream)
    if st != PA_OK:
        raise PagedAttnError(st, f"device error (index {detail})")


def qk_norm_rope_kv_write(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_norm_weight: torch.Tensor,
                          k_norm_weight: torch.Tensor, eps: float, cos_table: torch.Tensor, sin_table: torch.Tensor,
                          positions: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, q_out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q/k RMSNorm and rotary embedding at absolute positions, fused into the
    KV write: returns q_out (normed, rotated q; may be ``q`` itself) and stores
    the normed, rotated k and the unchanged v into their slots."""
    pool = make_pool(k_cache, v_cache)
    for name, t in (("q", q), ("k", k), ("v", v), ("q_norm_weight", q_norm_weight),
                    ("k_norm_weight", k_norm_weight), ("cos_table", cos_table), ("sin_table", sin_table)):
        _need(t, name, k_cache.dtype)
    _need(positions, "positions", torch.int32)
    _need(slot_mapping, "slot_mapping", torch.int64)
    T, hq, d = q.shape
    if k.shape != (T, pool.num_kv_heads, d) or v.shape != k.shape or positions.shape != (T,) \
            or slot_mapping.shape != (T,) or cos_table.dim() != 2 or cos_table.shape != sin_table.shape:
        raise ValueError("q [T, Hq, 128], k/v [T, Hkv, 128], positions/slot_mapping [T], tables [max_pos, 128]")
    if q_out is None:
        q_out = torch.empty_like(q)
    _need(q_out, "q_out", q.dtype)
    _check(load_library().pa_qk_norm_rope_kv_write(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), q_norm_weight.data_ptr(), k_norm_weight.data_ptr(), float(eps),
        cos_table.data_ptr(), sin_table.data_ptr(), cos_table.shape[0], positions.data_ptr(),
        slot_mapping.data_ptr(), T, hq, q_out.data_ptr(), ctypes.byref(pool), _stream(stream)),
        "pa_qk_norm_rope_kv_write")
    return q_out


# ---- copy-on-write block copy and the host-side block-table builder ---------------------

def kv_block_copy(pools, pairs: torch.Tensor, stream=None) -> None:
    """Copy block src onto block dst in K and V of every layer pool, for each
    row (src, dst) of ``pairs`` (int32 [n, 2] on the device).  ``pools`` is a
    sequence of (k_cache, v_cache) layer pools of one geometry."""
    descs = [make_pool(k, v) for k, v in pools]
    _need(pairs, "pairs", torch.int32)
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [n, 2] (src, dst)")
    arr = (KVPool * max(len(descs), 1))(*descs)
    _check(load_library().pa_kv_block_copy(arr, len(descs), pairs.data_ptr(), pairs.shape[0], _stream(stream)),
           "pa_kv_block_copy")


class BlockAllocator:
    """Host-side pool of ``num_blocks`` block ids with reference counts (the
    library's native allocator; no GPU involved)."""

    def __init__(self, num_blocks: int):
        self._lib = load_library()
        h = ctypes.c_void_p()
        _check(self._lib.pa_allocator_create(num_blocks, ctypes.byref(h)), "pa_allocator_create")
        self._h = h
        self._seqs = []

    @property
    def handle(self):
        return self._h

    def allocate(self, n: int = 1):
        out = (ctypes.c_int32 * max(n, 1))()
        _check(self._lib.pa_allocator_allocate(self._h, n, out), "pa_allocator_allocate")
        return list(out[:n])

    def retain(self, block: int) -> None:
        _check(self._lib.pa_allocator_retain(self._h, block), "pa_allocator_retain")

    def release(self, block: int) -> None:
        _check(self._lib.pa_allocator_release(self._h, block), "pa_allocator_release")

    def refcount(self, block: int) -> int:
        return int(self._lib.pa_allocator_refcount(self._h, block))

    def stats(self) -> dict:
        st = AllocatorStats()
        _check(self._lib.pa_allocator_stats_get(self._h, ctypes.byref(st)), "pa_allocator_stats_get")
        return {name: int(getattr(st, name)) for name, _ in AllocatorStats._fields_}

    def take_copies(self):
        """The recorded copy-on-write pairs [(src, dst), ...], cleared."""
        n = ctypes.c_int32()
        st = self._lib.pa_allocator_take_copies(self._h, None, 0, ctypes.byref(n))
        if st == PA_OK and n.value == 0:
            return []
        buf = (ctypes.c_int32 * (2 * n.value))()
        _check(self._lib.pa_allocator_take_copies(self._h, buf, n.value, ctypes.byref(n)),
               "pa_allocator_take_copies")
        return [(buf[2 * i], buf[2 * i + 1]) for i in range(n.value)]

    def sequence(self) -> "Sequence":
        return Sequence(self)

    def close(self) -> None:
        if self._h:
            for s in self._seqs:
                s.close()
            self._lib.pa_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Sequence:
    """One request's block table and committed length on a BlockAllocator."""

    def __init__(self, alloc: BlockAllocator):
        self._lib, self.alloc = alloc._lib, alloc
        h = ctypes.c_void_p()
        _check(self._lib.pa_sequence_create(alloc.handle, ctypes.byref(h)), "pa_sequence_create")
        self._h = h
        alloc._seqs.append(self)

    @property
    def handle(self):
        return self._h

    def reserve(self, n: int):
        """Room for n more tokens; returns their flat slots (block * 16 + offset)."""
        slots = (ctypes.c_int64 * max(n, 1))()
        _check(self._lib.pa_sequence_reserve(self._h, n, slots), "pa_sequence_reserve")
        return list(slots[:n])

    def commit(self, n: int) -> None:
        _check(self._lib.pa_sequence_commit(self._h, n), "pa_sequence_commit")

    def adopt_prefix(self, blocks) -> None:
        arr = (ctypes.c_int32 * max(len(blocks), 1))(*blocks)
        _check(self._lib.pa_sequence_adopt_prefix(self._h, arr, len(blocks)), "pa_sequence_adopt_prefix")

    def fork_from(self, other: "Sequence") -> None:
        _check(self._lib.pa_sequence_fork(self._h, other.handle), "pa_sequence_fork")

    def release(self) -> None:
        _check(self._lib.pa_sequence_release(self._h), "pa_sequence_release")

    @property
    def length(self) -> int:
        return int(self._lib.pa_sequence_length(self._h))

    @property
    def reserved(self) -> int:
        return int(self._lib.pa_sequence_reserved(self._h))

    @property
    def blocks(self):
        n = int(self._lib.pa_sequence_num_blocks(self._h))
        out = (ctypes.c_int32 * max(n, 1))()
        _check(self._lib.pa_sequence_blocks(self._h, out, n), "pa_sequence_blocks")
        return list(out[:n])

    def close(self) -> None:
        if self._h:
            self._lib.pa_sequence_destroy(self._h)
            self._h = None


def build_step_tables(seqs, max_blocks: int):
    """Host int32 arrays for the step's attention calls: block tables
    [n, max_blocks] (-1 padded), chunk starts (committed lengths), chunk lens
    (reserved tokens) and context lens (their sums)."""
    import numpy as np
    n = len(seqs)
    bt = np.empty((max(n, 1), max_blocks), np.int32)
    starts, lens, ctx = (np.empty(max(n, 1), np.int32) for _ in range(3))
    handles = (ctypes.c_void_p * max(n, 1))(*[s.handle for s in seqs])
    ip = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    _check(load_library().pa_build_step_tables(handles, n, max_blocks, ip(bt), ip(starts), ip(lens), ip(ctx)),
           "pa_build_step_tables")
    return bt[:n], starts[:n], lens[:n], ctx[:n]
