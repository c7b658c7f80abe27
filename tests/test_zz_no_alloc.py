"""The allocation-free decode entry point (pa_paged_attn_decode_noalloc).

It serves callers that cannot allocate device memory or pass a workspace, by
using a fixed scratch array inside the library.  These checks call it through
the C-ABI and compare its output with the workspace entry point
(pa_paged_attn_decode) on the same inputs, on two calls in a row (the second
call finds the first call's leftovers in the shared array), within the
tolerance the parity tests use.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_gqa_cache_gb300 as pa
import workloads
from gpu_util import check_close, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc_c_call(case, kc, vc, out):
    lib = pa.load_library()
    pool = pa.make_pool(kc, vc)
    return lib.pa_paged_attn_decode_noalloc(
        case.q[0].data_ptr(), ctypes.byref(pool), case.block_tables.data_ptr(), case.block_tables.shape[1],
        case.context_lens.data_ptr(), case.q[0].shape[0], case.hq, case.max_context_len, ctypes.c_float(case.scale),
        out.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cfg", [1, 4, 5])
def test_noalloc_decode_matches_the_workspace_entry_point_twice(cfg):
    case = workloads.BY_INDEX[cfg](device=DEV)
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    ref = pa.paged_attn_decode(case.q[0], kc, vc, case.block_tables, case.context_lens, case.scale,
                               max_context_len=case.max_context_len)
    torch.cuda.synchronize()
    ref64 = f64(ref)
    for call in range(2):
        out = torch.full_like(case.q[0], float("nan"))
        assert _noalloc_c_call(case, kc, vc, out) == pa.PA_OK
        torch.cuda.synchronize()
        check_close(out, ref64, f"{case.name} no-alloc call {call + 1}")
    assert pa.get_device_error() == (0, 0)


def test_noalloc_rejects_calls_beyond_its_fixed_scratch():
    # 8 query heads per KV head: the split-K scratch alone exceeds the fixed array
    case = workloads.build_case("ratio8", "bf16", 64, 8, seed=3, device=DEV, decode_lens=[40, 50])
    assert pa.decode_workspace_bytes(2, 64, 8, case.max_context_len) > (32 << 20)
    out = torch.zeros_like(case.q[0])
    st = _noalloc_c_call(case, case.k_cache[0], case.v_cache[0], out)
    assert st == pa.STATUS_CODE["PA_ERR_WORKSPACE"]
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0          # nothing was enqueued
