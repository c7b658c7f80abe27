"""The allocation-free decode entry point (pa_paged_attn_decode_noalloc).

Some callers cannot allocate device memory or hand the library a workspace: a
plugin inside a host application that owns all device memory, or a serving
step that must not allocate at all.  This entry point serves them with a
fixed scratch array inside the library.  The checks here call it through the
C-ABI:

* its output is bit-identical to pa_paged_attn_decode's on the same inputs
  (both run the same kernels; that reference call gets a NaN-filled workspace
  of its own, so neither side can lean on leftovers), and within tolerance of
  the fp64 oracle;
* on two calls in a row with different queries and lengths, so that scratch
  left behind by the first call would show in the second;
* every case runs the split-K path, the only one that touches the scratch
  (the tiny and Qwen3-0.6B workloads are pushed onto it by a wide block table
  and a length bound past the one-cluster limit);
* once the first call in the context has looked up the array's address, a
  call leaves the device's free memory unchanged: it allocates nothing;
* sizes beyond the array are refused with PA_ERR_WORKSPACE, enqueuing nothing.

This file is collected last (test_zz_...) so that, in a run that stops at the
first failure, a failure here comes after every other test has run.  It
depends on no other test and passes alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
import workloads
from gpu_util import ORACLE_DTYPE, bits, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc_c_call(q, kc, vc, bt, ctx, hq, mcl, scale, out):
    lib = pa.load_library()
    pool = pa.make_pool(kc, vc)
    return lib.pa_paged_attn_decode_noalloc(
        q.data_ptr(), ctypes.byref(pool), bt.data_ptr(), bt.shape[1], ctx.data_ptr(), q.shape[0], hq, mcl,
        ctypes.c_float(scale), out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _split_inputs(case):
    """Block table and length bound that put the call on the split-K path."""
    bt, mcl = case.block_tables, case.max_context_len
    if pa.decode_kernel_launches(bt.shape[0], case.hkv, mcl) != 2:
        wide = torch.full((bt.shape[0], 1024), -1, dtype=torch.int32, device=DEV)
        wide[:, :bt.shape[1]] = bt
        bt, mcl = wide, 16384
    assert pa.decode_kernel_launches(bt.shape[0], case.hkv, mcl) == 2
    return bt, mcl


def _second_inputs(case, seed):
    """New query values and shorter lengths for the second call (every position
    below the new lengths holds a cached token)."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    q2 = torch.randn(case.q[0].shape, generator=g, device=DEV, dtype=torch.float32).to(case.q[0].dtype)
    lens = case.context_lens.cpu().numpy()
    cut = np.random.default_rng(seed).integers(1, 40, size=lens.shape)
    lens2 = np.maximum(1, lens - cut).astype(np.int32)
    assert (lens2 != lens).all()
    return q2, torch.from_numpy(lens2).to(DEV)


@pytest.mark.parametrize("cfg", [1, 2, 4, 5])
def test_noalloc_decode_is_the_workspace_decode_on_two_different_calls(cfg):
    case = workloads.BY_INDEX[cfg](device=DEV, nan_fill=True)
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(case.k_new[0], case.v_new[0], case.slot_mapping, kc, vc)
    bt, mcl = _split_inputs(case)
    q2, ctx2 = _second_inputs(case, 100 + cfg)
    calls = [(case.q[0], case.context_lens), (q2, ctx2)]

    # the workspace entry point on the same inputs, each with a fresh NaN-filled workspace
    refs = []
    for q, ctx in calls:
        ws = pa.alloc_decode_workspace(q.shape[0], case.hq, case.hkv, mcl, q.device)
        ws.fill_(0xFF)
        refs.append(pa.paged_attn_decode(q, kc, vc, bt, ctx, case.scale, workspace=ws, max_context_len=mcl))
    outs = [torch.full_like(q, float("nan")) for q, _ in calls]
    torch.cuda.synchronize()

    # call 1 also does the context's one-time set-up (the scratch array's address)
    assert _noalloc_c_call(calls[0][0], kc, vc, bt, calls[0][1], case.hq, mcl, case.scale, outs[0]) == pa.PA_OK
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    assert _noalloc_c_call(calls[1][0], kc, vc, bt, calls[1][1], case.hq, mcl, case.scale, outs[1]) == pa.PA_OK
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, f"a call changed free device memory by {free_before - free_after} bytes"

    for i, (out, ref) in enumerate(zip(outs, refs)):
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
            f"{case.name}: no-alloc call {i + 1} differs from pa_paged_attn_decode"
    # and the second call against the oracle
    odt = ORACLE_DTYPE[case.dtype]
    ref64 = oracle.paged_attn_decode(bits(q2), bits(kc), bits(vc), bt.cpu().numpy(), ctx2.cpu().numpy(),
                                     case.scale, odt)
    check_close(outs[1], ref64, f"{case.name} no-alloc call 2 against the oracle")
    assert pa.get_device_error() == (0, 0)


def test_noalloc_rejects_calls_beyond_its_fixed_scratch():
    # 8 query heads per KV head: the split-K scratch alone exceeds the fixed array
    case = workloads.build_case("ratio8", "bf16", 64, 8, seed=3, device=DEV, decode_lens=[40, 50])
    assert pa.decode_workspace_bytes(2, 64, 8, case.max_context_len) > (32 << 20)
    out = torch.zeros_like(case.q[0])
    args = (case.k_cache[0], case.v_cache[0], case.block_tables, case.context_lens, case.hq, case.max_context_len,
            case.scale, out)
    assert _noalloc_c_call(case.q[0], *args) == pa.STATUS_CODE["PA_ERR_WORKSPACE"]
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0          # nothing was enqueued
