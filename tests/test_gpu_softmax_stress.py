"""Online-softmax stress on the GPU against the oracle: scores that grow along
the sequence (the running maximum moves in every key tile, so the prefill's
lazy rescale and the decode's per-page rescale fire over and over), scores
that shrink (the first key dominates), and very peaked rows (most weights
underflow to zero), for the prefill and both decode paths."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_cache_gb300 as pa
import workloads
from gpu_util import ORACLE_DTYPE, bits, check_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
D, BS = 128, 16
TDT = {"bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(autouse=True)
def _clean_error_word():
    pa.get_device_error()
    yield
    st, detail = pa.get_device_error()
    assert st == 0, f"unexpected device error {pa.STATUS.get(st, st)} at index {detail}"


def _ramp_keys(n, hkv, slope, dtype, seed):
    """Keys along one unit direction u with magnitude slope * (position - n / 2), plus noise."""
    g = torch.Generator().manual_seed(seed)
    u = torch.randn(D, generator=g)
    u = u / u.norm()
    pos = torch.arange(n, dtype=torch.float32)[:, None, None]
    k = u[None, None, :] * slope * (pos - n / 2) + 0.05 * torch.randn((n, hkv, D), generator=g)
    return k.to(TDT[dtype]), u


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("slope", [0.05, -0.05, 0.4])
def test_prefill_with_moving_maximum(dtype, slope):
    n, hq, hkv = 512, 16, 8
    case = workloads.build_case("ramp-prefill", dtype, hq, hkv, seed=7, device=DEV, chunks=[(0, n)])
    k, u = _ramp_keys(n, hkv, slope, dtype, seed=8)
    q = (u[None, None, :] * 6.0 + 0.05 * torch.randn((n, hq, D), generator=torch.Generator().manual_seed(9)))
    q = q.to(TDT[dtype]).to(DEV)
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    pa.kv_cache_write(k.to(DEV), case.v_new[0], case.slot_mapping, kc, vc)
    out = pa.paged_attn_prefill_chunk(q, case.chunk_starts, case.chunk_lens, kc, vc, case.chunk_block_tables,
                                      case.chunk_context_lens, case.scale, max_chunk_len=n)
    torch.cuda.synchronize()
    ref = oracle.paged_attn_prefill(bits(q), bits(kc), bits(vc), case.chunk_starts.cpu().numpy(),
                                    case.chunk_lens.cpu().numpy(), case.chunk_block_tables.cpu().numpy(),
                                    case.chunk_context_lens.cpu().numpy(), case.scale, ORACLE_DTYPE[dtype])
    check_close(out, ref, f"prefill, slope {slope}, {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("slope", [0.05, -0.05, 0.4])
@pytest.mark.parametrize("bound", [None, 16384])
def test_decode_with_moving_maximum(dtype, slope, bound):
    lens, hq, hkv = [3000, 777, 40], 32, 8
    case = workloads.build_case("ramp-decode", dtype, hq, hkv, seed=10, device=DEV, decode_lens=lens)
    kc, vc = case.k_cache[0].clone(), case.v_cache[0].clone()
    bt = case.block_tables.cpu().numpy()
    g = torch.Generator().manual_seed(11)
    qs = []
    for s, n in enumerate(lens):   # overwrite every key of each sequence with a ramp
        k, u = _ramp_keys(n, hkv, slope, dtype, seed=12 + s)
        j = np.arange(n)
        slots = torch.from_numpy(bt[s, j // BS].astype(np.int64) * BS + j % BS).to(DEV)
        vrows = torch.randn((n, hkv, D), generator=g).to(TDT[dtype]).to(DEV)
        pa.kv_cache_write(k.to(DEV), vrows, slots, kc, vc)
        qs.append(u[None, :] * 6.0 + 0.05 * torch.randn((hq, D), generator=g))
    q = torch.stack(qs).to(TDT[dtype]).to(DEV)
    wide = torch.full((3, 1024), -1, dtype=torch.int32, device=DEV)
    wide[:, :bt.shape[1]] = case.block_tables
    out = pa.paged_attn_decode(q, kc, vc, wide, case.context_lens, case.scale, max_context_len=bound or max(lens))
    torch.cuda.synchronize()
    ref = oracle.paged_attn_decode(bits(q), bits(kc), bits(vc), bt, case.context_lens.cpu().numpy(), case.scale,
                                   ORACLE_DTYPE[dtype])
    check_close(out, ref, f"decode, slope {slope}, {dtype}, bound {bound}")
