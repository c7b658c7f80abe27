"""Host-side checks of the C-ABI (no GPU needed): the library loads, exports
every entry point include/pagedattn.h declares, and rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

import paged_kv_gqa_cache_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedattn.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_gqa_cache_gb300 import _build
    _build.build()
    return pa.load_library()


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_three_calls_and_helpers():
    names = declared_entry_points()
    for n in ("pa_kv_cache_write", "pa_paged_attn_decode", "pa_paged_attn_prefill_chunk",
              "pa_decode_workspace_bytes", "pa_get_device_error"):
        assert n in names


def test_binding_constants_match_the_header():
    text = open(HEADER).read()
    defines = dict(re.findall(r"#define (PA_[A-Z0-9_]+) (\d+)u?\b", text))
    assert int(defines["PA_DECODE_EARLY_PAGES"]) == pa.DECODE_EARLY_PAGES
    assert int(defines["PA_DECODE_ZEROED_WORKSPACE"]) == pa.DECODE_ZEROED_WORKSPACE
    assert int(defines["PA_HEAD_DIM"]) == 128 and int(defines["PA_BLOCK_SIZE"]) == 16
    codes = dict((name, int(v)) for name, v in re.findall(r"(PA_(?:OK|ERR_[A-Z_]+)) = (-?\d+)", text))
    assert codes == pa.STATUS_CODE


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), f"{name} declared in pagedattn.h but not exported"
    assert set(pa.EXPORTS) <= set(declared_entry_points())


def test_only_c_entry_points_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith("pa_")}
    assert ours == set(declared_entry_points())


def test_abi_version_and_status_strings(lib):
    assert lib.pa_abi_version() == 10
    for code in range(0, -12, -1):
        assert lib.pa_status_string(code).decode().startswith(pa.STATUS[code])


def _pool(**kw):
    d = dict(k_cache=4096, v_cache=8192, num_blocks=64, block_size=16, num_kv_heads=8, head_dim=128, dtype=0)
    d.update(kw)
    return pa.KVPool(**d)


P = 1 << 20  # a fake, 16-byte aligned "device" address; never dereferenced by these calls


@pytest.mark.parametrize("pool,expected", [
    (None, -1),
    (_pool(k_cache=0), -1),
    (_pool(dtype=7), -3),
    (_pool(block_size=32), -4),
    (_pool(head_dim=64), -4),
    (_pool(num_blocks=0), -2),
    (_pool(k_cache=4100), -9),
])
def test_write_rejects_bad_pools(lib, pool, expected):
    ref = ctypes.byref(pool) if pool is not None else None
    assert lib.pa_kv_cache_write(P, P, P, 4, ref, None) == expected


def test_write_rejects_bad_arguments(lib):
    pool = _pool()
    assert lib.pa_kv_cache_write(P, P, P, -1, ctypes.byref(pool), None) == -2
    assert lib.pa_kv_cache_write(P, P, P, 0, ctypes.byref(pool), None) == 0      # empty: no-op
    assert lib.pa_kv_cache_write(0, P, P, 4, ctypes.byref(pool), None) == -1
    assert lib.pa_kv_cache_write(P + 8, P, P, 4, ctypes.byref(pool), None) == -9
    assert lib.pa_kv_cache_write(P, P, P + 4, 4, ctypes.byref(pool), None) == -9


def test_decode_rejects_bad_arguments(lib):
    pool = _pool()
    ws = lib.pa_decode_workspace_bytes(4, 16, 8, 256)
    call = lambda **kw: lib.pa_paged_attn_decode(
        kw.get("q", P), ctypes.byref(kw.get("pool", pool)), kw.get("bt", P), kw.get("mb", 16), kw.get("ctx", P),
        kw.get("S", 4), kw.get("hq", 16), kw.get("mcl", 256), kw.get("scale", 0.088), kw.get("out", P),
        kw.get("ws", P), kw.get("wsb", ws), None)
    assert call(S=0) == 0
    assert call(S=-1) == -2
    assert call(q=0) == -1
    assert call(ws=0) == -5
    assert call(wsb=ws - 1) == -5       # checked before any CUDA call
    assert call(hq=12) == -2            # 12 % 8 != 0
    assert call(hq=24) == -4            # group of 3
    assert call(pool=_pool(num_kv_heads=2), hq=32) == -4      # group of 16
    assert call(mcl=300) == -2          # beyond the block table (16 * 16)
    assert call(mcl=0) == -2
    assert call(scale=float("nan")) == -2
    assert call(scale=0.0) == -2
    assert call(out=P + 2) == -9
    assert call(bt=P + 2) == -9


def test_prefill_rejects_bad_arguments(lib):
    pool = _pool()
    call = lambda **kw: lib.pa_paged_attn_prefill_chunk(
        kw.get("q", P), kw.get("cs", P), kw.get("cl", P), ctypes.byref(kw.get("pool", pool)), kw.get("bt", P),
        kw.get("mb", 128), kw.get("ctx", P), kw.get("C", 3), kw.get("hq", 16), kw.get("T", 1536),
        kw.get("mcl", 512), kw.get("scale", 0.088), kw.get("out", P), None)
    assert call(C=0) == 0
    assert call(C=-1) == -2
    assert call(mcl=513) == -2          # chunks are at most 512 tokens
    assert call(mcl=0) == -2
    assert call(cs=0) == -1
    assert call(hq=20) == -2
    assert call(T=0) == -2
    assert call(q=P + 8) == -9
    assert call(pool=_pool(dtype=2)) == -3


def test_workspace_size_is_pure_host_and_monotone(lib):
    a = lib.pa_decode_workspace_bytes(8, 16, 8, 1024)
    b = lib.pa_decode_workspace_bytes(64, 32, 8, 4096)
    assert 0 < a < b
    assert lib.pa_decode_workspace_bytes(8, 12, 8, 1024) == 0
    assert lib.pa_decode_workspace_bytes(-1, 16, 8, 1024) == 0


def _pool_q8(**kw):
    f = dict(k_cache=P, v_cache=P + 4096, k_scale=P + 8192, v_scale=P + 12288, num_blocks=64, block_size=16,
             num_kv_heads=8, head_dim=128)
    f.update(kw)
    return pa.KVPoolQ8(**f)


@pytest.mark.parametrize("fn", ["pa_kv_cache_write_q8", "pa_kv_cache_write_f8"])
def test_write_q8_rejects_bad_arguments(lib, fn):
    call = lambda pool=None, **kw: getattr(lib, fn)(
        kw.get("k", P), kw.get("v", P), kw.get("dtype", 0), kw.get("slots", P), kw.get("n", 4),
        ctypes.byref(pool or _pool_q8()), None)
    assert call(n=0) == 0
    assert call(n=-1) == -2
    assert call(k=0) == -1
    assert call(pool=_pool_q8(k_scale=0)) == -1
    assert call(dtype=2) == -3
    assert call(pool=_pool_q8(block_size=32)) == -4
    assert call(pool=_pool_q8(head_dim=64)) == -4
    assert call(pool=_pool_q8(v_scale=P + 4)) == -9
    assert call(slots=P + 4) == -9
    assert call(k=P + 2) == -9


@pytest.mark.parametrize("fn", ["pa_paged_attn_decode_q8", "pa_paged_attn_decode_f8"])
def test_decode_q8_rejects_bad_arguments(lib, fn):
    ws = lib.pa_decode_workspace_bytes(4, 16, 8, 256)
    call = lambda pool=None, **kw: getattr(lib, fn)(
        kw.get("q", P), kw.get("dtype", 1), ctypes.byref(pool or _pool_q8()), kw.get("bt", P), kw.get("mb", 16),
        kw.get("ctx", P), kw.get("S", 4), kw.get("hq", 16), kw.get("mcl", 256), kw.get("scale", 0.088),
        kw.get("out", P), kw.get("ws", P), kw.get("wsb", ws), None)
    assert call(S=0) == 0
    assert call(S=-1) == -2
    assert call(q=0) == -1
    assert call(dtype=5) == -3
    assert call(pool=_pool_q8(v_cache=0)) == -1
    assert call(ws=0) == -5
    assert call(wsb=ws - 1) == -5
    assert call(hq=24) == -4
    assert call(mcl=300) == -2
    assert call(scale=float("inf")) == -2
    assert call(out=P + 2) == -9


def test_decode_ex_checks_its_arguments(lib):
    pool = _pool()
    ws = lib.pa_decode_workspace_bytes(4, 16, 8, 256)
    call = lambda **kw: lib.pa_paged_attn_decode_ex(
        P, ctypes.byref(pool), P, 16, P, 4, 16, 256, 0.088, kw.get("window", 0), kw.get("kn"), kw.get("vn"),
        kw.get("flags", 1), kw.get("out", P), P, ws, None)
    assert call(kn=P) == -1 and call(vn=P) == -1   # k_new and v_new go together
    assert call(kn=P, vn=P, window=64) == -4       # the fused write takes no window
    assert call(flags=4) == -4 and call(flags=0x80000001) == -4   # bits beyond the two flags
    assert call(window=-1) == -2
    assert call(out=P + 2) == -9                   # the plain call's checks still apply, before any CUDA call
    assert call(kn=P + 8, vn=P, out=P) == -9


def test_decode_q8_ex_checks_its_arguments(lib):
    ws = lib.pa_decode_workspace_bytes(4, 16, 8, 256)
    call = lambda **kw: lib.pa_paged_attn_decode_q8_ex(
        P, kw.get("dtype", 1), ctypes.byref(_pool_q8()), kw.get("codes", 0), P, 16, P, 4, 16, 256, 0.088,
        kw.get("flags", 1), kw.get("out", P), P, ws, None)
    assert call(codes=2) == -4 and call(codes=-1) == -4
    assert call(flags=4) == -4
    assert call(dtype=3) == -3
    assert call(codes=1, out=P + 2) == -9 and call(codes=0, out=P + 2) == -9


def test_prefill_q8_checks_its_arguments(lib):
    call = lambda **kw: lib.pa_paged_attn_prefill_chunk_q8(
        kw.get("q", P), kw.get("dtype", 1), P, P, ctypes.byref(kw.get("pool", _pool_q8())), kw.get("codes", 0), P,
        128, P, kw.get("C", 3), kw.get("hq", 16), 1536, kw.get("mcl", 512), kw.get("scale", 0.088),
        kw.get("out", P), None)
    assert call(C=0) == 0                           # nothing to do
    assert call(codes=2) == -4 and call(codes=-1) == -4
    assert call(dtype=3) == -3
    assert call(C=-1) == -2
    assert call(hq=12) == -2 and call(hq=24) == -4  # not a multiple of Hkv; a ratio outside {1, 2, 4, 8}
    assert call(mcl=0) == -2 and call(mcl=513) == -2
    assert call(scale=float("nan")) == -2
    assert call(q=0) == -1
    assert call(q=P + 8) == -9 and call(out=P + 2, codes=1) == -9   # every check before any CUDA call


def test_mixed_step_checks_its_arguments(lib):
    pool = _pool()
    ws = lib.pa_mixed_step_workspace_bytes(512, 16, 8)
    assert ws > lib.pa_decode_workspace_bytes(512, 16, 8, 1024)     # the launch's counters, then the decode's
    assert lib.pa_mixed_step_workspace_bytes(6001, 16, 8) == 0       # over the sequence bound
    assert lib.pa_mixed_step_workspace_bytes(4, 12, 8) == 0
    ws = lib.pa_mixed_step_workspace_bytes(4, 16, 8)   # the calls below have 4 sequences

    def call(**kw):
        T, C, S = kw.get("T", 4), kw.get("C", 3), kw.get("S", 4)
        return lib.pa_mixed_step(
            ctypes.byref(kw.get("pool", pool)), kw.get("hq", 16), kw.get("scale", 0.088),
            kw.get("k", P), P, kw.get("slots", P), T,
            kw.get("qc", P), P, P, P, 128, P, C, 1536, kw.get("mcl", 512), kw.get("oc", P),
            kw.get("q", P), kw.get("kd", P), kw.get("vd", P), P, 64, P, S, kw.get("out", P),
            kw.get("ws", P), kw.get("wsb", ws), None)
    assert call(T=0, C=0, S=0) == 0                       # nothing to do
    assert call(T=-1) == -2 and call(C=257) == -2 and call(S=6001) == -2
    assert call(hq=12) == -2 and call(hq=24) == -4        # not a multiple of Hkv; a ratio outside {1, 2, 4, 8}
    assert call(scale=float("nan")) == -2
    assert call(k=0) == -1 and call(qc=0) == -1 and call(q=0) == -1
    assert call(kd=0) == -1                               # the sequences' new K and V go together
    assert call(kd=0, vd=0, ws=0) == -5                   # (both absent: already in the pool)
    assert call(k=0, T=0, ws=0) == -5                     # a part with no work reads none of its pointers
    assert call(mcl=513) == -2
    assert call(qc=P + 8) == -9 and call(out=P + 2) == -9 and call(slots=P + 4) == -9 and call(kd=P + 8) == -9
    assert call(ws=0) == -5 and call(wsb=ws - 1) == -5 and call(ws=P + 8) == -9   # every check before any CUDA call


def test_window_calls_check_their_arguments(lib):
    pool = _pool()
    ws = lib.pa_decode_workspace_bytes(4, 16, 8, 256)
    dec = lambda w, out=P: lib.pa_paged_attn_decode_window(P, ctypes.byref(pool), P, 16, P, 4, 16, 256, 0.088, w,
                                                           out, P, ws, None)
    pre = lambda w, q=P: lib.pa_paged_attn_prefill_chunk_window(q, P, P, ctypes.byref(pool), P, 128, P, 3, 16,
                                                                1536, 512, 0.088, w, P, None)
    assert dec(-1) == -2 and pre(-1) == -2      # a negative window
    assert dec(40, out=P + 2) == -9             # the plain calls' checks still apply, before any CUDA call
    assert pre(40, q=P + 8) == -9


def test_fused_rope_write_checks_its_arguments(lib):
    pool = _pool()
    call = lambda **kw: lib.pa_qk_norm_rope_kv_write(
        kw.get("q", P), P, P, P, P, kw.get("eps", 1e-6), P, P, kw.get("maxpos", 4096), P, kw.get("slots", P),
        kw.get("T", 4), kw.get("hq", 16), kw.get("q_out", P), ctypes.byref(kw.get("pool", pool)), None)
    assert call(T=0) == 0
    assert call(T=-1) == -2
    assert call(q=0) == -1
    assert call(hq=0) == -2
    assert call(maxpos=0) == -2
    assert call(eps=float("nan")) == -2
    assert call(eps=-1.0) == -2
    assert call(q_out=P + 8) == -9
    assert call(slots=P + 4) == -9
    assert call(pool=_pool(dtype=3)) == -3


def test_decode_append_checks_its_arguments(lib):
    pool = _pool()
    ws = lib.pa_decode_workspace_bytes(4, 16, 8, 256)
    call = lambda **kw: lib.pa_paged_attn_decode_append(
        P, kw.get("kn", P), kw.get("vn", P), ctypes.byref(pool), P, 16, P, kw.get("S", 4), 16, 256, 0.088, P, P,
        ws, None)
    assert call(S=0) == 0
    assert call(kn=0) == -1
    assert call(vn=0) == -1
    assert call(kn=P + 8) == -9


def test_header_is_plain_c_and_links_against_the_library(lib, tmp_path):
    # a C99 translation unit that includes the header, takes the address of every
    # declared entry point, links against the library and calls the pure-host ones
    names = declared_entry_points()
    src = tmp_path / "use_header.c"
    refs = "\n".join(f"  (entry_fn)&{n}," for n in names)
    src.write_text(f"""#include <stdio.h>
#include "pagedattn.h"
typedef void (*entry_fn)(void);
static const entry_fn table[] = {{
{refs}
}};
int main(void) {{
  pa_allocator *a = NULL;
  int32_t ids[3];
  if (pa_abi_version() != PA_ABI_VERSION) return 1;
  if (pa_allocator_create(64, &a) != PA_OK) return 2;
  if (pa_allocator_allocate(a, 3, ids) != PA_OK || ids[0] != 0 || ids[2] != 2) return 3;
  pa_allocator_destroy(a);
  printf("%d %s\\n", (int)(sizeof(table) / sizeof(table[0])), pa_status_string(PA_ERR_NO_BLOCKS));
  return 0;
}}
""")
    import subprocess
    exe = tmp_path / "use_header"
    include = os.path.join(ROOT, "include")
    libdir = os.path.dirname(pa.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", include, str(src),
                        "-o", str(exe), "-L", libdir, "-lpagedattn", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert run.stdout.split()[0] == str(len(names)) and "PA_ERR_NO_BLOCKS" in run.stdout
