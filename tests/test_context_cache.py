"""Host-side checks (no GPU) of the per-context caches and of the order of the
allocation-free decode's checks.

The library keeps the device addresses of its own device variables (the error
word, the allocation-free decode's scratch array) per CUDA context, keyed on
the context's unique id (csrc/context_cache.h).  The cache is plain host code,
so a small C++ driver exercises it directly: a value is fetched once per
(device, context), fetched again when the same device is used from another
context (a driver-API context of a host application, or the primary context
recreated after cudaDeviceReset), never reused across devices, and not cached
when the fetch fails.
"""
import ctypes
import os
import subprocess

import pytest

import paged_kv_gqa_cache_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_gqa_cache_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include "context_cache.h"

static int fetches = 0;
static int next_value = 100;
static bool fail_next = false;

static bool fetch(int *v) {
  ++fetches;
  if (fail_next) { fail_next = false; return false; }
  *v = next_value++;
  return true;
}

#define CHECK(c) do { if (!(c)) { std::printf("FAIL line %d: %s\n", __LINE__, #c); return 1; } } while (0)

int main() {
  pa::ContextCache<int, 4> cache;
  int v = 0;
  // first use of (device 0, context 11): fetched once, then served from the cache
  CHECK(cache.get(0, 11, fetch, &v) && v == 100 && fetches == 1);
  CHECK(cache.get(0, 11, fetch, &v) && v == 100 && fetches == 1);
  // another device: its own entry
  CHECK(cache.get(1, 11, fetch, &v) && v == 101 && fetches == 2);
  CHECK(cache.get(0, 11, fetch, &v) && v == 100 && fetches == 2);
  // device 0 from another context (same device, new context id): fetched anew
  CHECK(cache.get(0, 12, fetch, &v) && v == 102 && fetches == 3);
  CHECK(cache.get(0, 12, fetch, &v) && v == 102 && fetches == 3);
  // back in the first context: the entry now belongs to context 12, so fetch again
  CHECK(cache.get(0, 11, fetch, &v) && v == 103 && fetches == 4);
  // a failed fetch caches nothing and leaves the previous entry untouched
  fail_next = true;
  v = -1;
  CHECK(!cache.get(0, 13, fetch, &v) && v == -1 && fetches == 5);
  CHECK(cache.get(0, 11, fetch, &v) && v == 103 && fetches == 5);
  CHECK(cache.get(0, 13, fetch, &v) && v == 104 && fetches == 6);
  // no context (id 0) and devices outside the table are refused without a fetch
  CHECK(!cache.get(0, 0, fetch, &v) && fetches == 6);
  CHECK(!cache.get(-1, 11, fetch, &v) && !cache.get(4, 11, fetch, &v) && fetches == 6);
  std::printf("ok\n");
  return 0;
}
"""


def test_context_cache_refetches_per_context(tmp_path):
    src = tmp_path / "driver.cpp"
    src.write_text(DRIVER)
    exe = tmp_path / "driver"
    r = subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-I", CSRC, str(src), "-o", str(exe),
                        "-pthread"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


@pytest.fixture(scope="module")
def lib():
    from paged_kv_gqa_cache_gb300 import _build
    _build.build()
    return pa.load_library()


P = 1 << 20  # a fake, 16-byte aligned "device" address; never dereferenced by these calls


def _noalloc(lib, q=P, pool=None, bt=P, ctx=P, n=4096, hq=64, mcl=4096, out=P):
    pool = pool or pa.KVPool(k_cache=P, v_cache=P, num_blocks=16384, block_size=16, num_kv_heads=8, head_dim=128,
                             dtype=1)
    return lib.pa_paged_attn_decode_noalloc(q, ctypes.byref(pool), bt, 256, ctx, n, hq, mcl, ctypes.c_float(0.088),
                                            out, None)


def test_noalloc_checks_arguments_before_its_scratch_size(lib):
    # 4096 sequences at a head ratio of 8 need far more than the fixed scratch
    assert pa.decode_workspace_bytes(4096, 64, 8, 4096) > (32 << 20)
    assert _noalloc(lib) == pa.STATUS_CODE["PA_ERR_WORKSPACE"]
    # the same oversized call with a bad argument returns that argument's error,
    # as pa_paged_attn_decode would
    assert _noalloc(lib, q=None) == pa.STATUS_CODE["PA_ERR_NULL"]
    assert _noalloc(lib, out=None) == pa.STATUS_CODE["PA_ERR_NULL"]
    assert _noalloc(lib, q=P + 8) == pa.STATUS_CODE["PA_ERR_ALIGN"]
    assert _noalloc(lib, hq=60) == pa.STATUS_CODE["PA_ERR_SHAPE"]
    assert _noalloc(lib, mcl=1 << 20) == pa.STATUS_CODE["PA_ERR_SHAPE"]
    assert _noalloc(lib, n=-1) == pa.STATUS_CODE["PA_ERR_SHAPE"]
    assert _noalloc(lib, n=0) == pa.PA_OK
