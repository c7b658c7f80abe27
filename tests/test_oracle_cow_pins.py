"""Pins for the oracle's copy-on-write block copy ("Модуль 12: Финальный
проект: мини-движок инференса", qwen_serve/paged.py, SequenceCache._cow_copy:
the fresh block receives the old block's K and V in every layer, and the old
block is left as it was).  Checks:

* numpy's advanced-index assignment k[:, dst] = k[:, src] over the stacked
  layers (a library routine, not the oracle's loops);
* the source block and every block outside the pairs keep their bits;
* pairs with a block outside the pool are counted and skipped;
* pairs apply in order (a chain a -> b -> c leaves a's content in c);
* planted mistakes in mutated copies of the oracle fail this battery.
"""
import os

import numpy as np
import pytest

import oracle

BS, D = 16, 128


def _pools(layers, nb, hkv, seed):
    rng = np.random.default_rng(seed)
    k = [rng.integers(0, 1 << 16, size=(nb, BS, hkv, D), dtype=np.uint16) for _ in range(layers)]
    v = [rng.integers(0, 1 << 16, size=(nb, BS, hkv, D), dtype=np.uint16) for _ in range(layers)]
    return k, v


def _copy_vs_numpy(layers=3, nb=20, hkv=2, seed=0):
    k, v = _pools(layers, nb, hkv, seed)
    ks, vs = np.stack(k), np.stack(v)
    pairs = np.array([[3, 7], [0, 19], [12, 5]], np.int32)
    assert oracle.kv_block_copy(k, v, pairs) == 0
    ks[:, pairs[:, 1]] = ks[:, pairs[:, 0]]     # distinct dst, none a src: order does not matter
    vs[:, pairs[:, 1]] = vs[:, pairs[:, 0]]
    return np.array_equal(np.stack(k), ks) and np.array_equal(np.stack(v), vs)


def test_copy_matches_numpy_advanced_indexing():
    assert _copy_vs_numpy()


def _numpy_pin():
    assert _copy_vs_numpy(layers=2, nb=24, hkv=1, seed=5)


def test_source_and_untouched_blocks_keep_their_bits():
    k, v = _pools(2, 10, 8, seed=1)
    k0, v0 = [x.copy() for x in k], [x.copy() for x in v]
    oracle.kv_block_copy(k, v, [[4, 9]])
    for l in range(2):
        for b in range(10):
            want = 4 if b == 9 else b
            assert np.array_equal(k[l][b], k0[l][want]) and np.array_equal(v[l][b], v0[l][want])


def test_pairs_outside_the_pool_are_skipped():
    k, v = _pools(1, 6, 1, seed=2)
    k0 = k[0].copy()
    assert oracle.kv_block_copy(k, v, [[-1, 2], [1, 6], [5, 0]]) == 2
    assert np.array_equal(k[0][0], k0[5]) and np.array_equal(k[0][1:], k0[1:])


def test_pairs_apply_in_order():
    k, v = _pools(1, 4, 1, seed=3)
    k0 = k[0].copy()
    oracle.kv_block_copy(k, v, [[0, 1], [1, 2]])
    assert np.array_equal(k[0][2], k0[0])


# ---- planted mistakes ----------------------------------------------------------------

def _battery():
    failed = []
    for name, fn in [("numpy", _numpy_pin),
                     ("untouched", test_source_and_untouched_blocks_keep_their_bits),
                     ("skipped", test_pairs_outside_the_pool_are_skipped),
                     ("order", test_pairs_apply_in_order)]:
        try:
            fn()
        except Exception:
            failed.append(name)
    return failed


MUTATIONS = {
    "value-not-copied": ("      v_cache[dst * per_block + x] = v_cache[src * per_block + x];\n", ""),
    "last-element-dropped": ("    for (int64_t x = 0; x < per_block; ++x) {\n      k_cache[dst * per_block + x]",
                             "    for (int64_t x = 0; x < per_block - 1; ++x) {\n      k_cache[dst * per_block + x]"),
    "direction-swapped": ("      k_cache[dst * per_block + x] = k_cache[src * per_block + x];",
                          "      k_cache[src * per_block + x] = k_cache[dst * per_block + x];"),
}


def test_block_copy_battery_passes_on_the_real_oracle():
    assert _battery() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_block_copy_mistake_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTATIONS[name]
    assert src.count(old) == 1, f"mutation anchor not found: {old}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "liboracle_mut.so"))
    with oracle.use_library(lib):
        failed = _battery()
    assert failed, f"planted mistake '{name}' was not caught by any pin"
