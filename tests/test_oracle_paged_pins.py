"""Pins for the oracle's paged storage (p1 "A strong answer", the reversal
condition: a block table and a paged kernel; p3 "Design choices worth
noticing": the paged cache).

Paged storage only moves where tokens live: any page assignment must give
the ordinary cache's result exactly; rows whose tables share prefix pages
must equal rows that hold copies of that prefix; an append writes only the
pages its row's table maps; an unmapped target page is rejected with
nothing written.
"""

import numpy as np
import pytest

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import workloads as wl


def _rand(seed, stream, shape):
    return wl.normal(seed, stream, shape).numpy()


def _calls(seed, B, n, hi):
    rng = np.random.default_rng(seed)
    return [rng.integers(0, hi + 1, size=B).astype(np.int64) for _ in range(n)]


@pytest.mark.parametrize("seed", range(6))
def test_any_page_assignment_equals_the_ordinary_cache(seed):
    B, Hkv, G, d, P, mpr = 3, 2, 2, 8, 4, 8
    rng = np.random.default_rng(seed)
    num_pages = B * mpr + 5
    table = rng.permutation(num_pages)[: B * mpr].reshape(B, mpr)
    paged = ref.PagedOracleCache(1, B, Hkv, P, num_pages, mpr, d)
    paged.set_block_table(table)
    plain = ref.OracleCache(1, B, Hkv, P * mpr, d)
    for ci, n_new in enumerate(_calls(seed, B, 8, 4)):
        T = max(int(n_new.max()), 1)
        k, v = _rand(seed, 10 + ci, (B, Hkv, T, d)), _rand(seed, 50 + ci, (B, Hkv, T, d))
        q = _rand(seed, 90 + ci, (B, Hkv * G, T, d))
        a = ref.paged_append_attention(paged, 0, q, k, v, n_new)
        b = ref.append_attention(plain, 0, q, k, v, n_new)
        assert np.array_equal(a, b)


def test_shared_prefix_pages_equal_copied_prefixes():
    B, Hkv, G, d, P, mpr = 2, 1, 2, 8, 4, 4
    prefix, tail = 8, 5
    shared = ref.PagedOracleCache(1, B, Hkv, P, 12, mpr, d)
    # both rows read the prefix from pages 0 and 1; their own tails go to different pages
    shared.set_block_table([[0, 1, 2, 3], [0, 1, 4, 5]])
    kp, vp = _rand(1, 1, (1, Hkv, prefix, d)), _rand(1, 2, (1, Hkv, prefix, d))
    shared.append(0, np.concatenate([kp, kp]), np.concatenate([vp, vp]), [prefix, 0])
    shared.lens[0, 1] = prefix  # row 1 adopts the shared prefix
    copied = ref.OracleCache(1, B, Hkv, P * mpr, d)
    copied.append(0, np.concatenate([kp, kp]), np.concatenate([vp, vp]), [prefix, prefix])
    k, v = _rand(1, 3, (B, Hkv, tail, d)), _rand(1, 4, (B, Hkv, tail, d))
    q = _rand(1, 5, (B, Hkv * G, tail, d))
    a = ref.paged_append_attention(shared, 0, q, k, v, [tail, tail])
    b = ref.append_attention(copied, 0, q, k, v, [tail, tail])
    assert np.array_equal(a, b)


def test_append_touches_only_mapped_pages():
    B, Hkv, d, P, mpr = 2, 1, 4, 4, 3
    c = ref.PagedOracleCache(1, B, Hkv, P, 8, mpr, d)
    c.set_block_table([[5, 2, -1], [1, -1, -1]])
    for layer_k in c.k:
        layer_k[:] = 7.0
    k = np.ones((B, Hkv, 6, d))
    c.append(0, k, k, [6, 3])
    touched = {5, 2, 1}
    for page in range(8):
        if page not in touched:
            assert np.all(c.k[0][page] == 7.0)
    assert np.all(c.k[0][5] == 1.0) and np.all(c.k[0][2, :, :2] == 1.0) and np.all(c.k[0][2, :, 2:] == 7.0)


def test_unmapped_page_rejected():
    c = ref.PagedOracleCache(1, 1, 1, 4, 4, 2, 4)
    c.set_block_table([[3, -1]])
    z = np.zeros((1, 1, 6, 4))
    with pytest.raises(ref.CacheError):
        c.append(0, z, z, [6])
    assert list(c.lens[0]) == [0] and np.all(c.k[0] == 0)
    with pytest.raises(ref.CacheError):
        c.set_block_table([[4, 0]])
