"""The benchmark's algorithmic work, checked against the oracle's definitions.

The FLOP count of a prefill step counts the visible (query, key) pairs only;
here that count is taken from the oracle's bottom-right causal mask, row by
row.  The decode byte count is the oracle's K/V byte formula over the live
lengths after the step's append.
"""

import numpy as np

import bench
import oracle.ref as ref
from gqa_attention_preallocated_gb300 import workloads as wl


def _pairs_by_mask(priors, n_new):
    return sum(int(ref.decode_causal_mask(int(n), int(p) + int(n)).sum()) for p, n in zip(priors, n_new))


def test_visible_pairs_equal_the_mask_count():
    rng = np.random.default_rng(0)
    for _ in range(20):
        B = int(rng.integers(1, 5))
        priors = rng.integers(0, 300, size=B)
        n_new = rng.integers(0, 70, size=B)
        assert bench.visible_pairs(priors, n_new) == _pairs_by_mask(priors, n_new)


def test_prefill_flops_full_and_ragged():
    for ragged in (False, True):
        w = bench.Workload("prefill", prefill_ragged=ragged)
        s = w.shape
        assert w.work(0) == 4 * s.d * w.Hq * _pairs_by_mask(w.lens0, w.n_new)
        if ragged:
            assert np.all((w.n_new >= 1) & (w.n_new <= 512)) and np.array_equal(w.n_new, wl.ragged_chunk(0, s.B))
        else:
            assert np.all(w.n_new == 512)


def test_decode_bytes_are_the_live_cache():
    w = bench.Workload("decode8b")
    s = w.shape
    for i in (0, 1, 255, 256):
        lens = w.lens0 + w.n_new * ((i % w.rollback_every) + 1)
        want = ref.kv_cache_bytes(1, 1, int(lens.sum()), s.Hkv, s.d, 2)
        assert w.work(i) == want
    # the FP8 cache reads one byte a value
    w8 = bench.Workload("decode8b", kv_dtype="fp8")
    assert w8.work(0) * 2 == w.work(0)
