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


def _library_row_limits():
    """The library's routing limits, read from its host source: query rows per KV head above
    which attention runs on the tcgen05 kernel (bf16, FP8), and the rows of the one MMA tile
    under which the split-KV kernel appends inside its attention launch."""
    import pathlib
    import re
    src = (pathlib.Path(bench.__file__).parent / "gqa_attention_preallocated_gb300" / "csrc" / "kvc_host.cu").read_text()
    bf16 = int(re.search(r"constexpr int kTcMinRows = (\d+);", src).group(1))
    fp8 = int(re.search(r"constexpr int kTcMinRowsFp8 = (\d+);", src).group(1))
    mt1 = int(re.search(r"pl->mt = pl->R <= (\d+) \? 1", src).group(1))
    assert re.search(r"pl\.mt == 1 && max_n > 0 && \(pl\.R <= tc_min_rows\(c\)", src)  # the fused-append rule
    return bf16, fp8, mt1


def test_bench_kernel_labels_follow_the_library_routing():
    bf16, fp8, mt1 = _library_row_limits()
    for kv_dtype, limit in (("bf16", bf16), ("fp8", fp8)):
        for t, g in ((1, 1), (2, 4), (4, 4), (8, 2), (4, 8), (8, 4), (8, 8), (16, 8)):
            w = bench.Workload("verify", verify_t=t, verify_g=g, kv_dtype=kv_dtype)
            rows = g * t
            assert w.tensor_core == (rows > limit), (kv_dtype, t, g)
            assert w.fused == (rows <= limit and rows <= mt1), (kv_dtype, t, g)
            assert w.kernel_source == ("prefill_tc.cu" if rows > limit else "decode_bf16.cu")
    # decode and long-context steps are one row per query head: split-KV with the append fused in
    for name in ("decode8b", "longctx"):
        for kv_dtype in ("bf16", "fp8"):
            w = bench.Workload(name, kv_dtype=kv_dtype)
            assert not w.tensor_core and w.fused
    assert bench.Workload("prefill").tensor_core
