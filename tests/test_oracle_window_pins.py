"""Pins for the oracle's sliding window and ring buffer (p2 "Write the causal
mask for a decode step...", "A strong answer" last paragraph and "Common
mistakes"; p3 "16. Prefill, decode and the KV cache", exercise 3).

Each check ties the windowed path to something other than itself: the plain
causal path it must reduce to, a single-key closed form, the linear cache it
must agree with when stored as a ring, PyTorch's attention with an explicit
band mask (float64), and closed-form mask counts.  A planted slot-index mask
(the p2 "Common mistakes" item) must fail.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import workloads as wl


def _rand(seed, stream, shape):
    return wl.normal(seed, stream, shape).numpy()


def _chunks(seed, B, n_calls, max_chunk):
    rng = np.random.default_rng(seed)
    return [rng.integers(0, max_chunk + 1, size=B).astype(np.int64) for _ in range(n_calls)]


def _run(cache, seed, G, calls):
    outs = []
    for ci, n_new in enumerate(calls):
        T = max(int(n_new.max()), 1)
        k = _rand(seed, 100 + 3 * ci, (cache.B, cache.Hkv, T, cache.d))
        v = _rand(seed, 101 + 3 * ci, (cache.B, cache.Hkv, T, cache.d))
        q = _rand(seed, 102 + 3 * ci, (cache.B, cache.Hkv * G, T, cache.d))
        outs.append(ref.append_attention(cache, 0, q, k, v, n_new))
    return outs


def test_wide_window_is_plain_causal():
    B, Hkv, G, d, L = 2, 2, 3, 8, 80
    calls = _chunks(1, B, 12, 6)
    plain = ref.OracleCache(1, B, Hkv, L, d)
    wide = ref.OracleCache(1, B, Hkv, L, d)
    wide.set_window(L)
    for a, b in zip(_run(plain, 1, G, calls), _run(wide, 1, G, calls)):
        assert np.array_equal(a, b)


def test_window_of_one_returns_own_value():
    B, Hkv, G, d = 2, 2, 2, 8
    c = ref.OracleCache(1, B, Hkv, 40, d)
    c.set_window(1)
    calls = _chunks(2, B, 5, 4)
    outs = _run(c, 2, G, calls)
    lens = np.zeros(B, dtype=np.int64)
    for n_new in calls:
        lens = lens + n_new
    n_last, out = calls[-1], outs[-1]
    for b in range(B):
        for h in range(Hkv * G):
            for t in range(int(n_last[b])):
                p = int(lens[b] - n_last[b] + t)
                assert np.array_equal(out[b, h, t], c.v[0][b, h // G, p])


@pytest.mark.parametrize("W,C", [(5, 8), (7, 16), (16, 16)])
def test_ring_equals_linear_with_the_same_window(W, C):
    B, Hkv, G, d = 3, 2, 2, 8
    max_chunk = C - W + 1
    calls = _chunks(3 + W, B, 25, max_chunk)
    total = int(sum(c.max() for c in calls)) + 1
    linear = ref.OracleCache(1, B, Hkv, total, d)
    linear.set_window(W)
    ring = ref.OracleCache(1, B, Hkv, C, d)
    ring.set_window(W, ring=True)
    for a, b in zip(_run(linear, 4, G, calls), _run(ring, 4, G, calls)):
        assert np.array_equal(a, b)
    assert np.any(ring.lens[0] > C)  # the ring wrapped during the run
    assert np.array_equal(ring.lens[0], linear.lens[0])


def test_slot_index_mask_is_caught(monkeypatch):
    """Masking by slot index instead of stored position (p2 "Common mistakes")
    agrees before the ring wraps and breaks after it."""
    W, C, B, Hkv, G, d = 5, 8, 2, 1, 2, 8

    def by_slot(stored, lens_b, p, window):
        slots = np.arange(stored.shape[0])
        ps = p % stored.shape[0]
        ok = (slots <= ps) & (slots > ps - window) & (stored >= 0)
        return np.nonzero(ok)[0]

    calls = _chunks(9, B, 12, C - W + 1)
    total = int(sum(c.max() for c in calls)) + 1
    linear = ref.OracleCache(1, B, Hkv, total, d)
    linear.set_window(W)
    want = _run(linear, 5, G, calls)
    monkeypatch.setattr(ref, "visible_slots", by_slot)
    ring = ref.OracleCache(1, B, Hkv, C, d)
    ring.set_window(W, ring=True)
    got = _run(ring, 5, G, calls)
    assert any(not np.allclose(a, b) for a, b in zip(want, got))


def test_window_against_library_attention():
    """PyTorch's float64 attention with an explicit band mask (keys p-W < j <= p)."""
    for seed in range(30):
        rng = np.random.default_rng(seed)
        Hkv, G, d = int(rng.integers(1, 3)), int(rng.integers(1, 4)), 8
        prior, T, W = int(rng.integers(0, 30)), int(rng.integers(1, 6)), int(rng.integers(1, 20))
        S = prior + T
        c = ref.OracleCache(1, 1, Hkv, S, d)
        c.set_window(W)
        k = _rand(seed, 1, (1, Hkv, S, d))
        v = _rand(seed, 2, (1, Hkv, S, d))
        q = _rand(seed, 3, (1, Hkv * G, T, d))
        if prior:
            ref.append_attention(c, 0, np.zeros((1, Hkv * G, prior, d)), k[:, :, :prior], v[:, :, :prior], [prior])
        got = ref.append_attention(c, 0, q, k[:, :, prior:], v[:, :, prior:], [T])
        mask = torch.zeros(T, S, dtype=torch.bool)
        for i in range(T):
            p = prior + i
            for j in range(S):
                mask[i, j] = (j <= p) and (j > p - W)
        kt = torch.from_numpy(k).repeat_interleave(G, dim=1)
        vt = torch.from_numpy(v).repeat_interleave(G, dim=1)
        want = F.scaled_dot_product_attention(torch.from_numpy(q), kt, vt, attn_mask=mask).numpy()
        assert np.max(np.abs(got - want)) < 1e-10, seed


@pytest.mark.parametrize("T,S,W", [(4, 4096, 1000), (8, 4096, 4096), (1, 100, 7), (5, 37, 3)])
def test_window_mask_counts(T, S, W):
    m = ref.decode_window_mask(T, S, W)
    assert int(m.sum()) == sum(min(W, S - T + i + 1) for i in range(T))
    if W >= S:
        assert np.array_equal(m, ref.decode_causal_mask(T, S))


def test_page_count_with_full_window():
    """p2's speculative-verify count: 6 of 16,384 entries masked (W covers S)."""
    m = ref.decode_window_mask(4, 4096, 4096)
    assert m.size - int(m.sum()) == 6


def test_ring_validation():
    c = ref.OracleCache(1, 1, 1, 8, 4)
    with pytest.raises(ref.CacheError):
        c.set_window(0, ring=True)
    c.set_window(5, ring=True)
    z = np.zeros((1, 1, 5, 4))
    with pytest.raises(ref.CacheError):
        c.append(0, z, z, [5])  # 5 > 8 - 5 + 1: the chunk does not fit beside its window
    for _ in range(5):
        c.append(0, z[:, :, :4], z[:, :, :4], [4])  # wraps freely
    assert int(c.lens[0, 0]) == 20
    with pytest.raises(ref.CacheError):
        c.truncate([15])  # more than 8 - 5 + 1 back
    c.truncate([16])
    with pytest.raises(ref.CacheError):
        c.set_window(5, ring=False)  # storage changes only when empty
    c.reset()
    c.set_window(0, ring=False)
