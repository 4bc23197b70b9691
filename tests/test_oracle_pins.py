"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

None of these compares the oracle with a retyped copy of itself.  They use
numbers the pages print (tests/golden/page_figures.json), closed forms,
invariants, special cases that reduce to a library routine (PyTorch's
scaled_dot_product_attention with its lower-right causal bias, in float64),
and brute force on small random inputs against that routine.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import workloads as wl

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")))


def _rand(seed, stream, shape):
    return wl.normal(seed, stream, shape).numpy()


def _fill_cache(seed, B, Hkv, G, d, max_len, calls):
    """Run a sequence of append+attend calls through the oracle; return outputs and cache."""
    cache = ref.OracleCache(1, B, Hkv, max_len, d)
    outs = []
    for ci, n_new in enumerate(calls):
        T = int(n_new.max()) if len(n_new) else 0
        k_new = _rand(seed, 100 + 3 * ci, (B, Hkv, T, d))
        v_new = _rand(seed, 101 + 3 * ci, (B, Hkv, T, d))
        q = _rand(seed, 102 + 3 * ci, (B, Hkv * G, T, d))
        outs.append((q, n_new.copy(), ref.append_attention(cache, 0, q, k_new, v_new, n_new)))
    return outs, cache


def _sdpa_row(q_rows, K, V, G):
    """Library attention for one row: q [Hq, n, d], K/V [Hkv, S, d], lower-right causal."""
    qt = torch.from_numpy(np.ascontiguousarray(q_rows))[None]
    kt = torch.from_numpy(np.ascontiguousarray(K))[None]
    vt = torch.from_numpy(np.ascontiguousarray(V))[None]
    n, S = qt.shape[2], kt.shape[2]
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=causal_lower_right(n, S), enable_gqa=(G > 1))
    return o[0].numpy()


# ---------------------------------------------------------------------------
# Pages' worked examples
# ---------------------------------------------------------------------------


def test_golden_byte_figures():
    g = GOLDEN
    i = g["llama31_8b_kv_bytes_per_token"]["inputs"]
    per_tok = ref.kv_cache_bytes(**i)
    assert per_tok == g["llama31_8b_kv_bytes_per_token"]["value"]
    copied_tokens = sum(range(4096))
    assert copied_tokens == g["concat_tokens_copied_4096_steps"]["value"]
    copied = copied_tokens * per_tok
    e = g["concat_bytes_copied_4096_steps"]
    assert abs(copied - e["value"]) <= e["rel_tol"] * e["value"]
    assert 4096 * per_tok == g["final_cache_4096_tokens_bytes"]["value"]
    e = g["concat_copy_seconds_at_3p35_tbs"]
    assert abs(2 * copied / e["bandwidth_bytes_per_s"] - e["value"]) <= e["rel_tol"] * e["value"] + 0.005
    assert ref.kv_cache_bytes(32, 32, 8192, 8, 128, 2) == g["reservation_32_rows_8192_tokens_bytes"]["value"]
    i = g["qwen3_0p6b_kv_bytes_per_token"]["inputs"]
    assert ref.kv_cache_bytes(**i) == g["qwen3_0p6b_kv_bytes_per_token"]["value"]
    assert ref.kv_cache_bytes(28, 1, 2048, 8, 128, 2) == g["qwen3_0p6b_kv_bytes_2048"]["value"]
    assert ref.kv_cache_bytes(28, 1, 32768, 8, 128, 2) == g["qwen3_0p6b_kv_bytes_32k"]["value"]
    e = g["gqa_vs_mha_8b_8k"]
    assert ref.kv_cache_bytes(32, 1, 8192, e["inputs"]["gqa_kv_heads"], 128, 2) == e["gqa_bytes"]
    assert ref.kv_cache_bytes(32, 1, 8192, e["inputs"]["mha_kv_heads"], 128, 2) == e["mha_bytes"]


def test_oracle_cache_bytes_matches_formula():
    c = ref.OracleCache(3, 2, 4, 10, 8)
    assert c.bytes() == ref.kv_cache_bytes(3, 2, 10, 4, 8, bytes_per_value=8)


def test_golden_mask_figures():
    e = GOLDEN["verify_t4_s4096_masked_entries"]
    m = ref.decode_causal_mask(e["T"], e["S"])
    assert m.size == e["total"] and int((~m).sum()) == e["masked"]
    e = GOLDEN["verify_t4_top_left_row0_visible"]
    assert int(ref.top_left_causal_mask(e["T"], e["S"])[0].sum()) == e["visible"]
    e = GOLDEN["prefix3_chunk2_mask"]
    assert np.array_equal(ref.decode_causal_mask(e["T"], e["S"]).astype(int), np.array(e["rows"]))


@pytest.mark.parametrize("T,S", [(1, 1), (1, 4096), (4, 4096), (8, 4096), (5, 37), (37, 37), (512, 1024)])
def test_mask_closed_forms(T, S):
    m = ref.decode_causal_mask(T, S)
    # masked count of a bottom-right causal T x S block (T <= S) is T(T-1)/2
    assert int((~m).sum()) == T * (T - 1) // 2
    if T == 1:
        assert m.all()  # decode: the single row needs no mask
    if T == S:
        assert np.array_equal(m, np.tril(np.ones((T, S), dtype=bool)))


# ---------------------------------------------------------------------------
# Incremental vs full-sequence (S = 37, T = 5) and the top-left control
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("Hkv,G", [(1, 1), (2, 4), (1, 8)])
def test_incremental_equals_full_causal(Hkv, G):
    S, T, d, seed = 37, 5, 16, 3
    Hq = Hkv * G
    k_all = _rand(seed, 1, (1, Hkv, S, d))
    v_all = _rand(seed, 2, (1, Hkv, S, d))
    q_all = _rand(seed, 3, (1, Hq, S, d))
    full_cache = ref.OracleCache(1, 1, Hkv, 64, d)
    full = ref.append_attention(full_cache, 0, q_all, k_all, v_all, np.array([S]))
    inc_cache = ref.OracleCache(1, 1, Hkv, 64, d)
    inc_cache.append(0, k_all[:, :, : S - T], v_all[:, :, : S - T], np.array([S - T]))
    inc = ref.append_attention(inc_cache, 0, q_all[:, :, S - T :], k_all[:, :, S - T :], v_all[:, :, S - T :], np.array([T]))
    assert np.max(np.abs(inc - full[:, :, S - T :])) == 0.0
    # full-sequence causal attention is the library routine with T == S
    lib = _sdpa_row(q_all[0], k_all[0], v_all[0], G)
    assert np.max(np.abs(full[0] - lib)) < 1e-12
    # top-left alignment on the same chunk is visibly wrong
    s = np.einsum("htd,hsd->hts", q_all[0, :, S - T :], np.repeat(k_all[0], G, axis=0)) / math.sqrt(d)
    s = np.where(ref.top_left_causal_mask(T, S)[None], s, -np.inf)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    top_left = np.einsum("hts,hsd->htd", p, np.repeat(v_all[0], G, axis=0))
    assert np.max(np.abs(top_left - inc[0])) > 1e-1


# ---------------------------------------------------------------------------
# Closed forms that pin scale, offset, head mapping, padding
# ---------------------------------------------------------------------------


def _ramp_case(priors, n_new, Hkv, G, d, ramp_head_const=False):
    """K = 0 (uniform weights) and V[j] = j: output of query t is mean(0..pos) = pos / 2."""
    B = len(priors)
    T = int(max(n_new)) if B else 0
    max_len = int(max(p + n for p, n in zip(priors, n_new))) + 3
    c = ref.OracleCache(1, B, Hkv, max_len, d)
    for b in range(B):
        for j in range(max_len):
            c.v[0][b, :, j, :] = j
        if ramp_head_const:
            for h in range(Hkv):
                c.v[0][b, h, :, :] = h
    c.lens[0] = np.asarray(priors) + np.asarray(n_new)
    q = _rand(5, 9, (B, Hkv * G, T, d))
    return c, q, ref.gqa_attention(q, c, 0, np.asarray(n_new))


def test_closed_form_offset_and_padding():
    priors, n_new, Hkv, G, d = [0, 7, 30], [5, 3, 0], 2, 3, 8
    _, _, out = _ramp_case(priors, n_new, Hkv, G, d)
    for b in range(3):
        for t in range(out.shape[2]):
            want = (priors[b] + t) / 2.0 if t < n_new[b] else 0.0
            assert np.allclose(out[b, :, t, :], want, rtol=0, atol=1e-12), (b, t)


def test_closed_form_head_mapping():
    Hkv, G = 4, 3
    _, _, out = _ramp_case([6], [2], Hkv, G, 4, ramp_head_const=True)
    for h in range(Hkv * G):
        assert np.allclose(out[0, h], h // G, atol=1e-12), h


def test_closed_form_scale_two_keys():
    d, a = 16, 4.0
    c = ref.OracleCache(1, 1, 1, 4, d)
    c.k[0][0, 0, 1, 0] = a  # key 0 = 0, key 1 = a * e0
    c.v[0][0, 0, 1, :] = 1.0  # value 0 = 0, value 1 = 1
    c.lens[0] = [2]
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    out = ref.gqa_attention(q, c, 0, np.array([1]))
    want = 1.0 / (1.0 + math.exp(-a / math.sqrt(d)))  # logistic(q.k1 / sqrt(d))
    assert abs(out[0, 0, 0, 0] - want) < 1e-15


def test_single_key_returns_its_value():
    c = ref.OracleCache(1, 1, 2, 8, 5)
    k_new = _rand(1, 1, (1, 2, 1, 5))
    v_new = _rand(1, 2, (1, 2, 1, 5))
    q = _rand(1, 3, (1, 6, 1, 5)) * 100.0
    out = ref.append_attention(c, 0, q, k_new, v_new, np.array([1]))
    for h in range(6):
        assert np.array_equal(out[0, h, 0], v_new[0, h // 3, 0])


def test_shift_invariance_and_large_scores():
    """Adding one vector u to every key shifts all scores of a query equally."""
    B, Hkv, G, d, S = 2, 2, 2, 8, 11
    k = _rand(2, 1, (B, Hkv, S, d))
    v = _rand(2, 2, (B, Hkv, S, d))
    q = _rand(2, 3, (B, Hkv * G, S, d)) * 30.0  # large logits: max-subtraction must hold
    c1 = ref.OracleCache(1, B, Hkv, S, d)
    o1 = ref.append_attention(c1, 0, q, k, v, np.array([S, S]))
    u = _rand(2, 4, (1, 1, 1, d)) * 5.0
    c2 = ref.OracleCache(1, B, Hkv, S, d)
    o2 = ref.append_attention(c2, 0, q, k + u, v, np.array([S, S]))
    assert np.all(np.isfinite(o1))
    assert np.max(np.abs(o1 - o2)) < 1e-9


# ---------------------------------------------------------------------------
# Brute force against the library routine (the pages' 200 randomized trials)
# ---------------------------------------------------------------------------


def _trial(seed):
    B, Hkv, G, d = wl.trial_geometry(seed)
    finals, calls = wl.tiny_schedule(seed, B)
    outs, cache = _fill_cache(seed, B, Hkv, G, d, 48, calls)
    lens = np.zeros(B, dtype=np.int64)
    n_cmp, worst = 0, 0.0
    for q, n_new, out in outs:
        lens = lens + n_new
        for b in range(B):
            n = int(n_new[b])
            S = int(lens[b])
            assert np.all(out[b, :, n:] == 0.0)
            if n == 0:
                continue
            lib = _sdpa_row(q[b, :, :n], cache.k[0][b, :, :S], cache.v[0][b, :, :S], G)
            worst = max(worst, float(np.max(np.abs(out[b, :, :n] - lib))))
            n_cmp += 1
    assert np.array_equal(cache.lens[0], finals)
    return n_cmp, worst


def test_randomized_trials_vs_library():
    total, worst = 0, 0.0
    for seed in range(200):
        n, w = _trial(seed)
        total += n
        worst = max(worst, w)
    assert worst <= 1e-10
    assert total > 500  # many per-row comparisons, like the pages' count


def test_mqa_and_mha_special_cases():
    for Hkv, G in [(1, 6), (5, 1)]:
        B, d, S = 2, 8, 13
        c = ref.OracleCache(1, B, Hkv, 20, d)
        k = _rand(7, 1, (B, Hkv, S, d))
        v = _rand(7, 2, (B, Hkv, S, d))
        c.append(0, k, v, np.array([S, S]))
        q = _rand(7, 3, (B, Hkv * G, 4, d))
        k2 = _rand(7, 4, (B, Hkv, 4, d))
        v2 = _rand(7, 5, (B, Hkv, 4, d))
        out = ref.append_attention(c, 0, q, k2, v2, np.array([4, 2]))
        for b, n in [(0, 4), (1, 2)]:
            lib = _sdpa_row(q[b, :, :n], c.k[0][b, :, : S + n], c.v[0][b, :, : S + n], G)
            assert np.max(np.abs(out[b, :, :n] - lib)) < 1e-12


# ---------------------------------------------------------------------------
# Cache semantics: overflow, empty cases, lengths, truncate
# ---------------------------------------------------------------------------


def test_overflow_raises_and_changes_nothing():
    c = ref.OracleCache(1, 3, 2, 10, 4)
    c.append(0, np.ones((3, 2, 8, 4)), np.ones((3, 2, 8, 4)), np.array([8, 2, 8]))
    k_before = c.k[0].copy()
    lens_before = c.lens.copy()
    with pytest.raises(ref.CacheError):
        c.append(0, np.full((3, 2, 3, 4), 7.0), np.full((3, 2, 3, 4), 7.0), np.array([1, 1, 3]))
    assert np.array_equal(c.lens, lens_before)
    assert np.array_equal(c.k[0], k_before)  # row 0 and row 1 were not written either


@pytest.mark.parametrize("bad", [np.array([4, 0]), np.array([-1, 0])])
def test_bad_n_new_rejected(bad):
    c = ref.OracleCache(1, 2, 1, 10, 4)
    with pytest.raises(ref.CacheError):
        c.append(0, np.ones((2, 1, 3, 4)), np.ones((2, 1, 3, 4)), bad)
    assert np.all(c.lens == 0)


def test_shape_mismatch_rejected():
    c = ref.OracleCache(1, 2, 2, 10, 4)
    with pytest.raises(ref.CacheError):
        c.append(0, np.ones((2, 1, 3, 4)), np.ones((2, 1, 3, 4)), np.array([1, 1]))
    with pytest.raises(ref.CacheError):
        c.append(0, np.ones((2, 2, 3, 5)), np.ones((2, 2, 3, 5)), np.array([1, 1]))
    with pytest.raises(ref.CacheError):
        ref.gqa_attention(np.ones((2, 3, 1, 4)), c, 0, np.array([0, 0]))  # Hq % Hkv != 0


def test_empty_cases_return_zeros():
    c0 = ref.OracleCache(1, 0, 2, 8, 4)
    out = ref.gqa_attention(np.zeros((0, 4, 3, 4)), c0, 0, np.zeros(0, dtype=np.int64))
    assert out.shape == (0, 4, 3, 4)
    c = ref.OracleCache(1, 2, 2, 8, 4)
    out = ref.gqa_attention(_rand(1, 1, (2, 4, 3, 4)), c, 0, np.array([0, 0]))
    assert out.shape == (2, 4, 3, 4) and np.all(out == 0)
    out = ref.append_attention(c, 0, np.zeros((2, 4, 0, 4)), np.zeros((2, 2, 0, 4)), np.zeros((2, 2, 0, 4)), np.array([0, 0]))
    assert out.shape == (2, 4, 0, 4)


def test_appended_slice_is_stored_in_place():
    c = ref.OracleCache(1, 2, 2, 16, 4)
    buf = c.k[0]
    k1 = _rand(1, 1, (2, 2, 5, 4))
    c.append(0, k1, k1, np.array([5, 3]))
    k2 = _rand(1, 2, (2, 2, 2, 4))
    c.append(0, k2, k2, np.array([1, 2]))
    assert c.k[0] is buf
    assert np.array_equal(buf[0, :, 0:5], k1[0]) and np.array_equal(buf[0, :, 5:6], k2[0, :, :1])
    assert np.array_equal(buf[1, :, 0:3], k1[1, :, :3]) and np.array_equal(buf[1, :, 3:5], k2[1])
    assert list(c.lens[0]) == [6, 5]


def test_layer_lengths_and_truncate():
    c = ref.OracleCache(3, 2, 1, 10, 2)
    for layer in range(3):
        c.append(layer, np.ones((2, 1, 4, 2)), np.ones((2, 1, 4, 2)), np.array([4, 2]))
    assert list(c.length()) == [4, 2]
    c.append(0, np.ones((2, 1, 1, 2)), np.ones((2, 1, 1, 2)), np.array([1, 1]))
    with pytest.raises(ref.CacheError):
        c.length()  # a forward pass stopped part-way
    with pytest.raises(ref.CacheError):
        c.truncate([3, 1])  # length() refuses, so truncate does too
    c.lens[0] = c.lens[1]
    c.truncate([3, 1])
    assert list(c.length()) == [3, 1]
    with pytest.raises(ref.CacheError):
        c.truncate([4, 1])  # cannot grow
    with pytest.raises(ref.CacheError):
        c.truncate([-1, 0])
    c.reset()
    assert list(c.length()) == [0, 0]


# ---------------------------------------------------------------------------
# Planted mistakes: each plausible error in the oracle makes some pin fail
# ---------------------------------------------------------------------------

PINS = [
    test_closed_form_offset_and_padding,
    test_closed_form_head_mapping,
    test_closed_form_scale_two_keys,
    lambda: test_incremental_equals_full_causal(2, 4),
    lambda: [(_ for _ in ()).throw(AssertionError()) for s in range(6) if _trial(s)[1] > 1e-10],
]


def _some_pin_fails():
    for pin in PINS:
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            return True
    return False


@pytest.mark.parametrize(
    "name,wrong",
    [
        ("kv_head_of", lambda h, G: h % G),  # interleaved groups (h % Hkv-style)
        ("query_position", lambda L, n, t: t),  # top-left alignment
        ("query_position", lambda L, n, t: L - n + t - 1),  # off by one
        ("score_scale", lambda d: 1.0),  # dropped 1/sqrt(d)
        ("score_scale", lambda d: 1.0 / d),  # wrong scale
    ],
)
def test_planted_mistakes_are_caught(monkeypatch, name, wrong):
    assert not _some_pin_fails()
    monkeypatch.setattr(ref, name, wrong)
    assert _some_pin_fails()
