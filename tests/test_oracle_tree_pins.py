"""Pins for the oracle's tree speculative verify (p2 "Write the causal mask for
a decode step...", "What interviewers probe next": tree-based speculative
decoding, an ancestor mask built from parent pointers for the T x T corner).

The tree path is tied to the plain path by invariants: a chain tree is the
ordinary causal chunk; any draft token's output equals the last output of its
root-to-token path appended as an ordinary chunk; a star tree equals one
single-token decode per draft token.  The triangle mask applied to a
branching tree must give a visibly different answer.
"""

import numpy as np
import pytest

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import workloads as wl


def _rand(seed, stream, shape):
    return wl.normal(seed, stream, shape).numpy()


def _setup(seed, B, Hkv, G, d, prior, T):
    c = ref.OracleCache(1, B, Hkv, prior + T + 4, d)
    kp, vp = _rand(seed, 1, (B, Hkv, prior, d)), _rand(seed, 2, (B, Hkv, prior, d))
    ref.append_attention(c, 0, np.zeros((B, Hkv * G, prior, d)), kp, vp, np.full(B, prior))
    k, v = _rand(seed, 3, (B, Hkv, T, d)), _rand(seed, 4, (B, Hkv, T, d))
    q = _rand(seed, 5, (B, Hkv * G, T, d))
    return c, kp, vp, k, v, q


def _random_tree(rng, T):
    return np.array([-1] + [int(rng.integers(-1, t)) for t in range(1, T)])


def test_chain_tree_is_the_causal_chunk():
    B, Hkv, G, d, prior, T = 2, 2, 2, 8, 11, 6
    c1, _, _, k, v, q = _setup(1, B, Hkv, G, d, prior, T)
    c2, _, _, _, _, _ = _setup(1, B, Hkv, G, d, prior, T)
    chain = np.tile(np.arange(-1, T - 1), (B, 1))
    a = ref.append_attention(c1, 0, q, k, v, np.full(B, T), parents=chain)
    b = ref.append_attention(c2, 0, q, k, v, np.full(B, T))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("seed", range(8))
def test_each_token_equals_its_path_as_a_chunk(seed):
    B, Hkv, G, d, prior, T = 2, 2, 3, 8, 9, 8
    rng = np.random.default_rng(seed)
    parents = np.stack([_random_tree(rng, T) for _ in range(B)])
    c, kp, vp, k, v, q = _setup(seed, B, Hkv, G, d, prior, T)
    got = ref.append_attention(c, 0, q, k, v, np.full(B, T), parents=parents)
    for b in range(B):
        for t in range(T):
            path = sorted(ref.tree_path(parents[b], t))
            cp = ref.OracleCache(1, 1, Hkv, prior + T, d)
            ref.append_attention(cp, 0, np.zeros((1, Hkv * G, prior, d)), kp[b:b + 1], vp[b:b + 1], [prior])
            n = len(path)
            qq = np.zeros((1, Hkv * G, n, d))
            qq[0, :, n - 1] = q[b, :, t]
            out = ref.append_attention(cp, 0, qq, k[b:b + 1][:, :, path], v[b:b + 1][:, :, path], [n])
            assert np.allclose(got[b, :, t], out[0, :, n - 1], rtol=0, atol=1e-12)


def test_star_tree_is_independent_single_token_steps():
    B, Hkv, G, d, prior, T = 2, 1, 4, 8, 7, 5
    c, kp, vp, k, v, q = _setup(3, B, Hkv, G, d, prior, T)
    star = np.full((B, T), -1)
    got = ref.append_attention(c, 0, q, k, v, np.full(B, T), parents=star)
    single = ref.OracleCache(1, B, Hkv, prior + 1, d)
    ref.append_attention(single, 0, np.zeros((B, Hkv * G, prior, d)), kp, vp, np.full(B, prior))
    for t in range(T):
        out = ref.append_attention(single, 0, q[:, :, t:t + 1], k[:, :, t:t + 1], v[:, :, t:t + 1], np.ones(B))
        assert np.allclose(got[:, :, t], out[:, :, 0], rtol=0, atol=1e-12)
        single.truncate(np.full(B, prior))


def test_triangle_mask_on_a_branching_tree_is_wrong():
    B, Hkv, G, d, prior, T = 1, 1, 2, 8, 5, 6
    c1, _, _, k, v, q = _setup(4, B, Hkv, G, d, prior, T)
    c2, _, _, _, _, _ = _setup(4, B, Hkv, G, d, prior, T)
    tree = np.array([[-1, 0, 0, 1, 2, 2]])
    a = ref.append_attention(c1, 0, q, k, v, [T], parents=tree)
    b = ref.append_attention(c2, 0, q, k, v, [T])
    assert np.max(np.abs(a - b)) > 1e-3


def test_corner_mask_counts_and_rules():
    tree = np.array([-1, 0, 0, 1, 2, 2, 5, -1])
    m = ref.tree_corner_mask(tree)
    depth = [len(ref.tree_path(tree, t)) for t in range(len(tree))]
    assert int(m.sum()) == sum(depth) == 1 + 2 + 2 + 3 + 3 + 3 + 4 + 1
    assert np.array_equal(ref.tree_corner_mask(np.arange(-1, 7)), np.tril(np.ones((8, 8), dtype=bool)))
    assert np.array_equal(ref.tree_corner_mask(np.full(8, -1)), np.eye(8, dtype=bool))
    c = ref.OracleCache(1, 1, 1, 8, 4)
    z = np.zeros((1, 1, 3, 4))
    with pytest.raises(ref.CacheError):
        ref.append_attention(c, 0, z, z, z, [3], parents=[[-1, 1, 0]])  # a parent after its child
    assert list(c.lens[0]) == [0]  # rejected before the append
