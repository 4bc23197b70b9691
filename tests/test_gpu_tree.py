"""Tree speculative verify on the GPU against the oracle ("Write the causal
mask for a decode step with a KV cache...", "What interviewers probe next":
each draft token attends to the cache plus its own ancestors, an ancestor
mask built from parent pointers for the T x T corner).

Random trees (plus a chain and a star), ragged prior lengths spanning many
key tiles, rows with fewer draft tokens than T, every output compared with
the float64 oracle (max-abs 1e-4 fp32, 2e-2 bf16).
"""

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import KVCache, KVCError
from gqa_attention_preallocated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _trees(rng, B, T):
    out = []
    for b in range(B):
        kind = b % 4
        if kind == 0:
            out.append(np.arange(-1, T - 1))               # a chain: the ordinary causal chunk
        elif kind == 1:
            out.append(np.full(T, -1))                     # a star: every draft off the prefix
        else:
            out.append(np.array([-1] + [int(rng.integers(-1, t)) for t in range(1, T)]))
    return np.stack(out)


def _case(seed, B, Hkv, G, T, d, dtype, prior_lo, prior_hi):
    _cuda_or_skip()
    rng = np.random.default_rng(seed)
    priors = rng.integers(prior_lo, prior_hi + 1, size=B)
    n_new = np.full(B, T)
    n_new[1::3] = rng.integers(1, T + 1, size=len(n_new[1::3]))  # some rows with fewer drafts
    max_len = int(priors.max()) + T + 8
    cache = KVCache(1, B, Hkv, max_len, d, dtype=dtype)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    orc = ref.OracleCache(1, B, Hkv, max_len, d)
    P = int(priors.max())
    kp = wl.to_storage(wl.normal(seed, 1, (B, Hkv, P, d)), dtype)
    vp = wl.to_storage(wl.normal(seed, 2, (B, Hkv, P, d)), dtype)
    cache.append(0, kp.cuda(), vp.cuda(), priors)
    orc.append(0, kp.double().numpy(), vp.double().numpy(), priors)
    parents = _trees(rng, B, T)
    k = wl.to_storage(wl.normal(seed, 3, (B, Hkv, T, d)), dtype)
    v = wl.to_storage(wl.normal(seed, 4, (B, Hkv, T, d)), dtype)
    q = wl.to_storage(wl.normal(seed, 5, (B, Hkv * G, T, d)), dtype)
    out = cache.append_attention_tree(0, q.cuda(), k.cuda(), v.cuda(), n_new, parents)
    want = ref.append_attention(orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), n_new,
                                parents=parents)
    got = out.double().cpu().numpy()
    assert np.array_equal(cache.lens(0), orc.lens[0])
    assert np.all(np.isfinite(got))
    for b in range(B):
        assert np.all(got[b, :, n_new[b]:] == 0.0)
    err = float(np.max(np.abs(got - want)))
    assert err <= TOL[dtype], err
    # the plain causal call must differ wherever a row's tree is not a chain
    assert cache.device_status() == 0
    return err


@pytest.mark.parametrize("B,Hkv,G,T", [(4, 2, 4, 4), (5, 2, 4, 8), (4, 2, 8, 8), (8, 3, 1, 16), (4, 1, 4, 16)])
def test_bf16_tree(B, Hkv, G, T):
    _case(B * 100 + T, B, Hkv, G, T, 128, torch.bfloat16, 40, 900)


@pytest.mark.parametrize("B,Hkv,G,T", [(3, 2, 2, 8), (2, 1, 1, 64), (4, 2, 4, 16)])
def test_f32_tree(B, Hkv, G, T):
    _case(B * 10 + T, B, Hkv, G, T, 16, torch.float32, 0, 60)


def test_bf16_tree_verify_shape():
    """The speculative-verify workload's shape (Hkv=8, G=4, S=4096, T=8) on 8 rows."""
    _case(77, 8, 8, 4, 8, 128, torch.bfloat16, 4088, 4088)


def test_tree_rejections():
    _cuda_or_skip()
    c = KVCache(1, 2, 2, 128, 128)
    c.append(0, torch.zeros((2, 2, 4, 128), dtype=torch.bfloat16, device="cuda"),
             torch.zeros((2, 2, 4, 128), dtype=torch.bfloat16, device="cuda"), [4, 4])
    q = torch.zeros((2, 8, 4, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(KVCError) as e:
        c.gqa_attention_tree(0, q, [4, 4], [[-1, 0, 3, 1], [-1, 0, 0, 0]])  # a parent after its child
    assert e.value.status == 2
    c2 = KVCache(1, 1, 1, 256, 128)
    c2.set_window(64)
    z = torch.zeros((1, 1, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(KVCError) as e:
        c2.append_attention_tree(0, torch.zeros((1, 1, 2, 128), dtype=torch.bfloat16, device="cuda"), z, z, [2],
                                 [[-1, 0]])
    assert e.value.status == 1
    assert list(c2.lens(0)) == [0]  # nothing appended


@pytest.mark.parametrize("dtype,d", [(torch.float32, 16), (torch.bfloat16, 64), (torch.bfloat16, 128)])
@pytest.mark.parametrize("T", [48, 64])
def test_star_trees_on_an_empty_prefix(dtype, d, T):
    """Every draft hangs off an empty prefix: query t sees its own token only,
    so key tiles before it hold no visible key for it (and nothing came
    before).  The outputs are the queries' own V rows."""
    _cuda_or_skip()
    B, Hkv, G = 2, 1, 1
    cache = KVCache(1, B, Hkv, T + 8, d, dtype=dtype)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    orc = ref.OracleCache(1, B, Hkv, T + 8, d)
    n_new = np.array([T, T - 5])
    parents = np.full((B, T), -1)
    k = wl.to_storage(wl.normal(9, 1, (B, Hkv, T, d)), dtype)
    v = wl.to_storage(wl.normal(9, 2, (B, Hkv, T, d)), dtype)
    q = wl.to_storage(wl.normal(9, 3, (B, Hkv * G, T, d)), dtype)
    out = cache.append_attention_tree(0, q.cuda(), k.cuda(), v.cuda(), n_new, parents)
    want = ref.append_attention(orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), n_new,
                                parents=parents)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(got - want))) <= TOL[dtype]
    for b in range(B):  # a single visible key: the output is that key's V row
        assert np.allclose(want[b, :, :n_new[b]], v.double().numpy()[b, :, :n_new[b]], atol=1e-12)
    assert cache.device_status() == 0
