"""Packed query rows on the tensor-core kernel, against the oracle.

"Implement grouped-query attention over a preallocated KV cache...", "A
strong answer" (gqa_attention: the G*T rows of one KV head share its keys,
query t at position prior + t) and "Write the causal mask for a decode
step...", "TL;DR" (bottom-right alignment).  With T < 128 the kernel packs
the rows g*T + t of one KV head into 128-row tiles; with at most 128 such
rows its two TMEM buffers take alternate key tiles and their softmax states
are merged at the end.  Every case compares outputs with the float64 oracle
(2e-2 bf16); cache slots past each row's length hold NaN.
"""

import heapq

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import KVCache, PagedKVCache
from gqa_attention_preallocated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _step(cache, orc, seed, ci, G, n_new, T=None, paged=False):
    B, Hkv, d = orc.B, orc.Hkv, orc.d
    n_new = np.asarray(n_new, dtype=np.int64)
    T = max(int(n_new.max()), 1) if T is None else T
    k = wl.to_storage(wl.normal(seed, 100 + 3 * ci, (B, Hkv, T, d)), torch.bfloat16)
    v = wl.to_storage(wl.normal(seed, 101 + 3 * ci, (B, Hkv, T, d)), torch.bfloat16)
    q = wl.to_storage(wl.normal(seed, 102 + 3 * ci, (B, Hkv * G, T, d)), torch.bfloat16)
    out = cache.append_attention(0, q.cuda(), k.cuda(), v.cuda(), n_new)
    args = (orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), n_new)
    want = ref.paged_append_attention(*args) if paged else ref.append_attention(*args)
    got = out.double().cpu().numpy()
    assert np.array_equal(cache.lens(0), orc.lens[0])
    assert np.all(np.isfinite(got))
    for b in range(B):
        assert np.all(got[b, :, n_new[b]:] == 0.0)
    err = float(np.max(np.abs(got - want)))
    assert err <= TOL, (ci, err)
    return err


def _poisoned(B, Hkv, max_len, window=0):
    cache = KVCache(1, B, Hkv, max_len, 128)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    orc = ref.OracleCache(1, B, Hkv, max_len, 128)
    if window:
        cache.set_window(window)
        orc.set_window(window)
    return cache, orc


@pytest.mark.parametrize(
    "B,Hkv,G,T",
    [
        (3, 2, 8, 12),   # 96 rows: one tile, alternate key tiles
        (2, 2, 16, 8),   # 128 rows: one full tile
        (2, 1, 1, 100),  # MHA-like single head, 100 rows
        (2, 2, 4, 17),   # 68 rows
        (2, 2, 8, 40),   # 320 rows: two tile pairs, the last with one tile
        (1, 2, 32, 8),   # 256 rows: one pair of full tiles
        (2, 1, 5, 100),  # 500 rows: two pairs, odd G
    ],
)
def test_packed_rows_every_output(B, Hkv, G, T):
    _cuda_or_skip()
    rng = np.random.default_rng(B * 1000 + G * 10 + T)
    prior = rng.integers(200, 900, size=B)
    max_len = int(prior.max()) + 2 * T + 8
    cache, orc = _poisoned(B, Hkv, max_len)
    _step(cache, orc, 3, 0, G, prior, T=int(prior.max()))
    n1 = rng.integers(0, T + 1, size=B)
    n1[0] = T
    _step(cache, orc, 3, 1, G, n1, T=T)          # ragged: some rows with fewer (or no) new tokens
    _step(cache, orc, 3, 2, G, np.full(B, T), T=T)
    assert cache.device_status() == 0


def test_packed_rows_short_rows():
    """Rows whose whole length fits in one or two key tiles (the odd-tile buffer
    left empty or holding a single tile)."""
    _cuda_or_skip()
    cache, orc = _poisoned(4, 2, 300)
    _step(cache, orc, 4, 0, 8, np.array([12, 0, 5, 12]), T=12)
    _step(cache, orc, 4, 1, 8, np.array([12, 12, 12, 1]), T=12)
    _step(cache, orc, 4, 2, 8, np.array([100, 120, 120, 120]), T=120)
    _step(cache, orc, 4, 3, 8, np.array([12, 12, 3, 12]), T=12)


def _cuts(items, nsm, start_cost=5, min_piece=8):
    """Cuts the library's schedule makes for items (key tiles, cost per tile):
    a longest-first list schedule on the SMs, items cut at the common finish.
    Restated only to show that a case exercises the in-kernel merge."""
    W = sum(n * h + start_cost for n, h in items)
    target = W // nsm + start_cost
    parts = [(-n * h, k, 0) for k, (n, h) in enumerate(items)]
    heapq.heapify(parts)
    sms = [(0, m) for m in range(nsm)]
    cuts = 0
    while parts:
        c, k, lo = heapq.heappop(parts)
        n, h = items[k]
        t, m = heapq.heappop(sms)
        hi, fit = n, max(0, target - t - start_cost) // h
        if -c + start_cost > target - t and fit >= min_piece and n - (lo + fit) >= min_piece:
            hi = lo + fit
            cuts += 1
            heapq.heappush(parts, (-(n - hi) * h, k, hi))
        heapq.heappush(sms, (t + start_cost + (hi - lo) * h, m))
    return cuts


@pytest.mark.parametrize("G,T,prior", [(8, 12, 30000), (8, 40, 20000)])
def test_packed_long_rows_cut_and_merged(G, T, prior):
    """Long rows on few items: the schedule cuts items into key-range pieces
    whose partials the last piece merges in the launch; sampled units."""
    _cuda_or_skip()
    from test_gpu_parity import _decode_case

    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    B, Hkv = 4, 8
    R = G * T
    per_item = [1] if R <= 128 else [min(2, (R - p * 256 + 127) // 128) for p in range((R + 255) // 256)]
    lens0 = np.array([prior, prior - 700, prior - 5000, prior - 128])
    n_new = np.array([T, T - 3, T, 1])
    items = [((int(L) + min(T, int(n)) - 1) // 128 + 1, c) for L, n in zip(lens0, n_new)
             for _ in range(Hkv) for c in per_item]
    assert _cuts(items, nsm) > 0
    s = wl.Shape("packed_long_rows", B=B, Hq=Hkv * G, Hkv=Hkv, d=128, max_len=prior + T + 8, dtype="bf16")
    _decode_case(s, Hkv * G, lens0, [T], [n_new], 17, [(0, 0), (1, 5), (3, 7)])


def test_packed_rows_with_window():
    _cuda_or_skip()
    cache, orc = _poisoned(3, 2, 1500, window=300)
    _step(cache, orc, 5, 0, 8, np.array([700, 300, 1000]), T=1000)
    for ci in range(1, 5):
        _step(cache, orc, 5, ci, 8, np.array([12, 7, 12]), T=12)


def test_packed_rows_over_pages():
    _cuda_or_skip()
    B, Hkv, G, page, mpr = 3, 2, 8, 128, 12
    cache = PagedKVCache(1, B, Hkv, page, B * mpr, mpr, 128)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    table = np.random.default_rng(6).permutation(B * mpr)
    cache.block_table.copy_(torch.as_tensor(table, dtype=torch.int32).view(B, mpr))
    orc = ref.PagedOracleCache(1, B, Hkv, page, B * mpr, mpr, 128)
    orc.set_block_table(table)
    _step(cache, orc, 6, 0, G, np.array([900, 400, 1200]), T=1200, paged=True)
    for ci in range(1, 4):
        _step(cache, orc, 6, ci, G, np.array([12, 12, 9]), T=12, paged=True)
    assert cache.device_status() == 0


def test_packed_rows_score_jumps_in_one_buffer():
    """Scores that jump by about 200 (log2 units) in an odd key tile only: the
    odd-tile state's maximum is far above the even one's, and the merge of the
    two states still matches the oracle."""
    _cuda_or_skip()
    B, Hkv, G, T, d, prior = 1, 2, 8, 12, 128, 1300
    rng = np.random.default_rng(12)
    u = np.ones(d)
    k0 = rng.standard_normal((B, Hkv, prior, d))
    for pos, alpha in ((200, 1.5), (700, 4.0)):  # key tiles 1 and 5: the odd buffer
        k0[:, :, pos] = alpha * u + 0.1 * rng.standard_normal(d)
    v0 = rng.standard_normal((B, Hkv, prior, d))
    kn = rng.standard_normal((B, Hkv, T, d))
    vn = rng.standard_normal((B, Hkv, T, d))
    q = np.tile(u, (B, Hkv * G, T, 1)) * 4.0 + 0.1 * rng.standard_normal((B, Hkv * G, T, d))
    st = [wl.to_storage(torch.from_numpy(x), torch.bfloat16) for x in (k0, v0, kn, vn, q)]
    cache, orc = _poisoned(B, Hkv, prior + T + 8)
    z = torch.zeros((B, Hkv * G, prior, d), dtype=torch.bfloat16)
    cache.append_attention(0, z.cuda(), st[0].cuda(), st[1].cuda(), [prior])
    orc.append(0, st[0].double().numpy(), st[1].double().numpy(), [prior])
    out = cache.append_attention(0, st[4].cuda(), st[2].cuda(), st[3].cuda(), [T])
    want = ref.append_attention(orc, 0, st[4].double().numpy(), st[2].double().numpy(), st[3].double().numpy(), [T])
    err = float(np.max(np.abs(out.double().cpu().numpy() - want)))
    assert err <= TOL, err
    assert cache.device_status() == 0
