"""Paged K/V storage behind a block table, on the GPU against the oracle.

"Implement grouped-query attention over a preallocated KV cache...", "A
strong answer" (the reversal condition: rows of very different lengths want
a block table instead of max_len per row) and "16. Prefill, decode and the KV
cache", "Design choices worth noticing": the attention of a row is that of
its logical sequence, wherever its pages sit.  Every call is compared with
the float64 paged oracle on the same inputs (max-abs 1e-4 fp32, 2e-2 bf16);
every written position is compared bit for bit in its physical page; pages
and slots never written hold NaN, so a read of them fails.
"""

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import KVCError, PagedKVCache
from gqa_attention_preallocated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _pair(B, Hkv, d, page, num_pages, mpr, dtype, table, window=0):
    cache = PagedKVCache(1, B, Hkv, page, num_pages, mpr, d, dtype=dtype)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    cache.block_table.copy_(torch.as_tensor(table, dtype=torch.int32).view(B, mpr))
    if window:
        cache.set_window(window)
    orc = ref.PagedOracleCache(1, B, Hkv, page, num_pages, mpr, d)
    orc.set_block_table(table)
    orc.window = window
    return cache, orc


def _check_pages(cache, orc):
    kc, vc = cache.k[0].double().cpu().numpy(), cache.v[0].double().cpu().numpy()
    for b in range(orc.B):
        for a in range(int(orc.lens[0, b])):
            page, off = orc.page_of(b, a)
            assert np.array_equal(kc[page, :, off], orc.k[0][page, :, off]), (b, a)
            assert np.array_equal(vc[page, :, off], orc.v[0][page, :, off]), (b, a)


def _step(cache, orc, seed, ci, G, n_new, dtype, parents=None):
    B, Hkv, d = orc.B, orc.Hkv, orc.d
    n_new = np.asarray(n_new, dtype=np.int64)
    T = max(int(n_new.max()), 1) if parents is None else np.asarray(parents).shape[1]
    k = wl.to_storage(wl.normal(seed, 100 + 3 * ci, (B, Hkv, T, d)), dtype)
    v = wl.to_storage(wl.normal(seed, 101 + 3 * ci, (B, Hkv, T, d)), dtype)
    q = wl.to_storage(wl.normal(seed, 102 + 3 * ci, (B, Hkv * G, T, d)), dtype)
    if parents is None:
        out = cache.append_attention(0, q.cuda(), k.cuda(), v.cuda(), n_new)
    else:
        out = cache.append_attention_tree(0, q.cuda(), k.cuda(), v.cuda(), n_new, parents)
    want = ref.paged_append_attention(orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), n_new,
                                      parents)
    got = out.double().cpu().numpy()
    assert np.array_equal(cache.lens(0), orc.lens[0])
    assert np.all(np.isfinite(got))
    for b in range(B):
        assert np.all(got[b, :, n_new[b]:] == 0.0)
    err = float(np.max(np.abs(got - want)))
    assert err <= TOL[dtype], (ci, err)
    return err


def _run(seed, B, Hkv, G, d, page, num_pages, mpr, dtype, calls, window=0, table=None):
    _cuda_or_skip()
    rng = np.random.default_rng(seed)
    if table is None:
        table = rng.permutation(num_pages)[: B * mpr]
    cache, orc = _pair(B, Hkv, d, page, num_pages, mpr, dtype, table, window)
    for ci, n_new in enumerate(calls):
        _step(cache, orc, seed, ci, G, n_new, dtype)
    _check_pages(cache, orc)
    assert cache.device_status() == 0
    return cache, orc


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("page,mpr,window", [(4, 12, 0), (8, 6, 0), (1, 40, 0), (4, 12, 7)])
def test_f32_paged_tiny(seed, page, mpr, window):
    B, Hkv, G, d = 3, 2, 3, 16
    rng = np.random.default_rng(seed)
    per_call = (page * mpr) // 8
    calls = [rng.integers(0, per_call + 1, size=B) for _ in range(8)]
    _run(seed, B, Hkv, G, d, page, B * mpr + 5, mpr, torch.float32, calls, window)


@pytest.mark.parametrize("T", [1, 4, 8])
def test_bf16_decode_paged(T):
    """Split-KV decode / verify over pages of 128 in a random order, ragged prefixes."""
    B, Hkv, G, d, page, mpr = 4, 2, 4, 128, 128, 12
    rng = np.random.default_rng(10 + T)
    calls = [rng.integers(100, 300, size=B) for _ in range(4)]
    calls += [np.full(B, T) if i % 3 else rng.integers(0, T + 1, size=B) for i in range(8)]
    _run(20 + T, B, Hkv, G, d, page, B * mpr + 3, mpr, torch.bfloat16, calls)


def test_bf16_prefill_paged():
    """Chunks of 256 query positions (the tensor-core prefill kernel) through permuted pages."""
    B, Hkv, G, d, page, mpr = 2, 2, 4, 128, 128, 16
    calls = [np.full(B, 256)] * 5 + [np.array([256, 131])]
    _run(31, B, Hkv, G, d, page, B * mpr, mpr, torch.bfloat16, calls)


def test_bf16_paged_with_window():
    B, Hkv, G, d, page, mpr = 2, 2, 4, 128, 128, 16
    calls = [np.full(B, 256)] * 4 + [np.array([200, 7])] + [np.full(B, 1)] * 3
    _run(32, B, Hkv, G, d, page, B * mpr, mpr, torch.bfloat16, calls, window=300)


def test_bf16_paged_uneven_rows_share_a_pool():
    """Rows of very different lengths drawing pages from one pool smaller than B * max_pages_per_row.

    Only the pages each row's length needs are mapped; the rest of its
    table is -1 and is never touched.
    """
    _cuda_or_skip()
    B, Hkv, G, d, page, mpr = 4, 2, 4, 128, 128, 24
    want_len = np.array([2900, 130, 1, 700])
    need = (want_len + page - 1) // page
    num_pages = int(need.sum()) + 2
    rng = np.random.default_rng(5)
    free = list(rng.permutation(num_pages))
    table = np.full((B, mpr), -1)
    for b in range(B):
        for i in range(int(need[b])):
            table[b, i] = free.pop()
    cache, orc = _pair(B, Hkv, d, page, num_pages, mpr, torch.bfloat16, table.reshape(-1))
    calls = [np.minimum(want_len - 1, 2899) // 4] * 4
    calls.append(want_len - 1 - 4 * calls[0])
    calls.append(np.ones(B, dtype=np.int64))
    for ci, n_new in enumerate(calls):
        _step(cache, orc, 5, ci, G, n_new, torch.bfloat16)
    assert np.array_equal(orc.lens[0], want_len)
    _check_pages(cache, orc)
    assert cache.device_status() == 0


@pytest.mark.parametrize("dtype,d,page", [(torch.bfloat16, 128, 128), (torch.float32, 16, 4)])
def test_shared_prefix_pages(dtype, d, page):
    """Rows whose tables point at the same prefix pages attend to that prefix without copying it."""
    _cuda_or_skip()
    B, Hkv, G, mpr = 3, 2, 4, 8
    npre = 3  # prefix pages
    num_pages = npre + B * (mpr - npre)
    table = np.full((B, mpr), -1)
    table[:, :npre] = np.arange(npre)
    rest = np.random.default_rng(6).permutation(np.arange(npre, num_pages))
    table[:, npre:] = rest.reshape(B, mpr - npre)
    cache, orc = _pair(B, Hkv, d, page, num_pages, mpr, dtype, table.reshape(-1))
    P = npre * page
    n0 = np.zeros(B, dtype=np.int64)
    n0[0] = P
    _step(cache, orc, 7, 0, G, n0, dtype)  # row 0 writes the prefix
    shared = np.full(B, P, dtype=np.int64)
    cache.set_lens(0, shared)  # every row now starts from it
    orc.lens[0] = shared
    rng = np.random.default_rng(8)
    for ci in range(1, 6):
        _step(cache, orc, 7, ci, G, rng.integers(1, page // 2 + 1, size=B), dtype)
    _check_pages(cache, orc)
    assert cache.device_status() == 0


def test_tree_verify_over_pages():
    _cuda_or_skip()
    B, Hkv, G, d, page, mpr, T = 4, 2, 4, 128, 128, 10, 8
    rng = np.random.default_rng(9)
    cache, orc = _pair(B, Hkv, d, page, B * mpr, mpr, torch.bfloat16, rng.permutation(B * mpr))
    _step(cache, orc, 9, 0, G, rng.integers(200, 1000, size=B), torch.bfloat16)
    parents = np.stack([np.array([-1] + [int(rng.integers(-1, t)) for t in range(1, T)]) for _ in range(B)])
    _step(cache, orc, 9, 1, G, np.full(B, T), torch.bfloat16, parents=parents)
    _check_pages(cache, orc)
    assert cache.device_status() == 0


def test_decode_step_over_pages_matches_host_path():
    _cuda_or_skip()
    B, Hkv, G, T, page, mpr = 8, 4, 4, 1, 128, 16
    rng = np.random.default_rng(11)
    table = torch.as_tensor(rng.permutation(B * mpr), dtype=torch.int32).view(B, mpr)
    caches = []
    for _ in range(2):
        c = PagedKVCache(1, B, Hkv, page, B * mpr, mpr, 128)
        c.block_table.copy_(table)
        wl.fill_normal_(c.k[0], 3, wl.STREAM_CACHE_K)
        wl.fill_normal_(c.v[0], 3, wl.STREAM_CACHE_V)
        c.set_lens(0, wl.decode_lens(3, B, 600, 1900))
        caches.append(c)
    host, dev = caches
    ws = dev.workspace(Hkv * G, T)
    dev.lens_to_device()
    out = torch.empty((B, Hkv * G, T, 128), dtype=torch.bfloat16, device="cuda")
    nn = torch.ones(B, dtype=torch.int32, device="cuda")
    for step in range(6):
        q = wl.to_storage(wl.normal(3, 5000 + step, (B, Hkv * G, T, 128)), torch.bfloat16).cuda()
        k = wl.to_storage(wl.normal(3, 1000 + step, (B, Hkv, T, 128)), torch.bfloat16).cuda()
        v = wl.to_storage(wl.normal(3, 2000 + step, (B, Hkv, T, 128)), torch.bfloat16).cuda()
        want = host.append_attention(0, q, k, v, np.ones(B))
        dev.decode_step(0, q, k, v, nn, out, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, want), step
    assert dev.device_status(ws) == 0
    dev.lens_from_device()
    assert np.array_equal(dev.lens(0), host.lens(0))
    assert torch.equal(dev.k[0], host.k[0]) and torch.equal(dev.v[0], host.v[0])


@pytest.mark.parametrize("T", [1, 256])
def test_unmapped_page_is_reported_not_read(T):
    """A -1 entry under an attended position: the kernel reads no page for it,
    writes nothing through it, and the workspace error word reports it."""
    _cuda_or_skip()
    B, Hkv, G, d, page, mpr = 2, 2, 4, 128, 128, 8
    cache = PagedKVCache(1, B, Hkv, page, B * mpr, mpr, d)
    cache.k[0].zero_()
    cache.v[0].zero_()
    cache.set_lens(0, [5 * page, 3 * page])
    cache.block_table[0, 2] = -1   # under row 0's attended keys
    cache.block_table[1, 3] = -1   # under row 1's appended positions
    before = (cache.k[0].clone(), cache.v[0].clone())
    q = torch.zeros((B, Hkv * G, T, d), dtype=torch.bfloat16, device="cuda")
    k = torch.ones((B, Hkv, T, d), dtype=torch.bfloat16, device="cuda")
    cache.append_attention(0, q, k, k, np.full(B, T))
    torch.cuda.synchronize()
    with pytest.raises(KVCError):
        cache.device_status()
    assert cache.device_status() == 0  # the word was cleared
    # row 1's positions in the unmapped page went nowhere; everything else is as before or the new rows
    changed = (cache.k[0] != before[0]).any(dim=-1).any(dim=1)  # [num_pages, page]
    pages_written = set(torch.nonzero(changed.any(dim=1)).flatten().tolist())
    span = range(1 + (T - 1) // page)  # logical pages a chunk of T starting on a page boundary covers
    allowed = {int(cache.block_table[0, 5 + i]) for i in span} | {int(cache.block_table[1, 3 + i]) for i in span}
    assert -1 in allowed and pages_written == allowed - {-1}
