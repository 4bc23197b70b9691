"""GPU parity for bf16 caches whose head dimension is not 128.

bf16 caches of d = 64 run on the split-KV kernel (TMA tiles of one 64-column
box, mma.sync) up to 64 query rows per KV head, appends fused into decode,
and on the generic kernel above that; other head dimensions run on the
generic kernel (values widened to fp32 in shared memory).  The bars are the
same as for every bf16 call: the append and the lengths bit-exact, outputs
within max-abs 2e-2 of the float64 oracle, padded queries exactly 0.  Slots
past the valid lengths hold NaN, so an output that touched one fails.  Head
dimensions: 16 and 64 (the sizes beside 128 the hot path names), 96 and 256
(the largest the generic kernel takes).
"""

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import KVCache, KVCError, PagedKVCache
from gqa_attention_preallocated_gb300 import workloads as wl
from oracle_rows import UnitOracle, max_error

pytestmark = pytest.mark.gpu

TOL = 2e-2
BF16 = torch.bfloat16


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _step(cache, orc, seed, ci, G, n_new, parents=None):
    B, Hkv, d = cache.B, cache.Hkv, cache.d
    n_new = np.asarray(n_new, dtype=np.int64)
    T = max(int(n_new.max()), 1)
    k = wl.to_storage(wl.normal(seed, 100 + 3 * ci, (B, Hkv, T, d)), BF16)
    v = wl.to_storage(wl.normal(seed, 101 + 3 * ci, (B, Hkv, T, d)), BF16)
    q = wl.to_storage(wl.normal(seed, 102 + 3 * ci, (B, Hkv * G, T, d)), BF16)
    if parents is None:
        out = cache.append_attention(0, q.cuda(), k.cuda(), v.cuda(), n_new)
    else:
        out = cache.append_attention_tree(0, q.cuda(), k.cuda(), v.cuda(), n_new, parents)
    want = ref.append_attention(orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), n_new,
                                parents=parents)
    assert out.dtype == BF16
    got = out.double().cpu().numpy()
    assert np.array_equal(cache.lens(0), orc.lens[0])
    assert np.all(np.isfinite(got))
    for b in range(B):
        assert np.all(got[b, :, n_new[b]:] == 0.0), "padded queries must be exactly 0"
    err = float(np.max(np.abs(got - want))) if got.size else 0.0
    assert err <= TOL, (ci, err)
    return err


def _contiguous(B, Hkv, d, max_len, window=0, ring=False):
    _cuda_or_skip()
    cache = KVCache(1, B, Hkv, max_len, d, dtype=BF16)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    orc = ref.OracleCache(1, B, Hkv, max_len, d)
    if window:
        cache.set_window(window, ring)
        orc.set_window(window, ring)
    return cache, orc


def _check_slots(cache, orc):
    kc, vc = cache.k[0].double().cpu().numpy(), cache.v[0].double().cpu().numpy()
    written = orc.pos[0] >= 0
    for b in range(cache.B):
        w = written[b]
        assert np.array_equal(kc[b][:, w], orc.k[0][b][:, w])
        assert np.array_equal(vc[b][:, w], orc.v[0][b][:, w])
    assert cache.device_status() == 0


@pytest.mark.parametrize("d", [16, 64, 96, 256])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_bf16_generic_chunks(d, G):
    """Prefill, ragged verify chunks and decode; row blocks and 32-key tiles with ragged tails."""
    B, Hkv = 3, 2
    rng = np.random.default_rng(d * 10 + G)
    chunks = [150, 7, 40, 1, 1, 33]
    calls = []
    for c in chunks:
        n = rng.integers(max(0, c - 5), c + 1, size=B)
        n[0] = c
        calls.append(n)
    cache, orc = _contiguous(B, Hkv, d, int(sum(chunks)) + 9)
    for ci, n in enumerate(calls):
        _step(cache, orc, 5, ci, G, n)
    _check_slots(cache, orc)


def test_bf16_generic_empty_rows_and_zero_tokens():
    cache, orc = _contiguous(3, 2, 64, 40)
    for ci, n in enumerate([[0, 5, 0], [3, 0, 0], [1, 1, 0], [0, 0, 0]]):
        _step(cache, orc, 9, ci, 4, n)
    _check_slots(cache, orc)


@pytest.mark.parametrize("window,ring,max_len", [(9, False, 200), (24, True, 128), (128, True, 128)])
def test_bf16_generic_window(window, ring, max_len):
    cache, orc = _contiguous(2, 2, 64, max_len, window, ring)
    rng = np.random.default_rng(window)
    cap = max_len - window + 1 if ring else 12
    n_calls = (4 * max_len) // min(12, cap) if ring else 10  # enough to wrap the ring
    calls = [rng.integers(0, min(12, cap) + 1, size=2) for _ in range(n_calls)]
    for ci, n in enumerate(calls):
        _step(cache, orc, 3, ci, 4, n)
    if ring:
        assert np.any(orc.lens[0] > max_len)  # the ring wrapped
    _check_slots(cache, orc)


def test_bf16_generic_tree():
    B, Hkv, G, T, d = 4, 2, 4, 8, 64
    cache, orc = _contiguous(B, Hkv, d, 400)
    _step(cache, orc, 1, 0, G, np.array([300, 211, 77, 5]))
    rng = np.random.default_rng(2)
    parents = np.stack([np.arange(-1, T - 1), np.full(T, -1)] +
                       [np.array([-1] + [int(rng.integers(-1, t)) for t in range(1, T)]) for _ in range(2)])
    _step(cache, orc, 1, 1, G, np.array([T, T, 5, T]), parents=parents)
    _check_slots(cache, orc)


@pytest.mark.parametrize("d,page", [(96, 16), (64, 128)])
def test_bf16_paged(d, page):
    """Pages in a shuffled pool: 16 tokens for d = 96 (any page size works off
    the TMA path), 128 for d = 64 (a 128-key split-KV tile lies in one page)."""
    _cuda_or_skip()
    B, Hkv, G, mpr = 3, 2, 4, 12
    num_pages = B * mpr + 4
    cache = PagedKVCache(1, B, Hkv, page, num_pages, mpr, d, dtype=BF16)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    table = np.random.default_rng(4).permutation(num_pages)[: B * mpr].astype(np.int32)
    cache.block_table.copy_(torch.as_tensor(table).view(B, mpr))
    orc = ref.OracleCache(1, B, Hkv, page * mpr, d)
    for ci, n in enumerate([[100, 37, 64], [5, 8, 1], [1, 1, 1], [1, 1, 0], [12, 0, 7]]):
        _step(cache, orc, 6, ci, G, n)
    # every stored row sits in its page, bit-exact
    kp, vp = cache.k[0].double().cpu().numpy(), cache.v[0].double().cpu().numpy()
    for b in range(B):
        for a in range(int(orc.lens[0][b])):
            pg, off = table[b * mpr + a // page], a % page
            assert np.array_equal(kp[pg, :, off], orc.k[0][b, :, a])
            assert np.array_equal(vp[pg, :, off], orc.v[0][b, :, a])
    assert cache.device_status() == 0


def test_bf16_generic_rejects_fast_path_only_calls():
    """Device-resident steps and the allocation-free call serve head_dim 128 and 64 only."""
    _cuda_or_skip()
    cache = KVCache(1, 2, 2, 64, 96, dtype=BF16)
    assert cache.workspace_bytes(8, 1) == 0
    q = torch.zeros((2, 8, 1, 96), dtype=BF16, device="cuda")
    with pytest.raises(KVCError):
        cache.gqa_attention_noalloc(0, q, [0, 0], out=torch.zeros_like(q))


@pytest.mark.parametrize("window", [0, 300])
def test_generic_split_key_range(window):
    """Few (row, KV head) units and long rows: the generic kernel splits each
    unit's key range across 16 CTAs and merges them (decode and verify)."""
    cache, orc = _contiguous(2, 2, 96, 2048, window)
    rng = np.random.default_rng(7 + window)
    calls = [np.array([1500, 1203]), np.ones(2, dtype=np.int64), np.array([4, 3]), np.ones(2, dtype=np.int64)]
    for ci, n in enumerate(calls):
        _step(cache, orc, 21, ci, 4, n)
    assert cache.workspace_bytes(8, 1) > 0  # decode splits the key range: partials need room
    _check_slots(cache, orc)


# ---------------------------------------------------------------------------
# d = 64 on the split-KV kernel
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("G,T", [(4, 1), (8, 2), (4, 8), (8, 8)])
def test_d64_split_kv_decode_shape_every_unit(G, T):
    """A Llama-style decode shape with 64-wide heads (B = 32, Hkv = 8, lengths
    in [1024, 4000]): three fused decode / verify steps (16 to 64 rows per KV
    head: one, two and four 16-row blocks), then every query of every (row,
    KV head) unit of the last step against the oracle."""
    _cuda_or_skip()
    B, Hkv, d, max_len, seed = 32, 8, 64, 4096, 12
    Hq = Hkv * G
    lens0 = wl.decode_lens(seed, B, 1024, 4000)
    cache = KVCache(1, B, Hkv, max_len, d, dtype=BF16)
    wl.fill_normal_(cache.k[0], seed, wl.STREAM_CACHE_K)
    wl.fill_normal_(cache.v[0], seed, wl.STREAM_CACHE_V)
    for b, L in enumerate(lens0):
        cache.k[0][b, :, int(L):] = float("nan")
        cache.v[0][b, :, int(L):] = float("nan")
    cache.set_lens(0, lens0)
    orc = UnitOracle(seed, B, Hkv, max_len, d, lens0)
    for step in range(3):
        nn = np.full(B, T, dtype=np.int64)
        nn[step] = 0  # a row that skips a step
        k = wl.to_storage(wl.normal(seed, 1000 + 2 * step, (B, Hkv, T, d)), BF16)
        v = wl.to_storage(wl.normal(seed, 1001 + 2 * step, (B, Hkv, T, d)), BF16)
        q = wl.to_storage(wl.normal(seed, 5000 + step, (B, Hq, T, d)), BF16)
        out = cache.append_attention(0, q.cuda(), k.cuda(), v.cuda(), nn)
        want = orc.step(q, k, v, nn)
    torch.cuda.synchronize()
    assert max_error(out, want, nn, orc.units, Hkv) <= TOL
    assert cache.device_status() == 0
    lens = cache.lens(0)
    for b, kvh in orc.units:  # every stored row bit-exact, appended ones included
        L = int(lens[b])
        assert np.array_equal(cache.k[0][b, kvh, :L].double().cpu().numpy(), orc.K[b, kvh][0])
        assert np.array_equal(cache.v[0][b, kvh, :L].double().cpu().numpy(), orc.V[b, kvh][0])


def test_d64_device_step_and_graph_replay():
    """kvc_decode_step on a d = 64 cache, eager then replayed from a CUDA graph:
    every output of every step against the oracle."""
    _cuda_or_skip()
    B, Hkv, G, T, d, max_len, seed = 8, 4, 4, 1, 64, 2048, 14
    Hq = Hkv * G
    lens0 = wl.decode_lens(seed, B, 600, 1800)
    cache = KVCache(1, B, Hkv, max_len, d, dtype=BF16)
    wl.fill_normal_(cache.k[0], seed, wl.STREAM_CACHE_K)
    wl.fill_normal_(cache.v[0], seed, wl.STREAM_CACHE_V)
    cache.set_lens(0, lens0)
    orc = UnitOracle(seed, B, Hkv, max_len, d, lens0)
    ws = cache.workspace(Hq, T)
    cache.lens_to_device()
    sq = torch.empty((B, Hq, T, d), dtype=BF16, device="cuda")
    sk = torch.empty((B, Hkv, T, d), dtype=BF16, device="cuda")
    sv = torch.empty_like(sk)
    snn = torch.ones(B, dtype=torch.int32, device="cuda")
    sout = torch.empty_like(sq)
    graph = None
    lens = lens0.copy()
    for step in range(6):
        nn = np.ones(B, dtype=np.int64)
        nn[step % B] = 0
        lens += nn
        k = wl.to_storage(wl.normal(seed, 1000 + 2 * step, (B, Hkv, T, d)), BF16)
        v = wl.to_storage(wl.normal(seed, 1001 + 2 * step, (B, Hkv, T, d)), BF16)
        q = wl.to_storage(wl.normal(seed, 5000 + step, (B, Hq, T, d)), BF16)
        sq.copy_(q), sk.copy_(k), sv.copy_(v)
        snn.copy_(torch.from_numpy(nn.astype(np.int32)))
        if step == 0:
            cache.decode_step(0, sq, sk, sv, snn, sout, ws)  # first use outside the capture
            graph = torch.cuda.CUDAGraph()
        elif step == 1:
            with torch.cuda.graph(graph):
                cache.decode_step(0, sq, sk, sv, snn, sout, ws)
            graph.replay()
        else:
            graph.replay()
        torch.cuda.synchronize()
        assert max_error(sout, orc.step(q, k, v, nn), nn, orc.units, Hkv) <= TOL, step
    assert cache.device_status(ws) == 0
    cache.lens_from_device()
    assert np.array_equal(cache.lens(0), lens)


def test_d64_noalloc_matches_oracle():
    """The allocation-free entry point on a d = 64 cache (split-KV kernel, static scratch)."""
    _cuda_or_skip()
    B, Hkv, G, d, max_len = 4, 2, 4, 64, 1024
    cache, orc = _contiguous(B, Hkv, d, max_len)
    _step(cache, orc, 8, 0, G, np.array([700, 520, 311, 64]))  # the prefill chunk: 2800 rows, generic kernel
    for ci in range(1, 3):
        n = np.ones(B, dtype=np.int64)
        k = wl.to_storage(wl.normal(8, 100 + 3 * ci, (B, Hkv, 1, d)), BF16)
        v = wl.to_storage(wl.normal(8, 101 + 3 * ci, (B, Hkv, 1, d)), BF16)
        q = wl.to_storage(wl.normal(8, 102 + 3 * ci, (B, Hkv * G, 1, d)), BF16)
        cache.append(0, k.cuda(), v.cuda(), n)
        orc.append(0, k.double().numpy(), v.double().numpy(), n)
        out = torch.full((B, Hkv * G, 1, d), float("nan"), dtype=BF16, device="cuda")
        cache.gqa_attention_noalloc(0, q.cuda(), n, out=out)
        want = ref.gqa_attention(q.double().numpy(), orc, 0, n)
        assert float(np.max(np.abs(out.double().cpu().numpy() - want))) <= TOL, ci
    assert cache.noalloc_status() == 0
