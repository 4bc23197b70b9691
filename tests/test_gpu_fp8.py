"""FP8 E4M3 cache on the GPU against the oracle.

"16. Prefill, decode and the KV cache", exercise 4: the cache is stored in
FP8 E4M3 with one scale per KV head and dequantized on read.  Appends
quantize bf16 rows (code of x * (1/s), float32 reciprocal and product, ties
to even, saturating at +-448); the stored codes must equal the oracle's bit
for bit, and every attention output must be within 2e-2 of the float64
oracle reading the same codes.  Slots never written hold the NaN code 0x7F,
so a read of them fails.
"""

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import KVCache, PagedKVCache
from gqa_attention_preallocated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 2e-2
FP8 = torch.float8_e4m3fn


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _scales(Hkv, seed, lo=2.0 / 448, hi=6.0 / 448):
    """Per-head scales: N(0,1) data saturates beyond 448 * s (about 2 to 6 sigma)."""
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, Hkv).astype(np.float32), rng.uniform(lo, hi, Hkv).astype(np.float32)


def _pair(B, Hkv, max_len, seed, window=0, paged=None, d=128):
    if paged is None:
        cache = KVCache(1, B, Hkv, max_len, d, dtype=FP8)
        orc = ref.OracleCache(1, B, Hkv, max_len, d)
    else:
        page, num_pages, mpr, table = paged
        cache = PagedKVCache(1, B, Hkv, page, num_pages, mpr, 128, dtype=FP8)
        cache.block_table.copy_(torch.as_tensor(table, dtype=torch.int32).view(B, mpr))
        orc = ref.OracleCache(1, B, Hkv, mpr * page, 128)
    cache.k[0].view(torch.uint8).fill_(0x7F)
    cache.v[0].view(torch.uint8).fill_(0x7F)
    ks, vs = _scales(Hkv, seed)
    cache.set_kv_scales(0, ks, vs)
    orc.set_fp8()
    orc.set_kv_scales(0, ks.astype(np.float64), vs.astype(np.float64))
    if window:
        cache.set_window(window)
        orc.set_window(window)
    return cache, orc


def _codes_of(cache, orc, paged=None):
    """Compare every written slot's codes with the oracle's, bit for bit."""
    kc = cache.k[0].view(torch.uint8).cpu().numpy()
    vc = cache.v[0].view(torch.uint8).cpu().numpy()
    for b in range(orc.B):
        for a in range(int(orc.lens[0, b])):
            if paged is None:
                got_k, got_v = kc[b, :, a], vc[b, :, a]
            else:
                page, _, mpr, table = paged
                pg = int(np.asarray(table).reshape(orc.B, mpr)[b, a // page])
                got_k, got_v = kc[pg, :, a % page], vc[pg, :, a % page]
            assert np.array_equal(got_k, orc.k_code[0][b, :, a]), (b, a)
            assert np.array_equal(got_v, orc.v_code[0][b, :, a]), (b, a)


def _step(cache, orc, seed, ci, G, n_new, T=None, parents=None):
    B, Hkv, d = orc.B, orc.Hkv, orc.d
    n_new = np.asarray(n_new, dtype=np.int64)
    T = (max(int(n_new.max()), 1) if T is None else T) if parents is None else np.asarray(parents).shape[1]
    bf = torch.bfloat16
    k = wl.to_storage(wl.normal(seed, 100 + 3 * ci, (B, Hkv, T, d)), bf)
    v = wl.to_storage(wl.normal(seed, 101 + 3 * ci, (B, Hkv, T, d)), bf)
    q = wl.to_storage(wl.normal(seed, 102 + 3 * ci, (B, Hkv * G, T, d)), bf)
    if parents is None:
        out = cache.append_attention(0, q.cuda(), k.cuda(), v.cuda(), n_new)
    else:
        out = cache.append_attention_tree(0, q.cuda(), k.cuda(), v.cuda(), n_new, parents)
    want = ref.append_attention(orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), n_new,
                                parents=parents)
    got = out.double().cpu().numpy()
    assert np.array_equal(cache.lens(0), orc.lens[0])
    assert np.all(np.isfinite(got))
    for b in range(B):
        assert np.all(got[b, :, n_new[b]:] == 0.0)
    err = float(np.max(np.abs(got - want)))
    assert err <= TOL, (ci, err)
    return err


@pytest.mark.parametrize(
    "B,Hkv,G,chunks",
    [
        (4, 2, 4, [300, 1, 1, 1]),        # prefill (tensor-core kernel), then decode (split-KV, append fused)
        (3, 2, 4, [200, 4, 4]),           # verify at 16 rows (split-KV kernel, append fused)
        (2, 2, 8, [150, 4, 8, 1]),        # 32 rows (split-KV) and 64 rows (tensor-core) per KV head
        (2, 1, 1, [77, 5, 16, 1]),        # MHA
        (1, 8, 4, [1, 63, 64, 65, 129]),  # tile boundaries
        (2, 2, 8, [150, 40, 17, 12]),     # packed rows on the tensor-core kernel: 320, 136 and 96 rows
    ],
)
def test_fp8_chunks_against_oracle(B, Hkv, G, chunks):
    _cuda_or_skip()
    rng = np.random.default_rng(B * 100 + Hkv * 10 + G)
    cache, orc = _pair(B, Hkv, int(sum(chunks)) + 7, B + G)
    for ci, c in enumerate(chunks):
        n = rng.integers(max(0, c - 3), c + 1, size=B)
        n[0] = c
        _step(cache, orc, 11, ci, G, n)
    _codes_of(cache, orc)
    assert cache.device_status() == 0


def test_fp8_long_rows_split_over_ctas():
    """Rows long enough that units straddle CTAs (partials merged by the combine kernel)."""
    _cuda_or_skip()
    B, Hkv, G = 2, 2, 4
    cache, orc = _pair(B, Hkv, 6000, 3)
    _step(cache, orc, 12, 0, G, [5000, 3300])
    for ci in range(1, 4):
        _step(cache, orc, 12, ci, G, [1, 1])
    _codes_of(cache, orc)


def test_fp8_with_window():
    _cuda_or_skip()
    cache, orc = _pair(2, 2, 1024, 4, window=300)
    _step(cache, orc, 13, 0, 4, [700, 500])
    for ci in range(1, 5):
        _step(cache, orc, 13, ci, 4, [1, 4], T=4)
    _codes_of(cache, orc)


def test_fp8_over_pages():
    _cuda_or_skip()
    B, Hkv, page, mpr = 3, 2, 128, 8
    table = np.random.default_rng(5).permutation(B * mpr)
    paged = (page, B * mpr, mpr, table)
    cache, orc = _pair(B, Hkv, None, 5, paged=paged)
    _step(cache, orc, 14, 0, 4, [600, 300, 900])
    for ci in range(1, 4):
        _step(cache, orc, 14, ci, 4, [1, 1, 1])
    _codes_of(cache, orc, paged=paged)
    assert cache.device_status() == 0


def test_fp8_tree_verify():
    _cuda_or_skip()
    B, Hkv, G, T = 4, 2, 4, 8
    cache, orc = _pair(B, Hkv, 1200, 6)
    _step(cache, orc, 15, 0, G, [700, 300, 1000, 128])
    rng = np.random.default_rng(7)
    parents = np.stack([np.array([-1] + [int(rng.integers(-1, t)) for t in range(1, T)]) for _ in range(B)])
    _step(cache, orc, 15, 1, G, np.full(B, T), parents=parents)


def test_fp8_decode_step_matches_host_path():
    _cuda_or_skip()
    B, Hkv, G, T = 8, 4, 4, 1
    caches = []
    for _ in range(2):
        c, _ = _pair(B, Hkv, 2048, 8)
        k = wl.to_storage(wl.normal(9, 1, (B, Hkv, 1500, 128)), torch.bfloat16).cuda()
        v = wl.to_storage(wl.normal(9, 2, (B, Hkv, 1500, 128)), torch.bfloat16).cuda()
        c.append(0, k, v, wl.decode_lens(9, B, 600, 1500))
        caches.append(c)
    host, dev = caches
    ws = dev.workspace(Hkv * G, T)
    dev.lens_to_device()
    out = torch.empty((B, Hkv * G, T, 128), dtype=torch.bfloat16, device="cuda")
    nn = torch.ones(B, dtype=torch.int32, device="cuda")
    for step in range(5):
        q = wl.to_storage(wl.normal(9, 500 + step, (B, Hkv * G, T, 128)), torch.bfloat16).cuda()
        k = wl.to_storage(wl.normal(9, 600 + step, (B, Hkv, T, 128)), torch.bfloat16).cuda()
        v = wl.to_storage(wl.normal(9, 700 + step, (B, Hkv, T, 128)), torch.bfloat16).cuda()
        want = host.append_attention(0, q, k, v, np.ones(B))
        dev.decode_step(0, q, k, v, nn, out, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, want), step
    assert dev.device_status(ws) == 0
    dev.lens_from_device()
    assert np.array_equal(dev.lens(0), host.lens(0))
    assert torch.equal(dev.k[0].view(torch.uint8), host.k[0].view(torch.uint8))


def test_fp8_against_bf16_cache_over_many_decode_steps():
    """The page's experiment, on attention outputs (no model here): the same
    1,000 decode steps through an FP8 cache and a bf16 cache.  The difference
    is the quantization error only; it is reported and must stay small."""
    _cuda_or_skip()
    B, Hkv, G, steps, d = 4, 2, 4, 1000, 128
    f8 = KVCache(1, B, Hkv, 2048, d, dtype=FP8)
    bf = KVCache(1, B, Hkv, 2048, d, dtype=torch.bfloat16)
    s = np.full(Hkv, 4.0 / 448, dtype=np.float32)  # N(0,1): 4 sigma maps to 448
    f8.set_kv_scales(0, s, s)
    k0 = wl.to_storage(wl.normal(10, 1, (B, Hkv, 512, d)), torch.bfloat16).cuda()
    v0 = wl.to_storage(wl.normal(10, 2, (B, Hkv, 512, d)), torch.bfloat16).cuda()
    for c in (f8, bf):
        c.append(0, k0, v0, np.full(B, 512))
    worst, total = 0.0, 0.0
    for step in range(steps):
        q = wl.to_storage(wl.normal(10, 10000 + step, (B, Hkv * G, 1, d), device="cuda"), torch.bfloat16)
        k = wl.to_storage(wl.normal(10, 20000 + step, (B, Hkv, 1, d), device="cuda"), torch.bfloat16)
        v = wl.to_storage(wl.normal(10, 30000 + step, (B, Hkv, 1, d), device="cuda"), torch.bfloat16)
        a = f8.append_attention(0, q, k, v, np.ones(B)).float()
        b = bf.append_attention(0, q, k, v, np.ones(B)).float()
        diff = (a - b).abs()
        worst = max(worst, float(diff.max()))
        total += float(diff.mean())
    print(f"fp8 vs bf16 cache over {steps} decode steps: max-abs {worst:.4f}, mean-abs {total / steps:.5f}")
    assert worst < 0.1 and total / steps < 0.01


@pytest.mark.parametrize("T,G", [(1, 4), (8, 8)])
def test_fp8_full_size_sampled(T, G):
    """The decode8b shape (B=32, Hkv=8, [32, 8, 8192, 128]) on an FP8 cache at full size, in the
    launch configuration the benchmark times: one step, then sampled (row, KV head) units checked
    query by query against the oracle reading the cache's own codes (T = 8, G = 8 runs on the
    tensor-core kernel's FP8 variant)."""
    _cuda_or_skip()
    s = wl.DECODE_8B
    B, Hkv, L, d = s.B, s.Hkv, s.max_len, s.d
    cache = KVCache(1, B, Hkv, L, d, dtype=FP8)
    sc = np.full(Hkv, 4.0 / 448, dtype=np.float32)
    cache.set_kv_scales(0, sc, sc)
    for buf, stream in ((cache.k[0], wl.STREAM_CACHE_K), (cache.v[0], wl.STREAM_CACHE_V)):
        flat = buf.view(-1)
        for start in range(0, flat.numel(), 1 << 26):
            stop = min(flat.numel(), start + (1 << 26))
            idx = torch.arange(start, stop, dtype=torch.int64, device="cuda")
            x = wl.normal_at(21, stream, idx).to(torch.float32) * (448 / 4.0)
            flat[start:stop] = x.clamp_(-448.0, 448.0).to(FP8)
    lens0 = wl.decode_lens(21, B, 1024, L - 256)
    cache.set_lens(0, lens0)
    Hq = Hkv * G
    q = wl.to_storage(wl.normal(21, 5, (B, Hq, T, d)), torch.bfloat16)
    k = wl.to_storage(wl.normal(21, 6, (B, Hkv, T, d)), torch.bfloat16)
    v = wl.to_storage(wl.normal(21, 7, (B, Hkv, T, d)), torch.bfloat16)
    nn = np.full(B, T)
    out = cache.append_attention(0, q.cuda(), k.cuda(), v.cuda(), nn).double().cpu().numpy()
    assert cache.device_status() == 0
    qd = q.double().numpy()
    worst = 0.0
    for b, kvh in [(0, 0), (int(np.argmax(lens0)), 7), (17, 3)]:
        Lb = int(lens0[b]) + T
        K = ref.e4m3_dequantize(cache.k[0][b, kvh, :Lb].view(torch.uint8).cpu().numpy(), sc[kvh])
        V = ref.e4m3_dequantize(cache.v[0][b, kvh, :Lb].view(torch.uint8).cpu().numpy(), sc[kvh])
        for g in range(G):
            for t in range(T):
                want = ref.attend_one_query(qd[b, kvh * G + g, t], K, V, ref.query_position(Lb, T, t))
                worst = max(worst, float(np.max(np.abs(out[b, kvh * G + g, t] - want))))
    assert worst <= TOL, worst


def test_fp8_ring_storage():
    """Ring storage (slot = position mod max_len) with a window over an FP8 cache, past the wrap."""
    _cuda_or_skip()
    B, Hkv, G, max_len, W = 2, 2, 4, 512, 300
    cache = KVCache(1, B, Hkv, max_len, 128, dtype=FP8)
    cache.k[0].view(torch.uint8).fill_(0x7F)
    cache.v[0].view(torch.uint8).fill_(0x7F)
    ks, vs = _scales(Hkv, 16)
    cache.set_kv_scales(0, ks, vs)
    cache.set_window(W, ring=True)
    orc = ref.OracleCache(1, B, Hkv, max_len, 128)
    orc.set_fp8()
    orc.set_kv_scales(0, ks.astype(np.float64), vs.astype(np.float64))
    orc.set_window(W, ring=True)
    rng = np.random.default_rng(17)
    for ci in range(6):
        _step(cache, orc, 18, ci, G, rng.integers(100, max_len - W + 2, size=B))
    for ci in range(6, 10):
        _step(cache, orc, 18, ci, G, [1, 1])
    assert np.all(orc.lens[0] > max_len)  # the ring wrapped
    assert cache.device_status() == 0


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("window", [0, 200])
def test_fp8_other_head_dims_on_the_generic_kernel(d, window):
    """FP8 caches of d != 128: codes bit-exact, outputs against the oracle's
    dequantized values.  A prefill chunk, then decode over long rows (the key
    range split across CTAs) and a verify chunk."""
    _cuda_or_skip()
    cache, orc = _pair(2, 2, 1600, 31 + d, window=window, d=d)
    for ci, n in enumerate([np.array([1200, 907]), np.array([1, 1]), np.array([4, 2]), np.array([1, 0])]):
        _step(cache, orc, 40 + d, ci, 4, n)
    _codes_of(cache, orc)
    assert cache.device_status() == 0


def test_fp8_head_dim_64_tree():
    _cuda_or_skip()
    cache, orc = _pair(3, 1, 400, 5, d=64)
    _step(cache, orc, 6, 0, 8, np.array([300, 211, 77]))
    parents = np.array([[-1, 0, 1, 2, 3, 4], [-1, -1, -1, -1, -1, -1], [-1, 0, 0, 1, 1, 2]])
    _step(cache, orc, 6, 1, 8, np.array([6, 6, 4]), parents=parents)
    _codes_of(cache, orc)
