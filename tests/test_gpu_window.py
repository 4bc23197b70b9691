"""Sliding window and ring storage on the GPU against the oracle.

"Write the causal mask for a decode step with a KV cache...", "A strong
answer" (last paragraph) and "Common mistakes": with a window W the query at
position p sees keys p - W < a <= p, and in a ring cache the comparison uses
stored positions, not slots.  Every call's output is compared with the
float64 oracle on the same inputs (max-abs 1e-4 fp32, 2e-2 bf16); the cache
slots holding the window are compared bit for bit; slots never written hold
NaN, so any read of them fails.
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


def _run(seed, B, Hkv, G, d, max_len, dtype, window, ring, calls):
    _cuda_or_skip()
    cache = KVCache(1, B, Hkv, max_len, d, dtype=dtype)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    cache.set_window(window, ring)
    orc = ref.OracleCache(1, B, Hkv, max_len, d)
    orc.set_window(window, ring)
    worst = 0.0
    for ci, n_new in enumerate(calls):
        n_new = np.asarray(n_new, dtype=np.int64)
        T = max(int(n_new.max()), 1)
        k = wl.to_storage(wl.normal(seed, 100 + 3 * ci, (B, Hkv, T, d)), dtype)
        v = wl.to_storage(wl.normal(seed, 101 + 3 * ci, (B, Hkv, T, d)), dtype)
        q = wl.to_storage(wl.normal(seed, 102 + 3 * ci, (B, Hkv * G, T, d)), dtype)
        out = cache.append_attention(0, q.cuda(), k.cuda(), v.cuda(), n_new)
        want = ref.append_attention(orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), n_new)
        got = out.double().cpu().numpy()
        assert np.array_equal(cache.lens(0), orc.lens[0])
        assert np.all(np.isfinite(got))
        for b in range(B):
            assert np.all(got[b, :, n_new[b]:] == 0.0)
        err = float(np.max(np.abs(got - want)))
        worst = max(worst, err)
        assert err <= TOL[dtype], (ci, err)
    # every slot the oracle has written holds the same bits
    kc, vc = cache.k[0].double().cpu().numpy(), cache.v[0].double().cpu().numpy()
    written = orc.pos[0] >= 0
    for b in range(B):
        w = written[b]
        assert np.array_equal(kc[b][:, w], orc.k[0][b][:, w]) and np.array_equal(vc[b][:, w], orc.v[0][b][:, w])
    assert cache.device_status() == 0
    return worst, orc


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("window,ring,max_len", [(1, False, 64), (5, False, 64), (17, False, 64), (7, True, 16),
                                                  (9, True, 16), (16, True, 16)])
def test_f32_window_tiny(seed, window, ring, max_len):
    B, Hkv, G, d = 2, 2, 4, 16
    rng = np.random.default_rng(seed)
    cap = max_len - window + 1 if ring else 8
    calls = [rng.integers(0, min(8, cap) + 1, size=B) for _ in range(40 if ring else 6)]
    _, orc = _run(seed, B, Hkv, G, d, max_len, torch.float32, window, ring, calls)
    if ring:
        assert np.any(orc.lens[0] > max_len)  # the ring wrapped


@pytest.mark.parametrize("window,ring,max_len,T", [(100, False, 2048, 1), (700, False, 2048, 4), (300, True, 512, 1),
                                                    (300, True, 512, 4), (512, True, 512, 1)])
def test_bf16_decode_window(window, ring, max_len, T):
    B, Hkv, G, d = 4, 2, 4, 128
    rng = np.random.default_rng(window + T)
    cap = max_len - window + 1 if ring else 256
    lo, hi = min(100, cap), min(cap, 256)
    n_fill = 4 if not ring else int(np.ceil(1.3 * max_len / ((lo + hi) / 2)))
    calls = [rng.integers(lo, hi + 1, size=B) for _ in range(n_fill)]
    calls += [np.full(B, T) if i % 3 else rng.integers(0, T + 1, size=B) for i in range(10)]
    _run(7, B, Hkv, G, d, max_len, torch.bfloat16, window, ring, calls)


@pytest.mark.parametrize("window,ring,max_len", [(600, False, 2048), (200, False, 2048), (600, True, 1024)])
def test_bf16_prefill_window(window, ring, max_len):
    """Chunks of 256 (the tensor-core prefill kernel) with a window, ragged last chunk."""
    B, Hkv, G, d = 2, 2, 4, 128
    calls = [np.full(B, 256)] * 6 + [np.array([256, 131])]
    _, orc = _run(9, B, Hkv, G, d, max_len, torch.bfloat16, window, ring, calls)
    if ring:
        assert np.all(orc.lens[0] > max_len)


def test_decode_step_with_window_matches_host_path():
    _cuda_or_skip()
    B, Hkv, G, T, max_len, W = 8, 4, 4, 1, 1024, 300
    caches = []
    for _ in range(2):
        c = KVCache(1, B, Hkv, max_len, 128)
        c.set_window(W, ring=True)
        wl.fill_normal_(c.k[0], 2, wl.STREAM_CACHE_K)
        wl.fill_normal_(c.v[0], 2, wl.STREAM_CACHE_V)
        c.set_lens(0, wl.decode_lens(2, B, 1500, 3000))  # positions past max_len: the ring has wrapped
        caches.append(c)
    host, dev = caches
    ws = dev.workspace(Hkv * G, T)
    dev.lens_to_device()
    out = torch.empty((B, Hkv * G, T, 128), dtype=torch.bfloat16, device="cuda")
    nn = torch.ones(B, dtype=torch.int32, device="cuda")
    for step in range(6):
        q = wl.to_storage(wl.normal(2, 5000 + step, (B, Hkv * G, T, 128)), torch.bfloat16).cuda()
        k = wl.to_storage(wl.normal(2, 1000 + step, (B, Hkv, T, 128)), torch.bfloat16).cuda()
        v = wl.to_storage(wl.normal(2, 2000 + step, (B, Hkv, T, 128)), torch.bfloat16).cuda()
        want = host.append_attention(0, q, k, v, np.ones(B))
        dev.decode_step(0, q, k, v, nn, out, ws)
        torch.cuda.synchronize()
        assert torch.equal(out, want), step
    assert dev.device_status(ws) == 0
    dev.lens_from_device()
    assert np.array_equal(dev.lens(0), host.lens(0))
