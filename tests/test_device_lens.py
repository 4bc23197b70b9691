"""Device-resident lengths: graph-capturable decode steps (kvc_decode_step).

The step reads and advances the lengths in device memory and computes its
work partition on the device, so it can be captured in a CUDA graph ("16.
Prefill, decode and the KV cache", the cache protocol paragraph after
"Design choices worth noticing": a static cache for CUDA graphs).  It must
give exactly what the host-planned path gives: both use one CTA per SM over
the same tile partition when the call has at least one tile per SM, so the
outputs are compared bit for bit, and one unit per case against the oracle.
"""

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import KVCache, KVCError
from gqa_attention_preallocated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _pair(B, Hkv, max_len, lens0, seed):
    """Two caches with the same content and lengths."""
    caches = []
    for _ in range(2):
        c = KVCache(1, B, Hkv, max_len, 128)
        wl.fill_normal_(c.k[0], seed, wl.STREAM_CACHE_K)
        wl.fill_normal_(c.v[0], seed, wl.STREAM_CACHE_V)
        c.set_lens(0, lens0)
        caches.append(c)
    return caches


def _step_inputs(seed, step, B, Hkv, Hq, T):
    k = wl.to_storage(wl.normal(seed, 1000 + 2 * step, (B, Hkv, T, 128)), torch.bfloat16).cuda()
    v = wl.to_storage(wl.normal(seed, 1001 + 2 * step, (B, Hkv, T, 128)), torch.bfloat16).cuda()
    q = wl.to_storage(wl.normal(seed, 5000 + step, (B, Hq, T, 128)), torch.bfloat16).cuda()
    return q, k, v


def _n_new(seed, step, B, T):
    rng = np.random.default_rng(seed * 100 + step)
    nn = rng.integers(0, T + 1, size=B)
    nn[0] = T  # at least one row with the full chunk
    return nn.astype(np.int64)


@pytest.mark.parametrize("T,G", [(1, 4), (4, 4), (2, 8)])
def test_decode_step_matches_host_path(T, G):
    _cuda_or_skip()
    B, Hkv, max_len, seed = 8, 8, 4096, 3
    Hq = Hkv * G
    lens0 = wl.decode_lens(seed, B, 1000, 3000)
    host, dev = _pair(B, Hkv, max_len, lens0, seed)
    ws = dev.workspace(Hq, T)
    dev.lens_to_device()
    out_dev = torch.empty((B, Hq, T, 128), dtype=torch.bfloat16, device="cuda")
    for step in range(5):
        q, k, v = _step_inputs(seed, step, B, Hkv, Hq, T)
        nn = _n_new(seed, step, B, T)
        want = host.append_attention(0, q, k, v, nn)
        dev.decode_step(0, q, k, v, torch.from_numpy(nn.astype(np.int32)).cuda(), out_dev, ws)
        torch.cuda.synchronize()
        if G * T <= 12:
            # both calls run the split-KV kernel: the same arithmetic, bit for bit
            assert torch.equal(out_dev, want), step
        else:
            # the host path runs above 12 rows per KV head on the tensor-core kernel
            assert float((out_dev.float() - want.float()).abs().max()) <= 2e-2, step
    assert dev.device_status(ws) == 0
    dev.lens_from_device()
    assert np.array_equal(dev.lens(0), host.lens(0))
    L = int(dev.lens(0)[0])
    assert torch.equal(dev.k[0][:, :, :L], host.k[0][:, :, :L]) and torch.equal(dev.v[0][:, :, :L], host.v[0][:, :, :L])
    # one unit of the last step against the oracle (row 0 took the full chunk)
    K = dev.k[0][0, 1, :L].double().cpu().numpy()
    V = dev.v[0][0, 1, :L].double().cpu().numpy()
    qd = q.double().cpu().numpy()
    for g in range(G):
        for t in range(T):
            w = ref.attend_one_query(qd[0, G + g, t], K, V, ref.query_position(L, T, t))
            assert np.max(np.abs(out_dev[0, G + g, t].double().cpu().numpy() - w)) <= 2e-2


def test_decode_step_replayed_from_a_cuda_graph():
    _cuda_or_skip()
    B, Hkv, G, T, max_len, seed = 16, 8, 4, 1, 8192, 7
    Hq = Hkv * G
    lens0 = wl.decode_lens(seed, B, 2000, 6000)
    host, dev = _pair(B, Hkv, max_len, lens0, seed)
    ws = dev.workspace(Hq, T)
    dev.lens_to_device()
    sq = torch.empty((B, Hq, T, 128), dtype=torch.bfloat16, device="cuda")
    sk = torch.empty((B, Hkv, T, 128), dtype=torch.bfloat16, device="cuda")
    sv = torch.empty_like(sk)
    snn = torch.ones(B, dtype=torch.int32, device="cuda")
    sout = torch.empty_like(sq)
    # step 0 runs eagerly (first-use set-up happens outside the capture)
    q, k, v = _step_inputs(seed, 0, B, Hkv, Hq, T)
    sq.copy_(q), sk.copy_(k), sv.copy_(v)
    dev.decode_step(0, sq, sk, sv, snn, sout, ws)
    want = host.append_attention(0, q, k, v, np.ones(B))
    torch.cuda.synchronize()
    assert torch.equal(sout, want)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dev.decode_step(0, sq, sk, sv, snn, sout, ws)
    for step in range(1, 9):
        q, k, v = _step_inputs(seed, step, B, Hkv, Hq, T)
        nn = np.ones(B, dtype=np.int64)
        nn[step % B] = 0  # a row that skips a step
        sq.copy_(q), sk.copy_(k), sv.copy_(v)
        snn.copy_(torch.from_numpy(nn.astype(np.int32)))
        g.replay()
        want = host.append_attention(0, q, k, v, nn)
        torch.cuda.synchronize()
        assert torch.equal(sout, want), step
    assert dev.device_status(ws) == 0
    dev.lens_from_device()
    assert np.array_equal(dev.lens(0), host.lens(0))


def test_decode_step_overflow_rejects_the_whole_step():
    _cuda_or_skip()
    B, Hkv, G, T, max_len = 4, 2, 4, 2, 256
    lens0 = np.array([10, 255, 100, 0])  # row 1 has room for one token only
    c = KVCache(1, B, Hkv, max_len, 128)
    wl.fill_normal_(c.k[0], 1, wl.STREAM_CACHE_K)
    wl.fill_normal_(c.v[0], 1, wl.STREAM_CACHE_V)
    c.set_lens(0, lens0)
    k_before, v_before = c.k[0].clone(), c.v[0].clone()
    ws = c.workspace(Hkv * G, T)
    c.lens_to_device()
    q, k, v = _step_inputs(1, 0, B, Hkv, Hkv * G, T)
    out = torch.full_like(q, 7.0)
    c.decode_step(0, q, k, v, torch.tensor([2, 2, 1, 0], dtype=torch.int32, device="cuda"), out, ws)
    with pytest.raises(KVCError) as e:
        c.device_status(ws)
    assert e.value.status == 3  # KVC_ERR_OVERFLOW
    assert torch.equal(c.k[0], k_before) and torch.equal(c.v[0], v_before)
    assert bool((out == 7.0).all())  # nothing written
    c.lens_from_device()
    assert list(c.lens(0)) == list(lens0)


def test_host_length_calls_refused_while_on_device():
    _cuda_or_skip()
    c = KVCache(2, 3, 2, 64, 128)
    c.set_lens(0, [1, 2, 3])
    c.set_lens(1, [1, 2, 3])
    c.lens_to_device()
    k = torch.zeros((3, 2, 1, 128), dtype=torch.bfloat16, device="cuda")
    for call in (lambda: c.append(0, k, k, [1, 1, 1]), lambda: c.length(), lambda: c.truncate([0, 0, 0]),
                 lambda: c.reset(), lambda: c.lens(0), lambda: c.set_lens(0, [0, 0, 0])):
        with pytest.raises(KVCError) as e:
            call()
        assert e.value.status == 1
    with pytest.raises(KVCError):
        c.lens_to_device()  # already there
    c.lens_from_device()
    assert list(c.length()) == [1, 2, 3]
