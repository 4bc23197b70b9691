"""Device-resident lengths: graph-capturable decode steps (kvc_decode_step).

The step reads and advances the lengths in device memory and computes its
work partition on the device, so it can be captured in a CUDA graph ("16.
Prefill, decode and the KV cache", the cache protocol paragraph after
"Design choices worth noticing": a static cache for CUDA graphs).  It must
give what the host-planned path gives.  Every output of every step (eager
and replayed from a CUDA graph) is compared with the float64 oracle; where
both paths run the same kernel over the same partition, the outputs are also
equal bit for bit.
"""

import numpy as np
import pytest
import torch

from gqa_attention_preallocated_gb300 import KVCache, KVCError
from gqa_attention_preallocated_gb300 import workloads as wl
from oracle_rows import UnitOracle, max_error

TOL_BF16 = 2e-2

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
    """A step's q, k_new, v_new as stored (bf16), on the CPU; the GPU copies are made by the caller."""
    k = wl.to_storage(wl.normal(seed, 1000 + 2 * step, (B, Hkv, T, 128)), torch.bfloat16)
    v = wl.to_storage(wl.normal(seed, 1001 + 2 * step, (B, Hkv, T, 128)), torch.bfloat16)
    q = wl.to_storage(wl.normal(seed, 5000 + step, (B, Hq, T, 128)), torch.bfloat16)
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
    orc = UnitOracle(seed, B, Hkv, max_len, 128, lens0)
    ws = dev.workspace(Hq, T)
    dev.lens_to_device()
    out_dev = torch.empty((B, Hq, T, 128), dtype=torch.bfloat16, device="cuda")
    for step in range(5):
        q, k, v = _step_inputs(seed, step, B, Hkv, Hq, T)
        nn = _n_new(seed, step, B, T)
        want_host = host.append_attention(0, q.cuda(), k.cuda(), v.cuda(), nn)
        dev.decode_step(0, q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(nn.astype(np.int32)).cuda(), out_dev, ws)
        torch.cuda.synchronize()
        want = orc.step(q, k, v, nn)
        assert max_error(out_dev, want, nn, orc.units, Hkv) <= TOL_BF16, step
        if G * T <= 12:
            # both calls run the split-KV kernel over the same partition: bit for bit
            assert torch.equal(out_dev, want_host), step
    assert dev.device_status(ws) == 0
    dev.lens_from_device()
    assert np.array_equal(dev.lens(0), host.lens(0))
    # every appended row as stored by the device step, bit for bit against the oracle's rows
    lens = dev.lens(0)
    for b, kvh in orc.units:
        L = int(lens[b])
        assert np.array_equal(dev.k[0][b, kvh, :L].double().cpu().numpy(), orc.K[b, kvh][0])
        assert np.array_equal(dev.v[0][b, kvh, :L].double().cpu().numpy(), orc.V[b, kvh][0])


def test_decode_step_replayed_from_a_cuda_graph():
    _cuda_or_skip()
    B, Hkv, G, T, max_len, seed = 16, 8, 4, 1, 8192, 7
    Hq = Hkv * G
    lens0 = wl.decode_lens(seed, B, 2000, 6000)
    host, dev = _pair(B, Hkv, max_len, lens0, seed)
    orc = UnitOracle(seed, B, Hkv, max_len, 128, lens0)
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
    want_host = host.append_attention(0, q.cuda(), k.cuda(), v.cuda(), np.ones(B))
    torch.cuda.synchronize()
    nn = np.ones(B, dtype=np.int64)
    assert max_error(sout, orc.step(q, k, v, nn), nn, orc.units, Hkv) <= TOL_BF16
    assert torch.equal(sout, want_host)
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
        want_host = host.append_attention(0, q.cuda(), k.cuda(), v.cuda(), nn)
        torch.cuda.synchronize()
        assert max_error(sout, orc.step(q, k, v, nn), nn, orc.units, Hkv) <= TOL_BF16, step
        assert torch.equal(sout, want_host), step
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
    q, k, v = (x.cuda() for x in _step_inputs(1, 0, B, Hkv, Hkv * G, T))
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
