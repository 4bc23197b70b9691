"""The host-buffer form of append + attention against the float64 oracle.

q, k_new, v_new and out live in page-locked host memory; the library copies
positions t < n_new[b] in and out on its own copy streams, through two device
staging slots that alternate from call to call.  Every case issues all of its
calls before waiting once, so inputs, compute and outputs of neighbouring
calls are in flight together and the slots are reused while earlier copies
may still run.  Each call's output is compared with the oracle ("A strong
answer": KVCache.append then gqa_attention); the positions of out_host at or
past n_new[b] must keep what they held, and the cache's stored rows must equal
the oracle's bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import KVCache, KVCError
from gqa_attention_preallocated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
FP8 = torch.float8_e4m3fn
SENTINEL = 7.0  # out_host's initial value: positions the call must not write keep it


def _cuda_or_skip():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _pair(B, Hkv, max_len, d, dtype, seed):
    cache = KVCache(1, B, Hkv, max_len, d, dtype=dtype)
    orc = ref.OracleCache(1, B, Hkv, max_len, d)
    if dtype == FP8:
        cache.k[0].view(torch.uint8).fill_(0x7F)
        cache.v[0].view(torch.uint8).fill_(0x7F)
        rng = np.random.default_rng(seed)
        ks = rng.uniform(2.0 / 448, 6.0 / 448, Hkv).astype(np.float32)
        vs = rng.uniform(2.0 / 448, 6.0 / 448, Hkv).astype(np.float32)
        cache.set_kv_scales(0, ks, vs)
        orc.set_fp8()
        orc.set_kv_scales(0, ks.astype(np.float64), vs.astype(np.float64))
    else:
        cache.k[0].fill_(float("nan"))
        cache.v[0].fill_(float("nan"))
    return cache, orc


def _inputs(seed, ci, B, Hkv, G, T, d, io):
    k = wl.to_storage(wl.normal(seed, 100 + 3 * ci, (B, Hkv, T, d)), io)
    v = wl.to_storage(wl.normal(seed, 101 + 3 * ci, (B, Hkv, T, d)), io)
    q = wl.to_storage(wl.normal(seed, 102 + 3 * ci, (B, Hkv * G, T, d)), io)
    return q, k, v


def _issue(cache, orc, seed, ci, G, n_new, io, T=None):
    """Enqueue one host-buffer call and the oracle's answer; return what to check after the wait."""
    B, Hkv, d = orc.B, orc.Hkv, orc.d
    n_new = np.asarray(n_new, dtype=np.int64)
    T = max(int(n_new.max()), 1) if T is None else T
    q, k, v = _inputs(seed, ci, B, Hkv, G, T, d, io)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    hout = torch.full((B, Hkv * G, T, d), SENTINEL, dtype=io).pin_memory()
    cache.append_attention_host(0, hq, hk, hv, n_new, hout)
    want = ref.append_attention(orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), n_new)
    return (hq, hk, hv, hout, want, n_new)


def _check(pending, tol):
    worst = 0.0
    for hq, hk, hv, hout, want, n_new in pending:
        got = hout.double().numpy()
        for b in range(got.shape[0]):
            n = int(n_new[b])
            assert np.all(got[b, :, n:] == SENTINEL), "positions at or past n_new must not be written"
            part = got[b, :, :n]
            assert np.all(np.isfinite(part))
            if part.size:
                worst = max(worst, float(np.max(np.abs(part - want[b, :, :n]))))
    assert worst <= tol, worst
    return worst


def _stored_rows_equal(cache, orc):
    lens = cache.lens(0)
    assert np.array_equal(lens, orc.lens[0])
    if cache.k[0].dtype == FP8:
        kc = cache.k[0].view(torch.uint8).cpu().numpy()
        vc = cache.v[0].view(torch.uint8).cpu().numpy()
        for b in range(orc.B):
            L = int(lens[b])
            assert np.array_equal(kc[b, :, :L], orc.k_code[0][b, :, :L])
            assert np.array_equal(vc[b, :, :L], orc.v_code[0][b, :, :L])
        return
    kc = cache.k[0].double().cpu().numpy()
    vc = cache.v[0].double().cpu().numpy()
    for b in range(orc.B):
        L = int(lens[b])
        assert np.array_equal(kc[b, :, :L], orc.k[0][b, :, :L])
        assert np.array_equal(vc[b, :, :L], orc.v[0][b, :, :L])


@pytest.mark.parametrize(
    "dtype,d,B,Hkv,G,chunks",
    [
        # bf16: prefill (tcgen05 kernel), decode (split-KV, append fused), verify, a larger chunk that grows
        # the staging slots while earlier calls are in flight, and a ragged chunk with an empty row
        (torch.bfloat16, 128, 3, 2, 4, [40, 1, 300, 1, 4, 130]),
        (torch.bfloat16, 64, 4, 2, 4, [100, 1, 1, 3]),       # d = 64 on the split-KV kernel
        (FP8, 128, 2, 2, 4, [150, 1, 4, 1, 64]),             # FP8 storage: quantizing append, both kernels
        (torch.float32, 16, 3, 1, 2, [5, 1, 3, 1]),          # fp32 on the generic kernel
    ],
)
def test_host_calls_against_oracle(dtype, d, B, Hkv, G, chunks):
    _cuda_or_skip()
    io = torch.bfloat16 if dtype == FP8 else dtype
    rng = np.random.default_rng(B * 100 + Hkv * 10 + G + d)
    cache, orc = _pair(B, Hkv, int(sum(chunks)) + 9, d, dtype, seed=d + B)
    pending = []
    for ci, c in enumerate(chunks):
        n = rng.integers(max(0, c - 5), c + 1, size=B)
        n[0] = c
        if ci == len(chunks) - 1 and B > 1:
            n[1] = 0  # a row with nothing new
        pending.append(_issue(cache, orc, 31, ci, G, n, io))
    cache.host_copies_done()
    torch.cuda.synchronize()
    _check(pending, TOL[torch.bfloat16] if dtype == FP8 else TOL[dtype])
    _stored_rows_equal(cache, orc)
    assert cache.device_status() == 0


def test_host_call_error_changes_nothing():
    """A call that overflows a row, issued between valid calls, is refused
    before it enqueues anything: lengths, stored rows and its out_host stay
    as they were, and the calls around it are unaffected."""
    _cuda_or_skip()
    B, Hkv, G, d = 2, 2, 4, 128
    cache, orc = _pair(B, Hkv, 60, d, torch.bfloat16, seed=3)
    pending = [_issue(cache, orc, 5, 0, G, [50, 20], torch.bfloat16)]
    q, k, v = _inputs(5, 1, B, Hkv, G, 12, d, torch.bfloat16)
    bad_out = torch.full((B, Hkv * G, 12, d), SENTINEL, dtype=torch.bfloat16).pin_memory()
    with pytest.raises(KVCError) as e:
        cache.append_attention_host(0, q.pin_memory(), k.pin_memory(), v.pin_memory(), [12, 1], bad_out)
    assert e.value.status_name == "KVC_ERR_OVERFLOW"
    assert list(cache.lens(0)) == [50, 20]
    pending.append(_issue(cache, orc, 5, 2, G, [1, 1], torch.bfloat16))
    cache.host_copies_done()
    torch.cuda.synchronize()
    assert torch.all(bad_out == SENTINEL)
    _check(pending, TOL[torch.bfloat16])
    _stored_rows_equal(cache, orc)
    assert cache.device_status() == 0


def test_host_decode_loop_matches_device_calls():
    """Sixty-four decode8b-shaped steps (one token a row, lengths 1,000 to 3,000)
    through the host form, every step's output compared with the oracle on two
    sampled units, and the last step's output equal bit for bit to the same
    step through the device-buffer call on a second cache."""
    _cuda_or_skip()
    B, Hkv, G, d, steps = 8, 4, 4, 128, 64
    lens0 = np.random.default_rng(9).integers(1000, 3000, size=B)
    caches = []
    for _ in range(2):
        c = KVCache(1, B, Hkv, 3200, d, dtype=torch.bfloat16)
        c.k[0].copy_(wl.to_storage(wl.normal(2, wl.STREAM_CACHE_K, (B, Hkv, 3200, d), device="cuda"),
                                   torch.bfloat16))
        c.v[0].copy_(wl.to_storage(wl.normal(2, wl.STREAM_CACHE_V, (B, Hkv, 3200, d), device="cuda"),
                                   torch.bfloat16))
        c.set_lens(0, lens0)
        caches.append(c)
    from oracle_rows import UnitOracle

    units = [(0, 0), (B - 1, Hkv - 1)]
    orc = UnitOracle(2, B, Hkv, 3200, d, lens0, units)
    ones = np.ones(B, dtype=np.int64)
    pending = []
    for i in range(steps):
        q, k, v = _inputs(4, i, B, Hkv, G, 1, d, torch.bfloat16)
        hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        hout = torch.full((B, Hkv * G, 1, d), SENTINEL, dtype=torch.bfloat16).pin_memory()
        caches[0].append_attention_host(0, hq, hk, hv, ones, hout)
        dev_out = caches[1].append_attention(0, q.cuda(), k.cuda(), v.cuda(), ones)
        pending.append((hq, hk, hv, hout, orc.step(q, k, v, ones), dev_out))
    caches[0].host_copies_done()
    torch.cuda.synchronize()
    worst = 0.0
    for hq, hk, hv, hout, want, dev_out in pending:
        got = hout.double().numpy()
        for (b, h, t), w in want.items():
            worst = max(worst, float(np.max(np.abs(got[b, h, t] - w))))
    assert worst <= TOL[torch.bfloat16], worst
    assert torch.equal(pending[-1][3], pending[-1][5].cpu())
    assert np.array_equal(caches[0].lens(0), lens0 + steps)
