"""GPU parity: the CUDA path through the C ABI against the float64 CPU oracle.

Every input comes from the seeded generators in ``workloads``; the oracle
sees the values exactly as stored (bf16 or fp32 widened to float64), so only
kernel error is measured.  Bars (stated for this method): the append and all
lengths bit-exact; outputs within max-abs 1e-4 for fp32 storage and 2e-2 for
bf16 storage; padded queries exactly 0.

Cache slots past the valid lengths are filled with NaN before each case
("poison"), so any output that touched them fails.
"""

import math

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


def _store(x64, dtype):
    return wl.to_storage(x64, dtype)


def _run_calls(seed, B, Hkv, G, d, max_len, dtype, calls, poison=True):
    """Feed the same appends+queries to the GPU cache and the oracle; compare every call."""
    _cuda_or_skip()
    cache = KVCache(1, B, Hkv, max_len, d, dtype=dtype)
    if poison:
        cache.k[0].fill_(float("nan"))
        cache.v[0].fill_(float("nan"))
    orc = ref.OracleCache(1, B, Hkv, max_len, d)
    tol = TOL[dtype]
    worst = 0.0
    for ci, n_new in enumerate(calls):
        n_new = np.asarray(n_new, dtype=np.int64)
        T = int(n_new.max()) if B else 0
        k_new = _store(wl.normal(seed, 100 + 3 * ci, (B, Hkv, T, d)), dtype)
        v_new = _store(wl.normal(seed, 101 + 3 * ci, (B, Hkv, T, d)), dtype)
        q = _store(wl.normal(seed, 102 + 3 * ci, (B, Hkv * G, T, d)), dtype)
        out = cache.append_attention(0, q.cuda(), k_new.cuda(), v_new.cuda(), n_new)
        want = ref.append_attention(orc, 0, q.double().numpy(), k_new.double().numpy(), v_new.double().numpy(), n_new)
        got = out.double().cpu().numpy()
        assert np.array_equal(cache.lens(0), orc.lens[0])
        for b in range(B):
            assert np.all(got[b, :, n_new[b]:] == 0.0), "padded queries must be exactly 0"
        assert np.all(np.isfinite(got))
        err = float(np.max(np.abs(got - want))) if got.size else 0.0
        worst = max(worst, err)
        assert err <= tol, (ci, err)
    # cache state: every valid slot bit-exact
    lens = cache.lens(0)
    kc = cache.k[0].double().cpu().numpy()
    vc = cache.v[0].double().cpu().numpy()
    for b in range(B):
        L = int(lens[b])
        assert np.array_equal(kc[b, :, :L], orc.k[0][b, :, :L])
        assert np.array_equal(vc[b, :, :L], orc.v[0][b, :, :L])
    assert cache.device_status() == 0
    return worst


# ---------------------------------------------------------------------------
# Tiny ragged configuration (fp32, d = 16) and the pages' randomized trials
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("seed", range(12))
def test_tiny_ragged_f32(seed):
    s = wl.TINY
    _, calls = wl.tiny_schedule(seed, s.B)
    _run_calls(seed, s.B, s.Hkv, s.G, s.d, s.max_len, torch.float32, calls)


def test_randomized_trials_f32():
    for seed in range(40):
        B, Hkv, G, d = wl.trial_geometry(seed)
        _, calls = wl.tiny_schedule(seed, B)
        _run_calls(seed, B, Hkv, G, d, 48, torch.float32, calls)


# ---------------------------------------------------------------------------
# bf16 split-KV kernel, small sizes that still span many tiles and CTAs
# ---------------------------------------------------------------------------


@pytest.mark.parametrize(
    "B,Hkv,G,chunks",
    [
        (3, 2, 4, [300, 1, 1, 1]),  # prefill then decode (G*T = 4 rows)
        (2, 1, 8, [130, 4, 8, 1]),  # MQA, verify chunks (32 and 64 rows)
        (3, 4, 1, [77, 5, 16, 1]),  # MHA
        (2, 2, 4, [520, 37, 100]),  # several row blocks per unit, ragged tails
        (1, 8, 4, [1, 63, 64, 65, 129]),  # tile boundaries
    ],
)
def test_bf16_chunked(B, Hkv, G, chunks):
    rng = np.random.default_rng(B * 100 + Hkv * 10 + G)
    calls = []
    for c in chunks:
        n = rng.integers(max(0, c - 3), c + 1, size=B)
        n[0] = c  # T = c
        calls.append(n)
    max_len = int(sum(chunks)) + 7
    _run_calls(11, B, Hkv, G, 128, max_len, torch.bfloat16, calls)


def test_bf16_rows_with_zero_tokens_and_empty_rows():
    calls = [np.array([0, 5, 0]), np.array([3, 0, 0]), np.array([1, 1, 0])]
    _run_calls(5, 3, 2, 4, 128, 40, torch.bfloat16, calls)


def test_bf16_many_short_units_sole_path():
    """Many units with total tiles >> SMs: most units finish inside one CTA."""
    B, Hkv, G = 64, 8, 4
    rng = np.random.default_rng(3)
    first = rng.integers(60, 200, size=B)
    calls = [first, np.ones(B, dtype=np.int64), np.ones(B, dtype=np.int64)]
    _run_calls(7, B, Hkv, G, 128, 256, torch.bfloat16, calls)


def test_bf16_maximum_batch():
    """KVC_MAX_BATCH rows, every output compared.  Calls:
    - a prefill chunk of up to 120 tokens: 480 packed rows per KV head, tensor cores;
    - decode steps: the split-KV kernel at its limit of 1024 (row, row block) groups;
    - verify chunks of 4 and 8: one packed tensor-core tile.
    Some rows take zero tokens."""
    B, Hkv, G, d, max_len = 1024, 1, 4, 128, 160
    rng = np.random.default_rng(1024)
    calls = [rng.integers(1, 121, size=B)]
    calls[0][0] = 120
    for T in (1, 1, 4, 8):
        n = rng.integers(0, T + 1, size=B)
        n[0] = T
        calls.append(n)
    _run_calls(13, B, Hkv, G, d, max_len, torch.bfloat16, calls)


@pytest.mark.parametrize("dtype,d", [(torch.float32, 16), (torch.bfloat16, 64)])
def test_generic_kernel_maximum_batch(dtype, d):
    """KVC_MAX_BATCH rows on the generic kernel: ragged chunks, then decode."""
    B, Hkv, G, max_len = 1024, 2, 2, 64
    rng = np.random.default_rng(d)
    calls = [rng.integers(0, 41, size=B), rng.integers(0, 2, size=B), rng.integers(0, 6, size=B)]
    for c in calls:
        c[0] = c.max()
    _run_calls(17, B, Hkv, G, d, max_len, dtype, calls)


def test_f32_split_key_range():
    """fp32 decode over long rows: the generic kernel splits each unit's keys across 16 CTAs."""
    calls = [np.array([1500, 1203]), np.ones(2, dtype=np.int64), np.array([4, 3]), np.array([1, 0])]
    _run_calls(23, 2, 2, 4, 16, 2048, torch.float32, calls)


def test_incremental_equals_full_on_gpu():
    """S = 37, T = 5: the chunked output and the full-sequence output both
    match the oracle's full-sequence causal output (whose last T rows the
    oracle's own incremental call reproduces exactly)."""
    _cuda_or_skip()
    S, T, d, Hkv, G = 37, 5, 128, 2, 4
    k = _store(wl.normal(3, 1, (1, Hkv, S, d)), torch.bfloat16)
    v = _store(wl.normal(3, 2, (1, Hkv, S, d)), torch.bfloat16)
    q = _store(wl.normal(3, 3, (1, Hkv * G, S, d)), torch.bfloat16)
    orc = ref.OracleCache(1, 1, Hkv, 64, d)
    want = ref.append_attention(orc, 0, q.double().numpy(), k.double().numpy(), v.double().numpy(), [S])
    k, v, q = k.cuda(), v.cuda(), q.cuda()
    full = KVCache(1, 1, Hkv, 64, d).append_attention(0, q, k, v, [S])
    inc_cache = KVCache(1, 1, Hkv, 64, d)
    inc_cache.append(0, k[:, :, : S - T].contiguous(), v[:, :, : S - T].contiguous(), [S - T])
    inc = inc_cache.append_attention(0, q[:, :, S - T :].contiguous(), k[:, :, S - T :].contiguous(),
                                     v[:, :, S - T :].contiguous(), [T])
    assert float(np.max(np.abs(full.double().cpu().numpy() - want))) <= 2e-2
    assert float(np.max(np.abs(inc.double().cpu().numpy() - want[:, :, S - T :]))) <= 2e-2


# ---------------------------------------------------------------------------
# Errors leave everything unchanged; canaries around every buffer
# ---------------------------------------------------------------------------


def test_overflow_on_gpu_changes_nothing():
    _cuda_or_skip()
    c = KVCache(1, 2, 2, 10, 128)
    k = _store(wl.normal(1, 1, (2, 2, 8, 128)), torch.bfloat16).cuda()
    c.append(0, k, k, [8, 3])
    before = c.k[0].clone()
    with pytest.raises(KVCError) as e:
        c.append(0, k, k, [1, 8])
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert torch.equal(c.k[0], before)
    assert list(c.lens(0)) == [8, 3]


def test_guard_regions_untouched():
    _cuda_or_skip()
    B, Hkv, G, d, max_len, T = 3, 2, 4, 128, 96, 9
    pad = 4096
    n_cache = B * Hkv * max_len * d
    n_q = B * Hkv * G * T * d
    sentinel = 1232.0  # exactly representable in bf16
    bufs = {name: torch.full((n + 2 * pad,), sentinel, dtype=torch.bfloat16, device="cuda")
            for name, n in (("k", n_cache), ("v", n_cache), ("out", n_q))}
    view = lambda name, n, shape: bufs[name][pad : pad + n].view(shape)
    k_buf = view("k", n_cache, (B, Hkv, max_len, d))
    v_buf = view("v", n_cache, (B, Hkv, max_len, d))
    out = view("out", n_q, (B, Hkv * G, T, d))
    c = KVCache(1, B, Hkv, max_len, d, k_bufs=[k_buf], v_bufs=[v_buf])
    for step, n in enumerate([[9, 4, 0], [9, 9, 9], [1, 2, 3]] * 3):
        q = _store(wl.normal(2, step, (B, Hkv * G, T, d)), torch.bfloat16).cuda()
        kn = _store(wl.normal(3, step, (B, Hkv, T, d)), torch.bfloat16).cuda()
        c.append_attention(0, q, kn, kn, n, out=out)
    torch.cuda.synchronize()
    for name, t in bufs.items():
        assert bool((t[:pad] == sentinel).all()) and bool((t[-pad:] == sentinel).all()), name


# ---------------------------------------------------------------------------
# Failure detection without a fault: the bounded wait expires and reports
# ---------------------------------------------------------------------------


def test_bounded_wait_reports_timeout():
    _cuda_or_skip()
    c = KVCache(1, 2, 2, 64, 128)
    ws = c.workspace(8, 1)
    assert c.device_status(ws) == 0
    c.selftest_bounded_wait(10_000_000, ws)  # 10 ms
    with pytest.raises(KVCError) as e:
        c.device_status(ws)
    assert e.value.status == 6
    assert c.device_status(ws) == 0  # the word was cleared
    # the context is still usable afterwards
    k = _store(wl.normal(1, 1, (2, 2, 3, 128)), torch.bfloat16).cuda()
    q = _store(wl.normal(1, 2, (2, 8, 3, 128)), torch.bfloat16).cuda()
    out = c.append_attention(0, q, k, k, [3, 2])
    assert bool(torch.isfinite(out.float()).all())


# ---------------------------------------------------------------------------
# Full-size workloads: sampled outputs against the oracle, one by one
# ---------------------------------------------------------------------------


def _seq_rows(seed, stream, B, H, max_len, d, b, h, lo, hi):
    """Generator rows [lo, hi) of unit (b, h) of a [B, H, max_len, d] sequence tensor, float64 on CPU."""
    base = ((b * H + h) * max_len + lo) * d
    idx = torch.arange(base, base + (hi - lo) * d, dtype=torch.int64)
    return wl.to_storage(wl.normal_at(seed, stream, idx), torch.bfloat16).double().reshape(hi - lo, d).numpy()


def _fill_poisoned(cache, layer, seed, lens):
    """Cache content from the generator; every slot at or past lens[b] set to NaN."""
    wl.fill_normal_(cache.k[layer], seed, wl.STREAM_CACHE_K)
    wl.fill_normal_(cache.v[layer], seed, wl.STREAM_CACHE_V)
    for b, L in enumerate(lens):
        cache.k[layer][b, :, int(L):] = float("nan")
        cache.v[layer][b, :, int(L):] = float("nan")
    cache.set_lens(layer, lens)


def _new_tokens(seed, step, B, Hkv, T, d):
    """Appended K/V of one step, generated on the CPU (the oracle regenerates the same values)."""
    k = _store(wl.normal(seed, 1000 + 2 * step, (B, Hkv, T, d)), torch.bfloat16)
    v = _store(wl.normal(seed, 1001 + 2 * step, (B, Hkv, T, d)), torch.bfloat16)
    return k, v


def _queries(seed, step, B, Hq, T, d):
    return _store(wl.normal(seed, 5000 + step, (B, Hq, T, d)), torch.bfloat16)


def _check_units(seed, shape, lens0, steps, q_last, n_last, out_last, units, T_last, Hq):
    """Oracle check of every query row of the sampled (b, kvh) units after the last step.

    The row's keys are the generator's cache content for positions < lens0[b]
    and the appended tokens after that (step s wrote position lens0[b] + ...).
    """
    d, Hkv, G = shape.d, shape.Hkv, Hq // shape.Hkv
    worst = 0.0
    q_np = q_last.double().numpy()
    got = out_last.double().cpu().numpy()
    for b, kvh in units:
        L0 = int(lens0[b])
        K = [_seq_rows(seed, wl.STREAM_CACHE_K, shape.B, Hkv, shape.max_len, d, b, kvh, 0, L0)]
        V = [_seq_rows(seed, wl.STREAM_CACHE_V, shape.B, Hkv, shape.max_len, d, b, kvh, 0, L0)]
        for step, (nn, T) in enumerate(steps):
            kn, vn = _new_tokens(seed, step, shape.B, Hkv, T, d)
            K.append(kn[b, kvh, : nn[b]].double().cpu().numpy())
            V.append(vn[b, kvh, : nn[b]].double().cpu().numpy())
        K = np.concatenate(K)
        V = np.concatenate(V)
        L = K.shape[0]
        for g in range(G):
            h = kvh * G + g
            for t in range(T_last):
                if t >= n_last[b]:
                    assert np.all(got[b, h, t] == 0.0)
                    continue
                pos = ref.query_position(L, int(n_last[b]), t)
                want = ref.attend_one_query(q_np[b, h, t], K, V, pos)
                worst = max(worst, float(np.max(np.abs(got[b, h, t] - want))))
    assert worst <= 2e-2, worst
    return worst


def _decode_case(shape, Hq, lens0, steps_T, n_steps_list, seed, units):
    _cuda_or_skip()
    cache = KVCache(1, shape.B, shape.Hkv, shape.max_len, shape.d)
    _fill_poisoned(cache, 0, seed, lens0)
    steps = []
    out = q = None
    for step, nn in enumerate(n_steps_list):
        T = int(steps_T[step])
        kn, vn = _new_tokens(seed, step, shape.B, shape.Hkv, T, shape.d)
        q = _queries(seed, step, shape.B, Hq, T, shape.d)
        out = cache.append_attention(0, q.cuda(), kn.cuda(), vn.cuda(), nn)
        steps.append((nn, T))
    torch.cuda.synchronize()
    assert np.array_equal(cache.lens(0), lens0 + sum(np.asarray(n) for n, _ in steps))
    assert bool(torch.isfinite(out.float()).all())
    assert cache.device_status() == 0
    return _check_units(seed, shape, lens0, steps, q, np.asarray(n_steps_list[-1]), out, units, int(steps_T[-1]), Hq)


def test_decode_llama8b_shape_every_unit():
    """The Llama-3.1-8B-shaped decode at full size (cache [32, 8, 8192, 128]):
    three steps, then every (row, KV head) unit of the last step, all 1,024
    query rows, against the oracle."""
    s = wl.DECODE_8B
    lens0 = wl.decode_lens(0, s.B, 1024, s.max_len - 256)
    n_steps = [np.ones(s.B, dtype=np.int64)] * 3
    units = [(b, h) for b in range(s.B) for h in range(s.Hkv)]
    _decode_case(s, s.Hq, lens0, [1, 1, 1], n_steps, 0, units)


def test_decode_many_short_split_units():
    """9,216 (row, KV head) units (1,024 rows x 9 KV heads) of 2 to 3 key tiles
    each: nearly every unit is split between warps and left to the combine
    kernel.  Two decode steps; 200 sampled units against the oracle, every
    output finite."""
    s = wl.Shape("many_units_decode", B=1024, Hq=9, Hkv=9, d=128, max_len=160, dtype="bf16")
    lens0 = wl.decode_lens(9, s.B, 70, 150)
    rng = np.random.default_rng(9)
    units = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, s.B, 200), rng.integers(0, s.Hkv, 200))})
    _decode_case(s, s.Hq, lens0, [1, 1], [np.ones(s.B, dtype=np.int64)] * 2, 9, units)


@pytest.mark.parametrize("T", [4, 8])
@pytest.mark.parametrize("Hq", [8, 16, 32, 64])
def test_verify_sampled_and_rollback(T, Hq):
    s = wl.VERIFY
    _cuda_or_skip()
    lens0 = np.full(s.B, s.max_len - T, dtype=np.int64)
    nn = np.full(s.B, T, dtype=np.int64)
    units = [(0, 0), (37, 5), (63, 7)]
    _decode_case(s, Hq, lens0, [T], [nn], 2, units)


def test_verify_truncate_loop():
    """Append T -> attend -> truncate back, repeatedly: lengths and outputs stay consistent."""
    _cuda_or_skip()
    s = wl.VERIFY
    B, T = 8, 4
    cache = KVCache(1, B, s.Hkv, s.max_len, s.d)
    lens0 = np.full(B, s.max_len - T, dtype=np.int64)
    _fill_poisoned(cache, 0, 4, lens0)
    outs = []
    for rep in range(3):
        kn, vn = _new_tokens(4, 0, B, s.Hkv, T, s.d)
        q = _queries(4, 0, B, s.Hq, T, s.d)
        outs.append(cache.append_attention(0, q.cuda(), kn.cuda(), vn.cuda(), np.full(B, T)))
        assert list(cache.length()) == [s.max_len] * B
        cache.truncate(lens0)
        assert list(cache.length()) == list(lens0)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


@pytest.mark.parametrize("B,Hq,T,prior", [
    (4, 32, 512, None),   # the chunked-prefill shape: 128-position tiles, cut blocks
    (4, 64, 40, 12000),   # packed rows in tile pairs, long rows cut across CTAs
    (8, 32, 4, 4092),     # one packed tile per (row, KV head): verify-sized, cut
])
def test_prefill_repeated_calls_identical(B, Hq, T, prior):
    """The same call four times (append, attend, truncate back) gives the same
    bits: pieces of a cut block are combined in a fixed order whichever of
    them finishes last, and nothing else in the launch depends on timing."""
    _cuda_or_skip()
    Hkv, d = 8, 128
    lens0 = wl.prefill_priors(3, B) if prior is None else np.full(B, prior, dtype=np.int64)
    max_len = int(lens0.max()) + T + 8
    cache = KVCache(1, B, Hkv, max_len, d)
    _fill_poisoned(cache, 0, 9, lens0)
    kn, vn = (x.cuda() for x in _new_tokens(9, 0, B, Hkv, T, d))
    q = _queries(9, 0, B, Hq, T, d).cuda()
    outs = []
    for _ in range(4):
        outs.append(cache.append_attention(0, q, kn, vn, np.full(B, T)))
        cache.truncate(lens0)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("ragged", [False, True])
def test_prefill_chunk_every_unit_of_a_row(ragged):
    """The chunked-prefill shape at full size: every KV head of the row with
    the longest prior (all 32 query heads x 512 queries), plus one unit of the
    shortest, against the oracle."""
    s = wl.PREFILL
    priors = wl.prefill_priors(0, s.B)
    T = 512
    nn = wl.ragged_chunk(0, s.B) if ragged else np.full(s.B, T, dtype=np.int64)
    units = [(int(np.argmax(priors)), h) for h in range(s.Hkv)] + [(int(np.argmin(priors)), 0)]
    _decode_case(s, s.Hq, priors, [T], [nn], 3, units)


@pytest.mark.parametrize("G,tails", [(4, [1, 31, 32, 33]), (8, [64, 65, 96, 97]), (3, [127, 40, 5, 100])])
def test_prefill_ragged_tails(G, tails):
    """Chunks of T >= 128 whose rows end in a partial 128-position block, with
    tails around every 32-row boundary and head counts that leave a head pair
    with one head; every output of both calls is compared with the oracle (the
    first call's rows end in tails of 116, 20 and 80 positions)."""
    B, Hkv = 4, 2
    priors = np.array([500, 1300, 0, 2000])
    chunk = np.array([128 + t for t in tails])
    _run_calls(17, B, Hkv, G, 128, 2000 + 300, torch.bfloat16, [priors, chunk])


def test_prefill_ragged_tail_cut_and_merged():
    """A long row with a partial last block on few items: the schedule cuts
    the items, the tail block's among them, and their pieces are merged in the
    launch; every output against the oracle."""
    _run_calls(23, 1, 4, 4, 128, 6300, torch.bfloat16, [np.array([6000]), np.array([200])])


@pytest.mark.parametrize("B,Hkv,G,prior,T", [(1, 2, 4, 3000, 256), (2, 1, 2, 700, 200), (1, 1, 3, 2500, 130)])
def test_prefill_few_long_items(B, Hkv, G, prior, T):
    """Few long prefill items on many SMs, every output compared (odd G also
    leaves a head pair with one head)."""
    calls = [np.full(B, prior), np.full(B, T)]
    _run_calls(13, B, Hkv, G, 128, prior + T + 5, torch.bfloat16, calls)


def _prefill_cuts(priors, n_new, Hkv, G, T, nsm, start_cost=5, min_piece=8):
    """Cuts made by the library's prefill schedule (a longest-first list
    schedule on the SMs, items cut at the SMs' common finish); restated here
    only to show that a test case exercises the in-kernel merge."""
    import heapq
    items = []
    for b, (pr, nn) in enumerate(zip(priors, n_new)):
        for _ in range(Hkv):
            for t0 in range(0, T, 128):
                if t0 >= nn:
                    continue
                nkt = (int(pr) + min(t0 + 127, int(nn) - 1)) // 128 + 1
                for pair in range((G + 1) // 2):
                    items.append((nkt, min(2, G - 2 * pair)))
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


@pytest.mark.parametrize("Hq,T", [(32, 512), (24, 256)])
def test_prefill_cut_blocks_merged_in_kernel(Hq, T):
    """Long blocks on one row: the schedule cuts most blocks into key-range
    pieces, whose partials the last piece merges inside the launch; sampled
    (b, kvh) units are compared query by query (G = 3 adds one-head pieces)."""
    _cuda_or_skip()
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    prior = 12000
    s = wl.Shape("one_row_long_prefill", B=1, Hq=Hq, Hkv=8, d=128, max_len=prior + T + 8, dtype="bf16")
    nn = np.full(1, T, dtype=np.int64)
    assert _prefill_cuts([prior], nn, s.Hkv, Hq // s.Hkv, T, nsm) > 0
    _decode_case(s, Hq, np.array([prior]), [T], [nn], 21, [(0, 0), (0, 7)])


def test_longctx_layer_sampled():
    """One layer of the long-context shape ([4, 8, 131072, 128] bf16, lengths
    in [32768, 131008]): two decode steps, sampled units against the oracle."""
    s = wl.LONGCTX
    lens0 = wl.decode_lens(0, s.B, 32768, s.max_len - 64)
    units = [(int(np.argmax(lens0)), 3), (int(np.argmin(lens0)), 6), (1, 0)]
    _decode_case(s, s.Hq, lens0, [1, 1], [np.ones(s.B, dtype=np.int64)] * 2, 5, units)


@pytest.mark.parametrize("T,G,d", [(1, 4, 128), (4, 2, 128), (1, 4, 64)])
def test_decode_score_jumps(T, G, d):
    """Decode and short verify on the split-KV kernel with scores that jump by
    tens to hundreds (log2 units) at keys spread over a 3,000-key row: the
    running maximum moves inside a warp's tiles, and the combine merges
    partials whose maxima differ by that much (each unit is cut across CTAs
    and warps); every output against the oracle."""
    _cuda_or_skip()
    B, Hkv, prior = 2, 2, 3000
    max_len = prior + T + 8
    rng = np.random.default_rng(13)
    u = np.ones(d)
    k0 = rng.standard_normal((B, Hkv, prior, d))
    for pos, alpha in ((300, 0.5), (1100, 1.5), (1900, 4.0), (2950, 4.0)):
        k0[:, :, pos] = alpha * u + 0.1 * rng.standard_normal(d)
    v0 = rng.standard_normal((B, Hkv, prior, d))
    kn = rng.standard_normal((B, Hkv, T, d))
    vn = rng.standard_normal((B, Hkv, T, d))
    q = rng.standard_normal((B, Hkv * G, T, d)) + 3.0 * u
    k0s, v0s, kns, vns, qs = (_store(torch.from_numpy(x), torch.bfloat16) for x in (k0, v0, kn, vn, q))
    cache = KVCache(1, B, Hkv, max_len, d)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    cache.append(0, k0s.cuda(), v0s.cuda(), [prior] * B)
    out = cache.append_attention(0, qs.cuda(), kns.cuda(), vns.cuda(), [T] * B)
    orc = ref.OracleCache(1, B, Hkv, max_len, d)
    ref.append_attention(orc, 0, np.zeros((B, Hkv * G, prior, d)), k0s.double().numpy(), v0s.double().numpy(),
                         [prior] * B)
    want = ref.append_attention(orc, 0, qs.double().numpy(), kns.double().numpy(), vns.double().numpy(), [T] * B)
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - want)))
    assert err <= 2e-2, err
    assert cache.device_status() == 0


@pytest.mark.parametrize("T", [256, 200])
def test_prefill_score_jumps(T):
    """Scores that jump by about 25, 75 and 200 (log2 units) at keys further into
    the row: the running maximum moves at the next tile (jumps above 8) or
    inside the tile (jumps above 64, in either 64-key half), and the result
    still matches the oracle."""
    _cuda_or_skip()
    B, Hkv, G, d, prior = 1, 2, 2, 128, 1300
    max_len = prior + T + 8
    rng = np.random.default_rng(11)
    u = np.ones(d)
    k0 = rng.standard_normal((B, Hkv, prior, d))
    for pos, alpha in ((300, 0.5), (700, 1.5), (868, 4.0), (1190, 4.0)):
        k0[:, :, pos] = alpha * u + 0.1 * rng.standard_normal(d)
    v0 = rng.standard_normal((B, Hkv, prior, d))
    kn = rng.standard_normal((B, Hkv, T, d))
    vn = rng.standard_normal((B, Hkv, T, d))
    q = rng.standard_normal((B, Hkv * G, T, d)) + 3.0 * u
    store = [_store(torch.from_numpy(x), torch.bfloat16) for x in (k0, v0, kn, vn, q)]
    k0s, v0s, kns, vns, qs = store
    cache = KVCache(1, B, Hkv, max_len, d)
    cache.k[0].fill_(float("nan"))
    cache.v[0].fill_(float("nan"))
    cache.append(0, k0s.cuda(), v0s.cuda(), [prior])
    out = cache.append_attention(0, qs.cuda(), kns.cuda(), vns.cuda(), [T])
    orc = ref.OracleCache(1, B, Hkv, max_len, d)
    ref.append_attention(orc, 0, np.zeros((B, Hkv * G, prior, d)), k0s.double().numpy(), v0s.double().numpy(), [prior])
    want = ref.append_attention(orc, 0, qs.double().numpy(), kns.double().numpy(), vns.double().numpy(), [T])
    got = out.double().cpu().numpy()
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got - want)))
    assert err <= 2e-2, err
    assert cache.device_status() == 0
