"""The allocation-free attention entry point against the workspace one.

kvc_gqa_attention_noalloc exists for callers that cannot allocate device
memory (a host program that owns the whole device-memory budget, or a loop
that cannot pay for cudaMalloc): its split-KV scratch is a static device
array inside the library instead of a caller-provided workspace.  Here it is
called through the C ABI on two calls in a row (different shapes, so the
scratch is reused with a different layout) and must give the existing
entry point's output within the bf16 tolerance of the parity tests.  This
file is collected last on purpose; it passes alone or after the others.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import KVCache, KVCError, PagedKVCache, _lib
from gqa_attention_preallocated_gb300 import workloads as wl
from gqa_attention_preallocated_gb300.build import build_library

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
I32P = ctypes.POINTER(ctypes.c_int32)


def _bf16(seed, stream, shape):
    return wl.to_storage(wl.normal(seed, stream, shape), torch.bfloat16).cuda()


def _noalloc(cache, q, n_new, out):
    nn = np.ascontiguousarray(np.asarray(n_new, dtype=np.int32))
    st = _lib.lib().kvc_gqa_attention_noalloc(cache._h, 0, q.data_ptr(), q.shape[1], q.shape[2],
                                              nn.ctypes.data_as(I32P), out.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
    return st


def _status():
    code = ctypes.c_int32(0)
    st = _lib.lib().kvc_noalloc_status(torch.cuda.current_stream().cuda_stream, ctypes.byref(code))
    return st, code.value


def test_noalloc_matches_workspace_entry_point_twice():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build_library()
    B, Hkv, G, d, max_len = 8, 4, 4, 128, 2048
    cache = KVCache(1, B, Hkv, max_len, d)
    orc = ref.OracleCache(1, B, Hkv, max_len, d)
    rng = np.random.default_rng(5)
    prefill = rng.integers(600, 1500, size=B)
    T0 = int(prefill.max())
    k0, v0 = _bf16(1, 1, (B, Hkv, T0, d)), _bf16(1, 2, (B, Hkv, T0, d))
    cache.append(0, k0, v0, prefill)
    orc.append(0, k0.double().cpu().numpy(), v0.double().cpu().numpy(), prefill)
    for call, T in enumerate([1, 4]):  # decode, then speculative verify
        n_new = np.full(B, T)
        k, v = _bf16(2, 10 + call, (B, Hkv, T, d)), _bf16(2, 20 + call, (B, Hkv, T, d))
        cache.append(0, k, v, n_new)
        orc.append(0, k.double().cpu().numpy(), v.double().cpu().numpy(), n_new)
        q = _bf16(3, 30 + call, (B, Hkv * G, T, d))
        ref_out = cache.gqa_attention(0, q, n_new)
        out = torch.full_like(q, float("nan"))
        assert _noalloc(cache, q, n_new, out) == 0, _lib.lib().kvc_last_error()
        torch.cuda.synchronize()
        assert bool(torch.isfinite(out.float()).all())
        err = float((out.float() - ref_out.float()).abs().max())
        assert err <= TOL_BF16, (call, err)
        # and against the float64 oracle on the stored values
        want = ref.gqa_attention(q.double().cpu().numpy(), orc, 0, n_new)
        assert float(np.max(np.abs(out.double().cpu().numpy() - want))) <= TOL_BF16, call
    assert _status() == (0, 0)


@pytest.mark.parametrize("T", [1, 256])
def test_noalloc_reports_a_bad_block_table_entry(T):
    """A paged cache whose block table holds -1 under attended keys: the
    kernels never dereference it and record it in the static scratch's error
    word, which kvc_noalloc_status then reports (KVC_ERR_ARG, code 7) and
    clears; a following clean call reports nothing."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build_library()
    B, Hkv, G, d, page, mpr = 2, 2, 4, 128, 128, 8
    cache = PagedKVCache(1, B, Hkv, page, B * mpr, mpr, d)
    cache.k[0].zero_()
    cache.v[0].zero_()
    cache.set_lens(0, [5 * page, 3 * page])
    good = int(cache.block_table[0, 2])
    cache.block_table[0, 2] = -1  # under row 0's attended keys
    q = torch.zeros((B, Hkv * G, T, d), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    assert _noalloc(cache, q, np.full(B, T), out) == 0, _lib.lib().kvc_last_error()
    assert _status() == (1, 7)  # KVC_ERR_ARG: a block-table entry outside 0 .. num_pages - 1
    assert _status() == (0, 0)  # read once, then cleared
    with pytest.raises(KVCError):  # the Python wrapper allocates nothing: out is required
        cache.gqa_attention_noalloc(0, q, np.full(B, T))
    cache.block_table[0, 2] = good
    cache.gqa_attention_noalloc(0, q, np.full(B, T), out=out)
    assert cache.noalloc_status() == 0


def test_noalloc_long_chunk_runs_in_the_static_scratch():
    """A long prefill chunk (the tensor-core path needs only the workspace
    header) runs through the static scratch and matches the workspace entry
    point, although its full workspace is larger than the scratch."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build_library()
    B, Hkv, G, d, T = 4, 8, 4, 128, 512
    cache = KVCache(1, B, Hkv, 1024, d)
    cache.append(0, _bf16(1, 1, (B, Hkv, T, d)), _bf16(1, 2, (B, Hkv, T, d)), np.full(B, T))
    assert cache.workspace_bytes(Hkv * G, T) > (32 << 20)
    q = _bf16(3, 3, (B, Hkv * G, T, d))
    ref_out = cache.gqa_attention(0, q, np.full(B, T))
    out = torch.full_like(q, float("nan"))
    assert _noalloc(cache, q, np.full(B, T), out) == 0, _lib.lib().kvc_last_error()
    torch.cuda.synchronize()
    assert float((out.float() - ref_out.float()).abs().max()) <= TOL_BF16


def test_noalloc_rejects_oversized_calls():
    """A decode call on a very large batch needs more split-KV scratch than the
    static array holds: refused before anything is enqueued."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build_library()
    B, Hkv, G, d, T = 512, 8, 8, 128, 1  # 8 rows per KV head: the split-KV kernel
    cache = KVCache(1, B, Hkv, 16, d)
    cache.set_lens(0, np.full(B, 8))
    assert cache.workspace_bytes(Hkv * G, T) > (32 << 20)
    q = _bf16(3, 3, (B, Hkv * G, T, d))
    out = torch.zeros_like(q)
    assert _noalloc(cache, q, np.full(B, T), out) == 7  # KVC_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert bool((out == 0).all())


def test_noalloc_fp8_cache():
    """An FP8 E4M3 cache through the static scratch: decode on the split-KV kernel and a 64-row verify on
    the tensor-core kernel, each equal to the workspace entry point (same kernel, same bits)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    build_library()
    B, Hkv, d, max_len = 8, 4, 128, 2048
    cache = KVCache(1, B, Hkv, max_len, d, dtype=torch.float8_e4m3fn)
    sc = np.full(Hkv, 4.0 / 448, dtype=np.float32)
    cache.set_kv_scales(0, sc, sc)
    prefill = np.random.default_rng(6).integers(600, 1500, size=B)
    T0 = int(prefill.max())
    cache.append(0, _bf16(4, 1, (B, Hkv, T0, d)), _bf16(4, 2, (B, Hkv, T0, d)), prefill)
    for call, (T, G) in enumerate([(1, 4), (8, 8)]):
        n_new = np.full(B, T)
        cache.append(0, _bf16(5, 10 + call, (B, Hkv, T, d)), _bf16(5, 20 + call, (B, Hkv, T, d)), n_new)
        q = _bf16(6, 30 + call, (B, Hkv * G, T, d))
        ref_out = cache.gqa_attention(0, q, n_new)
        out = torch.full_like(q, float("nan"))
        assert _noalloc(cache, q, n_new, out) == 0, _lib.lib().kvc_last_error()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), call
