"""CPU tests of the C ABI: the library loads, exports what include/kvc.h
declares, and its host logic (validation, lengths, truncate, layer
agreement) behaves as the pages state.  No compute call runs here: the
buffer pointers are fake, and every call tested either fails validation
before any CUDA call or is host-only.
"""

import ctypes
import os
import re

import numpy as np
import pytest

from gqa_attention_preallocated_gb300 import _lib
from gqa_attention_preallocated_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
I32P = ctypes.POINTER(ctypes.c_int32)
I64P = ctypes.POINTER(ctypes.c_int64)


@pytest.fixture(scope="module")
def L():
    build_library()
    return _lib.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "kvc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvc_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    declared = _declared()
    assert "kvc_create" in declared and "kvc_gqa_attention" in declared
    for name in declared:
        assert hasattr(L, name), name
    bound = {n for n, _, _ in _lib.SIGNATURES}
    assert set(declared) == bound  # the binding covers exactly the header


def _fake_buffers(layers):
    # 16-byte aligned fake device addresses; never dereferenced by these tests
    base = 1 << 40
    k = (ctypes.c_void_p * layers)(*[base + (2 * i) * (1 << 30) for i in range(layers)])
    v = (ctypes.c_void_p * layers)(*[base + (2 * i + 1) * (1 << 30) for i in range(layers)])
    return k, v


def _create(L, layers=2, B=3, Hkv=2, max_len=16, d=16, dtype=_lib.KVC_F32):
    h = ctypes.c_void_p()
    k, v = _fake_buffers(layers)
    st = L.kvc_create(ctypes.byref(h), layers, B, Hkv, max_len, d, dtype, k, v)
    return st, h


def _i32(*xs):
    a = np.array(xs, dtype=np.int32)
    return a, a.ctypes.data_as(I32P)


def _i64(*xs):
    a = np.array(xs, dtype=np.int64)
    return a, a.ctypes.data_as(I64P)


def _lens(L, h, layer, B):
    out = np.zeros(B, dtype=np.int64)
    assert L.kvc_get_lens(h, layer, out.ctypes.data_as(I64P)) == 0
    return out


def test_create_validation(L):
    h = ctypes.c_void_p()
    k, v = _fake_buffers(1)
    assert L.kvc_create(ctypes.byref(h), 0, 2, 2, 8, 16, 0, k, v) == 1
    assert L.kvc_create(ctypes.byref(h), 1, 2, 2, 8, 6, 0, k, v) == 1  # 6 * 4 B not a multiple of 16
    assert L.kvc_create(ctypes.byref(h), 1, 2, 2, 8, 12, 1, k, v) == 1  # 12 * 2 B not a multiple of 16
    assert L.kvc_create(ctypes.byref(h), 1, 2, 2, 8, 264, 1, k, v) == 1  # d <= 256
    assert L.kvc_create(ctypes.byref(h), 1, 2, 2, 8, 260, 0, k, v) == 1  # fp32 too
    assert L.kvc_create(ctypes.byref(h), 1, 2, 2, 8, 272, 2, k, v) == 1  # and FP8
    for dt, d in ((0, 256), (1, 256), (2, 256), (1, 72), (2, 48)):      # the largest, and other sizes
        assert L.kvc_create(ctypes.byref(h), 1, 2, 2, 8, d, dt, k, v) == 0, (dt, d)
        L.kvc_destroy(h)
    assert L.kvc_create(ctypes.byref(h), 1, _lib.KVC_MAX_BATCH + 1, 2, 8, 16, 0, k, v) == 1
    bad = (ctypes.c_void_p * 1)(12345)  # misaligned
    assert L.kvc_create(ctypes.byref(h), 1, 2, 2, 8, 16, 0, bad, v) == 1
    assert b"aligned" in L.kvc_last_error()
    st, h = _create(L)
    assert st == 0
    L.kvc_destroy(h)
    L.kvc_destroy(None)


def test_append_validation_leaves_state(L):
    st, h = _create(L, layers=1, B=3, max_len=10)
    assert st == 0
    _, full = _i64(8, 2, 10)
    assert L.kvc_set_lens(h, 0, full) == 0
    kn = ctypes.c_void_p(1 << 41)
    # overflow in the last row: nothing changes, including the earlier rows
    a, p = _i32(1, 1, 1)
    assert L.kvc_append(h, 0, kn, kn, 3, p, None) == 3
    assert b"max_len" in L.kvc_last_error()
    assert list(_lens(L, h, 0, 3)) == [8, 2, 10]
    # n_new outside 0..T
    a, p = _i32(4, 0, 0)
    assert L.kvc_append(h, 0, kn, kn, 3, p, None) == 2
    a, p = _i32(-1, 0, 0)
    assert L.kvc_append(h, 0, kn, kn, 3, p, None) == 2
    # bad layer, T < 0, misaligned inputs
    a, p = _i32(0, 0, 0)
    assert L.kvc_append(h, 1, kn, kn, 3, p, None) == 1
    assert L.kvc_append(h, 0, kn, kn, -1, p, None) == 1
    a, p = _i32(1, 0, 0)
    assert L.kvc_append(h, 0, ctypes.c_void_p((1 << 41) + 4), kn, 3, p, None) == 1
    # all-zero n_new is a no-op that needs no GPU
    a, p = _i32(0, 0, 0)
    assert L.kvc_append(h, 0, None, None, 3, p, None) == 0
    assert list(_lens(L, h, 0, 3)) == [8, 2, 10]
    L.kvc_destroy(h)


def test_attention_validation(L):
    st, h = _create(L, layers=1, B=2, Hkv=2, max_len=10, d=16)
    _, full = _i64(5, 0)
    assert L.kvc_set_lens(h, 0, full) == 0
    q = ctypes.c_void_p(1 << 42)
    a, p = _i32(1, 0)
    assert L.kvc_gqa_attention(h, 0, q, 3, 1, p, q, None, 0, None) == 2  # Hq % Hkv != 0
    a, p = _i32(2, 0)
    assert L.kvc_gqa_attention(h, 0, q, 4, 1, p, q, None, 0, None) == 2  # n_new > T
    a, p = _i32(0, 1)
    assert L.kvc_gqa_attention(h, 0, q, 4, 1, p, q, None, 0, None) == 2  # n_new > lens (row 1 empty)
    a, p = _i32(1, 0)
    assert L.kvc_gqa_attention(h, 0, None, 4, 1, p, q, None, 0, None) == 1  # null q
    # T = 0 and an empty batch are valid no-ops
    a, p = _i32(0, 0)
    assert L.kvc_gqa_attention(h, 0, None, 4, 0, p, None, None, 0, None) == 0
    L.kvc_destroy(h)
    st, h0 = _create(L, layers=1, B=0)
    assert st == 0
    assert L.kvc_gqa_attention(h0, 0, None, 4, 3, None, None, None, 0, None) == 0
    L.kvc_destroy(h0)


def test_append_attention_validates_both_steps_first(L):
    st, h = _create(L, layers=1, B=2, Hkv=2, max_len=10, d=16)
    kn = ctypes.c_void_p(1 << 41)
    a, p = _i32(1, 1)
    # the attention step is invalid (Hq = 3): the append must not happen
    assert L.kvc_append_attention(h, 0, kn, kn, kn, 3, 1, p, kn, None, 0, None) == 2
    assert list(_lens(L, h, 0, 2)) == [0, 0]
    L.kvc_destroy(h)


def test_host_buffer_call_validates_before_any_copy(L):
    # Every error of the host-buffer form is found before a copy is enqueued or
    # a host buffer read: the pointers here are fake, so a copy would crash.
    st, h = _create(L, layers=1, B=2, Hkv=2, max_len=10, d=16)
    x = ctypes.c_void_p(1 << 41)
    a, p = _i32(1, 1)
    assert L.kvc_append_attention_host(h, 0, x, x, x, 3, 1, p, x, None, 0, None) == 2  # Hq % Hkv != 0
    a, p = _i32(2, 0)
    assert L.kvc_append_attention_host(h, 0, x, x, x, 4, 1, p, x, None, 0, None) == 2  # n_new > T
    a, p = _i32(1, 1)
    assert L.kvc_append_attention_host(h, 0, None, x, x, 4, 1, p, x, None, 0, None) == 1  # null q
    assert L.kvc_append_attention_host(h, 0, x, x, x, 4, 1, p, None, None, 0, None) == 1  # null out
    assert L.kvc_append_attention_host(h, 0, x, None, x, 4, 1, p, x, None, 0, None) == 1  # null k_new
    odd = ctypes.c_void_p((1 << 41) + 8)
    assert L.kvc_append_attention_host(h, 0, odd, x, x, 4, 1, p, x, None, 0, None) == 1  # q not 16-byte aligned
    assert L.kvc_append_attention_host(h, 1, x, x, x, 4, 1, p, x, None, 0, None) == 1  # layer out of range
    _, full = _i64(9, 0)
    assert L.kvc_set_lens(h, 0, full) == 0
    a, p = _i32(2, 0)
    assert L.kvc_append_attention_host(h, 0, x, x, x, 4, 2, p, x, None, 0, None) == 3  # 9 + 2 > max_len
    assert list(_lens(L, h, 0, 2)) == [9, 0]
    # nothing to do: T = 0, or an empty batch
    a, p = _i32(0, 0)
    assert L.kvc_append_attention_host(h, 0, None, None, None, 4, 0, p, None, None, 0, None) == 0
    assert L.kvc_host_copies_done(h, None) == 0  # no host-buffer call has enqueued anything
    assert L.kvc_host_copies_done(None, None) == 1
    L.kvc_destroy(h)


def test_set_lens_truncate_reset_length(L):
    st, h = _create(L, layers=3, B=2, max_len=16)
    for layer in range(3):
        _, p = _i64(7, 3)
        assert L.kvc_set_lens(h, layer, p) == 0
    out = np.zeros(2, dtype=np.int64)
    assert L.kvc_length(h, out.ctypes.data_as(I64P)) == 0 and list(out) == [7, 3]
    _, p = _i64(17, 0)
    assert L.kvc_set_lens(h, 0, p) == 1  # past max_len
    # a forward pass that stopped part-way: layer 0 ahead of the others
    _, p = _i64(8, 4)
    assert L.kvc_set_lens(h, 0, p) == 0
    assert L.kvc_length(h, out.ctypes.data_as(I64P)) == 4
    assert b"part-way" in L.kvc_last_error()
    _, p = _i64(2, 2)
    assert L.kvc_truncate(h, p) == 4  # refuses while layers disagree
    _, p = _i64(7, 3)
    assert L.kvc_set_lens(h, 0, p) == 0
    _, p = _i64(8, 3)
    assert L.kvc_truncate(h, p) == 1  # cannot grow
    _, p = _i64(-1, 3)
    assert L.kvc_truncate(h, p) == 1
    _, p = _i64(5, 0)
    assert L.kvc_truncate(h, p) == 0
    for layer in range(3):
        assert list(_lens(L, h, layer, 2)) == [5, 0]
    assert L.kvc_reset(h) == 0
    assert L.kvc_length(h, out.ctypes.data_as(I64P)) == 0 and list(out) == [0, 0]
    assert L.kvc_get_lens(h, 3, out.ctypes.data_as(I64P)) == 1
    L.kvc_destroy(h)


def test_workspace_query_without_gpu_or_for_f32(L):
    st, h = _create(L, dtype=_lib.KVC_F32)
    assert L.kvc_workspace_bytes(h, 4, 1) == 0  # the f32 path needs no workspace
    L.kvc_destroy(h)
    assert L.kvc_workspace_bytes(None, 4, 1) == 0
    st, h = _create(L, d=96, dtype=_lib.KVC_BF16)  # bf16 of d other than 64 and 128: the generic kernel
    assert st == 0
    assert L.kvc_workspace_bytes(h, 4, 1) == 0
    _, n = _i32(3, 0)
    assert L.kvc_gqa_attention_noalloc(h, 0, None, 4, 1, n, None, None) == 1
    assert b"head_dim 128" in L.kvc_last_error()
    L.kvc_destroy(h)
    st, h = _create(L, d=64, dtype=_lib.KVC_BF16)  # bf16 of d = 64: the split-KV kernel (sizes need a device)
    assert st == 0
    L.kvc_destroy(h)


def test_device_lens_calls_without_device_state(L):
    st, h = _create(L, layers=2, B=3)
    assert L.kvc_device_lens_bytes(h) == 2 * 3 * 4
    assert L.kvc_lens_from_device(h, None) == 1  # the lengths are on the host
    q = ctypes.c_void_p(1 << 42)
    # a resident-length step before the lengths were handed over
    assert L.kvc_decode_step(h, 0, q, q, q, 4, 1, q, q, q, 1 << 20, None) == 1
    assert b"kvc_lens_to_device" in L.kvc_last_error()
    assert L.kvc_lens_to_device(h, None, None) == 1  # null array
    L.kvc_destroy(h)
    assert L.kvc_device_lens_bytes(None) == 0


def test_window_and_ring_host_rules(L):
    st, h = _create(L, layers=2, B=2, max_len=16, dtype=_lib.KVC_F32)
    assert L.kvc_set_window(h, -1, 0) == 1
    assert L.kvc_set_window(h, 0, 1) == 1    # a ring needs a window
    assert L.kvc_set_window(h, 17, 1) == 1   # window past max_len
    assert L.kvc_set_window(h, 5, 1) == 0
    kn = ctypes.c_void_p(1 << 41)
    _, p = _i32(13, 0)
    assert L.kvc_append(h, 0, kn, kn, 13, p, None) == 3  # 13 > 16 - 5 + 1
    _, big = _i64(40, 3)
    for layer in range(2):
        assert L.kvc_set_lens(h, layer, big) == 0       # a ring counts every position
    _, p = _i64(27, 3)
    assert L.kvc_truncate(h, p) == 1  # would need key 23; the ring holds 24..39
    _, p = _i64(28, 3)
    assert L.kvc_truncate(h, p) == 0  # needs keys 24..27
    assert L.kvc_set_window(h, 5, 0) == 1  # storage changes only on an empty cache
    assert L.kvc_reset(h) == 0
    assert L.kvc_set_window(h, 5, 0) == 0
    L.kvc_destroy(h)
    st, h = _create(L, layers=1, B=1, max_len=200, d=128, dtype=_lib.KVC_BF16)
    assert L.kvc_set_window(h, 50, 1) == 1  # bf16 ring: max_len % 128
    L.kvc_destroy(h)


def _create_paged(L, layers=1, B=2, Hkv=2, page=4, num_pages=5, mpr=3, d=16, dtype=_lib.KVC_F32, table=1 << 42):
    h = ctypes.c_void_p()
    k, v = _fake_buffers(layers)
    st = L.kvc_create_paged(ctypes.byref(h), layers, B, Hkv, page, num_pages, mpr, d, dtype, k, v,
                            ctypes.c_void_p(table))
    return st, h


def test_paged_host_rules(L):
    assert _create_paged(L, page=0)[0] == 1
    assert _create_paged(L, num_pages=0)[0] == 1
    assert _create_paged(L, mpr=0)[0] == 1
    assert _create_paged(L, table=0)[0] == 1          # no block table
    assert _create_paged(L, table=(1 << 42) + 2)[0] == 1  # misaligned table
    assert _create_paged(L, page=64, d=128, dtype=_lib.KVC_BF16)[0] == 1  # bf16 pages: multiples of 128
    st, h = _create_paged(L, page=16, d=96, dtype=_lib.KVC_BF16)  # off the TMA path any page size works
    assert st == 0
    L.kvc_destroy(h)
    assert _create_paged(L, page=16, d=64, dtype=_lib.KVC_BF16)[0] == 1  # d = 64: pages of multiples of 128
    assert _create_paged(L, page=64, d=64, dtype=_lib.KVC_BF16)[0] == 1
    st, h = _create_paged(L, page=128, d=64, dtype=_lib.KVC_BF16)
    assert st == 0
    L.kvc_destroy(h)
    st, h = _create_paged(L, page=128, d=128, dtype=_lib.KVC_BF16)
    assert st == 0
    L.kvc_destroy(h)
    st, h = _create_paged(L, B=2, page=4, mpr=3)
    assert st == 0
    _, big = _i64(12, 0)
    assert L.kvc_set_lens(h, 0, big) == 0   # logical max_len = 3 pages * 4
    _, over = _i64(13, 0)
    assert L.kvc_set_lens(h, 0, over) == 1
    kn = ctypes.c_void_p(1 << 41)
    _, p = _i32(1, 0)
    assert L.kvc_append(h, 0, kn, kn, 1, p, None) == 3  # row 0 is full
    assert L.kvc_set_window(h, 6, 1) == 1   # ring storage is not paged
    assert L.kvc_reset(h) == 0
    assert L.kvc_set_window(h, 6, 0) == 0   # a window over pages is fine
    L.kvc_destroy(h)


def test_fp8_host_rules(L):
    FP = ctypes.POINTER(ctypes.c_float)

    def scales(*xs):
        a = np.array(xs, dtype=np.float32)
        return a, a.ctypes.data_as(FP)

    assert _create(L, d=24, dtype=_lib.KVC_FP8_E4M3)[0] == 1      # 24 one-byte values: not a multiple of 16
    st, h = _create(L, d=64, dtype=_lib.KVC_FP8_E4M3)             # other head dims: the generic kernel
    assert st == 0
    L.kvc_destroy(h)
    assert _create(L, Hkv=65, d=128, dtype=_lib.KVC_FP8_E4M3)[0] == 1
    st, h = _create(L, layers=2, B=2, Hkv=2, max_len=256, d=128, dtype=_lib.KVC_FP8_E4M3)
    assert st == 0
    _, ok = scales(0.5, 2.0)
    assert L.kvc_set_kv_scales(h, 0, ok, ok) == 0
    assert L.kvc_set_kv_scales(h, 2, ok, ok) == 1                 # layer out of range
    for bad in [(0.0, 1.0), (-1.0, 1.0), (float("inf"), 1.0), (float("nan"), 1.0)]:
        _, b = scales(*bad)
        assert L.kvc_set_kv_scales(h, 0, b, ok) == 1
        assert L.kvc_set_kv_scales(h, 0, ok, b) == 1
    _, lens = _i64(3, 0)
    assert L.kvc_set_lens(h, 1, lens) == 0
    assert L.kvc_set_kv_scales(h, 1, ok, ok) == 1                 # layer 1 holds data
    assert L.kvc_set_kv_scales(h, 0, ok, ok) == 0                 # layer 0 is still empty
    assert L.kvc_reset(h) == 0
    assert L.kvc_set_kv_scales(h, 1, ok, ok) == 0
    L.kvc_destroy(h)
    st, h = _create(L, d=16)
    _, ok = scales(1.0, 1.0)
    assert L.kvc_set_kv_scales(h, 0, ok, ok) == 1                 # not an fp8 cache
    L.kvc_destroy(h)


def test_tree_validation_before_any_device_call(L):
    """A draft tree's parents, size and the window rule are checked on the
    host before anything touches a GPU (so these run without one)."""
    st, h = _create(L, layers=1, B=2, Hkv=1, max_len=80, d=16)
    assert st == 0
    _, lens = _i64(10, 10)
    assert L.kvc_set_lens(h, 0, lens) == 0
    q = ctypes.c_void_p(1 << 41)
    out = ctypes.c_void_p(1 << 42)
    _, nn = _i32(4, 4)
    bad, bad_p = _i32(-1, 0, 3, 1, -1, 0, 0, 0)          # row 0: token 2's parent comes after it
    assert L.kvc_gqa_attention_tree(h, 0, q, 1, 4, nn, bad_p, out, None, 0, None) == 2
    assert b"parent" in L.kvc_last_error()
    _, long_lens = _i64(70, 70)
    assert L.kvc_set_lens(h, 0, long_lens) == 0
    _, nn65 = _i32(65, 65)
    chain = np.concatenate([np.arange(-1, 64), np.arange(-1, 64)]).astype(np.int32)
    assert L.kvc_gqa_attention_tree(h, 0, q, 1, 65, nn65, chain.ctypes.data_as(I32P), out, None, 0, None) == 2
    assert b"64" in L.kvc_last_error()
    assert L.kvc_set_lens(h, 0, lens) == 0
    assert L.kvc_reset(h) == 0
    assert L.kvc_set_window(h, 5, 0) == 0
    assert L.kvc_set_lens(h, 0, lens) == 0
    ok, ok_p = _i32(-1, 0, 1, 2, -1, -1, -1, -1)
    assert L.kvc_gqa_attention_tree(h, 0, q, 1, 4, nn, ok_p, out, None, 0, None) == 1  # no window with a tree
    L.kvc_destroy(h)
