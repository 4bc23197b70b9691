"""Pins for the oracle's FP8 E4M3 storage ("16. Prefill, decode and the KV
cache", exercise 4: store the cache in FP8 E4M3 with one scale per head and
dequantize on read).

The format is tied to things other than the oracle's own formula: the
values the format's definition fixes by hand (1, 448, the smallest normal and
subnormal), PyTorch's float8_e4m3fn decoding of all 256 codes and its float32
-> e4m3 cast (a library routine) on in-range values, the round-to-nearest-even
rule at exact midpoints, the half-ulp error bound, and an FP8 cache whose
attention equals the ordinary cache fed the dequantized values.  Planted
mistakes (round half up, a scale left out on read) must fail.
"""

import math

import numpy as np
import pytest
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import workloads as wl


def test_hand_values_of_the_format():
    assert ref.e4m3_value(0x00) == 0.0
    assert ref.e4m3_value(0x01) == 2.0 ** -9          # smallest subnormal: 1/8 * 2^-6
    assert ref.e4m3_value(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert ref.e4m3_value(0x08) == 2.0 ** -6          # smallest normal
    assert ref.e4m3_value(0x38) == 1.0                # exponent field 7 = bias
    assert ref.e4m3_value(0x3C) == 1.5
    assert ref.e4m3_value(0x7E) == 448.0              # largest finite: 1.75 * 2^8
    assert math.isnan(ref.e4m3_value(0x7F)) and math.isnan(ref.e4m3_value(0xFF))
    assert ref.e4m3_value(0xB8) == -1.0
    finite = [ref.e4m3_value(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(finite, finite[1:]))  # codes 0..126 ascend


def test_decoding_matches_the_library_format():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([ref.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ours)
    assert np.array_equal(nan, np.isnan(lib))
    assert np.array_equal(ours[~nan], lib[~nan])


def test_every_finite_code_round_trips():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert ref.e4m3_encode(ref.e4m3_value(c)) == c, hex(c)


def test_midpoints_round_to_even():
    # 1.0625 lies halfway between 1.0 (mantissa 0) and 1.125 (mantissa 1): even is 1.0
    assert ref.e4m3_encode(1.0625) == 0x38
    # 1.1875 halfway between 1.125 (m = 1) and 1.25 (m = 2): even is 1.25
    assert ref.e4m3_encode(1.1875) == 0x3A
    assert ref.e4m3_encode(2.0 ** -10) == 0x00          # halfway between 0 and the smallest subnormal
    assert ref.e4m3_encode(3 * 2.0 ** -10) == 0x02      # halfway between m = 1 and m = 2 subnormals
    assert ref.e4m3_encode(1.0625 + 1e-9) == 0x39       # just above the midpoint
    assert ref.e4m3_encode(-1.1875) == 0xBA


def test_saturation_and_nan():
    assert ref.e4m3_encode(449.0) == 0x7E
    assert ref.e4m3_encode(1e9) == 0x7E
    assert ref.e4m3_encode(-1e9) == 0xFE
    assert ref.e4m3_encode(float("inf")) == 0x7E
    assert ref.e4m3_encode(float("nan")) == 0x7F


def test_encoder_matches_the_library_cast_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(50000) * 40, rng.standard_normal(20000) * 0.01,
                        rng.uniform(-448, 448, 20000)]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref.e4m3_encode_array(x.astype(np.float64)), lib)


def test_vectorised_encoder_equals_the_scalar_one():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 100, rng.standard_normal(5000) * 1e-3,
                        [0.0, -0.0, 448.0, 464.0, 465.0, 1e30, -1e30, np.nan]])
    assert np.array_equal(ref.e4m3_encode_array(x), np.array([ref.e4m3_encode(v) for v in x], dtype=np.uint8))


def test_half_ulp_error_bound():
    rng = np.random.default_rng(2)
    x = rng.uniform(-440, 440, 100000)
    back = ref.e4m3_dequantize(ref.e4m3_encode_array(x), 1.0)
    normal = np.abs(x) >= 2.0 ** -6
    assert np.all(np.abs(back - x)[normal] <= np.abs(x)[normal] * 2.0 ** -4 + 1e-300)
    assert np.all(np.abs(back - x)[~normal] <= 2.0 ** -10)


def test_quantize_decides_on_the_float32_product():
    # x * (1/s) straddles a midpoint: in float64 it is just above 1.0625, the
    # float32 product rounds onto it exactly (then to even, 1.0)
    s = 3.0
    x = 1.0625 * 3.0 + 2e-8
    assert 1.0625 < x * (1.0 / s)
    assert float(np.float32(np.float32(x) * (np.float32(1.0) / np.float32(s)))) == 1.0625
    assert int(ref.e4m3_quantize(np.array([x]), s)[0]) == 0x38


def _fp8_pair(seed, B=2, Hkv=2, d=16, max_len=48):
    c8 = ref.OracleCache(1, B, Hkv, max_len, d)
    c8.set_fp8()
    rng = np.random.default_rng(seed)
    ks, vs = rng.uniform(0.002, 0.02, Hkv), rng.uniform(0.002, 0.02, Hkv)
    c8.set_kv_scales(0, ks, vs)
    return c8, ks, vs


def test_fp8_cache_equals_ordinary_cache_on_dequantized_values():
    B, Hkv, G, d = 2, 2, 3, 16
    c8, ks, vs = _fp8_pair(3, B, Hkv, d)
    plain = ref.OracleCache(1, B, Hkv, 48, d)
    rng = np.random.default_rng(4)
    for step in range(6):
        n_new = rng.integers(0, 6, size=B)
        T = max(int(n_new.max()), 1)
        k = wl.normal(5, 10 + step, (B, Hkv, T, d)).numpy()
        v = wl.normal(5, 20 + step, (B, Hkv, T, d)).numpy()
        q = wl.normal(5, 30 + step, (B, Hkv * G, T, d)).numpy()
        # what the FP8 cache will hold, computed per head from the codes
        kd = np.stack([ref.e4m3_dequantize(ref.e4m3_quantize(k[:, h], ks[h]), ks[h]) for h in range(Hkv)], axis=1)
        vd = np.stack([ref.e4m3_dequantize(ref.e4m3_quantize(v[:, h], vs[h]), vs[h]) for h in range(Hkv)], axis=1)
        got = ref.append_attention(c8, 0, q, k, v, n_new)
        want = ref.append_attention(plain, 0, q, kd, vd, n_new)
        assert np.array_equal(got, want)
    # codes and values agree slot by slot
    L = int(c8.lens[0, 0])
    for h in range(Hkv):
        assert np.array_equal(ref.e4m3_dequantize(c8.k_code[0][0, h, :L], ks[h]), c8.k[0][0, h, :L])


def test_fp8_attention_close_to_exact_values():
    """Quantization error only: outputs stay within a few percent of the unquantized cache."""
    B, Hkv, G, d = 2, 2, 4, 16
    c8 = ref.OracleCache(1, B, Hkv, 64, d)
    c8.set_fp8()
    c8.set_kv_scales(0, [4.0 / 448] * Hkv, [4.0 / 448] * Hkv)  # N(0,1) data: 4 sigma maps to 448
    plain = ref.OracleCache(1, B, Hkv, 64, d)
    k = wl.normal(6, 1, (B, Hkv, 40, d)).numpy()
    v = wl.normal(6, 2, (B, Hkv, 40, d)).numpy()
    q = wl.normal(6, 3, (B, Hkv * G, 40, d)).numpy()
    n = np.array([40, 33])
    err = np.max(np.abs(ref.append_attention(c8, 0, q, k, v, n) - ref.append_attention(plain, 0, q, k, v, n)))
    assert 0 < err < 0.25  # a loose sanity bound: 3 mantissa bits give up to 6 % error per stored value


def test_scale_and_format_rules():
    c8, _, _ = _fp8_pair(7)
    with pytest.raises(ref.CacheError):
        c8.set_kv_scales(0, [1.0], [1.0, 1.0])
    with pytest.raises(ref.CacheError):
        c8.set_kv_scales(0, [0.0, 1.0], [1.0, 1.0])
    z = np.zeros((2, 2, 1, 16))
    c8.append(0, z, z, [1, 0])
    with pytest.raises(ref.CacheError):
        c8.set_kv_scales(0, [1.0, 1.0], [1.0, 1.0])  # the layer holds data
    with pytest.raises(ref.CacheError):
        c8.set_fp8()
    c8.reset()
    c8.set_kv_scales(0, [1.0, 1.0], [1.0, 1.0])


def test_planted_mistakes_are_caught(monkeypatch):
    true_encode, true_dequantize = ref.e4m3_encode_array, ref.e4m3_dequantize
    # round half away from zero instead of half to even: the midpoint 1.0625 must go to 1.0
    def half_up(x):
        x = np.asarray(x, dtype=np.float64)
        return true_encode(x + np.where(x >= 0, 1e-12, -1e-12) * np.abs(x))

    monkeypatch.setattr(ref, "e4m3_encode_array", half_up)
    assert ref.e4m3_quantize(np.array([1.0625]), 1.0)[0] != 0x38
    monkeypatch.undo()
    # dequantize on read without the scale
    c8, ks, vs = _fp8_pair(8)
    k = wl.normal(9, 1, (2, 2, 3, 16)).numpy()
    c8.append(0, k, k, [3, 3])
    monkeypatch.setattr(ref, "e4m3_dequantize", lambda codes, scale: true_dequantize(codes, 1.0))
    bad, _, _ = _fp8_pair(8)
    bad.append(0, k, k, [3, 3])
    assert not np.allclose(bad.k[0][:, :, :3], c8.k[0][:, :, :3])
