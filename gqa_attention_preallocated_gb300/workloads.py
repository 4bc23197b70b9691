"""Seeded synthetic inputs for the cache and attention workloads.

This module only draws numbers: it holds none of the attention arithmetic and
imports neither the CUDA library nor the CPU oracle, so both sides of every
comparison can take their inputs from here.

Values.  q, k and v are approximately N(0, 1): the sum of four uniforms on
(0, 1), centred and scaled to unit variance (the Irwin-Hall distribution with
n = 4).  The uniforms come from a counter-based hash, so the value of any
element can be recomputed on its own from (seed, stream, flat index) without
generating the rest of the tensor.  That is what lets the tests check sampled
outputs of a 68 GB cache on the CPU.

The hash is Chris Wellons' "lowbias32" integer hash (hash-prospector, 2018):
    x ^= x >> 16; x *= 0x7feb352d; x ^= x >> 15; x *= 0x846ca68b; x ^= x >> 16
(32-bit wrapping multiply).  It is evaluated with int64 torch tensors holding
32-bit values, with every multiply split so that no intermediate overflows, so
CPU and GPU give the same bits.  Float conversion: the four 16-bit fields u_i
give (u_i + 0.5) / 65536 exactly in float64; their sum minus 2 is exact; one
multiply by sqrt(3) rounds once (IEEE, same on both devices); storage types
are reached by an explicit float64 -> float32 -> (bfloat16) rounding chain.

Lengths and chunk sizes are drawn with ``numpy.random.default_rng(seed)``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_M32 = 0xFFFFFFFF


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for 0 <= x < 2**32, without int64 overflow."""
    lo = c & 0xFFFF
    hi = (c >> 16) & 0xFFFF
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _lowbias32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _stream_key(seed: int, stream: int) -> int:
    t = torch.tensor([((seed & _M32) * 0x9E3779B1 + (stream & _M32) * 0x85EBCA77 + 0x27D4EB2F) & _M32], dtype=torch.int64)
    return int(_lowbias32(_lowbias32(t) ^ ((seed >> 32) & _M32)).item())


def normal_at(seed: int, stream: int, flat_index: torch.Tensor) -> torch.Tensor:
    """Float64 approximately-N(0,1) values at the given flat indices (int64 tensor)."""
    idx = flat_index.to(torch.int64)
    key = _stream_key(seed, stream)
    lo = idx & _M32
    hi = idx >> 32
    a = _lowbias32(_lowbias32(lo ^ key) ^ hi)
    b = _lowbias32(a ^ 0x5BD1E995)
    s = (a & 0xFFFF).to(torch.float64)
    s = s + (a >> 16).to(torch.float64)
    s = s + (b & 0xFFFF).to(torch.float64)
    s = s + (b >> 16).to(torch.float64)
    # sum of four (u + 0.5) / 65536, minus 2, exactly: (s + 2) / 65536 - 2
    s = (s + 2.0) * (1.0 / 65536.0) - 2.0
    return s * math.sqrt(3.0)


def normal(seed: int, stream: int, shape, device="cpu", offset: int = 0) -> torch.Tensor:
    """Float64 tensor of ``shape`` whose element i (row-major) is normal_at(offset + i)."""
    n = int(np.prod(shape)) if len(shape) else 1
    idx = torch.arange(offset, offset + n, dtype=torch.int64, device=device)
    return normal_at(seed, stream, idx).reshape(shape)


def to_storage(x64: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Round float64 values to the storage type: float64 -> float32 (-> bfloat16)."""
    x32 = x64.to(torch.float32)
    if dtype == torch.float32:
        return x32
    if dtype == torch.bfloat16:
        return x32.to(torch.bfloat16)
    raise ValueError(f"unsupported storage dtype {dtype}")


def fill_normal_(dst: torch.Tensor, seed: int, stream: int, chunk: int = 1 << 26) -> torch.Tensor:
    """Fill a contiguous tensor (any device) in place with normal(seed, stream) values."""
    flat = dst.view(-1)
    n = flat.numel()
    for start in range(0, n, chunk):
        stop = min(n, start + chunk)
        idx = torch.arange(start, stop, dtype=torch.int64, device=dst.device)
        flat[start:stop] = to_storage(normal_at(seed, stream, idx), dst.dtype)
    return dst


# ---------------------------------------------------------------------------
# Workload shapes.  Names describe the workload; sizes follow the pages'
# examples (Llama-3.1-8B-shaped heads: Hq = 32, Hkv = 8, d = 128).
# ---------------------------------------------------------------------------

STREAM_CACHE_K = 1
STREAM_CACHE_V = 2
STREAM_Q = 3
STREAM_K_NEW = 4
STREAM_V_NEW = 5


@dataclass
class Shape:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    max_len: int
    dtype: str  # "f32" | "bf16"
    layers: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


TINY = Shape("tiny_ragged_gqa_b2_hq8_hkv2_d16_f32", B=2, Hq=8, Hkv=2, d=16, max_len=64, dtype="f32")
DECODE_8B = Shape("llama8b_decode_b32_hq32_hkv8_d128_len8192_bf16", B=32, Hq=32, Hkv=8, d=128, max_len=8192, dtype="bf16")
PREFILL = Shape("chunked_prefill_b4_hq32_hkv8_d128_len16384_chunk512_bf16", B=4, Hq=32, Hkv=8, d=128, max_len=16384, dtype="bf16")
VERIFY = Shape("spec_verify_b64_hkv8_d128_s4096_bf16", B=64, Hq=32, Hkv=8, d=128, max_len=4096, dtype="bf16")
LONGCTX = Shape("longctx_32layer_decode_b4_hq32_hkv8_d128_len131072_bf16", B=4, Hq=32, Hkv=8, d=128, max_len=131072, dtype="bf16", layers=32)


def tiny_schedule(seed: int, B: int, max_final: int = 40, max_chunk: int = 8):
    """Per-call n_new vectors for one ragged trial.

    Final lengths are uniform in 0..max_final per row; each call gives every
    unfinished row min(U{1..max_chunk}, remaining) tokens and finished rows 0;
    T of a call is the largest n_new in it.  Returns (finals, [n_new, ...]).
    """
    rng = np.random.default_rng(seed)
    finals = rng.integers(0, max_final + 1, size=B).astype(np.int64)
    lens = np.zeros(B, dtype=np.int64)
    calls = []
    while np.any(lens < finals):
        want = rng.integers(1, max_chunk + 1, size=B)
        n = np.minimum(want, finals - lens)
        n = np.where(lens < finals, n, 0).astype(np.int64)
        calls.append(n)
        lens += n
    return finals, calls


def trial_geometry(seed: int):
    """Random geometry of one brute-force trial: Hkv in {1,2,4}, G in 1..8, B in 1..3."""
    rng = np.random.default_rng(10_000 + seed)
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.integers(1, 9))
    B = int(rng.integers(1, 4))
    d = int(rng.choice([4, 8, 16]))
    return B, Hkv, G, d


def decode_lens(seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    """Initial row lengths uniform in [lo, hi] (inclusive)."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=B).astype(np.int64)


def prefill_priors(seed: int, B: int, chunk: int = 512, max_prior: int = 15872) -> np.ndarray:
    """Prior lengths: uniform multiples of ``chunk`` in [0, max_prior]."""
    rng = np.random.default_rng(seed)
    return (rng.integers(0, max_prior // chunk + 1, size=B) * chunk).astype(np.int64)


def ragged_chunk(seed: int, B: int, chunk: int = 512) -> np.ndarray:
    """Final ragged chunk sizes n_new uniform in 1..chunk."""
    rng = np.random.default_rng(seed + 7919)
    return rng.integers(1, chunk + 1, size=B).astype(np.int64)
