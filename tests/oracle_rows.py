"""Oracle side of the full-size and device-resident parity tests.

A cache filled by the seeded generator holds, for every (row b, KV head kvh),
generator rows below its initial length and then the chunks appended by the
calls under test.  This helper rebuilds those rows on the CPU from the
generator (never from the device) and gives the oracle's output of a call
query by query (``oracle.ref.attend_one_query`` at ``query_position``: the
pages' ``gqa_attention`` for one query, without materialising the KV repeat
for every head of a large cache).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle.ref as ref
from gqa_attention_preallocated_gb300 import workloads as wl


def generator_rows(seed, stream, B, H, max_len, d, b, h, lo, hi):
    """Rows [lo, hi) of unit (b, h) of a generator-filled [B, H, max_len, d] bf16 tensor, float64 on the CPU."""
    base = ((b * H + h) * max_len + lo) * d
    idx = torch.arange(base, base + (hi - lo) * d, dtype=torch.int64)
    return wl.to_storage(wl.normal_at(seed, stream, idx), torch.bfloat16).double().reshape(hi - lo, d).numpy()


class UnitOracle:
    """Stored K/V of chosen (b, kvh) units of one layer, and the oracle's outputs of each call."""

    def __init__(self, seed, B, Hkv, max_len, d, lens0, units=None):
        self.B, self.Hkv, self.d = B, Hkv, d
        self.units = list(units) if units is not None else [(b, h) for b in range(B) for h in range(Hkv)]
        self.K, self.V = {}, {}
        for b, h in self.units:
            L0 = int(lens0[b])
            self.K[b, h] = [generator_rows(seed, wl.STREAM_CACHE_K, B, Hkv, max_len, d, b, h, 0, L0)]
            self.V[b, h] = [generator_rows(seed, wl.STREAM_CACHE_V, B, Hkv, max_len, d, b, h, 0, L0)]

    def step(self, q, k_new, v_new, n_new):
        """One call: append n_new[b] tokens of k_new / v_new (CPU tensors, as stored) to every tracked unit,
        then the oracle's outputs {(b, h, t): float64 [d]} for the tracked units' valid queries."""
        q = q.double().cpu().numpy()
        kn = k_new.double().cpu().numpy()
        vn = v_new.double().cpu().numpy()
        G = q.shape[1] // self.Hkv
        want = {}
        for b, kvh in self.units:
            n = int(n_new[b])
            self.K[b, kvh].append(kn[b, kvh, :n])
            self.V[b, kvh].append(vn[b, kvh, :n])
            K = np.concatenate(self.K[b, kvh])
            V = np.concatenate(self.V[b, kvh])
            self.K[b, kvh], self.V[b, kvh] = [K], [V]
            L = K.shape[0]
            for g in range(G):
                h = kvh * G + g
                for t in range(n):
                    want[b, h, t] = ref.attend_one_query(q[b, h, t], K, V, ref.query_position(L, n, t))
        return want


def max_error(got, want, n_new, tracked_units, Hkv):
    """Largest |got - want| over the tracked queries; padded queries of tracked units must be exactly 0."""
    got = got.double().cpu().numpy()
    G = got.shape[1] // Hkv
    T = got.shape[2]
    worst = 0.0
    for b, kvh in tracked_units:
        for g in range(G):
            h = kvh * G + g
            for t in range(T):
                if t >= int(n_new[b]):
                    assert np.all(got[b, h, t] == 0.0), (b, h, t)
                    continue
                worst = max(worst, float(np.max(np.abs(got[b, h, t] - want[b, h, t]))))
    return worst
