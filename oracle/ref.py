"""CPU float64 oracle for grouped-query attention over a preallocated KV cache.

TEST INFRASTRUCTURE ONLY.  This module is the definition the GPU library is
checked against.  Only the test suite, the package smoke check and the CPU
baseline leg of the benchmark may import it; the product path never does, and
it shares no code with the CUDA library (no kernels, headers, helpers or
constants).  It is deliberately plain and slow: NumPy float64, an explicit
loop over every (row, query head, query), an explicit repeat of the KV heads
to the query heads, and a plain softmax over keys 0..position.

Sources (three web pages; "p1", "p2", "p3" below):

* p1  "Implement grouped-query attention over a preallocated KV cache, with no
       torch.cat, for both prefill chunks and decode" (inferenceinterviews.com)
       - section "A strong answer": the ``KVCache`` class (allocate
         [B, Hkv, max_len, d] once, write in place at the row's length, raise
         past max_len) and ``gqa_attention`` (scale 1/sqrt(d), query t at
         absolute position lens - n_new + t, keys past lens masked, padded
         queries masked, fully masked rows -> zeros).
       - "The decisions an interviewer reads for", items 1-3, and the
         paragraph after them: the direct reference this oracle restates
         (repeat KV heads, loop over every query, plain softmax over keys 0
         to its position).
       - "Common mistakes": h // G (not h % Hkv); increment lengths only
         after the write.
* p2  "Write the causal mask for a decode step with a KV cache, where the
       query is shorter than the keys" (inferenceinterviews.com)
       - TL;DR and "A strong answer": bottom-right mask j <= i + (S - T),
         ``decode_causal_mask``; the top-left ``tril(ones(T, S))`` as the
         wrong convention; the T = 4, S = 4096 count.
* p3  "16. Prefill, decode and the KV cache" (inference.shantanugoel.com)
       - "Layout and validity": per-layer lengths, ``length`` refusing when a
         forward pass stopped part-way, ``update`` shape checks,
         ``truncate`` / ``reset``.
       - "How big is the cache?": the KV byte formula.

Readings where the pages are silent or loose (each is also listed in the
design notes):

* Overflow in one row of a batch: p1's loop would already have written the
  earlier rows when it raises.  Here every row is validated first and nothing
  is written on error, so an error leaves data and lengths unchanged.
* ``n_new[b]`` must satisfy 0 <= n_new[b] <= T; anything else is an error.
* Lengths are kept per layer and per row (p3 keeps one length per layer, p1
  one per row).  ``truncate`` takes one new length per row, applies it to
  every layer, and requires 0 <= new <= current for every row.
* ``length`` returns the per-row lengths shared by all layers and raises if
  any two layers disagree.
* Output for a padded query (t >= n_new[b]), for an empty batch, an empty
  chunk (T = 0) or an empty cache is zero.

Sliding window and ring buffer (p2 "A strong answer", its last paragraph, and
"Common mistakes"; p3 exercise 3):

* With a window W >= 1, the query at absolute position p sees the keys at
  positions a with p - W < a <= p (the lower bound j > (S - T) + i - W).
* A ring cache keeps max_len slots; the token at position a lives in slot
  a mod max_len, and the cache records the position stored in every slot.
  Attention selects keys by those stored positions, never by slot index.
  Lengths count every token appended (they may pass max_len).
* A ring chunk must fit beside its window: n_new[b] <= max_len - W + 1
  (else the chunk's first query would need a key already overwritten).
  Truncation to a length n needs the keys n - W + 1 .. n - 1 still in the
  ring (or n = 0) for the same reason.

Tree speculative verify (p2 "What interviewers probe next", the tree-based
speculative decoding question): the chunk's T draft tokens form a tree given
by parent pointers.  Draft token t sees every key before the chunk plus the
draft tokens on its own path to the root (itself and its ancestors), so the
T x T corner is an ancestor mask instead of a triangle.  Readings: parents
precede their children (parent[t] < t) and parent -1 means the token hangs
directly off the cached prefix; trees do not combine with a window.

Paged storage (p1 "A strong answer", the reversal condition: wildly ragged
rows call for a block table and a paged kernel; p3 "Design choices worth
noticing": a paged cache avoids reserving max_len per row up front): K and
V live in pages of P tokens, and a per-row block table maps logical page
a // P of row b to a physical page.  Attention is defined on the logical
sequence: ``PagedOracleCache.view`` gathers every row through the table into
an ordinary cache, and the ordinary attention runs on that.

FP8 storage (p3 "16. Prefill, decode and the KV cache", exercise 4: keep the
cache in FP8 E4M3 with one scale per head and dequantize on read; the
bandwidth bullet of the same page gives the motive).  Readings where the page
is silent (each also listed in the design notes):

* E4M3 is the 8-bit format with 1 sign bit, 4 exponent bits (bias 7) and 3
  mantissa bits: exponent field 0 holds the subnormals m/8 * 2^-6, fields
  1..15 hold (1 + m/8) * 2^(e - 7), and exponent 15 with mantissa 7 is NaN;
  there is no infinity, so the largest finite value is 448.
* "One scale per head" is one positive scale per (layer, KV head), separate
  for K and V, set by the caller while the layer is empty.
* A value x is stored as the E4M3 code nearest to x * (1/s), where the
  reciprocal 1/s and the product are each rounded to float32; ties go to
  the code with an even mantissa, and values beyond +-448 saturate to +-448.
* Attention reads code value * s (dequantize on read) and is otherwise the
  ordinary attention.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "CacheError",
    "OracleCache",
    "kv_head_of",
    "query_position",
    "score_scale",
    "attend_one_query",
    "gqa_attention",
    "append_attention",
    "decode_causal_mask",
    "decode_window_mask",
    "top_left_causal_mask",
    "visible_slots",
    "tree_path",
    "tree_corner_mask",
    "PagedOracleCache",
    "kv_cache_bytes",
    "e4m3_value",
    "e4m3_encode",
    "e4m3_quantize",
]


class CacheError(ValueError):
    """Raised for every rejected cache operation (overflow, bad shape, ...)."""


# ---------------------------------------------------------------------------
# Small named steps.  Each is one rule from the pages; keeping them separate
# lets the self-check suite swap in a plausible wrong version and confirm
# that some check fails.
# ---------------------------------------------------------------------------


def kv_head_of(h: int, G: int) -> int:
    """KV head read by query head h: h // G (p1 TL;DR; p1 "Common mistakes")."""
    return h // G


def query_position(lens_b: int, n_new_b: int, t: int) -> int:
    """Absolute position of query t of the chunk just appended to row b.

    p1 TL;DR and ``gqa_attention``: the chunk's queries are the last n_new
    positions of the row, so query t sits at lens - n_new + t (p2 TL;DR: the
    same rule written as S - T + i).
    """
    return lens_b - n_new_b + t


def score_scale(d: int) -> float:
    """Scores are q.k / sqrt(d) (p1 ``gqa_attention``)."""
    return 1.0 / math.sqrt(d)


def attend_one_query(q_vec: np.ndarray, K_rows: np.ndarray, V_rows: np.ndarray, pos: int) -> np.ndarray:
    """Output of one query at absolute position ``pos`` against one head's keys.

    Plain softmax over keys 0..pos (p1, the direct reference described after
    "The decisions an interviewer reads for").  ``K_rows``/``V_rows`` are that
    head's [len, d] rows; only rows 0..pos are read.  A query that sees no key
    (pos < 0) returns zeros (p1 decision 3).
    """
    d = q_vec.shape[-1]
    if pos < 0:
        return np.zeros(d, dtype=np.float64)
    keys = np.asarray(K_rows[: pos + 1], dtype=np.float64)
    vals = np.asarray(V_rows[: pos + 1], dtype=np.float64)
    s = (keys @ np.asarray(q_vec, dtype=np.float64)) * score_scale(d)
    s = s - s.max()
    p = np.exp(s)
    p = p / p.sum()
    return p @ vals


# ---------------------------------------------------------------------------
# FP8 E4M3 (p3 exercise 4), written out from the format's definition.
# ---------------------------------------------------------------------------


def e4m3_value(code: int) -> float:
    """The real number an E4M3 byte encodes (NaN for the two NaN codes)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _e4m3_positive_table():
    """(value, code) for the 127 non-negative finite codes, ascending."""
    return [(e4m3_value(c), c) for c in range(0x7F)]


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code to x: ties to the even mantissa, beyond +-448 saturates to +-448, NaN to 0x7F."""
    x = float(x)
    if math.isnan(x):
        return 0x7F
    sign = 0x80 if (x < 0 or (x == 0 and math.copysign(1.0, x) < 0)) else 0x00
    a = abs(x)
    table = _e4m3_positive_table()
    if a >= table[-1][0]:
        return sign | table[-1][1]
    for i in range(len(table) - 1):
        lo, hi = table[i], table[i + 1]
        if lo[0] <= a <= hi[0]:
            if a - lo[0] < hi[0] - a:
                return sign | lo[1]
            if a - lo[0] > hi[0] - a:
                return sign | hi[1]
            return sign | (lo[1] if lo[1] % 2 == 0 else hi[1])
    raise AssertionError("unreachable")


def e4m3_encode_array(x) -> np.ndarray:
    """``e4m3_encode`` applied to every element (same rule, vectorised with a sorted table)."""
    x = np.asarray(x, dtype=np.float64)
    table = _e4m3_positive_table()
    vals = np.array([v for v, _ in table])
    codes = np.array([c for _, c in table], dtype=np.int64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 1, len(vals) - 1)  # vals[hi-1] < a <= vals[hi]
    lo = hi - 1
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[lo] % 2 == 1))
    out = np.where(pick_hi, codes[hi], codes[lo])
    out = np.where(a >= vals[-1], codes[-1], out)
    out = np.where(a == 0, 0, out)
    neg = np.signbit(x)
    out = np.where(neg, out | 0x80, out)
    out = np.where(np.isnan(x), 0x7F, out)
    return out.astype(np.uint8)


def e4m3_quantize(x, scale: float) -> np.ndarray:
    """Codes (uint8) of the values x stored with scale s: e4m3_encode(f32(x * f32(1/s)))."""
    inv = np.float32(1.0) / np.float32(scale)
    y = np.asarray(x, dtype=np.float64).astype(np.float32) * inv
    return e4m3_encode_array(np.asarray(y, dtype=np.float32).astype(np.float64))


def e4m3_dequantize(codes, scale: float) -> np.ndarray:
    """Values read back from codes stored with scale s: value(code) * s."""
    codes = np.asarray(codes, dtype=np.uint8)
    lut = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
    return lut[codes] * float(scale)


class OracleCache:
    """Preallocated KV cache with per-layer, per-row valid lengths.

    K and V of each layer are float64 arrays [B, Hkv, max_len, d] allocated
    once (p1 ``KVCache.__init__``; p3 "Layout and validity" with one buffer
    pair per layer).  ``lens[layer, b]`` counts the valid tokens of row b.
    """

    def __init__(self, layers: int, batch: int, kv_heads: int, max_len: int, head_dim: int):
        if layers < 1 or batch < 0 or kv_heads < 1 or max_len < 0 or head_dim < 1:
            raise CacheError("bad cache geometry")
        self.layers, self.B, self.Hkv, self.max_len, self.d = layers, batch, kv_heads, max_len, head_dim
        shape = (batch, kv_heads, max_len, head_dim)
        self.k = [np.zeros(shape, dtype=np.float64) for _ in range(layers)]
        self.v = [np.zeros(shape, dtype=np.float64) for _ in range(layers)]
        self.lens = np.zeros((layers, batch), dtype=np.int64)
        # absolute position stored in every slot (-1: never written)
        self.pos = [np.full((batch, max_len), -1, dtype=np.int64) for _ in range(layers)]
        self.window = 0   # 0: no window (keys 0..p)
        self.ring = False
        # FP8 E4M3 storage: codes per slot, one scale per (layer, KV head) for K and for V
        self.fp8 = False
        self.k_code = self.v_code = None
        self.k_scale = np.ones((layers, kv_heads))
        self.v_scale = np.ones((layers, kv_heads))

    def set_fp8(self) -> None:
        """Store K and V as E4M3 codes (p3 exercise 4); only on an empty cache."""
        if np.any(self.lens != 0):
            raise CacheError("the storage format can only change on an empty cache")
        self.fp8 = True
        shape = (self.B, self.Hkv, self.max_len, self.d)
        self.k_code = [np.zeros(shape, dtype=np.uint8) for _ in range(self.layers)]
        self.v_code = [np.zeros(shape, dtype=np.uint8) for _ in range(self.layers)]

    def set_kv_scales(self, layer: int, k_scale, v_scale) -> None:
        """One positive finite scale per KV head for K and for V; only while the layer is empty."""
        k_scale = np.asarray(k_scale, dtype=np.float64).reshape(-1)
        v_scale = np.asarray(v_scale, dtype=np.float64).reshape(-1)
        if k_scale.shape[0] != self.Hkv or v_scale.shape[0] != self.Hkv:
            raise CacheError("one scale per KV head")
        if not (np.all(np.isfinite(k_scale)) and np.all(np.isfinite(v_scale)) and np.all(k_scale > 0)
                and np.all(v_scale > 0)):
            raise CacheError("scales must be positive and finite")
        if np.any(self.lens[layer] != 0):
            raise CacheError("scales can only change while the layer is empty")
        self.k_scale[layer] = k_scale
        self.v_scale[layer] = v_scale

    def set_window(self, window: int, ring: bool = False) -> None:
        """Attention window W (0 = none) and ring storage (slot = position mod max_len).

        Ring storage needs a window of 1..max_len and may only be switched
        on or off while the cache is empty.
        """
        if window < 0:
            raise CacheError("window must be >= 0")
        if ring and not 1 <= window <= self.max_len:
            raise CacheError("a ring cache needs a window of 1..max_len")
        if bool(ring) != self.ring and np.any(self.lens != 0):
            raise CacheError("ring storage can only change on an empty cache")
        self.window, self.ring = int(window), bool(ring)

    def slot_of(self, position: int) -> int:
        """Slot holding an absolute position: the position itself, or position mod max_len in a ring."""
        return position % self.max_len if self.ring else position

    # -- p1 ``KVCache.append`` / p3 ``KVCache.update`` ----------------------
    def append(self, layer: int, k_new: np.ndarray, v_new: np.ndarray, n_new) -> None:
        """Write k_new[b, :, :n_new[b]] at rows lens[b] .. lens[b]+n_new[b]-1.

        All rows are checked before any write; lengths grow only after every
        write (p1 "Common mistakes", last item).  Raises ``CacheError`` on a
        shape mismatch (p3 ``update``), on n_new outside 0..T, or when a row
        would pass max_len (p1 ``append``, p3 ``update``).
        """
        if not 0 <= layer < self.layers:
            raise CacheError(f"layer {layer} out of range")
        k_new = np.asarray(k_new)
        v_new = np.asarray(v_new)
        if k_new.ndim != 4 or k_new.shape != v_new.shape:
            raise CacheError("k_new and v_new must both be [B, Hkv, T, d]")
        Bn, Hn, T, dn = k_new.shape
        if Bn != self.B or Hn != self.Hkv or dn != self.d:
            raise CacheError("cache batch/head/width shapes differ")
        n_new = np.asarray(n_new, dtype=np.int64).reshape(-1)
        if n_new.shape[0] != self.B:
            raise CacheError("n_new must have one entry per row")
        lens = self.lens[layer]
        for b in range(self.B):
            if n_new[b] < 0 or n_new[b] > T:
                raise CacheError(f"row {b}: n_new={n_new[b]} outside 0..{T}")
            if self.ring:
                if n_new[b] > self.max_len - self.window + 1:
                    raise CacheError(f"row {b}: a ring chunk of {n_new[b]} tokens does not fit beside its window")
            elif lens[b] + n_new[b] > self.max_len:
                raise CacheError(f"row {b}: {lens[b] + n_new[b]} tokens > max_len {self.max_len}")
        for b in range(self.B):
            for t in range(int(n_new[b])):
                a = int(lens[b]) + t
                slot = self.slot_of(a)
                if self.fp8:
                    for h in range(self.Hkv):
                        kc = e4m3_quantize(k_new[b, h, t], self.k_scale[layer, h])
                        vc = e4m3_quantize(v_new[b, h, t], self.v_scale[layer, h])
                        self.k_code[layer][b, h, slot] = kc
                        self.v_code[layer][b, h, slot] = vc
                        self.k[layer][b, h, slot] = e4m3_dequantize(kc, self.k_scale[layer, h])
                        self.v[layer][b, h, slot] = e4m3_dequantize(vc, self.v_scale[layer, h])
                else:
                    self.k[layer][b, :, slot] = k_new[b, :, t]
                    self.v[layer][b, :, slot] = v_new[b, :, t]
                self.pos[layer][b, slot] = a
        self.lens[layer] = lens + n_new

    def lens_of(self, layer: int) -> np.ndarray:
        return self.lens[layer].copy()

    # -- p3 ``length`` / ``truncate`` / ``reset`` -----------------------------
    def length(self) -> np.ndarray:
        """Per-row lengths shared by every layer; raises if layers disagree."""
        if self.layers > 1 and np.any(self.lens != self.lens[0][None, :]):
            raise CacheError("a forward pass stopped part-way; reset or truncate the cache")
        return self.lens[0].copy()

    def truncate(self, new_lens) -> None:
        """Forget everything after new_lens[b] tokens in every layer; no data moves."""
        new_lens = np.asarray(new_lens, dtype=np.int64).reshape(-1)
        if new_lens.shape[0] != self.B:
            raise CacheError("new_lens must have one entry per row")
        cur = self.length()
        if np.any(new_lens < 0) or np.any(new_lens > cur):
            raise CacheError("invalid truncation length")
        if self.ring:
            # Keys positions max(0, new - W + 1) .. new - 1 must still be in the
            # ring (it holds positions cur - max_len .. cur - 1); new = 0 needs none.
            for b in range(self.B):
                n = int(new_lens[b])
                if n > 0 and max(0, n - self.window + 1) < int(cur[b]) - self.max_len:
                    raise CacheError("a ring cache cannot go back past the keys it still holds")
        self.lens[:] = new_lens[None, :]

    def reset(self) -> None:
        self.truncate(np.zeros(self.B, dtype=np.int64))

    def bytes(self) -> int:
        """Bytes held by every K and V buffer (p3 ``bytes``), at 8 B a value."""
        return sum(a.nbytes for a in self.k + self.v)


def visible_slots(stored: np.ndarray, lens_b: int, p: int, window: int) -> np.ndarray:
    """Slots whose stored position a a query at position p may see.

    a must be a written, valid position (0 <= a < lens), at most p, and with a
    window above p - W (p2: the mask compares stored positions, never slot
    indices, and gains the lower bound j > (S - T) + i - W).  Ascending
    position order.
    """
    a = stored
    ok = (a >= 0) & (a < lens_b) & (a <= p)
    if window > 0:
        ok &= a > p - window
    slots = np.nonzero(ok)[0]
    return slots[np.argsort(a[slots], kind="stable")]


def attend_slots(q_vec: np.ndarray, K_rows: np.ndarray, V_rows: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Plain softmax attention of one query over the given slots (zeros if none)."""
    d = q_vec.shape[-1]
    if slots.size == 0:
        return np.zeros(d, dtype=np.float64)
    keys = np.asarray(K_rows[slots], dtype=np.float64)
    vals = np.asarray(V_rows[slots], dtype=np.float64)
    s = (keys @ np.asarray(q_vec, dtype=np.float64)) * score_scale(d)
    s = s - s.max()
    p = np.exp(s)
    p = p / p.sum()
    return p @ vals


def tree_path(parents_row, t: int) -> list:
    """Draft tokens token t may see: itself and its ancestors (p2, tree verify)."""
    path = []
    u = t
    while u >= 0:
        path.append(u)
        u = int(parents_row[u])
    return path


def tree_corner_mask(parents_row) -> np.ndarray:
    """Bool [T, T]: True where draft token t may see draft token u (u on t's path)."""
    T = len(parents_row)
    m = np.zeros((T, T), dtype=bool)
    for t in range(T):
        m[t, tree_path(parents_row, t)] = True
    return m


def check_parents(parents: np.ndarray, T: int) -> None:
    """parents[b, t] in -1 .. t-1 (a parent precedes its child)."""
    for b in range(parents.shape[0]):
        for t in range(T):
            if not -1 <= int(parents[b, t]) < t:
                raise CacheError(f"row {b}: parent of draft token {t} must be in -1..{t - 1}")


def gqa_attention(q: np.ndarray, cache: OracleCache, layer: int, n_new, parents=None) -> np.ndarray:
    """Attention of the T queries of the chunk just appended (p1 ``gqa_attention``).

    q is [B, Hq, T, d] with Hq a multiple of Hkv.  The KV heads are explicitly
    repeated to Hq heads, then every query (b, h, t) with t < n_new[b] attends
    to keys 0..lens[b]-n_new[b]+t of KV head h // G with a plain softmax.
    Padded queries and empty cases give zeros.  Returns float64 [B, Hq, T, d].
    With ``parents`` (int [B, T], a draft tree per row) query t sees the keys
    before the chunk plus the chunk's tokens on its path to the root.
    """
    q = np.asarray(q, dtype=np.float64)
    if q.ndim != 4:
        raise CacheError("q must be [B, Hq, T, d]")
    B, Hq, T, d = q.shape
    if B != cache.B or d != cache.d:
        raise CacheError("q batch/width differ from the cache")
    if Hq % cache.Hkv != 0:
        raise CacheError("Hq must be a multiple of Hkv")
    G = Hq // cache.Hkv
    n_new = np.asarray(n_new, dtype=np.int64).reshape(-1)
    if n_new.shape[0] != B:
        raise CacheError("n_new must have one entry per row")
    lens = cache.lens[layer]
    if np.any(n_new < 0) or np.any(n_new > T) or np.any(n_new > lens):
        raise CacheError("n_new must satisfy 0 <= n_new <= min(T, lens)")
    if parents is not None:
        parents = np.asarray(parents, dtype=np.int64).reshape(B, T)
        check_parents(parents, T)
        if cache.window or cache.ring:
            raise CacheError("a draft tree does not combine with a window")
    out = np.zeros((B, Hq, T, d), dtype=np.float64)
    if B == 0 or T == 0:
        return out
    # The direct reference materialises one copy of KV head h // G for every
    # query head h (the repeat the GPU path avoids).
    k_rep = np.stack([cache.k[layer][:, kv_head_of(h, G)] for h in range(Hq)], axis=1)
    v_rep = np.stack([cache.v[layer][:, kv_head_of(h, G)] for h in range(Hq)], axis=1)
    for b in range(B):
        for h in range(Hq):
            K_rows = k_rep[b, h]
            V_rows = v_rep[b, h]
            for t in range(T):
                if t >= n_new[b]:
                    continue  # padded query slot: stays zero
                pos = query_position(int(lens[b]), int(n_new[b]), t)
                if parents is not None:
                    prior = int(lens[b] - n_new[b])
                    keys = list(range(prior)) + sorted(prior + u for u in tree_path(parents[b], t))
                    out[b, h, t] = attend_slots(q[b, h, t], K_rows, V_rows, np.asarray(keys, dtype=np.int64))
                elif cache.window == 0 and not cache.ring:
                    out[b, h, t] = attend_one_query(q[b, h, t], K_rows, V_rows, pos)
                else:
                    slots = visible_slots(cache.pos[layer][b], int(lens[b]), pos, cache.window)
                    out[b, h, t] = attend_slots(q[b, h, t], K_rows, V_rows, slots)
    return out


def append_attention(cache: OracleCache, layer: int, q, k_new, v_new, n_new, parents=None) -> np.ndarray:
    """One call of the path: in-place append, then attention of the chunk."""
    if parents is not None:
        check_parents(np.asarray(parents, dtype=np.int64).reshape(cache.B, -1), np.asarray(k_new).shape[2])
    cache.append(layer, k_new, v_new, n_new)
    return gqa_attention(q, cache, layer, n_new, parents)


def decode_causal_mask(T: int, S: int) -> np.ndarray:
    """Bool [T, S], True where query i may see key j: j <= i + (S - T) (p2)."""
    q_pos = np.arange(S - T, S)[:, None]
    k_pos = np.arange(S)[None, :]
    return k_pos <= q_pos


def decode_window_mask(T: int, S: int, W: int) -> np.ndarray:
    """Bool [T, S] with a sliding window: (S - T) + i - W < j <= (S - T) + i (p2)."""
    q_pos = np.arange(S - T, S)[:, None]
    k_pos = np.arange(S)[None, :]
    return (k_pos <= q_pos) & (k_pos > q_pos - W)


def top_left_causal_mask(T: int, S: int) -> np.ndarray:
    """The wrong convention p2 warns about: tril(ones(T, S)), aligned top-left."""
    return np.tril(np.ones((T, S), dtype=bool))


def kv_cache_bytes(layers: int, batch: int, tokens: int, kv_heads: int, head_dim: int, bytes_per_value: int = 2) -> int:
    """2 (K and V) x layers x batch x tokens x Hkv x d x bytes (p3 "How big is the cache?")."""
    return 2 * layers * batch * tokens * kv_heads * head_dim * bytes_per_value


class PagedOracleCache:
    """K/V in pages [num_pages, Hkv, P, d] per layer behind a block table.

    ``table[b, i]`` is the physical page of row b's tokens i*P .. i*P+P-1
    (-1: not mapped).  Each row holds up to max_pages_per_row * P tokens.
    """

    def __init__(self, layers, batch, kv_heads, page_size, num_pages, max_pages_per_row, head_dim):
        if min(layers, kv_heads, page_size, num_pages, max_pages_per_row, head_dim) < 1 or batch < 0:
            raise CacheError("bad paged geometry")
        self.layers, self.B, self.Hkv, self.d = layers, batch, kv_heads, head_dim
        self.P, self.num_pages, self.mpr = page_size, num_pages, max_pages_per_row
        self.max_len = max_pages_per_row * page_size
        shape = (num_pages, kv_heads, page_size, head_dim)
        self.k = [np.zeros(shape, dtype=np.float64) for _ in range(layers)]
        self.v = [np.zeros(shape, dtype=np.float64) for _ in range(layers)]
        self.lens = np.zeros((layers, batch), dtype=np.int64)
        self.table = np.full((batch, max_pages_per_row), -1, dtype=np.int64)
        self.window = 0

    def set_block_table(self, table) -> None:
        table = np.asarray(table, dtype=np.int64).reshape(self.B, self.mpr)
        if np.any(table < -1) or np.any(table >= self.num_pages):
            raise CacheError("block table entry outside -1..num_pages-1")
        self.table = table.copy()

    def page_of(self, b: int, position: int) -> tuple:
        """(physical page, offset) of row b's token at a logical position."""
        return int(self.table[b, position // self.P]), position % self.P

    def append(self, layer, k_new, v_new, n_new) -> None:
        """Write row b's chunk at logical positions lens .. lens+n_new-1 through the table.

        Every row is checked first (n_new in 0..T, capacity, every target page
        mapped); nothing is written on error.
        """
        k_new, v_new = np.asarray(k_new), np.asarray(v_new)
        T = k_new.shape[2]
        n_new = np.asarray(n_new, dtype=np.int64).reshape(-1)
        lens = self.lens[layer]
        for b in range(self.B):
            if n_new[b] < 0 or n_new[b] > T:
                raise CacheError(f"row {b}: n_new={n_new[b]} outside 0..{T}")
            if lens[b] + n_new[b] > self.max_len:
                raise CacheError(f"row {b}: {lens[b] + n_new[b]} tokens > capacity {self.max_len}")
            for a in range(int(lens[b]), int(lens[b] + n_new[b])):
                if self.page_of(b, a)[0] < 0:
                    raise CacheError(f"row {b}: position {a} falls in an unmapped page")
        for b in range(self.B):
            for t in range(int(n_new[b])):
                page, off = self.page_of(b, int(lens[b]) + t)
                self.k[layer][page, :, off] = k_new[b, :, t]
                self.v[layer][page, :, off] = v_new[b, :, t]
        self.lens[layer] = lens + n_new

    def view(self, layer: int) -> OracleCache:
        """An ordinary cache holding every row's logical sequence, gathered through the table."""
        c = OracleCache(1, self.B, self.Hkv, self.max_len, self.d)
        c.set_window(self.window)
        for b in range(self.B):
            for a in range(int(self.lens[layer, b])):
                page, off = self.page_of(b, a)
                c.k[0][b, :, a] = self.k[layer][page, :, off]
                c.v[0][b, :, a] = self.v[layer][page, :, off]
                c.pos[0][b, a] = a
        c.lens[0] = self.lens[layer]
        return c


def paged_append_attention(cache: PagedOracleCache, layer: int, q, k_new, v_new, n_new, parents=None) -> np.ndarray:
    """One call on a paged cache: append through the table, then attention on the logical view."""
    if parents is not None:
        check_parents(np.asarray(parents, dtype=np.int64).reshape(cache.B, -1), np.asarray(k_new).shape[2])
    cache.append(layer, k_new, v_new, n_new)
    return gqa_attention(q, cache.view(layer), 0, n_new, parents)
