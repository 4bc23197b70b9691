"""Python binding: argument marshalling over the libkvc C ABI.

Every step of the path runs in libkvc's kernels; this module only allocates
device memory through PyTorch, checks tensor shapes, and passes raw pointers,
host length arrays and the current CUDA stream.

The API mirrors the pages' ``KVCache.append`` / ``gqa_attention``
("Implement grouped-query attention over a preallocated KV cache...",
"A strong answer") and ``truncate`` / ``reset`` / ``length`` ("16. Prefill,
decode and the KV cache", "Layout and validity").
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from ._lib import KVC_BF16, KVC_F32, KVC_FP8_E4M3, KVCError, check, lib

_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)

# storage dtype -> library dtype; an FP8 E4M3 cache takes bf16 q / k_new / v_new / out
_DTYPES = {torch.float32: KVC_F32, torch.bfloat16: KVC_BF16, torch.float8_e4m3fn: KVC_FP8_E4M3}


def _stream_ptr(device: torch.device, stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _i32(a, n: int) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int64).reshape(-1))
    if arr.shape[0] != n:
        raise KVCError(1, f"expected {n} per-row entries, got {arr.shape[0]}")
    if np.any(arr > np.iinfo(np.int32).max) or np.any(arr < np.iinfo(np.int32).min):
        raise KVCError(1, "per-row entry out of int32 range")
    return arr.astype(np.int32)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


class KVCache:
    """Preallocated K/V buffers [B, Hkv, max_len, d] per layer plus the C handle.

    ``k_bufs`` / ``v_bufs`` may be given (lists of contiguous CUDA tensors of
    that shape); otherwise they are allocated here with ``torch.empty``.  The
    handle borrows them; this object keeps them alive.
    """

    def __init__(self, layers: int, batch: int, kv_heads: int, max_len: int, head_dim: int,
                 dtype: torch.dtype = torch.bfloat16, device="cuda", k_bufs=None, v_bufs=None):
        if dtype not in _DTYPES:
            raise KVCError(1, f"unsupported dtype {dtype}")
        self.layers, self.B, self.Hkv, self.max_len, self.d = layers, batch, kv_heads, max_len, head_dim
        self.dtype = dtype
        self.io_dtype = torch.bfloat16 if dtype == torch.float8_e4m3fn else dtype
        dev = torch.device(device)
        if dev.type == "cuda" and dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        shape = (batch, kv_heads, max_len, head_dim)
        if k_bufs is None:
            k_bufs = [torch.empty(shape, dtype=dtype, device=self.device) for _ in range(layers)]
        if v_bufs is None:
            v_bufs = [torch.empty(shape, dtype=dtype, device=self.device) for _ in range(layers)]
        for t in list(k_bufs) + list(v_bufs):
            if tuple(t.shape) != shape or t.dtype != dtype or not t.is_contiguous():
                raise KVCError(1, f"cache buffers must be contiguous {shape} {dtype}")
        self.k, self.v = list(k_bufs), list(v_bufs)
        kp = (ctypes.c_void_p * layers)(*[t.data_ptr() for t in self.k])
        vp = (ctypes.c_void_p * layers)(*[t.data_ptr() for t in self.v])
        h = ctypes.c_void_p()
        check(lib().kvc_create(ctypes.byref(h), layers, batch, kv_heads, max_len, head_dim, _DTYPES[dtype], kp, vp))
        self._h = h
        self._ws = None
        self._dev_lens = None

    # ------------------------------------------------------------------ state
    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().kvc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def lens(self, layer: int = 0) -> np.ndarray:
        out = np.zeros(self.B, dtype=np.int64)
        check(lib().kvc_get_lens(self._h, layer, out.ctypes.data_as(_I64P)))
        return out

    def set_lens(self, layer: int, lens) -> None:
        """Adopt lengths for a layer whose buffers were filled by other means."""
        arr = np.ascontiguousarray(np.asarray(lens, dtype=np.int64).reshape(-1))
        if arr.shape[0] != self.B:
            raise KVCError(1, f"expected {self.B} lengths")
        check(lib().kvc_set_lens(self._h, layer, arr.ctypes.data_as(_I64P)))

    def length(self) -> np.ndarray:
        """Per-row length shared by every layer; raises if a forward pass stopped part-way."""
        out = np.zeros(self.B, dtype=np.int64)
        check(lib().kvc_length(self._h, out.ctypes.data_as(_I64P)))
        return out

    def truncate(self, new_lens) -> None:
        arr = np.ascontiguousarray(np.asarray(new_lens, dtype=np.int64).reshape(-1))
        if arr.shape[0] != self.B:
            raise KVCError(1, f"expected {self.B} lengths")
        check(lib().kvc_truncate(self._h, arr.ctypes.data_as(_I64P)))

    def reset(self) -> None:
        check(lib().kvc_reset(self._h))

    def set_kv_scales(self, layer: int, k_scale, v_scale) -> None:
        """One K and one V scale per KV head of an FP8 E4M3 cache's layer (only while it is empty)."""
        ks = np.ascontiguousarray(np.asarray(k_scale, dtype=np.float32).reshape(-1))
        vs = np.ascontiguousarray(np.asarray(v_scale, dtype=np.float32).reshape(-1))
        if ks.shape[0] != self.Hkv or vs.shape[0] != self.Hkv:
            raise KVCError(1, f"k_scale and v_scale need {self.Hkv} entries")
        fp = ctypes.POINTER(ctypes.c_float)
        check(lib().kvc_set_kv_scales(self._h, layer, ks.ctypes.data_as(fp), vs.ctypes.data_as(fp)))

    def set_window(self, window: int, ring: bool = False) -> None:
        """Sliding window (0 = none) and ring storage (slot = position mod max_len), for every layer."""
        check(lib().kvc_set_window(self._h, int(window), 1 if ring else 0))

    def kernel_launches(self) -> int:
        """Kernels this cache's handle has enqueued so far."""
        return int(lib().kvc_kernel_launches(self._h))

    # ------------------------------------------------------------------ compute
    def workspace_bytes(self, q_heads: int, T: int) -> int:
        return int(lib().kvc_workspace_bytes(self._h, q_heads, T))

    def workspace(self, q_heads: int, T: int) -> torch.Tensor | None:
        """A workspace buffer owned by this cache, grown as needed (reused across calls).

        Allocated zeroed, so its error word reads clean (device_status) even
        before a call has used it.
        """
        need = self.workspace_bytes(q_heads, T)
        if need == 0:
            return None
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(need, dtype=torch.uint8, device=self.device)
        return self._ws

    def _check_tensor(self, t: torch.Tensor, shape, name: str) -> None:
        if tuple(t.shape) != tuple(shape) or t.dtype != self.io_dtype or not t.is_contiguous() or t.device != self.device:
            raise KVCError(1, f"{name} must be a contiguous {self.io_dtype} tensor of shape {tuple(shape)} on {self.device}")

    def append(self, layer: int, k_new: torch.Tensor, v_new: torch.Tensor, n_new, stream=None) -> None:
        """Write k_new[b, :, :n_new[b]] at each row's current length (in place)."""
        T = k_new.shape[2] if k_new.dim() == 4 else -1
        self._check_tensor(k_new, (self.B, self.Hkv, T, self.d), "k_new")
        self._check_tensor(v_new, (self.B, self.Hkv, T, self.d), "v_new")
        nn = _i32(n_new, self.B)
        check(lib().kvc_append(self._h, layer, _ptr(k_new), _ptr(v_new), T, nn.ctypes.data_as(_I32P),
                               _stream_ptr(self.device, stream)))

    def gqa_attention(self, layer: int, q: torch.Tensor, n_new, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Attention of the chunk just appended: q [B, Hq, T, d] -> out [B, Hq, T, d]."""
        if q.dim() != 4:
            raise KVCError(1, "q must be [B, Hq, T, d]")
        B, Hq, T, d = q.shape
        self._check_tensor(q, (self.B, Hq, T, self.d), "q")
        if out is None:
            out = torch.empty_like(q)
        self._check_tensor(out, q.shape, "out")
        ws = workspace if workspace is not None else self.workspace(Hq, T)
        nn = _i32(n_new, self.B)
        check(lib().kvc_gqa_attention(self._h, layer, _ptr(q), Hq, T, nn.ctypes.data_as(_I32P), _ptr(out),
                                      _ptr(ws), 0 if ws is None else ws.numel(), _stream_ptr(self.device, stream)))
        return out

    def gqa_attention_noalloc(self, layer: int, q: torch.Tensor, n_new, out: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
        """``gqa_attention`` through the allocation-free entry point (library-owned static scratch).

        For callers that cannot allocate device memory, so ``out`` must be
        passed in: this wrapper allocates nothing either (``out=None`` raises).
        Shapes whose scratch exceeds the static array are rejected.  Errors of
        the kernels stay recorded in the scratch until ``noalloc_status``.
        """
        if q.dim() != 4:
            raise KVCError(1, "q must be [B, Hq, T, d]")
        B, Hq, T, d = q.shape
        self._check_tensor(q, (self.B, Hq, T, self.d), "q")
        if out is None:
            raise KVCError(1, "the allocation-free call takes a caller-owned out tensor (out is None)")
        self._check_tensor(out, q.shape, "out")
        nn = _i32(n_new, self.B)
        check(lib().kvc_gqa_attention_noalloc(self._h, layer, _ptr(q), Hq, T, nn.ctypes.data_as(_I32P), _ptr(out),
                                              _stream_ptr(self.device, stream)))
        return out

    def append_attention(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, n_new,
                         out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
        """Append then attend, validated together (an error runs neither step)."""
        if q.dim() != 4:
            raise KVCError(1, "q must be [B, Hq, T, d]")
        B, Hq, T, d = q.shape
        self._check_tensor(q, (self.B, Hq, T, self.d), "q")
        self._check_tensor(k_new, (self.B, self.Hkv, T, self.d), "k_new")
        self._check_tensor(v_new, (self.B, self.Hkv, T, self.d), "v_new")
        if out is None:
            out = torch.empty_like(q)
        self._check_tensor(out, q.shape, "out")
        ws = workspace if workspace is not None else self.workspace(Hq, T)
        nn = _i32(n_new, self.B)
        check(lib().kvc_append_attention(self._h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), Hq, T,
                                         nn.ctypes.data_as(_I32P), _ptr(out), _ptr(ws),
                                         0 if ws is None else ws.numel(), _stream_ptr(self.device, stream)))
        return out

    def append_attention_host(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, n_new,
                              out: torch.Tensor, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """``append_attention`` on CPU tensors (page-locked for the copies to overlap).

        The library copies positions t < n_new[b] of q, k_new and v_new to its
        own device staging, runs the step on ``stream`` and copies those
        positions of out back; out's other positions are left as they were.
        Returns once enqueued: after ``host_copies_done`` and a synchronize of
        that stream, ``out`` holds the result and the inputs may change.
        """
        if q.dim() != 4:
            raise KVCError(1, "q must be [B, Hq, T, d]")
        B, Hq, T, d = q.shape
        for t, shape, name in ((q, (self.B, Hq, T, self.d), "q"), (k_new, (self.B, self.Hkv, T, self.d), "k_new"),
                               (v_new, (self.B, self.Hkv, T, self.d), "v_new"), (out, (self.B, Hq, T, self.d), "out")):
            if tuple(t.shape) != shape or t.dtype != self.io_dtype or not t.is_contiguous() or t.device.type != "cpu":
                raise KVCError(1, f"{name} must be a contiguous {self.io_dtype} CPU tensor of shape {shape}")
        ws = workspace if workspace is not None else self.workspace(Hq, T)
        nn = _i32(n_new, self.B)
        check(lib().kvc_append_attention_host(self._h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), Hq, T,
                                              nn.ctypes.data_as(_I32P), _ptr(out), _ptr(ws),
                                              0 if ws is None else ws.numel(), _stream_ptr(self.device, stream)))
        return out

    def host_copies_done(self, stream=None) -> None:
        """Make ``stream`` wait for every output copy of the host-buffer calls enqueued so far."""
        check(lib().kvc_host_copies_done(self._h, _stream_ptr(self.device, stream)))

    # ------------------------------------------------ device-resident lengths
    def lens_to_device(self, stream=None) -> torch.Tensor:
        """Hand the lengths over to a device array (int32 [layers, B]) owned by this object.

        Until ``lens_from_device``, only ``decode_step`` may run: it reads and
        advances the device lengths, so a step can be captured in a CUDA graph.
        """
        n = int(lib().kvc_device_lens_bytes(self._h)) // 4
        self._dev_lens = torch.zeros(max(n, 1), dtype=torch.int32, device=self.device)
        check(lib().kvc_lens_to_device(self._h, self._dev_lens.data_ptr(), _stream_ptr(self.device, stream)))
        return self._dev_lens[:n].view(self.layers, self.B)

    def lens_from_device(self, stream=None) -> None:
        """Make the host lengths authoritative again (copies the device lengths back)."""
        check(lib().kvc_lens_from_device(self._h, _stream_ptr(self.device, stream)))

    def decode_step(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    n_new: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, stream=None) -> torch.Tensor:
        """``append_attention`` with the lengths on the device and ``n_new`` a device int32 [B].

        Nothing per-step comes from the host, so the call can be captured in a
        CUDA graph; ``out`` and ``workspace`` must be passed in.
        """
        if q.dim() != 4:
            raise KVCError(1, "q must be [B, Hq, T, d]")
        B, Hq, T, d = q.shape
        self._check_tensor(q, (self.B, Hq, T, self.d), "q")
        self._check_tensor(k_new, (self.B, self.Hkv, T, self.d), "k_new")
        self._check_tensor(v_new, (self.B, self.Hkv, T, self.d), "v_new")
        self._check_tensor(out, q.shape, "out")
        if n_new.dtype != torch.int32 or n_new.device != self.device or n_new.numel() != self.B or not n_new.is_contiguous():
            raise KVCError(1, f"n_new must be a contiguous int32 tensor of {self.B} entries on {self.device}")
        check(lib().kvc_decode_step(self._h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), Hq, T, n_new.data_ptr(),
                                    _ptr(out), _ptr(workspace), workspace.numel(), _stream_ptr(self.device, stream)))
        return out

    def append_attention_tree(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, n_new,
                              parents, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
        """``append_attention`` for a draft tree: parents [B, T] (-1 = off the cached prefix)."""
        if q.dim() != 4:
            raise KVCError(1, "q must be [B, Hq, T, d]")
        B, Hq, T, d = q.shape
        self._check_tensor(q, (self.B, Hq, T, self.d), "q")
        self._check_tensor(k_new, (self.B, self.Hkv, T, self.d), "k_new")
        self._check_tensor(v_new, (self.B, self.Hkv, T, self.d), "v_new")
        if out is None:
            out = torch.empty_like(q)
        self._check_tensor(out, q.shape, "out")
        ws = workspace if workspace is not None else self.workspace(Hq, T)
        nn = _i32(n_new, self.B)
        par = _i32(parents, self.B * T)
        check(lib().kvc_append_attention_tree(self._h, layer, _ptr(q), _ptr(k_new), _ptr(v_new), Hq, T,
                                              nn.ctypes.data_as(_I32P), par.ctypes.data_as(_I32P), _ptr(out),
                                              _ptr(ws), 0 if ws is None else ws.numel(),
                                              _stream_ptr(self.device, stream)))
        return out

    def gqa_attention_tree(self, layer: int, q: torch.Tensor, n_new, parents, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """``gqa_attention`` of a chunk already appended, for a draft tree (parents [B, T])."""
        if q.dim() != 4:
            raise KVCError(1, "q must be [B, Hq, T, d]")
        B, Hq, T, d = q.shape
        self._check_tensor(q, (self.B, Hq, T, self.d), "q")
        if out is None:
            out = torch.empty_like(q)
        self._check_tensor(out, q.shape, "out")
        ws = workspace if workspace is not None else self.workspace(Hq, T)
        nn = _i32(n_new, self.B)
        par = _i32(parents, self.B * T)
        check(lib().kvc_gqa_attention_tree(self._h, layer, _ptr(q), Hq, T, nn.ctypes.data_as(_I32P),
                                           par.ctypes.data_as(_I32P), _ptr(out), _ptr(ws),
                                           0 if ws is None else ws.numel(), _stream_ptr(self.device, stream)))
        return out

    def selftest_bounded_wait(self, limit_ns: int, workspace: torch.Tensor | None = None, stream=None) -> None:
        """Launch the bounded-wait self-test into the workspace's error word."""
        ws = workspace if workspace is not None else self._ws
        if ws is None:
            raise KVCError(7, "no workspace")
        check(lib().kvc_selftest_bounded_wait(_ptr(ws), int(limit_ns), _stream_ptr(self.device, stream)))

    def noalloc_status(self, stream=None) -> int:
        """Synchronize and read the allocation-free calls' error word (0 = clean); raises on a non-zero code."""
        code = ctypes.c_int32(0)
        check(lib().kvc_noalloc_status(_stream_ptr(self.device, stream), ctypes.byref(code)))
        return code.value

    def device_status(self, workspace: torch.Tensor | None = None, stream=None) -> int:
        """Synchronize and read the workspace error word (0 = clean); raises on a non-zero code."""
        ws = workspace if workspace is not None else self._ws
        if ws is None:
            return 0
        code = ctypes.c_int32(0)
        check(lib().kvc_device_status(self._h, _ptr(ws), _stream_ptr(self.device, stream), ctypes.byref(code)))
        return code.value


class PagedKVCache(KVCache):
    """K/V in pages [num_pages, Hkv, page_size, d] per layer behind a device block table.

    ``block_table`` (int32 [B, max_pages_per_row], on the device, owned by
    this object) maps row b's logical page i to a physical page; it starts as
    row b owning pages b * max_pages_per_row .. (as long as num_pages allows,
    else -1) and may be rewritten between calls.  Every call works on the
    logical sequence, with max_len = max_pages_per_row * page_size.
    """

    def __init__(self, layers: int, batch: int, kv_heads: int, page_size: int, num_pages: int,
                 max_pages_per_row: int, head_dim: int, dtype: torch.dtype = torch.bfloat16, device="cuda"):
        if dtype not in _DTYPES:
            raise KVCError(1, f"unsupported dtype {dtype}")
        dev = torch.device(device)
        if dev.type == "cuda" and dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.layers, self.B, self.Hkv, self.d = layers, batch, kv_heads, head_dim
        self.page_size, self.num_pages, self.max_pages_per_row = page_size, num_pages, max_pages_per_row
        self.max_len = max_pages_per_row * page_size
        self.dtype, self.device = dtype, dev
        self.io_dtype = torch.bfloat16 if dtype == torch.float8_e4m3fn else dtype
        shape = (num_pages, kv_heads, page_size, head_dim)
        self.k = [torch.empty(shape, dtype=dtype, device=dev) for _ in range(layers)]
        self.v = [torch.empty(shape, dtype=dtype, device=dev) for _ in range(layers)]
        ids = torch.arange(batch * max_pages_per_row, dtype=torch.int32, device=dev)
        self.block_table = torch.where(ids < num_pages, ids, torch.full_like(ids, -1)).view(batch, max_pages_per_row)
        kp = (ctypes.c_void_p * layers)(*[t.data_ptr() for t in self.k])
        vp = (ctypes.c_void_p * layers)(*[t.data_ptr() for t in self.v])
        h = ctypes.c_void_p()
        check(lib().kvc_create_paged(ctypes.byref(h), layers, batch, kv_heads, page_size, num_pages,
                                     max_pages_per_row, head_dim, _DTYPES[dtype], kp, vp,
                                     self.block_table.data_ptr()))
        self._h = h
        self._ws = None
        self._dev_lens = None


def gqa_attention(q: torch.Tensor, cache: KVCache, n_new, layer: int = 0, **kw) -> torch.Tensor:
    """Module-level form of ``KVCache.gqa_attention`` (the pages' call signature)."""
    return cache.gqa_attention(layer, q, n_new, **kw)
